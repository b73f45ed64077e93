// Pre-pass for an explicit boolean mask ("masked multi head attention in
// CUDA", section 2.2: a [B, N, N] matrix of kept / removed positions), run
// once per call before the attention kernel.
//
// The attention kernel reads the mask in the form it needs:
//   * bits: one bit per (b, query row, key), 16 bytes per (row, 128-key tile),
//     so a softmax thread fetches its 64 keys of a tile in one 8-byte load
//     instead of 64 bytes;
//   * flags: per (b, 128-row block, 128-key tile) 0 = no kept position (the
//     tile is skipped: no loads, no MMAs, no exponentials), 1 = every
//     position kept (no masking work), 2 = partial (the bits are applied);
//   * last: per (b, 128-row block) the last tile with a kept position, or -1
//     (a block with none writes O = 0 and LSE = -inf without the tensor core).
//
// One CTA of 128 threads per (b, row block, key tile); warp w packs rows
// w, w + 4, ...: for each row its 32 lanes read 32 consecutive mask bytes at a
// time (coalesced, any alignment and strides) and a ballot makes a 32-bit
// word.  HBM-bound: one byte read per mask element.
#include <stdint.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kTile = 128;
constexpr int kMaskThreads = 128;

__global__ void __launch_bounds__(kMaskThreads)
    mask_pack_kernel(const uint8_t* __restrict__ mask, int64_t sb, int64_t sr, int Lq, int Lk,
                     int n_mb, int n_kt, uint32_t* __restrict__ bits, uint8_t* __restrict__ flags,
                     int* __restrict__ last) {
  const int t = static_cast<int>(blockIdx.x) % n_kt;  // key tile
  const int mb = (static_cast<int>(blockIdx.x) / n_kt) % n_mb;
  const int b = static_cast<int>(blockIdx.x) / (n_kt * n_mb);
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x) & 31;
  bool any = false, all = true;  // over the kept / in-range positions of this warp's rows
  for (int r = warp; r < kTile; r += kMaskThreads / 32) {
    const int row = mb * kTile + r;
    if (row >= Lq) break;
    const uint8_t* src = mask + b * sb + static_cast<int64_t>(row) * sr;
    uint32_t word[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int key = t * kTile + q * 32 + lane;
      const bool in = key < Lk;
      word[q] = __ballot_sync(0xffffffffu, in && src[key] != 0);
      const uint32_t in_range = __ballot_sync(0xffffffffu, in);
      any = any || word[q] != 0u;
      all = all && word[q] == in_range;
    }
    if (lane < 4) {
      const uint32_t v = lane == 0 ? word[0] : lane == 1 ? word[1] : lane == 2 ? word[2] : word[3];
      bits[((static_cast<int64_t>(b) * Lq + row) * n_kt + t) * 4 + lane] = v;
    }
  }
  any = __syncthreads_or(any ? 1 : 0) != 0;
  all = __syncthreads_and(all ? 1 : 0) != 0;
  if (threadIdx.x == 0) {
    flags[(static_cast<int64_t>(b) * n_mb + mb) * n_kt + t] = !any ? 0 : (all ? 1 : 2);
    if (any) atomicMax(last + static_cast<int64_t>(b) * n_mb + mb, t);
  }
}

struct MaskSizes {
  int64_t n_mb, n_kt, bits, flags, last;
};

MaskSizes sizes(const Problem& p) {
  MaskSizes z;
  z.n_mb = (p.Lq + kTile - 1) / kTile;
  z.n_kt = (p.Lk + kTile - 1) / kTile;
  z.bits = static_cast<int64_t>(p.B) * p.Lq * z.n_kt * 16;
  z.flags = (static_cast<int64_t>(p.B) * z.n_mb * z.n_kt + 15) / 16 * 16;
  z.last = static_cast<int64_t>(p.B) * z.n_mb * 4;
  return z;
}

}  // namespace

int64_t mask_workspace_bytes(const Problem& p) {
  const MaskSizes z = sizes(p);
  return z.bits + z.flags + z.last;
}

void mask_arrays(Problem& p, void* ws) {
  const MaskSizes z = sizes(p);
  uint8_t* base = static_cast<uint8_t*>(ws);
  p.mbits = reinterpret_cast<const uint32_t*>(base);
  p.mflags = base + z.bits;
  p.mlast = reinterpret_cast<const int*>(base + z.bits + z.flags);
}

cudaError_t launch_mask_pack(const Problem& p) {
  const MaskSizes z = sizes(p);
  const int64_t blocks = static_cast<int64_t>(p.B) * z.n_mb * z.n_kt;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  // every block's last tile starts at -1 (all bytes 0xFF)
  cudaError_t e = cudaMemsetAsync(const_cast<int*>(p.mlast), 0xFF, static_cast<size_t>(z.last), p.stream);
  if (e != cudaSuccess) return e;
  mask_pack_kernel<<<static_cast<unsigned>(blocks), kMaskThreads, 0, p.stream>>>(
      p.mask, p.mask_sb, p.mask_sr, p.Lq, p.Lk, static_cast<int>(z.n_mb), static_cast<int>(z.n_kt),
      const_cast<uint32_t*>(p.mbits), const_cast<uint8_t*>(p.mflags), const_cast<int*>(p.mlast));
  return cudaGetLastError();
}

}  // namespace attn
