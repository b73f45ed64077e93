// Pre-pass for an explicit boolean mask ("masked multi head attention in
// CUDA", section 2.2: a [B, N, N] matrix of kept / removed positions), run
// once per call before the attention kernel.
//
// The attention kernel reads the mask in the form it needs:
//   * bits: one bit per (mask batch, query row, key), 16 bytes per (row,
//     128-key tile), so a softmax thread fetches its 64 keys of a tile in one
//     8-byte load instead of 64 bytes;
//   * vis / part: per (mask batch, 128-row block) one bit per 128-key tile in
//     32-bit words: vis = the tile has a kept position (tiles without one are
//     skipped: no loads, no MMAs, no exponentials), part = some but not all
//     positions are kept (the bits are applied; a full tile needs no masking
//     work).  Every role of the attention kernel walks the visited tiles from
//     these words, 32 tiles per load;
//   * last: per (mask batch, 128-row block) the last visited tile, or -1 (a
//     block with none writes O = 0 and LSE = -inf without the tensor core).
// A mask shared by every batch (batch stride 0) is packed once.
//
// One CTA of 128 threads per (mask batch, row block, key tile).  When the
// rows are 16-byte aligned, lane l of a warp reads 16 bytes of row 4i + l/8
// (four whole 128-byte rows per warp load); otherwise 32 lanes read 32
// consecutive bytes of one row at a time.  HBM-bound: one byte read per mask
// element.
#include <stdint.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kTile = 128;
constexpr int kMaskThreads = 128;

// 4-bit mask of the non-zero bytes of w (bit i: byte i, the lowest first).
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t w) {
  const uint32_t m = __vcmpne4(w, 0u) & 0x08040201u;  // byte i -> bit i of that byte
  return (m * 0x01010101u) >> 24;                        // sum of the four bytes
}

__global__ void __launch_bounds__(kMaskThreads)
    mask_pack_kernel(const uint8_t* __restrict__ mask, int64_t sb, int64_t sr, int Lq, int Lk,
                     int n_mb, int n_kt, int n_ch, bool vec, uint32_t* __restrict__ bits,
                     uint32_t* __restrict__ vis, uint32_t* __restrict__ part,
                     int* __restrict__ last) {
  const int t = static_cast<int>(blockIdx.x) % n_kt;  // key tile
  const int mb = (static_cast<int>(blockIdx.x) / n_kt) % n_mb;
  const int b = static_cast<int>(blockIdx.x) / (n_kt * n_mb);  // mask batch
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const int k0 = t * kTile;
  // in-range keys of this tile, as four 32-bit words (bit c of word w: key k0 + 32w + c)
  auto in_range = [&](int wd) -> uint32_t {
    const int n = Lk - (k0 + 32 * wd);
    return n >= 32 ? 0xFFFFFFFFu : (n <= 0 ? 0u : ((1u << n) - 1u));
  };
  bool any = false, all = true;  // over the in-range positions of this warp's rows
  if (vec) {
    // lane l: row 4i + l/8 of the warp's 32-row group, bytes 16(l%8) .. +15
    const int sub = lane & 7;
    for (int i = 0; i < 8; ++i) {
      const int r = warp * 32 + i * 4 + (lane >> 3);
      const int row = mb * kTile + r;
      const bool row_in = row < Lq;
      const int key = k0 + 16 * sub;
      uint32_t m16 = 0;  // bit c: key key + c kept
      if (row_in) {
        const uint8_t* src = mask + b * sb + static_cast<int64_t>(row) * sr + key;
        if (key + 16 <= Lk) {
          const uint4 x = *reinterpret_cast<const uint4*>(src);
          m16 = nonzero_bytes(x.x) | (nonzero_bytes(x.y) << 4) | (nonzero_bytes(x.z) << 8) |
                (nonzero_bytes(x.w) << 12);
        } else {
          for (int c = 0; c < 16 && key + c < Lk; ++c) m16 |= (src[c] != 0 ? 1u : 0u) << c;
        }
      }
      // the word of keys 32(sub/2) .. +31: this lane's 16 bits and its neighbour's
      const uint32_t other = __shfl_xor_sync(0xffffffffu, m16, 1);
      const uint32_t word = (sub & 1) ? (other | (m16 << 16)) : (m16 | (other << 16));
      if (row_in && (sub & 1) == 0) {
        const int wd = sub >> 1;
        bits[((static_cast<int64_t>(b) * Lq + row) * n_kt + t) * 4 + wd] = word;
        any = any || word != 0u;
        all = all && word == in_range(wd);
      }
    }
  } else {
    // warp w: rows w, w + 4, ...; 32 lanes read 32 consecutive bytes of one row
    for (int r = warp; r < kTile; r += kMaskThreads / 32) {
      const int row = mb * kTile + r;
      if (row >= Lq) break;
      const uint8_t* src = mask + b * sb + static_cast<int64_t>(row) * sr;
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        const int key = k0 + wd * 32 + lane;
        const uint32_t word = __ballot_sync(0xffffffffu, key < Lk && src[key] != 0);
        if (lane == wd) bits[((static_cast<int64_t>(b) * Lq + row) * n_kt + t) * 4 + wd] = word;
        any = any || word != 0u;
        all = all && word == in_range(wd);
      }
    }
  }
  any = __syncthreads_or(any ? 1 : 0) != 0;
  all = __syncthreads_and(all ? 1 : 0) != 0;
  if (threadIdx.x == 0 && any) {
    const int64_t blk = static_cast<int64_t>(b) * n_mb + mb;
    atomicOr(vis + blk * n_ch + t / 32, 1u << (t % 32));
    if (!all) atomicOr(part + blk * n_ch + t / 32, 1u << (t % 32));
    atomicMax(last + blk, t);
  }
}

struct MaskSizes {
  int64_t mB, n_mb, n_kt, n_ch, bits, words, last;
};

MaskSizes sizes(const Problem& p) {
  MaskSizes z;
  z.mB = p.mask_sb == 0 ? 1 : p.B;  // a shared mask is packed once
  z.n_mb = (p.Lq + kTile - 1) / kTile;
  z.n_kt = (p.Lk + kTile - 1) / kTile;
  z.n_ch = (z.n_kt + 31) / 32;
  z.bits = z.mB * p.Lq * z.n_kt * 16;
  z.words = z.mB * z.n_mb * z.n_ch * 4;  // vis, then part
  z.last = z.mB * z.n_mb * 4;
  return z;
}

}  // namespace

int64_t mask_workspace_bytes(const Problem& p) {
  const MaskSizes z = sizes(p);
  return z.bits + 2 * z.words + z.last;
}

void mask_arrays(Problem& p, void* ws) {
  const MaskSizes z = sizes(p);
  uint8_t* base = static_cast<uint8_t*>(ws);
  p.mbits = reinterpret_cast<const uint32_t*>(base);
  p.mvis = reinterpret_cast<const uint32_t*>(base + z.bits);
  p.mpart = reinterpret_cast<const uint32_t*>(base + z.bits + z.words);
  p.mlast = reinterpret_cast<const int*>(base + z.bits + 2 * z.words);
}

cudaError_t launch_mask_pack(const Problem& p) {
  const MaskSizes z = sizes(p);
  const int64_t blocks = z.mB * z.n_mb * z.n_kt;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  // vis and part start empty (0), every block's last tile at -1 (bytes 0xFF)
  cudaError_t e = cudaMemsetAsync(const_cast<uint32_t*>(p.mvis), 0, static_cast<size_t>(2 * z.words),
                                  p.stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(const_cast<int*>(p.mlast), 0xFF, static_cast<size_t>(z.last), p.stream);
  if (e != cudaSuccess) return e;
  const bool vec = reinterpret_cast<uintptr_t>(p.mask) % 16 == 0 && p.mask_sr % 16 == 0 &&
                   p.mask_sb % 16 == 0;
  mask_pack_kernel<<<static_cast<unsigned>(blocks), kMaskThreads, 0, p.stream>>>(
      p.mask, p.mask_sb, p.mask_sr, p.Lq, p.Lk, static_cast<int>(z.n_mb), static_cast<int>(z.n_kt),
      static_cast<int>(z.n_ch), vec, const_cast<uint32_t*>(p.mbits), const_cast<uint32_t*>(p.mvis),
      const_cast<uint32_t*>(p.mpart), const_cast<int*>(p.mlast));
  return cudaGetLastError();
}

}  // namespace attn
