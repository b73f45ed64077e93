// Pre-pass for bf16 inputs: an exact fp16 copy of V, tile by tile.
//
// The attention kernel multiplies P (probabilities in [0, 1]) by V on the
// tensor core, and both operands of one MMA must have the same type.  With
// bf16 V that would force bf16 P (unit roundoff 2^-8), too coarse for rows
// dominated by a few keys.  An fp16 copy of V lets P be fp16 (unit roundoff
// 2^-11).  The copy is exact for every finite bf16 value with |v| < 2^16
// (bf16 keeps 8 significant bits, fp16 keeps 11, and the largest bf16 value
// below 2^16 is 65280 < 65504, the fp16 maximum); below 2^-14 fp16 is
// subnormal and the copy is within 2^-25 absolutely.  A 128-key tile with any
// value outside that range (|v| >= 2^16, inf, NaN) gets flag 0 and no copy:
// the attention kernel then reads the bf16 tile and splits P into two bf16
// terms instead.
//
// One CTA per (b*Hkv + h, 128-key tile): 256 threads hold the tile in
// registers (16-byte loads), vote on the range check, and write the fp16
// tile and its flag.  V may be strided (any batch, head and row strides that
// are multiples of 8 elements); the copy is always a contiguous
// [B, Hkv, Lk, D] tensor.  HBM-bound: reads 2 bytes and writes 2 bytes per
// element.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kTileKeys = 128;
constexpr int kThreadsV = 256;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Larger of the two bf16 exponent fields of a packed pair (sign dropped).
__device__ __forceinline__ uint32_t exp_max(uint32_t w) {
  const uint32_t e = w & 0x7F807F80u;
  return max(e & 0xFFFFu, e >> 16);
}

// Two bf16 values (one 32-bit word) -> two fp16 values; exact in range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D>
__global__ void __launch_bounds__(kThreadsV) v_to_f16_kernel(const uint16_t* __restrict__ v,
                                                             uint16_t* __restrict__ v16,
                                                             int* __restrict__ flags, int L,
                                                             int n_kt, int Hkv, Strides sv) {
  constexpr int kVecPerRow = D / 8;                 // 16-byte vectors per row
  constexpr int kPer = kTileKeys * kVecPerRow / kThreadsV;
  static_assert(kPer >= 1 && kPer * kThreadsV == kTileKeys * kVecPerRow, "tile / thread split");
  const int z = static_cast<int>(blockIdx.x) / n_kt;  // b*Hkv + h
  const int tile = static_cast<int>(blockIdx.x) % n_kt;
  const int r0 = tile * kTileKeys;
  const int rows = min(kTileKeys, L - r0);
  const int nvec = rows * kVecPerRow;
  // source: row r0 of head (b, h) of V, rows sv.l elements apart
  const uint16_t* src = v + (z / Hkv) * sv.b + (z % Hkv) * sv.h + static_cast<int64_t>(r0) * sv.l;
  // destination: the contiguous copy, in 16-byte vectors
  uint4* dst = reinterpret_cast<uint4*>(v16) + (static_cast<int64_t>(z) * L + r0) * D / 8;

  uint4 x[kPer];
  uint32_t ex = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int idx = static_cast<int>(threadIdx.x) + kThreadsV * i;
    const uint4* a = reinterpret_cast<const uint4*>(src + (idx / kVecPerRow) * sv.l) + idx % kVecPerRow;
    x[i] = idx < nvec ? ld_stream(a) : make_uint4(0u, 0u, 0u, 0u);
    ex = max(ex, max(max(exp_max(x[i].x), exp_max(x[i].y)), max(exp_max(x[i].z), exp_max(x[i].w))));
  }
  // exponent field 143 (0x4780) and above: |v| >= 2^16, inf or NaN
  const int bad = __syncthreads_or(ex >= 0x4780u ? 1 : 0);
  if (!bad) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int idx = static_cast<int>(threadIdx.x) + kThreadsV * i;
      if (idx < nvec) {
        dst[idx] = make_uint4(bf16x2_to_f16x2(x[i].x), bf16x2_to_f16x2(x[i].y),
                              bf16x2_to_f16x2(x[i].z), bf16x2_to_f16x2(x[i].w));
      }
    }
  }
  if (threadIdx.x == 0) flags[blockIdx.x] = bad ? 0 : 1;
}

}  // namespace

int64_t vconv_workspace_bytes(const Problem& p) {
  const int64_t n_kt = (p.Lk + kTileKeys - 1) / kTileKeys;
  const int64_t v_bytes = static_cast<int64_t>(p.B) * p.Hkv * p.Lk * p.D * 2;
  return v_bytes + static_cast<int64_t>(p.B) * p.Hkv * n_kt * 4;
}

cudaError_t launch_vconv(const Problem& p, void* v16, int* flags) {
  const int64_t n_kt = (p.Lk + kTileKeys - 1) / kTileKeys;
  const int64_t blocks = static_cast<int64_t>(p.B) * p.Hkv * n_kt;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  const auto* v = static_cast<const uint16_t*>(p.v);
  auto* out = static_cast<uint16_t*>(v16);
  if (p.D == 16) {
    v_to_f16_kernel<16><<<static_cast<unsigned>(blocks), kThreadsV, 0, p.stream>>>(
        v, out, flags, p.Lk, static_cast<int>(n_kt), p.Hkv, p.sv);
  } else if (p.D == 32) {
    v_to_f16_kernel<32><<<static_cast<unsigned>(blocks), kThreadsV, 0, p.stream>>>(
        v, out, flags, p.Lk, static_cast<int>(n_kt), p.Hkv, p.sv);
  } else if (p.D == 64) {
    v_to_f16_kernel<64><<<static_cast<unsigned>(blocks), kThreadsV, 0, p.stream>>>(
        v, out, flags, p.Lk, static_cast<int>(n_kt), p.Hkv, p.sv);
  } else if (p.D == 128) {
    v_to_f16_kernel<128><<<static_cast<unsigned>(blocks), kThreadsV, 0, p.stream>>>(
        v, out, flags, p.Lk, static_cast<int>(n_kt), p.Hkv, p.sv);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace attn
