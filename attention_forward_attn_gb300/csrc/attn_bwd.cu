// Backward of the attention forward, for the log-sum-exp the forward stores.
//
// tiny_flash_attn_triton.py keeps L = m + log2(l) per row "for the backward
// pass"; the pages give no backward algorithm, so this computes the
// derivative of O = softmax(sm_scale Q K^T) V from its definition, with the
// softmax rebuilt from the stored LSE instead of a second max/sum pass:
//   P_ij  = exp(sm_scale q_i.k_j - LSE_i)          (visible keys; 0 otherwise)
//   delta_i = dO_i . O_i                            (= sum_j P_ij dP_ij)
//   dP_ij = dO_i . v_j,   dS_ij = P_ij (dP_ij - delta_i)
//   dQ_i = sm_scale sum_j dS_ij k_j,   dK_j = sm_scale sum_i dS_ij q_i,
//   dV_j = sum_i P_ij dO_i
// with K/V of head h_kv = h_q / (Hq/Hkv) and dK, dV summed over its query heads.
//
// Three SIMT kernels, fp32 arithmetic (FMA units, no tensor cores), inputs
// converted from fp16/bf16 when they are staged in shared memory:
//   * delta: one warp per query row;
//   * dQ: one CTA per (b, h_q, 64-row query tile); K and V stream through
//     shared memory in 64-key tiles; S, dP and dS of a 64x64 block are
//     computed once (one element per thread pass) and dS is kept in shared
//     memory for the dQ product;
//   * dK/dV: one CTA per (b, h_kv, 64-key tile) with K and V resident; every
//     query head of the group and every query tile that sees the keys stream
//     through; P and dS of each block stay in shared memory, dK and dV
//     accumulate in registers and are written once (no atomics).
// Shared-memory rows are padded by one float, so that threads reading the
// same column of different rows hit different banks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kT = 64;          // rows of a query tile / keys of a key tile
constexpr int kThreadsBwd = 256;

template <bool BF16>
__device__ __forceinline__ float ld16(const void* base, int64_t idx) {
  if constexpr (BF16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  } else {
    return __half2float(reinterpret_cast<const __half*>(base)[idx]);
  }
}

template <bool BF16>
__device__ __forceinline__ void st16(void* base, int64_t idx, float x) {
  if constexpr (BF16) {
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
  } else {
    reinterpret_cast<__half*>(base)[idx] = __float2half_rn(x);
  }
}

struct BwdProblem {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* delta;  // [B*Hq, L] workspace
  const int32_t* valid_len;
  int B, Hq, Hkv, L;
  float scale;
  int causal;
};

__device__ __forceinline__ int kv_len_of(const BwdProblem& p, int b) {
  if (p.valid_len == nullptr) return p.L;
  const int vl = p.valid_len[b];
  return vl < 0 ? 0 : (vl > p.L ? p.L : vl);
}

// Stage `rows` rows of a [.., L, D] 16-bit head (row r0 onwards) into fp32
// shared memory with row stride D + 1; rows past L are zeros.
template <int D, bool BF16>
__device__ __forceinline__ void stage(float* dst, const void* src, int64_t head_row0, int r0,
                                      int L) {
  for (int t = threadIdx.x; t < kT * D; t += kThreadsBwd) {
    const int r = t / D, c = t % D;
    dst[r * (D + 1) + c] = r0 + r < L ? ld16<BF16>(src, (head_row0 + r0 + r) * D + c) : 0.f;
  }
}

template <int D>
__device__ __forceinline__ float dot_rows(const float* a, const float* b) {
  float s = 0.f;
#pragma unroll 16
  for (int e = 0; e < D; ++e) s = fmaf(a[e], b[e], s);
  return s;
}

// ------------------------------------------------------------------ delta

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreadsBwd) bwd_delta_kernel(BwdProblem p, int64_t rows) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (kThreadsBwd / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int c = lane; c < D; c += 32) s = fmaf(ld16<BF16>(p.dO, r * D + c), ld16<BF16>(p.o, r * D + c), s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) p.delta[r] = s;
}

// ------------------------------------------------------------------ dQ

template <int D>
constexpr int dq_smem() {
  return (4 * kT * (D + 1) + kT * (kT + 1) + 2 * kT) * static_cast<int>(sizeof(float));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreadsBwd) bwd_dq_kernel(BwdProblem p) {
  extern __shared__ float sm[];
  float* qs = sm;                       // [kT][D+1]
  float* dos = qs + kT * (D + 1);       // [kT][D+1]
  float* ks = dos + kT * (D + 1);       // [kT][D+1]
  float* vs = ks + kT * (D + 1);        // [kT][D+1]
  float* ds = vs + kT * (D + 1);        // [kT][kT+1]  dS of the block
  float* lse_s = ds + kT * (kT + 1);    // [kT]
  float* del_s = lse_s + kT;            // [kT]
  constexpr int kGroups = kThreadsBwd / D;  // row groups of the dQ product
  constexpr int kRowsPer = kT / kGroups;    // dQ rows per thread
  const int bh = blockIdx.y;
  const int b = bh / p.Hq;
  const int h_kv = (bh % p.Hq) / (p.Hq / p.Hkv);
  const int i0 = blockIdx.x * kT;
  const int64_t q_row0 = static_cast<int64_t>(bh) * p.L;
  const int64_t kv_row0 = (static_cast<int64_t>(b) * p.Hkv + h_kv) * p.L;
  const int kv = kv_len_of(p, b);
  stage<D, BF16>(qs, p.q, q_row0, i0, p.L);
  stage<D, BF16>(dos, p.dO, q_row0, i0, p.L);
  for (int t = threadIdx.x; t < kT; t += kThreadsBwd) {
    const bool in = i0 + t < p.L;
    lse_s[t] = in ? p.lse[q_row0 + i0 + t] : -INFINITY;
    del_s[t] = in ? p.delta[q_row0 + i0 + t] : 0.f;
  }
  float acc[kRowsPer];
#pragma unroll
  for (int r = 0; r < kRowsPer; ++r) acc[r] = 0.f;
  const int dcol = threadIdx.x % D, rgrp = threadIdx.x / D;
  // keys any row of the tile sees: j < kv, and j <= the last row when causal
  const int j_end = p.causal ? min(kv, i0 + kT) : kv;
  for (int j0 = 0; j0 < j_end; j0 += kT) {
    __syncthreads();
    stage<D, BF16>(ks, p.k, kv_row0, j0, p.L);
    stage<D, BF16>(vs, p.v, kv_row0, j0, p.L);
    __syncthreads();
    // dS of the 64x64 block, one element per thread per pass
    for (int e = threadIdx.x; e < kT * kT; e += kThreadsBwd) {
      const int il = e / kT, jl = e % kT;
      const int i = i0 + il, j = j0 + jl;
      float d = 0.f;
      const float lse = lse_s[il];
      if (j < kv && (!p.causal || j <= i) && lse != -INFINITY) {
        const float s = dot_rows<D>(qs + il * (D + 1), ks + jl * (D + 1)) * p.scale;
        const float pr = expf(s - lse);
        const float dp = dot_rows<D>(dos + il * (D + 1), vs + jl * (D + 1));
        d = pr * (dp - del_s[il]);
      }
      ds[il * (kT + 1) + jl] = d;
    }
    __syncthreads();
    // dQ_i += sum_j dS_ij k_j
    for (int jl = 0; jl < kT; ++jl) {
      const float kv_ = ks[jl * (D + 1) + dcol];
#pragma unroll
      for (int r = 0; r < kRowsPer; ++r) acc[r] = fmaf(ds[(rgrp + kGroups * r) * (kT + 1) + jl], kv_, acc[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPer; ++r) {
    const int i = i0 + rgrp + kGroups * r;
    if (i < p.L) st16<BF16>(p.dq, (q_row0 + i) * D + dcol, acc[r] * p.scale);
  }
}

// ------------------------------------------------------------------ dK, dV

template <int D>
constexpr int dkv_smem() {
  return (4 * kT * (D + 1) + 2 * kT * (kT + 1) + 2 * kT) * static_cast<int>(sizeof(float));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreadsBwd) bwd_dkv_kernel(BwdProblem p) {
  extern __shared__ float sm[];
  float* ks = sm;                       // [kT][D+1] resident
  float* vs = ks + kT * (D + 1);        // [kT][D+1] resident
  float* qs = vs + kT * (D + 1);        // [kT][D+1]
  float* dos = qs + kT * (D + 1);       // [kT][D+1]
  float* pt = dos + kT * (D + 1);       // [kT keys][kT+1]  P^T of the block
  float* dst = pt + kT * (kT + 1);      // [kT keys][kT+1]  dS^T of the block
  float* lse_s = dst + kT * (kT + 1);   // [kT]
  float* del_s = lse_s + kT;            // [kT]
  constexpr int kGroups = kThreadsBwd / D;
  constexpr int kRowsPer = kT / kGroups;  // dK/dV rows per thread
  const int bkv = blockIdx.y;             // b * Hkv + h_kv
  const int b = bkv / p.Hkv;
  const int h_kv = bkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int j0 = blockIdx.x * kT;
  const int64_t kv_row0 = static_cast<int64_t>(bkv) * p.L;
  const int kv = kv_len_of(p, b);
  const int dcol = threadIdx.x % D, rgrp = threadIdx.x / D;
  float dk[kRowsPer], dv[kRowsPer];
#pragma unroll
  for (int r = 0; r < kRowsPer; ++r) dk[r] = dv[r] = 0.f;
  if (j0 < kv) {  // keys at or past valid_len have no gradient
    stage<D, BF16>(ks, p.k, kv_row0, j0, p.L);
    stage<D, BF16>(vs, p.v, kv_row0, j0, p.L);
    // query rows that can see a key of the tile: i >= j0 when causal
    const int i_begin = p.causal ? (j0 / kT) * kT : 0;
    for (int g = 0; g < G; ++g) {
      const int64_t q_row0 = (static_cast<int64_t>(b) * p.Hq + h_kv * G + g) * p.L;
      for (int i0 = i_begin; i0 < p.L; i0 += kT) {
        __syncthreads();
        stage<D, BF16>(qs, p.q, q_row0, i0, p.L);
        stage<D, BF16>(dos, p.dO, q_row0, i0, p.L);
        for (int t = threadIdx.x; t < kT; t += kThreadsBwd) {
          const bool in = i0 + t < p.L;
          lse_s[t] = in ? p.lse[q_row0 + i0 + t] : -INFINITY;
          del_s[t] = in ? p.delta[q_row0 + i0 + t] : 0.f;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kT * kT; e += kThreadsBwd) {
          const int jl = e / kT, il = e % kT;
          const int i = i0 + il, j = j0 + jl;
          float pr = 0.f, d = 0.f;
          const float lse = lse_s[il];
          if (j < kv && (!p.causal || j <= i) && lse != -INFINITY) {
            const float s = dot_rows<D>(qs + il * (D + 1), ks + jl * (D + 1)) * p.scale;
            pr = expf(s - lse);
            const float dp = dot_rows<D>(dos + il * (D + 1), vs + jl * (D + 1));
            d = pr * (dp - del_s[il]);
          }
          pt[jl * (kT + 1) + il] = pr;
          dst[jl * (kT + 1) + il] = d;
        }
        __syncthreads();
        // dV_j += sum_i P_ij dO_i,  dK_j += sum_i dS_ij q_i
        for (int il = 0; il < kT; ++il) {
          const float dov = dos[il * (D + 1) + dcol];
          const float qv = qs[il * (D + 1) + dcol];
#pragma unroll
          for (int r = 0; r < kRowsPer; ++r) {
            const int jl = rgrp + kGroups * r;
            dv[r] = fmaf(pt[jl * (kT + 1) + il], dov, dv[r]);
            dk[r] = fmaf(dst[jl * (kT + 1) + il], qv, dk[r]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPer; ++r) {
    const int j = j0 + rgrp + kGroups * r;
    if (j < p.L) {
      st16<BF16>(p.dk, (kv_row0 + j) * D + dcol, dk[r] * p.scale);
      st16<BF16>(p.dv, (kv_row0 + j) * D + dcol, dv[r]);
    }
  }
}

template <int D, bool BF16>
cudaError_t launch_bwd_d(const BwdProblem& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.L;
  bwd_delta_kernel<D, BF16><<<static_cast<unsigned>((rows + 7) / 8), kThreadsBwd, 0, stream>>>(p, rows);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int s_dq = dq_smem<D>();
  constexpr int s_dkv = dkv_smem<D>();
  e = cudaFuncSetAttribute(bwd_dq_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, s_dq);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_dkv_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, s_dkv);
  if (e != cudaSuccess) return e;
  const unsigned tiles = static_cast<unsigned>((p.L + kT - 1) / kT);
  bwd_dq_kernel<D, BF16><<<dim3(tiles, p.B * p.Hq), kThreadsBwd, s_dq, stream>>>(p);
  bwd_dkv_kernel<D, BF16><<<dim3(tiles, p.B * p.Hkv), kThreadsBwd, s_dkv, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int64_t bwd_workspace_bytes(int B, int Hq, int L) { return static_cast<int64_t>(B) * Hq * L * 4; }

cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, void* dq, void* dk, void* dv, float* delta, int B, int Hq,
                       int Hkv, int L, int D, float sm_scale, int causal, const int32_t* valid_len,
                       bool bf16, cudaStream_t stream) {
  BwdProblem p{q, k, v, o, dO, lse, dq, dk, dv, delta, valid_len, B, Hq, Hkv, L, sm_scale, causal};
  if (D == 64) return bf16 ? launch_bwd_d<64, true>(p, stream) : launch_bwd_d<64, false>(p, stream);
  if (D == 128) return bf16 ? launch_bwd_d<128, true>(p, stream) : launch_bwd_d<128, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
