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
// Each thread owns 4 x 4 blocks of (query, key) pairs and of the dQ / dK / dV
// products; the dot products read 16-byte vectors of transposed [D][64]
// shared-memory tiles (one pair of loads per 16 FMAs).
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

// Stage rows r0 .. r0+63 of a [.., L, D] 16-bit head into fp32 shared memory
// (rows past L are zeros).  Row-major [64][D]: consecutive threads take
// consecutive columns.  Transposed [D][64]: a thread loads 8 columns of one row
// with one 16-byte load and consecutive threads take consecutive rows, so a
// warp's stores of one column fill 32 banks.
template <int D, bool BF16>
__device__ __forceinline__ void stage_rm(float* rm, const void* src, int64_t head_row0, int r0,
                                         int L) {
  for (int t = threadIdx.x; t < kT * D; t += kThreadsBwd) {
    const int r = t / D, c = t % D;
    rm[r * D + c] = r0 + r < L ? ld16<BF16>(src, (head_row0 + r0 + r) * D + c) : 0.f;
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack16x2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

template <int D, bool BF16>
__device__ __forceinline__ void stage_tr(float* tr, const void* src, int64_t head_row0, int r0,
                                         int L) {
  for (int t = threadIdx.x; t < kT * (D / 8); t += kThreadsBwd) {
    const int r = t % kT, c0 = (t / kT) * 8;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (r0 + r < L)
      raw = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) +
                                            (head_row0 + r0 + r) * D + c0);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack16x2<BF16>(w[k]);
      tr[(c0 + 2 * k) * kT + r] = f.x;
      tr[(c0 + 2 * k + 1) * kT + r] = f.y;
    }
  }
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// 4x4 block of dot products: acc[a][b] += sum_e A[e][a0+a] B[e][b0+b] over
// transposed [D][64] tiles (one 16-byte load of each operand per e).
template <int D>
__device__ __forceinline__ void dot4x4(float (&acc)[4][4], const float* at, const float* bt, int a0,
                                       int b0) {
#pragma unroll 4
  for (int e = 0; e < D; ++e) {
    const float4 x = ld4(at + e * kT + a0);
    const float4 y = ld4(bt + e * kT + b0);
    const float xa[4] = {x.x, x.y, x.z, x.w};
    const float yb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xa[a], yb[b], acc[a][b]);
  }
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

// Thread (ti, tj) of a 16 x 16 grid owns the 4 x 4 block of (query, key)
// pairs (4 ti + a, 4 tj + b) of a 64 x 64 block, and the 4 x D/16 block of dQ
// (rows 4 ti + a, columns tj + 16 c).
template <int D>
constexpr int dq_smem() {
  // Q^T, dO^T, K^T, V^T [D][64]; K [64][D]; dS^T [64 keys][64]; LSE, delta
  return (5 * kT * D + kT * kT + 2 * kT) * static_cast<int>(sizeof(float));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreadsBwd) bwd_dq_kernel(BwdProblem p) {
  extern __shared__ float sm[];
  float* qt = sm;                 // [D][64]
  float* dot_ = qt + kT * D;      // [D][64]
  float* kt = dot_ + kT * D;      // [D][64]
  float* vt = kt + kT * D;        // [D][64]
  float* kr = vt + kT * D;        // [64][D]
  float* dst = kr + kT * D;       // [64 keys][64 queries]
  float* lse_s = dst + kT * kT;   // [64]
  float* del_s = lse_s + kT;      // [64]
  constexpr int CQ = D / 16;      // dQ columns per thread
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  const int bh = blockIdx.y;
  const int b = bh / p.Hq;
  const int h_kv = (bh % p.Hq) / (p.Hq / p.Hkv);
  const int i0 = blockIdx.x * kT;
  const int64_t q_row0 = static_cast<int64_t>(bh) * p.L;
  const int64_t kv_row0 = (static_cast<int64_t>(b) * p.Hkv + h_kv) * p.L;
  const int kv = kv_len_of(p, b);
  stage_tr<D, BF16>(qt, p.q, q_row0, i0, p.L);
  stage_tr<D, BF16>(dot_, p.dO, q_row0, i0, p.L);
  for (int t = threadIdx.x; t < kT; t += kThreadsBwd) {
    const bool in = i0 + t < p.L;
    lse_s[t] = in ? p.lse[q_row0 + i0 + t] : -INFINITY;
    del_s[t] = in ? p.delta[q_row0 + i0 + t] : 0.f;
  }
  float acc[4][CQ];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < CQ; ++c) acc[a][c] = 0.f;
  const int j_end = p.causal ? min(kv, i0 + kT) : kv;
  for (int j0 = 0; j0 < j_end; j0 += kT) {
    __syncthreads();
    stage_rm<D, BF16>(kr, p.k, kv_row0, j0, p.L);
    stage_tr<D, BF16>(kt, p.k, kv_row0, j0, p.L);
    stage_tr<D, BF16>(vt, p.v, kv_row0, j0, p.L);
    __syncthreads();
    float sc[4][4] = {}, dp[4][4] = {};
    dot4x4<D>(sc, qt, kt, 4 * ti, 4 * tj);
    dot4x4<D>(dp, dot_, vt, 4 * ti, 4 * tj);
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int il = 4 * ti + a, i = i0 + il;
      const float lse = lse_s[il];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const int jl = 4 * tj + bb, j = j0 + jl;
        float d = 0.f;
        if (j < kv && (!p.causal || j <= i) && lse != -INFINITY)
          d = expf(sc[a][bb] * p.scale - lse) * (dp[a][bb] - del_s[il]);
        dst[jl * kT + il] = d;
      }
    }
    __syncthreads();
    // dQ_i += sum_j dS_ij k_j
    for (int jl = 0; jl < kT; ++jl) {
      const float4 d4 = ld4(dst + jl * kT + 4 * ti);
      const float da[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
      for (int c = 0; c < CQ; ++c) {
        const float kv_ = kr[jl * D + tj + 16 * c];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a][c] = fmaf(da[a], kv_, acc[a][c]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = i0 + 4 * ti + a;
    if (i < p.L) {
#pragma unroll
      for (int c = 0; c < CQ; ++c) st16<BF16>(p.dq, (q_row0 + i) * D + tj + 16 * c, acc[a][c] * p.scale);
    }
  }
}

// ------------------------------------------------------------------ dK, dV

// Thread (ti, tj): the 4 x 4 block of (key, query) pairs (4 ti + a, 4 tj + b)
// of a 64 x 64 block, and the 4 x D/16 blocks of dK and dV (rows 4 ti + a,
// columns tj + 16 c).
template <int D>
constexpr int dkv_smem() {
  // K^T, V^T, Q^T, dO^T [D][64]; Q, dO [64][D]; P, dS [64 queries][64 keys]; LSE, delta
  return (6 * kT * D + 2 * kT * kT + 2 * kT) * static_cast<int>(sizeof(float));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreadsBwd) bwd_dkv_kernel(BwdProblem p) {
  extern __shared__ float sm[];
  float* kt = sm;                  // [D][64] resident
  float* vt = kt + kT * D;         // [D][64] resident
  float* qt = vt + kT * D;         // [D][64]
  float* dot_ = qt + kT * D;       // [D][64]
  float* qr = dot_ + kT * D;       // [64][D]
  float* dor = qr + kT * D;        // [64][D]
  float* pq = dor + kT * D;        // [64 queries][64 keys]  P
  float* dq = pq + kT * kT;        // [64 queries][64 keys]  dS
  float* lse_s = dq + kT * kT;     // [64]
  float* del_s = lse_s + kT;       // [64]
  constexpr int CK = D / 16;
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  const int bkv = blockIdx.y;      // b * Hkv + h_kv
  const int b = bkv / p.Hkv;
  const int h_kv = bkv % p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int j0 = blockIdx.x * kT;
  const int64_t kv_row0 = static_cast<int64_t>(bkv) * p.L;
  const int kv = kv_len_of(p, b);
  float dk[4][CK], dv[4][CK];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < CK; ++c) dk[a][c] = dv[a][c] = 0.f;
  if (j0 < kv) {  // keys at or past valid_len have no gradient
    stage_tr<D, BF16>(kt, p.k, kv_row0, j0, p.L);
    stage_tr<D, BF16>(vt, p.v, kv_row0, j0, p.L);
    const int i_begin = p.causal ? j0 : 0;  // rows that see a key of the tile
    for (int g = 0; g < G; ++g) {
      const int64_t q_row0 = (static_cast<int64_t>(b) * p.Hq + h_kv * G + g) * p.L;
      for (int i0 = i_begin; i0 < p.L; i0 += kT) {
        __syncthreads();
        stage_rm<D, BF16>(qr, p.q, q_row0, i0, p.L);
        stage_tr<D, BF16>(qt, p.q, q_row0, i0, p.L);
        stage_rm<D, BF16>(dor, p.dO, q_row0, i0, p.L);
        stage_tr<D, BF16>(dot_, p.dO, q_row0, i0, p.L);
        for (int t = threadIdx.x; t < kT; t += kThreadsBwd) {
          const bool in = i0 + t < p.L;
          lse_s[t] = in ? p.lse[q_row0 + i0 + t] : -INFINITY;
          del_s[t] = in ? p.delta[q_row0 + i0 + t] : 0.f;
        }
        __syncthreads();
        float sc[4][4] = {}, dp[4][4] = {};
        dot4x4<D>(sc, kt, qt, 4 * ti, 4 * tj);   // [key a][query b]
        dot4x4<D>(dp, vt, dot_, 4 * ti, 4 * tj);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const int jl = 4 * ti + a, j = j0 + jl;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const int il = 4 * tj + bb, i = i0 + il;
            const float lse = lse_s[il];
            float pr = 0.f, d = 0.f;
            if (j < kv && (!p.causal || j <= i) && lse != -INFINITY) {
              pr = expf(sc[a][bb] * p.scale - lse);
              d = pr * (dp[a][bb] - del_s[il]);
            }
            pq[il * kT + jl] = pr;
            dq[il * kT + jl] = d;
          }
        }
        __syncthreads();
        // dV_j += sum_i P_ij dO_i,  dK_j += sum_i dS_ij q_i
        for (int il = 0; il < kT; ++il) {
          const float4 p4 = ld4(pq + il * kT + 4 * ti);
          const float4 s4 = ld4(dq + il * kT + 4 * ti);
          const float pa[4] = {p4.x, p4.y, p4.z, p4.w};
          const float sa[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int c = 0; c < CK; ++c) {
            const float dov = dor[il * D + tj + 16 * c];
            const float qv = qr[il * D + tj + 16 * c];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              dv[a][c] = fmaf(pa[a], dov, dv[a][c]);
              dk[a][c] = fmaf(sa[a], qv, dk[a][c]);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = j0 + 4 * ti + a;
    if (j < p.L) {
#pragma unroll
      for (int c = 0; c < CK; ++c) {
        st16<BF16>(p.dk, (kv_row0 + j) * D + tj + 16 * c, dk[a][c] * p.scale);
        st16<BF16>(p.dv, (kv_row0 + j) * D + tj + 16 * c, dv[a][c]);
      }
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
