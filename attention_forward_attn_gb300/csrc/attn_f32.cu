// fp32 attention forward, three kernels written from the designs that
// "masked multi head attention in CUDA" (wzjinhao.cn) measures in section 6.1,
// for reproducing that section's comparison on GB300:
//
//   * naive (section 3.1): one block per (b*h, query), one thread per head
//     column; three passes over the keys -- the scores and their maximum, the
//     sum of exp(score - max), the exp-weighted sum of V rows divided by it;
//   * tiled, per-element online softmax (sections 4.1-4.2): one block per
//     (b*h, BLOCK_M = 64 queries) of 1024 threads, the Q tile resident in
//     shared memory and K/V streamed in BLOCK_N = 32-key tiles; 16 threads
//     per query, each owning D/16 output columns and updating its running
//     max, sum and accumulators after every key (two exponentials per score);
//   * tiled, block rowmax (section 4.3): the same tiling, but each thread first
//     takes the maximum of its query's BLOCK_N scores, rescales once per tile
//     and takes one exponential per score.
//
// As on the page, every thread of the tiled kernels computes its query's dot
// products itself (the threads of one query repeat them) and fp32 is used
// throughout (expf).  Masked keys are skipped, so a fully masked row gives
// O = 0 and LSE = -inf (section 3.2's "output 0" branch).  These kernels are
// the comparison, not the fast path.
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn {
namespace {

struct F32Problem {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  const int32_t* valid_len;
  int* status;
  int B, H, L;
  float scale;
  int causal;
};

__device__ __forceinline__ int key_end(const F32Problem& p, int b, int i) {
  int kv = p.L;
  if (p.valid_len != nullptr) {
    const int vl = p.valid_len[b];
    kv = vl < 0 ? 0 : (vl > p.L ? p.L : vl);
  }
  return p.causal ? min(kv, i + 1) : kv;  // keys j < key_end are visible to query i
}

__device__ __forceinline__ void flag_clamped(const F32Problem& p, int b) {
  if (p.valid_len != nullptr && (p.valid_len[b] < 0 || p.valid_len[b] > p.L))
    atomicOr(p.status, kStatusValidLenClamped);
}

// ------------------------------------------------------------------ naive

// Block sum of one value per thread (D threads, D a multiple of 32).
template <int D>
__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = x;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) s += red[i];
  __syncthreads();
  return s;
}

template <int D>
__global__ void __launch_bounds__(D) f32_naive_kernel(F32Problem p) {
  extern __shared__ float score[];  // L scores of this query
  __shared__ float red[D / 32];
  const int i = blockIdx.x;   // query
  const int bh = blockIdx.y;  // b * H + h
  const int b = bh / p.H;
  const int d = threadIdx.x;
  if (d == 0 && i == 0) flag_clamped(p, b);
  const int n = key_end(p, b, i);
  const int64_t row = static_cast<int64_t>(bh) * p.L;
  const float qd = p.q[(row + i) * D + d];
  // pass 1: the scores (one block-wide dot product per key) and their maximum
  float m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    const float s = block_sum<D>(qd * p.k[(row + j) * D + d], red) * p.scale;
    if (d == 0) score[j] = s;
    m = fmaxf(m, s);
  }
  __syncthreads();
  // pass 2: the sum of exp(score - max)
  float part = 0.f;
  for (int j = d; j < n; j += D) part += expf(score[j] - m);
  const float l = block_sum<D>(part, red);
  // pass 3: the exp-weighted sum of V rows, divided by the sum
  float acc = 0.f;
  for (int j = 0; j < n; ++j) acc = fmaf(expf(score[j] - m) / l, p.v[(row + j) * D + d], acc);
  p.o[(row + i) * D + d] = n > 0 ? acc : 0.f;
  if (d == 0 && p.lse != nullptr) p.lse[row + i] = n > 0 ? m + logf(l) : -INFINITY;
}

// ------------------------------------------------------------------ tiled

// Section 4.1's parameters: BLOCK_M = 64 queries, BLOCK_N = 32 keys, 1024
// threads; 16 threads per query, each owning D/16 output columns (4 at
// D = 64) and computing its query's dot products itself.
constexpr int kBlockN = 32;
constexpr int kBlockM = 64;
constexpr int kThreadsPerQuery = 16;

template <int D>
constexpr int f32_tiled_smem() {
  return (kBlockM * D + 2 * kBlockN * D) * static_cast<int>(sizeof(float));
}

template <int D, bool ROWMAX>
__global__ void __launch_bounds__(1024) f32_tiled_kernel(F32Problem p) {
  constexpr int CPT = D / kThreadsPerQuery;  // output columns per thread
  extern __shared__ float smem_f32[];
  float (*qs)[D] = reinterpret_cast<float (*)[D]>(smem_f32);
  float (*ks)[D] = reinterpret_cast<float (*)[D]>(smem_f32 + kBlockM * D);
  float (*vs)[D] = reinterpret_cast<float (*)[D]>(smem_f32 + kBlockM * D + kBlockN * D);
  const int ql = threadIdx.x / kThreadsPerQuery;        // query within the block
  const int c0 = (threadIdx.x % kThreadsPerQuery) * CPT;  // first output column
  const int bh = blockIdx.y;
  const int b = bh / p.H;
  const int i = blockIdx.x * kBlockM + ql;  // query
  const int64_t row = static_cast<int64_t>(bh) * p.L;
  if (threadIdx.x == 0 && blockIdx.x == 0) flag_clamped(p, b);
  for (int t = threadIdx.x; t < kBlockM * D; t += 1024) {
    const int qi = blockIdx.x * kBlockM + t / D;
    qs[t / D][t % D] = qi < p.L ? p.q[(row + qi) * D + t % D] : 0.f;
  }
  const int n = i < p.L ? key_end(p, b, i) : 0;
  // keys the block needs: up to its largest key_end
  const int n_blk = key_end(p, b, min(p.L - 1, blockIdx.x * kBlockM + kBlockM - 1));
  float m = -INFINITY, l = 0.f;
  float acc[CPT];
#pragma unroll
  for (int c = 0; c < CPT; ++c) acc[c] = 0.f;
  for (int k0 = 0; k0 < n_blk; k0 += kBlockN) {
    __syncthreads();
    for (int t = threadIdx.x; t < kBlockN * D; t += 1024) {
      const int j = k0 + t / D;
      ks[t / D][t % D] = j < p.L ? p.k[(row + j) * D + t % D] : 0.f;
      vs[t / D][t % D] = j < p.L ? p.v[(row + j) * D + t % D] : 0.f;
    }
    __syncthreads();
    const int cnt = min(kBlockN, n - k0);  // this query's visible keys of the tile
    if constexpr (!ROWMAX) {
      // per-element online softmax: after every key
      for (int j = 0; j < cnt; ++j) {
        float s = 0.f;
#pragma unroll 16
        for (int e = 0; e < D; ++e) s = fmaf(qs[ql][e], ks[j][e], s);
        s *= p.scale;
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);
        const float beta = expf(s - m_new);
        l = l * alpha + beta;
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] = acc[c] * alpha + beta * vs[j][c0 + c];
        m = m_new;
      }
    } else {
      // block rowmax: the tile's scores and their maximum first, one rescale,
      // then one exponential per score
      float sc[kBlockN];
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < kBlockN; ++j) {
        float s = -INFINITY;
        if (j < cnt) {
          s = 0.f;
#pragma unroll 16
          for (int e = 0; e < D; ++e) s = fmaf(qs[ql][e], ks[j][e], s);
          s *= p.scale;
        }
        sc[j] = s;
        mt = fmaxf(mt, s);
      }
      if (cnt > 0) {
        const float m_new = fmaxf(m, mt);
        const float alpha = expf(m - m_new);
        l *= alpha;
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[c] *= alpha;
#pragma unroll
        for (int j = 0; j < kBlockN; ++j) {
          if (j < cnt) {
            const float e = expf(sc[j] - m_new);
            l += e;
#pragma unroll
            for (int c = 0; c < CPT; ++c) acc[c] = fmaf(e, vs[j][c0 + c], acc[c]);
          }
        }
        m = m_new;
      }
    }
  }
  if (i < p.L) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) p.o[(row + i) * D + c0 + c] = n > 0 ? acc[c] / l : 0.f;
    if (c0 == 0 && p.lse != nullptr) p.lse[row + i] = n > 0 ? m + logf(l) : -INFINITY;
  }
}

template <int D>
cudaError_t launch_f32_d(const F32Problem& p, int kernel, cudaStream_t stream) {
  if (kernel == 0) {
    const size_t smem = static_cast<size_t>(p.L) * sizeof(float);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(f32_naive_kernel<D>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    f32_naive_kernel<D><<<dim3(p.L, p.B * p.H), D, smem, stream>>>(p);
  } else {
    const dim3 grid((p.L + kBlockM - 1) / kBlockM, p.B * p.H);
    constexpr int smem = f32_tiled_smem<D>();
    auto kern = kernel == 1 ? f32_tiled_kernel<D, false> : f32_tiled_kernel<D, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 1024, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                       int B, int H, int L, int D, float sm_scale, int causal,
                       const int32_t* valid_len, int kernel, int* status, cudaStream_t stream) {
  F32Problem p{q, k, v, o, lse, valid_len, status, B, H, L, sm_scale, causal};
  if (D == 64) return launch_f32_d<64>(p, kernel, stream);
  if (D == 128) return launch_f32_d<128>(p, kernel, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
