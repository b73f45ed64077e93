// SIMT cross-check kernel for the attention forward.
//
// One warp per query row.  For each block of 32 keys, lane j computes the
// score of key (kb + j) as an fp32 dot product over D, the warp takes the
// block maximum, and the online-softmax state (running max m, exp-sum l and
// the fp32 accumulator, one D/32 slice per lane) is rescaled by
// alpha = exp2(m_old - m_new) and updated with the block's weights -- the
// "block rowmax, then one exp per score" form of wzjinhao.cn section 4.3 and
// of the Triton-CUDA Attention page's online softmax (scores pre-multiplied by
// sm_scale*log2(e) so that exp2 can be used).  No tensor cores: this kernel
// exists to cross-check the tensor-core path, not for speed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kWarpsPerBlock = 8;

template <bool BF16>
__device__ __forceinline__ float load_elem(const void* base, int64_t idx) {
  if constexpr (BF16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  } else {
    return __half2float(reinterpret_cast<const __half*>(base)[idx]);
  }
}

template <bool BF16>
__device__ __forceinline__ void store_elem(void* base, int64_t idx, float x) {
  if constexpr (BF16) {
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(x);
  } else {
    reinterpret_cast<__half*>(base)[idx] = __float2half_rn(x);
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    attn_fwd_simt_kernel(Problem p, float scale_log2) {
  constexpr int kPerLane = (D + 31) / 32;  // accumulator columns lane + 32c (c < kPerLane, < D)
  __shared__ float q_sh[kWarpsPerBlock][D];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarpsPerBlock + warp;  // query row
  const int bh = blockIdx.y;                         // b * Hq + h_q
  if (i >= p.Lq) return;                             // whole warp leaves together
  const int b = bh / p.Hq;
  const int h_q = bh % p.Hq;
  const int h_kv = h_q / (p.Hq / p.Hkv);

  int kv_len = p.Lk;
  if (p.valid_len != nullptr) {
    int vl = p.valid_len[b];
    if (vl < 0 || vl > p.Lk) {
      if (lane == 0) atomicOr(p.status, kStatusValidLenClamped);
      vl = vl < 0 ? 0 : p.Lk;
    }
    kv_len = vl;
  }
  const int key_end = p.causal ? min(kv_len, i + 1) : kv_len;

  // element offsets of this row of Q and O, of key 0 of the K and V head, and
  // of this row of LSE ([B*Hq, Lq] contiguous)
  const int64_t q_row = b * p.sq.b + h_q * p.sq.h + i * p.sq.l;
  const int64_t o_row = b * p.so.b + h_q * p.so.h + i * p.so.l;
  const int64_t k_head = b * p.sk.b + h_kv * p.sk.h;
  const int64_t v_head = b * p.sv.b + h_kv * p.sv.h;
  const int64_t lse_row = static_cast<int64_t>(bh) * p.Lq + i;
  for (int d = lane; d < D; d += 32) q_sh[warp][d] = load_elem<BF16>(p.q, q_row + d);
  __syncwarp();

  float m = -INFINITY;  // running max of the scaled (log2-domain) scores
  float l = 0.f;
  float acc[kPerLane];
#pragma unroll
  for (int c = 0; c < kPerLane; ++c) acc[c] = 0.f;

  for (int kb = 0; kb < key_end; kb += 32) {
    const int key = kb + lane;
    float t = -INFINITY;
    if (key < key_end) {
      const int64_t k_row = k_head + key * p.sk.l;
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) dot = fmaf(q_sh[warp][d], load_elem<BF16>(p.k, k_row + d), dot);
      t = dot * scale_log2;
    }
    const float m_new = fmaxf(m, warp_max(t));  // finite: key kb is always visible
    const float alpha = exp2f(m - m_new);
    const float w = (key < key_end) ? exp2f(t - m_new) : 0.f;
    l = l * alpha + warp_sum(w);
#pragma unroll
    for (int c = 0; c < kPerLane; ++c) acc[c] *= alpha;
    const int n_keys = min(32, key_end - kb);
    for (int j = 0; j < n_keys; ++j) {
      const float wj = __shfl_sync(0xffffffffu, w, j);
      const int64_t v_row = v_head + (kb + j) * p.sv.l;
#pragma unroll
      for (int c = 0; c < kPerLane; ++c) {
        if (D % 32 == 0 || lane + 32 * c < D)
          acc[c] = fmaf(wj, load_elem<BF16>(p.v, v_row + lane + 32 * c), acc[c]);
      }
    }
    m = m_new;
  }

  const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < kPerLane; ++c) {
    if (D % 32 == 0 || lane + 32 * c < D) store_elem<BF16>(p.o, o_row + lane + 32 * c, acc[c] * inv_l);
  }
  if (p.lse != nullptr && lane == 0) {
    // natural log: ln(sum exp(s)) = ln2 * (m + log2 l) with m in log2 units
    p.lse[lse_row] = (l > 0.f) ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_simt(const Problem& p) {
  const float scale_log2 = p.sm_scale * 1.4426950408889634f;
  if (static_cast<int64_t>(p.B) * p.Hq > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((p.Lq + kWarpsPerBlock - 1) / kWarpsPerBlock, p.B * p.Hq);
  dim3 block(kWarpsPerBlock * 32);
  if (p.D == 16) {
    if (p.bf16) attn_fwd_simt_kernel<16, true><<<grid, block, 0, p.stream>>>(p, scale_log2);
    else attn_fwd_simt_kernel<16, false><<<grid, block, 0, p.stream>>>(p, scale_log2);
  } else if (p.D == 32) {
    if (p.bf16) attn_fwd_simt_kernel<32, true><<<grid, block, 0, p.stream>>>(p, scale_log2);
    else attn_fwd_simt_kernel<32, false><<<grid, block, 0, p.stream>>>(p, scale_log2);
  } else if (p.D == 64) {
    if (p.bf16) attn_fwd_simt_kernel<64, true><<<grid, block, 0, p.stream>>>(p, scale_log2);
    else attn_fwd_simt_kernel<64, false><<<grid, block, 0, p.stream>>>(p, scale_log2);
  } else if (p.D == 128) {
    if (p.bf16) attn_fwd_simt_kernel<128, true><<<grid, block, 0, p.stream>>>(p, scale_log2);
    else attn_fwd_simt_kernel<128, false><<<grid, block, 0, p.stream>>>(p, scale_log2);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace attn
