// Tensor-core attention backward for sm_103a (tcgen05 + TMA + TMEM).
//
// What it computes (the derivative of O = softmax(sm_scale Q K^T + Mask) V,
// with the softmax rebuilt from the LSE the forward stores "for the backward
// pass", tiny_flash_attn_triton.py; the pages give no backward algorithm):
//   P_ij = exp(sm_scale q_i.k_j - LSE_i) on visible keys, 0 elsewhere,
//   delta_i = dO_i.O_i,  dP_ij = dO_i.v_j,  dS_ij = P_ij (dP_ij - delta_i),
//   dQ = sm_scale dS K,  dK = sm_scale dS^T Q,  dV = P^T dO,
// dK and dV of a key/value head summed over the query heads that read it.
//
// How: a pre-pass and two kernels, every product on the tensor core with an
// fp32 accumulator in TMEM and P, dS rounded to the input dtype as operands:
//   * pre-pass (D/8 lanes per row): delta_i and -LSE_i log2(e) into rows
//     padded to a multiple of 128 (0 and -inf beyond Lq; -inf where the row
//     sees no key), so that both kernels fetch them with aligned bulk copies;
//   * dK/dV kernel, one CTA per (128-key tile, b, h_kv), K and V resident in
//     shared memory.  Every (query head of the group, 128-row query tile) that
//     sees the keys streams through a ring of Q, dO, LSE and delta stages.
//     Per step: S^T = K Q^T and dP^T = V dO^T (keys in TMEM lanes, two
//     128-column regions that swap roles every step), then two elementwise
//     warpgroups (each 64 query columns of every key row) write P^T and dS^T
//     as 16-bit pairs into the S^T region, and dV += P^T dO, dK += dS^T Q
//     read them from TMEM (dO and Q as MN-major operands); the next S^T goes
//     into the dP^T region as soon as dP^T has been read.  TMEM: the two
//     regions, dV, dK (512 columns at D = 128).  With too few key tiles for
//     the GPU (MQA), each key tile's steps are split over several CTAs that
//     write fp32 partials, summed in a fixed order by a reduction kernel;
//   * dQ kernel, one CTA per (128-row query tile, b, h_q), Q and dO resident,
//     K and V streaming: S = Q K^T, dP = dO V^T, dS written to its own TMEM
//     columns (two buffers), dQ += dS K (K as MN-major operand).  TMEM: S,
//     dP, dQ, dS x 2.
// Warp roles: warps 0-7 elementwise (TMEM lane = key row in the dK/dV kernel,
// query row in the dQ kernel; warps w and w + 4 share a lane quadrant and
// split the columns), warp 8 TMA producer, warp 9 MMA issuer (one elected
// lane issues) and TMEM owner.  Causal tiles above the diagonal and key tiles
// at or beyond valid_len[b] are never visited; masked (query, key) pairs get
// P = 0, hence dS = 0.  An explicit mask is packed into bits over keys and
// over queries by a pre-pass, which also lists the 128 x 128 blocks that keep
// any position; the MASK instances visit only those.  Separate query and key
// lengths (causal top-left) and strided operands throughout; D = 16 and 32 run
// the D = 64 instances on zero-filled columns.
//
// Every mbarrier wait is bounded as in the forward: on a timeout the waiting
// role records it in the device status word and raises the CTA's abort flag;
// the others leave too, the CTA drains its own copies and MMAs and frees its
// TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "attn_internal.h"
#include "ptx.cuh"

#ifndef ATTN_WAIT_LIMIT_NS
#define ATTN_WAIT_LIMIT_NS 2000000000ull
#endif

namespace attn {
namespace {

// Elementwise warpgroups per CTA: each takes T / kGroups columns of every
// 128 x 128 step.  Two (64 columns per thread) measured 2-4 % faster than
// four (32 columns, twice the warps per sub-partition).
#ifndef ATTN_BWD_EW_GROUPS
#define ATTN_BWD_EW_GROUPS 2
#endif
constexpr int T = 128;                       // query rows of a query tile = keys of a key tile
constexpr int kGroups = ATTN_BWD_EW_GROUPS;  // elementwise warpgroups
constexpr int TH = T / kGroups;              // columns of one elementwise warpgroup
constexpr int kEwThreads = 128 * kGroups;
constexpr int kLoadWarp = 4 * kGroups;
constexpr int kMmaWarp = 4 * kGroups + 1;
constexpr int kThreadsB = 32 * (4 * kGroups + 2);
static_assert(kGroups == 2 || kGroups == 4, "two or four elementwise warpgroups");
constexpr float kLog2e = 1.4426950408889634f;

struct BwdTcParams {
  const float* nlse2;  // [B*Hq, Lp] -LSE log2(e); -inf: no visible key, or row >= L
  const float* delta;  // [B*Hq, Lp] dO.O; 0 for rows >= L
  void* dq;
  void* dk;
  void* dv;
  const int32_t* valid_len;
  int* status;
  int B, Hq, Hkv, G;
  int Lq, Lk;      // query and key lengths
  int n_tq, n_tk;  // 128-row query tiles, 128-key tiles
  int Lqp;         // 128 n_tq: rows of the -LSE log2(e) and delta arrays
  int dg;                         // head dimension in memory: D, or 16 / 32 on the D = 64 kernels
  Strides sdq, sdk, sdv;          // element strides (batch, head, row) of the outputs
  int splits;                     // CTAs per key tile of the dK/dV kernel (see bwd_tc_splits)
  float* part;                    // splits > 1: fp32 partial dV, dK [splits][2][B*Hkv*L][dg]
  // explicit mask (bwd_mask_pack_kernel): bit i%32 of a word = the mask at
  // (query i, key j); rbits [mB][Lq][n_tk][4] words over the keys of a tile,
  // cbits [mB][Lk][n_tq][4] over the queries of a tile; mB = 1 when shared
  const uint32_t* rbits;
  const uint32_t* cbits;
  int mask_shared;
  // tiles with a kept position (bwd_mask_lists_kernel): per key tile the
  // query tiles to visit, ascending (klist [mB][n_tk][n_tq], kcount
  // [mB][n_tk]); per query tile the key tiles (qlist [mB][n_tq][n_tk], qcount)
  const int* klist;
  const int* kcount;
  const int* qlist;
  const int* qcount;
  float scale_log2;               // sm_scale log2(e)
  float sm_scale;
  int causal;
};

// Shared-memory layout and TMEM columns, both kernels.  Every tile is 128
// rows of 64-column (128-byte) swizzled slabs, 1024-byte aligned.
template <int D>
struct BCfg {
  static constexpr int kTile = T * D * 2;
  static constexpr int kSlab = T * 128;
  // dK/dV kernel: K, V resident; stages of Q, dO, -LSE log2(e), delta
  static constexpr int kvStages = (D == 128) ? 2 : 3;
  static constexpr int kvOffK = 0;
  static constexpr int kvOffV = kTile;
  static constexpr int kvOffIn = 2 * kTile;
  static constexpr int kvStageBytes = 2 * kTile + 1024;
  static constexpr int kvOffBar = kvOffIn + kvStages * kvStageBytes;
  // dQ kernel: Q, dO resident; a K ring and a V ring (V is released a step
  // earlier than K: after dP, K only after dQ)
  static constexpr int qKStages = (D == 128) ? 3 : 6;
  static constexpr int qVStages = (D == 128) ? 2 : 4;
  static constexpr int qOffQ = 0;
  static constexpr int qOffDO = kTile;
  static constexpr int qOffK = 2 * kTile;
  static constexpr int qOffV = qOffK + qKStages * kTile;
  static constexpr int qOffBar = qOffV + qVStages * kTile;
  static constexpr int kBarBytes = 256;  // barriers, TMEM base word, abort flag
  static constexpr int kvSmem = kvOffBar + kBarBytes + 1024;  // + slack to align the base
  static constexpr int qSmem = qOffBar + kBarBytes + 1024;
  static_assert(kvSmem <= 232448 && qSmem <= 232448, "shared-memory budget");
  // TMEM columns
  // dK/dV kernel: regions [0, 128) and [128, 256) hold S^T and dP^T of a
  // step, swapping every step (region_x / region_y); dQ kernel: S and dP
  static constexpr uint32_t kColS = 0;      // S (fp32, dQ kernel)
  static constexpr uint32_t kColDP = T;     // dP (fp32, dQ kernel)
  static constexpr uint32_t kColAcc0 = 2 * T;      // dV (dK/dV kernel) / dQ (dQ kernel)
  static constexpr uint32_t kColAcc1 = 2 * T + D;  // dK (dK/dV kernel) / dS (dQ kernel, 2 x 64 columns)
  static constexpr uint32_t kTmemCols = 512;
  static_assert(2 * T + 2 * D <= 512 && 2 * T + D + T <= 512, "TMEM budget");
};

// Barrier block: n_bars 8-byte barriers from `base`, then the TMEM base word
// and the abort flag.
struct BBars {
  uint32_t base;
  int n_bars;
  __device__ __forceinline__ uint32_t bar(int i) const { return base + 8u * static_cast<uint32_t>(i); }
  __device__ __forceinline__ uint32_t tmem_word() const { return bar(n_bars); }
  __device__ __forceinline__ uint32_t abort_word() const { return tmem_word() + 4u; }
};

// Bounded mbarrier wait.  False: timed out (recorded) or another role aborted.
__device__ __forceinline__ bool bwait(const BBars& br, int* status, uint32_t bar, uint32_t parity,
                                      int role) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (ptx::ld_shared_volatile(br.abort_word()) != 0u) return false;
    if (ptx::globaltimer_ns() - t0 > ATTN_WAIT_LIMIT_NS) {
      ptx::st_shared_volatile(br.abort_word(), 1u);
      atomicOr(status, kStatusTimeout | role);
      return false;
    }
  }
}

// Wait with a time limit and no abort check (draining in-flight work only).
__device__ __forceinline__ void bdrain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t0 < ATTN_WAIT_LIMIT_NS) {
  }
}

__device__ __forceinline__ bool elect() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void commit(uint32_t bar) {
  if (elect()) ptx::mma_commit(bar);
  __syncwarp();
}

__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Untiled bulk copy global -> shared of `bytes` bytes (both addresses 16-byte
// aligned, size a multiple of 16), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// d = A B^T over D with both operands K-major 128-row tiles (128 x 128 fp32
// result): S^T = K Q^T, dP^T = V dO^T, S = Q K^T, dP = dO V^T.
template <int D, bool BF16>
__device__ __forceinline__ void mma_rows(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint32_t idesc = ptx::idesc_f16(T, T, BF16, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * BCfg<D>::kSlab + (kk & 3) * 32u;
    ptx::mma_ss(d_tmem, dadd(a_desc, off), dadd(b_desc, off), idesc, kk > 0 ? 1u : 0u);
  }
}

// acc (+)= A X with A a 128 x 128 16-bit matrix in TMEM, one TH-column block
// per elementwise warpgroup, each packed into the first TH/2 columns of its
// block (P^T, dS^T: a_group = TH) or all packed contiguously (dS of the dQ
// kernel: a_group = TH/2), and X a 128-row tile used as an MN-major operand
// (X = dO, Q or K; 16 rows per MMA).
template <int D, bool BF16>
__device__ __forceinline__ void mma_acc(uint32_t acc, uint32_t a_tmem, uint32_t a_group,
                                        uint64_t x_mn, bool accumulate) {
  constexpr uint32_t idesc = ptx::idesc_f16(T, D, BF16, true);
  constexpr int kPerGroup = TH / 16;  // MMAs (16 K values each) per warpgroup block
#pragma unroll
  for (int kk = 0; kk < T / 16; ++kk) {
    ptx::mma_ts(acc, a_tmem + (kk / kPerGroup) * a_group + (kk % kPerGroup) * 8u,
                dadd(x_mn, kk * 2048u), idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// N = TH consecutive fp32 columns of this thread's TMEM lane; N/2 packed columns back.
template <int N>
__device__ __forceinline__ void ld_th(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 32 || N == 64, "32 or 64 columns");
  if constexpr (N == 64) {
    ptx::tmem_ld64(taddr, r);
  } else {
    ptx::tmem_ld32(taddr, r);
  }
}
template <int N>
__device__ __forceinline__ void st_th2(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 packed columns");
  if constexpr (N == 32) {
    ptx::tmem_st32(taddr, r);
  } else {
    ptx::tmem_st16(taddr, r);
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pk2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ int kv_len_of(const BwdTcParams& p, int b) {
  if (p.valid_len == nullptr) return p.Lk;
  const int vl = p.valid_len[b];
  return vl < 0 ? 0 : (vl > p.Lk ? p.Lk : vl);
}

// ------------------------------------------------------------------ pre-pass

// Padded rows r of [B*Hq, Lp], D/8 lanes per row (32*8/D rows per warp):
// delta = dO.O with 16-byte loads, and -LSE log2(e).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_tc_prep_kernel(const void* __restrict__ o,
                                                          const void* __restrict__ dO,
                                                          const float* __restrict__ lse,
                                                          float* nlse2, float* delta, int Hq, int L,
                                                          int Lp, int64_t rows, Strides so,
                                                          Strides sdo) {
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp
  const int lane = threadIdx.x & 31;
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * RPW + lane / LPR;
  const int sub = lane % LPR;
  const int64_t bh = r / Lp;
  const int i = static_cast<int>(r - bh * Lp);
  const bool live = r < rows && i < L;
  float s = 0.f;
  if (live) {
    const int64_t b = bh / Hq, h = bh - b * Hq;
    const int64_t eo = b * so.b + h * so.h + i * so.l + sub * 8;
    const int64_t eg = b * sdo.b + h * sdo.h + i * sdo.l + sub * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(o) + eo);
    const uint4 g = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(dO) + eg);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 fa, fg;
      if constexpr (BF16) {
        fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[k]));
        fg = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[k]));
      } else {
        fa = __half22float2(*reinterpret_cast<const __half2*>(&av[k]));
        fg = __half22float2(*reinterpret_cast<const __half2*>(&gv[k]));
      }
      s = fmaf(fa.x, fg.x, s);
      s = fmaf(fa.y, fg.y, s);
    }
  }
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (sub == 0 && r < rows) {
    float nl = -INFINITY;
    if (i < L) {
      const float x = lse[bh * L + i];
      nl = (x == -INFINITY) ? -INFINITY : -x * kLog2e;
    }
    nlse2[r] = nl;
    delta[r] = i < L ? s : 0.f;
  }
}

// Explicit mask -> bits, one CTA per (key tile, query tile, mask batch): the
// 128 x 128 block of mask bytes is staged in shared memory (rows padded to
// 132 bytes, so a warp reading one column touches 32 banks), then warp
// ballots write each query row's 128 key bits (rbits) and each key row's 128
// query bits (cbits).  Positions outside [0, Lq) x [0, Lk) are 0.
__global__ void __launch_bounds__(256) bwd_mask_pack_kernel(const uint8_t* __restrict__ mask,
                                                            int64_t msb, int64_t msr, int Lq,
                                                            int Lk, int n_tq, int n_tk,
                                                            uint32_t* rbits, uint32_t* cbits,
                                                            uint8_t* vis) {
  constexpr int kPitch = 132;
  __shared__ uint8_t blk[T * kPitch];
  __shared__ int any_kept;
  const int n = blockIdx.x, m = blockIdx.y, mb = blockIdx.z;
  if (threadIdx.x == 0) any_kept = 0;
  const uint8_t* src = mask + mb * msb;
  for (int idx = threadIdx.x; idx < T * T; idx += 256) {
    const int r = idx / T, c = idx % T;
    const int i = m * T + r, j = n * T + c;
    blk[r * kPitch + c] = (i < Lq && j < Lk) ? (src[static_cast<int64_t>(i) * msr + j] != 0) : 0;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = warp; r < T; r += 8) {  // query row r of the block: its 128 key bits
    uint32_t wd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) wd[q] = __ballot_sync(0xffffffffu, blk[r * kPitch + q * 32 + lane] != 0);
    const int i = m * T + r;
    if (lane == 0 && i < Lq)
      *reinterpret_cast<uint4*>(rbits + ((static_cast<int64_t>(mb) * Lq + i) * n_tk + n) * 4) =
          make_uint4(wd[0], wd[1], wd[2], wd[3]);
    if (lane == 0 && (wd[0] | wd[1] | wd[2] | wd[3]) != 0u) any_kept = 1;
  }
  for (int c = warp; c < T; c += 8) {  // key column c of the block: its 128 query bits
    uint32_t wd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) wd[q] = __ballot_sync(0xffffffffu, blk[(q * 32 + lane) * kPitch + c] != 0);
    const int j = n * T + c;
    if (lane == 0 && j < Lk)
      *reinterpret_cast<uint4*>(cbits + ((static_cast<int64_t>(mb) * Lk + j) * n_tq + m) * 4) =
          make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
  __syncthreads();
  if (threadIdx.x == 0) vis[(static_cast<int64_t>(mb) * n_tq + m) * n_tk + n] = any_kept ? 1 : 0;
}

// From the block flags: per key tile n the query tiles with a kept position
// (under causality only m >= n), per query tile m the key tiles (causal: only
// j <= m), each list ascending.  One thread per list.
__global__ void __launch_bounds__(256) bwd_mask_lists_kernel(const uint8_t* __restrict__ vis,
                                                             int mB, int n_tq, int n_tk,
                                                             int causal, int* klist, int* kcount,
                                                             int* qlist, int* qcount) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  const int64_t nk = static_cast<int64_t>(mB) * n_tk;
  if (t < nk) {
    const int64_t mb = t / n_tk;
    const int n = static_cast<int>(t - mb * n_tk);
    int c = 0;
    for (int m = causal ? n : 0; m < n_tq; ++m)
      if (vis[(mb * n_tq + m) * n_tk + n]) klist[t * n_tq + c++] = m;
    kcount[t] = c;
  } else if (t < nk + static_cast<int64_t>(mB) * n_tq) {
    const int64_t u = t - nk;
    const int64_t mb = u / n_tq;
    const int m = static_cast<int>(u - mb * n_tq);
    const int jend = causal ? min(m + 1, n_tk) : n_tk;
    int c = 0;
    for (int j = 0; j < jend; ++j)
      if (vis[(mb * n_tq + m) * n_tk + j]) qlist[u * n_tk + c++] = j;
    qcount[u] = c;
  }
}

// The TH mask bits of this thread's columns (bit c: column TH grp + c) from a
// 4-word row of 128 bits.
__device__ __forceinline__ uint64_t mask_bits(const uint32_t* words, int grp) {
  if constexpr (TH == 64) {
    return *reinterpret_cast<const uint64_t*>(words + 2 * grp);
  } else {
    return words[grp];
  }
}

// ------------------------------------------------------------------ dK, dV

// Barrier indices of the dK/dV kernel (NS input stages).
template <int NS>
struct KvIdx {
  static constexpr int kvFull = 0;            // K, V tiles landed
  static constexpr int inFull = 1;            // [NS] Q, dO, -LSE log2(e), delta of a step landed
  static constexpr int inEmpty = 1 + NS;      // [NS] the step's last MMA (dK) completed
  static constexpr int sFull = 1 + 2 * NS;    // S^T in TMEM
  static constexpr int dpFull = sFull + 1;    // dP^T in TMEM
  static constexpr int pReady = sFull + 2;    // P^T written (elementwise arrivals)
  static constexpr int dsReady = sFull + 3;   // dS^T written (elementwise arrivals)
  static constexpr int dpFree = sFull + 4;    // dP^T read (elementwise arrivals)
  static constexpr int dkDone = sFull + 5;    // dV and dK MMAs of the step completed
  static constexpr int accFull = sFull + 6;   // every MMA of the unit completed
  static constexpr int drain = sFull + 7;
  static constexpr int n = sFull + 8;
};

// Unit of the dK/dV kernel: split s of key tile n of (b, h_kv).  The steps of
// a key tile -- every query head of the group (fastest) for every query tile
// m >= m_lo -- are cut into `splits` contiguous ranges, one per CTA; with more
// than one, each CTA writes fp32 partial sums that bwd_dkv_reduce_kernel adds
// up.  Key tiles vary slowest over the grid, so under causality the units
// with the most query tiles start first.
struct KvUnit {
  int n, s, b, hkv, kv_len, m_lo, t0, steps;  // steps [t0, t0 + steps) of the key tile
  const int* tiles;  // explicit mask: the query tiles to visit (else every m >= m_lo)
};

// Query tile of step t of a dK/dV unit.
__device__ __forceinline__ int kv_qtile(const KvUnit& w, int G, int t) {
  const int k = (w.t0 + t) / G;
  return w.tiles != nullptr ? w.tiles[k] : w.m_lo + k;
}

template <bool SPLIT, bool MASK>
__device__ __forceinline__ KvUnit kv_unit(const BwdTcParams& p, int unit) {
  const int per = p.B * p.Hkv;
  const int splits = SPLIT ? p.splits : 1;
  KvUnit w;
  w.n = unit / (per * splits);
  const int r = unit - w.n * per * splits;
  w.s = SPLIT ? r / per : 0;
  const int z = r - w.s * per;
  w.b = z / p.Hkv;
  w.hkv = z - w.b * p.Hkv;
  w.kv_len = kv_len_of(p, w.b);
  w.m_lo = p.causal ? w.n : 0;
  int total = (w.n * T < w.kv_len && w.m_lo < p.n_tq) ? p.G * (p.n_tq - w.m_lo) : 0;
  w.tiles = nullptr;
  if constexpr (MASK) {  // only the query tiles with a kept position
    const int64_t kl = (p.mask_shared ? 0 : static_cast<int64_t>(w.b)) * p.n_tk + w.n;
    w.tiles = p.klist + kl * p.n_tq;
    total = (w.n * T < w.kv_len) ? p.G * p.kcount[kl] : 0;
  }
  if constexpr (SPLIT) {
    const int chunk = (total + splits - 1) / splits;
    w.t0 = min(total, w.s * chunk);
    w.steps = min(total, w.t0 + chunk) - w.t0;
  } else {
    w.t0 = 0;
    w.steps = total;
  }
  return w;
}

template <int D>
__device__ void dkv_producer(const BwdTcParams& p, const KvUnit& w, const BBars& br, uint32_t smem,
                             const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                             const CUtensorMap* tm_v, const CUtensorMap* tm_do) {
  using C = BCfg<D>;
  constexpr int NS = C::kvStages;
  using I = KvIdx<NS>;
  if (w.steps == 0) return;
  const uint64_t pol_keep = ptx::policy_evict_last();    // Q, dO: read by every key tile
  const uint64_t pol_once = ptx::policy_evict_first();   // K, V: read once here
  ptx::mbar_arrive_expect_tx(br.bar(I::kvFull), 2 * C::kTile);
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    ptx::tma_load_4d_hint(smem + C::kvOffK + h * C::kSlab, tm_k, br.bar(I::kvFull), h * 64, w.n * T,
                          w.hkv, w.b, pol_once);
    ptx::tma_load_4d_hint(smem + C::kvOffV + h * C::kSlab, tm_v, br.bar(I::kvFull), h * 64, w.n * T,
                          w.hkv, w.b, pol_once);
  }
  int t = 0;
  for (; t < w.steps; ++t) {
    const uint32_t s = static_cast<uint32_t>(t % NS);
    if (!bwait(br, p.status, br.bar(I::inEmpty + s), ((t / NS) & 1) ^ 1, kRoleProducer)) break;
    const int mi = kv_qtile(w, p.G, t);
    const int hq = w.hkv * p.G + (w.t0 + t) % p.G;
    const uint32_t st = smem + C::kvOffIn + s * C::kvStageBytes;
    const uint32_t full = br.bar(I::inFull + s);
    ptx::mbar_arrive_expect_tx(full, 2 * C::kTile + 1024);
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
      ptx::tma_load_4d_hint(st + h * C::kSlab, tm_q, full, h * 64, mi * T, hq, w.b, pol_keep);
      ptx::tma_load_4d_hint(st + C::kTile + h * C::kSlab, tm_do, full, h * 64, mi * T, hq, w.b,
                            pol_keep);
    }
    const int64_t row = (static_cast<int64_t>(w.b) * p.Hq + hq) * p.Lqp + static_cast<int64_t>(mi) * T;
    bulk_load(st + 2 * C::kTile, p.nlse2 + row, T * 4, full);
    bulk_load(st + 2 * C::kTile + T * 4, p.delta + row, T * 4, full);
  }
  // never leave with a copy in flight: the last load of every stage
  bdrain(br.bar(I::kvFull), 0);
  for (int k = (t > NS ? t - NS : 0); k < t; ++k) bdrain(br.bar(I::inFull + k % NS), (k / NS) & 1);
}

// TMEM regions: step t's S^T goes to X_t and its dP^T to Y_t, with X and Y
// swapping every step (X_t = A for even t, B for odd; A = columns [0, 128),
// B = [128, 256)).  P^T(t) and dS^T(t) are both written into X_t (each
// elementwise warpgroup packs them into the first and second 32 columns of
// its 64-column block), so Y_t is free as soon as dP^T(t) has been read.
// Issue order: S^T(0), dP^T(0), then per step t
//   dV(t) once P^T(t) is written;
//   S^T(t+1) into Y_t once dP^T(t) has been read (during the dS^T(t) math);
//   dK(t) once dS^T(t) is written;
//   dP^T(t+1) into X_t once dV(t) and dK(t), which read X_t, have completed.
__device__ __forceinline__ uint32_t region_x(int t) { return (t & 1) ? 128u : 0u; }
__device__ __forceinline__ uint32_t region_y(int t) { return (t & 1) ? 0u : 128u; }

template <int D, bool BF16>
__device__ void dkv_mma(const BwdTcParams& p, const KvUnit& w, const BBars& br, uint32_t smem,
                        uint32_t tmem) {
  using C = BCfg<D>;
  constexpr int NS = C::kvStages;
  using I = KvIdx<NS>;
  constexpr uint32_t kFull = 0xffffffffu;
  auto stage = [&](int t) { return smem + C::kvOffIn + static_cast<uint32_t>(t % NS) * C::kvStageBytes; };
  auto wait = [&](int bar, uint32_t parity) {
    return __all_sync(kFull, bwait(br, p.status, br.bar(bar), parity, kRoleMma));
  };
  if (w.steps > 0) {
    // K-major operands: 1024 bytes between 8-row groups; MN-major: 64-column
    // slabs kSlab apart
    const uint64_t k_desc = ptx::sdesc_sw128(smem + C::kvOffK, 16, 1024);
    const uint64_t v_desc = ptx::sdesc_sw128(smem + C::kvOffV, 16, 1024);
    auto issue_s = [&](int t) {  // S^T(t) = K Q(t)^T into X_t
      ptx::tc_fence_after();
      if (elect()) mma_rows<D, BF16>(tmem + region_x(t), k_desc, ptx::sdesc_sw128(stage(t), 16, 1024));
      __syncwarp();
      commit(br.bar(I::sFull));
    };
    auto issue_dp = [&](int t) {  // dP^T(t) = V dO(t)^T into Y_t
      ptx::tc_fence_after();
      if (elect())
        mma_rows<D, BF16>(tmem + region_y(t), v_desc, ptx::sdesc_sw128(stage(t) + C::kTile, 16, 1024));
      __syncwarp();
      commit(br.bar(I::dpFull));
    };
    bool ok = wait(I::kvFull, 0) && wait(I::inFull, 0);
    if (ok) {
      issue_s(0);
      issue_dp(0);
    }
    for (int t = 0; ok && t < w.steps; ++t) {
      const uint32_t st = stage(t);
      const bool more = t + 1 < w.steps;
      // dV += P^T dO
      if (!(ok = wait(I::pReady, t & 1))) break;
      ptx::tc_fence_after();
      if (elect())
        mma_acc<D, BF16>(tmem + C::kColAcc0, tmem + region_x(t), TH,
                         ptx::sdesc_sw128(st + C::kTile, C::kSlab, 1024), t > 0);
      __syncwarp();
      if (more) {
        if (!(ok = wait(I::inFull + (t + 1) % NS, ((t + 1) / NS) & 1) && wait(I::dpFree, t & 1))) break;
        issue_s(t + 1);
      }
      // dK += dS^T Q (unscaled; sm_scale is applied in the epilogue)
      if (!(ok = wait(I::dsReady, t & 1))) break;
      ptx::tc_fence_after();
      if (elect())
        mma_acc<D, BF16>(tmem + C::kColAcc1, tmem + region_x(t) + TH / 2, TH,
                         ptx::sdesc_sw128(st, C::kSlab, 1024), t > 0);
      __syncwarp();
      commit(br.bar(I::dkDone));
      commit(br.bar(I::inEmpty + t % NS));
      if (more) {
        if (!(ok = wait(I::dkDone, t & 1))) break;
        issue_dp(t + 1);
      } else {
        commit(br.bar(I::accFull));
      }
    }
  }
  // every MMA issued here completes before TMEM is released
  commit(br.bar(I::drain));
  bdrain(br.bar(I::drain), 0);
}

// Store the first `ncols` (a multiple of 8, at most 32) columns of a
// 32-column chunk of an fp32 TMEM row, times `mul`, as 16-bit values
// (16-byte stores; the thread owns the whole row).
template <bool BF16>
__device__ __forceinline__ void store_chunk(uint16_t* dst, const uint32_t (&r)[32], float mul,
                                            int ncols) {
  uint32_t o16[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    o16[i] = pk2<BF16>(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (q * 8 < ncols)
      reinterpret_cast<uint4*>(dst)[q] = make_uint4(o16[4 * q], o16[4 * q + 1], o16[4 * q + 2], o16[4 * q + 3]);
}

// Columns of [c_lo, c_lo + part) inside a row of dg columns.
__device__ __forceinline__ int cols_in(int dg, int c_lo, int part) {
  const int n = dg - c_lo;
  return n < 0 ? 0 : (n > part ? part : n);
}

// Elementwise warpgroups of the dK/dV kernel.  Thread: key row `row` of the
// tile (TMEM lane), query columns [TH grp, TH grp + TH) of every step.
//   P^T = exp2(S^T sm_scale log2(e) - LSE log2(e)), zero where the key is at
//   or beyond valid_len[b] or (diagonal tile, causal) after the query; kept in
//   fp32 registers for dS and written to TMEM as 16-bit pairs over the first
//   TH/2 S^T columns of the thread's block;
//   dS^T = P^T (dP^T - delta), written over the next TH/2.
// Epilogue: the first half of the warpgroups write dV, the second dK (x
// sm_scale), each a D / (kGroups / 2)-column part of the row.
template <int D, bool BF16, bool SPLIT, bool MASK>
__device__ void dkv_elementwise(const BwdTcParams& p, const KvUnit& w, const BBars& br,
                                uint32_t smem, uint32_t tmem) {
  using C = BCfg<D>;
  constexpr int NS = C::kvStages;
  using I = KvIdx<NS>;
  constexpr uint32_t kFull = 0xffffffffu;
  const int row = threadIdx.x & 127;
  const int grp = static_cast<int>(threadIdx.x) >> 7;
  const uint32_t lane_addr = (((threadIdx.x >> 5) & 3u) * 32u) << 16;
  const uint32_t t_grp = tmem + lane_addr + grp * TH;  // + region_x(t) / region_y(t)
  const bool key_ok = w.n * T + row < w.kv_len;
  const uint64_t sc2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
  bool ok = true;
  for (int t = 0; ok && t < w.steps; ++t) {
    const uint32_t s = static_cast<uint32_t>(t % NS);
    const uint32_t st = smem + C::kvOffIn + s * C::kvStageBytes;
    const int mi = MASK ? kv_qtile(w, p.G, t) : w.m_lo + ((SPLIT ? w.t0 : 0) + t) / p.G;
    // explicit mask: this key row's bits over the query tile (loaded first)
    uint64_t mbits = ~0ull;
    if constexpr (MASK) {
      const int j = w.n * T + row;
      const int64_t mb = p.mask_shared ? 0 : w.b;
      mbits = j < p.Lk ? mask_bits(p.cbits + ((mb * p.Lk + j) * p.n_tq + mi) * 4, grp) : 0ull;
    }
    // the stage's -LSE log2(e) and delta are read from shared memory
    ok = __all_sync(kFull, bwait(br, p.status, br.bar(I::inFull + s), (t / NS) & 1, kRoleSoftmax));
    if (ok) ok = __all_sync(kFull, bwait(br, p.status, br.bar(I::sFull), t & 1, kRoleSoftmax));
    if (!ok) break;
    const uint32_t t_s = t_grp + region_x(t);   // S^T(t), then P^T(t) and dS^T(t)
    const uint32_t t_dp = t_grp + region_y(t);  // dP^T(t)
    ptx::tc_fence_after();
    uint32_t r[TH];
    ld_th(t_s, r);
    float pr[TH];
    const uint32_t nl_addr = st + 2 * C::kTile + grp * TH * 4;
#pragma unroll
    for (int c = 0; c < TH; c += 4) {
      const uint4 nl = ptx::ld_shared_v4(nl_addr + c * 4);
      const uint64_t x01 = ptx::f2_fma(ptx::f2_pack(__uint_as_float(r[c]), __uint_as_float(r[c + 1])),
                                       sc2, ptx::f2_pack(__uint_as_float(nl.x), __uint_as_float(nl.y)));
      const uint64_t x23 = ptx::f2_fma(ptx::f2_pack(__uint_as_float(r[c + 2]), __uint_as_float(r[c + 3])),
                                       sc2, ptx::f2_pack(__uint_as_float(nl.z), __uint_as_float(nl.w)));
      float x0, x1, x2, x3;
      ptx::f2_unpack(x01, x0, x1);
      ptx::f2_unpack(x23, x2, x3);
      pr[c] = ptx::ex2_approx(x0);
      pr[c + 1] = ptx::ex2_approx(x1);
      pr[c + 2] = ptx::ex2_approx(x2);
      pr[c + 3] = ptx::ex2_approx(x3);
    }
    // columns c < cmin hold queries before this key (diagonal tile, causal)
    const int cmin = key_ok ? ((p.causal && mi == w.n) ? row - grp * TH : 0) : TH;
    if (cmin > 0) {
#pragma unroll
      for (int c = 0; c < TH; ++c) pr[c] = c < cmin ? 0.f : pr[c];
    }
    if constexpr (MASK) {
#pragma unroll
      for (int c = 0; c < TH; ++c) pr[c] = ((mbits >> c) & 1ull) ? pr[c] : 0.f;
    }
    uint32_t pk[TH / 2];
#pragma unroll
    for (int i = 0; i < TH / 2; ++i) pk[i] = pk2<BF16>(pr[2 * i], pr[2 * i + 1]);
    st_th2(t_s, pk);
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
    ptx::mbar_arrive(br.bar(I::pReady));

    ok = __all_sync(kFull, bwait(br, p.status, br.bar(I::dpFull), t & 1, kRoleSoftmax));
    if (!ok) break;
    ptx::tc_fence_after();
    ld_th(t_dp, r);
    ptx::tc_fence_before();
    ptx::mbar_arrive(br.bar(I::dpFree));  // the MMA issuer may now write S^T(t+1) there
    const uint32_t dl_addr = st + 2 * C::kTile + T * 4 + grp * TH * 4;
#pragma unroll
    for (int c = 0; c < TH; c += 4) {
      const uint4 dl = ptx::ld_shared_v4(dl_addr + c * 4);
      const uint64_t d01 = ptx::f2_mul(
          ptx::f2_pack(pr[c], pr[c + 1]),
          ptx::f2_sub(ptx::f2_pack(__uint_as_float(r[c]), __uint_as_float(r[c + 1])),
                      ptx::f2_pack(__uint_as_float(dl.x), __uint_as_float(dl.y))));
      const uint64_t d23 = ptx::f2_mul(
          ptx::f2_pack(pr[c + 2], pr[c + 3]),
          ptx::f2_sub(ptx::f2_pack(__uint_as_float(r[c + 2]), __uint_as_float(r[c + 3])),
                      ptx::f2_pack(__uint_as_float(dl.z), __uint_as_float(dl.w))));
      float a, b2, c2, d2;
      ptx::f2_unpack(d01, a, b2);
      ptx::f2_unpack(d23, c2, d2);
      pk[c / 2] = pk2<BF16>(a, b2);
      pk[c / 2 + 1] = pk2<BF16>(c2, d2);
    }
    st_th2(t_s + TH / 2, pk);
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
    ptx::mbar_arrive(br.bar(I::dsReady));
  }
  if (!ok) return;
  // epilogue: warpgroups [0, kGroups/2) the dV row, the others the dK row,
  // kPart columns each
  constexpr int kPart = D / (kGroups / 2);
  const bool is_dk = grp >= kGroups / 2;
  const int c_lo = (grp % (kGroups / 2)) * kPart;
  const int j = w.n * T + row;
  const int nv = j < p.Lk ? cols_in(p.dg, c_lo, kPart) : 0;  // columns this thread stores
  const Strides& so = is_dk ? p.sdk : p.sdv;
  uint16_t* dst = static_cast<uint16_t*>(is_dk ? p.dk : p.dv) + w.b * so.b + w.hkv * so.h +
                  static_cast<int64_t>(j) * so.l + c_lo;
  // split key tiles: unscaled fp32 partial rows, summed by bwd_dkv_reduce_kernel
  float* part = p.part + ((static_cast<int64_t>(w.s) * 2 + (is_dk ? 1 : 0)) * p.B * p.Hkv * p.Lk +
                          (static_cast<int64_t>(w.b) * p.Hkv + w.hkv) * p.Lk + j) * p.dg + c_lo;
  constexpr bool split = SPLIT;
  if (w.steps == 0) {  // no query sees these keys (in this split)
    for (int c = 0; c < nv / 8; ++c) {
      if (split) {
        reinterpret_cast<float4*>(part)[2 * c] = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4*>(part)[2 * c + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        reinterpret_cast<uint4*>(dst)[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }
  if (!__all_sync(kFull, bwait(br, p.status, br.bar(I::accFull), 0, kRoleEpilogue))) return;
  ptx::tc_fence_after();
  const uint32_t t_acc = tmem + lane_addr + (is_dk ? C::kColAcc1 : C::kColAcc0) + c_lo;
  const float mul = is_dk ? p.sm_scale : 1.f;
#pragma unroll 1
  for (int c0 = 0; c0 < kPart; c0 += 32) {
    uint32_t r[32];
    ptx::tmem_ld32(t_acc + c0, r);
    if (split) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c0 + q * 4 < nv)
          reinterpret_cast<float4*>(part + c0)[q] =
              make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                          __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
    } else {
      store_chunk<BF16>(dst + c0, r, mul, nv - c0);
    }
  }
}

// dV and dK of split key tiles: the `splits` fp32 partials of every element
// added in split order (deterministic), dK times sm_scale, rounded once to
// the input dtype.  One thread per 8 consecutive elements of a row.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_dkv_reduce_kernel(const BwdTcParams p) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hkv * p.Lk;
  const int64_t per_row = p.dg / 8;
  const int64_t v = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (v >= 2 * rows * per_row) return;
  const int which = static_cast<int>(v / (rows * per_row));  // 0: dV, 1: dK
  const int64_t e = v - which * rows * per_row;
  const int64_t row = e / per_row;
  const int col = static_cast<int>(e - row * per_row) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int sp = 0; sp < p.splits; ++sp) {
    const float4* src = reinterpret_cast<const float4*>(
        p.part + ((static_cast<int64_t>(sp) * 2 + which) * rows + row) * p.dg + col);
    const float4 a = src[0], b = src[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  const float mul = which ? p.sm_scale : 1.f;
  const int64_t z = row / p.Lk;  // b * Hkv + h_kv
  const int64_t j = row - z * p.Lk;
  const int64_t sb = which ? p.sdk.b : p.sdv.b;
  const int64_t sh = which ? p.sdk.h : p.sdv.h;
  const int64_t sl = which ? p.sdk.l : p.sdv.l;
  uint16_t* dst = static_cast<uint16_t*>(which ? p.dk : p.dv) + (z / p.Hkv) * sb + (z % p.Hkv) * sh +
                  j * sl + col;
  *reinterpret_cast<uint4*>(dst) = make_uint4(pk2<BF16>(acc[0] * mul, acc[1] * mul),
                                              pk2<BF16>(acc[2] * mul, acc[3] * mul),
                                              pk2<BF16>(acc[4] * mul, acc[5] * mul),
                                              pk2<BF16>(acc[6] * mul, acc[7] * mul));
}

// One CTA of the dK/dV kernel on unit `unit`.  SPLIT: key tiles split over
// several CTAs (p.splits > 1), fp32 partial rows.  MASK: an explicit mask.
template <int D, bool BF16, bool SPLIT, bool MASK>
__device__ __forceinline__ void dkv_cta(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                        const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                        const BwdTcParams& p, int unit) {
  using C = BCfg<D>;
  using I = KvIdx<C::kvStages>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const BBars br{smem + C::kvOffBar, I::n};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const KvUnit w = kv_unit<SPLIT, MASK>(p, unit);
  if (threadIdx.x == 0) {
    for (int i = 0; i < I::n; ++i) {
      const bool ew = (i == I::pReady || i == I::dsReady || i == I::dpFree);
      ptx::mbar_init(br.bar(i), ew ? kEwThreads : 1);
    }
    ptx::st_shared_volatile(br.abort_word(), 0u);
    ptx::fence_barrier_init();
    if (p.valid_len != nullptr && w.n == 0 && w.hkv == 0) {
      const int vl = p.valid_len[w.b];
      if (vl < 0 || vl > p.Lk) atomicOr(p.status, kStatusValidLenClamped);
    }
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::prefetch_tensormap(tm_q);
    ptx::prefetch_tensormap(tm_do);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(br.tmem_word(), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ptx::ld_shared_volatile(br.tmem_word());
  if (warp == kLoadWarp) {
    if (lane == 0) dkv_producer<D>(p, w, br, smem, tm_q, tm_k, tm_v, tm_do);
  } else if (warp == kMmaWarp) {
    dkv_mma<D, BF16>(p, w, br, smem, tmem);
  } else {
    dkv_elementwise<D, BF16, SPLIT, MASK>(p, w, br, smem, tmem);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ dQ

// Barrier indices of the dQ kernel (KS K stages, VS V stages, two dS buffers).
template <int KS, int VS>
struct QIdx {
  static constexpr int qdFull = 0;                // Q, dO tiles landed
  static constexpr int kFull = 1;                 // [KS] K tile landed
  static constexpr int kEmpty = 1 + KS;           // [KS] its last MMA (dQ) completed
  static constexpr int vFull = 1 + 2 * KS;        // [VS] V tile landed
  static constexpr int vEmpty = 1 + 2 * KS + VS;  // [VS] its MMA (dP) completed
  static constexpr int sFull = 1 + 2 * KS + 2 * VS;  // S in TMEM
  static constexpr int dpFull = sFull + 1;   // dP in TMEM
  static constexpr int sFree = sFull + 2;    // S read (256 arrivals)
  static constexpr int dpFree = sFull + 3;   // dP read (256 arrivals)
  static constexpr int dsReady = sFull + 4;  // [2] dS written into buffer b (256 arrivals)
  static constexpr int dqDone = sFull + 6;   // [2] dQ MMA reading buffer b completed
  static constexpr int accFull = sFull + 8;
  static constexpr int drain = sFull + 9;
  static constexpr int n = sFull + 10;
};

// Unit of the dQ kernel: query tile m of (b, h_q), key tiles [0, steps).
// Query tiles vary slowest, the last (longest under causality) first.
struct QUnit {
  int m, b, hq, hkv, kv_len, steps;
  const int* tiles;  // explicit mask: the key tiles to visit (else 0, 1, ...)
};

// Key tile of step j of a dQ unit.
__device__ __forceinline__ int q_ktile(const QUnit& w, int j) {
  return w.tiles != nullptr ? w.tiles[j] : j;
}

template <bool MASK>
__device__ __forceinline__ QUnit q_unit(const BwdTcParams& p, int unit) {
  const int per = p.B * p.Hq;
  const int u = unit / per;
  const int z = unit - u * per;
  QUnit w;
  w.m = p.n_tq - 1 - u;
  w.b = z / p.Hq;
  w.hq = z - w.b * p.Hq;
  w.hkv = w.hq / p.G;
  w.kv_len = kv_len_of(p, w.b);
  const int kt = (w.kv_len + T - 1) / T;
  w.steps = min(p.causal ? min(w.m + 1, p.n_tk) : p.n_tk, kt);
  w.tiles = nullptr;
  if constexpr (MASK) {  // the listed key tiles below the valid_len cut
    const int64_t ql = (p.mask_shared ? 0 : static_cast<int64_t>(w.b)) * p.n_tq + w.m;
    w.tiles = p.qlist + ql * p.n_tk;
    const int cnt = p.qcount[ql];
    int k = 0;
    while (k < cnt && w.tiles[k] < kt) ++k;
    w.steps = k;
  }
  return w;
}

template <int D>
__device__ void dq_producer(const BwdTcParams& p, const QUnit& w, const BBars& br, uint32_t smem,
                            const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                            const CUtensorMap* tm_v, const CUtensorMap* tm_do) {
  using C = BCfg<D>;
  constexpr int KS = C::qKStages, VS = C::qVStages;
  using I = QIdx<KS, VS>;
  if (w.steps == 0) return;
  const uint64_t pol_keep = ptx::policy_evict_last();   // K, V: read by every query tile
  const uint64_t pol_once = ptx::policy_evict_first();  // Q, dO: read once here
  ptx::mbar_arrive_expect_tx(br.bar(I::qdFull), 2 * C::kTile);
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    ptx::tma_load_4d_hint(smem + C::qOffQ + h * C::kSlab, tm_q, br.bar(I::qdFull), h * 64, w.m * T,
                          w.hq, w.b, pol_once);
    ptx::tma_load_4d_hint(smem + C::qOffDO + h * C::kSlab, tm_do, br.bar(I::qdFull), h * 64,
                          w.m * T, w.hq, w.b, pol_once);
  }
  // K(j) then V(j): K's slot frees after dQ(j - KS), V's after dP(j - VS),
  // which completes earlier
  int nk = 0, nv = 0;  // K and V tiles issued
  for (int j = 0; j < w.steps; ++j) {
    const int kj = q_ktile(w, j);  // the key tile of step j
    if (!bwait(br, p.status, br.bar(I::kEmpty + j % KS), ((j / KS) & 1) ^ 1, kRoleProducer)) break;
    const uint32_t kf = br.bar(I::kFull + j % KS);
    ptx::mbar_arrive_expect_tx(kf, C::kTile);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      ptx::tma_load_4d_hint(smem + C::qOffK + (j % KS) * C::kTile + h * C::kSlab, tm_k, kf, h * 64,
                            kj * T, w.hkv, w.b, pol_keep);
    ++nk;
    if (!bwait(br, p.status, br.bar(I::vEmpty + j % VS), ((j / VS) & 1) ^ 1, kRoleProducer)) break;
    const uint32_t vf = br.bar(I::vFull + j % VS);
    ptx::mbar_arrive_expect_tx(vf, C::kTile);
#pragma unroll
    for (int h = 0; h < D / 64; ++h)
      ptx::tma_load_4d_hint(smem + C::qOffV + (j % VS) * C::kTile + h * C::kSlab, tm_v, vf, h * 64,
                            kj * T, w.hkv, w.b, pol_keep);
    ++nv;
  }
  bdrain(br.bar(I::qdFull), 0);
  for (int k = (nk > KS ? nk - KS : 0); k < nk; ++k) bdrain(br.bar(I::kFull + k % KS), (k / KS) & 1);
  for (int k = (nv > VS ? nv - VS : 0); k < nv; ++k) bdrain(br.bar(I::vFull + k % VS), (k / VS) & 1);
}

// Issue order: S(0), dP(0), then per key tile j
//   S(j+1) once S(j) has been read, dP(j+1) once dP(j) has been read,
//   dQ += dS(j) K(j) once dS(j) is written (dS buffer j % 2);
// the elementwise warps compute dS(j) while S(j+1) and dP(j+1) run.
template <int D, bool BF16>
__device__ void dq_mma(const BwdTcParams& p, const QUnit& w, const BBars& br, uint32_t smem,
                       uint32_t tmem) {
  using C = BCfg<D>;
  constexpr int KS = C::qKStages, VS = C::qVStages;
  using I = QIdx<KS, VS>;
  constexpr uint32_t kFull = 0xffffffffu;
  auto k_tile = [&](int j) { return smem + C::qOffK + static_cast<uint32_t>(j % KS) * C::kTile; };
  auto v_tile = [&](int j) { return smem + C::qOffV + static_cast<uint32_t>(j % VS) * C::kTile; };
  auto wait = [&](int bar, uint32_t parity) {
    return __all_sync(kFull, bwait(br, p.status, br.bar(bar), parity, kRoleMma));
  };
  if (w.steps > 0) {
    const uint64_t q_desc = ptx::sdesc_sw128(smem + C::qOffQ, 16, 1024);
    const uint64_t do_desc = ptx::sdesc_sw128(smem + C::qOffDO, 16, 1024);
    auto issue_s = [&](int j) {  // S(j) = Q K(j)^T
      ptx::tc_fence_after();
      if (elect()) mma_rows<D, BF16>(tmem + C::kColS, q_desc, ptx::sdesc_sw128(k_tile(j), 16, 1024));
      __syncwarp();
      commit(br.bar(I::sFull));
    };
    auto issue_dp = [&](int j) {  // dP(j) = dO V(j)^T; V(j) is free once it completes
      ptx::tc_fence_after();
      if (elect())
        mma_rows<D, BF16>(tmem + C::kColDP, do_desc, ptx::sdesc_sw128(v_tile(j), 16, 1024));
      __syncwarp();
      commit(br.bar(I::dpFull));
      commit(br.bar(I::vEmpty + j % VS));
    };
    bool ok = wait(I::qdFull, 0) && wait(I::kFull, 0);
    if (ok) issue_s(0);
    if (ok && (ok = wait(I::vFull, 0))) issue_dp(0);
    for (int j = 0; ok && j < w.steps; ++j) {
      const int b = j & 1;
      if (j + 1 < w.steps) {
        if (!(ok = wait(I::kFull + (j + 1) % KS, ((j + 1) / KS) & 1) && wait(I::sFree, j & 1))) break;
        issue_s(j + 1);
        if (!(ok = wait(I::vFull + (j + 1) % VS, ((j + 1) / VS) & 1) && wait(I::dpFree, j & 1))) break;
        issue_dp(j + 1);
      }
      if (!(ok = wait(I::dsReady + b, (j >> 1) & 1))) break;
      ptx::tc_fence_after();
      if (elect())
        mma_acc<D, BF16>(tmem + C::kColAcc0, tmem + C::kColAcc1 + b * (T / 2), TH / 2,
                         ptx::sdesc_sw128(k_tile(j), C::kSlab, 1024), j > 0);
      __syncwarp();
      commit(br.bar(I::dqDone + b));
      commit(br.bar(I::kEmpty + j % KS));
      if (j + 1 == w.steps) commit(br.bar(I::accFull));
    }
  }
  commit(br.bar(I::drain));
  bdrain(br.bar(I::drain), 0);
}

// Elementwise warpgroups of the dQ kernel.  Thread: query row `row` (TMEM
// lane), key columns [TH grp, TH grp + TH) of every key tile; its LSE and
// delta are two registers.  P = exp2(S sm_scale log2(e) - LSE log2(e)), zero
// for keys at or beyond valid_len[b] and (diagonal tile, causal) after the
// query; dS = P (dP - delta) into dS buffer j % 2 (16-bit pairs) once the dQ
// MMA of key tile j - 2 has read it.  Epilogue: warpgroup g < kEpi writes dQ
// columns [g D/kEpi, (g + 1) D/kEpi) of its row, times sm_scale.
template <int D, bool BF16, bool MASK>
__device__ void dq_elementwise(const BwdTcParams& p, const QUnit& w, const BBars& br, uint32_t tmem) {
  using C = BCfg<D>;
  using I = QIdx<C::qKStages, C::qVStages>;
  constexpr uint32_t kFull = 0xffffffffu;
  const int row = threadIdx.x & 127;
  const int grp = static_cast<int>(threadIdx.x) >> 7;
  const uint32_t lane_addr = (((threadIdx.x >> 5) & 3u) * 32u) << 16;
  const uint32_t t_s = tmem + lane_addr + C::kColS + grp * TH;
  const uint32_t t_dp = tmem + lane_addr + C::kColDP + grp * TH;
  const uint32_t t_ds = tmem + lane_addr + C::kColAcc1 + grp * (TH / 2);  // + (j % 2) * 64
  const int64_t g_row = (static_cast<int64_t>(w.b) * p.Hq + w.hq) * p.Lqp + static_cast<int64_t>(w.m) * T + row;
  const float nl = w.steps > 0 ? p.nlse2[g_row] : 0.f;
  const float dl = w.steps > 0 ? p.delta[g_row] : 0.f;
  const uint64_t sc2 = ptx::f2_pack(p.scale_log2, p.scale_log2);
  const uint64_t nl2 = ptx::f2_pack(nl, nl);
  const uint64_t dl2 = ptx::f2_pack(dl, dl);
  bool ok = true;
  for (int j = 0; ok && j < w.steps; ++j) {
    // explicit mask: this query row's bits over the key tile (loaded first)
    uint64_t mbits = ~0ull;
    if constexpr (MASK) {
      const int i = w.m * T + row;
      const int64_t mb = p.mask_shared ? 0 : w.b;
      mbits = i < p.Lq ? mask_bits(p.rbits + ((mb * p.Lq + i) * p.n_tk + q_ktile(w, j)) * 4, grp)
                       : 0ull;
    }
    ok = __all_sync(kFull, bwait(br, p.status, br.bar(I::sFull), j & 1, kRoleSoftmax));
    if (!ok) break;
    ptx::tc_fence_after();
    uint32_t r[TH];
    ld_th(t_s, r);
    float pr[TH];
#pragma unroll
    for (int c = 0; c < TH; c += 2) {
      const uint64_t x = ptx::f2_fma(ptx::f2_pack(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), sc2, nl2);
      float x0, x1;
      ptx::f2_unpack(x, x0, x1);
      pr[c] = ptx::ex2_approx(x0);
      pr[c + 1] = ptx::ex2_approx(x1);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(br.bar(I::sFree));
    // visible key columns: c < climit (causal diagonal tile; last key tile)
    int climit = TH;
    const int kj = MASK ? q_ktile(w, j) : j;  // the key tile of step j
    if (p.causal && kj == w.m) climit = min(climit, row - grp * TH + 1);
    climit = min(climit, w.kv_len - kj * T - grp * TH);
    if (climit < TH) {
#pragma unroll
      for (int c = 0; c < TH; ++c) pr[c] = c < climit ? pr[c] : 0.f;
    }
    if constexpr (MASK) {
#pragma unroll
      for (int c = 0; c < TH; ++c) pr[c] = ((mbits >> c) & 1ull) ? pr[c] : 0.f;
    }
    ok = __all_sync(kFull, bwait(br, p.status, br.bar(I::dpFull), j & 1, kRoleSoftmax));
    if (!ok) break;
    ptx::tc_fence_after();
    ld_th(t_dp, r);
    ptx::tc_fence_before();
    ptx::mbar_arrive(br.bar(I::dpFree));
    uint32_t pk[TH / 2];
#pragma unroll
    for (int c = 0; c < TH; c += 2) {
      const uint64_t d = ptx::f2_mul(
          ptx::f2_pack(pr[c], pr[c + 1]),
          ptx::f2_sub(ptx::f2_pack(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), dl2));
      float a, b2;
      ptx::f2_unpack(d, a, b2);
      pk[c / 2] = pk2<BF16>(a, b2);
    }
    // buffer j % 2 held dS(j-2): wait until dQ(j-2) has read it
    const int b = j & 1;
    if (j >= 2)
      ok = __all_sync(kFull, bwait(br, p.status, br.bar(I::dqDone + b), ((j >> 1) - 1) & 1, kRoleSoftmax));
    if (!ok) break;
    ptx::tc_fence_after();
    st_th2(t_ds + b * (T / 2), pk);
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
    ptx::mbar_arrive(br.bar(I::dsReady + b));
  }
  // epilogue: kEpi warpgroups, kPart columns each (32-column loads)
  constexpr int kEpi = (kGroups < D / 32) ? kGroups : D / 32;
  constexpr int kPart = D / kEpi;
  if (!ok || grp >= kEpi) return;
  const int i = w.m * T + row;
  const int nv = i < p.Lq ? cols_in(p.dg, grp * kPart, kPart) : 0;  // columns this thread stores
  uint16_t* dst = static_cast<uint16_t*>(p.dq) + w.b * p.sdq.b + w.hq * p.sdq.h +
                  static_cast<int64_t>(i) * p.sdq.l + grp * kPart;
  if (w.steps == 0) {  // no visible key: dQ = 0
    for (int c = 0; c < nv / 8; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  if (!__all_sync(kFull, bwait(br, p.status, br.bar(I::accFull), 0, kRoleEpilogue))) return;
  ptx::tc_fence_after();
  const uint32_t t_acc = tmem + lane_addr + C::kColAcc0 + grp * kPart;
#pragma unroll 1
  for (int c0 = 0; c0 < kPart; c0 += 32) {
    uint32_t r[32];
    ptx::tmem_ld32(t_acc + c0, r);
    store_chunk<BF16>(dst + c0, r, p.sm_scale, nv - c0);
  }
}

// One CTA of the dQ kernel on unit `unit`.
template <int D, bool BF16, bool MASK>
__device__ __forceinline__ void dq_cta(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                       const CUtensorMap* tm_v, const CUtensorMap* tm_do,
                                       const BwdTcParams& p, int unit) {
  using C = BCfg<D>;
  using I = QIdx<C::qKStages, C::qVStages>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const BBars br{smem + C::qOffBar, I::n};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const QUnit w = q_unit<MASK>(p, unit);
  if (threadIdx.x == 0) {
    for (int i = 0; i < I::n; ++i) {
      const bool ew = (i == I::sFree || i == I::dpFree || i == I::dsReady || i == I::dsReady + 1);
      ptx::mbar_init(br.bar(i), ew ? kEwThreads : 1);
    }
    ptx::st_shared_volatile(br.abort_word(), 0u);
    ptx::fence_barrier_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::prefetch_tensormap(tm_k);
    ptx::prefetch_tensormap(tm_v);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(br.tmem_word(), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ptx::ld_shared_volatile(br.tmem_word());
  if (warp == kLoadWarp) {
    if (lane == 0) dq_producer<D>(p, w, br, smem, tm_q, tm_k, tm_v, tm_do);
  } else if (warp == kMmaWarp) {
    dq_mma<D, BF16>(p, w, br, smem, tmem);
  } else {
    dq_elementwise<D, BF16, MASK>(p, w, br, tmem);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// The dK/dV and dQ kernels: the same CTA bodies, launched one after the
// other, or (ATTN_BWD_FUSED) as one grid -- the dK/dV units first, then the
// dQ units -- so that dQ CTAs take the SMs the dK/dV kernel's tail leaves idle.
#ifndef ATTN_BWD_FUSED
#define ATTN_BWD_FUSED 1
#endif

template <int D, bool BF16, bool SPLIT, bool MASK>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do, const BwdTcParams p) {
  dkv_cta<D, BF16, SPLIT, MASK>(&tm_q, &tm_k, &tm_v, &tm_do, p, static_cast<int>(blockIdx.x));
}

template <int D, bool BF16, bool MASK>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do, const BwdTcParams p) {
  dq_cta<D, BF16, MASK>(&tm_q, &tm_k, &tm_v, &tm_do, p, static_cast<int>(blockIdx.x));
}

template <int D, bool BF16, bool SPLIT, bool MASK>
__global__ void __launch_bounds__(kThreadsB, 1)
    bwd_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_do, const BwdTcParams p,
                        int n_dkv) {
  const int u = static_cast<int>(blockIdx.x);
  if (u < n_dkv) {
    dkv_cta<D, BF16, SPLIT, MASK>(&tm_q, &tm_k, &tm_v, &tm_do, p, u);
  } else {
    dq_cta<D, BF16, MASK>(&tm_q, &tm_k, &tm_v, &tm_do, p, u - n_dkv);
  }
}

// The pre-pass for rows of DR columns in memory.
template <int DR, bool BF16>
void launch_prep(const BwdTcParams& p, const void* o, const Strides& so, const void* dO,
                 const Strides& sdo, const float* lse, float* nlse2, float* delta,
                 cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.Lqp;
  constexpr int kRowsPerBlock = 8 * (32 / (DR / 8));
  bwd_tc_prep_kernel<DR, BF16><<<static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock),
                                 256, 0, stream>>>(o, dO, lse, nlse2, delta, p.Hq, p.Lq, p.Lqp, rows,
                                                   so, sdo);
}

template <int D, bool BF16, bool MASK>
cudaError_t launch_bwd_tc_d(const CUtensorMap (&maps)[4], const BwdTcParams& p, const void* o,
                            const Strides& so, const void* dO, const Strides& sdo,
                            const float* lse, float* nlse2, float* delta, cudaStream_t stream) {
  using C = BCfg<D>;
  if (p.dg == 16) {
    launch_prep<16, BF16>(p, o, so, dO, sdo, lse, nlse2, delta, stream);
  } else if (p.dg == 32) {
    launch_prep<32, BF16>(p, o, so, dO, sdo, lse, nlse2, delta, stream);
  } else {
    launch_prep<D, BF16>(p, o, so, dO, sdo, lse, nlse2, delta, stream);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n_dkv = p.n_tk * p.B * p.Hkv * p.splits;
  const int n_dq = p.n_tq * p.B * p.Hq;
  if constexpr (ATTN_BWD_FUSED != 0) {
    constexpr int smem = C::kvSmem > C::qSmem ? C::kvSmem : C::qSmem;
    auto fused = p.splits > 1 ? bwd_fused_tc_kernel<D, BF16, true, MASK>
                              : bwd_fused_tc_kernel<D, BF16, false, MASK>;
    e = cudaFuncSetAttribute(fused, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    fused<<<static_cast<unsigned>(n_dkv + n_dq), kThreadsB, smem, stream>>>(maps[0], maps[1], maps[2],
                                                                           maps[3], p, n_dkv);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else {
    auto dkv = p.splits > 1 ? bwd_dkv_tc_kernel<D, BF16, true, MASK>
                            : bwd_dkv_tc_kernel<D, BF16, false, MASK>;
    e = cudaFuncSetAttribute(dkv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kvSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_dq_tc_kernel<D, BF16, MASK>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::qSmem);
    if (e != cudaSuccess) return e;
    dkv<<<static_cast<unsigned>(n_dkv), kThreadsB, C::kvSmem, stream>>>(maps[0], maps[1], maps[2],
                                                                       maps[3], p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq_tc_kernel<D, BF16, MASK><<<static_cast<unsigned>(n_dq), kThreadsB, C::qSmem, stream>>>(
        maps[0], maps[1], maps[2], maps[3], p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.splits > 1) {  // after every dK/dV CTA has written its partials
    const int64_t vecs = 2 * static_cast<int64_t>(p.B) * p.Hkv * p.Lk * (p.dg / 8);
    bwd_dkv_reduce_kernel<BF16><<<static_cast<unsigned>((vecs + 255) / 256), 256, 0, stream>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

template <int D, bool BF16>
cudaError_t launch_bwd_tc_m(const CUtensorMap (&maps)[4], const BwdTcParams& p, const void* o,
                            const Strides& so, const void* dO, const Strides& sdo,
                            const float* lse, float* nlse2, float* delta, cudaStream_t stream) {
  return p.rbits != nullptr
             ? launch_bwd_tc_d<D, BF16, true>(maps, p, o, so, dO, sdo, lse, nlse2, delta, stream)
             : launch_bwd_tc_d<D, BF16, false>(maps, p, o, so, dO, sdo, lse, nlse2, delta, stream);
}

}  // namespace

// CTAs per key tile of the dK/dV kernel: 1 when its (key tile, b, h_kv) units
// alone fill four waves of the GPU, else enough splits of each key tile's
// steps to do so (at most 16) -- with few K/V heads (MQA), one CTA per key
// tile would run every query head of the group and leave SMs idle.
int bwd_tc_splits(int B, int Hkv, int Lk, int num_sms) {
  const int64_t units = static_cast<int64_t>((Lk + T - 1) / T) * B * Hkv;
  const int64_t target = 4 * static_cast<int64_t>(num_sms > 0 ? num_sms : 1);
  if (units >= target) return 1;
  const int64_t s = (target + units - 1) / units;
  return static_cast<int>(s < 16 ? s : 16);
}

// Workspace: -LSE log2(e) and delta [B*Hq, Lq rounded up to 128], the fp32
// partials of split key tiles, the explicit mask's row and column bits.
int64_t bwd_tc_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D, int num_sms,
                               int mask_batches) {
  const int64_t lqp = (static_cast<int64_t>(Lq) + T - 1) / T * T;
  const int64_t lkp = (static_cast<int64_t>(Lk) + T - 1) / T * T;
  const int splits = bwd_tc_splits(B, Hkv, Lk, num_sms);
  const int64_t part = splits > 1 ? static_cast<int64_t>(splits) * 2 * B * Hkv * Lk * D * 4 : 0;
  const int64_t bits = static_cast<int64_t>(mask_batches) * (Lq * (lkp / 8) + Lk * (lqp / 8));
  const int64_t ntq = lqp / T, ntk = lkp / T;
  const int64_t flags = (static_cast<int64_t>(mask_batches) * ntq * ntk + 15) / 16 * 16;
  const int64_t lists = static_cast<int64_t>(mask_batches) * (2 * ntq * ntk + ntq + ntk) * 4;
  return 2 * static_cast<int64_t>(B) * Hq * lqp * 4 + part + bits + (mask_batches ? flags + lists : 0);
}

cudaError_t launch_bwd_tc(const CUtensorMap (&maps)[4], const void* o, const Strides& so,
                          const void* dO, const Strides& sdo, const float* lse, void* dq,
                          const Strides& sdq, void* dk, const Strides& sdk, void* dv,
                          const Strides& sdv, void* workspace, int B, int Hq, int Hkv, int Lq,
                          int Lk, int D, float sm_scale, int causal, const int32_t* valid_len,
                          const uint8_t* mask, int64_t mask_batch_stride, int64_t mask_row_stride,
                          bool bf16, int num_sms, int* status, cudaStream_t stream) {
  BwdTcParams p;
  p.splits = bwd_tc_splits(B, Hkv, Lk, num_sms);
  p.sdq = sdq;
  p.sdk = sdk;
  p.sdv = sdv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.n_tq = (Lq + T - 1) / T;
  p.n_tk = (Lk + T - 1) / T;
  p.Lqp = p.n_tq * T;
  float* nlse2 = static_cast<float*>(workspace);
  float* delta = nlse2 + static_cast<int64_t>(B) * Hq * p.Lqp;
  p.part = delta + static_cast<int64_t>(B) * Hq * p.Lqp;  // used when splits > 1
  const int64_t part_floats =
      p.splits > 1 ? static_cast<int64_t>(p.splits) * 2 * B * Hkv * Lk * D : 0;
  p.rbits = nullptr;
  p.cbits = nullptr;
  p.klist = p.kcount = p.qlist = p.qcount = nullptr;
  p.mask_shared = mask_batch_stride == 0 ? 1 : 0;
  if (mask != nullptr) {
    const int mB = p.mask_shared ? 1 : B;
    uint32_t* rbits = reinterpret_cast<uint32_t*>(p.part + part_floats);
    uint32_t* cbits = rbits + static_cast<int64_t>(mB) * Lq * ((Lk + T - 1) / T) * 4;
    const int ntq = (Lq + T - 1) / T, ntk = (Lk + T - 1) / T;
    uint8_t* vis = reinterpret_cast<uint8_t*>(cbits + static_cast<int64_t>(mB) * Lk * ntq * 4);
    int* klist = reinterpret_cast<int*>(vis + (static_cast<int64_t>(mB) * ntq * ntk + 15) / 16 * 16);
    int* kcount = klist + static_cast<int64_t>(mB) * ntk * ntq;
    int* qlist = kcount + static_cast<int64_t>(mB) * ntk;
    int* qcount = qlist + static_cast<int64_t>(mB) * ntq * ntk;
    p.rbits = rbits;
    p.cbits = cbits;
    p.klist = klist;
    p.kcount = kcount;
    p.qlist = qlist;
    p.qcount = qcount;
    bwd_mask_pack_kernel<<<dim3(ntk, ntq, mB), 256, 0, stream>>>(
        mask, mask_batch_stride, mask_row_stride, Lq, Lk, ntq, ntk, rbits, cbits, vis);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t nlists = static_cast<int64_t>(mB) * (ntk + ntq);
    bwd_mask_lists_kernel<<<static_cast<unsigned>((nlists + 255) / 256), 256, 0, stream>>>(
        vis, mB, ntq, ntk, causal, klist, kcount, qlist, qcount);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  p.nlse2 = nlse2;
  p.delta = delta;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.valid_len = valid_len;
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.scale_log2 = sm_scale * kLog2e;
  p.sm_scale = sm_scale;
  p.causal = causal;
  p.dg = D;
  // D = 16 and 32 run the D = 64 kernels: their tensor maps have an inner
  // extent of D with 64-column boxes, so TMA fills columns D..63 of every Q,
  // K, V and dO tile with zeros (S and dP unchanged; the extra columns of dQ,
  // dK and dV are 0) and the epilogues store only the D columns.
  if (D == 16 || D == 32 || D == 64)
    return bf16 ? launch_bwd_tc_m<64, true>(maps, p, o, so, dO, sdo, lse, nlse2, delta, stream)
                : launch_bwd_tc_m<64, false>(maps, p, o, so, dO, sdo, lse, nlse2, delta, stream);
  if (D == 128)
    return bf16 ? launch_bwd_tc_m<128, true>(maps, p, o, so, dO, sdo, lse, nlse2, delta, stream)
                : launch_bwd_tc_m<128, false>(maps, p, o, so, dO, sdo, lse, nlse2, delta, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
