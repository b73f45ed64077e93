// Tensor-core attention forward for sm_103a (tcgen05 + TMA + TMEM).
//
// What it computes: O = softmax(Q K^T * sm_scale + Mask) V and the per-row
// natural-log LSE, tile by tile with the online softmax of the Triton-CUDA
// Attention page ("Online Softmax core algorithm": running max m_i, exp-sum
// l_i, an fp32 accumulator rescaled by alpha = exp2(m_old - m_new), scores
// pre-multiplied by sm_scale*log2(e)); masks and head map as in include/attn.h.
//
// How (one CTA per SM, persistent over work units):
//   * work unit = (b, h_q, 256 query rows) = two 128-row query tiles that share
//     one stream of K/V tiles (128 keys each);
//   * warp 8 (producer): TMA loads of the two Q tiles and of the K and V rings
//     (2 + 3 stages at D=128, 4 + 4 at D=64), 128-byte swizzled;
//   * warps 9 and 10 (MMA issuers, one per query tile t): S_t = Q_t K^T into
//     TMEM (fp32), then O_t += P_t V with P_t read from TMEM.  For every key
//     tile j the issuers take turns -- PV_0(j) S_0(j+1), then PV_1(j)
//     S_1(j+1) -- so the tensor core runs one tile's group while that tile's
//     issuer does its barrier work and the other tile's softmax runs;
//   * warps 0-3 / 4-7 (softmax, one thread per query row = TMEM lane): load
//     the S row, mask (only on boundary tiles), row max, ex2.approx, row sum,
//     write P into TMEM over the S columns, rescale the O row in TMEM when the
//     max grew by more than 2^8 (exact after the final division), and finally
//     O / l -> global memory and the LSE.
// Causal units skip every key tile above the diagonal; padded units skip every
// key tile at or beyond valid_len[b]; a unit with no visible key writes O = 0
// and LSE = -inf without touching the tensor core.
//
// bf16 inputs: P.V runs with fp16 P (unit roundoff 2^-11) whenever the V tile
// has an exact fp16 copy -- made once per call by the pre-pass in
// attn_vconv.cu, which flags every 128-key tile whose values are all finite
// with |v| < 2^16 -- and the producer then loads that copy.  A tile without
// one stays bf16 and P is split into two bf16 terms (see the softmax).
// Without flags (no workspace) every bf16 tile takes the split form.
//
// Every mbarrier wait is bounded: after ATTN_WAIT_LIMIT_NS the waiting role
// records a timeout in the device status word, raises a CTA-wide abort flag
// and leaves its loop; the others see the flag and leave too; the CTA then
// waits (bounded) for its own copies and MMAs in flight and frees its TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"
#include "ptx.cuh"

#ifndef ATTN_WAIT_LIMIT_NS
#define ATTN_WAIT_LIMIT_NS 2000000000ull
#endif

namespace attn {
namespace {

constexpr int BM = 128;       // query rows per tile (TMEM lanes)
constexpr int QT = 2;         // query tiles per work unit
constexpr int BN = 128;       // keys per K/V tile
constexpr int kUnitRows = QT * BM;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp0 = 9;   // MMA issuer of query tile 0; tile 1 has warp 10
constexpr int kThreads = 384;  // warpgroups: softmax tile 0, softmax tile 1, producer/MMA
// Register split between warpgroups (setmaxnreg).  The CTA is launched with
// kLaunchRegs per thread (the __launch_bounds__(384, 1) ceiling: 3 warps per
// SM sub-partition); the split must add up to exactly that pool.  D = 128
// issues its MMAs from fully unrolled loops (fewer instructions between MMAs
// on the issuer warps), which needs more control registers; D = 64 keeps
// every register it can for the softmax.
constexpr int kLaunchRegs = 168;
template <int D>
struct RegSplit {
  static constexpr int kSoftmax = (D == 128) ? 216 : 224;
  static constexpr int kControl = (D == 128) ? 72 : 56;
  static_assert(2 * 128 * kSoftmax + 128 * kControl == kThreads * kLaunchRegs,
                "register split must equal the launch pool");
};
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.69314718055994531f;

template <int D>
struct Cfg {
  // separate rings for K and V tiles; V gets the extra stage (its tiles are
  // consumed later in each step than the K tiles)
  static constexpr int kKStages = (D == 128) ? 2 : 4;
  static constexpr int kVStages = (D == 128) ? 3 : 4;
  static constexpr int kHalves = D / 64;           // 64-column (128-byte) slabs per row
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kSlabQ = BM * 128;          // bytes of one 64-column slab of a Q tile
  static constexpr int kSlabKV = BN * 128;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = QT * kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kVStages * kKVBytes;
  // barrier block: q_full[QT] q_empty[QT] k_full[KS] k_empty[KS] v_full[VS]
  // v_empty[VS] s_full[QT] p_full[QT] o_full[QT] drain turn[QT], then 32-bit
  // words: TMEM base, abort flag
  static constexpr int kNumBars = 6 * QT + 2 * kKStages + 2 * kVStages + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kMiscBytes = 8;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + slack to align the base
  // TMEM columns: S_0, S_1 (fp32, BN each; P_t is written over S_t), then
  // O_0, O_1 (fp32, D each).
  static __device__ __forceinline__ uint32_t col_s(int t) { return static_cast<uint32_t>(t * BN); }
  static __device__ __forceinline__ uint32_t col_o(int t) {
    return static_cast<uint32_t>(2 * BN + t * D);
  }
  static constexpr uint32_t kTmemCols = 512;
  static_assert(2 * BN + 2 * D <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared-memory budget");
};

// Shared-memory addresses of the barriers (32-bit, one base + constants).
template <int D>
struct Bars {
  static constexpr uint32_t KS = Cfg<D>::kKStages;
  static constexpr uint32_t VS = Cfg<D>::kVStages;
  uint32_t base;
  __device__ __forceinline__ uint32_t q_full(int t) const { return base + 8u * t; }
  __device__ __forceinline__ uint32_t q_empty(int t) const { return base + 8u * (QT + t); }
  __device__ __forceinline__ uint32_t k_full(uint32_t s) const { return base + 8u * (2 * QT + s); }
  __device__ __forceinline__ uint32_t k_empty(uint32_t s) const {
    return base + 8u * (2 * QT + KS + s);
  }
  __device__ __forceinline__ uint32_t v_full(uint32_t s) const {
    return base + 8u * (2 * QT + 2 * KS + s);
  }
  __device__ __forceinline__ uint32_t v_empty(uint32_t s) const {
    return base + 8u * (2 * QT + 2 * KS + VS + s);
  }
  __device__ __forceinline__ uint32_t s_full(int t) const {
    return base + 8u * (2 * QT + 2 * KS + 2 * VS + t);
  }
  __device__ __forceinline__ uint32_t p_full(int t) const {
    return base + 8u * (3 * QT + 2 * KS + 2 * VS + t);
  }
  __device__ __forceinline__ uint32_t o_full(int t) const {
    return base + 8u * (4 * QT + 2 * KS + 2 * VS + t);
  }
  __device__ __forceinline__ uint32_t drain() const { return base + 8u * (5 * QT + 2 * KS + 2 * VS); }
  // issuer t may issue its MMA group of the current key tile
  __device__ __forceinline__ uint32_t turn(int t) const {
    return base + 8u * (5 * QT + 2 * KS + 2 * VS + 1 + t);
  }
  __device__ __forceinline__ uint32_t tmem_word() const {
    return base + 8u * (6 * QT + 2 * KS + 2 * VS + 1);
  }
  __device__ __forceinline__ uint32_t abort_word() const { return tmem_word() + 4u; }
};

struct KParams {
  void* o;
  float* lse;
  const int32_t* valid_len;
  int* status;
  // bf16 only: per (b, h_kv, 128-key tile) 1 = the fp16 copy of the V tile is
  // exact, 0 = use the bf16 tile; null = no fp16 copy exists
  const int* vflags;
  int n_kt;     // 128-key tiles per (b, h_kv)
  int B, Hq, Hkv, L, G;
  int n_mb;     // 256-row blocks per (b, h_q)
  int n_units;  // B * Hq * n_mb
  float scale_log2;
  int causal;
};

struct Unit {
  int bh, b, hkv, m0, kv_len;
  int n[QT];  // key tiles each query tile visits (0: tile absent or no visible key)
};

// Units are ordered so that causal work runs heaviest-first (last row blocks
// first) with heads innermost (query heads of one KV group are adjacent, so
// their K/V stay in L2), and non-causal work runs head by head.  CTA c takes
// the unit of round r at position c (r even) or gridDim.x-1-c (r odd): this
// "snake" keeps per-CTA totals within a few percent on heaviest-first lists.
__device__ __forceinline__ int unit_of(int round) {
  const int g = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  return round * g + ((round & 1) ? (g - 1 - c) : c);
}

__device__ __forceinline__ Unit decode_unit(const KParams& p, int u) {
  Unit w;
  const int BH = p.B * p.Hq;
  int mb;
  if (p.causal) {
    mb = p.n_mb - 1 - u / BH;
    w.bh = u % BH;
  } else {
    w.bh = u / p.n_mb;
    mb = u % p.n_mb;
  }
  w.b = w.bh / p.Hq;
  w.hkv = (w.bh % p.Hq) / p.G;
  w.m0 = mb * kUnitRows;
  int kv = p.L;
  if (p.valid_len != nullptr) {
    kv = p.valid_len[w.b];
    kv = kv < 0 ? 0 : (kv > p.L ? p.L : kv);
  }
  w.kv_len = kv;
#pragma unroll
  for (int t = 0; t < QT; ++t) {
    const int r0 = w.m0 + t * BM;
    if (r0 >= p.L) {
      w.n[t] = 0;
    } else {
      const int hi = p.causal ? min(kv, r0 + BM) : kv;
      w.n[t] = (hi + BN - 1) / BN;
    }
  }
  return w;
}

// Bounded mbarrier wait.  False: timed out (recorded) or another role aborted.
// (Everything is inlined: out-of-line calls do not mix with setmaxnreg.)
template <class BarsT>
__device__ __forceinline__ bool wait_bar(const BarsT& br, int* status, uint32_t bar,
                                         uint32_t parity, int role) {
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

// Wait with a time limit and no abort check (used only to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer_ns() - t0 < ATTN_WAIT_LIMIT_NS) {
  }
}

// bf16 inputs: true when P.V for key tile j of KV head z takes the split form
// (no exact fp16 copy of the V tile).  fp16 inputs: never.
template <bool BF16>
__device__ __forceinline__ bool v_split(const KParams& p, int z_kv, int j) {
  if constexpr (!BF16) {
    return false;
  } else {
    return p.vflags == nullptr || __ldg(p.vflags + static_cast<int64_t>(z_kv) * p.n_kt + j) == 0;
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// ------------------------------------------------------------------ producer

template <int D, bool BF16>
__device__ void producer_role(const KParams& p, const Bars<D>& br, uint32_t smem,
                              const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                              const CUtensorMap* tm_v, const CUtensorMap* tm_v16) {
  using C = Cfg<D>;
  uint32_t q_phase = 0;   // bit t: parity of tile t's next q_empty wait ^ 1
  uint32_t q_used = 0;    // bit t: a Q_t load was issued
  uint32_t k_used = 0, k_par = 0;  // per K stage: loaded at least once / parity of the last load
  uint32_t v_used = 0, v_par = 0;  // per V stage: the same
  uint32_t kit = 0, vit = 0;       // K and V ring items issued
  const uint64_t pol_keep = ptx::policy_evict_last();
  const uint64_t pol_stream = ptx::policy_evict_first();
  bool ok = true;

  // One K or V tile into the next slot of its ring.
  auto load_kv = [&](bool is_v, int j, int z_kv) -> bool {
    uint32_t& it = is_v ? vit : kit;
    const uint32_t ns = is_v ? C::kVStages : C::kKStages;
    const uint32_t s = it % ns;
    const uint32_t par = (it / ns) & 1u;
    if (!wait_bar(br, p.status, is_v ? br.v_empty(s) : br.k_empty(s), par ^ 1u, kRoleProducer))
      return false;
    ++it;
    const uint32_t full = is_v ? br.v_full(s) : br.k_full(s);
    const uint32_t dst = smem + (is_v ? C::kOffV : C::kOffK) + s * C::kKVBytes;
    // bf16 V: the exact fp16 copy of the tile when there is one
    const CUtensorMap* map = !is_v ? tm_k : ((!BF16 || v_split<BF16>(p, z_kv, j)) ? tm_v : tm_v16);
    ptx::mbar_arrive_expect_tx(full, C::kKVBytes);
#pragma unroll
    for (int h = 0; h < C::kHalves; ++h)
      ptx::tma_load_3d_hint(dst + h * C::kSlabKV, map, full, h * 64, j * BN, z_kv, pol_keep);
    if (is_v) {
      v_used |= 1u << s;
      v_par = (v_par & ~(1u << s)) | (par << s);
    } else {
      k_used |= 1u << s;
      k_par = (k_par & ~(1u << s)) | (par << s);
    }
    return true;
  };

  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  for (int r = 0; ok && r < rounds; ++r) {
    const int u = unit_of(r);
    if (u >= p.n_units) continue;
    const Unit w = decode_unit(p, u);
    const int n = max(w.n[0], w.n[1]);
    if (n == 0) continue;
    const int z_kv = w.b * p.Hkv + w.hkv;
#pragma unroll
    for (int t = 0; t < QT; ++t) {
      if (w.n[t] == 0) continue;
      if (!wait_bar(br, p.status, br.q_empty(t), ((q_phase >> t) & 1u) ^ 1u, kRoleProducer)) {
        ok = false;
        break;
      }
      q_phase ^= 1u << t;
      q_used |= 1u << t;
      const uint32_t dst = smem + C::kOffQ + t * C::kQBytes;
      ptx::mbar_arrive_expect_tx(br.q_full(t), C::kQBytes);
#pragma unroll
      for (int h = 0; h < C::kHalves; ++h)
        ptx::tma_load_3d_hint(dst + h * C::kSlabQ, tm_q, br.q_full(t), h * 64, w.m0 + t * BM,
                              w.bh, pol_stream);
    }
    // issue order K_0 V_0 | V_1 K_1 | V_2 K_2 ...: each V tile is requested as
    // soon as its (deeper) ring has room
    ok = ok && load_kv(false, 0, z_kv) && load_kv(true, 0, z_kv);
    for (int j = 1; ok && j < n; ++j) ok = load_kv(true, j, z_kv) && load_kv(false, j, z_kv);
  }
  // Never leave with a copy in flight: wait (bounded) for the last load of
  // every buffer.  In a normal run these phases completed long ago.
  for (uint32_t s = 0; s < C::kKStages; ++s)
    if ((k_used >> s) & 1u) drain_wait(br.k_full(s), (k_par >> s) & 1u);
  for (uint32_t s = 0; s < C::kVStages; ++s)
    if ((v_used >> s) & 1u) drain_wait(br.v_full(s), (v_par >> s) & 1u);
  for (int t = 0; t < QT; ++t)
    if ((q_used >> t) & 1u) drain_wait(br.q_full(t), ((q_phase >> t) & 1u) ^ 1u);
}

// ------------------------------------------------------------------ MMA issuer

// One lane of a converged warp, chosen by the hardware (elect.sync).  The MMA
// issuer runs on the whole warp so that descriptors and TMEM addresses stay
// warp-uniform values; only the tcgen05.mma / tcgen05.commit instructions
// themselves are executed by the elected lane.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void commit_one(uint32_t bar) {
  if (elect_one()) ptx::mma_commit(bar);
  __syncwarp();
}

// A descriptor's start address is its low 14 bits (address >> 4); a byte
// offset inside the same shared-memory window is added there directly.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) {
  return desc + (bytes >> 4);
}

// S = Q K^T over D: A = Q tile, B = K tile, both K-major 128-byte swizzled
// (64-column slabs); each MMA consumes 16 columns (32 bytes of a slab row).
template <int D, bool BF16>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  using C = Cfg<D>;
  constexpr uint32_t idesc = ptx::idesc_f16(BM, BN, BF16, false);
#pragma unroll (D == 128 ? D / 16 : 1)
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk & 3) * 32u;
    ptx::mma_ss(d_tmem, desc_add(q_desc, (kk / 4) * C::kSlabQ + off),
                desc_add(k_desc, (kk / 4) * C::kSlabKV + off), idesc, kk > 0 ? 1u : 0u);
  }
}

// O += P V: A = P from TMEM (16-bit pairs, 8 columns per 16 keys), B = V tile
// as an MN-major 128-byte-swizzled operand (16 keys = two 8-row groups).
// fp16 V tile (fp16 inputs, or the exact fp16 copy of a bf16 tile):
// O += P V with fp16 P.  bf16 V tile (split): O += [P_hi | P_lo] [V; V], the
// same V tile read twice.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         bool accumulate, bool split) {
  const uint32_t idesc = split ? ptx::idesc_f16(BM, D, true, true) : ptx::idesc_f16(BM, D, false, true);
#pragma unroll (D == 128 ? BN / 16 : 1)
  for (int kk = 0; kk < BN / 16; ++kk)
    ptx::mma_ts(d_tmem, p_tmem + kk * 8u, desc_add(v_desc, kk * 2048u), idesc,
                (accumulate || kk > 0) ? 1u : 0u);
  if (split) {
#pragma unroll 1
    for (int kk = 0; kk < BN / 16; ++kk)
      ptx::mma_ts(d_tmem, p_tmem + BN / 2 + kk * 8u, desc_add(v_desc, kk * 2048u), idesc, 1u);
  }
}

// Release of a K or V ring slot by an issuer warp: after the warp's MMAs that
// read it (commit), or at once when its tile does not use the slot.  Each
// slot's empty barrier expects one release from each of the two issuers.
__device__ __forceinline__ void release_slot(uint32_t bar, bool used) {
  if (used) {
    commit_one(bar);
  } else {
    if (elect_one()) ptx::mbar_arrive(bar);
    __syncwarp();
  }
}

// Issuer of query tile t (whole warp; one elected lane issues).  It walks
// every K and V ring item of every unit in the producer's order, so both
// issuers stay in phase with the rings even when one tile has fewer key tiles
// (causal diagonal) or none.
//
// Turns: for every key tile (counted over all units) issuer 0 issues its
// group (PV_0(j), S_0(j+1)) and hands the turn to issuer 1, which issues its
// group and hands it back.  The tensor core then works through whole groups
// in that order, so the two tiles' scores complete half a step apart and the
// two softmax warpgroups alternate instead of running at the same time.
template <int D, bool BF16>
__device__ void mma_role(const KParams& p, const Bars<D>& br, uint32_t smem, uint32_t tmem, int t) {
  using C = Cfg<D>;
  uint32_t q_phase = 0, p_phase = 0;
  uint32_t kit = 0, vit = 0;
  uint32_t step = 0;  // key tiles of all units so far (turn phase)
  // K-major operands (Q, K): leading byte offset unused with 128-byte swizzle,
  // 1024 bytes between 8-row groups.  MN-major V: 64-column slabs kSlabKV
  // apart (leading), 1024 bytes between 8-key groups (stride).
  const uint64_t q_desc = ptx::sdesc_sw128(smem + C::kOffQ + t * C::kQBytes, 16, 1024);
  const uint64_t k_desc0 = ptx::sdesc_sw128(smem + C::kOffK, 16, 1024);
  const uint64_t v_desc0 = ptx::sdesc_sw128(smem + C::kOffV, C::kSlabKV, 1024);
  const uint32_t t_s = tmem + C::col_s(t);
  const uint32_t t_o = tmem + C::col_o(t);
  bool ok = true;

  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  for (int r = 0; ok && r < rounds; ++r) {
    const int u = unit_of(r);
    if (u >= p.n_units) continue;
    const Unit w = decode_unit(p, u);
    const int n = max(w.n[0], w.n[1]);
    const int nt = t == 0 ? w.n[0] : w.n[1];  // (a select keeps Unit in registers)
    if (n == 0) continue;
    const int z_kv = w.b * p.Hkv + w.hkv;
    if (nt > 0) {
      if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.q_full(t), q_phase, kRoleMma))) break;
      q_phase ^= 1u;
    }
    // S_t(0)
    {
      const uint32_t sk = kit % C::kKStages;
      if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.k_full(sk),
                                            (kit / C::kKStages) & 1u, kRoleMma)))
        break;
      ++kit;
      if (nt > 0) {
        ptx::tc_fence_after();
        if (elect_one()) issue_qk<D, BF16>(t_s, q_desc, desc_add(k_desc0, sk * C::kKVBytes));
        __syncwarp();
        commit_one(br.s_full(t));
        if (nt == 1) commit_one(br.q_empty(t));
      }
      release_slot(br.k_empty(sk), nt > 0);
    }
    for (int j = 0; j < n; ++j, ++step) {
      const uint32_t sv = vit % C::kVStages;
      if (!__all_sync(0xffffffffu,
                      wait_bar(br, p.status, br.v_full(sv), (vit / C::kVStages) & 1u, kRoleMma))) {
        ok = false;
        break;
      }
      ++vit;
      const bool use_v = j < nt;
      const bool split = use_v && v_split<BF16>(p, z_kv, j);
      const bool has_next = j + 1 < n;
      uint32_t sk = 0;
      if (has_next) {
        sk = kit % C::kKStages;
        if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.k_full(sk),
                                              (kit / C::kKStages) & 1u, kRoleMma))) {
          ok = false;
          break;
        }
        ++kit;
      }
      const bool use_k = j + 1 < nt;
      // my turn: issuer 0 waits for issuer 1's previous group (none at the
      // first key tile: the fresh barrier's preceding phase counts as done),
      // issuer 1 for issuer 0's group of this key tile
      const uint32_t turn_par = (t == 0) ? ((step & 1u) ^ 1u) : (step & 1u);
      if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.turn(t), turn_par, kRoleMma))) {
        ok = false;
        break;
      }
      // P last: V, K and the turn are normally ready long before the softmax
      // finishes, so only this wait stands between P_t(j) and its MMAs
      if (use_v) {
        if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.p_full(t), p_phase, kRoleMma))) {
          ok = false;
          break;
        }
        p_phase ^= 1u;
      }
      ptx::tc_fence_after();
      if (elect_one()) {
        if (use_v) issue_pv<D>(t_o, t_s, desc_add(v_desc0, sv * C::kKVBytes), j > 0, split);
        if (use_k) issue_qk<D, BF16>(t_s, q_desc, desc_add(k_desc0, sk * C::kKVBytes));
        ptx::mbar_arrive(br.turn(t ^ 1));  // the other issuer's group may follow
      }
      __syncwarp();
      if (use_v && j == nt - 1) commit_one(br.o_full(t));
      release_slot(br.v_empty(sv), use_v);
      if (use_k) {
        commit_one(br.s_full(t));
        // Q_t is free once the unit's last S_t MMA completes: the producer
        // can load the next unit's Q_t while this unit finishes
        if (j + 2 == nt) commit_one(br.q_empty(t));
      }
      if (has_next) release_slot(br.k_empty(sk), use_k);
    }
  }
  // Every MMA issued by this warp completes before TMEM is released.
  commit_one(br.drain());
  drain_wait(br.drain(), 0);
}

// ------------------------------------------------------------------ softmax + epilogue

// P for one score row (128 keys in registers), 32 keys at a time, written
// over the row's S columns in TMEM; returns the row sum of P.  fp16 V tile:
// P rounded to fp16 in columns [0, 64).  bf16 V tile (SPLIT): P = P_hi + P_lo
// with P_hi = p truncated to bf16 (columns [0, 64)) and P_lo = bf16(p - P_hi)
// (columns [64, 128)); a single bf16 P (unit roundoff 2^-8) is too coarse for
// rows dominated by a few keys, the pair leaves a relative error below 2^-15.
// MASKED: columns c >= c_lim get P = 0.
template <bool MASKED, bool SPLIT>
__device__ __forceinline__ float exp_row(const uint32_t (&s)[BN], uint64_t sc2, uint64_t nm2, int c_lim,
                                         uint32_t t_s) {
  uint64_t rsum2[4];  // independent partial row sums, two lanes each
#pragma unroll
  for (int k = 0; k < 4; ++k) rsum2[k] = 0ull;
#pragma unroll
  for (int qtr = 0; qtr < 4; ++qtr) {
    uint32_t hi[16];
    uint32_t lo[SPLIT ? 16 : 1];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = qtr * 32 + 2 * i;
      // exponent argument s*scale - m for two keys in one instruction
      const uint64_t x2 =
          ptx::f2_fma(ptx::f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sc2, nm2);
      float x0, x1;
      ptx::f2_unpack(x2, x0, x1);
      float p0 = ptx::ex2_approx(x0);
      float p1 = ptx::ex2_approx(x1);
      if constexpr (MASKED) {
        p0 = (c < c_lim) ? p0 : 0.f;
        p1 = (c + 1 < c_lim) ? p1 : 0.f;
      }
      const uint64_t p2 = ptx::f2_pack(p0, p1);
      rsum2[i & 3] = ptx::f2_add(rsum2[i & 3], p2);
      if constexpr (SPLIT) {
        const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
        hi[i] = __byte_perm(b0, b1, 0x7632);  // upper halves: truncated bf16 pair
        const uint64_t r2 = ptx::f2_sub(
            p2, ptx::f2_pack(__uint_as_float(b0 & 0xFFFF0000u), __uint_as_float(b1 & 0xFFFF0000u)));
        float r0, r1;
        ptx::f2_unpack(r2, r0, r1);
        lo[i] = pack2<true>(r0, r1);
      } else {
        hi[i] = pack2<false>(p0, p1);
      }
    }
    ptx::tmem_st16(t_s + qtr * 16, hi);
    if constexpr (SPLIT) ptx::tmem_st16(t_s + BN / 2 + qtr * 16, lo);
  }
  float ra, rb;
  ptx::f2_unpack(ptx::f2_add(ptx::f2_add(rsum2[0], rsum2[1]), ptx::f2_add(rsum2[2], rsum2[3])), ra, rb);
  return ra + rb;
}

template <int D, bool BF16>
__device__ void softmax_role(const KParams& p, const Bars<D>& br, uint32_t tmem, int t) {
  using C = Cfg<D>;
  const int lane_row = threadIdx.x & 127;           // row within the tile = TMEM lane
  const uint32_t quad = (threadIdx.x >> 5) & 3u;    // this warp's 32-lane TMEM quadrant
  const uint32_t t_s = tmem + ((quad * 32u) << 16) + C::col_s(t);
  const uint32_t t_o = tmem + ((quad * 32u) << 16) + C::col_o(t);
  const float scale_log2 = p.scale_log2;
  uint32_t s_phase = 0, o_phase = 0;

  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  for (int r = 0; r < rounds; ++r) {
    const int u = unit_of(r);
    if (u >= p.n_units) continue;
    const Unit w = decode_unit(p, u);
    const int z_kv = w.b * p.Hkv + w.hkv;
    const int r0 = w.m0 + t * BM;
    if (r0 >= p.L) continue;
    const int row = r0 + lane_row;
    const bool row_ok = row < p.L;
    const int64_t grow = static_cast<int64_t>(w.bh) * p.L + row;
    if (t == 0 && threadIdx.x == 0 && p.valid_len != nullptr) {
      const int vl = p.valid_len[w.b];
      if (vl < 0 || vl > p.L) atomicOr(p.status, kStatusValidLenClamped);
    }
    const int nt = w.n[t];
    if (nt == 0) {  // no visible key: O = 0, LSE = -inf
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) + grow * D * 2);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        if (p.lse != nullptr) p.lse[grow] = -INFINITY;
      }
      continue;
    }
    // keys < key_lim are visible to this row
    const int key_lim = p.causal ? min(w.kv_len, row + 1) : w.kv_len;
    float m = -INFINITY;  // running max, log2 units (scaled)
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // P format of this key tile: fp16 P, or the bf16 pair (split)
      const bool split = v_split<BF16>(p, z_kv, j);
      ok = wait_bar(br, p.status, br.s_full(t), s_phase, kRoleSoftmax);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      s_phase ^= 1u;
      ptx::tc_fence_after();
      uint32_t s[BN];
      ptx::tmem_ld128(t_s, s);
      const int n0 = j * BN;
      const bool masked = (n0 + BN > w.kv_len) || (p.causal && n0 + BN - 1 > r0);
      const int c_lim = key_lim - n0;  // columns c < c_lim are visible
      // row max: 8 independent chains of 3-input maxima
      float mxk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mxk[k] = -INFINITY;
      if (masked) {
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) {
          const int c = 2 * i;
          mxk[i & 7] = ptx::max3(mxk[i & 7], (c < c_lim) ? __uint_as_float(s[c]) : -INFINITY,
                                 (c + 1 < c_lim) ? __uint_as_float(s[c + 1]) : -INFINITY);
        }
      } else {
#pragma unroll
        for (int i = 0; i < BN / 2; ++i)
          mxk[i & 7] = ptx::max3(mxk[i & 7], __uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
      }
      const float mx = ptx::max3(ptx::max3(mxk[0], mxk[1], mxk[2]), ptx::max3(mxk[3], mxk[4], mxk[5]),
                                 fmaxf(mxk[6], mxk[7]));
      const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * scale_log2;
      const float m_new = fmaxf(m, m_tile);
      float alpha = 1.f;
      bool rescale = false;
      if (m_new > m + kRescaleLog2) {  // also taken on the first tile (m = -inf)
        alpha = ptx::ex2_approx(m - m_new);
        m = m_new;
        rescale = true;
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      const uint64_t sc2 = ptx::f2_pack(scale_log2, scale_log2);
      const uint64_t nm2 = ptx::f2_pack(neg_m, neg_m);
      // P over the S columns (every S value is already in registers); the
      // masked form only on key tiles that need it, so full tiles carry no
      // per-key selects
      float rowsum;
      if (!split) {
        rowsum = masked ? exp_row<true, false>(s, sc2, nm2, c_lim, t_s)
                        : exp_row<false, false>(s, sc2, nm2, c_lim, t_s);
      } else if constexpr (BF16) {
        rowsum = masked ? exp_row<true, true>(s, sc2, nm2, c_lim, t_s)
                        : exp_row<false, true>(s, sc2, nm2, c_lim, t_s);
      } else {
        rowsum = 0.f;
      }
      l = l * alpha + rowsum;
      // O was accumulated against the old max: rescale it before PV_j runs.
      // PV_{j-1} is complete: the commit that signalled S_j came after it.
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          ptx::tmem_ld32(t_o + c0, o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          ptx::tmem_st32(t_o + c0, o);
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(br.p_full(t));
    }
    if (!ok) return;
    // epilogue
    ok = wait_bar(br, p.status, br.o_full(t), o_phase, kRoleEpilogue);
    if (!__all_sync(0xffffffffu, ok)) return;
    o_phase ^= 1u;
    ptx::tc_fence_after();
    const float inv_l = 1.f / l;
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t o[32];
      ptx::tmem_ld32(t_o + c0, o);
      uint32_t h[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        h[c] = pack2<BF16>(__uint_as_float(o[2 * c]) * inv_l, __uint_as_float(o[2 * c + 1]) * inv_l);
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) + (grow * D + c0) * 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
      }
    }
    if (row_ok && p.lse != nullptr) p.lse[grow] = (m + ptx::lg2_approx(l)) * kLn2;
  }
}

// ------------------------------------------------------------------ kernel

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_v16, const KParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const Bars<D> br{smem + C::kOffBar};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < QT; ++t) {
      ptx::mbar_init(br.q_full(t), 1);
      ptx::mbar_init(br.q_empty(t), 1);
      ptx::mbar_init(br.s_full(t), 1);
      ptx::mbar_init(br.p_full(t), BM);
      ptx::mbar_init(br.o_full(t), 1);
    }
    // ring slots and the final drain: one release from each MMA issuer
    for (int s = 0; s < C::kKStages; ++s) {
      ptx::mbar_init(br.k_full(s), 1);
      ptx::mbar_init(br.k_empty(s), QT);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      ptx::mbar_init(br.v_full(s), 1);
      ptx::mbar_init(br.v_empty(s), QT);
    }
    ptx::mbar_init(br.drain(), QT);
    ptx::mbar_init(br.turn(0), 1);
    ptx::mbar_init(br.turn(1), 1);
    ptx::st_shared_volatile(br.abort_word(), 0u);
    ptx::fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
    if constexpr (BF16) ptx::prefetch_tensormap(&tm_v16);
  }
  if (warp == kMmaWarp0) {
    ptx::tmem_alloc(br.tmem_word(), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ptx::ld_shared_volatile(br.tmem_word());

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegSplit<D>::kControl));
    if (warp == kProducerWarp) {
      if (lane == 0) producer_role<D, BF16>(p, br, smem, &tm_q, &tm_k, &tm_v, &tm_v16);
    } else if (warp < kMmaWarp0 + QT) {
      mma_role<D, BF16>(p, br, smem, tmem, warp - kMmaWarp0);  // whole warp
    }
    // warp 11 has no role
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RegSplit<D>::kSoftmax));
    softmax_role<D, BF16>(p, br, tmem, warp >> 2);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool BF16>
cudaError_t launch_instance(const Problem& pr, const CUtensorMap* maps, int num_sms) {
  using C = Cfg<D>;
  static bool configured = false;  // per (D, dtype) instance
  auto kern = attn_fwd_tc_kernel<D, BF16>;
  if (!configured) {
    // The setmaxnreg split is only safe when the CTA is launched with exactly
    // kLaunchRegs registers per thread; anything else could stall the
    // increasing warpgroups forever, so refuse to launch.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  KParams kp;
  kp.o = pr.o;
  kp.lse = pr.lse;
  kp.valid_len = pr.valid_len;
  kp.status = pr.status;
  kp.vflags = pr.vflags;
  kp.n_kt = (pr.L + BN - 1) / BN;
  kp.B = pr.B;
  kp.Hq = pr.Hq;
  kp.Hkv = pr.Hkv;
  kp.L = pr.L;
  kp.G = pr.Hq / pr.Hkv;
  kp.n_mb = (pr.L + kUnitRows - 1) / kUnitRows;
  kp.n_units = pr.B * pr.Hq * kp.n_mb;
  kp.scale_log2 = pr.sm_scale * 1.4426950408889634f;
  kp.causal = pr.causal;
  const int grid = kp.n_units < num_sms ? kp.n_units : num_sms;
  kern<<<grid, kThreads, C::kSmemBytes, pr.stream>>>(maps[0], maps[1], maps[2], maps[3], kp);
  return cudaGetLastError();
}

}  // namespace

bool tc_config(int D, TcConfig* out) {
  if (D == 64) {
    *out = {BM, QT, BN, Cfg<64>::kKStages + Cfg<64>::kVStages, kThreads, Cfg<64>::kSmemBytes,
            static_cast<int>(Cfg<64>::kTmemCols)};
    return true;
  }
  if (D == 128) {
    *out = {BM, QT, BN, Cfg<128>::kKStages + Cfg<128>::kVStages, kThreads, Cfg<128>::kSmemBytes,
            static_cast<int>(Cfg<128>::kTmemCols)};
    return true;
  }
  return false;
}

cudaError_t launch_tc(const Problem& p, const CUtensorMap* maps, int num_sms) {
  if (p.D == 64) {
    return p.bf16 ? launch_instance<64, true>(p, maps, num_sms)
                  : launch_instance<64, false>(p, maps, num_sms);
  }
  if (p.D == 128) {
    return p.bf16 ? launch_instance<128, true>(p, maps, num_sms)
                  : launch_instance<128, false>(p, maps, num_sms);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
