// Tensor-core attention forward for sm_103a (tcgen05 + TMA + TMEM).
//
// What it computes: O = softmax(Q K^T * sm_scale + Mask) V and the per-row
// natural-log LSE, tile by tile with the online softmax of the Triton-CUDA
// Attention page ("Online Softmax core algorithm": running max m_i, exp-sum
// l_i, an fp32 accumulator rescaled by alpha = exp2(m_old - m_new), scores
// pre-multiplied by sm_scale*log2(e)); masks and head map as in include/attn.h.
//
// How (one CTA per SM, persistent over work units):
//   * work unit = (b, h_q, 128 query rows), one query tile; K/V streamed in
//     tiles of 128 keys;
//   * warp 8 (producer): TMA loads of the Q tile and of the K and V rings
//     (2 + 3 stages at D=128, 6 + 6 at D=64), 128-byte swizzled;
//   * warps 9 and 10 (MMA issuers; one elected lane each issues): warp 10
//     issues S(j) = Q K_j^T into one of three TMEM score buffers, warp 9
//     issues the P.V products with P read from TMEM.  The scores run up to
//     three key tiles ahead of the softmax (S(j+3) goes into the buffer P(j)
//     came from, once PV(j) has completed), so the tensor core has work
//     queued while P(j) is being computed;
//   * warps 0-7 (softmax, two warpgroups; a TMEM lane is a query row): warp w
//     and warp w + 4 share the same 32 rows, warps 0-3 (half a) taking key
//     columns 0-63 of every tile and warps 4-7 (half b) columns 64-127.  Per
//     step a thread loads its 64 scores with their maximum (tcgen05.ld.red),
//     masks them (only on boundary tiles), ex2.approx, the sum, writes P into
//     TMEM over its S columns and rescales O in TMEM when the max grew by
//     more than 2^8 (exact after the final division).  D = 64: each half
//     keeps its own online softmax -- running max, sum and a partial
//     accumulator, O_a or O_b (O_h += P_h V_h) -- so the two never wait for
//     each other inside a unit, and the epilogue combines them
//     (O = (O_a 2^(m_a-m) + O_b 2^(m_b-m)) / l).  D = 128: TMEM holds three
//     score buffers only next to one 128-column accumulator, so the halves
//     share O and agree on the running max at every step through shared
//     memory.  The epilogue warpgroup stages O in shared memory in the TMA
//     layout and writes it with one TMA store per 64-column slab, and the
//     LSE.  The staging tile is the V ring stage of the unit's last key tile:
//     idle from its PV's completion until the producer refills it, so the
//     epilogue, not the PV issuer, releases that stage once the store has
//     read it.
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

#include <atomic>

#include "attn_internal.h"
#include "ptx.cuh"

#ifndef ATTN_WAIT_LIMIT_NS
#define ATTN_WAIT_LIMIT_NS 2000000000ull
#endif

namespace attn {
namespace {

constexpr int BM = 128;       // query rows per tile (TMEM lanes)
constexpr int BN = 128;       // keys per K/V tile
constexpr int BH = BN / 2;    // keys of one half tile (one softmax warpgroup's columns)
constexpr int kProducerWarp = 8;
constexpr int kPvWarp = 9;     // P.V issuer; also allocates TMEM
constexpr int kSWarp = 10;     // score issuer
constexpr int kDecodeWarp = 11;  // decodes the CTA's units ahead of the softmax
constexpr int kEpiWarp0 = 12;  // warps 12-15: epilogue (warp 12 + q reads TMEM lane quadrant q)
constexpr int kUnitSlots = 4;  // decoded units in flight (shared-memory ring)
constexpr int kUnitWords = 12; // 32-bit words per ring slot
// warpgroups: softmax half a, softmax half b, control (producer, two issuers,
// unit decoder), epilogue
constexpr int kThreads = 512;
constexpr int kSoftmaxThreads = 256;
constexpr int kEpiThreads = 128;
// Register split between warpgroups (setmaxnreg).  The CTA is launched with
// kLaunchRegs registers per thread (the __launch_bounds__(512, 1) ceiling);
// the softmax warpgroups take kSoftmaxRegs, the control and epilogue
// warpgroups kOtherRegs.  The split must add up to exactly the launch pool,
// or an increase could wait forever: launch_instance refuses a build whose
// register count differs.
constexpr int kLaunchRegs = 128;
constexpr int kSoftmaxRegs = 160;
constexpr int kOtherRegs = 96;
static_assert(2 * 128 * kSoftmaxRegs + 2 * 128 * kOtherRegs == kThreads * kLaunchRegs,
              "register split must equal the launch pool");
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8
constexpr float kLn2 = 0.69314718055994531f;

template <int D>
struct Cfg {
  // Three score buffers at both head dimensions.  D = 64: the two halves keep
  // separate accumulators O_a, O_b (TMEM: 3 x 128 + 64 + 64 = 512 columns).
  // D = 128: two 128-column accumulators would leave room for two score
  // buffers only, so the halves share one O (3 x 128 + 128) and agree on a
  // common running max every step (kSharedO, see the softmax).
  static constexpr bool kSharedO = (D == 128);
  static constexpr int kScoreBufs = 3;
  // D = 128: 2 K + 3 V stages (3 + 2 measured 3 % slower at C4 and C5)
  static constexpr int kKStages = (D == 128) ? 2 : 6;
  static constexpr int kVStages = (D == 128) ? 3 : 6;
  static constexpr int kHalves = D / 64;           // 64-column (128-byte) slabs per row
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kSlabQ = BM * 128;          // bytes of one 64-column slab of a Q tile
  static constexpr int kSlabKV = BN * 128;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kKStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kVStages * kKVBytes;
  static_assert(kQBytes == kKVBytes, "an O tile is staged in a V stage");
  // barrier block: q_full q_empty k_full[KS] k_empty[KS] v_full[VS] v_empty[VS]
  // s_full[SB] p_full[SB] pv_done[SB] o_full drain o_staged ml_full ml_empty
  // o_free unit_full[kUnitSlots] unit_empty[kUnitSlots], then 32-bit words:
  // TMEM base, abort flag; then the row statistics the softmax hands to the
  // epilogue (m_a, l_a, m_b, l_b per row); then the ring of decoded units
  static constexpr int kNumBars = 2 + 2 * kKStages + 2 * kVStages + 3 * kScoreBufs + 6 + 2 * kUnitSlots;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kMiscBytes = 8;
  static constexpr int kOffXch = (kOffMisc + kMiscBytes + 15) / 16 * 16;  // 16-byte aligned
  static constexpr int kOffRing = kOffXch + BM * 16;                      // 16-byte aligned
  // kSharedO: the per-step max exchange between the halves, one 32-bit word
  // per (step parity, half, row)
  static constexpr int kOffMx = kOffRing + kUnitSlots * kUnitWords * 4;
  static constexpr int kMxBytes = kSharedO ? 2 * 2 * BM * 4 : 0;
  // Dynamic shared memory starts 1024-byte aligned (the tiles need it); the
  // kernel checks that the layout fits what it was given.
  static constexpr int kSmemBytes = kOffMx + kMxBytes;
  // TMEM columns: score buffers S_b (fp32, BN each; each half's P is written
  // over the first columns of that half), then the accumulators: O_a (keys
  // of the first half of every tile) and O_b (second half), or the one
  // shared O (kColOa == kColOb).
  static __device__ __forceinline__ uint32_t col_s(uint32_t b) { return b * BN; }
  static constexpr uint32_t kColOa = kScoreBufs * BN;
  static constexpr uint32_t kColOb = kSharedO ? kColOa : kColOa + D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kScoreBufs * BN + (kSharedO ? 1 : 2) * D <= 512, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared-memory budget");
  static_assert(kOffRing % 16 == 0, "ring slots are read with 16-byte accesses");
};

// Shared-memory addresses of the barriers (32-bit, one base + constants).
template <int D>
struct Bars {
  static constexpr uint32_t KS = Cfg<D>::kKStages;
  static constexpr uint32_t VS = Cfg<D>::kVStages;
  static constexpr uint32_t SB = Cfg<D>::kScoreBufs;
  uint32_t base;
  __device__ __forceinline__ uint32_t q_full() const { return base; }
  __device__ __forceinline__ uint32_t q_empty() const { return base + 8u; }
  __device__ __forceinline__ uint32_t k_full(uint32_t s) const { return base + 8u * (2 + s); }
  __device__ __forceinline__ uint32_t k_empty(uint32_t s) const { return base + 8u * (2 + KS + s); }
  __device__ __forceinline__ uint32_t v_full(uint32_t s) const { return base + 8u * (2 + 2 * KS + s); }
  __device__ __forceinline__ uint32_t v_empty(uint32_t s) const {
    return base + 8u * (2 + 2 * KS + VS + s);
  }
  __device__ __forceinline__ uint32_t s_full(uint32_t b) const {
    return base + 8u * (2 + 2 * KS + 2 * VS + b);
  }
  __device__ __forceinline__ uint32_t p_full(uint32_t b) const {
    return base + 8u * (2 + 2 * KS + 2 * VS + SB + b);
  }
  // PV of the key tile whose P was in buffer b has completed
  __device__ __forceinline__ uint32_t pv_done(uint32_t b) const {
    return base + 8u * (2 + 2 * KS + 2 * VS + 2 * SB + b);
  }
  __device__ __forceinline__ uint32_t o_full() const { return base + 8u * (2 + 2 * KS + 2 * VS + 3 * SB); }
  __device__ __forceinline__ uint32_t drain() const { return base + 8u * (3 + 2 * KS + 2 * VS + 3 * SB); }
  // every epilogue thread has written its O row into the staging tile
  __device__ __forceinline__ uint32_t o_staged() const { return base + 8u * (4 + 2 * KS + 2 * VS + 3 * SB); }
  // the softmax has written the unit's row statistics / the epilogue has read them
  __device__ __forceinline__ uint32_t ml_full() const { return base + 8u * (5 + 2 * KS + 2 * VS + 3 * SB); }
  __device__ __forceinline__ uint32_t ml_empty() const { return base + 8u * (6 + 2 * KS + 2 * VS + 3 * SB); }
  // the epilogue has read O_a and O_b out of TMEM (the next unit may overwrite them)
  __device__ __forceinline__ uint32_t o_free() const { return base + 8u * (7 + 2 * KS + 2 * VS + 3 * SB); }
  // ring slot s holds a decoded unit / the softmax has read it
  __device__ __forceinline__ uint32_t unit_full(uint32_t s) const {
    return base + 8u * (8 + 2 * KS + 2 * VS + 3 * SB + s);
  }
  __device__ __forceinline__ uint32_t unit_empty(uint32_t s) const {
    return base + 8u * (8 + 2 * KS + 2 * VS + 3 * SB + kUnitSlots + s);
  }
  __device__ __forceinline__ uint32_t tmem_word() const {
    return base + 8u * (8 + 2 * KS + 2 * VS + 3 * SB + 2 * kUnitSlots);
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
  // explicit mask, packed by the pre-pass (null: none); see attn_mask.cu
  const uint32_t* mbits;
  const uint32_t* mvis;
  const uint32_t* mpart;
  const int* mlast;
  int n_ch;         // 32-tile words per row block in mvis / mpart
  int mask_shared;  // 1: one mask for every batch (mask batch 0)
  int n_kt;     // 128-key tiles per (b, h_kv)
  int B, Hq, Hkv, G;
  int Lq, Lk;   // query rows, key/value rows per head
  int d_o;      // elements per row of O in memory: the problem's D (<= the instance's D)
  int64_t o_sb, o_sh, o_sl;  // element strides of O (batch, head, row)
  int n_mb;     // 128-row query tiles per (b, h_q)
  int n_units;  // B * Hq * n_mb
  float scale_log2;
  int causal;
};

struct Unit {
  int bh, b, hq, hkv, mb, m0, kv_len;
  int mblk;  // explicit mask: (mask batch, row block) index of its packed words
  int n;     // key tiles in range of the causal and padding masks
  int last;  // last key tile the unit visits (-1: none; with an explicit mask,
             // tiles without a kept position are skipped)
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

template <bool MASK>
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
  w.hq = w.bh % p.Hq;
  w.hkv = w.hq / p.G;
  w.m0 = mb * BM;
  int kv = p.Lk;
  if (p.valid_len != nullptr) {
    kv = p.valid_len[w.b];
    kv = kv < 0 ? 0 : (kv > p.Lk ? p.Lk : kv);
  }
  w.kv_len = kv;
  const int hi = p.causal ? min(kv, w.m0 + BM) : kv;
  w.n = (hi + BN - 1) / BN;
  w.mb = mb;
  w.last = w.n - 1;
  w.mblk = 0;
  if constexpr (MASK) {
    w.mblk = (p.mask_shared ? 0 : w.b) * p.n_mb + mb;
    if (w.last >= 0) {
      // the last tile in range that has a kept position
      int last = min(w.last, __ldg(p.mlast + w.mblk));
      const uint32_t* vis = p.mvis + static_cast<int64_t>(w.mblk) * p.n_ch;
      while (last >= 0) {
        const uint32_t word = __ldg(vis + (last >> 5)) & (0xFFFFFFFFu >> (31 - (last & 31)));
        if (word != 0u) {
          last = (last & ~31) + 31 - __clz(word);
          break;
        }
        last = (last & ~31) - 1;
      }
      w.last = last;
    }
  }
  return w;
}

// The key tiles a unit visits, in order: 0 .. last without an explicit
// mask; with one, the tiles that have a kept position, read from the
// pre-pass's bit words 32 tiles at a time.  The kernel is instantiated with
// and without the mask (MASK) so that the unmasked kernel carries none of
// this code: its hot loop measured up to 25 % slower with it compiled in.
template <bool MASK>
struct TileWalk {
  const uint32_t* vis = nullptr;
  const uint32_t* part = nullptr;
  int chunk = -1;        // 32-tile word held in v / pt
  uint32_t v = 0, pt = 0;
  __device__ __forceinline__ void init(const KParams& p, const Unit& w) {
    if constexpr (MASK) {
      vis = p.mvis + static_cast<int64_t>(w.mblk) * p.n_ch;
      part = p.mpart + static_cast<int64_t>(w.mblk) * p.n_ch;
      chunk = -1;
    }
  }
  // the first visited tile >= j, or a value > last
  __device__ __forceinline__ int next(int j, int last) {
    if constexpr (MASK) {
      while (j <= last) {
        const int c = j >> 5;
        if (c != chunk) {
          chunk = c;
          v = __ldg(vis + c);
          pt = __ldg(part + c);
        }
        const uint32_t rest = v >> (j & 31);
        if (rest != 0u) return j + __ffs(static_cast<int>(rest)) - 1;
        j = (c + 1) << 5;
      }
    }
    return j;
  }
  // tile j (just returned by next) is partially kept
  __device__ __forceinline__ bool partial(int j) const {
    if constexpr (MASK) return ((pt >> (j & 31)) & 1u) != 0u;
    return false;
  }
};

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

// The same for key tiles [j0, j0 + 32) at once, as a bit mask (bit i: tile
// j0 + i has an exact fp16 copy): lane i reads one flag, a ballot combines
// them, so a warp touches global memory once per 32 key tiles.  Every lane
// of the warp must take part.  fp16 inputs and bf16 without flags: 0.
template <bool BF16>
__device__ __forceinline__ uint32_t v_fp16_mask(const KParams& p, int z_kv, int j0, int n) {
  if constexpr (!BF16) {
    return 0u;
  } else {
    const int j = j0 + static_cast<int>(threadIdx.x & 31);
    int f = 0;
    if (p.vflags != nullptr && j < n) f = __ldg(p.vflags + static_cast<int64_t>(z_kv) * p.n_kt + j);
    return __ballot_sync(0xffffffffu, f != 0);
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

template <int D, bool BF16, bool MASK>
__device__ void producer_role(const KParams& p, const Bars<D>& br, uint32_t smem,
                              const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                              const CUtensorMap* tm_v, const CUtensorMap* tm_v16) {
  using C = Cfg<D>;
  uint32_t q_loads = 0;            // Q tiles loaded so far (one buffer)
  uint32_t k_used = 0, k_par = 0;  // per K stage: loaded at least once / parity of the last load
  uint32_t v_used = 0, v_par = 0;  // per V stage: the same
  uint32_t kit = 0, vit = 0;       // K and V ring items issued
  const uint64_t pol_keep = ptx::policy_evict_last();
  const uint64_t pol_stream = ptx::policy_evict_first();
  bool ok = true;

  // One K or V tile into the next slot of its ring.
  auto load_kv = [&](bool is_v, int j, const Unit& w, int z_kv) -> bool {  // tile j of unit w
    uint32_t& it = is_v ? vit : kit;
    const uint32_t ns = is_v ? C::kVStages : C::kKStages;
    const uint32_t s = it % ns;
    const uint32_t par = (it / ns) & 1u;
    if (!wait_bar(br, p.status, is_v ? br.v_empty(s) : br.k_empty(s), par ^ 1u, kRoleProducer))
      return false;
    ++it;
#ifdef ATTN_TEST_DROP_K_LOAD
    // Test build only (a separate library, never libattn.so): CTA 0 skips
    // its first K-tile load, so the waits for that tile can end only by their
    // time limit -- the path that reports ATTN_ERR_TIMEOUT.
    if (!is_v && blockIdx.x == 0 && it == 1) return true;
#endif
    const uint32_t full = is_v ? br.v_full(s) : br.k_full(s);
    const uint32_t dst = smem + (is_v ? C::kOffV : C::kOffK) + s * C::kKVBytes;
    // bf16 V: the exact fp16 copy of the tile when there is one
    const CUtensorMap* map = !is_v ? tm_k : ((!BF16 || v_split<BF16>(p, z_kv, j)) ? tm_v : tm_v16);
    ptx::mbar_arrive_expect_tx(full, C::kKVBytes);
#pragma unroll
    for (int h = 0; h < C::kHalves; ++h)
      ptx::tma_load_4d_hint(dst + h * C::kSlabKV, map, full, h * 64, j * BN, w.hkv, w.b, pol_keep);
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
    const Unit w = decode_unit<MASK>(p, u);
    if (w.last < 0) continue;
    const int z_kv = w.b * p.Hkv + w.hkv;
    // Q: the buffer is free once the previous unit's last score MMA completed
    if (!wait_bar(br, p.status, br.q_empty(), (q_loads & 1u) ^ 1u, kRoleProducer)) break;
    ++q_loads;
    ptx::mbar_arrive_expect_tx(br.q_full(), C::kQBytes);
#pragma unroll
    for (int h = 0; h < C::kHalves; ++h)
      ptx::tma_load_4d_hint(smem + C::kOffQ + h * C::kSlabQ, tm_q, br.q_full(), h * 64, w.m0, w.hq,
                            w.b, pol_stream);
    // issue order = consumption order over the visited tiles t_0 t_1 ...:
    // K(t_0) .. K(t_SB-1) | V(t_0) K(t_SB) | V(t_1) K(t_SB+1) | ...
    TileWalk<MASK> kw, vw;  // K runs ahead of V: one walker each
    kw.init(p, w);
    vw.init(p, w);
    int kj = kw.next(0, w.last);  // next tile whose K is loaded
    for (int i = 0; ok && i < C::kScoreBufs && kj <= w.last; ++i) {
      ok = load_kv(false, kj, w, z_kv);
      kj = kw.next(kj + 1, w.last);
    }
    for (int j = vw.next(0, w.last); ok && j <= w.last; j = vw.next(j + 1, w.last)) {
      ok = load_kv(true, j, w, z_kv);
      if (ok && kj <= w.last) {
        ok = load_kv(false, kj, w, z_kv);
        kj = kw.next(kj + 1, w.last);
      }
    }
  }
  // Never leave with a copy in flight: wait (bounded) for the last load of
  // every buffer.  In a normal run these phases completed long ago.
  for (uint32_t s = 0; s < C::kKStages; ++s)
    if ((k_used >> s) & 1u) drain_wait(br.k_full(s), (k_par >> s) & 1u);
  for (uint32_t s = 0; s < C::kVStages; ++s)
    if ((v_used >> s) & 1u) drain_wait(br.v_full(s), (v_par >> s) & 1u);
  if (q_loads > 0) drain_wait(br.q_full(), (q_loads - 1u) & 1u);
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
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk & 3) * 32u;
    ptx::mma_ss(d_tmem, desc_add(q_desc, (kk / 4) * C::kSlabQ + off),
                desc_add(k_desc, (kk / 4) * C::kSlabKV + off), idesc, kk > 0 ? 1u : 0u);
  }
}

// O_h += P_h V_h for the two halves of a key tile (h = a: keys 0-63 into
// O_a, h = b: keys 64-127 into O_b; with a shared O both into it).  A = P_h
// from TMEM (16-bit pairs, 8 columns per 16 keys, at the start of its half's
// 64 score columns), B = the half's rows of the V tile as an MN-major
// 128-byte-swizzled operand (16 keys = two 8-row groups).  fp16 V tile (fp16
// inputs, or the exact fp16 copy of a bf16 tile): fp16 P.  bf16 V tile
// (split): O_h += [P_hi | P_lo] [V_h; V_h] with P_lo in the 32 columns after
// P_hi, the same V rows read twice.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t o_a, uint32_t o_b, uint32_t p_tmem,
                                         uint64_t v_desc, bool accumulate, bool split) {
  const uint32_t idesc = split ? ptx::idesc_f16(BM, D, true, true) : ptx::idesc_f16(BM, D, false, true);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    const int h = kk / (BH / 16);
    const int k4 = kk % (BH / 16);
    // a unit's first product starts its accumulator (the shared O: once)
    const bool acc = accumulate || (Cfg<D>::kSharedO ? kk > 0 : k4 > 0);
    ptx::mma_ts(h ? o_b : o_a, p_tmem + h * BH + k4 * 8u, desc_add(v_desc, kk * 2048u), idesc,
                acc ? 1u : 0u);
  }
  if (split) {
#pragma unroll 1
    for (int kk = 0; kk < BN / 16; ++kk) {
      const int h = kk / (BH / 16);
      const int k4 = kk % (BH / 16);
      ptx::mma_ts(h ? o_b : o_a, p_tmem + h * BH + BH / 2 + k4 * 8u, desc_add(v_desc, kk * 2048u),
                  idesc, 1u);
    }
  }
}


// Two issuer warps (one elected lane each issues), so that one warp's
// barrier waits and commits overlap the other's MMAs on the tensor core:
//   * the S issuer issues every score tile in order, S(g) into buffer
//     g % SB; before overwriting a buffer it waits until PV(g-SB), which
//     read P from it, has completed -- the scores run up to SB key tiles
//     ahead of the softmax;
//   * the PV issuer issues PV(j) (both halves) as soon as P(j) is in TMEM.
// Per-buffer completion barriers (pv_done[b]) cannot run two phases ahead of
// a waiter: PV(g+SB) needs S(g+SB), which the S issuer issues only after its
// wait for PV(g).
template <int D, bool BF16, bool MASK>
__device__ void s_issuer_role(const KParams& p, const Bars<D>& br, uint32_t smem, uint32_t tmem) {
  using C = Cfg<D>;
  constexpr uint32_t SB = C::kScoreBufs;
  uint32_t q_phase = 0;
  uint32_t kit = 0;
  uint32_t g = 0;  // score tiles of all units so far: tile g uses buffer g % SB
  // K-major operands (Q, K): leading byte offset unused with 128-byte swizzle,
  // 1024 bytes between 8-row groups
  const uint64_t q_desc = ptx::sdesc_sw128(smem + C::kOffQ, 16, 1024);
  const uint64_t k_desc0 = ptx::sdesc_sw128(smem + C::kOffK, 16, 1024);
  bool ok = true;

  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  for (int r = 0; ok && r < rounds; ++r) {
    const int u = unit_of(r);
    if (u >= p.n_units) continue;
    const Unit w = decode_unit<MASK>(p, u);
    if (w.last < 0) continue;
    if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.q_full(), q_phase, kRoleMma))) break;
    q_phase ^= 1u;
    TileWalk<MASK> tw;
    tw.init(p, w);
    for (int j = tw.next(0, w.last); j <= w.last; j = tw.next(j + 1, w.last), ++g) {
      const uint32_t b = g % SB;
      // the K tile first: it normally landed long ago, and the wait for the
      // buffer below is the one on the critical path
      const uint32_t sk = kit % C::kKStages;
      if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.k_full(sk),
                                            (kit / C::kKStages) & 1u, kRoleMma))) {
        ok = false;
        break;
      }
      ++kit;
      // buffer b held P(g-SB): wait until PV(g-SB) has read it
      if (g >= SB && !__all_sync(0xffffffffu, wait_bar(br, p.status, br.pv_done(b),
                                                       ((g - SB) / SB) & 1u, kRoleMma))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      if (elect_one()) issue_qk<D, BF16>(tmem + C::col_s(b), q_desc, desc_add(k_desc0, sk * C::kKVBytes));
      __syncwarp();
      commit_one(br.s_full(b));
      commit_one(br.k_empty(sk));
      if (j == w.last) commit_one(br.q_empty());  // Q is free once its last S completes
    }
  }
  // Every MMA issued by this warp completes before TMEM is released.
  commit_one(br.drain());
  drain_wait(br.drain(), 0);
}

template <int D, bool BF16, bool MASK>
__device__ void pv_issuer_role(const KParams& p, const Bars<D>& br, uint32_t smem, uint32_t tmem) {
  using C = Cfg<D>;
  constexpr uint32_t SB = C::kScoreBufs;
  uint32_t vit = 0;
  uint32_t g = 0;
  // MN-major V: 64-column slabs kSlabKV apart (leading), 1024 bytes between
  // 8-key groups (stride)
  const uint64_t v_desc0 = ptx::sdesc_sw128(smem + C::kOffV, C::kSlabKV, 1024);
  const uint32_t t_oa = tmem + C::kColOa;
  const uint32_t t_ob = tmem + C::kColOb;
  uint32_t units = 0;  // units with key tiles issued so far
  bool ok = true;

  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  for (int r = 0; ok && r < rounds; ++r) {
    const int u = unit_of(r);
    if (u >= p.n_units) continue;
    const Unit w = decode_unit<MASK>(p, u);
    if (w.last < 0) continue;
    const int z_kv = w.b * p.Hkv + w.hkv;
    uint32_t fmask = 0;
    int fchunk = -1;  // 32-tile chunk fmask holds
    bool first = true;
    TileWalk<MASK> tw;
    tw.init(p, w);
    for (int j = tw.next(0, w.last); j <= w.last; j = tw.next(j + 1, w.last), ++g) {
      if ((j >> 5) != fchunk) {
        fchunk = j >> 5;
        fmask = v_fp16_mask<BF16>(p, z_kv, j & ~31, w.n);
      }
      const uint32_t b = g % SB;
      const uint32_t sv = vit % C::kVStages;
      if (!__all_sync(0xffffffffu,
                      wait_bar(br, p.status, br.v_full(sv), (vit / C::kVStages) & 1u, kRoleMma))) {
        ok = false;
        break;
      }
      ++vit;
      const bool split = BF16 && ((fmask >> (j & 31)) & 1u) == 0u;
      // P last: V is normally in shared memory long before the softmax
      // delivers P(j)
      if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.p_full(b), (g / SB) & 1u, kRoleMma))) {
        ok = false;
        break;
      }
      // The unit's first P.V overwrites O_a and O_b: the epilogue must have
      // read the previous unit's out of TMEM (it normally has, long before)
      if (first && units > 0 &&
          !__all_sync(0xffffffffu, wait_bar(br, p.status, br.o_free(), (units - 1u) & 1u, kRoleMma))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      if (elect_one())
        issue_pv<D>(t_oa, t_ob, tmem + C::col_s(b), desc_add(v_desc0, sv * C::kKVBytes), !first,
                    split);
      __syncwarp();
      first = false;
      commit_one(br.pv_done(b));
      // the unit's last V stage is released by the epilogue (it stages O)
      if (j == w.last) {
        commit_one(br.o_full());
      } else {
        commit_one(br.v_empty(sv));
      }
    }
    ++units;
  }
  commit_one(br.drain());
  drain_wait(br.drain(), 0);
}

// ------------------------------------------------------------------ unit decoder

// A decoded unit and its fp16-flag mask in a ring slot (kUnitWords words).
__device__ __forceinline__ void write_unit(uint32_t slot_addr, const Unit& w, uint32_t fmask) {
  const uint32_t v[kUnitWords] = {static_cast<uint32_t>(w.bh), static_cast<uint32_t>(w.b),
                                  static_cast<uint32_t>(w.hq), static_cast<uint32_t>(w.hkv),
                                  static_cast<uint32_t>(w.mb), static_cast<uint32_t>(w.m0),
                                  static_cast<uint32_t>(w.kv_len), static_cast<uint32_t>(w.mblk),
                                  static_cast<uint32_t>(w.n), static_cast<uint32_t>(w.last), fmask, 0u};
#pragma unroll
  for (int i = 0; i < kUnitWords; i += 4)
    ptx::st_shared_v4(slot_addr + i * 4, make_uint4(v[i], v[i + 1], v[i + 2], v[i + 3]));
}

__device__ __forceinline__ Unit read_unit(uint32_t slot_addr, uint32_t* fmask) {
  const uint4 a = ptx::ld_shared_v4(slot_addr);
  const uint4 b = ptx::ld_shared_v4(slot_addr + 16u);
  const uint4 c = ptx::ld_shared_v4(slot_addr + 32u);
  Unit w;
  w.bh = static_cast<int>(a.x);
  w.b = static_cast<int>(a.y);
  w.hq = static_cast<int>(a.z);
  w.hkv = static_cast<int>(a.w);
  w.mb = static_cast<int>(b.x);
  w.m0 = static_cast<int>(b.y);
  w.kv_len = static_cast<int>(b.z);
  w.mblk = static_cast<int>(b.w);
  w.n = static_cast<int>(c.x);
  w.last = static_cast<int>(c.y);
  *fmask = c.z;
  return w;
}

// Warp 11: decodes the CTA's units in order, kUnitSlots ahead of the
// softmax, and checks valid_len (values outside [0, Lk] are clamped by the
// decode and reported in the status word).
template <int D, bool BF16, bool MASK>
__device__ void decoder_role(const KParams& p, const Bars<D>& br, uint32_t smem) {
  using C = Cfg<D>;
  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  const bool lead = (threadIdx.x & 31) == 0;
  for (int r = 0; r < rounds; ++r) {
    const int u = unit_of(r);
    if (u >= p.n_units) break;
    const Unit w = decode_unit<MASK>(p, u);
    const uint32_t fmask = v_fp16_mask<BF16>(p, w.b * p.Hkv + w.hkv, 0, w.n);  // whole warp
    if (lead && p.valid_len != nullptr) {
      const int vl = p.valid_len[w.b];
      if (vl < 0 || vl > p.Lk) atomicOr(p.status, kStatusValidLenClamped);
    }
    const uint32_t slot = static_cast<uint32_t>(r) % kUnitSlots;
    if (r >= kUnitSlots &&
        !__all_sync(0xffffffffu, wait_bar(br, p.status, br.unit_empty(slot),
                                          (static_cast<uint32_t>(r) / kUnitSlots - 1u) & 1u,
                                          kRoleProducer)))
      return;
    if (lead) {
      write_unit(smem + C::kOffRing + slot * (kUnitWords * 4), w, fmask);
      ptx::mbar_arrive(br.unit_full(slot));  // release: the slot's words before the arrive
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ softmax + epilogue

// P for one half row (64 keys in registers), 32 keys at a time, written over
// the half's S columns in TMEM; returns the half row's sum of P.  fp16 V
// tile: P rounded to fp16 in the half's columns [0, 32).  bf16 V tile
// (SPLIT): P = P_hi + P_lo with P_hi = p truncated to bf16 (columns [0, 32))
// and P_lo = bf16(p - P_hi) (columns [32, 64)); a single bf16 P (unit
// roundoff 2^-8) is too coarse for rows dominated by a few keys, the pair
// leaves a relative error below 2^-15.  Masked keys arrive as -inf scores and
// give P = 0.
template <bool SPLIT>
__device__ __forceinline__ float exp_half(const uint32_t (&s)[BH], uint64_t sc2, uint64_t nm2,
                                          uint32_t t_s) {
  uint64_t rsum2[4];  // independent partial sums, two lanes each
#pragma unroll
  for (int k = 0; k < 4; ++k) rsum2[k] = 0ull;
#pragma unroll
  for (int qtr = 0; qtr < BH / 32; ++qtr) {
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
      const float p0 = ptx::ex2_approx(x0);
      const float p1 = ptx::ex2_approx(x1);
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
    if constexpr (SPLIT) ptx::tmem_st16(t_s + BH / 2 + qtr * 16, lo);
  }
  float ra, rb;
  ptx::f2_unpack(ptx::f2_add(ptx::f2_add(rsum2[0], rsum2[1]), ptx::f2_add(rsum2[2], rsum2[3])), ra, rb);
  return ra + rb;
}

// Shared O (D = 128): the two halves of a row agree on one running max at
// every step.  Each thread writes its half row's maximum into a shared-memory
// word per (step parity, half, row); the two warps of a TMEM lane quadrant
// (warp q and q + 4) meet at named barrier kXBar0 + q, and each reads its
// partner's word.  Two parities: a word is rewritten two exchanges later, by
// when the partner has passed the exchange in between (so it has read it).
// Both halves take fmaxf of the same two values, so they agree (up to the
// sign of a zero maximum, which changes no exponential and no result).
// A named-barrier wait has no time limit, so a warp that leaves the softmax
// early (a bounded wait elsewhere gave up, which raises the CTA's abort flag)
// arrives once more at its quadrant's barrier on the way out: that releases
// the one exchange its partner can be waiting in or reach next, and the
// partner, reading the abort flag right after every exchange, leaves too.
constexpr uint32_t kXBar0 = 1;  // named barriers 1-4 (0 is __syncthreads)

template <class BarsT>
__device__ __forceinline__ bool exchange_max(const BarsT& br, uint32_t mine0, uint32_t other0,
                                             uint32_t quad, uint32_t& xs, float& mx) {
  const uint32_t off = (xs & 1u) * (2u * BM * 4u);
  ++xs;
  ptx::st_shared_f32(mine0 + off, mx);
  ptx::named_barrier_sync(kXBar0 + quad, 64);
  const float partner = ptx::ld_shared_f32(other0 + off);
  const bool abort = ptx::ld_shared_volatile(br.abort_word()) != 0u;
  mx = fmaxf(mx, partner);
  return !abort;
}

// O_h *= alpha over ncols columns of this thread's TMEM row, once PV(j-1)
// (barrier `bar`, phase `parity`) has completed -- the rare rescale of the
// softmax step, kept out of line so that the step's hot code stays compact.
// The wait is bounded like wait_bar's; false: it gave up (recorded) or the
// CTA is aborting.
__device__ __noinline__ bool rescale_o(uint32_t bar, uint32_t parity, uint32_t abort_word,
                                       int* status, uint32_t t_oh, int ncols, float alpha) {
  bool done = ptx::mbar_try_wait(bar, parity);
  if (!done) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
      if (ptx::mbar_try_wait(bar, parity)) {
        done = true;
        break;
      }
      if (ptx::ld_shared_volatile(abort_word) != 0u) break;
      if (ptx::globaltimer_ns() - t0 > ATTN_WAIT_LIMIT_NS) {
        ptx::st_shared_volatile(abort_word, 1u);
        atomicOr(status, kStatusTimeout | kRoleSoftmax);
        break;
      }
    }
  }
  if (!__all_sync(0xffffffffu, done)) return false;
  ptx::tc_fence_after();
#pragma unroll 1
  for (int c0 = 0; c0 < ncols; c0 += 32) {
    uint32_t o[32];
    ptx::tmem_ld32(t_oh + c0, o);
#pragma unroll
    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
    ptx::tmem_st32(t_oh + c0, o);
  }
  return true;
}

// Two softmax warpgroups share every query tile: warps 0-3 (half a) own key
// columns 0-63 of each key tile and warps 4-7 (half b) columns 64-127, for
// the same rows (warp w and w + 4 read the same TMEM lane quadrant).  At
// D = 64 each half runs its own online softmax -- running max m_h, sum l_h
// and the partial accumulator O_h over its keys only -- so the two never wait
// for each other while the tile streams; they meet once per unit, in the
// epilogue, where the partial results combine exactly:
//   m = max(m_a, m_b),  l = l_a 2^(m_a - m) + l_b 2^(m_b - m),
//   O = (O_a 2^(m_a - m) + O_b 2^(m_b - m)) / l.
// At D = 128 (shared O) the halves exchange their maxima every step, so
// m_a = m_b and the same formulas reduce to O / (l_a + l_b).
template <int D, bool BF16, bool MASK>
__device__ bool softmax_role(const KParams& p, const Bars<D>& br, uint32_t smem, uint32_t tmem) {
  using C = Cfg<D>;
  constexpr int SB = C::kScoreBufs;
  const int lane_row = threadIdx.x & 127;           // row within the tile = TMEM lane
  const int half = static_cast<int>(threadIdx.x) >> 7;  // 0: keys 0-63 of a tile, 1: 64-127
  const uint32_t quad = (threadIdx.x >> 5) & 3u;    // this warp's 32-lane TMEM quadrant
  const uint32_t lane_addr = (quad * 32u) << 16;
  // the O columns this half rescales: its own accumulator, or its half of
  // the shared one
  constexpr int kOCols = C::kSharedO ? D / 2 : D;
  const uint32_t t_oh =
      tmem + lane_addr + (C::kSharedO ? C::kColOa + half * kOCols : (half ? C::kColOb : C::kColOa));
  // this row's statistics for the epilogue: (m_a, l_a) then (m_b, l_b)
  const uint32_t xch = smem + C::kOffXch + static_cast<uint32_t>(lane_row) * 16u + half * 8u;
  // shared O: this thread's and its partner's max-exchange slots (parity 0)
  const uint32_t mx_mine = smem + C::kOffMx + static_cast<uint32_t>(half * BM + lane_row) * 4u;
  const uint32_t mx_other = smem + C::kOffMx + static_cast<uint32_t>((half ^ 1) * BM + lane_row) * 4u;
  uint32_t xs = 0;  // max exchanges so far
  const float scale_log2 = p.scale_log2;
  uint32_t epi = 0;  // units with key tiles done so far (their statistics handed over)
  uint32_t g = 0;    // score (and V) tiles of all units so far (buffer g % SB)

  // Units come decoded, with the fp16 flags of their first 32 key tiles,
  // from the decoder warp through a shared-memory ring: the integer
  // divisions and the global loads of valid_len and the flags stay off the
  // softmax warps.  Unit indices grow with the round, so the first one past
  // the end ends the loop.
  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  for (int r = 0; r < rounds; ++r) {
    if (unit_of(r) >= p.n_units) break;
    const uint32_t slot = static_cast<uint32_t>(r) % kUnitSlots;
    if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.unit_full(slot),
                                          (static_cast<uint32_t>(r) / kUnitSlots) & 1u, kRoleSoftmax)))
      return false;
    uint32_t fmask;
    const Unit w = read_unit(smem + C::kOffRing + slot * (kUnitWords * 4), &fmask);
    ptx::mbar_arrive(br.unit_empty(slot));
    const int row = w.m0 + lane_row;
    const bool row_ok = row < p.Lq;
    if (w.last < 0) continue;  // no visible key: the epilogue writes O = 0, LSE = -inf
    const int z_kv = w.b * p.Hkv + w.hkv;
    // keys < key_lim are visible to this row
    const int key_lim = p.causal ? min(w.kv_len, row + 1) : w.kv_len;
    float m = -INFINITY;  // running max of this half's keys, log2 units (scaled)
    float l = 0.f;
    bool ok = true;
    // S(gg) was seen complete by the look-ahead test of the previous step
    // (the test is an acquire like a wait): no blocking wait needed
    bool s_ready = false;
    int fchunk = 0;     // 32-tile chunk fmask holds
    uint32_t cnt = 0;   // key tiles of this unit visited so far
    TileWalk<MASK> tw;
    tw.init(p, w);
    // D = 64 without an explicit mask: the key tiles below j_plain are
    // visible to every row of the unit in both halves (the causal and padding
    // limits of the unit's first row lie beyond them), so they run in a first
    // pass whose copy of the step has no masking code at all (C2 +2.4 %, C3
    // +5.5 % against one loop carrying it); the rest -- the diagonal and the
    // padding edge -- in a second pass with it.  D = 128 (measured no faster)
    // and explicit masks: one pass.
    constexpr bool kSplit = !MASK && !C::kSharedO;
    const int j_plain = kSplit ? (p.causal ? min(w.kv_len, w.m0 + 1) : w.kv_len) / BN : 0;
    int j = tw.next(0, w.last);
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const bool plain = kSplit && pass == 0;  // compile-time in each unrolled copy
      if (!kSplit && pass == 0) continue;
      const int j_end = plain ? min(j_plain, w.last + 1) : w.last + 1;
      for (; j < j_end; j = tw.next(j + 1, w.last), ++cnt) {
        const uint32_t gg = g + cnt;
        const uint32_t b = gg % SB;
        const uint32_t t_s = tmem + lane_addr + C::col_s(b) + static_cast<uint32_t>(half * BH);
        // P format of this key tile: fp16 P, or the bf16 pair (split)
        if ((j >> 5) != fchunk) {
          fchunk = j >> 5;
          fmask = v_fp16_mask<BF16>(p, z_kv, j & ~31, w.n);
        }
        const bool split = BF16 && ((fmask >> (j & 31)) & 1u) == 0u;
        // explicit mask: this row's 64 bits of the half tile when the tile is
        // partial (loaded before the wait, to hide its latency)
        const bool partial = tw.partial(j);
        uint2 keep = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        if constexpr (MASK) {
          if (partial && row_ok) {
            const int64_t mrow = static_cast<int64_t>(p.mask_shared ? 0 : w.b) * p.Lq + row;
            keep = __ldg(reinterpret_cast<const uint2*>(p.mbits + (mrow * p.n_kt + j) * 4 + half * 2));
          }
        }
        if (!s_ready) {
          ok = wait_bar(br, p.status, br.s_full(b), (gg / SB) & 1u, kRoleSoftmax);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        ptx::tc_fence_after();
        // the half row's scores with their maximum, reduced by the load itself
        uint32_t s[BH];
        float mx = ptx::tmem_ld64_max(t_s, s);
        const int n0 = j * BN + half * BH;  // key of column 0 of this half
        const bool masked =
            !plain && (partial || (n0 + BH > w.kv_len) || (p.causal && n0 + BH - 1 > w.m0));
        const int c_lim = key_lim - n0;  // columns c < c_lim are visible
        // Boundary and partially masked tiles only: invisible scores become
        // -inf and the maximum is taken again over what is left, so the
        // exponentials below are the same code for every tile (one copy of the
        // unrolled loop keeps the hot code small); exp2(-inf * scale - m) = 0
        // because the scale is > 0 (a zero sm_scale arrives as FLT_MIN).
        if (masked) {
          if constexpr (MASK) {
            // columns >= c_lim leave the keep bits first; then per column one
            // prmt replicates its bit (moved to a byte's sign) over a word and
            // one logic op selects the score or -inf: about the cost of the
            // implicit masks' compare-and-select (a per-column bit test
            // measured ~30 % slower on every step, partial or not)
            uint32_t kw[2] = {keep.x, keep.y};
  #pragma unroll
            for (int wd = 0; wd < 2; ++wd) {
              const int n = c_lim - 32 * wd;  // columns of this word below c_lim
              kw[wd] &= n >= 32 ? 0xFFFFFFFFu : (n <= 0 ? 0u : (1u << n) - 1u);
            }
  #pragma unroll
            for (int wd = 0; wd < 2; ++wd) {
  #pragma unroll
              for (int c0 = 0; c0 < 8; ++c0) {
                const uint32_t t = kw[wd] << (7 - c0);  // bit c0 + 8k -> sign of byte k
  #pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint32_t m = ptx::prmt(t, 0u, 0x8888u + 0x1111u * k);
                  const int c = 32 * wd + 8 * k + c0;
                  s[c] = (s[c] & m) | (0xFF800000u & ~m);
                }
              }
            }
          } else {
  #pragma unroll
            for (int c = 0; c < BH; ++c) s[c] = (c < c_lim) ? s[c] : 0xFF800000u;
          }
          // max of the visible scores: 8 independent chains of 3-input maxima
          float mxk[8];
  #pragma unroll
          for (int k = 0; k < 8; ++k) mxk[k] = -INFINITY;
  #pragma unroll
          for (int i = 0; i < BH / 2; ++i)
            mxk[i & 7] = ptx::max3(mxk[i & 7], __uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
          mx = ptx::max3(ptx::max3(mxk[0], mxk[1], mxk[2]), ptx::max3(mxk[3], mxk[4], mxk[5]),
                         fmaxf(mxk[6], mxk[7]));
        }
        // shared O: the row's max over both halves (the same value in both)
        if constexpr (C::kSharedO) {
          if (!__all_sync(0xffffffffu, exchange_max(br, mx_mine, mx_other, quad, xs, mx))) {
            ok = false;
            break;
          }
        }
        const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * scale_log2;
        const float m_new = fmaxf(m, m_tile);
        float alpha = 1.f;
        bool rescale = false;
        if (m_new > m + kRescaleLog2) {  // also taken on the first visible key (m = -inf)
          alpha = ptx::ex2_approx(m - m_new);
          m = m_new;
          rescale = true;
        }
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        // look ahead (non-blocking): has S(gg+1) completed?  Its answer is used
        // at the next step, so the test's latency hides behind the exponentials.
        // S(gg+1) may be the next unit's first tile: g counts every tile.  With
        // three score buffers the scores are normally ready (with two, at
        // D = 128 before the shared O, it measured slower).
        if constexpr (SB > 2)
          s_ready = __all_sync(0xffffffffu, ptx::mbar_test_wait(br.s_full((gg + 1u) % SB), ((gg + 1u) / SB) & 1u));
        const uint64_t sc2 = ptx::f2_pack(scale_log2, scale_log2);
        const uint64_t nm2 = ptx::f2_pack(neg_m, neg_m);
        // P over the half's S columns (every S value is already in registers)
        float rowsum;
        if (!split) {
          rowsum = exp_half<false>(s, sc2, nm2, t_s);
        } else if constexpr (BF16) {
          rowsum = exp_half<true>(s, sc2, nm2, t_s);
        } else {
          rowsum = 0.f;
        }
        l = l * alpha + rowsum;
        // O_h was accumulated against the old max: rescale it before PV(j)
        // runs.  PV(j-SB) and earlier are complete (S(j) was issued after
        // PV(j-SB) completed); PV(j-1) may still be running: wait for it (the
        // tensor core completes them in order).
        if (cnt > 0 && __any_sync(0xffffffffu, rescale)) {
          const uint32_t done_bar = br.pv_done((gg - 1u) % SB);
          const uint32_t done_par = ((gg - 1u) / SB) & 1u;
          if constexpr (!C::kSharedO) {
            // D = 64: out of line (C2 +2.4 %, C3 +1 %); at D = 128 that measured
            // slower where rescales are frequent (C5, Q x 4)
            if (!rescale_o(done_bar, done_par, br.abort_word(), p.status, t_oh, kOCols, alpha)) {
              ok = false;
              break;
            }
          } else {
            ok = wait_bar(br, p.status, done_bar, done_par, kRoleSoftmax);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
  #pragma unroll 1
            for (int c0 = 0; c0 < kOCols; c0 += 32) {
              uint32_t o[32];
              ptx::tmem_ld32(t_oh + c0, o);
  #pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              ptx::tmem_st32(t_oh + c0, o);
            }
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(br.p_full(b));
      }
      if (!ok) break;
    }
    g += cnt;
    if (!ok) return false;
    // Hand this half's row statistics to the epilogue warpgroup, which
    // combines the halves and writes O and the LSE once the unit's last P.V
    // has completed; meanwhile this warp goes on with the next unit.  The
    // slot is free once the epilogue has read the previous unit's values.
    if (epi > 0) {
      ok = wait_bar(br, p.status, br.ml_empty(), (epi - 1u) & 1u, kRoleSoftmax);
      if (!__all_sync(0xffffffffu, ok)) return false;
    }
    ptx::st_shared_f32(xch, m);
    ptx::st_shared_f32(xch + 4u, l);
    ptx::mbar_arrive(br.ml_full());
    ++epi;
  }
  return true;
}

// ------------------------------------------------------------------ epilogue

// Warps 12-15, one query row per thread (warp 12 + q reads TMEM lane quadrant
// q), one unit behind the softmax.  Per unit: the two halves' statistics give
//   m = max(m_a, m_b),  l = l_a 2^(m_a - m) + l_b 2^(m_b - m),
//   O = (O_a 2^(m_a - m) + O_b 2^(m_b - m)) / l,  LSE = ln 2 (m + log2 l);
// O_a and O_b are read out of TMEM as soon as the unit's last P.V has
// completed (then o_free lets the next unit's first P.V overwrite them), O is
// staged in the V ring stage of the unit's last key tile in the TMA layout
// and written with one TMA store per 64-column slab, and the stage is handed
// back to the producer once the store has read it.  A unit with no visible
// key gets O = 0 and LSE = -inf with plain stores.
template <int D, bool BF16, bool MASK>
__device__ void epilogue_role(const KParams& p, const Bars<D>& br, uint32_t smem, uint32_t tmem,
                              const CUtensorMap* tm_o) {
  using C = Cfg<D>;
  const int t = static_cast<int>(threadIdx.x) - kEpiWarp0 * 32;  // row within the tile = TMEM lane
  const uint32_t quad = static_cast<uint32_t>(t) >> 5;
  const uint32_t lane_addr = (quad * 32u) << 16;
  const uint32_t t_oa = tmem + lane_addr + C::kColOa;
  const uint32_t t_ob = tmem + lane_addr + C::kColOb;
  const uint32_t xch = smem + C::kOffXch + static_cast<uint32_t>(t) * 16u;
  const bool leader = t == 0;  // issues the O stores
  uint32_t epi = 0;            // units with key tiles so far
  uint32_t g = 0;              // V tiles of all units so far (the staging stage)
  const int rounds = (p.n_units + gridDim.x - 1) / gridDim.x;
  for (int r = 0; r < rounds; ++r) {
    const int u = unit_of(r);
    if (u >= p.n_units) break;
    const Unit w = decode_unit<MASK>(p, u);
    const int row = w.m0 + t;
    const bool row_ok = row < p.Lq;
    const int64_t grow = static_cast<int64_t>(w.bh) * p.Lq + row;  // LSE row
    if (w.last < 0) {  // no visible key: O = 0, LSE = -inf
      if (row_ok) {
        // rows of O are d_o elements long (D = 16 and 32 run the D = 64 instance)
        const int64_t orow = w.b * p.o_sb + w.hq * p.o_sh + row * p.o_sl;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) + orow * 2);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          if (c < p.d_o / 8) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (p.lse != nullptr) p.lse[grow] = -INFINITY;
      }
      continue;
    }
    // visited key tiles of the unit (the staging stage is the last one's)
    uint32_t n_tiles = static_cast<uint32_t>(w.last) + 1u;
    if constexpr (MASK) {
      TileWalk<MASK> tw;
      tw.init(p, w);
      n_tiles = 0;
      for (int j = tw.next(0, w.last); j <= w.last; j = tw.next(j + 1, w.last)) ++n_tiles;
    }
    g += n_tiles;
    // the row statistics of both halves
    if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.ml_full(), epi & 1u, kRoleEpilogue)))
      return;
    const float ma = ptx::ld_shared_f32(xch), la = ptx::ld_shared_f32(xch + 4u);
    const float mb = ptx::ld_shared_f32(xch + 8u), lb = ptx::ld_shared_f32(xch + 12u);
    ptx::mbar_arrive(br.ml_empty());
    // a half (with an explicit mask: both) may have seen no visible key
    const float mm = fmaxf(ma, mb);
    const float ea = (ma == -INFINITY) ? 0.f : ptx::ex2_approx(ma - mm);
    const float eb = (mb == -INFINITY) ? 0.f : ptx::ex2_approx(mb - mm);
    const float ll = la * ea + lb * eb;
    const float inv_l = ll > 0.f ? 1.f / ll : 0.f;  // no visible key: O = 0
    const float sa = ea * inv_l, sb = eb * inv_l;
    if (row_ok && p.lse != nullptr)
      p.lse[grow] = ll > 0.f ? (mm + ptx::lg2_approx(ll)) * kLn2 : -INFINITY;
    // O_a and O_b: complete once the unit's last P.V is
    if (!__all_sync(0xffffffffu, wait_bar(br, p.status, br.o_full(), epi & 1u, kRoleEpilogue)))
      return;
    ptx::tc_fence_after();
    // staging tile: the V stage of this unit's last key tile; its P.V has
    // completed (o_full)
    const uint32_t vstage = (g - 1u) % C::kVStages;
    const uint32_t stage = smem + C::kOffV + vstage * C::kKVBytes;
    // O as 16-bit pairs into the staging tile: 64-column slabs of 128-byte
    // rows, the 16-byte chunk k of row r at chunk position k ^ (r % 8) (the
    // 128-byte swizzle of the O tensor map)
    const uint32_t stage_row = stage + static_cast<uint32_t>(t) * 128u;
    const uint32_t rsw = static_cast<uint32_t>(t) & 7u;
    const uint64_t sa2 = ptx::f2_pack(sa, sa);
    const uint64_t sb2 = ptx::f2_pack(sb, sb);
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 16) {
      uint32_t oa[16], ob[C::kSharedO ? 1 : 16];
      ptx::tmem_ld16(t_oa + c0, oa);
      if constexpr (!C::kSharedO) ptx::tmem_ld16(t_ob + c0, ob);
      if (c0 + 16 == D) {  // every TMEM read of this unit is done
        ptx::tc_fence_before();
        ptx::mbar_arrive(br.o_free());
      }
      uint32_t h[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint64_t a2 = ptx::f2_pack(__uint_as_float(oa[2 * c]), __uint_as_float(oa[2 * c + 1]));
        uint64_t o2;
        if constexpr (C::kSharedO) {
          o2 = ptx::f2_mul(a2, sa2);  // one accumulator: m_a = m_b, so sa = 1 / l
        } else {
          o2 = ptx::f2_fma(a2, sa2,
                           ptx::f2_mul(ptx::f2_pack(__uint_as_float(ob[2 * c]), __uint_as_float(ob[2 * c + 1])),
                                       sb2));
        }
        float o0, o1;
        ptx::f2_unpack(o2, o0, o1);
        h[c] = pack2<BF16>(o0, o1);
      }
      const uint32_t slab = stage_row + static_cast<uint32_t>(c0 / 64) * C::kSlabQ;
      const uint32_t k0 = static_cast<uint32_t>(c0 % 64) / 8u;
#pragma unroll
      for (int i = 0; i < 2; ++i)
        ptx::st_shared_v4(slab + (((k0 + i) ^ rsw) << 4),
                          make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]));
    }
    ptx::fence_proxy_async_shared();  // the generic-proxy writes, before the TMA reads them
    ptx::mbar_arrive(br.o_staged());
    if (leader) {
      // rows past Lq are outside the tensor map and are not written
      if (!wait_bar(br, p.status, br.o_staged(), epi & 1u, kRoleEpilogue)) return;
#pragma unroll
      for (int hs = 0; hs < C::kHalves; ++hs)
        ptx::tma_store_4d(tm_o, stage + hs * C::kSlabQ, hs * 64, w.m0, w.hq, w.b);
      ptx::bulk_commit_group();
      // once the store has read the staging tile, the producer may refill it
      ptx::bulk_wait_read_all();
      ptx::mbar_arrive(br.v_empty(vstage));
    }
    __syncwarp();
    ++epi;
  }
}

// ------------------------------------------------------------------ kernel

template <int D, bool BF16, bool MASK>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_v16,
                       const __grid_constant__ CUtensorMap tm_o, const KParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t smem = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  // the layout needs a 1024-byte aligned base and no more than kSmemBytes:
  // otherwise leave at once (every thread alike, before any barrier exists)
  if (smem != ptx::smem_u32(smem_raw)) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  const Bars<D> br{smem + C::kOffBar};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ptx::mbar_init(br.q_full(), 1);
    ptx::mbar_init(br.q_empty(), 1);
    for (int s = 0; s < C::kKStages; ++s) {
      ptx::mbar_init(br.k_full(s), 1);
      ptx::mbar_init(br.k_empty(s), 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      ptx::mbar_init(br.v_full(s), 1);
      ptx::mbar_init(br.v_empty(s), 1);
    }
    for (int b = 0; b < C::kScoreBufs; ++b) {
      ptx::mbar_init(br.s_full(b), 1);
      ptx::mbar_init(br.p_full(b), kSoftmaxThreads);
    }
    for (int b = 0; b < C::kScoreBufs; ++b) ptx::mbar_init(br.pv_done(b), 1);
    ptx::mbar_init(br.o_full(), 1);
    ptx::mbar_init(br.drain(), 2);  // one commit from each issuer
    ptx::mbar_init(br.o_staged(), kEpiThreads);
    ptx::mbar_init(br.ml_full(), kSoftmaxThreads);
    ptx::mbar_init(br.ml_empty(), kEpiThreads);
    ptx::mbar_init(br.o_free(), kEpiThreads);
    for (int s = 0; s < kUnitSlots; ++s) {
      ptx::mbar_init(br.unit_full(s), 1);
      ptx::mbar_init(br.unit_empty(s), kSoftmaxThreads);
    }
    ptx::st_shared_volatile(br.abort_word(), 0u);
    ptx::fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
    if constexpr (BF16) ptx::prefetch_tensormap(&tm_v16);
  }
  if (warp == kEpiWarp0 && lane == 0) ptx::prefetch_tensormap(&tm_o);
  if (warp == kPvWarp) {
    ptx::tmem_alloc(br.tmem_word(), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ptx::ld_shared_volatile(br.tmem_word());

  if (warp >= kEpiWarp0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    epilogue_role<D, BF16, MASK>(p, br, smem, tmem, &tm_o);  // warps 12-15
    // the last O store: complete before the CTA (and its shared memory) goes
    if (warp == kEpiWarp0 && lane == 0) ptx::bulk_wait_all();
  } else if (warp >= kProducerWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    if (warp == kProducerWarp) {
      if (lane == 0) producer_role<D, BF16, MASK>(p, br, smem, &tm_q, &tm_k, &tm_v, &tm_v16);
    } else if (warp == kPvWarp) {
      pv_issuer_role<D, BF16, MASK>(p, br, smem, tmem);  // whole warp
    } else if (warp == kSWarp) {
      s_issuer_role<D, BF16, MASK>(p, br, smem, tmem);  // whole warp
    } else {
      decoder_role<D, BF16, MASK>(p, br, smem);  // warp 11, whole warp
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    const bool done = softmax_role<D, BF16, MASK>(p, br, smem, tmem);  // warps 0-7
    // shared O: a half that left early releases its partner's next exchange
    if constexpr (C::kSharedO)
      if (!done) ptx::named_barrier_arrive(kXBar0 + ((threadIdx.x >> 5) & 3u), 64);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kPvWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool BF16, bool MASK>
cudaError_t launch_instance(const Problem& pr, const CUtensorMap* maps, int num_sms) {
  using C = Cfg<D>;
  // the shared-memory opt-in is per device; set once per (D, dtype) instance and device
  static std::atomic<uint64_t> configured{0};
  auto kern = attn_fwd_tc_kernel<D, BF16, MASK>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit == 0 || (configured.load(std::memory_order_relaxed) & bit) == 0) {
    // The setmaxnreg split is only safe when the CTA is launched with exactly
    // kLaunchRegs registers per thread: refuse to launch anything else.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidKernelImage;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_relaxed);
  }
  KParams kp;
  kp.o = pr.o;
  kp.lse = pr.lse;
  kp.valid_len = pr.valid_len;
  kp.status = pr.status;
  kp.vflags = pr.vflags;
  kp.mbits = pr.mbits;
  kp.mvis = pr.mvis;
  kp.mpart = pr.mpart;
  kp.mlast = pr.mlast;
  kp.mask_shared = pr.mask_sb == 0 ? 1 : 0;
  kp.n_kt = (pr.Lk + BN - 1) / BN;
  kp.B = pr.B;
  kp.Hq = pr.Hq;
  kp.Hkv = pr.Hkv;
  kp.Lq = pr.Lq;
  kp.Lk = pr.Lk;
  kp.G = pr.Hq / pr.Hkv;
  kp.d_o = pr.D;
  kp.o_sb = pr.so.b;
  kp.o_sh = pr.so.h;
  kp.o_sl = pr.so.l;
  kp.n_mb = (pr.Lq + BM - 1) / BM;
  kp.n_ch = (kp.n_kt + 31) / 32;
  kp.n_units = pr.B * pr.Hq * kp.n_mb;
  // A zero scale is passed as the smallest normal float: every product
  // s * scale then rounds to zero exactly as with 0 (all visible keys get
  // P = 1), while -inf (a masked score) times it stays -inf and gives P = 0.
  kp.scale_log2 = pr.sm_scale > 0.f ? pr.sm_scale * 1.4426950408889634f : 1.17549435e-38f;
  kp.causal = pr.causal;
  const int grid = kp.n_units < num_sms ? kp.n_units : num_sms;
  kern<<<grid, kThreads, C::kSmemBytes, pr.stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], kp);
  return cudaGetLastError();
}

}  // namespace

bool tc_config(int D, TcConfig* out) {
  if (D == 16 || D == 32 || D == 64) {  // D < 64: the D = 64 kernel on zero-filled columns
    *out = {BM, 1, BN, Cfg<64>::kKStages + Cfg<64>::kVStages, kThreads, Cfg<64>::kSmemBytes,
            static_cast<int>(Cfg<64>::kTmemCols)};
    return true;
  }
  if (D == 128) {
    *out = {BM, 1, BN, Cfg<128>::kKStages + Cfg<128>::kVStages, kThreads, Cfg<128>::kSmemBytes,
            static_cast<int>(Cfg<128>::kTmemCols)};
    return true;
  }
  return false;
}

// D = 16 and 32 run the D = 64 instance: their tensor maps have an inner
// extent of D with 64-column boxes, so TMA fills columns D..63 of every Q, K
// and V tile with zeros (Q.K^T and P.V unchanged; O's extra columns are 0)
// and the O store writes only the D columns inside the tensor.
cudaError_t launch_tc(const Problem& p, const CUtensorMap* maps, int num_sms) {
  const bool mask = p.mvis != nullptr;
  if (p.D == 16 || p.D == 32 || p.D == 64) {
    if (mask)
      return p.bf16 ? launch_instance<64, true, true>(p, maps, num_sms)
                    : launch_instance<64, false, true>(p, maps, num_sms);
    return p.bf16 ? launch_instance<64, true, false>(p, maps, num_sms)
                  : launch_instance<64, false, false>(p, maps, num_sms);
  }
  if (p.D == 128) {
    if (mask)
      return p.bf16 ? launch_instance<128, true, true>(p, maps, num_sms)
                    : launch_instance<128, false, true>(p, maps, num_sms);
    return p.bf16 ? launch_instance<128, true, false>(p, maps, num_sms)
                  : launch_instance<128, false, false>(p, maps, num_sms);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
