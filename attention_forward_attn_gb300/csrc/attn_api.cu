// Host side of libattn.so: the C ABI declared in include/attn.h.
//
// Validates arguments (no device synchronisation), keeps one device status
// word per GPU, encodes the TMA tensor maps of Q, K and V, and launches the
// kernels on the caller's stream.  Calls that need a workspace (bf16: the
// fp16 copy of V and its tile flags; an explicit mask: its packed form; the
// backward: its row statistics) take it from the caller (the *_ws entry
// points) or, when none is given, from a per-device stream-ordered pool owned
// here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

using attn::Problem;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool probed = false;
  bool arch_ok = false;
  int num_sms = 0;
  int* status = nullptr;  // one int of device memory
  cudaMemPool_t pool = nullptr;  // bf16 workspaces (created on first bf16 call)
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
thread_local int g_last_cuda_error = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace attn {

attn_status_t cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_CUDA;
}

// Argument checks that need no device.
attn_status_t validate(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                       const int32_t* valid_len, attn_dtype_t dtype) {
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1) return ATTN_ERR_SHAPE;
  if (D != 16 && D != 32 && D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  if (Hq % Hkv != 0) return ATTN_ERR_HEADS;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  if (!(sm_scale >= 0.f) || isinf(sm_scale)) return ATTN_ERR_SCALE;
  // every flat row index (b*Hq + h)*L + i fits in int32, and so does the unit count
  if (static_cast<int64_t>(B) * Hq * L > INT32_MAX) return ATTN_ERR_SHAPE;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return ATTN_ERR_ALIGN;
  if ((lse != nullptr && !aligned(lse, 4)) || (valid_len != nullptr && !aligned(valid_len, 4)))
    return ATTN_ERR_ALIGN;
  // (alignment is checked last: attn_fwd_host, whose host buffers need none,
  // treats ATTN_ERR_ALIGN as success)
  return ATTN_OK;
}

// The driver's cuTensorMapEncodeTiled, looked up once (no allocation).
attn_status_t tensor_map_encoder_ready() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &qr);
    if (e != cudaSuccess) return cuda_fail(e);
    if (qr != cudaDriverEntryPointSuccess || fn == nullptr) return cuda_fail(cudaErrorNotSupported);
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return ATTN_OK;
}

}  // namespace attn

namespace {

using attn::cuda_fail;
using attn::validate;

// Per-device probe and status-word allocation (first call on a device only).
attn_status_t device_state(int* dev_out, DeviceState** st_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_ARCH;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.probed) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    st.arch_ok = (prop.major == 10 && prop.minor == 3);
    st.num_sms = prop.multiProcessorCount;
    st.probed = true;
  }
  if (!st.arch_ok) return ATTN_ERR_ARCH;
  if (st.status == nullptr) {
    int* s = nullptr;
    e = cudaMalloc(&s, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemset(s, 0, sizeof(int));
    if (e != cudaSuccess) {
      cudaFree(s);
      return cuda_fail(e);
    }
    st.status = s;
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qr);
    if (e != cudaSuccess) return cuda_fail(e);
    if (qr != cudaDriverEntryPointSuccess || fn == nullptr) return cuda_fail(cudaErrorNotSupported);
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *dev_out = dev;
  *st_out = &st;
  return ATTN_OK;
}

// The device's workspace pool: memory stays reserved between calls (release
// threshold: never), so after the first bf16 call of a given size the
// stream-ordered allocation is a pool lookup.
attn_status_t workspace_pool(int dev, DeviceState* st, cudaMemPool_t* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (st->pool == nullptr) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    cudaError_t e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return cuda_fail(e);
    uint64_t keep = UINT64_MAX;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return cuda_fail(e);
    }
    st->pool = pool;
  }
  *out = st->pool;
  return ATTN_OK;
}

}  // namespace

namespace attn {

attn_status_t current_device(int* dev, int* num_sms, int** status) {
  DeviceState* st = nullptr;
  attn_status_t s = device_state(dev, &st);
  if (s != ATTN_OK) return s;
  *num_sms = st->num_sms;
  *status = st->status;
  return ATTN_OK;
}

attn_status_t device_pool(int dev, cudaMemPool_t* out) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_ARCH;
  return workspace_pool(dev, &g_dev[dev], out);
}

// Tensor map over a [B, H, L, D] 16-bit operand with element strides st,
// viewed as 4-D (D innermost, then L, H, B), boxes of 64 columns x `rows`
// rows x 1 head x 1 batch, 128-byte swizzle.  Strides are validated by the
// entry points (positive multiples of 8 elements where the extent is > 1);
// the stride of an extent-1 dimension is never used and is replaced by a
// valid one.
attn_status_t encode_map(CUtensorMap* map, const void* base, int B, int H, int L, int D,
                         const Strides& st, int rows, bool bf16) {
  const Strides c = contiguous_strides(H, L, D);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(L > 1 ? st.l : c.l) * 2,
                           static_cast<cuuint64_t>(H > 1 ? st.h : c.h) * 2,
                           static_cast<cuuint64_t>(B > 1 ? st.b : c.b) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(rows), 1, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        4, const_cast<void*>(base), dims, strides, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return ATTN_OK;
}

attn_status_t encode_problem_maps(const Problem& p, CUtensorMap (&maps)[5]) {
  TcConfig cfg;
  if (!tc_config(p.D, &cfg)) return ATTN_ERR_HEADDIM;
  const bool bf16 = p.bf16 != 0;
  attn_status_t s;
  if ((s = encode_map(&maps[0], p.q, p.B, p.Hq, p.Lq, p.D, p.sq, cfg.block_m, bf16)) != ATTN_OK)
    return s;
  if ((s = encode_map(&maps[1], p.k, p.B, p.Hkv, p.Lk, p.D, p.sk, cfg.block_n, bf16)) != ATTN_OK)
    return s;
  if ((s = encode_map(&maps[2], p.v, p.B, p.Hkv, p.Lk, p.D, p.sv, cfg.block_n, bf16)) != ATTN_OK)
    return s;
  maps[3] = maps[2];
  return encode_map(&maps[4], p.o, p.B, p.Hq, p.Lq, p.D, p.so, cfg.block_m, bf16);
}

Problem make_problem(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                     const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream,
                     int* status) {
  Problem p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.valid_len = valid_len;
  p.status = status;
  p.vflags = nullptr;
  p.mask = nullptr;
  p.mask_sb = p.mask_sr = 0;
  p.mbits = nullptr;
  p.mvis = nullptr;
  p.mpart = nullptr;
  p.mlast = nullptr;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = L;
  p.Lk = L;
  p.D = D;
  p.sq = p.so = contiguous_strides(Hq, L, D);
  p.sk = p.sv = contiguous_strides(Hkv, L, D);
  p.sm_scale = sm_scale;
  p.causal = causal;
  p.bf16 = dtype == ATTN_BF16 ? 1 : 0;
  p.stream = reinterpret_cast<cudaStream_t>(stream);
  return p;
}

}  // namespace attn

using attn::encode_map;
using attn::make_problem;

namespace {

// A workspace the caller supplies (the *_ws entry points).
struct CallerWorkspace {
  void* ptr;
  size_t bytes;
};

// Caller workspaces start on a 256-byte boundary (every part inside is
// placed at a multiple of 256 bytes from it).
constexpr uintptr_t kWorkspaceAlign = 256;

// Check a caller workspace against the bytes a call needs.
attn_status_t check_workspace(const CallerWorkspace* cws, int64_t need) {
  if (cws == nullptr || need == 0) return ATTN_OK;
  if (cws->ptr == nullptr || !aligned(cws->ptr, kWorkspaceAlign) ||
      cws->bytes < static_cast<size_t>(need))
    return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

// Bytes of the forward's workspace: for bf16 the contiguous fp16 copy of V
// and its per-tile flags (rounded up to 256 bytes), then for an explicit mask
// its packed form.
int64_t fwd_workspace_bytes(const Problem& p, int64_t* v_part) {
  const int64_t v_ws = p.bf16 ? (attn::vconv_workspace_bytes(p) + 255) / 256 * 256 : 0;
  const int64_t m_ws = p.mask != nullptr ? attn::mask_workspace_bytes(p) : 0;
  if (v_part != nullptr) *v_part = v_ws;
  return v_ws + m_ws;
}

// The tensor-core path for a validated problem on the current device: the
// workspace (the caller's, or a stream-ordered one from the pool), for bf16
// the V pre-pass, the mask pre-pass, then the attention kernel, then a pool
// workspace is returned to the pool.
attn_status_t run_tc(Problem& p, int dev, DeviceState* st, const CallerWorkspace* cws) {
  attn::TcConfig cfg;
  if (!attn::tc_config(p.D, &cfg)) return ATTN_ERR_HEADDIM;
  int64_t v_ws = 0;
  const int64_t need = fwd_workspace_bytes(p, &v_ws);
  attn_status_t s = check_workspace(cws, need);
  if (s != ATTN_OK) return s;
  CUtensorMap maps[5];
  s = attn::encode_problem_maps(p, maps);
  if (s != ATTN_OK) return s;
  void* ws = nullptr;
  const bool pooled = cws == nullptr && need > 0;
  if (need > 0) {
    cudaError_t e = cudaSuccess;
    if (pooled) {
      cudaMemPool_t pool = nullptr;
      if ((s = workspace_pool(dev, st, &pool)) != ATTN_OK) return s;
      e = cudaMallocFromPoolAsync(&ws, static_cast<size_t>(need), pool, p.stream);
      if (e != cudaSuccess) return cuda_fail(e);
    } else {
      ws = cws->ptr;
    }
    if (p.mask != nullptr) {
      attn::mask_arrays(p, static_cast<uint8_t*>(ws) + v_ws);
      e = attn::launch_mask_pack(p);
      if (e != cudaSuccess) s = cuda_fail(e);
    }
    if (s == ATTN_OK && p.bf16) {
      const size_t v_bytes = static_cast<size_t>(p.B) * p.Hkv * p.Lk * p.D * 2;
      int* flags = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + v_bytes);
      s = encode_map(&maps[3], ws, p.B, p.Hkv, p.Lk, p.D,
                     attn::contiguous_strides(p.Hkv, p.Lk, p.D), cfg.block_n, false);
      if (s == ATTN_OK) {
        e = attn::launch_vconv(p, ws, flags);
        if (e != cudaSuccess) s = cuda_fail(e);
      }
      p.vflags = flags;
    }
    if (s != ATTN_OK) {
      if (pooled) cudaFreeAsync(ws, p.stream);
      return s;
    }
  }
  cudaError_t e = attn::launch_tc(p, maps, st->num_sms);
  if (pooled) {
    const cudaError_t ef = cudaFreeAsync(ws, p.stream);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

// Strides of one operand: NULL means contiguous.  Every stride of a
// dimension with extent > 1 must be a positive multiple of 8 elements (16
// bytes: TMA strides and 16-byte row loads) below 2^39 elements (the tensor
// map's 2^40-byte limit); an extent-1 dimension's stride is not used.
attn_status_t strides_of(const attn_strides_t* in, int B, int H, int L, int D,
                         attn::Strides* out) {
  if (in == nullptr) {
    *out = attn::contiguous_strides(H, L, D);
    return ATTN_OK;
  }
  const int64_t v[3] = {in->batch, in->head, in->seq};
  const bool used[3] = {B > 1, H > 1, L > 1};
  for (int i = 0; i < 3; ++i) {
    if (!used[i]) continue;
    if (v[i] < 1 || v[i] % 8 != 0 || v[i] >= (int64_t(1) << 39)) return ATTN_ERR_STRIDE;
  }
  *out = attn::Strides{in->batch, in->head, in->seq};
  return ATTN_OK;
}

// O is written: no two of its elements may share an address.  With the
// dimensions of extent > 1 ordered by stride, each stride must step over the
// whole extent of the next smaller one (the row of D elements innermost).
bool no_self_overlap(const attn::Strides& s, int B, int H, int L, int D) {
  int64_t st[3] = {s.l, s.h, s.b};
  int64_t ext[3] = {L, H, B};
  // sort the three dimensions by stride (insertion sort)
  for (int i = 1; i < 3; ++i)
    for (int j = i; j > 0 && st[j] < st[j - 1]; --j) {
      const int64_t a = st[j], e = ext[j];
      st[j] = st[j - 1];
      ext[j] = ext[j - 1];
      st[j - 1] = a;
      ext[j - 1] = e;
    }
  int64_t span = D;  // elements covered by the dimensions below
  for (int i = 0; i < 3; ++i) {
    if (ext[i] == 1) continue;
    if (st[i] < span) return false;
    span = st[i] * ext[i];
  }
  return true;
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

attn_status_t fwd_contiguous(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                             const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream,
                             const CallerWorkspace* cws) {
  attn_status_t s = validate(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len, dtype);
  if (s != ATTN_OK) return s;
  Problem p = make_problem(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len, dtype,
                           stream, nullptr);
  // a caller workspace is checked before anything touches the device
  if ((s = check_workspace(cws, fwd_workspace_bytes(p, nullptr))) != ATTN_OK) return s;
  int dev = 0;
  DeviceState* st = nullptr;
  s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  p.status = st->status;
  return run_tc(p, dev, st, cws);
}

attn_status_t fwd_masked(const void* q, const attn_strides_t* q_strides, const void* k,
                         const attn_strides_t* k_strides, const void* v,
                         const attn_strides_t* v_strides, void* o, const attn_strides_t* o_strides,
                         float* lse, int B, int Hq, int Hkv, int Lq, int Lk, int D, float sm_scale,
                         int causal, const int32_t* valid_len, const uint8_t* mask,
                         int64_t mask_batch_stride, int64_t mask_row_stride, attn_dtype_t dtype,
                         attn_stream_t stream, const CallerWorkspace* cws) {
  // attn_fwd's checks with L = Lq, then the key length
  attn_status_t s =
      validate(q, k, v, o, lse, B, Hq, Hkv, Lq, D, sm_scale, causal, valid_len, dtype);
  if (s != ATTN_OK) return s;
  if (Lk < 1 || static_cast<int64_t>(B) * Hkv * Lk > INT32_MAX) return ATTN_ERR_SHAPE;
  attn::Strides sq, sk, sv, so;
  if ((s = strides_of(q_strides, B, Hq, Lq, D, &sq)) != ATTN_OK) return s;
  if ((s = strides_of(k_strides, B, Hkv, Lk, D, &sk)) != ATTN_OK) return s;
  if ((s = strides_of(v_strides, B, Hkv, Lk, D, &sv)) != ATTN_OK) return s;
  if ((s = strides_of(o_strides, B, Hq, Lq, D, &so)) != ATTN_OK) return s;
  if (!no_self_overlap(so, B, Hq, Lq, D)) return ATTN_ERR_STRIDE;
  if (mask != nullptr && (mask_batch_stride < 0 || mask_row_stride < 0)) return ATTN_ERR_STRIDE;
  // the mask pre-pass runs one CTA per (b, 128-row block, 128-key tile)
  if (mask != nullptr &&
      static_cast<int64_t>(B) * ((Lq + 127) / 128) * ((Lk + 127) / 128) > INT32_MAX)
    return ATTN_ERR_SHAPE;
  Problem p = make_problem(q, k, v, o, lse, B, Hq, Hkv, Lq, D, sm_scale, causal, valid_len, dtype,
                           stream, nullptr);
  p.Lk = Lk;
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.so = so;
  p.mask = mask;
  p.mask_sb = mask_batch_stride;
  p.mask_sr = mask_row_stride;
  if ((s = check_workspace(cws, fwd_workspace_bytes(p, nullptr))) != ATTN_OK) return s;
  int dev = 0;
  DeviceState* st = nullptr;
  s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  p.status = st->status;
  return run_tc(p, dev, st, cws);
}

}  // namespace

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                       const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream) {
  return fwd_contiguous(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len, dtype,
                        stream, nullptr);
}

attn_status_t attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                          const int32_t* valid_len, attn_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, attn_stream_t stream) {
  const CallerWorkspace cws{workspace, workspace_bytes};
  return fwd_contiguous(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len, dtype,
                        stream, &cws);
}

attn_status_t attn_fwd_masked(const void* q, const attn_strides_t* q_strides, const void* k,
                              const attn_strides_t* k_strides, const void* v,
                              const attn_strides_t* v_strides, void* o,
                              const attn_strides_t* o_strides, float* lse, int B, int Hq, int Hkv,
                              int Lq, int Lk, int D, float sm_scale, int causal,
                              const int32_t* valid_len, const uint8_t* mask,
                              int64_t mask_batch_stride, int64_t mask_row_stride,
                              attn_dtype_t dtype, attn_stream_t stream) {
  return fwd_masked(q, q_strides, k, k_strides, v, v_strides, o, o_strides, lse, B, Hq, Hkv, Lq,
                    Lk, D, sm_scale, causal, valid_len, mask, mask_batch_stride, mask_row_stride,
                    dtype, stream, nullptr);
}

attn_status_t attn_fwd_masked_ws(const void* q, const attn_strides_t* q_strides, const void* k,
                                 const attn_strides_t* k_strides, const void* v,
                                 const attn_strides_t* v_strides, void* o,
                                 const attn_strides_t* o_strides, float* lse, int B, int Hq,
                                 int Hkv, int Lq, int Lk, int D, float sm_scale, int causal,
                                 const int32_t* valid_len, const uint8_t* mask,
                                 int64_t mask_batch_stride, int64_t mask_row_stride,
                                 attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                 attn_stream_t stream) {
  const CallerWorkspace cws{workspace, workspace_bytes};
  return fwd_masked(q, q_strides, k, k_strides, v, v_strides, o, o_strides, lse, B, Hq, Hkv, Lq,
                    Lk, D, sm_scale, causal, valid_len, mask, mask_batch_stride, mask_row_stride,
                    dtype, stream, &cws);
}

attn_status_t attn_fwd_workspace_size(int B, int Hq, int Hkv, int Lq, int Lk, int D,
                                      attn_dtype_t dtype, int mask_batches, size_t* bytes) {
  if (bytes == nullptr) return ATTN_ERR_ARG;
  *bytes = 0;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1) return ATTN_ERR_SHAPE;
  if (D != 16 && D != 32 && D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  if (Hq % Hkv != 0) return ATTN_ERR_HEADS;
  if (mask_batches != 0 && mask_batches != 1 && mask_batches != B) return ATTN_ERR_ARG;
  Problem p = make_problem(nullptr, nullptr, nullptr, nullptr, nullptr, B, Hq, Hkv, Lq, D, 1.f, 0,
                           nullptr, dtype, nullptr, nullptr);
  p.Lk = Lk;
  if (mask_batches != 0) {
    p.mask = reinterpret_cast<const uint8_t*>(kWorkspaceAlign);  // only "a mask is given"
    p.mask_sb = mask_batches == 1 ? 0 : 1;  // 0: one mask shared by every batch
  }
  *bytes = static_cast<size_t>(fwd_workspace_bytes(p, nullptr));
  return ATTN_OK;
}

attn_status_t attn_fwd_strided(const void* q, const attn_strides_t* q_strides, const void* k,
                               const attn_strides_t* k_strides, const void* v,
                               const attn_strides_t* v_strides, void* o,
                               const attn_strides_t* o_strides, float* lse, int B, int Hq,
                               int Hkv, int Lq, int Lk, int D, float sm_scale, int causal,
                               const int32_t* valid_len, attn_dtype_t dtype,
                               attn_stream_t stream) {
  return attn_fwd_masked(q, q_strides, k, k_strides, v, v_strides, o, o_strides, lse, B, Hq, Hkv,
                         Lq, Lk, D, sm_scale, causal, valid_len, nullptr, 0, 0, dtype, stream);
}

attn_status_t attn_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                            const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream) {
  attn_status_t s = validate(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len, dtype);
  if (s != ATTN_OK) return s;
  if (static_cast<int64_t>(B) * Hq > 65535) return ATTN_ERR_SHAPE;
  int dev = 0;
  DeviceState* st = nullptr;
  s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  Problem p = make_problem(q, k, v, o, lse, B, Hq, Hkv, L, D, sm_scale, causal, valid_len, dtype,
                           stream, st->status);
  cudaError_t e = attn::launch_simt(p);
  if (e != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

attn_status_t attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                           int B, int H, int L, int D, float sm_scale, int causal,
                           const int32_t* valid_len, attn_f32_kernel_t kernel,
                           attn_stream_t stream) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_NULL;
  if (B < 1 || H < 1 || L < 1) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  if (kernel != ATTN_F32_NAIVE && kernel != ATTN_F32_TILED_ELEMENT &&
      kernel != ATTN_F32_TILED_ROWMAX)
    return ATTN_ERR_ARG;
  if (!(sm_scale >= 0.f) || isinf(sm_scale)) return ATTN_ERR_SCALE;
  // grid rows are (b, h) pairs; the naive kernel keeps a query's L scores in shared memory
  if (static_cast<int64_t>(B) * H > 65535 || static_cast<int64_t>(B) * H * L > INT32_MAX)
    return ATTN_ERR_SHAPE;
  if (kernel == ATTN_F32_NAIVE && L > 50000) return ATTN_ERR_SHAPE;
  if (!aligned(q, 4) || !aligned(k, 4) || !aligned(v, 4) || !aligned(o, 4) ||
      (lse != nullptr && !aligned(lse, 4)) || (valid_len != nullptr && !aligned(valid_len, 4)))
    return ATTN_ERR_ALIGN;
  int dev = 0;
  DeviceState* st = nullptr;
  attn_status_t s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  cudaError_t e = attn::launch_f32(q, k, v, o, lse, B, H, L, D, sm_scale, causal, valid_len,
                                   static_cast<int>(kernel), st->status,
                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

namespace {

// Arguments shared by the two backward entry points.
attn_status_t bwd_validate(const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                           int Hq, int Hkv, int Lq, int Lk, int D, float sm_scale, int causal,
                           const int32_t* valid_len, attn_dtype_t dtype, bool small_d) {
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr || dO == nullptr ||
      lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
    return ATTN_ERR_NULL;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1) return ATTN_ERR_SHAPE;
  if (D != 64 && D != 128 && !(small_d && (D == 16 || D == 32))) return ATTN_ERR_HEADDIM;
  if (Hq % Hkv != 0) return ATTN_ERR_HEADS;
  if (causal != 0 && causal != 1) return ATTN_ERR_ARG;
  if (!(sm_scale >= 0.f) || isinf(sm_scale)) return ATTN_ERR_SCALE;
  if (static_cast<int64_t>(B) * Hq * Lq > INT32_MAX || static_cast<int64_t>(B) * Hkv * Lk > INT32_MAX ||
      static_cast<int64_t>(B) * Hq > 65535)
    return ATTN_ERR_SHAPE;
  const void* p16[] = {q, k, v, o, dO, dq, dk, dv};  // TMA bases, 16-byte vector loads and stores
  for (const void* ptr : p16)
    if (!aligned(ptr, 16)) return ATTN_ERR_ALIGN;
  if (!aligned(lse, 4) || (valid_len != nullptr && !aligned(valid_len, 4))) return ATTN_ERR_ALIGN;
  return ATTN_OK;
}

}  // namespace

namespace {

attn_status_t bwd_masked(const void* q, const attn_strides_t* q_strides, const void* k,
                         const attn_strides_t* k_strides, const void* v,
                         const attn_strides_t* v_strides, const void* o,
                         const attn_strides_t* o_strides, const void* dO,
                         const attn_strides_t* do_strides, const float* lse, void* dq,
                         const attn_strides_t* dq_strides, void* dk,
                         const attn_strides_t* dk_strides, void* dv,
                         const attn_strides_t* dv_strides, int B, int Hq, int Hkv, int Lq, int Lk,
                         int D, float sm_scale, int causal, const int32_t* valid_len,
                         const uint8_t* mask, int64_t mask_batch_stride, int64_t mask_row_stride,
                         attn_dtype_t dtype, attn_stream_t stream, const CallerWorkspace* cws) {
  attn_status_t s = bwd_validate(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, sm_scale,
                                 causal, valid_len, dtype, true);
  if (s != ATTN_OK) return s;
  if (mask != nullptr && (mask_batch_stride < 0 || mask_row_stride < 0)) return ATTN_ERR_STRIDE;
  attn::Strides sq, sk, sv, so, sdo, sdq, sdk, sdv;
  if ((s = strides_of(q_strides, B, Hq, Lq, D, &sq)) != ATTN_OK ||
      (s = strides_of(k_strides, B, Hkv, Lk, D, &sk)) != ATTN_OK ||
      (s = strides_of(v_strides, B, Hkv, Lk, D, &sv)) != ATTN_OK ||
      (s = strides_of(o_strides, B, Hq, Lq, D, &so)) != ATTN_OK ||
      (s = strides_of(do_strides, B, Hq, Lq, D, &sdo)) != ATTN_OK ||
      (s = strides_of(dq_strides, B, Hq, Lq, D, &sdq)) != ATTN_OK ||
      (s = strides_of(dk_strides, B, Hkv, Lk, D, &sdk)) != ATTN_OK ||
      (s = strides_of(dv_strides, B, Hkv, Lk, D, &sdv)) != ATTN_OK)
    return s;
  if (!no_self_overlap(sdq, B, Hq, Lq, D) || !no_self_overlap(sdk, B, Hkv, Lk, D) ||
      !no_self_overlap(sdv, B, Hkv, Lk, D))
    return ATTN_ERR_STRIDE;
  // a caller workspace: pointer and alignment checked before the device is
  // touched (the backward always needs one); its size needs the SM count
  if (cws != nullptr && (cws->ptr == nullptr || !aligned(cws->ptr, kWorkspaceAlign)))
    return ATTN_ERR_WORKSPACE;
  int dev = 0;
  DeviceState* st = nullptr;
  if ((s = device_state(&dev, &st)) != ATTN_OK) return s;
  const bool bf16 = dtype == ATTN_BF16;
  CUtensorMap maps[4];
  if ((s = encode_map(&maps[0], q, B, Hq, Lq, D, sq, 128, bf16)) != ATTN_OK ||
      (s = encode_map(&maps[1], k, B, Hkv, Lk, D, sk, 128, bf16)) != ATTN_OK ||
      (s = encode_map(&maps[2], v, B, Hkv, Lk, D, sv, 128, bf16)) != ATTN_OK ||
      (s = encode_map(&maps[3], dO, B, Hq, Lq, D, sdo, 128, bf16)) != ATTN_OK)
    return s;
  const int64_t need = attn::bwd_tc_workspace_bytes(
      B, Hq, Hkv, Lq, Lk, D, st->num_sms, mask == nullptr ? 0 : (mask_batch_stride == 0 ? 1 : B));
  if ((s = check_workspace(cws, need)) != ATTN_OK) return s;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  cudaError_t e = cudaSuccess;
  if (cws != nullptr) {
    ws = cws->ptr;
  } else {
    cudaMemPool_t pool = nullptr;
    if ((s = workspace_pool(dev, st, &pool)) != ATTN_OK) return s;
    e = cudaMallocFromPoolAsync(&ws, static_cast<size_t>(need), pool, cs);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  e = attn::launch_bwd_tc(maps, o, so, dO, sdo, lse, dq, sdq, dk, sdk, dv, sdv, ws, B, Hq, Hkv, Lq,
                          Lk, D, sm_scale, causal, valid_len, mask, mask_batch_stride,
                          mask_row_stride, bf16, st->num_sms, st->status, cs);
  if (cws == nullptr) {
    const cudaError_t ef = cudaFreeAsync(ws, cs);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

}  // namespace

attn_status_t attn_bwd_masked(const void* q, const attn_strides_t* q_strides, const void* k,
                              const attn_strides_t* k_strides, const void* v,
                              const attn_strides_t* v_strides, const void* o,
                              const attn_strides_t* o_strides, const void* dO,
                              const attn_strides_t* do_strides, const float* lse, void* dq,
                              const attn_strides_t* dq_strides, void* dk,
                              const attn_strides_t* dk_strides, void* dv,
                              const attn_strides_t* dv_strides, int B, int Hq, int Hkv, int Lq,
                              int Lk, int D, float sm_scale, int causal, const int32_t* valid_len,
                              const uint8_t* mask, int64_t mask_batch_stride,
                              int64_t mask_row_stride, attn_dtype_t dtype, attn_stream_t stream) {
  return bwd_masked(q, q_strides, k, k_strides, v, v_strides, o, o_strides, dO, do_strides, lse,
                    dq, dq_strides, dk, dk_strides, dv, dv_strides, B, Hq, Hkv, Lq, Lk, D,
                    sm_scale, causal, valid_len, mask, mask_batch_stride, mask_row_stride, dtype,
                    stream, nullptr);
}

attn_status_t attn_bwd_masked_ws(const void* q, const attn_strides_t* q_strides, const void* k,
                                 const attn_strides_t* k_strides, const void* v,
                                 const attn_strides_t* v_strides, const void* o,
                                 const attn_strides_t* o_strides, const void* dO,
                                 const attn_strides_t* do_strides, const float* lse, void* dq,
                                 const attn_strides_t* dq_strides, void* dk,
                                 const attn_strides_t* dk_strides, void* dv,
                                 const attn_strides_t* dv_strides, int B, int Hq, int Hkv, int Lq,
                                 int Lk, int D, float sm_scale, int causal,
                                 const int32_t* valid_len, const uint8_t* mask,
                                 int64_t mask_batch_stride, int64_t mask_row_stride,
                                 attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                 attn_stream_t stream) {
  const CallerWorkspace cws{workspace, workspace_bytes};
  return bwd_masked(q, q_strides, k, k_strides, v, v_strides, o, o_strides, dO, do_strides, lse,
                    dq, dq_strides, dk, dk_strides, dv, dv_strides, B, Hq, Hkv, Lq, Lk, D,
                    sm_scale, causal, valid_len, mask, mask_batch_stride, mask_row_stride, dtype,
                    stream, &cws);
}

attn_status_t attn_bwd_ws(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                          int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                          const int32_t* valid_len, attn_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, attn_stream_t stream) {
  return attn_bwd_masked_ws(q, nullptr, k, nullptr, v, nullptr, o, nullptr, dO, nullptr, lse, dq,
                            nullptr, dk, nullptr, dv, nullptr, B, Hq, Hkv, L, L, D, sm_scale,
                            causal, valid_len, nullptr, 0, 0, dtype, workspace, workspace_bytes,
                            stream);
}

attn_status_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Lq, int Lk, int D,
                                      int mask_batches, size_t* bytes) {
  if (bytes == nullptr) return ATTN_ERR_ARG;
  *bytes = 0;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1) return ATTN_ERR_SHAPE;
  if (D != 16 && D != 32 && D != 64 && D != 128) return ATTN_ERR_HEADDIM;
  if (Hq % Hkv != 0) return ATTN_ERR_HEADS;
  if (mask_batches != 0 && mask_batches != 1 && mask_batches != B) return ATTN_ERR_ARG;
  int dev = 0;
  DeviceState* st = nullptr;
  attn_status_t s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  *bytes = static_cast<size_t>(
      attn::bwd_tc_workspace_bytes(B, Hq, Hkv, Lq, Lk, D, st->num_sms, mask_batches));
  return ATTN_OK;
}

attn_status_t attn_workspace_pool_stats(int reset_high_water, size_t* reserved_bytes,
                                        size_t* high_water_bytes) {
  if (reserved_bytes != nullptr) *reserved_bytes = 0;
  if (high_water_bytes != nullptr) *high_water_bytes = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_ARCH;
  cudaMemPool_t pool = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    pool = g_dev[dev].pool;
  }
  if (pool == nullptr) return ATTN_OK;
  uint64_t reserved = 0, high = 0;
  if ((e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrReservedMemCurrent, &reserved)) !=
          cudaSuccess ||
      (e = cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &high)) != cudaSuccess)
    return cuda_fail(e);
  if (reserved_bytes != nullptr) *reserved_bytes = static_cast<size_t>(reserved);
  if (high_water_bytes != nullptr) *high_water_bytes = static_cast<size_t>(high);
  if (reset_high_water) {
    uint64_t zero = 0;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return ATTN_OK;
}

attn_status_t attn_bwd_strided(const void* q, const attn_strides_t* q_strides, const void* k,
                               const attn_strides_t* k_strides, const void* v,
                               const attn_strides_t* v_strides, const void* o,
                               const attn_strides_t* o_strides, const void* dO,
                               const attn_strides_t* do_strides, const float* lse, void* dq,
                               const attn_strides_t* dq_strides, void* dk,
                               const attn_strides_t* dk_strides, void* dv,
                               const attn_strides_t* dv_strides, int B, int Hq, int Hkv, int Lq,
                               int Lk, int D, float sm_scale, int causal,
                               const int32_t* valid_len, attn_dtype_t dtype,
                               attn_stream_t stream) {
  return attn_bwd_masked(q, q_strides, k, k_strides, v, v_strides, o, o_strides, dO, do_strides,
                         lse, dq, dq_strides, dk, dk_strides, dv, dv_strides, B, Hq, Hkv, Lq, Lk, D,
                         sm_scale, causal, valid_len, nullptr, 0, 0, dtype, stream);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                       int L, int D, float sm_scale, int causal, const int32_t* valid_len,
                       attn_dtype_t dtype, attn_stream_t stream) {
  return attn_bwd_strided(q, nullptr, k, nullptr, v, nullptr, o, nullptr, dO, nullptr, lse, dq,
                          nullptr, dk, nullptr, dv, nullptr, B, Hq, Hkv, L, L, D, sm_scale, causal,
                          valid_len, dtype, stream);
}

attn_status_t attn_bwd_simt(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                            int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                            const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream) {
  attn_status_t s = bwd_validate(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, L, L, D, sm_scale,
                                 causal, valid_len, dtype, false);
  if (s != ATTN_OK) return s;
  int dev = 0;
  DeviceState* st = nullptr;
  if ((s = device_state(&dev, &st)) != ATTN_OK) return s;
  cudaMemPool_t pool = nullptr;
  if ((s = workspace_pool(dev, st, &pool)) != ATTN_OK) return s;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(&ws, static_cast<size_t>(attn::bwd_workspace_bytes(B, Hq, L)),
                                          pool, cs);
  if (e != cudaSuccess) return cuda_fail(e);
  e = attn::launch_bwd(q, k, v, o, dO, lse, dq, dk, dv, static_cast<float*>(ws), B, Hq, Hkv, L, D,
                       sm_scale, causal, valid_len, dtype == ATTN_BF16, cs);
  const cudaError_t ef = cudaFreeAsync(ws, cs);
  if (e == cudaSuccess) e = ef;
  if (e != cudaSuccess) return cuda_fail(e);
  return ATTN_OK;
}

attn_status_t attn_status(attn_stream_t stream, int* device_code) {
  if (device_code != nullptr) *device_code = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return ATTN_OK;
  int* word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    word = g_dev[dev].status;
  }
  int code = 0;
  if (word != nullptr) {
    e = cudaMemcpy(&code, word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (code != 0) {
      e = cudaMemset(word, 0, sizeof(int));
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }
  attn_status_t s = attn::noalloc_take_status(dev, &code);
  if (s != ATTN_OK) return s;
  if (device_code != nullptr) *device_code = code;
  if (code & attn::kStatusTimeout) return ATTN_ERR_TIMEOUT;
  if (code & attn::kStatusLayout) return ATTN_ERR_ARCH;
  if (code & attn::kStatusValidLenClamped) return ATTN_ERR_VALID_LEN;
  return ATTN_OK;
}

attn_status_t attn_query(int D, attn_dtype_t dtype, attn_caps_t* out) {
  if (out == nullptr) return ATTN_ERR_ARG;
  *out = attn_caps_t{};
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  attn::TcConfig cfg;
  if (!attn::tc_config(D, &cfg)) return ATTN_ERR_HEADDIM;
  out->block_m = cfg.block_m;
  out->q_tiles_per_cta = cfg.q_tiles;
  out->block_n = cfg.block_n;
  out->kv_stages = cfg.stages;
  out->threads = cfg.threads;
  out->smem_bytes = cfg.smem_bytes;
  out->tmem_cols = cfg.tmem_cols;
  out->lse_natural_log = 1;
  int n = 0;
  if (cudaGetDeviceCount(&n) == cudaSuccess && n > 0) {
    int dev = 0;
    cudaDeviceProp prop;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
      out->num_sms = prop.multiProcessorCount;
      out->supported = (prop.major == 10 && prop.minor == 3) ? 1 : 0;
    }
  } else {
    cudaGetLastError();  // clear the "no device" error
  }
  return ATTN_OK;
}

const char* attn_strerror(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "success";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_ALIGN: return "q/k/v/o must be 16-byte aligned, lse/valid_len 4-byte aligned";
    case ATTN_ERR_SHAPE: return "B, Hq, Hkv and L must be >= 1 and B*Hq*L must fit in int32";
    case ATTN_ERR_HEADS: return "Hq must be a multiple of Hkv";
    case ATTN_ERR_HEADDIM: return "unsupported head dimension (16, 32, 64 or 128)";
    case ATTN_ERR_DTYPE: return "dtype must be ATTN_F16 or ATTN_BF16";
    case ATTN_ERR_SCALE: return "sm_scale must be finite and >= 0";
    case ATTN_ERR_ARCH: return "no sm_103 (GB300) device is current";
    case ATTN_ERR_CUDA: return "a CUDA call failed (see attn_last_cuda_error)";
    case ATTN_ERR_TIMEOUT: return "a bounded wait inside the kernel timed out";
    case ATTN_ERR_VALID_LEN: return "a valid_len value was outside [0, L] and was clamped";
    case ATTN_ERR_ARG: return "invalid argument";
    case ATTN_ERR_SCRATCH:
      return "the call needs more scratch than attn_fwd_noalloc's static array holds";
    case ATTN_ERR_STRIDE:
      return "a stride is not a positive multiple of 8 elements below 2^39, or O's elements overlap";
    case ATTN_ERR_WORKSPACE:
      return "the workspace is NULL, not 256-byte aligned, or smaller than the call needs";
  }
  return "unknown status";
}

int attn_last_cuda_error(void) { return g_last_cuda_error; }

void attn_shutdown(void) {
  attn::host_path_shutdown();  // before g_mu: attn_fwd_host takes its own lock, then g_mu
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (int d = 0; d < kMaxDevices; ++d) {
    if (g_dev[d].status != nullptr) {
      if (cudaSetDevice(d) == cudaSuccess) cudaFree(g_dev[d].status);
      g_dev[d].status = nullptr;
    }
    if (g_dev[d].pool != nullptr) {
      // released once the workspaces still queued have been freed
      cudaMemPoolDestroy(g_dev[d].pool);
      g_dev[d].pool = nullptr;
    }
  }
  if (have_cur) cudaSetDevice(cur);
  cudaGetLastError();
}

}  // extern "C"
