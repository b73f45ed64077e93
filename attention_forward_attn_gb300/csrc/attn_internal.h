// Internal interface between the host API (attn_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"

namespace attn {

// Device status word bits (see attn_status in include/attn.h).
enum : int {
  kStatusTimeout = 1 << 0,
  kStatusValidLenClamped = 1 << 1,
  kStatusLayout = 1 << 2,  // a kernel's shared-memory layout did not fit what it was given
  kRoleProducer = 1 << 8,
  kRoleMma = 2 << 8,
  kRoleSoftmax = 4 << 8,
  kRoleEpilogue = 8 << 8,
};

// Element strides of one [B, H, L, D] operand (batch, head, sequence
// position); the D elements of a row are contiguous.
struct Strides {
  int64_t b, h, l;
};

// Strides of a contiguous [B, H, L, D] tensor.
inline Strides contiguous_strides(int H, int L, int D) {
  return {static_cast<int64_t>(H) * L * D, static_cast<int64_t>(L) * D, static_cast<int64_t>(D)};
}

// Problem description handed to a kernel launcher (already validated).
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;              // may be null
  const int32_t* valid_len;  // may be null
  int* status;             // device status word
  // bf16: per (b*Hkv + h, 128-key tile) flag from the V pre-pass (1 = exact
  // fp16 copy of the tile exists); null = no copy (every tile split)
  const int* vflags;
  // explicit mask (null: none): the caller's bytes, and the packed form made
  // by the mask pre-pass (attn_mask.cu)
  const uint8_t* mask;
  int64_t mask_sb, mask_sr;  // element strides of its batch (0: shared) and rows
  // (mB = 1 when the mask is shared by every batch, else B)
  const uint32_t* mbits;     // [mB, Lq, n_kt, 4] words: bit c of word w = key 128t + 32w + c
  const uint32_t* mvis;      // [mB, n_mb, ceil(n_kt/32)]: bit t%32 = tile t has a kept position
  const uint32_t* mpart;     // same layout: bit t%32 = tile t is partially kept
  const int* mlast;          // [mB, n_mb]: last key tile with a kept position, or -1
  int B, Hq, Hkv;
  int Lq, Lk;              // query rows, key/value rows per head
  int D;
  Strides sq, sk, sv, so;  // element strides of q, k, v and o
  float sm_scale;
  int causal;
  int bf16;                // 0 fp16, 1 bf16
  cudaStream_t stream;
};

// Static configuration of the tensor-core kernel for one head dimension.
struct TcConfig {
  int block_m;          // rows per query tile (= TMEM lanes)
  int q_tiles;          // query tiles per CTA
  int block_n;          // keys per K/V tile
  int stages;           // K/V ring stages
  int threads;
  int smem_bytes;
  int tmem_cols;
};

bool tc_config(int D, TcConfig* out);

// Tensor-core (tcgen05/TMA) forward.  maps: Q, K, V, the fp16 copy of V
// (bf16 inputs with p.vflags set; any valid map otherwise, it is not read)
// and O (boxes of 128 rows, the kernel's store map).
cudaError_t launch_tc(const Problem& p, const CUtensorMap* maps, int num_sms);

// bf16 V pre-pass (attn_vconv.cu): bytes of its workspace (the fp16 copy of
// V, then one int flag per (b*Hkv + h, 128-key tile)), and its launch.
int64_t vconv_workspace_bytes(const Problem& p);
cudaError_t launch_vconv(const Problem& p, void* v16, int* flags);

// Explicit-mask pre-pass (attn_mask.cu): bytes of its workspace for p, and
// its launch (clears mvis, mpart and mlast first).  The workspace holds
// mbits, mvis, mpart and mlast in that order; mask_arrays sets the four
// pointers of p into it.
int64_t mask_workspace_bytes(const Problem& p);
void mask_arrays(Problem& p, void* ws);
cudaError_t launch_mask_pack(const Problem& p);

// fp32 comparison kernels (attn_f32.cu): kernel 0 naive three-pass, 1 tiled
// per-element online softmax, 2 tiled block rowmax.
cudaError_t launch_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                       int B, int H, int L, int D, float sm_scale, int causal,
                       const int32_t* valid_len, int kernel, int* status, cudaStream_t stream);

// Backward (attn_bwd.cu): bytes of its workspace (delta, fp32 [B*Hq, L])
// and its launch (delta, dQ and dK/dV kernels on `stream`).
int64_t bwd_workspace_bytes(int B, int Hq, int L);
cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, void* dq, void* dk, void* dv, float* delta, int B, int Hq,
                       int Hkv, int L, int D, float sm_scale, int causal, const int32_t* valid_len,
                       bool bf16, cudaStream_t stream);

// Tensor-core backward (attn_bwd_tc.cu): bytes of its workspace (-LSE log2(e)
// and delta, fp32 [B*Hq, L rounded up to 128] each) and its launch (pre-pass,
// dK/dV and dQ kernels on `stream`).  maps: Q, K, V, dO as encode_map makes
// them with 128-row boxes.  so, sdo: element strides of O and dO (read by the
// pre-pass); sdq, sdk, sdv: of the outputs.  D 16, 32, 64 or 128.  With few
// key tiles per SM the dK/dV kernel splits each key tile over several CTAs
// (bwd_tc_splits) and the workspace also holds their fp32 partial sums.
int bwd_tc_splits(int B, int Hkv, int Lk, int num_sms);
int64_t bwd_tc_workspace_bytes(int B, int Hq, int Hkv, int Lq, int Lk, int D, int num_sms,
                               int mask_batches);
cudaError_t launch_bwd_tc(const CUtensorMap (&maps)[4], const void* o, const Strides& so,
                          const void* dO, const Strides& sdo, const float* lse, void* dq,
                          const Strides& sdq, void* dk, const Strides& sdk, void* dv,
                          const Strides& sdv, void* workspace, int B, int Hq, int Hkv, int Lq,
                          int Lk, int D, float sm_scale, int causal, const int32_t* valid_len,
                          const uint8_t* mask, int64_t mask_batch_stride, int64_t mask_row_stride,
                          bool bf16, int num_sms, int* status, cudaStream_t stream);

// SIMT cross-check forward.
cudaError_t launch_simt(const Problem& p);

// Host helpers shared by the entry points (attn_api.cu).
attn_status_t cuda_fail(cudaError_t e);  // records e for attn_last_cuda_error
attn_status_t validate(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                       const int32_t* valid_len, attn_dtype_t dtype);
attn_status_t tensor_map_encoder_ready();
// Tensor map over a [B, H, L, D] 16-bit operand with element strides st,
// viewed as 4-D (D innermost, then L, H, B); boxes of 64 columns x `rows`
// rows of one head, 128-byte swizzle.  Columns D..63 of a box (D < 64) and
// rows past L read as zeros and are not written by stores.
attn_status_t encode_map(CUtensorMap* map, const void* base, int B, int H, int L, int D,
                         const Strides& st, int rows, bool bf16);
// A problem over contiguous tensors with Lq = Lk = L.
Problem make_problem(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                     const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream,
                     int* status);

// The five tensor maps of the tensor-core kernel for p (Q, K, V, V again in
// place of the fp16 copy, O); launch_tc's caller replaces maps[3] when it
// makes the fp16 copy.
attn_status_t encode_problem_maps(const Problem& p, CUtensorMap (&maps)[5]);

// attn_noalloc.cu: OR the no-alloc path's status word on `dev` into *code
// and clear it (a no-op unless attn_fwd_noalloc ran on that device).
attn_status_t noalloc_take_status(int dev, int* code);

// attn_api.cu: the current device (probed, status word allocated, sm_103
// checked) with its SM count and status word, and its workspace pool
// (created on first use).
attn_status_t current_device(int* dev, int* num_sms, int** status);
attn_status_t device_pool(int dev, cudaMemPool_t* out);

// attn_host.cu: destroy the host path's per-device copy streams and events.
void host_path_shutdown();

}  // namespace attn
