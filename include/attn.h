/*
 * attn.h -- C ABI of libattn.so, a fused multi-head attention forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (one call = one forward over a whole batch):
 *
 *   O = softmax(Q K^T * sm_scale + Mask) V,   LSE = log sum exp(Q K^T * sm_scale + Mask)
 *
 * as defined in "masked multi head attention in CUDA" (wzjinhao.cn), section
 * 2.1, over [B, H, L, D] tensors, evaluated tile by tile with the online
 * softmax of the Triton-CUDA Attention page ("Online Softmax core algorithm":
 * running row max m_i, exp-sum l_i, fp32 accumulator rescaled by
 * alpha = exp2(m_old - m_new), scores pre-multiplied by sm_scale * log2(e)),
 * so the [B, H, L, L] score matrix never reaches device memory.
 *
 * All entry points are plain C: no C++ exceptions cross this boundary, every
 * call returns an attn_status_t, and no argument is a framework type.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same object as cudaStream_t / CUstream); NULL is the
 * legacy default stream. */
typedef struct CUstream_st* attn_stream_t;

/* Element type of Q, K, V and O.  The accumulation is always fp32. */
typedef enum {
  ATTN_F16 = 0,  /* IEEE binary16 */
  ATTN_BF16 = 1  /* bfloat16 */
} attn_dtype_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = 1,       /* a required pointer is NULL */
  ATTN_ERR_ALIGN = 2,      /* q, k, v or o is not 16-byte aligned, or lse / valid_len not 4-byte aligned */
  ATTN_ERR_SHAPE = 3,      /* B, Hq, Hkv or L < 1, or a size overflows the supported range */
  ATTN_ERR_HEADS = 4,      /* Hq is not a multiple of Hkv */
  ATTN_ERR_HEADDIM = 5,    /* D is not supported by this entry point */
  ATTN_ERR_DTYPE = 6,      /* dtype is not ATTN_F16 / ATTN_BF16 */
  ATTN_ERR_SCALE = 7,      /* sm_scale is negative, NaN or infinite */
  ATTN_ERR_ARCH = 8,       /* the current device is not an sm_103 GPU, or no device */
  ATTN_ERR_CUDA = 9,       /* a CUDA runtime/driver call failed (see attn_last_cuda_error) */
  ATTN_ERR_TIMEOUT = 10,   /* device side: a bounded wait inside a kernel gave up */
  ATTN_ERR_VALID_LEN = 11, /* device side: a valid_len value was outside [0, L] and was clamped */
  ATTN_ERR_ARG = 12,       /* another invalid argument (causal not 0/1, NULL out-pointer, ...) */
  ATTN_ERR_SCRATCH = 13,   /* attn_fwd_noalloc: the call needs more scratch than its static array holds */
  ATTN_ERR_STRIDE = 14,    /* a stride is invalid, or an output's elements overlap (strided entry points) */
  ATTN_ERR_WORKSPACE = 15  /* *_ws entry points: the workspace is NULL, misaligned or too small */
} attn_status_t;

/*
 * attn_fwd -- the fused attention forward.
 *
 * Defined by: the attention formula of wzjinhao.cn section 2.1; the implicit
 * causal mask (Triton-CUDA Attention page, "Causal Attention": key j is
 * visible to query i iff j <= i, square and top-left aligned); the padding
 * mask by per-batch valid length (wzjinhao.cn section 2.2: key j is masked
 * when j >= valid_len[b]); the GQA/MQA head map h_kv = h_q / (Hq / Hkv) with
 * integer division (Triton-CUDA Attention page, "GQA" and "MQA"); and the
 * per-row log-sum-exp that tiny_flash_attn_triton.py stores for the backward
 * pass, here in natural-log units.
 *
 * Arguments (all pointers are DEVICE pointers, owned by the caller):
 *   q         [B, Hq, L, D] contiguous, dtype elements, 16-byte aligned.
 *   k, v      [B, Hkv, L, D] contiguous, 16-byte aligned.  Hkv = 1 is
 *             multi-query attention; its bytes equal a squeezed [B, L, D].
 *   o         [B, Hq, L, D] contiguous output, dtype, 16-byte aligned.
 *   lse       [B*Hq, L] row-major fp32 output, natural log:
 *             lse[(b*Hq + h)*L + i] = log(sum_{j visible} exp(sm_scale * q_i . k_j)).
 *             NULL skips the store.
 *   B, Hq, Hkv, L   batch, query heads, key/value heads, sequence length (>= 1).
 *   D         head dimension: 16, 32, 64 or 128 (the Triton-CUDA Attention
 *             page's set).  D = 16 and 32 run the D = 64 kernel: its loads
 *             fill columns D..63 with zeros (scores and O unchanged) and its
 *             stores write only the D columns, so they cost as much as D = 64.
 *   sm_scale  score scale, finite and >= 0 (normally 1/sqrt(D)).
 *   causal    0 or 1.
 *   valid_len NULL (no padding mask) or a device array of B int32 values.
 *             Values outside [0, L] are clamped on the device and reported
 *             by attn_status as ATTN_ERR_VALID_LEN.
 *   dtype     ATTN_F16 or ATTN_BF16 (q, k, v and o share it).
 *   stream    the stream the work is queued on.
 *
 * A query row with no visible key (valid_len[b] == 0) gets O = 0 and
 * LSE = -inf (wzjinhao.cn section 3.2: such a row outputs 0, never NaN).
 *
 * Errors: argument errors are detected on the host before anything is
 * queued and returned immediately (nothing is written).  The call never
 * synchronises; device-side conditions (ATTN_ERR_TIMEOUT, ATTN_ERR_VALID_LEN)
 * are recorded in a per-device status word and reported by attn_status.
 *
 * Device memory owned by the library: the status word (one int per device,
 * cudaMalloc on first use) and, for ATTN_BF16, a per-call workspace of
 * B*Hkv*L*D*2 bytes plus 4 bytes per (b, h_kv, 128-key tile).  The workspace
 * holds an fp16 copy of V (exact where every value of a 128-key tile is
 * finite with |v| < 65536; flagged tiles keep bf16) so that P.V runs with fp16
 * probabilities.  It is taken with cudaMallocFromPoolAsync from a pool the
 * library creates per device (release threshold: never) and returned with
 * cudaFreeAsync on the same stream after the kernel, so calls on different
 * streams never share it and repeated calls reuse the pool's memory.
 * attn_shutdown destroys the pools.  ATTN_F16 calls take no workspace.
 * attn_fwd_ws is the same call with the workspace supplied by the caller.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                       const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_fwd_workspace_size -- bytes of device workspace one forward call needs
 * (attn_fwd_ws, attn_fwd_masked_ws) for these sizes.
 *
 * The pages say nothing about memory management; the contract is that the
 * caller's framework allocates all per-call device memory (the library only
 * owns its status word).  The workspace holds, for ATTN_BF16, the fp16 copy
 * of V and one flag per (b, h_kv, 128-key tile) that attn_fwd describes, and,
 * for an explicit mask, the packed bit form attn_fwd_masked describes.
 *   B, Hq, Hkv, Lq, Lk, D, dtype   as the call will pass them (Lq = Lk = L
 *                  for attn_fwd_ws).
 *   mask_batches   0 without an explicit mask, 1 for one [Lq, Lk] mask
 *                  shared by every batch (mask batch stride 0), B for one
 *                  mask per batch.
 *   bytes          receives the size; 0 when the call needs no workspace
 *                  (ATTN_F16 without a mask).
 * Host-only, needs no device.  Errors: ATTN_ERR_ARG (bytes NULL, or
 * mask_batches not 0, 1 or B), and attn_fwd's shape, head and dtype errors.
 */
attn_status_t attn_fwd_workspace_size(int B, int Hq, int Hkv, int Lq, int Lk, int D,
                                      attn_dtype_t dtype, int mask_batches, size_t* bytes);

/*
 * attn_fwd_ws -- attn_fwd with a caller-supplied workspace: the library
 * allocates no per-call device memory.
 *
 * Defined by: the same operation, arguments and results as attn_fwd, bit for
 * bit.  workspace: a DEVICE buffer owned by the caller, 256-byte aligned, of
 * at least workspace_bytes >= attn_fwd_workspace_size(...) bytes (NULL with 0
 * bytes is accepted when the size is 0).  Its contents on entry do not matter;
 * the call overwrites it on `stream` and reads it until its kernels finish, so
 * the caller must not reuse or free it before then (stream order is enough;
 * two calls in flight at once on different streams need two workspaces).
 * Errors: as attn_fwd, plus ATTN_ERR_WORKSPACE when the workspace is NULL,
 * misaligned or too small for the call (checked on the host, nothing queued).
 */
attn_status_t attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                          const int32_t* valid_len, attn_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, attn_stream_t stream);

/* Element strides of one [B, H, L, D] operand of attn_fwd_strided: how many
 * elements apart (b, h, i, d) and (b + 1, h, i, d), (b, h + 1, i, d) and
 * (b, h, i + 1, d) are.  The D elements of a row are always contiguous. */
typedef struct {
  int64_t batch;
  int64_t head;
  int64_t seq;
} attn_strides_t;

/*
 * attn_fwd_strided -- attn_fwd on strided operands, with a query length Lq and
 * a key/value length Lk.
 *
 * Defined by: the same operation as attn_fwd.  tiny_flash_attn_triton.py's
 * flash_attn_triton and the Triton-CUDA Attention page's standard Flash
 * Attention pass every operand to the kernel with its own batch, head,
 * sequence and dim strides; "masked multi head attention in CUDA"
 * (wzjinhao.cn) section 2.1 notes that frameworks hold Q, K and V either as
 * [B, N, H, D] or as [B, H, N, D].  Here both, and any other layout whose rows
 * of D elements are contiguous (a slice of a packed QKV tensor, for example),
 * are read and written in place, without a copy.  The pages use one sequence
 * length; with Lq != Lk the masks keep their comparisons on absolute
 * positions: key j is visible to query i iff (!causal || j <= i) and
 * (valid_len == NULL || j < valid_len[b]) -- the causal mask stays top-left
 * aligned.
 *
 * Arguments (device pointers, owned by the caller):
 *   q, o      base of query and output element (0, 0, 0, 0); Q and O are
 *             [B, Hq, Lq, D] in the index space, placed by q_strides and
 *             o_strides.
 *   k, v      base of K and V, [B, Hkv, Lk, D] in the index space.
 *   *_strides NULL for a contiguous [B, H, L, D] tensor, else its element
 *             strides.  Every stride of a dimension whose extent is > 1 must
 *             be a positive multiple of 8 elements (16 bytes) below 2^39;
 *             the stride of an extent-1 dimension is ignored.  O's elements
 *             must not overlap one another (ATTN_ERR_STRIDE); Q, K and V may
 *             overlap one another and themselves.  O must not overlap Q, K or
 *             V (not checked: the result is then undefined).
 *   lse       [B*Hq, Lq] contiguous fp32 output, lse[(b*Hq + h)*Lq + i], or
 *             NULL.
 *   Lq, Lk    query rows and key/value rows per head (>= 1); B*Hq*Lq and
 *             B*Hkv*Lk must fit in int32.
 *   valid_len NULL or B int32 values; values outside [0, Lk] are clamped and
 *             reported by attn_status as ATTN_ERR_VALID_LEN.
 *   the rest  as attn_fwd.
 *
 * Work and memory: attn_fwd's kernel, reading and writing through 4-D tensor
 * maps built from the strides.  For ATTN_BF16 the fp16 copy of V in the
 * per-call workspace is contiguous, B*Hkv*Lk*D*2 bytes (plus the tile flags).
 * Errors: as attn_fwd, plus ATTN_ERR_STRIDE; nothing is queued on an
 * argument error.
 */
attn_status_t attn_fwd_strided(const void* q, const attn_strides_t* q_strides, const void* k,
                               const attn_strides_t* k_strides, const void* v,
                               const attn_strides_t* v_strides, void* o,
                               const attn_strides_t* o_strides, float* lse, int B, int Hq,
                               int Hkv, int Lq, int Lk, int D, float sm_scale, int causal,
                               const int32_t* valid_len, attn_dtype_t dtype,
                               attn_stream_t stream);

/*
 * attn_fwd_masked -- attn_fwd_strided with an explicit boolean mask.
 *
 * Defined by: "masked multi head attention in CUDA" (wzjinhao.cn) section
 * 2.2: a padding mask given as a [B, N, N] boolean matrix, and the combined
 * mask as a float matrix of 0 (kept) and -inf (removed) added to the scores --
 * both name, per (b, query, key), whether the position takes part.  Here the
 * mask is a byte matrix: key j is visible to query i of batch b iff
 * mask[b*mask_batch_stride + i*mask_row_stride + j] != 0 (for every head) AND
 * the causal and valid_len conditions of attn_fwd_strided hold.  A row with
 * no visible key gets O = 0 and LSE = -inf.
 *
 * Arguments: as attn_fwd_strided, plus
 *   mask               device pointer to uint8 values, any alignment; NULL
 *                      makes the call identical to attn_fwd_strided.
 *   mask_batch_stride  elements between batches (0: one [Lq, Lk] mask shared
 *                      by every batch), >= 0.
 *   mask_row_stride    elements between query rows, >= 0.
 * The mask is read once per call by a pre-pass that packs it into bits and
 * marks every (b, 128-row block, 128-key tile) as having no kept position
 * (the attention kernel skips the tile: no loads, no tensor-core work), all
 * positions kept (no masking work) or some (the bits are applied).
 *
 * Device memory: the per-call workspace of attn_fwd (bf16) plus
 * B*Lq*ceil(Lk/128)*16 bytes of bits and a byte per tile.
 * Errors: as attn_fwd_strided; negative mask strides give ATTN_ERR_STRIDE.
 */
attn_status_t attn_fwd_masked(const void* q, const attn_strides_t* q_strides, const void* k,
                              const attn_strides_t* k_strides, const void* v,
                              const attn_strides_t* v_strides, void* o,
                              const attn_strides_t* o_strides, float* lse, int B, int Hq, int Hkv,
                              int Lq, int Lk, int D, float sm_scale, int causal,
                              const int32_t* valid_len, const uint8_t* mask,
                              int64_t mask_batch_stride, int64_t mask_row_stride,
                              attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_fwd_masked_ws -- attn_fwd_masked (and, with mask NULL,
 * attn_fwd_strided) with a caller-supplied workspace, on the terms of
 * attn_fwd_ws: same arguments, results and errors as attn_fwd_masked, plus
 * workspace / workspace_bytes sized by attn_fwd_workspace_size with
 * mask_batches = 0 (no mask), 1 (mask_batch_stride 0) or B.
 */
attn_status_t attn_fwd_masked_ws(const void* q, const attn_strides_t* q_strides, const void* k,
                                 const attn_strides_t* k_strides, const void* v,
                                 const attn_strides_t* v_strides, void* o,
                                 const attn_strides_t* o_strides, float* lse, int B, int Hq,
                                 int Hkv, int Lq, int Lk, int D, float sm_scale, int causal,
                                 const int32_t* valid_len, const uint8_t* mask,
                                 int64_t mask_batch_stride, int64_t mask_row_stride,
                                 attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                                 attn_stream_t stream);

/*
 * attn_fwd_simt -- the same operation, same arguments and same contract as
 * attn_fwd, computed by a plain SIMT kernel (one warp per query row, fp32
 * FMA dot products, online softmax over 32-key blocks; no tensor cores).
 * It is a slow cross-check of attn_fwd, not the fast path.  D is 16, 32, 64
 * or 128.
 */
attn_status_t attn_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                            const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_bwd -- gradients of attn_fwd: dQ, dK, dV for an output gradient dO.
 *
 * Defined by: tiny_flash_attn_triton.py stores the per-row log-sum-exp "for
 * the backward pass"; the pages give no backward algorithm, so this is the
 * derivative of O = softmax(sm_scale Q K^T + Mask) V from its definition,
 * with the softmax rebuilt from that LSE: P_ij = exp(sm_scale q_i.k_j - LSE_i)
 * on the visible keys, delta_i = dO_i . O_i, dS_ij = P_ij (dO_i.v_j - delta_i),
 * dQ = sm_scale dS K, dK = sm_scale dS^T Q, dV = P^T dO; dK and dV of a
 * key/value head sum over the query heads that read it (GQA/MQA).
 *
 * Arguments (device pointers, caller-owned; same layouts, dtype and masks as
 * attn_fwd, 16-byte aligned):
 *   q, k, v    the forward's inputs;  o the forward's output;
 *   dO         [B, Hq, L, D] output gradient;
 *   lse        [B*Hq, L] fp32, the forward's natural-log LSE (required);
 *   dq         [B, Hq, L, D] out;  dk, dv  [B, Hkv, L, D] out (overwritten).
 *   D          16, 32, 64 or 128 (16 and 32 run the D = 64 kernels on
 *              zero-filled columns).  B*Hq <= 65535.
 * Work: a pre-pass (delta and the LSE in base 2, in rows padded to 128) and
 * one launch of two tensor-core CTA kinds (tcgen05, fp32 accumulators in
 * tensor memory): dK/dV per 128-key tile with K and V resident and every query
 * tile and query head of the group streaming through; dQ per 128-row query
 * tile with K and V streaming.  When the (key tile, b, h_kv) units are too few
 * for the GPU (few K/V heads, e.g. MQA), each key tile's work is split over
 * several CTAs whose fp32 partials a reduction adds in a fixed order.  P and
 * dS are rounded to the input dtype as MMA operands, every sum is accumulated
 * in fp32, each result rounded once to the input dtype.  No atomics: the
 * result does not depend on scheduling.  Device memory: a stream-ordered
 * workspace from the library's pool of 2*B*Hq*ceil(L/128)*128*4 bytes, plus
 * splits*2*B*Hkv*L*D*4 bytes of partials when split (at most 16 splits).
 * Errors: argument errors as attn_fwd (nothing is queued); device-side
 * conditions (bounded-wait timeout, clamped valid_len) through attn_status.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                       int L, int D, float sm_scale, int causal, const int32_t* valid_len,
                       attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_bwd_strided -- attn_bwd on strided operands with separate query and
 * key lengths: q, o, dO, dq are [B, Hq, Lq, D], k, v, dk, dv [B, Hkv, Lk, D],
 * lse [B*Hq, Lq]; the masks as in attn_fwd_strided (causal keeps key j <= query
 * i, valid_len clamped to [0, Lk]).  Each of q, k, v, o, dO, dq, dk and dv
 * takes an attn_strides_t (NULL: contiguous) with the rules of
 * attn_fwd_strided (positive multiples of 8 elements below 2^39; the stride of
 * an extent-1 dimension is ignored; rows of D elements contiguous).  dq, dk
 * and dv must not overlap themselves (ATTN_ERR_STRIDE).  Everything else as
 * attn_bwd, which is this call with Lq = Lk = L and every stride NULL.
 */
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
                               attn_stream_t stream);

/*
 * attn_bwd_masked -- attn_bwd_strided with the explicit boolean mask of
 * attn_fwd_masked (mask[b*mask_batch_stride + i*mask_row_stride + j] != 0
 * keeps key j for query i; mask_batch_stride 0: one [Lq, Lk] mask for every
 * batch; intersected with causal and valid_len).  A pre-pass packs the mask
 * into bits over keys (for the dQ kernel) and over queries (for the dK/dV
 * kernel); every masked (query, key) pair gets P = 0.  The workspace grows by
 * 2 bits per position (1 for each layout) per mask batch.  Same arguments,
 * preconditions and errors as attn_bwd_strided; negative mask strides give
 * ATTN_ERR_STRIDE.
 */
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
                              int64_t mask_row_stride, attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace one tensor-core
 * backward call needs (attn_bwd_ws, attn_bwd_masked_ws): the row statistics
 * of its pre-pass, the fp32 partial sums when key tiles are split over
 * several CTAs, and the packed mask.  mask_batches: 0 without an explicit
 * mask, 1 for a mask shared by every batch, B for one per batch.  The size
 * depends on the current device's SM count (the split), so the call looks at
 * the current device (sm_103 required; on the first call on a device the
 * library also allocates its status word there).  Errors: ATTN_ERR_ARG
 * (bytes NULL, mask_batches not 0, 1 or B), the shape, head and head-dim
 * errors of attn_bwd, ATTN_ERR_ARCH, ATTN_ERR_CUDA.
 */
attn_status_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Lq, int Lk, int D,
                                      int mask_batches, size_t* bytes);

/*
 * attn_bwd_ws / attn_bwd_masked_ws -- attn_bwd and attn_bwd_masked (mask
 * NULL: attn_bwd_strided) with a caller-supplied workspace instead of one
 * from the library's pool: the library allocates no per-call device memory.
 * Same arguments, results and errors as those calls, plus workspace (a
 * 256-byte aligned DEVICE buffer owned by the caller, contents on entry
 * irrelevant, in use until the call's kernels finish on `stream`) of
 * workspace_bytes >= attn_bwd_workspace_size(...) bytes; ATTN_ERR_WORKSPACE
 * when it is NULL, misaligned or too small (nothing queued).
 */
attn_status_t attn_bwd_ws(const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                          int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                          const int32_t* valid_len, attn_dtype_t dtype, void* workspace,
                          size_t workspace_bytes, attn_stream_t stream);
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
                                 attn_stream_t stream);

/*
 * attn_workspace_pool_stats -- memory of the workspace pool the library keeps
 * on the current device for calls made without a caller workspace:
 * *reserved_bytes the pool's reserved device memory, *high_water_bytes the
 * most it had handed out at once since the last reset (both 0 when no call
 * on this device has needed the pool).  reset_high_water != 0 resets the
 * high-water mark after reading it.  Either pointer may be NULL.  Lets a
 * caller account for the library's memory, and check that its *_ws calls
 * take none from the pool.
 */
attn_status_t attn_workspace_pool_stats(int reset_high_water, size_t* reserved_bytes,
                                        size_t* high_water_bytes);

/*
 * attn_bwd_simt -- the same gradients computed by SIMT kernels with fp32
 * arithmetic throughout (P and dS are never rounded to 16 bits): delta; dQ per
 * 64-row query tile; dK/dV per 64-key tile with all query heads of its group;
 * 4 x 4 register blocks over transposed shared-memory tiles.  A cross-check of
 * attn_bwd, and much slower.  Same arguments, preconditions and errors
 * as attn_bwd except D: 64 or 128 only; workspace B*Hq*L*4 bytes.
 */
attn_status_t attn_bwd_simt(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                            int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                            const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream);

/* The fp32 comparison kernels of attn_fwd_f32. */
typedef enum {
  ATTN_F32_NAIVE = 0,          /* three passes over the keys per query */
  ATTN_F32_TILED_ELEMENT = 1,  /* tiled, online softmax updated after every key */
  ATTN_F32_TILED_ROWMAX = 2    /* tiled, block row max first, one exponential per score */
} attn_f32_kernel_t;

/*
 * attn_fwd_f32 -- the same operation on fp32 tensors, computed by one of the
 * three CUDA kernels that "masked multi head attention in CUDA" (wzjinhao.cn)
 * compares in section 6.1: the naive kernel of section 3.1 (one block per
 * query, one thread per head column, three passes: scores and max, sum of
 * exponentials, weighted sum of V), and the tiled kernels of sections
 * 4.1-4.3 (Q tile resident in shared memory, K/V tiles of 32 keys, one thread
 * per output element; online softmax after every key, or block row max with
 * one exponential per score).  fp32 throughout, no tensor cores.  They exist
 * to reproduce that comparison on this GPU; attn_fwd is the fast path.
 *
 * Arguments: q, k, v, o fp32 [B, H, L, D] contiguous device memory (4-byte
 * aligned; multi-head, K and V with the same H); lse fp32 [B*H, L] or NULL;
 * D 64 or 128; valid_len, causal, sm_scale as attn_fwd.  B*H <= 65535; the
 * naive kernel keeps a query's L scores in shared memory (L <= 50000).
 * Errors as attn_fwd (ATTN_ERR_ARG for an unknown kernel).
 */
attn_status_t attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                           int B, int H, int L, int D, float sm_scale, int causal,
                           const int32_t* valid_len, attn_f32_kernel_t kernel,
                           attn_stream_t stream);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that must not allocate device
 * memory.  The pages have no counterpart: this is a deployment variant.
 *
 * attn_fwd allocates one int of device memory (its device status word) with
 * cudaMalloc on its first call on a device.  Callers that cannot allow that
 * -- servers that reserve all device memory at start-up and forbid
 * allocations on the request path (cudaMalloc can synchronise the device and
 * stall every other stream); latency-bound loops that cannot afford an
 * allocation's unpredictable cost; runtimes whose memory accounting covers
 * only their own allocator -- use this entry point instead.  Same arguments,
 * same layouts and the same kernel as attn_fwd; it calls no cudaMalloc,
 * cudaFree or any other allocating routine.  Results: ATTN_F16 calls equal
 * attn_fwd's.  ATTN_BF16 calls cannot take attn_fwd's workspace (the fp16 copy
 * of V), so every key tile runs P.V with P split into two bf16 terms
 * (P_hi + P_lo), the form attn_fwd uses only for tiles outside fp16's range:
 * the same accuracy bound, about twice the P.V tensor-core work.
 *
 * Scratch: the kernel's status word lives in a fixed 256-byte array
 * (64 int32 words) of the library's static device memory, which every GPU
 * that loads libattn.so holds until the process exits.  One call uses one
 * word; a call that needed more than the array holds would be rejected with
 * ATTN_ERR_SCRATCH before anything is queued.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); if the CUDA driver has
 * not yet loaded the library's static device data on that device, this is
 * when it does (the array itself, a one-time cost).  Make that first call
 * before any stream capture begins on the device.
 *
 * Sharing: every call on a device uses the same array.  The status word
 * starts at zero when the library's device data is loaded, each call ORs its
 * conditions into it, and attn_status reads and clears it together with
 * attn_fwd's word -- so, as with attn_fwd, it holds every condition since the
 * last attn_status.  Nothing else in the array must start at zero.  Calls
 * whose executions overlap on the GPU (different streams without ordering)
 * race on the word's read-and-clear: order them, or read attn_status between
 * them, if their device-side status matters.
 */
attn_status_t attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                               const int32_t* valid_len, attn_dtype_t dtype,
                               attn_stream_t stream);

/*
 * attn_fwd_host -- attn_fwd with every buffer in HOST memory: the call a
 * program makes when its tensors are not yet on the GPU.  The pages define
 * only the device-side operation; this entry point adds the host<->device
 * transfers around it.
 *
 * Arguments: as attn_fwd, except that q, k, v, o, lse and valid_len are host
 * pointers (any alignment).  Page-locked memory (cudaHostAlloc,
 * cudaHostRegister, torch pin_memory) lets the copies overlap the kernels;
 * pageable memory gives the same results, but the CUDA driver then stages
 * each copy and this call blocks until it is done.  Pointers to device or
 * managed memory are accepted too (the copies use cudaMemcpyDefault).
 *
 * Work: the problem is cut into chunks of consecutive query heads -- see
 * attn_host_plan; each chunk is one contiguous slice of every tensor -- and
 * three queues run side by side: the host->device copies of Q, K and V
 * chunk by chunk on a copy stream the library owns, the attention of each
 * chunk (exactly attn_fwd's kernels, on `stream`) once its inputs have
 * landed, and the device->host copies of O and LSE of each finished chunk
 * on a second library-owned copy stream.  The host link is the bound: the
 * call moves 2*(B*Hq + 2*B*Hkv)*L*D bytes in and 2*B*Hq*L*D (+ 4*B*Hq*L
 * for lse) out.  Results are identical to attn_fwd's on the same inputs.
 *
 * Ordering: everything the call queues starts after the work already on
 * `stream`, and `stream` waits for all of it (both copy streams join it at
 * the end), so o and lse may be read once `stream` has synchronised
 * (attn_status(stream, ...) or cudaStreamSynchronize).  The call itself
 * returns after queueing (unless the memory is pageable).
 *
 * Device memory: one stream-ordered allocation from the library's
 * per-device pool holding the device copies of the whole problem
 * (2*(2*B*Hq + 2*B*Hkv)*L*D bytes, + lse, + valid_len), returned with
 * cudaFreeAsync on `stream` after the last copy; ATTN_BF16 chunks also take
 * attn_fwd's workspace.  The copy streams and their events are created on
 * the first call on a device and destroyed by attn_shutdown.  Calls on one
 * device are serialised while they are queued (a per-device lock); their
 * copies share the two copy streams.
 *
 * Errors: argument errors as attn_fwd (nothing is queued).  A CUDA error
 * while queueing stops the remaining chunks, still joins and frees what
 * was queued, and returns ATTN_ERR_CUDA.
 */
attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int L, int D, float sm_scale, int causal,
                            const int32_t* valid_len, attn_dtype_t dtype, attn_stream_t stream);

/* One chunk of attn_fwd_host.  Heads are flattened: query head h of batch b
 * is b*Hq + h, key/value head h_kv of batch b is b*Hkv + h_kv. */
typedef struct {
  int q_head0;   /* first query head of the chunk */
  int q_heads;   /* consecutive query heads in the chunk (>= 1) */
  int kv_head0;  /* first key/value head whose K and V this chunk copies in */
  int kv_heads;  /* K/V heads it copies in (0 when earlier chunks copied all it needs) */
  int calls;     /* attention calls it is computed in: the query heads are cut at
                    key/value-group and batch boundaries into calls of whole batches,
                    whole groups of one batch, or part of one group */
} attn_chunk_t;

/*
 * attn_host_plan -- the chunks attn_fwd_host cuts a problem into, in the
 * order it queues them.  Together the chunks copy every query head and
 * every key/value head in exactly once, in order, and each chunk's K/V heads
 * have landed no later than its own inputs.  A full chunk holds about an
 * eighth of the problem's input, kept within [8, 32] MiB (and larger only
 * when that would make over 48 chunks); the first chunks ramp up from 1/8
 * of a full chunk and the last ones ramp down, so that the first kernel
 * starts early and little is left once the last input lands.  A problem
 * under 12 MiB of input is one chunk.  Writes min(*n_chunks, cap)
 * entries to chunks (chunks may be NULL when cap is 0) and the full count
 * to *n_chunks.  Host-only: needs no device.  Returns attn_fwd's argument
 * errors for invalid sizes, ATTN_ERR_ARG for a NULL n_chunks or a negative
 * cap.
 */
attn_status_t attn_host_plan(int B, int Hq, int Hkv, int L, int D, attn_dtype_t dtype,
                             attn_chunk_t* chunks, int cap, int* n_chunks);

/*
 * attn_status -- synchronise `stream`, then read and clear the device status
 * word of the current device.  *device_code (may be NULL) receives the raw
 * word: bit 0 a bounded wait timed out, bit 1 a valid_len value was clamped,
 * bit 2 a kernel found its shared memory smaller or less aligned than its
 * layout needs (it then did nothing; reported as ATTN_ERR_ARCH);
 * bits 8..11 are a set of role flags, one per waiting role that timed out
 * (0x100 the TMA producer, 0x200 an MMA issuer, 0x400 the softmax, 0x800 the
 * epilogue), ORed over every timed-out wait of every CTA and call since the
 * word was last read.  Returns ATTN_OK, ATTN_ERR_TIMEOUT,
 * ATTN_ERR_VALID_LEN (timeout wins when both are set) or ATTN_ERR_CUDA when
 * the synchronisation itself reported an error (ATTN_ERR_ARCH for bit 2).
 */
attn_status_t attn_status(attn_stream_t stream, int* device_code);

/* Capabilities and launch configuration of attn_fwd for a head dimension. */
typedef struct {
  int supported;        /* 1 if attn_fwd accepts this (D, dtype) on the current device */
  int block_m;          /* query rows per tensor-core tile (TMEM lanes) */
  int q_tiles_per_cta;  /* query tiles a CTA keeps in flight (ping-pong) */
  int block_n;          /* keys per K/V tile */
  int kv_stages;        /* shared-memory ring stages (one K or one V tile each) */
  int threads;          /* threads per CTA */
  int smem_bytes;       /* dynamic shared memory per CTA */
  int tmem_cols;        /* tensor-memory columns allocated per CTA */
  int num_sms;          /* SMs on the current device (0 without a device) */
  int lse_natural_log;  /* 1: lse is in natural-log units */
} attn_caps_t;

/*
 * attn_query -- fill *out for head dimension D and dtype.  Does not need a
 * device for the static fields; num_sms is 0 and supported is 0 without an
 * sm_103 device.  Returns ATTN_ERR_ARG for a NULL out, ATTN_ERR_HEADDIM /
 * ATTN_ERR_DTYPE for unsupported values (out still describes nothing).
 */
attn_status_t attn_query(int D, attn_dtype_t dtype, attn_caps_t* out);

/* A static, human-readable description of a status code. */
const char* attn_strerror(attn_status_t status);

/* The CUDA error code (cudaError_t as int) of the most recent ATTN_ERR_CUDA
 * returned on this thread, or 0. */
int attn_last_cuda_error(void);

/* Free the per-device status words, destroy the per-device workspace pools
 * (their memory is released once every queued call that took a workspace
 * has completed) and attn_fwd_host's copy streams and events.  Optional, at process exit; attn_fwd may be called
 * again afterwards (they are re-created). */
void attn_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */
