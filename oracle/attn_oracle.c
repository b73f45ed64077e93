/*
 * Float64 CPU oracle for the fused multi-head attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the package
 * attention_forward_attn_gb300 and its CUDA library) may include, link, load
 * or call this file.  Only tests/, __graft_entry__.smoke() and the CPU-baseline
 * leg of bench.py use it.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it computes (plain definition, no blocking, no online softmax):
 *
 *   Attention(Q,K,V) = softmax(Q K^T * sm_scale + Mask) V
 *     -- "masked multi head attention in CUDA" (wzjinhao.cn), section 2.1,
 *        the attention formula over [B, H, N, D] with B and H merged.
 *
 * computed per query row in three passes, the structure of that page's
 * naive kernel (section 3.1): pass 1 scores and their maximum, pass 2 the sum
 * of exp(score - max), pass 3 the exp-weighted sum of V rows divided by
 * that sum.  Everything is float64 with libm exp/log.
 *
 * Masks (section 2.2 of the same page): the implicit causal mask removes
 * key j > query i (the Triton-CUDA Attention page, "Causal Attention":
 * the kept set is offs_m >= start_n + offs_n); the padding mask removes key
 * j >= valid_len[b].  A row whose key set is empty outputs 0 (section 3.2,
 * "output 0 for an all-invalid row") and its log-sum-exp is -inf (the log of
 * an empty sum).
 *
 * Head grouping (Triton-CUDA Attention page, "GQA"): h_kv = h_q // (Hq/Hkv),
 * integer division, never modulo.
 *
 * Explicit mask ("masked multi head attention in CUDA", section 2.2: a
 * [B, N, N] boolean matrix, or a float matrix of 0 for a kept and -inf for a
 * removed position added to the scores -- the same set of kept positions):
 * mask[b, i, j] == 0 removes key j from query i of batch b, for every head.
 * All masks combine by intersection of their kept sets (the page's
 * "combined mask").
 *
 * Query and key lengths: the pages use one sequence length for Q, K and V.
 * Here Q has Lq rows and K/V have Lk rows (Lq = Lk is the pages' case); the
 * masks keep the pages' comparisons on absolute positions, so the causal
 * mask stays top-left aligned (key j visible to query i iff j <= i) and the
 * padding mask still removes key j >= valid_len[b].
 *
 * Log-sum-exp: the natural-log LSE of the scaled scores,
 *   LSE[i] = log sum_{j in J} exp(sm_scale * q_i . k_j),
 * which is tiny_flash_attn_triton.py's stored m + log2(l) (base 2, in the
 * sm_scale*log2(e)-scaled domain) multiplied by ln 2.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE binary16 -> double, by its published bit layout
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits). */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double val;
  if (e == 0) {
    val = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
  } else if (e == 31) {
    val = (m == 0) ? INFINITY : NAN;
  } else {
    val = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return sign ? -val : val;
}

/* bfloat16 -> double: bfloat16 is the upper half of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t b) {
  uint32_t bits = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* dtype: 0 = fp16, 1 = bf16.  Decodes n 16-bit values into out. */
int oracle_decode(const uint16_t* in, double* out, int64_t n, int dtype) {
  if (dtype != 0 && dtype != 1) return 1;
  for (int64_t t = 0; t < n; ++t)
    out[t] = dtype == 0 ? oracle_f16_to_f64(in[t]) : oracle_bf16_to_f64(in[t]);
  return 0;
}

/* The explicit mask: element (b, i, j) at mask[b*batch_stride + i*row_stride + j]. */
typedef struct {
  const uint8_t* mask; /* NULL: no explicit mask */
  int64_t batch_stride, row_stride;
} oracle_mask_t;

/* Is key j visible to query i of batch b? */
static int key_visible(int64_t i, int64_t j, int b, int causal, const int32_t* valid_len,
                       const oracle_mask_t* mk) {
  if (causal && j > i) return 0;
  if (valid_len != NULL && j >= (int64_t)valid_len[b]) return 0;
  if (mk->mask != NULL && mk->mask[b * mk->batch_stride + i * mk->row_stride + j] == 0) return 0;
  return 1;
}

/*
 * One query row, three passes.  q_row: D values; k_head, v_head: Lk x D rows
 * of the mapped key/value head; s: scratch of Lk doubles.
 */
static void one_row(const double* q_row, const double* k_head, const double* v_head,
                    int64_t i, int b, int Lk, int D, double sm_scale, int causal,
                    const int32_t* valid_len, const oracle_mask_t* mk, double* s, double* o_row,
                    double* lse_out) {
  /* pass 1: scores of the visible keys and their maximum */
  double m = -INFINITY;
  int64_t n_visible = 0;
  for (int64_t j = 0; j < Lk; ++j) {
    if (!key_visible(i, j, b, causal, valid_len, mk)) continue;
    const double* k_row = k_head + j * (int64_t)D;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q_row[d] * k_row[d];
    s[j] = sm_scale * dot;
    if (s[j] > m) m = s[j];
    ++n_visible;
  }
  if (n_visible == 0) {
    for (int d = 0; d < D; ++d) o_row[d] = 0.0;
    *lse_out = -INFINITY;
    return;
  }
  /* pass 2: the normaliser l = sum_j exp(s_j - m); s_j is replaced by its weight */
  double l = 0.0;
  for (int64_t j = 0; j < Lk; ++j) {
    if (!key_visible(i, j, b, causal, valid_len, mk)) continue;
    s[j] = exp(s[j] - m);
    l += s[j];
  }
  /* pass 3: O = sum_j w_j v_j / l */
  for (int d = 0; d < D; ++d) o_row[d] = 0.0;
  for (int64_t j = 0; j < Lk; ++j) {
    if (!key_visible(i, j, b, causal, valid_len, mk)) continue;
    const double* v_row = v_head + j * (int64_t)D;
    for (int d = 0; d < D; ++d) o_row[d] += s[j] * v_row[d];
  }
  for (int d = 0; d < D; ++d) o_row[d] /= l;
  *lse_out = m + log(l);
}

/*
 * q: [B, Hq, Lq, D]; k, v: [B, Hkv, Lk, D] (contiguous, float64).
 * rows == NULL: every row r = (b*Hq + h_q)*Lq + i, written to o[r*D..], lse[r].
 * rows != NULL: row rows[n] written to o[n*D..], lse[n], for n < nrows.
 * valid_len: NULL (no padding mask) or B int32 values.
 * threads <= 0: OpenMP default.
 * Returns 0, or 1 on invalid arguments.
 */
int oracle_attn_fwd_f64(const double* q, const double* k, const double* v, double* o,
                        double* lse, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                        double sm_scale, int causal, const int32_t* valid_len,
                        const uint8_t* mask, int64_t mask_batch_stride, int64_t mask_row_stride,
                        const int64_t* rows, int64_t nrows, int threads) {
  const oracle_mask_t mk = {mask, mask_batch_stride, mask_row_stride};
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1 || D < 1 || Hq % Hkv != 0) return 1;
  const int G = Hq / Hkv;
  const int64_t total = (int64_t)B * Hq * Lq;
  const int64_t n_out = rows ? nrows : total;
  if (rows)
    for (int64_t n = 0; n < nrows; ++n)
      if (rows[n] < 0 || rows[n] >= total) return 1;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
    if (!s) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 16)
    for (int64_t n = 0; n < n_out; ++n) {
      if (!s) continue;
      const int64_t r = rows ? rows[n] : n;
      const int64_t bh = r / Lq;
      const int64_t i = r % Lq;
      const int b = (int)(bh / Hq);
      const int h_q = (int)(bh % Hq);
      const int h_kv = h_q / G; /* integer division, never modulo */
      const double* q_row = q + r * (int64_t)D;
      const double* k_head = k + ((int64_t)b * Hkv + h_kv) * Lk * (int64_t)D;
      const double* v_head = v + ((int64_t)b * Hkv + h_kv) * Lk * (int64_t)D;
      one_row(q_row, k_head, v_head, i, b, Lk, D, sm_scale, causal, valid_len, &mk, s,
              o + n * (int64_t)D, lse + n);
    }
    free(s);
  }
  return bad ? 2 : 0;
}

/* Same as oracle_attn_fwd_f64, on raw fp16 (dtype 0) or bf16 (dtype 1) bits. */
int oracle_attn_fwd_u16(const uint16_t* q, const uint16_t* k, const uint16_t* v, double* o,
                        double* lse, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                        double sm_scale, int causal, const int32_t* valid_len,
                        const uint8_t* mask, int64_t mask_batch_stride, int64_t mask_row_stride,
                        int dtype, const int64_t* rows, int64_t nrows, int threads) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1 || D < 1 || Hq % Hkv != 0) return 1;
  if (dtype != 0 && dtype != 1) return 1;
  const int64_t nq = (int64_t)B * Hq * Lq * D;
  const int64_t nkv = (int64_t)B * Hkv * Lk * D;
  double* qd = (double*)malloc(sizeof(double) * (size_t)nq);
  double* kd = (double*)malloc(sizeof(double) * (size_t)nkv);
  double* vd = (double*)malloc(sizeof(double) * (size_t)nkv);
  int rc = 2;
  if (qd && kd && vd) {
    oracle_decode(q, qd, nq, dtype);
    oracle_decode(k, kd, nkv, dtype);
    oracle_decode(v, vd, nkv, dtype);
    rc = oracle_attn_fwd_f64(qd, kd, vd, o, lse, B, Hq, Hkv, Lq, Lk, D, sm_scale, causal,
                             valid_len, mask, mask_batch_stride, mask_row_stride, rows, nrows,
                             threads);
  }
  free(qd);
  free(kd);
  free(vd);
  return rc;
}

/* Number of threads an OpenMP parallel region would use. */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Backward of the same operation, from its definition (the pages store the
 * log-sum-exp "for the backward pass" -- tiny_flash_attn_triton.py -- but give
 * no backward algorithm, so this is the derivative of
 *   O = softmax(S) V,  S = sm_scale * Q K^T restricted to the visible keys,
 * written out with the chain rule).  For a loss with gradient dO:
 *   P_ij = exp(S_ij) / sum_j' exp(S_ij')            (visible j; 0 otherwise)
 *   dV_j = sum_i P_ij dO_i
 *   dP_ij = dO_i . V_j
 *   dS_ij = P_ij (dP_ij - sum_j' P_ij' dP_ij')      (softmax Jacobian)
 *   dQ_i = sm_scale sum_j dS_ij K_j,   dK_j = sm_scale sum_i dS_ij Q_i
 * with K_j, V_j of head h_kv = h_q / (Hq/Hkv); dK and dV of a key/value head
 * sum over the query heads that read it.  Rows without a visible key give
 * nothing.  Float64, plain loops, one (b, h_kv) group per OpenMP task.
 *
 * q, dO: [B, Hq, L, D]; k, v: [B, Hkv, L, D]; dq like q, dk and dv like k.
 * Returns 0, 1 on invalid arguments, 2 when scratch could not be allocated.
 */
int oracle_attn_bwd_f64(const double* q, const double* k, const double* v, const double* dO,
                        double* dq, double* dk, double* dv, int B, int Hq, int Hkv, int L, int D,
                        double sm_scale, int causal, const int32_t* valid_len, int threads) {
  if (B < 1 || Hq < 1 || Hkv < 1 || L < 1 || D < 1 || Hq % Hkv != 0) return 1;
  const int G = Hq / Hkv;
  const oracle_mask_t mk = {NULL, 0, 0};
  memset(dq, 0, sizeof(double) * (size_t)B * Hq * L * D);
  memset(dk, 0, sizeof(double) * (size_t)B * Hkv * L * D);
  memset(dv, 0, sizeof(double) * (size_t)B * Hkv * L * D);
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  int bad = 0;
#pragma omp parallel
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)L);   /* P_i. of one row */
    double* dp = (double*)malloc(sizeof(double) * (size_t)L);  /* dP_i. of one row */
    if (!p || !dp) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t grp = 0; grp < (int64_t)B * Hkv; ++grp) {
      if (!p || !dp) continue;
      const int b = (int)(grp / Hkv);
      const int h_kv = (int)(grp % Hkv);
      const double* k_head = k + grp * L * (int64_t)D;
      const double* v_head = v + grp * L * (int64_t)D;
      double* dk_head = dk + grp * L * (int64_t)D;
      double* dv_head = dv + grp * L * (int64_t)D;
      for (int g = 0; g < G; ++g) {
        const int h_q = h_kv * G + g;
        const int64_t qh = (int64_t)b * Hq + h_q;
        for (int64_t i = 0; i < L; ++i) {
          const double* q_row = q + (qh * L + i) * D;
          const double* do_row = dO + (qh * L + i) * D;
          double* dq_row = dq + (qh * L + i) * D;
          /* P_i. by the definition (max subtracted for the exponentials) */
          double m = -INFINITY;
          int any = 0;
          for (int64_t j = 0; j < L; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q_row[d] * k_head[j * D + d];
            p[j] = sm_scale * dot;
            if (p[j] > m) m = p[j];
            any = 1;
          }
          if (!any) continue;
          double z = 0.0;
          for (int64_t j = 0; j < L; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            p[j] = exp(p[j] - m);
            z += p[j];
          }
          double pdp = 0.0; /* sum_j P_ij dP_ij */
          for (int64_t j = 0; j < L; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            p[j] /= z;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += do_row[d] * v_head[j * D + d];
            dp[j] = dot;
            pdp += p[j] * dot;
          }
          for (int64_t j = 0; j < L; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            const double ds = p[j] * (dp[j] - pdp);
            for (int d = 0; d < D; ++d) {
              dv_head[j * D + d] += p[j] * do_row[d];
              dq_row[d] += sm_scale * ds * k_head[j * D + d];
              dk_head[j * D + d] += sm_scale * ds * q_row[d];
            }
          }
        }
      }
    }
    free(p);
    free(dp);
  }
  return bad ? 2 : 0;
}
