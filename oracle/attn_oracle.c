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

/* Threads for one call: `threads` when > 0, else the OpenMP default. */
static int oracle_threads(int threads) {
#ifdef _OPENMP
  return threads > 0 ? threads : omp_get_max_threads();
#else
  (void)threads;
  return 1;
#endif
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
  /* the thread count of this call only (the process-wide default is left as it is) */
  const int nthr = oracle_threads(threads);
  int bad = 0;
#pragma omp parallel num_threads(nthr)
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
 * q, dO: [B, Hq, Lq, D]; k, v: [B, Hkv, Lk, D]; dq like q, dk and dv like k
 * (Lq = Lk is the pages' case; the masks compare absolute positions as in
 * the forward).  mask: the forward's explicit mask (NULL: none), combined
 * with the causal and padding masks by intersection.
 * Returns 0, 1 on invalid arguments, 2 when scratch could not be allocated.
 */
int oracle_attn_bwd_f64(const double* q, const double* k, const double* v, const double* dO,
                        double* dq, double* dk, double* dv, int B, int Hq, int Hkv, int Lq, int Lk, int D,
                        double sm_scale, int causal, const int32_t* valid_len, const uint8_t* mask,
                        int64_t mask_batch_stride, int64_t mask_row_stride, int threads) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1 || D < 1 || Hq % Hkv != 0) return 1;
  const int G = Hq / Hkv;
  const oracle_mask_t mk = {mask, mask_batch_stride, mask_row_stride};  /* explicit mask or none */
  memset(dq, 0, sizeof(double) * (size_t)B * Hq * Lq * D);
  memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Lk * D);
  memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Lk * D);
  /* the thread count of this call only (the process-wide default is left as it is) */
  const int nthr = oracle_threads(threads);
  int bad = 0;
#pragma omp parallel num_threads(nthr)
  {
    double* p = (double*)malloc(sizeof(double) * (size_t)Lk);   /* P_i. of one row */
    double* dp = (double*)malloc(sizeof(double) * (size_t)Lk);  /* dP_i. of one row */
    if (!p || !dp) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t grp = 0; grp < (int64_t)B * Hkv; ++grp) {
      if (!p || !dp) continue;
      const int b = (int)(grp / Hkv);
      const int h_kv = (int)(grp % Hkv);
      const double* k_head = k + grp * Lk * (int64_t)D;
      const double* v_head = v + grp * Lk * (int64_t)D;
      double* dk_head = dk + grp * Lk * (int64_t)D;
      double* dv_head = dv + grp * Lk * (int64_t)D;
      for (int g = 0; g < G; ++g) {
        const int h_q = h_kv * G + g;
        const int64_t qh = (int64_t)b * Hq + h_q;
        for (int64_t i = 0; i < Lq; ++i) {
          const double* q_row = q + (qh * Lq + i) * D;
          const double* do_row = dO + (qh * Lq + i) * D;
          double* dq_row = dq + (qh * Lq + i) * D;
          /* P_i. by the definition (max subtracted for the exponentials) */
          double m = -INFINITY;
          int any = 0;
          for (int64_t j = 0; j < Lk; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q_row[d] * k_head[j * D + d];
            p[j] = sm_scale * dot;
            if (p[j] > m) m = p[j];
            any = 1;
          }
          if (!any) continue;
          double z = 0.0;
          for (int64_t j = 0; j < Lk; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            p[j] = exp(p[j] - m);
            z += p[j];
          }
          double pdp = 0.0; /* sum_j P_ij dP_ij */
          for (int64_t j = 0; j < Lk; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            p[j] /= z;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += do_row[d] * v_head[j * D + d];
            dp[j] = dot;
            pdp += p[j] * dot;
          }
          for (int64_t j = 0; j < Lk; ++j) {
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

/*
 * Statistics of query row i (q_row, do_row) against the keys of its K/V head,
 * from the definition: the maximum m of the visible scores s_j = sm_scale *
 * q_i.k_j, z = sum_j exp(s_j - m), delta = sum_j P_ij dP_ij with
 * P_ij = exp(s_j - m) / z and dP_ij = dO_i.v_j.  s: scratch of Lk doubles.
 * Returns the number of visible keys (0: the row sees none; m, z, delta unset).
 */
static int64_t row_stats(const double* q_row, const double* do_row, const double* k_head,
                         const double* v_head, int64_t i, int b, int Lk, int D, double sm_scale,
                         int causal, const int32_t* valid_len, const oracle_mask_t* mkp,
                         double* s, double* m_out, double* z_out, double* delta_out) {
  const oracle_mask_t mk = *mkp;
  double m = -INFINITY;
  int64_t n = 0;
  for (int64_t j = 0; j < Lk; ++j) {
    if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q_row[d] * k_head[j * D + d];
    s[j] = sm_scale * dot;
    if (s[j] > m) m = s[j];
    ++n;
  }
  if (n == 0) return 0;
  double z = 0.0, acc = 0.0;
  for (int64_t j = 0; j < Lk; ++j) {
    if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
    const double e = exp(s[j] - m);
    double dp = 0.0;
    for (int d = 0; d < D; ++d) dp += do_row[d] * v_head[j * D + d];
    z += e;
    acc += e * dp;
  }
  *m_out = m;
  *z_out = z;
  *delta_out = acc / z;
  return n;
}

/*
 * Selected rows of the gradients of oracle_attn_bwd_f64 (same inputs and
 * definition), for checks at sizes where the full backward is too slow:
 *   dQ rows q_rows[r] (flat index (b*Hq + h_q)*Lq + i), r < n_q -> dq[r*D ..];
 *   dK, dV rows k_rows[r] (flat index (b*Hkv + h_kv)*Lk + j), r < n_k ->
 *   dk[r*D ..], dv[r*D ..].
 * A key row sums over every query row of its group's G query heads, so the
 * statistics of those rows are computed once per group that a sampled key
 * row belongs to.  Also, per row, magnitudes a tolerance can be built on
 * (w_i = sum_d |dO_id O_id|, O_i the forward's output row):
 *   qmag[3r ..]: sum_j |dS_ij|, w_i, visible keys;
 *   kmag[4r ..]: sum_i |dS_ij|, sum_i P_ij, sum_i P_ij w_i, visible queries
 * (sums over the G query heads of the key's group).  mask: as in
 * oracle_attn_bwd_f64.
 */
int oracle_attn_bwd_rows_f64(const double* q, const double* k, const double* v, const double* dO,
                             int B, int Hq, int Hkv, int Lq, int Lk, int D, double sm_scale,
                             int causal, const int32_t* valid_len, const uint8_t* mask,
                             int64_t mask_batch_stride, int64_t mask_row_stride,
                             const int64_t* q_rows, int64_t n_q,
                             double* dq, double* qmag, const int64_t* k_rows, int64_t n_k,
                             double* dk, double* dv, double* kmag, int threads) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lq < 1 || Lk < 1 || D < 1 || Hq % Hkv != 0) return 1;
  const int G = Hq / Hkv;
  const oracle_mask_t mk = {mask, mask_batch_stride, mask_row_stride};  /* the rows' key sets */
  for (int64_t r = 0; r < n_q; ++r)
    if (q_rows[r] < 0 || q_rows[r] >= (int64_t)B * Hq * Lq) return 1;
  for (int64_t r = 0; r < n_k; ++r)
    if (k_rows[r] < 0 || k_rows[r] >= (int64_t)B * Hkv * Lk) return 1;
  /* the thread count of this call only (the process-wide default is left as it is) */
  const int nthr = oracle_threads(threads);
  int bad = 0;
  /* dQ rows */
#pragma omp parallel num_threads(nthr)
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
    if (!s) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_q; ++r) {
      if (!s) continue;
      const int64_t qh = q_rows[r] / Lq;
      const int64_t i = q_rows[r] % Lq;
      const int b = (int)(qh / Hq);
      const int64_t kvh = (int64_t)b * Hkv + (qh % Hq) / G;
      const double* q_row = q + q_rows[r] * D;
      const double* do_row = dO + q_rows[r] * D;
      const double* k_head = k + kvh * Lk * (int64_t)D;
      const double* v_head = v + kvh * Lk * (int64_t)D;
      double* dq_row = dq + r * D;
      double m = 0.0, z = 1.0, delta = 0.0, sabs = 0.0, w = 0.0;
      for (int d = 0; d < D; ++d) dq_row[d] = 0.0;
      const int64_t n = row_stats(q_row, do_row, k_head, v_head, i, b, Lk, D, sm_scale, causal,
                                  valid_len, &mk, s, &m, &z, &delta);
      if (n > 0) {
        double* o_row = (double*)calloc((size_t)D, sizeof(double));
        for (int64_t j = 0; j < Lk; ++j) {
          if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
          const double p = exp(s[j] - m) / z;
          double dp = 0.0;
          for (int d = 0; d < D; ++d) dp += do_row[d] * v_head[j * D + d];
          const double ds = p * (dp - delta);
          const double* k_j = k_head + j * D;
          sabs += fabs(ds);
          for (int d = 0; d < D; ++d) {
            dq_row[d] += sm_scale * ds * k_j[d];
            if (o_row) o_row[d] += p * v_head[j * D + d];
          }
        }
        if (o_row) {
          for (int d = 0; d < D; ++d) w += fabs(do_row[d] * o_row[d]);
        } else {
#pragma omp atomic write
          bad = 1;
        }
        free(o_row);
      }
      qmag[3 * r] = sabs;
      qmag[3 * r + 1] = w;
      qmag[3 * r + 2] = (double)n;
    }
    free(s);
  }
  /* dK, dV rows: group by K/V head, row statistics of the group's query rows once */
  for (int64_t r0 = 0; r0 < n_k && !bad; ++r0) {
    const int64_t kvh = k_rows[r0] / Lk;
    int seen = 0;
    for (int64_t r = 0; r < r0; ++r) seen |= (k_rows[r] / Lk == kvh);
    if (seen) continue;
    const int b = (int)(kvh / Hkv);
    const int h_kv = (int)(kvh % Hkv);
    const double* k_head = k + kvh * Lk * (int64_t)D;
    const double* v_head = v + kvh * Lk * (int64_t)D;
    const int64_t nrow = (int64_t)G * Lq;
    double* st = (double*)malloc(sizeof(double) * 4 * (size_t)nrow);  /* m, z, delta, w */
    if (!st) return 2;
#pragma omp parallel num_threads(nthr)
    {
      double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
      double* o_row = (double*)malloc(sizeof(double) * (size_t)D);
      if (!s || !o_row) {
#pragma omp atomic write
        bad = 1;
      }
#pragma omp for schedule(dynamic, 16)
      for (int64_t gi = 0; gi < nrow; ++gi) {
        if (!s || !o_row) continue;
        const int64_t qrow = ((int64_t)b * Hq + (int64_t)h_kv * G + gi / Lq) * Lq + gi % Lq;
        const int64_t i = gi % Lq;
        double m = 0.0, z = 1.0, delta = 0.0, w = 0.0;
        const int64_t n = row_stats(q + qrow * D, dO + qrow * D, k_head, v_head, i, b, Lk, D,
                                    sm_scale, causal, valid_len, &mk, s, &m, &z, &delta);
        if (n > 0) {
          for (int d = 0; d < D; ++d) o_row[d] = 0.0;
          for (int64_t j = 0; j < Lk; ++j) {
            if (!key_visible(i, j, b, causal, valid_len, &mk)) continue;
            const double p = exp(s[j] - m) / z;
            for (int d = 0; d < D; ++d) o_row[d] += p * v_head[j * D + d];
          }
          for (int d = 0; d < D; ++d) w += fabs(dO[qrow * D + d] * o_row[d]);
        }
        st[4 * gi] = n > 0 ? m : INFINITY;  /* +inf: the row sees no key */
        st[4 * gi + 1] = z;
        st[4 * gi + 2] = delta;
        st[4 * gi + 3] = w;
      }
      free(s);
      free(o_row);
    }
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthr)
    for (int64_t r = r0; r < n_k; ++r) {
      if (k_rows[r] / Lk != kvh) continue;
      const int64_t j = k_rows[r] % Lk;
      const double* k_row = k_head + j * D;
      const double* v_row = v_head + j * D;
      double* dk_row = dk + r * D;
      double* dv_row = dv + r * D;
      double sabs = 0.0, psum = 0.0, pw = 0.0, nvis = 0.0;
      for (int d = 0; d < D; ++d) dk_row[d] = dv_row[d] = 0.0;
      for (int64_t gi = 0; gi < nrow; ++gi) {
        const int64_t i = gi % Lq;
        if (st[4 * gi] == INFINITY || !key_visible(i, j, b, causal, valid_len, &mk)) continue;
        const int64_t qrow = ((int64_t)b * Hq + (int64_t)h_kv * G + gi / Lq) * Lq + i;
        const double* q_row = q + qrow * D;
        const double* do_row = dO + qrow * D;
        double dot = 0.0, dp = 0.0;
        for (int d = 0; d < D; ++d) {
          dot += q_row[d] * k_row[d];
          dp += do_row[d] * v_row[d];
        }
        const double p = exp(sm_scale * dot - st[4 * gi]) / st[4 * gi + 1];
        const double ds = p * (dp - st[4 * gi + 2]);
        for (int d = 0; d < D; ++d) {
          dv_row[d] += p * do_row[d];
          dk_row[d] += sm_scale * ds * q_row[d];
        }
        sabs += fabs(ds);
        psum += p;
        pw += p * st[4 * gi + 3];
        nvis += 1.0;
      }
      kmag[4 * r] = sabs;
      kmag[4 * r + 1] = psum;
      kmag[4 * r + 2] = pw;
      kmag[4 * r + 3] = nvis;
    }
    free(st);
  }
  return bad ? 2 : 0;
}
