/*
 * swa_ref.c — plain, slow, obviously-correct fp64 CPU oracle for
 * sliding-window (BAND) / unmasked softmax attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * What it computes (restated from the sources cited per function):
 *   forward  (FlashAttentionVarLenScore doc, "计算公式";
 *             PyPTO-Gym FlashAttentionScoreGrad article, "前向公式"):
 *       s_ij = scale * q_i . k_j
 *       V_i  = keys visible to query i (sparse_mode 0: all keys of the
 *              sequence; sparse_mode 4 BAND: i - pre <= j <= i + next)
 *       m_i  = max_{j in V_i} s_ij                 -> softmax_max
 *       l_i  = sum_{j in V_i} exp(s_ij - m_i)      -> softmax_sum
 *       P_ij = exp(s_ij - m_i) / l_i  on V_i, 0 elsewhere
 *       O_i  = sum_j P_ij * z_ij / keep_prob * v_j (inverted dropout, z in {0,1})
 *   backward (PyPTO-Gym article, "反向公式"; aclnnFlashAttentionUnpadding-
 *             ScoreGradV2 article §2.3):
 *       D_i   = sum_d dY_id * O_id
 *       dP_ij = (dY_i . v_j) * z_ij / keep_prob
 *       dS_ij = P_ij * (dP_ij - D_i)
 *       dV_j  = sum_i P_ij * z_ij / keep_prob * dY_i
 *       dQ_i  = scale * sum_j dS_ij * k_j
 *       dK_j  = scale * sum_i dS_ij * q_i
 * Empty rows (V_i empty): O_i = 0, m_i = -inf, l_i = 0, no gradient flows.
 *
 * Grouped key/value heads (aclnnFlashAttentionUnpaddingScoreGradV2 article
 * §6.2: the query head count must be a non-zero integer multiple of the
 * key/value head count): query head n reads key/value head n / (N / N_kv),
 * and since that head is shared, its dK_j / dV_j are the sums of the
 * expressions above over the N / N_kv query heads that read it.
 *
 * Inputs are fp64 arrays (the bf16 values of the problem, converted exactly
 * by the caller); all arithmetic is double.  The
 * sequences of a TND problem use cumulative end offsets (no leading 0); a
 * drop in the cumulative array (trailing zeros) marks skipped batches.
 *
 * Parity pins for every exported function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t layout; /* 0 = BNSD [B,N,S,D]; 1 = TND [T,N,D] */
  int32_t sparse_mode; /* 0 = no mask, 4 = BAND */
  int64_t B, N, D;
  int64_t S_q, S_kv;      /* BNSD */
  int64_t T_q, T_kv;      /* TND */
  const int64_t *cu_q;    /* TND: cumulative ends, length B */
  const int64_t *cu_kv;
  double scale;
  int64_t pre_tokens, next_tokens;
  double keep_prob;
  int64_t N_kv; /* key/value heads; N is a multiple of N_kv */
} orc_params;

/* ------------------------------------------------------------ geometry -- */

/* Start offset and length of batch b's sequence (TND), from cumulative ends. */
static void seq_span(const int64_t *cu, int64_t b, int64_t *start, int64_t *len) {
  int64_t prev = (b == 0) ? 0 : cu[b - 1];
  int64_t end = cu[b];
  *start = prev;
  *len = end > prev ? end - prev : 0;
}

typedef struct {
  int64_t q_start, q_len, kv_start, kv_len; /* rows of this batch's sequence */
  int64_t mask_base;                        /* dropout bit index of (n=0,i=0,j=0) */
} orc_seq;

static orc_seq seq_of(const orc_params *p, int64_t b) {
  orc_seq s;
  if (p->layout == 0) {
    s.q_start = 0; s.q_len = p->S_q; s.kv_start = 0; s.kv_len = p->S_kv;
    s.mask_base = b * p->N * p->S_q * p->S_kv;
  } else {
    seq_span(p->cu_q, b, &s.q_start, &s.q_len);
    seq_span(p->cu_kv, b, &s.kv_start, &s.kv_len);
    /* masks of earlier batches are packed back to back, no padding */
    int64_t base = 0;
    for (int64_t bb = 0; bb < b; ++bb) {
      int64_t a, lq, c, lk;
      seq_span(p->cu_q, bb, &a, &lq);
      seq_span(p->cu_kv, bb, &c, &lk);
      base += p->N * lq * lk;
    }
    s.mask_base = base;
  }
  return s;
}

/* Element offset of row i (local to the sequence) of head n, batch b. */
static int64_t row_q(const orc_params *p, const orc_seq *s, int64_t b, int64_t n, int64_t i) {
  if (p->layout == 0) return ((b * p->N + n) * p->S_q + i) * p->D;
  return ((s->q_start + i) * p->N + n) * p->D;
}
/* Element offset of key row j of key/value head h, batch b. */
static int64_t row_kv(const orc_params *p, const orc_seq *s, int64_t b, int64_t h, int64_t j) {
  if (p->layout == 0) return ((b * p->N_kv + h) * p->S_kv + j) * p->D;
  return ((s->kv_start + j) * p->N_kv + h) * p->D;
}
/* The key/value head query head n reads. */
static int64_t kv_head(const orc_params *p, int64_t n) { return n / (p->N / p->N_kv); }
/* Index of the softmax statistics of query row i: [B,N,S] or [T,N]. */
static int64_t stat_q(const orc_params *p, const orc_seq *s, int64_t b, int64_t n, int64_t i) {
  if (p->layout == 0) return (b * p->N + n) * p->S_q + i;
  return (s->q_start + i) * p->N + n;
}

/* Visible key range of query i: sparse_mode 0 sees every key of its sequence;
 * BAND sees i - pre <= j <= i + next, clipped to [0, kv_len).  Returns 0 when
 * the set is empty. */
static int key_range(const orc_params *p, const orc_seq *s, int64_t i, int64_t *lo, int64_t *hi) {
  int64_t a = 0, b = s->kv_len - 1;
  if (p->sparse_mode == 4) {
    /* clamp pre/next into +-(S_q + S_kv): the window cannot reach further */
    int64_t lim = s->q_len + s->kv_len + 1;
    int64_t pre = p->pre_tokens > lim ? lim : (p->pre_tokens < -lim ? -lim : p->pre_tokens);
    int64_t nxt = p->next_tokens > lim ? lim : (p->next_tokens < -lim ? -lim : p->next_tokens);
    if (i - pre > a) a = i - pre;
    if (i + nxt < b) b = i + nxt;
  }
  *lo = a; *hi = b;
  return a <= b;
}
/* Query range that sees key j (the same inequality solved for i). */
static int query_range(const orc_params *p, const orc_seq *s, int64_t j, int64_t *lo, int64_t *hi) {
  int64_t a = 0, b = s->q_len - 1;
  if (j >= s->kv_len) return 0;
  if (p->sparse_mode == 4) {
    int64_t lim = s->q_len + s->kv_len + 1;
    int64_t pre = p->pre_tokens > lim ? lim : (p->pre_tokens < -lim ? -lim : p->pre_tokens);
    int64_t nxt = p->next_tokens > lim ? lim : (p->next_tokens < -lim ? -lim : p->next_tokens);
    if (j - nxt > a) a = j - nxt;
    if (j + pre < b) b = j + pre;
  }
  *lo = a; *hi = b;
  return a <= b;
}

/* Dropout keep bit z_ij: element e = mask_base + (n*Sq + i)*Skv + j of the
 * packed uint8 mask, LSB first, 1 = keep.  No mask means keep everything. */
static double keep_bit(const orc_seq *s, const uint8_t *mask, int64_t n, int64_t i,
                       int64_t j) {
  if (!mask) return 1.0;
  int64_t e = s->mask_base + (n * s->q_len + i) * s->kv_len + j;
  return (double)((mask[e >> 3] >> (e & 7)) & 1);
}

static double dot(const double *a, const double *b, int64_t D) {
  double acc = 0.0;
  for (int64_t d = 0; d < D; ++d) acc += a[d] * b[d];
  return acc;
}

/* ---------------------------------------------------------- per row ---- */

/* Forward for one query row: m, l and O (fp64). */
static void forward_row(const orc_params *p, const orc_seq *s, int64_t b, int64_t n, int64_t i,
                        const double *q, const double *k, const double *v, const uint8_t *mask,
                        double *o, double *m_out, double *l_out) {
  const int64_t D = p->D;
  int64_t lo, hi;
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  if (!key_range(p, s, i, &lo, &hi)) {
    *m_out = -INFINITY; *l_out = 0.0;
    return;
  }
  const double *qi = q + row_q(p, s, b, n, i);
  const int64_t h = kv_head(p, n);
  double m = -INFINITY;
  for (int64_t j = lo; j <= hi; ++j) {
    double sij = p->scale * dot(qi, k + row_kv(p, s, b, h, j), D);
    if (sij > m) m = sij;
  }
  double l = 0.0;
  for (int64_t j = lo; j <= hi; ++j) l += exp(p->scale * dot(qi, k + row_kv(p, s, b, h, j), D) - m);
  for (int64_t j = lo; j <= hi; ++j) {
    double pij = exp(p->scale * dot(qi, k + row_kv(p, s, b, h, j), D) - m) / l;
    double w = pij * keep_bit(s, mask, n, i, j) / p->keep_prob;
    const double *vj = v + row_kv(p, s, b, h, j);
    for (int64_t d = 0; d < D; ++d) o[d] += w * vj[d];
  }
  *m_out = m; *l_out = l;
}

/* Per-row data the backward needs: m, l and D_i = dY_i . O_i.  When the
 * caller supplies O / softmax_max / softmax_sum ("given-stats" mode) they
 * are used instead of the oracle's own forward. */
typedef struct { double m, l, Di; } row_data;

static row_data backward_row_data(const orc_params *p, const orc_seq *s, int64_t b, int64_t n, int64_t i,
                                  const double *q, const double *k, const double *v, const double *dy,
                                  const uint8_t *mask, const double *given_out, const double *given_max,
                                  const double *given_sum, double *scratch_o) {
  row_data r;
  const int64_t D = p->D;
  const double *dyi = dy + row_q(p, s, b, n, i);
  if (given_out) {
    int64_t st = stat_q(p, s, b, n, i);
    r.m = given_max[st]; r.l = given_sum[st];
    r.Di = dot(dyi, given_out + row_q(p, s, b, n, i), D);
  } else {
    forward_row(p, s, b, n, i, q, k, v, mask, scratch_o, &r.m, &r.l);
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d) acc += dyi[d] * scratch_o[d];
    r.Di = acc;
  }
  return r;
}

/* P_ij from the row statistics (the backward's recomputation). */
static double prob(const row_data *r, double sij) {
  if (r->l == 0.0) return 0.0;
  return exp(sij - r->m) / r->l;
}

/* dQ_i = scale * sum_j dS_ij k_j. */
static void dq_row(const orc_params *p, const orc_seq *s, int64_t b, int64_t n, int64_t i, const row_data *r,
                   const double *q, const double *k, const double *v, const double *dy,
                   const uint8_t *mask, double *dq) {
  const int64_t D = p->D;
  int64_t lo, hi;
  for (int64_t d = 0; d < D; ++d) dq[d] = 0.0;
  if (!key_range(p, s, i, &lo, &hi)) return;
  const double *qi = q + row_q(p, s, b, n, i);
  const double *dyi = dy + row_q(p, s, b, n, i);
  const int64_t h = kv_head(p, n);
  for (int64_t j = lo; j <= hi; ++j) {
    const double *kj = k + row_kv(p, s, b, h, j);
    double pij = prob(r, p->scale * dot(qi, kj, D));
    double dpij = dot(dyi, v + row_kv(p, s, b, h, j), D) * keep_bit(s, mask, n, i, j) / p->keep_prob;
    double dsij = pij * (dpij - r->Di);
    for (int64_t d = 0; d < D; ++d) dq[d] += p->scale * dsij * kj[d];
  }
}

/* dK_j and dV_j of key/value head h, gathering over the queries that see
 * key j in each of the query heads that read head h.  `rows` holds the row
 * data of those heads: rows[g * q_len + i] for the g-th head of the group. */
static void dkv_col(const orc_params *p, const orc_seq *s, int64_t b, int64_t h, int64_t j, const row_data *rows,
                    const double *q, const double *k, const double *v, const double *dy,
                    const uint8_t *mask, double *dk, double *dv) {
  const int64_t D = p->D, G = p->N / p->N_kv;
  int64_t lo, hi;
  for (int64_t d = 0; d < D; ++d) { dk[d] = 0.0; dv[d] = 0.0; }
  if (!query_range(p, s, j, &lo, &hi)) return;
  const double *kj = k + row_kv(p, s, b, h, j);
  const double *vj = v + row_kv(p, s, b, h, j);
  for (int64_t gi = 0; gi < G; ++gi) {
    const int64_t n = h * G + gi;
    for (int64_t i = lo; i <= hi; ++i) {
      const double *qi = q + row_q(p, s, b, n, i);
      const double *dyi = dy + row_q(p, s, b, n, i);
      const row_data *r = &rows[gi * s->q_len + i];
      double pij = prob(r, p->scale * dot(qi, kj, D));
      double z = keep_bit(s, mask, n, i, j) / p->keep_prob;
      double dsij = pij * (dot(dyi, vj, D) * z - r->Di);
      for (int64_t d = 0; d < D; ++d) {
        dv[d] += pij * z * dyi[d];
        dk[d] += p->scale * dsij * qi[d];
      }
    }
  }
}

/* Map a flat query-row id (the statistics index: (b*N+n)*S_q+i for BNSD,
 * t*N+n for TND) to (b, n, local i).  Returns 0 if the row belongs to no
 * sequence. */
static int locate_q(const orc_params *p, int64_t id, int64_t *b, int64_t *n, int64_t *i) {
  if (id < 0) return 0;
  if (p->layout == 0) {
    *i = id % p->S_q; *n = (id / p->S_q) % p->N; *b = id / (p->S_q * p->N);
    return *b < p->B;
  }
  int64_t t = id / p->N;
  *n = id % p->N;
  for (int64_t bb = 0; bb < p->B; ++bb) {
    int64_t st, len;
    seq_span(p->cu_q, bb, &st, &len);
    if (t >= st && t < st + len) { *b = bb; *i = t - st; return 1; }
  }
  return 0;
}
/* Map a flat key-row id ((b*N_kv+h)*S_kv+j for BNSD, t*N_kv+h for TND) to
 * (b, key/value head h, local j). */
static int locate_kv(const orc_params *p, int64_t id, int64_t *b, int64_t *n, int64_t *j) {
  if (id < 0) return 0;
  if (p->layout == 0) {
    *j = id % p->S_kv; *n = (id / p->S_kv) % p->N_kv; *b = id / (p->S_kv * p->N_kv);
    return *b < p->B;
  }
  int64_t t = id / p->N_kv;
  *n = id % p->N_kv;
  for (int64_t bb = 0; bb < p->B; ++bb) {
    int64_t st, len;
    seq_span(p->cu_kv, bb, &st, &len);
    if (t >= st && t < st + len) { *b = bb; *j = t - st; return 1; }
  }
  return 0;
}

static int64_t total_q_rows(const orc_params *p) { return p->layout == 0 ? p->B * p->S_q : p->T_q; }

/* ------------------------------------------------------------ exports -- */

/* Full forward: out (fp64, same layout as q), softmax_max / softmax_sum
 * ([B,N,S_q] or [T_q,N]). */
int orc_forward(const orc_params *p, const double *q, const double *k, const double *v,
                const uint8_t *mask, double *out, double *smax, double *ssum) {
  const int64_t nrows = total_q_rows(p) * p->N;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t id = 0; id < nrows; ++id) {
    int64_t b, n, i;
    if (!locate_q(p, id, &b, &n, &i)) continue;
    orc_seq s = seq_of(p, b);
    double m, l;
    forward_row(p, &s, b, n, i, q, k, v, mask, out + row_q(p, &s, b, n, i), &m, &l);
    smax[stat_q(p, &s, b, n, i)] = m;
    ssum[stat_q(p, &s, b, n, i)] = l;
  }
  return 0;
}

/* Forward for a list of query rows (flat statistics ids). */
int orc_forward_rows(const orc_params *p, const double *q, const double *k, const double *v,
                     const uint8_t *mask, int64_t nsel, const int64_t *sel, double *out, double *smax,
                     double *ssum) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < nsel; ++t) {
    int64_t b, n, i;
    if (!locate_q(p, sel[t], &b, &n, &i)) continue;
    orc_seq s = seq_of(p, b);
    forward_row(p, &s, b, n, i, q, k, v, mask, out + t * p->D, &smax[t], &ssum[t]);
  }
  return 0;
}

/* Full backward: dq, dk, dv (fp64, same layouts as q, k, v).  given_out /
 * given_max / given_sum may be NULL (exact mode: the oracle's own forward)
 * or the caller's forward results (given-stats mode). */
int orc_backward(const orc_params *p, const double *q, const double *k, const double *v, const double *dy,
                 const uint8_t *mask, const double *given_out, const double *given_max, const double *given_sum,
                 double *dq, double *dk, double *dv) {
  const int64_t D = p->D, G = p->N / p->N_kv;
  int64_t max_sq = 0;
  for (int64_t b = 0; b < p->B; ++b) { orc_seq s = seq_of(p, b); if (s.q_len > max_sq) max_sq = s.q_len; }
  row_data *rows = (row_data *)malloc(sizeof(row_data) * (size_t)(G * (max_sq > 0 ? max_sq : 1)));
  for (int64_t b = 0; b < p->B; ++b) {
    orc_seq s = seq_of(p, b);
    for (int64_t h = 0; h < p->N_kv; ++h) {
      for (int64_t gi = 0; gi < G; ++gi) {
        const int64_t n = h * G + gi;
        row_data *rg = rows + gi * s.q_len;
        /* 1) row statistics and D_i for every query of this (b, n) */
#pragma omp parallel
        {
          double *o = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 8)
          for (int64_t i = 0; i < s.q_len; ++i)
            rg[i] = backward_row_data(p, &s, b, n, i, q, k, v, dy, mask, given_out, given_max, given_sum, o);
          free(o);
        }
        /* 2) dQ rows */
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t i = 0; i < s.q_len; ++i)
          dq_row(p, &s, b, n, i, &rg[i], q, k, v, dy, mask, dq + row_q(p, &s, b, n, i));
      }
      /* 3) dK / dV columns of key/value head h, over its query heads */
#pragma omp parallel for schedule(dynamic, 8)
      for (int64_t j = 0; j < s.kv_len; ++j)
        dkv_col(p, &s, b, h, j, rows, q, k, v, dy, mask, dk + row_kv(p, &s, b, h, j), dv + row_kv(p, &s, b, h, j));
    }
  }
  free(rows);
  return 0;
}

/* dQ for a list of query rows (flat statistics ids), exact mode. */
int orc_backward_dq_rows(const orc_params *p, const double *q, const double *k, const double *v,
                         const double *dy, const uint8_t *mask, int64_t nsel, const int64_t *sel, double *dq) {
#pragma omp parallel
  {
    double *o = (double *)malloc(sizeof(double) * p->D);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < nsel; ++t) {
      int64_t b, n, i;
      for (int64_t d = 0; d < p->D; ++d) dq[t * p->D + d] = 0.0;
      if (!locate_q(p, sel[t], &b, &n, &i)) continue;
      orc_seq s = seq_of(p, b);
      row_data r = backward_row_data(p, &s, b, n, i, q, k, v, dy, mask, NULL, NULL, NULL, o);
      dq_row(p, &s, b, n, i, &r, q, k, v, dy, mask, dq + t * p->D);
    }
    free(o);
  }
  return 0;
}

/* dK / dV for a list of key rows (flat ids (b*N_kv+h)*S_kv+j or t*N_kv+h),
 * exact mode.  Computes the row data of exactly the queries that see each
 * key, in every query head of the key's group. */
int orc_backward_dkv_cols(const orc_params *p, const double *q, const double *k, const double *v,
                          const double *dy, const uint8_t *mask, int64_t nsel, const int64_t *sel, double *dk,
                          double *dv) {
  const int64_t G = p->N / p->N_kv;
  for (int64_t t = 0; t < nsel; ++t) {
    int64_t b, h, j, lo, hi;
    for (int64_t d = 0; d < p->D; ++d) { dk[t * p->D + d] = 0.0; dv[t * p->D + d] = 0.0; }
    if (!locate_kv(p, sel[t], &b, &h, &j)) continue;
    orc_seq s = seq_of(p, b);
    if (!query_range(p, &s, j, &lo, &hi)) continue;
    row_data *rows = (row_data *)calloc((size_t)(G * (s.q_len > 0 ? s.q_len : 1)), sizeof(row_data));
    for (int64_t gi = 0; gi < G; ++gi) {
      const int64_t n = h * G + gi;
#pragma omp parallel
      {
        double *o = (double *)malloc(sizeof(double) * p->D);
#pragma omp for schedule(dynamic, 8)
        for (int64_t i = lo; i <= hi; ++i)
          rows[gi * s.q_len + i] = backward_row_data(p, &s, b, n, i, q, k, v, dy, mask, NULL, NULL, NULL, o);
        free(o);
      }
    }
    dkv_col(p, &s, b, h, j, rows, q, k, v, dy, mask, dk + t * p->D, dv + t * p->D);
    free(rows);
  }
  return 0;
}

/* ------------------------------------------------- rounding budgets -- */

/* Test support, not part of what the method computes: sums of absolute
 * values that bound how far an evaluation of the same definitions may drift
 * when it rounds the operands of its matrix products to a float of unit
 * roundoff u.  Rounding every P~_ij = P_ij z_ij / keep (forward and dV) or
 * dS_ij (dQ and dK) to such a float moves, element by element over d, at
 * most by u times
 *   out_b[i] = sum_j |P~_ij| |v_j|,      dv_b[j] = sum_i |P~_ij| |dY_i|,
 *   dq_b[i]  = |scale| sum_j |dS_ij| |k_j|,  dk_b[j] = |scale| sum_i |dS_ij| |q_i|
 * (to first order: the error of a sum of rounded terms), with P and dS as
 * in the exact backward (the VarLen doc's forward formula; the PyPTO
 * article's backward formulas). */
static void budget_row(const orc_params *p, const orc_seq *s, int64_t b, int64_t n, int64_t i, const row_data *r,
                       const double *q, const double *k, const double *v, const double *dy, const uint8_t *mask,
                       double *out_b, double *dq_b) {
  const int64_t D = p->D;
  int64_t lo, hi;
  for (int64_t d = 0; d < D; ++d) { out_b[d] = 0.0; dq_b[d] = 0.0; }
  if (!key_range(p, s, i, &lo, &hi)) return;
  const double *qi = q + row_q(p, s, b, n, i);
  const double *dyi = dy + row_q(p, s, b, n, i);
  const int64_t h = kv_head(p, n);
  for (int64_t j = lo; j <= hi; ++j) {
    const double *kj = k + row_kv(p, s, b, h, j);
    const double *vj = v + row_kv(p, s, b, h, j);
    const double pij = prob(r, p->scale * dot(qi, kj, D));
    const double z = keep_bit(s, mask, n, i, j) / p->keep_prob;
    const double dsij = pij * (dot(dyi, vj, D) * z - r->Di);
    for (int64_t d = 0; d < D; ++d) {
      out_b[d] += fabs(pij * z) * fabs(vj[d]);
      dq_b[d] += fabs(p->scale) * fabs(dsij) * fabs(kj[d]);
    }
  }
}

static void budget_col(const orc_params *p, const orc_seq *s, int64_t b, int64_t h, int64_t j, const row_data *rows,
                       const double *q, const double *k, const double *v, const double *dy, const uint8_t *mask,
                       double *dk_b, double *dv_b) {
  const int64_t D = p->D, G = p->N / p->N_kv;
  int64_t lo, hi;
  for (int64_t d = 0; d < D; ++d) { dk_b[d] = 0.0; dv_b[d] = 0.0; }
  if (!query_range(p, s, j, &lo, &hi)) return;
  const double *kj = k + row_kv(p, s, b, h, j);
  const double *vj = v + row_kv(p, s, b, h, j);
  for (int64_t gi = 0; gi < G; ++gi) {
    const int64_t n = h * G + gi;
    for (int64_t i = lo; i <= hi; ++i) {
      const double *qi = q + row_q(p, s, b, n, i);
      const double *dyi = dy + row_q(p, s, b, n, i);
      const row_data *r = &rows[gi * s->q_len + i];
      const double pij = prob(r, p->scale * dot(qi, kj, D));
      const double z = keep_bit(s, mask, n, i, j) / p->keep_prob;
      const double dsij = pij * (dot(dyi, vj, D) * z - r->Di);
      for (int64_t d = 0; d < D; ++d) {
        dv_b[d] += fabs(pij * z) * fabs(dyi[d]);
        dk_b[d] += fabs(p->scale) * fabs(dsij) * fabs(qi[d]);
      }
    }
  }
}

/* The four budgets over the whole problem (fp64, the layouts of out / q and
 * of k / v), from the oracle's own forward (exact mode). */
int orc_rounding_budget(const orc_params *p, const double *q, const double *k, const double *v, const double *dy,
                        const uint8_t *mask, double *out_b, double *dq_b, double *dk_b, double *dv_b) {
  const int64_t D = p->D, G = p->N / p->N_kv;
  int64_t max_sq = 0;
  for (int64_t b = 0; b < p->B; ++b) { orc_seq s = seq_of(p, b); if (s.q_len > max_sq) max_sq = s.q_len; }
  row_data *rows = (row_data *)malloc(sizeof(row_data) * (size_t)(G * (max_sq > 0 ? max_sq : 1)));
  for (int64_t b = 0; b < p->B; ++b) {
    orc_seq s = seq_of(p, b);
    for (int64_t h = 0; h < p->N_kv; ++h) {
      for (int64_t gi = 0; gi < G; ++gi) {
        const int64_t n = h * G + gi;
        row_data *rg = rows + gi * s.q_len;
#pragma omp parallel
        {
          double *o = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 8)
          for (int64_t i = 0; i < s.q_len; ++i)
            rg[i] = backward_row_data(p, &s, b, n, i, q, k, v, dy, mask, NULL, NULL, NULL, o);
          free(o);
        }
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t i = 0; i < s.q_len; ++i)
          budget_row(p, &s, b, n, i, &rg[i], q, k, v, dy, mask, out_b + row_q(p, &s, b, n, i),
                     dq_b + row_q(p, &s, b, n, i));
      }
#pragma omp parallel for schedule(dynamic, 8)
      for (int64_t j = 0; j < s.kv_len; ++j)
        budget_col(p, &s, b, h, j, rows, q, k, v, dy, mask, dk_b + row_kv(p, &s, b, h, j),
                   dv_b + row_kv(p, &s, b, h, j));
    }
  }
  free(rows);
  return 0;
}

/* First-order error bounds of an evaluation that rounds P~ (the forward's
 * and dV's operand), dS (dQ's and dK's) and the stored output O to a float
 * of unit roundoff u, and computes everything else exactly (test support):
 *   out_e = u out_b,   dv_e = u dv_b,
 *   dq_e[i] = u dq_b[i] + |scale| dD_i sum_j P_ij |k_j|,
 *   dk_e[j] = u dk_b[j] + |scale| sum_i dD_i P_ij |q_i|,
 * where dD_i = u sum_d |dY_id| (out_b[i,d] + |O_id|) bounds the error of
 * D_i = dY_i . O_i formed from that O (its operand-rounding error plus its
 * own rounding), and dS_ij moves by -P_ij times it. */
static double row_dD(const orc_params *p, const orc_seq *s, int64_t b, int64_t n, int64_t i, const row_data *r,
                     const double *q, const double *k, const double *v, const double *dy, const uint8_t *mask,
                     double u, double *o, double *ob, double *scratch) {
  const int64_t D = p->D;
  double m, l;
  forward_row(p, s, b, n, i, q, k, v, mask, o, &m, &l);
  budget_row(p, s, b, n, i, r, q, k, v, dy, mask, ob, scratch);
  const double *dyi = dy + row_q(p, s, b, n, i);
  double acc = 0.0;
  for (int64_t d = 0; d < D; ++d) acc += fabs(dyi[d]) * (ob[d] + fabs(o[d]));
  return u * acc;
}

int orc_rounding_error(const orc_params *p, const double *q, const double *k, const double *v, const double *dy,
                       const uint8_t *mask, double u, double *out_e, double *dq_e, double *dk_e, double *dv_e) {
  const int64_t D = p->D, G = p->N / p->N_kv;
  orc_rounding_budget(p, q, k, v, dy, mask, out_e, dq_e, dk_e, dv_e);
  const int64_t nq = total_q_rows(p) * p->N, nk = (p->layout == 0 ? p->B * p->S_kv : p->T_kv) * p->N_kv;
  for (int64_t t = 0; t < nq * D; ++t) { out_e[t] *= u; dq_e[t] *= u; }
  for (int64_t t = 0; t < nk * D; ++t) { dk_e[t] *= u; dv_e[t] *= u; }
  int64_t max_sq = 0;
  for (int64_t b = 0; b < p->B; ++b) { orc_seq s = seq_of(p, b); if (s.q_len > max_sq) max_sq = s.q_len; }
  const size_t nrows = (size_t)(G * (max_sq > 0 ? max_sq : 1));
  row_data *rows = (row_data *)malloc(sizeof(row_data) * nrows);
  double *dD = (double *)malloc(sizeof(double) * nrows);
  for (int64_t b = 0; b < p->B; ++b) {
    orc_seq s = seq_of(p, b);
    for (int64_t h = 0; h < p->N_kv; ++h) {
      for (int64_t gi = 0; gi < G; ++gi) {
        const int64_t n = h * G + gi;
        row_data *rg = rows + gi * s.q_len;
        double *dg = dD + gi * s.q_len;
#pragma omp parallel
        {
          double *o = (double *)malloc(sizeof(double) * D);
          double *ob = (double *)malloc(sizeof(double) * D);
          double *sc = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 8)
          for (int64_t i = 0; i < s.q_len; ++i) {
            rg[i] = backward_row_data(p, &s, b, n, i, q, k, v, dy, mask, NULL, NULL, NULL, o);
            dg[i] = row_dD(p, &s, b, n, i, &rg[i], q, k, v, dy, mask, u, o, ob, sc);
          }
          free(o); free(ob); free(sc);
        }
        /* dQ_i moves by -scale dD_i sum_j P_ij k_j */
#pragma omp parallel for schedule(dynamic, 8)
        for (int64_t i = 0; i < s.q_len; ++i) {
          int64_t lo, hi;
          if (!key_range(p, &s, i, &lo, &hi)) continue;
          const double *qi = q + row_q(p, &s, b, n, i);
          double *e = dq_e + row_q(p, &s, b, n, i);
          for (int64_t j = lo; j <= hi; ++j) {
            const double *kj = k + row_kv(p, &s, b, h, j);
            const double pij = prob(&rg[i], p->scale * dot(qi, kj, D));
            for (int64_t d = 0; d < D; ++d) e[d] += fabs(p->scale) * dg[i] * pij * fabs(kj[d]);
          }
        }
      }
      /* dK_j moves by -scale sum_i dD_i P_ij q_i, over the group's query heads */
#pragma omp parallel for schedule(dynamic, 8)
      for (int64_t j = 0; j < s.kv_len; ++j) {
        int64_t lo, hi;
        if (!query_range(p, &s, j, &lo, &hi)) continue;
        const double *kj = k + row_kv(p, &s, b, h, j);
        double *e = dk_e + row_kv(p, &s, b, h, j);
        for (int64_t gi = 0; gi < G; ++gi) {
          const int64_t n = h * G + gi;
          for (int64_t i = lo; i <= hi; ++i) {
            const double *qi = q + row_q(p, &s, b, n, i);
            const double pij = prob(&rows[gi * s.q_len + i], p->scale * dot(qi, kj, D));
            for (int64_t d = 0; d < D; ++d) e[d] += fabs(p->scale) * dD[gi * s.q_len + i] * pij * fabs(qi[d]);
          }
        }
      }
    }
  }
  free(rows);
  free(dD);
  return 0;
}

/* ------------------------------------------------ generated dropout -- */

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplications by
 * 0xD2511F53 and 0xCD9E8D57 on counter words 0 and 2; the new counter is
 * (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)); the key is
 * bumped by (0x9E3779B9, 0xBB67AE85) after every round. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
    const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n1 = (uint32_t)p1;
    const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1, n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The keep mask a seed / offset pair stands for, written in the packed
 * element order of the drop_mask input (bit e of byte e>>3, LSB first).
 * Element (query row r = statistics id, local key j) keeps iff
 *   byte (j mod 16) of Philox4x32-10(counter = (j/16, lo32 r, hi32 r,
 *   lo32 offset), key = (lo32 seed, hi32 seed)) < threshold,
 * bytes taken little-endian across the four output words, threshold =
 * round(keep_prob * 256) in [0, 256]. */
int orc_generate_keep_mask(const orc_params *p, uint64_t seed, uint64_t offset, uint8_t *mask) {
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  long thr = lround(p->keep_prob * 256.0);
  if (thr < 0) thr = 0;
  if (thr > 256) thr = 256;
  for (int64_t b = 0; b < p->B; ++b) {
    orc_seq s = seq_of(p, b);
    for (int64_t n = 0; n < p->N; ++n)
      for (int64_t i = 0; i < s.q_len; ++i) {
        const int64_t r = stat_q(p, &s, b, n, i);
        for (int64_t j = 0; j < s.kv_len; ++j) {
          const uint32_t ctr[4] = {(uint32_t)(j >> 4), (uint32_t)r, (uint32_t)((uint64_t)r >> 32), (uint32_t)offset};
          uint32_t o[4];
          orc_philox4x32_10(ctr, key, o);
          const uint32_t byte = (o[(j & 15) >> 2] >> (8 * (j & 3))) & 0xFFu;
          const int64_t e = s.mask_base + (n * s.q_len + i) * s.kv_len + j;
          if ((long)byte < thr) mask[e >> 3] |= (uint8_t)(1u << (e & 7));
          else mask[e >> 3] &= (uint8_t)~(1u << (e & 7));
        }
      }
  }
  return 0;
}

/* Visible key range [lo, hi] of each query row (flat statistics ids); lo > hi
 * for an empty row.  Used to compare masked sets exactly. */
int orc_key_ranges(const orc_params *p, int64_t nsel, const int64_t *sel, int64_t *lo, int64_t *hi) {
  for (int64_t t = 0; t < nsel; ++t) {
    int64_t b, n, i;
    lo[t] = 0; hi[t] = -1;
    if (!locate_q(p, sel[t], &b, &n, &i)) continue;
    orc_seq s = seq_of(p, b);
    if (!key_range(p, &s, i, &lo[t], &hi[t])) { lo[t] = 0; hi[t] = -1; }
  }
  return 0;
}
