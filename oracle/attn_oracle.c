/*
 * Oracle for non-causal DiT self-attention, its KV-chunk decomposition and the
 * log-sum-exp merge of chunk partials.  TEST INFRASTRUCTURE ONLY: it is used by
 * the tests, by the smoke check and by the bench's CPU-baseline leg, never by
 * the product path.  It shares no code, header or constant with the CUDA path.
 *
 * Everything is computed in IEEE fp64 with plain loops, in the order of the
 * definitions below; there is no blocking, no online softmax and no fusion.
 *
 * Definitions followed:
 *  - Attention per head (b, h), query row i, over key rows j of one KV range:
 *        s_ij  = scale * sum_d q_id k_jd
 *        m_i   = max_j s_ij
 *        l_i   = sum_j exp(s_ij - m_i)
 *        lse_i = m_i + ln l_i                      (natural log of the scaled scores)
 *        o_id  = sum_j exp(s_ij - m_i) v_jd / l_i
 *    Source: MindIE-SD parallelism docs, "Ring Sequence Parallel" usage example
 *    (local_attn: scores q.k^T / sqrt(dim), softmax over keys, times v);
 *    arganzheng.life multi-GPU diffusion parallelism, section 4.1 Ulysses (each
 *    head does full attention over all N tokens); "AIGC distributed inference:
 *    understanding DP/TP/CP/SP/PP from Wan2.2", Ulysses section (heads are
 *    independent, tokens are not).  Subtracting m_i is the usual exact rewrite
 *    of softmax; it changes nothing but the range of the exponentials.
 *  - A KV chunk (one virtual ring rank) is the same formula with j restricted
 *    to that chunk's rows.  Source: arganzheng.life, section 4.2 Ring (round i
 *    uses the K/V block of rank (r+i) mod p; after p rounds every query has
 *    seen all keys).
 *  - Merge of p partials (O_c, lse_c) of one query row:
 *        M   = max_c lse_c
 *        lse = M + ln sum_c exp(lse_c - M)
 *        o   = sum_c exp(lse_c - lse) o_c
 *    This is the exact combination of per-chunk softmaxes that the Ring
 *    section's "online softmax accumulation" over rounds implies.  A chunk with
 *    lse_c = -inf contributes nothing; if every lse_c is -inf the row is o = 0,
 *    lse = -inf.  (The MindIE Ring usage example adds normalised per-chunk
 *    outputs, out += local_attn(...); that sum is not attention and is not
 *    followed here.)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const uint16_t *q, *k, *v;
  int64_t bh_count, n_q, n_kv, d;
  int64_t q_head_stride, kv_head_stride;
  double scale;
  const int64_t *rows; /* NULL: all rows 0..n_q-1 */
  int64_t n_rows;
  double *out, *lse;
  int64_t item_begin, item_end; /* items are (bh, row) pairs, row-major */
  int status;
} attn_job;

static void attention_row(const attn_job *j, int64_t bh, int64_t qi, double *o, double *lse_out,
                          double *s, double *qrow) {
  const int64_t D = j->d, n = j->n_kv;
  const uint16_t *qp = j->q + bh * j->q_head_stride + qi * D;
  const uint16_t *kb = j->k + bh * j->kv_head_stride;
  const uint16_t *vb = j->v + bh * j->kv_head_stride;
  for (int64_t d = 0; d < D; ++d) qrow[d] = bf16_to_f64(qp[d]);

  /* scores */
  for (int64_t kj = 0; kj < n; ++kj) {
    const uint16_t *kp = kb + kj * D;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d) dot += qrow[d] * bf16_to_f64(kp[d]);
    s[kj] = j->scale * dot;
  }
  /* max */
  double m = -INFINITY;
  for (int64_t kj = 0; kj < n; ++kj)
    if (s[kj] > m) m = s[kj];
  /* unnormalised weights and their sum */
  double l = 0.0;
  for (int64_t kj = 0; kj < n; ++kj) {
    s[kj] = exp(s[kj] - m);
    l += s[kj];
  }
  /* weighted sum of values, then normalise */
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int64_t kj = 0; kj < n; ++kj) {
    const uint16_t *vp = vb + kj * D;
    const double w = s[kj];
    for (int64_t d = 0; d < D; ++d) o[d] += w * bf16_to_f64(vp[d]);
  }
  for (int64_t d = 0; d < D; ++d) o[d] /= l;
  *lse_out = m + log(l);
}

static void *attention_worker(void *arg) {
  attn_job *j = (attn_job *)arg;
  double *s = (double *)malloc(sizeof(double) * (size_t)(j->n_kv > 0 ? j->n_kv : 1));
  double *qrow = (double *)malloc(sizeof(double) * (size_t)j->d);
  if (!s || !qrow) {
    j->status = -2;
    free(s);
    free(qrow);
    return NULL;
  }
  for (int64_t it = j->item_begin; it < j->item_end; ++it) {
    const int64_t bh = it / j->n_rows, r = it % j->n_rows;
    const int64_t qi = j->rows ? j->rows[r] : r;
    attention_row(j, bh, qi, j->out + it * j->d, j->lse + it, s, qrow);
  }
  free(s);
  free(qrow);
  j->status = 0;
  return NULL;
}

static int clamp_threads(int nthreads, int64_t items) {
  if (nthreads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = c > 0 ? (int)c : 1;
  }
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > items) nthreads = (int)(items > 0 ? items : 1);
  return nthreads;
}

/*
 * Attention of every listed query row against key/value rows [0, n_kv).
 *  q: bf16 bits, head (b*H+h) at q + bh*q_head_stride, row i at + i*d.
 *  k, v: bf16 bits, head at + bh*kv_head_stride, row j at + j*d (a chunk is
 *        passed as pointers already offset to its first row).
 *  rows: n_rows query indices (or NULL with n_rows == n_q for all rows).
 *  out: fp64 [bh_count][n_rows][d];  lse: fp64 [bh_count][n_rows].
 *  nthreads <= 0 uses every online core.  Returns 0, or -1 on bad arguments,
 *  -2 if a worker could not allocate.
 */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t bh_count,
                     int64_t n_q, int64_t n_kv, int64_t d, int64_t q_head_stride,
                     int64_t kv_head_stride, double scale, const int64_t *rows, int64_t n_rows,
                     double *out, double *lse, int nthreads) {
  if (!q || !k || !v || !out || !lse || bh_count < 1 || n_q < 1 || n_kv < 1 || d < 1) return -1;
  if (!rows && n_rows != n_q) return -1;
  if (rows)
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= n_q) return -1;
  const int64_t items = bh_count * n_rows;
  nthreads = clamp_threads(nthreads, items);
  attn_job *jobs = (attn_job *)calloc((size_t)nthreads, sizeof(attn_job));
  pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return -2;
  }
  for (int t = 0; t < nthreads; ++t) {
    attn_job *j = &jobs[t];
    j->q = q; j->k = k; j->v = v;
    j->bh_count = bh_count; j->n_q = n_q; j->n_kv = n_kv; j->d = d;
    j->q_head_stride = q_head_stride; j->kv_head_stride = kv_head_stride;
    j->scale = scale; j->rows = rows; j->n_rows = n_rows; j->out = out; j->lse = lse;
    j->item_begin = items * t / nthreads;
    j->item_end = items * (t + 1) / nthreads;
    j->status = -2;
  }
  int rc = 0;
  for (int t = 1; t < nthreads; ++t)
    if (pthread_create(&tids[t], NULL, attention_worker, &jobs[t]) != 0) {
      attention_worker(&jobs[t]); /* run inline if a thread cannot start */
      tids[t] = 0;
    }
  attention_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (tids[t]) pthread_join(tids[t], NULL);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != 0) rc = jobs[t].status;
  free(jobs);
  free(tids);
  return rc;
}

/*
 * Merge of p chunk partials for `rows` independent query rows.
 *  partials: fp64 [p][rows][d];  lses: fp64 [p][rows]
 *  out: fp64 [rows][d];          lse: fp64 [rows]
 */
int oracle_lse_merge(const double *partials, const double *lses, int64_t p, int64_t rows,
                     int64_t d, double *out, double *lse) {
  if (!partials || !lses || !out || !lse || p < 1 || rows < 1 || d < 1) return -1;
  for (int64_t r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int64_t c = 0; c < p; ++c)
      if (lses[c * rows + r] > M) M = lses[c * rows + r];
    double *o = out + r * d;
    for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int64_t c = 0; c < p; ++c) sum += exp(lses[c * rows + r] - M);
    const double L = M + log(sum);
    for (int64_t c = 0; c < p; ++c) {
      const double w = exp(lses[c * rows + r] - L);
      const double *oc = partials + (c * rows + r) * d;
      for (int64_t e = 0; e < d; ++e) o[e] += w * oc[e];
    }
    lse[r] = L;
  }
  return 0;
}

/* Number of worker threads oracle_attention would start for `nthreads`. */
int oracle_threads_used(int nthreads, int64_t items) { return clamp_threads(nthreads, items); }
