/*
 * attn_oracle.c -- float64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * What it computes is the plain definition of attention, written out without
 * tiling, fusion or reordering:
 *
 *   S = scale * Q K^T        [FlashAttention深度攻略 §2 (standard attention);
 *                             FlashAttention (PKM page), "standard attention, IO view"]
 *   S_ij = -inf where causal and j > i
 *                            [FlashAttention深度攻略, live-coding section,
 *                             standard_attention: upper-triangular mask above the
 *                             diagonal, i.e. key j hidden from query i iff j > i]
 *   P = row softmax of S with the row max subtracted
 *                            [FlashAttention深度攻略 §4, numerically stable softmax]
 *   O = P V
 *   LSE_i = m_i + ln sum_j exp(S_ij - m_i)
 *                            [the single per-row statistic kept in place of (m, l):
 *                             FlashAttention (PKM page) §3 Recomputation;
 *                             FlashAttention深度攻略 §6]
 *
 * and the analytic backward of L = <O, dO> [FlashAttention深度攻略 §6, the
 * recomputation backward; its printed dQ formula is garbled, so the standard
 * derivation is used]:
 *
 *   dP = dO V^T,  D_i = sum_k dO_ik O_ik,  dS = P o (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 *
 * Layout: every [B,H,N,d] tensor is row-major float64, viewed as BH = B*H
 * independent heads of [N][d]; lse is [BH][N].
 *
 * Block-sparse variant (FlashAttention深度攻略, 进阶追问 "Sparse FlashAttention"
 * and its note separating tiling from block-sparse attention): an optional
 * mask [mask_heads][nb][nb] of bytes, head h using mask h % mask_heads, hides
 * key j from query i unless mask[i / blk][j / blk] != 0 (on top of the causal
 * rule).  A row that sees no key at all has O = 0 and LSE = -inf.
 *
 * Work is spread over threads by (head, block of rows) or (head, block of key
 * columns); each row or column is computed exactly as the definition reads,
 * so threading changes no arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ROWS_PER_ITEM 16

typedef struct {
  const double *q, *k, *v, *o, *dO, *lse, *Dvec;
  double *o_out, *lse_out, *p_out, *dq, *dk, *dv;
  double *P_head, *dS_head; /* per-head N x N scratch (backward only) */
  int64_t BH, N, d;
  double scale;
  int causal;
  /* optional block mask */
  const uint8_t *bmask;
  int64_t mask_heads, nb, blk;
  /* sampled rows / columns */
  const int64_t *bh_idx, *idx;
  int64_t nsel;
  /* work distribution */
  int64_t nitems;
  int64_t next;
  pthread_mutex_t mu;
  int head; /* current head for per-head phases */
} job_t;

static int64_t take_item(job_t *j) {
  pthread_mutex_lock(&j->mu);
  int64_t it = j->next++;
  pthread_mutex_unlock(&j->mu);
  return it < j->nitems ? it : -1;
}

static int run_threads(void *(*fn)(void *), job_t *j, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, fn, j) != 0) break;
    started = t;
  }
  fn(j);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  return 0;
}

/* Visibility rule of one query row: causal flag and (optional) its row of the block mask. */
typedef struct {
  int causal;
  const uint8_t *mrow; /* mask row of query i's block (nb entries) or NULL */
  int64_t blk;
} vis_t;

/* Is key j visible to query i? */
static int visible(vis_t v, int64_t i, int64_t j) {
  return (!v.causal || j <= i) && (!v.mrow || v.mrow[j / v.blk]);
}

static vis_t vis_for(const job_t *J, int64_t h, int64_t i) {
  vis_t v;
  v.causal = J->causal;
  v.blk = J->blk;
  v.mrow = J->bmask ? J->bmask + ((h % J->mask_heads) * J->nb + i / J->blk) * J->nb : NULL;
  return v;
}

/* One query row of one head, materialising its row of S and P.
 * s_row, p_row: scratch of length N.  Writes o_row[d], *lse_out, and p_row. */
static void forward_row(const double *qh, const double *kh, const double *vh, int64_t N,
                        int64_t d, double scale, vis_t vis, int64_t i, double *s_row,
                        double *p_row, double *o_row, double *lse_out) {
  const double *qi = qh + i * d;
  double m = -INFINITY;
  for (int64_t j = 0; j < N; ++j) {
    if (!visible(vis, i, j)) {
      s_row[j] = -INFINITY;
      continue;
    }
    const double *kj = kh + j * d;
    double acc = 0.0;
    for (int64_t c = 0; c < d; ++c) acc += qi[c] * kj[c];
    s_row[j] = scale * acc;
    if (s_row[j] > m) m = s_row[j];
  }
  if (m == -INFINITY) { /* no visible key: O = 0, LSE = -inf */
    for (int64_t j = 0; j < N; ++j) p_row[j] = 0.0;
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    *lse_out = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int64_t j = 0; j < N; ++j) {
    p_row[j] = (s_row[j] == -INFINITY) ? 0.0 : exp(s_row[j] - m);
    l += p_row[j];
  }
  for (int64_t j = 0; j < N; ++j) p_row[j] /= l;
  for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
  for (int64_t j = 0; j < N; ++j) {
    if (p_row[j] == 0.0) continue;
    const double *vj = vh + j * d;
    for (int64_t c = 0; c < d; ++c) o_row[c] += p_row[j] * vj[c];
  }
  *lse_out = m + log(l);
}

/* ---------------------------------------------------------------- forward */

static void *fwd_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int64_t N = J->N, d = J->d;
  const int64_t blocks = (N + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
  double *s_row = (double *)malloc(sizeof(double) * N);
  double *p_tmp = (double *)malloc(sizeof(double) * N);
  for (int64_t it; (it = take_item(J)) >= 0;) {
    const int64_t h = it / blocks, rb = it % blocks;
    const double *qh = J->q + h * N * d, *kh = J->k + h * N * d, *vh = J->v + h * N * d;
    for (int64_t i = rb * ROWS_PER_ITEM; i < N && i < (rb + 1) * ROWS_PER_ITEM; ++i) {
      double *p_row = J->p_out ? J->p_out + (h * N + i) * N : p_tmp;
      forward_row(qh, kh, vh, N, d, J->scale, vis_for(J, h, i), i, s_row, p_row,
                  J->o_out + (h * N + i) * d, J->lse_out + h * N + i);
    }
  }
  free(s_row);
  free(p_tmp);
  return NULL;
}

/* O = softmax(scale Q K^T [+ causal mask]) V and LSE for all heads.
 * p_out: optional [BH][N][N] probabilities (NULL to skip). */
int oracle_forward_masked(const double *q, const double *k, const double *v, double *o,
                          double *lse, double *p_out, int64_t BH, int64_t N, int64_t d,
                          double scale, int causal, const uint8_t *bmask, int64_t mask_heads,
                          int64_t blk, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !o || !lse) return 1;
  if (bmask && (mask_heads < 1 || blk < 1)) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.bmask = bmask; J.mask_heads = mask_heads; J.blk = blk > 0 ? blk : 1;
  J.nb = (N + J.blk - 1) / J.blk;
  J.q = q; J.k = k; J.v = v; J.o_out = o; J.lse_out = lse; J.p_out = p_out;
  J.BH = BH; J.N = N; J.d = d; J.scale = scale; J.causal = causal;
  J.nitems = BH * ((N + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM);
  pthread_mutex_init(&J.mu, NULL);
  run_threads(fwd_worker, &J, nthreads);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

int oracle_forward(const double *q, const double *k, const double *v, double *o, double *lse,
                   double *p_out, int64_t BH, int64_t N, int64_t d, double scale, int causal,
                   int nthreads) {
  return oracle_forward_masked(q, k, v, o, lse, p_out, BH, N, d, scale, causal, NULL, 0, 0,
                               nthreads);
}

/* --------------------------------------------------------------- backward */

/* Phase 1 (rows of one head): P row, dP row, D_i, dS row, dQ row. */
static void *bwd_rows_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int64_t N = J->N, d = J->d, h = J->head;
  const double *qh = J->q + h * N * d, *kh = J->k + h * N * d, *vh = J->v + h * N * d;
  const double *oh = J->o + h * N * d, *doh = J->dO + h * N * d;
  double *s_row = (double *)malloc(sizeof(double) * N);
  double *o_row = (double *)malloc(sizeof(double) * d);
  for (int64_t it; (it = take_item(J)) >= 0;) {
    for (int64_t i = it * ROWS_PER_ITEM; i < N && i < (it + 1) * ROWS_PER_ITEM; ++i) {
      double *p_row = J->P_head + i * N, *ds_row = J->dS_head + i * N;
      double lse_unused;
      forward_row(qh, kh, vh, N, d, J->scale, vis_for(J, h, i), i, s_row, p_row, o_row, &lse_unused);
      const double *doi = doh + i * d, *oi = oh + i * d;
      double Di = 0.0;
      for (int64_t c = 0; c < d; ++c) Di += doi[c] * oi[c];
      for (int64_t j = 0; j < N; ++j) {
        if (p_row[j] == 0.0) { ds_row[j] = 0.0; continue; }
        const double *vj = vh + j * d;
        double dp = 0.0;
        for (int64_t c = 0; c < d; ++c) dp += doi[c] * vj[c];
        ds_row[j] = p_row[j] * (dp - Di);
      }
      double *dqi = J->dq + (h * N + i) * d;
      for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
      for (int64_t j = 0; j < N; ++j) {
        if (ds_row[j] == 0.0) continue;
        const double *kj = kh + j * d;
        for (int64_t c = 0; c < d; ++c) dqi[c] += ds_row[j] * kj[c];
      }
      for (int64_t c = 0; c < d; ++c) dqi[c] *= J->scale;
    }
  }
  free(s_row);
  free(o_row);
  return NULL;
}

/* Phase 2 (key columns of one head): dV_j = sum_i P_ij dO_i, dK_j = scale sum_i dS_ij Q_i. */
static void *bwd_cols_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int64_t N = J->N, d = J->d, h = J->head;
  const double *qh = J->q + h * N * d, *doh = J->dO + h * N * d;
  for (int64_t it; (it = take_item(J)) >= 0;) {
    for (int64_t j = it * ROWS_PER_ITEM; j < N && j < (it + 1) * ROWS_PER_ITEM; ++j) {
      double *dvj = J->dv + (h * N + j) * d, *dkj = J->dk + (h * N + j) * d;
      for (int64_t c = 0; c < d; ++c) { dvj[c] = 0.0; dkj[c] = 0.0; }
      for (int64_t i = 0; i < N; ++i) {
        const double p = J->P_head[i * N + j], ds = J->dS_head[i * N + j];
        const double *doi = doh + i * d, *qi = qh + i * d;
        if (p != 0.0)
          for (int64_t c = 0; c < d; ++c) dvj[c] += p * doi[c];
        if (ds != 0.0)
          for (int64_t c = 0; c < d; ++c) dkj[c] += ds * qi[c];
      }
      for (int64_t c = 0; c < d; ++c) dkj[c] *= J->scale;
    }
  }
  return NULL;
}

/* Analytic backward.  o must be the forward output of the same inputs (the
 * oracle's own float64 O).  Materialises P and dS one head at a time
 * (2 * N * N doubles). */
int oracle_backward_masked(const double *q, const double *k, const double *v, const double *o,
                           const double *dO, double *dq, double *dk, double *dv, int64_t BH,
                           int64_t N, int64_t d, double scale, int causal, const uint8_t *bmask,
                           int64_t mask_heads, int64_t blk, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !o || !dO || !dq || !dk || !dv) return 1;
  if (bmask && (mask_heads < 1 || blk < 1)) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.bmask = bmask; J.mask_heads = mask_heads; J.blk = blk > 0 ? blk : 1;
  J.nb = (N + J.blk - 1) / J.blk;
  J.q = q; J.k = k; J.v = v; J.o = o; J.dO = dO; J.dq = dq; J.dk = dk; J.dv = dv;
  J.BH = BH; J.N = N; J.d = d; J.scale = scale; J.causal = causal;
  J.P_head = (double *)malloc(sizeof(double) * N * N);
  J.dS_head = (double *)malloc(sizeof(double) * N * N);
  if (!J.P_head || !J.dS_head) { free(J.P_head); free(J.dS_head); return 2; }
  pthread_mutex_init(&J.mu, NULL);
  const int64_t blocks = (N + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
  for (int64_t h = 0; h < BH; ++h) {
    J.head = (int)h;
    J.nitems = blocks; J.next = 0;
    run_threads(bwd_rows_worker, &J, nthreads);
    J.nitems = blocks; J.next = 0;
    run_threads(bwd_cols_worker, &J, nthreads);
  }
  pthread_mutex_destroy(&J.mu);
  free(J.P_head);
  free(J.dS_head);
  return 0;
}

int oracle_backward(const double *q, const double *k, const double *v, const double *o,
                    const double *dO, double *dq, double *dk, double *dv, int64_t BH, int64_t N,
                    int64_t d, double scale, int causal, int nthreads) {
  return oracle_backward_masked(q, k, v, o, dO, dq, dk, dv, BH, N, d, scale, causal, NULL, 0, 0,
                                nthreads);
}

/* ------------------------------------------------------- sampled query rows */

/* For each selected (head, row) pair: O row, LSE and dQ row, straight from the
 * definition (D_i uses the oracle's own O row).  Cost O(N d) per row, so it
 * scales to sequence lengths where a whole head cannot be materialised.
 * o_rows/dq_rows: [nsel][d]; lse_rows: [nsel]; dq_rows may be NULL. */
static void *rows_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int64_t N = J->N, d = J->d;
  double *s_row = (double *)malloc(sizeof(double) * N);
  double *p_row = (double *)malloc(sizeof(double) * N);
  for (int64_t r; (r = take_item(J)) >= 0;) {
    const int64_t h = J->bh_idx[r], i = J->idx[r];
    const double *qh = J->q + h * N * d, *kh = J->k + h * N * d, *vh = J->v + h * N * d;
    double *oi = J->o_out + r * d;
    forward_row(qh, kh, vh, N, d, J->scale, vis_for(J, h, i), i, s_row, p_row, oi, J->lse_out + r);
    if (!J->dq) continue;
    const double *doi = J->dO + (h * N + i) * d;
    double Di = 0.0;
    for (int64_t c = 0; c < d; ++c) Di += doi[c] * oi[c];
    double *dqi = J->dq + r * d;
    for (int64_t c = 0; c < d; ++c) dqi[c] = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      if (p_row[j] == 0.0) continue;
      const double *vj = vh + j * d, *kj = kh + j * d;
      double dp = 0.0;
      for (int64_t c = 0; c < d; ++c) dp += doi[c] * vj[c];
      const double ds = p_row[j] * (dp - Di);
      for (int64_t c = 0; c < d; ++c) dqi[c] += ds * kj[c];
    }
    for (int64_t c = 0; c < d; ++c) dqi[c] *= J->scale;
  }
  free(s_row);
  free(p_row);
  return NULL;
}

int oracle_rows(const double *q, const double *k, const double *v, const double *dO,
                int64_t BH, int64_t N, int64_t d, double scale, int causal,
                const int64_t *bh_idx, const int64_t *row_idx, int64_t nsel, double *o_rows,
                double *lse_rows, double *dq_rows, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !bh_idx || !row_idx || !o_rows || !lse_rows)
    return 1;
  if (dq_rows && !dO) return 1;
  for (int64_t r = 0; r < nsel; ++r)
    if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= N) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.dO = dO; J.o_out = o_rows; J.lse_out = lse_rows; J.dq = dq_rows;
  J.BH = BH; J.N = N; J.d = d; J.scale = scale; J.causal = causal;
  J.bh_idx = bh_idx; J.idx = row_idx; J.nsel = nsel; J.nitems = nsel;
  pthread_mutex_init(&J.mu, NULL);
  run_threads(rows_worker, &J, nthreads);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

/* ----------------------------------------------------- sampled key columns */

/* For each selected (head, key) pair: dK and dV rows.  Needs every row's LSE
 * and D_i = sum_k dO_ik O_ik of that head (from oracle_rows or
 * oracle_forward), so that P_ij = exp(S_ij - LSE_i) is the definition's
 * probability.  lse_all, D_all: [BH][N]; dk_rows/dv_rows: [nsel][d]. */
static void *cols_worker(void *arg) {
  job_t *J = (job_t *)arg;
  const int64_t N = J->N, d = J->d;
  for (int64_t r; (r = take_item(J)) >= 0;) {
    const int64_t h = J->bh_idx[r], j = J->idx[r];
    const double *qh = J->q + h * N * d, *kj = J->k + (h * N + j) * d,
                 *vj = J->v + (h * N + j) * d, *doh = J->dO + h * N * d;
    double *dkj = J->dk + r * d, *dvj = J->dv + r * d;
    for (int64_t c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
    for (int64_t i = 0; i < N; ++i) {
      if (!visible(vis_for(J, h, i), i, j)) continue;
      const double *qi = qh + i * d, *doi = doh + i * d;
      double acc = 0.0, dp = 0.0;
      for (int64_t c = 0; c < d; ++c) { acc += qi[c] * kj[c]; dp += doi[c] * vj[c]; }
      const double p = exp(J->scale * acc - J->lse[h * N + i]);
      const double ds = p * (dp - J->Dvec[h * N + i]);
      for (int64_t c = 0; c < d; ++c) { dvj[c] += p * doi[c]; dkj[c] += ds * qi[c]; }
    }
    for (int64_t c = 0; c < d; ++c) dkj[c] *= J->scale;
  }
  return NULL;
}

int oracle_cols(const double *q, const double *k, const double *v, const double *dO,
                const double *lse_all, const double *D_all, int64_t BH, int64_t N, int64_t d,
                double scale, int causal, const int64_t *bh_idx, const int64_t *col_idx,
                int64_t nsel, double *dk_rows, double *dv_rows, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !dO || !lse_all || !D_all || !bh_idx ||
      !col_idx || !dk_rows || !dv_rows)
    return 1;
  for (int64_t r = 0; r < nsel; ++r)
    if (bh_idx[r] < 0 || bh_idx[r] >= BH || col_idx[r] < 0 || col_idx[r] >= N) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  J.q = q; J.k = k; J.v = v; J.dO = dO; J.lse = lse_all; J.Dvec = D_all;
  J.dk = dk_rows; J.dv = dv_rows;
  J.BH = BH; J.N = N; J.d = d; J.scale = scale; J.causal = causal;
  J.bh_idx = bh_idx; J.idx = col_idx; J.nsel = nsel; J.nitems = nsel;
  pthread_mutex_init(&J.mu, NULL);
  run_threads(cols_worker, &J, nthreads);
  pthread_mutex_destroy(&J.mu);
  return 0;
}
