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
 * Dropout variant (FlashAttention深度攻略 §7, operator fusion: the softmax
 * step of the fused kernel also applies dropout).  The pages name the step
 * and nothing more, so the usual inverted dropout on the attention
 * probabilities is taken:
 *
 *   O_i   = sum_j  keep_ij * (256 / t) * P_ij * V_j       (P undropped softmax)
 *   LSE_i = log sum_j exp(S_ij)                           (statistics undropped)
 *   dV_j  = sum_i  keep_ij * (256 / t) * P_ij * dO_i
 *   dP_ij = keep_ij * (256 / t) * dO_i . V_j,   D_i = dO_i . O_i,
 *   dS    = P o (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
 *
 * keep_ij is 1 iff the byte u_ij < t, where t = floor((1 - p) * 256 + 0.5)
 * (the keep probability rounded to a multiple of 1/256, 1 <= t <= 256) and
 * u_ij is byte (j mod 4) of word floor((j mod 16) / 4) of
 *   Philox4x32-10(counter = (floor(j / 16), i, bh, offset), key = (seed lo, seed hi))
 * -- the counter-based generator of Salmon, Moraes, Dror and Shaw, "Parallel
 * Random Numbers: As Easy as 1, 2, 3" (SC'11): ten rounds of two 32x32->64
 * bit multiplies with a Weyl-sequence key schedule.  One call yields the
 * bytes of 16 consecutive keys of one query row.
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

/* ---------------------------------------------------------------- Philox */

/* Philox4x32 with 10 rounds (Salmon et al., SC'11): each round multiplies
 * words 0 and 2 by the two round multipliers, takes the high halves XORed
 * with the other two words and the round key, and permutes; the key advances
 * by the Weyl constants (golden ratio and sqrt(3) - 1, as 32-bit fractions)
 * between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint64_t p0 = (uint64_t)0xD2511F53u * x0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
    x0 = y0;
    x1 = lo1;
    x2 = y2;
    x3 = lo0;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Dropout parameters: on = 0 disables dropout entirely. */
typedef struct {
  int on;
  uint32_t t;      /* keep iff byte < t, 1 <= t <= 256 */
  uint32_t key[2]; /* seed, low and high words */
  uint32_t offset;
  double rscale;   /* 256 / t */
} drop_t;

/* The dropout byte u_ij of head bh. */
static uint32_t drop_byte(const drop_t *dr, int64_t bh, int64_t i, int64_t j) {
  const uint32_t ctr[4] = {(uint32_t)(j >> 4), (uint32_t)i, (uint32_t)bh, dr->offset};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, dr->key, out);
  return (out[(j & 15) >> 2] >> (8 * (j & 3))) & 0xFFu;
}

/* Weight the dropout gives P_ij: 0 (dropped), 256 / t (kept), 1 without dropout. */
static double drop_weight(const drop_t *dr, int64_t bh, int64_t i, int64_t j) {
  if (!dr->on) return 1.0;
  return drop_byte(dr, bh, i, j) < dr->t ? dr->rscale : 0.0;
}

/* p in [0, 1) -> keep threshold t in [1, 256]; 0 when p is out of range. */
static uint32_t drop_threshold(double p) {
  if (!(p >= 0.0 && p < 1.0)) return 0;
  const double t = floor((1.0 - p) * 256.0 + 0.5);
  return t < 1.0 ? 0u : (uint32_t)t;
}

static int drop_init(drop_t *dr, double p, uint64_t seed, uint32_t offset) {
  memset(dr, 0, sizeof *dr);
  dr->t = drop_threshold(p);
  if (dr->t == 0) return 1;
  dr->on = 1;
  dr->key[0] = (uint32_t)seed;
  dr->key[1] = (uint32_t)(seed >> 32);
  dr->offset = offset;
  dr->rscale = 256.0 / (double)dr->t;
  return 0;
}

/* keep_ij (0/1) of head bh for rows [0, n_rows) and keys [0, n_cols): out[n_rows][n_cols]. */
int oracle_dropout_keep(double p, uint64_t seed, uint32_t offset, int64_t bh, int64_t n_rows,
                        int64_t n_cols, uint8_t *out) {
  drop_t dr;
  if (drop_init(&dr, p, seed, offset) || n_rows < 0 || n_cols < 0 || !out) return 1;
  for (int64_t i = 0; i < n_rows; ++i)
    for (int64_t j = 0; j < n_cols; ++j) out[i * n_cols + j] = drop_byte(&dr, bh, i, j) < dr.t;
  return 0;
}

typedef struct {
  const double *q, *k, *v, *o, *dO, *lse, *Dvec;
  double *o_out, *lse_out, *p_out, *dq, *dk, *dv;
  double *P_head, *dS_head; /* per-head N x N scratch (backward only) */
  int64_t BH, N, d;
  double scale;
  int causal;
  drop_t drop;
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

/* One query row of head h, materialising its row of S and P.
 * s_row, p_row: scratch of length N.  Writes o_row[d], *lse_out, and p_row
 * (the softmax probabilities before dropout). */
static void forward_row(const double *qh, const double *kh, const double *vh, int64_t N,
                        int64_t d, double scale, vis_t vis, const drop_t *dr, int64_t h,
                        int64_t i, double *s_row, double *p_row, double *o_row,
                        double *lse_out) {
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
    const double w = p_row[j] * drop_weight(dr, h, i, j);
    if (w == 0.0) continue;
    const double *vj = vh + j * d;
    for (int64_t c = 0; c < d; ++c) o_row[c] += w * vj[c];
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
      forward_row(qh, kh, vh, N, d, J->scale, vis_for(J, h, i), &J->drop, h, i, s_row, p_row,
                  J->o_out + (h * N + i) * d, J->lse_out + h * N + i);
    }
  }
  free(s_row);
  free(p_tmp);
  return NULL;
}

/* O = softmax(scale Q K^T [+ causal mask]) V and LSE for all heads.
 * p_out: optional [BH][N][N] probabilities (NULL to skip). */
static int forward_job(const double *q, const double *k, const double *v, double *o, double *lse,
                       double *p_out, int64_t BH, int64_t N, int64_t d, double scale, int causal,
                       const uint8_t *bmask, int64_t mask_heads, int64_t blk, const drop_t *dr,
                       int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !o || !lse) return 1;
  if (bmask && (mask_heads < 1 || blk < 1)) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  if (dr) J.drop = *dr;
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

int oracle_forward_masked(const double *q, const double *k, const double *v, double *o,
                          double *lse, double *p_out, int64_t BH, int64_t N, int64_t d,
                          double scale, int causal, const uint8_t *bmask, int64_t mask_heads,
                          int64_t blk, int nthreads) {
  return forward_job(q, k, v, o, lse, p_out, BH, N, d, scale, causal, bmask, mask_heads, blk,
                     NULL, nthreads);
}

/* Forward with dropout of probability p (p_out, if given, holds P before dropout). */
int oracle_forward_dropout(const double *q, const double *k, const double *v, double *o,
                           double *lse, double *p_out, int64_t BH, int64_t N, int64_t d,
                           double scale, int causal, double p, uint64_t seed, uint32_t offset,
                           int nthreads) {
  drop_t dr;
  if (drop_init(&dr, p, seed, offset)) return 1;
  return forward_job(q, k, v, o, lse, p_out, BH, N, d, scale, causal, NULL, 0, 0, &dr, nthreads);
}

/* Block mask and dropout together: key j reaches O_i with weight
 * P_ij * keep_ij * 256 / t when it is visible (mask and causal rule), 0
 * otherwise; P is the softmax over the visible keys, before dropout. */
int oracle_forward_masked_dropout(const double *q, const double *k, const double *v, double *o,
                                  double *lse, double *p_out, int64_t BH, int64_t N, int64_t d,
                                  double scale, int causal, const uint8_t *bmask, int64_t mask_heads,
                                  int64_t blk, double p, uint64_t seed, uint32_t offset, int nthreads) {
  drop_t dr;
  if (!bmask || drop_init(&dr, p, seed, offset)) return 1;
  return forward_job(q, k, v, o, lse, p_out, BH, N, d, scale, causal, bmask, mask_heads, blk, &dr,
                     nthreads);
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
      forward_row(qh, kh, vh, N, d, J->scale, vis_for(J, h, i), &J->drop, h, i, s_row, p_row,
                  o_row, &lse_unused);
      const double *doi = doh + i * d, *oi = oh + i * d;
      double Di = 0.0;
      for (int64_t c = 0; c < d; ++c) Di += doi[c] * oi[c];
      for (int64_t j = 0; j < N; ++j) {
        if (p_row[j] == 0.0) { ds_row[j] = 0.0; continue; }
        const double w = drop_weight(&J->drop, h, i, j);
        const double *vj = vh + j * d;
        double dp = 0.0;
        for (int64_t c = 0; c < d; ++c) dp += doi[c] * vj[c];
        ds_row[j] = p_row[j] * (w * dp - Di);
        p_row[j] *= w; /* the weight dV sees */
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

/* Phase 2 (key columns of one head): dV_j = sum_i P_ij dO_i (P after dropout),
 * dK_j = scale sum_i dS_ij Q_i. */
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
static int backward_job(const double *q, const double *k, const double *v, const double *o,
                        const double *dO, double *dq, double *dk, double *dv, int64_t BH,
                        int64_t N, int64_t d, double scale, int causal, const uint8_t *bmask,
                        int64_t mask_heads, int64_t blk, const drop_t *dr, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !o || !dO || !dq || !dk || !dv) return 1;
  if (bmask && (mask_heads < 1 || blk < 1)) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  if (dr) J.drop = *dr;
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

int oracle_backward_masked(const double *q, const double *k, const double *v, const double *o,
                           const double *dO, double *dq, double *dk, double *dv, int64_t BH,
                           int64_t N, int64_t d, double scale, int causal, const uint8_t *bmask,
                           int64_t mask_heads, int64_t blk, int nthreads) {
  return backward_job(q, k, v, o, dO, dq, dk, dv, BH, N, d, scale, causal, bmask, mask_heads, blk,
                      NULL, nthreads);
}

/* Backward with dropout; o must be the dropout forward's output for the same
 * p, seed and offset. */
int oracle_backward_dropout(const double *q, const double *k, const double *v, const double *o,
                            const double *dO, double *dq, double *dk, double *dv, int64_t BH,
                            int64_t N, int64_t d, double scale, int causal, double p,
                            uint64_t seed, uint32_t offset, int nthreads) {
  drop_t dr;
  if (drop_init(&dr, p, seed, offset)) return 1;
  return backward_job(q, k, v, o, dO, dq, dk, dv, BH, N, d, scale, causal, NULL, 0, 0, &dr,
                      nthreads);
}

/* Backward of oracle_forward_masked_dropout (o its output for the same mask,
 * p, seed and offset). */
int oracle_backward_masked_dropout(const double *q, const double *k, const double *v, const double *o,
                                   const double *dO, double *dq, double *dk, double *dv, int64_t BH,
                                   int64_t N, int64_t d, double scale, int causal, const uint8_t *bmask,
                                   int64_t mask_heads, int64_t blk, double p, uint64_t seed,
                                   uint32_t offset, int nthreads) {
  drop_t dr;
  if (!bmask || drop_init(&dr, p, seed, offset)) return 1;
  return backward_job(q, k, v, o, dO, dq, dk, dv, BH, N, d, scale, causal, bmask, mask_heads, blk, &dr,
                      nthreads);
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
    forward_row(qh, kh, vh, N, d, J->scale, vis_for(J, h, i), &J->drop, h, i, s_row, p_row, oi,
                J->lse_out + r);
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
      const double ds = p_row[j] * (drop_weight(&J->drop, h, i, j) * dp - Di);
      for (int64_t c = 0; c < d; ++c) dqi[c] += ds * kj[c];
    }
    for (int64_t c = 0; c < d; ++c) dqi[c] *= J->scale;
  }
  free(s_row);
  free(p_row);
  return NULL;
}

static int rows_job(const double *q, const double *k, const double *v, const double *dO,
                    int64_t BH, int64_t N, int64_t d, double scale, int causal,
                    const int64_t *bh_idx, const int64_t *row_idx, int64_t nsel, double *o_rows,
                    double *lse_rows, double *dq_rows, const drop_t *dr, int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !bh_idx || !row_idx || !o_rows || !lse_rows)
    return 1;
  if (dq_rows && !dO) return 1;
  for (int64_t r = 0; r < nsel; ++r)
    if (bh_idx[r] < 0 || bh_idx[r] >= BH || row_idx[r] < 0 || row_idx[r] >= N) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  if (dr) J.drop = *dr;
  J.q = q; J.k = k; J.v = v; J.dO = dO; J.o_out = o_rows; J.lse_out = lse_rows; J.dq = dq_rows;
  J.BH = BH; J.N = N; J.d = d; J.scale = scale; J.causal = causal;
  J.bh_idx = bh_idx; J.idx = row_idx; J.nsel = nsel; J.nitems = nsel;
  pthread_mutex_init(&J.mu, NULL);
  run_threads(rows_worker, &J, nthreads);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

int oracle_rows(const double *q, const double *k, const double *v, const double *dO,
                int64_t BH, int64_t N, int64_t d, double scale, int causal,
                const int64_t *bh_idx, const int64_t *row_idx, int64_t nsel, double *o_rows,
                double *lse_rows, double *dq_rows, int nthreads) {
  return rows_job(q, k, v, dO, BH, N, d, scale, causal, bh_idx, row_idx, nsel, o_rows, lse_rows,
                  dq_rows, NULL, nthreads);
}

int oracle_rows_dropout(const double *q, const double *k, const double *v, const double *dO,
                        int64_t BH, int64_t N, int64_t d, double scale, int causal, double p,
                        uint64_t seed, uint32_t offset, const int64_t *bh_idx,
                        const int64_t *row_idx, int64_t nsel, double *o_rows, double *lse_rows,
                        double *dq_rows, int nthreads) {
  drop_t dr;
  if (drop_init(&dr, p, seed, offset)) return 1;
  return rows_job(q, k, v, dO, BH, N, d, scale, causal, bh_idx, row_idx, nsel, o_rows, lse_rows,
                  dq_rows, &dr, nthreads);
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
      const double w = drop_weight(&J->drop, h, i, j);
      const double ds = p * (w * dp - J->Dvec[h * N + i]);
      for (int64_t c = 0; c < d; ++c) { dvj[c] += w * p * doi[c]; dkj[c] += ds * qi[c]; }
    }
    for (int64_t c = 0; c < d; ++c) dkj[c] *= J->scale;
  }
  return NULL;
}

static int cols_job(const double *q, const double *k, const double *v, const double *dO,
                    const double *lse_all, const double *D_all, int64_t BH, int64_t N, int64_t d,
                    double scale, int causal, const int64_t *bh_idx, const int64_t *col_idx,
                    int64_t nsel, double *dk_rows, double *dv_rows, const drop_t *dr,
                    int nthreads) {
  if (BH < 1 || N < 1 || d < 1 || !q || !k || !v || !dO || !lse_all || !D_all || !bh_idx ||
      !col_idx || !dk_rows || !dv_rows)
    return 1;
  for (int64_t r = 0; r < nsel; ++r)
    if (bh_idx[r] < 0 || bh_idx[r] >= BH || col_idx[r] < 0 || col_idx[r] >= N) return 1;
  job_t J;
  memset(&J, 0, sizeof J);
  if (dr) J.drop = *dr;
  J.q = q; J.k = k; J.v = v; J.dO = dO; J.lse = lse_all; J.Dvec = D_all;
  J.dk = dk_rows; J.dv = dv_rows;
  J.BH = BH; J.N = N; J.d = d; J.scale = scale; J.causal = causal;
  J.bh_idx = bh_idx; J.idx = col_idx; J.nsel = nsel; J.nitems = nsel;
  pthread_mutex_init(&J.mu, NULL);
  run_threads(cols_worker, &J, nthreads);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

int oracle_cols(const double *q, const double *k, const double *v, const double *dO,
                const double *lse_all, const double *D_all, int64_t BH, int64_t N, int64_t d,
                double scale, int causal, const int64_t *bh_idx, const int64_t *col_idx,
                int64_t nsel, double *dk_rows, double *dv_rows, int nthreads) {
  return cols_job(q, k, v, dO, lse_all, D_all, BH, N, d, scale, causal, bh_idx, col_idx, nsel,
                  dk_rows, dv_rows, NULL, nthreads);
}

int oracle_cols_dropout(const double *q, const double *k, const double *v, const double *dO,
                        const double *lse_all, const double *D_all, int64_t BH, int64_t N,
                        int64_t d, double scale, int causal, double p, uint64_t seed,
                        uint32_t offset, const int64_t *bh_idx, const int64_t *col_idx,
                        int64_t nsel, double *dk_rows, double *dv_rows, int nthreads) {
  drop_t dr;
  if (drop_init(&dr, p, seed, offset)) return 1;
  return cols_job(q, k, v, dO, lse_all, D_all, BH, N, d, scale, causal, bh_idx, col_idx, nsel,
                  dk_rows, dv_rows, &dr, nthreads);
}
