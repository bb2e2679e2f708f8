/*
 * topo_oracle.c -- CPU oracle for condensate-set ("topological") attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg call into this file.  It shares no code with
 * the CUDA library, and the CUDA library never calls it.
 *
 * It is written to be read against the method's definition, not to be fast:
 * one query row at a time, every step in the order the method states it.
 *
 * What it computes (The Condensate Theorem, arXiv 2602.06317, as restated by
 * the gist.science explainer pages):
 *   - Condensate set, Technical Summary section 2 ("Condensate Set C_i"): for
 *     query position i, C_i = {anchor 0} U {the W most recent causal
 *     positions} U {the k remaining positions with the largest q_i . k_j}.
 *   - Topological attention, Technical Summary section 3: the softmax is taken
 *     over the indices in C_i only and the output is the weighted sum of V.
 *   - Dense causal attention (the full-attention comparison, and the "pillar
 *     layer" of the Methodology section).
 *   - Excluded mass: the dense-softmax probability that falls outside C_i, and
 *     the largest such single weight; these are the quantities the pages'
 *     float32-ULP exactness argument is about (Technical Summary section 3,
 *     "numerical equivalence").
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - The window is the W most recent causal positions INCLUDING the query's
 *     own position p: {max(0, p-W+1), ..., p}.
 *   - Top-k candidates are the positions 1..p-W (not the anchor, not the
 *     window); with fewer than k candidates all of them are taken.
 *   - Ranking uses a float32 score (the precision the GPU decides in):
 *     acc = +0.0f; for c = 0..d-1: acc = fmaf(q[c], k[c], acc).  Order is
 *     (score descending, index ascending), so equal scores go to the lower
 *     index.
 *   - Query head h reads KV head h / (Hq/Hkv); query row r sits at position
 *     n - nq + r.
 *   - Softmax and weighted sums are evaluated in float64 from the exact input
 *     values (bf16 / f32 widened exactly), with logits scale * (q . k_j).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t B, Hq, Hkv, d;
  int64_t n, nq, kv_stride;
  int32_t W, k;
  float scale;
  int32_t dtype; /* 0: float32 inputs, 1: bfloat16 inputs (raw uint16 bits) */
} orc_params;

/* ---- input access -------------------------------------------------------- */

static float orc_elem(const void *base, int dtype, int64_t i) {
  if (dtype == 0) return ((const float *)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

/* ---- step 1: scores ------------------------------------------------------ */

/* The float32 ranking score: a left-to-right chain of fused multiply-adds,
 * starting from +0.0f.  fmaf rounds once per step (IEEE-754 fusedMultiplyAdd). */
float orc_score_f32(const float *q, const float *kr, int d) {
  float acc = 0.0f;
  for (int c = 0; c < d; ++c) acc = fmaf(q[c], kr[c], acc);
  return acc;
}

/* The float64 dot product used for logits.  Products of two float32 values
 * are exact in float64; the sum rounds in float64. */
static double orc_dot_f64(const double *q, const double *kr, int d) {
  double acc = 0.0;
  for (int c = 0; c < d; ++c) acc += q[c] * kr[c];
  return acc;
}

/* ---- step 2: the ranking order ------------------------------------------ */

typedef struct {
  float s;
  int64_t j;
} orc_cand;

/* Total order: larger score first; on equal score, smaller index first. */
static int orc_cand_cmp(const void *a, const void *b) {
  const orc_cand *x = (const orc_cand *)a, *y = (const orc_cand *)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  if (x->j < y->j) return -1;
  if (x->j > y->j) return 1;
  return 0;
}

/* ---- per-row work -------------------------------------------------------- */

typedef struct {
  const orc_params *P;
  const void *q, *k, *v;
  const int64_t *rows; /* flat (b, h, r) ids, or NULL for all rows */
  int64_t nrows;
  /* outputs, one slot per listed row */
  double *out;      /* [nrows, d] sparse output, or NULL */
  int32_t *idx;     /* [nrows, 1+W+k] condensate set, ascending, -1 padded, or NULL */
  double *dense;    /* [nrows, d] dense output, or NULL */
  double *excl;     /* [nrows] excluded dense mass, or NULL */
  double *wmax;     /* [nrows] largest excluded dense weight, or NULL */
  double *p0;       /* [nrows] dense weight of the anchor, or NULL */
  int64_t next;     /* shared row counter */
  pthread_mutex_t mu;
} orc_job;

static void orc_row(orc_job *J, int64_t slot, int64_t flat, float *s32, double *s64,
                    orc_cand *cand, unsigned char *inC, double *q64, float *q32,
                    double *k64, float *k32) {
  const orc_params *P = J->P;
  const int d = P->d;
  const int64_t r = flat % P->nq;
  const int64_t h = (flat / P->nq) % P->Hq;
  const int64_t b = flat / (P->nq * P->Hq);
  const int64_t g = P->Hq / P->Hkv;
  const int64_t kvh = h / g;
  const int64_t p = P->n - P->nq + r; /* absolute position of this query row */
  const int64_t W = P->W, K = P->k;
  const int64_t cmax = 1 + W + K;
  const double scale = (double)P->scale;

  const int64_t qoff = ((b * P->Hq + h) * P->nq + r) * d;
  for (int c = 0; c < d; ++c) {
    q32[c] = orc_elem(J->q, P->dtype, qoff + c);
    q64[c] = (double)q32[c];
  }
  const int64_t kbase = (b * P->Hkv + kvh) * P->kv_stride;

  /* scores of every causal position 0..p */
  for (int64_t j = 0; j <= p; ++j) {
    const int64_t off = (kbase + j) * d;
    for (int c = 0; c < d; ++c) {
      k32[c] = orc_elem(J->k, P->dtype, off + c);
      k64[c] = (double)k32[c];
    }
    s32[j] = orc_score_f32(q32, k32, d);
    s64[j] = orc_dot_f64(q64, k64, d);
  }

  /* anchor + window */
  memset(inC, 0, (size_t)(p + 1));
  inC[0] = 1;
  const int64_t wlo = (p - W + 1 > 0) ? p - W + 1 : 0;
  for (int64_t j = wlo; j <= p; ++j) inC[j] = 1;

  /* top-k of the remaining positions 1..p-W */
  int64_t nc = 0;
  for (int64_t j = 1; j <= p - W; ++j) {
    cand[nc].s = s32[j];
    cand[nc].j = j;
    ++nc;
  }
  qsort(cand, (size_t)nc, sizeof(orc_cand), orc_cand_cmp);
  const int64_t take = nc < K ? nc : K;
  for (int64_t t = 0; t < take; ++t) inC[cand[t].j] = 1;

  /* C_i ascending, -1 padded */
  if (J->idx) {
    int32_t *row = J->idx + slot * cmax;
    int64_t m = 0;
    for (int64_t j = 0; j <= p; ++j)
      if (inC[j]) row[m++] = (int32_t)j;
    for (; m < cmax; ++m) row[m] = -1;
  }

  /* softmax over C_i (float64) and the weighted sum of V */
  const int64_t vbase = (b * P->Hkv + kvh) * P->kv_stride;
  if (J->out) {
    double mx = -INFINITY;
    for (int64_t j = 0; j <= p; ++j)
      if (inC[j] && scale * s64[j] > mx) mx = scale * s64[j];
    double Z = 0.0;
    double *o = J->out + slot * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t j = 0; j <= p; ++j) {
      if (!inC[j]) continue;
      const double w = exp(scale * s64[j] - mx);
      Z += w;
      const int64_t off = (vbase + j) * d;
      for (int c = 0; c < d; ++c) o[c] += w * (double)orc_elem(J->v, P->dtype, off + c);
    }
    for (int c = 0; c < d; ++c) o[c] /= Z;
  }

  /* dense causal softmax over 0..p, and the mass it puts outside C_i */
  if (J->dense || J->excl || J->wmax || J->p0) {
    double mx = -INFINITY;
    for (int64_t j = 0; j <= p; ++j)
      if (scale * s64[j] > mx) mx = scale * s64[j];
    double Z = 0.0, Zx = 0.0, wx = 0.0;
    for (int64_t j = 0; j <= p; ++j) {
      const double w = exp(scale * s64[j] - mx);
      Z += w;
      if (!inC[j]) {
        Zx += w;
        if (w > wx) wx = w;
      }
    }
    if (J->excl) J->excl[slot] = Zx / Z;
    if (J->wmax) J->wmax[slot] = wx / Z;
    if (J->p0) J->p0[slot] = exp(scale * s64[0] - mx) / Z;
    if (J->dense) {
      double *o = J->dense + slot * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int64_t j = 0; j <= p; ++j) {
        const double w = exp(scale * s64[j] - mx);
        const int64_t off = (vbase + j) * d;
        for (int c = 0; c < d; ++c) o[c] += w * (double)orc_elem(J->v, P->dtype, off + c);
      }
      for (int c = 0; c < d; ++c) o[c] /= Z;
    }
  }
}

static void *orc_worker(void *arg) {
  orc_job *J = (orc_job *)arg;
  const orc_params *P = J->P;
  const int64_t n = P->n, d = P->d;
  float *s32 = (float *)malloc(sizeof(float) * (size_t)n);
  double *s64 = (double *)malloc(sizeof(double) * (size_t)n);
  orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)n);
  unsigned char *inC = (unsigned char *)malloc((size_t)n);
  double *q64 = (double *)malloc(sizeof(double) * (size_t)d);
  double *k64 = (double *)malloc(sizeof(double) * (size_t)d);
  float *q32 = (float *)malloc(sizeof(float) * (size_t)d);
  float *k32 = (float *)malloc(sizeof(float) * (size_t)d);
  if (s32 && s64 && cand && inC && q64 && k64 && q32 && k32) {
    for (;;) {
      pthread_mutex_lock(&J->mu);
      const int64_t slot = J->next++;
      pthread_mutex_unlock(&J->mu);
      if (slot >= J->nrows) break;
      const int64_t flat = J->rows ? J->rows[slot] : slot;
      orc_row(J, slot, flat, s32, s64, cand, inC, q64, q32, k64, k32);
    }
  }
  free(s32); free(s64); free(cand); free(inC);
  free(q64); free(k64); free(q32); free(k32);
  return NULL;
}

/* Argument check shared by the entry points; returns 0 when usable. */
static int orc_check(const orc_params *P) {
  if (!P) return -1;
  if (P->B < 1 || P->Hq < 1 || P->Hkv < 1 || P->d < 1 || P->Hq % P->Hkv) return -1;
  if (P->n < 1 || P->nq < 1 || P->nq > P->n || P->kv_stride < P->n) return -1;
  if (P->W < 1 || P->k < 0 || (P->dtype != 0 && P->dtype != 1)) return -1;
  return 0;
}

/*
 * Condensate-set attention for the listed rows (all rows when rows == NULL).
 * A row id is flat over [B, Hq, nq].  Every output pointer may be NULL.
 * Returns 0, or -1 on bad arguments.
 */
int orc_topo_attn(const orc_params *P, const void *q, const void *k, const void *v,
                  const int64_t *rows, int64_t nrows, double *out, int32_t *idx,
                  double *dense, double *excl, double *wmax, double *p0, int nthreads) {
  if (orc_check(P)) return -1;
  orc_job J;
  memset(&J, 0, sizeof J);
  J.P = P; J.q = q; J.k = k; J.v = v;
  J.rows = rows;
  J.nrows = rows ? nrows : (int64_t)P->B * P->Hq * P->nq;
  J.out = out; J.idx = idx; J.dense = dense; J.excl = excl; J.wmax = wmax; J.p0 = p0;
  pthread_mutex_init(&J.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if (nthreads > J.nrows) nthreads = (int)(J.nrows > 0 ? J.nrows : 1);
  pthread_t th[512];
  int started = 0;
  for (int t = 1; t < nthreads; ++t)
    if (pthread_create(&th[started], NULL, orc_worker, &J) == 0) ++started;
  orc_worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.mu);
  return 0;
}

/* ---- group-shared selection (GQA) ---------------------------------------- */
/*
 * A variant the pages allow for grouped-query attention models (the method is
 * validated on GQA architectures, Technical Summary section 4): one
 * condensate set per (sequence, KV head, query row), shared by the g query
 * heads that read that KV head.  Reading fixed here (the pages give no rule):
 * the top-k ranks candidate j by the group score
 *     shat_j = max over the group's heads h of s_{h,j}
 * (s: the float32 ranking score of step 1), larger first, ties to the smaller
 * index.  Anchor and window are as for one head.  Each head then takes its
 * own float64 softmax over the shared set, with its own logits.
 */
typedef struct {
  const orc_params *P;
  const void *q, *k, *v;
  const int64_t *rows; /* flat (b, kvh, r) ids over [B, Hkv, nq], or NULL for all */
  int64_t nrows;
  double *out;   /* [nrows, g, d], or NULL */
  int32_t *idx;  /* [nrows, 1+W+k], or NULL */
  int64_t next;
  pthread_mutex_t mu;
} orc_gjob;

static void orc_group_row(orc_gjob *J, int64_t slot, int64_t flat, float *shat, double *s64,
                          orc_cand *cand, unsigned char *inC, float *q32, float *k32) {
  const orc_params *P = J->P;
  const int d = P->d;
  const int64_t g = P->Hq / P->Hkv;
  const int64_t r = flat % P->nq;
  const int64_t kvh = (flat / P->nq) % P->Hkv;
  const int64_t b = flat / (P->nq * P->Hkv);
  const int64_t p = P->n - P->nq + r;
  const int64_t W = P->W, K = P->k;
  const int64_t cmax = 1 + W + K;
  const double scale = (double)P->scale;
  const int64_t kbase = (b * P->Hkv + kvh) * P->kv_stride;

  /* group score of every causal position: the largest of the heads' scores */
  for (int64_t j = 0; j <= p; ++j) shat[j] = -INFINITY;
  for (int64_t hh = 0; hh < g; ++hh) {
    const int64_t h = kvh * g + hh;
    const int64_t qoff = ((b * P->Hq + h) * P->nq + r) * d;
    for (int c = 0; c < d; ++c) q32[c] = orc_elem(J->q, P->dtype, qoff + c);
    for (int64_t j = 0; j <= p; ++j) {
      const int64_t off = (kbase + j) * d;
      for (int c = 0; c < d; ++c) k32[c] = orc_elem(J->k, P->dtype, off + c);
      const float s = orc_score_f32(q32, k32, d);
      if (s > shat[j]) shat[j] = s;
    }
  }

  /* anchor + window, then the top-k of 1..p-W by the group score */
  memset(inC, 0, (size_t)(p + 1));
  inC[0] = 1;
  const int64_t wlo = (p - W + 1 > 0) ? p - W + 1 : 0;
  for (int64_t j = wlo; j <= p; ++j) inC[j] = 1;
  int64_t nc = 0;
  for (int64_t j = 1; j <= p - W; ++j) {
    cand[nc].s = shat[j];
    cand[nc].j = j;
    ++nc;
  }
  qsort(cand, (size_t)nc, sizeof(orc_cand), orc_cand_cmp);
  const int64_t take = nc < K ? nc : K;
  for (int64_t t = 0; t < take; ++t) inC[cand[t].j] = 1;

  if (J->idx) {
    int32_t *row = J->idx + slot * cmax;
    int64_t m = 0;
    for (int64_t j = 0; j <= p; ++j)
      if (inC[j]) row[m++] = (int32_t)j;
    for (; m < cmax; ++m) row[m] = -1;
  }

  /* each head: float64 softmax over the shared set and the weighted sum of V */
  if (J->out) {
    for (int64_t hh = 0; hh < g; ++hh) {
      const int64_t h = kvh * g + hh;
      const int64_t qoff = ((b * P->Hq + h) * P->nq + r) * d;
      double mx = -INFINITY;
      for (int64_t j = 0; j <= p; ++j) {
        s64[j] = -INFINITY;
        if (!inC[j]) continue;
        const int64_t off = (kbase + j) * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
          acc += (double)orc_elem(J->q, P->dtype, qoff + c) *
                 (double)orc_elem(J->k, P->dtype, off + c);
        s64[j] = scale * acc;
        if (s64[j] > mx) mx = s64[j];
      }
      double Z = 0.0;
      double *o = J->out + (slot * g + hh) * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int64_t j = 0; j <= p; ++j) {
        if (!inC[j]) continue;
        const double w = exp(s64[j] - mx);
        Z += w;
        const int64_t off = (kbase + j) * d;
        for (int c = 0; c < d; ++c) o[c] += w * (double)orc_elem(J->v, P->dtype, off + c);
      }
      for (int c = 0; c < d; ++c) o[c] /= Z;
    }
  }
}

static void *orc_gworker(void *arg) {
  orc_gjob *J = (orc_gjob *)arg;
  const int64_t n = J->P->n, d = J->P->d;
  float *shat = (float *)malloc(sizeof(float) * (size_t)n);
  double *s64 = (double *)malloc(sizeof(double) * (size_t)n);
  orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)n);
  unsigned char *inC = (unsigned char *)malloc((size_t)n);
  float *q32 = (float *)malloc(sizeof(float) * (size_t)d);
  float *k32 = (float *)malloc(sizeof(float) * (size_t)d);
  if (shat && s64 && cand && inC && q32 && k32) {
    for (;;) {
      pthread_mutex_lock(&J->mu);
      const int64_t slot = J->next++;
      pthread_mutex_unlock(&J->mu);
      if (slot >= J->nrows) break;
      const int64_t flat = J->rows ? J->rows[slot] : slot;
      orc_group_row(J, slot, flat, shat, s64, cand, inC, q32, k32);
    }
  }
  free(shat); free(s64); free(cand); free(inC); free(q32); free(k32);
  return NULL;
}

/*
 * Group-shared condensate-set attention for the listed group rows (all when
 * rows == NULL); a row id is flat over [B, Hkv, nq].  out: [nrows, g, d]
 * (head hh of the group at [slot, hh]); idx: [nrows, 1+W+k].  Either may be
 * NULL.  Returns 0, or -1 on bad arguments.
 */
int orc_topo_attn_group(const orc_params *P, const void *q, const void *k, const void *v,
                        const int64_t *rows, int64_t nrows, double *out, int32_t *idx,
                        int nthreads) {
  if (orc_check(P)) return -1;
  orc_gjob J;
  memset(&J, 0, sizeof J);
  J.P = P; J.q = q; J.k = k; J.v = v;
  J.rows = rows;
  J.nrows = rows ? nrows : (int64_t)P->B * P->Hkv * P->nq;
  J.out = out; J.idx = idx;
  pthread_mutex_init(&J.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if (nthreads > J.nrows) nthreads = (int)(J.nrows > 0 ? J.nrows : 1);
  pthread_t th[512];
  int started = 0;
  for (int t = 1; t < nthreads; ++t)
    if (pthread_create(&th[started], NULL, orc_gworker, &J) == 0) ++started;
  orc_gworker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.mu);
  return 0;
}
