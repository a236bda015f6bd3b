/*
 * TEST INFRASTRUCTURE ONLY: the CPU oracle of the Tensor-Train embedding bag.
 * Only tests, the smoke check and the benchmark's CPU-baseline arm may call
 * it; the product path never does.  It shares no code with the CUDA path.
 *
 * What it computes (plain definitions, evaluated naively in fp64):
 *
 *  - A table of M = m1*m2*m3 rows of width D = n1*n2*n3 is stored as three
 *    TT cores (a table replaced by a series of small tensor cores whose
 *    product gives the rows: FlowTT summary card, problem statement; TT-Rec
 *    press article, method paragraph).  Core k is float32 [m_k][R_{k-1}][n_k][R_k] with
 *    R_0 = R_3 = 1.
 *  - Row index r is split mixed-radix with i1 most significant:
 *    r = (i1*m2 + i2)*m3 + i3.  Output position j = (j1*n2 + j2)*n3 + j3.
 *  - A lookup is the chain of contractions over the cores, one core after
 *    the other (FlowTT summary card, problem statement):
 *        T1  = G1[i1]                (n1 x R1)
 *        T12 = T1 . G2[i2]           (n1 x n2*R2)  ==  (n1*n2 x R2)
 *        row = T12 . G3[i3]          (n1*n2 x n3)  ==  D values
 *    i.e. row(r)[j] = sum_{a,b} G1[i1][0][j1][a] G2[i2][a][j2][b] G3[i3][b][j3][0].
 *  - Bags are CSR offsets (B+1 entries); out[b] = sum of the rows of the
 *    lookups offsets[b] .. offsets[b+1]-1 (the embedding-bag operator of
 *    TT-Rec, abstract).  Empty bags give zero rows.
 *  - The two other pooling rules of an embedding bag: a weighted sum, each
 *    row scaled by its lookup's per-sample weight w[l], and the mean, the sum
 *    divided by the bag's number of lookups (an empty bag stays zero).  The
 *    weights go with the sum only.  For the weighted sum the gradient of
 *    <grad_out, out> with respect to w[l] is <grad_out[bag(l)], row(r_l)>.
 *  - Backward: the exact gradient of <grad_out, out> with respect to each
 *    core, accumulated lookup by lookup (training latency, FlowTT abstract).
 *  - SGD: G <- G - lr*dG.
 *  - Grouping reference: lookups stably sorted by the key (i2, i1, i3), then
 *    unique runs of rows and of (i1, i2) prefixes (lookups that share the
 *    leading core indices grouped together, FlowTT summary card, key
 *    innovations).
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TTO_OK 0
#define TTO_ERR_ARG (-1)
#define TTO_ERR_INDEX (-2)
#define TTO_ERR_OFFSETS (-3)
#define TTO_ERR_NOMEM (-4)

typedef struct {
  const float *G1, *G2, *G3;
  int64_t m1, m2, m3;
  int n1, n2, n3, R1, R2;
} tto_tt;

static int tto_init(tto_tt *t, const float *G1, const float *G2, const float *G3,
                    const int64_t *m, const int32_t *n, const int32_t *R) {
  if (!G1 || !G2 || !G3 || !m || !n || !R) return TTO_ERR_ARG;
  if (R[0] != 1 || R[3] != 1) return TTO_ERR_ARG;
  for (int k = 0; k < 3; ++k)
    if (m[k] < 1 || n[k] < 1) return TTO_ERR_ARG;
  if (R[1] < 1 || R[2] < 1) return TTO_ERR_ARG;
  t->G1 = G1; t->G2 = G2; t->G3 = G3;
  t->m1 = m[0]; t->m2 = m[1]; t->m3 = m[2];
  t->n1 = n[0]; t->n2 = n[1]; t->n3 = n[2];
  t->R1 = R[1]; t->R2 = R[2];
  return TTO_OK;
}

/* Mixed-radix split of a row index, i1 most significant. */
static void tto_split(const tto_tt *t, int64_t r, int64_t *i1, int64_t *i2, int64_t *i3) {
  *i3 = r % t->m3;
  int64_t q = r / t->m3;
  *i2 = q % t->m2;
  *i1 = q / t->m2;
}

/* Element accessors in the [m_k][R_{k-1}][n_k][R_k] layout. */
static double g1(const tto_tt *t, int64_t i1, int j1, int a) {
  return (double)t->G1[(i1 * t->n1 + j1) * t->R1 + a];
}
static double g2(const tto_tt *t, int64_t i2, int a, int j2, int b) {
  return (double)t->G2[((i2 * t->R1 + a) * t->n2 + j2) * t->R2 + b];
}
static double g3(const tto_tt *t, int64_t i3, int b, int j3) {
  return (double)t->G3[(i3 * t->R2 + b) * t->n3 + j3];
}

/* T12[(j1*n2 + j2)*R2 + b] = sum_a G1[i1][0][j1][a] * G2[i2][a][j2][b]. */
static void tto_prefix(const tto_tt *t, int64_t i1, int64_t i2, double *T12) {
  for (int j1 = 0; j1 < t->n1; ++j1)
    for (int j2 = 0; j2 < t->n2; ++j2)
      for (int b = 0; b < t->R2; ++b) {
        double s = 0.0;
        for (int a = 0; a < t->R1; ++a) s += g1(t, i1, j1, a) * g2(t, i2, a, j2, b);
        T12[(j1 * t->n2 + j2) * t->R2 + b] = s;
      }
}

/* row[(j1*n2 + j2)*n3 + j3] = sum_b T12[(j1*n2 + j2)*R2 + b] * G3[i3][b][j3][0]. */
static void tto_row(const tto_tt *t, const double *T12, int64_t i3, double *row) {
  int n12 = t->n1 * t->n2;
  for (int j12 = 0; j12 < n12; ++j12)
    for (int j3 = 0; j3 < t->n3; ++j3) {
      double s = 0.0;
      for (int b = 0; b < t->R2; ++b) s += T12[j12 * t->R2 + b] * g3(t, i3, b, j3);
      row[j12 * t->n3 + j3] = s;
    }
}

static int tto_check_offsets(const int64_t *offsets, int64_t B, int64_t nnz) {
  if (!offsets || B < 0) return TTO_ERR_ARG;
  if (offsets[0] != 0 || offsets[B] != nnz) return TTO_ERR_OFFSETS;
  for (int64_t b = 0; b < B; ++b)
    if (offsets[b + 1] < offsets[b]) return TTO_ERR_OFFSETS;
  return TTO_OK;
}

/* ---------------- threads: a plain split of [0, count) ---------------- */

typedef struct tto_job {
  void (*fn)(struct tto_job *, int64_t, int64_t);
  const void *ctx;
  int64_t lo, hi;
  int err;
  double *scratch;   /* per-thread accumulators (backward) */
} tto_job;

static void *tto_thread_main(void *p) {
  tto_job *j = (tto_job *)p;
  j->fn(j, j->lo, j->hi);
  return NULL;
}

static int tto_parallel(void (*fn)(tto_job *, int64_t, int64_t), const void *ctx, int64_t count,
                        int threads, tto_job *jobs) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_t tid[256];
  for (int k = 0; k < threads; ++k) {
    jobs[k].fn = fn;
    jobs[k].ctx = ctx;
    jobs[k].lo = count * k / threads;
    jobs[k].hi = count * (k + 1) / threads;
    jobs[k].err = TTO_OK;
  }
  for (int k = 1; k < threads; ++k) pthread_create(&tid[k], NULL, tto_thread_main, &jobs[k]);
  tto_thread_main(&jobs[0]);
  for (int k = 1; k < threads; ++k) pthread_join(tid[k], NULL);
  int err = TTO_OK;
  for (int k = 0; k < threads; ++k)
    if (jobs[k].err != TTO_OK) err = jobs[k].err;
  return err;
}

/* ---------------- forward ---------------- */

typedef struct {
  tto_tt t;
  const int64_t *indices, *offsets;
  const float *weights;     /* per-sample weights [nnz], or NULL */
  int mean;                 /* 1: divide each bag's sum by its length */
  double *out;
} tto_fwd_ctx;

static void tto_fwd_bags(tto_job *job, int64_t b0, int64_t b1) {
  const tto_fwd_ctx *c = (const tto_fwd_ctx *)job->ctx;
  const tto_tt *t = &c->t;
  int D = t->n1 * t->n2 * t->n3;
  int64_t M = t->m1 * t->m2 * t->m3;
  double *T12 = (double *)malloc(sizeof(double) * t->n1 * t->n2 * t->R2);
  double *row = (double *)malloc(sizeof(double) * D);
  if (!T12 || !row) { job->err = TTO_ERR_NOMEM; free(T12); free(row); return; }
  for (int64_t b = b0; b < b1; ++b) {
    double *o = c->out + b * D;
    for (int j = 0; j < D; ++j) o[j] = 0.0;
    for (int64_t l = c->offsets[b]; l < c->offsets[b + 1]; ++l) {
      int64_t r = c->indices[l];
      if (r < 0 || r >= M) { job->err = TTO_ERR_INDEX; continue; }
      int64_t i1, i2, i3;
      tto_split(t, r, &i1, &i2, &i3);
      tto_prefix(t, i1, i2, T12);
      tto_row(t, T12, i3, row);
      double w = c->weights ? (double)c->weights[l] : 1.0;
      for (int j = 0; j < D; ++j) o[j] += w * row[j];
    }
    int64_t len = c->offsets[b + 1] - c->offsets[b];
    if (c->mean && len > 0)
      for (int j = 0; j < D; ++j) o[j] /= (double)len;
  }
  free(T12);
  free(row);
}

/* out: double [B][D], overwritten.  Out-of-range indices contribute nothing
 * and make the call return TTO_ERR_INDEX.  weights: float [nnz] or NULL;
 * mean != 0 divides every non-empty bag by its length (not with weights). */
int tto_forward_ex(const float *G1, const float *G2, const float *G3, const int64_t *m,
                   const int32_t *n, const int32_t *R, const int64_t *indices, int64_t nnz,
                   const int64_t *offsets, int64_t B, const float *weights, int mean,
                   double *out, int threads) {
  tto_fwd_ctx c;
  int e = tto_init(&c.t, G1, G2, G3, m, n, R);
  if (e) return e;
  if (nnz < 0 || (nnz > 0 && !indices) || (B > 0 && !out)) return TTO_ERR_ARG;
  if (mean && weights) return TTO_ERR_ARG;
  e = tto_check_offsets(offsets, B, nnz);
  if (e) return e;
  c.indices = indices; c.offsets = offsets; c.out = out;
  c.weights = weights; c.mean = mean != 0;
  tto_job jobs[256];
  return tto_parallel(tto_fwd_bags, &c, B, threads, jobs);
}

/* Plain sum pooling. */
int tto_forward(const float *G1, const float *G2, const float *G3, const int64_t *m,
                const int32_t *n, const int32_t *R, const int64_t *indices, int64_t nnz,
                const int64_t *offsets, int64_t B, double *out, int threads) {
  return tto_forward_ex(G1, G2, G3, m, n, R, indices, nnz, offsets, B, NULL, 0, out, threads);
}

/* ---------------- backward ---------------- */

typedef struct {
  tto_tt t;
  const int64_t *indices, *offsets;
  const float *grad_out;
  const float *weights;     /* per-sample weights [nnz], or NULL */
  int mean;                 /* 1: bags were divided by their length */
  double *dW;               /* [nnz] gradient of the weights, or NULL */
  int filter_core;          /* 0: all lookups; k in 1..3: only lookups with i_k == filter_value */
  int64_t filter_value;
  size_t n1g, n2g, n3g;     /* element counts of the three core gradients */
} tto_bwd_ctx;

static void tto_bwd_bags(tto_job *job, int64_t b0, int64_t b1) {
  const tto_bwd_ctx *c = (const tto_bwd_ctx *)job->ctx;
  const tto_tt *t = &c->t;
  int n1 = t->n1, n2 = t->n2, n3 = t->n3, R1 = t->R1, R2 = t->R2;
  int D = n1 * n2 * n3;
  int64_t M = t->m1 * t->m2 * t->m3;
  double *dG1 = job->scratch, *dG2 = dG1 + c->n1g, *dG3 = dG2 + c->n2g;
  double *T12 = (double *)malloc(sizeof(double) * n1 * n2 * R2);
  double *dT12 = (double *)malloc(sizeof(double) * n1 * n2 * R2);
  double *g = (double *)malloc(sizeof(double) * D);
  double *row = (double *)malloc(sizeof(double) * D);
  if (!T12 || !dT12 || !g || !row) {
    job->err = TTO_ERR_NOMEM; free(T12); free(dT12); free(g); free(row); return;
  }
  for (int64_t b = b0; b < b1; ++b) {
    const float *gb = c->grad_out + b * D;
    int64_t len = c->offsets[b + 1] - c->offsets[b];
    for (int64_t l = c->offsets[b]; l < c->offsets[b + 1]; ++l) {
      int64_t r = c->indices[l];
      if (c->dW) c->dW[l] = 0.0;
      if (r < 0 || r >= M) { job->err = TTO_ERR_INDEX; continue; }
      int64_t i1, i2, i3;
      tto_split(t, r, &i1, &i2, &i3);
      if (c->dW) {
        /* d<grad_out, out>/dw_l = <grad_out[b], row(r)> */
        tto_prefix(t, i1, i2, T12);
        tto_row(t, T12, i3, row);
        double s = 0.0;
        for (int j = 0; j < D; ++j) s += (double)gb[j] * row[j];
        c->dW[l] = s;
      }
      if (c->filter_core == 1 && i1 != c->filter_value) continue;
      if (c->filter_core == 2 && i2 != c->filter_value) continue;
      if (c->filter_core == 3 && i3 != c->filter_value) continue;
      /* the lookup's row enters out[b] with the factor w_l (weighted sum),
       * 1/len (mean) or 1 (sum): its share of grad_out[b] is that factor times it */
      double f = c->weights ? (double)c->weights[l] : (c->mean ? 1.0 / (double)len : 1.0);
      for (int j = 0; j < D; ++j) g[j] = f * (double)gb[j];
      tto_prefix(t, i1, i2, T12);
      /* dG3[i3][b][j3] += sum_{j12} T12[j12][b] * g[j12][j3] */
      for (int bb = 0; bb < R2; ++bb)
        for (int j3 = 0; j3 < n3; ++j3) {
          double s = 0.0;
          for (int j12 = 0; j12 < n1 * n2; ++j12)
            s += T12[j12 * R2 + bb] * g[j12 * n3 + j3];
          dG3[(i3 * R2 + bb) * n3 + j3] += s;
        }
      /* dT12[j12][b] = sum_{j3} g[j12][j3] * G3[i3][b][j3] */
      for (int j12 = 0; j12 < n1 * n2; ++j12)
        for (int bb = 0; bb < R2; ++bb) {
          double s = 0.0;
          for (int j3 = 0; j3 < n3; ++j3) s += g[j12 * n3 + j3] * g3(t, i3, bb, j3);
          dT12[j12 * R2 + bb] = s;
        }
      /* dG2[i2][a][j2][b] += sum_{j1} G1[i1][j1][a] * dT12[j1][j2][b] */
      for (int a = 0; a < R1; ++a)
        for (int j2 = 0; j2 < n2; ++j2)
          for (int bb = 0; bb < R2; ++bb) {
            double s = 0.0;
            for (int j1 = 0; j1 < n1; ++j1) s += g1(t, i1, j1, a) * dT12[(j1 * n2 + j2) * R2 + bb];
            dG2[((i2 * R1 + a) * n2 + j2) * R2 + bb] += s;
          }
      /* dG1[i1][j1][a] += sum_{j2,b} dT12[j1][j2][b] * G2[i2][a][j2][b] */
      for (int j1 = 0; j1 < n1; ++j1)
        for (int a = 0; a < R1; ++a) {
          double s = 0.0;
          for (int j2 = 0; j2 < n2; ++j2)
            for (int bb = 0; bb < R2; ++bb)
              s += dT12[(j1 * n2 + j2) * R2 + bb] * g2(t, i2, a, j2, bb);
          dG1[(i1 * n1 + j1) * R1 + a] += s;
        }
    }
  }
  free(T12);
  free(dT12);
  free(g);
  free(row);
}

/* dG1, dG2, dG3: double, same layouts as the cores, ACCUMULATED (+=).
 * filter_core in 1..3 restricts the sum to lookups whose i_k equals
 * filter_value, which gives slice filter_value of dG_k exactly at a fraction
 * of the cost (the other slices then hold partial sums).  weights / mean as
 * for tto_forward_ex; dW (double [nnz], overwritten; needs weights and no
 * filter) receives the gradient of the weights, 0 for out-of-range lookups. */
int tto_backward_ex(const float *grad_out, const float *G1, const float *G2, const float *G3,
                    const int64_t *m, const int32_t *n, const int32_t *R, const int64_t *indices,
                    int64_t nnz, const int64_t *offsets, int64_t B, const float *weights,
                    int mean, double *dG1, double *dG2, double *dG3, double *dW,
                    int filter_core, int64_t filter_value, int threads) {
  tto_bwd_ctx c;
  int e = tto_init(&c.t, G1, G2, G3, m, n, R);
  if (e) return e;
  if (nnz < 0 || (nnz > 0 && !indices) || (B > 0 && !grad_out)) return TTO_ERR_ARG;
  if (!dG1 || !dG2 || !dG3 || filter_core < 0 || filter_core > 3) return TTO_ERR_ARG;
  if ((mean && weights) || (dW && (!weights || filter_core != 0))) return TTO_ERR_ARG;
  e = tto_check_offsets(offsets, B, nnz);
  if (e) return e;
  c.indices = indices; c.offsets = offsets; c.grad_out = grad_out;
  c.weights = weights; c.mean = mean != 0; c.dW = dW;
  c.filter_core = filter_core; c.filter_value = filter_value;
  c.n1g = (size_t)m[0] * n[0] * R[1];
  c.n2g = (size_t)m[1] * R[1] * n[1] * R[2];
  c.n3g = (size_t)m[2] * R[2] * n[2];
  size_t per = c.n1g + c.n2g + c.n3g;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  double *scratch = (double *)calloc(per * (size_t)threads, sizeof(double));
  if (!scratch) return TTO_ERR_NOMEM;
  tto_job jobs[256];
  for (int k = 0; k < threads; ++k) jobs[k].scratch = scratch + per * (size_t)k;
  e = tto_parallel(tto_bwd_bags, &c, B, threads, jobs);
  /* reduce the per-thread sums in thread order */
  for (int k = 0; k < threads; ++k) {
    const double *s = scratch + per * (size_t)k;
    for (size_t i = 0; i < c.n1g; ++i) dG1[i] += s[i];
    for (size_t i = 0; i < c.n2g; ++i) dG2[i] += s[c.n1g + i];
    for (size_t i = 0; i < c.n3g; ++i) dG3[i] += s[c.n1g + c.n2g + i];
  }
  free(scratch);
  return e;
}

/* Plain sum pooling. */
int tto_backward(const float *grad_out, const float *G1, const float *G2, const float *G3,
                 const int64_t *m, const int32_t *n, const int32_t *R, const int64_t *indices,
                 int64_t nnz, const int64_t *offsets, int64_t B, double *dG1, double *dG2,
                 double *dG3, int filter_core, int64_t filter_value, int threads) {
  return tto_backward_ex(grad_out, G1, G2, G3, m, n, R, indices, nnz, offsets, B, NULL, 0, dG1,
                         dG2, dG3, NULL, filter_core, filter_value, threads);
}

/* out[i] = G[i] - lr * dG[i] in fp64. */
void tto_sgd(const float *G, const double *dG, int64_t count, double lr, double *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = (double)G[i] - lr * dG[i];
}

/* ---------------- grouping reference ---------------- */

typedef struct {
  uint64_t key;   /* (i2*m1 + i1)*m3 + i3 */
  int64_t l;      /* lookup position */
} tto_kl;

static int tto_kl_cmp(const void *pa, const void *pb) {
  const tto_kl *a = (const tto_kl *)pa, *b = (const tto_kl *)pb;
  if (a->key != b->key) return a->key < b->key ? -1 : 1;
  return a->l < b->l ? -1 : (a->l > b->l ? 1 : 0);
}

/* Sorts the valid lookups by (key, l) with key = (i2*m1 + i1)*m3 + i3 and
 * reports the unique runs.  Output arrays must hold nnz (+1) entries:
 *   perm[k]            lookup position of the k-th sorted valid lookup
 *   row_start[u]       first sorted position of unique row u (row_start[U_r] = n_valid)
 *   row_index[u]       the row index r of unique row u
 *   row_pair[u]        the unique prefix (pair) that row u belongs to
 *   pair_row_start[p]  first unique row of pair p (pair_row_start[U_12] = U_r)
 *   pair_i1[p], pair_i2[p]
 *   uid[l]             unique row of lookup l, -1 for an out-of-range index
 *   counts[0..2]       n_valid, U_r, U_12
 * Returns TTO_ERR_INDEX if any index was out of range (the rest is still valid). */
int tto_group(const int64_t *indices, int64_t nnz, const int64_t *m, int32_t *perm,
              int32_t *row_start, int64_t *row_index, int32_t *row_pair,
              int32_t *pair_row_start, int32_t *pair_i1, int32_t *pair_i2, int32_t *uid,
              int64_t *counts) {
  if (!m || nnz < 0 || (nnz > 0 && !indices)) return TTO_ERR_ARG;
  int64_t m1 = m[0], m2 = m[1], m3 = m[2], M = m1 * m2 * m3;
  tto_kl *kl = (tto_kl *)malloc(sizeof(tto_kl) * (size_t)(nnz > 0 ? nnz : 1));
  if (!kl) return TTO_ERR_NOMEM;
  int err = TTO_OK;
  int64_t nv = 0;
  for (int64_t l = 0; l < nnz; ++l) {
    int64_t r = indices[l];
    uid[l] = -1;
    if (r < 0 || r >= M) { err = TTO_ERR_INDEX; continue; }
    int64_t i3 = r % m3, i2 = (r / m3) % m2, i1 = r / (m2 * m3);
    kl[nv].key = (uint64_t)((i2 * m1 + i1) * m3 + i3);
    kl[nv].l = l;
    ++nv;
  }
  qsort(kl, (size_t)nv, sizeof(tto_kl), tto_kl_cmp);
  int64_t ur = 0, up = 0;
  for (int64_t k = 0; k < nv; ++k) {
    uint64_t key = kl[k].key;
    int new_row = (k == 0) || key != kl[k - 1].key;
    int new_pair = (k == 0) || (key / (uint64_t)m3) != (kl[k - 1].key / (uint64_t)m3);
    if (new_pair) {
      uint64_t q = key / (uint64_t)m3;
      pair_row_start[up] = (int32_t)ur;
      pair_i1[up] = (int32_t)(q % (uint64_t)m1);
      pair_i2[up] = (int32_t)(q / (uint64_t)m1);
      ++up;
    }
    if (new_row) {
      int64_t i3 = (int64_t)(key % (uint64_t)m3);
      row_start[ur] = (int32_t)k;
      row_index[ur] = ((int64_t)pair_i1[up - 1] * m2 + pair_i2[up - 1]) * m3 + i3;
      row_pair[ur] = (int32_t)(up - 1);
      ++ur;
    }
    perm[k] = (int32_t)kl[k].l;
    uid[kl[k].l] = (int32_t)(ur - 1);
  }
  row_start[ur] = (int32_t)nv;
  pair_row_start[up] = (int32_t)ur;
  counts[0] = nv;
  counts[1] = ur;
  counts[2] = up;
  free(kl);
  return err;
}

/* ---------------- d cores ----------------
 *
 * The same definitions for a chain of d >= 2 cores (the pages contract a
 * chain of cores without fixing their number, FlowTT summary card, problem
 * statement; three cores is the case above).  Core k (0-based) is float32
 * [m_k][R_k][n_k][R_{k+1}] with R_0 = R_d = 1; the row index splits
 * mixed-radix with i_0 most significant, the output position likewise with
 * j_0 most significant.  Per lookup the chain T_0 = G_0[i_0] (n_0 x R_1),
 * T_k = T_{k-1} . G_k[i_k] ((n_0..n_{k-1}) x R_k times R_k x (n_k R_{k+1}),
 * viewed as (n_0..n_k) x R_{k+1}), row = T_{d-1}; bags are summed.  The
 * backward keeps the chain and walks it back: dG_k[i_k] += T_{k-1}^T . dT_k,
 * dT_{k-1} = dT_k . G_k[i_k]^T, dG_0[i_0] += dT_0. */

#define TTO_MAXD 8

typedef struct {
  int d;
  const float *G[TTO_MAXD];
  int64_t m[TTO_MAXD];
  int n[TTO_MAXD], R[TTO_MAXD + 1];
  int64_t M;
  int D;
} tto_ttd;

static int tto_initd(tto_ttd *t, int d, const float *const *G, const int64_t *m, const int32_t *n,
                     const int32_t *R) {
  if (d < 2 || d > TTO_MAXD || !G || !m || !n || !R) return TTO_ERR_ARG;
  if (R[0] != 1 || R[d] != 1) return TTO_ERR_ARG;
  t->d = d;
  t->M = 1;
  t->D = 1;
  t->R[0] = 1;
  for (int k = 0; k < d; ++k) {
    if (!G[k] || m[k] < 1 || n[k] < 1 || R[k + 1] < 1) return TTO_ERR_ARG;
    t->G[k] = G[k];
    t->m[k] = m[k];
    t->n[k] = n[k];
    t->R[k + 1] = R[k + 1];
    t->M *= m[k];
    t->D *= n[k];
  }
  return TTO_OK;
}

/* digits of r, i_0 most significant */
static void tto_splitd(const tto_ttd *t, int64_t r, int64_t *ik) {
  for (int k = t->d - 1; k >= 0; --k) {
    ik[k] = r % t->m[k];
    r /= t->m[k];
  }
}

/* chain T_0 .. T_{d-1} of one lookup into T (T_k at offset off[k]; N_k = n_0..n_k rows) */
static void tto_chaind(const tto_ttd *t, const int64_t *ik, double *T, const size_t *off) {
  int N = t->n[0];
  const float *g0 = t->G[0] + ik[0] * (int64_t)t->n[0] * t->R[1];
  for (int e = 0; e < N * t->R[1]; ++e) T[off[0] + e] = (double)g0[e];
  for (int k = 1; k < t->d; ++k) {
    const int Ra = t->R[k], nk = t->n[k], Rb = t->R[k + 1];
    const float *gk = t->G[k] + ik[k] * (int64_t)Ra * nk * Rb;
    const double *A = T + off[k - 1];
    double *C = T + off[k];
    for (int J = 0; J < N; ++J)
      for (int j = 0; j < nk; ++j)
        for (int b = 0; b < Rb; ++b) {
          double s = 0.0;
          for (int a = 0; a < Ra; ++a) s += A[J * Ra + a] * (double)gk[(a * nk + j) * Rb + b];
          C[(J * nk + j) * Rb + b] = s;
        }
    N *= nk;
  }
}

static size_t tto_chain_offsets(const tto_ttd *t, size_t *off) {
  size_t o = 0;
  int N = 1;
  for (int k = 0; k < t->d; ++k) {
    N *= t->n[k];
    off[k] = o;
    o += (size_t)N * t->R[k + 1];
  }
  return o;
}

/* out: double [B][D], overwritten; as tto_forward for d cores (sum pooling). */
int tto_forward_d(int d, const float *const *G, const int64_t *m, const int32_t *n,
                  const int32_t *R, const int64_t *indices, int64_t nnz, const int64_t *offsets,
                  int64_t B, double *out) {
  tto_ttd t;
  int e = tto_initd(&t, d, G, m, n, R);
  if (e) return e;
  if (nnz < 0 || (nnz > 0 && !indices) || (B > 0 && !out)) return TTO_ERR_ARG;
  e = tto_check_offsets(offsets, B, nnz);
  if (e) return e;
  size_t off[TTO_MAXD];
  const size_t tot = tto_chain_offsets(&t, off);
  double *T = (double *)malloc(sizeof(double) * tot);
  if (!T) return TTO_ERR_NOMEM;
  int err = TTO_OK;
  int64_t ik[TTO_MAXD];
  for (int64_t b = 0; b < B; ++b) {
    double *o = out + b * t.D;
    for (int j = 0; j < t.D; ++j) o[j] = 0.0;
    for (int64_t l = offsets[b]; l < offsets[b + 1]; ++l) {
      const int64_t r = indices[l];
      if (r < 0 || r >= t.M) { err = TTO_ERR_INDEX; continue; }
      tto_splitd(&t, r, ik);
      tto_chaind(&t, ik, T, off);
      const double *row = T + off[d - 1];
      for (int j = 0; j < t.D; ++j) o[j] += row[j];
    }
  }
  free(T);
  return err;
}

/* dG[k]: double, same layouts as the cores, ACCUMULATED (+=). */
int tto_backward_d(int d, const float *grad_out, const float *const *G, const int64_t *m,
                   const int32_t *n, const int32_t *R, const int64_t *indices, int64_t nnz,
                   const int64_t *offsets, int64_t B, double *const *dG) {
  tto_ttd t;
  int e = tto_initd(&t, d, G, m, n, R);
  if (e) return e;
  if (nnz < 0 || (nnz > 0 && !indices) || (B > 0 && !grad_out) || !dG) return TTO_ERR_ARG;
  for (int k = 0; k < d; ++k)
    if (!dG[k]) return TTO_ERR_ARG;
  e = tto_check_offsets(offsets, B, nnz);
  if (e) return e;
  size_t off[TTO_MAXD];
  const size_t tot = tto_chain_offsets(&t, off);
  double *T = (double *)malloc(sizeof(double) * tot);
  double *dT = (double *)malloc(sizeof(double) * tot);
  if (!T || !dT) { free(T); free(dT); return TTO_ERR_NOMEM; }
  int err = TTO_OK;
  int64_t ik[TTO_MAXD];
  for (int64_t b = 0; b < B; ++b) {
    const float *g = grad_out + b * t.D;
    for (int64_t l = offsets[b]; l < offsets[b + 1]; ++l) {
      const int64_t r = indices[l];
      if (r < 0 || r >= t.M) { err = TTO_ERR_INDEX; continue; }
      tto_splitd(&t, r, ik);
      tto_chaind(&t, ik, T, off);
      for (int j = 0; j < t.D; ++j) dT[off[d - 1] + j] = (double)g[j];
      int N = t.D;
      for (int k = d - 1; k >= 1; --k) {
        const int Ra = t.R[k], nk = t.n[k], Rb = t.R[k + 1];
        N /= nk;                                   /* rows of T_{k-1} */
        const float *gk = t.G[k] + ik[k] * (int64_t)Ra * nk * Rb;
        double *dgk = dG[k] + ik[k] * (int64_t)Ra * nk * Rb;
        const double *A = T + off[k - 1], *dC = dT + off[k];
        double *dA = dT + off[k - 1];
        /* dG_k[i_k][a][j][b] += sum_J A[J][a] dC[(J, j)][b] */
        for (int a = 0; a < Ra; ++a)
          for (int j = 0; j < nk; ++j)
            for (int bb = 0; bb < Rb; ++bb) {
              double s = 0.0;
              for (int J = 0; J < N; ++J) s += A[J * Ra + a] * dC[(J * nk + j) * Rb + bb];
              dgk[(a * nk + j) * Rb + bb] += s;
            }
        /* dA[J][a] = sum_{j, b} dC[(J, j)][b] G_k[i_k][a][j][b] */
        for (int J = 0; J < N; ++J)
          for (int a = 0; a < Ra; ++a) {
            double s = 0.0;
            for (int j = 0; j < nk; ++j)
              for (int bb = 0; bb < Rb; ++bb)
                s += dC[(J * nk + j) * Rb + bb] * (double)gk[(a * nk + j) * Rb + bb];
            dA[J * Ra + a] = s;
          }
      }
      double *dg0 = dG[0] + ik[0] * (int64_t)t.n[0] * t.R[1];
      for (int e2 = 0; e2 < t.n[0] * t.R[1]; ++e2) dg0[e2] += dT[off[0] + e2];
    }
  }
  free(T);
  free(dT);
  return err;
}
