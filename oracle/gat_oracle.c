/*
 * Plain fp64 CPU oracle for the fused GAT neighbour aggregation.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (per destination node i and head k):
 *   s_dst(i,k) = a_dst[k] . h[i][k]       s_src(j,k) = a_src[k] . h[j][k]
 *   z_ij = s_dst(i,k) + s_src(j,k)        e_ij = LeakyReLU(z_ij) (slope for z <= 0)
 *   alpha_ij = softmax over the in-neighbours j of i of e_ij
 *   out[i][k] = sum_j alpha_ij h[j][k]    lse(i,k) = log sum_j exp(e_ij)
 * The score is the additive single-layer attention of Graph Attention Networks
 * (Velickovic et al., ICLR 2018, eqs. 1-3), with the projection W applied
 * outside this operation and a = [a_dst || a_src] split into its two halves.
 * "On Efficient Scaling of GNNs via IO-Aware Layers Implementations",
 * Technical Summary > Methodology, attention-based layers: score computation,
 * softmax normalisation and value aggregation over a node's neighbours, with a
 * per-node log-sum-exp kept for the backward pass.  This oracle reaches that
 * result by the textbook two-pass softmax (max, then sum of exponentials),
 * not by the streaming form, so it shares no algorithm with the GPU kernels.
 *
 * Backward: the gradient of L = sum(out * dout) w.r.t. h, a_src and a_dst,
 * written out by the chain rule:
 *   da_ij  = dout[i][k] . h[j][k]              (d L / d alpha_ij)
 *   Delta_i = sum_j alpha_ij da_ij
 *   de_ij  = alpha_ij (da_ij - Delta_i)        (softmax Jacobian)
 *   dz_ij  = de_ij * (z_ij > 0 ? 1 : slope)    (LeakyReLU; slope at z = 0)
 *   ds_dst(i) = sum_j dz_ij,  ds_src(j) = sum_{i : j in N(i)} dz_ij
 *   dh[j]  = sum_i alpha_ij dout[i] + ds_src(j) a_src + ds_dst(j) a_dst
 *   da_src = sum_j ds_src(j) h[j],  da_dst = sum_i ds_dst(i) h[i]
 * Multi-edges count with their multiplicity.  A node with no in-neighbours has
 * out = 0, lse = -inf and contributes nothing as a destination.
 *
 * Inputs: the exact arrays given to the GPU (float32, or bfloat16 bit
 * patterns), widened exactly to double as they are read; float64 features are
 * also accepted (finite-difference checks).  a_src / a_dst are passed as
 * double (float32 values widen exactly).  All outputs double.
 * Optional "mag" outputs give, per output element, the sum of the absolute
 * values of the terms that make it up (used by tests to bound float32
 * summation error where a result cancels).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int64_t n;
  const int32_t* row_ptr;
  const int32_t* col;
  int H, D, dtype; /* dtype 0: float32, 1: bfloat16 bit patterns, 2: float64 */
  const void* h;
  const double* a_src;
  const double* a_dst;
  double slope;
} gat_inputs;

static double widen(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  if (dtype == 2) return ((const double*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double feat(const gat_inputs* g, const void* arr, int64_t node, int k, int d) {
  return widen(arr, g->dtype, (node * g->H + k) * (int64_t)g->D + d);
}

static double leaky(double z, double slope) { return z > 0.0 ? z : slope * z; }
static double leaky_grad(double z, double slope) { return z > 0.0 ? 1.0 : slope; }

/* a[k] . x[v][k] in double */
static double head_dot(const gat_inputs* g, const double* a, const void* x, int64_t v, int k) {
  double s = 0.0;
  for (int d = 0; d < g->D; ++d) s += a[k * g->D + d] * feat(g, x, v, k, d);
  return s;
}

static int64_t max_in_degree(const gat_inputs* g) {
  int64_t m = 0;
  for (int64_t i = 0; i < g->n; ++i) {
    int64_t d = (int64_t)g->row_ptr[i + 1] - g->row_ptr[i];
    if (d > m) m = d;
  }
  return m;
}

/*
 * Two-pass softmax over the in-neighbours of (i, k).  Fills z[q] and alpha[q]
 * for q = 0 .. deg(i)-1 and returns the log-sum-exp (-inf when deg(i) = 0).
 */
static double row_softmax(const gat_inputs* g, int64_t i, int k, double* z, double* alpha) {
  const int64_t b = g->row_ptr[i], deg = (int64_t)g->row_ptr[i + 1] - b;
  if (deg <= 0) return -INFINITY;
  const double sd = head_dot(g, g->a_dst, g->h, i, k);
  double m = -INFINITY;
  for (int64_t q = 0; q < deg; ++q) {
    const int64_t j = g->col[b + q];
    z[q] = sd + head_dot(g, g->a_src, g->h, j, k);
    const double e = leaky(z[q], g->slope);
    alpha[q] = e;
    if (e > m) m = e;
  }
  double l = 0.0;
  for (int64_t q = 0; q < deg; ++q) l += exp(alpha[q] - m);
  for (int64_t q = 0; q < deg; ++q) alpha[q] = exp(alpha[q] - m) / l;
  return m + log(l);
}

/*
 * Destination-side statistics of (i, k): fills da[q] = dout_i . h_j for every
 * in-edge and returns Delta_i; *ds_dst = sum_q dz_iq and *dz_mag = the sum of
 * |alpha| (|da| + |Delta|) over the edges.
 */
static double row_backward_stats(const gat_inputs* g, const void* dout, int64_t i, int k,
                                 const double* z, const double* alpha, double* da,
                                 double* ds_dst, double* dz_mag) {
  const int64_t b = g->row_ptr[i], deg = (int64_t)g->row_ptr[i + 1] - b;
  double delta = 0.0;
  for (int64_t q = 0; q < deg; ++q) {
    const int64_t j = g->col[b + q];
    double s = 0.0;
    for (int d = 0; d < g->D; ++d) s += feat(g, dout, i, k, d) * feat(g, g->h, j, k, d);
    da[q] = s;
    delta += alpha[q] * s;
  }
  double ds = 0.0, mag = 0.0;
  for (int64_t q = 0; q < deg; ++q) {
    ds += alpha[q] * (da[q] - delta) * leaky_grad(z[q], g->slope);
    mag += alpha[q] * (fabs(da[q]) + fabs(delta));
  }
  *ds_dst = ds;
  *dz_mag = mag;
  return delta;
}

/* sum_d |a[k][d] x[v][k][d]|: the size of a score half, for the rounding
 * bound of its float32 value. */
static double head_dot_mag(const gat_inputs* g, const double* a, const void* x, int64_t v, int k) {
  double s = 0.0;
  for (int d = 0; d < g->D; ++d) s += fabs(a[k * g->D + d] * feat(g, x, v, k, d));
  return s;
}

/* Largest |z| at which a float32 evaluation of z = s_dst(i) + s_src(j) (two
 * sums of D products, then their sum) can still have the wrong sign: the
 * worst-case rounding bound (D + 2) 2^-24 (|s_dst|_mag + |s_src|_mag), with a
 * factor of two to spare. */
static double kink_width(const gat_inputs* g, double mag_dst, double mag_src) {
  return (double)(g->D + 4) * ldexp(1.0, -23) * (mag_dst + mag_src);
}

/*
 * The LeakyReLU derivative of an edge is a decision on the sign of z_ij.
 * Within the rounding bound of a float32 z both derivatives are results of
 * the method at that precision, so a check must accept either.  amb[q]
 * (q = 0 .. deg(i)-1) receives |1 - slope| alpha_q |da_q - Delta| for the
 * in-edges of (i, k) whose |z| is within that bound and 0 for the others:
 * how far dz_iq, and with it ds_dst(i) and ds_src(j), can move between the
 * two derivatives.  Returns the sum over the row.
 */
static double row_kink(const gat_inputs* g, int64_t i, int k, const double* z,
                       const double* alpha, const double* da, double delta, double* amb) {
  const int64_t b = g->row_ptr[i], deg = (int64_t)g->row_ptr[i + 1] - b;
  const double md = head_dot_mag(g, g->a_dst, g->h, i, k);
  double tot = 0.0;
  for (int64_t q = 0; q < deg; ++q) {
    const int64_t j = g->col[b + q];
    const double tau = kink_width(g, md, head_dot_mag(g, g->a_src, g->h, j, k));
    amb[q] = fabs(z[q]) <= tau ? fabs(1.0 - g->slope) * alpha[q] * fabs(da[q] - delta) : 0.0;
    tot += amb[q];
  }
  return tot;
}

static int check_inputs(const gat_inputs* g) {
  if (g->n < 0 || g->H < 1 || g->D < 1 || g->dtype < 0 || g->dtype > 2) return 1;
  if (!g->row_ptr || (g->n > 0 && (!g->h || !g->a_src || !g->a_dst))) return 1;
  if (g->row_ptr[0] != 0) return 2;
  for (int64_t i = 0; i < g->n; ++i)
    if (g->row_ptr[i + 1] < g->row_ptr[i]) return 2;
  const int64_t E = g->row_ptr[g->n];
  for (int64_t p = 0; p < E; ++p)
    if (g->col[p] < 0 || g->col[p] >= g->n) return 2;
  return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for the oracle's later parallel regions (timing on fewer cores). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * Forward.  sel = NULL computes every node (n_out = n); otherwise the n_sel
 * listed nodes, output row t belonging to node sel[t].
 * out [n_out][H][D], lse [n_out][H]; out_mag and alpha_sum may be NULL.
 * Returns 0, or nonzero for bad arguments / an invalid CSR.
 */
int oracle_gat_forward(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                       int dtype, const void* h, const double* a_src, const double* a_dst,
                       double slope, int64_t n_sel, const int64_t* sel, double* out,
                       double* lse, double* out_mag, double* alpha_sum) {
  gat_inputs g = {n, row_ptr, col, H, D, dtype, h, a_src, a_dst, slope};
  int rc = check_inputs(&g);
  if (rc) return rc;
  const int64_t n_out = sel ? n_sel : n;
  for (int64_t t = 0; sel && t < n_sel; ++t)
    if (sel[t] < 0 || sel[t] >= n) return 1;
  const int64_t maxdeg = max_in_degree(&g);
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t t = 0; t < n_out; ++t) {
      const int64_t i = sel ? sel[t] : t;
      const int64_t b = row_ptr[i], deg = (int64_t)row_ptr[i + 1] - b;
      for (int k = 0; k < H; ++k) {
        const double l = row_softmax(&g, i, k, z, alpha);
        lse[t * H + k] = l;
        double asum = 0.0;
        for (int64_t q = 0; q < deg; ++q) asum += alpha[q];
        if (alpha_sum) alpha_sum[t * H + k] = asum;
        for (int d = 0; d < D; ++d) {
          double acc = 0.0, mag = 0.0;
          for (int64_t q = 0; q < deg; ++q) {
            const double x = feat(&g, h, col[b + q], k, d);
            acc += alpha[q] * x;
            mag += alpha[q] * fabs(x);
          }
          out[(t * H + k) * (int64_t)D + d] = acc;
          if (out_mag) out_mag[(t * H + k) * (int64_t)D + d] = mag;
        }
      }
    }
    free(z);
    free(alpha);
  }
  return 0;
}

/*
 * Per-node destination statistics for the n_sel listed nodes (sel = NULL: all):
 * lse, Delta = sum_j alpha_ij (dout_i . h_j) and ds_dst, each [n_out][H].
 */
int oracle_gat_node_stats(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                          int dtype, const void* h, const double* a_src, const double* a_dst,
                          double slope, const void* dout, int64_t n_sel, const int64_t* sel,
                          double* lse, double* delta, double* ds_dst) {
  gat_inputs g = {n, row_ptr, col, H, D, dtype, h, a_src, a_dst, slope};
  int rc = check_inputs(&g);
  if (rc) return rc;
  if (!dout && n > 0) return 1;
  const int64_t n_out = sel ? n_sel : n;
  for (int64_t t = 0; sel && t < n_sel; ++t)
    if (sel[t] < 0 || sel[t] >= n) return 1;
  const int64_t maxdeg = max_in_degree(&g);
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t t = 0; t < n_out; ++t) {
      const int64_t i = sel ? sel[t] : t;
      for (int k = 0; k < H; ++k) {
        double ds = 0.0, mag = 0.0, dl = 0.0;
        const double l = row_softmax(&g, i, k, z, alpha);
        if (row_ptr[i + 1] > row_ptr[i]) dl = row_backward_stats(&g, dout, i, k, z, alpha, da, &ds, &mag);
        if (lse) lse[t * H + k] = l;
        if (delta) delta[t * H + k] = dl;
        if (ds_dst) ds_dst[t * H + k] = ds;
      }
    }
    free(z);
    free(alpha);
    free(da);
  }
  return 0;
}

/*
 * Backward over the whole graph: dh [n][H][D], da_src and da_dst [H][D].
 * dh_mag [n][H][D] and da_mag [2][H][D] (src, dst) may be NULL, and so may
 * dh_kink [n][H][D] and da_kink [2][H][D]: per element, how far the result
 * can move between the two LeakyReLU derivatives of edges at the kink
 * (row_kink).  Destination statistics are computed in parallel over nodes;
 * the source-side scatter runs in edge order on one thread, so the result is
 * deterministic.
 */
int oracle_gat_backward(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                        int dtype, const void* h, const double* a_src, const double* a_dst,
                        double slope, const void* dout, double* dh, double* da_src,
                        double* da_dst, double* dh_mag, double* da_mag, double* dh_kink,
                        double* da_kink) {
  gat_inputs g = {n, row_ptr, col, H, D, dtype, h, a_src, a_dst, slope};
  int rc = check_inputs(&g);
  if (rc) return rc;
  if (!dout && n > 0) return 1;
  const int64_t NH = n * H, NHD = NH * D;
  const int64_t maxdeg = max_in_degree(&g);
  double* ds_dst = (double*)calloc((size_t)NH + 1, sizeof(double));
  double* ds_src = (double*)calloc((size_t)NH + 1, sizeof(double));
  double* delta = (double*)calloc((size_t)NH + 1, sizeof(double));
  double* mag_dst = (double*)calloc((size_t)NH + 1, sizeof(double));
  double* mag_src = (double*)calloc((size_t)NH + 1, sizeof(double));
  const int kink = dh_kink || da_kink;
  double* kink_dst = kink ? (double*)calloc((size_t)NH + 1, sizeof(double)) : NULL;
  double* kink_src = kink ? (double*)calloc((size_t)NH + 1, sizeof(double)) : NULL;
  if (!ds_dst || !ds_src || !delta || !mag_dst || !mag_src || (kink && (!kink_dst || !kink_src))) {
    free(ds_dst); free(ds_src); free(delta); free(mag_dst); free(mag_src);
    free(kink_dst); free(kink_src);
    return 3;
  }
  /* destination side: Delta_i and ds_dst(i) */
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* amb = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t i = 0; i < n; ++i) {
      if (row_ptr[i + 1] == row_ptr[i]) continue;
      for (int k = 0; k < H; ++k) {
        row_softmax(&g, i, k, z, alpha);
        delta[i * H + k] = row_backward_stats(&g, dout, i, k, z, alpha, da, &ds_dst[i * H + k],
                                              &mag_dst[i * H + k]);
        if (kink) kink_dst[i * H + k] = row_kink(&g, i, k, z, alpha, da, delta[i * H + k], amb);
      }
    }
    free(z);
    free(alpha);
    free(da);
    free(amb);
  }
  /* source side: scatter alpha_ij dout_i and dz_ij onto j, in edge order */
  memset(dh, 0, sizeof(double) * (size_t)NHD);
  if (dh_mag) memset(dh_mag, 0, sizeof(double) * (size_t)NHD);
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    for (int64_t i = 0; i < n; ++i) {
      const int64_t b = row_ptr[i], deg = (int64_t)row_ptr[i + 1] - b;
      if (deg == 0) continue;
      for (int k = 0; k < H; ++k) {
        row_softmax(&g, i, k, z, alpha);
        const double dl = delta[i * H + k];
        for (int64_t q = 0; q < deg; ++q) {
          const int64_t j = col[b + q];
          double da = 0.0;
          for (int d = 0; d < D; ++d) da += feat(&g, dout, i, k, d) * feat(&g, h, j, k, d);
          ds_src[j * H + k] += alpha[q] * (da - dl) * leaky_grad(z[q], slope);
          mag_src[j * H + k] += alpha[q] * (fabs(da) + fabs(dl));
          if (kink &&
              fabs(z[q]) <= kink_width(&g, head_dot_mag(&g, a_dst, h, i, k),
                                       head_dot_mag(&g, a_src, h, j, k)))
            kink_src[j * H + k] += fabs(1.0 - slope) * alpha[q] * fabs(da - dl);
          for (int d = 0; d < D; ++d) {
            const double x = feat(&g, dout, i, k, d);
            dh[(j * H + k) * (int64_t)D + d] += alpha[q] * x;
            if (dh_mag) dh_mag[(j * H + k) * (int64_t)D + d] += alpha[q] * fabs(x);
          }
        }
      }
    }
    free(z);
    free(alpha);
  }
  /* score terms and the attention-vector gradients */
  for (int k = 0; k < H; ++k)
    for (int d = 0; d < D; ++d) {
      da_src[k * D + d] = 0.0;
      da_dst[k * D + d] = 0.0;
      if (da_mag) da_mag[k * D + d] = da_mag[(H + k) * D + d] = 0.0;
      if (da_kink) da_kink[k * D + d] = da_kink[(H + k) * D + d] = 0.0;
    }
  for (int64_t j = 0; j < n; ++j)
    for (int k = 0; k < H; ++k)
      for (int d = 0; d < D; ++d) {
        const int64_t x = (j * H + k) * (int64_t)D + d;
        const double as = a_src[k * D + d], ad = a_dst[k * D + d], hv = feat(&g, h, j, k, d);
        dh[x] += ds_src[j * H + k] * as + ds_dst[j * H + k] * ad;
        if (dh_mag) dh_mag[x] += mag_src[j * H + k] * fabs(as) + mag_dst[j * H + k] * fabs(ad);
        da_src[k * D + d] += ds_src[j * H + k] * hv;
        da_dst[k * D + d] += ds_dst[j * H + k] * hv;
        if (da_mag) {
          da_mag[k * D + d] += mag_src[j * H + k] * fabs(hv);
          da_mag[(H + k) * D + d] += mag_dst[j * H + k] * fabs(hv);
        }
        if (dh_kink)
          dh_kink[x] = kink_src[j * H + k] * fabs(as) + kink_dst[j * H + k] * fabs(ad);
        if (da_kink) {
          da_kink[k * D + d] += kink_src[j * H + k] * fabs(hv);
          da_kink[(H + k) * D + d] += kink_dst[j * H + k] * fabs(hv);
        }
      }
  free(ds_dst); free(ds_src); free(delta); free(mag_dst); free(mag_src);
  free(kink_dst); free(kink_src);
  return 0;
}

/*
 * Backward for selected nodes only: dh rows of the n_sel listed (distinct)
 * nodes.  Row j gathers the value term and ds_src(j) from every edge j -> i
 * (found by a scan of the whole CSR, ascending edge position) and ds_dst(j)
 * from its own in-edges.  Two phases, so that a source with many
 * out-neighbours costs one pass over their rows, not one per edge:
 *   1. for every destination i that an edge from a listed node reaches, and
 *      for every listed node itself: the softmax statistics of each head,
 *      s_dst(i), lse_i, Delta_i (and ds_dst for the listed nodes), from the
 *      row's two-pass softmax;
 *   2. for each listed j and each such edge: alpha_ij = exp(e_ij - lse_i),
 *      da_ij = dout_i . h_j, dz_ij = alpha_ij (da_ij - Delta_i) g_ij, and
 *      dh_j = sum alpha_ij dout_i + ds_src(j) a_src + ds_dst(j) a_dst.
 * dh [n_sel][H][D]; dh_mag and dh_kink (as for oracle_gat_backward) may be
 * NULL.  Used where the whole-graph oracle would take too long.
 */
int oracle_gat_backward_rows(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                             int dtype, const void* h, const double* a_src, const double* a_dst,
                             double slope, const void* dout, int64_t n_sel, const int64_t* sel,
                             double* dh, double* dh_mag, double* dh_kink) {
  gat_inputs g = {n, row_ptr, col, H, D, dtype, h, a_src, a_dst, slope};
  int rc = check_inputs(&g);
  if (rc) return rc;
  if (!dout || !sel || n_sel < 0) return 1;
  int64_t* target = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  if (!target || !slot) { free(target); free(slot); return 3; }
  for (int64_t v = 0; v < n; ++v) target[v] = slot[v] = -1;
  for (int64_t t = 0; t < n_sel; ++t) {
    if (sel[t] < 0 || sel[t] >= n || target[sel[t]] >= 0) { free(target); free(slot); return 1; }
    target[sel[t]] = t;
  }
  /* out-edge lists of the targets: (destination i, edge position p - row_ptr[i]),
     ascending p; destinations needing statistics get a slot */
  int64_t* cnt = (int64_t*)calloc((size_t)n_sel + 1, sizeof(int64_t));
  const int64_t E = row_ptr[n];
  for (int64_t p = 0; p < E; ++p)
    if (target[col[p]] >= 0) cnt[target[col[p]] + 1]++;
  for (int64_t t = 0; t < n_sel; ++t) cnt[t + 1] += cnt[t];
  int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_sel + 1));
  int64_t* edge_dst = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cnt[n_sel] + 1));
  int64_t* edge_pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cnt[n_sel] + 1));
  memcpy(fill, cnt, sizeof(int64_t) * (size_t)(n_sel + 1));
  int64_t n_u = 0;
  for (int64_t i = 0; i < n; ++i) {
    int needed = target[i] >= 0;
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p)
      if (target[col[p]] >= 0) {
        const int64_t t = target[col[p]];
        edge_dst[fill[t]] = i;
        edge_pos[fill[t]] = p - row_ptr[i];
        fill[t]++;
        needed = 1;
      }
    if (needed) slot[i] = n_u++;
  }
  int64_t* u_node = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_u + 1));
  /* per slot and head: s_dst, lse, Delta, ds_dst, |dz| sum, |s_dst| size,
     kink ambiguity of ds_dst */
  enum { NS = 7 };
  double* st = (double*)malloc(sizeof(double) * (size_t)(NS * n_u * H + 1));
  for (int64_t i = 0; i < n; ++i)
    if (slot[i] >= 0) u_node[slot[i]] = i;
  const int64_t maxdeg = max_in_degree(&g);
  /* phase 1: statistics of every needed destination, from its own row */
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* amb = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t u = 0; u < n_u; ++u) {
      const int64_t i = u_node[u];
      for (int k = 0; k < H; ++k) {
        double* s = st + (u * H + k) * NS;
        s[0] = head_dot(&g, a_dst, h, i, k);
        s[1] = -INFINITY;
        s[2] = s[3] = s[4] = s[6] = 0.0;
        s[5] = head_dot_mag(&g, a_dst, h, i, k);
        if (row_ptr[i + 1] > row_ptr[i]) {
          s[1] = row_softmax(&g, i, k, z, alpha);
          s[2] = row_backward_stats(&g, dout, i, k, z, alpha, da, &s[3], &s[4]);
          if (dh_kink) s[6] = row_kink(&g, i, k, z, alpha, da, s[2], amb);
        }
      }
    }
    free(z);
    free(alpha);
    free(da);
    free(amb);
  }
  /* phase 2: each listed source from the statistics of its out-neighbours */
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < n_sel; ++t) {
    const int64_t j = sel[t];
    for (int k = 0; k < H; ++k) {
      double* row = dh + (t * H + k) * (int64_t)D;
      double* rmag = dh_mag ? dh_mag + (t * H + k) * (int64_t)D : NULL;
      for (int d = 0; d < D; ++d) {
        row[d] = 0.0;
        if (rmag) rmag[d] = 0.0;
      }
      const double ss = head_dot(&g, a_src, h, j, k);
      const double ss_mag = head_dot_mag(&g, a_src, h, j, k);
      double ds_src = 0.0, msrc = 0.0, ksrc = 0.0;
      for (int64_t x = cnt[t]; x < cnt[t + 1]; ++x) {
        const int64_t i = edge_dst[x];
        const double* s = st + (slot[i] * H + k) * NS;
        const double zz = s[0] + ss;
        const double alpha = exp(leaky(zz, slope) - s[1]);
        double da = 0.0;
        for (int d = 0; d < D; ++d) da += feat(&g, dout, i, k, d) * feat(&g, h, j, k, d);
        ds_src += alpha * (da - s[2]) * leaky_grad(zz, slope);
        msrc += alpha * (fabs(da) + fabs(s[2]));
        if (fabs(zz) <= kink_width(&g, s[5], ss_mag))
          ksrc += fabs(1.0 - slope) * alpha * fabs(da - s[2]);
        for (int d = 0; d < D; ++d) {
          const double xv = feat(&g, dout, i, k, d);
          row[d] += alpha * xv;
          if (rmag) rmag[d] += alpha * fabs(xv);
        }
      }
      const double* sj = st + (slot[j] * H + k) * NS;
      for (int d = 0; d < D; ++d) {
        const double as = a_src[k * D + d], ad = a_dst[k * D + d];
        row[d] += ds_src * as + sj[3] * ad;
        if (rmag) rmag[d] += msrc * fabs(as) + sj[4] * fabs(ad);
        if (dh_kink) dh_kink[(t * H + k) * (int64_t)D + d] = ksrc * fabs(as) + sj[6] * fabs(ad);
      }
    }
  }
  free(target); free(slot); free(cnt); free(fill); free(edge_dst); free(edge_pos);
  free(u_node); free(st);
  return 0;
}

/*
 * Attention-vector gradients only, summed per destination row so the work
 * parallelises over rows: da_src = sum_i sum_{j in N(i)} dz_ij h_j and
 * da_dst = sum_i ds_dst(i) h_i.  (The same sums as oracle_gat_backward's,
 * grouped by destination instead of by source.)  Rows are split statically
 * over threads and the per-thread float64 sums are added in thread order.
 * da_src, da_dst [H][D]; da_mag and da_kink [2][H][D] (as for
 * oracle_gat_backward) may be NULL.
 */
int oracle_gat_att_grads(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                         int dtype, const void* h, const double* a_src, const double* a_dst,
                         double slope, const void* dout, double* da_src, double* da_dst,
                         double* da_mag, double* da_kink) {
  gat_inputs g = {n, row_ptr, col, H, D, dtype, h, a_src, a_dst, slope};
  int rc = check_inputs(&g);
  if (rc) return rc;
  if (!dout && n > 0) return 1;
  const int64_t HD = (int64_t)H * D;
  const int64_t maxdeg = max_in_degree(&g);
  int nt = oracle_num_threads();
  /* per thread: src, dst, src mag, dst mag, src kink, dst kink */
  double* part = (double*)calloc((size_t)(nt * 6 * HD), sizeof(double));
  if (!part) return 3;
#pragma omp parallel num_threads(nt)
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    double* ps = part + (int64_t)t * 6 * HD;
    double* z = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* amb = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
      const int64_t b = row_ptr[i], deg = (int64_t)row_ptr[i + 1] - b;
      if (deg == 0) continue;
      for (int k = 0; k < H; ++k) {
        double ds, mag;
        row_softmax(&g, i, k, z, alpha);
        const double dl = row_backward_stats(&g, dout, i, k, z, alpha, da, &ds, &mag);
        const double kd = da_kink ? row_kink(&g, i, k, z, alpha, da, dl, amb) : 0.0;
        for (int64_t q = 0; q < deg; ++q) {
          const int64_t j = col[b + q];
          const double dz = alpha[q] * (da[q] - dl) * leaky_grad(z[q], slope);
          const double dm = alpha[q] * (fabs(da[q]) + fabs(dl));
          for (int d = 0; d < D; ++d) {
            const double x = feat(&g, h, j, k, d);
            ps[k * D + d] += dz * x;
            ps[2 * HD + k * D + d] += dm * fabs(x);
            if (da_kink) ps[4 * HD + k * D + d] += amb[q] * fabs(x);
          }
        }
        for (int d = 0; d < D; ++d) {
          const double x = feat(&g, h, i, k, d);
          ps[HD + k * D + d] += ds * x;
          ps[3 * HD + k * D + d] += mag * fabs(x);
          ps[5 * HD + k * D + d] += kd * fabs(x);
        }
      }
    }
    free(z);
    free(alpha);
    free(da);
    free(amb);
  }
  for (int64_t x = 0; x < HD; ++x) {
    double s = 0.0, d = 0.0, ms = 0.0, md = 0.0, ks = 0.0, kd = 0.0;
    for (int t = 0; t < nt; ++t) {
      s += part[(int64_t)t * 6 * HD + x];
      d += part[(int64_t)t * 6 * HD + HD + x];
      ms += part[(int64_t)t * 6 * HD + 2 * HD + x];
      md += part[(int64_t)t * 6 * HD + 3 * HD + x];
      ks += part[(int64_t)t * 6 * HD + 4 * HD + x];
      kd += part[(int64_t)t * 6 * HD + 5 * HD + x];
    }
    da_src[x] = s;
    da_dst[x] = d;
    if (da_mag) {
      da_mag[x] = ms;
      da_mag[HD + x] = md;
    }
    if (da_kink) {
      da_kink[x] = ks;
      da_kink[HD + x] = kd;
    }
  }
  free(part);
  return 0;
}
