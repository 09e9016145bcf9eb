/*
 * Plain fp64 CPU oracle for the fused GATv2 neighbour aggregation.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, per destination i and head k ("On Efficient Scaling of
 * GNNs via IO-Aware Layers Implementations", Technical Summary > Methodology,
 * attention-based layers, GATv2; the score of Brody, Alon and Yahav, "How
 * Attentive are Graph Attention Networks?", ICLR 2022, eq. 7, with the two
 * halves of W applied by the caller: xl = W_l h on the source side, which is
 * also the aggregated value, and xr = W_r h on the destination side):
 *   z_ij[d] = xr[i][k][d] + xl[j][k][d]
 *   e_ij    = sum_d att[k][d] LeakyReLU(z_ij[d])      (slope for z <= 0)
 *   alpha_ij = softmax over the in-neighbours j of i of e_ij
 *   out[i][k] = sum_j alpha_ij xl[j][k],   lse(i, k) = log sum_j exp(e_ij)
 * by the textbook two-pass softmax.  A node with no in-neighbours gets
 * out = 0 and lse = -inf.  Multi-edges count with their multiplicity.
 *
 * Backward of L = sum(out * dout), by the chain rule:
 *   da_ij  = dout[i][k] . xl[j][k],   Delta_i = sum_j alpha_ij da_ij
 *   de_ij  = alpha_ij (da_ij - Delta_i)
 *   dz_ij[d] = de_ij att[k][d] LeakyReLU'(z_ij[d])    (slope at z = 0)
 *   dxl[j] = sum_i (alpha_ij dout[i] + dz_ij),   dxr[i] = sum_j dz_ij
 *   datt[k][d] = sum_ij de_ij LeakyReLU(z_ij[d])
 *
 * Inputs: the exact arrays given to the GPU (float32 or bfloat16 bit
 * patterns, widened exactly; float64 accepted).  att as double.  Outputs
 * double.  "mag" outputs hold per element the sum of |terms| (tests bound
 * float32 rounding with them).
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
  int H, D, dtype;
  const void* xl;
  const void* xr;
  const double* att;
  double slope;
} v2_inputs;

static double v2_widen(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  if (dtype == 2) return ((const double*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double v2_feat(const v2_inputs* g, const void* a, int64_t v, int k, int d) {
  return v2_widen(a, g->dtype, ((int64_t)v * g->H + k) * g->D + d);
}

static double v2_leaky(double z, double s) { return z > 0.0 ? z : s * z; }
static double v2_leaky_grad(double z, double s) { return z > 0.0 ? 1.0 : s; }

static int v2_check(const v2_inputs* g) {
  if (g->n < 0 || g->H < 1 || g->D < 1 || g->dtype < 0 || g->dtype > 2 || !g->row_ptr) return 1;
  if (g->n > 0 && (!g->xl || !g->xr || !g->att)) return 1;
  if (g->row_ptr[0] != 0) return 2;
  for (int64_t i = 0; i < g->n; ++i)
    if (g->row_ptr[i + 1] < g->row_ptr[i]) return 2;
  for (int64_t p = 0; p < g->row_ptr[g->n]; ++p)
    if (g->col[p] < 0 || g->col[p] >= g->n) return 2;
  return 0;
}

static int64_t v2_max_deg(const v2_inputs* g) {
  int64_t m = 0;
  for (int64_t i = 0; i < g->n; ++i)
    if (g->row_ptr[i + 1] - g->row_ptr[i] > m) m = g->row_ptr[i + 1] - g->row_ptr[i];
  return m;
}

/* score e_ij of the edge at position p (source col[p]) of row i, head k */
static double v2_score(const v2_inputs* g, int64_t i, int64_t j, int k) {
  double e = 0.0;
  for (int d = 0; d < g->D; ++d)
    e += g->att[k * g->D + d] *
         v2_leaky(v2_feat(g, g->xr, i, k, d) + v2_feat(g, g->xl, j, k, d), g->slope);
  return e;
}

/* Two-pass softmax of row i, head k: alpha[q] for q < deg(i); returns lse. */
static double v2_softmax(const v2_inputs* g, int64_t i, int k, double* alpha) {
  const int64_t b = g->row_ptr[i], deg = g->row_ptr[i + 1] - b;
  if (deg == 0) return -INFINITY;
  double m = -INFINITY;
  for (int64_t q = 0; q < deg; ++q) {
    alpha[q] = v2_score(g, i, g->col[b + q], k);
    if (alpha[q] > m) m = alpha[q];
  }
  double l = 0.0;
  for (int64_t q = 0; q < deg; ++q) l += exp(alpha[q] - m);
  for (int64_t q = 0; q < deg; ++q) alpha[q] = exp(alpha[q] - m) / l;
  return m + log(l);
}

/* da[q] = dout_i . xl_j for every in-edge; returns Delta_i */
static double v2_delta(const v2_inputs* g, const void* dout, int64_t i, int k,
                       const double* alpha, double* da) {
  const int64_t b = g->row_ptr[i], deg = g->row_ptr[i + 1] - b;
  double delta = 0.0;
  for (int64_t q = 0; q < deg; ++q) {
    double s = 0.0;
    for (int d = 0; d < g->D; ++d)
      s += v2_feat(g, dout, i, k, d) * v2_feat(g, g->xl, g->col[b + q], k, d);
    da[q] = s;
    delta += alpha[q] * s;
  }
  return delta;
}

int oracle_gatv2_forward(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                         int dtype, const void* xl, const void* xr, const double* att,
                         double slope, int64_t n_sel, const int64_t* sel, double* out,
                         double* lse, double* out_mag, double* alpha_sum) {
  v2_inputs g = {n, row_ptr, col, H, D, dtype, xl, xr, att, slope};
  int rc = v2_check(&g);
  if (rc) return rc;
  const int64_t n_out = sel ? n_sel : n;
  for (int64_t t = 0; sel && t < n_sel; ++t)
    if (sel[t] < 0 || sel[t] >= n) return 1;
  const int64_t maxdeg = v2_max_deg(&g);
#pragma omp parallel
  {
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t t = 0; t < n_out; ++t) {
      const int64_t i = sel ? sel[t] : t;
      const int64_t b = row_ptr[i], deg = row_ptr[i + 1] - b;
      for (int k = 0; k < H; ++k) {
        lse[t * H + k] = v2_softmax(&g, i, k, alpha);
        double asum = 0.0;
        for (int64_t q = 0; q < deg; ++q) asum += alpha[q];
        if (alpha_sum) alpha_sum[t * H + k] = asum;
        for (int d = 0; d < D; ++d) {
          double acc = 0.0, mag = 0.0;
          for (int64_t q = 0; q < deg; ++q) {
            const double x = v2_feat(&g, xl, col[b + q], k, d);
            acc += alpha[q] * x;
            mag += alpha[q] * fabs(x);
          }
          out[(t * H + k) * (int64_t)D + d] = acc;
          if (out_mag) out_mag[(t * H + k) * (int64_t)D + d] = mag;
        }
      }
    }
    free(alpha);
  }
  return 0;
}

/* Delta_i = sum_j alpha_ij dout_i . xl_j for the listed nodes (sel = NULL: all). */
int oracle_gatv2_delta(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                       int dtype, const void* xl, const void* xr, const double* att,
                       double slope, const void* dout, int64_t n_sel, const int64_t* sel,
                       double* delta) {
  v2_inputs g = {n, row_ptr, col, H, D, dtype, xl, xr, att, slope};
  int rc = v2_check(&g);
  if (rc) return rc;
  const int64_t n_out = sel ? n_sel : n;
  const int64_t maxdeg = v2_max_deg(&g);
#pragma omp parallel
  {
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t t = 0; t < n_out; ++t) {
      const int64_t i = sel ? sel[t] : t;
      for (int k = 0; k < H; ++k) {
        v2_softmax(&g, i, k, alpha);
        delta[t * H + k] = v2_delta(&g, dout, i, k, alpha, da);
      }
    }
    free(alpha);
    free(da);
  }
  return 0;
}

/*
 * Backward.  Destination-side terms (dxr, datt) per destination row in
 * parallel, with per-thread datt sums added in thread order; the source-side
 * scatter into dxl runs on one thread in edge order.  sel = NULL: whole
 * graph, dxl and dxr [n][H][D].  With sel: dxl and dxr rows of the listed
 * (distinct) nodes only (dxl from a scan for the edges that leave them),
 * datt still over the whole graph.  Mags may be NULL.
 */
int oracle_gatv2_backward(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                          int dtype, const void* xl, const void* xr, const double* att,
                          double slope, const void* dout, int64_t n_sel, const int64_t* sel,
                          double* dxl, double* dxr, double* datt, double* dxl_mag,
                          double* dxr_mag, double* datt_mag) {
  v2_inputs g = {n, row_ptr, col, H, D, dtype, xl, xr, att, slope};
  int rc = v2_check(&g);
  if (rc) return rc;
  if (!dout && n > 0) return 1;
  const int64_t HD = (int64_t)H * D;
  const int64_t m = sel ? n_sel : n;
  int64_t* target = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  if (!target) return 3;
  for (int64_t v = 0; v < n; ++v) target[v] = sel ? -1 : v;
  for (int64_t t = 0; sel && t < n_sel; ++t) {
    if (sel[t] < 0 || sel[t] >= n || target[sel[t]] >= 0) {
      free(target);
      return 1;
    }
    target[sel[t]] = t;
  }
  memset(dxl, 0, sizeof(double) * (size_t)(m * HD));
  memset(dxr, 0, sizeof(double) * (size_t)(m * HD));
  if (dxl_mag) memset(dxl_mag, 0, sizeof(double) * (size_t)(m * HD));
  if (dxr_mag) memset(dxr_mag, 0, sizeof(double) * (size_t)(m * HD));
  const int64_t maxdeg = v2_max_deg(&g);
  int nt = 1;
#ifdef _OPENMP
  nt = omp_get_max_threads();
#endif
  double* part = (double*)calloc((size_t)(nt * 2 * HD), sizeof(double));
  if (!part) {
    free(target);
    return 3;
  }
  /* destination side: dxr rows, datt */
#pragma omp parallel num_threads(nt)
  {
    int th = 0;
#ifdef _OPENMP
    th = omp_get_thread_num();
#endif
    double* pa = part + (int64_t)th * 2 * HD;
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
      const int64_t b = row_ptr[i], deg = row_ptr[i + 1] - b;
      if (deg == 0) continue;
      for (int k = 0; k < H; ++k) {
        v2_softmax(&g, i, k, alpha);
        const double delta = v2_delta(&g, dout, i, k, alpha, da);
        for (int64_t q = 0; q < deg; ++q) {
          const int64_t j = col[b + q];
          const double de = alpha[q] * (da[q] - delta);
          const double dm = alpha[q] * (fabs(da[q]) + fabs(delta));
          for (int d = 0; d < D; ++d) {
            const double z = v2_feat(&g, xr, i, k, d) + v2_feat(&g, xl, j, k, d);
            const double a = att[k * D + d];
            pa[k * D + d] += de * v2_leaky(z, slope);
            pa[HD + k * D + d] += dm * fabs(v2_leaky(z, slope));
            if (target[i] >= 0) {
              const int64_t x = (target[i] * H + k) * (int64_t)D + d;
              dxr[x] += de * a * v2_leaky_grad(z, slope);
              if (dxr_mag) dxr_mag[x] += dm * fabs(a) * v2_leaky_grad(z, slope);
            }
          }
        }
      }
    }
    free(alpha);
    free(da);
  }
  for (int64_t x = 0; x < HD; ++x) {
    double s = 0.0, ms = 0.0;
    for (int t = 0; t < nt; ++t) {
      s += part[(int64_t)t * 2 * HD + x];
      ms += part[(int64_t)t * 2 * HD + HD + x];
    }
    datt[x] = s;
    if (datt_mag) datt_mag[x] = ms;
  }
  free(part);
  /* source side: scatter alpha dout_i + dz onto the listed sources, edge order */
  {
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
    for (int64_t i = 0; i < n; ++i) {
      const int64_t b = row_ptr[i], deg = row_ptr[i + 1] - b;
      int hit = 0;
      for (int64_t q = 0; q < deg && !hit; ++q) hit = target[col[b + q]] >= 0;
      if (!hit) continue;
      for (int k = 0; k < H; ++k) {
        v2_softmax(&g, i, k, alpha);
        const double delta = v2_delta(&g, dout, i, k, alpha, da);
        for (int64_t q = 0; q < deg; ++q) {
          const int64_t t = target[col[b + q]];
          if (t < 0) continue;
          const int64_t j = col[b + q];
          const double de = alpha[q] * (da[q] - delta);
          const double dm = alpha[q] * (fabs(da[q]) + fabs(delta));
          for (int d = 0; d < D; ++d) {
            const double z = v2_feat(&g, xr, i, k, d) + v2_feat(&g, xl, j, k, d);
            const double a = att[k * D + d], gd = v2_feat(&g, dout, i, k, d);
            const int64_t x = (t * H + k) * (int64_t)D + d;
            dxl[x] += alpha[q] * gd + de * a * v2_leaky_grad(z, slope);
            if (dxl_mag)
              dxl_mag[x] += alpha[q] * fabs(gd) + dm * fabs(a) * v2_leaky_grad(z, slope);
          }
        }
      }
    }
    free(alpha);
    free(da);
  }
  free(target);
  return 0;
}
