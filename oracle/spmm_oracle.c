/*
 * Plain fp64 CPU oracle for the SpMM-family neighbour aggregation (GCN /
 * GraphConv propagation).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes: out = A~ x for the CSR graph (row i lists the sources j of
 * the edges j -> i, with multiplicity) and a feature matrix x [N][F], where
 * A~ is the propagation matrix of the layer H' = sigma(A~ H W) ("On Efficient
 * Scaling of GNNs via IO-Aware Layers Implementations", Technical Summary >
 * Methodology, SpMM-based convolutions; W and sigma act outside this
 * operation).  Per edge j -> i the coefficient is
 *   norm 0 ("sum"):  1
 *   norm 1 ("mean"): 1 / deg(i)
 *   norm 2 ("sym"):  1 / sqrt(deg(i) deg(j))   (the renormalised adjacency
 *                    D^-1/2 A D^-1/2 of Kipf & Welling, ICLR 2017, eq. 2)
 * with deg(v) the number of in-edges of v (the length of CSR row v, so the
 * row sums of A; self-loops count when the graph has them).  A node of
 * degree 0 has coefficient 0 wherever its degree appears in a denominator.
 * A multi-edge contributes once per copy.
 *
 * Backward: the gradient of L = sum(out * dout) w.r.t. x, dx = A~^T dout:
 * every edge j -> i adds coef(i, j) dout[i] to dx[j].  A~ does not depend on
 * x, so there is no other gradient.
 *
 * Inputs: the exact arrays given to the GPU (float32, or bfloat16 bit
 * patterns), widened exactly to double; float64 is also accepted.  Outputs
 * double.  Optional "mag" outputs hold, per output element, the sum of the
 * absolute values of its terms (used by tests to bound float32 rounding).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double spmm_widen(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  if (dtype == 2) return ((const double*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int64_t spmm_deg(const int32_t* row_ptr, int64_t v) {
  return (int64_t)row_ptr[v + 1] - row_ptr[v];
}

/* coefficient of the edge j -> i */
static double spmm_coef(int norm, const int32_t* row_ptr, int64_t i, int64_t j) {
  const int64_t di = spmm_deg(row_ptr, i), dj = spmm_deg(row_ptr, j);
  if (norm == 0) return 1.0;
  if (norm == 1) return di > 0 ? 1.0 / (double)di : 0.0;
  if (di == 0 || dj == 0) return 0.0;
  return 1.0 / sqrt((double)di * (double)dj);
}

static int spmm_check(int64_t n, const int32_t* row_ptr, const int32_t* col, int64_t F,
                      int dtype, int norm) {
  if (n < 0 || F < 1 || dtype < 0 || dtype > 2 || norm < 0 || norm > 2 || !row_ptr) return 1;
  if (row_ptr[0] != 0) return 2;
  for (int64_t i = 0; i < n; ++i)
    if (row_ptr[i + 1] < row_ptr[i]) return 2;
  for (int64_t p = 0; p < row_ptr[n]; ++p)
    if (col[p] < 0 || col[p] >= n) return 2;
  return 0;
}

/*
 * Forward for every node (sel = NULL) or for the n_sel listed nodes (output
 * row t is node sel[t]): out [n_out][F]; out_mag may be NULL.
 */
int oracle_spmm_forward(int64_t n, const int32_t* row_ptr, const int32_t* col, int64_t F,
                        int dtype, const void* x, int norm, int64_t n_sel, const int64_t* sel,
                        double* out, double* out_mag) {
  int rc = spmm_check(n, row_ptr, col, F, dtype, norm);
  if (rc) return rc;
  const int64_t n_out = sel ? n_sel : n;
  for (int64_t t = 0; sel && t < n_sel; ++t)
    if (sel[t] < 0 || sel[t] >= n) return 1;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t t = 0; t < n_out; ++t) {
    const int64_t i = sel ? sel[t] : t;
    double* o = out + t * F;
    double* m = out_mag ? out_mag + t * F : NULL;
    for (int64_t f = 0; f < F; ++f) {
      o[f] = 0.0;
      if (m) m[f] = 0.0;
    }
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const int64_t j = col[p];
      const double c = spmm_coef(norm, row_ptr, i, j);
      for (int64_t f = 0; f < F; ++f) {
        const double v = spmm_widen(x, dtype, j * F + f);
        o[f] += c * v;
        if (m) m[f] += fabs(c * v);
      }
    }
  }
  return 0;
}

/*
 * Backward over the whole graph: dx [n][F] = A~^T dout, scattered in edge
 * order (deterministic).  dx_mag may be NULL.
 */
int oracle_spmm_backward(int64_t n, const int32_t* row_ptr, const int32_t* col, int64_t F,
                         int dtype, const void* dout, int norm, double* dx, double* dx_mag) {
  int rc = spmm_check(n, row_ptr, col, F, dtype, norm);
  if (rc) return rc;
  memset(dx, 0, sizeof(double) * (size_t)(n * F));
  if (dx_mag) memset(dx_mag, 0, sizeof(double) * (size_t)(n * F));
  for (int64_t i = 0; i < n; ++i)
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const int64_t j = col[p];
      const double c = spmm_coef(norm, row_ptr, i, j);
      for (int64_t f = 0; f < F; ++f) {
        const double v = spmm_widen(dout, dtype, i * F + f);
        dx[j * F + f] += c * v;
        if (dx_mag) dx_mag[j * F + f] += fabs(c * v);
      }
    }
  return 0;
}

/*
 * Backward rows of the n_sel listed (distinct) nodes only: dx [n_sel][F],
 * from a scan of the whole CSR for the edges that leave each listed node.
 */
int oracle_spmm_backward_rows(int64_t n, const int32_t* row_ptr, const int32_t* col, int64_t F,
                              int dtype, const void* dout, int norm, int64_t n_sel,
                              const int64_t* sel, double* dx, double* dx_mag) {
  int rc = spmm_check(n, row_ptr, col, F, dtype, norm);
  if (rc) return rc;
  if (!sel || n_sel < 0) return 1;
  int64_t* target = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  if (!target) return 3;
  for (int64_t v = 0; v < n; ++v) target[v] = -1;
  for (int64_t t = 0; t < n_sel; ++t) {
    if (sel[t] < 0 || sel[t] >= n || target[sel[t]] >= 0) {
      free(target);
      return 1;
    }
    target[sel[t]] = t;
  }
  memset(dx, 0, sizeof(double) * (size_t)(n_sel * F));
  if (dx_mag) memset(dx_mag, 0, sizeof(double) * (size_t)(n_sel * F));
  for (int64_t i = 0; i < n; ++i)
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const int64_t t = target[col[p]];
      if (t < 0) continue;
      const double c = spmm_coef(norm, row_ptr, i, col[p]);
      for (int64_t f = 0; f < F; ++f) {
        const double v = spmm_widen(dout, dtype, i * F + f);
        dx[t * F + f] += c * v;
        if (dx_mag) dx_mag[t * F + f] += fabs(c * v);
      }
    }
  free(target);
  return 0;
}
