/*
 * Plain fp64 CPU oracle for the reduction-family neighbour aggregation
 * (max / min pooling over in-neighbours).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes ("On Efficient Scaling of GNNs via IO-Aware Layers
 * Implementations", Technical Summary > Methodology, reduction-based
 * aggregations: a per-edge message followed by a neighbourhood max or min;
 * the message here is the source row x_j itself, any per-node transform
 * such as an MLP being applied by the caller):
 *   out[i][f] = max (or min) over the in-neighbours j of i of x[j][f]
 *   arg[i][f] = the j that attains it; among equal values the smallest j
 * A node with no in-neighbours gets out = 0 and arg = -1.  Values are
 * compared exactly as given (float32 or bfloat16 widened exactly to double),
 * so out is always one of the inputs.  Multi-edges change nothing.
 *
 * Backward: the gradient of L = sum(out * dout) w.r.t. x: each destination
 * i with in-neighbours passes dout[i][f] to the single source arg[i][f]:
 *   dx[j][f] = sum over i with arg[i][f] = j of dout[i][f]
 * (the arg array is the one the forward pass returns).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double red_widen(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  if (dtype == 2) return ((const double*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int red_check(int64_t n, const int32_t* row_ptr, const int32_t* col, int64_t F,
                     int dtype) {
  if (n < 0 || F < 1 || dtype < 0 || dtype > 2 || !row_ptr) return 1;
  if (row_ptr[0] != 0) return 2;
  for (int64_t i = 0; i < n; ++i)
    if (row_ptr[i + 1] < row_ptr[i]) return 2;
  for (int64_t p = 0; p < row_ptr[n]; ++p)
    if (col[p] < 0 || col[p] >= n) return 2;
  return 0;
}

/* The reduction of row i, feature f: *who receives the winning source (-1
 * for an empty row) and the value is returned (0 for an empty row). */
static double red_row(const int32_t* row_ptr, const int32_t* col, int64_t F, int dtype,
                      const void* x, int op, int64_t i, int64_t f, int64_t* who) {
  double best = 0.0;
  *who = -1;
  for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
    const int64_t j = col[p];
    const double v = red_widen(x, dtype, j * F + f);
    const int better = op == 0 ? v > best : v < best;
    if (*who < 0 || better || (v == best && j < *who)) {
      best = v;
      *who = j;
    }
  }
  return best;
}

/*
 * Forward.  op 0 = max, 1 = min.  sel = NULL: every node; otherwise output
 * row t is node sel[t].  out [n_out][F] double, arg [n_out][F] int32.
 */
int oracle_reduce_forward(int64_t n, const int32_t* row_ptr, const int32_t* col, int64_t F,
                          int dtype, const void* x, int op, int64_t n_sel, const int64_t* sel,
                          double* out, int32_t* arg) {
  int rc = red_check(n, row_ptr, col, F, dtype);
  if (rc) return rc;
  if (op != 0 && op != 1) return 1;
  const int64_t n_out = sel ? n_sel : n;
  for (int64_t t = 0; sel && t < n_sel; ++t)
    if (sel[t] < 0 || sel[t] >= n) return 1;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t t = 0; t < n_out; ++t) {
    const int64_t i = sel ? sel[t] : t;
    for (int64_t f = 0; f < F; ++f) {
      int64_t who;
      out[t * F + f] = red_row(row_ptr, col, F, dtype, x, op, i, f, &who);
      arg[t * F + f] = (int32_t)who;
    }
  }
  return 0;
}

/*
 * Backward: dx [n][F] from arg [n][F] (int32, -1 = no source) and dout
 * [n][F], summed in ascending destination order.  dx_mag (may be NULL) is
 * the sum of |terms| per element.
 */
int oracle_reduce_backward(int64_t n, int64_t F, int dtype, const int32_t* arg,
                           const void* dout, double* dx, double* dx_mag) {
  if (n < 0 || F < 1 || dtype < 0 || dtype > 2) return 1;
  for (int64_t x = 0; x < n * F; ++x)
    if (arg[x] < -1 || arg[x] >= n) return 2;
  memset(dx, 0, sizeof(double) * (size_t)(n * F));
  if (dx_mag) memset(dx_mag, 0, sizeof(double) * (size_t)(n * F));
  for (int64_t i = 0; i < n; ++i)
    for (int64_t f = 0; f < F; ++f) {
      const int64_t j = arg[i * F + f];
      if (j < 0) continue;
      const double g = red_widen(dout, dtype, i * F + f);
      dx[j * F + f] += g;
      if (dx_mag) dx_mag[j * F + f] += fabs(g);
    }
  return 0;
}

/*
 * Backward rows of the n_sel listed (distinct) sources only, straight from
 * the inputs: every destination whose row holds a listed source has its
 * reduction recomputed, and passes dout[i][f] to the winner when that is a
 * listed node.  dx [n_sel][F]; dx_mag may be NULL.
 */
int oracle_reduce_backward_rows(int64_t n, const int32_t* row_ptr, const int32_t* col,
                                int64_t F, int dtype, const void* x, int op, const void* dout,
                                int64_t n_sel, const int64_t* sel, double* dx, double* dx_mag) {
  int rc = red_check(n, row_ptr, col, F, dtype);
  if (rc) return rc;
  if ((op != 0 && op != 1) || !sel || n_sel < 0) return 1;
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
  for (int64_t i = 0; i < n; ++i) {
    int hit = 0;
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1] && !hit; ++p) hit = target[col[p]] >= 0;
    if (!hit) continue;
    for (int64_t f = 0; f < F; ++f) {
      int64_t who;
      red_row(row_ptr, col, F, dtype, x, op, i, f, &who);
      if (who < 0 || target[who] < 0) continue;
      const double g = red_widen(dout, dtype, i * F + f);
      dx[target[who] * F + f] += g;
      if (dx_mag) dx_mag[target[who] * F + f] += fabs(g);
    }
  }
  free(target);
  return 0;
}
