/*
 * Plain fp64 CPU oracle for the fused graph-transformer neighbour attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, per destination i and head k ("On Efficient Scaling of
 * GNNs via IO-Aware Layers Implementations", Technical Summary > Methodology,
 * attention-based layers, Graph Transformer; the attention of Shi et al.,
 * "Masked Label Prediction: Unified Message Passing Model for Semi-Supervised
 * Classification", IJCAI 2021, eqs. 3-4, restricted to the neighbourhood,
 * with the query, key and value projections applied by the caller):
 *   e_ij  = scale * q[i][k] . key[j][k]      (scale = 1/sqrt(D) in that paper)
 *   alpha_ij = softmax over the in-neighbours j of i of e_ij
 *   out[i][k] = sum_j alpha_ij val[j][k],  lse(i, k) = log sum_j exp(e_ij)
 * by the textbook two-pass softmax.  A node with no in-neighbours gets
 * out = 0 and lse = -inf.  Multi-edges count with their multiplicity.
 *
 * Backward of L = sum(out * dout):
 *   da_ij  = dout[i][k] . val[j][k],  Delta_i = sum_j alpha_ij da_ij
 *   de_ij  = alpha_ij (da_ij - Delta_i)
 *   dq[i]  = scale * sum_j de_ij key[j]
 *   dkey[j] = scale * sum_i de_ij q[i],   dval[j] = sum_i alpha_ij dout[i]
 *
 * Inputs: the exact arrays given to the GPU (float32 or bfloat16 bit
 * patterns, widened exactly; float64 accepted).  Outputs double; "mag"
 * outputs hold per element the sum of |terms|.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int64_t n;
  const int32_t* row_ptr;
  const int32_t* col;
  int H, D, dtype;
  const void* q;
  const void* key;
  const void* val;
  double scale;
} gt_inputs;

static double gt_widen(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  if (dtype == 2) return ((const double*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double gt_feat(const gt_inputs* g, const void* a, int64_t v, int k, int d) {
  return gt_widen(a, g->dtype, ((int64_t)v * g->H + k) * g->D + d);
}

static int gt_check(const gt_inputs* g) {
  if (g->n < 0 || g->H < 1 || g->D < 1 || g->dtype < 0 || g->dtype > 2 || !g->row_ptr) return 1;
  if (g->n > 0 && (!g->q || !g->key || !g->val)) return 1;
  if (g->row_ptr[0] != 0) return 2;
  for (int64_t i = 0; i < g->n; ++i)
    if (g->row_ptr[i + 1] < g->row_ptr[i]) return 2;
  for (int64_t p = 0; p < g->row_ptr[g->n]; ++p)
    if (g->col[p] < 0 || g->col[p] >= g->n) return 2;
  return 0;
}

static int64_t gt_max_deg(const gt_inputs* g) {
  int64_t m = 0;
  for (int64_t i = 0; i < g->n; ++i)
    if (g->row_ptr[i + 1] - g->row_ptr[i] > m) m = g->row_ptr[i + 1] - g->row_ptr[i];
  return m;
}

static double gt_dot(const gt_inputs* g, const void* a, int64_t u, const void* b, int64_t v,
                     int k) {
  double s = 0.0;
  for (int d = 0; d < g->D; ++d) s += gt_feat(g, a, u, k, d) * gt_feat(g, b, v, k, d);
  return s;
}

/* alpha[q] of row i, head k; returns lse (-inf for an empty row) */
static double gt_softmax(const gt_inputs* g, int64_t i, int k, double* alpha) {
  const int64_t b = g->row_ptr[i], deg = g->row_ptr[i + 1] - b;
  if (deg == 0) return -INFINITY;
  double m = -INFINITY;
  for (int64_t q = 0; q < deg; ++q) {
    alpha[q] = g->scale * gt_dot(g, g->q, i, g->key, g->col[b + q], k);
    if (alpha[q] > m) m = alpha[q];
  }
  double l = 0.0;
  for (int64_t q = 0; q < deg; ++q) l += exp(alpha[q] - m);
  for (int64_t q = 0; q < deg; ++q) alpha[q] = exp(alpha[q] - m) / l;
  return m + log(l);
}

static double gt_delta(const gt_inputs* g, const void* dout, int64_t i, int k,
                       const double* alpha, double* da) {
  const int64_t b = g->row_ptr[i], deg = g->row_ptr[i + 1] - b;
  double delta = 0.0;
  for (int64_t q = 0; q < deg; ++q) {
    da[q] = gt_dot(g, dout, i, g->val, g->col[b + q], k);
    delta += alpha[q] * da[q];
  }
  return delta;
}

int oracle_gt_forward(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                      int dtype, const void* q, const void* key, const void* val, double scale,
                      int64_t n_sel, const int64_t* sel, double* out, double* lse,
                      double* out_mag, double* alpha_sum) {
  gt_inputs g = {n, row_ptr, col, H, D, dtype, q, key, val, scale};
  int rc = gt_check(&g);
  if (rc) return rc;
  const int64_t n_out = sel ? n_sel : n;
  for (int64_t t = 0; sel && t < n_sel; ++t)
    if (sel[t] < 0 || sel[t] >= n) return 1;
  const int64_t maxdeg = gt_max_deg(&g);
#pragma omp parallel
  {
    double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t t = 0; t < n_out; ++t) {
      const int64_t i = sel ? sel[t] : t;
      const int64_t b = row_ptr[i], deg = row_ptr[i + 1] - b;
      for (int k = 0; k < H; ++k) {
        lse[t * H + k] = gt_softmax(&g, i, k, alpha);
        double asum = 0.0;
        for (int64_t e = 0; e < deg; ++e) asum += alpha[e];
        if (alpha_sum) alpha_sum[t * H + k] = asum;
        for (int d = 0; d < D; ++d) {
          double acc = 0.0, mag = 0.0;
          for (int64_t e = 0; e < deg; ++e) {
            const double x = gt_feat(&g, val, col[b + e], k, d);
            acc += alpha[e] * x;
            mag += alpha[e] * fabs(x);
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

/*
 * Backward.  sel = NULL: every node; otherwise rows of the listed (distinct)
 * nodes only: dq from the node's own row, dkey and dval from a scan for the
 * edges that leave it.  dq, dkey, dval [m][H][D]; mags may be NULL.
 */
int oracle_gt_backward(int64_t n, const int32_t* row_ptr, const int32_t* col, int H, int D,
                       int dtype, const void* q, const void* key, const void* val,
                       double scale, const void* dout, int64_t n_sel, const int64_t* sel,
                       double* dq, double* dkey, double* dval, double* dq_mag,
                       double* dkey_mag, double* dval_mag) {
  gt_inputs g = {n, row_ptr, col, H, D, dtype, q, key, val, scale};
  int rc = gt_check(&g);
  if (rc) return rc;
  if (!dout && n > 0) return 1;
  const int64_t HD = (int64_t)H * D, m = sel ? n_sel : n;
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
  double* outs[3] = {dq, dkey, dval};
  double* mags[3] = {dq_mag, dkey_mag, dval_mag};
  for (int a = 0; a < 3; ++a) {
    memset(outs[a], 0, sizeof(double) * (size_t)(m * HD));
    if (mags[a]) memset(mags[a], 0, sizeof(double) * (size_t)(m * HD));
  }
  const int64_t maxdeg = gt_max_deg(&g);
  double* alpha = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
  double* da = (double*)malloc(sizeof(double) * (size_t)(maxdeg + 1));
  for (int64_t i = 0; i < n; ++i) {
    const int64_t b = row_ptr[i], deg = row_ptr[i + 1] - b;
    int hit = target[i] >= 0 && deg > 0;
    for (int64_t e = 0; e < deg && !hit; ++e) hit = target[col[b + e]] >= 0;
    if (!hit) continue;
    for (int k = 0; k < H; ++k) {
      gt_softmax(&g, i, k, alpha);
      const double delta = gt_delta(&g, dout, i, k, alpha, da);
      for (int64_t e = 0; e < deg; ++e) {
        const int64_t j = col[b + e];
        const double de = alpha[e] * (da[e] - delta);
        const double dm = alpha[e] * (fabs(da[e]) + fabs(delta));
        for (int d = 0; d < D; ++d) {
          if (target[i] >= 0) {
            const double kv = gt_feat(&g, key, j, k, d);
            const int64_t x = (target[i] * H + k) * (int64_t)D + d;
            dq[x] += scale * de * kv;
            if (dq_mag) dq_mag[x] += fabs(scale) * dm * fabs(kv);
          }
          if (target[j] >= 0) {
            const double qv = gt_feat(&g, q, i, k, d), gv = gt_feat(&g, dout, i, k, d);
            const int64_t x = (target[j] * H + k) * (int64_t)D + d;
            dkey[x] += scale * de * qv;
            dval[x] += alpha[e] * gv;
            if (dkey_mag) dkey_mag[x] += fabs(scale) * dm * fabs(qv);
            if (dval_mag) dval_mag[x] += alpha[e] * fabs(gv);
          }
        }
      }
    }
  }
  free(alpha);
  free(da);
  free(target);
  return 0;
}
