// C-ABI entry points: argument checks, workspace layout, dispatch.
#include <new>

#include "internal.h"

namespace gnn {

bool make_shape(int H, int D, gnn_dtype dt, Shape* s) {
  if (H < 1 || D < 1 || H > 4096 || D > 4096) return false;
  if (dt != GNN_F32 && dt != GNN_BF16) return false;
  s->H = H;
  s->D = D;
  s->esize = dt == GNN_F32 ? 4 : 2;
  const int head_bytes = D * s->esize;
  if (head_bytes % 16) return false;
  s->hv = head_bytes / 16;
  if (s->hv > 32 || (s->hv & (s->hv - 1))) return false;
  const int64_t rv = int64_t(H) * s->hv;
  if (rv * 16 > 2048) return false;
  s->rv = int(rv);
  if (s->rv <= 32) {
    s->lpr = 1;
    while (s->lpr < s->rv) s->lpr <<= 1;
    s->nv = 1;
  } else {
    s->lpr = 32;
    s->nv = (s->rv + 31) / 32;
    if (s->nv == 3) s->nv = 4;
  }
  s->hv_log2 = 0;
  while ((1 << s->hv_log2) < s->hv) ++s->hv_log2;
  s->lpr_log2 = 0;
  while ((1 << s->lpr_log2) < s->lpr) ++s->lpr_log2;
  return true;
}

bool make_wide_shape(const Shape& s, Shape* w) {
  if (s.hv < 2 || s.rv > 64) return false;
  *w = s;
  w->rv = s.rv / 2;
  w->hv = s.hv / 2;
  w->lpr = 1;
  while (w->lpr < w->rv) w->lpr <<= 1;
  w->nv = 1;
  w->hv_log2 = s.hv_log2 - 1;
  w->lpr_log2 = 0;
  while ((1 << w->lpr_log2) < w->lpr) ++w->lpr_log2;
  return true;
}

WsLayout ws_layout(const gnn_graph* g, const Shape& s) {
  WsLayout L;
  const size_t HD = size_t(s.H) * s.D;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t r = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return r;
  };
  // forward: work counters, hub chunk partials of the CSR direction
  L.fwd_ctr = take(kCounters * 4);
  L.fwd_scores = take(size_t(g->n) * s.H * 8);  // s_src [N][H] then s_dst [N][H]
  L.fwd_acc = take(size_t(g->csr.n_hub_chunks) * HD * 4);
  L.fwd_ml = take(size_t(g->csr.n_hub_chunks) * s.H * 8);
  L.fwd_total = off;
  // backward
  off = 0;
  L.bwd_ctr = take(kCounters * 4);
  L.bwd_scores = take(size_t(g->n) * s.H * 8);
  L.stats = take(size_t(g->n) * s.H * 16);
  L.ds_src = take(size_t(g->n) * s.H * 4);
  L.dst_part = take(size_t(g->csr.n_hub_chunks) * s.H * 16);
  L.src_acc = take(size_t(g->csc.n_hub_chunks) * HD * 4);
  L.src_sum = take(size_t(g->csc.n_hub_chunks) * s.H * 4);
  // attention-vector partial sums: up to 8 blocks per SM, each warp summing
  // at least 16 nodes before its block's float64 fold
  const int64_t cap = int64_t(g->sm_count > 0 ? g->sm_count : 1) * 8;
  int64_t blocks = (g->n + 127) / 128;
  if (blocks < 1) blocks = 1;
  if (blocks > cap) blocks = cap;
  L.da_blocks = int(blocks);
  L.da_part = take(size_t(blocks) * 2 * HD * 8);
  L.bwd_total = off;
  return L;
}

}  // namespace gnn

using gnn::Shape;
using gnn::WsLayout;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool tiling_ok(const gnn_tiling& t) {
  return t.light_max_deg >= GNN_LIGHT_AUTO && t.cta_max_deg >= 0 &&
         t.cta_max_deg >= t.light_max_deg && t.cta_max_deg <= 16384 && t.hub_chunk >= 1 &&
         t.hub_chunk <= 16384;
}

// The tiling that bounds the prepared graph's buffers: an automatic light
// threshold is never below its floor (or cta_max_deg), and fewer light nodes
// only mean more block items, which the bound covers.
gnn_tiling bound_tiling(gnn_tiling t) {
  if (t.light_max_deg == GNN_LIGHT_AUTO)
    t.light_max_deg = t.cta_max_deg < gnn::kLightAutoMin ? t.cta_max_deg : gnn::kLightAutoMin;
  return t;
}

gnn_tiling resolve_tiling(const gnn_tiling* t) {
  gnn_tiling r;
  gnn_default_tiling(&r);
  if (t) r = *t;
  return r;
}

bool sizes_ok(int64_t n, int64_t e) {
  return n >= 0 && e >= 0 && n < (int64_t(1) << 31) - 1 && e < (int64_t(1) << 31) - 1;
}

gnn_status check_call(const gnn_graph* g, int H, int D, gnn_dtype dt, Shape* s) {
  if (!g) return GNN_ERR_INVALID_ARG;
  if (dt != GNN_F32 && dt != GNN_BF16) return GNN_ERR_INVALID_ARG;
  if (H < 1 || D < 1) return GNN_ERR_INVALID_ARG;
  if (!gnn::make_shape(H, D, dt, s)) return GNN_ERR_UNSUPPORTED;
  return GNN_OK;
}

gnn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GNN_OK : GNN_ERR_CUDA; }

}  // namespace

extern "C" {

void gnn_default_tiling(gnn_tiling* t) {
  if (!t) return;
  t->light_max_deg = GNN_LIGHT_AUTO;
  t->cta_max_deg = 4096;
  t->hub_chunk = 2048;
}

int gnn_abi_version(void) { return GNNAGG_ABI_VERSION; }

const char* gnn_status_string(gnn_status s) {
  switch (s) {
    case GNN_OK: return "ok";
    case GNN_ERR_INVALID_ARG: return "invalid argument";
    case GNN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case GNN_ERR_INVALID_GRAPH: return "invalid CSR graph";
    case GNN_ERR_WORKSPACE_TOO_SMALL: return "buffer or workspace too small";
    case GNN_ERR_CUDA: return "CUDA error";
    case GNN_ERR_DEVICE_ASSERT: return "device-side consistency check failed";
    case GNN_ERR_TIMEOUT: return "a bounded device wait timed out";
  }
  return "unknown status";
}

size_t gnn_graph_buffer_bytes(int64_t n_nodes, int64_t n_edges, const gnn_tiling* tiling) {
  const gnn_tiling t = resolve_tiling(tiling);
  if (!sizes_ok(n_nodes, n_edges) || !tiling_ok(t)) return 0;
  return gnn::graph_buffer_bytes(n_nodes, n_edges, bound_tiling(t));
}

size_t gnn_graph_scratch_bytes(int64_t n_nodes, int64_t n_edges) {
  if (!sizes_ok(n_nodes, n_edges)) return 0;
  return gnn::graph_scratch_bytes(n_nodes, n_edges);
}

gnn_status gnn_graph_prepare(int64_t n_nodes, int64_t n_edges, const int32_t* row_ptr_d,
                             const int32_t* col_idx_d, void* buffer_d, size_t buffer_bytes,
                             void* scratch_d, size_t scratch_bytes, const gnn_tiling* tiling,
                             void* stream, gnn_graph** out) {
  if (!out) return GNN_ERR_INVALID_ARG;
  *out = nullptr;
  const gnn_tiling t = resolve_tiling(tiling);
  if (!sizes_ok(n_nodes, n_edges) || !tiling_ok(t)) return GNN_ERR_INVALID_ARG;
  if (!row_ptr_d || !buffer_d || !scratch_d || (n_edges > 0 && !col_idx_d))
    return GNN_ERR_INVALID_ARG;
  if (!aligned(row_ptr_d, 4) || !aligned(col_idx_d, 16) || !aligned(buffer_d, 256) ||
      !aligned(scratch_d, 256))
    return GNN_ERR_INVALID_ARG;
  if (buffer_bytes < gnn::graph_buffer_bytes(n_nodes, n_edges, bound_tiling(t)) ||
      scratch_bytes < gnn::graph_scratch_bytes(n_nodes, n_edges))
    return GNN_ERR_WORKSPACE_TOO_SMALL;
  gnn_graph* g = new (std::nothrow) gnn_graph;
  if (!g) return GNN_ERR_INVALID_ARG;
  g->n = n_nodes;
  g->e = n_edges;
  g->tiling = t;
  if (cudaGetDevice(&g->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&g->sm_count, cudaDevAttrMultiProcessorCount, g->device) !=
          cudaSuccess) {
    delete g;
    return GNN_ERR_CUDA;
  }
  if (t.light_max_deg == GNN_LIGHT_AUTO)
    g->tiling.light_max_deg = gnn::auto_light_max(n_edges, g->sm_count, t.cta_max_deg);
  const gnn_status s =
      gnn::prepare_graph(g, row_ptr_d, col_idx_d, static_cast<char*>(buffer_d), buffer_bytes,
                         static_cast<char*>(scratch_d), scratch_bytes,
                         static_cast<cudaStream_t>(stream));
  if (s != GNN_OK) {
    delete g;
    return s;
  }
  *out = g;
  return GNN_OK;
}

gnn_status gnn_graph_destroy(gnn_graph* g) {
  delete g;
  return GNN_OK;
}

gnn_status gnn_graph_stats(const gnn_graph* g, int64_t* st, int n) {
  if (!g || !st || n < 16) return GNN_ERR_INVALID_ARG;
  st[0] = g->n;
  st[1] = g->e;
  const gnn::Dir* d[2] = {&g->csr, &g->csc};
  for (int k = 0; k < 2; ++k) {
    int64_t* o = st + 2 + 6 * k;
    o[0] = d[k]->n_light;
    o[1] = d[k]->n_items;
    o[2] = d[k]->n_hubs;
    o[3] = d[k]->n_hub_chunks;
    o[4] = d[k]->max_deg;
    o[5] = d[k]->max_item;
  }
  st[14] = g->tiling.light_max_deg;
  st[15] = g->tiling.cta_max_deg;
  for (int k = 16; k < n; ++k) st[k] = 0;
  return GNN_OK;
}

gnn_status gnn_graph_arrays(const gnn_graph* g, const void** p, int n) {
  if (!g || !p || n < 8) return GNN_ERR_INVALID_ARG;
  p[0] = g->csc.ptr;
  p[1] = g->csc.idx;
  p[2] = g->csr.light;
  p[3] = g->csr.items;
  p[4] = g->csr.hubs;
  p[5] = g->csc.light;
  p[6] = g->csc.items;
  p[7] = g->csc.hubs;
  for (int k = 8; k < n; ++k) p[k] = nullptr;
  return GNN_OK;
}

size_t gat_agg_workspace_bytes(const gnn_graph* g, int H, int D, gnn_dtype dtype) {
  Shape s;
  if (check_call(g, H, D, dtype, &s) != GNN_OK) return 0;
  const WsLayout L = gnn::ws_layout(g, s);
  return L.fwd_total > L.bwd_total ? L.fwd_total : L.bwd_total;
}

gnn_status gat_agg_forward_timed(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* h,
                                 const float* a_src, const float* a_dst, float slope, void* out,
                                 float* lse, void* ws, size_t ws_bytes, void* stream,
                                 void* const* events, int n_events) {
  if (events && n_events < 4) return GNN_ERR_INVALID_ARG;
  Shape s;
  gnn_status r = check_call(g, H, D, dtype, &s);
  if (r != GNN_OK) return r;
  if (g->n == 0) return GNN_OK;
  if (!h || !a_src || !a_dst || !out || !lse) return GNN_ERR_INVALID_ARG;
  if (!aligned(h, 16) || !aligned(out, 16) || !aligned(a_src, 16) || !aligned(a_dst, 16) ||
      !aligned(lse, 4))
    return GNN_ERR_INVALID_ARG;
  const WsLayout L = gnn::ws_layout(g, s);
  if (ws_bytes < L.fwd_total) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_forward(g, s, dtype, h, a_src, a_dst, slope, out, lse,
                                       static_cast<char*>(ws), L,
                                       static_cast<cudaStream_t>(stream),
                                       reinterpret_cast<const cudaEvent_t*>(events)));
}

gnn_status gat_agg_forward(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* h,
                           const float* a_src, const float* a_dst, float slope, void* out,
                           float* lse, void* ws, size_t ws_bytes, void* stream) {
  return gat_agg_forward_timed(g, H, D, dtype, h, a_src, a_dst, slope, out, lse, ws, ws_bytes,
                               stream, nullptr, 0);
}

}  // extern "C"

namespace {

gnn_status backward_call(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* h,
                         const float* a_src, const float* a_dst, float slope, const float* lse,
                         const void* dout, void* dh, float* da_src, float* da_dst, void* ws,
                         size_t ws_bytes, void* stream, void* const* events, int n_events,
                         bool reuse_scores) {
  if (events && n_events < 8) return GNN_ERR_INVALID_ARG;
  Shape s;
  gnn_status r = check_call(g, H, D, dtype, &s);
  if (r != GNN_OK) return r;
  if (!a_src || !a_dst || !da_src || !da_dst) return GNN_ERR_INVALID_ARG;
  if (!aligned(a_src, 16) || !aligned(a_dst, 16) || !aligned(da_src, 4) || !aligned(da_dst, 4))
    return GNN_ERR_INVALID_ARG;
  if (g->n > 0) {
    if (!h || !lse || !dout || !dh) return GNN_ERR_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(dout, 16) || !aligned(dh, 16) || !aligned(lse, 4))
      return GNN_ERR_INVALID_ARG;
  }
  const WsLayout L = gnn::ws_layout(g, s);
  if (ws_bytes < L.bwd_total) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  // both calls keep the per-node scores at the same offset of ws
  if (reuse_scores && L.fwd_scores != L.bwd_scores) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_backward(g, s, dtype, h, a_src, a_dst, slope, lse, dout, dh,
                                        da_src, da_dst, static_cast<char*>(ws), L,
                                        static_cast<cudaStream_t>(stream),
                                        reinterpret_cast<const cudaEvent_t*>(events),
                                        reuse_scores));
}

}  // namespace

extern "C" {

gnn_status gat_agg_backward_timed(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                  const void* h, const float* a_src, const float* a_dst,
                                  float slope, const float* lse, const void* dout, void* dh,
                                  float* da_src, float* da_dst, void* ws, size_t ws_bytes,
                                  void* stream, void* const* events, int n_events) {
  return backward_call(g, H, D, dtype, h, a_src, a_dst, slope, lse, dout, dh, da_src, da_dst,
                       ws, ws_bytes, stream, events, n_events, false);
}

gnn_status gat_agg_backward_reuse(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                  const void* h, const float* a_src, const float* a_dst,
                                  float slope, const float* lse, const void* dout, void* dh,
                                  float* da_src, float* da_dst, void* ws, size_t ws_bytes,
                                  void* stream, void* const* events, int n_events) {
  return backward_call(g, H, D, dtype, h, a_src, a_dst, slope, lse, dout, dh, da_src, da_dst,
                       ws, ws_bytes, stream, events, n_events, true);
}

gnn_status gat_agg_backward(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* h,
                            const float* a_src, const float* a_dst, float slope,
                            const float* lse, const void* dout, void* dh, float* da_src,
                            float* da_dst, void* ws, size_t ws_bytes, void* stream) {
  return gat_agg_backward_timed(g, H, D, dtype, h, a_src, a_dst, slope, lse, dout, dh, da_src,
                                da_dst, ws, ws_bytes, stream, nullptr, 0);
}

}  // extern "C"

// ---- SpMM-family propagation ---------------------------------------------

namespace {

// A row of F elements as F * size / 16 one-vector "heads".
gnn_status spmm_shape(const gnn_graph* g, int F, gnn_dtype dt, Shape* s) {
  if (!g || F < 1 || (dt != GNN_F32 && dt != GNN_BF16)) return GNN_ERR_INVALID_ARG;
  const int64_t bytes = int64_t(F) * (dt == GNN_F32 ? 4 : 2);
  if (bytes % 16 || bytes > 2048) return GNN_ERR_UNSUPPORTED;
  return gnn::make_shape(int(bytes / 16), dt == GNN_F32 ? 4 : 8, dt, s) ? GNN_OK
                                                                         : GNN_ERR_UNSUPPORTED;
}

gnn_status spmm_call(const gnn_graph* g, int F, gnn_dtype dt, gnn_norm norm, const void* x,
                     void* out, void* ws, size_t ws_bytes, void* stream, bool transpose) {
  Shape s;
  gnn_status r = spmm_shape(g, F, dt, &s);
  if (r != GNN_OK) return r;
  if (norm != GNN_NORM_SUM && norm != GNN_NORM_MEAN && norm != GNN_NORM_SYM)
    return GNN_ERR_INVALID_ARG;
  if (g->n == 0) return GNN_OK;
  if (!x || !out || !aligned(x, 16) || !aligned(out, 16)) return GNN_ERR_INVALID_ARG;
  if (ws_bytes < gnn::spmm_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_spmm(g, s, dt, int(norm), transpose, x, out,
                                    static_cast<char*>(ws), static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

size_t gcn_agg_workspace_bytes(const gnn_graph* g, int F, gnn_dtype dtype) {
  Shape s;
  if (spmm_shape(g, F, dtype, &s) != GNN_OK) return 0;
  return gnn::spmm_ws_bytes(g, s);
}

gnn_status gcn_agg_forward(const gnn_graph* g, int F, gnn_dtype dtype, gnn_norm norm,
                           const void* x, void* out, void* ws, size_t ws_bytes, void* stream) {
  return spmm_call(g, F, dtype, norm, x, out, ws, ws_bytes, stream, false);
}

gnn_status gcn_agg_backward(const gnn_graph* g, int F, gnn_dtype dtype, gnn_norm norm,
                            const void* dout, void* dx, void* ws, size_t ws_bytes,
                            void* stream) {
  return spmm_call(g, F, dtype, norm, dout, dx, ws, ws_bytes, stream, true);
}

}  // extern "C"

namespace {

gnn_status gatv2_shape(const gnn_graph* g, int H, int D, gnn_dtype dt, Shape* s) {
  gnn_status r = check_call(g, H, D, dt, s);
  if (r != GNN_OK) return r;
  return s->nv == 1 ? GNN_OK : GNN_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

size_t gatv2_agg_workspace_bytes(const gnn_graph* g, int H, int D, gnn_dtype dtype) {
  Shape s;
  if (gatv2_shape(g, H, D, dtype, &s) != GNN_OK) return 0;
  return gnn::gatv2_ws_bytes(g, s);
}

gnn_status gatv2_agg_forward(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* xl,
                             const void* xr, const float* att, float slope, void* out,
                             float* lse, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  gnn_status r = gatv2_shape(g, H, D, dtype, &s);
  if (r != GNN_OK) return r;
  if (g->n == 0) return GNN_OK;
  if (!xl || !xr || !att || !out || !lse) return GNN_ERR_INVALID_ARG;
  if (!aligned(xl, 16) || !aligned(xr, 16) || !aligned(att, 16) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return GNN_ERR_INVALID_ARG;
  if (ws_bytes < gnn::gatv2_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_gatv2_forward(g, s, dtype, xl, xr, att, slope, out, lse,
                                             static_cast<char*>(ws),
                                             static_cast<cudaStream_t>(stream)));
}

gnn_status gatv2_agg_backward(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                              const void* xl, const void* xr, const float* att, float slope,
                              const float* lse, const void* dout, void* dxl, void* dxr,
                              float* datt, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  gnn_status r = gatv2_shape(g, H, D, dtype, &s);
  if (r != GNN_OK) return r;
  if (!att || !datt || !aligned(att, 16) || !aligned(datt, 4)) return GNN_ERR_INVALID_ARG;
  if (g->n > 0) {
    if (!xl || !xr || !lse || !dout || !dxl || !dxr) return GNN_ERR_INVALID_ARG;
    if (!aligned(xl, 16) || !aligned(xr, 16) || !aligned(dout, 16) || !aligned(dxl, 16) ||
        !aligned(dxr, 16) || !aligned(lse, 4))
      return GNN_ERR_INVALID_ARG;
  }
  if (ws_bytes < gnn::gatv2_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_gatv2_backward(g, s, dtype, xl, xr, att, slope, lse, dout, dxl,
                                              dxr, datt, static_cast<char*>(ws),
                                              static_cast<cudaStream_t>(stream)));
}

size_t transformer_agg_workspace_bytes(const gnn_graph* g, int H, int D, gnn_dtype dtype) {
  Shape s;
  if (gatv2_shape(g, H, D, dtype, &s) != GNN_OK) return 0;
  return gnn::transformer_ws_bytes(g, s);
}

gnn_status transformer_agg_forward(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                   const void* q, const void* key, const void* val, float scale,
                                   void* out, float* lse, void* ws, size_t ws_bytes,
                                   void* stream) {
  Shape s;
  gnn_status r = gatv2_shape(g, H, D, dtype, &s);
  if (r != GNN_OK) return r;
  if (g->n == 0) return GNN_OK;
  if (!q || !key || !val || !out || !lse) return GNN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(key, 16) || !aligned(val, 16) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return GNN_ERR_INVALID_ARG;
  if (ws_bytes < gnn::transformer_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_transformer_forward(g, s, dtype, q, key, val, scale, out, lse,
                                                   static_cast<char*>(ws),
                                                   static_cast<cudaStream_t>(stream)));
}

gnn_status transformer_agg_backward(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                    const void* q, const void* key, const void* val, float scale,
                                    const float* lse, const void* dout, void* dq, void* dkey,
                                    void* dval, void* ws, size_t ws_bytes, void* stream) {
  Shape s;
  gnn_status r = gatv2_shape(g, H, D, dtype, &s);
  if (r != GNN_OK) return r;
  if (g->n == 0) return GNN_OK;
  if (!q || !key || !val || !lse || !dout || !dq || !dkey || !dval) return GNN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(key, 16) || !aligned(val, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dkey, 16) || !aligned(dval, 16) || !aligned(lse, 4))
    return GNN_ERR_INVALID_ARG;
  if (ws_bytes < gnn::transformer_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_transformer_backward(g, s, dtype, q, key, val, scale, lse, dout,
                                                    dq, dkey, dval, static_cast<char*>(ws),
                                                    static_cast<cudaStream_t>(stream)));
}

size_t reduce_agg_workspace_bytes(const gnn_graph* g, int F, gnn_dtype dtype) {
  Shape s;
  if (spmm_shape(g, F, dtype, &s) != GNN_OK) return 0;
  return gnn::reduce_ws_bytes(g, s);
}

gnn_status reduce_agg_forward(const gnn_graph* g, int F, gnn_dtype dtype, gnn_reduce_op op,
                              const void* x, void* out, int32_t* arg, void* ws, size_t ws_bytes,
                              void* stream) {
  Shape s;
  gnn_status r = spmm_shape(g, F, dtype, &s);
  if (r != GNN_OK) return r;
  if (op != GNN_REDUCE_MAX && op != GNN_REDUCE_MIN) return GNN_ERR_INVALID_ARG;
  if (g->n == 0) return GNN_OK;
  if (!x || !out || !arg || !aligned(x, 16) || !aligned(out, 16) || !aligned(arg, 16))
    return GNN_ERR_INVALID_ARG;
  if (ws_bytes < gnn::reduce_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_reduce_forward(g, s, dtype, int(op), x, out, arg,
                                              static_cast<char*>(ws),
                                              static_cast<cudaStream_t>(stream)));
}

gnn_status reduce_agg_backward(const gnn_graph* g, int F, gnn_dtype dtype, const int32_t* arg,
                               const void* dout, void* dx, void* ws, size_t ws_bytes,
                               void* stream) {
  Shape s;
  gnn_status r = spmm_shape(g, F, dtype, &s);
  if (r != GNN_OK) return r;
  if (g->n == 0) return GNN_OK;
  if (!arg || !dout || !dx || !aligned(arg, 16) || !aligned(dout, 16) || !aligned(dx, 16))
    return GNN_ERR_INVALID_ARG;
  if (ws_bytes < gnn::reduce_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_reduce_backward(g, s, dtype, arg, dout, dx,
                                               static_cast<char*>(ws),
                                               static_cast<cudaStream_t>(stream)));
}

gnn_status reduce_agg_backward_ordered(const gnn_graph* g, int F, gnn_dtype dtype,
                                       const int32_t* arg, const void* dout, void* dx, void* ws,
                                       size_t ws_bytes, void* stream) {
  Shape s;
  gnn_status r = spmm_shape(g, F, dtype, &s);
  if (r != GNN_OK) return r;
  if (g->n == 0) return GNN_OK;
  if (!arg || !dout || !dx || !aligned(arg, 16) || !aligned(dout, 16) || !aligned(dx, 16))
    return GNN_ERR_INVALID_ARG;
  if (ws_bytes < gnn::reduce_ws_bytes(g, s)) return GNN_ERR_WORKSPACE_TOO_SMALL;
  if (!ws || !aligned(ws, 256)) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_reduce_backward_ordered(g, s, dtype, arg, dout, dx,
                                                       static_cast<char*>(ws),
                                                       static_cast<cudaStream_t>(stream)));
}

gnn_status gnn_wait_selftest(const gnn_graph* g, int polls, void* stream) {
  if (!g || !g->err || polls < 1 || polls > 1000000) return GNN_ERR_INVALID_ARG;
  return from_cuda(gnn::launch_wait_selftest(g, polls, static_cast<cudaStream_t>(stream)));
}

gnn_status gnn_check_device_error(const gnn_graph* g, void* stream, int32_t* info) {
  if (!g || !g->err) return GNN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t w = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GNN_ERR_CUDA;
  if (cudaMemcpy(&w, g->err, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) return GNN_ERR_CUDA;
  if (w != 0 && cudaMemset(g->err, 0, sizeof w) != cudaSuccess) return GNN_ERR_CUDA;
  if (info) *info = w;
  if (w & gnn::DEVERR_TIMEOUT) return GNN_ERR_TIMEOUT;
  if (w) return GNN_ERR_DEVICE_ASSERT;
  return GNN_OK;
}

}  // extern "C"
