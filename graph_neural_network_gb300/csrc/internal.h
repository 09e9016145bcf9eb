// Internal structures shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gnnagg.h"

namespace gnn {

// Device status word bits.
enum : int32_t {
  DEVERR_BAD_ROW_PTR = 1 << 0,  // row_ptr[0] != 0, decreasing, or row_ptr[N] != E
  DEVERR_BAD_COL = 1 << 1,      // col_idx outside [0, N)
  DEVERR_TIMEOUT = 1 << 4,      // a bounded mbarrier wait ran out
  DEVERR_INTERNAL = 1 << 5,     // an internal consistency check failed
};

// One direction of the adjacency with its degree buckets.
//   CSR: ptr/idx = caller's row_ptr/col_idx, grouped by destination (in-edges)
//   CSC: ptr/idx = transpose built by prepare, grouped by source (out-edges)
// items: {node, begin, end, slot}; slot >= 0 marks one chunk of a hub (its
// partial state goes to workspace slot `slot`), slot < 0 a whole mid node.
// Hub chunks come first (ascending node, then chunk), then mid nodes.
// hubs: {node, first_slot, n_chunks, 0}.
struct Dir {
  const int32_t* ptr = nullptr;
  const int32_t* idx = nullptr;
  int32_t* light = nullptr;
  int4* items = nullptr;
  int4* hubs = nullptr;
  int64_t n_light = 0, n_items = 0, n_hubs = 0, n_hub_chunks = 0;
  int32_t max_deg = 0, max_item = 0;
};

}  // namespace gnn

struct gnn_graph {
  int64_t n = 0, e = 0;
  gnn_tiling tiling{};
  gnn::Dir csr, csc;
  int32_t* err = nullptr;  // device status word (in the caller's buffer)
  bool csr_sorted = true;  // every CSR row lists its sources in non-decreasing order
  int device = 0;
  int sm_count = 0;
};

namespace gnn {

// Per-call shape of the feature rows.
struct Shape {
  int H = 0, D = 0;
  int esize = 0;  // bytes per element
  int rv = 0;     // 16-byte vectors per row (H * D * esize / 16)
  int hv = 0;     // 16-byte vectors per head (power of two, <= 32)
  int lpr = 0;    // lanes per row (power of two, <= 32)
  int nv = 0;     // vectors per lane (1, 2 or 4)
  int hv_log2 = 0, lpr_log2 = 0;
};

// Workspace layout of one call (byte offsets into ws, 256-aligned).
struct WsLayout {
  size_t fwd_ctr = 0, fwd_scores = 0, fwd_acc = 0, fwd_ml = 0, fwd_total = 0;
  size_t bwd_ctr = 0, bwd_scores = 0, stats = 0, ds_src = 0, dst_part = 0, src_acc = 0,
         src_sum = 0, da_part = 0, bwd_total = 0;
  int da_blocks = 0;
};

// Work counters at the head of each call's workspace, zeroed by the launcher
// before the persistent kernels pull work from them.
constexpr int kCounters = 8;

// Automatic light-node threshold.  A light node runs on one warp or
// sub-group with no barrier and no merge, while a block item pays a work
// pull, the staging of its edge list and a block-wide merge; so as many
// nodes as possible should be light, as long as the largest light node (its
// edges walked by one sub-group) stays short beside the work of one resident
// warp.  With 32 resident warps per SM, E / (SMs * 32) edges per warp, the
// threshold is a sixteenth of that, rounded to a power of two, within
// [kLightAutoMin, kLightAutoMax] and at most cta_max_deg.  On GB300 this is
// 256 for 18.7M edges and 1024 for 118M or more.
constexpr int kLightAutoMin = 64;
constexpr int kLightAutoMax = 1024;
inline int auto_light_max(int64_t e, int sm_count, int cta_max_deg) {
  const double per = double(e) / (double(sm_count > 0 ? sm_count : 1) * 32.0 * 16.0);
  int t = kLightAutoMin;
  // nearest power of two on a log scale: double while per >= t * sqrt(2)
  while (t < kLightAutoMax && per >= double(t) * 1.4142135623730951) t *= 2;
  return t < cta_max_deg ? t : cta_max_deg;
}

bool make_shape(int H, int D, gnn_dtype dt, Shape* s);
// The geometry of 32-byte lane vectors for the same rows (false when a head
// spans less than 32 bytes or a row more than 1024).
bool make_wide_shape(const Shape& s, Shape* w);
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
WsLayout ws_layout(const gnn_graph* g, const Shape& s);

// Kernel launchers (gat_fwd.cu, gat_bwd.cu); return the launch error.
cudaError_t launch_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt, const void* h,
                           const float* a_src, const float* a_dst, float slope, void* out,
                           float* lse, char* ws, const WsLayout& L, cudaStream_t st,
                           const cudaEvent_t* ev);
cudaError_t launch_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt, const void* h,
                            const float* a_src, const float* a_dst, float slope,
                            const float* lse, const void* dout, void* dh, float* da_src,
                            float* da_dst, char* ws, const WsLayout& L, cudaStream_t st,
                            const cudaEvent_t* ev, bool reuse_scores);

// Per-node base-2 score halves s_src, s_dst [N][H] (scores.cu).
cudaError_t launch_node_scores(const Shape& s, gnn_dtype dt, const void* h, const float* a_src,
                               const float* a_dst, int64_t n, float* ssrc, float* sdst,
                               int sm_count, cudaStream_t st);

// SpMM-family propagation (spmm.cu): out = A~ x over the CSR, or A~^T x
// over the CSC (transpose).  Workspace: counters, then the per-node
// coefficients at kSpmmCoefOffset, then the hub partial sums.
constexpr size_t kSpmmCoefOffset = 256;
// win (optional): the masked mode of the max / min backward, edge terms kept
// only where the gathered row's winner is the output node (norm "sum").
cudaError_t launch_spmm(const gnn_graph* g, const Shape& s, gnn_dtype dt, int norm, bool transpose,
                        const void* x, void* out, char* ws, cudaStream_t st,
                        const int32_t* win = nullptr);
size_t spmm_ws_bytes(const gnn_graph* g, const Shape& s);

// Max / min neighbourhood reduction (reduce.cu).  Workspace: counters,
// packed hub keys, float32 gradient accumulator.
size_t reduce_ws_bytes(const gnn_graph* g, const Shape& s);
cudaError_t launch_reduce_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt, int op,
                                  const void* x, void* out, int32_t* arg, char* ws,
                                  cudaStream_t st);
cudaError_t launch_reduce_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                   const int32_t* arg, const void* dout, void* dx, char* ws,
                                   cudaStream_t st);
// The same gradient without atomics: a gather over the cached CSC in a fixed
// order (bitwise reproducible).
cudaError_t launch_reduce_backward_ordered(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                           const int32_t* arg, const void* dout, void* dx,
                                           char* ws, cudaStream_t st);

// GATv2 attention (gatv2.cu), rows of at most 512 bytes.
size_t gatv2_ws_bytes(const gnn_graph* g, const Shape& s);
cudaError_t launch_gatv2_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                 const void* xl, const void* xr, const float* att, float slope,
                                 void* out, float* lse, char* ws, cudaStream_t st);
cudaError_t launch_gatv2_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                  const void* xl, const void* xr, const float* att, float slope,
                                  const float* lse, const void* dout, void* dxl, void* dxr,
                                  float* datt, char* ws, cudaStream_t st);

// Graph-transformer attention (transformer.cu), rows of at most 512 bytes.
size_t transformer_ws_bytes(const gnn_graph* g, const Shape& s);
cudaError_t launch_transformer_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                       const void* q, const void* key, const void* val,
                                       float scale, void* out, float* lse, char* ws,
                                       cudaStream_t st);
cudaError_t launch_transformer_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                        const void* q, const void* key, const void* val,
                                        float scale, const float* lse, const void* dout,
                                        void* dq, void* dkey, void* dval, char* ws,
                                        cudaStream_t st);

// Bounded-wait self-test (diag.cu).
cudaError_t launch_wait_selftest(const gnn_graph* g, int polls, cudaStream_t st);

// Graph preparation (prepare.cu).
gnn_status prepare_graph(gnn_graph* g, const int32_t* row_ptr, const int32_t* col,
                         char* buffer, size_t buffer_bytes, char* scratch, size_t scratch_bytes,
                         cudaStream_t st);
size_t graph_buffer_bytes(int64_t n, int64_t e, const gnn_tiling& t);
size_t graph_scratch_bytes(int64_t n, int64_t e);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace gnn
