/*
 * gnnagg.h -- IO-aware fused GAT neighbour aggregation for one GPU (sm_103a).
 *
 * The operation.  For a directed graph in CSR form (row i lists the sources j
 * of the edges j -> i) and node features h[N][H][D] (H heads of width D), each
 * destination i and head k gets
 *
 *     e_ij   = LeakyReLU(a_dst[k] . h_i[k] + a_src[k] . h_j[k])
 *     alpha  = softmax over the in-neighbours j of i of e_ij
 *     out_i[k] = sum_j alpha_ij h_j[k],   lse_i[k] = log sum_j exp(e_ij)
 *
 * The score is the additive attention of Graph Attention Networks (Velickovic
 * et al., ICLR 2018, eqs. 1-3) with the projection W applied by the caller.
 * Following "On Efficient Scaling of GNNs via IO-Aware Layers Implementations"
 * (Technical Summary > Methodology, attention-based layers), the forward pass
 * computes scores, softmax and aggregation in one streaming pass over each
 * node's neighbours with an online softmax, so no per-edge score, weight or
 * message is ever written to device memory; it keeps the per-node
 * log-sum-exp, from which the backward pass recomputes alpha on the fly.
 * The backward pass walks the CSR for the destination-side gradient terms
 * and a cached transposed adjacency (CSC, built once per graph; same page,
 * SpMM bullet: transposed adjacency cached for the backward pass) for the
 * source-side terms.  Degree-aware tiling (same page, reduction bullet:
 * light and heavy nodes split by a degree threshold, heavy nodes tiled over
 * edge chunks) assigns a warp to each light node, a thread block to each
 * mid-degree node and several thread blocks to each hub, whose partial
 * (max, sum, accumulator) states are merged in a fixed order.  Results are
 * bitwise reproducible run to run.
 *
 * Conventions.
 *   - Every pointer argument named *_d or listed as "device" is a device
 *     pointer on the current device; all device memory is owned by the
 *     caller.  The library keeps only a small host-side struct per graph.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Compute calls are asynchronous on that stream and never synchronise,
 *     except gnn_graph_prepare (two synchronisations) and
 *     gnn_check_device_error (one).
 *   - Feature layout: h, out, dout, dh are [N][H][D] row-major, contiguous,
 *     of the given dtype; lse is float [N][H] (natural log, -inf for a node
 *     with no in-neighbours); a_src, a_dst, da_src, da_dst are float [H][D].
 *   - Supported shapes: D * sizeof(dtype) a multiple of 16 bytes with
 *     D * sizeof(dtype) / 16 a power of two no larger than 32, and
 *     H * D * sizeof(dtype) <= 2048 bytes.  Others return GNN_ERR_UNSUPPORTED.
 *   - h, out, dout, dh, a_src, a_dst must be 16-byte aligned, the workspace
 *     256-byte aligned, col_idx 16-byte aligned.
 *   - Multi-edges count with their multiplicity.  The library adds no
 *     self-loops.  n_edges must be below 2^31.
 *   - Errors never abort, trap or print; every call returns a gnn_status.
 */
#ifndef GNNAGG_H_
#define GNNAGG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GNNAGG_ABI_VERSION 1

typedef enum {
  GNN_OK = 0,
  GNN_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad size, bad enum */
  GNN_ERR_UNSUPPORTED = 2,        /* (H, D, dtype) outside the supported set */
  GNN_ERR_INVALID_GRAPH = 3,      /* CSR failed validation in gnn_graph_prepare */
  GNN_ERR_WORKSPACE_TOO_SMALL = 4,
  GNN_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
  GNN_ERR_DEVICE_ASSERT = 6,      /* a kernel recorded an internal consistency error */
  GNN_ERR_TIMEOUT = 7             /* a kernel gave up a bounded wait (see gnn_check_device_error) */
} gnn_status;

typedef enum { GNN_F32 = 0, GNN_BF16 = 1 } gnn_dtype;

/* Degree-aware tiling thresholds (in edges).  A node of in-degree (CSR) or
 * out-degree (CSC) d is "light" when d <= light_max_deg and gets one warp
 * (or a sub-group of one, for rows narrower than a warp); "mid" when
 * light_max_deg < d <= cta_max_deg and gets one thread block; a "hub"
 * otherwise, split into chunks of hub_chunk edges, one thread block each.
 * light_max_deg = GNN_LIGHT_AUTO lets gnn_graph_prepare choose it from the
 * edge count and the device's SM count: E / (SMs * 512) rounded to a power of
 * two, within [64, 1024] and at most cta_max_deg (gnn_graph_stats reports the
 * value chosen).  Constraints: light_max_deg = GNN_LIGHT_AUTO or
 * 0 <= light_max_deg <= cta_max_deg; cta_max_deg <= 16384;
 * 1 <= hub_chunk <= 16384. */
#define GNN_LIGHT_AUTO (-1)
typedef struct {
  int32_t light_max_deg;
  int32_t cta_max_deg;
  int32_t hub_chunk;
} gnn_tiling;

/* Fills *t with the default thresholds: an automatic light threshold,
 * cta_max_deg 4096, hub_chunk 2048. */
void gnn_default_tiling(gnn_tiling* t);

typedef struct gnn_graph gnn_graph; /* opaque; immutable after prepare */

/* Bytes of caller-owned device memory the prepared graph keeps (CSC
 * transpose, degree buckets, hub chunk tables, status word).  An upper bound
 * computed from sizes only; tiling NULL = defaults.  Returns 0 for invalid
 * sizes. */
size_t gnn_graph_buffer_bytes(int64_t n_nodes, int64_t n_edges, const gnn_tiling* tiling);

/* Bytes of temporary device memory gnn_graph_prepare needs during the call
 * (radix-sort ping-pong buffers, degree arrays, scan partials). */
size_t gnn_graph_scratch_bytes(int64_t n_nodes, int64_t n_edges);

/* Validate a CSR graph and build everything the aggregation kernels read.
 *   row_ptr_d [n_nodes + 1], col_idx_d [n_edges]: device, int32; must stay
 *     alive and unchanged for the lifetime of *out (they are read, not copied).
 *   buffer_d / buffer_bytes: device memory that holds the prepared structures
 *     for the lifetime of *out (>= gnn_graph_buffer_bytes, 256-byte aligned).
 *   scratch_d / scratch_bytes: device memory used only during this call
 *     (>= gnn_graph_scratch_bytes, 256-byte aligned).
 *   tiling: NULL = defaults.
 * Validation: row_ptr[0] = 0, non-decreasing, row_ptr[n] = n_edges, every
 * col_idx in [0, n_nodes); a failure returns GNN_ERR_INVALID_GRAPH.  The CSC
 * lists each column's rows in ascending order (deterministic).  Each light
 * list holds its nodes by descending degree, ties by ascending id, so that
 * the nodes one warp takes at a time have nearly the same edge count (the
 * order of work only: results do not depend on it).  The call
 * synchronises `stream` twice (after validation, and to read bucket counts).
 * On success *out receives a handle owned by the caller (gnn_graph_destroy). */
gnn_status gnn_graph_prepare(int64_t n_nodes, int64_t n_edges, const int32_t* row_ptr_d,
                             const int32_t* col_idx_d, void* buffer_d, size_t buffer_bytes,
                             void* scratch_d, size_t scratch_bytes, const gnn_tiling* tiling,
                             void* stream, gnn_graph** out);

/* Frees the host-side handle only (the device buffer belongs to the caller). */
gnn_status gnn_graph_destroy(gnn_graph* g);

/* Host-side counts recorded by prepare, 16 int64 values:
 *   [0] n_nodes [1] n_edges
 *   [2..7]  CSR (by in-degree):  light nodes, block items, hubs, hub chunks,
 *           max in-degree, longest block item
 *   [8..13] CSC (by out-degree): the same six
 *   [14] light_max_deg in use (the chosen value when it was GNN_LIGHT_AUTO)
 *   [15] cta_max_deg
 * n must be >= 16. */
gnn_status gnn_graph_stats(const gnn_graph* g, int64_t* stats, int n);

/* Device pointers of the prepared structures, for inspection and tests.
 * ptrs[8] receives: CSC col_ptr [N+1], CSC row_idx [E] (int32); CSR light
 * list [light], CSR block items [items] (int4 {node, begin, end, slot}), CSR
 * hubs [hubs] (int4 {node, first slot, chunks, 0}); CSC light, items, hubs.
 * Counts are those of gnn_graph_stats.  All lie inside the caller's buffer. */
gnn_status gnn_graph_arrays(const gnn_graph* g, const void** ptrs, int n);

/* Device memory the compute calls need as workspace, for either pass (the
 * larger of the two), 256-byte aligned sizes.  Grows with the number of hub
 * chunks and with N * H, never with E * H.  Returns 0 for unsupported shapes. */
size_t gat_agg_workspace_bytes(const gnn_graph* g, int H, int D, gnn_dtype dtype);

/* Forward pass.  Writes every element of out [N][H][D] (dtype) and lse
 * [N][H] (float).  h [N][H][D] dtype, a_src/a_dst [H][D] float, all device.
 * slope: LeakyReLU negative slope.  ws: device workspace of ws_bytes bytes
 * (>= gat_agg_workspace_bytes; may be NULL when that is 0).
 * Asynchronous; returns GNN_ERR_CUDA on a launch failure. */
gnn_status gat_agg_forward(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* h,
                           const float* a_src, const float* a_dst, float slope, void* out,
                           float* lse, void* ws, size_t ws_bytes, void* stream);

/* Backward pass of L(out) given dout = dL/dout [N][H][D] (dtype) and the lse
 * [N][H] written by gat_agg_forward on the same inputs.  Writes every element
 * of dh [N][H][D] (dtype), da_src and da_dst [H][D] (float): nothing is
 * accumulated into, so no output needs zeroing.  alpha is recomputed from
 * lse; the only intermediates are O(N * H) per-node statistics and the hub
 * partials in ws.  Asynchronous. */
gnn_status gat_agg_backward(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* h,
                            const float* a_src, const float* a_dst, float slope,
                            const float* lse, const void* dout, void* dh, float* da_src,
                            float* da_dst, void* ws, size_t ws_bytes, void* stream);

/* gat_agg_forward / gat_agg_backward that also record the caller's CUDA
 * events (cudaEvent_t passed as void*) on `stream` between their kernels, for
 * per-kernel timing.  Forward: n_events = 4 -- before the per-node score
 * pre-pass, before the main kernel, after it, after the hub merge.
 * Backward: n_events = 8 -- before the score pre-pass, before the
 * destination-side pass, after its main kernel, after its hub merge, after
 * the source-side main kernel, after its hub merge, after the
 * attention-vector partial sums, at the end.  A kernel with no work records
 * its events back to back.  Other behaviour as the untimed calls. */
gnn_status gat_agg_forward_timed(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* h,
                                 const float* a_src, const float* a_dst, float slope, void* out,
                                 float* lse, void* ws, size_t ws_bytes, void* stream,
                                 void* const* events, int n_events);
gnn_status gat_agg_backward_timed(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                  const void* h, const float* a_src, const float* a_dst,
                                  float slope, const float* lse, const void* dout, void* dh,
                                  float* da_src, float* da_dst, void* ws, size_t ws_bytes,
                                  void* stream, void* const* events, int n_events);

/* gat_agg_backward_timed (events may be NULL) that reuses the per-node score
 * halves a_src . h_n and a_dst . h_n which gat_agg_forward computed into its
 * workspace, instead of computing them again: ws must be the workspace of
 * the forward call on the same h, a_src and a_dst, with nothing written to
 * it since (a training step that passes one workspace to both calls; the
 * caller vouches for that, the library cannot check it).  The page's
 * backward keeps compact per-node statistics from the forward pass; these
 * are two more of them.  Results are bitwise those of gat_agg_backward; the
 * score pre-pass interval of the events is empty. */
gnn_status gat_agg_backward_reuse(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                  const void* h, const float* a_src, const float* a_dst,
                                  float slope, const float* lse, const void* dout, void* dh,
                                  float* da_src, float* da_dst, void* ws, size_t ws_bytes,
                                  void* stream, void* const* events, int n_events);

/* Forward pass that allocates nothing and takes no workspace.  The page has
 * no counterpart to this call; it exists for callers that must not allocate
 * device memory -- for example code that runs under another framework's
 * memory pool, an inference runtime with a static memory plan, or a
 * latency-critical path where an allocation (and the synchronisation it can
 * imply) is not allowed.  Such callers still pass h, a_src, a_dst, out and
 * lse, exactly as for gat_agg_forward, and get the same results.
 * The per-node scores and hub partial states that gat_agg_forward keeps in
 * `ws` go instead to a fixed array inside this library of
 * gat_agg_forward_noalloc_capacity() bytes (16 MiB) on each GPU that loads
 * the library, held until the process exits.  A graph whose forward workspace (gat_agg_workspace_bytes' forward
 * part: about 8 * N * H bytes of per-node scores plus hub chunks * H *
 * (D + 2) * 4 bytes) exceeds that size is rejected with
 * GNN_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and caches it together with
 * the id of the current context; make that first call before any stream
 * capture.  After a device reset (or a new primary context) the next call
 * sees another context id and looks the address up again, so make that
 * call before any capture too.  The device must be the one the graph was
 * prepared on (else GNN_ERR_INVALID_ARG).
 * Every call shares the one array: calls that overlap on the GPU (on
 * different streams, or from several threads) race and must be serialised
 * by the caller.  The array keeps the last call's contents; the call zeroes
 * the few work counters it needs and writes every score and partial before
 * reading it. */
gnn_status gat_agg_forward_noalloc(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                   const void* h, const float* a_src, const float* a_dst,
                                   float slope, void* out, float* lse, void* stream);

/* Size in bytes of the array gat_agg_forward_noalloc uses. */
size_t gat_agg_forward_noalloc_capacity(void);

/* ---- SpMM-family propagation (GCN / GraphConv) --------------------------
 *
 * out = A~ x for node features x[N][F], the propagation step of the layer
 * H' = sigma(A~ H W) ("On Efficient Scaling of GNNs via IO-Aware Layers
 * Implementations", Technical Summary > Methodology, SpMM-based
 * convolutions; W and sigma are the caller's).  For each edge j -> i of the
 * prepared graph (multi-edges with multiplicity):
 *   GNN_NORM_SUM:  A~_ij = 1
 *   GNN_NORM_MEAN: A~_ij = 1 / deg(i)
 *   GNN_NORM_SYM:  A~_ij = 1 / sqrt(deg(i) deg(j))  (D^-1/2 A D^-1/2 of
 *                  Kipf & Welling, ICLR 2017; add self-loops to the graph
 *                  for their A + I)
 * deg(v) = in-degree of v (length of CSR row v); a degree of 0 makes the
 * coefficient 0.  The backward pass dx = A~^T dout walks the cached CSC
 * transpose (same page: transposed adjacency cached for the backward
 * pass); it is the only gradient (A~ does not depend on x).  Both passes
 * use the degree-aware tiling of the attention kernels, write every output
 * element, use no atomics on values and are bitwise reproducible.
 * Shapes: F * sizeof(dtype) a multiple of 16 bytes, at most 2048 bytes.
 * x, out, dout, dx: [N][F] dtype, device, 16-byte aligned; ws: device,
 * 256-byte aligned, >= gcn_agg_workspace_bytes (counters, N per-node
 * coefficients, hub-chunk partial sums).  Asynchronous on `stream`. */
typedef enum { GNN_NORM_SUM = 0, GNN_NORM_MEAN = 1, GNN_NORM_SYM = 2 } gnn_norm;

/* Workspace bytes of gcn_agg_forward / gcn_agg_backward (the same for both);
 * 0 for an unsupported (F, dtype). */
size_t gcn_agg_workspace_bytes(const gnn_graph* g, int F, gnn_dtype dtype);

/* out [N][F] = A~ x. */
gnn_status gcn_agg_forward(const gnn_graph* g, int F, gnn_dtype dtype, gnn_norm norm,
                           const void* x, void* out, void* ws, size_t ws_bytes, void* stream);

/* dx [N][F] = A~^T dout. */
gnn_status gcn_agg_backward(const gnn_graph* g, int F, gnn_dtype dtype, gnn_norm norm,
                            const void* dout, void* dx, void* ws, size_t ws_bytes,
                            void* stream);

/* ---- GATv2 attention -------------------------------------------------------
 *
 * For each destination i and head k, with xl = W_l h (source side; also the
 * aggregated value) and xr = W_r h (destination side) computed by the caller:
 *     e_ij     = att[k] . LeakyReLU(xr_i[k] + xl_j[k])
 *     alpha    = softmax over the in-neighbours j of i of e_ij
 *     out_i[k] = sum_j alpha_ij xl_j[k],   lse_i[k] = log sum_j exp(e_ij)
 * (Brody et al., "How Attentive are Graph Attention Networks?", ICLR 2022,
 * eq. 7; the GATv2 layer of "On Efficient Scaling of GNNs via IO-Aware
 * Layers Implementations", Technical Summary > Methodology, attention-based
 * layers).  Same streaming design as the GAT calls: one pass over each
 * node's in-neighbours with an online softmax, no per-edge tensor in device
 * memory, lse kept for the backward, which walks the CSR (destination side:
 * dxr) and the cached CSC (source side: dxl); each pass adds its per-node
 * share of datt.  Results, datt included, are bitwise reproducible.
 * Layout: xl, xr, out, dout, dxl, dxr [N][H][D] dtype; att, datt [H][D]
 * float; lse [N][H] float.  Shapes as for the GAT calls, with the further
 * limit H * D * sizeof(dtype) <= 512 bytes.  Pointers 16-byte aligned (lse
 * 4), ws 256-byte aligned and >= gatv2_agg_workspace_bytes (hub-chunk
 * partial states, an 8-byte per-(node, head) record, per-block float64
 * datt sums).  Asynchronous on `stream`. */
size_t gatv2_agg_workspace_bytes(const gnn_graph* g, int H, int D, gnn_dtype dtype);

gnn_status gatv2_agg_forward(const gnn_graph* g, int H, int D, gnn_dtype dtype, const void* xl,
                             const void* xr, const float* att, float slope, void* out,
                             float* lse, void* ws, size_t ws_bytes, void* stream);

/* Gradients of L(out) given dout and the forward's lse: writes every element
 * of dxl, dxr (dtype) and datt (float). */
gnn_status gatv2_agg_backward(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                              const void* xl, const void* xr, const float* att, float slope,
                              const float* lse, const void* dout, void* dxl, void* dxr,
                              float* datt, void* ws, size_t ws_bytes, void* stream);

/* ---- Graph-transformer attention -------------------------------------------
 *
 * For each destination i and head k, with the query, key and value
 * projections q, key, val computed by the caller:
 *     e_ij     = scale * q_i[k] . key_j[k]        (scale = 1/sqrt(D) usually)
 *     alpha    = softmax over the in-neighbours j of i of e_ij
 *     out_i[k] = sum_j alpha_ij val_j[k],   lse_i[k] = log sum_j exp(e_ij)
 * (Shi et al., "Masked Label Prediction: Unified Message Passing Model for
 * Semi-Supervised Classification", IJCAI 2021, eqs. 3-4; the Graph
 * Transformer layer of "On Efficient Scaling of GNNs via IO-Aware Layers
 * Implementations", Technical Summary > Methodology, attention-based
 * layers).  One streaming pass per node with an online softmax; no per-edge
 * tensor in device memory; the backward recomputes alpha from lse, walking
 * the CSR for dq and the cached CSC for dkey and dval.  Bitwise
 * reproducible.
 * Layout: q, key, val, out, dout, dq, dkey, dval [N][H][D] dtype; lse [N][H]
 * float.  Shapes as for gatv2 (H * D * sizeof(dtype) <= 512 bytes).
 * Pointers 16-byte aligned (lse 4), ws 256-byte aligned and >=
 * transformer_agg_workspace_bytes.  Asynchronous on `stream`. */
size_t transformer_agg_workspace_bytes(const gnn_graph* g, int H, int D, gnn_dtype dtype);

gnn_status transformer_agg_forward(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                   const void* q, const void* key, const void* val, float scale,
                                   void* out, float* lse, void* ws, size_t ws_bytes,
                                   void* stream);

/* Writes every element of dq, dkey and dval. */
gnn_status transformer_agg_backward(const gnn_graph* g, int H, int D, gnn_dtype dtype,
                                    const void* q, const void* key, const void* val, float scale,
                                    const float* lse, const void* dout, void* dq, void* dkey,
                                    void* dval, void* ws, size_t ws_bytes, void* stream);

/* ---- Max / min neighbourhood reduction -----------------------------------
 *
 * out[i][f] = max (or min) over the in-neighbours j of i of x[j][f], and
 * arg[i][f] = the winning j (the smallest j among equal values); a node with
 * no in-neighbours gets out = 0 and arg = -1.  The reduction-based
 * aggregation of "On Efficient Scaling of GNNs via IO-Aware Layers
 * Implementations" (Technical Summary > Methodology, reduction-based
 * aggregations: per-edge message, then a neighbourhood max or min) with the
 * message x_j (per-node transforms are the caller's).  Degree-aware tiling
 * as on that page: a warp per light node, a block per mid node, hubs split
 * into edge chunks merged by 64-bit atomicMax on packed (value, source)
 * keys.  out and arg are exact (out is always an input value) and bitwise
 * reproducible.  Inputs must not hold NaN.
 * Backward: dx[j][f] = sum of dout[i][f] over the i with arg[i][f] = j,
 * accumulated with float32 atomic adds; where several destinations share a
 * winner the order of those additions, and so the last bits of dx, may vary
 * from run to run.
 * Shapes as for the GCN calls (F * sizeof(dtype) a multiple of 16, at most
 * 2048 bytes).  x, out, dout, dx: [N][F] dtype; arg: [N][F] int32; all
 * device, 16-byte aligned; ws 256-byte aligned, >= reduce_agg_workspace_bytes
 * (counters, N_hub_chunks * F packed keys, and N * F floats for the
 * backward's accumulator; at least the SpMM workspace size, which the
 * ordered backward uses).  Asynchronous on `stream`. */
typedef enum { GNN_REDUCE_MAX = 0, GNN_REDUCE_MIN = 1 } gnn_reduce_op;

size_t reduce_agg_workspace_bytes(const gnn_graph* g, int F, gnn_dtype dtype);

gnn_status reduce_agg_forward(const gnn_graph* g, int F, gnn_dtype dtype, gnn_reduce_op op,
                              const void* x, void* out, int32_t* arg, void* ws, size_t ws_bytes,
                              void* stream);

/* dx [N][F] from the forward's arg and dout; writes every element of dx. */
gnn_status reduce_agg_backward(const gnn_graph* g, int F, gnn_dtype dtype, const int32_t* arg,
                               const void* dout, void* dx, void* ws, size_t ws_bytes,
                               void* stream);

/* The same dx without atomics, bitwise reproducible: for each source j, the
 * cached CSC transpose (rows ascending) is walked and dout[i][f] is added
 * where arg[i][f] = j, with the degree-aware tiling of the SpMM backward
 * (hub chunks summed in chunk order).  It reads the winners and dout rows
 * once per edge rather than once per node, so it moves more bytes than
 * reduce_agg_backward.  Arguments, workspace and errors as
 * reduce_agg_backward. */
gnn_status reduce_agg_backward_ordered(const gnn_graph* g, int F, gnn_dtype dtype,
                                       const int32_t* arg, const void* dout, void* dx, void* ws,
                                       size_t ws_bytes, void* stream);

/* Synchronises `stream`, reads and clears the graph's device status word.
 * Returns GNN_OK, GNN_ERR_TIMEOUT (a bounded wait on an asynchronous copy ran
 * out) or GNN_ERR_DEVICE_ASSERT; *info (may be NULL) receives the raw word. */
gnn_status gnn_check_device_error(const gnn_graph* g, void* stream, int32_t* info);

/* Diagnostic with no counterpart on the page: makes one bounded device wait
 * run out, to exercise the error path that replaces a hang.  A single thread
 * waits on a shared-memory mbarrier that nothing will complete, gives up
 * after `polls` polls (1 .. 1,000,000), sets the timeout bit of g's status
 * word and returns; nothing stays in flight and the context remains usable.
 * A following gnn_check_device_error returns GNN_ERR_TIMEOUT (and clears the
 * word).  Asynchronous on `stream`. */
gnn_status gnn_wait_selftest(const gnn_graph* g, int polls, void* stream);

/* Static description of a status code. */
const char* gnn_status_string(gnn_status s);

/* GNNAGG_ABI_VERSION of the loaded library. */
int gnn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GNNAGG_H_ */
