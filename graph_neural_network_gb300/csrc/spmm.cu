// SpMM-family neighbour aggregation: the propagation out = A~ x of GCN /
// GraphConv layers, H' = sigma(A~ H W) ("On Efficient Scaling of GNNs via
// IO-Aware Layers Implementations", Technical Summary > Methodology,
// SpMM-based convolutions), with W and sigma outside.  For the edge j -> i
//   sum:  A~_ij = 1      mean: A~_ij = 1 / deg(i)
//   sym:  A~_ij = 1 / sqrt(deg(i) deg(j))   (Kipf & Welling's D^-1/2 A D^-1/2)
// deg = in-degree (CSR row length); a degree of 0 gives a coefficient of 0.
// The backward pass dx = A~^T dout runs the same kernel over the cached CSC
// transpose (same page: transposed adjacency cached for the backward pass),
// so no atomics or scatters are needed and results are reproducible bit for
// bit.
//
// A~ factors as diag(c_out) A diag(c_in) with per-node coefficients (1/deg
// or deg^-1/2) computed once per call from row_ptr; each edge gathers one
// feature row and one float.  Degree-aware tiling as in the attention
// kernels: light nodes get a warp, or a sub-group of their own where a row is
// narrower than a warp, mid nodes a block (edge list staged in shared memory
// by a bulk copy), hubs are split into edge chunks whose partial sums a
// second kernel adds in chunk order.  Rows that start on 32-byte boundaries
// and hold an even number of 16-byte vectors (up to 1024 bytes) are read as
// 32-byte lane vectors.
#include "device.cuh"

namespace gnn {
namespace {

constexpr int kGrab = 4;  // light nodes a warp takes per counter access

struct SpmmArgs {
  Shape s;           // one 16-byte vector per "head": no per-head arithmetic
  const int32_t* ptr;
  const int32_t* idx;
  const int32_t* light;
  int64_t n_light;
  const int4* items;
  int64_t n_items;
  const int4* hubs;
  int64_t n_hubs;
  const void* x;
  void* out;
  const float* c_out;  // [N] coefficient of the output node, or null (= 1)
  const float* c_in;   // [N] coefficient of the gathered node, or null (= 1)
  const int32_t* win;  // masked mode: [N][F] winners; edge term kept where win == node
  float* part;         // [hub chunks][row floats]
  int* ctr;            // [0] block items taken, [1] light nodes taken
  int32_t* err;
  int col_off;         // bytes of shared memory before the per-warp sums
};

// Per-node coefficient from the in-degree: mode 1 -> 1/deg, mode 2 -> deg^-1/2
// (0 where deg = 0).
__global__ void spmm_coef(const int32_t* ptr, int64_t n, int mode, float* c) {
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < n;
       v += int64_t(gridDim.x) * blockDim.x) {
    const int d = ptr[v + 1] - ptr[v];
    c[v] = d <= 0 ? 0.f : (mode == 1 ? 1.f / float(d) : rsqrtf(float(d)));
  }
}

// Edges in flight per lane: 64 bytes of rows (4 edges of 16-byte lane
// vectors, 2 of 32-byte ones), or two in the masked mode (each edge also
// gathers the row's winners, four bytes per feature; 16-byte vectors only).
template <bool kMask, int VB>
struct SpmmUnroll {
  static constexpr int value = kMask ? 2 : UnrollOf<VB>::value;
};

// acc += c_in(j) x_j over the edges beg + sg, beg + sg + SG, ... < end
// (sg, SG: this lane's sub-group and the sub-groups sharing the node; 0, 1
// when a sub-group has the node to itself).  Masked mode (the max / min
// backward over the CSC, `self` the output node whose list starts at edge
// `colstart`): acc[f] += x_j[f] where win[j][f] == self, once per destination
// j -- a repeated edge (the same j right before it in the ascending list)
// adds nothing, since a winner is counted per destination, not per edge.
template <typename T, int NV, int VB, bool kMask>
__device__ __forceinline__ void spmm_edges(const SpmmArgs& A, const Lane<NV>& L, int self,
                                           int colstart, const int32_t* cols, int colbase,
                                           int beg, int end, int sg, int SG, int step,
                                           int (&jn)[SpmmUnroll<kMask, VB>::value],
                                           float (&acc)[NV][ElemsOf<T, VB>::n]) {
  static_assert(!kMask || VB == 16, "masked mode uses 16-byte lane vectors");
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = SpmmUnroll<kMask, VB>::value;
  const int row_f = A.s.rv * V;
  for (int base = beg; base < end; base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    RawV<VB> raw[U][NV];
    float w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int v = 0; v < NV; ++v)
        raw[u][v] = (j[u] >= 0 && L.ok[v])
                        ? ldv<VB>(row_at<VB>(A.x, j[u], A.s.rv) + VB * L.q[v])
                        : zero_raw<VB>();
      w[u] = j[u] < 0 ? 0.f : (A.c_in ? __ldg(A.c_in + j[u]) : 1.f);
    }
    int wn[kMask ? U : 1][kMask ? NV : 1][kMask ? V : 1];
    if constexpr (kMask) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = base + u * SG + sg;
        const bool repeat = j[u] >= 0 && e > colstart && __ldg(A.idx + e - 1) == j[u];
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int c4 = 0; c4 < V; c4 += 4) {
            const int4 a = (j[u] >= 0 && !repeat && L.ok[v])
                               ? __ldg(reinterpret_cast<const int4*>(
                                     A.win + int64_t(j[u]) * row_f + L.q[v] * V + c4))
                               : make_int4(-1, -1, -1, -1);
            wn[u][v][c4] = a.x;
            wn[u][v][c4 + 1] = a.y;
            wn[u][v][c4 + 2] = a.z;
            wn[u][v][c4 + 3] = a.w;
          }
      }
    }
    if (base + step < end) batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float xv[V];
        unpackv<T, VB>(raw[u][v], xv);
        if constexpr (kMask) {
#pragma unroll
          for (int c = 0; c < V; ++c) acc[v][c] += wn[u][v][c] == self ? xv[c] : 0.f;
        } else {
          axpy<V>(acc[v], w[u], xv);
        }
      }
  }
}

template <typename T, int NV, int VB>
__device__ __forceinline__ void zero(float (&acc)[NV][ElemsOf<T, VB>::n]) {
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int c = 0; c < ElemsOf<T, VB>::n; ++c) acc[v][c] = 0.f;
}

// Sum the accumulators of the warp's sub-groups (every lane ends with the total).
template <typename T, int NV, int VB>
__device__ __forceinline__ void subgroup_sums(const Shape& s,
                                              float (&acc)[NV][ElemsOf<T, VB>::n]) {
  for (int o = s.lpr; o < 32; o <<= 1)
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int c = 0; c < ElemsOf<T, VB>::n; ++c)
        acc[v][c] += __shfl_xor_sync(kFull, acc[v][c], o);
}

// out_node = c_out(node) * acc.
template <typename T, int NV, int VB>
__device__ __forceinline__ void write_row(const SpmmArgs& A, const Lane<NV>& L, int64_t node,
                                          float (&acc)[NV][ElemsOf<T, VB>::n]) {
  const float c = A.c_out ? __ldg(A.c_out + node) : 1.f;
  char* orow = reinterpret_cast<char*>(A.out) + node * int64_t(A.s.rv) * VB;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!L.ok[v]) continue;
    scale<ElemsOf<T, VB>::n>(acc[v], c);
    storev<T, VB>(orow + VB * L.q[v], acc[v]);
  }
}

template <typename T, int NV, int VB, bool kMask, bool kSub>
__global__ void __launch_bounds__(kThreads, MinBlocksLean<NV>::value) spmm_main(const SpmmArgs A) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = SpmmUnroll<kMask, VB>::value;
  const Lane<NV> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  float acc[NV][V];

  // ---- block items: mid nodes and hub chunks -----------------------------
  if (A.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    float* wacc = reinterpret_cast<float*>(smem + A.col_off);  // [kWarps][row_f]
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 0, 1);
      __syncthreads();
      const int it_i = s_item;
      if (it_i >= A.n_items) break;
      const int4 it = A.items[it_i];
      if (!stage_edges(cols, A.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of U * G edges dealt to the warps in turn
      const int wb = it.y + wid * U * L.G;
      const int colbase = it.y & ~3;
      int jn[U];
      batch_ids<U>(cols, colbase, wb, it.z, L.g, L.G, jn);
      zero<T, NV, VB>(acc);
      spmm_edges<T, NV, VB, kMask>(A, L, it.x, kMask ? A.ptr[it.x] : 0, cols, colbase, wb, it.z,
                                   L.g, L.G, kWarps * U * L.G, jn, acc);
      subgroup_sums<T, NV, VB>(A.s, acc);
      if (L.g == 0)
#pragma unroll
        for (int v = 0; v < NV; ++v)
          if (L.ok[v])
#pragma unroll
            for (int c = 0; c < V; ++c) wacc[wid * row_f + L.q[v] * V + c] = acc[v][c];
      __syncthreads();
      if (wid == 0 && L.g == 0) {
        // warp 0 adds the warps' sums in warp order
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int c = 0; c < V; ++c) {
            float t = 0.f;
            if (L.ok[v])
              for (int w = 0; w < kWarps; ++w) t += wacc[w * row_f + L.q[v] * V + c];
            acc[v][c] = t;
          }
        if (it.w < 0) {
          write_row<T, NV, VB>(A, L, it.x, acc);
        } else {
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            if (!L.ok[v]) continue;
            float* pa = A.part + int64_t(it.w) * row_f + L.q[v] * V;
#pragma unroll
            for (int c4 = 0; c4 < V; c4 += 4)
              *reinterpret_cast<float4*>(pa + c4) =
                  make_float4(acc[v][c4], acc[v][c4 + 1], acc[v][c4 + 2], acc[v][c4 + 3]);
          }
        }
      }
      __syncthreads();  // shared memory is reused by the next item
    }
  }

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  if constexpr (kSub) {
    // a pull takes two nodes per sub-group, four where a warp holds two
    // sub-groups (eight per pull: 2 % faster on 512-byte rows); the edge loop
    // has no shuffles, so the sub-groups of a warp run their own trip counts
    // (the light list is sorted by degree, so they are nearly equal)
    const int R = L.G == 2 ? 4 : 2;
    const int npull = R * L.G;
    for (;;) {
      int t0 = 0;
      if (L.lane == 0) t0 = atomicAdd(A.ctr + 1, npull);
      t0 = __shfl_sync(kFull, t0, 0);
      if (t0 >= A.n_light) break;
#pragma unroll 1
      for (int r = 0; r < R; ++r) {
        const int64_t t = int64_t(t0) + r * L.G + L.g;
        if (t >= A.n_light) break;
        const int i = __ldg(A.light + t);
        const int beg = __ldg(A.ptr + i), end = __ldg(A.ptr + i + 1);
        int jn[U];
        batch_ids<U>(A.idx, 0, beg, end, 0, 1, jn);
        zero<T, NV, VB>(acc);
        spmm_edges<T, NV, VB, kMask>(A, L, i, beg, A.idx, 0, beg, end, 0, 1, U, jn, acc);
        write_row<T, NV, VB>(A, L, i, acc);
      }
    }
    return;
  }

  // ---- light nodes, rows of a whole warp: one warp each, kGrab at a time --
  for (;;) {
    int t0 = 0;
    if (L.lane == 0) t0 = atomicAdd(A.ctr + 1, kGrab);
    t0 = __shfl_sync(kFull, t0, 0);
    if (t0 >= A.n_light) break;
    int my_i = -1, my_b = 0, my_e = 0;
    if (L.lane < kGrab && t0 + L.lane < A.n_light) {
      my_i = A.light[t0 + L.lane];
      my_b = A.ptr[my_i];
      my_e = A.ptr[my_i + 1];
    }
    int i = __shfl_sync(kFull, my_i, 0);
    int beg = __shfl_sync(kFull, my_b, 0), end = __shfl_sync(kFull, my_e, 0);
    int jn[U];
    batch_ids<U>(A.idx, 0, beg, end, L.g, L.G, jn);
    for (int q = 0; q < kGrab && i >= 0; ++q) {
      const int nq = (q + 1) & (kGrab - 1);
      const int i2 = q + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[U];
      batch_ids<U>(A.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      zero<T, NV, VB>(acc);
      spmm_edges<T, NV, VB, kMask>(A, L, i, beg, A.idx, 0, beg, end, L.g, L.G, U * L.G, jn, acc);
      subgroup_sums<T, NV, VB>(A.s, acc);
      if (L.g == 0) write_row<T, NV, VB>(A, L, i, acc);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < U; ++u) jn[u] = jn2[u];
    }
  }
}

// One warp per hub: add its chunk partials in chunk order.
template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) spmm_merge(const SpmmArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<NV> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.n_hubs || L.g != 0) return;
  const int4 hb = A.hubs[t];
  const int row_f = A.s.rv * V;
  float acc[NV][V], cmp[NV][V];
  zero<T, NV, 16>(acc);
  zero<T, NV, 16>(cmp);
  for (int c = 0; c < hb.z; ++c) {
    const int64_t slot = int64_t(hb.y) + c;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      if (!L.ok[v]) continue;
      const float* pa = A.part + slot * row_f + L.q[v] * V;
#pragma unroll
      for (int c4 = 0; c4 < V; c4 += 4) {
        const float4 p = *reinterpret_cast<const float4*>(pa + c4);
        kahan_add(acc[v][c4], cmp[v][c4], p.x);
        kahan_add(acc[v][c4 + 1], cmp[v][c4 + 1], p.y);
        kahan_add(acc[v][c4 + 2], cmp[v][c4 + 2], p.z);
        kahan_add(acc[v][c4 + 3], cmp[v][c4 + 3], p.w);
      }
    }
  }
  write_row<T, NV, 16>(A, L, hb.x, acc);
}

// The persistent kernel for A's shape: a sub-group per light node where a
// row is narrower than a warp.
template <typename T, int NV, int VB>
cudaError_t launch_main(const SpmmArgs& A, int sm_count, cudaStream_t st) {
  constexpr int V = ElemsOf<T, VB>::n;
  if (A.n_items + A.n_light <= 0) return cudaSuccess;
  const bool sub = A.s.lpr < 32;
  void (*kernel)(const SpmmArgs);
  if constexpr (VB == 32) {
    kernel = sub ? spmm_main<T, NV, VB, false, true> : spmm_main<T, NV, VB, false, false>;
  } else if constexpr (NV == 1) {
    if (A.win)
      kernel = sub ? spmm_main<T, NV, VB, true, true> : spmm_main<T, NV, VB, true, false>;
    else
      kernel = sub ? spmm_main<T, NV, VB, false, true> : spmm_main<T, NV, VB, false, false>;
  } else {
    kernel = A.win ? spmm_main<T, NV, VB, true, false> : spmm_main<T, NV, VB, false, false>;
  }
  const size_t smem = size_t(A.col_off) + size_t(kWarps) * A.s.rv * V * 4;
  cudaError_t e;
  if (smem > 48 * 1024 &&
      (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(smem))) != cudaSuccess)
    return e;
  const int64_t work = A.n_items + (A.n_light + kWarps * kGrab - 1) / (kWarps * kGrab);
  const int64_t cap = persistent_blocks(kernel, smem, sm_count);
  const int64_t blocks = work < cap ? work : cap;
  kernel<<<unsigned(blocks), kThreads, smem, st>>>(A);
  return cudaGetLastError();
}

// Hub merge over the 16-byte-vector shape of the row (the chunk partials are
// plain float rows whatever lane vectors the main kernel used).
template <typename T>
cudaError_t launch_merge(const SpmmArgs& A16, cudaStream_t st) {
  if (A16.n_hubs <= 0) return cudaSuccess;
  const unsigned grid = unsigned((A16.n_hubs + kWarps - 1) / kWarps);
  switch (A16.s.nv) {
    case 1: spmm_merge<T, 1><<<grid, kThreads, 0, st>>>(A16); break;
    case 2: spmm_merge<T, 2><<<grid, kThreads, 0, st>>>(A16); break;
    case 4: spmm_merge<T, 4><<<grid, kThreads, 0, st>>>(A16); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// 32-byte lane vectors: rows of an even number of 16-byte vectors up to
// 1024 bytes, one vector per lane.
bool spmm_wide_shape(const Shape& s, Shape* w) {
  if (s.rv % 2 || s.rv > 64) return false;
  *w = s;
  w->rv = s.rv / 2;
  w->hv = 1;
  w->hv_log2 = 0;
  w->nv = 1;
  w->lpr = 1;
  while (w->lpr < w->rv) w->lpr <<= 1;
  w->lpr_log2 = 0;
  while ((1 << w->lpr_log2) < w->lpr) ++w->lpr_log2;
  return true;
}

template <typename T>
cudaError_t launch_all(const SpmmArgs& A16, int sm_count, cudaStream_t st) {
  cudaError_t e;
  Shape w;
  if (!A16.win && spmm_wide_shape(A16.s, &w) && aligned32(A16.x)) {
    SpmmArgs A = A16;
    A.s = w;
    e = launch_main<T, 1, 32>(A, sm_count, st);
  } else {
    switch (A16.s.nv) {
      case 1: e = launch_main<T, 1, 16>(A16, sm_count, st); break;
      case 2: e = launch_main<T, 2, 16>(A16, sm_count, st); break;
      case 4: e = launch_main<T, 4, 16>(A16, sm_count, st); break;
      default: return cudaErrorInvalidValue;
    }
  }
  if (e != cudaSuccess) return e;
  return launch_merge<T>(A16, st);
}

}  // namespace

cudaError_t launch_spmm(const gnn_graph* g, const Shape& s, gnn_dtype dt, int norm, bool transpose,
                        const void* x, void* out, char* ws, cudaStream_t st,
                        const int32_t* win) {
  const Dir& d = transpose ? g->csc : g->csr;
  SpmmArgs A{};
  A.s = s;
  A.ptr = d.ptr;
  A.idx = d.idx;
  A.light = d.light;
  A.n_light = d.n_light;
  A.items = d.items;
  A.n_items = d.n_items;
  A.hubs = d.hubs;
  A.n_hubs = d.n_hubs;
  A.x = x;
  A.out = out;
  A.win = win;
  A.ctr = reinterpret_cast<int*>(ws);
  float* coef = reinterpret_cast<float*>(ws + kSpmmCoefOffset);
  A.part = reinterpret_cast<float*>(ws + kSpmmCoefOffset + align_up(size_t(g->n) * 4, 256));
  A.err = g->err;
  A.col_off = int(16 + align_up(size_t(d.max_item + 4) * 4, 16));
  // A~ = diag(c_out) A diag(c_in): forward over the CSR, A~^T over the CSC
  if (norm == GNN_NORM_MEAN) {
    (transpose ? A.c_in : A.c_out) = coef;
  } else if (norm == GNN_NORM_SYM) {
    A.c_in = coef;
    A.c_out = coef;
  }
  cudaError_t e;
  if ((e = cudaMemsetAsync(A.ctr, 0, kCounters * sizeof(int), st)) != cudaSuccess) return e;
  if (norm != GNN_NORM_SUM && g->n > 0) {
    int64_t blocks = (g->n + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(g->sm_count > 0 ? g->sm_count : 1) * 8;
    if (blocks > cap) blocks = cap;
    spmm_coef<<<unsigned(blocks), kThreads, 0, st>>>(g->csr.ptr, g->n,
                                                     norm == GNN_NORM_MEAN ? 1 : 2, coef);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (dt == GNN_F32) return launch_all<float>(A, g->sm_count, st);
  return launch_all<__nv_bfloat16>(A, g->sm_count, st);
}

size_t spmm_ws_bytes(const gnn_graph* g, const Shape& s) {
  int64_t chunks = g->csr.n_hub_chunks > g->csc.n_hub_chunks ? g->csr.n_hub_chunks
                                                             : g->csc.n_hub_chunks;
  const size_t row_f = size_t(s.rv) * 16 / s.esize;
  return kSpmmCoefOffset + align_up(size_t(g->n) * 4, 256) +
         align_up(size_t(chunks) * row_f * 4 + 1, 256);
}

}  // namespace gnn
