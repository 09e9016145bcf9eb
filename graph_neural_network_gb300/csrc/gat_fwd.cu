// Forward pass of the fused GAT neighbour aggregation.
//
// One streaming pass over each destination's in-neighbours: the source row
// h_j is gathered once (16-byte vector loads spread over the lanes of a
// sub-group), its score half a_src . h_j is reduced across the lanes of each
// head, and an online softmax keeps the running (max, sum, accumulator) in
// registers ("On Efficient Scaling of GNNs via IO-Aware Layers
// Implementations", Technical Summary > Methodology, attention-based layers:
// fused CSR kernel, online softmax in registers, per-node log-sum-exp).  No
// per-edge score, weight or message is stored.
//
// Scores are kept in base 2 (a_src and a_dst are pre-scaled by log2 e, which
// commutes with LeakyReLU), so every exponential is one exp2f; lse is stored
// in natural log.
//
// Degree-aware tiling: light nodes get one warp each; mid-degree nodes one
// thread block whose warps split the edge list (staged in shared memory by a
// bulk copy) and merge their states in warp order; hubs are split into edge
// chunks, one block each, whose partial states a second kernel folds in chunk
// order.  Every merge has a fixed order, so results are reproducible.
#include "device.cuh"

namespace gnn {
namespace {

struct FwdArgs {
  Shape s;
  const int32_t* ptr;
  const int32_t* idx;
  const int32_t* light;
  int64_t n_light;
  const int4* items;
  int64_t n_items;
  const int4* hubs;
  int64_t n_hubs;
  const void* h;
  const float* a_src;
  const float* a_dst;
  float slope;
  void* out;
  float* lse;
  float* part_acc;   // [hub chunks][H * D]
  float2* part_ml;   // [hub chunks][H]  (max in base 2, sum)
  int32_t* err;
  int col_off;       // bytes of shared memory before the per-warp states
};

// Running softmax state of the vectors a lane owns.
template <typename T, int NV>
struct Online {
  static constexpr int V = VecOf<T>::n;
  float m[NV], l[NV], acc[NV][V];

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      m[v] = -INFINITY;
      l[v] = 0.f;
#pragma unroll
      for (int c = 0; c < V; ++c) acc[v][c] = 0.f;
    }
  }

  // Fold the state (mb, lb, ab) of a disjoint edge set into vector slot v.
  __device__ __forceinline__ void merge(int v, float mb, float lb, const float (&ab)[V]) {
    const float M = fmaxf(m[v], mb);
    const float Mr = (M == -INFINITY) ? 0.f : M;
    const float sa = exp2f(m[v] - Mr), sb = exp2f(mb - Mr);
    l[v] = l[v] * sa + lb * sb;
#pragma unroll
    for (int c = 0; c < V; ++c) acc[v][c] = acc[v][c] * sa + ab[c] * sb;
    m[v] = M;
  }

  // Combine the G sub-groups of the warp (butterfly; every lane ends with the
  // state of all edges the warp saw).
  __device__ __forceinline__ void merge_subgroups(const Shape& s) {
    for (int o = s.lpr; o < 32; o <<= 1) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float mb = __shfl_xor_sync(kFull, m[v], o);
        const float lb = __shfl_xor_sync(kFull, l[v], o);
        float ab[V];
#pragma unroll
        for (int c = 0; c < V; ++c) ab[c] = __shfl_xor_sync(kFull, acc[v][c], o);
        merge(v, mb, lb, ab);
      }
    }
  }
};

// Stream the edges beg, beg + G, ... < end of this lane's sub-group through
// the online softmax.  cols[x - colbase] is the source of edge x.
template <typename T, int NV>
__device__ __forceinline__ void fwd_edges(const FwdArgs& A, const Lane<NV>& L,
                                          const int32_t* cols, int colbase, int beg, int end,
                                          const float (&as2)[NV][VecOf<T>::n],
                                          const float (&sd2)[NV], Online<T, NV>& st) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kUnroll;
  const int step = L.G * U;
  int jn[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int e = beg + u * L.G + L.g;
    jn[u] = e < end ? cols[e - colbase] : -1;
  }
  for (int base = beg; base < end; base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    if (base + step < end) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = base + step + u * L.G + L.g;
        jn[u] = e < end ? cols[e - colbase] : -1;
      }
    }
    uint4 raw[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v)
        raw[u][v] = (j[u] >= 0 && L.ok[v]) ? ld16(row_base<T>(A.h, j[u], A.s.rv) + 16 * L.q[v])
                                           : make_uint4(0, 0, 0, 0);
    float sc[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float x[V];
        unpack<T>(raw[u][v], x);
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < V; ++c) d = fmaf(x[c], as2[v][c], d);
        sc[u][v] = d;
      }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float z = sd2[v] + head_sum(sc[u][v], A.s.hv);
        const float e = z > 0.f ? z : A.slope * z;
        sc[u][v] = j[u] >= 0 ? e : -INFINITY;
      }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float bm = sc[0][v];
#pragma unroll
      for (int u = 1; u < U; ++u) bm = fmaxf(bm, sc[u][v]);
      const float mn = fmaxf(st.m[v], bm);
      const float mr = (mn == -INFINITY) ? 0.f : mn;
      const float s0 = exp2f(st.m[v] - mr);
      st.l[v] *= s0;
#pragma unroll
      for (int c = 0; c < V; ++c) st.acc[v][c] *= s0;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float pu = exp2f(sc[u][v] - mr);
        st.l[v] += pu;
        float x[V];
        unpack_alt<T>(raw[u][v], x);
#pragma unroll
        for (int c = 0; c < V; ++c) st.acc[v][c] = fmaf(pu, x[c], st.acc[v][c]);
      }
      st.m[v] = mn;
    }
  }
}

// out = acc / l, lse = (m + log2 l) ln 2; a node without edges gets 0 and -inf.
template <typename T, int NV>
__device__ __forceinline__ void write_node(const FwdArgs& A, const Lane<NV>& L, int64_t node,
                                           const Online<T, NV>& st) {
  constexpr int V = VecOf<T>::n;
  char* orow = reinterpret_cast<char*>(A.out) + node * int64_t(A.s.rv) * 16;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!L.ok[v]) continue;
    const float inv = st.l[v] > 0.f ? 1.f / st.l[v] : 0.f;
    float x[V];
#pragma unroll
    for (int c = 0; c < V; ++c) x[c] = st.acc[v][c] * inv;
    st16(orow + 16 * L.q[v], pack<T>(x));
    if (L.head_leader(A.s, v))
      A.lse[node * A.s.H + L.k[v]] =
          st.l[v] > 0.f ? (st.m[v] + log2f(st.l[v])) * kLn2 : -INFINITY;
  }
}

template <typename T, int NV>
__global__ void __launch_bounds__(kThreads, MinBlocks<NV>::value) fwd_main(const FwdArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<NV> L(A.s);
  const int wid = threadIdx.x >> 5;
  float as2[NV][V], ad2[NV][V];
  load_att<T, NV>(A.a_src, L, kLog2e, as2);
  load_att<T, NV>(A.a_dst, L, kLog2e, ad2);
  Online<T, NV> st;
  st.init();

  if (blockIdx.x >= A.n_items) {
    // ---- light node: one warp ------------------------------------------
    const int64_t t = (int64_t(blockIdx.x) - A.n_items) * kWarps + wid;
    if (t >= A.n_light) return;
    const int i = A.light[t];
    const int beg = A.ptr[i], end = A.ptr[i + 1];
    float sd2[NV];
    row_dot<T, NV>(A.h, i, A.s, L, ad2, sd2);
    fwd_edges<T, NV>(A, L, A.idx, 0, beg, end, as2, sd2, st);
    st.merge_subgroups(A.s);
    if (L.g == 0) write_node<T, NV>(A, L, i, st);
    return;
  }

  // ---- block item: a mid node, or one chunk of a hub ---------------------
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
  float* wm = reinterpret_cast<float*>(smem + A.col_off);
  float* wl = wm + kWarps * A.s.H;
  float* wacc = wl + kWarps * A.s.H;
  const int row_f = A.s.rv * V;  // floats per accumulator row

  const int4 it = A.items[blockIdx.x];
  const int i = it.x, beg = it.y, end = it.z, slot = it.w;
  if (!stage_edges(cols, A.idx, beg, end, bar, A.err)) return;
  float sd2[NV];
  row_dot<T, NV>(A.h, i, A.s, L, ad2, sd2);
  const int len = end - beg;
  const int per = (len + kWarps - 1) / kWarps;
  const int wb = min(end, beg + wid * per), we = min(end, wb + per);
  fwd_edges<T, NV>(A, L, cols, beg & ~3, wb, we, as2, sd2, st);
  st.merge_subgroups(A.s);
  if (L.g == 0) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      if (!L.ok[v]) continue;
#pragma unroll
      for (int c = 0; c < V; ++c) wacc[wid * row_f + L.q[v] * V + c] = st.acc[v][c];
      if (L.head_leader(A.s, v)) {
        wm[wid * A.s.H + L.k[v]] = st.m[v];
        wl[wid * A.s.H + L.k[v]] = st.l[v];
      }
    }
  }
  __syncthreads();
  if (wid != 0 || L.g != 0) return;
  // warp 0 folds the warps' states in warp order
  Online<T, NV> tot;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    tot.m[v] = L.ok[v] ? wm[L.k[v]] : -INFINITY;
    tot.l[v] = L.ok[v] ? wl[L.k[v]] : 0.f;
#pragma unroll
    for (int c = 0; c < V; ++c) tot.acc[v][c] = L.ok[v] ? wacc[L.q[v] * V + c] : 0.f;
  }
  for (int w = 1; w < kWarps; ++w) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      if (!L.ok[v]) continue;
      float ab[V];
#pragma unroll
      for (int c = 0; c < V; ++c) ab[c] = wacc[w * row_f + L.q[v] * V + c];
      tot.merge(v, wm[w * A.s.H + L.k[v]], wl[w * A.s.H + L.k[v]], ab);
    }
  }
  if (slot < 0) {
    write_node<T, NV>(A, L, i, tot);
    return;
  }
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!L.ok[v]) continue;
    float* pa = A.part_acc + int64_t(slot) * row_f + L.q[v] * V;
#pragma unroll
    for (int c4 = 0; c4 < V; c4 += 4)
      *reinterpret_cast<float4*>(pa + c4) =
          make_float4(tot.acc[v][c4], tot.acc[v][c4 + 1], tot.acc[v][c4 + 2], tot.acc[v][c4 + 3]);
    if (L.head_leader(A.s, v)) A.part_ml[int64_t(slot) * A.s.H + L.k[v]] = make_float2(tot.m[v], tot.l[v]);
  }
}

// One warp per hub: fold its chunk partials in chunk order.
template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) fwd_merge(const FwdArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<NV> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.n_hubs || L.g != 0) return;
  const int4 hb = A.hubs[t];
  const int row_f = A.s.rv * V;
  Online<T, NV> st;
  st.init();
  for (int c = 0; c < hb.z; ++c) {
    const int64_t slot = int64_t(hb.y) + c;
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      if (!L.ok[v]) continue;
      const float2 ml = A.part_ml[slot * A.s.H + L.k[v]];
      float ab[V];
      const float* pa = A.part_acc + slot * row_f + L.q[v] * V;
#pragma unroll
      for (int c4 = 0; c4 < V; c4 += 4) {
        const float4 q = *reinterpret_cast<const float4*>(pa + c4);
        ab[c4] = q.x;
        ab[c4 + 1] = q.y;
        ab[c4 + 2] = q.z;
        ab[c4 + 3] = q.w;
      }
      st.merge(v, ml.x, ml.y, ab);
    }
  }
  write_node<T, NV>(A, L, hb.x, st);
}

template <typename T, int NV>
cudaError_t launch_t(const FwdArgs& A0, cudaStream_t stream, const cudaEvent_t* ev) {
  FwdArgs A = A0;
  constexpr int V = VecOf<T>::n;
  const int64_t blocks = A.n_items + (A.n_light + kWarps - 1) / kWarps;
  if (ev) cudaEventRecord(ev[0], stream);
  if (blocks > 0) {
    const size_t smem = size_t(A.col_off) + size_t(kWarps) * (2 * A.s.H + A.s.rv * V) * 4;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(fwd_main<T, NV>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return e;
    }
    fwd_main<T, NV><<<unsigned(blocks), kThreads, smem, stream>>>(A);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[1], stream);
  if (A.n_hubs > 0) {
    fwd_merge<T, NV><<<unsigned((A.n_hubs + kWarps - 1) / kWarps), kThreads, 0, stream>>>(A);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[2], stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt, const void* h,
                           const float* a_src, const float* a_dst, float slope, void* out,
                           float* lse, char* ws, const WsLayout& L, cudaStream_t st,
                           const cudaEvent_t* ev) {
  FwdArgs A{};
  A.s = s;
  A.ptr = g->csr.ptr;
  A.idx = g->csr.idx;
  A.light = g->csr.light;
  A.n_light = g->csr.n_light;
  A.items = g->csr.items;
  A.n_items = g->csr.n_items;
  A.hubs = g->csr.hubs;
  A.n_hubs = g->csr.n_hubs;
  A.h = h;
  A.a_src = a_src;
  A.a_dst = a_dst;
  A.slope = slope;
  A.out = out;
  A.lse = lse;
  A.part_acc = reinterpret_cast<float*>(ws + L.fwd_acc);
  A.part_ml = reinterpret_cast<float2*>(ws + L.fwd_ml);
  A.err = g->err;
  A.col_off = int(16 + align_up(size_t(g->csr.max_item + 4) * 4, 16));
  if (dt == GNN_F32) {
    switch (s.nv) {
      case 1: return launch_t<float, 1>(A, st, ev);
      case 2: return launch_t<float, 2>(A, st, ev);
      case 4: return launch_t<float, 4>(A, st, ev);
    }
  } else {
    switch (s.nv) {
      case 1: return launch_t<__nv_bfloat16, 1>(A, st, ev);
      case 2: return launch_t<__nv_bfloat16, 2>(A, st, ev);
      case 4: return launch_t<__nv_bfloat16, 4>(A, st, ev);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace gnn
