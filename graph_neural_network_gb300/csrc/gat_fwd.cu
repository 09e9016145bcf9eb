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
// commutes with LeakyReLU), so every exponential is one ex2; lse is stored
// in natural log.  Both score halves of every node come from a streaming
// pre-pass (scores.cu), so the edge loop gathers one float per edge and head
// next to the row it aggregates.
//
// Degree-aware tiling: mid-degree nodes get one thread block whose warps split
// the edge list (staged in shared memory by a bulk copy) and merge their
// states in warp order; hubs are split into edge chunks, one block each, whose
// partial states a second kernel folds in chunk order; light nodes get one
// warp each.  Blocks are persistent: each first pulls block items (hub chunks
// first, then mid nodes) from a work counter, then its warps pull light
// nodes in groups.  Which block or warp handles a node never changes the
// arithmetic applied to it, and every merge has a fixed order, so results
// are reproducible bit for bit.
#include "device.cuh"

namespace gnn {
namespace {

constexpr int kGrab = 4;  // light nodes a warp takes per counter access
// How far (base 2) a score may exceed the running state's reference value
// before the state is rescaled to it.
constexpr float kSlack = 16.f;

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
  const float* ssrc;  // [N][H] base-2 a_src . h_n
  const float* sdst;  // [N][H] base-2 a_dst . h_n
  float slope;
  void* out;
  float* lse;
  float* part_acc;   // [hub chunks][H * D]
  float2* part_ml;   // [hub chunks][H]  (max in base 2, sum)
  int* ctr;          // [0] block items taken, [1] light nodes taken
  int32_t* err;
  int col_off;       // bytes of shared memory before the per-warp states
};

// Running softmax state of the vectors a lane owns (VB-byte lane vectors).
template <typename T, int NV, int VB = 16>
struct Online {
  static constexpr int V = ElemsOf<T, VB>::n;
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
    const float sa = ex2(m[v] - Mr), sb = ex2(mb - Mr);
    l[v] = l[v] * sa + lb * sb;
    scale<V>(acc[v], sa);
    axpy<V>(acc[v], sb, ab);
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

// Stream edges through the online softmax, kUnroll edges per lane and batch:
// the batch at `base` holds edges base + sg + u * SG (u < kUnroll), and the
// next batch starts `step` edges further (SG * kUnroll when one warp takes
// every batch, more when the batches are dealt out to several warps).  Runs
// until end (kFixed false; every lane of the warp then has the same beg and
// end), or for exactly `trips` batches (kFixed true; the same count on every
// lane, batches past end change nothing).
// cols[x - colbase] is the source of edge x; jn holds the sources of the
// first batch (already loaded).
template <typename T, int NV, int VB, bool kFixed>
__device__ __forceinline__ void fwd_edges(const FwdArgs& A, const Lane<NV>& L,
                                          const int32_t* cols, int colbase, int beg, int end,
                                          int sg, int SG, int step, int trips,
                                          int (&jn)[UnrollOf<VB>::value], const float (&sd2)[NV],
                                          Online<T, NV, VB>& st) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = UnrollOf<VB>::value;
  const int H = A.s.H;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    RawV<VB> raw[U][NV];
    float sc[U * NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const bool ok = j[u] >= 0 && L.ok[v];
        raw[u][v] = ok ? ldv<VB>(row_at<VB>(A.h, j[u], A.s.rv) + VB * L.q[v]) : zero_raw<VB>();
        sc[u * NV + v] = ok ? __ldg(A.ssrc + int64_t(j[u]) * H + L.k[v]) : 0.f;
      }
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float z = sd2[v] + sc[u * NV + v];
        const float e = z > 0.f ? z : A.slope * z;
        sc[u * NV + v] = j[u] >= 0 ? e : -INFINITY;
      }
    // The reference value m of the running state is raised only when a score
    // exceeds it by more than kSlack (base 2), which after a node's first
    // batch is rare: most batches skip rescaling the accumulator.  Weights
    // stay below 2^kSlack, and out = acc / l, lse = m + log2 l hold for any
    // reference value.  The vote keeps the branch uniform over the warp.
    bool raise = false;
    float bmx[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      float bm = sc[v];
#pragma unroll
      for (int u = 1; u < U; ++u) bm = fmaxf(bm, sc[u * NV + v]);
      bmx[v] = bm;
      raise |= bm > st.m[v] + kSlack;
    }
    if (__any_sync(kFull, raise)) {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        if (!(bmx[v] > st.m[v] + kSlack)) continue;
        const float s0 = ex2(st.m[v] - bmx[v]);
        st.l[v] *= s0;
        scale<V>(st.acc[v], s0);
        st.m[v] = bmx[v];
      }
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const float mr = (st.m[v] == -INFINITY) ? 0.f : st.m[v];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float pu = ex2(sc[u * NV + v] - mr);
        st.l[v] += pu;
        float x[V];
        unpackv<T, VB>(raw[u][v], x);
        axpy<V>(st.acc[v], pu, x);
      }
    }
  }
}

// The edges of one node from beg on, spread over the warp's sub-groups
// (every lane sees the same beg and end), batches `step` edges apart.
template <typename T, int NV, int VB>
__device__ __forceinline__ void fwd_edges(const FwdArgs& A, const Lane<NV>& L,
                                          const int32_t* cols, int colbase, int beg, int end,
                                          int step, int (&jn)[UnrollOf<VB>::value],
                                          const float (&sd2)[NV], Online<T, NV, VB>& st) {
  fwd_edges<T, NV, VB, false>(A, L, cols, colbase, beg, end, L.g, L.G, step, 0, jn, sd2, st);
}

// This lane's base-2 destination score halves of node i.
template <int NV>
__device__ __forceinline__ void node_sdst(const FwdArgs& A, const Lane<NV>& L, int64_t i,
                                          float (&sd2)[NV]) {
#pragma unroll
  for (int v = 0; v < NV; ++v) sd2[v] = L.ok[v] ? __ldg(A.sdst + i * A.s.H + L.k[v]) : 0.f;
}

// out = acc / l, lse = (m + log2 l) ln 2; a node without edges gets 0 and -inf.
template <typename T, int NV, int VB>
__device__ __forceinline__ void write_node(const FwdArgs& A, const Lane<NV>& L, int64_t node,
                                           const Online<T, NV, VB>& st) {
  constexpr int V = ElemsOf<T, VB>::n;
  char* orow = reinterpret_cast<char*>(A.out) + node * int64_t(A.s.rv) * VB;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!L.ok[v]) continue;
    const float inv = st.l[v] > 0.f ? __frcp_rn(st.l[v]) : 0.f;
    float x[V];
#pragma unroll
    for (int c = 0; c < V; ++c) x[c] = st.acc[v][c];
    scale<V>(x, inv);
    storev<T, VB>(orow + VB * L.q[v], x);
    if (L.head_leader(A.s, v))
      A.lse[node * A.s.H + L.k[v]] =
          st.l[v] > 0.f ? (st.m[v] + __log2f(st.l[v])) * kLn2 : -INFINITY;
  }
}

// One block item: a whole mid node (slot < 0) or one chunk of a hub.
template <typename T, int NV, int VB>
__device__ __forceinline__ bool fwd_item(const FwdArgs& A, const Lane<NV>& L, int wid,
                                         const int4 it, unsigned char* smem, uint32_t& parity) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = UnrollOf<VB>::value;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
  float* wm = reinterpret_cast<float*>(smem + A.col_off);
  float* wl = wm + kWarps * A.s.H;
  float* wacc = wl + kWarps * A.s.H;
  const int row_f = A.s.rv * V;
  const int i = it.x, beg = it.y, end = it.z, slot = it.w;
  if (!stage_edges(cols, A.idx, beg, end, bar, parity, A.err)) return false;
  // batches of kUnroll * G edges are dealt to the warps in turn: warp w
  // takes batches w, w + kWarps, ... (at most one batch of padding per item)
  const int batch = U * L.G;
  const int wb = beg + wid * batch;
  const int colbase = beg & ~3;
  int jn[U];
  batch_ids<U>(cols, colbase, wb, end, L.g, L.G, jn);
  float sd2[NV];
  node_sdst<NV>(A, L, i, sd2);
  Online<T, NV, VB> st;
  st.init();
  fwd_edges<T, NV, VB>(A, L, cols, colbase, wb, end, kWarps * batch, jn, sd2, st);
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
  if (wid == 0 && L.g == 0) {
    // warp 0 folds the warps' states in warp order
    Online<T, NV, VB> tot;
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
      write_node<T, NV, VB>(A, L, i, tot);
    } else {
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        if (!L.ok[v]) continue;
        float* pa = A.part_acc + int64_t(slot) * row_f + L.q[v] * V;
#pragma unroll
        for (int c4 = 0; c4 < V; c4 += 4)
          *reinterpret_cast<float4*>(pa + c4) = make_float4(tot.acc[v][c4], tot.acc[v][c4 + 1],
                                                            tot.acc[v][c4 + 2], tot.acc[v][c4 + 3]);
        if (L.head_leader(A.s, v))
          A.part_ml[int64_t(slot) * A.s.H + L.k[v]] = make_float2(tot.m[v], tot.l[v]);
      }
    }
  }
  __syncthreads();  // shared memory is reused by the next item
  return true;
}

// kSub: light nodes take one sub-group each (rows narrower than a warp);
// otherwise one warp each.  Two instantiations keep each loop's register
// allocation its own.
template <typename T, int NV, int VB, bool kSub>
__global__ void __launch_bounds__(kThreads, MinBlocksLean<NV>::value) fwd_main(const FwdArgs A) {
  constexpr int U = UnrollOf<VB>::value;
  const Lane<NV> L(A.s);
  const int wid = threadIdx.x >> 5;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;

  // ---- block items: mid nodes and hub chunks -----------------------------
  if (A.n_items > 0) {
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(reinterpret_cast<uint64_t*>(smem), 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 0, 1);
      __syncthreads();
      const int it = s_item;
      if (it >= A.n_items) break;
      if (!fwd_item<T, NV, VB>(A, L, wid, A.items[it], smem, parity)) return;
    }
  }

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  // (a node's edges stay in one sub-group, so no cross-sub-group merge; the
  // sub-groups of a warp run as many batches as the longest of their nodes)
  if (kSub) {
    // nodes per sub-group per pull: four where a warp holds two sub-groups
    // (eight nodes per pull; measured 1 % faster than two on 512-byte rows),
    // two otherwise
    const int R = L.G >= 32 ? 1 : (L.G == 2 ? 4 : 2);
    const int npull = R * L.G;        // <= 32
    for (;;) {
      int t0 = 0;
      if (L.lane == 0) t0 = atomicAdd(A.ctr + 1, npull);
      t0 = __shfl_sync(kFull, t0, 0);
      if (t0 >= A.n_light) break;
      int my_i = -1, my_b = 0, my_e = 0;
      if (L.lane < npull && t0 + L.lane < A.n_light) {
        my_i = A.light[t0 + L.lane];
        my_b = A.ptr[my_i];
        my_e = A.ptr[my_i + 1];
      }
      for (int r = 0; r < R; ++r) {
        const int src = r * L.G + L.g;
        const int i = __shfl_sync(kFull, my_i, src);
        const int beg = __shfl_sync(kFull, my_b, src);
        const int e0 = __shfl_sync(kFull, my_e, src);  // every lane shuffles
        const int end = i >= 0 ? e0 : beg;
        if (!__any_sync(kFull, i >= 0)) break;
        int trips = (end - beg + U - 1) / U;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) trips = max(trips, __shfl_xor_sync(kFull, trips, o));
        int jn[U];
        batch_ids<U>(A.idx, 0, beg, end, 0, 1, jn);
        float sd2[NV];
        node_sdst<NV>(A, L, i >= 0 ? i : 0, sd2);
        Online<T, NV, VB> st;
        st.init();
        fwd_edges<T, NV, VB, true>(A, L, A.idx, 0, beg, end, 0, 1, U, trips, jn, sd2, st);
        if (i >= 0) write_node<T, NV, VB>(A, L, i, st);
      }
    }
    return;
  }

  // ---- light nodes, rows of a whole warp: one warp each, kGrab per pull ---
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
      // the next node's range and first sources, loaded while this one runs
      const int nq = (q + 1) & (kGrab - 1);
      const int i2 = q + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[U];
      batch_ids<U>(A.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      float sd2[NV];
      node_sdst<NV>(A, L, i, sd2);
      Online<T, NV, VB> st;
      st.init();
      fwd_edges<T, NV, VB>(A, L, A.idx, 0, beg, end, U * L.G, jn, sd2, st);
      st.merge_subgroups(A.s);
      if (L.g == 0) write_node<T, NV, VB>(A, L, i, st);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < U; ++u) jn[u] = jn2[u];
    }
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
  Online<T, NV, 16> st;
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
  write_node<T, NV, 16>(A, L, hb.x, st);
}

template <typename T>
cudaError_t launch_merge(const FwdArgs& M, cudaStream_t stream) {
  const unsigned grid = unsigned((M.n_hubs + kWarps - 1) / kWarps);
  switch (M.s.nv) {
    case 1: fwd_merge<T, 1><<<grid, kThreads, 0, stream>>>(M); break;
    case 2: fwd_merge<T, 2><<<grid, kThreads, 0, stream>>>(M); break;
    default: fwd_merge<T, 4><<<grid, kThreads, 0, stream>>>(M); break;
  }
  return cudaGetLastError();
}

// A.s is the lane geometry of the main kernel (VB-byte lane vectors); s16
// the one of 16-byte vectors, used by the score pre-pass and the hub merge.
template <typename T, int NV, int VB>
cudaError_t launch_t(const FwdArgs& A, const Shape& s16, gnn_dtype dt, const float* a_src,
                     const float* a_dst, int64_t n, int sm_count, cudaStream_t stream,
                     const cudaEvent_t* ev) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(A.ctr, 0, kCounters * sizeof(int), stream)) != cudaSuccess) return e;
  if (ev) cudaEventRecord(ev[0], stream);
  if ((e = launch_node_scores(s16, dt, A.h, a_src, a_dst, n, const_cast<float*>(A.ssrc),
                              const_cast<float*>(A.sdst), sm_count, stream)) != cudaSuccess)
    return e;
  if (ev) cudaEventRecord(ev[1], stream);
  if (A.n_items + A.n_light > 0) {
    const size_t smem = size_t(A.col_off) + size_t(kWarps) * (2 * A.s.H + A.s.H * A.s.D) * 4;
    // rows that do not fill the warp give each light node a sub-group (NV = 1)
    auto kernel = (NV == 1 && A.s.lpr < 32) ? fwd_main<T, NV, VB, NV == 1>
                                             : fwd_main<T, NV, VB, false>;
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem))) != cudaSuccess)
      return e;
    const int64_t work = A.n_items + (A.n_light + kWarps * kGrab - 1) / (kWarps * kGrab);
    const int64_t cap = persistent_blocks(kernel, smem, sm_count);
    const int64_t blocks = work < cap ? work : cap;
    kernel<<<unsigned(blocks), kThreads, smem, stream>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[2], stream);
  if (A.n_hubs > 0) {
    FwdArgs M = A;
    M.s = s16;
    if ((e = launch_merge<T>(M, stream)) != cudaSuccess) return e;
  }
  if (ev) cudaEventRecord(ev[3], stream);
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
  A.ssrc = reinterpret_cast<const float*>(ws + L.fwd_scores);
  A.sdst = A.ssrc + g->n * s.H;
  A.slope = slope;
  A.out = out;
  A.lse = lse;
  A.part_acc = reinterpret_cast<float*>(ws + L.fwd_acc);
  A.part_ml = reinterpret_cast<float2*>(ws + L.fwd_ml);
  A.ctr = reinterpret_cast<int*>(ws + L.fwd_ctr);
  A.err = g->err;
  A.col_off = int(16 + align_up(size_t(g->csr.max_item + 4) * 4, 16));
  // 32-byte lane vectors where a head spans 32 bytes or more, the row fits
  // one warp and the feature rows start on 32-byte boundaries
  Shape w;
  if (make_wide_shape(s, &w) && aligned32(h)) {
    A.s = w;
    if (dt == GNN_F32)
      return launch_t<float, 1, 32>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
    return launch_t<__nv_bfloat16, 1, 32>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
  }
  if (dt == GNN_F32) {
    switch (s.nv) {
      case 1: return launch_t<float, 1, 16>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
      case 2: return launch_t<float, 2, 16>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
      case 4: return launch_t<float, 4, 16>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
    }
  } else {
    switch (s.nv) {
      case 1:
        return launch_t<__nv_bfloat16, 1, 16>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
      case 2:
        return launch_t<__nv_bfloat16, 2, 16>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
      case 4:
        return launch_t<__nv_bfloat16, 4, 16>(A, s, dt, a_src, a_dst, g->n, g->sm_count, st, ev);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace gnn
