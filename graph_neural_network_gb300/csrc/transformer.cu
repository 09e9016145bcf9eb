// Fused graph-transformer neighbour attention, forward and backward.
//
// Per destination i and head k, with the query, key and value projections
// q, key, val given by the caller:
//   e_ij = scale * q_i[k] . key_j[k],  alpha = softmax over in-neighbours,
//   out_i[k] = sum_j alpha_ij val_j[k],  lse_i[k] = log sum_j exp e_ij
// (Shi et al., "Masked Label Prediction", eqs. 3-4, on the neighbourhood; the
// Graph Transformer layer of "On Efficient Scaling of GNNs via IO-Aware
// Layers Implementations", Technical Summary > Methodology, attention-based
// layers: fused CSR kernel, one streaming pass with an online softmax, the
// log-sum-exp kept so that the backward pass recomputes alpha).  Each edge
// gathers two rows, key_j and val_j.
//
// Backward, with da_ij = dout_i . val_j, Delta_i = sum_j alpha_ij da_ij and
// de_ij = alpha_ij (da_ij - Delta_i):
//   pass 1, destination side (CSR): sums Delta, P = sum alpha da key_j and
//     Q = sum alpha key_j in one streaming pass, so dq_i = scale (P - Delta Q);
//     the per-node record {lse, Delta} goes to the workspace.
//   pass 2, source side (cached CSC): dkey_j = scale sum_i de_ij q_i and
//     dval_j = sum_i alpha_ij dout_i, gathering q_i, dout_i and i's record.
// No reduction crosses nodes, so work is pulled dynamically and results are
// still reproducible bit for bit.  Rows up to 512 bytes; degree-aware tiling
// and hub merges as in the other attention kernels.
#include "device.cuh"

namespace gnn {
namespace {

constexpr int kGrab = 4;
// Edges in flight per lane: two (not kUnroll = 4; each edge gathers two rows)
// fits every kernel here in 80 registers, three blocks per SM, which
// measured faster on GB300.
constexpr int kU = 2;

struct GtDir {
  const int32_t* ptr;
  const int32_t* idx;
  const int32_t* light;
  int64_t n_light;
  const int4* items;
  int64_t n_items;
  const int4* hubs;
  int64_t n_hubs;
  int col_off;
};

struct GtArgs {
  Shape s;
  GtDir csr, csc;
  const void* q;
  const void* key;
  const void* val;
  float scale;        // natural units
  float scale2;       // scale * log2(e)
  void* out;
  float* lse;
  float* f_acc;       // [CSR hub chunks][row_f]
  float2* f_ml;       // [CSR hub chunks][H]
  const float* lse_in;
  const void* dout;
  void* dq;
  void* dkey;
  void* dval;
  float2* stats;      // [N][H] {lse (base 2), Delta}
  float* d_delta;     // [CSR hub chunks][H]
  float* d_vec;       // [CSR hub chunks][2][row_f]  (P, Q)
  float* s_vec;       // [CSC hub chunks][2][row_f]  (dkey, dval)
  int* ctr;
  int32_t* err;
};

template <typename T>
__device__ __forceinline__ uint4 gather(const void* x, int node, const Shape& s,
                                        const Lane<1>& L) {
  return (node >= 0 && L.ok[0]) ? ld16(row_base<T>(x, node, s.rv) + 16 * L.q[0])
                                : make_uint4(0, 0, 0, 0);
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

template <typename T>
struct GtOnline {
  static constexpr int V = VecOf<T>::n;
  float m, l, acc[V];
  __device__ __forceinline__ void init() {
    m = -INFINITY;
    l = 0.f;
    zero<V>(acc);
  }
  __device__ __forceinline__ void merge(float mb, float lb, const float (&ab)[V]) {
    const float M = fmaxf(m, mb);
    const float Mr = (M == -INFINITY) ? 0.f : M;
    const float sa = ex2(m - Mr), sb = ex2(mb - Mr);
    l = l * sa + lb * sb;
    scale<V>(acc, sa);
    axpy<V>(acc, sb, ab);
    m = M;
  }
  __device__ __forceinline__ void merge_subgroups(const Shape& s) {
    for (int o = s.lpr; o < 32; o <<= 1) {
      const float mb = __shfl_xor_sync(kFull, m, o);
      const float lb = __shfl_xor_sync(kFull, l, o);
      float ab[V];
#pragma unroll
      for (int c = 0; c < V; ++c) ab[c] = __shfl_xor_sync(kFull, acc[c], o);
      merge(mb, lb, ab);
    }
  }
};

template <typename T, bool kFixed>
__device__ __forceinline__ void fwd_edges(const GtArgs& A, const Lane<1>& L, const int32_t* cols,
                                          int colbase, int beg, int end, int sg, int SG,
                                          int step, int trips, int (&jn)[kU],
                                          const float (&qs)[VecOf<T>::n], GtOnline<T>& st) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kU;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    uint4 rk[U], rv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      rk[u] = gather<T>(A.key, j[u], A.s, L);
      rv[u] = gather<T>(A.val, j[u], A.s, L);
    }
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
    float sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[V];
      unpack<T>(rk[u], x);
      sc[u] = dot<V>(x, qs);
    }
    head_sums<U>(sc, A.s.hv_log2);
    float bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      sc[u] = j[u] >= 0 ? sc[u] : -INFINITY;
      bm = fmaxf(bm, sc[u]);
    }
    const float mn = fmaxf(st.m, bm);
    const float mr = (mn == -INFINITY) ? 0.f : mn;
    const float s0 = ex2(st.m - mr);
    st.l *= s0;
    scale<V>(st.acc, s0);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float p = ex2(sc[u] - mr);
      st.l += p;
      float x[V];
      unpack<T>(rv[u], x);
      axpy<V>(st.acc, p, x);
    }
    st.m = mn;
  }
}

template <typename T>
__device__ __forceinline__ void fwd_write(const GtArgs& A, const Lane<1>& L, int64_t node,
                                          const GtOnline<T>& st) {
  constexpr int V = VecOf<T>::n;
  if (!L.ok[0]) return;
  const float inv = st.l > 0.f ? __frcp_rn(st.l) : 0.f;
  float x[V];
#pragma unroll
  for (int c = 0; c < V; ++c) x[c] = st.acc[c];
  scale<V>(x, inv);
  st16(reinterpret_cast<char*>(A.out) + node * int64_t(A.s.rv) * 16 + 16 * L.q[0], pack<T>(x));
  if (L.head_leader(A.s, 0))
    A.lse[node * A.s.H + L.k[0]] = st.l > 0.f ? (st.m + __log2f(st.l)) * kLn2 : -INFINITY;
}

// q_i scaled into base-2 score units.
template <typename T>
__device__ __forceinline__ void query(const GtArgs& A, const Lane<1>& L, int64_t i,
                                      float (&qs)[VecOf<T>::n]) {
  own_row<T>(A.q, i, A.s, L, qs);
  scale<VecOf<T>::n>(qs, A.scale2);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 3) gt_fwd_main(const GtArgs A) {
  constexpr int V = VecOf<T>::n;
  const GtDir& D = A.csr;
  const Lane<1> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  const int H = A.s.H;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  float qs[V];

  if (D.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    float* wm = reinterpret_cast<float*>(smem + D.col_off);
    float* wl = wm + kWarps * H;
    float* wacc = wl + kWarps * H;
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 0, 1);
      __syncthreads();
      const int it_i = s_item;
      if (it_i >= D.n_items) break;
      const int4 it = D.items[it_i];
      if (!stage_edges(cols, D.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kU * G edges dealt to the warps in turn
      const int wb = it.y + wid * kU * L.G, we = it.z;
      const int colbase = it.y & ~3;
      int jn[kU];
      batch_ids<kU>(cols, colbase, wb, we, L.g, L.G, jn);
      query<T>(A, L, it.x, qs);
      GtOnline<T> st;
      st.init();
      fwd_edges<T, false>(A, L, cols, colbase, wb, we, L.g, L.G, kWarps * kU * L.G, 0, jn, qs, st);
      st.merge_subgroups(A.s);
      if (L.g == 0 && L.ok[0]) {
#pragma unroll
        for (int c = 0; c < V; ++c) wacc[wid * row_f + L.q[0] * V + c] = st.acc[c];
        if (L.head_leader(A.s, 0)) {
          wm[wid * H + L.k[0]] = st.m;
          wl[wid * H + L.k[0]] = st.l;
        }
      }
      __syncthreads();
      if (wid == 0 && L.g == 0 && L.ok[0]) {
        GtOnline<T> tot;
        tot.m = wm[L.k[0]];
        tot.l = wl[L.k[0]];
#pragma unroll
        for (int c = 0; c < V; ++c) tot.acc[c] = wacc[L.q[0] * V + c];
        for (int w = 1; w < kWarps; ++w) {
          float ab[V];
#pragma unroll
          for (int c = 0; c < V; ++c) ab[c] = wacc[w * row_f + L.q[0] * V + c];
          tot.merge(wm[w * H + L.k[0]], wl[w * H + L.k[0]], ab);
        }
        if (it.w < 0) {
          fwd_write<T>(A, L, it.x, tot);
        } else {
          float* pa = A.f_acc + int64_t(it.w) * row_f + L.q[0] * V;
#pragma unroll
          for (int c4 = 0; c4 < V; c4 += 4)
            *reinterpret_cast<float4*>(pa + c4) =
                make_float4(tot.acc[c4], tot.acc[c4 + 1], tot.acc[c4 + 2], tot.acc[c4 + 3]);
          if (L.head_leader(A.s, 0)) A.f_ml[int64_t(it.w) * H + L.k[0]] = make_float2(tot.m, tot.l);
        }
      }
      __syncthreads();
    }
  }

  // ---- light nodes, rows of a whole warp: one warp each -----------------
  for (;;) {
    int t0 = 0;
    if (L.lane == 0) t0 = atomicAdd(A.ctr + 1, kGrab);
    t0 = __shfl_sync(kFull, t0, 0);
    if (t0 >= D.n_light) break;
    int my_i = -1, my_b = 0, my_e = 0;
    if (L.lane < kGrab && t0 + L.lane < D.n_light) {
      my_i = D.light[t0 + L.lane];
      my_b = D.ptr[my_i];
      my_e = D.ptr[my_i + 1];
    }
    int i = __shfl_sync(kFull, my_i, 0);
    int beg = __shfl_sync(kFull, my_b, 0), end = __shfl_sync(kFull, my_e, 0);
    int jn[kU];
    batch_ids<kU>(D.idx, 0, beg, end, L.g, L.G, jn);
    for (int qq = 0; qq < kGrab && i >= 0; ++qq) {
      const int nq = (qq + 1) & (kGrab - 1);
      const int i2 = qq + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[kU];
      batch_ids<kU>(D.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      query<T>(A, L, i, qs);
      GtOnline<T> st;
      st.init();
      fwd_edges<T, false>(A, L, D.idx, 0, beg, end, L.g, L.G, kU * L.G, 0, jn, qs, st);
      st.merge_subgroups(A.s);
      if (L.g == 0) fwd_write<T>(A, L, i, st);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < kU; ++u) jn[u] = jn2[u];
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) gt_fwd_merge(const GtArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<1> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.csr.n_hubs || L.g != 0 || !L.ok[0]) return;
  const int4 hb = A.csr.hubs[t];
  const int row_f = A.s.rv * V;
  GtOnline<T> st;
  st.init();
  for (int c = 0; c < hb.z; ++c) {
    const int64_t slot = int64_t(hb.y) + c;
    const float2 ml = A.f_ml[slot * A.s.H + L.k[0]];
    float ab[V];
    const float* pa = A.f_acc + slot * row_f + L.q[0] * V;
#pragma unroll
    for (int c4 = 0; c4 < V; c4 += 4) {
      const float4 p = *reinterpret_cast<const float4*>(pa + c4);
      ab[c4] = p.x;
      ab[c4 + 1] = p.y;
      ab[c4 + 2] = p.z;
      ab[c4 + 3] = p.w;
    }
    st.merge(ml.x, ml.y, ab);
  }
  fwd_write<T>(A, L, hb.x, st);
}

// ---------------------------------------------------------------------------
// backward pass 1: destination side
// ---------------------------------------------------------------------------

template <typename T>
struct GtDst {
  static constexpr int V = VecOf<T>::n;
  float delta, P[V], Q[V];
  __device__ __forceinline__ void init() {
    delta = 0.f;
    zero<V>(P);
    zero<V>(Q);
  }
  __device__ __forceinline__ void subgroup_total(const Shape& s) {
    delta = subgroup_sum(delta, s);
    subgroup_sums<V>(P, s);
    subgroup_sums<V>(Q, s);
  }
};

template <typename T, bool kFixed>
__device__ __forceinline__ void dst_edges(const GtArgs& A, const Lane<1>& L, const int32_t* cols,
                                          int colbase, int beg, int end, int sg, int SG,
                                          int step, int trips, int (&jn)[kU],
                                          const float (&qs)[VecOf<T>::n],
                                          const float (&gi)[VecOf<T>::n], float lse2,
                                          GtDst<T>& sm) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kU;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    uint4 rk[U], rv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      rk[u] = gather<T>(A.key, j[u], A.s, L);
      rv[u] = gather<T>(A.val, j[u], A.s, L);
    }
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
    float red[2 * U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[V], y[V];
      unpack<T>(rk[u], x);
      unpack<T>(rv[u], y);
      red[u] = dot<V>(x, qs);
      red[U + u] = dot<V>(y, gi);
    }
    head_sums<2 * U>(red, A.s.hv_log2);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float al = j[u] >= 0 ? ex2(red[u] - lse2) : 0.f;
      const float ad = al * red[U + u];
      sm.delta += ad;
      float x[V];
      unpack_alt<T>(rk[u], x);
      axpy<V>(sm.P, ad, x);
      axpy<V>(sm.Q, al, x);
    }
  }
}

template <typename T>
__device__ __forceinline__ void dst_finish(const GtArgs& A, const Lane<1>& L, int64_t i,
                                           const GtDst<T>& sm, float lse2) {
  constexpr int V = VecOf<T>::n;
  if (!L.ok[0]) return;
  float y[V];
#pragma unroll
  for (int c = 0; c < V; ++c) y[c] = A.scale * fmaf(-sm.delta, sm.Q[c], sm.P[c]);
  st16(reinterpret_cast<char*>(A.dq) + i * int64_t(A.s.rv) * 16 + 16 * L.q[0], pack<T>(y));
  if (L.head_leader(A.s, 0)) A.stats[i * A.s.H + L.k[0]] = make_float2(lse2, sm.delta);
}

// kSub: light nodes take one sub-group each (rows narrower than a warp).
template <typename T, bool kSub>
__global__ void __launch_bounds__(kThreads, 3) gt_dst_main(const GtArgs A) {
  constexpr int V = VecOf<T>::n;
  const GtDir& D = A.csr;
  const Lane<1> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  const int H = A.s.H;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  float qs[V], gi[V];

  if (D.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    float* wbuf = reinterpret_cast<float*>(smem + D.col_off);  // [kWarps][H + 2 row_f]
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 0, 1);
      __syncthreads();
      const int it_i = s_item;
      if (it_i >= D.n_items) break;
      const int4 it = D.items[it_i];
      if (!stage_edges(cols, D.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kU * G edges dealt to the warps in turn
      const int wb = it.y + wid * kU * L.G, we = it.z;
      const int colbase = it.y & ~3;
      int jn[kU];
      batch_ids<kU>(cols, colbase, wb, we, L.g, L.G, jn);
      query<T>(A, L, it.x, qs);
      own_row<T>(A.dout, it.x, A.s, L, gi);
      const float lse2 = L.ok[0] ? A.lse_in[int64_t(it.x) * H + L.k[0]] * kLog2e : 0.f;
      GtDst<T> sm;
      sm.init();
      dst_edges<T, false>(A, L, cols, colbase, wb, we, L.g, L.G, kWarps * kU * L.G, 0, jn, qs, gi, lse2, sm);
      sm.subgroup_total(A.s);
      float* mine = wbuf + wid * (H + 2 * row_f);
      if (L.g == 0 && L.ok[0]) {
        if (L.head_leader(A.s, 0)) mine[L.k[0]] = sm.delta;
#pragma unroll
        for (int c = 0; c < V; ++c) {
          mine[H + L.q[0] * V + c] = sm.P[c];
          mine[H + row_f + L.q[0] * V + c] = sm.Q[c];
        }
      }
      __syncthreads();
      if (wid == 0 && L.g == 0 && L.ok[0]) {
        GtDst<T> tot;
        tot.init();
        for (int w = 0; w < kWarps; ++w) {
          const float* o = wbuf + w * (H + 2 * row_f);
          tot.delta += o[L.k[0]];
#pragma unroll
          for (int c = 0; c < V; ++c) {
            tot.P[c] += o[H + L.q[0] * V + c];
            tot.Q[c] += o[H + row_f + L.q[0] * V + c];
          }
        }
        if (it.w < 0) {
          dst_finish<T>(A, L, it.x, tot, lse2);
        } else {
          if (L.head_leader(A.s, 0)) A.d_delta[int64_t(it.w) * H + L.k[0]] = tot.delta;
          float* pv = A.d_vec + int64_t(it.w) * 2 * row_f + L.q[0] * V;
#pragma unroll
          for (int c = 0; c < V; ++c) {
            pv[c] = tot.P[c];
            pv[row_f + c] = tot.Q[c];
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  if (kSub) {
    // nodes per sub-group per pull: four where a warp holds two sub-groups,
    // two otherwise
    const int R = L.G >= 32 ? 1 : (L.G == 2 ? 4 : 2);
    const int npull = R * L.G;
    for (;;) {
      int t0 = 0;
      if (L.lane == 0) t0 = atomicAdd(A.ctr + 1, npull);
      t0 = __shfl_sync(kFull, t0, 0);
      if (t0 >= D.n_light) break;
      int my_n = -1, my_b = 0, my_e = 0;
      if (L.lane < npull && t0 + L.lane < D.n_light) {
        my_n = D.light[t0 + L.lane];
        my_b = D.ptr[my_n];
        my_e = D.ptr[my_n + 1];
      }
      for (int r = 0; r < R; ++r) {
        const int src = r * L.G + L.g;
        const int i = __shfl_sync(kFull, my_n, src);
        const int beg = __shfl_sync(kFull, my_b, src);
        const int e0 = __shfl_sync(kFull, my_e, src);  // every lane shuffles
        const int end = i >= 0 ? e0 : beg;
        if (!__any_sync(kFull, i >= 0)) break;
        int trips = (end - beg + kU - 1) / kU;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) trips = max(trips, __shfl_xor_sync(kFull, trips, o));
        int jn[kU];
        batch_ids<kU>(D.idx, 0, beg, end, 0, 1, jn);
        const int ii = i >= 0 ? i : 0;
        query<T>(A, L, ii, qs);
        own_row<T>(A.dout, ii, A.s, L, gi);
        const float lse2 = L.ok[0] ? A.lse_in[int64_t(ii) * H + L.k[0]] * kLog2e : 0.f;
        GtDst<T> sm;
        sm.init();
        dst_edges<T, true>(A, L, D.idx, 0, beg, end, 0, 1, kU, trips, jn, qs, gi, lse2, sm);
        if (i >= 0) dst_finish<T>(A, L, i, sm, lse2);
      }
    }
    return;
  }

  // ---- light nodes, rows of a whole warp: one warp each -----------------
  for (;;) {
    int t0 = 0;
    if (L.lane == 0) t0 = atomicAdd(A.ctr + 1, kGrab);
    t0 = __shfl_sync(kFull, t0, 0);
    if (t0 >= D.n_light) break;
    int my_i = -1, my_b = 0, my_e = 0;
    if (L.lane < kGrab && t0 + L.lane < D.n_light) {
      my_i = D.light[t0 + L.lane];
      my_b = D.ptr[my_i];
      my_e = D.ptr[my_i + 1];
    }
    int i = __shfl_sync(kFull, my_i, 0);
    int beg = __shfl_sync(kFull, my_b, 0), end = __shfl_sync(kFull, my_e, 0);
    int jn[kU];
    batch_ids<kU>(D.idx, 0, beg, end, L.g, L.G, jn);
    for (int qq = 0; qq < kGrab && i >= 0; ++qq) {
      const int nq = (qq + 1) & (kGrab - 1);
      const int i2 = qq + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[kU];
      batch_ids<kU>(D.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      query<T>(A, L, i, qs);
      own_row<T>(A.dout, i, A.s, L, gi);
      const float lse2 = L.ok[0] ? A.lse_in[int64_t(i) * H + L.k[0]] * kLog2e : 0.f;
      GtDst<T> sm;
      sm.init();
      dst_edges<T, false>(A, L, D.idx, 0, beg, end, L.g, L.G, kU * L.G, 0, jn, qs, gi, lse2, sm);
      sm.subgroup_total(A.s);
      if (L.g == 0) dst_finish<T>(A, L, i, sm, lse2);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < kU; ++u) jn[u] = jn2[u];
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) gt_dst_merge(const GtArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<1> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.csr.n_hubs || L.g != 0 || !L.ok[0]) return;
  const int4 hb = A.csr.hubs[t];
  const int row_f = A.s.rv * V;
  const int H = A.s.H;
  GtDst<T> tot;
  tot.init();
  for (int c = 0; c < hb.z; ++c) {
    const int64_t slot = int64_t(hb.y) + c;
    tot.delta += A.d_delta[slot * H + L.k[0]];
    const float* pv = A.d_vec + slot * 2 * row_f + L.q[0] * V;
#pragma unroll
    for (int e = 0; e < V; ++e) {
      tot.P[e] += pv[e];
      tot.Q[e] += pv[row_f + e];
    }
  }
  dst_finish<T>(A, L, hb.x, tot, A.lse_in[int64_t(hb.x) * H + L.k[0]] * kLog2e);
}

// ---------------------------------------------------------------------------
// backward pass 2: source side
// ---------------------------------------------------------------------------

template <typename T, bool kFixed>
__device__ __forceinline__ void src_edges(const GtArgs& A, const Lane<1>& L, const int32_t* cols,
                                          int colbase, int beg, int end, int sg, int SG,
                                          int step, int trips, int (&in)[kU],
                                          const float (&ks)[VecOf<T>::n],
                                          const float (&vj)[VecOf<T>::n],
                                          float (&dk)[VecOf<T>::n], float (&dv)[VecOf<T>::n]) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kU;
  const int H = A.s.H;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int i[U];
#pragma unroll
    for (int u = 0; u < U; ++u) i[u] = in[u];
    uint4 rq[U], rg[U];
    float2 st[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      rq[u] = gather<T>(A.q, i[u], A.s, L);
      rg[u] = gather<T>(A.dout, i[u], A.s, L);
      st[u] = (i[u] >= 0 && L.ok[0]) ? __ldg(A.stats + int64_t(i[u]) * H + L.k[0])
                                     : make_float2(0.f, 0.f);
    }
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, in);
    float red[2 * U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[V], y[V];
      unpack<T>(rq[u], x);
      unpack<T>(rg[u], y);
      red[u] = dot<V>(x, ks);
      red[U + u] = dot<V>(y, vj);
    }
    head_sums<2 * U>(red, A.s.hv_log2);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float al = i[u] >= 0 ? ex2(red[u] - st[u].x) : 0.f;
      const float de = al * (red[U + u] - st[u].y) * A.scale;
      float x[V], y[V];
      unpack_alt<T>(rq[u], x);
      unpack_alt<T>(rg[u], y);
      axpy<V>(dk, de, x);
      axpy<V>(dv, al, y);
    }
  }
}

template <typename T>
__device__ __forceinline__ void src_write(const GtArgs& A, const Lane<1>& L, int64_t j,
                                          const float (&dk)[VecOf<T>::n],
                                          const float (&dv)[VecOf<T>::n]) {
  if (!L.ok[0]) return;
  const int64_t off = j * int64_t(A.s.rv) * 16 + 16 * L.q[0];
  st16(reinterpret_cast<char*>(A.dkey) + off, pack<T>(dk));
  st16(reinterpret_cast<char*>(A.dval) + off, pack<T>(dv));
}

// kSub: light nodes take one sub-group each (rows narrower than a warp).
template <typename T, bool kSub>
__global__ void __launch_bounds__(kThreads, 3) gt_src_main(const GtArgs A) {
  constexpr int V = VecOf<T>::n;
  const GtDir& D = A.csc;
  const Lane<1> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  float ks[V], vj[V], dk[V], dv[V];

  if (D.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    float* wbuf = reinterpret_cast<float*>(smem + D.col_off);  // [kWarps][2 row_f]
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 2, 1);
      __syncthreads();
      const int it_i = s_item;
      if (it_i >= D.n_items) break;
      const int4 it = D.items[it_i];
      if (!stage_edges(cols, D.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kU * G edges dealt to the warps in turn
      const int wb = it.y + wid * kU * L.G, we = it.z;
      const int colbase = it.y & ~3;
      int in[kU];
      batch_ids<kU>(cols, colbase, wb, we, L.g, L.G, in);
      own_row<T>(A.key, it.x, A.s, L, ks);
      scale<V>(ks, A.scale2);
      own_row<T>(A.val, it.x, A.s, L, vj);
      zero<V>(dk);
      zero<V>(dv);
      src_edges<T, false>(A, L, cols, colbase, wb, we, L.g, L.G, kWarps * kU * L.G, 0, in, ks, vj, dk, dv);
      subgroup_sums<V>(dk, A.s);
      subgroup_sums<V>(dv, A.s);
      if (L.g == 0 && L.ok[0])
#pragma unroll
        for (int c = 0; c < V; ++c) {
          wbuf[wid * 2 * row_f + L.q[0] * V + c] = dk[c];
          wbuf[wid * 2 * row_f + row_f + L.q[0] * V + c] = dv[c];
        }
      __syncthreads();
      if (wid == 0 && L.g == 0 && L.ok[0]) {
#pragma unroll
        for (int c = 0; c < V; ++c) {
          float a = 0.f, b = 0.f;
          for (int w = 0; w < kWarps; ++w) {
            a += wbuf[w * 2 * row_f + L.q[0] * V + c];
            b += wbuf[w * 2 * row_f + row_f + L.q[0] * V + c];
          }
          dk[c] = a;
          dv[c] = b;
        }
        if (it.w < 0) {
          src_write<T>(A, L, it.x, dk, dv);
        } else {
          float* pa = A.s_vec + int64_t(it.w) * 2 * row_f + L.q[0] * V;
#pragma unroll
          for (int c = 0; c < V; ++c) {
            pa[c] = dk[c];
            pa[row_f + c] = dv[c];
          }
        }
      }
      __syncthreads();
    }
  }

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  if (kSub) {
    // nodes per sub-group per pull: four where a warp holds two sub-groups,
    // two otherwise
    const int R = L.G >= 32 ? 1 : (L.G == 2 ? 4 : 2);
    const int npull = R * L.G;
    for (;;) {
      int t0 = 0;
      if (L.lane == 0) t0 = atomicAdd(A.ctr + 3, npull);
      t0 = __shfl_sync(kFull, t0, 0);
      if (t0 >= D.n_light) break;
      int my_n = -1, my_b = 0, my_e = 0;
      if (L.lane < npull && t0 + L.lane < D.n_light) {
        my_n = D.light[t0 + L.lane];
        my_b = D.ptr[my_n];
        my_e = D.ptr[my_n + 1];
      }
      for (int r = 0; r < R; ++r) {
        const int src = r * L.G + L.g;
        const int j = __shfl_sync(kFull, my_n, src);
        const int beg = __shfl_sync(kFull, my_b, src);
        const int e0 = __shfl_sync(kFull, my_e, src);  // every lane shuffles
        const int end = j >= 0 ? e0 : beg;
        if (!__any_sync(kFull, j >= 0)) break;
        int trips = (end - beg + kU - 1) / kU;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) trips = max(trips, __shfl_xor_sync(kFull, trips, o));
        int in[kU];
        batch_ids<kU>(D.idx, 0, beg, end, 0, 1, in);
        const int jj = j >= 0 ? j : 0;
        own_row<T>(A.key, jj, A.s, L, ks);
        scale<V>(ks, A.scale2);
        own_row<T>(A.val, jj, A.s, L, vj);
        zero<V>(dk);
        zero<V>(dv);
        src_edges<T, true>(A, L, D.idx, 0, beg, end, 0, 1, kU, trips, in, ks, vj, dk, dv);
        if (j >= 0) src_write<T>(A, L, j, dk, dv);
      }
    }
    return;
  }

  // ---- light nodes, rows of a whole warp: one warp each -----------------
  for (;;) {
    int t0 = 0;
    if (L.lane == 0) t0 = atomicAdd(A.ctr + 3, kGrab);
    t0 = __shfl_sync(kFull, t0, 0);
    if (t0 >= D.n_light) break;
    int my_j = -1, my_b = 0, my_e = 0;
    if (L.lane < kGrab && t0 + L.lane < D.n_light) {
      my_j = D.light[t0 + L.lane];
      my_b = D.ptr[my_j];
      my_e = D.ptr[my_j + 1];
    }
    int j = __shfl_sync(kFull, my_j, 0);
    int beg = __shfl_sync(kFull, my_b, 0), end = __shfl_sync(kFull, my_e, 0);
    int in[kU];
    batch_ids<kU>(D.idx, 0, beg, end, L.g, L.G, in);
    for (int qq = 0; qq < kGrab && j >= 0; ++qq) {
      const int nq = (qq + 1) & (kGrab - 1);
      const int j2 = qq + 1 < kGrab ? __shfl_sync(kFull, my_j, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int in2[kU];
      batch_ids<kU>(D.idx, 0, b2, j2 >= 0 ? e2 : b2, L.g, L.G, in2);
      own_row<T>(A.key, j, A.s, L, ks);
      scale<V>(ks, A.scale2);
      own_row<T>(A.val, j, A.s, L, vj);
      zero<V>(dk);
      zero<V>(dv);
      src_edges<T, false>(A, L, D.idx, 0, beg, end, L.g, L.G, kU * L.G, 0, in, ks, vj, dk, dv);
      subgroup_sums<V>(dk, A.s);
      subgroup_sums<V>(dv, A.s);
      if (L.g == 0) src_write<T>(A, L, j, dk, dv);
      j = j2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < kU; ++u) in[u] = in2[u];
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) gt_src_merge(const GtArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<1> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.csc.n_hubs || L.g != 0 || !L.ok[0]) return;
  const int4 hb = A.csc.hubs[t];
  const int row_f = A.s.rv * V;
  float dk[V], dv[V], ck[V], cv[V];
  zero<V>(dk);
  zero<V>(dv);
  zero<V>(ck);
  zero<V>(cv);
  for (int c = 0; c < hb.z; ++c) {
    const float* pa = A.s_vec + (int64_t(hb.y) + c) * 2 * row_f + L.q[0] * V;
#pragma unroll
    for (int e = 0; e < V; ++e) {
      kahan_add(dk[e], ck[e], pa[e]);
      kahan_add(dv[e], cv[e], pa[row_f + e]);
    }
  }
  src_write<T>(A, L, hb.x, dk, dv);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

template <typename T, typename K>
cudaError_t persistent_launch(K kernel, const GtArgs& A, const GtDir& D, size_t smem,
                              int sm_count, cudaStream_t st) {
  if (D.n_items + D.n_light == 0) return cudaSuccess;
  cudaError_t e;
  if ((e = set_smem(kernel, smem)) != cudaSuccess) return e;
  const int64_t work = D.n_items + (D.n_light + kWarps * kGrab - 1) / (kWarps * kGrab);
  const int64_t cap = persistent_blocks(kernel, smem, sm_count);
  kernel<<<unsigned(work < cap ? work : cap), kThreads, smem, st>>>(A);
  return cudaGetLastError();
}

template <typename T>
cudaError_t fwd_t(const GtArgs& A, int sm_count, cudaStream_t st) {
  constexpr int V = VecOf<T>::n;
  const int row_f = A.s.rv * V;
  cudaError_t e;
  if ((e = cudaMemsetAsync(A.ctr, 0, kCounters * sizeof(int), st)) != cudaSuccess) return e;
  const size_t smem = size_t(A.csr.col_off) + size_t(kWarps) * (2 * A.s.H + row_f) * 4;
  if ((e = persistent_launch<T>(gt_fwd_main<T>, A, A.csr, smem, sm_count, st)) != cudaSuccess)
    return e;
  if (A.csr.n_hubs > 0) {
    gt_fwd_merge<T><<<unsigned((A.csr.n_hubs + kWarps - 1) / kWarps), kThreads, 0, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T>
cudaError_t bwd_t(const GtArgs& A, int sm_count, cudaStream_t st) {
  constexpr int V = VecOf<T>::n;
  const int row_f = A.s.rv * V;
  cudaError_t e;
  if ((e = cudaMemsetAsync(A.ctr, 0, kCounters * sizeof(int), st)) != cudaSuccess) return e;
  const size_t smem1 = size_t(A.csr.col_off) + size_t(kWarps) * (A.s.H + 2 * row_f) * 4;
  if ((e = persistent_launch<T>(A.s.lpr < 32 ? gt_dst_main<T, true> : gt_dst_main<T, false>, A, A.csr,
                                    smem1, sm_count, st)) != cudaSuccess)
    return e;
  if (A.csr.n_hubs > 0) {
    gt_dst_merge<T><<<unsigned((A.csr.n_hubs + kWarps - 1) / kWarps), kThreads, 0, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t smem2 = size_t(A.csc.col_off) + size_t(kWarps) * 2 * row_f * 4;
  if ((e = persistent_launch<T>(A.s.lpr < 32 ? gt_src_main<T, true> : gt_src_main<T, false>, A, A.csc,
                                    smem2, sm_count, st)) != cudaSuccess)
    return e;
  if (A.csc.n_hubs > 0) {
    gt_src_merge<T><<<unsigned((A.csc.n_hubs + kWarps - 1) / kWarps), kThreads, 0, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

GtDir gt_dir(const Dir& d) {
  GtDir a{};
  a.ptr = d.ptr;
  a.idx = d.idx;
  a.light = d.light;
  a.n_light = d.n_light;
  a.items = d.items;
  a.n_items = d.n_items;
  a.hubs = d.hubs;
  a.n_hubs = d.n_hubs;
  a.col_off = int(16 + align_up(size_t(d.max_item + 4) * 4, 16));
  return a;
}

struct GtLayout {
  size_t ctr, f_acc, f_ml, stats, d_delta, d_vec, s_vec, total;
};

GtLayout gt_layout(const gnn_graph* g, const Shape& s) {
  const size_t row_f = size_t(s.rv) * 16 / s.esize;
  const size_t cc = size_t(g->csr.n_hub_chunks), sc = size_t(g->csc.n_hub_chunks);
  GtLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t r = off;
    off += align_up(bytes > 0 ? bytes : 1, 256);
    return r;
  };
  L.ctr = take(kCounters * 4);
  L.f_acc = take(cc * row_f * 4);
  L.f_ml = take(cc * s.H * 8);
  L.stats = take(size_t(g->n) * s.H * 8);
  L.d_delta = take(cc * s.H * 4);
  L.d_vec = take(cc * 2 * row_f * 4);
  L.s_vec = take(sc * 2 * row_f * 4);
  L.total = off;
  return L;
}

GtArgs gt_args(const gnn_graph* g, const Shape& s, const void* q, const void* key,
               const void* val, float scale, char* ws) {
  const GtLayout W = gt_layout(g, s);
  GtArgs A{};
  A.s = s;
  A.csr = gt_dir(g->csr);
  A.csc = gt_dir(g->csc);
  A.q = q;
  A.key = key;
  A.val = val;
  A.scale = scale;
  A.scale2 = scale * kLog2e;
  A.ctr = reinterpret_cast<int*>(ws + W.ctr);
  A.f_acc = reinterpret_cast<float*>(ws + W.f_acc);
  A.f_ml = reinterpret_cast<float2*>(ws + W.f_ml);
  A.stats = reinterpret_cast<float2*>(ws + W.stats);
  A.d_delta = reinterpret_cast<float*>(ws + W.d_delta);
  A.d_vec = reinterpret_cast<float*>(ws + W.d_vec);
  A.s_vec = reinterpret_cast<float*>(ws + W.s_vec);
  A.err = g->err;
  return A;
}

}  // namespace

size_t transformer_ws_bytes(const gnn_graph* g, const Shape& s) { return gt_layout(g, s).total; }

cudaError_t launch_transformer_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                       const void* q, const void* key, const void* val,
                                       float scale, void* out, float* lse, char* ws,
                                       cudaStream_t st) {
  GtArgs A = gt_args(g, s, q, key, val, scale, ws);
  A.out = out;
  A.lse = lse;
  return dt == GNN_F32 ? fwd_t<float>(A, g->sm_count, st)
                       : fwd_t<__nv_bfloat16>(A, g->sm_count, st);
}

cudaError_t launch_transformer_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                        const void* q, const void* key, const void* val,
                                        float scale, const float* lse, const void* dout,
                                        void* dq, void* dkey, void* dval, char* ws,
                                        cudaStream_t st) {
  GtArgs A = gt_args(g, s, q, key, val, scale, ws);
  A.lse_in = lse;
  A.dout = dout;
  A.dq = dq;
  A.dkey = dkey;
  A.dval = dval;
  return dt == GNN_F32 ? bwd_t<float>(A, g->sm_count, st)
                       : bwd_t<__nv_bfloat16>(A, g->sm_count, st);
}

}  // namespace gnn
