// Fused GATv2 neighbour aggregation, forward and backward.
//
// Per destination i and head k, with xl = W_l h (source side, also the
// aggregated value) and xr = W_r h (destination side) given by the caller:
//   e_ij = att[k] . LeakyReLU(xr_i[k] + xl_j[k]),  alpha = softmax_j e_ij,
//   out_i[k] = sum_j alpha_ij xl_j[k],  lse_i[k] = log sum_j exp e_ij
// (Brody et al., "How Attentive are Graph Attention Networks?", eq. 7; the
// GATv2 layer of "On Efficient Scaling of GNNs via IO-Aware Layers
// Implementations", Technical Summary > Methodology, attention-based layers:
// fused CSR kernel, one streaming pass, online softmax, log-sum-exp kept for
// the backward pass).  Unlike the GAT score, this one does not split into
// per-node halves: every edge evaluates LeakyReLU on a D-vector, so the
// score is computed from the gathered row inside the edge loop.
//
// Backward, with da_ij = dout_i . xl_j, Delta_i = sum_j alpha_ij da_ij,
// de_ij = alpha_ij (da_ij - Delta_i), g = LeakyReLU'(z) and l = LeakyReLU(z):
//   pass 1, destination side (CSR), one streaming pass per node that sums
//     Delta, P = sum alpha da g and Q = sum alpha g (D-vectors), so that
//     u_i = sum_j de_ij g_ij = P - Delta Q and dxr_i = att u_i; the per-node
//     record {lse, Delta} goes to the workspace.
//   pass 2, source side (cached CSC): w_j = sum_i de_ij g_ij and
//     dxl_j = sum_i alpha_ij dout_i + att w_j, gathering xr_i, dout_i and
//     i's record per edge.
// datt = sum over edges of de l.  Since l_ij = g_ij (xr_i + xl_j), it splits
// into per-node terms, datt = sum_i xr_i u_i + sum_j xl_j w_j, so each pass
// adds one product per node instead of one per edge.  Both passes assign
// work to blocks and warps statically, each block folds its warps' sums in a
// fixed order, and a last kernel adds the block sums in a fixed order in
// float64: datt is deterministic.
//
// Rows up to 512 bytes (one 16-byte vector per lane).  Degree-aware tiling
// and hub merges as in the GAT kernels.
#include "device.cuh"

namespace gnn {
namespace {

constexpr int kGrab = 4;
// Edges in flight per lane in the backward passes: two (not kUnroll = 4)
// lets them run three blocks per SM, which measured faster on GB300.
constexpr int kUB = 2;

struct V2Dir {
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

struct V2Args {
  Shape s;
  V2Dir csr, csc;
  int64_t n;
  const void* xl;
  const void* xr;
  const float* att;
  float slope;
  // forward
  void* out;
  float* lse;
  float* f_acc;      // [CSR hub chunks][row_f]
  float2* f_ml;      // [CSR hub chunks][H] (max in base 2, sum)
  // backward
  const float* lse_in;
  const void* dout;
  void* dxl;
  void* dxr;
  float* datt;
  float2* stats;     // [N][H] {lse (base 2), Delta}
  float* d_delta;    // [CSR hub chunks][H]
  float* d_vec;      // [CSR hub chunks][2][row_f]  (P, Q)
  float* s_acc;      // [CSC hub chunks][row_f]
  double* da_part;   // [da rows][row_f]
  int da_main_rows;  // rows of da_part written by pass 1 (one per block)
  int da_src_row0;   // first da_part row of pass 2 (one per block)
  int* ctr;
  int32_t* err;
};

__device__ __forceinline__ float leaky_g(float z, float s) { return z > 0.f ? 1.f : s; }

// For z = r + x elementwise: g = LeakyReLU'(z) and lz = LeakyReLU(z) = g z,
// with the additions and products done two lanes of data at a time.
template <int V>
__device__ __forceinline__ void leaky_terms(const float (&r)[V], const float (&x)[V],
                                            float slope, float (&g)[V], float (&lz)[V]) {
#pragma unroll
  for (int c = 0; c < V; c += 2) {
    float z0, z1;
    add2(z0, z1, r[c], r[c + 1], x[c], x[c + 1]);
    g[c] = leaky_g(z0, slope);
    g[c + 1] = leaky_g(z1, slope);
    mul2v(lz[c], lz[c + 1], z0, z1, g[c], g[c + 1]);
  }
}

// The score att . LeakyReLU(r + x) (att given as w) for the forward, with
// LeakyReLU(z) = c1 z + c2 |z|, c1 = (1 + s) / 2, c2 = (1 - s) / 2: the sums
// of w z and of w |z| take multiply-adds only (|z| is an operand modifier),
// where max(z, s z) or a select would take the integer/logic pipe.
template <int V>
__device__ __forceinline__ float score_abs(const float (&r)[V], const float (&x)[V],
                                           const float (&w)[V], float c1, float c2) {
  float d0 = 0.f, d1 = 0.f, e0 = 0.f, e1 = 0.f;
#pragma unroll
  for (int c = 0; c < V; c += 2) {
    float z0, z1;
    add2(z0, z1, r[c], r[c + 1], x[c], x[c + 1]);
    fma2(d0, d1, z0, z1, w[c], w[c + 1]);
    e0 = fmaf(w[c], fabsf(z0), e0);
    e1 = fmaf(w[c + 1], fabsf(z1), e1);
  }
  return fmaf(c1, d0 + d1, c2 * (e0 + e1));
}

template <typename T>
__device__ __forceinline__ void att_slice(const float* att, const Lane<1>& L, float scale,
                                          float (&w)[VecOf<T>::n]) {
  float tmp[1][VecOf<T>::n];
  load_att<T, 1>(att, L, scale, tmp);
#pragma unroll
  for (int c = 0; c < VecOf<T>::n; ++c) w[c] = tmp[0][c];
}

// ---------------------------------------------------------------------------
// forward
// ---------------------------------------------------------------------------

template <typename T>
struct V2Online {
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
__device__ __forceinline__ void fwd_edges(const V2Args& A, const Lane<1>& L, const int32_t* cols,
                                          int colbase, int beg, int end, int sg, int SG, int step,
                                          int trips, int (&jn)[kUnroll],
                                          const float (&xr)[VecOf<T>::n],
                                          const float (&a2)[VecOf<T>::n], V2Online<T>& st) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kUnroll;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      raw[u] = (j[u] >= 0 && L.ok[0]) ? ld16(row_base<T>(A.xl, j[u], A.s.rv) + 16 * L.q[0])
                                      : make_uint4(0, 0, 0, 0);
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
    float sc[U];
    const float c1 = 0.5f * (1.f + A.slope), c2 = 0.5f * (1.f - A.slope);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[V];
      unpack<T>(raw[u], x);
      sc[u] = score_abs<V>(xr, x, a2, c1, c2);
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
      unpack_alt<T>(raw[u], x);
      axpy<V>(st.acc, p, x);
    }
    st.m = mn;
  }
}

template <typename T>
__device__ __forceinline__ void fwd_write(const V2Args& A, const Lane<1>& L, int64_t node,
                                          const V2Online<T>& st) {
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

// kSub: light nodes take one sub-group each (rows narrower than a warp).
template <typename T, bool kSub>
__global__ void __launch_bounds__(kThreads, 3) v2_fwd_main(const V2Args A) {
  constexpr int V = VecOf<T>::n;
  const V2Dir& D = A.csr;
  const Lane<1> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  const int H = A.s.H;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  float a2[V], xr[V];
  att_slice<T>(A.att, L, kLog2e, a2);

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
      // batches of kUnroll * G edges dealt to the warps in turn
      const int wb = it.y + wid * kUnroll * L.G;
      const int colbase = it.y & ~3;
      int jn[kUnroll];
      batch_ids<kUnroll>(cols, colbase, wb, it.z, L.g, L.G, jn);
      own_row<T>(A.xr, it.x, A.s, L, xr);
      V2Online<T> st;
      st.init();
      fwd_edges<T, false>(A, L, cols, colbase, wb, it.z, L.g, L.G, kWarps * kUnroll * L.G, 0, jn,
                          xr, a2, st);
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
        V2Online<T> tot;
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

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  if (kSub) {
    // nodes per sub-group per pull: four where a warp holds two sub-groups
    // (3 % faster than two on 256-byte rows), two otherwise; the backward
    // passes keep two (four measured 3 % slower there)
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
        int trips = (end - beg + kUnroll - 1) / kUnroll;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) trips = max(trips, __shfl_xor_sync(kFull, trips, o));
        int jn[kUnroll];
        batch_ids<kUnroll>(D.idx, 0, beg, end, 0, 1, jn);
        own_row<T>(A.xr, i >= 0 ? i : 0, A.s, L, xr);
        V2Online<T> st;
        st.init();
        fwd_edges<T, true>(A, L, D.idx, 0, beg, end, 0, 1, kUnroll, trips, jn, xr, a2, st);
        if (i >= 0) fwd_write<T>(A, L, i, st);
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
    int jn[kUnroll];
    batch_ids<kUnroll>(D.idx, 0, beg, end, L.g, L.G, jn);
    for (int q = 0; q < kGrab && i >= 0; ++q) {
      const int nq = (q + 1) & (kGrab - 1);
      const int i2 = q + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[kUnroll];
      batch_ids<kUnroll>(D.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      own_row<T>(A.xr, i, A.s, L, xr);
      V2Online<T> st;
      st.init();
      fwd_edges<T, false>(A, L, D.idx, 0, beg, end, L.g, L.G, kUnroll * L.G, 0, jn, xr, a2, st);
      st.merge_subgroups(A.s);
      if (L.g == 0) fwd_write<T>(A, L, i, st);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) jn[u] = jn2[u];
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) v2_fwd_merge(const V2Args A) {
  constexpr int V = VecOf<T>::n;
  const Lane<1> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.csr.n_hubs || L.g != 0 || !L.ok[0]) return;
  const int4 hb = A.csr.hubs[t];
  const int row_f = A.s.rv * V;
  V2Online<T> st;
  st.init();
  for (int c = 0; c < hb.z; ++c) {
    const int64_t slot = int64_t(hb.y) + c;
    const float2 ml = A.f_ml[slot * A.s.H + L.k[0]];
    float ab[V];
    const float* pa = A.f_acc + slot * row_f + L.q[0] * V;
#pragma unroll
    for (int c4 = 0; c4 < V; c4 += 4) {
      const float4 q = *reinterpret_cast<const float4*>(pa + c4);
      ab[c4] = q.x;
      ab[c4 + 1] = q.y;
      ab[c4 + 2] = q.z;
      ab[c4 + 3] = q.w;
    }
    st.merge(ml.x, ml.y, ab);
  }
  fwd_write<T>(A, L, hb.x, st);
}

// ---------------------------------------------------------------------------
// backward pass 1: destination side
// ---------------------------------------------------------------------------

template <typename T>
struct DstSums {
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

// The LeakyReLU slopes g of a batch stay in registers between the score
// (which needs l = g z) and the sums (which need g alone).  The batch at
// `base` holds edges base + sg + u * SG; until end (kFixed false), or for
// exactly `trips` batches (kFixed true, the same count on every lane of the
// warp; batches past end add nothing).
template <typename T, bool kFixed>
__device__ __forceinline__ void dst_edges(const V2Args& A, const Lane<1>& L, const int32_t* cols,
                                          int colbase, int beg, int end, int sg, int SG,
                                          int step, int trips, int (&jn)[kUB],
                                          const float (&xr)[VecOf<T>::n],
                                          const float (&gi)[VecOf<T>::n],
                                          const float (&a2)[VecOf<T>::n], float lse2,
                                          DstSums<T>& sm) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kUB;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      raw[u] = (j[u] >= 0 && L.ok[0]) ? ld16(row_base<T>(A.xl, j[u], A.s.rv) + 16 * L.q[0])
                                      : make_uint4(0, 0, 0, 0);
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
    float red[2 * U];  // scores (base 2), then dout_i . xl_j
    float g[U][V];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[V], lz[V];
      unpack<T>(raw[u], x);
      leaky_terms<V>(xr, x, A.slope, g[u], lz);
      red[u] = dot<V>(lz, a2);
      red[U + u] = dot<V>(x, gi);
    }
    head_sums<2 * U>(red, A.s.hv_log2);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float al = j[u] >= 0 ? ex2(red[u] - lse2) : 0.f;
      const float ad = al * red[U + u];
      sm.delta += ad;
      axpy<V>(sm.P, ad, g[u]);
      axpy<V>(sm.Q, al, g[u]);
    }
  }
}

// From the totals of node i: u = P - Delta Q; write dxr_i = att u and i's
// record, add i's datt term xr_i u into this warp's datt sums dslot[row_f]
// (shared memory; the lane's own elements, so no other lane touches them).
template <typename T>
__device__ __forceinline__ void dst_finish(const V2Args& A, const Lane<1>& L, int64_t i,
                                           const DstSums<T>& sm, float lse2,
                                           const float (&xr)[VecOf<T>::n], float* dslot) {
  constexpr int V = VecOf<T>::n;
  if (!L.ok[0]) return;
  float a[V], y[V];
  att_slice<T>(A.att, L, 1.f, a);
  float* d = dslot + L.q[0] * V;
#pragma unroll
  for (int c = 0; c < V; ++c) {
    const float u = fmaf(-sm.delta, sm.Q[c], sm.P[c]);
    y[c] = a[c] * u;
    d[c] = fmaf(xr[c], u, d[c]);
  }
  st16(reinterpret_cast<char*>(A.dxr) + i * int64_t(A.s.rv) * 16 + 16 * L.q[0], pack<T>(y));
  if (L.head_leader(A.s, 0)) A.stats[i * A.s.H + L.k[0]] = make_float2(lse2, sm.delta);
}

// Zero this lane's elements of its datt slot (with kSub every sub-group has
// a slot of its own; otherwise the g == 0 lanes own the warp's one).
template <int V, bool kSub>
__device__ __forceinline__ void zero_da(const Lane<1>& L, float* dslot) {
  if ((kSub || L.g == 0) && L.ok[0])
#pragma unroll
    for (int c = 0; c < V; ++c) dslot[L.q[0] * V + c] = 0.f;
}

// Fold the datt slots buf[slots][row_f] of this block (slot order: warp, then
// sub-group) into da_part[row].
__device__ __forceinline__ void fold_da(const V2Args& A, int row_f, const float* buf, int slots,
                                        int64_t row) {
  __syncthreads();
  for (int t = threadIdx.x; t < row_f; t += blockDim.x) {
    double s = 0.0;
    for (int w = 0; w < slots; ++w) s += double(buf[w * row_f + t]);
    A.da_part[row * row_f + t] = s;
  }
}

// kSub: light nodes take one sub-group each (rows narrower than a warp), each
// sub-group with its own datt slot; otherwise one warp each.
template <typename T, bool kSub>
__global__ void __launch_bounds__(kThreads, 3) v2_dst_main(const V2Args A) {
  constexpr int V = VecOf<T>::n;
  const V2Dir& D = A.csr;
  const Lane<1> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  const int H = A.s.H;
  const int nsub = kSub ? L.G : 1;
  extern __shared__ __align__(16) unsigned char smem[];
  float a2[V], xr[V], gi[V];
  att_slice<T>(A.att, L, kLog2e, a2);
  float* wbuf = reinterpret_cast<float*>(smem + D.col_off);  // [kWarps][H + 2 row_f]
  float* dsum = wbuf + kWarps * (H + 2 * row_f);              // [kWarps * nsub][row_f]
  float* dslot = dsum + (wid * nsub + (kSub ? L.g : 0)) * row_f;
  zero_da<V, kSub>(L, dslot);

  // ---- block items, assigned statically: item b, b + B, ... -------------
  if (D.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    __syncthreads();
    for (int64_t it_i = blockIdx.x; it_i < D.n_items; it_i += gridDim.x) {
      const int4 it = D.items[it_i];
      if (!stage_edges(cols, D.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kUB * G edges dealt to the warps in turn
      const int wb = it.y + wid * kUB * L.G;
      const int colbase = it.y & ~3;
      int jn[kUB];
      batch_ids<kUB>(cols, colbase, wb, it.z, L.g, L.G, jn);
      own_row<T>(A.xr, it.x, A.s, L, xr);
      own_row<T>(A.dout, it.x, A.s, L, gi);
      const float lse2 = L.ok[0] ? A.lse_in[int64_t(it.x) * H + L.k[0]] * kLog2e : 0.f;
      DstSums<T> sm;
      sm.init();
      dst_edges<T, false>(A, L, cols, colbase, wb, it.z, L.g, L.G, kWarps * kUB * L.G, 0, jn, xr,
                          gi, a2, lse2, sm);
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
        DstSums<T> tot;
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
          dst_finish<T>(A, L, it.x, tot, lse2, xr, dslot);
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

  const int64_t gw = int64_t(blockIdx.x) * kWarps + wid;
  const int64_t W = int64_t(gridDim.x) * kWarps;
  // ---- light nodes, rows narrower than a warp: one sub-group each, groups
  // of R * G nodes per warp assigned statically ------------------------------
  if (kSub) {
    const int R = L.G >= 32 ? 1 : 2;  // nodes per sub-group per group
    const int npull = R * L.G;
    for (int64_t t0 = gw * npull; t0 < D.n_light; t0 += W * npull) {
      int my_i = -1, my_b = 0, my_e = 0;
      if (L.lane < npull && t0 + L.lane < D.n_light) {
        my_i = D.light[t0 + L.lane];
        my_b = D.ptr[my_i];
        my_e = D.ptr[my_i + 1];
      }
      for (int r = 0; r < R; ++r) {
        const int from = r * L.G + L.g;
        const int i = __shfl_sync(kFull, my_i, from);
        const int beg = __shfl_sync(kFull, my_b, from);
        const int e0 = __shfl_sync(kFull, my_e, from);  // every lane shuffles
        const int end = i >= 0 ? e0 : beg;
        if (!__any_sync(kFull, i >= 0)) break;
        int trips = (end - beg + kUB - 1) / kUB;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) trips = max(trips, __shfl_xor_sync(kFull, trips, o));
        int jn[kUB];
        batch_ids<kUB>(D.idx, 0, beg, end, 0, 1, jn);
        const int ii = i >= 0 ? i : 0;
        own_row<T>(A.xr, ii, A.s, L, xr);
        own_row<T>(A.dout, ii, A.s, L, gi);
        const float lse2 = L.ok[0] ? A.lse_in[int64_t(ii) * H + L.k[0]] * kLog2e : 0.f;
        DstSums<T> sm;
        sm.init();
        dst_edges<T, true>(A, L, D.idx, 0, beg, end, 0, 1, kUB, trips, jn, xr, gi, a2, lse2, sm);
        if (i >= 0) dst_finish<T>(A, L, i, sm, lse2, xr, dslot);
      }
    }
    fold_da(A, row_f, dsum, kWarps * nsub, blockIdx.x);
    return;
  }

  // ---- light nodes, rows of a whole warp: groups of kGrab per warp,
  // assigned statically -------------------------------------------------------
  for (int64_t t0 = gw * kGrab; t0 < D.n_light; t0 += W * kGrab) {
    int my_i = -1, my_b = 0, my_e = 0;
    if (L.lane < kGrab && t0 + L.lane < D.n_light) {
      my_i = D.light[t0 + L.lane];
      my_b = D.ptr[my_i];
      my_e = D.ptr[my_i + 1];
    }
    int i = __shfl_sync(kFull, my_i, 0);
    int beg = __shfl_sync(kFull, my_b, 0), end = __shfl_sync(kFull, my_e, 0);
    int jn[kUB];
    batch_ids<kUB>(D.idx, 0, beg, end, L.g, L.G, jn);
    for (int q = 0; q < kGrab && i >= 0; ++q) {
      const int nq = (q + 1) & (kGrab - 1);
      const int i2 = q + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[kUB];
      batch_ids<kUB>(D.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      own_row<T>(A.xr, i, A.s, L, xr);
      own_row<T>(A.dout, i, A.s, L, gi);
      const float lse2 = L.ok[0] ? A.lse_in[int64_t(i) * H + L.k[0]] * kLog2e : 0.f;
      DstSums<T> sm;
      sm.init();
      dst_edges<T, false>(A, L, D.idx, 0, beg, end, L.g, L.G, kUB * L.G, 0, jn, xr, gi, a2, lse2,
                          sm);
      sm.subgroup_total(A.s);
      if (L.g == 0) dst_finish<T>(A, L, i, sm, lse2, xr, dslot);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < kUB; ++u) jn[u] = jn2[u];
    }
  }
  fold_da(A, row_f, dsum, kWarps * nsub, blockIdx.x);
}

// One warp per CSR hub (static): add its chunk sums in chunk order, finish the
// node; each block's datt terms go to da_part[da_main_rows + block].
template <typename T>
__global__ void __launch_bounds__(kThreads) v2_dst_merge(const V2Args A) {
  constexpr int V = VecOf<T>::n;
  const Lane<1> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int64_t t = int64_t(blockIdx.x) * kWarps + wid;
  const int row_f = A.s.rv * V;
  const int H = A.s.H;
  __shared__ float buf[kWarps * 256];  // rows of at most 512 bytes: <= 256 floats
  float* dslot = buf + wid * row_f;
  zero_da<V, false>(L, dslot);
  if (t < A.csr.n_hubs && L.g == 0 && L.ok[0]) {
    const int4 hb = A.csr.hubs[t];
    DstSums<T> tot;
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
    float xr[V];
    own_row<T>(A.xr, hb.x, A.s, L, xr);
    const float lse2 = A.lse_in[int64_t(hb.x) * H + L.k[0]] * kLog2e;
    dst_finish<T>(A, L, hb.x, tot, lse2, xr, dslot);
  }
  fold_da(A, row_f, buf, kWarps, A.da_main_rows + blockIdx.x);
}

// ---------------------------------------------------------------------------
// backward pass 2: source side
// ---------------------------------------------------------------------------

// acc += alpha_ij dout_i and w += de_ij g_ij over the batch; the slopes g of
// a batch stay in registers between the score and the sums.
template <typename T, bool kFixed>
__device__ __forceinline__ void src_edges(const V2Args& A, const Lane<1>& L, const int32_t* cols,
                                          int colbase, int beg, int end, int sg, int SG,
                                          int step, int trips, int (&in)[kUB],
                                          const float (&xl)[VecOf<T>::n],
                                          const float (&a2)[VecOf<T>::n],
                                          float (&acc)[VecOf<T>::n], float (&w)[VecOf<T>::n]) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kUB;
  const int H = A.s.H;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int i[U];
#pragma unroll
    for (int u = 0; u < U; ++u) i[u] = in[u];
    uint4 rr[U], rg[U];
    float2 st[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool ok = i[u] >= 0 && L.ok[0];
      rr[u] = ok ? ld16(row_base<T>(A.xr, i[u], A.s.rv) + 16 * L.q[0]) : make_uint4(0, 0, 0, 0);
      rg[u] = ok ? ld16(row_base<T>(A.dout, i[u], A.s.rv) + 16 * L.q[0]) : make_uint4(0, 0, 0, 0);
      st[u] = ok ? __ldg(A.stats + int64_t(i[u]) * H + L.k[0]) : make_float2(0.f, 0.f);
    }
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, in);
    float red[2 * U];
    float g[U][V];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float r[V], gd[V], lz[V];
      unpack<T>(rr[u], r);
      unpack<T>(rg[u], gd);
      leaky_terms<V>(r, xl, A.slope, g[u], lz);
      red[u] = dot<V>(lz, a2);
      red[U + u] = dot<V>(gd, xl);
    }
    head_sums<2 * U>(red, A.s.hv_log2);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float al = i[u] >= 0 ? ex2(red[u] - st[u].x) : 0.f;
      const float de = al * (red[U + u] - st[u].y);
      float gd[V];
      unpack_alt<T>(rg[u], gd);
      axpy<V>(acc, al, gd);
      axpy<V>(w, de, g[u]);
    }
  }
}

// Totals of node j's (partial) sums: add the datt term xl_j w into the datt
// slot and turn acc into acc + att w.  Split (a node's edges spread over the
// warp's sub-groups): the sub-group sums are added first and the lanes with
// g == 0 finish; otherwise each sub-group holds a node of its own.
template <typename T, bool kSplit>
__device__ __forceinline__ void src_combine(const V2Args& A, const Lane<1>& L,
                                            const float (&xl)[VecOf<T>::n],
                                            float (&acc)[VecOf<T>::n],
                                            float (&w)[VecOf<T>::n], float* dslot) {
  constexpr int V = VecOf<T>::n;
  if (kSplit) {
    subgroup_sums<V>(acc, A.s);
    subgroup_sums<V>(w, A.s);
    if (L.g != 0) return;
  }
  if (!L.ok[0]) return;
  float a[V];
  att_slice<T>(A.att, L, 1.f, a);
  float* d = dslot + L.q[0] * V;
#pragma unroll
  for (int c = 0; c < V; ++c) {
    d[c] = fmaf(xl[c], w[c], d[c]);
    acc[c] = fmaf(a[c], w[c], acc[c]);
  }
}

template <typename T>
__device__ __forceinline__ void src_write(const V2Args& A, const Lane<1>& L, int64_t j,
                                          const float (&acc)[VecOf<T>::n]) {
  if (!L.ok[0]) return;
  st16(reinterpret_cast<char*>(A.dxl) + j * int64_t(A.s.rv) * 16 + 16 * L.q[0], pack<T>(acc));
}

// Work is assigned statically (block items b, b + B, ...; light groups by
// warp), so that the per-block datt sums, folded into da_part[da_src_row0 +
// block], do not depend on timing.
template <typename T, bool kSub>
__global__ void __launch_bounds__(kThreads, 3) v2_src_main(const V2Args A) {
  constexpr int V = VecOf<T>::n;
  const V2Dir& D = A.csc;
  const Lane<1> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  const int nsub = kSub ? L.G : 1;
  extern __shared__ __align__(16) unsigned char smem[];
  float a2[V], xl[V], acc[V], w[V];
  att_slice<T>(A.att, L, kLog2e, a2);
  float* wacc = reinterpret_cast<float*>(smem + D.col_off);  // [kWarps][row_f]
  float* dsum = wacc + kWarps * row_f;                        // [kWarps * nsub][row_f]
  float* dslot = dsum + (wid * nsub + (kSub ? L.g : 0)) * row_f;
  zero_da<V, kSub>(L, dslot);

  if (D.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    __syncthreads();
    for (int64_t it_i = blockIdx.x; it_i < D.n_items; it_i += gridDim.x) {
      const int4 it = D.items[it_i];
      if (!stage_edges(cols, D.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kUB * G edges dealt to the warps in turn
      const int wb = it.y + wid * kUB * L.G;
      const int colbase = it.y & ~3;
      int in[kUB];
      batch_ids<kUB>(cols, colbase, wb, it.z, L.g, L.G, in);
      own_row<T>(A.xl, it.x, A.s, L, xl);
      zero<V>(acc);
      zero<V>(w);
      src_edges<T, false>(A, L, cols, colbase, wb, it.z, L.g, L.G, kWarps * kUB * L.G, 0, in, xl,
                          a2, acc, w);
      src_combine<T, true>(A, L, xl, acc, w, dslot);
      if (L.g == 0 && L.ok[0])
#pragma unroll
        for (int c = 0; c < V; ++c) wacc[wid * row_f + L.q[0] * V + c] = acc[c];
      __syncthreads();
      if (wid == 0 && L.g == 0 && L.ok[0]) {
#pragma unroll
        for (int c = 0; c < V; ++c) {
          float s = 0.f;
          for (int k = 0; k < kWarps; ++k) s += wacc[k * row_f + L.q[0] * V + c];
          acc[c] = s;
        }
        if (it.w < 0) {
          src_write<T>(A, L, it.x, acc);
        } else {
          float* pa = A.s_acc + int64_t(it.w) * row_f + L.q[0] * V;
#pragma unroll
          for (int c4 = 0; c4 < V; c4 += 4)
            *reinterpret_cast<float4*>(pa + c4) =
                make_float4(acc[c4], acc[c4 + 1], acc[c4 + 2], acc[c4 + 3]);
        }
      }
      __syncthreads();
    }
  }

  const int64_t gw = int64_t(blockIdx.x) * kWarps + wid;
  const int64_t W = int64_t(gridDim.x) * kWarps;
  // ---- light nodes, rows narrower than a warp: one sub-group each, groups
  // of R * G nodes per warp assigned statically ------------------------------
  if (kSub) {
    const int R = L.G >= 32 ? 1 : 2;
    const int npull = R * L.G;
    for (int64_t t0 = gw * npull; t0 < D.n_light; t0 += W * npull) {
      int my_j = -1, my_b = 0, my_e = 0;
      if (L.lane < npull && t0 + L.lane < D.n_light) {
        my_j = D.light[t0 + L.lane];
        my_b = D.ptr[my_j];
        my_e = D.ptr[my_j + 1];
      }
      for (int r = 0; r < R; ++r) {
        const int from = r * L.G + L.g;
        const int j = __shfl_sync(kFull, my_j, from);
        const int beg = __shfl_sync(kFull, my_b, from);
        const int e0 = __shfl_sync(kFull, my_e, from);  // every lane shuffles
        const int end = j >= 0 ? e0 : beg;
        if (!__any_sync(kFull, j >= 0)) break;
        int trips = (end - beg + kUB - 1) / kUB;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) trips = max(trips, __shfl_xor_sync(kFull, trips, o));
        int in[kUB];
        batch_ids<kUB>(D.idx, 0, beg, end, 0, 1, in);
        own_row<T>(A.xl, j >= 0 ? j : 0, A.s, L, xl);
        zero<V>(acc);
        zero<V>(w);
        src_edges<T, true>(A, L, D.idx, 0, beg, end, 0, 1, kUB, trips, in, xl, a2, acc, w);
        if (j >= 0) {
          src_combine<T, false>(A, L, xl, acc, w, dslot);
          src_write<T>(A, L, j, acc);
        }
      }
    }
    fold_da(A, row_f, dsum, kWarps * nsub, A.da_src_row0 + blockIdx.x);
    return;
  }

  // ---- light nodes, rows of a whole warp: groups of kGrab per warp,
  // assigned statically -------------------------------------------------------
  for (int64_t t0 = gw * kGrab; t0 < D.n_light; t0 += W * kGrab) {
    int my_j = -1, my_b = 0, my_e = 0;
    if (L.lane < kGrab && t0 + L.lane < D.n_light) {
      my_j = D.light[t0 + L.lane];
      my_b = D.ptr[my_j];
      my_e = D.ptr[my_j + 1];
    }
    int j = __shfl_sync(kFull, my_j, 0);
    int beg = __shfl_sync(kFull, my_b, 0), end = __shfl_sync(kFull, my_e, 0);
    int in[kUB];
    batch_ids<kUB>(D.idx, 0, beg, end, L.g, L.G, in);
    for (int q = 0; q < kGrab && j >= 0; ++q) {
      const int nq = (q + 1) & (kGrab - 1);
      const int j2 = q + 1 < kGrab ? __shfl_sync(kFull, my_j, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int in2[kUB];
      batch_ids<kUB>(D.idx, 0, b2, j2 >= 0 ? e2 : b2, L.g, L.G, in2);
      own_row<T>(A.xl, j, A.s, L, xl);
      zero<V>(acc);
      zero<V>(w);
      src_edges<T, false>(A, L, D.idx, 0, beg, end, L.g, L.G, kUB * L.G, 0, in, xl, a2, acc, w);
      src_combine<T, true>(A, L, xl, acc, w, dslot);
      if (L.g == 0) src_write<T>(A, L, j, acc);
      j = j2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < kUB; ++u) in[u] = in2[u];
    }
  }
  fold_da(A, row_f, dsum, kWarps * nsub, A.da_src_row0 + blockIdx.x);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) v2_src_merge(const V2Args A) {
  constexpr int V = VecOf<T>::n;
  const Lane<1> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.csc.n_hubs || L.g != 0 || !L.ok[0]) return;
  const int4 hb = A.csc.hubs[t];
  const int row_f = A.s.rv * V;
  float acc[V], cmp[V];
  zero<V>(acc);
  zero<V>(cmp);
  for (int c = 0; c < hb.z; ++c) {
    const float* pa = A.s_acc + (int64_t(hb.y) + c) * row_f + L.q[0] * V;
#pragma unroll
    for (int e = 0; e < V; ++e) kahan_add(acc[e], cmp[e], pa[e]);
  }
  src_write<T>(A, L, hb.x, acc);
}

// datt = fixed-order float64 sum of the da_part rows (one warp per element).
__global__ void __launch_bounds__(kThreads) v2_datt_final(const double* part, int rows,
                                                          int row_f, float* datt) {
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= row_f) return;
  double s = 0.0;
#pragma unroll 8
  for (int r = lane; r < rows; r += 32) s += part[int64_t(r) * row_f + t];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
  if (lane == 0) datt[t] = float(s);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

template <typename T>
cudaError_t fwd_t(const V2Args& A, int sm_count, cudaStream_t st) {
  constexpr int V = VecOf<T>::n;
  const int row_f = A.s.rv * V;
  cudaError_t e;
  if ((e = cudaMemsetAsync(A.ctr, 0, kCounters * sizeof(int), st)) != cudaSuccess) return e;
  const V2Dir& D = A.csr;
  if (D.n_items + D.n_light > 0) {
    const size_t smem = size_t(D.col_off) + size_t(kWarps) * (2 * A.s.H + row_f) * 4;
    auto kernel = A.s.lpr < 32 ? v2_fwd_main<T, true> : v2_fwd_main<T, false>;
    if ((e = set_smem(kernel, smem)) != cudaSuccess) return e;
    const int64_t work = D.n_items + (D.n_light + kWarps * kGrab - 1) / (kWarps * kGrab);
    const int64_t cap = persistent_blocks(kernel, smem, sm_count);
    kernel<<<unsigned(work < cap ? work : cap), kThreads, smem, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (D.n_hubs > 0) {
    v2_fwd_merge<T><<<unsigned((D.n_hubs + kWarps - 1) / kWarps), kThreads, 0, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename T>
cudaError_t bwd_t(V2Args A, int sm_count, cudaStream_t st) {
  constexpr int V = VecOf<T>::n;
  const int row_f = A.s.rv * V;
  const int64_t cap = int64_t(sm_count > 0 ? sm_count : 1) * 8;
  // rows narrower than a warp: light nodes one sub-group each, with a datt
  // slot per sub-group
  const bool sub = A.s.lpr < 32;
  const int nsub = sub ? 32 / A.s.lpr : 1;
  cudaError_t e;
  // pass 1: a fixed grid (static work assignment), one da_part row per block
  {
    const V2Dir& D = A.csr;
    const size_t smem =
        size_t(D.col_off) + size_t(kWarps) * (A.s.H + 2 * row_f + nsub * row_f) * 4;
    auto kernel = sub ? v2_dst_main<T, true> : v2_dst_main<T, false>;
    if ((e = set_smem(kernel, smem)) != cudaSuccess) return e;
    int64_t blocks = persistent_blocks(kernel, smem, sm_count);
    if (blocks > cap) blocks = cap;
    A.da_main_rows = int(blocks);
    kernel<<<unsigned(blocks), kThreads, smem, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t mblocks = (D.n_hubs + kWarps - 1) / kWarps;
    if (mblocks > 0) {
      v2_dst_merge<T><<<unsigned(mblocks), kThreads, 0, st>>>(A);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    A.da_src_row0 = int(blocks + mblocks);
  }
  // pass 2: likewise a fixed grid, one da_part row per block
  {
    const V2Dir& D = A.csc;
    const size_t smem = size_t(D.col_off) + size_t(kWarps) * (1 + nsub) * row_f * 4;
    auto kernel = sub ? v2_src_main<T, true> : v2_src_main<T, false>;
    if ((e = set_smem(kernel, smem)) != cudaSuccess) return e;
    int64_t blocks = persistent_blocks(kernel, smem, sm_count);
    if (blocks > cap) blocks = cap;
    kernel<<<unsigned(blocks), kThreads, smem, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (D.n_hubs > 0) {
      v2_src_merge<T><<<unsigned((D.n_hubs + kWarps - 1) / kWarps), kThreads, 0, st>>>(A);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    v2_datt_final<<<unsigned((row_f + kWarps - 1) / kWarps), kThreads, 0, st>>>(
        A.da_part, int(A.da_src_row0 + blocks), row_f, A.datt);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

V2Dir v2_dir(const Dir& d) {
  V2Dir a{};
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

struct V2Layout {
  size_t ctr, f_acc, f_ml, stats, d_delta, d_vec, s_acc, da_part, total;
};

V2Layout v2_layout(const gnn_graph* g, const Shape& s) {
  const size_t row_f = size_t(s.rv) * 16 / s.esize;
  const size_t cc = size_t(g->csr.n_hub_chunks), sc = size_t(g->csc.n_hub_chunks);
  // one row per block of each pass (at most 8 per SM) and per hub-merge block
  const size_t da_rows = size_t(g->sm_count > 0 ? g->sm_count : 1) * 16 +
                         size_t((g->csr.n_hubs + kWarps - 1) / kWarps);
  V2Layout L{};
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
  L.s_acc = take(sc * row_f * 4);
  L.da_part = take(da_rows * row_f * 8);
  L.total = off;
  return L;
}

V2Args v2_args(const gnn_graph* g, const Shape& s, const void* xl, const void* xr,
               const float* att, float slope, char* ws) {
  const V2Layout W = v2_layout(g, s);
  V2Args A{};
  A.s = s;
  A.csr = v2_dir(g->csr);
  A.csc = v2_dir(g->csc);
  A.n = g->n;
  A.xl = xl;
  A.xr = xr;
  A.att = att;
  A.slope = slope;
  A.ctr = reinterpret_cast<int*>(ws + W.ctr);
  A.f_acc = reinterpret_cast<float*>(ws + W.f_acc);
  A.f_ml = reinterpret_cast<float2*>(ws + W.f_ml);
  A.stats = reinterpret_cast<float2*>(ws + W.stats);
  A.d_delta = reinterpret_cast<float*>(ws + W.d_delta);
  A.d_vec = reinterpret_cast<float*>(ws + W.d_vec);
  A.s_acc = reinterpret_cast<float*>(ws + W.s_acc);
  A.da_part = reinterpret_cast<double*>(ws + W.da_part);
  A.err = g->err;
  return A;
}

}  // namespace

size_t gatv2_ws_bytes(const gnn_graph* g, const Shape& s) { return v2_layout(g, s).total; }

cudaError_t launch_gatv2_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                 const void* xl, const void* xr, const float* att, float slope,
                                 void* out, float* lse, char* ws, cudaStream_t st) {
  V2Args A = v2_args(g, s, xl, xr, att, slope, ws);
  A.out = out;
  A.lse = lse;
  return dt == GNN_F32 ? fwd_t<float>(A, g->sm_count, st)
                       : fwd_t<__nv_bfloat16>(A, g->sm_count, st);
}

cudaError_t launch_gatv2_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                  const void* xl, const void* xr, const float* att, float slope,
                                  const float* lse, const void* dout, void* dxl, void* dxr,
                                  float* datt, char* ws, cudaStream_t st) {
  V2Args A = v2_args(g, s, xl, xr, att, slope, ws);
  A.lse_in = lse;
  A.dout = dout;
  A.dxl = dxl;
  A.dxr = dxr;
  A.datt = datt;
  return dt == GNN_F32 ? bwd_t<float>(A, g->sm_count, st)
                       : bwd_t<__nv_bfloat16>(A, g->sm_count, st);
}

}  // namespace gnn
