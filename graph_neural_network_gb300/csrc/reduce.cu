// Reduction-family neighbour aggregation: max or min over the in-neighbours
// of each node, feature by feature, with the winning source ("On Efficient
// Scaling of GNNs via IO-Aware Layers Implementations", Technical Summary >
// Methodology, reduction-based aggregations).
//
//   out[i][f] = max_j x[j][f]  (or min),  arg[i][f] = the winning j,
//   equal values going to the smallest j; a node with no in-neighbours gets
//   out = 0 and arg = -1.
//
// Candidates are ordered by (s * value descending, source ascending), with
// s = +1 for max and -1 for min: a total order, so the winner does not
// depend on the order edges are visited and every merge below is exact and
// reproducible.  Degree-aware tiling as on the page: light nodes get a warp
// (feature-parallel lanes, edges split over sub-groups), or a sub-group of
// their own where a row is narrower than a warp, mid nodes a thread block,
// and hubs are split into edge chunks whose winners are merged with
// 64-bit atomicMax on packed (value, source) keys -- the page's atomic merge
// of packed (value, index) pairs -- then decoded by a small kernel.
//
// Backward: dx[j][f] = sum of dout[i][f] over the i whose winner for f is
// j.  One coalesced pass over (arg, dout) adds each term into a float32
// accumulator with atomic adds; when several destinations share a winner
// the order of their additions, and so the last bits of dx, can vary from
// run to run (out and arg never do).  (Splitting the features into slabs
// whose accumulator part stays in L2 measured 2.5x slower on GB300.)  The
// ordered variant gathers the same terms over the cached CSC instead, in a
// fixed order and without atomics.
#include "device.cuh"

namespace gnn {
namespace {

constexpr int kGrab = 4;
constexpr int kNone = 0x7fffffff;  // "no candidate yet"

struct RedArgs {
  Shape s;
  const int32_t* ptr;
  const int32_t* idx;
  const int32_t* light;
  int64_t n_light;
  const int4* items;
  int64_t n_items;
  const int4* hubs;
  int64_t n_hubs;
  int hub_chunk;
  const void* x;
  float sign;                   // +1 max, -1 min
  void* out;
  int32_t* arg;
  unsigned long long* keys;     // [hub chunks][row floats], indexed by the hub's first slot
  int* ctr;
  int32_t* err;
  int col_off;
};

// Does (v, j) come before (bv, bj) in the order (value desc, source asc)?
__device__ __forceinline__ bool wins(float v, int j, float bv, int bj) {
  return v > bv || (v == bv && j < bj);
}

// Float bits mapped to an unsigned integer with the same order (callers add
// +0.0 first so that -0.0 and +0.0, equal as floats, get one key).
__device__ __forceinline__ uint32_t ordered(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unordered(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

template <typename T, int NV>
struct Best {
  static constexpr int V = VecOf<T>::n;
  float v[NV][V];  // sign * value
  int j[NV][V];
  bool have;       // a candidate has been taken (ascending streams only)
  __device__ __forceinline__ void init() {
    have = false;
#pragma unroll
    for (int a = 0; a < NV; ++a)
#pragma unroll
      for (int c = 0; c < V; ++c) {
        v[a][c] = -INFINITY;
        j[a][c] = kNone;
      }
  }
  __device__ __forceinline__ void take(int a, int c, float bv, int bj) {
    if (wins(bv, bj, v[a][c], j[a][c])) {
      v[a][c] = bv;
      j[a][c] = bj;
    }
  }
  // every lane of the warp ends with the winner over all sub-groups
  __device__ __forceinline__ void merge_subgroups(const Shape& s) {
    for (int o = s.lpr; o < 32; o <<= 1)
#pragma unroll
      for (int a = 0; a < NV; ++a)
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const float bv = __shfl_xor_sync(kFull, v[a][c], o);
          const int bj = __shfl_xor_sync(kFull, j[a][c], o);
          take(a, c, bv, bj);
        }
  }
};

// b takes the edges beg + sg, beg + sg + SG, ... < end (sg, SG: this lane's
// sub-group and the sub-groups sharing the node; 0, 1 for a node of its own).
// kAsc: the CSR rows list their sources in non-decreasing order, so a lane
// meets its candidates by ascending source and an equal value never displaces
// the one it holds: after the lane's first candidate (taken whole), one
// strict comparison per element decides.  Otherwise the full order (value,
// then source) is compared.  kMin: the values enter negated.
template <typename T, int NV, bool kMin, bool kAsc>
__device__ __forceinline__ void red_edges(const RedArgs& A, const Lane<NV>& L,
                                          const int32_t* cols, int colbase, int beg, int end,
                                          int sg, int SG, int step, int (&jn)[kUnroll],
                                          Best<T, NV>& b) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kUnroll;
  for (int base = beg; base < end; base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    uint4 raw[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int a = 0; a < NV; ++a)
        raw[u][a] = (j[u] >= 0 && L.ok[a]) ? ld16(row_base<T>(A.x, j[u], A.s.rv) + 16 * L.q[a])
                                           : make_uint4(0, 0, 0, 0);
    if (base + step < end) batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (j[u] < 0) continue;
      const bool first = kAsc && !b.have;
#pragma unroll
      for (int a = 0; a < NV; ++a) {
        float xv[V];
        unpack<T>(raw[u][a], xv);
#pragma unroll
        for (int c = 0; c < V; ++c) {
          const float sv = kMin ? -xv[c] : xv[c];
          if (kAsc) {
            if (first || sv > b.v[a][c]) {
              b.v[a][c] = sv;
              b.j[a][c] = j[u];
            }
          } else {
            b.take(a, c, sv, j[u]);
          }
        }
      }
      if (kAsc) b.have = true;
    }
  }
}

template <typename T, int NV>
__device__ __forceinline__ void write_best(const RedArgs& A, const Lane<NV>& L, int64_t node,
                                           const Best<T, NV>& b) {
  constexpr int V = VecOf<T>::n;
  char* orow = reinterpret_cast<char*>(A.out) + node * int64_t(A.s.rv) * 16;
  int32_t* arow = A.arg + node * int64_t(A.s.rv) * V;
#pragma unroll
  for (int a = 0; a < NV; ++a) {
    if (!L.ok[a]) continue;
    float y[V];
    int w[V];
#pragma unroll
    for (int c = 0; c < V; ++c) {
      const bool none = b.j[a][c] == kNone;
      y[c] = none ? 0.f : A.sign * b.v[a][c];
      w[c] = none ? -1 : b.j[a][c];
    }
    st16(orow + 16 * L.q[a], pack<T>(y));
#pragma unroll
    for (int c4 = 0; c4 < V; c4 += 4)
      st16(arow + L.q[a] * V + c4, make_uint4(w[c4], w[c4 + 1], w[c4 + 2], w[c4 + 3]));
  }
}

template <typename T, int NV, bool kSub, bool kMin, bool kAsc>
__global__ void __launch_bounds__(kThreads, MinBlocksLean<NV>::value) red_fwd_main(const RedArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<NV> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int row_f = A.s.rv * V;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  Best<T, NV> b;

  if (A.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    float* wv = reinterpret_cast<float*>(smem + A.col_off);  // [kWarps][row_f]
    int* wj = reinterpret_cast<int*>(wv + kWarps * row_f);    // [kWarps][row_f]
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 0, 1);
      __syncthreads();
      const int it_i = s_item;
      if (it_i >= A.n_items) break;
      const int4 it = A.items[it_i];
      if (!stage_edges(cols, A.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kUnroll * G edges dealt to the warps in turn
      const int wb = it.y + wid * kUnroll * L.G;
      const int colbase = it.y & ~3;
      int jn[kUnroll];
      batch_ids<kUnroll>(cols, colbase, wb, it.z, L.g, L.G, jn);
      b.init();
      red_edges<T, NV, kMin, kAsc>(A, L, cols, colbase, wb, it.z, L.g, L.G,
                                   kWarps * kUnroll * L.G, jn, b);
      b.merge_subgroups(A.s);
      if (L.g == 0)
#pragma unroll
        for (int a = 0; a < NV; ++a)
          if (L.ok[a])
#pragma unroll
            for (int c = 0; c < V; ++c) {
              wv[wid * row_f + L.q[a] * V + c] = b.v[a][c];
              wj[wid * row_f + L.q[a] * V + c] = b.j[a][c];
            }
      __syncthreads();
      if (wid == 0 && L.g == 0) {
        b.init();
#pragma unroll
        for (int a = 0; a < NV; ++a)
          if (L.ok[a])
#pragma unroll
            for (int c = 0; c < V; ++c)
              for (int w = 0; w < kWarps; ++w)
                b.take(a, c, wv[w * row_f + L.q[a] * V + c], wj[w * row_f + L.q[a] * V + c]);
        if (it.w < 0) {
          write_best<T, NV>(A, L, it.x, b);
        } else {
          // hub chunk: fold into the hub's packed keys (slot of its first chunk)
          const int first = it.w - (it.y - A.ptr[it.x]) / A.hub_chunk;
          unsigned long long* key = A.keys + int64_t(first) * row_f;
#pragma unroll
          for (int a = 0; a < NV; ++a)
            if (L.ok[a])
#pragma unroll
              for (int c = 0; c < V; ++c)
                if (b.j[a][c] != kNone)
                  atomicMax(key + L.q[a] * V + c,
                            (static_cast<unsigned long long>(ordered(b.v[a][c] + 0.f)) << 32) |
                                static_cast<uint32_t>(~b.j[a][c]));
        }
      }
      __syncthreads();
    }
  }

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  if constexpr (kSub) {
    // two nodes per sub-group per pull, four where a warp holds two
    // sub-groups; no shuffles in the edge loop, so the sub-groups run their
    // own trip counts
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
        int jn[kUnroll];
        batch_ids<kUnroll>(A.idx, 0, beg, end, 0, 1, jn);
        b.init();
        red_edges<T, NV, kMin, kAsc>(A, L, A.idx, 0, beg, end, 0, 1, kUnroll, jn, b);
        write_best<T, NV>(A, L, i, b);
      }
    }
    return;
  }

  // ---- light nodes, rows of a whole warp: one warp each --------------------
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
    int jn[kUnroll];
    batch_ids<kUnroll>(A.idx, 0, beg, end, L.g, L.G, jn);
    for (int q = 0; q < kGrab && i >= 0; ++q) {
      const int nq = (q + 1) & (kGrab - 1);
      const int i2 = q + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[kUnroll];
      batch_ids<kUnroll>(A.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      b.init();
      red_edges<T, NV, kMin, kAsc>(A, L, A.idx, 0, beg, end, L.g, L.G, kUnroll * L.G, jn, b);
      b.merge_subgroups(A.s);
      if (L.g == 0) write_best<T, NV>(A, L, i, b);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) jn[u] = jn2[u];
    }
  }
}

// One warp per hub: decode its packed keys into out and arg.
template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) red_fwd_hubs(const RedArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<NV> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.n_hubs || L.g != 0) return;
  const int4 hb = A.hubs[t];
  const int row_f = A.s.rv * V;
  const unsigned long long* key = A.keys + int64_t(hb.y) * row_f;
  Best<T, NV> b;
  b.init();
#pragma unroll
  for (int a = 0; a < NV; ++a)
    if (L.ok[a])
#pragma unroll
      for (int c = 0; c < V; ++c) {
        const unsigned long long k = key[L.q[a] * V + c];
        if (k != 0ull) {
          b.v[a][c] = unordered(uint32_t(k >> 32));
          b.j[a][c] = int(~uint32_t(k));
        }
      }
  write_best<T, NV>(A, L, hb.x, b);
}

// dx accumulation: every (i, f) with a winner adds dout[i][f] at
// acc[arg[i][f]][f].  One thread per 4 features, coalesced over (arg, dout).
template <typename T>
__global__ void red_bwd_scatter(const int32_t* arg, const void* dout, int64_t n4, int64_t F,
                                float* acc) {
  for (int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < n4;
       q += int64_t(gridDim.x) * blockDim.x) {
    const int4 w = __ldg(reinterpret_cast<const int4*>(arg) + q);
    float g[4];
    if (sizeof(T) == 4) {
      const float4 d = __ldg(reinterpret_cast<const float4*>(dout) + q);
      g[0] = d.x; g[1] = d.y; g[2] = d.z; g[3] = d.w;
    } else {
      const uint2 d = __ldg(reinterpret_cast<const uint2*>(dout) + q);
      g[0] = __uint_as_float(d.x << 16);
      g[1] = __uint_as_float(d.x & 0xffff0000u);
      g[2] = __uint_as_float(d.y << 16);
      g[3] = __uint_as_float(d.y & 0xffff0000u);
    }
    const int64_t f = (q * 4) % F;
    const int ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (ws[c] >= 0) atomicAdd(acc + int64_t(ws[c]) * F + f + c, g[c]);
  }
}

// dx (bfloat16) = acc rounded to nearest even, 8 features per thread.
__global__ void red_bwd_convert(const float* acc, int64_t n8, void* dx) {
  for (int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < n8;
       q += int64_t(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + 2 * q);
    const float4 b = __ldg(reinterpret_cast<const float4*>(acc) + 2 * q + 1);
    reinterpret_cast<uint4*>(dx)[q] =
        make_uint4(bf2(a.x, a.y), bf2(a.z, a.w), bf2(b.x, b.y), bf2(b.z, b.w));
  }
}

template <typename T, int NV>
cudaError_t launch_fwd_t(const RedArgs& A, bool asc, int sm_count, cudaStream_t st) {
  constexpr int V = VecOf<T>::n;
  cudaError_t e;
  if (A.n_items + A.n_light > 0) {
    const size_t smem = size_t(A.col_off) + size_t(kWarps) * A.s.rv * V * 8;
    const bool mn = A.sign < 0.f;
    void (*kernel)(const RedArgs);
    if constexpr (NV == 1) {
      // a sub-group per light node where the row is narrower than a warp;
      // the strict comparison where the CSR rows are in ascending order
      const bool sub = A.s.lpr < 32;
      if (asc)
        kernel = sub ? (mn ? red_fwd_main<T, NV, true, true, true> : red_fwd_main<T, NV, true, false, true>)
                     : (mn ? red_fwd_main<T, NV, false, true, true> : red_fwd_main<T, NV, false, false, true>);
      else
        kernel = sub ? (mn ? red_fwd_main<T, NV, true, true, false> : red_fwd_main<T, NV, true, false, false>)
                     : (mn ? red_fwd_main<T, NV, false, true, false> : red_fwd_main<T, NV, false, false, false>);
    } else {
      kernel = mn ? red_fwd_main<T, NV, false, true, false> : red_fwd_main<T, NV, false, false, false>;
    }
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem))) != cudaSuccess)
      return e;
    const int64_t work = A.n_items + (A.n_light + kWarps * kGrab - 1) / (kWarps * kGrab);
    const int64_t cap = persistent_blocks(kernel, smem, sm_count);
    const int64_t blocks = work < cap ? work : cap;
    kernel<<<unsigned(blocks), kThreads, smem, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (A.n_hubs > 0) {
    red_fwd_hubs<T, NV><<<unsigned((A.n_hubs + kWarps - 1) / kWarps), kThreads, 0, st>>>(A);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

unsigned grid_for(int64_t items, int sm_count) {
  int64_t blocks = (items + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(sm_count > 0 ? sm_count : 1) * 8;
  if (blocks > cap) blocks = cap;
  return unsigned(blocks < 1 ? 1 : blocks);
}

}  // namespace

size_t reduce_ws_bytes(const gnn_graph* g, const Shape& s) {
  const size_t row_f = size_t(s.rv) * 16 / s.esize;
  // counters, hub keys, float32 accumulator of the backward pass; the ordered
  // backward lays the same bytes out as the SpMM workspace
  const size_t own = 256 + align_up(size_t(g->csr.n_hub_chunks) * row_f * 8 + 1, 256) +
                     align_up(size_t(g->n) * row_f * 4 + 1, 256);
  const size_t ordered = spmm_ws_bytes(g, s);
  return own > ordered ? own : ordered;
}

cudaError_t launch_reduce_forward(const gnn_graph* g, const Shape& s, gnn_dtype dt, int op,
                                  const void* x, void* out, int32_t* arg, char* ws,
                                  cudaStream_t st) {
  const Dir& d = g->csr;
  const size_t row_f = size_t(s.rv) * 16 / s.esize;
  RedArgs A{};
  A.s = s;
  A.ptr = d.ptr;
  A.idx = d.idx;
  A.light = d.light;
  A.n_light = d.n_light;
  A.items = d.items;
  A.n_items = d.n_items;
  A.hubs = d.hubs;
  A.n_hubs = d.n_hubs;
  A.hub_chunk = g->tiling.hub_chunk;
  A.x = x;
  A.sign = op == GNN_REDUCE_MIN ? -1.f : 1.f;
  A.out = out;
  A.arg = arg;
  A.ctr = reinterpret_cast<int*>(ws);
  A.keys = reinterpret_cast<unsigned long long*>(ws + 256);
  A.err = g->err;
  A.col_off = int(16 + align_up(size_t(d.max_item + 4) * 4, 16));
  cudaError_t e;
  if ((e = cudaMemsetAsync(A.ctr, 0, kCounters * sizeof(int), st)) != cudaSuccess) return e;
  if (d.n_hub_chunks > 0 &&
      (e = cudaMemsetAsync(A.keys, 0, size_t(d.n_hub_chunks) * row_f * 8, st)) != cudaSuccess)
    return e;
  if (dt == GNN_F32) {
    switch (s.nv) {
      case 1: return launch_fwd_t<float, 1>(A, g->csr_sorted, g->sm_count, st);
      case 2: return launch_fwd_t<float, 2>(A, g->csr_sorted, g->sm_count, st);
      case 4: return launch_fwd_t<float, 4>(A, g->csr_sorted, g->sm_count, st);
    }
  } else {
    switch (s.nv) {
      case 1: return launch_fwd_t<__nv_bfloat16, 1>(A, g->csr_sorted, g->sm_count, st);
      case 2: return launch_fwd_t<__nv_bfloat16, 2>(A, g->csr_sorted, g->sm_count, st);
      case 4: return launch_fwd_t<__nv_bfloat16, 4>(A, g->csr_sorted, g->sm_count, st);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_reduce_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                   const int32_t* arg, const void* dout, void* dx, char* ws,
                                   cudaStream_t st) {
  const int64_t F = int64_t(s.rv) * 16 / s.esize;
  const int64_t nf = g->n * F;
  float* acc = dt == GNN_F32 ? static_cast<float*>(dx)
                             : reinterpret_cast<float*>(
                                   ws + 256 + align_up(size_t(g->csr.n_hub_chunks) * F * 8 + 1,
                                                       256));
  cudaError_t e;
  if ((e = cudaMemsetAsync(acc, 0, size_t(nf) * 4, st)) != cudaSuccess) return e;
  const unsigned grid = grid_for(nf / 4, g->sm_count);
  if (dt == GNN_F32)
    red_bwd_scatter<float><<<grid, kThreads, 0, st>>>(arg, dout, nf / 4, F, acc);
  else
    red_bwd_scatter<__nv_bfloat16><<<grid, kThreads, 0, st>>>(arg, dout, nf / 4, F, acc);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (dt != GNN_F32) {
    red_bwd_convert<<<grid_for(nf / 8, g->sm_count), kThreads, 0, st>>>(acc, nf / 8, dx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// dx[j][f] = sum over the out-edges j -> i (cached CSC, rows ascending) of
// dout[i][f] where arg[i][f] == j: the SpMM transpose pass with each term
// masked by the winner, hubs chunked and merged in chunk order.  No atomics,
// so dx is the same bit for bit on every run; it reads the winners and dout
// rows once per edge instead of once per node.
cudaError_t launch_reduce_backward_ordered(const gnn_graph* g, const Shape& s, gnn_dtype dt,
                                           const int32_t* arg, const void* dout, void* dx,
                                           char* ws, cudaStream_t st) {
  return launch_spmm(g, s, dt, GNN_NORM_SUM, true, dout, dx, ws, st, arg);
}

}  // namespace gnn
