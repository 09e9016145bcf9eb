// Graph preparation, once per graph: validation, the cached CSC transpose and
// the degree buckets of both directions.
//
// The transpose is built by a stable least-significant-digit radix sort of
// the (source, destination) pairs on the source id: since the CSR lists edges
// by ascending destination, each CSC column comes out with its rows in
// ascending order, whatever the scheduling (integer counts only, no
// order-dependent atomics).  "On Efficient Scaling of GNNs via IO-Aware Layers
// Implementations", Technical Summary > Methodology: the transposed adjacency
// is precomputed once and cached for the backward pass; nodes are split into
// light and heavy by a degree threshold, heavy ones tiled over edge chunks.
#include <algorithm>

#include "device.cuh"

namespace gnn {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 16;
constexpr int kScanTile = kScanThreads * kScanItems;
constexpr int kSortWarps = 8;
constexpr int kSortSteps = 8;
constexpr int kSortTile = kSortWarps * kSortSteps * 32;  // 2048 edges per block

// Counters the host reads back at the end of prepare.
struct Counters {
  int32_t err;
  int32_t unsorted;  // some CSR row lists a source after a larger one
  int32_t pad[2];
  int32_t csr[8];  // light, mid, hubs, hub chunks, max degree
  int32_t csc[8];
};

unsigned grid_for(int64_t n, int threads, int64_t cap = 65536) {
  int64_t b = (n + threads - 1) / threads;
  return unsigned(std::max<int64_t>(1, std::min(b, cap)));
}

__global__ void k_validate(const int32_t* row_ptr, const int32_t* col, int64_t n, int64_t e,
                           int32_t* err) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t m = n + 1 > e ? n + 1 : e;
  for (int64_t x = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; x < m; x += stride) {
    if (x <= n) {
      const int32_t r = row_ptr[x];
      if ((x == 0 && r != 0) || (x == n && int64_t(r) != e) || (x < n && row_ptr[x + 1] < r))
        atomicOr(err, DEVERR_BAD_ROW_PTR);
    }
    if (x < e) {
      const int32_t c = col[x];
      if (c < 0 || int64_t(c) >= n) atomicOr(err, DEVERR_BAD_COL);
    }
  }
}

__global__ void k_out_degree(const int32_t* col, int64_t e, int32_t* deg) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t x = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; x < e; x += stride)
    atomicAdd(deg + col[x], 1);
}

// Flags a CSR row whose sources are not in non-decreasing order (rows[x]:
// the row of position x).
__global__ void k_row_order(const int32_t* rows, const int32_t* col, int64_t e, int32_t* flag) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t x = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; x + 1 < e; x += stride)
    if (rows[x] == rows[x + 1] && col[x] > col[x + 1]) atomicOr(flag, 1);
}

// row id of every CSR position: the last r with row_ptr[r] <= x
__global__ void k_expand_rows(const int32_t* row_ptr, int64_t n, int64_t e, int32_t* rows) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t x = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; x < e; x += stride) {
    int64_t lo = 0, hi = n;  // row_ptr[lo] <= x < row_ptr[hi]
    while (hi - lo > 1) {
      const int64_t mid = (lo + hi) >> 1;
      if (row_ptr[mid] <= x)
        lo = mid;
      else
        hi = mid;
    }
    rows[x] = int32_t(lo);
  }
}

// ---- exclusive scan of int32 (reduce, scan partials, apply) ----------------

__device__ __forceinline__ int32_t block_excl_scan(int32_t v, int32_t* total) {
  __shared__ int32_t warp_tot[kScanThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[wid] = inc;
  __syncthreads();
  int32_t base = 0, all = 0;
  for (int w = 0; w < kScanThreads / 32; ++w) {
    if (w < wid) base += warp_tot[w];
    all += warp_tot[w];
  }
  __syncthreads();
  *total = all;
  return base + inc - v;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(const int32_t* in, int64_t n,
                                                              int32_t* partial) {
  const int64_t base = int64_t(blockIdx.x) * kScanTile + threadIdx.x * kScanItems;
  int32_t s = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k)
    if (base + k < n) s += in[base + k];
  int32_t tot;
  block_excl_scan(s, &tot);
  if (threadIdx.x == 0) partial[blockIdx.x] = tot;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_partials(int32_t* partial, int64_t nb,
                                                                int32_t* total) {
  int32_t carry = 0;
  for (int64_t off = 0; off < nb; off += kScanThreads) {
    const int64_t x = off + threadIdx.x;
    const int32_t v = x < nb ? partial[x] : 0;
    int32_t tot;
    const int32_t ex = block_excl_scan(v, &tot);
    if (x < nb) partial[x] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0 && total) *total = carry;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_apply(const int32_t* in, int32_t* out,
                                                             int64_t n, const int32_t* partial) {
  const int64_t base = int64_t(blockIdx.x) * kScanTile + threadIdx.x * kScanItems;
  int32_t v[kScanItems];
  int32_t s = 0;
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    v[k] = base + k < n ? in[base + k] : 0;
    s += v[k];
  }
  int32_t tot;
  int32_t run = block_excl_scan(s, &tot) + partial[blockIdx.x];
#pragma unroll
  for (int k = 0; k < kScanItems; ++k) {
    if (base + k < n) out[base + k] = run;
    run += v[k];
  }
}

cudaError_t scan_excl(const int32_t* in, int32_t* out, int64_t n, int32_t* total,
                      int32_t* partial, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t nb = (n + kScanTile - 1) / kScanTile;
  k_scan_reduce<<<unsigned(nb), kScanThreads, 0, st>>>(in, n, partial);
  k_scan_partials<<<1, kScanThreads, 0, st>>>(partial, nb, total);
  k_scan_apply<<<unsigned(nb), kScanThreads, 0, st>>>(in, out, n, partial);
  return cudaGetLastError();
}

// ---- stable LSD radix sort pass (8-bit digits) ----------------------------

__global__ void __launch_bounds__(kSortWarps * 32) k_radix_hist(const int32_t* keys, int64_t e,
                                                                int shift, int32_t* hist,
                                                                int64_t nb) {
  __shared__ int32_t h[256];
  h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = int64_t(blockIdx.x) * kSortTile;
  for (int x = threadIdx.x; x < kSortTile; x += blockDim.x)
    if (base + x < e) atomicAdd(&h[(uint32_t(keys[base + x]) >> shift) & 255u], 1);
  __syncthreads();
  hist[int64_t(threadIdx.x) * nb + blockIdx.x] = h[threadIdx.x];
}

// hist holds, after the exclusive scan, the first output position of each
// (digit, block).  Within a block, warp w owns elements [w*256, w*256 + 256)
// of the tile; ranks among equal digits follow element order, so the pass is
// stable.
__global__ void __launch_bounds__(kSortWarps * 32) k_radix_scatter(
    const int32_t* kin, const int32_t* vin, int32_t* kout, int32_t* vout, int64_t e, int shift,
    const int32_t* hist, int64_t nb) {
  __shared__ int32_t cnt[kSortWarps][256];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int x = threadIdx.x; x < kSortWarps * 256; x += blockDim.x) (&cnt[0][0])[x] = 0;
  __syncthreads();
  const int64_t wbase = int64_t(blockIdx.x) * kSortTile + wid * (kSortSteps * 32);
#pragma unroll
  for (int s = 0; s < kSortSteps; ++s) {
    const int64_t x = wbase + s * 32 + lane;
    if (x < e) atomicAdd(&cnt[wid][(uint32_t(kin[x]) >> shift) & 255u], 1);
  }
  __syncthreads();
  {
    const int d = threadIdx.x;  // one thread per digit
    int32_t run = hist[int64_t(d) * nb + blockIdx.x];
    for (int w = 0; w < kSortWarps; ++w) {
      const int32_t c = cnt[w][d];
      cnt[w][d] = run;
      run += c;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll 1
  for (int s = 0; s < kSortSteps; ++s) {
    const int64_t x = wbase + s * 32 + lane;
    const bool in = x < e;
    const int32_t key = in ? kin[x] : 0;
    const int32_t val = in ? vin[x] : 0;
    const unsigned d = in ? ((uint32_t(key) >> shift) & 255u) : 256u;
    const unsigned peers = __match_any_sync(kFull, d);
    const int rank = __popc(peers & lt);
    const int32_t pos = in ? cnt[wid][d] + rank : 0;
    __syncwarp();
    if (in && rank == 0) cnt[wid][d] += __popc(peers);
    __syncwarp();
    if (in) {
      if (kout) kout[pos] = key;
      vout[pos] = val;
    }
  }
}

// ---- degree buckets -------------------------------------------------------

// Also writes the key and value arrays of the light-list sort: light nodes
// get key light_max_deg - degree (descending degree first), every other node
// light_max_deg + 1 (after all light nodes); the value is the node id.
__global__ void k_classify(const int32_t* ptr, int64_t n, gnn_tiling t, int32_t* f_light,
                           int32_t* f_mid, int32_t* f_hub, int32_t* f_chunks, int32_t* max_deg,
                           int32_t* light_key, int32_t* light_id) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  int32_t mx = 0;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < n; v += stride) {
    const int32_t d = ptr[v + 1] - ptr[v];
    mx = max(mx, d);
    const bool light = d <= t.light_max_deg;
    const bool mid = !light && d <= t.cta_max_deg;
    const bool hub = !light && !mid;
    light_key[v] = light ? t.light_max_deg - d : t.light_max_deg + 1;
    light_id[v] = int32_t(v);
    f_light[v] = light;
    f_mid[v] = mid;
    f_hub[v] = hub;
    f_chunks[v] = hub ? (d + t.hub_chunk - 1) / t.hub_chunk : 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(kFull, mx, o));
  if ((threadIdx.x & 31) == 0) atomicMax(max_deg, mx);
}

// After the scans f_* hold each node's position in its bucket list.  The
// light list is written by the sort instead.
__global__ void k_fill_buckets(const int32_t* ptr, int64_t n, gnn_tiling t,
                               const int32_t* p_mid, const int32_t* p_hub,
                               const int32_t* p_chunk, const int32_t* n_chunks_total,
                               int4* items, int4* hubs) {
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int32_t nch_total = *n_chunks_total;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < n; v += stride) {
    const int32_t b = ptr[v], e = ptr[v + 1], d = e - b;
    if (d <= t.light_max_deg) {
      // light: placed by the degree sort
    } else if (d <= t.cta_max_deg) {
      items[nch_total + p_mid[v]] = make_int4(int32_t(v), b, e, -1);
    } else {
      const int32_t first = p_chunk[v];
      const int32_t nch = (d + t.hub_chunk - 1) / t.hub_chunk;
      hubs[p_hub[v]] = make_int4(int32_t(v), first, nch, 0);
      for (int32_t c = 0; c < nch; ++c) {
        const int32_t cb = b + c * t.hub_chunk;
        items[first + c] = make_int4(int32_t(v), cb, min(e, cb + t.hub_chunk), first + c);
      }
    }
  }
}

// Sequential 256-byte-aligned sub-allocation of a caller-owned buffer (or,
// with base 0, just the byte count).
struct Carve {
  uintptr_t base;
  size_t off;
  size_t cap;
  template <typename T>
  T* take(int64_t count) {
    T* r = reinterpret_cast<T*>(base + off);
    off += align_up(size_t(std::max<int64_t>(count, 1)) * sizeof(T), 256);
    return r;
  }
  bool ok() const { return off <= cap; }
};

int64_t cap_items(int64_t n, int64_t e, const gnn_tiling& t) {
  return std::min<int64_t>(n, e / (int64_t(t.light_max_deg) + 1)) + e / t.hub_chunk + 1;
}
int64_t cap_hubs(int64_t n, int64_t e, const gnn_tiling& t) {
  return std::min<int64_t>(n, e / (int64_t(t.cta_max_deg) + 1)) + 1;
}

struct DirBuffers {
  int32_t* light;
  int4* items;
  int4* hubs;
};

DirBuffers carve_dir(Carve& c, int64_t n, int64_t e, const gnn_tiling& t) {
  DirBuffers d;
  d.light = c.take<int32_t>(n);
  d.items = c.take<int4>(cap_items(n, e, t));
  d.hubs = c.take<int4>(cap_hubs(n, e, t));
  return d;
}

struct ScratchBuffers {
  int32_t *f_light, *f_mid, *f_hub, *f_chunk, *outdeg;
  int32_t *k1, *v1, *k2, *v2;
  int32_t *hist, *partial, *totals;
};

int64_t sort_blocks(int64_t e) { return std::max<int64_t>(1, (e + kSortTile - 1) / kSortTile); }

ScratchBuffers carve_scratch(Carve& c, int64_t n, int64_t e) {
  ScratchBuffers s;
  s.f_light = c.take<int32_t>(n + 1);
  s.f_mid = c.take<int32_t>(n + 1);
  s.f_hub = c.take<int32_t>(n + 1);
  s.f_chunk = c.take<int32_t>(n + 1);
  s.outdeg = c.take<int32_t>(n + 1);
  // sort buffers serve the CSC sort (e pairs) and the light-list sort (n pairs)
  const int64_t m = std::max(n, e);
  s.k1 = c.take<int32_t>(m);
  s.v1 = c.take<int32_t>(m);
  s.k2 = c.take<int32_t>(m);
  s.v2 = c.take<int32_t>(m);
  const int64_t hist_n = 256 * sort_blocks(m);
  s.hist = c.take<int32_t>(hist_n);
  s.partial = c.take<int32_t>((std::max(hist_n, n + 1) + kScanTile - 1) / kScanTile + 1);
  s.totals = c.take<int32_t>(16);
  return s;
}

// Stable LSD radix sort of m (key, value) pairs on the low `bits` bits of the
// keys (8 bits per pass); the sorted values go to vout.  Intermediate passes
// use s.k1/v1 then s.k2/v2 alternately, so kin and vin must not be s.k1 or
// s.v1.
cudaError_t radix_sort_pairs(const int32_t* kin, const int32_t* vin, int64_t m, int bits,
                             int32_t* vout, const ScratchBuffers& s, cudaStream_t st) {
  const int passes = std::max(1, (bits + 7) / 8);
  const int64_t nb = sort_blocks(m);
  int32_t* kb[2] = {s.k1, s.k2};
  int32_t* vb[2] = {s.v1, s.v2};
  cudaError_t e;
  for (int p = 0; p < passes; ++p) {
    const bool last = p == passes - 1;
    int32_t* ko = last ? nullptr : kb[p & 1];
    int32_t* vo = last ? vout : vb[p & 1];
    k_radix_hist<<<unsigned(nb), kSortWarps * 32, 0, st>>>(kin, m, 8 * p, s.hist, nb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = scan_excl(s.hist, s.hist, 256 * nb, s.totals + 1, s.partial, st)) != cudaSuccess)
      return e;
    k_radix_scatter<<<unsigned(nb), kSortWarps * 32, 0, st>>>(kin, vin, ko, vo, m, 8 * p, s.hist,
                                                              nb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kin = ko;
    vin = vo;
  }
  return cudaSuccess;
}

cudaError_t build_buckets(const int32_t* ptr, int64_t n, const gnn_tiling& t,
                          const DirBuffers& d, const ScratchBuffers& s, int32_t* counters,
                          cudaStream_t st) {
  // counters: [0] light [1] mid [2] hubs [3] hub chunks [4] max degree
  cudaError_t e;
  if (n == 0) return cudaSuccess;
  k_classify<<<grid_for(n, 256), 256, 0, st>>>(ptr, n, t, s.f_light, s.f_mid, s.f_hub,
                                                s.f_chunk, counters + 4, s.k2, s.v2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = scan_excl(s.f_light, s.f_light, n, counters + 0, s.partial, st)) != cudaSuccess) return e;
  if ((e = scan_excl(s.f_mid, s.f_mid, n, counters + 1, s.partial, st)) != cudaSuccess) return e;
  if ((e = scan_excl(s.f_hub, s.f_hub, n, counters + 2, s.partial, st)) != cudaSuccess) return e;
  if ((e = scan_excl(s.f_chunk, s.f_chunk, n, counters + 3, s.partial, st)) != cudaSuccess) return e;
  k_fill_buckets<<<grid_for(n, 256), 256, 0, st>>>(ptr, n, t, s.f_mid, s.f_hub, s.f_chunk,
                                                   counters + 3, d.items, d.hubs);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // light list: light nodes by descending degree, ties by ascending id (the
  // sort is stable), so that the nodes a warp takes at once have nearly the
  // same number of edges; the non-light nodes sorted after them fill the
  // rest of the n-entry array and are never read
  int bits = 1;
  while ((int64_t(1) << bits) <= int64_t(t.light_max_deg) + 1) ++bits;
  return radix_sort_pairs(s.k2, s.v2, n, bits, d.light, s, st);
}

}  // namespace

size_t graph_buffer_bytes(int64_t n, int64_t e, const gnn_tiling& t) {
  Carve c{0, 0, 0};
  c.take<Counters>(1);
  c.take<int32_t>(n + 1);  // col_ptr
  c.take<int32_t>(e);      // row_idx
  carve_dir(c, n, e, t);
  carve_dir(c, n, e, t);
  return c.off;
}

size_t graph_scratch_bytes(int64_t n, int64_t e) {
  Carve c{0, 0, 0};
  carve_scratch(c, n, e);
  return c.off;
}

gnn_status prepare_graph(gnn_graph* g, const int32_t* row_ptr, const int32_t* col,
                         char* buffer, size_t buffer_bytes, char* scratch, size_t scratch_bytes,
                         cudaStream_t st) {
  const int64_t n = g->n, e = g->e;
  const gnn_tiling t = g->tiling;
  Carve cb{reinterpret_cast<uintptr_t>(buffer), 0, buffer_bytes};
  Counters* cnt = cb.take<Counters>(1);
  int32_t* col_ptr = cb.take<int32_t>(n + 1);
  int32_t* row_idx = cb.take<int32_t>(e);
  DirBuffers dcsr = carve_dir(cb, n, e, t);
  DirBuffers dcsc = carve_dir(cb, n, e, t);
  Carve cs{reinterpret_cast<uintptr_t>(scratch), 0, scratch_bytes};
  ScratchBuffers s = carve_scratch(cs, n, e);
  if (!cb.ok() || !cs.ok()) return GNN_ERR_WORKSPACE_TOO_SMALL;

  Counters host{};
  auto cuda_fail = [](cudaError_t x) { return x != cudaSuccess; };
  if (cuda_fail(cudaMemsetAsync(cnt, 0, sizeof(Counters), st))) return GNN_ERR_CUDA;
  k_validate<<<grid_for(std::max(n + 1, e), 256), 256, 0, st>>>(row_ptr, col, n, e, &cnt->err);
  if (cuda_fail(cudaGetLastError())) return GNN_ERR_CUDA;
  if (cuda_fail(cudaMemcpyAsync(&host.err, &cnt->err, sizeof(int32_t), cudaMemcpyDeviceToHost, st)) ||
      cuda_fail(cudaStreamSynchronize(st)))
    return GNN_ERR_CUDA;
  if (host.err & (DEVERR_BAD_ROW_PTR | DEVERR_BAD_COL)) return GNN_ERR_INVALID_GRAPH;

  // CSC column pointers: exclusive scan of the out-degrees
  if (cuda_fail(cudaMemsetAsync(s.outdeg, 0, sizeof(int32_t) * (n + 1), st))) return GNN_ERR_CUDA;
  if (e > 0) {
    k_out_degree<<<grid_for(e, 256), 256, 0, st>>>(col, e, s.outdeg);
    if (cuda_fail(cudaGetLastError())) return GNN_ERR_CUDA;
  }
  if (cuda_fail(scan_excl(s.outdeg, col_ptr, n + 1, s.totals, s.partial, st))) return GNN_ERR_CUDA;

  // CSC row lists: stable radix sort of the CSR positions by source id
  if (e > 0) {
    int bits = 0;
    while (bits < 31 && (int64_t(1) << bits) < n) ++bits;
    int32_t* v0 = s.k2;  // row id per CSR position; consumed by pass 0
    k_expand_rows<<<grid_for(e, 256), 256, 0, st>>>(row_ptr, n, e, v0);
    if (cuda_fail(cudaGetLastError())) return GNN_ERR_CUDA;
    k_row_order<<<grid_for(e, 256), 256, 0, st>>>(v0, col, e, &cnt->unsorted);
    if (cuda_fail(cudaGetLastError())) return GNN_ERR_CUDA;
    if (cuda_fail(radix_sort_pairs(col, v0, e, bits, row_idx, s, st))) return GNN_ERR_CUDA;
  }

  // degree buckets of both directions
  if (cuda_fail(build_buckets(row_ptr, n, t, dcsr, s, cnt->csr, st))) return GNN_ERR_CUDA;
  if (cuda_fail(build_buckets(col_ptr, n, t, dcsc, s, cnt->csc, st))) return GNN_ERR_CUDA;
  if (cuda_fail(cudaMemcpyAsync(&host, cnt, sizeof(Counters), cudaMemcpyDeviceToHost, st)) ||
      cuda_fail(cudaStreamSynchronize(st)))
    return GNN_ERR_CUDA;

  g->err = &cnt->err;
  g->csr_sorted = host.unsorted == 0;
  auto fill = [&](Dir& d, const int32_t* ptr, const int32_t* idx, const DirBuffers& b,
                  const int32_t* c) {
    d.ptr = ptr;
    d.idx = idx;
    d.light = b.light;
    d.items = b.items;
    d.hubs = b.hubs;
    d.n_light = c[0];
    d.n_items = int64_t(c[1]) + c[3];
    d.n_hubs = c[2];
    d.n_hub_chunks = c[3];
    d.max_deg = c[4];
    d.max_item = d.n_items > 0 ? std::min(d.max_deg, std::max(t.cta_max_deg, t.hub_chunk)) : 0;
  };
  fill(g->csr, row_ptr, col, dcsr, host.csr);
  fill(g->csc, col_ptr, row_idx, dcsc, host.csc);
  if (g->csr.n_light + g->csr.n_items - g->csr.n_hub_chunks + g->csr.n_hubs != n ||
      g->csc.n_light + g->csc.n_items - g->csc.n_hub_chunks + g->csc.n_hubs != n)
    return GNN_ERR_DEVICE_ASSERT;
  return GNN_OK;
}

}  // namespace gnn
