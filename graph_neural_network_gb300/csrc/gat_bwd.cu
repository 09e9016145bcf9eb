// Backward pass of the fused GAT neighbour aggregation.
//
// alpha is never stored: both passes recompute it from the per-node
// log-sum-exp the forward pass kept ("On Efficient Scaling of GNNs via
// IO-Aware Layers Implementations", Technical Summary > Methodology,
// attention-based layers, backward: compact per-node statistics instead of
// edge weights, attention recomputed on the fly).  With da_ij = dout_i . h_j,
// Delta_i = sum_j alpha_ij da_ij, dz_ij = alpha_ij (da_ij - Delta_i) g_ij and
// g_ij the LeakyReLU slope factor:
//
//   pass 1, destination side, over the CSR (one streaming pass per node):
//     SA = sum alpha da g,  SB = sum alpha g,  SD = sum alpha da = Delta_i,
//     ds_dst(i) = SA - Delta_i SB = sum_j dz_ij
//     -> per-node record {s_dst (base 2), lse (base 2), Delta, ds_dst} per head
//   pass 2, source side, over the cached CSC transpose (same page, SpMM
//   bullet: transposed adjacency cached for the backward pass):
//     dh_j = sum_i alpha_ij dout_i + ds_src(j) a_src + ds_dst(j) a_dst,
//     ds_src(j) = sum_i dz_ij, gathering dout_i and i's record per edge
//   da_src = sum_j ds_src(j) h_j, da_dst = sum_i ds_dst(i) h_i: per-block
//     partial sums, then a fixed-order float64 sum over blocks.
//
// Both passes use the same degree-aware tiling as the forward pass (warp per
// light node, block per mid node, chunked hubs with fixed-order merges), over
// in-degrees for pass 1 and out-degrees for pass 2.
#include "device.cuh"

namespace gnn {
namespace {

struct DirArgs {
  const int32_t* ptr;
  const int32_t* idx;
  const int32_t* light;
  int64_t n_light;
  const int4* items;
  int64_t n_items;
  const int4* hubs;
  int64_t n_hubs;
  int col_off;  // bytes of shared memory before the per-warp partials
};

struct BwdArgs {
  Shape s;
  DirArgs csr, csc;
  int64_t n;
  const void* h;
  const float* a_src;
  const float* a_dst;
  const float* ssrc;  // [N][H] base-2 a_src . h_n (pre-pass)
  const float* sdst;  // [N][H] base-2 a_dst . h_n (pre-pass)
  float slope;
  const float* lse;
  const void* dout;
  void* dh;
  float* da_src;
  float* da_dst;
  float4* stats;     // [N][H] {s_dst2, lse2, Delta, ds_dst}
  float* ds_src;     // [N][H]
  float4* dst_part;  // [CSR hub chunks][H] {SA, SB, SD, s_dst2}
  float* src_acc;    // [CSC hub chunks][H * D]
  float* src_sum;    // [CSC hub chunks][H]
  double* da_part;   // [da blocks][2][H * D]
  int da_blocks;
  int* ctr;          // work counters: [0], [1] pass 1 items / light; [2], [3] pass 2
  int32_t* err;
};

constexpr int kGrab = 4;  // light nodes a warp takes per counter access

__device__ __forceinline__ float leaky(float z, float slope) { return z > 0.f ? z : slope * z; }
__device__ __forceinline__ float leaky_grad(float z, float slope) { return z > 0.f ? 1.f : slope; }

// ---------------------------------------------------------------------------
// pass 1: destination side (CSR)
// ---------------------------------------------------------------------------

// Batches of kUnroll edges per lane: the batch at `base` holds edges
// base + sg + u * SG, the next one starts `step` edges further; until end
// (kFixed false) or in exactly `trips` batches (kFixed true; the same count
// on every lane of the warp, batches past end add nothing).
template <typename T, int NV, int VB, bool kFixed>
__device__ __forceinline__ void dst_edges(const BwdArgs& A, const Lane<NV>& L,
                                          const int32_t* cols, int colbase, int beg, int end,
                                          int sg, int SG, int step, int trips,
                                          int (&jn)[UnrollOf<VB>::value],
                                          const OwnVec<T, VB> (&gi)[NV],
                                          const float (&sd2)[NV], const float (&lse2)[NV],
                                          float (&SA)[NV], float (&SB)[NV], float (&SD)[NV]) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = UnrollOf<VB>::value;
  const int H = A.s.H;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int j[U];
#pragma unroll
    for (int u = 0; u < U; ++u) j[u] = jn[u];
    RawV<VB> raw[U][NV];
    float ss[U * NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const bool ok = j[u] >= 0 && L.ok[v];
        raw[u][v] = ok ? ldv<VB>(row_at<VB>(A.h, j[u], A.s.rv) + VB * L.q[v]) : zero_raw<VB>();
        ss[u * NV + v] = ok ? __ldg(A.ssrc + int64_t(j[u]) * H + L.k[v]) : 0.f;
      }
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, jn);
    float dd[U * NV];  // dout_i . h_j per head
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        dd[u * NV + v] = gi[v].dot_with(raw[u][v]);
      }
    head_sums<U * NV>(dd, A.s.hv_log2);
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float z = sd2[v] + ss[u * NV + v];
        const float da = dd[u * NV + v];
        const float al = j[u] >= 0 ? ex2(leaky(z, A.slope) - lse2[v]) : 0.f;
        const float g = leaky_grad(z, A.slope);
        const float ad = al * da;
        SA[v] = fmaf(ad, g, SA[v]);
        SB[v] = fmaf(al, g, SB[v]);
        SD[v] += ad;
      }
  }
}

// Destination-side sums of node i over its edges [beg, end).  split: the
// edges are spread over the warp's sub-groups (beg + g, beg + g + G, ...)
// and the sums added over them; otherwise this lane's sub-group takes them
// all in `trips` batches.  jn: sources of the first batch.
template <typename T, int NV, int VB>
__device__ __forceinline__ void dst_node(const BwdArgs& A, const Lane<NV>& L, int i,
                                         const int32_t* cols, int colbase, int beg, int end,
                                         bool split, int step, int trips,
                                         int (&jn)[UnrollOf<VB>::value], float (&sd2)[NV],
                                         float (&lse2)[NV], float (&SA)[NV], float (&SB)[NV],
                                         float (&SD)[NV]) {
  constexpr int U = UnrollOf<VB>::value;
  OwnVec<T, VB> gi[NV];
  {
    const char* row = row_at<VB>(A.dout, i, A.s.rv);
#pragma unroll
    for (int v = 0; v < NV; ++v) gi[v].set(L.ok[v] ? ldv<VB>(row + VB * L.q[v]) : zero_raw<VB>());
  }
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    sd2[v] = L.ok[v] ? __ldg(A.sdst + int64_t(i) * A.s.H + L.k[v]) : 0.f;
    lse2[v] = L.ok[v] ? A.lse[int64_t(i) * A.s.H + L.k[v]] * kLog2e : 0.f;
    SA[v] = SB[v] = SD[v] = 0.f;
  }
  if (split) {
    dst_edges<T, NV, VB, false>(A, L, cols, colbase, beg, end, L.g, L.G, step, 0, jn, gi, sd2,
                                lse2, SA, SB, SD);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      SA[v] = subgroup_sum(SA[v], A.s);
      SB[v] = subgroup_sum(SB[v], A.s);
      SD[v] = subgroup_sum(SD[v], A.s);
    }
  } else {
    dst_edges<T, NV, VB, true>(A, L, cols, colbase, beg, end, 0, 1, U, trips, jn, gi, sd2, lse2,
                               SA, SB, SD);
  }
}

// kSub: light nodes take one sub-group each (rows narrower than a warp);
// otherwise one warp each.
template <typename T, int NV, int VB, bool kSub>
__global__ void __launch_bounds__(kThreads, MinBlocksLean<NV>::value) bwd_dst_main(const BwdArgs A) {
  constexpr int U = UnrollOf<VB>::value;
  const DirArgs& D = A.csr;
  const Lane<NV> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int H = A.s.H;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  float sd2[NV], lse2[NV], SA[NV], SB[NV], SD[NV];

  // ---- block items -------------------------------------------------------
  if (D.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    float* wp = reinterpret_cast<float*>(smem + D.col_off);  // [kWarps][H][3]
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 0, 1);
      __syncthreads();
      const int idx = s_item;
      if (idx >= D.n_items) break;
      const int4 it = D.items[idx];
      if (!stage_edges(cols, D.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kUnroll * G edges dealt to the warps in turn
      const int batch = U * L.G;
      const int wb = it.y + wid * batch;
      int jn[U];
      batch_ids<U>(cols, it.y & ~3, wb, it.z, L.g, L.G, jn);
      dst_node<T, NV, VB>(A, L, it.x, cols, it.y & ~3, wb, it.z, true, kWarps * batch, 0, jn, sd2,
                          lse2, SA, SB, SD);
      if (L.g == 0)
#pragma unroll
        for (int v = 0; v < NV; ++v)
          if (L.head_leader(A.s, v)) {
            float* p = wp + (wid * H + L.k[v]) * 3;
            p[0] = SA[v];
            p[1] = SB[v];
            p[2] = SD[v];
          }
      __syncthreads();
      if (wid == 0 && L.g == 0) {
        // warp 0 folds the warps' partial sums in warp order
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          if (!L.head_leader(A.s, v)) continue;
          float a = 0.f, b = 0.f, d = 0.f;
          for (int w = 0; w < kWarps; ++w) {
            const float* p = wp + (w * H + L.k[v]) * 3;
            a += p[0];
            b += p[1];
            d += p[2];
          }
          if (it.w < 0)
            A.stats[int64_t(it.x) * H + L.k[v]] = make_float4(sd2[v], lse2[v], d, a - d * b);
          else
            A.dst_part[int64_t(it.w) * H + L.k[v]] = make_float4(a, b, d, sd2[v]);
        }
      }
      __syncthreads();  // shared memory is reused by the next item
    }
  }

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  if (kSub) {
    // nodes per sub-group per pull: four where a warp holds two sub-groups
    // (eight nodes per pull; measured 12 % faster than two on 512-byte rows),
    // two otherwise
    const int R = L.G >= 32 ? 1 : (L.G == 2 ? 4 : 2);
    const int npull = R * L.G;
    for (;;) {
      int t0 = 0;
      if (L.lane == 0) t0 = atomicAdd(A.ctr + 1, npull);
      t0 = __shfl_sync(kFull, t0, 0);
      if (t0 >= D.n_light) break;
      int my_i = -1, my_b = 0, my_e = 0;
      if (L.lane < npull && t0 + L.lane < D.n_light) {
        my_i = D.light[t0 + L.lane];
        my_b = D.ptr[my_i];
        my_e = D.ptr[my_i + 1];
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
        batch_ids<U>(D.idx, 0, beg, end, 0, 1, jn);
        dst_node<T, NV, VB>(A, L, i >= 0 ? i : 0, D.idx, 0, beg, end, false, 0, trips, jn, sd2, lse2,
                            SA, SB, SD);
        if (i >= 0)
#pragma unroll
          for (int v = 0; v < NV; ++v)
            if (L.head_leader(A.s, v))
              A.stats[int64_t(i) * H + L.k[v]] =
                  make_float4(sd2[v], lse2[v], SD[v], SA[v] - SD[v] * SB[v]);
      }
    }
    return;
  }

  // ---- light nodes, rows of a whole warp: one warp each ---------------------
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
    int jn[U];
    batch_ids<U>(D.idx, 0, beg, end, L.g, L.G, jn);
    for (int q = 0; q < kGrab && i >= 0; ++q) {
      const int nq = (q + 1) & (kGrab - 1);
      const int i2 = q + 1 < kGrab ? __shfl_sync(kFull, my_i, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int jn2[U];
      batch_ids<U>(D.idx, 0, b2, i2 >= 0 ? e2 : b2, L.g, L.G, jn2);
      dst_node<T, NV, VB>(A, L, i, D.idx, 0, beg, end, true, U * L.G, 0, jn, sd2, lse2, SA, SB,
                          SD);
      if (L.g == 0)
#pragma unroll
        for (int v = 0; v < NV; ++v)
          if (L.head_leader(A.s, v))
            A.stats[int64_t(i) * H + L.k[v]] =
                make_float4(sd2[v], lse2[v], SD[v], SA[v] - SD[v] * SB[v]);
      i = i2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < U; ++u) jn[u] = jn2[u];
    }
  }
}

template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) bwd_dst_merge(const BwdArgs A) {
  const Lane<NV> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.csr.n_hubs || L.g != 0) return;
  const int4 hb = A.csr.hubs[t];
  const int H = A.s.H;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!L.head_leader(A.s, v)) continue;
    float a = 0.f, b = 0.f, d = 0.f;
    for (int c = 0; c < hb.z; ++c) {
      const float4 p = A.dst_part[(int64_t(hb.y) + c) * H + L.k[v]];
      a += p.x;
      b += p.y;
      d += p.z;
    }
    const float sd2 = A.dst_part[int64_t(hb.y) * H + L.k[v]].w;
    const float lse2 = A.lse[int64_t(hb.x) * H + L.k[v]] * kLog2e;
    A.stats[int64_t(hb.x) * H + L.k[v]] = make_float4(sd2, lse2, d, a - d * b);
  }
}

// ---------------------------------------------------------------------------
// pass 2: source side (CSC)
// ---------------------------------------------------------------------------

// The source pass's own bf16 row with 32-byte lane vectors, kept in shared
// memory (each lane's 32 bytes in a slot of its own) and re-read per edge
// instead of held in 8 registers through the loop: at 4 blocks per SM the
// pass then spills far less (measured 6-9 % faster).  Only the owning lane
// writes and reads its slot, so no barrier is needed.
struct SmemOwn {
  uint32_t addr;  // this lane's first 16 bytes; the second 16 at addr + 512
  __device__ __forceinline__ void set(const RawV<32>& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.a.x), "r"(v.a.y),
                 "r"(v.a.z), "r"(v.a.w)
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr + 512), "r"(v.b.x),
                 "r"(v.b.y), "r"(v.b.z), "r"(v.b.w)
                 : "memory");
  }
  __device__ __forceinline__ float dot_with(const RawV<32>& g) const {
    RawV<32> r;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w)
                 : "r"(addr));
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.b.x), "=r"(r.b.y), "=r"(r.b.z), "=r"(r.b.w)
                 : "r"(addr + 512));
    return dot_bf16<32>(g, r);
  }
};
template <typename T, int VB>
struct SrcOwn {
  using type = OwnVec<T, VB>;
};
template <>
struct SrcOwn<__nv_bfloat16, 32> {
  using type = SmemOwn;
};
template <typename O>
__device__ __forceinline__ void own_init(O&, uint32_t) {}
__device__ __forceinline__ void own_init(SmemOwn& o, uint32_t base) {
  o.addr = base + (threadIdx.x & ~31) * 32 + (threadIdx.x & 31) * 16;
}

template <typename T, int NV, int VB, bool kFixed>
__device__ __forceinline__ void src_edges(const BwdArgs& A, const Lane<NV>& L,
                                          const int32_t* cols, int colbase, int beg, int end,
                                          int sg, int SG, int step, int trips,
                                          int (&in)[UnrollOf<VB>::value],
                                          const typename SrcOwn<T, VB>::type (&xj)[NV],
                                          const float (&ss2)[NV],
                                          float (&acc)[NV][ElemsOf<T, VB>::n], float (&SZ)[NV]) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = UnrollOf<VB>::value;
  const int H = A.s.H;
  int base = beg;
  for (int t = 0; kFixed ? t < trips : base < end; ++t, base += step) {
    int i[U];
#pragma unroll
    for (int u = 0; u < U; ++u) i[u] = in[u];
    RawV<VB> raw[U][NV];
    float3 st[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const bool ok = i[u] >= 0 && L.ok[v];
        raw[u][v] = ok ? ldv<VB>(row_at<VB>(A.dout, i[u], A.s.rv) + VB * L.q[v]) : zero_raw<VB>();
        st[u][v] = make_float3(0.f, 0.f, 0.f);
        if (ok)  // {s_dst, lse, Delta}; the record's ds_dst is not needed here
          asm("ld.global.nc.v4.f32 {%0, %1, %2, _}, [%3];"
              : "=f"(st[u][v].x), "=f"(st[u][v].y), "=f"(st[u][v].z)
              : "l"(A.stats + int64_t(i[u]) * H + L.k[v]));
      }
    if (kFixed ? t + 1 < trips : base + step < end)
      batch_ids<U>(cols, colbase, base + step, end, sg, SG, in);
    float dd[U * NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        dd[u * NV + v] = xj[v].dot_with(raw[u][v]);
      }
    head_sums<U * NV>(dd, A.s.hv_log2);
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const float da = dd[u * NV + v];
        const float z = st[u][v].x + ss2[v];
        const float al = i[u] >= 0 ? ex2(leaky(z, A.slope) - st[u][v].y) : 0.f;
        SZ[v] = fmaf(al * (da - st[u][v].z), leaky_grad(z, A.slope), SZ[v]);
        float g[V];
        unpack_altv<T, VB>(raw[u][v], g);
        axpy<V>(acc[v], al, g);
      }
  }
}

// Source-side sums of node j over its out-edges [beg, end) (in:
// destinations of the first batch).  split / trips as for dst_node.
template <typename T, int NV, int VB>
__device__ __forceinline__ void src_node(const BwdArgs& A, const Lane<NV>& L, int j,
                                         const int32_t* cols, int colbase, int beg, int end,
                                         bool split, int step, int trips,
                                         int (&in)[UnrollOf<VB>::value],
                                         float (&acc)[NV][ElemsOf<T, VB>::n], float (&SZ)[NV]) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = UnrollOf<VB>::value;
  static_assert(!(VB == 32 && sizeof(T) == 2) || NV == 1, "one own-row slot per lane");
  __shared__ __align__(16) uint4 s_own[kThreads * 2];
  typename SrcOwn<T, VB>::type xj[NV];
  float ss2[NV];
  {
#pragma unroll
    for (int v = 0; v < NV; ++v) own_init(xj[v], smem_u32(s_own));
    const char* row = row_at<VB>(A.h, j, A.s.rv);
#pragma unroll
    for (int v = 0; v < NV; ++v) xj[v].set(L.ok[v] ? ldv<VB>(row + VB * L.q[v]) : zero_raw<VB>());
  }
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    ss2[v] = L.ok[v] ? __ldg(A.ssrc + int64_t(j) * A.s.H + L.k[v]) : 0.f;
    SZ[v] = 0.f;
#pragma unroll
    for (int c = 0; c < V; ++c) acc[v][c] = 0.f;
  }
  if (split) {
    src_edges<T, NV, VB, false>(A, L, cols, colbase, beg, end, L.g, L.G, step, 0, in, xj, ss2,
                                acc, SZ);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      SZ[v] = subgroup_sum(SZ[v], A.s);
#pragma unroll
      for (int c = 0; c < V; ++c) acc[v][c] = subgroup_sum(acc[v][c], A.s);
    }
  } else {
    src_edges<T, NV, VB, true>(A, L, cols, colbase, beg, end, 0, 1, U, trips, in, xj, ss2, acc,
                               SZ);
  }
}

// dh_j = acc + ds_src a_src + ds_dst a_dst (natural units), ds_src(j) = SZ.
template <typename T, int NV, int VB>
__device__ __forceinline__ void write_src(const BwdArgs& A, const Lane<NV>& L, int64_t j,
                                          const float (&acc)[NV][ElemsOf<T, VB>::n],
                                          const float (&SZ)[NV]) {
  constexpr int V = ElemsOf<T, VB>::n;
  float as[NV][V], ad[NV][V];
  load_att_v<T, NV, VB>(A.a_src, L, 1.f, as);
  load_att_v<T, NV, VB>(A.a_dst, L, 1.f, ad);
  char* orow = reinterpret_cast<char*>(A.dh) + j * int64_t(A.s.rv) * VB;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!L.ok[v]) continue;
    const float dsd = A.stats[j * A.s.H + L.k[v]].w;
    float x[V];
#pragma unroll
    for (int c = 0; c < V; ++c) x[c] = fmaf(dsd, ad[v][c], fmaf(SZ[v], as[v][c], acc[v][c]));
    storev<T, VB>(orow + VB * L.q[v], x);
    if (L.head_leader(A.s, v)) A.ds_src[j * A.s.H + L.k[v]] = SZ[v];
  }
}

// With 32-byte lane vectors the source pass runs 4 blocks per SM (64
// registers and a few spilled bytes), which measured 6-8 % faster than 3
// blocks without spills; with 16-byte vectors it runs 3.
template <int NV, int VB>
struct SrcBlocks {
  static constexpr int value = VB == 32 ? 4 : MinBlocks<NV>::value;
};

template <typename T, int NV, int VB, bool kSub>
__global__ void __launch_bounds__(kThreads, SrcBlocks<NV, VB>::value) bwd_src_main(const BwdArgs A) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = UnrollOf<VB>::value;
  const DirArgs& D = A.csc;
  const Lane<NV> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int H = A.s.H;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_item;
  float acc[NV][V], SZ[NV];

  // ---- block items -------------------------------------------------------
  if (D.n_items > 0) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cols = reinterpret_cast<int32_t*>(smem + 16);
    const int row_f = A.s.rv * V;
    float* wsum = reinterpret_cast<float*>(smem + D.col_off);  // [kWarps][H]
    float* wacc = wsum + kWarps * H;                            // [kWarps][H * D]
    uint32_t parity = 0;
    if (threadIdx.x == 0) mbar_init(bar, 1);
    for (;;) {
      if (threadIdx.x == 0) s_item = atomicAdd(A.ctr + 2, 1);
      __syncthreads();
      const int idx = s_item;
      if (idx >= D.n_items) break;
      const int4 it = D.items[idx];
      if (!stage_edges(cols, D.idx, it.y, it.z, bar, parity, A.err)) return;
      // batches of kUnroll * G edges dealt to the warps in turn
      const int batch = U * L.G;
      const int wb = it.y + wid * batch;
      int in[U];
      batch_ids<U>(cols, it.y & ~3, wb, it.z, L.g, L.G, in);
      src_node<T, NV, VB>(A, L, it.x, cols, it.y & ~3, wb, it.z, true, kWarps * batch, 0, in, acc,
                          SZ);
      if (L.g == 0)
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          if (!L.ok[v]) continue;
#pragma unroll
          for (int c = 0; c < V; ++c) wacc[wid * row_f + L.q[v] * V + c] = acc[v][c];
          if (L.head_leader(A.s, v)) wsum[wid * H + L.k[v]] = SZ[v];
        }
      __syncthreads();
      if (wid == 0 && L.g == 0) {
        // warp 0 folds the warps' partial sums in warp order
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          SZ[v] = 0.f;
#pragma unroll
          for (int c = 0; c < V; ++c) acc[v][c] = 0.f;
          if (!L.ok[v]) continue;
          for (int w = 0; w < kWarps; ++w) {
            SZ[v] += wsum[w * H + L.k[v]];
#pragma unroll
            for (int c = 0; c < V; ++c) acc[v][c] += wacc[w * row_f + L.q[v] * V + c];
          }
        }
        if (it.w < 0) {
          write_src<T, NV, VB>(A, L, it.x, acc, SZ);
        } else {
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            if (!L.ok[v]) continue;
            float* pa = A.src_acc + int64_t(it.w) * row_f + L.q[v] * V;
#pragma unroll
            for (int c4 = 0; c4 < V; c4 += 4)
              *reinterpret_cast<float4*>(pa + c4) =
                  make_float4(acc[v][c4], acc[v][c4 + 1], acc[v][c4 + 2], acc[v][c4 + 3]);
            if (L.head_leader(A.s, v)) A.src_sum[int64_t(it.w) * H + L.k[v]] = SZ[v];
          }
        }
      }
      __syncthreads();  // shared memory is reused by the next item
    }
  }

  // ---- light nodes, rows narrower than a warp: one sub-group each --------
  if (kSub) {
    const int R = L.G >= 32 ? 1 : 2;
    const int npull = R * L.G;
    for (;;) {
      int t0 = 0;
      if (L.lane == 0) t0 = atomicAdd(A.ctr + 3, npull);
      t0 = __shfl_sync(kFull, t0, 0);
      if (t0 >= D.n_light) break;
      for (int r = 0; r < R; ++r) {
        // each sub-group reads its node's entry itself (the same address on
        // all its lanes) instead of keeping the pull's entries in registers
        const int64_t t = int64_t(t0) + r * L.G + L.g;
        const int j = t < D.n_light ? __ldg(D.light + t) : -1;
        const int beg = j >= 0 ? __ldg(D.ptr + j) : 0;
        const int end = j >= 0 ? __ldg(D.ptr + j + 1) : beg;
        if (!__any_sync(kFull, j >= 0)) break;
        int trips = (end - beg + U - 1) / U;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) trips = max(trips, __shfl_xor_sync(kFull, trips, o));
        int in[U];
        batch_ids<U>(D.idx, 0, beg, end, 0, 1, in);
        src_node<T, NV, VB>(A, L, j >= 0 ? j : 0, D.idx, 0, beg, end, false, 0, trips, in, acc, SZ);
        if (j >= 0) write_src<T, NV, VB>(A, L, j, acc, SZ);
      }
    }
    return;
  }

  // ---- light nodes, rows of a whole warp: one warp each ---------------------
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
    int in[U];
    batch_ids<U>(D.idx, 0, beg, end, L.g, L.G, in);
    for (int q = 0; q < kGrab && j >= 0; ++q) {
      const int nq = (q + 1) & (kGrab - 1);
      const int j2 = q + 1 < kGrab ? __shfl_sync(kFull, my_j, nq) : -1;
      const int b2 = __shfl_sync(kFull, my_b, nq);
      const int e2 = __shfl_sync(kFull, my_e, nq);
      int in2[U];
      batch_ids<U>(D.idx, 0, b2, j2 >= 0 ? e2 : b2, L.g, L.G, in2);
      src_node<T, NV, VB>(A, L, j, D.idx, 0, beg, end, true, U * L.G, 0, in, acc, SZ);
      if (L.g == 0) write_src<T, NV, VB>(A, L, j, acc, SZ);
      j = j2;
      beg = b2;
      end = e2;
#pragma unroll
      for (int u = 0; u < U; ++u) in[u] = in2[u];
    }
  }
}

template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) bwd_src_merge(const BwdArgs A) {
  constexpr int V = VecOf<T>::n;
  const Lane<NV> L(A.s);
  const int64_t t = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (t >= A.csc.n_hubs || L.g != 0) return;
  const int4 hb = A.csc.hubs[t];
  const int H = A.s.H;
  const int row_f = A.s.rv * V;
  float acc[NV][V], SZ[NV];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    SZ[v] = 0.f;
#pragma unroll
    for (int c = 0; c < V; ++c) acc[v][c] = 0.f;
    if (!L.ok[v]) continue;
    for (int c = 0; c < hb.z; ++c) {
      const int64_t slot = int64_t(hb.y) + c;
      SZ[v] += A.src_sum[slot * H + L.k[v]];
      const float* pa = A.src_acc + slot * row_f + L.q[v] * V;
#pragma unroll
      for (int c4 = 0; c4 < V; c4 += 4) {
        const float4 q = *reinterpret_cast<const float4*>(pa + c4);
        acc[v][c4] += q.x;
        acc[v][c4 + 1] += q.y;
        acc[v][c4 + 2] += q.z;
        acc[v][c4 + 3] += q.w;
      }
    }
  }
  write_src<T, NV, 16>(A, L, hb.x, acc, SZ);
}

// ---------------------------------------------------------------------------
// attention-vector gradients
// ---------------------------------------------------------------------------

// Block b sums ds_src(n) h_n and ds_dst(n) h_n over its nodes n = b, b + B,
// ... (per sub-group: every G-th of them, kDaRows rows in flight) in
// float32, then folds its warps' and sub-groups' sums in float64 in a fixed
// order into da_part[b].
constexpr int kDaRows = 4;

template <typename T, int NV>
__global__ void __launch_bounds__(kThreads) da_partial(const BwdArgs A) {
  constexpr int V = VecOf<T>::n;
  constexpr int U = kDaRows;
  const Lane<NV> L(A.s);
  const int wid = threadIdx.x >> 5;
  const int H = A.s.H;
  const int row_f = A.s.rv * V;
  float s_acc[NV][V], d_acc[NV][V];
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int c = 0; c < V; ++c) s_acc[v][c] = d_acc[v][c] = 0.f;
  const float* dsd = reinterpret_cast<const float*>(A.stats);  // .w of each record
  const int64_t stride = int64_t(A.da_blocks) * kWarps * L.G;
  for (int64_t n0 = (int64_t(blockIdx.x) * kWarps + wid) * L.G + L.g; n0 < A.n;
       n0 += U * stride) {
    uint4 raw[U][NV];
    float ds[U][NV], dd[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t n = n0 + u * stride;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        const bool ok = n < A.n && L.ok[v];
        raw[u][v] = ok ? ld16(row_base<T>(A.h, n, A.s.rv) + 16 * L.q[v]) : make_uint4(0, 0, 0, 0);
        ds[u][v] = ok ? __ldg(A.ds_src + n * H + L.k[v]) : 0.f;
        dd[u][v] = ok ? __ldg(dsd + (n * H + L.k[v]) * 4 + 3) : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float x[V];
        unpack<T>(raw[u][v], x);
        axpy<V>(s_acc[v], ds[u][v], x);
        axpy<V>(d_acc[v], dd[u][v], x);
      }
  }
  extern __shared__ __align__(16) unsigned char smem[];
  float* buf = reinterpret_cast<float*>(smem);  // [kWarps * G][2][row_f]
  const int sub = wid * L.G + L.g;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    if (!L.ok[v]) continue;
#pragma unroll
    for (int c = 0; c < V; ++c) {
      buf[(sub * 2 + 0) * row_f + L.q[v] * V + c] = s_acc[v][c];
      buf[(sub * 2 + 1) * row_f + L.q[v] * V + c] = d_acc[v][c];
    }
  }
  __syncthreads();
  const int nsub = kWarps * L.G;
  for (int t = threadIdx.x; t < 2 * row_f; t += blockDim.x) {
    const int which = t / row_f, e = t - which * row_f;
    double s = 0.0;
    for (int q = 0; q < nsub; ++q) s += double(buf[(q * 2 + which) * row_f + e]);
    A.da_part[int64_t(blockIdx.x) * 2 * row_f + t] = s;
  }
}

// One warp per output element: lane l sums the block partials l, l + 32, ...
// in order, then a fixed butterfly adds the 32 lane sums.
__global__ void __launch_bounds__(kThreads) da_final(const double* part, int blocks, int row_f,
                                                     float* da_src, float* da_dst) {
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= 2 * row_f) return;
  double s = 0.0;
#pragma unroll 8
  for (int b = lane; b < blocks; b += 32) s += part[int64_t(b) * 2 * row_f + t];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
  if (lane == 0) {
    if (t < row_f)
      da_src[t] = float(s);
    else
      da_dst[t - row_f] = float(s);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

// Launch a kernel template instantiated for the 16-byte lane geometry M.s.
template <typename T, template <typename, int> class K>
cudaError_t launch16(const BwdArgs& M, unsigned grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  switch (M.s.nv) {
    case 1: e = K<T, 1>::launch(M, grid, smem, st); break;
    case 2: e = K<T, 2>::launch(M, grid, smem, st); break;
    default: e = K<T, 4>::launch(M, grid, smem, st); break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, int NV>
struct DstMerge {
  static cudaError_t launch(const BwdArgs& M, unsigned grid, size_t, cudaStream_t st) {
    bwd_dst_merge<T, NV><<<grid, kThreads, 0, st>>>(M);
    return cudaSuccess;
  }
};
template <typename T, int NV>
struct SrcMerge {
  static cudaError_t launch(const BwdArgs& M, unsigned grid, size_t, cudaStream_t st) {
    bwd_src_merge<T, NV><<<grid, kThreads, 0, st>>>(M);
    return cudaSuccess;
  }
};
template <typename T, int NV>
struct DaPartial {
  static cudaError_t launch(const BwdArgs& M, unsigned grid, size_t smem, cudaStream_t st) {
    cudaError_t e = set_smem(da_partial<T, NV>, smem);
    if (e != cudaSuccess) return e;
    da_partial<T, NV><<<grid, kThreads, smem, st>>>(M);
    return cudaSuccess;
  }
};

// A.s is the lane geometry of the two main kernels (VB-byte lane vectors);
// s16 the one of 16-byte vectors, used by the score pre-pass, the hub merges
// and the attention-vector gradients.
template <typename T, int NV, int VB>
cudaError_t launch_t(const BwdArgs& A, const Shape& s16, gnn_dtype dt, int sm_count,
                     cudaStream_t st, const cudaEvent_t* ev, bool reuse_scores) {
  const int H = A.s.H, row_f = A.s.H * A.s.D;
  BwdArgs M = A;
  M.s = s16;
  cudaError_t e;
  auto mark = [&](int k) {
    if (ev) cudaEventRecord(ev[k], st);
  };
  if ((e = cudaMemsetAsync(A.ctr, 0, kCounters * sizeof(int), st)) != cudaSuccess) return e;
  // rows narrower than a warp: light nodes one sub-group each (NV = 1)
  const bool sub = NV == 1 && A.s.lpr < 32;
  mark(0);
  // the forward call left the same scores at the same place in ws
  if (!reuse_scores &&
      (e = launch_node_scores(s16, dt, A.h, A.a_src, A.a_dst, A.n, const_cast<float*>(A.ssrc),
                              const_cast<float*>(A.sdst), sm_count, st)) != cudaSuccess)
    return e;
  mark(1);
  // pass 1
  {
    const int64_t work = A.csr.n_items + (A.csr.n_light + kWarps * kGrab - 1) / (kWarps * kGrab);
    const size_t smem = size_t(A.csr.col_off) + size_t(kWarps) * H * 3 * 4;
    if (work > 0) {
      auto kernel = sub ? bwd_dst_main<T, NV, VB, NV == 1> : bwd_dst_main<T, NV, VB, false>;
      if ((e = set_smem(kernel, smem)) != cudaSuccess) return e;
      const int64_t cap = persistent_blocks(kernel, smem, sm_count);
      const int64_t blocks = work < cap ? work : cap;
      kernel<<<unsigned(blocks), kThreads, smem, st>>>(A);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    mark(2);
    if (A.csr.n_hubs > 0 &&
        (e = launch16<T, DstMerge>(M, unsigned((A.csr.n_hubs + kWarps - 1) / kWarps), 0, st)) !=
            cudaSuccess)
      return e;
    mark(3);
  }
  // pass 2
  {
    const int64_t work = A.csc.n_items + (A.csc.n_light + kWarps * kGrab - 1) / (kWarps * kGrab);
    const size_t smem = size_t(A.csc.col_off) + size_t(kWarps) * (H + row_f) * 4;
    if (work > 0) {
      auto kernel = sub ? bwd_src_main<T, NV, VB, NV == 1> : bwd_src_main<T, NV, VB, false>;
      if ((e = set_smem(kernel, smem)) != cudaSuccess) return e;
      const int64_t cap = persistent_blocks(kernel, smem, sm_count);
      const int64_t blocks = work < cap ? work : cap;
      kernel<<<unsigned(blocks), kThreads, smem, st>>>(A);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    mark(4);
    if (A.csc.n_hubs > 0 &&
        (e = launch16<T, SrcMerge>(M, unsigned((A.csc.n_hubs + kWarps - 1) / kWarps), 0, st)) !=
            cudaSuccess)
      return e;
    mark(5);
  }
  // attention-vector gradients: as many blocks as are resident at once (at
  // most the workspace's rows), so that no second partial wave trails
  {
    const size_t smem = size_t(kWarps) * (32 / s16.lpr) * 2 * row_f * 4;
    void (*dk)(const BwdArgs) =
        M.s.nv == 1 ? da_partial<T, 1> : (M.s.nv == 2 ? da_partial<T, 2> : da_partial<T, 4>);
    if ((e = set_smem(dk, smem)) != cudaSuccess) return e;
    BwdArgs Md = M;
    const int64_t resident = persistent_blocks(dk, smem, sm_count);
    if (resident < Md.da_blocks) Md.da_blocks = int(resident);
    if ((e = launch16<T, DaPartial>(Md, unsigned(Md.da_blocks), smem, st)) != cudaSuccess)
      return e;
    mark(6);
    da_final<<<unsigned((2 * row_f + kWarps - 1) / kWarps), kThreads, 0, st>>>(
        A.da_part, Md.da_blocks, row_f, A.da_src, A.da_dst);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    mark(7);
  }
  return cudaGetLastError();
}

DirArgs dir_args(const Dir& d) {
  DirArgs a{};
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

}  // namespace

cudaError_t launch_backward(const gnn_graph* g, const Shape& s, gnn_dtype dt, const void* h,
                            const float* a_src, const float* a_dst, float slope,
                            const float* lse, const void* dout, void* dh, float* da_src,
                            float* da_dst, char* ws, const WsLayout& L, cudaStream_t st,
                            const cudaEvent_t* ev, bool reuse_scores) {
  BwdArgs A{};
  A.s = s;
  A.csr = dir_args(g->csr);
  A.csc = dir_args(g->csc);
  A.n = g->n;
  A.h = h;
  A.a_src = a_src;
  A.a_dst = a_dst;
  A.ssrc = reinterpret_cast<const float*>(ws + L.bwd_scores);
  A.sdst = A.ssrc + g->n * s.H;
  A.slope = slope;
  A.lse = lse;
  A.dout = dout;
  A.dh = dh;
  A.da_src = da_src;
  A.da_dst = da_dst;
  A.stats = reinterpret_cast<float4*>(ws + L.stats);
  A.ds_src = reinterpret_cast<float*>(ws + L.ds_src);
  A.dst_part = reinterpret_cast<float4*>(ws + L.dst_part);
  A.src_acc = reinterpret_cast<float*>(ws + L.src_acc);
  A.src_sum = reinterpret_cast<float*>(ws + L.src_sum);
  A.da_part = reinterpret_cast<double*>(ws + L.da_part);
  A.da_blocks = L.da_blocks;
  A.ctr = reinterpret_cast<int*>(ws + L.bwd_ctr);
  A.err = g->err;
  // 32-byte lane vectors where a head spans 32 bytes or more, the row fits
  // one warp and the gathered and own rows start on 32-byte boundaries
  Shape w;
  if (make_wide_shape(s, &w) && aligned32(h) && aligned32(dout)) {
    A.s = w;
    if (dt == GNN_F32) return launch_t<float, 1, 32>(A, s, dt, g->sm_count, st, ev, reuse_scores);
    return launch_t<__nv_bfloat16, 1, 32>(A, s, dt, g->sm_count, st, ev, reuse_scores);
  }
  if (dt == GNN_F32) {
    switch (s.nv) {
      case 1: return launch_t<float, 1, 16>(A, s, dt, g->sm_count, st, ev, reuse_scores);
      case 2: return launch_t<float, 2, 16>(A, s, dt, g->sm_count, st, ev, reuse_scores);
      case 4: return launch_t<float, 4, 16>(A, s, dt, g->sm_count, st, ev, reuse_scores);
    }
  } else {
    switch (s.nv) {
      case 1: return launch_t<__nv_bfloat16, 1, 16>(A, s, dt, g->sm_count, st, ev, reuse_scores);
      case 2: return launch_t<__nv_bfloat16, 2, 16>(A, s, dt, g->sm_count, st, ev, reuse_scores);
      case 4: return launch_t<__nv_bfloat16, 4, 16>(A, s, dt, g->sm_count, st, ev, reuse_scores);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace gnn
