// Per-node score halves, once per call: s_src(n, k) = log2(e) a_src[k] . h_n[k]
// and s_dst(n, k) = log2(e) a_dst[k] . h_n[k] (base-2 units, float [N][H]).
// The edge loops then gather one float per edge and head instead of
// re-deriving a_src . h_j from every gathered row.  One streaming read of h.
#include "device.cuh"

namespace gnn {
namespace {

constexpr int kNodesPerIter = 4;  // node rows in flight per sub-group

template <typename T, int NV, int VB>
__global__ void __launch_bounds__(kThreads) node_scores(const Shape s, const void* h,
                                                        const float* a_src, const float* a_dst,
                                                        int64_t n, float* ssrc, float* sdst) {
  constexpr int V = ElemsOf<T, VB>::n;
  constexpr int U = kNodesPerIter * 16 / VB;  // the same bytes in flight per lane
  const Lane<NV> L(s);
  float as2[NV][V], ad2[NV][V];
  load_att_v<T, NV, VB>(a_src, L, kLog2e, as2);
  load_att_v<T, NV, VB>(a_dst, L, kLog2e, ad2);
  const int64_t stride = int64_t(gridDim.x) * kWarps * L.G;
  // warp-uniform loop over groups of G consecutive nodes; sub-group g takes
  // node base + g of each group
  for (int64_t base = (int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * L.G; base < n;
       base += U * stride) {
    RawV<VB> raw[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t node = base + u * stride + L.g;
#pragma unroll
      for (int v = 0; v < NV; ++v)
        raw[u][v] = (node < n && L.ok[v]) ? ldv<VB>(row_at<VB>(h, node, s.rv) + VB * L.q[v])
                                          : zero_raw<VB>();
    }
    float d[2 * U * NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float x[V];
        unpackv<T, VB>(raw[u][v], x);
        d[u * NV + v] = dot<V>(x, as2[v]);
        d[U * NV + u * NV + v] = dot<V>(x, ad2[v]);
      }
    head_sums<2 * U * NV>(d, s.hv_log2);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t node = base + u * stride + L.g;
      if (node >= n) continue;
#pragma unroll
      for (int v = 0; v < NV; ++v)
        if (L.head_leader(s, v)) {
          ssrc[node * s.H + L.k[v]] = d[u * NV + v];
          sdst[node * s.H + L.k[v]] = d[U * NV + u * NV + v];
        }
    }
  }
}

template <typename T, int NV, int VB>
cudaError_t launch_t(const Shape& s, const void* h, const float* a_src, const float* a_dst,
                     int64_t n, float* ssrc, float* sdst, int sm_count, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t per_block = int64_t(kWarps) * (32 >> s.lpr_log2) * (kNodesPerIter * 16 / VB);
  int64_t blocks = (n + per_block - 1) / per_block;
  // as many blocks as are resident at once: one wave, no trailing partial one
  const int64_t cap = persistent_blocks(node_scores<T, NV, VB>, 0, sm_count);
  if (blocks > cap) blocks = cap;
  node_scores<T, NV, VB><<<unsigned(blocks), kThreads, 0, st>>>(s, h, a_src, a_dst, n, ssrc,
                                                                sdst);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_node_scores(const Shape& s, gnn_dtype dt, const void* h, const float* a_src,
                               const float* a_dst, int64_t n, float* ssrc, float* sdst,
                               int sm_count, cudaStream_t st) {
  // 32-byte lane vectors where the attention kernels use them
  Shape w;
  if (make_wide_shape(s, &w) && aligned32(h)) {
    if (dt == GNN_F32)
      return launch_t<float, 1, 32>(w, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
    return launch_t<__nv_bfloat16, 1, 32>(w, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
  }
  if (dt == GNN_F32) {
    switch (s.nv) {
      case 1: return launch_t<float, 1, 16>(s, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
      case 2: return launch_t<float, 2, 16>(s, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
      case 4: return launch_t<float, 4, 16>(s, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
    }
  } else {
    switch (s.nv) {
      case 1:
        return launch_t<__nv_bfloat16, 1, 16>(s, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
      case 2:
        return launch_t<__nv_bfloat16, 2, 16>(s, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
      case 4:
        return launch_t<__nv_bfloat16, 4, 16>(s, h, a_src, a_dst, n, ssrc, sdst, sm_count, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace gnn
