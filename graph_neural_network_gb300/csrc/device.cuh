// Device-side helpers shared by the aggregation kernels: 16-byte row
// vectors, per-head warp reductions, the lane geometry of a feature row, and
// the bulk-copy staging of an edge list into shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace gnn {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kWarps = 8;      // warps per thread block in every aggregation kernel
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 4;     // edges in flight per lane and batch

// Resident blocks per SM the main kernels are compiled for (register cap).
// Rows up to 512 bytes: 4 blocks (32 warps, <= 64 registers) for the
// kernels that gather one row per edge and keep little state, 3 blocks
// (24 warps, <= 80 registers) for the source-side backward pass with
// 16-byte vectors, which gathers a row and a statistics record and keeps a
// row accumulator (at 64 registers it spills and runs slower).  Measured on
// GB300 over the power-law workloads.
template <int NV>
struct MinBlocks {
  static constexpr int value = NV == 1 ? 3 : (NV == 2 ? 2 : 1);
};
template <int NV>
struct MinBlocksLean {
  static constexpr int value = NV == 1 ? 4 : (NV == 2 ? 2 : 1);
};

template <typename T>
struct VecOf;
template <>
struct VecOf<float> {
  static constexpr int n = 4;
};
template <>
struct VecOf<__nv_bfloat16> {
  static constexpr int n = 8;
};

// Read-only 16-byte load (gathered feature rows, edge lists, statistics).
__device__ __forceinline__ uint4 ld16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ float4 ld16f(const void* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

template <typename T>
__device__ __forceinline__ void unpack(const uint4& r, float (&x)[VecOf<T>::n]);

template <>
__device__ __forceinline__ void unpack<float>(const uint4& r, float (&x)[4]) {
  x[0] = __uint_as_float(r.x);
  x[1] = __uint_as_float(r.y);
  x[2] = __uint_as_float(r.z);
  x[3] = __uint_as_float(r.w);
}

// bfloat16 -> float32 is exact: the 16 bits become the high half of a float.
template <>
__device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4& r, float (&x)[8]) {
  x[0] = __uint_as_float(r.x << 16);
  x[1] = __uint_as_float(r.x & 0xffff0000u);
  x[2] = __uint_as_float(r.y << 16);
  x[3] = __uint_as_float(r.y & 0xffff0000u);
  x[4] = __uint_as_float(r.z << 16);
  x[5] = __uint_as_float(r.z & 0xffff0000u);
  x[6] = __uint_as_float(r.w << 16);
  x[7] = __uint_as_float(r.w & 0xffff0000u);
}

// Same values as unpack(), computed with byte permutes instead of shifts.  The
// kernels widen each gathered vector twice (once for the score, once for the
// accumulation); the different instruction sequence keeps the compiler from
// holding all widened values of a batch live in registers between the two.
template <typename T>
__device__ __forceinline__ void unpack_alt(const uint4& r, float (&x)[VecOf<T>::n]);

template <>
__device__ __forceinline__ void unpack_alt<float>(const uint4& r, float (&x)[4]) {
  unpack<float>(r, x);
}

template <>
__device__ __forceinline__ void unpack_alt<__nv_bfloat16>(const uint4& r, float (&x)[8]) {
  x[0] = __uint_as_float(__byte_perm(r.x, 0u, 0x1054));
  x[1] = __uint_as_float(__byte_perm(r.x, 0u, 0x3244));
  x[2] = __uint_as_float(__byte_perm(r.y, 0u, 0x1054));
  x[3] = __uint_as_float(__byte_perm(r.y, 0u, 0x3244));
  x[4] = __uint_as_float(__byte_perm(r.z, 0u, 0x1054));
  x[5] = __uint_as_float(__byte_perm(r.z, 0u, 0x3244));
  x[6] = __uint_as_float(__byte_perm(r.w, 0u, 0x1054));
  x[7] = __uint_as_float(__byte_perm(r.w, 0u, 0x3244));
}

template <typename T>
__device__ __forceinline__ uint4 pack(const float (&x)[VecOf<T>::n]);

template <>
__device__ __forceinline__ uint4 pack<float>(const float (&x)[4]) {
  return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                    __float_as_uint(x[3]));
}

__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

template <>
__device__ __forceinline__ uint4 pack<__nv_bfloat16>(const float (&x)[8]) {
  return make_uint4(bf2(x[0], x[1]), bf2(x[2], x[3]), bf2(x[4], x[5]), bf2(x[6], x[7]));
}

__device__ __forceinline__ void st16(void* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// 2^x with the SFU instruction (relative error about 2^-22; results below
// 2^-126 flush to zero, which a softmax weight can ignore).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed two-wide float32 arithmetic (one instruction for two lanes of
// data on sm_100 and later).
__device__ __forceinline__ unsigned long long pk(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
// (d0, d1) = (a0, a1) * (b0, b1) + (d0, d1)
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk(a0, a1)), "l"(pk(b0, b1)),
      "l"(pk(d0, d1)));
  upk(d, d0, d1);
}
// (d0, d1) *= (s, s)
__device__ __forceinline__ void mul2(float& d0, float& d1, float s) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(d0, d1)), "l"(pk(s, s)));
  upk(d, d0, d1);
}

// (d0, d1) = (a0, a1) + (b0, b1)
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0,
                                     float b1) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a0, a1)), "l"(pk(b0, b1)));
  upk(d, d0, d1);
}
// (d0, d1) = (a0, a1) * (b0, b1)
__device__ __forceinline__ void mul2v(float& d0, float& d1, float a0, float a1, float b0,
                                      float b1) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk(a0, a1)), "l"(pk(b0, b1)));
  upk(d, d0, d1);
}

// x . w over V elements (two interleaved partial sums, added at the end).
template <int V>
__device__ __forceinline__ float dot(const float (&x)[V], const float (&w)[V]) {
  float d0 = 0.f, d1 = 0.f;
#pragma unroll
  for (int c = 0; c < V; c += 2) fma2(d0, d1, x[c], x[c + 1], w[c], w[c + 1]);
  return d0 + d1;
}

// acc += p * x over V elements.
template <int V>
__device__ __forceinline__ void axpy(float (&acc)[V], float p, const float (&x)[V]) {
#pragma unroll
  for (int c = 0; c < V; c += 2) fma2(acc[c], acc[c + 1], x[c], x[c + 1], p, p);
}

// acc *= s over V elements.
template <int V>
__device__ __forceinline__ void scale(float (&acc)[V], float s) {
#pragma unroll
  for (int c = 0; c < V; c += 2) mul2(acc[c], acc[c + 1], s);
}

// Butterfly sums over aligned groups of 2^L lanes, for every element of x.
template <int L, int N>
__device__ __forceinline__ void group_sum(float (&x)[N]) {
#pragma unroll
  for (int o = 1; o < (1 << L); o <<= 1)
#pragma unroll
    for (int n = 0; n < N; ++n) x[n] += __shfl_xor_sync(kFull, x[n], o);
}

// Sum each element of x over the 2^hv_log2 lanes of its head.  One uniform
// branch per call; the shuffles themselves are unrolled for the head width.
template <int N>
__device__ __forceinline__ void head_sums(float (&x)[N], int hv_log2) {
  switch (hv_log2) {
    case 0: break;
    case 1: group_sum<1, N>(x); break;
    case 2: group_sum<2, N>(x); break;
    case 3: group_sum<3, N>(x); break;
    case 4: group_sum<4, N>(x); break;
    default: group_sum<5, N>(x); break;
  }
}

// Where one lane sits in a feature row.  A row of rv 16-byte vectors is spread
// over lpr lanes (a power of two); a warp therefore handles G = 32 / lpr rows
// (edges) at once, sub-group g = lane / lpr.  With nv > 1 (rows wider than
// 512 bytes) lpr = 32 and lane p holds vectors p, p + 32, ...
template <int NV>
struct Lane {
  int lane, g, G, p;
  int q[NV];     // vector index within the row
  bool ok[NV];   // q < rv
  int k[NV];     // head of the vector
  __device__ __forceinline__ Lane(const Shape& s) {
    lane = threadIdx.x & 31;
    g = lane >> s.lpr_log2;
    G = 32 >> s.lpr_log2;
    p = lane & (s.lpr - 1);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      q[v] = p + (v << s.lpr_log2);
      ok[v] = q[v] < s.rv;
      k[v] = ok[v] ? q[v] >> s.hv_log2 : 0;
    }
  }
  // lane writes the per-head scalar of vector v (one lane per head)
  __device__ __forceinline__ bool head_leader(const Shape& s, int v) const {
    return ok[v] && (q[v] & (s.hv - 1)) == 0;
  }
};

template <typename T>
__device__ __forceinline__ const char* row_base(const void* base, int64_t node, int rv) {
  return reinterpret_cast<const char*>(base) + node * int64_t(rv) * 16;
}

// This lane's slice of an attention vector [H][D] (float), times `scale`.
template <typename T, int NV>
__device__ __forceinline__ void load_att(const float* a, const Lane<NV>& L, float scale,
                                         float (&w)[NV][VecOf<T>::n]) {
  constexpr int V = VecOf<T>::n;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
#pragma unroll
    for (int c4 = 0; c4 < V; c4 += 4) {
      float4 t = L.ok[v] ? ld16f(a + L.q[v] * V + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      w[v][c4 + 0] = t.x * scale;
      w[v][c4 + 1] = t.y * scale;
      w[v][c4 + 2] = t.z * scale;
      w[v][c4 + 3] = t.w * scale;
    }
  }
}

// This lane's vectors of row `node` of x, widened to float (zeros where q >= rv).
template <typename T, int NV>
__device__ __forceinline__ void load_row(const void* x, int64_t node, const Shape& s,
                                         const Lane<NV>& L, float (&r)[NV][VecOf<T>::n]) {
  const char* row = row_base<T>(x, node, s.rv);
#pragma unroll
  for (int v = 0; v < NV; ++v)
    unpack<T>(L.ok[v] ? ld16(row + 16 * L.q[v]) : make_uint4(0, 0, 0, 0), r[v]);
}

// Per-head dot product w[k] . x[node][k] for the heads this lane touches.
template <typename T, int NV>
__device__ __forceinline__ void row_dot(const void* x, int64_t node, const Shape& s,
                                        const Lane<NV>& L, const float (&w)[NV][VecOf<T>::n],
                                        float (&out)[NV]) {
  constexpr int V = VecOf<T>::n;
  float r[NV][V];
  load_row<T, NV>(x, node, s, L, r);
#pragma unroll
  for (int v = 0; v < NV; ++v) out[v] = dot<V>(r[v], w[v]);
  head_sums<NV>(out, s.hv_log2);
}

// The sources (or destinations) of the batch of edges starting at beg that
// this lane's sub-group takes: edges beg + g, beg + g + G, ... (U of them)
// below end, read from cols[edge - colbase]; -1 past the end.
template <int U>
__device__ __forceinline__ void batch_ids(const int32_t* cols, int colbase, int beg, int end,
                                          int g, int G, int (&j)[U]) {
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int e = beg + u * G + g;
    j[u] = e < end ? cols[e - colbase] : -1;
  }
}

// Butterfly sum over the warp's sub-groups (every lane ends with the total).
__device__ __forceinline__ float subgroup_sum(float x, const Shape& s) {
  for (int o = s.lpr; o < 32; o <<= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

template <int V>
__device__ __forceinline__ void subgroup_sums(float (&x)[V], const Shape& s) {
#pragma unroll
  for (int c = 0; c < V; ++c) x[c] = subgroup_sum(x[c], s);
}

template <int V>
__device__ __forceinline__ void zero(float (&x)[V]) {
#pragma unroll
  for (int c = 0; c < V; ++c) x[c] = 0.f;
}

// s += x with the rounding error of the addition carried in c (Kahan's
// compensated summation), for merges that add thousands of hub-chunk
// partials, where a plain running sum loses accuracy with their number.
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = __fsub_rn(x, c);
  const float t = __fadd_rn(s, y);
  c = __fsub_rn(__fsub_rn(t, s), y);
  s = t;
}

// ---- lane vectors of 16 or 32 bytes -------------------------------------------
//
// The attention kernels can give each lane 32 contiguous bytes of a row (two
// 16-byte halves, loaded by one 256-bit load) instead of 16, where a head
// spans at least 32 bytes: the per-edge work that does not depend on the
// number of elements a lane holds (addresses, the per-edge statistics, the
// score and its exponential) is then shared by twice as many elements.

template <int VB>
struct RawV;
template <>
struct RawV<16> {
  uint4 a;
};
template <>
struct RawV<32> {
  uint4 a, b;
};

// Elements of T in a VB-byte lane vector, and edges each lane keeps in flight
// per batch (the same 64 bytes either way).
template <typename T, int VB>
struct ElemsOf {
  static constexpr int n = VB / int(sizeof(T));
};
template <int VB>
struct UnrollOf {
  static constexpr int value = 64 / VB;
};

template <int VB>
__device__ __forceinline__ RawV<VB> ldv(const void* p);
template <>
__device__ __forceinline__ RawV<16> ldv<16>(const void* p) {
  return RawV<16>{ld16(p)};
}
// One 256-bit read-only load (32-byte aligned).
template <>
__device__ __forceinline__ RawV<32> ldv<32>(const void* p) {
  RawV<32> r;
  asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w), "=r"(r.b.x), "=r"(r.b.y),
        "=r"(r.b.z), "=r"(r.b.w)
      : "l"(p));
  return r;
}

template <int VB>
__device__ __forceinline__ RawV<VB> zero_raw();
template <>
__device__ __forceinline__ RawV<16> zero_raw<16>() {
  return RawV<16>{make_uint4(0, 0, 0, 0)};
}
template <>
__device__ __forceinline__ RawV<32> zero_raw<32>() {
  return RawV<32>{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
}

// Widen a lane vector to float (two spellings, as unpack / unpack_alt).
template <typename T, int VB>
__device__ __forceinline__ void unpackv(const RawV<VB>& r, float (&x)[ElemsOf<T, VB>::n]) {
  constexpr int H16 = VecOf<T>::n;
  float* p = x;
  unpack<T>(r.a, *reinterpret_cast<float(*)[H16]>(p));
  if constexpr (VB == 32) unpack<T>(r.b, *reinterpret_cast<float(*)[H16]>(p + H16));
}
template <typename T, int VB>
__device__ __forceinline__ void unpack_altv(const RawV<VB>& r, float (&x)[ElemsOf<T, VB>::n]) {
  constexpr int H16 = VecOf<T>::n;
  float* p = x;
  unpack_alt<T>(r.a, *reinterpret_cast<float(*)[H16]>(p));
  if constexpr (VB == 32) unpack_alt<T>(r.b, *reinterpret_cast<float(*)[H16]>(p + H16));
}

// Narrow and store a lane vector (plain stores, 16 bytes each).
template <typename T, int VB>
__device__ __forceinline__ void storev(void* dst, const float (&x)[ElemsOf<T, VB>::n]) {
  constexpr int H16 = VecOf<T>::n;
  const float* p = x;
  st16(dst, pack<T>(*reinterpret_cast<const float(*)[H16]>(p)));
  if constexpr (VB == 32)
    st16(reinterpret_cast<char*>(dst) + 16, pack<T>(*reinterpret_cast<const float(*)[H16]>(p + H16)));
}

// a . b over the bfloat16 elements of two lane vectors in float32: every
// product of two bfloat16 values is exact in float32, so each step is one
// fused multiply-add of the widened values; even and odd elements go to two
// sums added at the end (the same order as dot() on widened vectors, so the
// result is bit for bit the same).
template <int VB>
__device__ __forceinline__ float dot_bf16(const RawV<VB>& a, const RawV<VB>& b) {
  const uint32_t* pa = reinterpret_cast<const uint32_t*>(&a);
  const uint32_t* pb = reinterpret_cast<const uint32_t*>(&b);
  float d0 = 0.f, d1 = 0.f;
#pragma unroll
  for (int w = 0; w < VB / 4; ++w)
    asm("{\n .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
        " fma.rn.f32.bf16 %0, al, bl, %0;\n fma.rn.f32.bf16 %1, ah, bh, %1;\n}"
        : "+f"(d0), "+f"(d1)
        : "r"(pa[w]), "r"(pb[w]));
  return d0 + d1;
}

// A node's own row vector that is dotted with one gathered vector per edge:
// float32 rows are kept widened; bfloat16 rows stay packed and go through
// dot_bf16 (no widening of either operand).
template <typename T, int VB>
struct OwnVec {
  float x[ElemsOf<T, VB>::n];
  __device__ __forceinline__ void set(const RawV<VB>& r) { unpackv<T, VB>(r, x); }
  __device__ __forceinline__ float dot_with(const RawV<VB>& g) const {
    constexpr int V = ElemsOf<T, VB>::n;
    float y[V];
    unpackv<T, VB>(g, y);
    return dot<V>(y, x);
  }
};
template <int VB>
struct OwnVec<__nv_bfloat16, VB> {
  RawV<VB> r;
  __device__ __forceinline__ void set(const RawV<VB>& v) { r = v; }
  __device__ __forceinline__ float dot_with(const RawV<VB>& g) const { return dot_bf16<VB>(g, r); }
};

template <int VB>
__device__ __forceinline__ const char* row_at(const void* base, int64_t node, int rv) {
  return reinterpret_cast<const char*>(base) + node * int64_t(rv) * VB;
}

// This lane's slices of an attention vector [H][D] (float) for VB-byte lane
// vectors, times `scale`.
template <typename T, int NV, int VB>
__device__ __forceinline__ void load_att_v(const float* a, const Lane<NV>& L, float scale,
                                           float (&w)[NV][ElemsOf<T, VB>::n]) {
  constexpr int V = ElemsOf<T, VB>::n;
#pragma unroll
  for (int v = 0; v < NV; ++v) {
#pragma unroll
    for (int c4 = 0; c4 < V; c4 += 4) {
      float4 t = L.ok[v] ? ld16f(a + L.q[v] * V + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      w[v][c4 + 0] = t.x * scale;
      w[v][c4 + 1] = t.y * scale;
      w[v][c4 + 2] = t.z * scale;
      w[v][c4 + 3] = t.w * scale;
    }
  }
}

// This lane's vectors of row `node` of x (VB-byte lane vectors), widened
// (zeros where q >= rv).
template <typename T, int NV, int VB>
__device__ __forceinline__ void load_row_v(const void* x, int64_t node, const Shape& s,
                                           const Lane<NV>& L, float (&r)[NV][ElemsOf<T, VB>::n]) {
  const char* row = row_at<VB>(x, node, s.rv);
#pragma unroll
  for (int v = 0; v < NV; ++v)
    unpackv<T, VB>(L.ok[v] ? ldv<VB>(row + VB * L.q[v]) : zero_raw<VB>(), r[v]);
}

// This lane's slice (vector q) of row `node` when a row needs at most one
// vector per lane, widened (zeros when !ok).
template <typename T>
__device__ __forceinline__ void own_row(const void* x, int64_t node, const Shape& s,
                                        const Lane<1>& L, float (&r)[VecOf<T>::n]) {
  unpack<T>(L.ok[0] ? ld16(row_base<T>(x, node, s.rv) + 16 * L.q[0]) : make_uint4(0, 0, 0, 0),
            r);
}

// ---- mbarrier + bulk copy (shared::cta) --------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One-dimensional bulk copy global -> shared, completing on `bar`.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait on phase `parity`; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int limit) {
  const uint32_t a = smem_u32(bar);
  for (int it = 0; it < limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

constexpr int kWaitLimit = 1 << 20;

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Stage idx[beg, end) into shared memory `dst` (16-byte aligned) such that
// element x lands at dst[x - (beg & ~3)].  The 16-byte-aligned interior moves
// with one bulk copy completing on `bar` (initialised once per kernel with
// mbar_init(bar, 1); `parity` tracks its phase across calls); the ragged
// ends (< 4 elements each) move with plain loads.  Must be called by all
// threads of the block, after a __syncthreads that ends every read of the
// previous contents.  Returns false (after recording a timeout in *err and
// letting the copy land) when the bulk copy did not complete within the
// limit.
__device__ __forceinline__ bool stage_edges(int32_t* dst, const int32_t* idx, int beg, int end,
                                            uint64_t* bar, uint32_t& parity, int32_t* err) {
  const int base = beg & ~3;
  const int a0 = (beg + 3) & ~3;
  const int a1 = end & ~3;
  const bool bulk = a1 > a0;
  if (threadIdx.x == 0 && bulk) {
    fence_proxy_async();  // earlier generic-proxy reads of dst come first
    mbar_expect_tx(bar, uint32_t(a1 - a0) * 4u);
    bulk_g2s(dst + (a0 - base), idx + a0, uint32_t(a1 - a0) * 4u, bar);
  }
  // ragged head and tail (or everything when the item is short)
  const int h1 = bulk ? a0 : end;
  for (int x = beg + int(threadIdx.x); x < h1; x += blockDim.x) dst[x - base] = __ldg(idx + x);
  if (bulk)
    for (int x = a1 + int(threadIdx.x); x < end; x += blockDim.x) dst[x - base] = __ldg(idx + x);
  bool timed_out = false;
  if (bulk) timed_out = !mbar_wait(bar, parity, kWaitLimit);
  if (__syncthreads_or(timed_out)) {
    if (threadIdx.x == 0) {
      atomicOr(err, DEVERR_TIMEOUT);
      mbar_wait(bar, parity, kWaitLimit);  // let the copy land before the block exits
    }
    return false;
  }
  if (bulk) parity ^= 1u;
  return true;
}

// Number of persistent blocks for a kernel: what fits on every SM at once.
template <typename K>
__host__ int persistent_blocks(K kernel, size_t smem, int sm_count) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm * (sm_count > 0 ? sm_count : 1);
}

}  // namespace gnn
