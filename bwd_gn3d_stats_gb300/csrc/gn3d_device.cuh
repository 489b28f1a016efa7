// gn3d_device.cuh -- device building blocks shared by the GroupNorm kernels:
// vector loads/stores, fixed-order block reductions, the group merge of the
// per-unit statistics.
//
// Every floating-point operation that feeds a statistic or an output is written
// with an explicit round-to-nearest intrinsic (__fadd_rn, __fmul_rn, __fmaf_rn,
// ...).  The compiler never contracts or reorders those, so the arithmetic --
// and the bits -- are the same in every template instantiation (bf16 or fp32
// input, bf16 or fp32 output) and in every kernel variant that uses them.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "gn3d_plan.cuh"

namespace gn3d {

__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float ffma(float a, float b, float c) { return __fmaf_rn(a, b, c); }

// ------------------------------------------------------------- element I/O
// A "vector" is 8 consecutive elements starting at a flat index that is a
// multiple of 8; with a 16-byte aligned base this is one 16-byte access for
// bf16 and two for fp32.

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <class T> struct IO;

template <> struct IO<__nv_bfloat16> {
  static __device__ __forceinline__ void load8(const __nv_bfloat16* p, float v[8]) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    v[0] = bf16_lo(r.x); v[1] = bf16_hi(r.x); v[2] = bf16_lo(r.y); v[3] = bf16_hi(r.y);
    v[4] = bf16_lo(r.z); v[5] = bf16_hi(r.z); v[6] = bf16_lo(r.w); v[7] = bf16_hi(r.w);
  }
  static __device__ __forceinline__ float load1(const __nv_bfloat16* p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short*>(p)) << 16);
  }
  static __device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // round to nearest even, low half = a
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ void store8(__nv_bfloat16* p, const float v[8]) {
    uint4 r;
    r.x = pack2(v[0], v[1]); r.y = pack2(v[2], v[3]); r.z = pack2(v[4], v[5]); r.w = pack2(v[6], v[7]);
    __stcs(reinterpret_cast<uint4*>(p), r);
  }
  static __device__ __forceinline__ void store1(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
};

template <> struct IO<float> {
  static __device__ __forceinline__ void load8(const float* p, float v[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ float load1(const float* p) { return *p; }
  static __device__ __forceinline__ void store8(float* p, const float v[8]) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<float4*>(p + 4), make_float4(v[4], v[5], v[6], v[7]));
  }
  static __device__ __forceinline__ void store1(float* p, float v) { *p = v; }
};

// ------------------------------------------------------ block reductions
// Sum of (a, b) over the CTA in a fixed order: an xor butterfly inside each warp
// (every lane ends with the same bits, since IEEE addition is commutative), then
// the warp totals added in warp order.  Every thread returns the total.

__device__ __forceinline__ float2 block_sum2(float a, float b, float2* sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fadd(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    b = fadd(b, __shfl_xor_sync(0xFFFFFFFFu, b, o));
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) sh[w] = make_float2(a, b);
  __syncthreads();
  float2 r = sh[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) {
    r.x = fadd(r.x, sh[i].x);
    r.y = fadd(r.y, sh[i].y);
  }
  __syncthreads();
  return r;
}

// ------------------------------------------------------ group statistics
// Per-unit record of the forward statistics (16 bytes): the unit's mean as the
// unevaluated pair m1 + cn (m1 = sum/n in fp32, cn = sum(x - m1)/n), its M2 =
// sum((x - mean)^2) and its element count.
struct Part {
  float m1, m2;
  int n;
  float cn;
};

// Merge of the unit partials of one group (the parallel-variance combine of
// Chan, Golub & LeVeque in its shifted-sum form): with the shift K = the first
// unit's mean and d_u = mean_u - K,
//   mean = K + (sum n_u d_u) / M,   M2 = sum (M2_u + n_u d_u^2) - (sum n_u d_u)^2 / M.
// The merge runs in fp64 (the per-element accumulation is fp32): the group
// mean then keeps the digits an fp32 mean of a large-offset group loses, which
// the normalize uses as a hi/lo pair.  Fixed shape: thread t sums its
// contiguous slice in order, a shfl_down tree sums each warp into lane 0, and
// thread 0 adds the warp sums in warp order.  Result valid in thread 0.
struct GroupMoments {
  double mean, m2;
};

__device__ __forceinline__ double dadd(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ double dmul(double a, double b) { return __dmul_rn(a, b); }

__device__ __forceinline__ GroupMoments combine_parts(const Part* parts, int64_t cnt, int64_t M, double2* sh) {
  const float4 r0 = __ldcg(reinterpret_cast<const float4*>(parts));
  const double K = dadd((double)r0.x, (double)r0.w);
  const int64_t per = (cnt + kThreads - 1) / kThreads;
  int64_t lo = (int64_t)threadIdx.x * per, hi = lo + per;
  if (hi > cnt) hi = cnt;
  double S = 0.0, Q = 0.0;
  for (int64_t i = lo; i < hi; ++i) {
    const float4 r = __ldcg(reinterpret_cast<const float4*>(parts + i));
    const int n = __float_as_int(r.z);
    if (n == 0) continue;
    const double d = dadd(dadd((double)r.x, -K), (double)r.w);
    const double nd = dmul((double)n, d);
    S = dadd(S, nd);
    Q = dadd(Q, dadd((double)r.y, dmul(nd, d)));
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double a = __shfl_down_sync(0xFFFFFFFFu, S, o);
    const double b = __shfl_down_sync(0xFFFFFFFFu, Q, o);
    if (lane + o < 32) { S = dadd(S, a); Q = dadd(Q, b); }
  }
  if (lane == 0) sh[threadIdx.x >> 5] = make_double2(S, Q);
  __syncthreads();
  GroupMoments g = {0.0, 0.0};
  if (threadIdx.x == 0) {
    S = sh[0].x;
    Q = sh[0].y;
    for (int i = 1; i < kWarps; ++i) { S = dadd(S, sh[i].x); Q = dadd(Q, sh[i].y); }
    const double sm = __ddiv_rn(S, (double)M);
    g.mean = dadd(K, sm);
    g.m2 = dadd(Q, -dmul(S, sm));
    if (g.m2 < 0.0) g.m2 = 0.0;  // rounding only; NaN is kept
  }
  __syncthreads();
  return g;
}

// ---------------------------------------------------------- unit loaders
// Loads one unit into registers: kVecPerThread vectors per thread (vector j of
// the body goes to thread j % kThreads, slot j / kThreads) plus at most one
// head/tail scalar (scalar s goes to thread s).  Absent values are 0 and flagged.
template <class T>
struct UnitRegs {
  float v[kVecPerThread][8];
  bool vok[kVecPerThread];
  float s;
  bool sok;

  __device__ __forceinline__ void load(const T* __restrict__ p, const URange& q) {
    const int64_t nv = (q.b1 - q.b0) / kVec;
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int64_t j = threadIdx.x + (int64_t)i * kThreads;
      vok[i] = j < nv;
      if (vok[i]) IO<T>::load8(p + q.b0 + j * kVec, v[i]);
      else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[i][e] = 0.f;
      }
    }
    sok = (int)threadIdx.x < scalar_count(q);
    s = sok ? IO<T>::load1(p + scalar_index(q, threadIdx.x)) : 0.f;
  }
};

}  // namespace gn3d
