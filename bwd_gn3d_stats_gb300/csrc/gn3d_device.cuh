// gn3d_device.cuh -- the GroupNorm arithmetic, shared by both launch forms:
// vector I/O, warp reductions, the per-unit statistics, the block and group
// merges, and the elementwise passes.
//
// Every floating-point operation that feeds a statistic or an output is written
// with an explicit round-to-nearest intrinsic (__fadd_rn, __fmul_rn, __fmaf_rn,
// ...).  The compiler never contracts or reorders those, so the arithmetic --
// and the bits -- are the same in every template instantiation (bf16 or fp32
// input, bf16 or fp32 output) and in both launch forms.
//
// Completion across warps and CTAs uses integer counters with acquire/release
// semantics (never float atomics): the warp that brings a block's counter to
// its size merges the block, and the warp that completes a group's last block
// merges the group and publishes it with a release store on the group's flag.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "gn3d_plan.cuh"

namespace gn3d {

__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float ffma(float a, float b, float c) { return __fmaf_rn(a, b, c); }

constexpr unsigned kFull = 0xFFFFFFFFu;

// ------------------------------------------------------------- element I/O
// A "vector" is 8 consecutive elements starting at a flat index that is a
// multiple of 8; with a 16-byte aligned base this is one 16-byte access for
// bf16 and two for fp32.  load8 takes a generic pointer (shared memory in the
// persistent kernels, global memory in the streaming ones).

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
  static __device__ __forceinline__ void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
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

// -------------------------------------------------------- warp reductions
// xor butterfly: every lane ends with the same bits (IEEE addition commutes).
__device__ __forceinline__ float warp_sum(float a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fadd(a, __shfl_xor_sync(kFull, a, o));
  return a;
}

__device__ __forceinline__ float2 warp_sum2(float a, float b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fadd(a, __shfl_xor_sync(kFull, a, o));
    b = fadd(b, __shfl_xor_sync(kFull, b, o));
  }
  return make_float2(a, b);
}

// The fixed meeting tree of a lane's 8 running sums.
__device__ __forceinline__ float tree8(const float c[8]) {
  return fadd(fadd(fadd(c[0], c[1]), fadd(c[2], c[3])), fadd(fadd(c[4], c[5]), fadd(c[6], c[7])));
}

// -------------------------------------------------- acquire/release words
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Lane 0 adds one arrival to *ctr; every lane learns whether it was the last of
// `total`.  The release half orders lane 0's earlier stores before the arrival,
// the acquire half (with the __syncwarp) orders the warp's later loads after it.
__device__ __forceinline__ bool warp_arrive_last(uint32_t* ctr, uint32_t total) {
  uint32_t old = 0;
  if ((threadIdx.x & 31) == 0) old = atom_add_acq_rel(ctr, 1u);
  old = __shfl_sync(kFull, old, 0);
  __syncwarp();
  return old + 1u == total;
}

// ------------------------------------------------------------- moments
// Moments of a set of elements: the mean as the unevaluated pair m1 + cn, M2 =
// sum((x - mean)^2), and the count (16 bytes, one per unit, block and group).
struct Part {
  float m1, m2;
  int n;
  float cn;
};

// --------------------------------------------------------- body readers
// Where a unit's body vectors come from: a bulk-copied shared-memory slot or
// global memory.  A vector is kRaw 16-byte words.  Shared-memory reads are plain
// loads: the compiler schedules them freely, and the "memory" clobber of the
// mbarrier wait keeps them after the copy has landed.
struct FromShared {
  static __device__ __forceinline__ uint4 word(const void* p) { return *reinterpret_cast<const uint4*>(p); }
};

struct FromGlobal {
  static __device__ __forceinline__ uint4 word(const void* p) { return *reinterpret_cast<const uint4*>(p); }
};

// ----------------------------------------------------------- fp32 pairs
// Two fp32 values in one 64-bit register pair, for the paired fp32
// instructions of sm_100-class GPUs (add/sub/mul/fma .rn.f32x2).  Each half is
// rounded exactly as the scalar instruction would round it, so pair code gives
// the same bits as the scalar code it replaces -- at half the instructions.
typedef unsigned long long f2;

__device__ __forceinline__ f2 f2_of(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ f2 f2_bits(uint32_t lo, uint32_t hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(f2 a) {
  float lo;
  asm("{\n .reg .f32 t;\n mov.b64 {%0, t}, %1;\n}" : "=f"(lo) : "l"(a));
  return lo;
}
__device__ __forceinline__ float f2_hi(f2 a) {
  float hi;
  asm("{\n .reg .f32 t;\n mov.b64 {t, %0}, %1;\n}" : "=f"(hi) : "l"(a));
  return hi;
}
__device__ __forceinline__ f2 f2_splat(float a) { return f2_of(a, a); }
__device__ __forceinline__ f2 f2add(f2 a, f2 b) {
  f2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 f2sub(f2 a, f2 b) {
  f2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2 f2fma(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// 0xFFFF in each 16-bit half of w that holds a bf16 value <= 0 (NaN: 0).
__device__ __forceinline__ uint32_t bf16x2_le0(uint32_t w) {
  uint32_t m;
  asm("set.le.u32.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(w), "r"(0u));
  return m;
}

// (lo - k, hi - k) for the two bf16 halves of w, as an fp32 pair.
__device__ __forceinline__ f2 bf16_pair_minus(uint32_t w, float k) {
  f2 d;
  asm("{\n .reg .b16 l, h;\n .reg .f32 dl, dh;\n mov.b32 {l, h}, %1;\n sub.rn.f32.bf16 dl, l, %2;\n"
      " sub.rn.f32.bf16 dh, h, %2;\n mov.b64 %0, {dl, dh};\n}"
      : "=l"(d)
      : "r"(w), "f"(k));
  return d;
}

template <class T> struct Vec;

// A vector of 8 elements as 4 pairs: pair k holds elements 2k and 2k+1.
template <> struct Vec<__nv_bfloat16> {
  static constexpr int kRaw = 1;
  template <class Src>
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, uint4 r[kRaw]) { r[0] = Src::word(p); }
  static __device__ __forceinline__ void unpack(const uint4 r[kRaw], float v[8]) {
    v[0] = bf16_lo(r[0].x); v[1] = bf16_hi(r[0].x); v[2] = bf16_lo(r[0].y); v[3] = bf16_hi(r[0].y);
    v[4] = bf16_lo(r[0].z); v[5] = bf16_hi(r[0].z); v[6] = bf16_lo(r[0].w); v[7] = bf16_hi(r[0].w);
  }
  static __device__ __forceinline__ void pairs(const uint4 r[kRaw], f2 p[4]) {
    p[0] = f2_of(bf16_lo(r[0].x), bf16_hi(r[0].x));
    p[1] = f2_of(bf16_lo(r[0].y), bf16_hi(r[0].y));
    p[2] = f2_of(bf16_lo(r[0].z), bf16_hi(r[0].z));
    p[3] = f2_of(bf16_lo(r[0].w), bf16_hi(r[0].w));
  }
  // x - k as pairs: one mixed-precision subtraction per element (bf16 operand,
  // fp32 result, rounded once -- the same value as converting x first).
  static __device__ __forceinline__ void diff(const uint4 r[kRaw], float k, f2 d[4]) {
    d[0] = bf16_pair_minus(r[0].x, k);
    d[1] = bf16_pair_minus(r[0].y, k);
    d[2] = bf16_pair_minus(r[0].z, k);
    d[3] = bf16_pair_minus(r[0].w, k);
  }
  // Zero the elements of d where the result o is <= 0 (ordered compare: a NaN
  // result keeps its gradient) -- threshold_backward's gate, two halves at once.
  static __device__ __forceinline__ void gate(const uint4 o[kRaw], uint4 d[kRaw]) {
    d[0].x &= ~bf16x2_le0(o[0].x);
    d[0].y &= ~bf16x2_le0(o[0].y);
    d[0].z &= ~bf16x2_le0(o[0].z);
    d[0].w &= ~bf16x2_le0(o[0].w);
  }
};

template <> struct Vec<float> {
  static constexpr int kRaw = 2;
  template <class Src>
  static __device__ __forceinline__ void load(const float* p, uint4 r[kRaw]) {
    r[0] = Src::word(p);
    r[1] = Src::word(p + 4);
  }
  static __device__ __forceinline__ void unpack(const uint4 r[kRaw], float v[8]) {
    v[0] = __uint_as_float(r[0].x); v[1] = __uint_as_float(r[0].y);
    v[2] = __uint_as_float(r[0].z); v[3] = __uint_as_float(r[0].w);
    v[4] = __uint_as_float(r[1].x); v[5] = __uint_as_float(r[1].y);
    v[6] = __uint_as_float(r[1].z); v[7] = __uint_as_float(r[1].w);
  }
  static __device__ __forceinline__ void pairs(const uint4 r[kRaw], f2 p[4]) {
    p[0] = f2_bits(r[0].x, r[0].y);
    p[1] = f2_bits(r[0].z, r[0].w);
    p[2] = f2_bits(r[1].x, r[1].y);
    p[3] = f2_bits(r[1].z, r[1].w);
  }
  static __device__ __forceinline__ void diff(const uint4 r[kRaw], float k, f2 d[4]) {
    f2 p[4];
    pairs(r, p);
    const f2 k2 = f2_splat(k);
#pragma unroll
    for (int e = 0; e < 4; ++e) d[e] = f2sub(p[e], k2);
  }
  static __device__ __forceinline__ void gate(const uint4 o[kRaw], uint4 d[kRaw]) {
#pragma unroll
    for (int t = 0; t < kRaw; ++t) {
      d[t].x = __uint_as_float(o[t].x) <= 0.f ? 0u : d[t].x;
      d[t].y = __uint_as_float(o[t].y) <= 0.f ? 0u : d[t].y;
      d[t].z = __uint_as_float(o[t].z) <= 0.f ? 0u : d[t].z;
      d[t].w = __uint_as_float(o[t].w) <= 0.f ? 0u : d[t].w;
    }
  }
};

// Store of 8 results given as 4 pairs (one rounding to the output type, RNE).
template <class T>
__device__ __forceinline__ void store8p(T* p, const f2 v[4]);

template <>
__device__ __forceinline__ void store8p<__nv_bfloat16>(__nv_bfloat16* p, const f2 v[4]) {
  uint4 r;
  r.x = IO<__nv_bfloat16>::pack2(f2_lo(v[0]), f2_hi(v[0]));
  r.y = IO<__nv_bfloat16>::pack2(f2_lo(v[1]), f2_hi(v[1]));
  r.z = IO<__nv_bfloat16>::pack2(f2_lo(v[2]), f2_hi(v[2]));
  r.w = IO<__nv_bfloat16>::pack2(f2_lo(v[3]), f2_hi(v[3]));
  __stcs(reinterpret_cast<uint4*>(p), r);
}

template <>
__device__ __forceinline__ void store8p<float>(float* p, const f2 v[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(f2_lo(v[0]), f2_hi(v[0]), f2_lo(v[1]), f2_hi(v[1])));
  __stcs(reinterpret_cast<float4*>(p + 4), make_float4(f2_lo(v[2]), f2_hi(v[2]), f2_lo(v[3]), f2_hi(v[3])));
}

// The 8 running sums of a lane, kept as 4 pairs, meeting in the fixed tree.
__device__ __forceinline__ float tree8p(const f2 a[4]) {
  const float c[8] = {f2_lo(a[0]), f2_hi(a[0]), f2_lo(a[1]), f2_hi(a[1]),
                      f2_lo(a[2]), f2_hi(a[2]), f2_lo(a[3]), f2_hi(a[3])};
  return fadd(fadd(fadd(c[0], c[1]), fadd(c[2], c[3])), fadd(fadd(c[4], c[5]), fadd(c[6], c[7])));
}

template <class T, class Src>
__device__ __forceinline__ void load_vec(const T* body, int j, float v[8]) {
  uint4 r[Vec<T>::kRaw];
  Vec<T>::template load<Src>(body + j * kVec, r);
  Vec<T>::unpack(r, v);
}

// ------------------------------------------------------------ unit views
// A unit's body as one warp sees it: lane l owns vectors l, l+32, ..., l+480.
// RegView holds the lane's vectors in registers (loaded once, from shared or
// global memory); MemView reads them from memory on every access.  Both give
// the same values in the same order, so every function below does the same
// arithmetic whichever view it is handed.
template <class T>
struct RegView {
  uint4 w[kVecPerLane][Vec<T>::kRaw];
  int nv;
  template <class Src>
  __device__ __forceinline__ void load(const T* body, int nv_) {
    nv = nv_;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i)
      if (lane + 32 * i < nv) Vec<T>::template load<Src>(body + (lane + 32 * i) * kVec, w[i]);
  }
  // all 16 vectors present (a full unit)
  template <class Src>
  __device__ __forceinline__ void load_full(const T* body) {
    nv = kUnitVecs;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i) Vec<T>::template load<Src>(body + (lane + 32 * i) * kVec, w[i]);
  }
  __device__ __forceinline__ bool has(int i) const { return (int)(threadIdx.x & 31) + 32 * i < nv; }
  __device__ __forceinline__ void get(int i, f2 p[4]) const { Vec<T>::pairs(w[i], p); }
  __device__ __forceinline__ void diff(int i, float k, f2 d[4]) const { Vec<T>::diff(w[i], k, d); }
};

template <class T, class Src>
struct MemView {
  const T* body;
  int nv;
  __device__ __forceinline__ bool has(int i) const { return (int)(threadIdx.x & 31) + 32 * i < nv; }
  __device__ __forceinline__ void get(int i, f2 p[4]) const {
    uint4 r[Vec<T>::kRaw];
    Vec<T>::template load<Src>(body + ((int)(threadIdx.x & 31) + 32 * i) * kVec, r);
    Vec<T>::pairs(r, p);
  }
  __device__ __forceinline__ void diff(int i, float k, f2 d[4]) const {
    uint4 r[Vec<T>::kRaw];
    Vec<T>::template load<Src>(body + ((int)(threadIdx.x & 31) + 32 * i) * kVec, r);
    Vec<T>::diff(r, k, d);
  }
};

// Shifted-sum merge (the parallel-variance combine of Chan, Golub & LeVeque):
// with the shift K and d_i = mean_i - K,  S = sum n_i d_i,  Q = sum (M2_i + n_i d_i^2);
// the union has mean K + S/n and M2 = Q - S*(S/n).
__device__ __forceinline__ void shifted_terms(const Part& a, float K, float& S, float& Q) {
  if (a.n == 0) { S = 0.f; Q = 0.f; return; }
  const float d = fadd(fsub(a.m1, K), a.cn);
  const float nd = fmul((float)a.n, d);
  S = nd;
  Q = fadd(a.m2, fmul(nd, d));
}

__device__ __forceinline__ Part finish_merge(float K, float S, float Q, int64_t n) {
  Part r;
  r.m1 = K;
  r.n = (int)n;
  const float fn = (float)n;
  r.cn = __fdiv_rn(S, fn);
  r.m2 = fsub(Q, fmul(S, r.cn));
  if (r.m2 < 0.f) r.m2 = 0.f;
  return r;
}

// Loads issued together by the lane-strided merges (their sums keep lane order).
constexpr int kMergeBatch = 8;

__device__ __forceinline__ Part ldcg_part(const Part* p) {
  const float4 r = __ldcg(reinterpret_cast<const float4*>(p));
  return Part{r.x, r.y, __float_as_int(r.z), r.w};
}

__device__ __forceinline__ void stcg_unit(Part* p, const Part& a) {
  __stcg(reinterpret_cast<float4*>(p), make_float4(a.m1, a.m2, __int_as_float(a.n), a.cn));
}
__device__ __forceinline__ void stcg_unit(float2* p, float2 a) { __stcg(p, a); }
__device__ __forceinline__ Part ldcg_unit(const Part* p) { return ldcg_part(p); }
__device__ __forceinline__ float2 ldcg_unit(const float2* p) { return __ldcg(p); }

// A merge block cut between two warps' shares, by one warp: lanes lo..hi hold
// the results of units lo..hi of the block (unit i in lane i).  They publish
// them to parts[lane] and add hi-lo+1 arrivals to *ctr; true in the warp whose
// arrivals complete the block's bsz units, which then reads all of parts back
// (ldcg_unit) and merges the block exactly as a warp holding it whole would.
template <class V>
__device__ __forceinline__ bool split_block_arrive(V* parts, uint32_t* ctr, int lo, int hi, int bsz, const V& a) {
  const int lane = threadIdx.x & 31;
  if (lane >= lo && lane <= hi) stcg_unit(parts + lane, a);
  __threadfence();  // every lane's publication before lane 0's arrival
  __syncwarp();
  const uint32_t n = (uint32_t)(hi - lo + 1);
  uint32_t old = 0;
  if (lane == 0) old = atom_add_acq_rel(ctr, n);
  old = __shfl_sync(kFull, old, 0);
  __syncwarp();
  return old + n == (uint32_t)bsz;
}

// Block merge of a block's unit partials, by one warp: lane l holds unit l's
// partial (lanes past the block's size hold an empty one).
__device__ __forceinline__ Part merge_block(const Part a) {
  const float K = __shfl_sync(kFull, fadd(a.m1, a.cn), 0);
  float S, Q;
  shifted_terms(a, K, S, Q);
  const float2 t = warp_sum2(S, Q);
  int n = a.n;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(kFull, n, o);
  return finish_merge(K, t.x, t.y, n);
}

// Merge of the 32 lanes' partials of one unit (total count n), by one warp.
__device__ __forceinline__ Part merge_lanes(const Part a, int n) {
  const float K = __shfl_sync(kFull, fadd(a.m1, a.cn), 0);
  float S, Q;
  shifted_terms(a, K, S, Q);
  const float2 t = warp_sum2(S, Q);
  return finish_merge(K, t.x, t.y, n);
}

// Group merge of its Cg*nb block partials, by one warp: lane l takes blocks l,
// l+32, ... in order, then the butterfly.  Returns the group's moments (mean =
// m1 + cn, M2).  ld(i) gives block i's partial (from global memory, or from
// shared memory in the cluster kernels).
template <class Load>
__device__ __forceinline__ Part merge_group_part_from(Load ld, int64_t nblk, int64_t M) {
  const int lane = threadIdx.x & 31;
  const Part b0 = ld(0);
  const float K = fadd(b0.m1, b0.cn);
  float S = 0.f, Q = 0.f;
  // loads in batches of kMergeBatch (independent), sums in the same order
  for (int64_t i0 = lane; i0 < nblk; i0 += 32 * kMergeBatch) {
    Part v[kMergeBatch];
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (i0 + 32 * j < nblk) v[j] = ld(i0 + 32 * j);
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j) {
      if (i0 + 32 * j < nblk) {
        float s, q;
        shifted_terms(v[j], K, s, q);
        S = fadd(S, s);
        Q = fadd(Q, q);
      }
    }
  }
  const float2 t = warp_sum2(S, Q);
  return finish_merge(K, t.x, t.y, M);
}

// The group merge of Cg*nb contiguous block partials in global memory.
__device__ __forceinline__ Part merge_group_part(const Part* blocks, int64_t nblk, int64_t M) {
  return merge_group_part_from([&](int64_t i) { return ldcg_part(blocks + i); }, nblk, M);
}

// A group's statistics from its moments over M elements: (mean hi, mean lo,
// rstd) with rstd = 1/sqrt(M2/M + eps).
__device__ __forceinline__ float4 group_stats(const Part& g, int64_t M, float eps) {
  const float var = __fdiv_rn(g.m2, (float)M);
  return make_float4(g.m1, g.cn, __frsqrt_rn(fadd(var, eps)), 0.f);
}

__device__ __forceinline__ float4 merge_group(const Part* blocks, int64_t nblk, int64_t M, float eps) {
  return group_stats(merge_group_part(blocks, nblk, M), M, eps);
}

// The gradient arriving at GroupNorm behind a fused ReLU: dy read from `body`,
// zeroed where the forward's result (read from `res`, laid out like dy) is
// <= 0 -- torch's threshold_backward on the saved result.
template <class T, class Src>
struct GatedView {
  const T* body;
  const T* res;
  int nv;
  __device__ __forceinline__ bool has(int i) const { return (int)(threadIdx.x & 31) + 32 * i < nv; }
  __device__ __forceinline__ void get(int i, f2 p[4]) const {
    const int v = (int)(threadIdx.x & 31) + 32 * i;
    uint4 d[Vec<T>::kRaw], o[Vec<T>::kRaw];
    Vec<T>::template load<Src>(body + v * kVec, d);
    Vec<T>::template load<Src>(res + v * kVec, o);
    Vec<T>::gate(o, d);
    Vec<T>::pairs(d, p);
  }
};

// Moments of one unit, by one warp, in one pass over its elements.  Lane l
// first takes a pilot mean K_l of its first kPilotVecs vectors, then sums
// d = x - K_l and d^2 over all its elements: its partial is n_l, mean
// K_l + c/n_l (kept as the pair K_l, c/n_l) and M2 = q - c*(c/n_l).  The
// lanes' partials then merge with the shifted-sum formula below, shifted by
// lane 0's mean.  Shifting by the mean of a quarter of the lane's elements
// bounds the cancellation of the one pass: by Cauchy-Schwarz,
// sum d^2 <= (n_l / pilot) * M2 = 4 * M2 (ScaFFold PR #93 keeps per-tile
// partials merged with Chan's formula; this is that merge one level down).
// kFull: a unit of 4096 body elements and no head or tail scalars, every lane
// full -- the same arithmetic as the general path, without its checks.
constexpr int kPilotVecs = 4;

// The lane's head or tail scalar of a general unit, 0 where it has none.  The
// streaming reduction kernels load it a unit ahead: read where it is used, its
// DRAM latency would stall the warp once per unit.
template <bool kFull, class T>
__device__ __forceinline__ float unit_scalar(const T* __restrict__ x, const URange& q) {
  const int lane = threadIdx.x & 31;
  return !kFull && lane < scalar_count(q) ? IO<T>::load1(x + scalar_index(q, lane)) : 0.f;
}

// sv: the lane's scalar, as unit_scalar gives it.
template <bool kFull, class T, class View>
__device__ __forceinline__ Part unit_moments_sv(const View& u, float sv, const URange& q) {
  if (!kFull && q.n == 0) return Part{0.f, 0.f, 0, 0.f};
  const int lane = threadIdx.x & 31;
  const f2 z2 = f2_splat(0.f);
  f2 pa[4] = {z2, z2, z2, z2};
  int npv = 0;
#pragma unroll
  for (int i = 0; i < kPilotVecs; ++i) {
    if (kFull || u.has(i)) {
      f2 v[4];
      u.get(i, v);
#pragma unroll
      for (int k = 0; k < 4; ++k) pa[k] = f2add(pa[k], v[k]);
      ++npv;
    }
  }
  const bool hs = !kFull && lane < scalar_count(q);
  // the shift: the pilot mean (an exact power-of-two scaling when the lane is full),
  // else the lane's scalar, else 0 for an empty lane
  float K;
  if (kFull) K = fmul(tree8p(pa), 1.f / (float)(kVec * kPilotVecs));
  else K = npv > 0 ? __fdiv_rn(tree8p(pa), (float)(kVec * npv)) : sv;
  f2 c[4] = {z2, z2, z2, z2};
  f2 qq[4] = {z2, z2, z2, z2};
  int nvl = 0;
#pragma unroll
  for (int i = 0; i < kVecPerLane; ++i) {
    if (kFull || u.has(i)) {
      f2 d[4];
      u.diff(i, K, d);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        c[k] = f2add(c[k], d[k]);
        qq[k] = f2fma(d[k], d[k], qq[k]);
      }
      ++nvl;
    }
  }
  float cs = tree8p(c), qs = tree8p(qq);
  if (hs) {
    const float d = fsub(sv, K);
    cs = fadd(cs, d);
    qs = ffma(d, d, qs);
  }
  Part lp;
  lp.m1 = K;
  if (kFull) {
    lp.n = kVec * kVecPerLane;
    lp.cn = fmul(cs, 1.f / (float)(kVec * kVecPerLane));
  } else {
    lp.n = kVec * nvl + (hs ? 1 : 0);
    lp.cn = lp.n > 0 ? __fdiv_rn(cs, (float)lp.n) : 0.f;
  }
  lp.m2 = fsub(qs, fmul(cs, lp.cn));
  if (lp.m2 < 0.f) lp.m2 = 0.f;  // rounding only; NaN is kept
  return merge_lanes(lp, kFull ? kUnitElems : q.n);
}

template <bool kFull, class T, class View>
__device__ __forceinline__ Part unit_moments(const View& u, const T* __restrict__ x, const URange& q) {
  return unit_moments_sv<kFull, T>(u, unit_scalar<kFull, T>(x, q), q);
}

// --------------------------------------------------------------- forward
// The moments of one group as the C ABI exports them (gn3d_moments).
struct Moments {
  long long count;
  float mean_hi, mean_lo, m2, reserved;
};

struct FwdWs {
  Part* parts;      // [units]
  Part* bparts;     // [NC * nb]
  float4* stats;    // [NG] (mean hi, mean lo, rstd, 0)
  uint32_t* bcnt;   // [NC * nb] unit arrivals per block
  uint32_t* gcnt;   // [NG] block arrivals per group
  uint32_t* ready;  // [NG] 1 once stats[g] is published
  Moments* moments; // [NG] or null: export each group's moments instead of its statistics
};

// A completed forward block, by one warp: publish its partial, arrive on the
// group, and merge and publish the group if this completes it.
__device__ __forceinline__ void fwd_block_done(const Plan& p, const FwdWs& ws, int64_t blk, const Part& b,
                                               float eps, float* mean_out, float* rstd_out) {
  const int lane = threadIdx.x & 31;
  if (lane == 0) ws.bparts[blk] = b;
  const int64_t g = (blk / p.nb) / p.Cg;
  if (!warp_arrive_last(ws.gcnt + g, (uint32_t)(p.Cg * p.nb))) return;
  const Part gp = merge_group_part(ws.bparts + g * p.Cg * p.nb, p.Cg * p.nb, p.M);
  if (ws.moments) {  // the group's moments only (a shard's partial statistics)
    if (lane == 0) ws.moments[g] = Moments{(long long)p.M, gp.m1, gp.cn, gp.m2, 0.f};
    return;
  }
  const float4 st = group_stats(gp, p.M, eps);
  if (lane == 0) {
    ws.stats[g] = st;
    if (mean_out) mean_out[g] = fadd(st.x, st.y);
    if (rstd_out) rstd_out[g] = st.z;
    st_release(ws.ready + g, 1u);
  }
}

// NORM of one forward unit, by one warp: y = (x - hi)*sc + (beta - lo*sc), sc = rstd*gamma.
// The fused ReLU of the forward: F.relu of the value the store will round to,
// computed before the store.  Rounding to TO and then v < 0 ? +0 : v keeps -0.0
// for the values that round to -0.0 (below half the smallest bf16 subnormal,
// 2^-134, in magnitude) and gives +0 for every other negative.
template <class TO> struct OutRelu;
template <> struct OutRelu<float> {
  static __device__ __forceinline__ float apply(float v) { return v < 0.f ? 0.f : v; }
};
template <> struct OutRelu<__nv_bfloat16> {
  static __device__ __forceinline__ float apply(float v) {
    return v < 0.f ? (v >= -0x1p-134f ? -0.f : 0.f) : v;
  }
};

template <bool kFull, class TI, class TO, class View, bool kRelu = false>
__device__ __forceinline__ void fwd_norm(const View& u, const TI* __restrict__ x, TO* __restrict__ y,
                                         const URange& q, float4 st, float gam, float bet) {
  const int lane = threadIdx.x & 31;
  const float sc = fmul(st.z, gam);
  const float sh = ffma(-st.y, sc, bet);
  const f2 sc2 = f2_splat(sc), sh2 = f2_splat(sh);
#pragma unroll
  for (int i = 0; i < kVecPerLane; ++i) {
    if (kFull || u.has(i)) {
      f2 v[4];
      u.diff(i, st.x, v);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[k] = f2fma(v[k], sc2, sh2);
        if (kRelu) v[k] = f2_of(OutRelu<TO>::apply(f2_lo(v[k])), OutRelu<TO>::apply(f2_hi(v[k])));
      }
      store8p<TO>(y + q.b0 + (int64_t)(lane + 32 * i) * kVec, v);
    }
  }
  if (!kFull && lane < scalar_count(q)) {
    const int64_t idx = scalar_index(q, lane);
    const float r = ffma(fsub(IO<TI>::load1(x + idx), st.x), sc, sh);
    IO<TO>::store1(y + idx, kRelu ? OutRelu<TO>::apply(r) : r);
  }
}

// -------------------------------------------------------------- backward
struct BwdWs {
  float2* parts;    // [units] (S1, S2)
  float2* bparts;   // [NC * nb]
  float2* rows;     // [NC] per-row (S1, S2)
  float2* coef;     // [NG] (a, b)
  uint32_t* bcnt;   // [NC * nb]
  uint32_t* gcnt;   // [NG]
  uint32_t* ready;  // [NG]
  uint32_t* done;   // [1] groups finalized
};

// S1 = sum dy, S2 = sum dy*(x - mean) of one unit, by one warp, in two steps:
// bwd_accum adds the lane's vectors i0 <= i < i1 to its running sums (a unit's
// body may arrive in parts), bwd_finish meets the sums in the fixed tree, adds
// the lane's scalar and sums the lanes.
template <bool kFull, class T, class XView, class DView>
__device__ __forceinline__ void bwd_accum(const XView& ux, const DView& ud, int i0, int i1, float mu, f2 a1[4],
                                          f2 a2[4]) {
#pragma unroll
  for (int i = 0; i < kVecPerLane; ++i) {
    if (i >= i0 && i < i1 && (kFull || ux.has(i))) {
      f2 xm[4], vd[4];
      ux.diff(i, mu, xm);
      ud.get(i, vd);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        a1[k] = f2add(a1[k], vd[k]);
        a2[k] = f2fma(vd[k], xm[k], a2[k]);
      }
    }
  }
}

// The gradient at scalar element idx: dy, zeroed behind a fused ReLU (res !=
// nullptr) where the forward's result is <= 0.
template <class T>
__device__ __forceinline__ float grad_at(const T* __restrict__ dy, const T* __restrict__ res, int64_t idx) {
  const float d = IO<T>::load1(dy + idx);
  return res && IO<T>::load1(res + idx) <= 0.f ? 0.f : d;
}

// The lane's scalar of a general unit for the backward sums: its gradient and
// its x (zeros where it has none), loaded a unit ahead by the reduction kernel.
struct BwdScalar {
  float d, x;
};
template <bool kFull, class T>
__device__ __forceinline__ BwdScalar bwd_scalar(const T* __restrict__ x, const T* __restrict__ dy,
                                                const T* __restrict__ res, const URange& q) {
  const int lane = threadIdx.x & 31;
  if (kFull || lane >= scalar_count(q)) return BwdScalar{0.f, 0.f};
  const int64_t idx = scalar_index(q, lane);
  return BwdScalar{grad_at(dy, res, idx), IO<T>::load1(x + idx)};
}

template <bool kFull>
__device__ __forceinline__ float2 bwd_finish_sv(const f2 a1[4], const f2 a2[4], BwdScalar sc, const URange& q,
                                                float mu) {
  const int lane = threadIdx.x & 31;
  float s1 = tree8p(a1), s2 = tree8p(a2);
  if (!kFull && lane < scalar_count(q)) {
    s1 = fadd(s1, sc.d);
    s2 = ffma(sc.d, fsub(sc.x, mu), s2);
  }
  return warp_sum2(s1, s2);
}

template <bool kFull, class T>
__device__ __forceinline__ float2 bwd_finish(const f2 a1[4], const f2 a2[4], const T* __restrict__ x,
                                             const T* __restrict__ dy, const URange& q, float mu,
                                             const T* __restrict__ res = nullptr) {
  return bwd_finish_sv<kFull>(a1, a2, bwd_scalar<kFull, T>(x, dy, res, q), q, mu);
}

template <bool kFull, class T, class View>
__device__ __forceinline__ float2 unit_bwd_sums(const View& ux, const View& ud, const T* __restrict__ x,
                                                const T* __restrict__ dy, const URange& q, float mu) {
  const f2 z2 = f2_splat(0.f);
  f2 a1[4] = {z2, z2, z2, z2};
  f2 a2[4] = {z2, z2, z2, z2};
  bwd_accum<kFull, T>(ux, ud, 0, kVecPerLane, mu, a1, a2);
  return bwd_finish<kFull, T>(a1, a2, x, dy, q, mu);
}

// Group finalize of the backward, by one warp: per-row totals of the block sums
// (rows of more than 32 blocks: lane l takes blocks l, l+32, ... of the row,
// then the butterfly; shorter rows: one lane per row, below), then
// A = sum_c gamma_c*S1_c and B = rstd * sum_c gamma_c*S2_c in channel order;
// returns (a, b) = (A/M, B/M).  ld(i) gives block i of the group (row-major:
// row cl, block kb at cl*nb + kb); row(cl, t) receives row cl's totals.
template <class Load, class Row>
__device__ __forceinline__ float2 bwd_group_from(const Plan& p, int64_t g, const float* rstd, const float* gamma,
                                                 Load ld, Row row) {
  const int lane = threadIdx.x & 31;
  float A = 0.f, B = 0.f;
  // rows of at most 32 blocks: lane c takes row c of each pass of 32 rows and
  // forms the row's totals as warp_sum2 would with lane k holding block k
  // (lanes >= nb zero) -- the xor butterfly's additions on the same operands,
  // so the same bits -- then every lane takes the pass's totals in channel
  // order from the row lanes.  A group of many short rows costs one L2 round
  // trip per pass, not one butterfly and round trip per row.
  for (int64_t cl0 = 0; p.nb <= 32 && cl0 < p.Cg; cl0 += 32) {
    const int64_t cl = cl0 + lane;
    float2 t = make_float2(0.f, 0.f);
    float gm = 1.f;
    if (cl < p.Cg) {
      const int64_t bb = cl * p.nb;
      float bx[16], by[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 lo = k < p.nb ? ld(bb + k) : make_float2(0.f, 0.f);
        const float2 hi = k + 16 < p.nb ? ld(bb + k + 16) : make_float2(0.f, 0.f);
        bx[k] = fadd(k < p.nb ? fadd(0.f, lo.x) : 0.f, k + 16 < p.nb ? fadd(0.f, hi.x) : 0.f);
        by[k] = fadd(k < p.nb ? fadd(0.f, lo.y) : 0.f, k + 16 < p.nb ? fadd(0.f, hi.y) : 0.f);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1)
#pragma unroll
        for (int k = 0; k < o; ++k) {
          bx[k] = fadd(bx[k], bx[k + o]);
          by[k] = fadd(by[k], by[k + o]);
        }
      t = make_float2(bx[0], by[0]);
      row(cl, t);
      gm = gamma ? gamma[(g % p.G) * p.Cg + cl] : 1.f;
    }
    const int nr = p.Cg - cl0 < 32 ? (int)(p.Cg - cl0) : 32;
    for (int j = 0; j < nr; ++j) {
      const float tx = __shfl_sync(kFull, t.x, j), ty = __shfl_sync(kFull, t.y, j);
      const float gj = __shfl_sync(kFull, gm, j);
      A = fadd(A, fmul(gj, tx));
      B = fadd(B, fmul(gj, ty));
    }
  }
  for (int64_t cl = 0; p.nb > 32 && cl < p.Cg; ++cl) {
    const int64_t bb = cl * p.nb;
    float s1 = 0.f, s2 = 0.f;
    for (int64_t i0 = lane; i0 < p.nb; i0 += 32 * kMergeBatch) {
      float2 v[kMergeBatch];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j)
        if (i0 + 32 * j < p.nb) v[j] = ld(bb + i0 + 32 * j);
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        if (i0 + 32 * j < p.nb) {
          s1 = fadd(s1, v[j].x);
          s2 = fadd(s2, v[j].y);
        }
      }
    }
    const float2 t = warp_sum2(s1, s2);
    if (lane == 0) row(cl, t);
    const float gm = gamma ? gamma[(g % p.G) * p.Cg + cl] : 1.f;
    A = fadd(A, fmul(gm, t.x));
    B = fadd(B, fmul(gm, t.y));
  }
  B = fmul(rstd[g], B);
  const float fM = (float)p.M;
  return make_float2(__fdiv_rn(A, fM), __fdiv_rn(B, fM));
}

// The streaming kernels' group step: block sums from global memory, row totals
// and (a, b) stored to the workspace.
__device__ __forceinline__ void bwd_group(const Plan& p, const BwdWs& ws, int64_t g, const float* rstd,
                                          const float* gamma) {
  const float2* bp = ws.bparts + g * p.Cg * p.nb;
  float2* rows = ws.rows + g * p.Cg;
  const float2 ab = bwd_group_from(
      p, g, rstd, gamma, [&](int64_t i) { return __ldcg(bp + i); }, [&](int64_t cl, float2 t) { rows[cl] = t; });
  if ((threadIdx.x & 31) == 0) ws.coef[g] = ab;
  // every lane's row stores before lane 0's release arrivals (the warp that
  // completes the last group reads all rows for the parameter gradients)
  __threadfence();
  __syncwarp();
}

// dgamma_c = sum_n rstd[n,g] * S2[n,c], dbeta_c = sum_n S1[n,c], in n order, by one warp.
__device__ __forceinline__ void bwd_param_grads(const Plan& p, const float* rstd, const float2* rows,
                                                float* dgamma, float* dbeta) {
  // one sample: the loads of kMergeBatch channels per lane go out together
  for (int64_t c0 = threadIdx.x & 31; p.N == 1 && c0 < p.C; c0 += 32 * kMergeBatch) {
    float2 rs[kMergeBatch];
    float r[kMergeBatch];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const int64_t c = c0 + 32 * k;
      if (c < p.C) {
        rs[k] = __ldcg(rows + c);
        r[k] = rstd[c / p.Cg];
      }
    }
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      const int64_t c = c0 + 32 * k;
      if (c >= p.C) break;
      const float dg = fadd(0.f, fmul(r[k], rs[k].y)), db = fadd(0.f, rs[k].x);
      if (dgamma) dgamma[c] = dg;
      if (dbeta) dbeta[c] = db;
    }
  }
  for (int64_t c = threadIdx.x & 31; p.N > 1 && c < p.C; c += 32) {
    const int64_t g = c / p.Cg;
    float dg = 0.f, db = 0.f;
    for (int64_t n0 = 0; n0 < p.N; n0 += kMergeBatch) {
      float2 rs[kMergeBatch];
      float r[kMergeBatch];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        if (n0 + j < p.N) {
          rs[j] = __ldcg(rows + (n0 + j) * p.C + c);
          r[j] = rstd[(n0 + j) * p.G + g];
        }
      }
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        if (n0 + j < p.N) {
          dg = fadd(dg, fmul(r[j], rs[j].y));
          db = fadd(db, rs[j].x);
        }
      }
    }
    if (dgamma) dgamma[c] = dg;
    if (dbeta) dbeta[c] = db;
  }
}

// A completed backward block, by one warp (lane l holds unit l's sums): the
// block sums, the group arrival, and the group and parameter-gradient merges
// if this completes them.
__device__ __forceinline__ void bwd_block_done(const Plan& p, const BwdWs& ws, int64_t blk, float2 v,
                                               const float* rstd, const float* gamma, float* dgamma,
                                               float* dbeta) {
  const int lane = threadIdx.x & 31;
  const float2 t = warp_sum2(v.x, v.y);
  if (lane == 0) ws.bparts[blk] = t;
  const int64_t g = (blk / p.nb) / p.Cg;
  if (!warp_arrive_last(ws.gcnt + g, (uint32_t)(p.Cg * p.nb))) return;
  bwd_group(p, ws, g, rstd, gamma);
  if (lane == 0) st_release(ws.ready + g, 1u);
  if (!warp_arrive_last(ws.done, (uint32_t)p.NG)) return;
  bwd_param_grads(p, rstd, ws.rows, dgamma, dbeta);
}

// Per-group coefficients of dx = dy*p1 - (x - mean)*p2 - p3, with p1 = rstd*gamma,
// p2 = rstd^2 * b, p3 = rstd * a  (= rstd*((dy*gamma - a) - xhat*b)).
struct DxCoef {
  float mu, r, a, b;
  bool single;  // one element per group: dx is exactly 0
};

// NORM of one backward unit, by one warp.
template <bool kFull, class T, class XView, class DView>
__device__ __forceinline__ void bwd_norm(const XView& ux, const DView& ud, const T* __restrict__ x,
                                         const T* __restrict__ dy, T* __restrict__ dx, const URange& q,
                                         const DxCoef& k, float gam, const T* __restrict__ res = nullptr) {
  const int lane = threadIdx.x & 31;
  const float p1 = k.single ? 0.f : fmul(k.r, gam);
  const float p2 = k.single ? 0.f : fmul(fmul(k.r, k.r), k.b);
  const float p3 = k.single ? 0.f : fmul(k.r, k.a);
  const f2 p12 = f2_splat(p1), np22 = f2_splat(-p2), np32 = f2_splat(-p3);
#pragma unroll
  for (int i = 0; i < kVecPerLane; ++i) {
    if (kFull || ux.has(i)) {
      f2 xm[4], vd[4];
      ux.diff(i, k.mu, xm);
      ud.get(i, vd);
#pragma unroll
      for (int e = 0; e < 4; ++e) vd[e] = f2fma(vd[e], p12, f2fma(np22, xm[e], np32));
      store8p<T>(dx + q.b0 + (int64_t)(lane + 32 * i) * kVec, vd);
    }
  }
  if (!kFull && lane < scalar_count(q)) {
    const int64_t idx = scalar_index(q, lane);
    const float d = grad_at(dy, res, idx);
    IO<T>::store1(dx + idx, ffma(d, p1, ffma(-p2, fsub(IO<T>::load1(x + idx), k.mu), -p3)));
  }
}

// bwd_norm of a general unit read from global memory, with the loads of kB
// vectors of each tensor issued together before any of them is used: where
// every vector is behind its own bounds check, the compiler otherwise keeps
// each vector's loads after the previous vector's store, one DRAM round trip
// per vector.  The same arithmetic as bwd_norm, element for element.
template <class T, bool kRelu, int kB>
__device__ __forceinline__ void bwd_norm_staged(const T* __restrict__ x, const T* __restrict__ dy,
                                                const T* __restrict__ res, T* __restrict__ dx, const URange& q,
                                                const DxCoef& k, float gam) {
  static_assert(kVecPerLane % kB == 0, "whole batches");
  constexpr int kR = Vec<T>::kRaw;
  const int lane = threadIdx.x & 31;
  const int nv = (int)((q.b1 - q.b0) / kVec);
  const float p1 = k.single ? 0.f : fmul(k.r, gam);
  const float p2 = k.single ? 0.f : fmul(fmul(k.r, k.r), k.b);
  const float p3 = k.single ? 0.f : fmul(k.r, k.a);
  const f2 p12 = f2_splat(p1), np22 = f2_splat(-p2), np32 = f2_splat(-p3);
  // the scalar first: its loads overlap the body's
  const bool hs = lane < scalar_count(q);
  const int64_t sidx = hs ? scalar_index(q, lane) : 0;
  const float sd = hs ? grad_at(dy, kRelu ? res : nullptr, sidx) : 0.f;
  const float sx = hs ? IO<T>::load1(x + sidx) : 0.f;
#pragma unroll
  for (int i0 = 0; i0 < kVecPerLane; i0 += kB) {
    if (lane + 32 * i0 >= nv) break;
    uint4 rx[kB][kR], rd[kB][kR], rr[kRelu ? kB : 1][kR];
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int v = lane + 32 * (i0 + j);
      if (v < nv) {
        Vec<T>::template load<FromGlobal>(x + q.b0 + (int64_t)v * kVec, rx[j]);
        Vec<T>::template load<FromGlobal>(dy + q.b0 + (int64_t)v * kVec, rd[j]);
        if constexpr (kRelu) Vec<T>::template load<FromGlobal>(res + q.b0 + (int64_t)v * kVec, rr[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int v = lane + 32 * (i0 + j);
      if (v < nv) {
        f2 xm[4], vd[4];
        Vec<T>::diff(rx[j], k.mu, xm);
        if constexpr (kRelu) Vec<T>::gate(rr[j], rd[j]);
        Vec<T>::pairs(rd[j], vd);
#pragma unroll
        for (int e = 0; e < 4; ++e) vd[e] = f2fma(vd[e], p12, f2fma(np22, xm[e], np32));
        store8p<T>(dx + q.b0 + (int64_t)v * kVec, vd);
      }
    }
  }
  if (hs) IO<T>::store1(dx + sidx, ffma(sd, p1, ffma(-p2, fsub(sx, k.mu), -p3)));
}

// Row -> channel, in 32 bits when the indices allow it.
__device__ __forceinline__ int64_t channel_of(int64_t row, int64_t C) {
  if (row < 0x7FFFFFFF && C < 0x7FFFFFFF) return (int64_t)((uint32_t)row % (uint32_t)C);
  return row % C;
}

}  // namespace gn3d
