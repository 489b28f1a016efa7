// gn3d_kernels.cuh -- the GroupNorm forward/backward kernels (unit-streaming form).
//
// Forward  (ScaFFold PR #93 "Optimize GroupNorm": split-group statistics, a
//           corrected two-pass per tile merged with Chan's formula, then a
//           normalize that rounds once on the store, PR #105):
//   fwd_stats : per unit (count, mean, M2); the CTA that completes a group
//               merges its partials in a fixed tree and writes mean/rstd.
//   fwd_norm  : y = (x - mean) * (rstd*gamma_c) + beta_c, units in reverse order
//               so the tail of the statistics pass is re-read from L2.
// Backward (the same PR's _bwd_finalize/_dwdb_reduce/_dx split):
//   bwd_reduce: per unit S1 = sum dy, S2 = sum dy*(x - mean); the CTA that
//               completes a group forms per-row sums, the group coefficients
//               a = sum(g)/M, b = sum(g*xhat)/M, and the CTA that completes the
//               last group forms dgamma/dbeta in fixed n order.
//   bwd_dx    : dx = rstd * ((dy*gamma - a) - xhat*b), units in reverse order.
//
// Completion is detected with integer counters only (no float atomics); the
// counters live in per-call scratch that the host zeroes before the launch.
#pragma once
#include "gn3d_device.cuh"

namespace gn3d {

struct FwdWs {
  Part* parts;      // [units]
  float4* stats;    // [NG] (mean hi, mean lo, rstd, 0)
  unsigned* cnt;    // [NG] arrivals per group
};

struct BwdWs {
  float2* parts;    // [units] (S1, S2)
  float2* rows;     // [NC] per-row (S1, S2)
  float2* coef;     // [NG] (a, b)
  unsigned* cnt;    // [NG + 1] arrivals per group, then groups done
};

// Corrected two-pass moments of one unit held in registers: m1 = sum/n, then
// c = sum(x - m1), q = sum((x - m1)^2); the unit mean is m1 + c/n (kept as the
// pair) and M2 = q - c*c/n (the correction term keeps M2 exact to first order
// in the error of m1).
template <class T>
__device__ __forceinline__ Part unit_moments(const UnitRegs<T>& u, int n, float2* red) {
  Part m = {0.f, 0.f, 0, 0.f};
  if (n == 0) return m;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i)
    if (u.vok[i]) {
#pragma unroll
      for (int e = 0; e < 8; ++e) s = fadd(s, u.v[i][e]);
    }
  if (u.sok) s = fadd(s, u.s);
  const float fn = (float)n;
  const float m1 = __fdiv_rn(block_sum2(s, 0.f, red).x, fn);
  float c = 0.f, q = 0.f;
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i)
    if (u.vok[i]) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float d = fsub(u.v[i][e], m1);
        c = fadd(c, d);
        q = ffma(d, d, q);
      }
    }
  if (u.sok) {
    const float d = fsub(u.s, m1);
    c = fadd(c, d);
    q = ffma(d, d, q);
  }
  const float2 t = block_sum2(c, q, red);
  m.m1 = m1;
  m.cn = __fdiv_rn(t.x, fn);
  m.m2 = fsub(t.y, fmul(t.x, m.cn));
  if (m.m2 < 0.f) m.m2 = 0.f;  // rounding only; NaN is kept
  m.n = n;
  return m;
}

// Finalize of one group from its unit partials: mean, rstd = 1/sqrt(M2/M + eps)
// (fp64, rounded once to fp32); the workspace keeps the mean as a hi/lo fp32 pair.
__device__ __forceinline__ void finalize_group(const Plan& p, int64_t ng, const Part* parts, float eps,
                                               float4* stats, float* mean_out, float* rstd_out,
                                               double2* sh) {
  const GroupMoments m = combine_parts(parts + ng * p.upg, p.upg, p.M, sh);
  if (threadIdx.x == 0) {
    const double var = __ddiv_rn(m.m2, (double)p.M);
    const float r = (float)__drcp_rn(__dsqrt_rn(dadd(var, (double)eps)));
    const float hi = (float)m.mean;
    const float lo = (float)dadd(m.mean, -(double)hi);
    stats[ng] = make_float4(hi, lo, r, 0.f);
    if (mean_out) mean_out[ng] = hi;
    if (rstd_out) rstd_out[ng] = r;
  }
}

template <class TI>
__global__ void __launch_bounds__(kThreads) k_fwd_stats(const TI* __restrict__ x, Plan p, FwdWs ws,
                                                        float eps, float* mean_out, float* rstd_out) {
  __shared__ float2 red[kWarps];
  __shared__ double2 msh[kWarps];
  __shared__ int s_last;
  for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
    const URange q = unit_range(p, u);
    UnitRegs<TI> r;
    r.load(x, q);
    const Part m = unit_moments(r, q.n, red);
    const int64_t ng = q.row / p.Cg;
    if (threadIdx.x == 0) {
      ws.parts[u] = m;
      __threadfence();
      s_last = atomicAdd(&ws.cnt[ng], 1u) == (unsigned)(p.upg - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      finalize_group(p, ng, ws.parts, eps, ws.stats, mean_out, rstd_out, msh);
    }
    __syncthreads();
  }
}

template <class TI, class TO>
__global__ void __launch_bounds__(kThreads) k_fwd_norm(const TI* __restrict__ x, TO* __restrict__ y, Plan p,
                                                       const float4* __restrict__ stats,
                                                       const float* __restrict__ gamma,
                                                       const float* __restrict__ beta) {
  for (int64_t i = blockIdx.x; i < p.units; i += gridDim.x) {
    const int64_t u = p.units - 1 - i;
    const URange q = unit_range(p, u);
    const int64_t c = q.row % p.C, ng = q.row / p.Cg;
    const float4 st = stats[ng];
    const float sc = gamma ? fmul(st.z, gamma[c]) : st.z;
    const float sh = beta ? beta[c] : 0.f;
    const int64_t nv = (q.b1 - q.b0) / kVec;
    float v[kVecPerThread][8];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t j = threadIdx.x + (int64_t)k * kThreads;
      if (j < nv) IO<TI>::load8(x + q.b0 + j * kVec, v[k]);
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t j = threadIdx.x + (int64_t)k * kThreads;
      if (j < nv) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[k][e] = ffma(fsub(fsub(v[k][e], st.x), st.y), sc, sh);
        IO<TO>::store8(y + q.b0 + j * kVec, v[k]);
      }
    }
    if ((int)threadIdx.x < scalar_count(q)) {
      const int64_t idx = scalar_index(q, threadIdx.x);
      IO<TO>::store1(y + idx, ffma(fsub(fsub(IO<TI>::load1(x + idx), st.x), st.y), sc, sh));
    }
  }
}

// Backward partial sums of one unit: S1 = sum dy, S2 = sum dy*(x - mean).
template <class T>
__device__ __forceinline__ float2 unit_bwd_sums(const UnitRegs<T>& d, const UnitRegs<T>& xr, float mu,
                                                float2* red) {
  float s1 = 0.f, s2 = 0.f;
#pragma unroll
  for (int i = 0; i < kVecPerThread; ++i)
    if (d.vok[i]) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        s1 = fadd(s1, d.v[i][e]);
        s2 = ffma(d.v[i][e], fsub(xr.v[i][e], mu), s2);
      }
    }
  if (d.sok) {
    s1 = fadd(s1, d.s);
    s2 = ffma(d.s, fsub(xr.s, mu), s2);
  }
  return block_sum2(s1, s2, red);
}

// Group finalize of the backward: per-row totals (warp w takes rows w, w+8, ...;
// lane l sums units l, l+32, ... in order, then a shfl_down tree), then
// A = sum_c gamma_c*S1_c and B = rstd * sum_c gamma_c*S2_c in channel order.
__device__ __forceinline__ void bwd_finalize_group(const Plan& p, int64_t ng, const float* rstd,
                                                   const float* gamma, BwdWs ws) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t cl = w; cl < p.Cg; cl += kWarps) {
    const int64_t row = ng * p.Cg + cl;
    const float2* pr = ws.parts + row * p.R;
    float s1 = 0.f, s2 = 0.f;
    for (int64_t k = lane; k < p.R; k += 32) {
      const float2 v = __ldcg(pr + k);
      s1 = fadd(s1, v.x);
      s2 = fadd(s2, v.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float a = __shfl_down_sync(0xFFFFFFFFu, s1, o);
      const float b = __shfl_down_sync(0xFFFFFFFFu, s2, o);
      if (lane + o < 32) { s1 = fadd(s1, a); s2 = fadd(s2, b); }
    }
    if (lane == 0) ws.rows[row] = make_float2(s1, s2);
  }
  __threadfence_block();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t g = ng % p.G;
    float A = 0.f, B = 0.f;
    for (int64_t cl = 0; cl < p.Cg; ++cl) {
      const float2 rs = ws.rows[ng * p.Cg + cl];
      const float gm = gamma ? gamma[g * p.Cg + cl] : 1.f;
      A = fadd(A, fmul(gm, rs.x));
      B = fadd(B, fmul(gm, rs.y));
    }
    B = fmul(rstd[ng], B);
    const float fM = (float)p.M;
    ws.coef[ng] = make_float2(__fdiv_rn(A, fM), __fdiv_rn(B, fM));
  }
}

// dgamma_c = sum_n rstd[n,g] * S2[n,c], dbeta_c = sum_n S1[n,c], in n order.
__device__ __forceinline__ void bwd_param_grads(const Plan& p, const float* rstd, const float2* rows,
                                                float* dgamma, float* dbeta) {
  for (int64_t c = threadIdx.x; c < p.C; c += kThreads) {
    const int64_t g = c / p.Cg;
    float dg = 0.f, db = 0.f;
    for (int64_t n = 0; n < p.N; ++n) {
      const float2 rs = __ldcg(rows + n * p.C + c);
      dg = fadd(dg, fmul(rstd[n * p.G + g], rs.y));
      db = fadd(db, rs.x);
    }
    if (dgamma) dgamma[c] = dg;
    if (dbeta) dbeta[c] = db;
  }
}

template <class T>
__global__ void __launch_bounds__(kThreads) k_bwd_reduce(const T* __restrict__ dy, const T* __restrict__ x,
                                                         Plan p, const float* __restrict__ mean,
                                                         const float* __restrict__ rstd,
                                                         const float* __restrict__ gamma, BwdWs ws,
                                                         float* dgamma, float* dbeta) {
  __shared__ float2 red[kWarps];
  __shared__ int s_last, s_all;
  for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
    const URange q = unit_range(p, u);
    const int64_t ng = q.row / p.Cg;
    UnitRegs<T> rd, rx;
    rd.load(dy, q);
    rx.load(x, q);
    const float2 s = unit_bwd_sums(rd, rx, mean[ng], red);
    if (threadIdx.x == 0) {
      ws.parts[u] = s;
      __threadfence();
      s_last = atomicAdd(&ws.cnt[ng], 1u) == (unsigned)(p.upg - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      bwd_finalize_group(p, ng, rstd, gamma, ws);
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        s_all = atomicAdd(&ws.cnt[p.NG], 1u) == (unsigned)(p.NG - 1);
      }
      __syncthreads();
      if (s_all) {
        __threadfence();
        bwd_param_grads(p, rstd, ws.rows, dgamma, dbeta);
      }
    }
    __syncthreads();
  }
}

template <class T>
__global__ void __launch_bounds__(kThreads) k_bwd_dx(const T* __restrict__ dy, const T* __restrict__ x,
                                                     T* __restrict__ dx, Plan p,
                                                     const float* __restrict__ mean,
                                                     const float* __restrict__ rstd,
                                                     const float* __restrict__ gamma,
                                                     const float2* __restrict__ coef) {
  for (int64_t i = blockIdx.x; i < p.units; i += gridDim.x) {
    const int64_t u = p.units - 1 - i;
    const URange q = unit_range(p, u);
    const int64_t c = q.row % p.C, ng = q.row / p.Cg;
    const float mu = mean[ng], r = rstd[ng];
    const float gm = gamma ? gamma[c] : 1.f;
    const float2 ab = coef[ng];
    const int64_t nv = (q.b1 - q.b0) / kVec;
    float vd[kVecPerThread][8], vx[kVecPerThread][8];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t j = threadIdx.x + (int64_t)k * kThreads;
      if (j < nv) {
        IO<T>::load8(dy + q.b0 + j * kVec, vd[k]);
        IO<T>::load8(x + q.b0 + j * kVec, vx[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t j = threadIdx.x + (int64_t)k * kThreads;
      if (j < nv) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float t = fsub(fmul(vd[k][e], gm), ab.x);   // never contracted: exact 0 when M == 1
          const float xh = fmul(fsub(vx[k][e], mu), r);
          vd[k][e] = fmul(r, ffma(-xh, ab.y, t));
        }
        IO<T>::store8(dx + q.b0 + j * kVec, vd[k]);
      }
    }
    if ((int)threadIdx.x < scalar_count(q)) {
      const int64_t idx = scalar_index(q, threadIdx.x);
      const float t = fsub(fmul(IO<T>::load1(dy + idx), gm), ab.x);
      const float xh = fmul(fsub(IO<T>::load1(x + idx), mu), r);
      IO<T>::store1(dx + idx, fmul(r, ffma(-xh, ab.y, t)));
    }
  }
}

// Empty groups (M == 0): mean 0, rstd 1/sqrt(eps).
__global__ void k_fill_empty_stats(float* mean, float* rstd, int64_t ng, float eps) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i < ng) {
    if (mean) mean[i] = 0.f;
    if (rstd) rstd[i] = __frsqrt_rn(eps);
  }
}

}  // namespace gn3d
