// gn3d_kernels.cuh -- the streaming launch form: two kernels per direction.
//
// Forward  (ScaFFold PR #93 "Optimize GroupNorm": split-group statistics, a
//           corrected two-pass per tile merged with Chan's formula, then a
//           normalize that rounds once on the store, PR #105):
//   k_fwd_stats : each warp takes units in turn (fwd_stat); the warp that
//                 completes a block or a group merges it.
//   k_fwd_norm  : each warp normalizes units, last unit first, so the tail of
//                 the statistics pass is re-read from L2.
// Backward (the same PR's _bwd_finalize/_dwdb_reduce/_dx split):
//   k_bwd_reduce: S1 = sum dy, S2 = sum dy*(x - mean) per unit; group and
//                 parameter-gradient merges by the completing warps.
//   k_bwd_dx    : dx per unit, last unit first.
// These read unit bodies straight from global memory and use exactly the
// arithmetic of the persistent kernels (gn3d_device.cuh), so the two launch
// forms give bit-identical results.
#pragma once
#include "gn3d_device.cuh"

namespace gn3d {

constexpr int kStreamWarps = 8;

__device__ __forceinline__ int64_t warp_global() {
  return (int64_t)blockIdx.x * kStreamWarps + (threadIdx.x >> 5);
}

template <class TI>
__global__ void __launch_bounds__(32 * kStreamWarps)
    k_fwd_stats(const TI* __restrict__ x, Plan p, FwdWs ws, float eps, float* mean_out, float* rstd_out) {
  const int64_t nw = (int64_t)gridDim.x * kStreamWarps;
  for (int64_t u = warp_global(); u < p.units; u += nw) {
    const int64_t row = u / p.R, kr = u - row * p.R;
    const URange q = unit_range_rk(p, row, kr);
    fwd_stat_global<TI>(p, ws, x + q.b0, x, q, u, kr, eps, mean_out, rstd_out);
  }
}

template <class TI, class TO>
__global__ void __launch_bounds__(32 * kStreamWarps)
    k_fwd_norm(const TI* __restrict__ x, TO* __restrict__ y, Plan p, const float4* __restrict__ stats,
               const float* __restrict__ gamma, const float* __restrict__ beta) {
  const int64_t nw = (int64_t)gridDim.x * kStreamWarps;
  for (int64_t i = warp_global(); i < p.units; i += nw) {
    const int64_t u = p.units - 1 - i;
    const int64_t row = u / p.R;
    const URange q = unit_range_rk(p, row, u - row * p.R);
    const int64_t c = channel_of(row, p.C), g = row / p.Cg;
    const MemView<TI, FromGlobal> v{x + q.b0, (int)((q.b1 - q.b0) / kVec)};
    fwd_norm<TI, TO>(v, x, y, q, __ldcg(stats + g), gamma ? gamma[c] : 1.f, beta ? beta[c] : 0.f);
  }
}

template <class T>
__global__ void __launch_bounds__(32 * kStreamWarps)
    k_bwd_reduce(const T* __restrict__ dy, const T* __restrict__ x, Plan p, const float* __restrict__ mean,
                 const float* __restrict__ rstd, const float* __restrict__ gamma, BwdWs ws, float* dgamma,
                 float* dbeta) {
  const int64_t nw = (int64_t)gridDim.x * kStreamWarps;
  for (int64_t u = warp_global(); u < p.units; u += nw) {
    const int64_t row = u / p.R, kr = u - row * p.R;
    const URange q = unit_range_rk(p, row, kr);
    bwd_stat_global<T>(p, ws, x + q.b0, dy + q.b0, x, dy, q, u, kr, mean, rstd, gamma, dgamma, dbeta);
  }
}

template <class T>
__global__ void __launch_bounds__(32 * kStreamWarps)
    k_bwd_dx(const T* __restrict__ dy, const T* __restrict__ x, T* __restrict__ dx, Plan p,
             const float* __restrict__ mean, const float* __restrict__ rstd, const float* __restrict__ gamma,
             const float2* __restrict__ coef) {
  const int64_t nw = (int64_t)gridDim.x * kStreamWarps;
  for (int64_t i = warp_global(); i < p.units; i += nw) {
    const int64_t u = p.units - 1 - i;
    const int64_t row = u / p.R;
    const URange q = unit_range_rk(p, row, u - row * p.R);
    const int64_t c = channel_of(row, p.C), g = row / p.Cg;
    const float2 ab = __ldcg(coef + g);
    const DxCoef k{mean[g], rstd[g], ab.x, ab.y, p.M == 1};
    const int nv = (int)((q.b1 - q.b0) / kVec);
    bwd_norm<T>(MemView<T, FromGlobal>{x + q.b0, nv}, MemView<T, FromGlobal>{dy + q.b0, nv}, x, dy, dx, q, k,
                gamma ? gamma[c] : 1.f);
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
