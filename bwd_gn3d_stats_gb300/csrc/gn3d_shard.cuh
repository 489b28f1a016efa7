// gn3d_shard.cuh -- global statistics for a volume split into shards (spatial
// sharding, e.g. one D-slab per rank): the small kernels around the streaming
// ones that turn per-shard partial results into the whole volume's.
//
// Forward: each shard's per-group moments (count, mean as hi + lo, M2 -- the
// group merge of the statistics kernel, stopped before rstd) are exchanged by
// the caller and combined here in rank order with the shifted-sum form of
// Chan's parallel-variance merge, the same form every merge of the library
// uses; the combined moments give (mean, rstd) and the normalize pass runs on
// the shard with them.  Backward: each shard's per-row sums S1 = sum dy, S2 =
// sum dy*(x - mean) at the global statistics are exchanged and added in rank
// order; the group coefficients a, b and dgamma, dbeta follow from the totals
// exactly as in the backward's group step, and the dx pass runs on the shard.
// (The ScaFFold GroupNorm pages keep statistics per shard under DistConv and
// leave global statistics open; this is the exchange that closes it.)
//
// With one shard every step is the identity, and the results are bit-identical
// to gn3d_forward / gn3d_backward on the whole tensor.
#pragma once
#include "gn3d_device.cuh"

namespace gn3d {

// Combine K shards' moments of each group in rank order: shards[k * ng + g].
__global__ void k_moments_combine(const Moments* __restrict__ shards, int64_t K, int64_t ng,
                                  Moments* __restrict__ out) {
  const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (g >= ng) return;
  const Moments m0 = shards[g];
  if (K == 1) {
    out[g] = m0;
    return;
  }
  // shifted sums about the first non-empty shard's mean: S = sum n_k d_k,
  // Q = sum (M2_k + n_k d_k^2), d_k = (mean_k - K); then mean = K + S/n and
  // M2 = Q - S*(S/n)
  float Ksh = 0.f;
  for (int64_t k = 0; k < K; ++k) {
    const Moments m = shards[k * ng + g];
    if (m.count > 0) {
      Ksh = fadd(m.mean_hi, m.mean_lo);
      break;
    }
  }
  float S = 0.f, Q = 0.f;
  long long n = 0;
  for (int64_t k = 0; k < K; ++k) {
    const Moments m = shards[k * ng + g];
    if (m.count <= 0) continue;
    const float d = fadd(fsub(m.mean_hi, Ksh), m.mean_lo);
    const float nd = fmul((float)m.count, d);
    S = fadd(S, nd);
    Q = fadd(Q, fadd(m.m2, fmul(nd, d)));
    n += m.count;
  }
  Moments r{n, Ksh, 0.f, 0.f, 0.f};
  if (n > 0) {
    r.mean_lo = __fdiv_rn(S, (float)n);
    r.m2 = fsub(Q, fmul(S, r.mean_lo));
    if (r.m2 < 0.f) r.m2 = 0.f;
  }
  out[g] = r;
}

// (mean hi, mean lo, rstd) of each group from its moments, as the group step of
// the statistics kernel forms them; mean and rstd outputs where requested.
__global__ void k_stats_from_moments(const Moments* __restrict__ m, int64_t ng, float eps, float4* __restrict__ stats,
                                     float* mean, float* rstd) {
  const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (g >= ng) return;
  const Moments v = m[g];
  const Part p{v.mean_hi, v.m2, (int)v.count, v.mean_lo};
  const float4 st = v.count > 0 ? group_stats(p, v.count, eps) : make_float4(0.f, 0.f, __frsqrt_rn(eps), 0.f);
  stats[g] = st;
  if (mean) mean[g] = fadd(st.x, st.y);
  if (rstd) rstd[g] = st.z;
}

// Sum K shards' per-row sums in rank order: shards[k * nc + row].
__global__ void k_sums_combine(const float2* __restrict__ shards, int64_t K, int64_t nc, float2* __restrict__ out) {
  const int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (r >= nc) return;
  float2 t = shards[r];
  for (int64_t k = 1; k < K; ++k) {
    const float2 v = shards[k * nc + r];
    t.x = fadd(t.x, v.x);
    t.y = fadd(t.y, v.y);
  }
  out[r] = t;
}

// Per group (a, b) from the row totals, over M elements of the whole group: A =
// sum_c gamma_c*S1_c and B = rstd * sum_c gamma_c*S2_c in channel order, a =
// A/M, b = B/M -- the backward's group step, operation for operation.
__global__ void k_coef_from_sums(Plan p, const float2* __restrict__ rows, const float* __restrict__ rstd,
                                 const float* __restrict__ gamma, int64_t M, float2* __restrict__ coef) {
  const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (g >= p.NG) return;
  float A = 0.f, B = 0.f;
  for (int64_t cl = 0; cl < p.Cg; ++cl) {
    const float2 t = rows[g * p.Cg + cl];
    const float gm = gamma ? gamma[(g % p.G) * p.Cg + cl] : 1.f;
    A = fadd(A, fmul(gm, t.x));
    B = fadd(B, fmul(gm, t.y));
  }
  B = fmul(rstd[g], B);
  const float fM = (float)M;
  coef[g] = make_float2(__fdiv_rn(A, fM), __fdiv_rn(B, fM));
}

// dgamma and dbeta from the row totals (one warp).
__global__ void k_param_grads(Plan p, const float* __restrict__ rstd, const float2* __restrict__ rows, float* dgamma,
                              float* dbeta) {
  bwd_param_grads(p, rstd, rows, dgamma, dbeta);
}

}  // namespace gn3d
