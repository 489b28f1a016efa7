// gn3d_ndhwc_plan.cuh -- the launch plan of the channels-last (NDHWC) kernels:
// channel ranges, units, merge blocks and pieces, as pure functions of the
// shape (N, C, S = D*H*W, G).  Nothing here depends on the dtype or on the GPU,
// so neither does any reduction order.  Host and device share these functions.
#pragma once
#include <stdint.h>

#ifndef __CUDACC__
#define __host__
#define __device__
#endif

namespace gn3d {

constexpr int kNVec = 8;     // elements per vector: 8 channels of one position
constexpr int kNSpan = 32;   // vectors per channel range (256 channels)
constexpr int kNSteps = 64;  // steps (vectors per lane) per unit, at most
constexpr int kNMinSteps = 16;     // ... and at least (one pilot-shifted chunk)
// Units wanted before a unit is halved.  The forward's statistics kernel merges
// each unit's lanes into channels and pieces, so it keeps long units unless
// they are very few (a quarter of a 152-CTA grid's reduction warps); the
// backward's reduction and dx kernels want one unit per elementwise warp of that
// grid.  The backward takes the statistics as inputs, so the two directions'
// plans need not agree.
constexpr int64_t kNMinUnitsFwd = 304;
constexpr int64_t kNMinUnitsBwd = 2432;
constexpr int kNChunk = 16;  // steps of a lane's first chunk (pilot-shifted)
constexpr int kNPilot = 4;   // steps of the pilot mean
constexpr int kNRedWarps = 8;    // warps per CTA of the statistics and reduction kernels
constexpr int kNElemWarps = 16;  // warps per CTA of the normalize and dx kernels

struct NPlan {
  int64_t N, C, S, G, Cg, NG, M;
  int64_t V;      // vectors per position (C / 8)
  int64_t nr;     // channel ranges
  int64_t steps;  // steps per unit: kNSteps, halved while units are fewer than wanted
  int64_t Pu;     // positions per unit
  int64_t R;      // units per row
  int64_t P;      // pieces (groups met) per range, the most of any range
  int64_t rows;   // N * nr
  int64_t units;  // rows * R
};

// Range r: vectors [32r, 32r + vr), channels [c0, c1), groups g0 .. g1.
struct NRange {
  int vr, lp, lw;
  int64_t c0, c1, g0, g1;
};

__host__ __device__ inline NRange n_range(const NPlan& p, int64_t r) {
  NRange q;
  const int64_t v = p.V - r * kNSpan;
  q.vr = (int)(v < kNSpan ? v : kNSpan);
  q.lp = 32 / q.vr;
  q.lw = q.lp * q.vr;
  q.c0 = r * kNSpan * kNVec;
  q.c1 = q.c0 + (int64_t)kNVec * q.vr;
  q.g0 = q.c0 / p.Cg;
  q.g1 = (q.c1 - 1) / p.Cg;
  return q;
}

// min_units: kNMinUnitsFwd for the forward, kNMinUnitsBwd for the backward.
inline NPlan make_nplan(int64_t N, int64_t C, int64_t S, int64_t G, int64_t min_units) {
  NPlan p;
  p.N = N; p.C = C; p.S = S; p.G = G;
  p.Cg = C / G;
  p.NG = N * G;
  p.M = p.Cg * S;
  p.V = C / kNVec;
  p.nr = (p.V + kNSpan - 1) / kNSpan;
  const int64_t v0 = p.V < kNSpan ? p.V : kNSpan;
  // small volumes: shorter units, so that their work spreads over the grid
  p.steps = kNSteps;
  for (;;) {
    p.Pu = p.steps * (32 / v0);
    p.R = S > 0 ? (S + p.Pu - 1) / p.Pu : 0;
    if (p.steps <= kNMinSteps || N * p.nr * p.R >= min_units) break;
    p.steps /= 2;
  }
  p.P = 0;
  for (int64_t r = 0; r < p.nr; ++r) {
    const NRange q = n_range(p, r);
    if (q.g1 - q.g0 + 1 > p.P) p.P = q.g1 - q.g0 + 1;
  }
  p.rows = N * p.nr;
  p.units = p.rows * p.R;
  return p;
}

// One unit as the calling lane sees it.
struct NUnit {
  int64_t row, k, n, r;
  NRange rg;
  int m, b;          // the lane's position in the step and its vector in the range
  int64_t u0, len;   // first position of the unit and its positions
  int cnt;           // vectors this lane reads
  int64_t off;       // element offset of the lane's first vector
  int64_t step;      // elements between the lane's consecutive vectors (lp * C)
};

__host__ __device__ inline NUnit n_unit(const NPlan& p, int64_t u, int lane) {
  NUnit q;
  q.row = u / p.R;
  q.k = u - q.row * p.R;
  q.n = q.row / p.nr;
  q.r = q.row - q.n * p.nr;
  q.rg = n_range(p, q.r);
  q.m = lane / q.rg.vr;
  q.b = lane - q.m * q.rg.vr;
  q.u0 = q.k * p.Pu;
  q.len = p.S - q.u0 < p.Pu ? p.S - q.u0 : p.Pu;
  const bool active = lane < q.rg.lw && q.len > q.m;
  q.cnt = active ? (int)((q.len - q.m + q.rg.lp - 1) / q.rg.lp) : 0;
  q.off = (q.n * p.S + q.u0 + q.m) * p.C + q.rg.c0 + (int64_t)kNVec * q.b;
  q.step = (int64_t)q.rg.lp * p.C;
  return q;
}

// Channels [c0, c1) of piece j (group g0 + j) of a range, relative to the range.
__host__ __device__ inline void n_piece(const NPlan& p, const NRange& rg, int64_t j, int64_t& c0, int64_t& c1) {
  const int64_t g = rg.g0 + j;
  const int64_t a = g * p.Cg, e = a + p.Cg;
  c0 = (a > rg.c0 ? a : rg.c0) - rg.c0;
  c1 = (e < rg.c1 ? e : rg.c1) - rg.c0;
}

// Ring form (one channel range, so a unit is one contiguous span of len*C
// elements and step i its 8*lw elements from i*8*lw on): the steps of unit u,
// and part `part` of kPS steps -- elements [e0, e0 + n) -- returning whether it
// is the unit's last part.
__host__ __device__ inline int n_unit_steps(const NPlan& p, const NRange& rg, int64_t u) {
  const int64_t k = u % p.R, len = p.S - k * p.Pu < p.Pu ? p.S - k * p.Pu : p.Pu;
  return (int)((len + rg.lp - 1) / rg.lp);
}

__host__ __device__ inline bool n_ring_part(const NPlan& p, const NRange& rg, int64_t u, int part, int kPS,
                                            int64_t& e0, int64_t& n) {
  const int64_t k = u % p.R, s = u / p.R;
  const int64_t len = p.S - k * p.Pu < p.Pu ? p.S - k * p.Pu : p.Pu;
  const int64_t span = (int64_t)kPS * kNVec * rg.lw, total = len * p.C;
  e0 = (s * p.S + k * p.Pu) * p.C + part * span;
  const int64_t rest = total - part * span;
  n = rest < span ? rest : span;
  return (int64_t)(part + 1) * span >= total;
}

}  // namespace gn3d
