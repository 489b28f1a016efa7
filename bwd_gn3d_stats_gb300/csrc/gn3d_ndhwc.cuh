// gn3d_ndhwc.cuh -- GroupNorm over channels-last (NDHWC) volumes: the plan and
// the four streaming kernels (statistics, normalize, backward reduction, dx).
//
// Layout.  x[n][s][c], s = (d*H + h)*W + w -- the channels_last_3d memory
// format of an NCDHW tensor (ScaFFold's Triton GroupNorm reads channels-last
// activations: a dense run of positions x C channels, viewed as (G, C/G)).
// Sample n is S*C contiguous elements; group g of sample n is the column block
// [g*Cg, (g+1)*Cg) of that S x C matrix.  C is a multiple of 8, so a vector (8
// elements: 16 B of bf16, 32 B of fp32) holds 8 channels of one position.
//
// Ranges and lanes.  The channels are cut into ranges of up to kNSpan vectors
// (256 channels).  In a range of vr vectors a warp takes lp = 32 / vr positions
// per step: lane l = m*vr + b reads vector b of position m of the step, so a
// warp-wide load is lp*vr*16 contiguous bytes of bf16 (one position's range
// slice when vr = 32) and each lane keeps the same 8 channels throughout
// (lanes >= lp*vr idle).
//
// Units, blocks, groups.  Row (n, r) -- sample n, range r -- is cut into units of
// Pu = kNSteps * lp0 positions (lp0: the lp of range 0, the widest), one warp
// per unit, at most kNSteps vectors per lane.  B consecutive units of a row form
// a merge block.  Statistics merge in a fixed tree that depends on the shape
// alone: lane -> channel (the lp lanes of a channel, pairwise) -> piece (the
// channels of one group inside the range) per unit -> piece per block (the
// warp that completes the block) -> group (the last CTA to finish).  The
// backward keeps per-channel sums (the weight gradient needs them): unit ->
// block -> row (n, c) -> group coefficients and parameter gradients.
//
// Every floating-point step uses the round-to-nearest intrinsics of
// gn3d_device.cuh, so the result bits depend on the shape only.
#pragma once
#include "gn3d_device.cuh"
#include "gn3d_ndhwc_plan.cuh"
#include "gn3d_sync.cuh"

namespace gn3d {

// ------------------------------------------------------------- workspaces
struct NFwdWs {
  Part* upart;     // [rows][P][R]  unit pieces
  Part* bpart;     // [rows][P][nb] block pieces
  float4* stats;   // [NG] (mean hi, mean lo, rstd, 0)
  uint32_t* bcnt;  // [nblk] unit arrivals per block
  uint32_t* done;  // [1] CTAs finished
};

struct NBwdWs {
  float2* usum;    // [N*C][R]  unit sums per channel (S1, S2)
  float2* bsum;    // [N*C][nb] block sums per channel
  float2* rows;    // [N*C]     row totals
  float2* coef;    // [NG]      (a, b)
  uint32_t* bcnt;  // [nblk]
  uint32_t* done;  // [1]
};

// ------------------------------------------------------------- lane sums
// Vectors of each tensor loaded together, per kernel (statistics and reduction:
// 8 warps, up to 255 registers; normalize and dx: 16 warps, up to 128).
template <class T, bool kRelu = false> struct NBatch {
  static constexpr int kRaw = Vec<T>::kRaw;
  static constexpr int kStats = 16 / kRaw;
  static constexpr int kNorm = 8 / kRaw;
  static constexpr int kReduce = (kRelu ? 4 : 8) / kRaw;
  static constexpr int kDx = (kRelu ? 2 : 4) / kRaw;
};

// (v - k) for the 8 elements of a vector as pairs, each pair with its own shift.
template <class T>
__device__ __forceinline__ void n_diff(const uint4 r[Vec<T>::kRaw], const f2 k[4], f2 d[4]) {
  f2 v[4];
  Vec<T>::pairs(r, v);
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = f2sub(v[e], k[e]);
}

__device__ __forceinline__ float n_slot(const f2 a[4], int s) { return s & 1 ? f2_hi(a[s >> 1]) : f2_lo(a[s >> 1]); }

// Moments of the lane's elements of each of its 8 channels, one pass.  The
// first chunk (kNChunk vectors) is shifted by its pilot mean (the first kNPilot
// vectors); the rest by the first chunk's mean.  With shift K and d = x - K,
// a chunk's sums c = sum d, q = sum d^2 give M2 = q - c*(c/n); a shift that is
// the mean of a quarter of the chunk keeps q <= 5 M2 (Cauchy-Schwarz), and the
// second chunk, shifted by the mean of the first 16 of its up to 64 elements,
// the same bound (ScaFFold PR #93: per-tile corrected two-pass partials merged
// with Chan's formula; here the pass is one, the correction its shift).
// Returns the 8 slot partials as (m1, cn, m2) pairs and the count.
template <class T>
__device__ __forceinline__ int n_lane_moments(const T* __restrict__ x, const NUnit& q, f2 m1[4], f2 cn[4],
                                              f2 m2[4]) {
  constexpr int kB = NBatch<T>::kStats, kRaw = Vec<T>::kRaw;
  const f2 z2 = f2_splat(0.f);
  const T* base = x + q.off;
  const int cnt = q.cnt;
  const int nA = cnt < kNChunk ? cnt : kNChunk;
  f2 K[4] = {z2, z2, z2, z2}, c[4] = {z2, z2, z2, z2}, s2[4] = {z2, z2, z2, z2};
#pragma unroll
  for (int t0 = 0; t0 < kNChunk; t0 += kB) {
    if (t0 < nA) {
      uint4 w[kB][kRaw];
#pragma unroll
      for (int t = 0; t < kB; ++t)
        if (t0 + t < nA) Vec<T>::template load<FromGlobal>(base + (int64_t)(t0 + t) * q.step, w[t]);
      if (t0 == 0) {
        f2 pa[4] = {z2, z2, z2, z2};
#pragma unroll
        for (int t = 0; t < kNPilot; ++t) {
          if (t < nA) {
            f2 v[4];
            Vec<T>::pairs(w[t], v);
#pragma unroll
            for (int e = 0; e < 4; ++e) pa[e] = f2add(pa[e], v[e]);
          }
        }
        const int np = nA < kNPilot ? nA : kNPilot;
        const f2 inv = f2_splat(np == kNPilot ? 1.f / (float)kNPilot : __frcp_rn((float)np));
#pragma unroll
        for (int e = 0; e < 4; ++e) K[e] = f2fma(pa[e], inv, z2);
      }
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t0 + t < nA) {
          f2 d[4];
          n_diff<T>(w[t], K, d);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            c[e] = f2add(c[e], d[e]);
            s2[e] = f2fma(d[e], d[e], s2[e]);
          }
        }
      }
    }
  }
  if (nA == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) m1[e] = cn[e] = m2[e] = z2;
    return 0;
  }
  // the first chunk's partial
  const f2 invA = f2_splat(nA == kNChunk ? 1.f / (float)kNChunk : __frcp_rn((float)nA));
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    m1[e] = K[e];
    cn[e] = f2fma(c[e], invA, z2);
    m2[e] = f2sub(s2[e], f2fma(c[e], cn[e], z2));
  }
  if (cnt > nA) {
    // the rest, shifted by the first chunk's mean
    f2 K2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      K2[e] = f2add(m1[e], cn[e]);
      c[e] = z2;
      s2[e] = z2;
    }
    for (int t0 = kNChunk; t0 < cnt; t0 += kB) {
      uint4 w[kB][kRaw];
#pragma unroll
      for (int t = 0; t < kB; ++t)
        if (t0 + t < cnt) Vec<T>::template load<FromGlobal>(base + (int64_t)(t0 + t) * q.step, w[t]);
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t0 + t < cnt) {
          f2 d[4];
          n_diff<T>(w[t], K2, d);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            c[e] = f2add(c[e], d[e]);
            s2[e] = f2fma(d[e], d[e], s2[e]);
          }
        }
      }
    }
    // merge: the first chunk's terms about K2, plus the rest's sums
    const f2 fa = f2_splat((float)nA);
    const f2 inv = f2_splat(cnt == kNSteps ? 1.f / (float)kNSteps : __frcp_rn((float)cnt));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const f2 d = f2add(f2sub(m1[e], K2[e]), cn[e]);
      const f2 nd = f2fma(fa, d, z2);
      const f2 S = f2add(nd, c[e]);
      const f2 Q = f2add(f2fma(nd, d, m2[e]), s2[e]);
      m1[e] = K2[e];
      cn[e] = f2fma(S, inv, z2);
      m2[e] = f2sub(Q, f2fma(S, cn[e], z2));
    }
  }
  return cnt;
}

// Sum over the lp lanes that share a vector b (lane m*vr + b), pairwise over m;
// the totals land in the m = 0 lanes.  All 32 lanes call.
__device__ __forceinline__ float n_msum(float v, const NRange& rg, int m) {
  for (int s = 1; s < rg.lp; s <<= 1) {
    const float o = __shfl_down_sync(kFull, v, s * rg.vr);
    if ((m & (2 * s - 1)) == 0 && m + s < rg.lp) v = fadd(v, o);
  }
  return v;
}

__device__ __forceinline__ float n_shifted_s(float m1, float cn, int n, float K, float& Q, float m2) {
  if (n == 0) {
    Q = 0.f;
    return 0.f;
  }
  const float d = fadd(fsub(m1, K), cn);
  const float nd = fmul((float)n, d);
  Q = fadd(m2, fmul(nd, d));
  return nd;
}

// ------------------------------------------------------- forward statistics
// Error-free transformations (Knuth's TwoSum, the fma TwoProduct): s + e = a + b
// and p + e = a * b exactly.
__device__ __forceinline__ float n_two_sum(float a, float b, float& e) {
  const float s = fadd(a, b);
  const float bb = fsub(s, a);
  e = fadd(fsub(a, fsub(s, bb)), fsub(b, bb));
  return s;
}

__device__ __forceinline__ float n_two_prod(float a, float b, float& e) {
  const float p = fmul(a, b);
  e = ffma(a, b, -p);
  return p;
}

// The unit's channel partials (in shared memory, warp-private) merged into
// pieces: piece j is written to upart.  Lanes work in segments of L lanes per
// piece (L a power of two); sub-lane s takes the piece's channels s, s+L, ...
// and the segment sums pairwise.  The channels of a group can have means far
// apart, so this merge is the one place where the shifted terms n*(mean - K)
// are large: the shift K is the centre of the piece's channel means (their
// plain average, the same bits in every sub-lane), and S = sum n*(mean - K) is
// carried as an unevaluated pair, each term split exactly (TwoSum, TwoProduct),
// so S is exact but for the rounding of the small low parts.
__device__ __forceinline__ void n_unit_pieces(const NPlan& p, const NUnit& q, const Part* sp, Part* upart) {
  const int lane = threadIdx.x & 31;
  const int64_t np = q.rg.g1 - q.rg.g0 + 1;
  int L = 1;
  while (L * 2 * np <= 32) L *= 2;
  const int segs = 32 / L, sg = lane / L, s = lane - sg * L;
  for (int64_t j0 = 0; j0 < np; j0 += segs) {
    const int64_t j = j0 + sg;
    int64_t c0 = 0, c1 = 0;
    if (j < np) n_piece(p, q.rg, j, c0, c1);
    float K = 0.f, Sh = 0.f, Sl = 0.f, Q = 0.f;
    if (c1 > c0) {
      for (int64_t c = c0; c < c1; ++c) K = fadd(K, fadd(sp[c].m1, sp[c].cn));
      K = fmul(K, __frcp_rn((float)(c1 - c0)));
      for (int64_t c = c0 + s; c < c1; c += L) {
        const Part a = sp[c];
        const float fn = (float)a.n;
        float ed, ep, es;
        const float dh = n_two_sum(a.m1, -K, ed);  // dh + ed = m1 - K
        const float dl = fadd(ed, a.cn);           // mean - K = dh + dl
        const float ph = n_two_prod(fn, dh, ep);
        Sh = n_two_sum(Sh, ph, es);
        Sl = fadd(Sl, fadd(es, ffma(fn, dl, ep)));
        const float d = fadd(dh, dl);
        Q = fadd(Q, fadd(a.m2, fmul(fmul(fn, d), d)));
      }
    }
    for (int o = 1; o < L; o <<= 1) {
      const float ho = __shfl_down_sync(kFull, Sh, o), lo = __shfl_down_sync(kFull, Sl, o);
      const float qo = __shfl_down_sync(kFull, Q, o);
      if ((s & (2 * o - 1)) == 0) {
        float e;
        Sh = n_two_sum(Sh, ho, e);
        Sl = fadd(Sl, fadd(lo, e));
        Q = fadd(Q, qo);
      }
    }
    if (s == 0 && j < np)
      upart[(q.row * p.P + j) * p.R + q.k] = finish_merge(K, fadd(Sh, Sl), Q, q.len * (c1 - c0));
  }
}

// Sum over the B lanes of a segment (lanes cl*B .. cl*B + B - 1, B a power of
// two): an xor butterfly inside the segment, every lane ends with the total.
__device__ __forceinline__ float n_segsum(float v, int B) {
  for (int o = B >> 1; o > 0; o >>= 1) v = fadd(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Block kb of row `row` is complete: merge each piece's unit partials into
// bpart, by one warp.  The warp works as 32/B segments of B lanes, one piece
// per segment, lane kk of a segment holding unit kk of the block.
__device__ __forceinline__ void n_fwd_block(const NPlan& p, const NFwdWs& ws, int64_t row, int64_t kb) {
  const int lane = threadIdx.x & 31, B = (int)p.B, per = 32 / B, cl = lane / B, kk = lane - cl * B;
  const NRange rg = n_range(p, row % p.nr);
  const int64_t np = rg.g1 - rg.g0 + 1;
  const int bsz = n_block_size(p, kb);
  const int64_t pos = n_block_positions(p, kb);
  for (int64_t j0 = 0; j0 < np; j0 += (int64_t)per * kMergeBatch) {
    Part v[kMergeBatch];
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t) {
      const int64_t j = j0 + (int64_t)t * per + cl;
      v[t] = j < np && kk < bsz ? ldcg_part(ws.upart + ((row * p.P + j) * p.R + kb * p.B + kk))
                                : Part{0.f, 0.f, 0, 0.f};
    }
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t) {
      if (j0 + (int64_t)t * per >= np) break;
      const int64_t j = j0 + (int64_t)t * per + cl;
      const float K = __shfl_sync(kFull, fadd(v[t].m1, v[t].cn), cl * B);
      float S, Q;
      shifted_terms(v[t], K, S, Q);
      S = n_segsum(S, B);
      Q = n_segsum(Q, B);
      if (kk == 0 && j < np) {
        int64_t c0, c1;
        n_piece(p, rg, j, c0, c1);
        ws.bpart[(row * p.P + j) * p.nb + kb] = finish_merge(K, S, Q, pos * (c1 - c0));
      }
    }
  }
}

// Group gi = n*G + g from its block pieces (every range the group meets, block
// by block), by one warp: lane l takes parts l, l+32, ... in order.
__device__ __forceinline__ void n_fwd_group(const NPlan& p, const NFwdWs& ws, int64_t gi, float eps, float* mean_out,
                                            float* rstd_out) {
  const int lane = threadIdx.x & 31;
  const int64_t n = gi / p.G, g = gi - n * p.G;
  const int64_t r_lo = (g * p.Cg) / (kNSpan * kVec), r_hi = ((g + 1) * p.Cg - 1) / (kNSpan * kVec);
  const int64_t total = (r_hi - r_lo + 1) * p.nb;
  auto at = [&](int64_t i) {
    const int64_t r = r_lo + i / p.nb, kb = i - (i / p.nb) * p.nb;
    const int64_t j = g - n_range(p, r).g0;
    return ws.bpart + ((n * p.nr + r) * p.P + j) * p.nb + kb;
  };
  const Part b0 = ldcg_part(at(0));
  const float K = fadd(b0.m1, b0.cn);
  float S = 0.f, Q = 0.f;
  for (int64_t i0 = lane; i0 < total; i0 += 32 * kMergeBatch) {
    Part v[kMergeBatch];
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t)
      if (i0 + 32 * t < total) v[t] = ldcg_part(at(i0 + 32 * t));
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t) {
      if (i0 + 32 * t < total) {
        float s, q;
        shifted_terms(v[t], K, s, q);
        S = fadd(S, s);
        Q = fadd(Q, q);
      }
    }
  }
  const float2 tq = warp_sum2(S, Q);
  const Part gp = finish_merge(K, tq.x, tq.y, p.M);
  const float rs = __frsqrt_rn(fadd(__fdiv_rn(gp.m2, (float)p.M), eps));
  if (lane == 0) {
    ws.stats[gi] = make_float4(gp.m1, gp.cn, rs, 0.f);
    if (mean_out) mean_out[gi] = fadd(gp.m1, gp.cn);
    if (rstd_out) rstd_out[gi] = rs;
  }
}

// Everything this CTA wrote is published; true in the last CTA to finish, which
// then sees every other CTA's results.
__device__ __forceinline__ bool n_last_cta(uint32_t* done) {
  __shared__ uint32_t last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atom_add_acq_rel(done, 1u) + 1u == gridDim.x ? 1u : 0u;
  __syncthreads();
  const bool l = last != 0;
  if (l) __threadfence();
  return l;
}

// Reduction warp w = warp*grid + cta takes units w, w + W, w + 2W, ... (W =
// grid * kNRedWarps).  An elementwise warp takes the units of reduction warp
// warp % kNRedWarps of the same CTA, last first, every kSplit-th: what that
// warp read last is read again first, while it is still in L2.
__device__ __forceinline__ int64_t n_first_unit() {
  return (int64_t)(threadIdx.x >> 5) * gridDim.x + blockIdx.x;
}

struct NOwned {
  static constexpr int kSplit = kNElemWarps / kNRedWarps;
  int64_t u0, W, t;  // the owner's first unit, its stride, the current step (-1: done)
  __device__ __forceinline__ NOwned(const NPlan& p) {
    const int warp = threadIdx.x >> 5;
    u0 = (int64_t)(warp % kNRedWarps) * gridDim.x + blockIdx.x;
    W = (int64_t)gridDim.x * kNRedWarps;
    t = u0 < p.units ? (p.units - 1 - u0) / W - warp / kNRedWarps : -1;
  }
  __device__ __forceinline__ bool more() const { return t >= 0; }
  __device__ __forceinline__ int64_t unit() const { return u0 + t * W; }
  __device__ __forceinline__ void next() { t -= kSplit; }
};

template <class T>
__global__ void __launch_bounds__(32 * kNRedWarps, 1)
    k_ndhwc_stats(const T* __restrict__ x, NPlan p, NFwdWs ws, float eps, float* mean_out, float* rstd_out) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Part* sp = reinterpret_cast<Part*>(smem) + (size_t)warp * (kNSpan * kVec);
  pdl_launch_dependents();
  const int64_t W = (int64_t)gridDim.x * kNRedWarps;
  for (int64_t u = n_first_unit(); u < p.units; u += W) {
    const NUnit q = n_unit(p, u, lane);
    f2 m1[4], cn[4], m2[4];
    const int cnt = n_lane_moments<T>(x, q, m1, cn, m2);
    // the lp lanes of each channel: shift by the m = 0 lane's mean, sum pairwise
#pragma unroll
    for (int sl = 0; sl < 8; ++sl) {
      const float a1 = n_slot(m1, sl), ac = n_slot(cn, sl), a2 = n_slot(m2, sl);
      const float K = __shfl_sync(kFull, fadd(a1, ac), q.b);
      float Q;
      float S = n_shifted_s(a1, ac, cnt, K, Q, a2 < 0.f ? 0.f : a2);
      S = n_msum(S, q.rg, q.m);
      Q = n_msum(Q, q.rg, q.m);
      if (q.m == 0 && lane < q.rg.vr) sp[kVec * q.b + sl] = finish_merge(K, S, Q, q.len);
    }
    __syncwarp();
    n_unit_pieces(p, q, sp, ws.upart);
    // the pieces (written by several lanes) are published before lane 0's arrival
    __threadfence();
    __syncwarp();
    const int64_t kb = q.k / p.B;
    if (warp_arrive_last(ws.bcnt + q.row * p.nb + kb, (uint32_t)n_block_size(p, kb))) n_fwd_block(p, ws, q.row, kb);
  }
  if (!n_last_cta(ws.done)) return;
  for (int64_t gi = warp; gi < p.NG; gi += kNRedWarps) n_fwd_group(p, ws, gi, eps, mean_out, rstd_out);
}

// ------------------------------------------------------------- normalize
// Per-channel coefficients of the lane's 8 channels: y = (x - hi)*sc + sh with
// sc = rstd*gamma, sh = beta - lo*sc (mean = hi + lo), the forward's formula.
template <class TI, class TO, bool kRelu>
__global__ void __launch_bounds__(32 * kNElemWarps, 1)
    k_ndhwc_norm(const TI* __restrict__ x, TO* __restrict__ y, NPlan p, const float4* __restrict__ stats,
                 const float* __restrict__ gamma, const float* __restrict__ beta) {
  constexpr int kB = NBatch<TI>::kNorm, kRaw = Vec<TI>::kRaw;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  for (NOwned own(p); own.more(); own.next()) {
    const int64_t u = own.unit();
    const NUnit q = n_unit(p, u, lane);
    if (q.cnt == 0) continue;
    f2 hi[4], sc[4], sh[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float h[2], a[2], b[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int64_t c = q.rg.c0 + kVec * q.b + 2 * e + t;
        const float4 st = __ldcg(stats + q.n * p.G + c / p.Cg);
        const float gm = gamma ? gamma[c] : 1.f, bt = beta ? beta[c] : 0.f;
        h[t] = st.x;
        a[t] = fmul(st.z, gm);
        b[t] = ffma(-st.y, a[t], bt);
      }
      hi[e] = f2_of(h[0], h[1]);
      sc[e] = f2_of(a[0], a[1]);
      sh[e] = f2_of(b[0], b[1]);
    }
    const TI* xb = x + q.off;
    TO* yb = y + q.off;
    for (int t0 = 0; t0 < q.cnt; t0 += kB) {
      uint4 w[kB][kRaw];
#pragma unroll
      for (int t = 0; t < kB; ++t)
        if (t0 + t < q.cnt) Vec<TI>::template load<FromGlobal>(xb + (int64_t)(t0 + t) * q.step, w[t]);
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t0 + t < q.cnt) {
          f2 v[4];
          n_diff<TI>(w[t], hi, v);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[e] = f2fma(v[e], sc[e], sh[e]);
            if (kRelu) v[e] = f2_of(OutRelu<TO>::apply(f2_lo(v[e])), OutRelu<TO>::apply(f2_hi(v[e])));
          }
          store8p<TO>(yb + (int64_t)(t0 + t) * q.step, v);
        }
      }
    }
  }
}

// ------------------------------------------------------------- backward
// The lane's gradient vector: dy, zeroed where the fused ReLU's result <= 0.
template <class T, bool kRelu>
__device__ __forceinline__ void n_grad(const T* dy, const T* res, int64_t o, uint4 d[Vec<T>::kRaw]) {
  Vec<T>::template load<FromGlobal>(dy + o, d);
  if constexpr (kRelu) {
    uint4 r[Vec<T>::kRaw];
    Vec<T>::template load<FromGlobal>(res + o, r);
    Vec<T>::gate(r, d);
  }
}

// Block kb of row `row` is complete: per channel of the range, the sum of its
// unit sums, by one warp working as 32/B segments (one channel per segment,
// lane kk holding unit kk of the block).
__device__ __forceinline__ void n_bwd_block(const NPlan& p, const NBwdWs& ws, int64_t row, int64_t kb) {
  const int lane = threadIdx.x & 31, B = (int)p.B, per = 32 / B, cl = lane / B, kk = lane - cl * B;
  const int64_t n = row / p.nr;
  const NRange rg = n_range(p, row - n * p.nr);
  const int bsz = n_block_size(p, kb);
  for (int64_t c0 = rg.c0; c0 < rg.c1; c0 += (int64_t)per * kMergeBatch) {
    float2 v[kMergeBatch];
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t) {
      const int64_t c = c0 + (int64_t)t * per + cl;
      v[t] = c < rg.c1 && kk < bsz ? __ldcg(ws.usum + (n * p.C + c) * p.R + kb * p.B + kk) : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int t = 0; t < kMergeBatch; ++t) {
      if (c0 + (int64_t)t * per >= rg.c1) break;
      const int64_t c = c0 + (int64_t)t * per + cl;
      const float s1 = n_segsum(v[t].x, B), s2 = n_segsum(v[t].y, B);
      if (kk == 0 && c < rg.c1) ws.bsum[(n * p.C + c) * p.nb + kb] = make_float2(s1, s2);
    }
  }
}

template <class T, bool kRelu>
__global__ void __launch_bounds__(32 * kNRedWarps, 1)
    k_ndhwc_reduce(const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ res, NPlan p,
                   const float* __restrict__ mean, const float* __restrict__ rstd, const float* __restrict__ gamma,
                   NBwdWs ws, float* dgamma, float* dbeta) {
  constexpr int kB = NBatch<T, kRelu>::kReduce, kRaw = Vec<T>::kRaw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  const int64_t W = (int64_t)gridDim.x * kNRedWarps;
  const f2 z2 = f2_splat(0.f);
  for (int64_t u = n_first_unit(); u < p.units; u += W) {
    const NUnit q = n_unit(p, u, lane);
    f2 mu[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t c = q.rg.c0 + kVec * q.b + 2 * e;
      const float* mg = mean + q.n * p.G;
      mu[e] = q.cnt ? f2_of(mg[c / p.Cg], mg[(c + 1) / p.Cg]) : z2;
    }
    f2 a1[4] = {z2, z2, z2, z2}, a2[4] = {z2, z2, z2, z2};
    for (int t0 = 0; t0 < q.cnt; t0 += kB) {
      uint4 wx[kB][kRaw], wd[kB][kRaw];
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t0 + t < q.cnt) {
          const int64_t o = q.off + (int64_t)(t0 + t) * q.step;
          Vec<T>::template load<FromGlobal>(x + o, wx[t]);
          n_grad<T, kRelu>(dy, res, o, wd[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t0 + t < q.cnt) {
          f2 xm[4], vd[4];
          n_diff<T>(wx[t], mu, xm);
          Vec<T>::pairs(wd[t], vd);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            a1[e] = f2add(a1[e], vd[e]);
            a2[e] = f2fma(vd[e], xm[e], a2[e]);
          }
        }
      }
    }
#pragma unroll
    for (int sl = 0; sl < 8; ++sl) {
      const float s1 = n_msum(n_slot(a1, sl), q.rg, q.m), s2 = n_msum(n_slot(a2, sl), q.rg, q.m);
      if (q.m == 0 && lane < q.rg.vr)
        ws.usum[(q.n * p.C + q.rg.c0 + kVec * q.b + sl) * p.R + q.k] = make_float2(s1, s2);
    }
    __threadfence();
    __syncwarp();
    const int64_t kb = q.k / p.B;
    if (warp_arrive_last(ws.bcnt + q.row * p.nb + kb, (uint32_t)n_block_size(p, kb))) n_bwd_block(p, ws, q.row, kb);
  }
  if (!n_last_cta(ws.done)) return;
  // row totals (n, c): warp per row, lane l takes blocks l, l+32, ...
  for (int64_t rc = warp; rc < p.N * p.C; rc += kNRedWarps) {
    const float2* bp = ws.bsum + rc * p.nb;
    float s1 = 0.f, s2 = 0.f;
    for (int64_t i0 = lane; i0 < p.nb; i0 += 32 * kMergeBatch) {
      float2 v[kMergeBatch];
#pragma unroll
      for (int t = 0; t < kMergeBatch; ++t)
        if (i0 + 32 * t < p.nb) v[t] = __ldcg(bp + i0 + 32 * t);
#pragma unroll
      for (int t = 0; t < kMergeBatch; ++t) {
        if (i0 + 32 * t < p.nb) {
          s1 = fadd(s1, v[t].x);
          s2 = fadd(s2, v[t].y);
        }
      }
    }
    const float2 t = warp_sum2(s1, s2);
    if (lane == 0) ws.rows[rc] = t;
  }
  __syncthreads();
  // group coefficients: A = sum_c gamma_c*S1_c and B = rstd * sum_c gamma_c*S2_c
  // in channel order; a = A/M, b = B/M
  for (int64_t gi = threadIdx.x; gi < p.NG; gi += blockDim.x) {
    const int64_t n = gi / p.G, g = gi - n * p.G;
    float A = 0.f, Bs = 0.f;
    for (int64_t cl = 0; cl < p.Cg; ++cl) {
      const int64_t c = g * p.Cg + cl;
      const float2 t = __ldcg(ws.rows + n * p.C + c);
      const float gm = gamma ? gamma[c] : 1.f;
      A = fadd(A, fmul(gm, t.x));
      Bs = fadd(Bs, fmul(gm, t.y));
    }
    Bs = fmul(rstd[gi], Bs);
    const float fM = (float)p.M;
    ws.coef[gi] = make_float2(__fdiv_rn(A, fM), __fdiv_rn(Bs, fM));
  }
  // dgamma_c = sum_n rstd[n,g]*S2[n,c], dbeta_c = sum_n S1[n,c], in n order
  for (int64_t c = threadIdx.x; c < p.C; c += blockDim.x) {
    const int64_t g = c / p.Cg;
    float dg = 0.f, db = 0.f;
    for (int64_t n = 0; n < p.N; ++n) {
      const float2 t = __ldcg(ws.rows + n * p.C + c);
      dg = fadd(dg, fmul(rstd[n * p.G + g], t.y));
      db = fadd(db, t.x);
    }
    if (dgamma) dgamma[c] = dg;
    if (dbeta) dbeta[c] = db;
  }
}

// dx = dy*p1 - (x - mean)*p2 - p3 per channel, with p1 = rstd*gamma,
// p2 = rstd^2 * b, p3 = rstd * a (a single-element group has dx = 0).
template <class T, bool kRelu>
__global__ void __launch_bounds__(32 * kNElemWarps, 1)
    k_ndhwc_dx(const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ res, T* __restrict__ dx,
               NPlan p, const float* __restrict__ mean, const float* __restrict__ rstd,
               const float* __restrict__ gamma, const float2* __restrict__ coef) {
  constexpr int kB = NBatch<T, kRelu>::kDx, kRaw = Vec<T>::kRaw;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const bool single = p.M == 1;
  for (NOwned own(p); own.more(); own.next()) {
    const int64_t u = own.unit();
    const NUnit q = n_unit(p, u, lane);
    if (q.cnt == 0) continue;
    f2 mu[4], p1[4], np2[4], np3[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float a[4][2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int64_t c = q.rg.c0 + kVec * q.b + 2 * e + t;
        const int64_t gi = q.n * p.G + c / p.Cg;
        const float2 ab = __ldcg(coef + gi);
        const float r = rstd[gi], gm = gamma ? gamma[c] : 1.f;
        a[0][t] = mean[gi];
        a[1][t] = single ? 0.f : fmul(r, gm);
        a[2][t] = single ? 0.f : -fmul(fmul(r, r), ab.y);
        a[3][t] = single ? 0.f : -fmul(r, ab.x);
      }
      mu[e] = f2_of(a[0][0], a[0][1]);
      p1[e] = f2_of(a[1][0], a[1][1]);
      np2[e] = f2_of(a[2][0], a[2][1]);
      np3[e] = f2_of(a[3][0], a[3][1]);
    }
    for (int t0 = 0; t0 < q.cnt; t0 += kB) {
      uint4 wx[kB][kRaw], wd[kB][kRaw];
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t0 + t < q.cnt) {
          const int64_t o = q.off + (int64_t)(t0 + t) * q.step;
          Vec<T>::template load<FromGlobal>(x + o, wx[t]);
          n_grad<T, kRelu>(dy, res, o, wd[t]);
        }
      }
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t0 + t < q.cnt) {
          f2 xm[4], vd[4];
          n_diff<T>(wx[t], mu, xm);
          Vec<T>::pairs(wd[t], vd);
#pragma unroll
          for (int e = 0; e < 4; ++e) vd[e] = f2fma(vd[e], p1[e], f2fma(np2[e], xm[e], np3[e]));
          store8p<T>(dx + q.off + (int64_t)(t0 + t) * q.step, vd);
        }
      }
    }
  }
}

}  // namespace gn3d
