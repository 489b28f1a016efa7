// gn3d_ndhwc.cuh -- GroupNorm over channels-last (NDHWC) volumes: six kernels,
// three per direction (streaming statistics, finalize, normalize; streaming
// reduction, finalize, dx), chained by dependent launches.  The plan is in
// gn3d_ndhwc_plan.cuh.
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
// Units and groups.  Row (n, r) -- sample n, range r -- is cut into units of
// Pu = steps * lp0 positions (lp0: the lp of range 0, the widest; steps = kNSteps,
// halved down to kNMinSteps for small volumes), one warp per unit, at most
// steps vectors per lane.  Statistics merge in a fixed tree
// that depends on the shape alone: lane -> channel (the lp lanes of a channel,
// pairwise) -> piece (the channels of one group inside the range), per unit,
// in the streaming kernel; the pieces -> group in the finalize kernel, one CTA
// per chunk of kNFinChunk units, then the chunk partials in order.  The
// backward keeps per-channel sums (the weight gradient needs them): unit -> row
// (n, c) the same way -> group coefficients and parameter gradients.  With one
// channel range (C <= 256) the streaming kernels read through warp-private
// rings of bulk copies; otherwise with vector loads.  They only store their
// unit results: a round trip
// to L2 (an arrival counter, a merge's loads) costs microseconds while the
// stream saturates DRAM, and a warp that waits for one falls behind.
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
  uint32_t* never; // [1] zero, never set (the forced-timeout test waits on it)
  Part* upart;     // [rows][P][R]       unit pieces
  Part* fpart;     // [NG][maxr * nkc]   finalize chunk partials
  uint32_t* gcnt;  // [NG]               finalize chunks done per group
  float4* stats;   // [NG]               (mean hi, mean lo, rstd, 0)
};

struct NBwdWs {
  float2* usum;    // [N*C][R]    unit sums per channel (S1, S2)
  float2* rpart;   // [N*C][nkc]  finalize chunk sums
  uint32_t* rcnt;  // [N*C]       finalize chunks done per row
  float2* rows;    // [N*C]       row totals
  float2* coef;    // [NG]        (a, b)
  uint32_t* done;  // [1]         rows finished
};

// ------------------------------------------------------------- lane sums
// Vectors of each tensor loaded together, per kernel (statistics and reduction:
// 8 warps, up to 255 registers; normalize and dx: 16 warps, up to 128).
template <class T, bool kRelu = false> struct NBatch {
  static constexpr int kRaw = Vec<T>::kRaw;
  static constexpr int kStats = 16 / kRaw;
  static constexpr int kNorm = 16 / kRaw;
  static constexpr int kReduce = (kRelu ? 4 : 8) / kRaw;
  static constexpr int kDx = (kRelu ? 4 : 8) / kRaw;
};

// (lo - k.lo, hi - k.hi) for the two bf16 halves of w: one mixed-precision
// subtraction per element (bf16 operand, fp32 shift and result, rounded once --
// the value of widening first).
__device__ __forceinline__ f2 n_bf16_pair_minus(uint32_t w, f2 k) {
  f2 d;
  asm("{\n .reg .b16 l, h;\n .reg .f32 kl, kh, dl, dh;\n mov.b32 {l, h}, %1;\n mov.b64 {kl, kh}, %2;\n"
      " sub.rn.f32.bf16 dl, l, kl;\n sub.rn.f32.bf16 dh, h, kh;\n mov.b64 %0, {dl, dh};\n}"
      : "=l"(d)
      : "r"(w), "l"(k));
  return d;
}

// (v - k) for the 8 elements of a vector as pairs, each pair with its own shift.
template <class T>
__device__ __forceinline__ void n_diff(const uint4 r[Vec<T>::kRaw], const f2 k[4], f2 d[4]) {
  if constexpr (Vec<T>::kRaw == 1) {
    d[0] = n_bf16_pair_minus(r[0].x, k[0]);
    d[1] = n_bf16_pair_minus(r[0].y, k[1]);
    d[2] = n_bf16_pair_minus(r[0].z, k[2]);
    d[3] = n_bf16_pair_minus(r[0].w, k[3]);
  } else {
    f2 v[4];
    Vec<T>::pairs(r, v);
#pragma unroll
    for (int e = 0; e < 4; ++e) d[e] = f2sub(v[e], k[e]);
  }
}

__device__ __forceinline__ float n_slot(const f2 a[4], int s) { return s & 1 ? f2_hi(a[s >> 1]) : f2_lo(a[s >> 1]); }

// Moments of the lane's elements of each of its 8 channels, one pass.  The
// first chunk (kNChunk vectors) is shifted by its pilot mean (the first kNPilot
// vectors); the rest by the first chunk's mean.  With shift K and d = x - K,
// a chunk's sums c = sum d, q = sum d^2 give M2 = q - c*(c/n); a shift that is
// the mean of a quarter of the chunk keeps q <= 5 M2 (Cauchy-Schwarz), and the
// rest, shifted by the mean of the first 16 of the lane's up to kNSteps
// elements, q <= (kNSteps / 16 + 1) M2 (ScaFFold PR #93: per-tile corrected two-pass partials merged
// with Chan's formula; here the pass is one, the correction its shift).
// The vectors arrive in batches of kB consecutive steps (kB divides kNChunk),
// from global memory or from a shared-memory slot; the arithmetic is the same.
template <class T>
struct NMoments {
  f2 K[4], c[4], s2[4];  // the current chunk: shift and sums
  f2 c1[4], q1[4];       // second set of sums (odd steps), added to c, s2 at a chunk's end
  f2 m1[4], cn[4], m2[4];  // the first chunk's partial, then the lane's (pairs of channels)
  int nA = 0;

  // Steps t0 .. t0 + nv - 1 of the lane (nv >= 1), w[t] holding step t0 + t.
  template <int kB>
  __device__ __forceinline__ void batch(const uint4 (&w)[kB][Vec<T>::kRaw], int t0, int nv, int cnt) {
    static_assert(kNChunk % kB == 0 && kB >= kNPilot, "batches inside chunks, the pilot in the first");
    const f2 z2 = f2_splat(0.f);
    if (t0 == 0) {
      f2 pa[4] = {z2, z2, z2, z2};
#pragma unroll
      for (int t = 0; t < kNPilot; ++t) {
        if (t < nv) {
          f2 v[4];
          Vec<T>::pairs(w[t], v);
#pragma unroll
          for (int e = 0; e < 4; ++e) pa[e] = f2add(pa[e], v[e]);
        }
      }
      const int np = nv < kNPilot ? nv : kNPilot;
      const f2 inv = f2_splat(np == kNPilot ? 1.f / (float)kNPilot : __frcp_rn((float)np));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        K[e] = f2fma(pa[e], inv, z2);
        c[e] = s2[e] = c1[e] = q1[e] = z2;
      }
    }
    // even steps into (c, s2), odd steps into (c1, q1): two chains per sum
#pragma unroll
    for (int t = 0; t < kB; ++t) {
      if (t < nv) {
        f2 d[4];
        n_diff<T>(w[t], K, d);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (t & 1) {
            c1[e] = f2add(c1[e], d[e]);
            q1[e] = f2fma(d[e], d[e], q1[e]);
          } else {
            c[e] = f2add(c[e], d[e]);
            s2[e] = f2fma(d[e], d[e], s2[e]);
          }
        }
      }
    }
    // the first chunk ends with step min(cnt, kNChunk) - 1: its partial, and the
    // rest's shift (its mean)
    const int endA = cnt < kNChunk ? cnt : kNChunk;
    if (t0 < kNChunk && t0 + nv >= endA) {
      nA = endA;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        c[e] = f2add(c[e], c1[e]);
        s2[e] = f2add(s2[e], q1[e]);
      }
      const f2 invA = f2_splat(nA == kNChunk ? 1.f / (float)kNChunk : __frcp_rn((float)nA));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        m1[e] = K[e];
        cn[e] = f2fma(c[e], invA, z2);
        m2[e] = f2sub(s2[e], f2fma(c[e], cn[e], z2));
        K[e] = f2add(m1[e], cn[e]);
        c[e] = s2[e] = c1[e] = q1[e] = z2;
      }
    }
  }

  // After every step: the lane's partial of each channel in (m1, cn, m2); count cnt.
  __device__ __forceinline__ void finish(int cnt) {
    const f2 z2 = f2_splat(0.f);
    if (cnt == 0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) m1[e] = cn[e] = m2[e] = z2;
      return;
    }
    if (cnt == nA) return;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      c[e] = f2add(c[e], c1[e]);
      s2[e] = f2add(s2[e], q1[e]);
    }
    // merge: the first chunk's terms about the rest's shift K, plus the rest's sums
    const f2 fa = f2_splat((float)nA);
    const f2 inv = f2_splat(cnt == kNSteps ? 1.f / (float)kNSteps : __frcp_rn((float)cnt));
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const f2 d = f2add(f2sub(m1[e], K[e]), cn[e]);
      const f2 nd = f2fma(fa, d, z2);
      const f2 S = f2add(nd, c[e]);
      const f2 Q = f2add(f2fma(nd, d, m2[e]), s2[e]);
      m1[e] = K[e];
      cn[e] = f2fma(S, inv, z2);
      m2[e] = f2sub(Q, f2fma(S, cn[e], z2));
    }
  }
};

// The direct form: the lane's vectors read from global memory, kB at a time.
template <class T>
__device__ __forceinline__ void n_lane_moments(const T* __restrict__ x, const NUnit& q, NMoments<T>& mom) {
  constexpr int kB = NBatch<T>::kStats, kRaw = Vec<T>::kRaw;
  const T* base = x + q.off;
  for (int t0 = 0; t0 < q.cnt; t0 += kB) {
    const int nv = q.cnt - t0 < kB ? q.cnt - t0 : kB;
    uint4 w[kB][kRaw];
#pragma unroll
    for (int t = 0; t < kB; ++t)
      if (t < nv) Vec<T>::template load<FromGlobal>(base + (int64_t)(t0 + t) * q.step, w[t]);
    mom.batch(w, t0, nv, q.cnt);
  }
  mom.finish(q.cnt);
}

// Sums over the lp lanes that share a vector b (lane m*vr + b), pairwise over
// m, of kV values at once (the shuffles of one level issue together); the
// totals land in the m = 0 lanes.  All 32 lanes call.
template <int kV>
__device__ __forceinline__ void n_msum(float (&v)[kV], const NRange& rg, int m) {
  for (int s = 1; s < rg.lp; s <<= 1) {
    float o[kV];
#pragma unroll
    for (int i = 0; i < kV; ++i) o[i] = __shfl_down_sync(kFull, v[i], s * rg.vr);
    if ((m & (2 * s - 1)) == 0 && m + s < rg.lp) {
#pragma unroll
      for (int i = 0; i < kV; ++i) v[i] = fadd(v[i], o[i]);
    }
  }
}

// The merged partial from shift K and sums S, Q over n elements, with inv = 1/n
// (rounded; exact when n is a power of two).
__device__ __forceinline__ Part n_finish(float K, float S, float Q, int n, float inv) {
  Part r;
  r.m1 = K;
  r.n = n;
  r.cn = fmul(S, inv);
  r.m2 = fsub(Q, fmul(S, r.cn));
  if (r.m2 < 0.f) r.m2 = 0.f;
  return r;
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

// A unit's lane partials -> channel partials (the lp lanes of each channel,
// shifted by the m = 0 lane's mean, summed pairwise) -> pieces, stored to upart.
// Nothing waits here: the finalize kernel merges the pieces once every unit is
// done, so the streaming warps never stop for a round trip to L2.
template <class T>
__device__ __forceinline__ void n_stats_unit_done(const NPlan& p, const NFwdWs& ws, const NUnit& q,
                                                  const NMoments<T>& mom, Part* sp) {
  const int lane = threadIdx.x & 31;
  float K[8], v[16];  // v: S of the 8 channels, then Q
#pragma unroll
  for (int sl = 0; sl < 8; ++sl) K[sl] = __shfl_sync(kFull, fadd(n_slot(mom.m1, sl), n_slot(mom.cn, sl)), q.b);
#pragma unroll
  for (int sl = 0; sl < 8; ++sl) {
    const float a2 = n_slot(mom.m2, sl);
    v[sl] = n_shifted_s(n_slot(mom.m1, sl), n_slot(mom.cn, sl), q.cnt, K[sl], v[8 + sl], a2 < 0.f ? 0.f : a2);
  }
  n_msum(v, q.rg, q.m);
  if (q.m == 0 && lane < q.rg.vr) {
    const float inv = __frcp_rn((float)q.len);
#pragma unroll
    for (int sl = 0; sl < 8; ++sl) sp[kVec * q.b + sl] = n_finish(K[sl], v[sl], v[8 + sl], (int)q.len, inv);
  }
  __syncwarp();
  n_unit_pieces(p, q, sp, ws.upart);
  __syncwarp();  // sp is rewritten by the next unit
}

// The direct statistics kernel (any channel count).
template <class T>
__global__ void __launch_bounds__(32 * kNRedWarps, 1)
    k_ndhwc_stats(const T* __restrict__ x, NPlan p, NFwdWs ws) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Part* sp = reinterpret_cast<Part*>(smem) + (size_t)warp * (kNSpan * kVec);
  pdl_launch_dependents();
  const int64_t W = (int64_t)gridDim.x * kNRedWarps;
  for (int64_t u = n_first_unit(); u < p.units; u += W) {
    const NUnit q = n_unit(p, u, lane);
    NMoments<T> mom;
    n_lane_moments<T>(x, q, mom);
    n_stats_unit_done<T>(p, ws, q, mom, sp);
  }
}

// A bounded wait gave up: GN3D_ERR_TIMEOUT in the device status word.
__device__ __forceinline__ void n_record_timeout(uint32_t* status) {
  if ((threadIdx.x & 31) == 0) atomicExch(status, 4u);
}

// ---------------------------------------------------------- bulk-copy rings
// With one channel range (C <= 256) a unit is one contiguous span: len*C
// elements, step i the 8*lw elements from i*8*lw on (lane l < lw holding
// vector l of the step).  The ring kernels stream the spans of the warp's units
// through a warp-private ring of kSlots shared-memory slots, kPS steps per
// slot, filled by 1-D bulk copies (the TMA engine) issued by lane 0, so several
// parts of a warp's units are in flight at every moment.
template <class T, int kTensors, int kSlots, int kPS>
struct NRing {
  static constexpr int kTensorBytes = kPS * kNSpan * kVec * (int)sizeof(T);
  static constexpr int kSlotBytes = kTensors * kTensorBytes;
  static constexpr int kWarpBytes = (kSlots * (kSlotBytes + 8) + 127) / 128 * 128;
  static_assert(kTensorBytes % 128 == 0 && kSlotBytes % 8 == 0, "slot alignment");
  unsigned char* data;
  uint64_t* bar;
  int64_t issued = 0, taken = 0;

  __device__ __forceinline__ void init(unsigned char* base) {
    data = base;
    bar = reinterpret_cast<uint64_t*>(base + (size_t)kSlots * kSlotBytes);
    if ((threadIdx.x & 31) == 0) {
      for (int i = 0; i < kSlots; ++i) mbar_init(&bar[i], 1);
      fence_mbar_init();
    }
    __syncwarp();
  }
  // Copy elements [e0, e0 + n) of each tensor into the next slot (all lanes call;
  // lane 0 copies).  e0 and n are multiples of 8 (16-byte aligned, 16-byte sizes).
  __device__ __forceinline__ void issue(const T* const* src, int64_t e0, int64_t n) {
    const int slot = (int)(issued % kSlots);
    if ((threadIdx.x & 31) == 0) {
      const uint32_t bytes = (uint32_t)(n * (int64_t)sizeof(T));
      unsigned char* dst = data + (size_t)slot * kSlotBytes;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bar[slot], bytes * kTensors);
#pragma unroll
      for (int t = 0; t < kTensors; ++t) bulk_g2s(dst + t * kTensorBytes, src[t] + e0, bytes, &bar[slot]);
    }
    ++issued;
  }
  // Wait (bounded) for the next slot; its data, or nullptr in every lane.
  __device__ __forceinline__ const unsigned char* take(unsigned long long spin) {
    const int slot = (int)(taken % kSlots);
    const bool ok = __all_sync(kFull, mbar_wait_bounded(&bar[slot], (uint32_t)((taken / kSlots) & 1), spin));
    if (!ok) return nullptr;
    ++taken;
    return data + (size_t)slot * kSlotBytes;
  }
  __device__ __forceinline__ void drain(unsigned long long spin) {
    for (int64_t t = taken; t < issued; ++t)
      mbar_wait_bounded(&bar[t % kSlots], (uint32_t)((t / kSlots) & 1), spin);
  }
};

// Steps of unit u (one range: lp positions per step).
// The loader of a ring: part `part` of unit u (n_ring_part), over the warp's units.
template <int kPS>
struct NLoader {
  int64_t u;
  int part;
  template <class Ring, class T>
  __device__ __forceinline__ void issue_next(const NPlan& p, const NRange& rg, int64_t W, Ring& ring,
                                             const T* const* src) {
    if (u >= p.units) return;
    int64_t e0, n;
    const bool last = n_ring_part(p, rg, u, part, kPS, e0, n);
    ring.issue(src, e0, n);
    if (last) {
      part = 0;
      u += W;
    } else {
      ++part;
    }
  }
};

template <class T> struct NStatRing {
  static constexpr int kSlots = 3;
  static constexpr int kPS = NBatch<T>::kStats;  // 8 KB slots
  using Ring = NRing<T, 1, kSlots, kPS>;
  static constexpr int kSmem = kNRedWarps * (Ring::kWarpBytes + kNSpan * kVec * (int)sizeof(Part));
};

// The ring statistics kernel (one channel range).
template <class T>
__global__ void __launch_bounds__(32 * kNRedWarps, 1)
    k_ndhwc_stats_ring(const T* __restrict__ x, NPlan p, NFwdWs ws, unsigned long long spin, uint32_t* status,
                       int force_timeout) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Sh = NStatRing<T>;
  constexpr int kPS = Sh::kPS, kRaw = Vec<T>::kRaw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  typename Sh::Ring ring;
  ring.init(smem + (size_t)warp * Sh::Ring::kWarpBytes);
  Part* sp = reinterpret_cast<Part*>(smem + (size_t)kNRedWarps * Sh::Ring::kWarpBytes) + (size_t)warp * (kNSpan * kVec);
  pdl_launch_dependents();
  const int64_t W = (int64_t)gridDim.x * kNRedWarps;
  const NRange rg = n_range(p, 0);
  const T* src[1] = {x};
  NLoader<kPS> ld{n_first_unit(), 0};
  for (int i = 0; i < Sh::kSlots; ++i) ld.issue_next(p, rg, W, ring, src);
  bool failed = false;
  if (force_timeout) {  // testing: a bounded wait on a word nothing sets, with copies in flight
    unsigned long long i = 0;
    while (i < spin && ld_acquire(ws.never) == 0u) ++i;
    failed = ld_acquire(ws.never) == 0u;
  }
  for (int64_t u = n_first_unit(); u < p.units && !failed; u += W) {
    const NUnit q = n_unit(p, u, lane);
    const int steps = n_unit_steps(p, rg, u);
    NMoments<T> mom;
    for (int t0 = 0; t0 < steps; t0 += kPS) {
      const unsigned char* slot = ring.take(spin);
      if (!slot) {
        failed = true;
        break;
      }
      const T* sb = reinterpret_cast<const T*>(slot) + kVec * lane;
      const int nv = q.cnt - t0 < kPS ? q.cnt - t0 : kPS;
      uint4 w[kPS][kRaw];
#pragma unroll
      for (int t = 0; t < kPS; ++t)
        if (t < nv) Vec<T>::template load<FromShared>(sb + t * kVec * rg.lw, w[t]);
      __syncwarp();
      ld.issue_next(p, rg, W, ring, src);
      if (nv > 0) mom.batch(w, t0, nv, q.cnt);
    }
    if (failed) break;
    mom.finish(q.cnt);
    n_stats_unit_done<T>(p, ws, q, mom, sp);
  }
  if (failed) n_record_timeout(status);
  ring.drain(kDrainPolls);
}

// ------------------------------------------------------ forward finalize
// The unit pieces of group gi = n*G + g (range by range, unit by unit) are cut
// into chunks of kNFinChunk units; one CTA of kNFinThreads threads merges a
// chunk (thread t takes units t, t + kNFinThreads, ... in order, then the
// warps' butterflies, then the warps in order) and the CTA that completes a
// group merges its chunk partials in order.  Every merge is the shifted-sum
// merge with the shift = the mean of the first part merged.  Chunk boundaries
// depend on the shape only.
constexpr int kNFinThreads = 256;
constexpr int64_t kNFinChunk = 4096;

// Ranges a group can meet (the most of any group) and chunks per range.
__host__ __device__ inline int64_t n_fin_maxr(const NPlan& p) {
  int64_t m = 1;
  for (int64_t g = 0; g < p.G; ++g) {
    const int64_t r = ((g + 1) * p.Cg - 1) / (kNSpan * kVec) - (g * p.Cg) / (kNSpan * kVec) + 1;
    if (r > m) m = r;
  }
  return m;
}
__host__ __device__ inline int64_t n_fin_nkc(const NPlan& p) { return (p.R + kNFinChunk - 1) / kNFinChunk; }

// Rows of at most kNFinShortRow units: the backward finalize sums each with one
// warp instead of one CTA.
constexpr int64_t kNFinShortRow = 512;
__host__ __device__ inline bool n_fin_short_rows(const NPlan& p) { return p.R <= kNFinShortRow; }

__device__ __forceinline__ float2 n_cta_sum2(float a, float b) {
  __shared__ float2 part[kNFinThreads / 32];
  const float2 t = warp_sum2(a, b);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = t;
  __syncthreads();
  float2 r = part[0];
  for (int w = 1; w < kNFinThreads / 32; ++w) r = make_float2(fadd(r.x, part[w].x), fadd(r.y, part[w].y));
  __syncthreads();  // part is reused by the next call
  return r;
}

// Thread 0 adds the CTA's arrival on *ctr after the CTA's stores; every thread
// learns whether it was the last of `total` (and then sees the others' stores).
__device__ __forceinline__ bool n_cta_arrive_last(uint32_t* ctr, uint32_t total) {
  __shared__ uint32_t last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atom_add_acq_rel(ctr, 1u) + 1u == total ? 1u : 0u;
  __syncthreads();
  const bool l = last != 0;
  if (l) __threadfence();
  __syncthreads();  // last is reused by the next call
  return l;
}

__global__ void __launch_bounds__(kNFinThreads)
    k_ndhwc_stats_final(NPlan p, NFwdWs ws, float eps, float* mean_out, float* rstd_out) {
  pdl_launch_dependents();
  pdl_wait();  // the statistics kernel's unit pieces
  const int64_t maxr = n_fin_maxr(p), nkc = n_fin_nkc(p), per = maxr * nkc;
  for (int64_t t = blockIdx.x; t < p.NG * per; t += gridDim.x) {
    const int64_t gi = t / per, rem = t - gi * per, ri = rem / nkc, kc = rem - ri * nkc;
    const int64_t n = gi / p.G, g = gi - n * p.G;
    const int64_t r = (g * p.Cg) / (kNSpan * kVec) + ri, r_hi = ((g + 1) * p.Cg - 1) / (kNSpan * kVec);
    Part part{0.f, 0.f, 0, 0.f};
    if (r <= r_hi) {
      const NRange rg = n_range(p, r);
      const int64_t j = g - rg.g0;
      int64_t c0, c1;
      n_piece(p, rg, j, c0, c1);
      const Part* base = ws.upart + ((n * p.nr + r) * p.P + j) * p.R;
      const int64_t k0 = kc * kNFinChunk, k1 = k0 + kNFinChunk < p.R ? k0 + kNFinChunk : p.R;
      const Part b0 = ldcg_part(base + k0);
      const float K = fadd(b0.m1, b0.cn);
      float S = 0.f, Q = 0.f;
      constexpr int kBatch = 16, kPer = (int)(kNFinChunk / kNFinThreads);
#pragma unroll
      for (int i0 = 0; i0 < kPer; i0 += kBatch) {
        Part v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int64_t k = k0 + threadIdx.x + (int64_t)(i0 + i) * kNFinThreads;
          if (k < k1) v[i] = ldcg_part(base + k);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          if (k0 + threadIdx.x + (int64_t)(i0 + i) * kNFinThreads < k1) {
            float s1, q1;
            shifted_terms(v[i], K, s1, q1);
            S = fadd(S, s1);
            Q = fadd(Q, q1);
          }
        }
      }
      const float2 tq = n_cta_sum2(S, Q);
      const int64_t pos = (k1 * p.Pu < p.S ? k1 * p.Pu : p.S) - k0 * p.Pu;
      part = finish_merge(K, tq.x, tq.y, pos * (c1 - c0));
    }
    if (per == 1) {  // one chunk: it is the group
      if (threadIdx.x == 0) {
        const float rs = __frsqrt_rn(fadd(__fdiv_rn(part.m2, (float)p.M), eps));
        ws.stats[gi] = make_float4(part.m1, part.cn, rs, 0.f);
        if (mean_out) mean_out[gi] = fadd(part.m1, part.cn);
        if (rstd_out) rstd_out[gi] = rs;
      }
      continue;
    }
    if (threadIdx.x == 0) ws.fpart[t] = part;
    if (!n_cta_arrive_last(ws.gcnt + gi, (uint32_t)per)) continue;
    if (threadIdx.x < 32) {
      // the group's chunk partials in order (the first one is never empty)
      const Part* fp = ws.fpart + gi * per;
      const Part a0 = ldcg_part(fp);
      const float K = fadd(a0.m1, a0.cn);
      float S = 0.f, Q = 0.f;
      for (int64_t i = threadIdx.x; i < per; i += 32) {
        float s1, q1;
        shifted_terms(ldcg_part(fp + i), K, s1, q1);
        S = fadd(S, s1);
        Q = fadd(Q, q1);
      }
      const float2 tq = warp_sum2(S, Q);
      if (threadIdx.x == 0) {
        const Part gp = finish_merge(K, tq.x, tq.y, p.M);
        const float rs = __frsqrt_rn(fadd(__fdiv_rn(gp.m2, (float)p.M), eps));
        ws.stats[gi] = make_float4(gp.m1, gp.cn, rs, 0.f);
        if (mean_out) mean_out[gi] = fadd(gp.m1, gp.cn);
        if (rstd_out) rstd_out[gi] = rs;
      }
    }
  }
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
  NOwned own(p);
  // the first batch of the first unit is loaded before the statistics are
  // complete (x is not written there); everything else after pdl_wait
  uint4 w[kB][kRaw];
  bool pre = false;
  if (own.more()) {
    const NUnit q = n_unit(p, own.unit(), lane);
#pragma unroll
    for (int t = 0; t < kB; ++t)
      if (t < q.cnt) Vec<TI>::template load<FromGlobal>(x + q.off + (int64_t)t * q.step, w[t]);
    pre = true;
  }
  pdl_wait();
  f2 hi[4], sc[4], sh[4];
  int64_t have = -1;  // the row (n, r) whose coefficients are loaded
  for (; own.more(); own.next()) {
    const NUnit q = n_unit(p, own.unit(), lane);
    if (q.cnt == 0) {
      pre = false;
      continue;
    }
    // a warp's units mostly share the row: the coefficients are reloaded only
    // when it changes
#pragma unroll
    for (int e = 0; e < 4 && have != q.row; ++e) {
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
    have = q.row;
    const TI* xb = x + q.off;
    TO* yb = y + q.off;
    for (int t0 = 0; t0 < q.cnt; t0 += kB) {
      if (!pre) {
#pragma unroll
        for (int t = 0; t < kB; ++t)
          if (t0 + t < q.cnt) Vec<TI>::template load<FromGlobal>(xb + (int64_t)(t0 + t) * q.step, w[t]);
      }
      pre = false;
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

// S1 += dy, S2 += dy*(x - mean) over a batch of nv steps (wx: x, wd: the gradient).
// Even steps go to (a1, a2), odd steps to (b1, b2): two chains per sum; the
// caller adds the two sets when the unit is done.
template <class T, int kB>
__device__ __forceinline__ void n_bwd_batch(const uint4 (&wx)[kB][Vec<T>::kRaw], const uint4 (&wd)[kB][Vec<T>::kRaw],
                                            int nv, const f2 mu[4], f2 a1[4], f2 a2[4], f2 b1[4], f2 b2[4]) {
#pragma unroll
  for (int t = 0; t < kB; ++t) {
    if (t < nv) {
      f2 xm[4], vd[4];
      n_diff<T>(wx[t], mu, xm);
      Vec<T>::pairs(wd[t], vd);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (t & 1) {
          b1[e] = f2add(b1[e], vd[e]);
          b2[e] = f2fma(vd[e], xm[e], b2[e]);
        } else {
          a1[e] = f2add(a1[e], vd[e]);
          a2[e] = f2fma(vd[e], xm[e], a2[e]);
        }
      }
    }
  }
}

// The lane's 8 group means (pairs of channels).
template <class T>
__device__ __forceinline__ void n_lane_means(const NPlan& p, const NUnit& q, const float* __restrict__ mean,
                                             f2 mu[4]) {
  const float* mg = mean + q.n * p.G;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int64_t c = q.rg.c0 + kVec * q.b + 2 * e;
    mu[e] = q.cnt ? f2_of(mg[c / p.Cg], mg[(c + 1) / p.Cg]) : f2_splat(0.f);
  }
}

// A unit's lane sums -> channel sums (pairwise over the lp lanes of a channel),
// stored to usum (the finalize kernel sums them).
__device__ __forceinline__ void n_reduce_unit_done(const NPlan& p, const NBwdWs& ws, const NUnit& q, const f2 a1[4],
                                                   const f2 a2[4]) {
  const int lane = threadIdx.x & 31;
  float v[16];  // S1 of the 8 channels, then S2
#pragma unroll
  for (int sl = 0; sl < 8; ++sl) {
    v[sl] = n_slot(a1, sl);
    v[8 + sl] = n_slot(a2, sl);
  }
  n_msum(v, q.rg, q.m);
  if (q.m == 0 && lane < q.rg.vr) {
#pragma unroll
    for (int sl = 0; sl < 8; ++sl)
      ws.usum[(q.n * p.C + q.rg.c0 + kVec * q.b + sl) * p.R + q.k] = make_float2(v[sl], v[8 + sl]);
  }
}

// ----------------------------------------------------- backward finalize
// Row (n, c): rows of at most kNFinShortRow units are summed one warp per row,
// with one CTA arrival per pass of the CTA's warps.  Longer rows: the unit sums
// cut into chunks of kNFinChunk units; one CTA sums a
// chunk (thread t takes units t, t + kNFinThreads, ... in order, then the warps'
// butterflies, then the warps in order); the CTA that completes a row adds its
// chunk sums in order (S1, S2 of the row); the CTA that completes the last row
// forms the group coefficients, A = sum_c gamma_c*S1_c and
// B = rstd * sum_c gamma_c*S2_c (one warp per group: lane-strided over the
// channels, then the butterfly; a = A/M, b = B/M), and
// dgamma_c = sum_n rstd[n,g]*S2[n,c], dbeta_c = sum_n S1[n,c] in n order.
__global__ void __launch_bounds__(kNFinThreads)
    k_ndhwc_reduce_final(NPlan p, NBwdWs ws, const float* __restrict__ rstd, const float* __restrict__ gamma,
                         float* dgamma, float* dbeta) {
  pdl_launch_dependents();
  pdl_wait();  // the reduction kernel's unit sums
  const int64_t nkc = n_fin_nkc(p), NC = p.N * p.C;
  bool last_row = false;
  if (n_fin_short_rows(p)) {
    // short rows: one warp per row (lane l takes units l, l + 32, ... in order,
    // then the butterfly) and one CTA arrival per pass of the CTA's warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = kNFinThreads / 32;
    const int64_t passes = (NC + nw - 1) / nw;
    for (int64_t ps = blockIdx.x; ps < passes; ps += gridDim.x) {
      const int64_t rc = ps * nw + warp;
      if (rc < NC) {
        const float2* us = ws.usum + rc * p.R;
        float2 v[kNFinShortRow / 32];
#pragma unroll
        for (int k = 0; k < kNFinShortRow / 32; ++k)
          if (lane + 32 * k < p.R) v[k] = __ldcg(us + lane + 32 * k);
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int k = 0; k < kNFinShortRow / 32; ++k) {
          if (lane + 32 * k < p.R) {
            s1 = fadd(s1, v[k].x);
            s2 = fadd(s2, v[k].y);
          }
        }
        const float2 row = warp_sum2(s1, s2);
        if (lane == 0) ws.rows[rc] = row;
      }
      if (n_cta_arrive_last(ws.done, (uint32_t)passes)) last_row = true;
    }
  }
  for (int64_t t = n_fin_short_rows(p) ? NC * nkc : blockIdx.x; t < NC * nkc; t += gridDim.x) {
    const int64_t rc = t / nkc, kc = t - rc * nkc;
    const float2* us = ws.usum + rc * p.R;
    const int64_t k0 = kc * kNFinChunk, k1 = k0 + kNFinChunk < p.R ? k0 + kNFinChunk : p.R;
    float s1 = 0.f, s2 = 0.f;
    constexpr int kPer = (int)(kNFinChunk / kNFinThreads);
    float2 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int64_t k = k0 + threadIdx.x + (int64_t)i * kNFinThreads;
      if (k < k1) v[i] = __ldcg(us + k);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      if (k0 + threadIdx.x + (int64_t)i * kNFinThreads < k1) {
        s1 = fadd(s1, v[i].x);
        s2 = fadd(s2, v[i].y);
      }
    }
    const float2 sum = n_cta_sum2(s1, s2);
    if (nkc == 1) {  // one chunk: it is the row
      if (threadIdx.x == 0) ws.rows[rc] = sum;
    } else {
      if (threadIdx.x == 0) ws.rpart[t] = sum;
      if (!n_cta_arrive_last(ws.rcnt + rc, (uint32_t)nkc)) continue;
    }
    if (nkc > 1 && threadIdx.x < 32) {
      float a1 = 0.f, a2 = 0.f;
      for (int64_t i = threadIdx.x; i < nkc; i += 32) {
        const float2 v = __ldcg(ws.rpart + rc * nkc + i);
        a1 = fadd(a1, v.x);
        a2 = fadd(a2, v.y);
      }
      const float2 row = warp_sum2(a1, a2);
      if (threadIdx.x == 0) ws.rows[rc] = row;
    }
    if (n_cta_arrive_last(ws.done, (uint32_t)NC)) last_row = true;
  }
  if (!last_row) return;
  // one warp per group: lane l takes the group's channels l, l + 32, ... in
  // order (their loads issued kNCoefBatch at a time), then the butterfly
  constexpr int kNCoefBatch = 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t gi = warp; gi < p.NG; gi += blockDim.x >> 5) {
    const int64_t n = gi / p.G, g = gi - n * p.G;
    float A = 0.f, Bs = 0.f;
    for (int64_t c0 = 0; c0 < p.Cg; c0 += 32 * kNCoefBatch) {
      float2 v[kNCoefBatch];
      float gm[kNCoefBatch];
#pragma unroll
      for (int k = 0; k < kNCoefBatch; ++k) {
        const int64_t cl = c0 + lane + 32 * k;
        if (cl < p.Cg) {
          const int64_t c = g * p.Cg + cl;
          v[k] = __ldcg(ws.rows + n * p.C + c);
          gm[k] = gamma ? gamma[c] : 1.f;
        }
      }
#pragma unroll
      for (int k = 0; k < kNCoefBatch; ++k) {
        if (c0 + lane + 32 * k < p.Cg) {
          A = fadd(A, fmul(gm[k], v[k].x));
          Bs = fadd(Bs, fmul(gm[k], v[k].y));
        }
      }
    }
    const float2 t = warp_sum2(A, Bs);
    if (lane == 0) {
      const float fM = (float)p.M;
      ws.coef[gi] = make_float2(__fdiv_rn(t.x, fM), __fdiv_rn(fmul(rstd[gi], t.y), fM));
    }
  }
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

// The direct reduction kernel (any channel count).
template <class T, bool kRelu>
__global__ void __launch_bounds__(32 * kNRedWarps, 1)
    k_ndhwc_reduce(const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ res, NPlan p,
                   const float* __restrict__ mean, NBwdWs ws) {
  constexpr int kB = NBatch<T, kRelu>::kReduce, kRaw = Vec<T>::kRaw;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();
  const int64_t W = (int64_t)gridDim.x * kNRedWarps;
  const f2 z2 = f2_splat(0.f);
  f2 mu[4];
  int64_t have = -1;  // the row (n, r) whose means are loaded
  for (int64_t u = n_first_unit(); u < p.units; u += W) {
    const NUnit q = n_unit(p, u, lane);
    if (have != q.row && q.cnt) {
      n_lane_means<T>(p, q, mean, mu);
      have = q.row;
    }
    f2 a1[4] = {z2, z2, z2, z2}, a2[4] = {z2, z2, z2, z2}, b1[4] = {z2, z2, z2, z2}, b2[4] = {z2, z2, z2, z2};
    for (int t0 = 0; t0 < q.cnt; t0 += kB) {
      const int nv = q.cnt - t0 < kB ? q.cnt - t0 : kB;
      uint4 wx[kB][kRaw], wd[kB][kRaw];
#pragma unroll
      for (int t = 0; t < kB; ++t) {
        if (t < nv) {
          const int64_t o = q.off + (int64_t)(t0 + t) * q.step;
          Vec<T>::template load<FromGlobal>(x + o, wx[t]);
          n_grad<T, kRelu>(dy, res, o, wd[t]);
        }
      }
      n_bwd_batch<T>(wx, wd, nv, mu, a1, a2, b1, b2);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a1[e] = f2add(a1[e], b1[e]);
      a2[e] = f2add(a2[e], b2[e]);
    }
    n_reduce_unit_done(p, ws, q, a1, a2);
  }
}

template <class T, bool kRelu> struct NRedRing {
  static constexpr int kSlots = kRelu ? 4 : 3;
  static constexpr int kTensors = kRelu ? 3 : 2;
  static constexpr int kPS = NBatch<T, kRelu>::kReduce;  // 4 KB (2 KB behind a ReLU) of each tensor per slot
  using Ring = NRing<T, kTensors, kSlots, kPS>;
  static constexpr int kSmem = kNRedWarps * Ring::kWarpBytes;
};

// The ring reduction kernel (one channel range).
template <class T, bool kRelu>
__global__ void __launch_bounds__(32 * kNRedWarps, 1)
    k_ndhwc_reduce_ring(const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ res, NPlan p,
                        const float* __restrict__ mean, NBwdWs ws, unsigned long long spin, uint32_t* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Sh = NRedRing<T, kRelu>;
  using Ring = typename Sh::Ring;
  constexpr int kPS = Sh::kPS, kRaw = Vec<T>::kRaw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ring ring;
  ring.init(smem + (size_t)warp * Ring::kWarpBytes);
  pdl_launch_dependents();
  const int64_t W = (int64_t)gridDim.x * kNRedWarps;
  const NRange rg = n_range(p, 0);
  const T* src[3] = {x, dy, res};
  NLoader<kPS> ld{n_first_unit(), 0};
  for (int i = 0; i < Sh::kSlots; ++i) ld.issue_next(p, rg, W, ring, src);
  const f2 z2 = f2_splat(0.f);
  bool failed = false;
  f2 mu[4];
  int64_t have = -1;  // the row (n, r) whose means are loaded
  for (int64_t u = n_first_unit(); u < p.units && !failed; u += W) {
    const NUnit q = n_unit(p, u, lane);
    const int steps = n_unit_steps(p, rg, u);
    if (have != q.row && q.cnt) {
      n_lane_means<T>(p, q, mean, mu);
      have = q.row;
    }
    f2 a1[4] = {z2, z2, z2, z2}, a2[4] = {z2, z2, z2, z2}, b1[4] = {z2, z2, z2, z2}, b2[4] = {z2, z2, z2, z2};
    for (int t0 = 0; t0 < steps; t0 += kPS) {
      const unsigned char* slot = ring.take(spin);
      if (!slot) {
        failed = true;
        break;
      }
      const int nv = q.cnt - t0 < kPS ? q.cnt - t0 : kPS;
      const T* xs = reinterpret_cast<const T*>(slot) + kVec * lane;
      const T* ds = reinterpret_cast<const T*>(slot + Ring::kTensorBytes) + kVec * lane;
      uint4 wx[kPS][kRaw], wd[kPS][kRaw];
#pragma unroll
      for (int t = 0; t < kPS; ++t) {
        if (t < nv) {
          Vec<T>::template load<FromShared>(xs + t * kVec * rg.lw, wx[t]);
          Vec<T>::template load<FromShared>(ds + t * kVec * rg.lw, wd[t]);
          if constexpr (kRelu) {
            const T* rs = reinterpret_cast<const T*>(slot + 2 * Ring::kTensorBytes) + kVec * lane;
            uint4 o[kRaw];
            Vec<T>::template load<FromShared>(rs + t * kVec * rg.lw, o);
            Vec<T>::gate(o, wd[t]);
          }
        }
      }
      __syncwarp();
      ld.issue_next(p, rg, W, ring, src);
      n_bwd_batch<T>(wx, wd, nv, mu, a1, a2, b1, b2);
    }
    if (failed) break;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      a1[e] = f2add(a1[e], b1[e]);
      a2[e] = f2add(a2[e], b2[e]);
    }
    n_reduce_unit_done(p, ws, q, a1, a2);
  }
  if (failed) n_record_timeout(status);
  ring.drain(kDrainPolls);
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
  NOwned own(p);
  // the first batch is loaded before the coefficients exist (x, dy and the
  // forward's result are inputs); the coefficients after pdl_wait
  uint4 wx[kB][kRaw], wd[kB][kRaw];
  bool pre = false;
  if (own.more()) {
    const NUnit q = n_unit(p, own.unit(), lane);
#pragma unroll
    for (int t = 0; t < kB; ++t) {
      if (t < q.cnt) {
        const int64_t o = q.off + (int64_t)t * q.step;
        Vec<T>::template load<FromGlobal>(x + o, wx[t]);
        n_grad<T, kRelu>(dy, res, o, wd[t]);
      }
    }
    pre = true;
  }
  pdl_wait();
  const bool single = p.M == 1;
  f2 mu[4], p1[4], np2[4], np3[4];
  int64_t have = -1;  // the row (n, r) whose coefficients are loaded
  for (; own.more(); own.next()) {
    const NUnit q = n_unit(p, own.unit(), lane);
    if (q.cnt == 0) {
      pre = false;
      continue;
    }
#pragma unroll
    for (int e = 0; e < 4 && have != q.row; ++e) {
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
    have = q.row;
    for (int t0 = 0; t0 < q.cnt; t0 += kB) {
      if (!pre) {
#pragma unroll
        for (int t = 0; t < kB; ++t) {
          if (t0 + t < q.cnt) {
            const int64_t o = q.off + (int64_t)(t0 + t) * q.step;
            Vec<T>::template load<FromGlobal>(x + o, wx[t]);
            n_grad<T, kRelu>(dy, res, o, wd[t]);
          }
        }
      }
      pre = false;
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
