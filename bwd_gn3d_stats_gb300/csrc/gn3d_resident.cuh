// gn3d_resident.cuh -- the group-wave launch form: one persistent cooperative
// kernel per direction in which every CTA holds a share of every group, reads
// it from HBM once, and normalizes it while the next groups stream in.
//
// Work placement (gn3d_resident_plan.cuh).  Every group is cut into one
// contiguous run of units per CTA (its "share"); the CTAs walk their shares in
// group order, so all CTAs finish a group's reduction at about the same time.
// Unit j of a share of n units is
//   held  (the last nh = min(n, rh) units): its body stays in a shared-memory
//         slot of the held ring until the elementwise pass has used it;
//   pass  (the others): its slot in the pass ring is released once the
//         reduction has read it, and the elementwise pass reads it again from
//         global memory (L2: the producer runs at most `window` units ahead of
//         the elementwise pass, so it was read a few microseconds before).
//
// Warp roles (one CTA per SM):
//   producer     one lane issues the 1-D bulk copies (the TMA engine) of the
//                sequence's units, in order, into the rings' slots, each on the
//                slot's "full" mbarrier once the slot's "empty" mbarrier shows
//                its previous use was released;
//   reduction    slot s of either ring is read by reduction warp s mod kRed
//                (both rings hold a multiple of kRed slots): the unit's
//                partial -- the streaming kernels' per-unit arithmetic -- goes
//                to global memory, and the warp that completes the CTA's share
//                of a group makes the CTA's one arrival on the group's counter;
//   elementwise  per group (the CTA's shares in order): once every CTA holding
//                a share has arrived, all elementwise warps merge the group
//                from its unit partials -- every block exactly as merge_block
//                and the group exactly as the group merge of the streaming
//                kernels, so every CTA obtains the same bits -- and then write
//                y (or dx) of the share's units, last unit first.
// Every CTA merges every group it holds a share of (a few hundred merge_block
// calls per group spread over the elementwise warps), which replaces the
// streaming kernels' chain of block and group arrivals by one arrival per CTA
// and one load of the group's partials.  (The ScaFFold GroupNorm kernels split
// a group "to fill the device" and read it twice; here the split keeps the
// first read on chip or in L2.)
//
// Deadlock freedom: all CTAs are co-resident (cooperative launch).  Loading a
// share of group g waits at most for slots held by groups < g, and for the
// elementwise pass of groups < g (the window); those wait only for the
// reductions of groups < g, whose units every CTA loaded before g's.  The
// elementwise warps of a CTA meet at named barriers and decide together
// whether to go on, so none waits at a barrier for a warp that left.  Every
// wait is bounded: on timeout the kernel records GN3D_ERR_TIMEOUT, raises the
// abort word, which every other wait watches, and returns; the producer drains
// its bulk copies in flight before it returns.
#pragma once
#include "gn3d_device.cuh"
#include "gn3d_resident_plan.cuh"
#include "gn3d_sync.cuh"

namespace gn3d {

constexpr int kCtrRing = 256;  // per-CTA group counters (more than groups in flight: window < kCtrRing)

struct ResCfg {
  ResGeo geo;              // placement: CTAs, share sizes, held units per share, rings
  long long window;        // units the producer may run ahead of the elementwise pass (< kCtrRing)
  int force_timeout;       // testing hook: the first group wait targets a word nothing sets
  unsigned long long spin; // poll budget of every bounded wait
};

struct ResSync {
  uint32_t* abort;   // [1] raised by a warp that gave up waiting
  uint32_t* never;   // [1] stays 0
  uint32_t* status;  // device status word (GN3D_ERR_TIMEOUT on a timeout)
};

constexpr uint32_t kResTimeout = 4;  // GN3D_ERR_TIMEOUT

__device__ __forceinline__ bool res_aborted(const ResSync& rs) { return ld_relaxed(rs.abort) != 0; }

__device__ __forceinline__ void res_fail(const ResSync& rs) {
  atomicExch(rs.status, kResTimeout);
  atomicExch(rs.abort, 1u);
}

// Bounded mbarrier wait that also watches the abort word (every 64 polls), by one lane.
__device__ __forceinline__ bool res_mbar_wait(uint64_t* bar, uint32_t parity, const ResCfg& c, const ResSync& rs) {
  for (unsigned long long i = 0; i < c.spin; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && res_aborted(rs)) return false;
  }
  return false;
}

// The same wait by a warp: lane 0 polls and the warp learns the outcome, so the
// lanes never disagree; on success every lane then observes the completed phase
// itself (which orders the bulk copy's data before its reads).
__device__ __forceinline__ bool warp_mbar_wait(uint64_t* bar, uint32_t parity, const ResCfg& c, const ResSync& rs) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = res_mbar_wait(bar, parity, c, rs);
  if (__shfl_sync(kFull, ok ? 1 : 0, 0) == 0) return false;
  return mbar_try_wait(bar, parity);
}

// Bounded wait, by one lane, until a counter reaches `want` (acquire).
__device__ __forceinline__ bool res_wait_count(const uint32_t* ctr, uint32_t want, const ResCfg& c,
                                               const ResSync& rs) {
  for (unsigned long long it = 1; ld_acquire(ctr) < want; ++it) {
    if (it > c.spin || ((it & 63) == 0 && res_aborted(rs))) return false;
  }
  return true;
}

// A barrier among the elementwise warps only (named barrier 1).
template <int kThreads>
__device__ __forceinline__ void elem_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

// The shared-memory layout of a group-wave kernel: held slots, pass slots, the
// rings' mbarriers, the per-group unit counters, the finalize staging area
// (one round of block results), the elementwise progress counter and the
// elementwise warps' shared decision word.
template <int kSlotBytes, class StageT, int kStage>
struct ResLayout {
  unsigned char* held;
  unsigned char* pass;
  uint64_t *hfull, *hempty, *pfull, *pempty;
  uint32_t* gctr;
  StageT* stage;
  int* normed;
  int* go;
  __device__ __forceinline__ void carve(unsigned char* smem, const ResGeo& G) {
    held = smem;
    pass = held + (size_t)G.kh * kSlotBytes;
    hfull = reinterpret_cast<uint64_t*>(pass + (size_t)G.kp * kSlotBytes);
    hempty = hfull + G.kh;
    pfull = hempty + G.kh;
    pempty = pfull + G.kp;
    stage = reinterpret_cast<StageT*>(pempty + G.kp);
    gctr = reinterpret_cast<uint32_t*>(stage + kStage);
    normed = reinterpret_cast<int*>(gctr + kCtrRing);
    go = normed + 1;
  }
  static __host__ __device__ constexpr int bytes(int kh, int kp) {
    return (kh + kp) * kSlotBytes + 2 * (kh + kp) * 8 + kStage * (int)sizeof(StageT) + kCtrRing * 4 + 16;
  }
  __device__ __forceinline__ void init(const ResGeo& G) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < G.kh; ++i) {
        mbar_init(&hfull[i], 1);
        mbar_init(&hempty[i], 1);
      }
      for (int i = 0; i < G.kp; ++i) {
        mbar_init(&pfull[i], 1);
        mbar_init(&pempty[i], 1);
      }
      fence_mbar_init();
      *normed = 0;
      *go = 0;
    }
    for (int i = threadIdx.x; i < kCtrRing; i += blockDim.x) gctr[i] = 0;
  }
  __device__ __forceinline__ const unsigned char* slot_data(bool hd, int slot) const {
    return (hd ? held : pass) + (size_t)slot * kSlotBytes;
  }
};

// The producer (one lane): bulk copies of the CTA's shares into the rings, in
// sequence order (each share's pass units, then its held units), kTensors
// tensors per unit, each kUnitElems elements of T, side by side in a slot.
template <class T, int kTensors, class Layout>
__device__ __forceinline__ void res_produce(const Plan& p, const ResCfg& c, const ResSync& rs, const Layout& L,
                                            const T* const* src) {
  constexpr uint32_t kTensorBytes = kUnitElems * (uint32_t)sizeof(T);
  const ResGeo& G = c.geo;
  const int cta = blockIdx.x;
  RingPos hr, qr;
  hr.at(0, G.kh > 0 ? G.kh : 1);
  qr.at(0, G.kp);
  int64_t pos = 0, lead = 0;  // units issued; issue allowed while pos < lead
  bool ok = true;
  for (int64_t g = 0; g < p.NG && ok; ++g) {
    const ResShare sh = res_share(p, G, g, cta);
    const int npass = sh.n - sh.nh;
    for (int j = 0; j < sh.n; ++j, ++pos) {
      const bool hd = j >= npass;
      RingPos& r = hd ? hr : qr;
      const int nr = hd ? G.kh : G.kp;
      // the slot's previous use (of the other parity) must have been released
      if (r.uses >= nr && !res_mbar_wait(&(hd ? L.hempty : L.pempty)[r.slot], r.par ^ 1u, c, rs)) {
        ok = false;
        break;
      }
      // at most `window` units ahead of the elementwise pass
      for (unsigned long long it = 0; pos >= lead; ++it) {
        lead = *(volatile int*)L.normed + c.window;
        if (pos < lead) break;
        if (it >= c.spin || ((it & 63) == 63 && res_aborted(rs))) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      unsigned char* dst = const_cast<unsigned char*>(L.slot_data(hd, r.slot));
      uint64_t* full = &(hd ? L.hfull : L.pfull)[r.slot];
      const int64_t b0 = (sh.start + j) * kUnitElems;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(full, kTensorBytes * kTensors);
#pragma unroll
      for (int t = 0; t < kTensors; ++t) bulk_g2s(dst + t * kTensorBytes, src[t] + b0, kTensorBytes, full);
      r.step(1, nr);
    }
  }
  if (!ok) res_fail(rs);
  // every copy issued must land before the CTA may exit: wait for the last
  // phase of each slot that was used
  for (int sl = 0; sl < G.kh; ++sl)
    if (hr.uses > sl) mbar_wait_bounded(&L.hfull[sl], (uint32_t)(((hr.uses - 1 - sl) / G.kh) & 1), kDrainPolls);
  for (int sl = 0; sl < G.kp; ++sl)
    if (qr.uses > sl) mbar_wait_bounded(&L.pfull[sl], (uint32_t)(((qr.uses - 1 - sl) / G.kp) & 1), kDrainPolls);
}

// The reduction warps' loop: in each share, warp w takes the pass units at pass
// ring positions = w (mod kRed), then the held units at held positions = w
// (mod kRed) -- both rings hold a multiple of kRed slots, so every slot is read
// by one reduction warp only, which takes its uses in order: the parity wait
// cannot be met by an older phase of the same parity.  unit(data, hd, slot, g)
// computes one unit's partial (one warp; it releases a pass slot itself once
// the data is read), which lane 0 stores to parts[u].  The warp whose unit
// completes the CTA's share of a group makes the CTA's arrival on gcnt[g]: the
// other warps' stores are ordered before it by their block-scope fences and the
// shared counter, and by its device-scope fence (cumulative) before the arrival.
template <int kRed, class PartT, class Layout, class Unit>
__device__ __forceinline__ bool res_reduce(const Plan& p, const ResCfg& c, const ResSync& rs, const Layout& L,
                                           PartT* parts, uint32_t* gcnt, Unit unit) {
  const ResGeo& G = c.geo;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int h = 0, q = 0;  // held / pass units of the sequence before the share
  for (int64_t g = 0; g < p.NG; ++g) {
    const ResShare sh = res_share(p, G, g, blockIdx.x);
    if (sh.n == 0) continue;
    const int npass = sh.n - sh.nh;
    for (int part = 0; part < 2; ++part) {  // the share's pass units, then its held units
      const bool hd = part == 1;
      const int first = hd ? npass : 0, count = hd ? sh.nh : npass, before = hd ? h : q;
      const int nr = hd ? G.kh : G.kp;
      int j = res_first_of_warp(before, warp, kRed);  // this warp's first unit of the part
      if (j >= count) continue;
      RingPos r;
      r.at(before + j, nr);
      for (; j < count; j += kRed, r.step(kRed, nr)) {
        if (!warp_mbar_wait(&(hd ? L.hfull : L.pfull)[r.slot], r.par, c, rs)) return false;
        const int64_t u = sh.start + first + j;
        const PartT m = unit(L.slot_data(hd, r.slot), hd, r.slot, g);
        if (lane == 0) {
          stcg_unit(parts + u, m);
          __threadfence_block();
          uint32_t* ctr = L.gctr + ((uint32_t)g & (kCtrRing - 1));
          if (atomicAdd(ctr, 1u) + 1u == (uint32_t)sh.n) {  // the CTA's share of group g is reduced
            *ctr = 0;
            __threadfence();
            atomicAdd(gcnt + g, 1u);
          }
        }
        __syncwarp();
      }
    }
    h += sh.nh;
    q += npass;
  }
  return true;
}

// The elementwise warps' loop over the CTA's shares, in group order.  Warp 0
// waits until every CTA holding a share of the group has arrived, and all
// elementwise warps learn the outcome at a barrier; fin(g, writer) merges the
// group (all elementwise warps; writer: this CTA writes the group's outputs);
// held(u, row, data) and pass(u, row) write one unit's result from its held slot
// or from global memory.  Unit r of the share's last-first order goes to
// elementwise warp r mod kElem.
template <int kRed, int kElem, class Layout, class Fin, class Held, class Pass>
__device__ __forceinline__ bool res_elementwise(const Plan& p, const ResCfg& c, const ResSync& rs, const Layout& L,
                                                const uint32_t* gcnt, Fin fin, Held held, Pass pass) {
  const ResGeo& G = c.geo;
  const int ew = (threadIdx.x >> 5) - kRed, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const uint32_t arrivals = G.q > 0 ? (uint32_t)G.P : (uint32_t)G.r;  // CTAs holding a share of each group
  bool forced = c.force_timeout != 0;
  int64_t hg = 0;  // held units of the sequence before this share
  for (int64_t g = 0; g < p.NG; ++g) {
    const ResShare sh = res_share(p, G, g, cta);
    if (sh.n == 0) continue;
    if (ew == 0 && lane == 0)
      *(volatile int*)L.go = res_wait_count(forced ? rs.never : gcnt + g, forced ? 1u : arrivals, c, rs) ? 1 : 0;
    forced = false;
    elem_sync<32 * kElem>();
    if (*(volatile int*)L.go == 0) return false;  // every elementwise warp leaves together
    fin(g, sh.start == g * p.upg);
    const int hs0 = G.kh > 0 ? (int)((uint64_t)hg % (uint64_t)G.kh) : 0;
    const uint32_t hp0 = G.kh > 0 ? (uint32_t)(((uint64_t)hg / (uint64_t)G.kh) & 1) : 0u;
    for (int r = ew; r < sh.n; r += kElem) {
      const int j = sh.n - 1 - r;
      const int64_t u = sh.start + j;
      const int64_t row = res_row_of(u, p.R);
      if (j >= sh.n - sh.nh) {  // held: at most one wrap past the share's first held slot
        int slot = hs0 + (j - (sh.n - sh.nh));
        uint32_t par = hp0;
        if (slot >= G.kh) {
          slot -= G.kh;
          par ^= 1u;
        }
        // the reduction warp saw this phase complete before the CTA arrived;
        // waiting on it here orders the bulk copy's data before this warp's reads
        if (!warp_mbar_wait(&L.hfull[slot], par, c, rs)) {
          if (lane == 0) res_fail(rs);
          continue;  // the next group's decision sees the abort word
        }
        held(u, row, L.slot_data(true, slot));
        __syncwarp();
        if (lane == 0) mbar_arrive(&L.hempty[slot]);
      } else {
        pass(u, row);
      }
      if (lane == 0) atomicAdd(L.normed, 1);
    }
    hg += sh.nh;
  }
  return true;
}

// Block i of group g (row-major over the group's rows): its first unit and size.
__device__ __forceinline__ void res_block(const Plan& p, int64_t g, int64_t i, int64_t& b0, int& bsz) {
  const int64_t cl = i / p.nb, kb = i - cl * p.nb;
  b0 = (g * p.Cg + cl) * p.R + kb * kBlockUnits;
  bsz = block_size(p, kb);
}

// ------------------------------------------------------------- forward
template <class TI>
struct ResFwdShape {
  static constexpr int kRed = 4;    // reduction warps
  static constexpr int kElem = 7;   // elementwise warps (12 warps: 3 per SM sub-partition)
  static constexpr int kWarps = kRed + kElem + 1;
  static constexpr int kRound = 32 * kElem;  // blocks per finalize round
  static constexpr int kSlotBytes = kUnitElems * (int)sizeof(TI);
};

// The value every lane of a warp holds after the xor butterfly of warp_sum
// (offsets 16, 8, 4, 2, 1), computed by one thread from the 32 lane values: the
// same additions on the same operands (IEEE addition commutes), so the same bits.
struct Butterfly {
  float b[16];  // after the offset-16 step, lanes 0 .. 15
  __device__ __forceinline__ float finish() {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
#pragma unroll
      for (int l = 0; l < o; ++l) b[l] = fadd(b[l], b[l + o]);
    return b[0];
  }
};

// merge_block of block (b0, bsz), by one thread: the partials of its units (lane
// i of merge_block holds unit i; lanes from bsz on hold an empty partial).
__device__ __forceinline__ Part thread_merge_block(const Part* __restrict__ parts, int64_t b0, int bsz) {
  Part a[kBlockUnits];
#pragma unroll
  for (int i = 0; i < kBlockUnits; ++i) a[i] = i < bsz ? ldcg_part(parts + b0 + i) : Part{0.f, 0.f, 0, 0.f};
  const float K = fadd(a[0].m1, a[0].cn);
  Butterfly S, Q;
  int n = 0;
#pragma unroll
  for (int i = 0; i < kBlockUnits; ++i) {
    float s, q;
    shifted_terms(a[i], K, s, q);  // lanes 16 .. 31: empty partials, terms +0
    S.b[i] = fadd(s, 0.f);
    Q.b[i] = fadd(q, 0.f);
    n += a[i].n;
  }
  const float St = S.finish(), Qt = Q.finish();
  return finish_merge(K, St, Qt, n);
}

// The group's statistics from its unit partials, by every elementwise warp ew
// of kElem: rounds of kRound blocks, block i of a round merged by lane (i mod
// 32) of elementwise warp (i / 32) into the staging area, exactly as
// merge_block would; then lane l adds blocks l, l + 32, ... in order with the
// shifted sums of the group merge.  The same operations in the same order as
// merge_block and merge_group, so every warp of every CTA ends with the same
// bits as the streaming kernels.
template <int kElem>
__device__ __forceinline__ float4 res_group_stats(const Plan& p, int64_t g, int ew, const Part* __restrict__ parts,
                                                  Part* stage, float eps) {
  constexpr int kRound = 32 * kElem;
  const int lane = threadIdx.x & 31;
  const int64_t nbg = p.Cg * p.nb;
  float K = 0.f, S = 0.f, Q = 0.f;
  for (int64_t base = 0; base < nbg; base += kRound) {
    const int cnt = (int)(nbg - base < kRound ? nbg - base : kRound);
    const int i = 32 * ew + lane;
    if (i < cnt) {
      int64_t b0;
      int bsz;
      res_block(p, g, base + i, b0, bsz);
      stage[i] = thread_merge_block(parts, b0, bsz);
    }
    elem_sync<32 * kElem>();
    if (base == 0) K = fadd(stage[0].m1, stage[0].cn);
#pragma unroll
    for (int m = 0; m < kElem; ++m) {
      const int k = 32 * m + lane;
      if (k < cnt) {
        float s, q;
        shifted_terms(stage[k], K, s, q);
        S = fadd(S, s);
        Q = fadd(Q, q);
      }
    }
    elem_sync<32 * kElem>();
  }
  const float2 t = warp_sum2(S, Q);
  const Part gp = finish_merge(K, t.x, t.y, p.M);
  const float var = __fdiv_rn(gp.m2, (float)p.M);
  return make_float4(gp.m1, gp.cn, __frsqrt_rn(fadd(var, eps)), 0.f);
}

template <class TI, class TO, bool kRelu>
__global__ void __launch_bounds__(32 * ResFwdShape<TI>::kWarps, 1)
    k_fwd_resident(const TI* __restrict__ x, TO* __restrict__ y, Plan p, FwdWs ws, ResCfg c, ResSync rs, float eps,
                   const float* __restrict__ gamma, const float* __restrict__ beta, float* mean_out,
                   float* rstd_out) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Shape = ResFwdShape<TI>;
  ResLayout<Shape::kSlotBytes, Part, Shape::kRound> L;
  L.carve(smem, c.geo);
  L.init(c.geo);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == Shape::kRed + Shape::kElem) {  // the producer
    if (lane == 0) {
      const TI* src[1] = {x};
      res_produce<TI, 1>(p, c, rs, L, src);
    }
    return;
  }
  bool ok;
  if (warp < Shape::kRed) {
    auto unit = [&](const unsigned char* data, bool hd, int slot, int64_t) {
      const TI* body = reinterpret_cast<const TI*>(data);
      Part m;
      if constexpr (Vec<TI>::kRaw == 1) {  // bf16: the unit goes to registers, a pass slot is released at once
        RegView<TI> v;
        v.template load_full<FromShared>(body);
        __syncwarp();
        if (!hd && lane == 0) mbar_arrive(&L.pempty[slot]);
        m = unit_moments_sv<true, TI>(v, 0.f, URange{});
      } else {
        m = unit_moments_sv<true, TI>(MemView<TI, FromShared>{body, kUnitVecs}, 0.f, URange{});
        __syncwarp();
        if (!hd && lane == 0) mbar_arrive(&L.pempty[slot]);
      }
      return m;
    };
    ok = res_reduce<Shape::kRed>(p, c, rs, L, ws.parts, ws.gcnt, unit);
  } else {
    const int ew = warp - Shape::kRed;
    float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
    int64_t crow = -1;
    float gm = 1.f, bt = 0.f;
    auto coef = [&](int64_t row) {
      if (row == crow) return;
      crow = row;
      const int64_t ch = channel_of(row, p.C);
      gm = gamma ? gamma[ch] : 1.f;
      bt = beta ? beta[ch] : 0.f;
    };
    auto fin = [&](int64_t g, bool writer) {
      st = res_group_stats<Shape::kElem>(p, g, ew, ws.parts, L.stage, eps);
      if (writer && ew == 0 && lane == 0) {
        if (mean_out) mean_out[g] = fadd(st.x, st.y);
        if (rstd_out) rstd_out[g] = st.z;
      }
    };
    auto held = [&](int64_t u, int64_t row, const unsigned char* data) {
      coef(row);
      const URange q = full_range(p, row, u - row * p.R);
      fwd_norm<true, TI, TO, MemView<TI, FromShared>, kRelu>(
          MemView<TI, FromShared>{reinterpret_cast<const TI*>(data), kUnitVecs}, x, y, q, st, gm, bt);
    };
    auto pass = [&](int64_t u, int64_t row) {
      coef(row);
      const URange q = full_range(p, row, u - row * p.R);
      if constexpr (Vec<TI>::kRaw == 1) {  // from L2, all 16 vectors in flight
        RegView<TI> v;
        v.template load_full<FromGlobal>(x + q.b0);
        fwd_norm<true, TI, TO, RegView<TI>, kRelu>(v, x, y, q, st, gm, bt);
      } else {
        fwd_norm<true, TI, TO, MemView<TI, FromGlobal>, kRelu>(MemView<TI, FromGlobal>{x + q.b0, kUnitVecs}, x,
                                                                y, q, st, gm, bt);
      }
    };
    ok = res_elementwise<Shape::kRed, Shape::kElem>(p, c, rs, L, ws.gcnt, fin, held, pass);
  }
  if (!ok && lane == 0) res_fail(rs);
}

// ------------------------------------------------------------ backward
template <class T>
struct ResBwdShape {
  static constexpr int kRed = 4;
  static constexpr int kElem = 7;
  static constexpr int kWarps = kRed + kElem + 1;
  static constexpr int kRound = 32 * kElem;
  static constexpr int kSlotBytes = 2 * kUnitElems * (int)sizeof(T);  // x, then dy
};

// The group's coefficients (a, b) from its unit sums, by every elementwise warp:
// each block's sums (warp_sum2 of its 16 unit sums, as the streaming kernels'
// block step), then per row lane l adds blocks l, l + 32, ... in order, the row
// totals meet in the butterfly, and A = sum_c gamma_c*S1_c, B = rstd * sum_c
// gamma_c*S2_c in channel order: the group step of the streaming kernels.  With
// `writer`, warp 0 also stores the row totals (for dgamma, dbeta).
template <int kElem>
__device__ __forceinline__ float2 res_group_coef(const Plan& p, int64_t g, int ew, const float2* __restrict__ parts,
                                                 float2* stage, const float* __restrict__ rstd,
                                                 const float* __restrict__ gamma, float2* rows, bool writer) {
  constexpr int kRound = 32 * kElem;
  const int lane = threadIdx.x & 31;
  const int64_t nbg = p.Cg * p.nb;
  float A = 0.f, B = 0.f, s1 = 0.f, s2 = 0.f;
  for (int64_t base = 0; base < nbg; base += kRound) {
    const int cnt = (int)(nbg - base < kRound ? nbg - base : kRound);
    const int i = 32 * ew + lane;
    if (i < cnt) {  // the block's sums: warp_sum2 of its unit sums, by one thread
      int64_t b0;
      int bsz;
      res_block(p, g, base + i, b0, bsz);
      float2 v[kBlockUnits];
#pragma unroll
      for (int k = 0; k < kBlockUnits; ++k) v[k] = k < bsz ? ldcg_unit(parts + b0 + k) : make_float2(0.f, 0.f);
      Butterfly X, Y;
#pragma unroll
      for (int k = 0; k < kBlockUnits; ++k) {
        X.b[k] = fadd(v[k].x, 0.f);
        Y.b[k] = fadd(v[k].y, 0.f);
      }
      const float bx = X.finish(), by = Y.finish();
      stage[i] = make_float2(bx, by);
    }
    elem_sync<32 * kElem>();
    // the rows met in this round: lane l adds the row's blocks l, l + 32, ...
    const int64_t end = base + cnt;
    for (int64_t cl = base / p.nb; cl * p.nb < end; ++cl) {
      const int64_t r0 = cl * p.nb, r1 = r0 + p.nb;
      const int64_t lo = r0 > base ? r0 : base, hi = r1 < end ? r1 : end;
      // first block of this row in [lo, hi) that is lane l's (kb = l mod 32)
      int64_t kb = lo - r0;
      kb += ((int64_t)lane - kb % 32 + 32) % 32;
      for (; r0 + kb < hi; kb += 32) {
        const float2 b = stage[r0 + kb - base];
        s1 = fadd(s1, b.x);
        s2 = fadd(s2, b.y);
      }
      if (hi == r1) {  // the row is complete
        const float2 t = warp_sum2(s1, s2);
        const int64_t row = g * p.Cg + cl;
        if (writer && ew == 0 && lane == 0) rows[row] = t;
        const float gm = gamma ? gamma[(g % p.G) * p.Cg + cl] : 1.f;
        A = fadd(A, fmul(gm, t.x));
        B = fadd(B, fmul(gm, t.y));
        s1 = 0.f;
        s2 = 0.f;
      }
    }
    elem_sync<32 * kElem>();
  }
  B = fmul(rstd[g], B);
  const float fM = (float)p.M;
  return make_float2(__fdiv_rn(A, fM), __fdiv_rn(B, fM));
}

template <class T>
__global__ void __launch_bounds__(32 * ResBwdShape<T>::kWarps, 1)
    k_bwd_resident(const T* __restrict__ dy, const T* __restrict__ x, T* __restrict__ dx, Plan p,
                   const float* __restrict__ mean, const float* __restrict__ rstd, const float* __restrict__ gamma,
                   BwdWs ws, ResCfg c, ResSync rs, float* dgamma, float* dbeta) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Shape = ResBwdShape<T>;
  constexpr int kTensorBytes = kUnitElems * (int)sizeof(T);
  ResLayout<Shape::kSlotBytes, float2, Shape::kRound> L;
  L.carve(smem, c.geo);
  L.init(c.geo);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == Shape::kRed + Shape::kElem) {
    if (lane == 0) {
      const T* src[2] = {x, dy};
      res_produce<T, 2>(p, c, rs, L, src);
    }
    return;
  }
  bool ok;
  if (warp < Shape::kRed) {
    auto unit = [&](const unsigned char* data, bool hd, int slot, int64_t g) {
      const float mu = mean[g];
      const f2 z2 = f2_splat(0.f);
      f2 a1[4] = {z2, z2, z2, z2};
      f2 a2[4] = {z2, z2, z2, z2};
      bwd_accum<true, T>(MemView<T, FromShared>{reinterpret_cast<const T*>(data), kUnitVecs},
                         MemView<T, FromShared>{reinterpret_cast<const T*>(data + kTensorBytes), kUnitVecs}, 0,
                         kVecPerLane, mu, a1, a2);
      __syncwarp();
      if (!hd && lane == 0) mbar_arrive(&L.pempty[slot]);
      return bwd_finish_sv<true>(a1, a2, BwdScalar{0.f, 0.f}, URange{}, mu);
    };
    ok = res_reduce<Shape::kRed>(p, c, rs, L, ws.parts, ws.gcnt, unit);
  } else {
    const int ew = warp - Shape::kRed;
    DxCoef kc{0.f, 0.f, 0.f, 0.f, false};
    int64_t crow = -1;
    float gm = 1.f;
    auto fin = [&](int64_t g, bool writer) {
      const float2 ab = res_group_coef<Shape::kElem>(p, g, ew, ws.parts, L.stage, rstd, gamma, ws.rows, writer);
      kc = DxCoef{mean[g], rstd[g], ab.x, ab.y, p.M == 1};
      if (writer && ew == 0) {
        // the group's rows are stored: the writer of the last group to finish
        // forms dgamma and dbeta in n order from every group's rows
        if (lane == 0) ws.coef[g] = ab;
        if (warp_arrive_last(ws.done, (uint32_t)p.NG)) bwd_param_grads(p, rstd, ws.rows, dgamma, dbeta);
      }
    };
    auto coef = [&](int64_t row) {
      if (row == crow) return;
      crow = row;
      gm = gamma ? gamma[channel_of(row, p.C)] : 1.f;
    };
    auto held = [&](int64_t u, int64_t row, const unsigned char* data) {
      coef(row);
      const URange q = full_range(p, row, u - row * p.R);
      bwd_norm<true, T>(MemView<T, FromShared>{reinterpret_cast<const T*>(data), kUnitVecs},
                        MemView<T, FromShared>{reinterpret_cast<const T*>(data + kTensorBytes), kUnitVecs}, x, dy,
                        dx, q, kc, gm);
    };
    auto pass = [&](int64_t u, int64_t row) {  // from L2, 8 vectors of each tensor in flight per lane
      coef(row);
      const URange q = full_range(p, row, u - row * p.R);
      bwd_norm_staged<T, false, 8 / Vec<T>::kRaw>(x, dy, nullptr, dx, q, kc, gm);
    };
    ok = res_elementwise<Shape::kRed, Shape::kElem>(p, c, rs, L, ws.gcnt, fin, held, pass);
  }
  if (!ok && lane == 0) res_fail(rs);
}

}  // namespace gn3d
