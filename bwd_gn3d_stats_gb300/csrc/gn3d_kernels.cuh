// gn3d_kernels.cuh -- the streaming launch form: two kernels per direction.
//
// Forward  (ScaFFold PR #93 "Optimize GroupNorm": split-group statistics, a
//           corrected two-pass per tile merged with Chan's formula, then a
//           normalize that rounds once on the store, PR #105):
//   k_fwd_stats : each warp takes an equal share of consecutive units
//                 (UnitWalk) and streams their bodies through a private ring of
//                 shared-memory slots filled by 1-D bulk copies (the TMA
//                 engine), so several units per warp are always in flight; it
//                 merges each merge block it holds whole in registers, a block
//                 cut between two shares is merged by the warp completing it,
//                 and the warp that completes a group merges the group.
//   k_fwd_norm  : normalizes the units of each statistics warp's share, on the
//                 same CTA index (so, for identical launches, the same SM), last
//                 unit first: what that SM read last is read again first, while
//                 it is still in L2.
// Backward (the same PR's _bwd_finalize/_dwdb_reduce/_dx split):
//   k_bwd_reduce: S1 = sum dy, S2 = sum dy*(x - mean) per unit, through the same
//                 kind of ring; group and parameter-gradient merges by the
//                 completing warps.
//   k_bwd_dx    : dx over the reduction warps' shares, the same way.
// These use exactly the units, merge blocks and arithmetic of the persistent
// kernels (gn3d_device.cuh), so the two launch forms give bit-identical results.
#pragma once
#include "gn3d_device.cuh"
#include "gn3d_sync.cuh"

namespace gn3d {

// ---------------------------------------------------------- unit rings
// The worker index of warp w of CTA c, of grid*warps: in unit shares c*warps +
// w (each CTA a run of consecutive shares), in strided blocks w*grid + c (every
// CTA blocks from all over the tensor); either way every SM gets an equal part.
template <int kWarps>
__device__ __forceinline__ int64_t worker_index(bool cut, int warp) {
  return cut ? (int64_t)blockIdx.x * kWarps + warp : (int64_t)warp * gridDim.x + blockIdx.x;
}

// A warp's private ring: kSlots slots, each holding kElems consecutive body
// elements of each of kTensors tensors (a whole unit, or one of its
// kUnitElems / kElems parts), one "full" mbarrier per slot.  Lane 0 issues the
// bulk copies; the warp reads a slot only after its barrier phase completed,
// and refills it only after every lane's reads of it (a __syncwarp, then the
// proxy fence) -- no other warp touches it.
template <class T, int kTensors, int kSlots, int kElems = kUnitElems>
struct WarpRing {
  static constexpr int kTensorBytes = kElems * (int)sizeof(T);
  static constexpr int kSlotBytes = kTensors * kTensorBytes;
  static constexpr int kParts = kUnitElems / kElems;
  // a warp's region: its slots, then its barriers, rounded up so that every
  // warp's slots start on a 128-byte boundary (bulk copies need 16)
  static constexpr int kWarpBytes = (kSlots * (kSlotBytes + 8) + 127) / 128 * 128;
  static_assert(kUnitElems % kElems == 0 && kElems % (32 * kVec) == 0, "parts of whole lane rows");
  static_assert(kSlotBytes % 128 == 0 && kTensorBytes % 16 == 0, "slot alignment");
  static_assert((kSlots * kSlotBytes) % 8 == 0, "mbarrier alignment");
  unsigned char* data;   // kSlots * kSlotBytes
  uint64_t* bar;         // kSlots
  int64_t issued = 0;    // copies issued
  int64_t taken = 0;     // slots consumed

  __device__ __forceinline__ void init(unsigned char* base) {
    data = base;
    bar = reinterpret_cast<uint64_t*>(base + (size_t)kSlots * kSlotBytes);
    if ((threadIdx.x & 31) == 0) {
      for (int i = 0; i < kSlots; ++i) mbar_init(&bar[i], 1);
      fence_mbar_init();
    }
    __syncwarp();
  }
  // Issue part `part` of the body of unit q into the next slot (all lanes call;
  // lane 0 copies).  A part past the end of a short body is empty: its barrier
  // phase completes on the arrival alone.
  __device__ __forceinline__ void issue(const URange& q, int part, const T* const* src) {
    const int slot = (int)(issued % kSlots);
    if ((threadIdx.x & 31) == 0) {
      const int64_t body = q.b1 - q.b0;
      const int64_t e0 = min((int64_t)part * kElems, body), e1 = min((int64_t)(part + 1) * kElems, body);
      const uint32_t bytes = (uint32_t)((e1 - e0) * (int64_t)sizeof(T));
      unsigned char* dst = data + (size_t)slot * kSlotBytes;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bar[slot], bytes * kTensors);
      if (bytes) {
#pragma unroll
        for (int t = 0; t < kTensors; ++t) bulk_g2s(dst + t * kTensorBytes, src[t] + q.b0 + e0, bytes, &bar[slot]);
      }
    }
    ++issued;
  }
  // Wait (bounded) for the next slot's copy; returns its data or nullptr.
  __device__ __forceinline__ const unsigned char* take(unsigned long long spin) {
    const int slot = (int)(taken % kSlots);
    if (!mbar_wait_bounded(&bar[slot], (uint32_t)((taken / kSlots) & 1), spin)) return nullptr;
    ++taken;
    return data + (size_t)slot * kSlotBytes;
  }
  // Wait (bounded) for every copy still in flight, after a failure.
  __device__ __forceinline__ void drain(unsigned long long spin) {
    for (int64_t t = taken; t < issued; ++t)
      mbar_wait_bounded(&bar[t % kSlots], (uint32_t)((t / kSlots) & 1), spin);
  }
};

// The load-ahead position of a ring: a block walk plus the part of the unit.
struct PartWalk {
  UnitWalk w;
  int part = 0;
  __device__ __forceinline__ void next(const Plan& p, int parts) {
    if (++part < parts) return;
    part = 0;
    w.next(p);
  }
};

// Unit k of a row: the general range, or its closed form when every unit is full.
template <bool kFull>
__device__ __forceinline__ URange urange(const Plan& p, int64_t row, int64_t k) {
  return kFull ? full_range(p, row, k) : unit_range_rk(p, row, k);
}

__device__ __forceinline__ void record_timeout(uint32_t* status) {
  if ((threadIdx.x & 31) == 0) atomicExch(status, 4u);  // GN3D_ERR_TIMEOUT
}

// Ring shapes per kernel and dtype: warps per CTA and slots per warp, one CTA
// per SM, every ring in 192 KB of shared memory.
template <class T> struct FwdStatShape {
  static constexpr int kWarps = sizeof(T) == 2 ? 8 : 4;
  static constexpr int kSlots = 3;
};
template <class T, bool kRelu = false> struct BwdRedShape {
  // a slot: 4 KB of each of x and dy (8 KB), or -- behind a fused ReLU, with the
  // forward's result as a third tensor -- 2 KB of each (6 KB, four slots)
  static constexpr int kWarps = 8;
  static constexpr int kSlots = kRelu ? 4 : 3;
  static constexpr int kTensors = kRelu ? 3 : 2;
  static constexpr int kElems = (kRelu ? 2048 : 4096) / (int)sizeof(T);
};

template <class TI, bool kFull, bool kCut>
__global__ void __launch_bounds__(32 * FwdStatShape<TI>::kWarps, 1)
    k_fwd_stats(const TI* __restrict__ x, Plan p, FwdWs ws, float eps, float* mean_out, float* rstd_out,
                unsigned long long spin, uint32_t* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Shape = FwdStatShape<TI>;
  using Ring = WarpRing<TI, 1, Shape::kSlots>;
  constexpr bool kRegs = Vec<TI>::kRaw == 1;  // bf16: the unit goes to registers, the slot is refilled at once
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();  // the normalize kernel may take SMs as this one leaves them
  Ring ring;
  ring.init(smem + (size_t)warp * Ring::kWarpBytes);
  const TI* src[1] = {x};
  UnitWalk ld, cu;
  ld.set(p, worker_index<Shape::kWarps>(kCut, warp), (int64_t)gridDim.x * Shape::kWarps, kCut);
  cu = ld;
  for (int i = 0; i < Shape::kSlots && !ld.end; ++i) {
    ring.issue(urange<kFull>(p, ld.row, ld.k), 0, src);
    ld.next(p);
  }
  const Part empty{0.f, 0.f, 0, 0.f};
  Part a = empty;  // lane l: the partial of unit l of the current block
  float sv = cu.end ? 0.f : unit_scalar<kFull, TI>(x, urange<kFull>(p, cu.row, cu.k));
  while (!cu.end) {
    const URange q = urange<kFull>(p, cu.row, cu.k);
    const int nv = (int)((q.b1 - q.b0) / kVec);
    float sv_next = 0.f;  // the next unit's scalar, in flight while this unit is summed
    if (!kFull) {
      UnitWalk nx = cu;
      nx.next(p);
      if (!nx.end) sv_next = unit_scalar<kFull, TI>(x, urange<kFull>(p, nx.row, nx.k));
    }
    const unsigned char* slot = ring.take(spin);
    if (!slot) {
      record_timeout(status);
      break;
    }
    // a full unit of a ragged plan takes the full-unit code: the same
    // operations on the same operands, so the same bits (unit_moments_sv)
    const bool fu = kFull || unit_is_full(q);
    Part m;
    if (kRegs) {
      RegView<TI> v;
      if (fu) v.template load_full<FromShared>(reinterpret_cast<const TI*>(slot));
      else v.template load<FromShared>(reinterpret_cast<const TI*>(slot), nv);
      __syncwarp();
      if (!ld.end) {
        ring.issue(urange<kFull>(p, ld.row, ld.k), 0, src);
        ld.next(p);
      }
      m = fu ? unit_moments_sv<true, TI>(v, sv, q) : unit_moments_sv<kFull, TI>(v, sv, q);
    } else {
      const MemView<TI, FromShared> v{reinterpret_cast<const TI*>(slot), nv};
      m = fu ? unit_moments_sv<true, TI>(v, sv, q) : unit_moments_sv<kFull, TI>(v, sv, q);
      __syncwarp();
      if (!ld.end) {
        ring.issue(urange<kFull>(p, ld.row, ld.k), 0, src);
        ld.next(p);
      }
    }
    const int ui = cu.ui(), bsz = block_size(p, cu.kb());
    if (lane == ui) a = m;
    if (ui == bsz - 1 || (kCut && cu.u + 1 == cu.u1)) {  // the block, or this warp's part of it, is done
      const int64_t blk = cu.row * p.nb + cu.kb();
      bool merge = ui == bsz - 1;
      Part v = lane < bsz ? a : empty;
      if constexpr (kCut) {
        const int64_t ub = cu.u - ui;
        const int lo = ub >= cu.u0 ? 0 : (int)(cu.u0 - ub);
        if (lo > 0 || ui < bsz - 1) {  // a cut block: the warp completing it merges it
          merge = split_block_arrive(ws.parts + ub, ws.bcnt + blk, lo, ui, bsz, a);
          if (merge) v = lane < bsz ? ldcg_unit(ws.parts + ub + lane) : empty;
        }
      }
      if (merge) fwd_block_done(p, ws, blk, merge_block(v), eps, mean_out, rstd_out);
      a = empty;
    }
    sv = sv_next;
    cu.next(p);
  }
  ring.drain(kDrainPolls);
}

// Elementwise passes: 16 warps per CTA, on the reduction kernel's grid, each
// taking units so that what the reduction read last is read again first, while
// it is still in L2.  Under unit shares warp w takes the units of reduction
// warp w % kOwners of the same CTA, every (16 / kOwners)-th, in the reverse of
// that warp's order (UnitWalkDown).  Under strided blocks the units are spread
// evenly over all the grid's warps, freshest first (UnitWalkFresh): a block is
// one reduction warp's whole work there, so following the owner would leave
// the warps of idle owners idle.  Placement only decides what is found in L2,
// never a result.
constexpr int kElemWarps = 16;

template <int kOwners, bool kCut>
__device__ __forceinline__ auto owned_units(const Plan& p) {
  const int warp = threadIdx.x >> 5;
  if constexpr (kCut) {
    UnitWalkDown w;
    w.set(p, worker_index<kOwners>(kCut, warp % kOwners), (int64_t)gridDim.x * kOwners, kCut, warp / kOwners,
          kElemWarps / kOwners);
    return w;
  } else {
    UnitWalkFresh w;
    w.set(p, (int64_t)warp * gridDim.x + blockIdx.x, (int64_t)gridDim.x * kElemWarps, (int64_t)gridDim.x * kOwners);
    return w;
  }
}

template <class TI, class TO, bool kFull, bool kRelu, bool kCut>
__global__ void __launch_bounds__(32 * kElemWarps, 1)
    k_fwd_norm(const TI* __restrict__ x, TO* __restrict__ y, Plan p, const float4* __restrict__ stats,
               const float* __restrict__ gamma, const float* __restrict__ beta) {
  constexpr bool kRegs = Vec<TI>::kRaw == 1;  // bf16: all 16 loads in flight before any use
  auto w = owned_units<FwdStatShape<TI>::kWarps, kCut>(p);
  // The warp's first unit is read before the statistics kernel has finished
  // (x is not written there); everything the statistics kernel writes is read
  // after pdl_wait.
  RegView<TI> v;
  bool pre = false;
  if (kRegs && !w.end()) {
    const URange q = urange<kFull>(p, w.row, w.k);
    if (kFull) v.template load_full<FromGlobal>(x + q.b0);
    else v.template load<FromGlobal>(x + q.b0, (int)((q.b1 - q.b0) / kVec));
    pre = true;
  }
  pdl_wait();
  int64_t row = -1;
  float4 st;
  float gm = 1.f, bt = 0.f;
  for (; !w.end(); w.next(p)) {
    if (w.row != row) {  // the row's coefficients
      row = w.row;
      const int64_t c = channel_of(row, p.C);
      st = __ldcg(stats + row / p.Cg);
      gm = gamma ? gamma[c] : 1.f;
      bt = beta ? beta[c] : 0.f;
    }
    const URange q = urange<kFull>(p, w.row, w.k);
    const int nv = (int)((q.b1 - q.b0) / kVec);
    const bool fu = kFull || unit_is_full(q);  // a full unit of a ragged plan: the full-unit code, the same bits
    if (kRegs) {
      if (!pre) {
        if (fu) v.template load_full<FromGlobal>(x + q.b0);
        else v.template load<FromGlobal>(x + q.b0, nv);
      }
      pre = false;
      if (fu) fwd_norm<true, TI, TO, RegView<TI>, kRelu>(v, x, y, q, st, gm, bt);
      else fwd_norm<kFull, TI, TO, RegView<TI>, kRelu>(v, x, y, q, st, gm, bt);
    } else {
      const MemView<TI, FromGlobal> mv{x + q.b0, nv};
      if (fu) fwd_norm<true, TI, TO, MemView<TI, FromGlobal>, kRelu>(mv, x, y, q, st, gm, bt);
      else fwd_norm<kFull, TI, TO, MemView<TI, FromGlobal>, kRelu>(mv, x, y, q, st, gm, bt);
    }
  }
}

template <class T, bool kFull, bool kRelu, bool kCut>
__global__ void __launch_bounds__(32 * BwdRedShape<T, kRelu>::kWarps, 1)
    k_bwd_reduce(const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ res, Plan p,
                 const float* __restrict__ mean, const float* __restrict__ rstd, const float* __restrict__ gamma,
                 BwdWs ws, float* dgamma, float* dbeta, unsigned long long spin, uint32_t* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  using Shape = BwdRedShape<T, kRelu>;
  using Ring = WarpRing<T, Shape::kTensors, Shape::kSlots, Shape::kElems>;
  constexpr int kParts = Ring::kParts, kPartVecs = kVecPerLane / kParts;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();  // the dx kernel may take SMs as this one leaves them
  Ring ring;
  ring.init(smem + (size_t)warp * Ring::kWarpBytes);
  const T* src[3] = {x, dy, res};
  PartWalk ld;
  ld.w.set(p, worker_index<Shape::kWarps>(kCut, warp), (int64_t)gridDim.x * Shape::kWarps, kCut);
  UnitWalk cu = ld.w;
  for (int i = 0; i < Shape::kSlots && !ld.w.end; ++i) {
    ring.issue(urange<kFull>(p, ld.w.row, ld.w.k), ld.part, src);
    ld.next(p, kParts);
  }
  const float2 zero = make_float2(0.f, 0.f);
  float2 a = zero;  // lane l: the sums of unit l of the current block
  bool failed = false;
  const T* gate = kRelu ? res : nullptr;
  BwdScalar sc = cu.end ? BwdScalar{0.f, 0.f} : bwd_scalar<kFull, T>(x, dy, gate, urange<kFull>(p, cu.row, cu.k));
  while (!cu.end) {
    const URange q = urange<kFull>(p, cu.row, cu.k);
    const int nv = (int)((q.b1 - q.b0) / kVec);
    const float mu = mean[q.row / p.Cg];
    BwdScalar sc_next{0.f, 0.f};  // the next unit's scalar, in flight while this unit is summed
    if (!kFull) {
      UnitWalk nx = cu;
      nx.next(p);
      if (!nx.end) sc_next = bwd_scalar<kFull, T>(x, dy, gate, urange<kFull>(p, nx.row, nx.k));
    }
    const f2 z2 = f2_splat(0.f);
    f2 a1[4] = {z2, z2, z2, z2};
    f2 a2[4] = {z2, z2, z2, z2};
    // a full unit of a ragged plan takes the full-unit code: the same
    // operations on the same operands, so the same bits (bwd_accum, bwd_finish_sv)
    const bool fu = kFull || unit_is_full(q);
#pragma unroll
    for (int part = 0; part < kParts; ++part) {
      const unsigned char* slot = ring.take(spin);
      if (!slot) {
        failed = true;
        break;
      }
      // views placed so that vector i of the unit is read from this part's slot
      const T* xs = reinterpret_cast<const T*>(slot) - (size_t)part * Shape::kElems;
      const T* ds = reinterpret_cast<const T*>(slot + Ring::kTensorBytes) - (size_t)part * Shape::kElems;
      const int i0 = part * kPartVecs, i1 = (part + 1) * kPartVecs;
      if constexpr (kRelu) {
        const T* rs = reinterpret_cast<const T*>(slot + 2 * Ring::kTensorBytes) - (size_t)part * Shape::kElems;
        const MemView<T, FromShared> vx{xs, nv};
        const GatedView<T, FromShared> vd{ds, rs, nv};
        if (fu) bwd_accum<true, T>(vx, vd, i0, i1, mu, a1, a2);
        else bwd_accum<kFull, T>(vx, vd, i0, i1, mu, a1, a2);
      } else {
        const MemView<T, FromShared> vx{xs, nv}, vd{ds, nv};
        if (fu) bwd_accum<true, T>(vx, vd, i0, i1, mu, a1, a2);
        else bwd_accum<kFull, T>(vx, vd, i0, i1, mu, a1, a2);
      }
      __syncwarp();
      if (!ld.w.end) {
        ring.issue(urange<kFull>(p, ld.w.row, ld.w.k), ld.part, src);
        ld.next(p, kParts);
      }
    }
    if (failed) {
      record_timeout(status);
      break;
    }
    const float2 v = fu ? bwd_finish_sv<true>(a1, a2, sc, q, mu) : bwd_finish_sv<kFull>(a1, a2, sc, q, mu);
    const int ui = cu.ui(), bsz = block_size(p, cu.kb());
    if (lane == ui) a = v;
    if (ui == bsz - 1 || (kCut && cu.u + 1 == cu.u1)) {  // the block, or this warp's part of it, is done
      const int64_t blk = cu.row * p.nb + cu.kb();
      bool merge = ui == bsz - 1;
      float2 bs = lane < bsz ? a : zero;
      if constexpr (kCut) {
        const int64_t ub = cu.u - ui;
        const int lo = ub >= cu.u0 ? 0 : (int)(cu.u0 - ub);
        if (lo > 0 || ui < bsz - 1) {  // a cut block: the warp completing it merges it
          merge = split_block_arrive(ws.parts + ub, ws.bcnt + blk, lo, ui, bsz, a);
          if (merge) bs = lane < bsz ? ldcg_unit(ws.parts + ub + lane) : zero;
        }
      }
      if (merge) bwd_block_done(p, ws, blk, bs, rstd, gamma, dgamma, dbeta);
      a = zero;
    }
    sc = sc_next;
    cu.next(p);
  }
  ring.drain(kDrainPolls);
}

template <class T, bool kFull, bool kRelu, bool kCut>
__global__ void __launch_bounds__(32 * kElemWarps, 1)
    k_bwd_dx(const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ res, T* __restrict__ dx,
             Plan p, const float* __restrict__ mean, const float* __restrict__ rstd,
             const float* __restrict__ gamma, const float2* __restrict__ coef) {
  auto w = owned_units<BwdRedShape<T, kRelu>::kWarps, kCut>(p);
  pdl_wait();  // the reduction kernel's coefficients
  int64_t row = -1;
  DxCoef k{0.f, 0.f, 0.f, 0.f, false};
  float gm = 1.f;
  for (; !w.end(); w.next(p)) {
    if (w.row != row) {  // the row's coefficients
      row = w.row;
      const int64_t c = channel_of(row, p.C), g = row / p.Cg;
      const float2 ab = __ldcg(coef + g);
      k = DxCoef{mean[g], rstd[g], ab.x, ab.y, p.M == 1};
      gm = gamma ? gamma[c] : 1.f;
    }
    const URange q = urange<kFull>(p, w.row, w.k);
    const int nv = (int)((q.b1 - q.b0) / kVec);
    if constexpr (!kFull) {
      bwd_norm_staged<T, kRelu, (kRelu ? 4 : 8) / Vec<T>::kRaw>(x, dy, res, dx, q, k, gm);
    } else if constexpr (kRelu) {
      bwd_norm<kFull, T>(MemView<T, FromGlobal>{x + q.b0, nv}, GatedView<T, FromGlobal>{dy + q.b0, res + q.b0, nv},
                         x, dy, dx, q, k, gm, res);
    } else {
      bwd_norm<kFull, T>(MemView<T, FromGlobal>{x + q.b0, nv}, MemView<T, FromGlobal>{dy + q.b0, nv}, x, dy, dx,
                         q, k, gm);
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
