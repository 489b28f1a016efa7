// gn3d_kernels.cuh -- the streaming launch form: two kernels per direction.
//
// Forward  (ScaFFold PR #93 "Optimize GroupNorm": split-group statistics, a
//           corrected two-pass per tile merged with Chan's formula, then a
//           normalize that rounds once on the store, PR #105):
//   k_fwd_stats : each warp owns whole merge blocks (up to 16 consecutive units
//                 of a row) and streams their bodies through a private ring of
//                 shared-memory slots filled by 1-D bulk copies (the TMA
//                 engine), so several units per warp are always in flight; it
//                 merges each block in registers and the warp that completes a
//                 group merges the group.
//   k_fwd_norm  : normalizes the blocks each statistics warp owned, on the same
//                 CTA index (so, for identical launches, the same SM), last
//                 block and last unit first: what that SM read last is read
//                 again first, while it is still in L2.
// Backward (the same PR's _bwd_finalize/_dwdb_reduce/_dx split):
//   k_bwd_reduce: S1 = sum dy, S2 = sum dy*(x - mean) per unit, through the same
//                 kind of ring; group and parameter-gradient merges by the
//                 completing warps.
//   k_bwd_dx    : dx over the reduction warps' blocks, the same way.
// These use exactly the units, merge blocks and arithmetic of the persistent
// kernels (gn3d_device.cuh), so the two launch forms give bit-identical results.
#pragma once
#include "gn3d_device.cuh"
#include "gn3d_sync.cuh"

namespace gn3d {

// ---------------------------------------------------------- block rings
// Warp w of CTA c walks merge blocks b = w*grid + c, then b + warps*grid, ...
// (every SM gets an equal share of each part of the tensor), unit by unit.
struct BlockWalk {
  int64_t b, row, kb;  // current block, its row and index in the row
  int bsz, ui;         // its unit count; the current unit in it
  bool end;
  __device__ __forceinline__ void set(const Plan& p, int64_t b_, int64_t nblk) {
    b = b_;
    end = b >= nblk;
    if (!end) {
      row = b / p.nb;
      kb = b - row * p.nb;
      bsz = block_size(p, kb);
      ui = 0;
    }
  }
  __device__ __forceinline__ void next(const Plan& p, int64_t stride, int64_t nblk) {
    if (++ui >= bsz) set(p, b + stride, nblk);
  }
  __device__ __forceinline__ int64_t k() const { return kb * kBlockUnits + ui; }
};

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
  BlockWalk w;
  int part = 0;
  __device__ __forceinline__ void next(const Plan& p, int64_t stride, int64_t nblk, int parts) {
    if (++part < parts) return;
    part = 0;
    w.next(p, stride, nblk);
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

template <class TI, bool kFull>
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
  const int64_t nblk = p.NC * p.nb, stride = (int64_t)gridDim.x * Shape::kWarps;
  const int64_t first = (int64_t)warp * gridDim.x + blockIdx.x;
  const TI* src[1] = {x};
  BlockWalk ld, cu;
  ld.set(p, first, nblk);
  cu = ld;
  for (int i = 0; i < Shape::kSlots && !ld.end; ++i) {
    ring.issue(urange<kFull>(p, ld.row, ld.k()), 0, src);
    ld.next(p, stride, nblk);
  }
  Part a{0.f, 0.f, 0, 0.f};  // lane l: the partial of unit l of the current block
  while (!cu.end) {
    const unsigned char* slot = ring.take(spin);
    if (!slot) {
      record_timeout(status);
      break;
    }
    const URange q = urange<kFull>(p, cu.row, cu.k());
    const int nv = (int)((q.b1 - q.b0) / kVec);
    Part m;
    if (kRegs) {
      RegView<TI> v;
      if (kFull) v.template load_full<FromShared>(reinterpret_cast<const TI*>(slot));
      else v.template load<FromShared>(reinterpret_cast<const TI*>(slot), nv);
      __syncwarp();
      if (!ld.end) {
        ring.issue(urange<kFull>(p, ld.row, ld.k()), 0, src);
        ld.next(p, stride, nblk);
      }
      m = unit_moments<kFull, TI>(v, x, q);
    } else {
      m = unit_moments<kFull, TI>(MemView<TI, FromShared>{reinterpret_cast<const TI*>(slot), nv}, x, q);
      __syncwarp();
      if (!ld.end) {
        ring.issue(urange<kFull>(p, ld.row, ld.k()), 0, src);
        ld.next(p, stride, nblk);
      }
    }
    if (lane == cu.ui) a = m;
    if (cu.ui == cu.bsz - 1) {
      fwd_block_done(p, ws, cu.b, merge_block(lane < cu.bsz ? a : Part{0.f, 0.f, 0, 0.f}), eps, mean_out,
                     rstd_out);
      a = Part{0.f, 0.f, 0, 0.f};
    }
    cu.next(p, stride, nblk);
  }
  ring.drain(kDrainPolls);
}

// Elementwise passes: 16 warps per CTA, on the reduction kernel's grid.  Warp w
// takes the blocks of reduction warp w % kOwners of the same CTA, from its last
// block back to its first, and in each block every (16 / kOwners)-th unit from
// the last one down.  Placement only decides what is found in L2, never a result.
constexpr int kElemWarps = 16;

template <int kOwners>
struct OwnedBlocks {
  static constexpr int kSplit = kElemWarps / kOwners;
  int64_t b0, stride;
  int share;
  __device__ __forceinline__ OwnedBlocks() {
    const int warp = threadIdx.x >> 5;
    stride = (int64_t)gridDim.x * kOwners;
    b0 = (int64_t)(warp % kOwners) * gridDim.x + blockIdx.x;
    share = warp / kOwners;
  }
  // the owner's last block, or -1
  __device__ __forceinline__ int64_t last(int64_t nblk) const {
    return b0 < nblk ? b0 + (nblk - 1 - b0) / stride * stride : -1;
  }
};

template <class TI, class TO, bool kFull, bool kRelu>
__global__ void __launch_bounds__(32 * kElemWarps, 1)
    k_fwd_norm(const TI* __restrict__ x, TO* __restrict__ y, Plan p, const float4* __restrict__ stats,
               const float* __restrict__ gamma, const float* __restrict__ beta) {
  using Own = OwnedBlocks<FwdStatShape<TI>::kWarps>;
  constexpr bool kRegs = Vec<TI>::kRaw == 1;  // bf16: all 16 loads in flight before any use
  const Own own;
  const int64_t nblk = p.NC * p.nb;
  // The warp's first unit is read before the statistics kernel has finished
  // (x is not written there); everything the statistics kernel writes is read
  // after pdl_wait.
  RegView<TI> v;
  bool pre = false;
  const int64_t b_first = own.last(nblk);
  if (kRegs && b_first >= own.b0) {
    const int64_t row = b_first / p.nb, kb = b_first - row * p.nb;
    const int ui = block_size(p, kb) - 1 - own.share;
    if (ui >= 0) {
      const URange q = urange<kFull>(p, row, kb * kBlockUnits + ui);
      if (kFull) v.template load_full<FromGlobal>(x + q.b0);
      else v.template load<FromGlobal>(x + q.b0, (int)((q.b1 - q.b0) / kVec));
      pre = true;
    }
  }
  pdl_wait();
  for (int64_t b = b_first; b >= own.b0; b -= own.stride) {
    const int64_t row = b / p.nb, kb = b - row * p.nb;
    const int bsz = block_size(p, kb);
    const int64_t c = channel_of(row, p.C), g = row / p.Cg;
    const float4 st = __ldcg(stats + g);
    const float gm = gamma ? gamma[c] : 1.f, bt = beta ? beta[c] : 0.f;
    for (int ui = bsz - 1 - own.share; ui >= 0; ui -= Own::kSplit) {
      const URange q = urange<kFull>(p, row, kb * kBlockUnits + ui);
      const int nv = (int)((q.b1 - q.b0) / kVec);
      if (kRegs) {
        if (!pre) {
          if (kFull) v.template load_full<FromGlobal>(x + q.b0);
          else v.template load<FromGlobal>(x + q.b0, nv);
        }
        pre = false;
        fwd_norm<kFull, TI, TO, RegView<TI>, kRelu>(v, x, y, q, st, gm, bt);
      } else {
        fwd_norm<kFull, TI, TO, MemView<TI, FromGlobal>, kRelu>(MemView<TI, FromGlobal>{x + q.b0, nv}, x, y, q, st,
                                                                gm, bt);
      }
    }
  }
}

template <class T, bool kFull, bool kRelu>
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
  const int64_t nblk = p.NC * p.nb, stride = (int64_t)gridDim.x * Shape::kWarps;
  const int64_t first = (int64_t)warp * gridDim.x + blockIdx.x;
  const T* src[3] = {x, dy, res};
  PartWalk ld;
  ld.w.set(p, first, nblk);
  BlockWalk cu = ld.w;
  for (int i = 0; i < Shape::kSlots && !ld.w.end; ++i) {
    ring.issue(urange<kFull>(p, ld.w.row, ld.w.k()), ld.part, src);
    ld.next(p, stride, nblk, kParts);
  }
  float2 a = make_float2(0.f, 0.f);  // lane l: the sums of unit l of the current block
  bool failed = false;
  while (!cu.end) {
    const URange q = urange<kFull>(p, cu.row, cu.k());
    const int nv = (int)((q.b1 - q.b0) / kVec);
    const float mu = mean[q.row / p.Cg];
    const f2 z2 = f2_splat(0.f);
    f2 a1[4] = {z2, z2, z2, z2};
    f2 a2[4] = {z2, z2, z2, z2};
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
      if constexpr (kRelu) {
        const T* rs = reinterpret_cast<const T*>(slot + 2 * Ring::kTensorBytes) - (size_t)part * Shape::kElems;
        bwd_accum<kFull, T>(MemView<T, FromShared>{xs, nv}, GatedView<T, FromShared>{ds, rs, nv},
                            part * kPartVecs, (part + 1) * kPartVecs, mu, a1, a2);
      } else {
        bwd_accum<kFull, T>(MemView<T, FromShared>{xs, nv}, MemView<T, FromShared>{ds, nv}, part * kPartVecs,
                            (part + 1) * kPartVecs, mu, a1, a2);
      }
      __syncwarp();
      if (!ld.w.end) {
        ring.issue(urange<kFull>(p, ld.w.row, ld.w.k()), ld.part, src);
        ld.next(p, stride, nblk, kParts);
      }
    }
    if (failed) {
      record_timeout(status);
      break;
    }
    const float2 v = bwd_finish<kFull, T>(a1, a2, x, dy, q, mu, kRelu ? res : nullptr);
    if (lane == cu.ui) a = v;
    if (cu.ui == cu.bsz - 1) {
      bwd_block_done(p, ws, cu.b, lane < cu.bsz ? a : make_float2(0.f, 0.f), rstd, gamma, dgamma, dbeta);
      a = make_float2(0.f, 0.f);
    }
    cu.next(p, stride, nblk);
  }
  ring.drain(kDrainPolls);
}

template <class T, bool kFull, bool kRelu>
__global__ void __launch_bounds__(32 * kElemWarps, 1)
    k_bwd_dx(const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ res, T* __restrict__ dx,
             Plan p, const float* __restrict__ mean, const float* __restrict__ rstd,
             const float* __restrict__ gamma, const float2* __restrict__ coef) {
  using Own = OwnedBlocks<BwdRedShape<T, kRelu>::kWarps>;
  const Own own;
  const int64_t nblk = p.NC * p.nb;
  pdl_wait();  // the reduction kernel's coefficients
  for (int64_t b = own.last(nblk); b >= own.b0; b -= own.stride) {
    const int64_t row = b / p.nb, kb = b - row * p.nb;
    const int bsz = block_size(p, kb);
    const int64_t c = channel_of(row, p.C), g = row / p.Cg;
    const float2 ab = __ldcg(coef + g);
    const DxCoef k{mean[g], rstd[g], ab.x, ab.y, p.M == 1};
    const float gm = gamma ? gamma[c] : 1.f;
    for (int ui = bsz - 1 - own.share; ui >= 0; ui -= Own::kSplit) {
      const URange q = urange<kFull>(p, row, kb * kBlockUnits + ui);
      const int nv = (int)((q.b1 - q.b0) / kVec);
      if constexpr (kRelu) {
        bwd_norm<kFull, T>(MemView<T, FromGlobal>{x + q.b0, nv}, GatedView<T, FromGlobal>{dy + q.b0, res + q.b0, nv},
                           x, dy, dx, q, k, gm, res);
      } else {
        bwd_norm<kFull, T>(MemView<T, FromGlobal>{x + q.b0, nv}, MemView<T, FromGlobal>{dy + q.b0, nv}, x, dy,
                           dx, q, k, gm);
      }
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
