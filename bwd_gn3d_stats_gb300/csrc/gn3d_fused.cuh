// gn3d_fused.cuh -- persistent, warp-specialized forward and backward kernels.
//
// One CTA per SM: kConsumerWarps consumer warps and one producer warp.  CTA p
// owns the merge blocks b = p (mod the grid) -- each block is up to 16
// consecutive units of one row -- and walks them in group order as a sequence
// of unit tasks:
//   STAT(g): statistics of the CTA's units of group g.  A unit's partial goes to
//            a block record in shared memory; the warp that completes the block
//            merges it there, publishes the block partial and arrives on the
//            group; the warp that completes the group merges and publishes it
//            with a release store on the group's ready flag.
//   NORM(g): the elementwise pass over the same units (y or dx), in reverse
//            order, once group g is ready.
// Order, with a lag of L groups: STAT(0) .. STAT(L-1), then STAT(L) NORM(0)
// STAT(L+1) NORM(1) ..., then the last L NORMs.  The wait for a group's
// statistics hides behind the next L groups' statistics passes while L+1
// groups stay resident in L2 for their second read.  Task i goes to consumer
// warp i mod kConsumerWarps.
//
// The producer warp moves each task's unit body global -> shared memory with a
// 1-D bulk copy (the TMA engine) into slot i mod nslots, on that slot's "full"
// mbarrier (lane l of the producer warp serves slot l); the consumer warp
// releases the slot on its "empty" mbarrier.  The
// consumers never synchronize as a block: each unit is one warp's work, with
// warp shuffles only, and only one global arrival is made per 16 units.  (The
// ScaFFold GroupNorm kernels are split-group Triton programs; this is that
// split-group reduction re-cut for sm_103a.)  Both launch forms use the same
// units, merge blocks and arithmetic, so their results are bit-identical.
//
// Deadlock freedom: all CTAs are co-resident (cooperative launch).  A STAT(h)
// task precedes every NORM(h) task in each CTA's sequence and waits only for
// its own bulk copy, whose slot is released by an earlier task; so the lowest
// group anyone waits for always completes.  Every wait is still bounded: on
// timeout the CTA records GN3D_ERR_TIMEOUT, raises the abort word (which the
// other CTAs' waits watch), drains its own bulk copies and returns.
#pragma once
#include "gn3d_device.cuh"
#include "gn3d_sync.cuh"

namespace gn3d {

constexpr int kMaxSlots = 32;  // one producer lane per slot
constexpr uint32_t kStatusTimeout = 4;  // GN3D_ERR_TIMEOUT
constexpr int kMaxLag = 8;

struct FusedCfg {
  int slots;                // shared-memory slots (>= 1)
  int recs;                 // block records (> slots: see record reuse below)
  int lag;                  // groups of lookahead between the two passes (0 .. kMaxLag)
  int force_timeout;        // testing hook: the first group wait targets a word nothing sets
  unsigned long long spin;  // poll budget of every bounded wait
};

struct FusedSync {
  uint32_t* abort;   // [1] raised by a CTA that gave up waiting
  uint32_t* never;   // [1] stays 0
  uint32_t* status;  // device status word (GN3D_ERR_TIMEOUT on a timeout)
};

// Shared-memory record of one block in its STAT phase: the unit partials, an
// arrival count, and the sequence number of the CTA's STAT block allowed to
// use it next.  Records are reused round-robin over the CTA's STAT blocks
// (block j uses record j mod recs); a warp writes into a record only once the
// previous block there has been merged (next == j), which in practice it always
// has -- recs exceeds the slots, so block j + recs starts long after block j.
template <class PartT>
struct BlockRec {
  PartT part[kBlockUnits];
  int cnt;
  long long next;
};

// ------------------------------------------------------------ scheduling
struct Sched {
  int64_t P, pid, NG, nbg, nb, R;  // nbg = merge blocks per group
  const Plan* plan;
  int lag;

  __device__ __forceinline__ int64_t first(int64_t g) const {
    const int64_t base = g * nbg;
    int64_t off = (pid - base % P) % P;
    if (off < 0) off += P;
    return base + off;
  }
  __device__ __forceinline__ int64_t count_from(int64_t g, int64_t b0) const {
    const int64_t end = (g + 1) * nbg;
    return b0 < end ? (end - 1 - b0) / P + 1 : 0;
  }
  // Phase k (0 <= k < 2*NG) -> (kind, group), with L = min(lag, NG):
  //   STAT(0) .. STAT(L-1), then STAT(L) NORM(0) STAT(L+1) NORM(1) ..., then the
  //   last L NORMs.  NORM(h) always follows STAT(h') for every h' <= h + L.
  __device__ __forceinline__ bool phase(int64_t k, int& kind, int64_t& g) const {
    const int64_t L = lag < NG ? lag : NG;
    if (k < L) {
      kind = kStatPhase;
      g = k;
    } else if (k >= 2 * NG - L) {
      kind = kNormPhase;
      g = k - NG;
    } else {
      const int64_t m = k - L;
      kind = (m & 1) ? kNormPhase : kStatPhase;
      g = (m & 1) ? (m - 1) >> 1 : L + (m >> 1);
    }
    return true;
  }
  __device__ __forceinline__ int64_t last_phase() const { return 2 * NG - 1; }
  static constexpr int kStatPhase = 0, kNormPhase = 1;
};

enum { kStat = 0, kNorm = 1, kEnd = 2 };

// Position in the task sequence: a few divisions per block, only additions per unit.
struct TaskIt {
  int64_t k;
  int kind;
  int64_t g;
  int64_t fb, nblk, bi;  // phase: first block, block count, block index
  int64_t b, row, kb;    // current block
  int bsz, ui;           // its unit count; units done in it
  int64_t kr;            // current unit within its row
  int64_t sblk;          // STAT blocks finished before this one (record sequence)

  __device__ __forceinline__ void set_block(const Sched& s) {
    const int64_t j = kind == kStat ? bi : nblk - 1 - bi;
    b = fb + j * s.P;
    row = b / s.nb;
    kb = b - row * s.nb;
    bsz = block_size(*s.plan, kb);
    ui = 0;
    kr = kb * kBlockUnits + (kind == kStat ? 0 : bsz - 1);
  }
  __device__ __forceinline__ void seek(const Sched& s) {
    for (;; ++k) {
      if (k > s.last_phase()) { kind = kEnd; return; }
      int kd;
      int64_t gg;
      if (!s.phase(k, kd, gg)) continue;
      const int64_t f = s.first(gg);
      const int64_t c = s.count_from(gg, f);
      if (c > 0) {
        kind = kd; g = gg; fb = f; nblk = c; bi = 0;
        set_block(s);
        return;
      }
    }
  }
  __device__ __forceinline__ void start(const Sched& s) { k = 0; sblk = 0; seek(s); }
  __device__ __forceinline__ void next(const Sched& s) {
    if (++ui < bsz) { kr += kind == kStat ? 1 : -1; return; }
    if (kind == kStat) ++sblk;
    if (++bi < nblk) { set_block(s); return; }
    ++k;
    seek(s);
  }
  // n steps of next(), skipping whole blocks at a time.
  __device__ __forceinline__ void advance(const Sched& s, int n) {
    while (n > 0 && kind != kEnd) {
      const int rest = bsz - ui;  // units left in this block, the current one included
      if (n < rest) {
        ui += n;
        kr += kind == kStat ? n : -n;
        return;
      }
      n -= rest;
      ui = bsz - 1;
      next(s);  // leaves the block
    }
  }
};

// Bounded wait for a group's ready flag (one lane); watches the abort word.
__device__ __forceinline__ bool wait_ready(const uint32_t* flag, const FusedSync& fs, unsigned long long spin) {
  unsigned long long it = 0;
  while (ld_acquire(flag) == 0) {
    if (ld_relaxed(fs.abort) != 0) return false;
    if (++it > spin) return false;
    __nanosleep(32);
  }
  return true;
}

// Bounded wait until a slot carries the given task tag (all lanes poll).
__device__ __forceinline__ bool wait_tag(const volatile unsigned long long* tag, unsigned long long want,
                                         unsigned long long spin, const volatile int* stop) {
  for (unsigned long long it = 0; it < spin; ++it) {
    if (*tag == want) return true;
    if (*stop) return false;
    __nanosleep(20);
  }
  return false;
}

// ------------------------------------------------------------- the kernel
// Op supplies the direction-specific parts:
//   Elem, PartT, kTensors       element type; unit partial type; tensors per slot
//   kWarps                      consumer warps (the producer warp comes after them)
//   kEarly, Held                Held is what a warp keeps of a unit: its body in
//                               registers (kEarly: the slot is released as soon as
//                               the registers are loaded) or a view of the slot
//   src(t)                      base pointer of tensor t (0: x, 1: dy)
//   ready(g)                    the group's ready flag
//   hold(h, slot, q)            take the unit from its slot
//   unit(h, q)                  the unit's partial (one warp)
//   block_done(blk, a)          a completed block, lane l holding unit l's partial
//   prepare(g)                  load group g's published statistics (one warp)
//   norm(h, q, row)             NORM of one unit (one warp)
template <class Op>
__device__ __forceinline__ void run_fused(Op& op, const Plan& p, const FusedCfg& cfg, const FusedSync& fs) {
  extern __shared__ __align__(128) unsigned char smem[];
  using T = typename Op::Elem;
  using PartT = typename Op::PartT;
  constexpr int kConsumerWarps = Op::kWarps;
  constexpr int kTensorBytes = kUnitElems * (int)sizeof(T);
  constexpr int kSlotBytes = Op::kTensors * kTensorBytes;
  const int nslots = cfg.slots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)nslots * kSlotBytes);
  uint64_t* empty = full + nslots;
  BlockRec<PartT>* recs = reinterpret_cast<BlockRec<PartT>*>(empty + nslots);
  __shared__ volatile int s_fail;
  __shared__ uint32_t s_issued[kMaxSlots];  // bulk copies issued per slot (producer)
  // Task loaded (or being loaded) into each slot, plus one.  Several consumer
  // warps share a slot's mbarrier; a warp first waits until its own task is the
  // slot's current one -- which implies the previous round has completed -- so
  // its parity wait cannot be satisfied by an older phase of the same parity.
  __shared__ volatile unsigned long long s_tag[kMaxSlots];

  Sched s;
  s.P = gridDim.x;
  s.pid = blockIdx.x;
  s.NG = p.NG;
  s.nbg = p.Cg * p.nb;
  s.nb = p.nb;
  s.R = p.R;
  s.plan = &p;
  s.lag = cfg.lag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nslots; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      s_issued[i] = 0;
      s_tag[i] = 0;
    }
    fence_mbar_init();
    s_fail = 0;
  }
  for (int i = threadIdx.x; i < cfg.recs; i += blockDim.x) {
    recs[i].cnt = 0;
    recs[i].next = i;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer
    // Lane l owns slot l: it loads tasks l, l + nslots, l + 2*nslots, ... each
    // once the slot's previous task has been released, so the lanes issue their
    // bulk copies independently of one another.
    if (lane < nslots) {
      const int slot = lane;
      TaskIt it;
      it.start(s);
      it.advance(s, slot);
      for (uint64_t round = 0; it.kind != kEnd; ++round) {
        if (round > 0 && !mbar_wait(&empty[slot], (uint32_t)((round - 1) & 1u), cfg.spin, &s_fail)) {
          s_fail = 1;
          break;
        }
        if (s_fail) break;  // a consumer warp gave up (only shared memory is polled here)
        const URange q = unit_range_rk(p, it.row, it.kr);
        const uint32_t bytes = (uint32_t)((q.b1 - q.b0) * (int64_t)sizeof(T));
        unsigned char* dst = smem + (size_t)slot * kSlotBytes;
        fence_proxy_async_smem();
        s_tag[slot] = round * (uint64_t)nslots + (uint64_t)slot + 1;
        mbar_arrive_expect_tx(&full[slot], bytes * Op::kTensors);
        if (bytes) {
#pragma unroll
          for (int tn = 0; tn < Op::kTensors; ++tn)
            bulk_g2s(dst + tn * kTensorBytes, op.src(tn) + q.b0, bytes, &full[slot]);
        }
        s_issued[slot] = (uint32_t)round + 1;
        it.advance(s, nslots);
      }
    }
  } else {
    // --------------------------------------------------------- consumers
    TaskIt it;
    it.start(s);
    it.advance(s, warp);
    int64_t norm_group = -1;
    bool forced = cfg.force_timeout != 0;
    for (uint64_t i = warp; it.kind != kEnd; i += kConsumerWarps) {
      const int slot = (int)(i % (uint64_t)nslots);
      const uint64_t round = i / (uint64_t)nslots;
      const URange q = unit_range_rk(p, it.row, it.kr);
      if (it.kind == kNorm && it.g != norm_group) {
        int ok = 1;
        if (lane == 0) ok = wait_ready(forced ? fs.never : op.ready(it.g), fs, cfg.spin) ? 1 : 0;
        ok = __shfl_sync(kFull, ok, 0);
        forced = false;
        if (!ok) {
          s_fail = 1;
          break;
        }
        __syncwarp();
        op.prepare(it.g);
        norm_group = it.g;
      }
      if (!wait_tag(&s_tag[slot], i + 1, cfg.spin, &s_fail) ||
          !mbar_wait(&full[slot], (uint32_t)(round & 1u), cfg.spin, &s_fail)) {
        s_fail = 1;
        break;
      }
      const unsigned char* data = smem + (size_t)slot * kSlotBytes;
      typename Op::Held h;
      op.hold(h, data, q);
      if (Op::kEarly) {  // the unit is in registers: hand the slot back before computing
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      if (it.kind == kStat) {
        const PartT v = op.unit(h, q);
        BlockRec<PartT>& rec = recs[it.sblk % cfg.recs];
        int last = 0, ok = 1;
        if (lane == 0) {
          // the record's previous block must have been merged (bounded wait)
          const volatile long long* next = &rec.next;
          for (unsigned long long w = 0; *next != it.sblk; ++w)
            if (w > cfg.spin || s_fail) { ok = 0; break; }
          if (ok) {
            rec.part[it.kr - it.kb * kBlockUnits] = v;
            __threadfence_block();  // the partial before the arrival
            last = atomicAdd(&rec.cnt, 1) == it.bsz - 1;
            if (last) __threadfence_block();  // the other warps' partials after it
          }
        }
        __syncwarp();
        if (!__shfl_sync(kFull, ok, 0)) {
          s_fail = 1;
          break;
        }
        last = __shfl_sync(kFull, last, 0);
        if (last) {
          const PartT a = lane < it.bsz ? rec.part[lane] : PartT{};
          __syncwarp();
          if (lane == 0) {
            rec.cnt = 0;
            __threadfence_block();
            *(volatile long long*)&rec.next = it.sblk + cfg.recs;  // the record is free
          }
          op.block_done(it.b, a);
        }
      } else {
        op.norm(h, q, it.row);
      }
      if (!Op::kEarly) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
      }
      it.advance(s, kConsumerWarps);
    }
  }

  __syncthreads();
  if (s_fail && threadIdx.x == 0) {
    atomicExch(fs.status, kStatusTimeout);
    atomicExch(fs.abort, 1u);
    // drain this CTA's bulk copies in flight: wait for the last issued phase of every slot
    const volatile int no_stop = 0;
    for (int i = 0; i < nslots; ++i)
      if (s_issued[i] > 0) mbar_wait(&full[i], (s_issued[i] - 1) & 1u, kDrainPolls, &no_stop);
  }
}

// ------------------------------------------------------------- forward op
// bf16 units (8 KB) are loaded into registers and their slot released at once,
// with 11 consumer warps; fp32 units stay in their slot, with 7.  With the
// producer warp the CTA is 12 or 8 warps, so every thread keeps 168 or 255
// registers (register files are allocated in 4-warp steps).
template <class T> struct FwdPolicy {
  static constexpr bool kEarly = Vec<T>::kRaw == 1;
  static constexpr int kWarps = kEarly ? 11 : 7;
};

template <class TI, class TO>
struct FwdOp {
  using Elem = TI;
  using PartT = Part;
  static constexpr int kTensors = 1;
  static constexpr int kWarps = FwdPolicy<TI>::kWarps;
  static constexpr bool kEarly = FwdPolicy<TI>::kEarly;
  struct Held {
    RegView<TI> r;                 // kEarly
    MemView<TI, FromShared> m;     // otherwise
  };
  const TI* x;
  TO* y;
  Plan p;
  FwdWs ws;
  float eps;
  const float* gamma;
  const float* beta;
  float* mean_out;
  float* rstd_out;
  float4 st;

  __device__ __forceinline__ const TI* src(int) const { return x; }
  __device__ __forceinline__ const uint32_t* ready(int64_t g) const { return ws.ready + g; }
  __device__ __forceinline__ void hold(Held& h, const unsigned char* slot, const URange& q) const {
    const int nv = (int)((q.b1 - q.b0) / kVec);
    if (kEarly) h.r.template load<FromShared>(reinterpret_cast<const TI*>(slot), nv);
    else h.m = MemView<TI, FromShared>{reinterpret_cast<const TI*>(slot), nv};
  }
  __device__ __forceinline__ Part unit(const Held& h, const URange& q) const {
    return kEarly ? unit_moments<false, TI>(h.r, x, q) : unit_moments<false, TI>(h.m, x, q);
  }
  __device__ __forceinline__ void block_done(int64_t blk, const Part& a) {
    fwd_block_done(p, ws, blk, merge_block(a), eps, mean_out, rstd_out);
  }
  __device__ __forceinline__ void prepare(int64_t g) { st = __ldcg(ws.stats + g); }
  __device__ __forceinline__ void norm(const Held& h, const URange& q, int64_t row) {
    const int64_t c = channel_of(row, p.C);
    const float gm = gamma ? gamma[c] : 1.f, bt = beta ? beta[c] : 0.f;
    if (kEarly) fwd_norm<false, TI, TO>(h.r, x, y, q, st, gm, bt);
    else fwd_norm<false, TI, TO>(h.m, x, y, q, st, gm, bt);
  }
};

template <class TI, class TO>
__global__ void __launch_bounds__(32 * (FwdPolicy<TI>::kWarps + 1), 1)
    k_fwd_fused(const TI* __restrict__ x, TO* __restrict__ y, Plan p, FwdWs ws, FusedCfg cfg, FusedSync fs,
                float eps, const float* __restrict__ gamma, const float* __restrict__ beta, float* mean_out,
                float* rstd_out) {
  FwdOp<TI, TO> op{x, y, p, ws, eps, gamma, beta, mean_out, rstd_out, make_float4(0.f, 0.f, 0.f, 0.f)};
  run_fused(op, p, cfg, fs);
}

// ------------------------------------------------------------ backward op
// bf16 units (x and dy, 16 KB) go to registers (128 per lane) and release their
// slot at once, with 7 consumer warps (8 with the producer: 255 registers per
// thread); fp32 units stay in their slot.
template <class T> struct BwdPolicy {
  static constexpr bool kEarly = Vec<T>::kRaw == 1;
  static constexpr int kWarps = 7;
};

template <class T>
struct BwdOp {
  using Elem = T;
  using PartT = float2;
  static constexpr int kTensors = 2;  // slot: x body, then dy body
  static constexpr int kWarps = BwdPolicy<T>::kWarps;
  static constexpr bool kEarly = BwdPolicy<T>::kEarly;
  struct Held {
    RegView<T> rx, rd;                // kEarly
    MemView<T, FromShared> mx, md;    // otherwise
  };
  const T* dy;
  const T* x;
  T* dx;
  Plan p;
  const float* mean;
  const float* rstd;
  const float* gamma;
  BwdWs ws;
  float* dgamma;
  float* dbeta;
  DxCoef k;

  __device__ __forceinline__ const T* src(int t) const { return t == 0 ? x : dy; }
  __device__ __forceinline__ const uint32_t* ready(int64_t g) const { return ws.ready + g; }
  __device__ __forceinline__ void hold(Held& h, const unsigned char* slot, const URange& q) const {
    const T* xb = reinterpret_cast<const T*>(slot);
    const int nv = (int)((q.b1 - q.b0) / kVec);
    if (kEarly) {
      h.rx.template load<FromShared>(xb, nv);
      h.rd.template load<FromShared>(xb + kUnitElems, nv);
    } else {
      h.mx = MemView<T, FromShared>{xb, nv};
      h.md = MemView<T, FromShared>{xb + kUnitElems, nv};
    }
  }
  __device__ __forceinline__ float2 unit(const Held& h, const URange& q) const {
    const float mu = mean[q.row / p.Cg];
    return kEarly ? unit_bwd_sums<false, T>(h.rx, h.rd, x, dy, q, mu)
                  : unit_bwd_sums<false, T>(h.mx, h.md, x, dy, q, mu);
  }
  __device__ __forceinline__ void block_done(int64_t blk, const float2& a) {
    bwd_block_done(p, ws, blk, a, rstd, gamma, dgamma, dbeta);
  }
  __device__ __forceinline__ void prepare(int64_t g) {
    const float2 ab = __ldcg(ws.coef + g);
    k = DxCoef{mean[g], rstd[g], ab.x, ab.y, p.M == 1};
  }
  __device__ __forceinline__ void norm(const Held& h, const URange& q, int64_t row) {
    const int64_t c = channel_of(row, p.C);
    const float gm = gamma ? gamma[c] : 1.f;
    if (kEarly) bwd_norm<false, T>(h.rx, h.rd, x, dy, dx, q, k, gm);
    else bwd_norm<false, T>(h.mx, h.md, x, dy, dx, q, k, gm);
  }
};

template <class T>
__global__ void __launch_bounds__(32 * (BwdPolicy<T>::kWarps + 1), 1)
    k_bwd_fused(const T* __restrict__ dy, const T* __restrict__ x, T* __restrict__ dx, Plan p,
                const float* __restrict__ mean, const float* __restrict__ rstd, const float* __restrict__ gamma,
                BwdWs ws, FusedCfg cfg, FusedSync fs, float* dgamma, float* dbeta) {
  BwdOp<T> op{dy, x, dx, p, mean, rstd, gamma, ws, dgamma, dbeta, DxCoef{0.f, 0.f, 0.f, 0.f, false}};
  run_fused(op, p, cfg, fs);
}

}  // namespace gn3d
