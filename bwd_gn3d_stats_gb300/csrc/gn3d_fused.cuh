// gn3d_fused.cuh -- persistent, cooperative forward and backward kernels.
//
// One CTA per SM walks the units of the plan (the same units, thread mapping
// and reduction trees as the streaming kernels, so results are bit-identical)
// in group order, as a sequence of tasks:
//   STAT(g): the statistics pass over this CTA's units of group g (forward:
//            unit moments; backward: S1 = sum dy, S2 = sum dy*(x - mean)); the
//            CTA that completes a group merges its partials, publishes the
//            group's statistics and raises the group's ready flag.
//   NORM(g): the elementwise pass over the same units (forward: y; backward:
//            dx), in reverse order, once group g is ready.
// The order is STAT(0) STAT(1) NORM(0) STAT(2) NORM(1) ... (lag 1: the wait for
// a group's statistics hides behind the next group's statistics pass, and two
// groups stay resident in L2), or STAT(0) NORM(0) STAT(1) NORM(1) ... (lag 0,
// for groups too large for two to fit in L2).
//
// Unit bodies move global -> shared memory with 1-D bulk copies (the TMA engine)
// on per-slot mbarriers, issued ahead by thread 0 into
//   * a FIFO ring of stream slots (units read once per pass), and
//   * two stash areas (even/odd groups) that keep the last units of a group
//     from its STAT task to its NORM task, so those are not read twice.
// The ScaFFold GroupNorm kernels are split-group Triton programs; this is the
// same split-group reduction re-cut for sm_103a: persistent CTAs, TMA staging,
// and group-ordered passes so the second read of a group hits shared memory
// or L2 instead of HBM.
//
// Deadlock freedom: all CTAs are co-resident (cooperative launch).  A CTA waits
// for group h only in NORM(h), after its STAT(h') for every h' <= h + lag, so
// the lowest group anyone waits for has all its STAT work done or in progress.
// Every wait is still bounded: on timeout the CTA records GN3D_ERR_TIMEOUT,
// raises the abort word (which the other CTAs' waits also watch), drains its
// own bulk copies and returns.
#pragma once
#include "gn3d_kernels.cuh"
#include "gn3d_sync.cuh"

namespace gn3d {

constexpr int kMaxSlots = 30;
constexpr int kFusedCtasPerSm = 2;
constexpr uint32_t kStatusTimeout = 4;  // GN3D_ERR_TIMEOUT

struct FusedCfg {
  int ring;            // stream slots (>= 1)
  int stash;           // stash slots per group parity (>= 0)
  int lag;             // 0 or 1
  int force_timeout;   // testing hook: the first group wait targets a word nothing sets
  unsigned long long spin;  // poll budget of every bounded wait
};

struct FusedSync {
  uint32_t* cnt;       // [NG + 1] STAT arrivals per group (+ groups finalized, backward)
  uint32_t* ready;     // [NG] 1 once the group's statistics are published
  uint32_t* abort;     // [1] raised by a CTA that gave up waiting
  uint32_t* never;     // [1] stays 0
  uint32_t* status;    // device status word (GN3D_ERR_TIMEOUT on a timeout)
};

// ------------------------------------------------------------ scheduling
// CTA pid of P owns the units u = pid (mod P); inside group g these are
// first(g), first(g) + P, ...  Phases: STAT(g) in increasing unit order, NORM(g)
// in decreasing order; the stashed units are the last `stash` of each group.
struct Sched {
  int64_t P, pid, NG, upg, R;
  int64_t qP, rP;  // P / R and P % R: stepping u by P moves (row, k) by these
  int stash, lag;

  __device__ __forceinline__ int64_t first(int64_t g) const {
    const int64_t base = g * upg;
    int64_t off = (pid - base % P) % P;
    if (off < 0) off += P;
    return base + off;
  }
  __device__ __forceinline__ int64_t count_from(int64_t g, int64_t u0) const {
    const int64_t end = (g + 1) * upg;
    return u0 < end ? (end - 1 - u0) / P + 1 : 0;
  }
  // phase k -> (kind, group); false when k names no phase (STAT beyond the last group)
  __device__ __forceinline__ bool phase(int64_t k, int& kind, int64_t& g) const {
    if (lag == 0) {
      kind = (int)(k & 1);
      g = k >> 1;
    } else if (k == 0) {
      kind = 0;
      g = 0;
    } else {
      const int64_t m = k - 1;
      kind = (m & 1) ? 1 : 0;
      g = (m & 1) ? (m >> 1) : (m >> 1) + 1;
    }
    return g < NG;
  }
  __device__ __forceinline__ int64_t last_phase() const { return lag == 0 ? 2 * NG - 1 : 2 * NG; }
  __device__ __forceinline__ int64_t norm_phase(int64_t g) const { return lag == 0 ? 2 * g + 1 : 2 * g + 2; }
};

enum { kStat = 0, kNorm = 1, kEnd = 2 };

struct Task {
  int kind;
  int64_t g, u, row, kr;
  bool stashed, last_in_phase;
  int sidx;  // stash slot within the group's parity area
};

// Position in the task sequence.  Per phase it costs a few divisions; per task
// it only adds or subtracts, so thread 0 can run it ahead cheaply.
struct TaskIt {
  int64_t k, idx, n, ns, u0;
  int kind;
  int64_t g;
  int64_t u, row, kr;

  __device__ __forceinline__ void seek(const Sched& s) {
    for (;; ++k) {
      if (k > s.last_phase()) { kind = kEnd; return; }
      int kd;
      int64_t gg;
      if (!s.phase(k, kd, gg)) continue;
      const int64_t f = s.first(gg);
      const int64_t c = s.count_from(gg, f);
      if (c > 0) {
        kind = kd; g = gg; n = c; idx = 0; u0 = f;
        ns = c < s.stash ? c : s.stash;
        u = kind == kStat ? f : f + (c - 1) * s.P;
        row = u / s.R;
        kr = u - row * s.R;
        return;
      }
    }
  }
  __device__ __forceinline__ void start(const Sched& s) { k = 0; seek(s); }
  __device__ __forceinline__ void next(const Sched& s) {
    if (++idx >= n) { ++k; seek(s); return; }
    if (kind == kStat) {
      u += s.P; row += s.qP; kr += s.rP;
      if (kr >= s.R) { kr -= s.R; ++row; }
    } else {
      u -= s.P; row -= s.qP; kr -= s.rP;
      if (kr < 0) { kr += s.R; --row; }
    }
  }
  __device__ __forceinline__ Task cur() const {
    Task t;
    t.kind = kind;
    t.g = g;
    t.u = u;
    t.row = row;
    t.kr = kr;
    const int64_t j = kind == kStat ? idx : n - 1 - idx;
    t.stashed = j >= n - ns;
    t.sidx = (int)(j - (n - ns));
    t.last_in_phase = idx == n - 1;
    return t;
  }
};

// Shared-memory slot layout: [ring stream slots][stash even][stash odd]
__device__ __forceinline__ int stash_slot(const FusedCfg& c, int64_t g, int sidx) {
  return c.ring + (int)(g & 1) * c.stash + sidx;
}

// Bounded wait for a group's ready flag (thread 0); watches the abort word.
__device__ __forceinline__ bool wait_ready(const uint32_t* flag, const FusedSync& fs, unsigned long long spin) {
  unsigned long long it = 0;
  while (ld_acquire(flag) == 0) {
    if (ld_relaxed(fs.abort) != 0) return false;
    if (++it > spin) return false;
    __nanosleep(32);
  }
  return true;
}

// Row -> channel, in 32 bits when the row index allows it.
__device__ __forceinline__ int64_t channel_of(int64_t row, int64_t C) {
  if (row < 0x7FFFFFFF && C < 0x7FFFFFFF) return (int64_t)((uint32_t)row % (uint32_t)C);
  return row % C;
}

// ------------------------------------------------------------- the kernel
// Op supplies the direction-specific parts:
//   kTensors                          tensors per unit in a slot (1: x; 2: x then dy)
//   src(t)                            base pointer of tensor t
//   stat(slot, q, u, g, arrive, n)    statistics of one unit (all threads); when
//                                     `arrive`, also the CTA's arrival for group g
//                                     with its n units (and the group finalize if last)
//   prepare(g)                        load group g's published statistics (all threads)
//   norm(slot, q)                     elementwise pass of one unit (all threads)
template <class Op>
__device__ __forceinline__ void run_fused(Op& op, const Plan& p, const FusedCfg& cfg, const FusedSync& fs) {
  extern __shared__ __align__(128) unsigned char smem[];
  using T = typename Op::Elem;
  constexpr int kSlotBytes = Op::kTensors * kUnitElems * (int)sizeof(T);
  const int nslots = cfg.ring + 2 * cfg.stash;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)nslots * kSlotBytes);
  __shared__ int s_fail;
  __shared__ uint32_t s_issued[kMaxSlots];  // loads issued per slot (thread 0)

  Sched s;
  s.P = gridDim.x;
  s.pid = blockIdx.x;
  s.NG = p.NG;
  s.upg = p.upg;
  s.R = p.R;
  s.qP = s.P / s.R;
  s.rP = s.P - s.qP * s.R;
  s.stash = cfg.stash;
  s.lag = cfg.lag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nslots; ++i) {
      mbar_init(&bars[i], 1);
      s_issued[i] = 0;
    }
    fence_mbar_init();
    s_fail = 0;
  }
  __syncthreads();

  TaskIt ct;  // consumer position (all threads, identical)
  ct.start(s);
  TaskIt pt = ct;  // producer position (thread 0)
  uint64_t lc = 0;      // stream loads consumed (all threads)
  uint64_t lp = 0;      // stream loads issued (thread 0)
  uint32_t stash_par = 0;  // parity bit per stash slot, consumer side (all threads)
  int64_t norm_group = -1;
  bool forced = cfg.force_timeout != 0;

  while (ct.kind != kEnd) {
    // ---- producer: issue bulk copies ahead while their slots are free
    if (threadIdx.x == 0) {
      while (pt.kind != kEnd) {
        const Task t = pt.cur();
        int slot;
        if (t.stashed) {
          if (t.kind == kNorm) { pt.next(s); continue; }     // data stays from STAT
          if (t.g >= 2 && ct.k <= s.norm_phase(t.g - 2)) break;  // stash area still in use
          slot = stash_slot(cfg, t.g, t.sidx);
        } else {
          if (lp >= lc + (uint64_t)cfg.ring) break;          // ring full
          slot = (int)(lp % (uint64_t)cfg.ring);
        }
        const URange q = unit_range_rk(p, t.row, t.kr);
        const uint32_t bytes = (uint32_t)((q.b1 - q.b0) * (int64_t)sizeof(T));
        unsigned char* dst = smem + (size_t)slot * kSlotBytes;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[slot], bytes * Op::kTensors);
        if (bytes) {
#pragma unroll
          for (int tn = 0; tn < Op::kTensors; ++tn)
            bulk_g2s(dst + tn * kUnitElems * sizeof(T), op.src(tn) + q.b0, bytes, &bars[slot]);
        }
        ++s_issued[slot];
        if (!t.stashed) ++lp;
        pt.next(s);
      }
    }

    // ---- consumer
    const Task t = ct.cur();
    const URange q = unit_range_rk(p, t.row, t.kr);
    if (t.kind == kNorm && t.g != norm_group) {
      if (threadIdx.x == 0) {
        const uint32_t* flag = forced ? fs.never : fs.ready + t.g;
        if (!wait_ready(flag, fs, cfg.spin)) s_fail = 1;
      }
      forced = false;
      __syncthreads();
      if (s_fail) break;
      op.prepare(t.g);
      norm_group = t.g;
    }
    int slot;
    bool waited = false;
    if (t.stashed) {
      slot = stash_slot(cfg, t.g, t.sidx);
      if (t.kind == kStat) {
        waited = true;
        if (!mbar_wait(&bars[slot], (stash_par >> (slot - cfg.ring)) & 1u, cfg.spin)) s_fail = 1;
      }
    } else {
      slot = (int)(lc % (uint64_t)cfg.ring);
      waited = true;
      if (!mbar_wait(&bars[slot], (uint32_t)((lc / (uint64_t)cfg.ring) & 1u), cfg.spin)) s_fail = 1;
    }
    if (waited) {
      __syncthreads();
      if (s_fail) break;
    }
    const unsigned char* data = smem + (size_t)slot * kSlotBytes;
    if (t.kind == kStat) op.stat(data, q, t.u, t.g, t.last_in_phase, ct.n);
    else op.norm(data, q, channel_of(t.row, p.C));
    __syncthreads();  // every thread is done with the slot
    if (!t.stashed) ++lc;
    else if (t.kind == kStat) stash_par ^= 1u << (slot - cfg.ring);
    ct.next(s);
  }

  if (s_fail) {
    if (threadIdx.x == 0) {
      atomicExch(fs.status, kStatusTimeout);
      atomicExch(fs.abort, 1u);
      // drain this CTA's bulk copies in flight: wait for the last issued phase of every slot
      for (int i = 0; i < nslots; ++i)
        if (s_issued[i] > 0) mbar_wait(&bars[i], (s_issued[i] - 1) & 1u, cfg.spin);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------- forward op
template <class TI, class TO>
struct FwdOp {
  using Elem = TI;
  static constexpr int kTensors = 1;
  const TI* x;
  TO* y;
  Plan p;
  FwdWs ws;
  float eps;
  const float* gamma;
  const float* beta;
  float* mean_out;
  float* rstd_out;
  FusedSync fs;
  float2* red;
  double2* msh;
  int* s_last;
  float4 st;

  __device__ __forceinline__ const TI* src(int) const { return x; }

  __device__ __forceinline__ void load_regs(const unsigned char* slot, const URange& q, UnitRegs<TI>& r) const {
    const TI* sp = reinterpret_cast<const TI*>(slot);
    const int64_t nv = (q.b1 - q.b0) / kVec;
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int64_t j = threadIdx.x + (int64_t)i * kThreads;
      r.vok[i] = j < nv;
      if (r.vok[i]) IO<TI>::load8(sp + j * kVec, r.v[i]);
      else {
#pragma unroll
        for (int e = 0; e < 8; ++e) r.v[i][e] = 0.f;
      }
    }
    r.sok = (int)threadIdx.x < scalar_count(q);
    r.s = r.sok ? IO<TI>::load1(x + scalar_index(q, threadIdx.x)) : 0.f;
  }

  __device__ __forceinline__ void stat(const unsigned char* slot, const URange& q, int64_t u, int64_t g,
                                      bool arrive, int64_t n) {
    UnitRegs<TI> r;
    load_regs(slot, q, r);
    const Part m = unit_moments(r, q.n, red);
    if (threadIdx.x == 0) {
      ws.parts[u] = m;
      if (arrive) {
        __threadfence();
        *s_last = atomicAdd(&fs.cnt[g], (unsigned)n) + (unsigned)n == (unsigned)p.upg;
      }
    }
    if (!arrive) return;
    __syncthreads();
    if (*s_last) {
      __threadfence();
      finalize_group(p, g, ws.parts, eps, ws.stats, mean_out, rstd_out, msh);
      if (threadIdx.x == 0) {
        __threadfence();
        st_release(fs.ready + g, 1u);
      }
    }
  }

  __device__ __forceinline__ void prepare(int64_t g) { st = __ldcg(ws.stats + g); }

  __device__ __forceinline__ void norm(const unsigned char* slot, const URange& q, int64_t c) {
    const float sc = gamma ? fmul(st.z, gamma[c]) : st.z;
    const float sh = beta ? beta[c] : 0.f;
    const TI* sp = reinterpret_cast<const TI*>(slot);
    const int64_t nv = (q.b1 - q.b0) / kVec;
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t j = threadIdx.x + (int64_t)k * kThreads;
      if (j < nv) {
        float v[8];
        IO<TI>::load8(sp + j * kVec, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = ffma(fsub(fsub(v[e], st.x), st.y), sc, sh);
        IO<TO>::store8(y + q.b0 + j * kVec, v);
      }
    }
    if ((int)threadIdx.x < scalar_count(q)) {
      const int64_t idx = scalar_index(q, threadIdx.x);
      IO<TO>::store1(y + idx, ffma(fsub(fsub(IO<TI>::load1(x + idx), st.x), st.y), sc, sh));
    }
  }
};

template <class TI, class TO>
__global__ void __launch_bounds__(kThreads, kFusedCtasPerSm)
    k_fwd_fused(const TI* __restrict__ x, TO* __restrict__ y, Plan p, FwdWs ws, FusedCfg cfg, FusedSync fs,
                float eps, const float* __restrict__ gamma, const float* __restrict__ beta, float* mean_out,
                float* rstd_out) {
  __shared__ float2 red[kWarps];
  __shared__ double2 msh[kWarps];
  __shared__ int s_last;
  FwdOp<TI, TO> op{x, y, p, ws, eps, gamma, beta, mean_out, rstd_out, fs, red, msh, &s_last,
                   make_float4(0.f, 0.f, 0.f, 0.f)};
  run_fused(op, p, cfg, fs);
}

// ------------------------------------------------------------ backward op
template <class T>
struct BwdOp {
  using Elem = T;
  static constexpr int kTensors = 2;  // slot: x body, then dy body
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
  FusedSync fs;
  float2* red;
  int* s_flags;  // [0]: last of group, [1]: last group overall
  float mu, r, a, b;

  __device__ __forceinline__ const T* src(int t) const { return t == 0 ? x : dy; }

  __device__ __forceinline__ void load_pair(const unsigned char* slot, const URange& q, UnitRegs<T>& rx,
                                            UnitRegs<T>& rd) const {
    const T* sx = reinterpret_cast<const T*>(slot);
    const T* sd = sx + kUnitElems;
    const int64_t nv = (q.b1 - q.b0) / kVec;
#pragma unroll
    for (int i = 0; i < kVecPerThread; ++i) {
      const int64_t j = threadIdx.x + (int64_t)i * kThreads;
      rx.vok[i] = rd.vok[i] = j < nv;
      if (rx.vok[i]) {
        IO<T>::load8(sx + j * kVec, rx.v[i]);
        IO<T>::load8(sd + j * kVec, rd.v[i]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) rx.v[i][e] = rd.v[i][e] = 0.f;
      }
    }
    rx.sok = rd.sok = (int)threadIdx.x < scalar_count(q);
    if (rx.sok) {
      const int64_t idx = scalar_index(q, threadIdx.x);
      rx.s = IO<T>::load1(x + idx);
      rd.s = IO<T>::load1(dy + idx);
    } else {
      rx.s = rd.s = 0.f;
    }
  }

  __device__ __forceinline__ void stat(const unsigned char* slot, const URange& q, int64_t u, int64_t g,
                                      bool arrive, int64_t n) {
    UnitRegs<T> rx, rd;
    load_pair(slot, q, rx, rd);
    const float2 sums = unit_bwd_sums(rd, rx, mean[g], red);
    if (threadIdx.x == 0) {
      ws.parts[u] = sums;
      if (arrive) {
        __threadfence();
        s_flags[0] = atomicAdd(&fs.cnt[g], (unsigned)n) + (unsigned)n == (unsigned)p.upg;
      }
    }
    if (!arrive) return;
    __syncthreads();
    if (s_flags[0]) {
      __threadfence();
      bwd_finalize_group(p, g, rstd, gamma, ws);
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        st_release(fs.ready + g, 1u);
        s_flags[1] = atomicAdd(&fs.cnt[p.NG], 1u) == (unsigned)(p.NG - 1);
      }
      __syncthreads();
      if (s_flags[1]) {
        __threadfence();
        bwd_param_grads(p, rstd, ws.rows, dgamma, dbeta);
      }
    }
  }

  __device__ __forceinline__ void prepare(int64_t g) {
    mu = mean[g];
    r = rstd[g];
    const float2 ab = __ldcg(ws.coef + g);
    a = ab.x;
    b = ab.y;
  }

  __device__ __forceinline__ void norm(const unsigned char* slot, const URange& q, int64_t c) {
    const float gm = gamma ? gamma[c] : 1.f;
    const T* sx = reinterpret_cast<const T*>(slot);
    const T* sd = sx + kUnitElems;
    const int64_t nv = (q.b1 - q.b0) / kVec;
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t j = threadIdx.x + (int64_t)k * kThreads;
      if (j < nv) {
        float vx[8], vd[8];
        IO<T>::load8(sx + j * kVec, vx);
        IO<T>::load8(sd + j * kVec, vd);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float t = fsub(fmul(vd[e], gm), a);
          const float xh = fmul(fsub(vx[e], mu), r);
          vd[e] = fmul(r, ffma(-xh, b, t));
        }
        IO<T>::store8(dx + q.b0 + j * kVec, vd);
      }
    }
    if ((int)threadIdx.x < scalar_count(q)) {
      const int64_t idx = scalar_index(q, threadIdx.x);
      const float t = fsub(fmul(IO<T>::load1(dy + idx), gm), a);
      const float xh = fmul(fsub(IO<T>::load1(x + idx), mu), r);
      IO<T>::store1(dx + idx, fmul(r, ffma(-xh, b, t)));
    }
  }
};

template <class T>
__global__ void __launch_bounds__(kThreads, kFusedCtasPerSm)
    k_bwd_fused(const T* __restrict__ dy, const T* __restrict__ x, T* __restrict__ dx, Plan p,
                const float* __restrict__ mean, const float* __restrict__ rstd, const float* __restrict__ gamma,
                BwdWs ws, FusedCfg cfg, FusedSync fs, float* dgamma, float* dbeta) {
  __shared__ float2 red[kWarps];
  __shared__ int s_flags[2];
  BwdOp<T> op{dy, x, dx, p, mean, rstd, gamma, ws, dgamma, dbeta, fs, red, s_flags, 0.f, 0.f, 0.f, 0.f};
  run_fused(op, p, cfg, fs);
}

}  // namespace gn3d
