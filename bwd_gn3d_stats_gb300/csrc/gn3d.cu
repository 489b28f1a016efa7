// gn3d.cu -- libgn3d's C ABI: argument checks, the launch plan, per-call scratch
// and the kernel launches for GroupNorm forward and backward (include/gn3d.h).
//
// Four launch forms run the same units with the same arithmetic (bit-identical
// results): the streaming kernels (gn3d_kernels.cuh, two launches per
// direction); the cluster kernels (gn3d_cluster.cuh, one launch per direction,
// one thread-block cluster per group holding its units in shared memory); the
// persistent cooperative kernels (gn3d_fused.cuh); and the group-wave kernels
// (gn3d_resident.cuh, one cooperative launch per direction, each group's share
// held on chip between the two passes).  The automatic choice takes the cluster
// form where every group's cluster is resident at once and the streaming
// kernels otherwise; the testing build's gn3d_debug_set selects any form, for
// cross-checks and A/B timing.  The channels-last entry points run their own
// kernels (gn3d_ndhwc.cuh).
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/gn3d.h"
#include "gn3d_cluster.cuh"
#include "gn3d_fused.cuh"
#include "gn3d_kernels.cuh"
#include "gn3d_ndhwc.cuh"
#include "gn3d_resident.cuh"
#include "gn3d_shard.cuh"

namespace gn3d {

// Device status word: bounded waits that give up record GN3D_ERR_TIMEOUT here.
__device__ uint32_t g_status_word;

namespace {

thread_local std::string g_detail;
thread_local std::string g_msg;
std::atomic<uint64_t> g_launches{0};

// testing / tuning hooks (gn3d_debug_set)
std::atomic<long long> g_hook_path{0};  // 0 auto, 1 streaming, 2 persistent, 3 group-wave, 4 cluster
std::atomic<long long> g_hook_spin{0};     // 0 default poll budget
std::atomic<long long> g_hook_timeout{0};  // 1: the next fused launch waits on a flag nothing sets
std::atomic<long long> g_hook_lag{-1};     // -1 auto
std::atomic<long long> g_hook_slots{-1};   // -1 auto
std::atomic<int> g_hook_shares{-1};        // -1 auto, 0 strided blocks, 1 unit shares
std::atomic<long long> g_hook_rheld{-1};   // -1 auto: held units per share of the group-wave kernels
std::atomic<long long> g_hook_window{-1};  // -1 auto: the group-wave producer's lead, in units
std::atomic<long long> g_hook_rpass{-1};   // -1 auto: pass-ring slots of the group-wave kernels
#ifdef GN3D_TESTING
std::atomic<int> g_inject{0};              // 1: the next scratch allocation fails, 2: the next launch
#endif

constexpr unsigned long long kDefaultSpin = 1ull << 26;  // ~4 s of polls at 64 ns sleeps

int cuda_fail(cudaError_t e, const char* what) {
  g_detail = std::string(what) + ": " + cudaGetErrorString(e);
  return GN3D_ERR_CUDA;
}

int arg_fail(const char* what) {
  g_detail = what;
  return GN3D_ERR_INVALID_ARG;
}

#define GN3D_CUDA(call, what)                          \
  do {                                                 \
    cudaError_t e_ = (call);                           \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// Per-device facts and objects, created once.
struct DevInfo {
  bool ready = false;
  int dev = 0;
  int sms = 0;
  int l2_bytes = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
  cudaMemPool_t pool = nullptr;
  uint32_t* status = nullptr;
  std::vector<cudaEvent_t> free_events;                // timing events of this device, for reuse
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
// The dynamic shared memory each kernel's attribute was raised to, per device:
// one table for every launch path, so no path can believe an attribute is
// higher than another path left it.
std::vector<std::pair<const void*, int>> g_attr_smem[kMaxDevices];

int device_info(int dev, DevInfo** out) {
  if (dev < 0 || dev >= kMaxDevices) return arg_fail("device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.ready) {
    d.dev = dev;
    GN3D_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev), "device attribute");
    GN3D_CUDA(cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev), "device attribute");
    GN3D_CUDA(cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
              "device attribute");
    GN3D_CUDA(cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev),
              "device attribute");
    // A pool of our own for the per-call scratch: the default pool trims
    // freed memory at every synchronization, which makes the next call remap.
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    GN3D_CUDA(cudaMemPoolCreate(&d.pool, &props), "cudaMemPoolCreate");
    uint64_t keep = 64ull << 20;
    GN3D_CUDA(cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep), "pool attribute");
    void* sym = nullptr;
    GN3D_CUDA(cudaGetSymbolAddress(&sym, g_status_word), "cudaGetSymbolAddress");
    d.status = static_cast<uint32_t*>(sym);
    d.ready = true;
  }
  *out = &d;
  return GN3D_OK;
}

// A tensor argument must be device (or managed) memory of the current device.
int check_ptr(const void* p, int dev, const char* name) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    g_detail = std::string(name) + ": not a CUDA allocation";
    return GN3D_ERR_DEVICE;
  }
  if (a.type == cudaMemoryTypeManaged) return GN3D_OK;
  if (a.type == cudaMemoryTypeDevice && a.device == dev) return GN3D_OK;
  g_detail = std::string(name) + (a.type == cudaMemoryTypeDevice ? ": on another device" : ": not device memory");
  return GN3D_ERR_DEVICE;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check_shape(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int64_t G) {
  if (N < 0 || C < 0 || D < 0 || H < 0 || W < 0) return arg_fail("negative dimension");
  if (G <= 0) return arg_fail("G must be >= 1");
  if (C % G != 0) return arg_fail("C must be divisible by G");
  const double total = (double)N * (double)C * (double)D * (double)H * (double)W;
  if (total > 4.0e18) return arg_fail("tensor too large");
  if (C > 0 && N * (C / G) * D * H * W == 1)
    return arg_fail("expected more than 1 value per group (N*(C/G)*D*H*W == 1)");
  return GN3D_OK;
}

int grid_for(const DevInfo& di, int64_t units, int per_sm) {
  int64_t g = (int64_t)di.sms * per_sm;
  if (g > units) g = units;
  return (int)(g < 1 ? 1 : g);
}

// Strided blocks or unit shares for the NCDHW streaming kernels' nw warps
// (placement only).
bool unit_shares(const Plan& p, int64_t nw) {
  const int h = g_hook_shares.load();
  return h < 0 ? use_unit_shares(p, nw) : h == 1;
}

// The per-call scratch allocation, stream-ordered from the library's pool.  In
// the testing build an armed injection (GN3D_DEBUG_FAIL_NEXT) makes it fail as
// an out-of-memory would, to exercise the callers' error paths.
cudaError_t scratch_alloc(void** p, int64_t bytes, const DevInfo& di, cudaStream_t st) {
#ifdef GN3D_TESTING
  int armed = 1;
  if (g_inject.compare_exchange_strong(armed, 0)) return cudaErrorMemoryAllocation;
#endif
  return cudaMallocFromPoolAsync(p, (size_t)bytes, di.pool, st);
}

// Called before a call's first kernel launch: cudaSuccess, or (testing build,
// injection armed) the error a failed launch returns.
cudaError_t injected_launch_error() {
#ifdef GN3D_TESTING
  int armed = 2;
  if (g_inject.compare_exchange_strong(armed, 0)) return cudaErrorLaunchFailure;
#endif
  return cudaSuccess;
}

// Scratch carved out of one stream-ordered allocation, 256-byte aligned pieces.
struct Scratch {
  void* base = nullptr;
  char* cur = nullptr;
  template <class T>
  T* take(int64_t count) {
    T* p = reinterpret_cast<T*>(cur);
    cur += ((count * (int64_t)sizeof(T) + 255) / 256) * 256;
    return p;
  }
};

int64_t rup(int64_t b) { return ((b + 255) / 256) * 256; }

// ------------------------------------------------------------ kernel timing
// While timing is on (gn3d_timing), each kernel launch is bracketed by two
// CUDA events on its stream; gn3d_kernel_time resolves them per kernel.
enum {
  KK_FWD_FUSED, KK_BWD_FUSED, KK_FWD_STATS, KK_FWD_NORM, KK_BWD_REDUCE, KK_BWD_DX,
  KK_N_STATS, KK_N_STATS_FINAL, KK_N_NORM, KK_N_REDUCE, KK_N_REDUCE_FINAL, KK_N_DX, KK_FWD_RES, KK_BWD_RES,
  KK_FWD_CLUSTER, KK_BWD_CLUSTER,
  KK_COUNT
};
const char* const kKernelNames[KK_COUNT] = {
    "k_fwd_fused",   "k_bwd_fused",         "k_fwd_stats",  "k_fwd_norm",     "k_bwd_reduce",
    "k_bwd_dx",      "k_ndhwc_stats",       "k_ndhwc_stats_final", "k_ndhwc_norm", "k_ndhwc_reduce",
    "k_ndhwc_reduce_final", "k_ndhwc_dx", "k_fwd_resident", "k_bwd_resident", "k_fwd_cluster", "k_bwd_cluster"};
std::atomic<int> g_timing{0};
std::mutex g_tmu;
struct TimedLaunch {
  int kind;
  DevInfo* dev;  // owner of the events
  cudaEvent_t a, b;
};
std::vector<TimedLaunch> g_timed;
double g_kernel_ms[KK_COUNT];
uint64_t g_kernel_n[KK_COUNT];

// An event of this device: a recycled one, else a new one (timing only).
cudaEvent_t take_event(DevInfo& di) {
  {
    std::lock_guard<std::mutex> lk(g_tmu);
    if (!di.free_events.empty()) {
      cudaEvent_t e = di.free_events.back();
      di.free_events.pop_back();
      return e;
    }
  }
  cudaEvent_t e = nullptr;
  return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
}

struct LaunchTimer {
  int kind;
  cudaStream_t st;
  DevInfo& di;
  cudaEvent_t a = nullptr;
  LaunchTimer(int k, cudaStream_t s, DevInfo& d) : kind(k), st(s), di(d) {
    if (!g_timing.load()) return;
    a = take_event(di);
    if (a && cudaEventRecord(a, st) != cudaSuccess) {
      cudaEventDestroy(a);
      a = nullptr;
    }
  }
  void done() {
    if (!a) return;
    cudaEvent_t b = take_event(di);
    std::lock_guard<std::mutex> lk(g_tmu);
    if (b && cudaEventRecord(b, st) == cudaSuccess) {
      g_timed.push_back(TimedLaunch{kind, &di, a, b});
    } else {
      di.free_events.push_back(a);
      if (b) di.free_events.push_back(b);
    }
    a = nullptr;
  }
};

unsigned long long spin_budget() {
  const long long s = g_hook_spin.load();
  return s > 0 ? (unsigned long long)s : kDefaultSpin;
}

bool use_fused() { return g_hook_path.load() == 2; }

// The cluster kernels run wherever they apply, unless a testing hook picks
// another launch form (path 4 asks for them explicitly).
bool want_cluster() {
  const long long h = g_hook_path.load();
  return h == 0 || h == 4;
}

// The group-wave (resident) kernels: every unit full, enough units for every
// SM to hold a share of each group most of the time.
bool use_resident(const Plan& p, const DevInfo& di) {
  const long long h = g_hook_path.load();
  if (h == 3) return plan_all_full(p);
  if (h != 0) return false;
  return false;
}

// Ring sizes of a group-wave launch: as many slots as fit next to the piece
// records, three of them in the pass ring; held units per share: half the held
// ring (so a share of the next group loads while the current one waits for its
// statistics); the producer's lead: half of L2's share per SM.
ResCfg resident_cfg(const DevInfo& di, const Plan& p, int kred, int slot_bytes, int fixed_bytes, int* smem) {
  ResCfg c;
  const int fixed = 2048 + fixed_bytes;  // 2 KB: static shared memory and slack
  const int nslots = (di.smem_optin - fixed) / (slot_bytes + 16);
  // both rings a multiple of the reduction warps (each slot read by one warp)
  const long long hp = g_hook_rpass.load();
  int kp = hp >= 1 ? (int)hp : kred;
  kp = (kp + kred - 1) / kred * kred;
  if (kp > nslots - kred) kp = (nslots - kred) / kred * kred;
  const int kh = (nslots - kp) / kred * kred;
  int rh = kh / 2 > 0 ? kh / 2 : 1;
  const long long hr = g_hook_rheld.load(), hw = g_hook_window.load();
  if (hr >= 0 && hr <= kh) rh = (int)hr;
  c.geo = res_geo(p, di.sms, rh, kh, kp, 0);
  c.window = (long long)di.l2_bytes / 2 / di.sms / slot_bytes;
  if (c.window < nslots) c.window = nslots;
  if (hw >= 1) c.window = hw;
  // a whole share of a group must fit in the lead, else nothing could ever be normalized
  if (c.window < res_min_window(p, di.sms)) c.window = res_min_window(p, di.sms);
  c.force_timeout = g_hook_timeout.exchange(0) != 0;
  c.spin = spin_budget();
  *smem = (kh + kp) * slot_bytes + 2 * (kh + kp) * 8 + fixed_bytes;
  return c;
}

// The lead's bound from the per-CTA group counters: fewer groups in flight than
// the counters (each group in flight holds at least max(q, 1) of the lead's units).
bool resident_lead_ok(const ResCfg& c) {
  const long long per = c.geo.q > 0 ? c.geo.q : 1;
  return c.window / per + 2 < kCtrRing;
}


// Shared-memory slots of a persistent launch (one CTA per SM) and its schedule.
// Dynamic shared memory: slots, two mbarriers per slot, slots + 2 block records.
FusedCfg fused_cfg(const DevInfo& di, int slot_bytes, int rec_bytes, int64_t group_bytes) {
  FusedCfg c;
  int n = (di.smem_optin - 2048 - 2 * rec_bytes) / (slot_bytes + 16 + rec_bytes);  // 2 KB: static smem
  if (n > kMaxSlots) n = kMaxSlots;
  const long long hs = g_hook_slots.load(), hl = g_hook_lag.load();
  if (hs >= 1 && hs < n) n = (int)hs;
  c.slots = n;
  c.recs = n + 2;
  // Lag: as many groups of lookahead as leave each group's second read in L2
  // (lag + 1 groups resident, with room for the writes), at least one -- a
  // lookahead of one group beats stalling at every group boundary even when a
  // group alone outgrows L2.
  int64_t lag = group_bytes > 0 ? (int64_t)di.l2_bytes / (2 * group_bytes) - 1 : kMaxLag;
  if (lag < 1) lag = 1;
  if (lag > kMaxLag) lag = kMaxLag;
  c.lag = (int)lag;
  if (hl >= 0) c.lag = (int)hl;
  c.force_timeout = g_hook_timeout.exchange(0) != 0;
  c.spin = spin_budget();
  return c;
}

// Raise a kernel's dynamic shared memory limit to at least `bytes` on the
// device (the limit only ever goes up, so a smaller launch never lowers it
// under a larger one).
int raise_smem(const void* func, int bytes, const DevInfo& di) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& e : g_attr_smem[di.dev]) {
    if (e.first != func) continue;
    if (e.second < bytes) {
      GN3D_CUDA(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                "cudaFuncSetAttribute");
      e.second = bytes;
    }
    return GN3D_OK;
  }
  GN3D_CUDA(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), "cudaFuncSetAttribute");
  g_attr_smem[di.dev].emplace_back(func, bytes);
  return GN3D_OK;
}

// How many clusters of cs CTAs with `smem` bytes of shared memory each kernel
// `k` can have resident at once on this device (0: none): its attributes
// raised, then the occupancy calculator asked.  The answer is kept per kernel,
// cluster size and shared memory; a refusal is an answer (the call takes
// another launch form), so its error is cleared.
struct ClusterFit {
  const void* k;
  int cs, smem, active;
};
std::vector<ClusterFit> g_cluster_fit[kMaxDevices];

int cluster_active(const void* k, int cs, int smem, DevInfo& di) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const ClusterFit& f : g_cluster_fit[di.dev])
      if (f.k == k && f.cs == cs && f.smem == smem) return f.active;
  }
  int n = 0;
  bool ok = smem <= di.smem_optin && raise_smem(k, smem, di) == GN3D_OK;
  if (ok && cs > 8) ok = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs);
    cfg.blockDim = dim3(32 * kClusterWarps);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = cs;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    ok = cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess;
  }
  if (!ok) {
    n = 0;
    cudaGetLastError();
  }
  std::lock_guard<std::mutex> lk(g_mu);
  std::vector<ClusterFit>& fits = g_cluster_fit[di.dev];
  if (fits.size() >= 4096) fits.clear();  // many distinct shapes: start the cache over
  fits.push_back(ClusterFit{k, cs, smem, n});
  return n;
}

// The cluster form runs only when every group's cluster is resident at once:
// a second wave of clusters costs more than the streaming kernels' second pass
// (measured: 256 channels at 32^3, 7 of 8 clusters resident, 26 against 23 us).
bool cluster_one_wave(const void* k, const Plan& p, int cs, int smem, DevInfo& di) {
  return smem > 0 && p.NG <= (int64_t)cluster_active(k, cs, smem, di);
}

// A launch in clusters of cs CTAs (one cluster per group).
template <class... KArgs, class... Args>
cudaError_t launch_cluster(void (*k)(KArgs...), int grid, int cs, int smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * kClusterWarps);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = cs;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

// The cluster form's shared memory per CTA for a plan, or 0 where it does not
// apply: whole units only, and the CTA's units, their results and the group's
// block results must fit.
template <class T, int kTensors, class V>
int cluster_smem(const Plan& p, const ClusterGeo& c, const DevInfo& di) {
  if (!plan_all_full(p) || p.NG < 1 || c.upc < 1 || p.NG * c.cs > (int64_t)0x7fffffff) return 0;
  const int64_t b = ClusterLayout<T, kTensors, V>::bytes(c.upc, c.nbg);
  return b <= di.smem_optin ? (int)b : 0;
}

// The forward in one cluster launch, where it applies (*done); nothing is
// allocated.
template <class TI, class TO>
int launch_forward_cluster(const void* x, const float* gamma, const float* beta, const Plan& p, float eps, void* y,
                           float* mean, float* rstd, cudaStream_t st, DevInfo& di, bool relu, bool* done) {
  *done = false;
  if (!want_cluster()) return GN3D_OK;
  const ClusterGeo c = cluster_geo(p);
  const int smem = cluster_smem<TI, 1, Part>(p, c, di);
  auto k = relu ? k_fwd_cluster<TI, TO, true> : k_fwd_cluster<TI, TO, false>;
  if (!cluster_one_wave((const void*)k, p, c.cs, smem, di)) return GN3D_OK;
  *done = true;
  cudaError_t e = injected_launch_error();
  if (e == cudaSuccess) {
    g_launches += 1;
    LaunchTimer tm(KK_FWD_CLUSTER, st, di);
    e = launch_cluster(k, (int)(p.NG * c.cs), c.cs, smem, st, static_cast<const TI*>(x), static_cast<TO*>(y), p, c,
                       eps, gamma, beta, mean, rstd, spin_budget(), di.status, g_hook_timeout.exchange(0) != 0 ? 1 : 0);
    tm.done();
  }
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  return GN3D_OK;
}

// Launch of a kernel that may start before the previous kernel on the stream
// has finished (programmatic dependent launch); it waits in-kernel (pdl_wait)
// before reading that kernel's results.
template <class... KArgs, class... Args>
cudaError_t launch_dependent(void (*k)(KArgs...), int grid, int threads, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

// Grid of a persistent launch: one CTA per SM, all resident at once.
int coop_grid(const void* func, int threads, int smem, const DevInfo& di, int* grid) {
  int per_sm = 0;
  GN3D_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, threads, (size_t)smem),
            "occupancy");
  if (per_sm < 1) {
    g_detail = "persistent kernel does not fit on an SM";
    return GN3D_ERR_CUDA;
  }
  *grid = di.sms;
  return GN3D_OK;
}

// --------------------------------------------------------------- forward
// The normalize kernel for a plan: full units or not, fused ReLU or not, layout.
template <class TI, class TO>
auto norm_kernel(bool full, bool relu, bool cut) {
  using K = decltype(&k_fwd_norm<TI, TO, true, true, true>);
  const K ks[8] = {k_fwd_norm<TI, TO, false, false, false>, k_fwd_norm<TI, TO, false, false, true>,
                   k_fwd_norm<TI, TO, false, true, false>,  k_fwd_norm<TI, TO, false, true, true>,
                   k_fwd_norm<TI, TO, true, false, false>,  k_fwd_norm<TI, TO, true, false, true>,
                   k_fwd_norm<TI, TO, true, true, false>,   k_fwd_norm<TI, TO, true, true, true>};
  return ks[(full ? 4 : 0) + (relu ? 2 : 0) + (cut ? 1 : 0)];
}

template <class TI, class TO>
int launch_forward(const void* x, const float* gamma, const float* beta, const Plan& p, float eps, void* y,
                   float* mean, float* rstd, cudaStream_t st, DevInfo& di, bool relu) {
  bool done = false;
  const int rc = launch_forward_cluster<TI, TO>(x, gamma, beta, p, eps, y, mean, rstd, st, di, relu, &done);
  if (done) return rc;
  const bool fused = use_fused() && !relu;  // the fused ReLU runs in the streaming kernels
  const int64_t nblk = p.NC * p.nb;
  const int64_t nsync = nblk + 2 * p.NG + 2;  // bcnt, gcnt, ready, abort, never
  const int64_t bytes = rup(nsync * 4) + rup(p.units * (int64_t)sizeof(Part)) +
                        rup(nblk * (int64_t)sizeof(Part)) + rup(p.NG * (int64_t)sizeof(float4));
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, bytes, di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  uint32_t* sync = s.take<uint32_t>(nsync);
  FwdWs w;
  w.moments = nullptr;
  w.bcnt = sync;
  w.gcnt = sync + nblk;
  w.ready = sync + nblk + p.NG;
  w.parts = s.take<Part>(p.units);
  w.bparts = s.take<Part>(nblk);
  w.stats = s.take<float4>(p.NG);
  FusedSync fs{sync + nblk + 2 * p.NG, sync + nblk + 2 * p.NG + 1, di.status};
  cudaError_t e = cudaMemsetAsync(sync, 0, (size_t)nsync * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = injected_launch_error();
  const TI* xp = static_cast<const TI*>(x);
  TO* yp = static_cast<TO*>(y);
  if (e == cudaSuccess && use_resident(p, di)) {
    int smem = 0;
    using Shape = ResFwdShape<TI>;
    using Lay = ResLayout<Shape::kSlotBytes, Part, Shape::kRound>;
    ResCfg cfg = resident_cfg(di, p, Shape::kRed, Shape::kSlotBytes, Lay::bytes(0, 0), &smem);
    auto k = relu ? k_fwd_resident<TI, TO, true> : k_fwd_resident<TI, TO, false>;
    int rc = resident_lead_ok(cfg) ? raise_smem((const void*)k, smem, di) : arg_fail("group-wave lead too long");
    const int threads = 32 * ResFwdShape<TI>::kWarps;
    int grid = 0;
    if (!rc) rc = coop_grid((const void*)k, threads, smem, di, &grid);
    if (rc) { cudaFreeAsync(s.base, st); return rc; }
    ResSync rs{fs.abort, fs.never, fs.status};
    void* args[] = {(void*)&xp, (void*)&yp, (void*)&p, (void*)&w, (void*)&cfg, (void*)&rs, (void*)&eps,
                    (void*)&gamma, (void*)&beta, (void*)&mean, (void*)&rstd};
    g_launches += 1;
    LaunchTimer tm(KK_FWD_RES, st, di);
    e = cudaLaunchCooperativeKernel((const void*)k, dim3(grid), dim3(threads), args, (size_t)smem, st);
    tm.done();
  } else if (e == cudaSuccess && fused) {
    const int slot = kUnitElems * (int)sizeof(TI);
    const int rec = (int)sizeof(BlockRec<Part>);
    FusedCfg cfg = fused_cfg(di, slot, rec, p.M * (int64_t)sizeof(TI));
    const int smem = cfg.slots * (slot + 16) + cfg.recs * rec;
    auto k = k_fwd_fused<TI, TO>;
    int rc = raise_smem((const void*)k, smem, di);
    const int threads = 32 * (FwdPolicy<TI>::kWarps + 1);
    int grid = 0;
    if (!rc) rc = coop_grid((const void*)k, threads, smem, di, &grid);
    if (rc) { cudaFreeAsync(s.base, st); return rc; }
    void* args[] = {(void*)&xp, (void*)&yp, (void*)&p, (void*)&w, (void*)&cfg, (void*)&fs, (void*)&eps,
                    (void*)&gamma, (void*)&beta, (void*)&mean, (void*)&rstd};
    g_launches += 1;
    LaunchTimer tm(KK_FWD_FUSED, st, di);
    e = cudaLaunchCooperativeKernel((const void*)k, dim3(grid), dim3(threads), args, (size_t)smem, st);
    tm.done();
  } else if (e == cudaSuccess) {
    using Shape = FwdStatShape<TI>;
    const int smem = Shape::kWarps * WarpRing<TI, 1, Shape::kSlots>::kWarpBytes;
    const bool full = plan_all_full(p);
    // one CTA per SM (fewer only when there are fewer units than SMs), every SM
    // an equal part of the work in either layout
    const int sgrid = grid_for(di, p.units, 1);
    const bool cut = unit_shares(p, (int64_t)sgrid * Shape::kWarps);
    auto ks = full ? (cut ? k_fwd_stats<TI, true, true> : k_fwd_stats<TI, true, false>)
                   : (cut ? k_fwd_stats<TI, false, true> : k_fwd_stats<TI, false, false>);
    int rc = raise_smem((const void*)ks, smem, di);
    if (rc) { cudaFreeAsync(s.base, st); return rc; }
    g_launches += 2;
    LaunchTimer t1(KK_FWD_STATS, st, di);
    ks<<<sgrid, 32 * Shape::kWarps, smem, st>>>(xp, p, w, eps, mean, rstd, spin_budget(), di.status);
    t1.done();
    e = cudaGetLastError();
    if (e == cudaSuccess) {
      LaunchTimer t2(KK_FWD_NORM, st, di);
      auto kn = norm_kernel<TI, TO>(full, relu, cut);
      e = launch_dependent(kn, sgrid, 32 * kElemWarps, st, xp, yp, p, (const float4*)w.stats, gamma, beta);
      t2.done();
    }
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

// -------------------------------------------------------------- backward
// The streaming backward launches; kRelu: behind a fused ReLU, dy gated by the
// forward's result `res`.
template <class T, bool kRelu>
cudaError_t launch_backward_streaming(const T* dyp, const T* xp, const T* resp, T* dxp, const Plan& p,
                                      const float* mean, const float* rstd, const float* gamma, BwdWs& w,
                                      float* dgamma, float* dbeta, cudaStream_t st, DevInfo& di, int* rc) {
  using Shape = BwdRedShape<T, kRelu>;
  const int smem = Shape::kWarps * WarpRing<T, Shape::kTensors, Shape::kSlots, Shape::kElems>::kWarpBytes;
  const bool full = plan_all_full(p);
  const int rgrid = grid_for(di, p.units, 1);
  const bool cut = unit_shares(p, (int64_t)rgrid * Shape::kWarps);
  auto kr = full ? (cut ? k_bwd_reduce<T, true, kRelu, true> : k_bwd_reduce<T, true, kRelu, false>)
                 : (cut ? k_bwd_reduce<T, false, kRelu, true> : k_bwd_reduce<T, false, kRelu, false>);
  *rc = raise_smem((const void*)kr, smem, di);
  if (*rc) return cudaSuccess;
  g_launches += 2;
  LaunchTimer t1(KK_BWD_REDUCE, st, di);
  kr<<<rgrid, 32 * Shape::kWarps, smem, st>>>(dyp, xp, resp, p, mean, rstd, gamma, w, dgamma, dbeta,
                                             spin_budget(), di.status);
  t1.done();
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    LaunchTimer t2(KK_BWD_DX, st, di);
    auto kd = full ? (cut ? k_bwd_dx<T, true, kRelu, true> : k_bwd_dx<T, true, kRelu, false>)
                   : (cut ? k_bwd_dx<T, false, kRelu, true> : k_bwd_dx<T, false, kRelu, false>);
    e = launch_dependent(kd, rgrid, 32 * kElemWarps, st, dyp, xp, resp, dxp, p, mean, rstd, gamma,
                         (const float2*)w.coef);
    t2.done();
  }
  return e;
}

template <class T>
int launch_backward(const void* dy, const void* x, const void* res, const float* mean, const float* rstd,
                    const float* gamma, const Plan& p, void* dx, float* dgamma, float* dbeta, cudaStream_t st,
                    DevInfo& di) {
  const bool fused = use_fused() && !res;  // the fused ReLU's gate runs in the streaming kernels
  const int64_t nblk = p.NC * p.nb;
  const int64_t nsync = nblk + 2 * p.NG + 3;  // bcnt, gcnt, ready, done, abort, never
  const int64_t bytes = rup(nsync * 4) + rup(p.units * (int64_t)sizeof(float2)) +
                        rup(nblk * (int64_t)sizeof(float2)) + rup(p.NC * (int64_t)sizeof(float2)) +
                        rup(p.NG * (int64_t)sizeof(float2));
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, bytes, di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  uint32_t* sync = s.take<uint32_t>(nsync);
  BwdWs w;
  w.bcnt = sync;
  w.gcnt = sync + nblk;
  w.ready = sync + nblk + p.NG;
  w.done = sync + nblk + 2 * p.NG;
  w.parts = s.take<float2>(p.units);
  w.bparts = s.take<float2>(nblk);
  w.rows = s.take<float2>(p.NC);
  w.coef = s.take<float2>(p.NG);
  FusedSync fs{sync + nblk + 2 * p.NG + 1, sync + nblk + 2 * p.NG + 2, di.status};
  cudaError_t e = cudaMemsetAsync(sync, 0, (size_t)nsync * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = injected_launch_error();
  const T* dyp = static_cast<const T*>(dy);
  const T* xp = static_cast<const T*>(x);
  T* dxp = static_cast<T*>(dx);
  const ClusterGeo cg = cluster_geo(p);
  const int csmem = !res && want_cluster() ? cluster_smem<T, 2, float2>(p, cg, di) : 0;
  if (e == cudaSuccess && cluster_one_wave((const void*)k_bwd_cluster<T>, p, cg.cs, csmem, di)) {
    g_launches += 1;
    LaunchTimer tm(KK_BWD_CLUSTER, st, di);
    e = launch_cluster(k_bwd_cluster<T>, (int)(p.NG * cg.cs), cg.cs, csmem, st, dyp, xp, dxp, p, cg, mean, rstd,
                       gamma, w.rows, w.done, dgamma, dbeta, spin_budget(), di.status,
                       g_hook_timeout.exchange(0) != 0 ? 1 : 0);
    tm.done();
  } else if (e == cudaSuccess && !res && sizeof(T) == 2 && use_resident(p, di)) {
    int smem = 0;
    using Shape = ResBwdShape<T>;
    using Lay = ResLayout<Shape::kSlotBytes, float2, Shape::kRound>;
    ResCfg cfg = resident_cfg(di, p, Shape::kRed, Shape::kSlotBytes, Lay::bytes(0, 0), &smem);
    auto k = k_bwd_resident<T>;
    int rc = resident_lead_ok(cfg) ? raise_smem((const void*)k, smem, di) : arg_fail("group-wave lead too long");
    const int threads = 32 * ResBwdShape<T>::kWarps;
    int grid = 0;
    if (!rc) rc = coop_grid((const void*)k, threads, smem, di, &grid);
    if (rc) { cudaFreeAsync(s.base, st); return rc; }
    ResSync rs{fs.abort, fs.never, fs.status};
    void* args[] = {(void*)&dyp, (void*)&xp, (void*)&dxp, (void*)&p, (void*)&mean, (void*)&rstd, (void*)&gamma,
                    (void*)&w, (void*)&cfg, (void*)&rs, (void*)&dgamma, (void*)&dbeta};
    g_launches += 1;
    LaunchTimer tm(KK_BWD_RES, st, di);
    e = cudaLaunchCooperativeKernel((const void*)k, dim3(grid), dim3(threads), args, (size_t)smem, st);
    tm.done();
  } else if (e == cudaSuccess && fused) {
    const int slot = 2 * kUnitElems * (int)sizeof(T);
    const int rec = (int)sizeof(BlockRec<float2>);
    FusedCfg cfg = fused_cfg(di, slot, rec, 2 * p.M * (int64_t)sizeof(T));
    const int smem = cfg.slots * (slot + 16) + cfg.recs * rec;
    auto k = k_bwd_fused<T>;
    int rc = raise_smem((const void*)k, smem, di);
    const int threads = 32 * (BwdPolicy<T>::kWarps + 1);
    int grid = 0;
    if (!rc) rc = coop_grid((const void*)k, threads, smem, di, &grid);
    if (rc) { cudaFreeAsync(s.base, st); return rc; }
    void* args[] = {(void*)&dyp, (void*)&xp, (void*)&dxp, (void*)&p, (void*)&mean, (void*)&rstd, (void*)&gamma,
                    (void*)&w, (void*)&cfg, (void*)&fs, (void*)&dgamma, (void*)&dbeta};
    g_launches += 1;
    LaunchTimer tm(KK_BWD_FUSED, st, di);
    e = cudaLaunchCooperativeKernel((const void*)k, dim3(grid), dim3(threads), args, (size_t)smem, st);
    tm.done();
  } else if (e == cudaSuccess) {
    int rc = GN3D_OK;
    const T* resp = static_cast<const T*>(res);
    e = res ? launch_backward_streaming<T, true>(dyp, xp, resp, dxp, p, mean, rstd, gamma, w, dgamma, dbeta, st,
                                                 di, &rc)
            : launch_backward_streaming<T, false>(dyp, xp, nullptr, dxp, p, mean, rstd, gamma, w, dgamma, dbeta,
                                                  st, di, &rc);
    if (rc) { cudaFreeAsync(s.base, st); return rc; }
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

// ---------------------------------------------------- channels-last (NDHWC)
// Three dependent launches per direction (gn3d_ndhwc.cuh): the streaming
// reduction on min(SMs, units) CTAs, the finalize (one CTA per group / per row),
// then the elementwise pass on the reduction's grid.
template <class TI, class TO>
int launch_forward_ndhwc(const void* x, const float* gamma, const float* beta, const NPlan& p, float eps, void* y,
                         float* mean, float* rstd, cudaStream_t st, DevInfo& di, bool relu) {
  const int64_t tasks = p.NG * n_fin_maxr(p) * n_fin_nkc(p);  // finalize chunks
  const int64_t bytes = rup((p.NG + 1) * 4) + rup(p.rows * p.P * p.R * (int64_t)sizeof(Part)) +
                        rup(tasks * (int64_t)sizeof(Part)) + rup(p.NG * (int64_t)sizeof(float4));
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, bytes, di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  NFwdWs w;
  w.gcnt = s.take<uint32_t>(p.NG + 1);
  w.never = w.gcnt + p.NG;
  w.upart = s.take<Part>(p.rows * p.P * p.R);
  w.fpart = s.take<Part>(tasks);
  w.stats = s.take<float4>(p.NG);
  const TI* xp = static_cast<const TI*>(x);
  TO* yp = static_cast<TO*>(y);
  // one channel range: the bulk-copy ring kernel; else the direct one (per warp:
  // one unit's channel partials in shared memory, plus the ring's slots)
  const bool ring = p.nr == 1;
  const int smem = ring ? NStatRing<TI>::kSmem : kNRedWarps * kNSpan * kNVec * (int)sizeof(Part);
  const void* kfn = ring ? (const void*)k_ndhwc_stats_ring<TI> : (const void*)k_ndhwc_stats<TI>;
  int rc = raise_smem(kfn, smem, di);
  if (rc) { cudaFreeAsync(s.base, st); return rc; }
  const int grid = grid_for(di, p.units, 1);
  cudaError_t e = cudaMemsetAsync(w.gcnt, 0, (size_t)(p.NG + 1) * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = injected_launch_error();
  if (e == cudaSuccess) {
    g_launches += 3;
    LaunchTimer t1(KK_N_STATS, st, di);
    if (ring)
      k_ndhwc_stats_ring<TI><<<grid, 32 * kNRedWarps, smem, st>>>(xp, p, w, spin_budget(), di.status,
                                                                  g_hook_timeout.exchange(0) != 0 ? 1 : 0);
    else
      k_ndhwc_stats<TI><<<grid, 32 * kNRedWarps, smem, st>>>(xp, p, w);
    t1.done();
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    LaunchTimer t2(KK_N_STATS_FINAL, st, di);
    e = launch_dependent(k_ndhwc_stats_final, grid_for(di, tasks, 4), kNFinThreads, st, p, w, eps, mean, rstd);
    t2.done();
  }
  if (e == cudaSuccess) {
    LaunchTimer t3(KK_N_NORM, st, di);
    auto kn = relu ? k_ndhwc_norm<TI, TO, true> : k_ndhwc_norm<TI, TO, false>;
    e = launch_dependent(kn, grid, 32 * kNElemWarps, st, xp, yp, p, (const float4*)w.stats, gamma, beta);
    t3.done();
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

template <class T>
int launch_backward_ndhwc(const void* dy, const void* x, const void* res, const float* mean, const float* rstd,
                          const float* gamma, const NPlan& p, void* dx, float* dgamma, float* dbeta, cudaStream_t st,
                          DevInfo& di) {
  const int64_t NC = p.N * p.C, tasks = NC * n_fin_nkc(p);
  const int64_t nsync = NC + 1;  // chunks done per row, rows done
  const int64_t bytes = rup(nsync * 4) + rup(NC * p.R * (int64_t)sizeof(float2)) +
                        rup(tasks * (int64_t)sizeof(float2)) + rup(NC * (int64_t)sizeof(float2)) +
                        rup(p.NG * (int64_t)sizeof(float2));
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, bytes, di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  NBwdWs w;
  uint32_t* sync = s.take<uint32_t>(nsync);
  w.rcnt = sync;
  w.done = sync + NC;
  w.usum = s.take<float2>(NC * p.R);
  w.rpart = s.take<float2>(tasks);
  w.rows = s.take<float2>(NC);
  w.coef = s.take<float2>(p.NG);
  cudaError_t e = cudaMemsetAsync(sync, 0, (size_t)nsync * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = injected_launch_error();
  const T* dyp = static_cast<const T*>(dy);
  const T* xp = static_cast<const T*>(x);
  const T* resp = static_cast<const T*>(res);
  T* dxp = static_cast<T*>(dx);
  const int grid = grid_for(di, p.units, 1);
  const bool ring = p.nr == 1;  // one channel range: the bulk-copy ring kernel
  if (ring) {
    const int smem = res ? NRedRing<T, true>::kSmem : NRedRing<T, false>::kSmem;
    int rc = raise_smem(res ? (const void*)k_ndhwc_reduce_ring<T, true> : (const void*)k_ndhwc_reduce_ring<T, false>,
                        smem, di);
    if (rc) { cudaFreeAsync(s.base, st); return rc; }
  }
  if (e == cudaSuccess) {
    g_launches += 3;
    LaunchTimer t1(KK_N_REDUCE, st, di);
    const unsigned long long spin = spin_budget();
    if (ring && res)
      k_ndhwc_reduce_ring<T, true><<<grid, 32 * kNRedWarps, NRedRing<T, true>::kSmem, st>>>(dyp, xp, resp, p, mean, w,
                                                                                            spin, di.status);
    else if (ring)
      k_ndhwc_reduce_ring<T, false><<<grid, 32 * kNRedWarps, NRedRing<T, false>::kSmem, st>>>(dyp, xp, nullptr, p,
                                                                                              mean, w, spin, di.status);
    else if (res)
      k_ndhwc_reduce<T, true><<<grid, 32 * kNRedWarps, 0, st>>>(dyp, xp, resp, p, mean, w);
    else
      k_ndhwc_reduce<T, false><<<grid, 32 * kNRedWarps, 0, st>>>(dyp, xp, nullptr, p, mean, w);
    t1.done();
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    LaunchTimer t2(KK_N_REDUCE_FINAL, st, di);
    const int64_t ftasks = n_fin_short_rows(p) ? (NC + kNFinThreads / 32 - 1) / (kNFinThreads / 32) : tasks;
    e = launch_dependent(k_ndhwc_reduce_final, grid_for(di, ftasks, 4), kNFinThreads, st, p, w, rstd, gamma, dgamma,
                         dbeta);
    t2.done();
  }
  if (e == cudaSuccess) {
    LaunchTimer t3(KK_N_DX, st, di);
    auto kd = res ? k_ndhwc_dx<T, true> : k_ndhwc_dx<T, false>;
    e = launch_dependent(kd, grid, 32 * kNElemWarps, st, dyp, xp, resp, dxp, p, mean, rstd, gamma, (const float2*)w.coef);
    t3.done();
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

bool valid_dtype(int d) { return d == GN3D_F32 || d == GN3D_BF16; }

// ------------------------------------------------------ sharded statistics
// The forward statistics kernel alone, exporting each group's moments.
template <class TI>
int launch_moments(const void* x, const Plan& p, Moments* moments, cudaStream_t st, DevInfo& di) {
  const int64_t nblk = p.NC * p.nb;
  const int64_t nsync = nblk + 2 * p.NG;
  const int64_t bytes = rup(nsync * 4) + rup(p.units * (int64_t)sizeof(Part)) + rup(nblk * (int64_t)sizeof(Part));
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, bytes, di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  uint32_t* sync = s.take<uint32_t>(nsync);
  FwdWs w;
  w.moments = moments;
  w.bcnt = sync;
  w.gcnt = sync + nblk;
  w.ready = sync + nblk + p.NG;
  w.parts = s.take<Part>(p.units);
  w.bparts = s.take<Part>(nblk);
  w.stats = nullptr;
  cudaError_t e = cudaMemsetAsync(sync, 0, (size_t)nsync * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = injected_launch_error();
  using Shape = FwdStatShape<TI>;
  const int smem = Shape::kWarps * WarpRing<TI, 1, Shape::kSlots>::kWarpBytes;
  const bool full = plan_all_full(p);
  const int sgrid = grid_for(di, p.units, 1);
  const bool cut = unit_shares(p, (int64_t)sgrid * Shape::kWarps);
  auto ks = full ? (cut ? k_fwd_stats<TI, true, true> : k_fwd_stats<TI, true, false>)
                 : (cut ? k_fwd_stats<TI, false, true> : k_fwd_stats<TI, false, false>);
  int rc = raise_smem((const void*)ks, smem, di);
  if (rc) { cudaFreeAsync(s.base, st); return rc; }
  if (e == cudaSuccess) {
    g_launches += 1;
    LaunchTimer t1(KK_FWD_STATS, st, di);
    ks<<<sgrid, 32 * Shape::kWarps, smem, st>>>(static_cast<const TI*>(x), p, w, 1.f, nullptr, nullptr,
                                                spin_budget(), di.status);
    t1.done();
    e = cudaGetLastError();
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "moments launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

// The normalize pass with statistics formed from given (combined) moments.
template <class TI, class TO>
int launch_apply(const void* x, const float* gamma, const float* beta, const Plan& p, float eps,
                 const Moments* moments, void* y, float* mean, float* rstd, cudaStream_t st, DevInfo& di) {
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, rup(p.NG * (int64_t)sizeof(float4)), di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  float4* stats = s.take<float4>(p.NG);
  cudaError_t e = injected_launch_error();
  if (e == cudaSuccess) {
    g_launches += 2;
    k_stats_from_moments<<<(unsigned)((p.NG + 127) / 128), 128, 0, st>>>(moments, p.NG, eps, stats, mean, rstd);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    using Shape = FwdStatShape<TI>;
    const bool full = plan_all_full(p);
    const int sgrid = grid_for(di, p.units, 1);
    const bool cut = unit_shares(p, (int64_t)sgrid * Shape::kWarps);
    LaunchTimer t2(KK_FWD_NORM, st, di);
    auto kn = norm_kernel<TI, TO>(full, false, cut);
    e = launch_dependent(kn, sgrid, 32 * kElemWarps, st, static_cast<const TI*>(x), static_cast<TO*>(y), p,
                         (const float4*)stats, gamma, beta);
    t2.done();
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "apply launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

// The backward reduction alone, its per-row totals written to `sums`.
template <class T>
int launch_row_sums(const void* dy, const void* x, const float* mean, const float* rstd, const Plan& p,
                    float2* sums, cudaStream_t st, DevInfo& di) {
  const int64_t nblk = p.NC * p.nb;
  const int64_t nsync = nblk + 2 * p.NG + 1;  // bcnt, gcnt, ready, done
  const int64_t bytes = rup(nsync * 4) + rup(p.units * (int64_t)sizeof(float2)) +
                        rup(nblk * (int64_t)sizeof(float2)) + rup(p.NG * (int64_t)sizeof(float2));
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, bytes, di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  uint32_t* sync = s.take<uint32_t>(nsync);
  BwdWs w;
  w.bcnt = sync;
  w.gcnt = sync + nblk;
  w.ready = sync + nblk + p.NG;
  w.done = sync + nblk + 2 * p.NG;
  w.parts = s.take<float2>(p.units);
  w.bparts = s.take<float2>(nblk);
  w.rows = sums;
  w.coef = s.take<float2>(p.NG);
  cudaError_t e = cudaMemsetAsync(sync, 0, (size_t)nsync * sizeof(uint32_t), st);
  if (e == cudaSuccess) e = injected_launch_error();
  using Shape = BwdRedShape<T, false>;
  const int smem = Shape::kWarps * WarpRing<T, Shape::kTensors, Shape::kSlots, Shape::kElems>::kWarpBytes;
  const bool full = plan_all_full(p);
  const int rgrid = grid_for(di, p.units, 1);
  const bool cut = unit_shares(p, (int64_t)rgrid * Shape::kWarps);
  auto kr = full ? (cut ? k_bwd_reduce<T, true, false, true> : k_bwd_reduce<T, true, false, false>)
                 : (cut ? k_bwd_reduce<T, false, false, true> : k_bwd_reduce<T, false, false, false>);
  int rc = raise_smem((const void*)kr, smem, di);
  if (rc) { cudaFreeAsync(s.base, st); return rc; }
  if (e == cudaSuccess) {
    g_launches += 1;
    LaunchTimer t1(KK_BWD_REDUCE, st, di);
    kr<<<rgrid, 32 * Shape::kWarps, smem, st>>>(static_cast<const T*>(dy), static_cast<const T*>(x), nullptr, p,
                                               mean, rstd, nullptr, w, nullptr, nullptr, spin_budget(), di.status);
    t1.done();
    e = cudaGetLastError();
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "sums launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

// The dx pass (and dgamma, dbeta) from given per-row totals over groups of M elements.
template <class T>
int launch_dx_from_sums(const void* dy, const void* x, const float* mean, const float* rstd, const float* gamma,
                        const float2* sums, int64_t M, const Plan& p, void* dx, float* dgamma, float* dbeta,
                        cudaStream_t st, DevInfo& di) {
  Scratch s;
  GN3D_CUDA(scratch_alloc(&s.base, rup(p.NG * (int64_t)sizeof(float2)), di, st), "scratch allocation");
  s.cur = static_cast<char*>(s.base);
  float2* coef = s.take<float2>(p.NG);
  cudaError_t e = injected_launch_error();
  if (e == cudaSuccess) {
    g_launches += 1;
    k_coef_from_sums<<<(unsigned)((p.NG + 127) / 128), 128, 0, st>>>(p, sums, rstd, gamma, M, coef);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess && (dgamma || dbeta)) {
    g_launches += 1;
    k_param_grads<<<1, 32, 0, st>>>(p, rstd, sums, dgamma, dbeta);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    using Shape = BwdRedShape<T, false>;
    const bool full = plan_all_full(p);
    const int rgrid = grid_for(di, p.units, 1);
    const bool cut = unit_shares(p, (int64_t)rgrid * Shape::kWarps);
    g_launches += 1;
    LaunchTimer t2(KK_BWD_DX, st, di);
    auto kd = full ? (cut ? k_bwd_dx<T, true, false, true> : k_bwd_dx<T, true, false, false>)
                   : (cut ? k_bwd_dx<T, false, false, true> : k_bwd_dx<T, false, false, false>);
    e = launch_dependent(kd, rgrid, 32 * kElemWarps, st, static_cast<const T*>(dy), static_cast<const T*>(x),
                         (const T*)nullptr, static_cast<T*>(dx), p, mean, rstd, gamma, (const float2*)coef);
    t2.done();
  }
  cudaError_t ef = cudaFreeAsync(s.base, st);
  if (e != cudaSuccess) return cuda_fail(e, "dx launch");
  if (ef != cudaSuccess) return cuda_fail(ef, "scratch free");
  return GN3D_OK;
}

// ------------------------------------------------- allocation-free forward
// Scratch of gn3d_forward_noalloc: one fixed area in the module's global memory,
// present on every device that loads the library, for as long as it is loaded.
// Host code never touches it by name: the name is only a host-side handle, so
// its device address is looked up once per device (cudaGetSymbolAddress, with
// that device current) and passed to the kernel.
constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDev {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  uint32_t* status = nullptr;        // device address of the status word
  DevInfo facts;                     // SM count, L2 and shared-memory sizes (no pool)
};
NoAllocDev g_noalloc[kMaxDevices];

int noalloc_setup(int dev, NoAllocDev** out) {
  if (dev < 0 || dev >= kMaxDevices) return arg_fail("device ordinal out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  NoAllocDev& d = g_noalloc[dev];
  if (!d.ready) {
    d.facts.dev = dev;
    GN3D_CUDA(cudaDeviceGetAttribute(&d.facts.sms, cudaDevAttrMultiProcessorCount, dev), "device attribute");
    GN3D_CUDA(cudaDeviceGetAttribute(&d.facts.l2_bytes, cudaDevAttrL2CacheSize, dev), "device attribute");
    GN3D_CUDA(cudaDeviceGetAttribute(&d.facts.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev),
              "device attribute");
    void* sym = nullptr;
    GN3D_CUDA(cudaGetSymbolAddress(&sym, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)");
    d.scratch = static_cast<unsigned char*>(sym);
    GN3D_CUDA(cudaGetSymbolAddress(&sym, g_status_word), "cudaGetSymbolAddress(status)");
    d.status = static_cast<uint32_t*>(sym);
    d.ready = true;
  }
  *out = &d;
  return GN3D_OK;
}

// The forward's scratch layout (sync words, unit partials, block partials, group
// statistics) laid over the static area; the same layout gn3d_forward allocates.
int64_t noalloc_bytes(const Plan& p) {
  const int64_t nblk = p.NC * p.nb;
  return rup((nblk + 2 * p.NG + 2) * 4) + rup(p.units * (int64_t)sizeof(Part)) +
         rup(nblk * (int64_t)sizeof(Part)) + rup(p.NG * (int64_t)sizeof(float4));
}

template <class TI, class TO>
int launch_forward_noalloc(const void* x, const float* gamma, const float* beta, const Plan& p, float eps,
                           void* y, float* mean, float* rstd, cudaStream_t st, NoAllocDev& nd) {
  const int64_t nblk = p.NC * p.nb;
  const int64_t nsync = nblk + 2 * p.NG + 2;
  Scratch s;
  s.base = nd.scratch;
  s.cur = reinterpret_cast<char*>(nd.scratch);
  uint32_t* sync = s.take<uint32_t>(nsync);
  FwdWs w;
  w.moments = nullptr;
  w.bcnt = sync;
  w.gcnt = sync + nblk;
  w.ready = sync + nblk + p.NG;
  w.parts = s.take<Part>(p.units);
  w.bparts = s.take<Part>(nblk);
  w.stats = s.take<float4>(p.NG);
  FusedSync fs{sync + nblk + 2 * p.NG, sync + nblk + 2 * p.NG + 1, nd.status};
  // the area keeps the previous call's contents: the counters and flags start at zero
  GN3D_CUDA(cudaMemsetAsync(sync, 0, (size_t)nsync * sizeof(uint32_t), st), "memset");
  const int slot = kUnitElems * (int)sizeof(TI);
  const int rec = (int)sizeof(BlockRec<Part>);
  FusedCfg cfg = fused_cfg(nd.facts, slot, rec, p.M * (int64_t)sizeof(TI));
  const int smem = cfg.slots * (slot + 16) + cfg.recs * rec;
  auto k = k_fwd_fused<TI, TO>;
  int rc = raise_smem((const void*)k, smem, nd.facts);
  if (rc) return rc;
  const int threads = 32 * (FwdPolicy<TI>::kWarps + 1);
  int grid = 0;
  rc = coop_grid((const void*)k, threads, smem, nd.facts, &grid);
  if (rc) return rc;
  const TI* xp = static_cast<const TI*>(x);
  TO* yp = static_cast<TO*>(y);
  void* args[] = {(void*)&xp, (void*)&yp, (void*)&p, (void*)&w, (void*)&cfg, (void*)&fs, (void*)&eps,
                  (void*)&gamma, (void*)&beta, (void*)&mean, (void*)&rstd};
  g_launches += 1;
  GN3D_CUDA(cudaLaunchCooperativeKernel((const void*)k, dim3(grid), dim3(threads), args, (size_t)smem, st),
            "forward launch");
  return GN3D_OK;
}

}  // namespace
}  // namespace gn3d

using namespace gn3d;

namespace {
int forward_impl(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C, int64_t D, int64_t H,
                 int64_t W, int64_t G, double eps, gn3d_dtype in_dtype, gn3d_dtype out_dtype, void* y, float* mean,
                 float* rstd, void* stream, bool relu, bool ndhwc = false) {
  int rc = check_shape(N, C, D, H, W, G);
  if (rc) return rc;
  if (ndhwc && C % kNVec != 0 && N * D * H * W > 0) return arg_fail("the NDHWC layout needs C % 8 == 0");
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return arg_fail("unsupported dtype");
  if (!(eps >= 0.0) || !isfinite(eps)) return arg_fail("eps must be finite and >= 0");
  const float feps = (float)eps;
  const Plan p = make_plan(N, C, D * H * W, G);
  const int64_t numel = p.NC * p.S;
  int dev = 0;
  GN3D_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DevInfo* di = nullptr;
  if ((rc = device_info(dev, &di))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (numel > 0) {
    if (!x || !y) return arg_fail("x and y are required");
    if (!aligned16(x) || !aligned16(y)) return arg_fail("x and y must be 16-byte aligned");
    if ((rc = check_ptr(x, dev, "x")) || (rc = check_ptr(y, dev, "y"))) return rc;
  }
  if (p.NG > 0) {
    if (mean && (rc = check_ptr(mean, dev, "mean"))) return rc;
    if (rstd && (rc = check_ptr(rstd, dev, "rstd"))) return rc;
  }
  if (C > 0) {
    if (gamma && (rc = check_ptr(gamma, dev, "gamma"))) return rc;
    if (beta && (rc = check_ptr(beta, dev, "beta"))) return rc;
  }
  if (numel == 0) {
    if (p.NG > 0 && (mean || rstd)) {
      g_launches += 1;
      k_fill_empty_stats<<<(unsigned)((p.NG + 255) / 256), 256, 0, st>>>(mean, rstd, p.NG, feps);
      GN3D_CUDA(cudaGetLastError(), "fill launch");
    }
    return GN3D_OK;
  }
  using bf = __nv_bfloat16;
  if (ndhwc) {
    const NPlan np = make_nplan(N, C, D * H * W, G, kNMinUnitsFwd);
    if (in_dtype == GN3D_BF16 && out_dtype == GN3D_BF16)
      return launch_forward_ndhwc<bf, bf>(x, gamma, beta, np, feps, y, mean, rstd, st, *di, relu);
    if (in_dtype == GN3D_BF16 && out_dtype == GN3D_F32)
      return launch_forward_ndhwc<bf, float>(x, gamma, beta, np, feps, y, mean, rstd, st, *di, relu);
    if (in_dtype == GN3D_F32 && out_dtype == GN3D_BF16)
      return launch_forward_ndhwc<float, bf>(x, gamma, beta, np, feps, y, mean, rstd, st, *di, relu);
    return launch_forward_ndhwc<float, float>(x, gamma, beta, np, feps, y, mean, rstd, st, *di, relu);
  }
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_BF16)
    return launch_forward<bf, bf>(x, gamma, beta, p, feps, y, mean, rstd, st, *di, relu);
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_F32)
    return launch_forward<bf, float>(x, gamma, beta, p, feps, y, mean, rstd, st, *di, relu);
  if (in_dtype == GN3D_F32 && out_dtype == GN3D_BF16)
    return launch_forward<float, bf>(x, gamma, beta, p, feps, y, mean, rstd, st, *di, relu);
  return launch_forward<float, float>(x, gamma, beta, p, feps, y, mean, rstd, st, *di, relu);
}

int backward_impl(const void* dy, const void* x, const void* res, const float* mean, const float* rstd,
                  const float* gamma, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int64_t G,
                  gn3d_dtype dtype, void* dx, float* dgamma, float* dbeta, void* stream, bool relu,
                  bool ndhwc = false) {
  int rc = check_shape(N, C, D, H, W, G);
  if (rc) return rc;
  if (ndhwc && C % kNVec != 0 && N * D * H * W > 0) return arg_fail("the NDHWC layout needs C % 8 == 0");
  if (!valid_dtype(dtype)) return arg_fail("unsupported dtype");
  const Plan p = make_plan(N, C, D * H * W, G);
  const int64_t numel = p.NC * p.S;
  int dev = 0;
  GN3D_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DevInfo* di = nullptr;
  if ((rc = device_info(dev, &di))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (C > 0) {
    if (gamma && (rc = check_ptr(gamma, dev, "gamma"))) return rc;
    if (dgamma && (rc = check_ptr(dgamma, dev, "dgamma"))) return rc;
    if (dbeta && (rc = check_ptr(dbeta, dev, "dbeta"))) return rc;
  }
  if (numel == 0) {
    if (dgamma && C > 0) GN3D_CUDA(cudaMemsetAsync(dgamma, 0, (size_t)C * sizeof(float), st), "memset");
    if (dbeta && C > 0) GN3D_CUDA(cudaMemsetAsync(dbeta, 0, (size_t)C * sizeof(float), st), "memset");
    return GN3D_OK;
  }
  if (!dy || !x || !dx || !mean || !rstd) return arg_fail("dy, x, dx, mean and rstd are required");
  if (!aligned16(dy) || !aligned16(x) || !aligned16(dx)) return arg_fail("dy, x and dx must be 16-byte aligned");
  if ((rc = check_ptr(dy, dev, "dy")) || (rc = check_ptr(x, dev, "x")) || (rc = check_ptr(dx, dev, "dx")) ||
      (rc = check_ptr(mean, dev, "mean")) || (rc = check_ptr(rstd, dev, "rstd")))
    return rc;
  if (relu) {
    if (!res) return arg_fail("out (the forward's result) is required");
    if (!aligned16(res)) return arg_fail("out must be 16-byte aligned");
    if ((rc = check_ptr(res, dev, "out"))) return rc;
  }
  if (ndhwc) {
    const NPlan np = make_nplan(N, C, D * H * W, G, kNMinUnitsBwd);
    if (dtype == GN3D_BF16)
      return launch_backward_ndhwc<__nv_bfloat16>(dy, x, relu ? res : nullptr, mean, rstd, gamma, np, dx, dgamma,
                                                  dbeta, st, *di);
    return launch_backward_ndhwc<float>(dy, x, relu ? res : nullptr, mean, rstd, gamma, np, dx, dgamma, dbeta, st,
                                        *di);
  }
  if (dtype == GN3D_BF16)
    return launch_backward<__nv_bfloat16>(dy, x, relu ? res : nullptr, mean, rstd, gamma, p, dx, dgamma, dbeta,
                                          st, *di);
  return launch_backward<float>(dy, x, relu ? res : nullptr, mean, rstd, gamma, p, dx, dgamma, dbeta, st, *di);
}
}  // namespace

extern "C" int gn3d_forward(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                            int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                            gn3d_dtype out_dtype, void* y, float* mean, float* rstd, void* stream) {
  return forward_impl(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd, stream, false);
}

extern "C" int gn3d_forward_relu(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                                 int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                                 gn3d_dtype out_dtype, void* out, float* mean, float* rstd, void* stream) {
  return forward_impl(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, out, mean, rstd, stream, true);
}

// The forward without any allocation: the same kernel as gn3d_forward, with its
// scratch in the library's static device area (see include/gn3d.h).
extern "C" int gn3d_forward_noalloc(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                                    int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                                    gn3d_dtype out_dtype, void* y, float* mean, float* rstd, void* stream) {
  int rc = check_shape(N, C, D, H, W, G);
  if (rc) return rc;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return arg_fail("unsupported dtype");
  if (!(eps >= 0.0) || !isfinite(eps)) return arg_fail("eps must be finite and >= 0");
  const float feps = (float)eps;
  const Plan p = make_plan(N, C, D * H * W, G);
  const int64_t numel = p.NC * p.S;
  if (numel == 0) return arg_fail("gn3d_forward_noalloc needs a non-empty tensor");
  const int64_t need = noalloc_bytes(p);
  if (need > (int64_t)kNoAllocScratchBytes) {
    g_detail = "gn3d_forward_noalloc: this shape needs " + std::to_string(need) +
               " bytes of scratch; the static area holds " + std::to_string(kNoAllocScratchBytes);
    return GN3D_ERR_INVALID_ARG;
  }
  int dev = 0;
  GN3D_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  NoAllocDev* nd = nullptr;
  if ((rc = noalloc_setup(dev, &nd))) return rc;
  if (!x || !y) return arg_fail("x and y are required");
  if (!aligned16(x) || !aligned16(y)) return arg_fail("x and y must be 16-byte aligned");
  if ((rc = check_ptr(x, dev, "x")) || (rc = check_ptr(y, dev, "y"))) return rc;
  if (mean && (rc = check_ptr(mean, dev, "mean"))) return rc;
  if (rstd && (rc = check_ptr(rstd, dev, "rstd"))) return rc;
  if (gamma && (rc = check_ptr(gamma, dev, "gamma"))) return rc;
  if (beta && (rc = check_ptr(beta, dev, "beta"))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  using bf = __nv_bfloat16;
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_BF16)
    return launch_forward_noalloc<bf, bf>(x, gamma, beta, p, feps, y, mean, rstd, st, *nd);
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_F32)
    return launch_forward_noalloc<bf, float>(x, gamma, beta, p, feps, y, mean, rstd, st, *nd);
  if (in_dtype == GN3D_F32 && out_dtype == GN3D_BF16)
    return launch_forward_noalloc<float, bf>(x, gamma, beta, p, feps, y, mean, rstd, st, *nd);
  return launch_forward_noalloc<float, float>(x, gamma, beta, p, feps, y, mean, rstd, st, *nd);
}

extern "C" int gn3d_backward(const void* dy, const void* x, const float* mean, const float* rstd,
                             const float* gamma, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                             int64_t G, gn3d_dtype dtype, void* dx, float* dgamma, float* dbeta, void* stream) {
  return backward_impl(dy, x, nullptr, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream,
                       false);
}

extern "C" int gn3d_backward_relu(const void* dy, const void* x, const void* out, const float* mean,
                                  const float* rstd, const float* gamma, int64_t N, int64_t C, int64_t D,
                                  int64_t H, int64_t W, int64_t G, gn3d_dtype dtype, void* dx, float* dgamma,
                                  float* dbeta, void* stream) {
  return backward_impl(dy, x, out, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream, true);
}

extern "C" int gn3d_forward_ndhwc(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                                  int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                                  gn3d_dtype out_dtype, void* y, float* mean, float* rstd, void* stream) {
  return forward_impl(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd, stream, false, true);
}

extern "C" int gn3d_forward_ndhwc_relu(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                                       int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                                       gn3d_dtype out_dtype, void* out, float* mean, float* rstd, void* stream) {
  return forward_impl(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, out, mean, rstd, stream, true, true);
}

extern "C" int gn3d_backward_ndhwc(const void* dy, const void* x, const float* mean, const float* rstd,
                                   const float* gamma, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                                   int64_t G, gn3d_dtype dtype, void* dx, float* dgamma, float* dbeta, void* stream) {
  return backward_impl(dy, x, nullptr, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream, false,
                       true);
}

extern "C" int gn3d_backward_ndhwc_relu(const void* dy, const void* x, const void* out, const float* mean,
                                        const float* rstd, const float* gamma, int64_t N, int64_t C, int64_t D,
                                        int64_t H, int64_t W, int64_t G, gn3d_dtype dtype, void* dx, float* dgamma,
                                        float* dbeta, void* stream) {
  return backward_impl(dy, x, out, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream, true, true);
}

// ------------------------------------------------------ sharded statistics
namespace {
// Shapes of one shard: a shard may hold a single element of a group.
int check_dims(int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int64_t G) {
  if (N < 0 || C < 0 || D < 0 || H < 0 || W < 0) return arg_fail("negative dimension");
  if (G <= 0) return arg_fail("G must be >= 1");
  if (C % G != 0) return arg_fail("C must be divisible by G");
  const double total = (double)N * (double)C * (double)D * (double)H * (double)W;
  if (total > 4.0e18) return arg_fail("tensor too large");
  return GN3D_OK;
}

bool aligned8(const void* p) { return ((uintptr_t)p & 7u) == 0; }

// The current device's facts and a device pointer check of each non-null argument.
int setup(DevInfo** di, int* dev) {
  GN3D_CUDA(cudaGetDevice(dev), "cudaGetDevice");
  return device_info(*dev, di);
}
}  // namespace

extern "C" int gn3d_forward_moments(const void* x, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int64_t G,
                                    gn3d_dtype in_dtype, gn3d_moments* moments, void* stream) {
  static_assert(sizeof(gn3d_moments) == sizeof(Moments), "gn3d_moments layout");
  int rc = check_dims(N, C, D, H, W, G);
  if (rc) return rc;
  if (!valid_dtype(in_dtype)) return arg_fail("unsupported dtype");
  const Plan p = make_plan(N, C, D * H * W, G);
  int dev = 0;
  DevInfo* di = nullptr;
  if ((rc = setup(&di, &dev))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.NG == 0) return GN3D_OK;
  if (!moments || !aligned8(moments)) return arg_fail("moments is required, 8-byte aligned");
  if ((rc = check_ptr(moments, dev, "moments"))) return rc;
  if (p.NC * p.S == 0) {  // no elements: count 0, mean 0, M2 0
    GN3D_CUDA(cudaMemsetAsync(moments, 0, (size_t)p.NG * sizeof(gn3d_moments), st), "memset");
    return GN3D_OK;
  }
  if (!x || !aligned16(x)) return arg_fail("x is required, 16-byte aligned");
  if ((rc = check_ptr(x, dev, "x"))) return rc;
  Moments* m = reinterpret_cast<Moments*>(moments);
  return in_dtype == GN3D_BF16 ? launch_moments<__nv_bfloat16>(x, p, m, st, *di) : launch_moments<float>(x, p, m, st, *di);
}

extern "C" int gn3d_moments_combine(const gn3d_moments* shards, int64_t K, int64_t NG, gn3d_moments* combined,
                                    void* stream) {
  if (K < 1 || NG < 0) return arg_fail("K >= 1 shards, NG >= 0 groups");
  int dev = 0, rc;
  DevInfo* di = nullptr;
  if ((rc = setup(&di, &dev))) return rc;
  if (NG == 0) return GN3D_OK;
  if (!shards || !combined || !aligned8(shards) || !aligned8(combined))
    return arg_fail("shards and combined are required, 8-byte aligned");
  if ((rc = check_ptr(shards, dev, "shards")) || (rc = check_ptr(combined, dev, "combined"))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  g_launches += 1;
  k_moments_combine<<<(unsigned)((NG + 127) / 128), 128, 0, st>>>(reinterpret_cast<const Moments*>(shards), K, NG,
                                                                  reinterpret_cast<Moments*>(combined));
  GN3D_CUDA(cudaGetLastError(), "combine launch");
  return GN3D_OK;
}

extern "C" int gn3d_forward_apply(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                                  int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                                  gn3d_dtype out_dtype, const gn3d_moments* moments, void* y, float* mean, float* rstd,
                                  void* stream) {
  int rc = check_dims(N, C, D, H, W, G);
  if (rc) return rc;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return arg_fail("unsupported dtype");
  if (!(eps >= 0.0) || !isfinite(eps)) return arg_fail("eps must be finite and >= 0");
  const Plan p = make_plan(N, C, D * H * W, G);
  int dev = 0;
  DevInfo* di = nullptr;
  if ((rc = setup(&di, &dev))) return rc;
  if (p.NG == 0) return GN3D_OK;
  if (!moments || !aligned8(moments)) return arg_fail("moments is required, 8-byte aligned");
  if ((rc = check_ptr(moments, dev, "moments"))) return rc;
  if (p.NC * p.S > 0) {
    if (!x || !y) return arg_fail("x and y are required");
    if (!aligned16(x) || !aligned16(y)) return arg_fail("x and y must be 16-byte aligned");
    if ((rc = check_ptr(x, dev, "x")) || (rc = check_ptr(y, dev, "y"))) return rc;
  }
  if (mean && (rc = check_ptr(mean, dev, "mean"))) return rc;
  if (rstd && (rc = check_ptr(rstd, dev, "rstd"))) return rc;
  if (gamma && (rc = check_ptr(gamma, dev, "gamma"))) return rc;
  if (beta && (rc = check_ptr(beta, dev, "beta"))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float feps = (float)eps;
  const Moments* m = reinterpret_cast<const Moments*>(moments);
  using bf = __nv_bfloat16;
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_BF16)
    return launch_apply<bf, bf>(x, gamma, beta, p, feps, m, y, mean, rstd, st, *di);
  if (in_dtype == GN3D_BF16 && out_dtype == GN3D_F32)
    return launch_apply<bf, float>(x, gamma, beta, p, feps, m, y, mean, rstd, st, *di);
  if (in_dtype == GN3D_F32 && out_dtype == GN3D_BF16)
    return launch_apply<float, bf>(x, gamma, beta, p, feps, m, y, mean, rstd, st, *di);
  return launch_apply<float, float>(x, gamma, beta, p, feps, m, y, mean, rstd, st, *di);
}

extern "C" int gn3d_backward_sums(const void* dy, const void* x, const float* mean, const float* rstd, int64_t N,
                                  int64_t C, int64_t D, int64_t H, int64_t W, int64_t G, gn3d_dtype dtype, float* sums,
                                  void* stream) {
  int rc = check_dims(N, C, D, H, W, G);
  if (rc) return rc;
  if (!valid_dtype(dtype)) return arg_fail("unsupported dtype");
  const Plan p = make_plan(N, C, D * H * W, G);
  int dev = 0;
  DevInfo* di = nullptr;
  if ((rc = setup(&di, &dev))) return rc;
  if (p.NC == 0) return GN3D_OK;
  if (!sums || !aligned8(sums)) return arg_fail("sums is required, 8-byte aligned");
  if ((rc = check_ptr(sums, dev, "sums"))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.NC * p.S == 0) {
    GN3D_CUDA(cudaMemsetAsync(sums, 0, (size_t)p.NC * 2 * sizeof(float), st), "memset");
    return GN3D_OK;
  }
  if (!dy || !x || !mean || !rstd) return arg_fail("dy, x, mean and rstd are required");
  if (!aligned16(dy) || !aligned16(x)) return arg_fail("dy and x must be 16-byte aligned");
  if ((rc = check_ptr(dy, dev, "dy")) || (rc = check_ptr(x, dev, "x")) || (rc = check_ptr(mean, dev, "mean")) ||
      (rc = check_ptr(rstd, dev, "rstd")))
    return rc;
  float2* s2 = reinterpret_cast<float2*>(sums);
  return dtype == GN3D_BF16 ? launch_row_sums<__nv_bfloat16>(dy, x, mean, rstd, p, s2, st, *di)
                            : launch_row_sums<float>(dy, x, mean, rstd, p, s2, st, *di);
}

extern "C" int gn3d_sums_combine(const float* shards, int64_t K, int64_t NC, float* total, void* stream) {
  if (K < 1 || NC < 0) return arg_fail("K >= 1 shards, NC >= 0 rows");
  int dev = 0, rc;
  DevInfo* di = nullptr;
  if ((rc = setup(&di, &dev))) return rc;
  if (NC == 0) return GN3D_OK;
  if (!shards || !total || !aligned8(shards) || !aligned8(total))
    return arg_fail("shards and total are required, 8-byte aligned");
  if ((rc = check_ptr(shards, dev, "shards")) || (rc = check_ptr(total, dev, "total"))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  g_launches += 1;
  k_sums_combine<<<(unsigned)((NC + 127) / 128), 128, 0, st>>>(reinterpret_cast<const float2*>(shards), K, NC,
                                                              reinterpret_cast<float2*>(total));
  GN3D_CUDA(cudaGetLastError(), "combine launch");
  return GN3D_OK;
}

extern "C" int gn3d_backward_dx_from_sums(const void* dy, const void* x, const float* mean, const float* rstd,
                                          const float* gamma, const float* sums, int64_t group_count, int64_t N,
                                          int64_t C, int64_t D, int64_t H, int64_t W, int64_t G, gn3d_dtype dtype,
                                          void* dx, float* dgamma, float* dbeta, void* stream) {
  int rc = check_dims(N, C, D, H, W, G);
  if (rc) return rc;
  if (!valid_dtype(dtype)) return arg_fail("unsupported dtype");
  if (group_count < 1) return arg_fail("group_count (elements per group of the whole tensor) must be >= 1");
  const Plan p = make_plan(N, C, D * H * W, G);
  int dev = 0;
  DevInfo* di = nullptr;
  if ((rc = setup(&di, &dev))) return rc;
  if (p.NC == 0) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dgamma && C > 0) GN3D_CUDA(cudaMemsetAsync(dgamma, 0, (size_t)C * sizeof(float), st), "memset");
    if (dbeta && C > 0) GN3D_CUDA(cudaMemsetAsync(dbeta, 0, (size_t)C * sizeof(float), st), "memset");
    return GN3D_OK;
  }
  if (!sums || !mean || !rstd || !aligned8(sums)) return arg_fail("sums (8-byte aligned), mean and rstd are required");
  if ((rc = check_ptr(sums, dev, "sums")) || (rc = check_ptr(mean, dev, "mean")) ||
      (rc = check_ptr(rstd, dev, "rstd")))
    return rc;
  if (p.NC * p.S > 0) {
    if (!dy || !x || !dx) return arg_fail("dy, x and dx are required");
    if (!aligned16(dy) || !aligned16(x) || !aligned16(dx)) return arg_fail("dy, x and dx must be 16-byte aligned");
    if ((rc = check_ptr(dy, dev, "dy")) || (rc = check_ptr(x, dev, "x")) || (rc = check_ptr(dx, dev, "dx")))
      return rc;
  }
  if (gamma && (rc = check_ptr(gamma, dev, "gamma"))) return rc;
  if (dgamma && (rc = check_ptr(dgamma, dev, "dgamma"))) return rc;
  if (dbeta && (rc = check_ptr(dbeta, dev, "dbeta"))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float2* s2 = reinterpret_cast<const float2*>(sums);
  return dtype == GN3D_BF16
             ? launch_dx_from_sums<__nv_bfloat16>(dy, x, mean, rstd, gamma, s2, group_count, p, dx, dgamma, dbeta, st,
                                                  *di)
             : launch_dx_from_sums<float>(dy, x, mean, rstd, gamma, s2, group_count, p, dx, dgamma, dbeta, st, *di);
}

extern "C" int gn3d_stream_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream");
  int dev = 0;
  GN3D_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  DevInfo* di = nullptr;
  int rc = device_info(dev, &di);
  if (rc) return rc;
  uint32_t word = 0;
  GN3D_CUDA(cudaMemcpy(&word, di->status, sizeof(word), cudaMemcpyDeviceToHost), "status read");
  if (word != 0) {
    const uint32_t zero = 0;
    GN3D_CUDA(cudaMemcpy(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice), "status clear");
    return (int)word;
  }
  return GN3D_OK;
}

#ifdef GN3D_TESTING
extern "C" int gn3d_debug_set(int what, long long value) {
  switch (what) {
    case GN3D_DEBUG_PATH:
      if (value < 0 || value > 4) return arg_fail("path: 0 .. 4");
      g_hook_path = value;
      break;
    case GN3D_DEBUG_SPIN_LIMIT:
      if (value < 0) return arg_fail("spin limit >= 0");
      g_hook_spin = value;
      break;
    case GN3D_DEBUG_FORCE_TIMEOUT:
      g_hook_timeout = value ? 1 : 0;
      break;
    case GN3D_DEBUG_LAG:
      if (value < -1 || value > kMaxLag) return arg_fail("lag: -1 .. 8");
      g_hook_lag = value;
      break;
    case GN3D_DEBUG_SLOTS:
      if (value < -1 || value == 0 || value > 32) return arg_fail("slots: -1, 1 .. 32");
      g_hook_slots = value;
      break;
    case GN3D_DEBUG_FAIL_NEXT:
      if (value < 0 || value > 2) return arg_fail("fail next: 0 none, 1 allocation, 2 launch");
      g_inject = (int)value;
      break;
    case GN3D_DEBUG_SHARES:
      if (value < -1 || value > 1) return arg_fail("shares: -1, 0 or 1");
      g_hook_shares = (int)value;
      break;
    case GN3D_DEBUG_RES_HELD:
      if (value < -1) return arg_fail("held units: -1 or >= 0");
      g_hook_rheld = value;
      break;
    case GN3D_DEBUG_RES_PASS:
      if (value < -1 || value == 0) return arg_fail("pass slots: -1 or >= 1");
      g_hook_rpass = value;
      break;
    case GN3D_DEBUG_RES_WINDOW:
      if (value < -1 || value == 0) return arg_fail("window: -1 or >= 1");
      g_hook_window = value;
      break;
    default:
      return arg_fail("unknown debug setting");
  }
  return GN3D_OK;
}

extern "C" int gn3d_debug_get(int what, long long* value) {
  if (!value) return arg_fail("gn3d_debug_get: NULL value");
  switch (what) {
    case GN3D_DEBUG_POOL_USED: {
      int dev = 0;
      GN3D_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
      DevInfo* di = nullptr;
      int rc = device_info(dev, &di);
      if (rc) return rc;
      unsigned long long used = 0;  // the attribute is a 64-bit count
      GN3D_CUDA(cudaMemPoolGetAttribute(di->pool, cudaMemPoolAttrUsedMemCurrent, &used), "pool attribute");
      *value = (long long)used;
      return GN3D_OK;
    }
    default:
      return arg_fail("unknown debug query");
  }
}
#endif  // GN3D_TESTING

extern "C" int gn3d_timing(int on) {
  if (on != 0 && on != 1) return arg_fail("gn3d_timing: 0 or 1");
  std::lock_guard<std::mutex> lk(g_tmu);
  if (on) {
    for (TimedLaunch& t : g_timed) {
      t.dev->free_events.push_back(t.a);
      t.dev->free_events.push_back(t.b);
    }
    g_timed.clear();
    for (int k = 0; k < KK_COUNT; ++k) {
      g_kernel_ms[k] = 0.0;
      g_kernel_n[k] = 0;
    }
  }
  g_timing = on;
  return GN3D_OK;
}

extern "C" const char* gn3d_error_string(int status) {
  switch (status) {
    case GN3D_OK: return "ok";
    case GN3D_ERR_INVALID_ARG: g_msg = "invalid argument: " + g_detail; return g_msg.c_str();
    case GN3D_ERR_DEVICE: g_msg = "device mismatch: " + g_detail; return g_msg.c_str();
    case GN3D_ERR_CUDA: g_msg = "CUDA error: " + g_detail; return g_msg.c_str();
    case GN3D_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    default: return "unknown status";
  }
}

extern "C" uint64_t gn3d_launch_count(void) { return g_launches.load(); }

extern "C" int gn3d_kernel_time(const char* name, double* ms, uint64_t* launches) {
  if (!name || !ms || !launches) return arg_fail("gn3d_kernel_time: NULL argument");
  int kind = -1;
  for (int k = 0; k < KK_COUNT; ++k)
    if (std::string(name) == kKernelNames[k]) kind = k;
  if (kind < 0) return arg_fail("gn3d_kernel_time: unknown kernel name");
  std::lock_guard<std::mutex> lk(g_tmu);
  cudaError_t err = cudaSuccess;
  for (TimedLaunch& t : g_timed) {
    float e = 0.f;
    cudaError_t r = cudaEventSynchronize(t.b);
    if (r == cudaSuccess) r = cudaEventElapsedTime(&e, t.a, t.b);
    if (r == cudaSuccess) {
      g_kernel_ms[t.kind] += e;
      g_kernel_n[t.kind] += 1;
    } else if (err == cudaSuccess) {
      err = r;
    }
    t.dev->free_events.push_back(t.a);
    t.dev->free_events.push_back(t.b);
  }
  g_timed.clear();
  if (err != cudaSuccess) return cuda_fail(err, "kernel timing events");
  *ms = g_kernel_ms[kind];
  *launches = g_kernel_n[kind];
  return GN3D_OK;
}

extern "C" const char* gn3d_version(void) { return "gn3d 0.4.0 sm_103a"; }
