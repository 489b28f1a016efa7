// gn3d_cluster.cuh -- one launch per direction for groups that one thread-block
// cluster holds in shared memory (the small sites of a volumetric UNet:
// 512 channels at 16^3, 256 at 32^3, and shapes like them).
//
// One cluster per group (the split is in gn3d_cluster_plan.cuh).  Each CTA
// bulk-copies all of its units into shared memory at once, one mbarrier per
// unit.  Then, with the streaming kernels' arithmetic throughout:
//   1. each warp computes its units' results (moments forward, S1 and S2
//      backward) into shared memory;
//   2. each warp merges whole blocks of the CTA and stores the block results
//      into CTA 0's shared memory (distributed shared memory);
//   3. after a cluster barrier, warp 0 of CTA 0 merges the group exactly as the
//      streaming kernels' group step does and stores what every CTA needs into
//      each CTA's shared memory;
//   4. after a second barrier, every CTA normalizes (or forms dx for) its units
//      from the copies it still holds.
// x (and dy) are read once from HBM and y (dx) written once; the group merge
// goes through distributed shared memory instead of global counters.  Every
// wait on a copy is bounded; a CTA whose wait gave up reports
// GN3D_ERR_TIMEOUT, and every CTA still meets both cluster barriers, so the
// cluster never waits on a CTA that left.
#pragma once
#include "gn3d_cluster_plan.cuh"
#include "gn3d_device.cuh"
#include "gn3d_sync.cuh"

namespace gn3d {

// A word nothing writes: the forced-timeout test of the cluster kernels waits on it.
__device__ uint32_t g_cluster_never = 0;

__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return (int)r;
}

// Every thread of every CTA of the cluster: the CTA's earlier memory operations
// (shared memory of other CTAs included) are released, the others' acquired.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address of this CTA's shared variable *p in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void* p, int rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void st_cluster(uint32_t a, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, const Part& v) {
  st_cluster(a, make_float4(v.m1, v.m2, __int_as_float(v.n), v.cn));
}
__device__ __forceinline__ void st_cluster(uint32_t a, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// A CTA's shared memory: its units' data (kTensors tensors of a unit, unit by
// unit), one mbarrier per unit, the unit results, the group's block results
// (filled in CTA 0 only) and, from warp 0 of CTA 0, the group's coefficients
// and whether every copy of the cluster arrived.
template <class T, int kTensors, class V>
struct ClusterLayout {
  static constexpr int kTensorBytes = kUnitElems * (int)sizeof(T);
  static constexpr int kUnitBytes = kTensors * kTensorBytes;
  static __host__ __device__ int64_t r16(int64_t b) { return (b + 15) / 16 * 16; }
  static __host__ __device__ int64_t off_bar(int upc) { return (int64_t)upc * kUnitBytes; }
  static __host__ __device__ int64_t off_unit(int upc) { return r16(off_bar(upc) + 8 * (int64_t)upc); }
  static __host__ __device__ int64_t off_blk(int upc) { return r16(off_unit(upc) + (int64_t)sizeof(V) * upc); }
  static __host__ __device__ int64_t off_coef(int upc, int64_t nbg) { return r16(off_blk(upc) + (int64_t)sizeof(V) * nbg); }
  static __host__ __device__ int64_t bytes(int upc, int64_t nbg) { return off_coef(upc, nbg) + 32; }
  unsigned char* data;
  uint64_t* bar;
  V* unit;
  V* blk;
  float4* coef;
  int* ok;
  __device__ __forceinline__ void carve(unsigned char* s, int upc, int64_t nbg) {
    data = s;
    bar = reinterpret_cast<uint64_t*>(s + off_bar(upc));
    unit = reinterpret_cast<V*>(s + off_unit(upc));
    blk = reinterpret_cast<V*>(s + off_blk(upc));
    coef = reinterpret_cast<float4*>(s + off_coef(upc, nbg));
    ok = reinterpret_cast<int*>(s + off_coef(upc, nbg) + 16);
  }
};

// The CTA's share: group g, blocks [b0, b1), nu units.
struct ClusterShare {
  int r;
  int64_t g, b0, b1;
  int nu;
  __device__ __forceinline__ ClusterShare(const Plan& p, const ClusterGeo& c) {
    r = cluster_rank();
    g = blockIdx.x / c.cs;
    b0 = cl_block_begin(c.nbg, c.cs, r);
    b1 = cl_block_begin(c.nbg, c.cs, r + 1);
    nu = cl_units(p, b0, b1);
  }
  // unit j of the CTA: its element range
  __device__ __forceinline__ URange range(const Plan& p, int j) const {
    int64_t b, row, k;
    int ui;
    cl_unit(p, b0, j, b, ui);
    cl_row_k(p, g, b, ui, row, k);
    return full_range(p, row, k);
  }
};

// Barriers set up, then every unit's bulk copies in flight at once (issued by
// lane 0 of the warp that reads the unit), then the first cluster barrier:
// every CTA of the cluster has started before any writes another's shared
// memory.
template <int kTensors, class T, class Layout>
__device__ __forceinline__ void cluster_load(const Plan& p, const ClusterShare& sh, const Layout& s,
                                             const T* const* src) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int j = 0; j < sh.nu; ++j) mbar_init(&s.bar[j], 1);
    *s.ok = 1;
    fence_mbar_init();
  }
  __syncthreads();
  for (int j = warp; j < sh.nu; j += kClusterWarps) {
    if (lane == 0) {
      const URange q = sh.range(p, j);
      unsigned char* dst = s.data + (size_t)j * Layout::kUnitBytes;
      mbar_arrive_expect_tx(&s.bar[j], (uint32_t)Layout::kUnitBytes);
#pragma unroll
      for (int t = 0; t < kTensors; ++t)
        bulk_g2s(dst + t * Layout::kTensorBytes, src[t] + q.b0, (uint32_t)Layout::kTensorBytes, &s.bar[j]);
    }
  }
  cluster_sync_all();
}

// Unit results (fn(j, data) for each of the warp's units), then the CTA's
// blocks merged (merge(values of the block's units, lanes past its size get
// `empty`)) into CTA 0's block array, then the second cluster barrier.  A
// failed wait marks the cluster's result invalid in CTA 0.
template <class Layout, class V, class Unit, class Merge>
__device__ __forceinline__ void cluster_reduce(const Plan& p, const ClusterShare& sh, const Layout& s,
                                               unsigned long long spin, uint32_t* status, V empty, Unit unit,
                                               Merge merge) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool failed = false;
  for (int j = warp; j < sh.nu; j += kClusterWarps) {
    // every lane observes the copy's completion itself (its acquire), and the
    // warp decides together whether to use the unit
    if (!__all_sync(kFull, mbar_wait_bounded(&s.bar[j], 0, spin))) {
      failed = true;
      continue;
    }
    const V v = unit(j, s.data + (size_t)j * Layout::kUnitBytes);
    if (lane == 0) s.unit[j] = v;
  }
  if (__any_sync(kFull, failed) && lane == 0) {
    atomicExch(status, 4u);  // GN3D_ERR_TIMEOUT
    st_cluster(cluster_map(s.ok, 0), 0);
  }
  __syncthreads();
  int start = 0;  // CTA-local index of block kb's first unit
  int kb0 = 0;
  for (int kb = warp; kb < (int)(sh.b1 - sh.b0); kb += kClusterWarps) {
    for (; kb0 < kb; ++kb0) start += cl_block_units(p, sh.b0 + kb0);
    const int bsz = cl_block_units(p, sh.b0 + kb);
    const V a = lane < bsz ? s.unit[start + lane] : empty;
    const V m = merge(a);
    if (lane == 0) st_cluster(cluster_map(&s.blk[sh.b0 + kb], 0), m);
  }
  cluster_sync_all();
}

// Warp 0 of CTA 0: whether the cluster's copies all arrived (and, forced for
// the failure-path test, a bounded wait on a word nothing writes).
__device__ __forceinline__ bool cluster_group_ok(const int* ok, unsigned long long spin, uint32_t* status,
                                                 int force_timeout) {
  const int lane = threadIdx.x & 31;
  bool good = *(volatile const int*)ok != 0;
  if (good && force_timeout) {
    if (lane == 0) {
      const volatile uint32_t* w = &g_cluster_never;
      unsigned long long it = 0;
      while (*w == 0u && it < spin) ++it;
      good = *w != 0u;
      if (!good) atomicExch(status, 4u);  // GN3D_ERR_TIMEOUT
    }
    good = __shfl_sync(kFull, good ? 1 : 0, 0) != 0;
  }
  return good;
}

// After a failed wait: wait (bounded, with the drain budget) for the copies
// still in flight into this CTA's shared memory, before it exits.
template <class Layout>
__device__ __forceinline__ void cluster_drain(const ClusterShare& sh, const Layout& s) {
  const int warp = threadIdx.x >> 5;
  for (int j = warp; j < sh.nu; j += kClusterWarps) mbar_wait_bounded(&s.bar[j], 0, kDrainPolls);
}

// ------------------------------------------------------------- forward
template <class TI, class TO, bool kRelu>
__global__ void __launch_bounds__(32 * kClusterWarps, 1)
    k_fwd_cluster(const TI* __restrict__ x, TO* __restrict__ y, Plan p, ClusterGeo c, float eps,
                  const float* __restrict__ gamma, const float* __restrict__ beta, float* mean_out, float* rstd_out,
                  unsigned long long spin, uint32_t* status, int force_timeout) {
  extern __shared__ __align__(128) unsigned char smem[];
  using L = ClusterLayout<TI, 1, Part>;
  L s;
  s.carve(smem, c.upc, c.nbg);
  const ClusterShare sh(p, c);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TI* src[1] = {x};
  cluster_load<1>(p, sh, s, src);
  const Part empty{0.f, 0.f, 0, 0.f};
  cluster_reduce(
      p, sh, s, spin, status, empty,
      [&](int j, const unsigned char* d) {
        const URange q = sh.range(p, j);
        if constexpr (Vec<TI>::kRaw == 1) {
          RegView<TI> v;
          v.template load_full<FromShared>(reinterpret_cast<const TI*>(d));
          return unit_moments_sv<true, TI>(v, 0.f, q);
        } else {
          return unit_moments_sv<true, TI>(MemView<TI, FromShared>{reinterpret_cast<const TI*>(d), kUnitVecs}, 0.f, q);
        }
      },
      [](const Part& a) { return merge_block(a); });
  if (sh.r == 0 && warp == 0) {  // the group step of the streaming statistics kernel
    const bool good = cluster_group_ok(s.ok, spin, status, force_timeout);
    float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
    if (good) {
      const Part gp = merge_group_part_from([&](int64_t i) { return s.blk[i]; }, c.nbg, p.M);
      st = group_stats(gp, p.M, eps);
      if (lane == 0) {
        if (mean_out) mean_out[sh.g] = fadd(st.x, st.y);
        if (rstd_out) rstd_out[sh.g] = st.z;
      }
    }
    if (lane < c.cs) {
      st_cluster(cluster_map(s.coef, lane), st);
      st_cluster(cluster_map(s.ok, lane), good ? 1 : 0);
    }
  }
  cluster_sync_all();  // no shared memory of another CTA is touched after this
  if (*(volatile int*)s.ok) {
    const float4 st = *s.coef;
    for (int j = warp; j < sh.nu; j += kClusterWarps) {
      const URange q = sh.range(p, j);
      const int64_t ch = channel_of(q.row, p.C);
      const float gm = gamma ? gamma[ch] : 1.f, bt = beta ? beta[ch] : 0.f;
      const TI* d = reinterpret_cast<const TI*>(s.data + (size_t)j * L::kUnitBytes);
      if constexpr (Vec<TI>::kRaw == 1) {
        RegView<TI> v;
        v.template load_full<FromShared>(d);
        fwd_norm<true, TI, TO, RegView<TI>, kRelu>(v, x, y, q, st, gm, bt);
      } else {
        fwd_norm<true, TI, TO, MemView<TI, FromShared>, kRelu>(MemView<TI, FromShared>{d, kUnitVecs}, x, y, q, st,
                                                               gm, bt);
      }
    }
  } else {
    cluster_drain(sh, s);
  }
}

// ------------------------------------------------------------- backward
template <class T>
__global__ void __launch_bounds__(32 * kClusterWarps, 1)
    k_bwd_cluster(const T* __restrict__ dy, const T* __restrict__ x, T* __restrict__ dx, Plan p, ClusterGeo c,
                  const float* __restrict__ mean, const float* __restrict__ rstd, const float* __restrict__ gamma,
                  float2* rows, uint32_t* done, float* dgamma, float* dbeta, unsigned long long spin,
                  uint32_t* status, int force_timeout) {
  extern __shared__ __align__(128) unsigned char smem[];
  using L = ClusterLayout<T, 2, float2>;
  L s;
  s.carve(smem, c.upc, c.nbg);
  const ClusterShare sh(p, c);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* src[2] = {x, dy};
  cluster_load<2>(p, sh, s, src);
  const float mu = mean[sh.g];
  cluster_reduce(
      p, sh, s, spin, status, make_float2(0.f, 0.f),
      [&](int j, const unsigned char* d) {
        const URange q = sh.range(p, j);
        const f2 z2 = f2_splat(0.f);
        f2 a1[4] = {z2, z2, z2, z2};
        f2 a2[4] = {z2, z2, z2, z2};
        bwd_accum<true, T>(MemView<T, FromShared>{reinterpret_cast<const T*>(d), kUnitVecs},
                           MemView<T, FromShared>{reinterpret_cast<const T*>(d + L::kTensorBytes), kUnitVecs}, 0,
                           kVecPerLane, mu, a1, a2);
        return bwd_finish_sv<true>(a1, a2, BwdScalar{0.f, 0.f}, q, mu);
      },
      [](const float2& a) { return warp_sum2(a.x, a.y); });
  if (sh.r == 0 && warp == 0) {  // the group step of the streaming reduction kernel
    const bool good = cluster_group_ok(s.ok, spin, status, force_timeout);
    float2 ab = make_float2(0.f, 0.f);
    if (good) {
      float2* grow = rows + sh.g * p.Cg;
      ab = bwd_group_from(
          p, sh.g, rstd, gamma, [&](int64_t i) { return s.blk[i]; }, [&](int64_t cl, float2 t) { grow[cl] = t; });
    }
    if (lane < c.cs) {
      st_cluster(cluster_map(s.coef, lane), make_float4(ab.x, ab.y, mu, rstd[sh.g]));
      st_cluster(cluster_map(s.ok, lane), good ? 1 : 0);
    }
    // every lane's row stores before the arrival; the cluster completing the
    // last group forms dgamma and dbeta in n order from every group's rows
    __threadfence();
    __syncwarp();
    if (warp_arrive_last(done, (uint32_t)p.NG)) bwd_param_grads(p, rstd, rows, dgamma, dbeta);
  }
  cluster_sync_all();  // no shared memory of another CTA is touched after this
  if (*(volatile int*)s.ok) {
    const float4 k4 = *s.coef;
    const DxCoef kc{k4.z, k4.w, k4.x, k4.y, p.M == 1};
    for (int j = warp; j < sh.nu; j += kClusterWarps) {
      const URange q = sh.range(p, j);
      const float gm = gamma ? gamma[channel_of(q.row, p.C)] : 1.f;
      const unsigned char* d = s.data + (size_t)j * L::kUnitBytes;
      bwd_norm<true, T>(MemView<T, FromShared>{reinterpret_cast<const T*>(d), kUnitVecs},
                        MemView<T, FromShared>{reinterpret_cast<const T*>(d + L::kTensorBytes), kUnitVecs}, x, dy,
                        dx, q, kc, gm);
    }
  } else {
    cluster_drain(sh, s);
  }
}

}  // namespace gn3d
