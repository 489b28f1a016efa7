// gn3d_cluster_plan.cuh -- the work split of the cluster kernels (host and
// device code; the CPU walk in tests/plan_walk.cpp checks it).
//
// One thread-block cluster per group: its cs CTAs split the group's merge
// blocks (row-major: row cl of the group, block kb of the row, at index
// cl*nb + kb) into contiguous runs, CTA r taking blocks
// [nbg*r/cs, nbg*(r+1)/cs).  A CTA's units are its blocks' units in block
// order; its warp w takes units w, w + kClusterWarps, ....  The split decides
// only where a unit is computed: every unit, block and group merge is the one
// the streaming kernels perform, so the results are the same bits.
#pragma once
#include "gn3d_plan.cuh"

namespace gn3d {

constexpr int kClusterWarps = 8;
constexpr int kClusterMaxCTAs = 16;  // non-portable cluster size (GB300 allows 16)

struct ClusterGeo {
  int cs;       // CTAs per cluster (one cluster per group)
  int upc;      // the most units any CTA of a cluster holds
  int64_t nbg;  // merge blocks per group (Cg * nb)
};

__host__ __device__ inline int64_t cl_block_begin(int64_t nbg, int cs, int r) { return nbg * r / cs; }

// Units of group-local block b.
__host__ __device__ inline int cl_block_units(const Plan& p, int64_t b) { return block_size(p, b % p.nb); }

// Units of the blocks [b0, b1).
__host__ __device__ inline int cl_units(const Plan& p, int64_t b0, int64_t b1) {
  int n = 0;
  for (int64_t b = b0; b < b1; ++b) n += cl_block_units(p, b);
  return n;
}

// CTA-local unit j of the blocks starting at b0: its group-local block b and
// its unit ui in the block.
__host__ __device__ inline void cl_unit(const Plan& p, int64_t b0, int j, int64_t& b, int& ui) {
  b = b0;
  for (int n = cl_block_units(p, b); j >= n; n = cl_block_units(p, b)) {
    j -= n;
    ++b;
  }
  ui = j;
}

// The row (n*C + c) and unit-in-row of group g's block b, unit ui.
__host__ __device__ inline void cl_row_k(const Plan& p, int64_t g, int64_t b, int ui, int64_t& row, int64_t& k) {
  row = g * p.Cg + b / p.nb;
  k = (b % p.nb) * kBlockUnits + ui;
}

// The cluster size: the largest power of two, at most kClusterMaxCTAs, that
// leaves every CTA at least one block and, on average, two units; and the most
// units a CTA of it then holds.
inline ClusterGeo cluster_geo(const Plan& p) {
  ClusterGeo c;
  c.nbg = p.Cg * p.nb;
  int cs = 1;
  while (cs < kClusterMaxCTAs && 2 * cs <= c.nbg && 4 * cs <= p.upg) cs *= 2;
  c.cs = cs;
  c.upc = 0;
  for (int r = 0; r < cs; ++r) {
    const int n = cl_units(p, cl_block_begin(c.nbg, cs, r), cl_block_begin(c.nbg, cs, r + 1));
    if (n > c.upc) c.upc = n;
  }
  return c;
}

}  // namespace gn3d
