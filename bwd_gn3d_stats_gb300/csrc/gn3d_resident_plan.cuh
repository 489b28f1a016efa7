// gn3d_resident_plan.cuh -- work placement of the group-wave kernels
// (gn3d_resident.cuh): each CTA's share of every group, the order in which a
// CTA's producer and reduction warps walk its shares, with every unit's ring
// slot and phase and its piece record, and the order of its elementwise pass.
// Host-compilable, so the placement can be replayed on the CPU.  Placement
// decides which CTA reads which unit and where the unit is kept between the two
// passes; it never changes a unit, block or group merge.
//
// The group-wave kernels take plans whose rows are whole units (plan_all_full),
// so unit u's body is elements [u * kUnitElems, (u + 1) * kUnitElems).  Walks
// advance by additions only: the divisions are done once per share.
#pragma once
#include <stdint.h>

#include "gn3d_plan.cuh"

namespace gn3d {

// The placement's constants for one launch (computed on the host).
struct ResGeo {
  int P;        // CTAs
  int r;        // upg mod P: the number of shares one unit longer than q
  int64_t q;    // upg / P
  int rh;       // held units per share, at most
  int kh, kp;   // held / pass ring slots
  int recs;     // piece records
};

__host__ __device__ __forceinline__ ResGeo res_geo(const Plan& p, int P, int rh, int kh, int kp, int recs) {
  ResGeo g;
  g.P = P;
  g.q = p.upg / P;
  g.r = (int)(p.upg - g.q * P);
  g.rh = rh;
  g.kh = kh;
  g.kp = kp;
  g.recs = recs;
  return g;
}

// CTA `cta`'s share of group g: units [start, start + n) (global unit indices),
// the last nh of them held.  The r CTAs with one more unit are the cyclic
// interval [a, a + r) with a = g*r mod P: consecutive groups deal the extra
// units out around the CTAs in turn.
struct ResShare {
  int64_t start;
  int n, nh;
};

__host__ __device__ __forceinline__ ResShare res_share(const Plan& p, const ResGeo& G, int64_t g, int cta) {
  const int P = G.P, r = G.r;
  const int a = (int)((uint64_t)((uint32_t)(g % P)) * (uint32_t)r % (uint32_t)P);
  int before;  // extra units among CTAs 0 .. cta-1
  bool extra;
  if (a + r <= P) {
    before = cta - a < 0 ? 0 : (cta - a > r ? r : cta - a);
    extra = cta >= a && cta < a + r;
  } else {
    const int w = a + r - P;  // the interval wraps: [a, P) and [0, w)
    before = (cta < w ? cta : w) + (cta - a > 0 ? cta - a : 0);
    extra = cta >= a || cta < w;
  }
  ResShare s;
  s.start = g * p.upg + (int64_t)cta * G.q + before;
  s.n = (int)G.q + (extra ? 1 : 0);
  s.nh = s.n < G.rh ? s.n : G.rh;
  return s;
}

// The smallest producer lead (window, in units) that lets a CTA load a whole
// share of a group before any of it has been normalized -- which the group's
// statistics need: the largest share, ceil(upg / P).
__host__ __device__ __forceinline__ int64_t res_min_window(const Plan& p, int P) { return (p.upg + P - 1) / P; }

// Unit -> row, in 32 bits when the indices allow it.
__host__ __device__ __forceinline__ int64_t res_row_of(int64_t u, int64_t R) {
  if (u < 0x7FFFFFFF && R < 0x7FFFFFFF) return (int64_t)((uint32_t)u / (uint32_t)R);
  return u / R;
}

// A CTA's sequence: its shares of groups 0, 1, ... in order, pass units first.
// For the current unit: its group, place in the share, index in its row, and
// ring (held or pass) with slot and phase parity.  Per-CTA counts fit in 32
// bits (a CTA holds fewer than 2^31 units of any tensor).
struct ResSeq {
  int64_t g;
  ResShare sh;
  int j;              // unit in the share
  int64_t u;          // the global unit
  int k;              // its index in its row
  int h, q;           // held / pass units before this one in the sequence
  int hs, qs;         // the next held / pass slot
  uint32_t hp, qp;    // its phase parity
  bool end;

  __host__ __device__ __forceinline__ void enter(const Plan& p, const ResGeo& G, int cta) {
    for (; g < p.NG; ++g) {
      sh = res_share(p, G, g, cta);
      if (sh.n > 0) {
        j = 0;
        u = sh.start;
        k = (int)(u - res_row_of(u, p.R) * p.R);
        return;
      }
    }
    end = true;
  }
  __host__ __device__ __forceinline__ void begin(const Plan& p, const ResGeo& G, int cta) {
    g = 0;
    h = q = 0;
    hs = qs = 0;
    hp = qp = 0;
    end = false;
    enter(p, G, cta);
  }
  __host__ __device__ __forceinline__ bool held() const { return j >= sh.n - sh.nh; }
  __host__ __device__ __forceinline__ int64_t unit_index() const { return u; }
  __host__ __device__ __forceinline__ int slot() const { return held() ? hs : qs; }
  __host__ __device__ __forceinline__ uint32_t parity() const { return held() ? hp : qp; }
  __host__ __device__ __forceinline__ int ring_index() const { return held() ? h : q; }
  __host__ __device__ __forceinline__ void next(const Plan& p, const ResGeo& G, int cta) {
    if (held()) {
      ++h;
      if (++hs == G.kh) { hs = 0; hp ^= 1u; }
    } else {
      ++q;
      if (++qs == G.kp) { qs = 0; qp ^= 1u; }
    }
    ++u;
    if (++k == p.R) k = 0;
    if (++j == sh.n) {
      ++g;
      enter(p, G, cta);
    }
  }
  // The current unit's merge block: its first unit, its size, and this share's
  // piece of it (block units lo .. hi).
  __host__ __device__ __forceinline__ void piece_span(const Plan& p, int64_t& b0, int& lo, int& hi, int& bsz) const {
    const int kb = k / kBlockUnits;
    b0 = u - (k - kb * kBlockUnits);
    bsz = block_size(p, kb);
    const int64_t s0 = sh.start, s1 = sh.start + sh.n;
    lo = (int)((s0 > b0 ? s0 : b0) - b0);
    hi = (int)((s1 < b0 + bsz ? s1 : b0 + bsz) - 1 - b0);
  }
  __host__ __device__ __forceinline__ int64_t block(const Plan& p) const {
    return res_row_of(u, p.R) * p.nb + k / kBlockUnits;
  }
};

// One ring's position: slot and phase parity of a use, and how many uses came
// before it.  The kernels walk a share's units with it (additions only).
struct RingPos {
  int slot;
  uint32_t par;
  int uses;
  __host__ __device__ __forceinline__ void at(int i, int n) {  // use i of a ring of n slots
    uses = i;
    slot = i % n;
    par = (uint32_t)((i / n) & 1);
  }
  __host__ __device__ __forceinline__ void step(int d, int n) {  // d <= n
    uses += d;
    slot += d;
    if (slot >= n) {
      slot -= n;
      par ^= 1u;
    }
  }
};

// The first unit of a share's pass (or held) part that reduction warp `warp`
// of kRed reads, when `before` uses of that ring came before the part: the ring
// position before + j must be = warp (mod kRed).
__host__ __device__ __forceinline__ int res_first_of_warp(int before, int warp, int kRed) {
  return (warp - before % kRed + kRed) % kRed;
}

// The elementwise order of a CTA: each share's units from the last to the
// first, advanced `step` positions at a time.  A held unit's slot and parity
// come from the share's first held slot, found once per share.
struct ResElemSeq {
  int64_t g;
  ResShare sh;
  int r;          // position in the share's elementwise order (unit n - 1 - r)
  int64_t hg;     // held units of the sequence before this share
  int hs0;        // slot of the share's first held unit
  uint32_t hp0;   // its phase parity
  bool end;
  __host__ __device__ __forceinline__ void enter(const Plan& p, const ResGeo& G, int cta) {
    for (; g < p.NG; ++g) {
      sh = res_share(p, G, g, cta);
      if (sh.n > 0) {
        hs0 = G.kh > 0 ? (int)(hg % G.kh) : 0;
        hp0 = G.kh > 0 ? (uint32_t)((hg / G.kh) & 1) : 0u;
        return;
      }
    }
    end = true;
  }
  __host__ __device__ __forceinline__ void begin(const Plan& p, const ResGeo& G, int cta) {
    g = 0;
    hg = 0;
    r = 0;
    end = false;
    enter(p, G, cta);
  }
  __host__ __device__ __forceinline__ int j() const { return sh.n - 1 - r; }
  __host__ __device__ __forceinline__ int64_t unit() const { return sh.start + j(); }
  __host__ __device__ __forceinline__ bool held() const { return j() >= sh.n - sh.nh; }
  __host__ __device__ __forceinline__ int64_t hidx() const { return hg + (j() - (sh.n - sh.nh)); }
  // slot and parity of the current (held) unit: at most one wrap past the first
  __host__ __device__ __forceinline__ void held_slot(const ResGeo& G, int& slot, uint32_t& par) const {
    slot = hs0 + (j() - (sh.n - sh.nh));
    par = hp0;
    if (slot >= G.kh) {
      slot -= G.kh;
      par ^= 1u;
    }
  }
  __host__ __device__ __forceinline__ void advance(const Plan& p, const ResGeo& G, int cta, int step) {
    r += step;
    while (!end && r >= sh.n) {
      r -= sh.n;
      hg += sh.nh;
      ++g;
      enter(p, G, cta);
    }
  }
};

}  // namespace gn3d
