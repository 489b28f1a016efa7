// gn3d_plan.cuh -- the launch plan: how a GroupNorm shape is cut into work units.
//
// The plan is a pure function of (N, C, D*H*W, G).  It never looks at the dtype,
// the GPU's SM count or the grid a kernel happens to be launched with, so the
// order of every floating-point reduction -- and therefore every output bit --
// depends on the shape alone (ScaFFold PR #105: "_plan takes no dtype"; PR #93's
// launch-folding commit: grid, split count, tiles and reduction order are pure
// functions of the shape).
//
// Units.  Row (n, c) is the contiguous span of S = D*H*W elements at flat offset
// (n*C + c)*S.  Each row is cut into R = ceil(S / kUnitElems) units.  Inside a
// row, the "body" is the part between the first and last flat index that is a
// multiple of 8 (kVec); body unit k covers body elements [k*kUnitElems,
// (k+1)*kUnitElems), read as 8-element vectors (16 B of bf16, 32 B of fp32).
// The up to 7 elements before the body (the head) belong to unit 0 and the up to
// 7 after it (the tail) to unit R-1; a row too short to hold an aligned 8-block
// is all head.  Groups are Cg = C/G consecutive rows, so group (n, g) owns the
// Cg*R consecutive units starting at ((n*C + g*Cg) * R).
//
// Reduction tree.  One warp reduces one unit: lane l takes body vectors l,
// l+32, l+64, ... and keeps one running sum per vector position (8 chains), the
// chains meet in a fixed pairwise tree, the lane's head/tail scalar (scalar l)
// is added, and an xor butterfly sums the lanes.  Within a row, units form
// blocks of kBlockUnits consecutive units (the last block of a row may be
// shorter); a block's unit partials are merged one per lane with the same
// butterfly.  A group merges its blocks row by row in a fixed order.
#pragma once
#include <stdint.h>

namespace gn3d {

constexpr int kVec = 8;             // elements per vector
constexpr int kUnitElems = 4096;    // body elements per unit (multiple of kVec)
constexpr int kUnitVecs = kUnitElems / kVec;  // 512
constexpr int kVecPerLane = kUnitVecs / 32;   // 16
constexpr int kBlockUnits = 16;     // units per merge block (one per lane; <= 32)
constexpr int kMaxScalars = 14;     // head + tail elements of one unit, at most

struct Plan {
  int64_t N, C, S, G;
  int64_t Cg;     // channels per group
  int64_t M;      // elements per group = Cg * S
  int64_t NG;     // N * G groups
  int64_t NC;     // N * C rows
  int64_t R;      // units per row
  int64_t nb;     // merge blocks per row = ceil(R / kBlockUnits)
  int64_t upg;    // units per group = Cg * R
  int64_t units;  // total units = NC * R
};

inline Plan make_plan(int64_t N, int64_t C, int64_t S, int64_t G) {
  Plan p;
  p.N = N; p.C = C; p.S = S; p.G = G;
  p.Cg = C / G;
  p.M = p.Cg * S;
  p.NG = N * G;
  p.NC = N * C;
  p.R = S > 0 ? (S + kUnitElems - 1) / kUnitElems : 0;
  p.nb = (p.R + kBlockUnits - 1) / kBlockUnits;
  p.upg = p.Cg * p.R;
  p.units = p.NC * p.R;
  return p;
}

// Element ranges of one unit (flat indices into the NCDHW tensor).
struct URange {
  int64_t row;
  int64_t h0, h1;   // head scalars (or the whole row when it has no body)
  int64_t b0, b1;   // body: multiple-of-8 aligned, possibly empty
  int64_t t0, t1;   // tail scalars
  int n;            // element count
};

// Unit k of row `row` (u = row * R + k).
__host__ __device__ inline URange unit_range_rk(const Plan& p, int64_t row, int64_t k) {
  URange q;
  const int64_t r0 = row * p.S, r1 = r0 + p.S;
  const int64_t bl = (r0 + kVec - 1) & ~(int64_t)(kVec - 1);
  const int64_t bh = r1 & ~(int64_t)(kVec - 1);
  q.row = row;
  if (bh <= bl) {
    q.h0 = r0; q.h1 = (k == 0) ? r1 : r0;
    q.b0 = q.b1 = r0;
    q.t0 = q.t1 = r1;
  } else {
    q.h0 = r0; q.h1 = (k == 0) ? bl : r0;
    const int64_t lo = bl + k * (int64_t)kUnitElems, hi = lo + kUnitElems;
    q.b0 = lo < bh ? lo : bh;
    q.b1 = hi < bh ? hi : bh;
    q.t0 = bh; q.t1 = (k == p.R - 1) ? r1 : bh;
  }
  q.n = (int)((q.h1 - q.h0) + (q.b1 - q.b0) + (q.t1 - q.t0));
  return q;
}

__host__ __device__ inline URange unit_range(const Plan& p, int64_t u) {
  const int64_t row = u / p.R;
  return unit_range_rk(p, row, u - row * p.R);
}

// A unit whose 4096 elements are all body (no head or tail scalars).
__host__ __device__ inline bool unit_is_full(const URange& q) {
  return q.n == kUnitElems && q.b1 - q.b0 == kUnitElems;
}

// Every unit of the plan is full: rows are whole multiples of kUnitElems, so
// every row also starts on a vector boundary.
__host__ __device__ inline bool plan_all_full(const Plan& p) { return p.S > 0 && p.S % kUnitElems == 0; }

// Unit k of row `row` when plan_all_full (the same range unit_range_rk gives).
__host__ __device__ inline URange full_range(const Plan& p, int64_t row, int64_t k) {
  URange q;
  q.row = row;
  q.b0 = row * p.S + k * (int64_t)kUnitElems;
  q.b1 = q.b0 + kUnitElems;
  q.h0 = q.h1 = row * p.S;
  q.t0 = q.t1 = row * p.S + p.S;
  q.n = kUnitElems;
  return q;
}

// Flat index of scalar number s (0 <= s < head+tail) of a unit: head first, then tail.
__host__ __device__ inline int64_t scalar_index(const URange& q, int s) {
  const int64_t nh = q.h1 - q.h0;
  return s < nh ? q.h0 + s : q.t0 + (s - nh);
}

__host__ __device__ inline int scalar_count(const URange& q) {
  return (int)((q.h1 - q.h0) + (q.t1 - q.t0));
}

// Merge block of unit (row, k): block id row * nb + k / kBlockUnits, and its size.
__host__ __device__ inline int64_t block_of(const Plan& p, int64_t row, int64_t k) {
  return row * p.nb + k / kBlockUnits;
}

__host__ __device__ inline int block_size(const Plan& p, int64_t kb) {
  const int64_t first = kb * kBlockUnits, rest = p.R - first;
  return (int)(rest < kBlockUnits ? rest : kBlockUnits);
}

// Work shares of the streaming kernels, in one of two layouts:
//   strided blocks (cut = false): worker w of W takes whole merge blocks w,
//     w + W, w + 2W, ...; no block is ever split;
//   unit shares (cut = true): worker w takes the contiguous units
//     [units*w/W, units*(w+1)/W) in (row, k) order, so shares differ by at most
//     one unit; a block cut by a share boundary is merged by whichever worker
//     completes it.
// Shares decide placement only: every unit, block and group merge is the same
// whatever W and the layout are.
__host__ __device__ inline int64_t share_begin(const Plan& p, int64_t w, int64_t nw) { return p.units * w / nw; }

// The first unit of unit u's merge block, and one past its last.
__host__ __device__ inline void block_span(const Plan& p, int64_t u, int64_t& b0, int64_t& b1) {
  const int64_t row = u / p.R, k = u - row * p.R, kb0 = k / kBlockUnits * kBlockUnits;
  b0 = row * p.R + kb0;
  b1 = row * p.R + (kb0 + kBlockUnits < p.R ? kb0 + kBlockUnits : p.R);
}

// Where a unit share's walk starts.  When a block is cut at the share's end,
// the walk takes that piece first and then wraps to the share's start: both
// cut pieces (their merges need global round trips between workers) are then
// done early, and the walk ends on whole blocks, merged in registers.
__host__ __device__ inline int64_t share_walk_start(const Plan& p, int64_t u0, int64_t u1) {
  if (u0 >= u1) return u0;
  int64_t lb, le;
  block_span(p, u1 - 1, lb, le);
  return (le > u1 && lb > u0) ? lb : u0;
}

// A worker's units in the reduction kernels' order.  Unit shares: a .. u1-1,
// then u0 .. a-1 (a = share_walk_start).  Strided blocks: each block's units
// in order, blocks w, w + W, ...  A block ends where ui() == its size - 1 or,
// in a unit share, at u1 - 1; it is cut when this worker holds only part of it.
struct UnitWalk {
  int64_t u, row, k;     // the current unit, its row and index in the row
  int64_t u0, u1, a;     // unit share [u0, u1), walk start a (strided: 0, max, 0)
  int64_t b, bstride;    // strided: the current block, the block stride
  bool cut, end;
  __host__ __device__ void go(const Plan& p, int64_t v) {
    u = v;
    row = v / p.R;
    k = v - row * p.R;
  }
  __host__ __device__ void go_block(const Plan& p) {
    row = b / p.nb;
    k = (b - row * p.nb) * kBlockUnits;
    u = row * p.R + k;
  }
  __host__ __device__ void set(const Plan& p, int64_t w, int64_t nw, bool cut_) {
    cut = cut_;
    u = row = k = 0;
    b = w;
    bstride = nw;
    if (cut) {
      u0 = share_begin(p, w, nw);
      u1 = share_begin(p, w + 1, nw);
      a = share_walk_start(p, u0, u1);
      end = u0 >= u1;
      if (!end) go(p, a);
    } else {
      u0 = a = 0;
      u1 = INT64_MAX;
      end = b >= p.NC * p.nb;
      if (!end) go_block(p);
    }
  }
  __host__ __device__ void next(const Plan& p) {
    ++u;
    ++k;
    if (!cut) {
      if (k % kBlockUnits == 0 || k == p.R) {  // the block is done
        b += bstride;
        end = b >= p.NC * p.nb;
        if (!end) go_block(p);
      }
      return;
    }
    if (k == p.R) {
      k = 0;
      ++row;
    }
    if (u == u1) {
      if (a == u0) end = true;
      else go(p, u0);  // wrap to the share's start
    } else if (u == a) {
      end = true;
    }
  }
  __host__ __device__ int ui() const { return (int)(k % kBlockUnits); }  // unit in its block
  __host__ __device__ int64_t kb() const { return k / kBlockUnits; }     // block in its row
};

// A worker's units in the elementwise kernels' order, `step` warps splitting
// them (this one starts `skip` in), so that what the reduction read last is
// read again first.  Unit shares: positions skip, skip+step, ... of the reverse
// of UnitWalk's order.  Strided blocks: the blocks from the last one down, in
// each block units size-1-skip, size-1-skip-step, ... down.
struct UnitWalkDown {
  int64_t u, row, k;       // the current unit
  int64_t u0, u1, a, i;    // unit shares: the share, walk start, position
  int64_t b, b0, bstride;  // strided: the current block, the first block, the stride
  int64_t kb;              // strided: the current block's index in its row
  int ui, skip, step;
  bool cut, done;
  __host__ __device__ void at_share(const Plan& p) {
    u = i < a - u0 ? a - 1 - i : u1 - 1 - (i - (a - u0));
    row = u / p.R;
    k = u - row * p.R;
  }
  // strided: block b, or the next one down that holds a unit for this warp
  __host__ __device__ void enter_block(const Plan& p) {
    for (; b >= b0; b -= bstride) {
      row = b / p.nb;
      kb = b - row * p.nb;
      ui = block_size(p, kb) - 1 - skip;
      if (ui >= 0) {
        k = kb * kBlockUnits + ui;
        u = row * p.R + k;
        return;
      }
    }
    done = true;
  }
  __host__ __device__ void set(const Plan& p, int64_t w, int64_t nw, bool cut_, int skip_, int step_) {
    cut = cut_;
    skip = skip_;
    step = step_;
    u = row = k = kb = 0;
    ui = 0;
    done = false;
    if (cut) {
      u0 = share_begin(p, w, nw);
      u1 = share_begin(p, w + 1, nw);
      a = share_walk_start(p, u0, u1);
      i = skip;
      done = i >= u1 - u0;
      if (!done) at_share(p);
    } else {
      const int64_t nblk = p.NC * p.nb;
      b0 = w;
      bstride = nw;
      b = b0 < nblk ? b0 + (nblk - 1 - b0) / nw * nw : -1;  // the last block
      enter_block(p);
    }
  }
  __host__ __device__ bool end() const { return done; }
  __host__ __device__ void next(const Plan& p) {
    if (cut) {
      i += step;
      done = i >= u1 - u0;
      if (!done) at_share(p);
    } else if (ui - step >= 0) {
      ui -= step;
      k -= step;
      u -= step;
    } else {
      b -= bstride;
      enter_block(p);
    }
  }
};

// The elementwise kernels' units under strided blocks, spread evenly over all
// their warps, freshest first.  Reduction worker v (of Wr) reads its blocks v,
// v + Wr, ... in rounds, each block's units in order, so unit p of a block of
// round r is read at about r*kBlockUnits + p.  Items enumerate (round from the
// last, position p from kBlockUnits - 1 down, block of the round): what the
// reduction read last comes first, while it is still in L2.  Warp w of W takes
// items w, w + W, ... (positions past a short block's size are skipped).
// Placement only: no result depends on it.
struct UnitWalkFresh {
  int64_t u, row, k;  // the current unit
  int64_t i, W, Wr, nitems, nrounds, nblk;
  bool done;
  __host__ __device__ bool item(const Plan& p) {  // the unit of item i, if it exists
    const int64_t per = Wr * kBlockUnits;
    const int64_t r = nrounds - 1 - i / per, rem = i % per;
    const int64_t pos = kBlockUnits - 1 - rem / Wr;
    const int64_t b = r * Wr + rem % Wr;
    if (b >= nblk) return false;
    const int64_t kb = b % p.nb;
    if (pos >= block_size(p, kb)) return false;
    row = b / p.nb;
    k = kb * kBlockUnits + pos;
    u = row * p.R + k;
    return true;
  }
  __host__ __device__ void seek(const Plan& p) {
    for (; i < nitems; i += W)
      if (item(p)) return;
    done = true;
  }
  __host__ __device__ void set(const Plan& p, int64_t w, int64_t W_, int64_t Wr_) {
    W = W_;
    Wr = Wr_;
    nblk = p.NC * p.nb;
    nrounds = (nblk + Wr - 1) / Wr;
    nitems = nrounds * Wr * kBlockUnits;
    i = w;
    u = row = k = 0;
    done = false;
    seek(p);
  }
  __host__ __device__ bool end() const { return done; }
  __host__ __device__ void next(const Plan& p) {
    i += W;
    seek(p);
  }
};

// Unit shares pay two cut blocks per worker and suit large tensors (contiguous
// runs per SM); they are used when shares hold two merge blocks or more on
// average, and when there are so few merge blocks (a third of the workers or
// fewer) that strided blocks would leave most warps idle and the rest each a
// long serial run; strided blocks otherwise.
__host__ __device__ inline bool use_unit_shares(const Plan& p, int64_t nw) {
  const int64_t nblk = p.NC * p.nb;
  return p.units >= 2 * kBlockUnits * nw || (3 * nblk <= nw && p.units > nblk);
}

}  // namespace gn3d
