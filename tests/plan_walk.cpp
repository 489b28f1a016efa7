// CPU walk of the launch plans' index arithmetic (host logic test, built and run
// by tests/test_plan_walk.py).  For many shapes it replays what the kernels touch:
//   NCDHW plan (gn3d_plan.cuh): every element of every row belongs to exactly one
//     unit (8-element body vectors at aligned offsets, or head/tail scalars),
//     units tile merge blocks, and every element is inside the tensor;
//   NDHWC plan (gn3d_ndhwc_plan.cuh): every element is read by exactly one lane
//     vector in a unit, vectors are 8-aligned and inside the unit's position range
//     and channel range; the lp lanes of a channel cover the unit's positions;
//     group pieces tile each range's channels and every group's pieces exist; the
//     ring parts (n_ring_part) of one-range shapes are aligned, inside the tensor,
//     fit a slot, and hold exactly each lane's vectors of their steps.
//   work shares (gn3d_plan.cuh), strided blocks and unit shares: the reduction
//     kernels' walks visit every unit once, whole and cut merge blocks complete
//     exactly once, and the elementwise kernels' walks cover every unit once.
// Prints "ok <shapes>" or the first failure.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#include "../bwd_gn3d_stats_gb300/csrc/gn3d_plan.cuh"
#include "../bwd_gn3d_stats_gb300/csrc/gn3d_ndhwc_plan.cuh"

using namespace gn3d;

static const char* g_what = "";
static int64_t g_rotated = 0;  // shares whose walk starts with the piece cut at their end
static int64_t g_shape[4];
#define CHECK(c)                                                                                     \
  do {                                                                                               \
    if (!(c)) {                                                                                      \
      printf("FAIL %s: %s (line %d) at N=%lld C=%lld S=%lld G=%lld\n", g_what, #c, __LINE__,          \
             (long long)g_shape[0], (long long)g_shape[1], (long long)g_shape[2], (long long)g_shape[3]); \
      exit(1);                                                                                       \
    }                                                                                                \
  } while (0)

static void walk_ncdhw(int64_t N, int64_t C, int64_t S, int64_t G) {
  g_what = "ncdhw";
  const Plan p = make_plan(N, C, S, G);
  const int64_t numel = N * C * S;
  std::vector<uint8_t> cover(numel, 0);
  for (int64_t row = 0; row < p.NC; ++row) {
    int64_t units_in_blocks = 0;
    for (int64_t kb = 0; kb < p.nb; ++kb) units_in_blocks += block_size(p, kb);
    CHECK(units_in_blocks == p.R);
    for (int64_t k = 0; k < p.R; ++k) {
      const URange q = unit_range_rk(p, row, k);
      CHECK(q.b0 <= q.b1);
      if (q.b1 > q.b0) CHECK(q.b0 % kVec == 0 && q.b1 % kVec == 0);  // vectors start 16-byte aligned
      CHECK(q.b1 - q.b0 <= kUnitElems && scalar_count(q) <= kMaxScalars);
      for (int64_t e = q.b0; e < q.b1; ++e) {
        CHECK(e >= row * S && e < row * S + S);
        CHECK(cover[e] == 0);
        cover[e] = 1;
      }
      for (int s = 0; s < scalar_count(q); ++s) {
        const int64_t e = scalar_index(q, s);
        CHECK(e >= row * S && e < row * S + S);
        CHECK(cover[e] == 0);
        cover[e] = 1;
      }
      CHECK(q.n == (q.b1 - q.b0) + scalar_count(q));
      if (plan_all_full(p)) {
        const URange f = full_range(p, row, k);
        CHECK(f.b0 == q.b0 && f.b1 == q.b1 && f.n == q.n);
      }
    }
  }
  for (int64_t e = 0; e < numel; ++e) CHECK(cover[e] == 1);
}

// The streaming kernels' work shares (UnitWalk, UnitWalkDown), in both layouts
// and for several worker counts: every unit is visited once with consistent
// (row, k); unit shares tile [0, units) in order; at each block end, whole
// blocks are merged once and the pieces of a cut block publish disjoint lanes
// that add up to its size; strided blocks cut none; the downward walks of a
// worker's `step` warps cover its units exactly once (for unit shares, in the
// reverse of the upward walk's order).
static void walk_shares(int64_t N, int64_t C, int64_t S, int64_t G) {
  g_what = "shares";
  const Plan p = make_plan(N, C, S, G);
  const int64_t nblk = p.NC * p.nb;
  for (bool cut : {false, true})
    for (int64_t nw : {(int64_t)1, (int64_t)7, (int64_t)608, (int64_t)1216, p.units + 3}) {
      std::vector<int64_t> cnt(nblk, 0), whole(nblk, 0);
      std::vector<uint32_t> lanes(nblk, 0);
      std::vector<uint8_t> seen(p.units, 0);
      int64_t prev_u1 = 0;
      for (int64_t w = 0; w < nw; ++w) {
        UnitWalk cu;
        cu.set(p, w, nw, cut);
        if (cut) {
          CHECK(cu.u0 == prev_u1 && cu.u1 >= cu.u0 && cu.u1 - cu.u0 <= p.units / nw + 1);
          prev_u1 = cu.u1;
          if (cu.a != cu.u0) ++g_rotated;
        }
        int64_t visited = 0;
        for (; !cu.end; cu.next(p)) {
          CHECK(cu.u >= 0 && cu.u < p.units && seen[cu.u] == 0);
          if (cut) CHECK(cu.u >= cu.u0 && cu.u < cu.u1);
          seen[cu.u] = 1;
          ++visited;
          CHECK(cu.u == cu.row * p.R + cu.k && cu.k >= 0 && cu.k < p.R && cu.row < p.NC);
          const int ui = cu.ui(), bsz = block_size(p, cu.kb());
          CHECK(ui < bsz && (int64_t)ui == cu.k - cu.kb() * kBlockUnits);
          if (!cut) CHECK((cu.row * p.nb + cu.kb()) % nw == w);
          if (ui == bsz - 1 || cu.u + 1 == cu.u1) {
            const int64_t ub = cu.u - ui, blk = cu.row * p.nb + cu.kb();
            const int lo = ub >= cu.u0 ? 0 : (int)(cu.u0 - ub);
            CHECK(lo >= 0 && lo <= ui && blk < nblk);
            if (lo == 0 && ui == bsz - 1) {
              ++whole[blk];
            } else {
              CHECK(cut);
              for (int l = lo; l <= ui; ++l) {
                CHECK(!(lanes[blk] >> l & 1u));
                lanes[blk] |= 1u << l;
              }
              cnt[blk] += ui - lo + 1;
            }
          }
        }
        if (cut) CHECK(visited == cu.u1 - cu.u0);
      }
      if (cut) CHECK(prev_u1 == p.units);
      for (int64_t u = 0; u < p.units; ++u) CHECK(seen[u] == 1);
      for (int64_t b = 0; b < nblk; ++b) {
        const int bsz = block_size(p, b % p.nb);
        CHECK((whole[b] == 1 && cnt[b] == 0) || (whole[b] == 0 && cnt[b] == bsz));
      }
      for (int step : {2, 4}) {
        if (nw % step) continue;
        const int64_t owners = nw / step;
        std::vector<uint8_t> hit(p.units, 0);
        for (int64_t w = 0; w < owners; ++w) {
          UnitWalk up;
          up.set(p, w, owners, cut);
          std::vector<int64_t> seq;
          for (; !up.end; up.next(p)) seq.push_back(up.u);
          std::vector<uint8_t> mine(p.units, 0);
          for (int64_t v : seq) mine[v] = 1;
          for (int skip = 0; skip < step; ++skip) {
            UnitWalkDown d;
            d.set(p, w, owners, cut, skip, step);
            for (int64_t j = skip; !d.end(); d.next(p), j += step) {
              CHECK(d.u >= 0 && d.u < p.units && mine[d.u] == 1);
              if (cut) CHECK(j < (int64_t)seq.size() && d.u == seq[seq.size() - 1 - j]);
              CHECK(d.u == d.row * p.R + d.k && d.k >= 0 && d.k < p.R);
              CHECK(hit[d.u] == 0);
              hit[d.u] = 1;
            }
          }
        }
        for (int64_t u = 0; u < p.units; ++u) CHECK(hit[u] == 1);
      }
    }
}

static void walk_ndhwc(int64_t N, int64_t C, int64_t S, int64_t G) {
  g_what = "ndhwc";
  const NPlan p = make_nplan(N, C, S, G);
  const int64_t numel = N * S * C;
  std::vector<uint8_t> cover(numel, 0);
  std::vector<uint8_t> piece(p.rows * p.P * p.R, 0);
  CHECK(p.P >= 1 && p.P <= kNSpan * kNVec);
  for (int64_t u = 0; u < p.units; ++u) {
    const NUnit q0 = n_unit(p, u, 0);
    std::vector<int64_t> chan(kNSpan * kNVec, 0);
    for (int lane = 0; lane < 32; ++lane) {
      const NUnit q = n_unit(p, u, lane);
      CHECK(q.row == q0.row && q.k == q0.k && q.len == q0.len && q.len >= 1);
      CHECK(q.cnt <= kNSteps && q.b >= 0 && q.b < q.rg.vr);
      if (lane < q.rg.vr) CHECK(q.m == 0 && q.cnt >= 1);  // the lanes whose means shift the others
      for (int t = 0; t < q.cnt; ++t) {
        const int64_t o = q.off + t * q.step;
        CHECK(o % kNVec == 0 && o >= 0 && o + kNVec <= numel);
        const int64_t n = o / (S * C), pos = (o / C) % S, c = o % C;
        CHECK(n == q.n && pos >= q.u0 && pos < q.u0 + q.len && c >= q.rg.c0 && c + kNVec <= q.rg.c1);
        for (int e = 0; e < kNVec; ++e) {
          CHECK(cover[o + e] == 0);
          cover[o + e] = 1;
        }
      }
      if (lane < q.rg.lw)
        for (int sl = 0; sl < kNVec; ++sl) chan[kNVec * q.b + sl] += q.cnt;
    }
    for (int64_t cc = 0; cc < kNVec * q0.rg.vr; ++cc) CHECK(chan[cc] == q0.len);
    const int64_t np = q0.rg.g1 - q0.rg.g0 + 1;
    CHECK(np <= p.P);
    int64_t chans = 0;
    for (int64_t j = 0; j < np; ++j) {
      int64_t c0, c1;
      n_piece(p, q0.rg, j, c0, c1);
      CHECK(c0 >= 0 && c1 <= kNVec * q0.rg.vr && c1 > c0);
      chans += c1 - c0;
      const int64_t idx = (q0.row * p.P + j) * p.R + q0.k;
      CHECK(idx < (int64_t)piece.size() && piece[idx] == 0);
      piece[idx] = 1;
    }
    CHECK(chans == kNVec * q0.rg.vr);
  }
  for (int64_t e = 0; e < numel; ++e) CHECK(cover[e] == 1);
  // every group's pieces, range by range and unit by unit, were written
  for (int64_t gi = 0; gi < p.NG; ++gi) {
    const int64_t n = gi / G, g = gi % G;
    const int64_t r_lo = (g * p.Cg) / (kNSpan * kNVec), r_hi = ((g + 1) * p.Cg - 1) / (kNSpan * kNVec);
    CHECK(r_hi < p.nr);
    int64_t chans = 0;
    for (int64_t r = r_lo; r <= r_hi; ++r) {
      const NRange rg = n_range(p, r);
      const int64_t j = g - rg.g0;
      CHECK(j >= 0 && j <= rg.g1 - rg.g0);
      int64_t c0, c1;
      n_piece(p, rg, j, c0, c1);
      chans += c1 - c0;
      for (int64_t k = 0; k < p.R; ++k) CHECK(piece[((n * p.nr + r) * p.P + j) * p.R + k] == 1);
    }
    CHECK(chans == p.Cg);
  }
  if (p.nr != 1) return;
  // ring parts of the one-range kernels: every warp's walk, for the part sizes they use
  g_what = "ndhwc ring";
  const NRange rg = n_range(p, 0);
  for (int kPS : {2, 4, 8, 16}) {
    const int64_t cap = (int64_t)kPS * kNSpan * kNVec;  // slot capacity in elements
    for (int64_t W : {(int64_t)1, (int64_t)7, (int64_t)1216}) {
      for (int64_t first = 0; first < W && first < p.units; ++first) {
        for (int64_t u = first; u < p.units; u += W) {
          const int steps = n_unit_steps(p, rg, u);
          int part = 0;
          for (int t0 = 0; t0 < steps; t0 += kPS, ++part) {
            int64_t e0, n;
            const bool last = n_ring_part(p, rg, u, part, kPS, e0, n);
            CHECK(last == (t0 + kPS >= steps));
            CHECK(n > 0 && n <= cap && e0 % kNVec == 0 && n % kNVec == 0 && e0 + n <= numel);
            for (int lane = 0; lane < 32; ++lane) {
              const NUnit q = n_unit(p, u, lane);
              const int nv = q.cnt - t0 < kPS ? q.cnt - t0 : kPS;
              for (int t = 0; t < nv; ++t) {
                const int64_t lo = (int64_t)t * kNVec * rg.lw + kNVec * lane;  // in the slot
                CHECK(lo + kNVec <= n);
                CHECK(e0 + lo == q.off + (int64_t)(t0 + t) * q.step);
              }
            }
          }
        }
      }
    }
  }
}

// The layout each bench volume gets on 152 SMs x 8 reduction warps: strided
// blocks below two merge blocks per warp (128^3, 96^3, the ragged 97^3 site),
// unit shares above (256^3).
static void layouts_of_the_bench_volumes() {
  g_what = "layouts";
  const int64_t nw = 152 * 8;
  CHECK(!use_unit_shares(make_plan(1, 32, 128 * 128 * 128, 8), nw));
  CHECK(!use_unit_shares(make_plan(2, 64, 96 * 96 * 96, 32), nw));
  CHECK(!use_unit_shares(make_plan(1, 48, 97 * 97 * 97, 8), nw));
  CHECK(use_unit_shares(make_plan(1, 32, 256 * 256 * 256, 8), nw));
}

int main() {
  int shapes = 0;
  layouts_of_the_bench_volumes();
  const int64_t Cs[] = {1, 3, 4, 6, 8, 16, 24, 32, 40, 48, 64, 96, 128, 192, 256, 264, 320, 512, 768};
  const int64_t Ss[] = {1, 2, 3, 7, 8, 9, 63, 64, 65, 255, 256, 257, 1000, 4096, 4097, 8191, 12345};
  for (int64_t C : Cs)
    for (int64_t S : Ss)
      for (int64_t G : {(int64_t)1, (int64_t)2, (int64_t)3, C / 8, C / 2, C}) {
        if (G < 1 || C % G) continue;
        for (int64_t N : {(int64_t)1, (int64_t)2}) {
          if (N * C * S > 4000000) continue;
          g_shape[0] = N; g_shape[1] = C; g_shape[2] = S; g_shape[3] = G;
          walk_ncdhw(N, C, S, G);
          walk_shares(N, C, S, G);
          if (C % kNVec == 0) walk_ndhwc(N, C, S, G);
          ++shapes;
        }
      }
  if (g_rotated == 0) {
    printf("FAIL no share walk started at its end's cut piece\n");
    return 1;
  }
  printf("ok %d\n", shapes);
  return 0;
}
