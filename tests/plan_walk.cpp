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
//   group-wave placement (gn3d_resident_plan.cuh): the shares of every group
//     tile it in CTA order and every CTA's total differs from every other's by
//     at most one unit; each CTA's sequence visits its units in order with
//     consistent (row, k), group, held/pass ring positions and piece spans; the
//     pieces of each merge block cover its units exactly once; the elementwise
//     order covers the same units once (also split over several warps) and
//     finds each held unit at the held position the sequence gave it.
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
#ifndef __forceinline__
#define __forceinline__ inline
#endif
#include "../bwd_gn3d_stats_gb300/csrc/gn3d_plan.cuh"
#include "../bwd_gn3d_stats_gb300/csrc/gn3d_ndhwc_plan.cuh"
#include "../bwd_gn3d_stats_gb300/csrc/gn3d_resident_plan.cuh"
#include "../bwd_gn3d_stats_gb300/csrc/gn3d_cluster_plan.cuh"

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
      if (!cut) {  // the elementwise kernels' even walk: every unit once, freshest round first
        for (int64_t ew : {(int64_t)16, (int64_t)4, (int64_t)9}) {
          const int64_t W = nw * ew / 8 > 0 ? nw * ew / 8 : 1;  // nw: the reduction warps, grid * 8
          std::vector<uint8_t> hit(p.units, 0);
          for (int64_t w = 0; w < W; ++w) {
            UnitWalkFresh f;
            f.set(p, w, W, nw);
            int64_t last_i = -1;
            for (; !f.end(); f.next(p)) {
              CHECK(f.u >= 0 && f.u < p.units && f.u == f.row * p.R + f.k && f.k >= 0 && f.k < p.R);
              CHECK(f.i > last_i && f.i % W == w);
              last_i = f.i;
              CHECK(hit[f.u] == 0);
              hit[f.u] = 1;
            }
          }
          for (int64_t u = 0; u < p.units; ++u) CHECK(hit[u] == 1);
        }
      }
    }
}

static void walk_ndhwc(int64_t N, int64_t C, int64_t S, int64_t G, int64_t min_units) {
  g_what = "ndhwc";
  const NPlan p = make_nplan(N, C, S, G, min_units);
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
      CHECK(q.cnt <= p.steps && p.steps <= kNSteps && p.steps >= kNMinSteps && q.b >= 0 && q.b < q.rg.vr);
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

// The group-wave kernels' placement for P CTAs, rh held units per share and
// rings of kh held and kp pass slots.
static void walk_resident(const Plan& p, int P, int rh, int kh, int kp, int recs) {
  g_what = "resident";
  const ResGeo G = res_geo(p, P, rh, kh, kp, recs);
  const int64_t nblk = p.NC * p.nb;
  std::vector<int32_t> owner(p.units, -1);
  std::vector<int64_t> held_at(p.units, -1);
  std::vector<int64_t> block_units(nblk, 0);
  std::vector<uint32_t> block_lanes(nblk, 0);
  std::vector<int64_t> total(P, 0);
  for (int64_t g = 0; g < p.NG; ++g) {  // shares tile the group in CTA order
    int64_t at = g * p.upg;
    for (int c = 0; c < P; ++c) {
      const ResShare sh = res_share(p, G, g, c);
      CHECK(sh.start == at && sh.n >= 0 && sh.nh == (sh.n < rh ? sh.n : rh));
      at += sh.n;
      total[c] += sh.n;
    }
    CHECK(at == (g + 1) * p.upg);
  }
  int64_t tmin = INT64_MAX, tmax = 0;
  for (int c = 0; c < P; ++c) {
    tmin = total[c] < tmin ? total[c] : tmin;
    tmax = total[c] > tmax ? total[c] : tmax;
  }
  CHECK(tmax - tmin <= 1);
  for (int c = 0; c < P; ++c) {
    ResSeq s;
    s.begin(p, G, c);
    int64_t h = 0, q = 0, piece = -1, pblk = -1, n = 0;
    int plo = -1, phi = -1;
    std::vector<int64_t> order;
    while (!s.end) {
      const int64_t u = s.unit_index();
      CHECK(u >= 0 && u < p.units && s.k == u % p.R && s.g == (u / p.R) / p.Cg);
      CHECK(u >= s.sh.start && u < s.sh.start + s.sh.n && s.j == u - s.sh.start);
      CHECK(s.h == h && s.q == q);
      CHECK(owner[u] == -1);
      owner[u] = c;
      const bool hd = s.held();
      CHECK(hd == (s.j >= s.sh.n - s.sh.nh));
      const int64_t ri = hd ? h : q, rn = hd ? kh : kp;
      CHECK(s.ring_index() == ri && s.slot() == ri % rn && s.parity() == (uint32_t)((ri / rn) & 1));
      if (hd) held_at[u] = h++;
      else ++q;
      int64_t b0;
      int lo, hi, bsz;
      s.piece_span(p, b0, lo, hi, bsz);
      const int ui = (int)(s.k % kBlockUnits);
      const int64_t blk = (u / p.R) * p.nb + s.k / kBlockUnits;
      CHECK(s.block(p) == blk && b0 == u - ui && lo >= 0 && lo <= ui && ui <= hi && hi < bsz && bsz <= kBlockUnits);
      if (blk != pblk) {  // a new piece
        ++piece;
        pblk = blk;
        plo = lo;
        phi = hi;
        const uint32_t m = (uint32_t)((((uint64_t)1 << (hi + 1)) - 1) & ~(((uint64_t)1 << lo) - 1));
        CHECK((block_lanes[blk] & m) == 0);
        block_lanes[blk] |= m;
        block_units[blk] += hi - lo + 1;
      } else {
        CHECK(lo == plo && hi == phi);
      }
      order.push_back(u);
      ++n;
      s.next(p, G, c);
    }
    CHECK(n == total[c] && s.h + s.q == n);
    // the kernels' per-share walks: the producer's order is the sequence; each
    // reduction warp takes, per share, the pass units then the held units at
    // ring positions = warp (mod 4), with the slot and parity the sequence gave
    for (int w = 0; w < 4 && kh % 4 == 0 && kp % 4 == 0; ++w) {
      std::vector<int64_t> mine;  // (unit) in the warp's order, from the sequence
      std::vector<std::pair<int, uint32_t>> ring;
      ResSeq t;
      t.begin(p, G, c);
      for (; !t.end; t.next(p, G, c))
        if (t.slot() % 4 == w) {
          mine.push_back(t.unit_index());
          ring.push_back({t.slot(), t.parity()});
        }
      size_t at = 0;
      int hb = 0, qb = 0;
      for (int64_t g = 0; g < p.NG; ++g) {
        const ResShare sh = res_share(p, G, g, c);
        if (sh.n == 0) continue;
        const int npass = sh.n - sh.nh;
        for (int part = 0; part < 2; ++part) {
          const bool hd = part == 1;
          const int first = hd ? npass : 0, count = hd ? sh.nh : npass, before = hd ? hb : qb;
          const int nr = hd ? kh : kp;
          int j = res_first_of_warp(before, w, 4);
          if (j >= count) continue;
          RingPos r;
          r.at(before + j, nr);
          for (; j < count; j += 4, r.step(4, nr)) {
            CHECK(at < mine.size() && mine[at] == sh.start + first + j);
            CHECK(ring[at].first == r.slot && ring[at].second == r.par);
            ++at;
          }
        }
        hb += sh.nh;
        qb += npass;
      }
      CHECK(at == mine.size());
    }
    std::vector<int64_t> pos_of(p.units, -1);
    for (int64_t i = 0; i < (int64_t)order.size(); ++i) pos_of[order[i]] = i;
    // the elementwise order: the same units, each share last unit first, held
    // units at the slots the sequence gave them; split over 1 or 7 warps
    for (int step : {1, 7}) {
      std::vector<uint8_t> got(order.size(), 0);
      int64_t count = 0;
      for (int w = 0; w < step; ++w) {
        ResElemSeq e;
        e.begin(p, G, c);
        e.advance(p, G, c, w);
        while (!e.end) {
          const int64_t u = e.unit();
          CHECK(u >= 0 && u < p.units && owner[u] == c);
          CHECK(e.j() >= 0 && e.j() < e.sh.n && e.g == (u / p.R) / p.Cg);
          CHECK(e.held() == (held_at[u] >= 0));
          if (e.held()) {
            CHECK(e.hidx() == held_at[u]);
            int slot;
            uint32_t par;
            e.held_slot(G, slot, par);
            CHECK(slot == held_at[u] % kh && par == (uint32_t)((held_at[u] / kh) & 1));
          }
          const int64_t pos = pos_of[u];
          CHECK(pos >= 0 && got[pos] == 0);
          got[pos] = 1;
          ++count;
          e.advance(p, G, c, step);
        }
      }
      CHECK(count == (int64_t)order.size());
    }
  }
  for (int64_t u = 0; u < p.units; ++u) CHECK(owner[u] >= 0);
  for (int64_t b = 0; b < nblk; ++b) {
    const int bsz = block_size(p, b % p.nb);
    CHECK(block_units[b] == bsz && block_lanes[b] == (uint32_t)((((uint64_t)1) << bsz) - 1));
  }
}

static void walk_resident_shapes() {
  // rows of whole units (the group-wave kernels' domain), the bench volumes among them
  struct Sh { int64_t N, C, S, G; };
  const Sh shapes[] = {{1, 32, 128 * 128 * 128, 8}, {1, 32, 256 * 256 * 256, 8}, {2, 64, 96 * 96 * 96, 32},
                       {1, 64, 128 * 128 * 128, 8}, {1, 128, 64 * 64 * 64, 8}, {1, 256, 32 * 32 * 32, 8},
                       {1, 512, 16 * 16 * 16, 8},   {2, 16, 16 * 16 * 16, 4},   {1, 4, 4096, 1},
                       {3, 6, 4096 * 5, 3},          {1, 12, 4096 * 33, 4},      {2, 40, 4096 * 17, 8},
                       {1, 1, 4096 * 3, 1},          {1, 8, 4096 * 300, 2}};
  for (const Sh& sh : shapes) {
    g_shape[0] = sh.N; g_shape[1] = sh.C; g_shape[2] = sh.S; g_shape[3] = sh.G;
    const Plan p = make_plan(sh.N, sh.C, sh.S, sh.G);
    CHECK(plan_all_full(p));
    for (int P : {1, 7, 152, 160})
      for (int rh : {1, 5, 10, 1000}) {
        if ((P > 1 && p.units > 200000 && rh != 10) || (p.units > 50000 && P < 152)) continue;  // bounded run time
        walk_resident(p, P, rh < 20 ? rh : 20, 20, 4, 16);
        if (rh == 5) walk_resident(p, P, rh, 8, 4, 3);
      }
  }
}

// The group-wave kernels' synchronization, simulated: per CTA a producer that
// issues the sequence's copies in order (a held or pass slot's next use only
// after its previous use was released, and at most `window` units ahead of the
// elementwise pass), kRed reduction warps (slot s of either ring read by warp
// s mod kRed, in order; a pass slot released after the reduction; a group is
// ready once every unit of it is reduced), and the elementwise warps, which
// move through the CTA's shares together (named barriers), a share once its
// group is ready, releasing its held slots.  Agents take enabled steps in a
// seeded random order; the run must finish every unit with no state in which
// nothing can move.
struct SimPos { int64_t u, g, use; bool held; int slot; };
static void sim_resident(const Plan& p, int P, int kh, int kp, int rh, int64_t window, int kRed, uint64_t seed) {
  g_what = "resident-sim";
  std::vector<int64_t> gleft(p.NG, p.upg);
  std::vector<uint8_t> ready(p.NG, 0);
  struct Cta {
    std::vector<SimPos> seq;                 // sequence order
    std::vector<std::vector<int64_t>> shares;  // per share (group order): its positions
    int64_t issued = 0, normed = 0, next_share = 0;
    std::vector<int64_t> hrel, prel;         // uses released per slot
    std::vector<std::vector<int64_t>> rpos;  // positions of each reduction warp, in order
    std::vector<int64_t> rnext;
  };
  std::vector<Cta> ctas(P);
  int64_t total = 0;
  const ResGeo G = res_geo(p, P, rh, kh, kp, 0);
  for (int c = 0; c < P; ++c) {
    Cta& t = ctas[c];
    ResSeq s;
    s.begin(p, G, c);
    int64_t gprev = -1;
    while (!s.end) {
      const bool hd = s.held();
      const int64_t i = s.ring_index();
      if (s.g != gprev) {
        t.shares.push_back({});
        gprev = s.g;
      }
      t.shares.back().push_back((int64_t)t.seq.size());
      t.seq.push_back(SimPos{s.unit_index(), s.g, i / (hd ? kh : kp), hd, s.slot()});
      s.next(p, G, c);
    }
    t.hrel.assign(kh, 0);
    t.prel.assign(kp, 0);
    t.rpos.assign(kRed, {});
    for (int64_t i = 0; i < (int64_t)t.seq.size(); ++i) t.rpos[t.seq[i].slot % kRed].push_back(i);
    t.rnext.assign(kRed, 0);
    total += (int64_t)t.seq.size();
  }
  uint64_t rng = seed * 0x9E3779B97F4A7C15ull + 1;
  auto rnd = [&](uint64_t n) {
    rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17;
    return rng % n;
  };
  const int agents = 2 + kRed;  // producer, reduction warps, the elementwise warps together
  auto step = [&](Cta& t, int a) -> bool {
    if (a == 0) {  // producer
      if (t.issued >= (int64_t)t.seq.size()) return false;
      const SimPos& q = t.seq[t.issued];
      const int64_t rel = q.held ? t.hrel[q.slot] : t.prel[q.slot];
      if (rel < q.use) return false;  // the slot's previous use not yet released
      if (t.issued >= t.normed + window) return false;
      ++t.issued;
      return true;
    }
    if (a <= kRed) {  // reduction warp
      int64_t& k = t.rnext[a - 1];
      const std::vector<int64_t>& mine = t.rpos[a - 1];
      if (k >= (int64_t)mine.size() || mine[k] >= t.issued) return false;
      const SimPos& q = t.seq[mine[k]];
      if (!q.held) ++t.prel[q.slot];
      if (--gleft[q.g] == 0) ready[q.g] = 1;
      ++k;
      return true;
    }
    // the elementwise warps: the next share, once its group is ready
    if (t.next_share >= (int64_t)t.shares.size()) return false;
    const std::vector<int64_t>& sh = t.shares[t.next_share];
    if (!ready[t.seq[sh[0]].g]) return false;
    for (int64_t i : sh) {
      const SimPos& q = t.seq[i];
      if (q.held) {
        CHECK(t.hrel[q.slot] == q.use);  // released in use order
        ++t.hrel[q.slot];
      }
    }
    t.normed += (int64_t)sh.size();
    ++t.next_share;
    return true;
  };
  for (;;) {
    bool moved = false;
    const int c0 = (int)rnd(P);
    for (int dc = 0; dc < P && !moved; ++dc) {
      Cta& t = ctas[(c0 + dc) % P];
      const int a0 = (int)rnd(agents);
      for (int da = 0; da < agents && !moved; ++da)
        if (step(t, (a0 + da) % agents)) moved = true;
    }
    if (!moved) break;
  }
  int64_t done = 0;
  for (const Cta& t : ctas) done += t.normed;
  CHECK(done == total);  // else: no agent could move -- a deadlock
  for (int64_t g = 0; g < p.NG; ++g) CHECK(ready[g]);
}

static void sim_resident_shapes() {
  struct Sh { int64_t N, C, S, G; };
  const Sh shapes[] = {{1, 32, 128 * 128 * 128, 8}, {2, 64, 96 * 96 * 96, 32}, {1, 512, 16 * 16 * 16, 8},
                       {1, 256, 32 * 32 * 32, 8},   {3, 6, 4096 * 5, 3},        {1, 12, 4096 * 33, 4}};
  for (const Sh& sh : shapes) {
    g_shape[0] = sh.N; g_shape[1] = sh.C; g_shape[2] = sh.S; g_shape[3] = sh.G;
    const Plan p = make_plan(sh.N, sh.C, sh.S, sh.G);
    // forward bf16 rings (20 held + 4 pass), backward bf16 rings (8 + 4), minimal
    // rings; held slots a multiple of the 4 reduction warps
    const int rings[3][2] = {{20, 4}, {8, 4}, {4, 4}};
    for (const auto& rg : rings)
      for (int rh : {0, rg[0] / 2, rg[0]})
        // the window must admit a whole share of a group (its statistics need it)
        for (int64_t window : {res_min_window(p, 152), res_min_window(p, 152) + rg[0] + rg[1], (int64_t)1000000})
          for (uint64_t seed : {1ull, 2ull})
            sim_resident(p, 152, rg[0], rg[1], rh, window, 4, seed);
  }
}

// The cluster kernels' split of a group: the CTAs' block runs tile the group's
// blocks in order; CTA-local unit j is unit ui of the run's blocks in block
// order (consecutive units of a row); every unit of the group is visited
// exactly once; upc is the largest CTA's unit count; the cluster size keeps a
// block and two units per CTA on average.
static void walk_cluster(int64_t N, int64_t C, int64_t S, int64_t G) {
  g_what = "cluster";
  const Plan p = make_plan(N, C, S, G);
  if (!plan_all_full(p)) return;
  const ClusterGeo c = cluster_geo(p);
  CHECK(c.nbg == p.Cg * p.nb);
  CHECK(c.cs >= 1 && c.cs <= kClusterMaxCTAs && (c.cs & (c.cs - 1)) == 0);
  CHECK(c.cs == 1 || (c.cs <= c.nbg && 2 * c.cs <= p.upg));
  CHECK(c.cs == kClusterMaxCTAs || 2 * c.cs > c.nbg || 4 * c.cs > p.upg);  // the largest such size
  for (int64_t g : {(int64_t)0, p.NG - 1}) {
    std::vector<int> seen((size_t)p.upg, 0);
    int upc = 0;
    int64_t prev = 0;
    for (int r = 0; r < c.cs; ++r) {
      const int64_t b0 = cl_block_begin(c.nbg, c.cs, r), b1 = cl_block_begin(c.nbg, c.cs, r + 1);
      CHECK(b0 == prev && b1 >= b0);
      prev = b1;
      const int nu = cl_units(p, b0, b1);
      if (nu > upc) upc = nu;
      int64_t lastb = -1;
      int lastui = -1;
      for (int j = 0; j < nu; ++j) {
        int64_t b, row, k;
        int ui;
        cl_unit(p, b0, j, b, ui);
        CHECK(b >= b0 && b < b1 && ui >= 0 && ui < cl_block_units(p, b));
        CHECK((b == lastb && ui == lastui + 1) || (b == lastb + 1 && ui == 0) || (j == 0 && b == b0 && ui == 0));
        lastb = b;
        lastui = ui;
        cl_row_k(p, g, b, ui, row, k);
        CHECK(row >= g * p.Cg && row < (g + 1) * p.Cg && k >= 0 && k < p.R);
        CHECK(k / kBlockUnits == b % p.nb && row - g * p.Cg == b / p.nb);
        seen[(size_t)((row - g * p.Cg) * p.R + k)] += 1;
      }
    }
    CHECK(prev == c.nbg);
    CHECK(upc == c.upc);
    for (int v : seen) CHECK(v == 1);
  }
}

static void layouts_of_the_bench_volumes() {
  g_what = "layouts";
  const int64_t nw = 152 * 8;
  CHECK(!use_unit_shares(make_plan(1, 32, 128 * 128 * 128, 8), nw));
  CHECK(!use_unit_shares(make_plan(2, 64, 96 * 96 * 96, 32), nw));
  CHECK(!use_unit_shares(make_plan(1, 48, 97 * 97 * 97, 8), nw));
  CHECK(use_unit_shares(make_plan(1, 32, 256 * 256 * 256, 8), nw));
  // few merge blocks: 256 rows of 8 units (shares), 512 rows of one unit (no
  // unit to share out), 512 blocks of 16 units (strided)
  CHECK(use_unit_shares(make_plan(1, 256, 32 * 32 * 32, 8), nw));
  CHECK(!use_unit_shares(make_plan(1, 512, 16 * 16 * 16, 8), nw));
  CHECK(!use_unit_shares(make_plan(1, 128, 64 * 64 * 64, 8), nw));
  // the cluster form's split at the UNet's small sites and the small fp32 volume
  g_what = "cluster sizes";
  CHECK(cluster_geo(make_plan(1, 512, 16 * 16 * 16, 8)).cs == 16 && cluster_geo(make_plan(1, 512, 4096, 8)).upc == 4);
  CHECK(cluster_geo(make_plan(1, 256, 32 * 32 * 32, 8)).cs == 16 && cluster_geo(make_plan(1, 256, 32768, 8)).upc == 16);
  CHECK(cluster_geo(make_plan(2, 16, 16 * 16 * 16, 4)).cs == 2 && cluster_geo(make_plan(2, 16, 4096, 4)).upc == 2);
}

int main() {
  int shapes = 0;
  layouts_of_the_bench_volumes();
  walk_resident_shapes();
  sim_resident_shapes();
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
          if (C % kNVec == 0) {
            walk_ndhwc(N, C, S, G, kNMinUnitsFwd);
            walk_ndhwc(N, C, S, G, kNMinUnitsBwd);
          }
          ++shapes;
        }
      }
  // whole-unit rows for the cluster split (rows of 1 .. 40 units)
  for (int64_t C : Cs)
    for (int64_t R : {1, 2, 3, 8, 15, 16, 17, 31, 33, 40})
      for (int64_t G : {(int64_t)1, (int64_t)2, (int64_t)3, C / 8, C / 2, C}) {
        if (G < 1 || C % G) continue;
        for (int64_t N : {(int64_t)1, (int64_t)2}) {
          g_shape[0] = N; g_shape[1] = C; g_shape[2] = R * kUnitElems; g_shape[3] = G;
          walk_cluster(N, C, R * kUnitElems, G);
        }
      }
  if (g_rotated == 0) {
    printf("FAIL no share walk started at its end's cut piece\n");
    return 1;
  }
  printf("ok %d\n", shapes);
  return 0;
}
