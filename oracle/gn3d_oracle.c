/*
 * gn3d_oracle.c -- plain fp64 CPU oracle for GroupNorm over NCDHW volumes.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity reference for the CUDA
 * library; it is called from tests/, from __graft_entry__.smoke() and from
 * bench.py's cpu_baseline / reference leg, and from nowhere else.  It shares
 * no code, header, table or constant with the CUDA path.
 *
 * What it computes is the plain definition of GroupNorm (the semantics of
 * torch's nn.GroupNorm, which the ScaFFold "Optimize GroupNorm" PR #93 keeps
 * as a drop-in: same weight and bias, same results), written out in fp64:
 *
 *   group (n,g) = channels g*C/G .. (g+1)*C/G-1 of sample n, all D*H*W
 *                 positions: M = (C/G)*S elements, contiguous in NCDHW;
 *   mu    = (1/M) sum x                      (biased statistics)
 *   var   = (1/M) sum (x - mu)^2
 *   rstd  = 1 / sqrt(var + eps)              (eps inside the root: with a
 *           zero-variance group and eps = 1e-5 this gives rstd = 316, the
 *           value PR #93's review of the single-element-group case quotes)
 *   y     = (x - mu) * rstd * gamma_c + beta_c
 *
 * and the backward of that map at given statistics (mu, rstd):
 *
 *   xhat = (x - mu) * rstd,  g = dy * gamma_c
 *   a = mean_group(g),  b = mean_group(g * xhat)
 *   dx = rstd * (g - a - xhat * b)
 *   dgamma_c = sum_{n, spatial} dy * xhat,   dbeta_c = sum_{n, spatial} dy
 *
 * The fused ReLU (the ScaFFold GroupNorm pages: FastGroupNorm's activation
 * argument, and the fix that makes it bit-identical to unfused GroupNorm then
 * F.relu on NaN, both infinities and -0.0) is, forward, F.relu of the rounded
 * output: out = (v < 0) ? +0 : v on v = y rounded to the output type -- NaN,
 * +Inf and -0.0 pass, -Inf and negatives become +0 -- and, backward, torch's
 * threshold_backward on the forward's result: the gradient reaching GroupNorm
 * is dy where the result is not <= 0 (a NaN result passes it) and 0 elsewhere.
 *
 * Every sum is a Neumaier-compensated fp64 sum (Neumaier 1974), so results are
 * the exact values to well below the GPU's fp32 error.  Inputs arrive as the
 * raw bytes the GPU sees (fp32 or bf16), widened exactly to fp64 here.  eps is
 * rounded to fp32 and widened, because the library's API takes a double but
 * computes with its fp32 value.  Rounding the fp64 result to the output type
 * is done once, round-to-nearest-even, straight from fp64 (PR #105 "Preserve
 * GroupNorm dtype": the output is the fp32-computed answer rounded once; the
 * oracle's is the exact answer rounded once).
 *
 * OpenMP, where present, only spreads independent groups / channels over
 * threads; the arithmetic inside each group is the same sequential sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_EINVAL 1

/* ---------------------------------------------------------------- inputs */

static double widen(const void* p, int dtype, int64_t i) {
  if (dtype == ORC_F32) return (double)((const float*)p)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;  /* bf16 is the high half of an fp32 */
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double eps_as_used(double eps) { return (double)(float)eps; }

static double param(const float* p, int64_t c, double dflt) {
  return p ? (double)p[c] : dflt;
}

/* ------------------------------------------------------ compensated sums */

typedef struct { double s, c; } nsum;

static void nsum_add(nsum* a, double v) {
  double t = a->s + v;
  if (fabs(a->s) >= fabs(v)) a->c += (a->s - t) + v;
  else a->c += (v - t) + a->s;
  a->s = t;
}

static double nsum_val(const nsum* a) { return a->s + a->c; }

static int check_shape(int64_t N, int64_t C, int64_t S, int64_t G) {
  if (N < 0 || C < 0 || S < 0 || G <= 0) return ORC_EINVAL;
  if (C % G != 0) return ORC_EINVAL;
  return ORC_OK;
}

/* ------------------------------------------------------------ statistics */

/* Per-group mean, biased variance and rstd.  mean/var/rstd: [N*G] (any may be NULL). */
int gn3d_oracle_stats(const void* x, int dtype, int64_t N, int64_t C, int64_t S, int64_t G,
                      double eps, double* mean, double* var, double* rstd) {
  if (check_shape(N, C, S, G) || (dtype != ORC_F32 && dtype != ORC_BF16)) return ORC_EINVAL;
  const int64_t M = (C / G) * S;
  const double e = eps_as_used(eps);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ng = 0; ng < N * G; ++ng) {
    const int64_t base = ng * M;
    nsum s1 = {0, 0};
    for (int64_t i = 0; i < M; ++i) nsum_add(&s1, widen(x, dtype, base + i));
    const double mu = M ? nsum_val(&s1) / (double)M : 0.0;
    nsum s2 = {0, 0};
    for (int64_t i = 0; i < M; ++i) {
      const double d = widen(x, dtype, base + i) - mu;
      nsum_add(&s2, d * d);
    }
    const double v = M ? nsum_val(&s2) / (double)M : 0.0;
    if (mean) mean[ng] = mu;
    if (var) var[ng] = v;
    if (rstd) rstd[ng] = 1.0 / sqrt(v + e);
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------- forward */

static double y_of(double xv, double mu, double r, double gam, double bet) {
  return (xv - mu) * r * gam + bet;
}

/* Full forward.  y: [N*C*S] fp64 (exact result before the output rounding).
 * mean/rstd: [N*G] fp64, may be NULL.  gamma/beta: [C] fp32 or NULL (1 / 0). */
int gn3d_oracle_forward(const void* x, int dtype, const float* gamma, const float* beta,
                        int64_t N, int64_t C, int64_t S, int64_t G, double eps,
                        double* y, double* mean, double* rstd) {
  if (check_shape(N, C, S, G)) return ORC_EINVAL;
  double* mu = (double*)malloc(sizeof(double) * (size_t)(N * G + 1));
  double* rs = (double*)malloc(sizeof(double) * (size_t)(N * G + 1));
  if (!mu || !rs) { free(mu); free(rs); return ORC_EINVAL; }
  int st = gn3d_oracle_stats(x, dtype, N, C, S, G, eps, mu, NULL, rs);
  if (st) { free(mu); free(rs); return st; }
  const int64_t Cg = C / G;
#pragma omp parallel for schedule(static)
  for (int64_t nc = 0; nc < N * C; ++nc) {
    const int64_t n = nc / C, c = nc % C, ng = n * G + c / Cg;
    const double gam = param(gamma, c, 1.0), bet = param(beta, c, 0.0);
    for (int64_t s = 0; s < S; ++s) {
      const int64_t i = nc * S + s;
      y[i] = y_of(widen(x, dtype, i), mu[ng], rs[ng], gam, bet);
    }
  }
  if (mean) memcpy(mean, mu, sizeof(double) * (size_t)(N * G));
  if (rstd) memcpy(rstd, rs, sizeof(double) * (size_t)(N * G));
  free(mu);
  free(rs);
  return ORC_OK;
}

/* Forward at k flat indices, given statistics (fp64 [N*G]). */
int gn3d_oracle_forward_at(const void* x, int dtype, const float* gamma, const float* beta,
                           int64_t N, int64_t C, int64_t S, int64_t G,
                           const double* mean, const double* rstd,
                           const int64_t* idx, int64_t k, double* y) {
  if (check_shape(N, C, S, G)) return ORC_EINVAL;
  const int64_t Cg = C / G, L = N * C * S;
  for (int64_t j = 0; j < k; ++j) {
    const int64_t i = idx[j];
    if (i < 0 || i >= L) return ORC_EINVAL;
    const int64_t nc = i / S, n = nc / C, c = nc % C, ng = n * G + c / Cg;
    y[j] = y_of(widen(x, dtype, i), mean[ng], rstd[ng], param(gamma, c, 1.0), param(beta, c, 0.0));
  }
  return ORC_OK;
}

/* --------------------------------------------------------------- backward */

/* Group sums a = mean(g), b = mean(g*xhat) per (n,g), and per-(n,c) partial
 * dgamma/dbeta sums, all at the given statistics. */
/* The gradient arriving at GroupNorm at element i: dy, or -- behind the fused
 * ReLU -- 0 where the forward's result `gate` is <= 0 (NaN compares false, so
 * a NaN result passes the gradient). */
static double grad_in(const void* dy, const void* gate, int dtype, int64_t i) {
  const double d = widen(dy, dtype, i);
  if (gate && widen(gate, dtype, i) <= 0.0) return 0.0;
  return d;
}

static void bwd_sums(const void* dy, const void* gate, const void* x, int dtype, const double* mean,
                     const double* rstd, const float* gamma, int64_t N, int64_t C, int64_t S, int64_t G,
                     double* a, double* b, double* dg_nc, double* db_nc) {
  const int64_t Cg = C / G, M = Cg * S;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t ng = 0; ng < N * G; ++ng) {
    const int64_t n = ng / G, g = ng % G;
    nsum sg = {0, 0}, sgx = {0, 0};
    for (int64_t cl = 0; cl < Cg; ++cl) {
      const int64_t c = g * Cg + cl, nc = n * C + c;
      const double gam = param(gamma, c, 1.0);
      nsum sdy = {0, 0}, sdyx = {0, 0};
      for (int64_t s = 0; s < S; ++s) {
        const int64_t i = nc * S + s;
        const double d = grad_in(dy, gate, dtype, i);
        const double xh = (widen(x, dtype, i) - mean[ng]) * rstd[ng];
        nsum_add(&sg, d * gam);
        nsum_add(&sgx, d * gam * xh);
        nsum_add(&sdy, d);
        nsum_add(&sdyx, d * xh);
      }
      db_nc[nc] = nsum_val(&sdy);
      dg_nc[nc] = nsum_val(&sdyx);
    }
    a[ng] = M ? nsum_val(&sg) / (double)M : 0.0;
    b[ng] = M ? nsum_val(&sgx) / (double)M : 0.0;
  }
}

static double dx_of(double dyv, double xv, double mu, double r, double gam, double a, double b) {
  const double xh = (xv - mu) * r;
  return r * (dyv * gam - a - xh * b);
}

static void reduce_params(const double* dg_nc, const double* db_nc, int64_t N, int64_t C,
                          double* dgamma, double* dbeta) {
  for (int64_t c = 0; c < C; ++c) {
    nsum sg = {0, 0}, sb = {0, 0};
    for (int64_t n = 0; n < N; ++n) {
      nsum_add(&sg, dg_nc[n * C + c]);
      nsum_add(&sb, db_nc[n * C + c]);
    }
    if (dgamma) dgamma[c] = nsum_val(&sg);
    if (dbeta) dbeta[c] = nsum_val(&sb);
  }
}

static int backward_impl(const void* dy, const void* gate, const void* x, int dtype, const double* mean,
                         const double* rstd, const float* gamma, int64_t N, int64_t C, int64_t S,
                         int64_t G, double* dx, double* dgamma, double* dbeta) {
  if (check_shape(N, C, S, G)) return ORC_EINVAL;
  const int64_t NG = N * G, NC = N * C, Cg = C / G;
  double* a = (double*)malloc(sizeof(double) * (size_t)(NG + 1));
  double* b = (double*)malloc(sizeof(double) * (size_t)(NG + 1));
  double* dg = (double*)malloc(sizeof(double) * (size_t)(NC + 1));
  double* db = (double*)malloc(sizeof(double) * (size_t)(NC + 1));
  if (!a || !b || !dg || !db) { free(a); free(b); free(dg); free(db); return ORC_EINVAL; }
  bwd_sums(dy, gate, x, dtype, mean, rstd, gamma, N, C, S, G, a, b, dg, db);
  if (dx) {
#pragma omp parallel for schedule(static)
    for (int64_t nc = 0; nc < NC; ++nc) {
      const int64_t n = nc / C, c = nc % C, ng = n * G + c / Cg;
      const double gam = param(gamma, c, 1.0);
      for (int64_t s = 0; s < S; ++s) {
        const int64_t i = nc * S + s;
        dx[i] = dx_of(grad_in(dy, gate, dtype, i), widen(x, dtype, i), mean[ng], rstd[ng], gam, a[ng], b[ng]);
      }
    }
  }
  reduce_params(dg, db, N, C, dgamma, dbeta);
  free(a); free(b); free(dg); free(db);
  return ORC_OK;
}

/* Backward at given statistics (fp64 [N*G]).  dx: [N*C*S] fp64 or NULL;
 * dgamma/dbeta: [C] fp64 or NULL. */
int gn3d_oracle_backward(const void* dy, const void* x, int dtype, const double* mean,
                         const double* rstd, const float* gamma, int64_t N, int64_t C, int64_t S,
                         int64_t G, double* dx, double* dgamma, double* dbeta) {
  return backward_impl(dy, NULL, x, dtype, mean, rstd, gamma, N, C, S, G, dx, dgamma, dbeta);
}

/* Backward of relu(GroupNorm(x)): `out` is the forward's result (x's dtype). */
int gn3d_oracle_backward_relu(const void* dy, const void* x, const void* out, int dtype, const double* mean,
                              const double* rstd, const float* gamma, int64_t N, int64_t C, int64_t S,
                              int64_t G, double* dx, double* dgamma, double* dbeta) {
  if (!out) return ORC_EINVAL;
  return backward_impl(dy, out, x, dtype, mean, rstd, gamma, N, C, S, G, dx, dgamma, dbeta);
}

static int backward_at_impl(const void* dy, const void* gate, const void* x, int dtype, const double* mean,
                            const double* rstd, const float* gamma, int64_t N, int64_t C,
                            int64_t S, int64_t G, const int64_t* idx, int64_t k, double* dx,
                            double* dgamma, double* dbeta) {
  if (check_shape(N, C, S, G)) return ORC_EINVAL;
  const int64_t NG = N * G, NC = N * C, Cg = C / G, L = N * C * S;
  double* a = (double*)malloc(sizeof(double) * (size_t)(NG + 1));
  double* b = (double*)malloc(sizeof(double) * (size_t)(NG + 1));
  double* dg = (double*)malloc(sizeof(double) * (size_t)(NC + 1));
  double* db = (double*)malloc(sizeof(double) * (size_t)(NC + 1));
  if (!a || !b || !dg || !db) { free(a); free(b); free(dg); free(db); return ORC_EINVAL; }
  bwd_sums(dy, gate, x, dtype, mean, rstd, gamma, N, C, S, G, a, b, dg, db);
  int st = ORC_OK;
  for (int64_t j = 0; j < k; ++j) {
    const int64_t i = idx[j];
    if (i < 0 || i >= L) { st = ORC_EINVAL; break; }
    const int64_t nc = i / S, n = nc / C, c = nc % C, ng = n * G + c / Cg;
    dx[j] = dx_of(grad_in(dy, gate, dtype, i), widen(x, dtype, i), mean[ng], rstd[ng],
                  param(gamma, c, 1.0), a[ng], b[ng]);
  }
  reduce_params(dg, db, N, C, dgamma, dbeta);
  free(a); free(b); free(dg); free(db);
  return st;
}

/* Backward: dx at k flat indices only, dgamma/dbeta in full. */
int gn3d_oracle_backward_at(const void* dy, const void* x, int dtype, const double* mean,
                            const double* rstd, const float* gamma, int64_t N, int64_t C,
                            int64_t S, int64_t G, const int64_t* idx, int64_t k, double* dx,
                            double* dgamma, double* dbeta) {
  return backward_at_impl(dy, NULL, x, dtype, mean, rstd, gamma, N, C, S, G, idx, k, dx, dgamma, dbeta);
}

int gn3d_oracle_backward_relu_at(const void* dy, const void* x, const void* out, int dtype, const double* mean,
                                 const double* rstd, const float* gamma, int64_t N, int64_t C, int64_t S,
                                 int64_t G, const int64_t* idx, int64_t k, double* dx, double* dgamma,
                                 double* dbeta) {
  if (!out) return ORC_EINVAL;
  return backward_at_impl(dy, out, x, dtype, mean, rstd, gamma, N, C, S, G, idx, k, dx, dgamma, dbeta);
}

/* The backward's sums at given statistics: per group a = mean(g), b =
 * mean(g * xhat); per (n, c) row s1 = sum dy and s2 = sum dy * xhat (dbeta and
 * dgamma before the sum over n).  `gate` (the fused ReLU forward's result, or
 * NULL) zeroes dy where it is <= 0.  a, b: [N*G]; s1, s2: [N*C] (any may be NULL). */
int gn3d_oracle_backward_sums(const void* dy, const void* gate, const void* x, int dtype, const double* mean,
                              const double* rstd, const float* gamma, int64_t N, int64_t C, int64_t S, int64_t G,
                              double* a, double* b, double* s1, double* s2) {
  if (check_shape(N, C, S, G)) return ORC_EINVAL;
  const int64_t NG = N * G, NC = N * C;
  double* ta = (double*)malloc(sizeof(double) * (size_t)(NG + 1));
  double* tb = (double*)malloc(sizeof(double) * (size_t)(NG + 1));
  double* dg = (double*)malloc(sizeof(double) * (size_t)(NC + 1));
  double* db = (double*)malloc(sizeof(double) * (size_t)(NC + 1));
  if (!ta || !tb || !dg || !db) { free(ta); free(tb); free(dg); free(db); return ORC_EINVAL; }
  bwd_sums(dy, gate, x, dtype, mean, rstd, gamma, N, C, S, G, ta, tb, dg, db);
  if (a) memcpy(a, ta, sizeof(double) * (size_t)NG);
  if (b) memcpy(b, tb, sizeof(double) * (size_t)NG);
  if (s1) memcpy(s1, db, sizeof(double) * (size_t)NC);
  if (s2) memcpy(s2, dg, sizeof(double) * (size_t)NC);
  free(ta); free(tb); free(dg); free(db);
  return ORC_OK;
}

/* ------------------------------------------------------------- fused ReLU */

/* F.relu on values already rounded to the output type (widened to fp64):
 * out = (v < 0) ? +0 : v (NaN, +Inf and -0.0 pass; -Inf and negatives become +0). */
void gn3d_oracle_relu(const double* v, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (v[i] < 0.0) ? 0.0 : v[i];
}

/* -------------------------------------------------------- output rounding */

/* Round-to-nearest-even of an fp64 value to bf16 (8 significant bits,
 * fp32's exponent range), done directly from fp64 -- not through fp32, which
 * would round twice.  Returns the bf16 bit pattern. */
static uint16_t round_bf16(double v) {
  if (isnan(v)) return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
  const uint16_t sign = (uint16_t)(signbit(v) ? 0x8000u : 0u);
  double a = fabs(v);
  if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                     /* a = m * 2^e, 0.5 <= m < 1 */
  int q = e - 8;                    /* spacing of 8-bit significands at this binade */
  if (q < -133) q = -133;           /* bf16 subnormal spacing: 2^-126 * 2^-7 */
  double k = nearbyint(ldexp(a, -q));   /* exact scaling; nearbyint rounds half to even */
  double r = ldexp(k, q);
  if (r >= 0x1p128) return (uint16_t)(sign | 0x7F80u);  /* overflow to infinity */
  float f = (float)r;               /* exact: r has at most 8 significant bits */
  uint32_t bits;
  memcpy(&bits, &f, sizeof bits);
  return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFFu));
}

void gn3d_oracle_round_bf16(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = round_bf16(v[i]);
}

/* Round-to-nearest-even of fp64 to fp32 (the C conversion, default rounding). */
void gn3d_oracle_round_f32(const double* v, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (float)v[i];
}
