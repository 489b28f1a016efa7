/*
 * gn3d.h -- C ABI of libgn3d: GroupNorm forward and backward over contiguous
 * NCDHW volumes on an NVIDIA GB300 (sm_103a).
 *
 * (The entry points named *_ndhwc take the channels-last layout instead; see
 * their declaration below.)
 *
 * Operation (ScaFFold PR #93 "Optimize GroupNorm": a drop-in for torch's
 * nn.GroupNorm, same weight and bias; PR #105 "Preserve GroupNorm dtype":
 * statistics accumulated in fp32, the normalized value computed in fp32, only
 * the store narrows):
 *
 *   x has shape [N, C, D, H, W], contiguous.  Group (n, g), 0 <= g < G, is the
 *   channel block g*C/G .. (g+1)*C/G - 1 of sample n: M = (C/G)*D*H*W
 *   elements, one contiguous span.
 *     mean = sum(x)/M,  var = sum((x-mean)^2)/M  (biased),
 *     rstd = 1/sqrt(var + eps)
 *     y    = (x - mean) * rstd * gamma[c] + beta[c]
 *   Backward at the saved (mean, rstd), with xhat = (x-mean)*rstd and
 *   g = dy*gamma[c]:
 *     dx       = rstd * (g - mean_group(g) - xhat * mean_group(g*xhat))
 *     dgamma_c = sum over n and positions of dy*xhat,   dbeta_c = sum of dy
 *
 * Determinism: every reduction runs in a fixed order chosen from the shape
 * alone (never from the dtype, the GPU's SM count or timing) and no float
 * atomics are used, so repeated calls give bit-identical results, and fp32
 * and bf16 inputs that hold the same values give bit-identical mean, rstd,
 * dgamma and dbeta (PR #105: the launch plan takes no dtype).
 *
 * Conventions for every entry point:
 *   - Tensors are dense, contiguous NCDHW, in device memory of the CURRENT
 *     device (cudaSetDevice), 16-byte aligned.  A pointer on another device or
 *     in unregistered host memory is rejected with GN3D_ERR_DEVICE (PR #93's
 *     review found a kernel launched on the wrong device faulting; this library
 *     checks instead of switching devices).
 *   - gamma, beta, mean, rstd, dgamma, dbeta are fp32 arrays.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous with respect to the host and ordered on
 *     `stream`; results are ready when the stream reaches the call.
 *   - Ownership: the caller owns every buffer; the library keeps no pointer
 *     after a call returns.  Per-call scratch is allocated and freed
 *     stream-ordered on `stream` (cudaMallocAsync / cudaFreeAsync), so calls
 *     can be captured into a CUDA graph and replayed (make one call on the
 *     device first, outside the capture).
 *   - Return value: GN3D_OK, or an error code below; on error nothing has been
 *     enqueued.  gn3d_error_string() describes the code and, for
 *     GN3D_ERR_CUDA, the CUDA error of the calling thread's last failure.
 *   - Empty tensors (N, C or D*H*W zero) are a successful no-op, except that
 *     dgamma/dbeta are zero-filled and, for M == 0 groups, mean = 0 and
 *     rstd = 1/sqrt(eps) are written.
 *   - Shapes with N*(C/G)*D*H*W == 1 are rejected (GN3D_ERR_INVALID_ARG), as
 *     stock GroupNorm raises for them (PR #93 review: "(1,C,1,1,1) ... where
 *     stock raises").
 */
#ifndef GN3D_H_
#define GN3D_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GN3D_F32 = 0, GN3D_BF16 = 1 } gn3d_dtype;

enum {
  GN3D_OK = 0,
  GN3D_ERR_INVALID_ARG = 1, /* bad shape, dtype, NULL required pointer, misalignment */
  GN3D_ERR_DEVICE = 2,      /* a pointer is not device memory of the current device */
  GN3D_ERR_CUDA = 3,        /* a CUDA runtime call (allocation, launch) failed */
  GN3D_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (see gn3d_stream_status) */
};

/*
 * GroupNorm forward.
 *   x      [N,C,D,H,W] in_dtype, read only.
 *   gamma  [C] fp32 or NULL (gamma = 1);  beta [C] fp32 or NULL (beta = 0).
 *   G      number of groups, G >= 1, C % G == 0.
 *   eps    added to the variance inside the square root; used as its fp32
 *          value (finite, >= 0).
 *   in_dtype / out_dtype: GN3D_BF16 or GN3D_F32, any pair.  y is the fp32
 *          result rounded once (round to nearest even) to out_dtype.
 *   y      [N,C,D,H,W] out_dtype, written; must not overlap x.
 *   mean, rstd  [N*G] fp32 (row-major (n, g)), written, or NULL (not saved).
 */
int gn3d_forward(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                 int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                 gn3d_dtype out_dtype, void* y, float* mean, float* rstd, void* stream);

/*
 * GroupNorm forward that allocates nothing.  The pages have no counterpart of
 * this entry point; it exists for callers that must not allocate device memory
 * during the call -- for example code running under a fixed memory budget, or
 * inside another allocator's critical section, where cudaMalloc (which may
 * synchronize the device) or a stream-ordered pool allocation is not allowed.
 *
 * Same arguments, results and errors as gn3d_forward (computed by the
 * persistent forward kernel, whose results are bit-identical to the streaming
 * kernels'), except:
 *   - Scratch comes from a static area of 8 MiB inside the library's device
 *     code, which every GPU that loads the library holds until the process
 *     exits.  The scratch is about 17 bytes per 4096 elements of each (n, c)
 *     row, so up to about 2 billion elements fit when rows are long, fewer
 *     when D*H*W is small.  A shape whose scratch would not fit is rejected
 *     with GN3D_ERR_INVALID_ARG, and gn3d_error_string says how many bytes it
 *     needed.  Empty tensors are rejected too.
 *   - The first call on a device looks up the area's device address; make that
 *     first call before any stream capture.
 *   - All calls share the one area (each call clears the counters it needs), so
 *     calls that can overlap on the GPU -- on different streams, or from
 *     different threads -- race and give wrong results.  Serialize them.
 * No cudaMalloc, cudaFree or memory-pool call is made.
 */
int gn3d_forward_noalloc(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                         int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                         gn3d_dtype out_dtype, void* y, float* mean, float* rstd, void* stream);

/*
 * GroupNorm backward at the forward's saved statistics.
 *   dy, x  [N,C,D,H,W] dtype, read only.
 *   mean, rstd  [N*G] fp32 as written by gn3d_forward for the same x, G, eps.
 *   gamma  [C] fp32 or NULL (gamma = 1).
 *   dx     [N,C,D,H,W] dtype, written (the fp32 result rounded once); must not
 *          overlap dy or x.
 *   dgamma, dbeta  [C] fp32, written (overwritten, not accumulated), or NULL.
 */
int gn3d_backward(const void* dy, const void* x, const float* mean, const float* rstd,
                  const float* gamma, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                  int64_t G, gn3d_dtype dtype, void* dx, float* dgamma, float* dbeta,
                  void* stream);

/*
 * GroupNorm followed by ReLU, the ReLU fused into the store (the ScaFFold
 * GroupNorm pages move the ReLU that follows every GroupNorm of the UNet inside
 * it: FastGroupNorm's activation argument).  Same arguments, errors, mean and
 * rstd as gn3d_forward; `out` receives F.relu of the rounded GroupNorm result,
 *   out = v < 0 ? +0 : v,   v = y rounded once to out_dtype,
 * so NaN, +Inf and -0.0 pass and -Inf and every other negative become +0: bit
 * for bit gn3d_forward followed by F.relu on its output (the pages' fix makes the
 * fused ReLU match F.relu on NaN, both infinities and -0.0).  Always runs the
 * streaming kernels (GN3D_DEBUG_PATH 2 does not apply to it).
 */
int gn3d_forward_relu(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                      int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                      gn3d_dtype out_dtype, void* out, float* mean, float* rstd, void* stream);

/*
 * Backward of relu(GroupNorm(x)).
 *   out  [N,C,D,H,W] dtype (the dtype of x, dy and dx), read only: the
 *        forward's result (gn3d_forward_relu's out).  The gradient reaching
 *        GroupNorm is torch's threshold_backward on it: dy where out is not <= 0
 *        (a NaN result passes the gradient, as the pages' fix requires), 0 where
 *        out <= 0 (either zero included).
 * Everything else as gn3d_backward; the results are bit for bit gn3d_backward's
 * on that gated dy.  dx must not overlap out.  Always runs the streaming kernels.
 */
int gn3d_backward_relu(const void* dy, const void* x, const void* out, const float* mean,
                       const float* rstd, const float* gamma, int64_t N, int64_t C, int64_t D,
                       int64_t H, int64_t W, int64_t G, gn3d_dtype dtype, void* dx, float* dgamma,
                       float* dbeta, void* stream);

/*
 * Channels-last (NDHWC) layout: the same four operations on tensors stored as
 * x[n][d][h][w][c] -- the channels_last_3d memory format of an [N,C,D,H,W]
 * tensor, as channels-last convolutions produce it (the ScaFFold GroupNorm
 * pages' Triton kernel reads channels-last activations: a dense run of
 * positions x C channels viewed as (G, C/G); their layout-tax measurements show
 * a layout conversion around GroupNorm costing more than GroupNorm itself).
 * Element (n, c, d, h, w) is at offset ((n*D + d)*H + h)*W + w)*C + c; group
 * (n, g) is channels g*C/G .. (g+1)*C/G - 1 of every position of sample n.
 *   - Same arguments, formulas, dtypes, ownership, empty-tensor handling and
 *     errors as gn3d_forward / gn3d_forward_relu / gn3d_backward /
 *     gn3d_backward_relu; y, dx, out and dy use the same NDHWC layout as x, and
 *     mean, rstd ([N*G]), gamma, beta, dgamma, dbeta ([C]) are unchanged.
 *   - C must be a multiple of 8 (a 16-byte vector then holds 8 channels of one
 *     position); otherwise GN3D_ERR_INVALID_ARG.
 *   - Deterministic (a fixed reduction order chosen from the shape alone; no
 *     float atomics).  The order differs from the NCDHW entry points', so the
 *     two layouts agree to rounding, not bit for bit.
 *   - Three kernels per direction: k_ndhwc_stats, k_ndhwc_stats_final,
 *     k_ndhwc_norm forward; k_ndhwc_reduce, k_ndhwc_reduce_final, k_ndhwc_dx
 *     backward.  GN3D_DEBUG_PATH does not apply.
 */
int gn3d_forward_ndhwc(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                       int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                       gn3d_dtype out_dtype, void* y, float* mean, float* rstd, void* stream);

int gn3d_forward_ndhwc_relu(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C,
                            int64_t D, int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype,
                            gn3d_dtype out_dtype, void* out, float* mean, float* rstd, void* stream);

int gn3d_backward_ndhwc(const void* dy, const void* x, const float* mean, const float* rstd,
                        const float* gamma, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W,
                        int64_t G, gn3d_dtype dtype, void* dx, float* dgamma, float* dbeta,
                        void* stream);

int gn3d_backward_ndhwc_relu(const void* dy, const void* x, const void* out, const float* mean,
                             const float* rstd, const float* gamma, int64_t N, int64_t C, int64_t D,
                             int64_t H, int64_t W, int64_t G, gn3d_dtype dtype, void* dx, float* dgamma,
                             float* dbeta, void* stream);

/*
 * Global statistics under spatial sharding, and a backward driven by
 * externally produced sums.
 *
 * A volume split into shards -- e.g. one D-slab per rank under DistConv, each
 * held as its own contiguous [N, C, D_k, H, W] tensor -- needs the GroupNorm
 * of the whole volume, whose statistics span every shard.  The ScaFFold
 * GroupNorm pages (PR #93, the commit that unwraps DCTensors) normalize each
 * shard with its own statistics and leave global statistics as an open
 * question; these entry points implement the one exchange per direction that
 * gives the whole volume's result:
 *
 *   forward:  gn3d_forward_moments on each shard -> exchange the [N*G]
 *             moments (e.g. all-gather, rank order) -> gn3d_moments_combine
 *             -> gn3d_forward_apply on each shard with the combined moments;
 *   backward: gn3d_backward_sums on each shard at the global (mean, rstd) ->
 *             exchange the [N*C] sums -> gn3d_sums_combine ->
 *             gn3d_backward_dx_from_sums on each shard with the totals.
 *
 * The moments of a group are combined in rank order with the parallel-variance
 * merge of Chan, Golub and LeVeque (the merge the pages name for partial
 * statistics), in the shifted-sum form used by every merge of this library;
 * the sums are added in rank order.  With one shard every combine is the
 * identity and the results are bit-identical to gn3d_forward / gn3d_backward.
 * The exchange itself is the caller's (this library makes no collective
 * call).  NCDHW layout, no fused ReLU.  All pointers are device memory of the
 * current device; calls are ordered on `stream`.
 *
 * gn3d_backward_dx_from_sums is also the dx pass for a caller that produces
 * the backward's sums itself (for example fused into the kernel that produces
 * dy): it reads x and dy once and writes dx, with no reduction pass.
 */
typedef struct {
  int64_t count;   /* elements of the group in this shard */
  float mean_hi;   /* the group mean is mean_hi + mean_lo (an unevaluated pair) */
  float mean_lo;
  float m2;        /* sum of (x - mean)^2 */
  float reserved;
} gn3d_moments;    /* 24 bytes */

/* Per group (n, g) moments of x [N,C,D,H,W] (a shard): moments[n*G + g].
 * x 16-byte aligned, moments 8-byte aligned.  A shard may hold any number of a
 * group's elements (zero gives count 0). */
int gn3d_forward_moments(const void* x, int64_t N, int64_t C, int64_t D, int64_t H, int64_t W, int64_t G,
                         gn3d_dtype in_dtype, gn3d_moments* moments, void* stream);

/* Combine K shards' moments, shards[k*NG + i] (rank-major), per group i in rank
 * order into combined[i] (may not alias shards). */
int gn3d_moments_combine(const gn3d_moments* shards, int64_t K, int64_t NG, gn3d_moments* combined, void* stream);

/* The forward's normalize pass of a shard with the whole volume's moments
 * [N*G]: y as gn3d_forward writes it, and mean [N*G] / rstd [N*G] (either may
 * be NULL) with rstd = 1/sqrt(M2/count + eps). */
int gn3d_forward_apply(const void* x, const float* gamma, const float* beta, int64_t N, int64_t C, int64_t D,
                       int64_t H, int64_t W, int64_t G, double eps, gn3d_dtype in_dtype, gn3d_dtype out_dtype,
                       const gn3d_moments* moments, void* y, float* mean, float* rstd, void* stream);

/* Per row (n, c) of a shard at the given (global) statistics: sums[2*(n*C+c)] =
 * sum dy, sums[2*(n*C+c)+1] = sum dy*(x - mean).  dy, x 16-byte aligned, sums
 * 8-byte aligned. */
int gn3d_backward_sums(const void* dy, const void* x, const float* mean, const float* rstd, int64_t N, int64_t C,
                       int64_t D, int64_t H, int64_t W, int64_t G, gn3d_dtype dtype, float* sums, void* stream);

/* Add K shards' row sums, shards[(k*NC + r)*2 + {0,1}], per row in rank order
 * into total[NC*2] (may not alias shards). */
int gn3d_sums_combine(const float* shards, int64_t K, int64_t NC, float* total, void* stream);

/* The backward's dx pass of a shard from the whole volume's row sums
 * [N*C*2] (as gn3d_backward_sums defines them): with M = group_count (the
 * elements of one group of the whole volume), per group a = A/M, b = B/M with
 * A = sum_c gamma_c*S1_c, B = rstd * sum_c gamma_c*S2_c, and dx = rstd*((dy*gamma
 * - a) - xhat*b); dgamma_c = sum_n rstd*S2, dbeta_c = sum_n S1 (either may be
 * NULL).  GN3D_ERR_INVALID_ARG if group_count < 1. */
int gn3d_backward_dx_from_sums(const void* dy, const void* x, const float* mean, const float* rstd,
                               const float* gamma, const float* sums, int64_t group_count, int64_t N, int64_t C,
                               int64_t D, int64_t H, int64_t W, int64_t G, gn3d_dtype dtype, void* dx,
                               float* dgamma, float* dbeta, void* stream);

/*
 * Synchronizes `stream`, then returns and clears the device-side error word
 * that bounded waits inside the kernels set (GN3D_ERR_TIMEOUT), or
 * GN3D_ERR_CUDA if the stream reports a CUDA error, else GN3D_OK.
 */
int gn3d_stream_status(void* stream);

/* Static description of a status code (thread-local detail for GN3D_ERR_CUDA). */
const char* gn3d_error_string(int status);

/* Number of CUDA kernels libgn3d has launched in this process, all devices and
 * threads together (diagnostics: lets a caller count the kernels of a timed
 * region).  Memory-set and copy operations are not counted. */
uint64_t gn3d_launch_count(void);

#ifdef GN3D_TESTING
/*
 * Testing and tuning hooks, present only in the testing build of the library
 * (compiled with GN3D_TESTING; the tests load it, the shipped library has none
 * of them).  Process-wide, not thread-scoped; every setting defaults to
 * automatic.  None of them changes a result bit: every launch form runs the
 * same units and reduction trees.
 *   GN3D_DEBUG_PATH          0 automatic (the cluster kernels where they
 *                            apply -- whole 4096-element units, a group held
 *                            in the shared memory of one cluster of at most 16
 *                            CTAs, every group's cluster resident at once, no
 *                            fused ReLU in the backward -- else the
 *                            streaming kernels: two launches per direction),
 *                            1 streaming, 2 persistent (one cooperative launch
 *                            per direction), 4 cluster where they apply (else
 *                            streaming), 3 group-wave
 *                            (one cooperative launch per direction; every CTA
 *                            holds a share of every group in shared memory
 *                            between the two passes; shapes whose rows are
 *                            whole 4096-element units, and not the fused-ReLU
 *                            or fp32 backward, which stay on the streaming
 *                            kernels).
 *   GN3D_DEBUG_SPIN_LIMIT    poll budget of every bounded device-side wait
 *                            (0 = default, about four seconds).  A kernel
 *                            whose wait gave up still waits for its own bulk
 *                            copies in flight with the default budget before
 *                            it exits.
 *   GN3D_DEBUG_FORCE_TIMEOUT 1: the next persistent, group-wave or cluster
 *                            launch (or the next channels-last statistics
 *                            launch with C <= 256)
 *                            waits for a flag that nothing sets, so its bounded
 *                            wait runs out and gn3d_stream_status reports
 *                            GN3D_ERR_TIMEOUT (tests the failure path without a
 *                            fault or a hang).
 *   GN3D_DEBUG_LAG           -1 automatic, else 0 .. 8: groups of lookahead
 *                            between the statistics pass and the elementwise pass.
 *   GN3D_DEBUG_SLOTS         -1 automatic, else the number of shared-memory
 *                            slots of the persistent kernels (at most what fits).
 *   GN3D_DEBUG_SHARES        -1 automatic, 0 strided blocks, 1 unit shares:
 *                            how the NCDHW streaming kernels split the units
 *                            among their warps (whole merge blocks dealt out in
 *                            turn, or equal contiguous runs of units that may
 *                            cut a block between two warps).  Placement only.
 *   GN3D_DEBUG_RES_HELD      -1 automatic, else >= 0: units of each CTA's share
 *                            of a group the group-wave kernels keep in shared
 *                            memory (the others are read again from L2).
 *   GN3D_DEBUG_RES_WINDOW    -1 automatic, else >= 1: units the group-wave
 *                            producer may run ahead of the elementwise pass (at
 *                            least one share of a group is always allowed).
 *   GN3D_DEBUG_RES_PASS      -1 automatic, else >= 1: slots of the group-wave
 *                            kernels' pass ring (rounded up to a multiple of
 *                            their reduction warps).
 *   GN3D_DEBUG_FAIL_NEXT     1: the next per-call scratch allocation fails as an
 *                            out-of-memory would; 2: the next call's first
 *                            kernel launch fails; 0 disarms.  The call returns
 *                            GN3D_ERR_CUDA having enqueued no kernel and freed
 *                            its scratch (a host-side fault injection: nothing
 *                            faults on the GPU).
 * Returns GN3D_OK or GN3D_ERR_INVALID_ARG for an unknown setting or value.
 */
enum {
  GN3D_DEBUG_PATH = 0,
  GN3D_DEBUG_SPIN_LIMIT = 1,
  GN3D_DEBUG_FORCE_TIMEOUT = 2,
  GN3D_DEBUG_LAG = 3,
  GN3D_DEBUG_SLOTS = 4,
  GN3D_DEBUG_SHARES = 6,
  GN3D_DEBUG_RES_HELD = 7,
  GN3D_DEBUG_RES_WINDOW = 8,
  GN3D_DEBUG_RES_PASS = 9,
  GN3D_DEBUG_FAIL_NEXT = 10
};
int gn3d_debug_set(int what, long long value);

/* Testing build: GN3D_DEBUG_POOL_USED writes the bytes currently allocated from
 * the current device's scratch pool (0 once every call's scratch is freed and
 * the stream has reached the frees).  GN3D_OK or GN3D_ERR_INVALID_ARG. */
enum { GN3D_DEBUG_POOL_USED = 0 };
int gn3d_debug_get(int what, long long* value);
#endif /* GN3D_TESTING */

/*
 * Per-kernel timing (diagnostics): gn3d_timing(1) clears the recorded times
 * and starts recording -- every kernel launch is then bracketed by two CUDA
 * events on its stream (see gn3d_kernel_time); gn3d_timing(0) stops.  Returns
 * GN3D_OK or GN3D_ERR_INVALID_ARG (value other than 0 or 1).
 */
int gn3d_timing(int on);

/*
 * Device time of one kernel, summed over the launches recorded since
 * gn3d_timing(1) was last called.  `name` is one of "k_fwd_fused",
 * "k_bwd_fused", "k_fwd_stats", "k_fwd_norm", "k_bwd_reduce", "k_bwd_dx",
 * "k_ndhwc_stats", "k_ndhwc_stats_final", "k_ndhwc_norm", "k_ndhwc_reduce",
 * "k_ndhwc_reduce_final", "k_ndhwc_dx", "k_fwd_resident", "k_bwd_resident",
 * "k_fwd_cluster", "k_bwd_cluster".
 * Waits for the recorded events (host-blocking), then writes the total
 * milliseconds to *ms and the launch count to *launches.  Returns GN3D_OK,
 * GN3D_ERR_INVALID_ARG (NULL argument, unknown name) or GN3D_ERR_CUDA.
 */
int gn3d_kernel_time(const char* name, double* ms, uint64_t* launches);

/* Library version, e.g. "gn3d 0.4.0 sm_103a". */
const char* gn3d_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GN3D_H_ */
