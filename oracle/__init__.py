"""fp64 CPU oracle for GroupNorm-3D forward/backward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg import this package.  The CUDA library never does, and this
package never imports the library: the two share no code.  The arithmetic
lives in ``gn3d_oracle.c`` (plain C, fp64, compensated sums); this module only
compiles it with gcc and marshals numpy arrays through ctypes.

Functions (all cite the ScaFFold pages' GroupNorm definition; see the C file):
  stats(x, dtype, N, C, S, G, eps)            -> mean, var, rstd   (fp64 [N*G])
  forward(x, dtype, gamma, beta, N, C, S, G, eps) -> y64, mean, rstd
  forward_at(..., mean, rstd, idx)             -> y64 at flat indices
  backward(dy, x, dtype, mean, rstd, gamma, N, C, S, G) -> dx64, dgamma, dbeta
  backward_at(..., idx)                        -> dx64 at indices, dgamma, dbeta
  backward_sums(dy, x, mean, rstd, gamma, N, C, S, G, out=None)
                                               -> a, b (per group), s1 = sum dy, s2 = sum dy*xhat (per row)
  backward_relu / backward_relu_at             -> the backward behind the fused ReLU (out: its result)
  moments(x, N, C, S, G) / combine_moments(list) -> sharded statistics: per-shard (count, mean, M2),
                                               combined in rank order (Chan's parallel formula)
  round_bf16(v64) -> uint16 bit patterns (RNE straight from fp64)
  round_f32(v64)  -> float32 (RNE)
Channels-last (NDHWC) tensors: the same GroupNorm of the same logical tensor,
only stored position-major (element (n, c, s) at flat index (n*S + s)*C + c).
  ndhwc_to_ncdhw(a, N, C, S) / ncdhw_to_ndhwc(a, N, C, S)  -> the layout change
  ndhwc_index(idx, N, C, S)  -> NCDHW flat indices of NDHWC flat indices
  forward_ndhwc / backward_ndhwc / backward_relu_ndhwc  -> as above, NDHWC in/out
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gn3d_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libgn3d_oracle.so")

F32, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """gcc -> shared library, with the oracle's flags (OpenMP, no FMA contraction,
    IEEE math).  The tests also use it to build deliberately broken copies."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle (once; again when the source is newer)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        compile_source(_SRC, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # GN3D_ORACLE_LIB: a library built from a modified copy of the source
            # (tests/test_oracle_mutants.py checks that the pins reject such copies)
            lib = ctypes.CDLL(os.environ.get("GN3D_ORACLE_LIB") or build())
            i64, vp, dp, fp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            lib.gn3d_oracle_stats.argtypes = [vp, ctypes.c_int, i64, i64, i64, i64, ctypes.c_double, dp, dp, dp]
            lib.gn3d_oracle_forward.argtypes = [vp, ctypes.c_int, fp, fp, i64, i64, i64, i64,
                                                ctypes.c_double, dp, dp, dp]
            lib.gn3d_oracle_forward_at.argtypes = [vp, ctypes.c_int, fp, fp, i64, i64, i64, i64, dp, dp,
                                                   vp, i64, dp]
            lib.gn3d_oracle_backward.argtypes = [vp, vp, ctypes.c_int, dp, dp, fp, i64, i64, i64, i64,
                                                 dp, dp, dp]
            lib.gn3d_oracle_backward_at.argtypes = [vp, vp, ctypes.c_int, dp, dp, fp, i64, i64, i64, i64,
                                                    vp, i64, dp, dp, dp]
            lib.gn3d_oracle_backward_relu.argtypes = [vp, vp, vp, ctypes.c_int, dp, dp, fp, i64, i64, i64, i64,
                                                      dp, dp, dp]
            lib.gn3d_oracle_backward_relu_at.argtypes = [vp, vp, vp, ctypes.c_int, dp, dp, fp, i64, i64, i64,
                                                         i64, vp, i64, dp, dp, dp]
            lib.gn3d_oracle_backward_sums.argtypes = [vp, vp, vp, ctypes.c_int, dp, dp, fp, i64, i64, i64, i64,
                                                      dp, dp, dp, dp]
            lib.gn3d_oracle_relu.argtypes = [dp, i64, dp]
            lib.gn3d_oracle_relu.restype = None
            lib.gn3d_oracle_round_bf16.argtypes = [dp, i64, vp]
            lib.gn3d_oracle_round_f32.argtypes = [dp, i64, fp]
            for f in ("stats", "forward", "forward_at", "backward", "backward_at", "backward_relu",
                      "backward_relu_at", "backward_sums"):
                getattr(lib, "gn3d_oracle_" + f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _raw(x: np.ndarray):
    """Input bytes as the GPU sees them: float32 array, or uint16 bf16 bit patterns."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"oracle inputs are float32 or uint16 (bf16 bits), got {x.dtype}")


def _params(p):
    return None if p is None else np.ascontiguousarray(p, dtype=np.float32)


def _check(rc):
    if rc != 0:
        raise ValueError("oracle rejected the arguments")


def stats(x, N, C, S, G, eps):
    xr, dt = _raw(x)
    mean, var, rstd = (np.empty(N * G) for _ in range(3))
    _check(_load().gn3d_oracle_stats(_ptr(xr), dt, N, C, S, G, eps, _ptr(mean), _ptr(var), _ptr(rstd)))
    return mean, var, rstd


def forward(x, gamma, beta, N, C, S, G, eps):
    xr, dt = _raw(x)
    g, b = _params(gamma), _params(beta)
    y = np.empty(N * C * S)
    mean, rstd = np.empty(N * G), np.empty(N * G)
    _check(_load().gn3d_oracle_forward(_ptr(xr), dt, _ptr(g), _ptr(b), N, C, S, G, eps, _ptr(y),
                                       _ptr(mean), _ptr(rstd)))
    return y, mean, rstd


def forward_at(x, gamma, beta, N, C, S, G, mean, rstd, idx):
    xr, dt = _raw(x)
    g, b = _params(gamma), _params(beta)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    y = np.empty(idx.size)
    _check(_load().gn3d_oracle_forward_at(_ptr(xr), dt, _ptr(g), _ptr(b), N, C, S, G, _ptr(mean),
                                          _ptr(rstd), _ptr(idx), idx.size, _ptr(y)))
    return y


def backward(dy, x, mean, rstd, gamma, N, C, S, G, want_dx=True):
    xr, dt = _raw(x)
    dyr, dt2 = _raw(dy)
    if dt != dt2:
        raise TypeError("dy and x must share a dtype")
    g = _params(gamma)
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    dx = np.empty(N * C * S) if want_dx else None
    dgamma, dbeta = np.empty(C), np.empty(C)
    _check(_load().gn3d_oracle_backward(_ptr(dyr), _ptr(xr), dt, _ptr(mean), _ptr(rstd), _ptr(g),
                                        N, C, S, G, _ptr(dx), _ptr(dgamma), _ptr(dbeta)))
    return dx, dgamma, dbeta


def backward_at(dy, x, mean, rstd, gamma, N, C, S, G, idx):
    xr, dt = _raw(x)
    dyr, _ = _raw(dy)
    g = _params(gamma)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    dx = np.empty(idx.size)
    dgamma, dbeta = np.empty(C), np.empty(C)
    _check(_load().gn3d_oracle_backward_at(_ptr(dyr), _ptr(xr), dt, _ptr(mean), _ptr(rstd), _ptr(g),
                                           N, C, S, G, _ptr(idx), idx.size, _ptr(dx), _ptr(dgamma),
                                           _ptr(dbeta)))
    return dx, dgamma, dbeta


def backward_sums(dy, x, mean, rstd, gamma, N, C, S, G, out=None):
    """The backward's sums at given statistics: a = mean(dy*gamma), b =
    mean(dy*gamma*xhat) per group [N*G]; s1 = sum dy, s2 = sum dy*xhat per row
    (n, c) [N*C].  With `out` (the fused ReLU forward's result), dy is zeroed
    where out <= 0 first."""
    xr, dt = _raw(x)
    dyr, dt2 = _raw(dy)
    outr = None
    if out is not None:
        outr, dt3 = _raw(out)
        if dt3 != dt:
            raise TypeError("out must share x's dtype")
    if dt != dt2:
        raise TypeError("dy and x must share a dtype")
    g = _params(gamma)
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    a, b = np.empty(N * G), np.empty(N * G)
    s1, s2 = np.empty(N * C), np.empty(N * C)
    _check(_load().gn3d_oracle_backward_sums(_ptr(dyr), _ptr(outr), _ptr(xr), dt, _ptr(mean), _ptr(rstd), _ptr(g),
                                             N, C, S, G, _ptr(a), _ptr(b), _ptr(s1), _ptr(s2)))
    return a, b, s1, s2


# ------------------------------------------------------- sharded statistics
# A volume cut into K shards along D (each rank's slab, its own contiguous
# [N, C, D_k, H, W] tensor) has per-shard moments (count, mean, M2) per group;
# the global statistics are those moments combined in rank order with the
# parallel-variance formula of Chan, Golub and LeVeque, which the ScaFFold
# GroupNorm pages name for merging partial statistics.

def moments(x, N, C, S, G):
    """Per group (n, g) of this tensor: count, mean and M2 = sum (x - mean)^2,
    fp64 (the definition: two compensated passes, as stats())."""
    mean, var, _ = stats(x, N, C, S, G, 0.0)
    count = np.full(N * G, (C // G) * S, dtype=np.float64)
    return count, mean, var * count


def combine_moments(parts):
    """Combine [(count, mean, M2), ...] (one per shard, rank order) pairwise left
    to right: n = na + nb, d = mb - ma, mean = ma + d*nb/n, M2 = M2a + M2b +
    d^2*na*nb/n.  Returns (count, mean, M2)."""
    n, m, q = (np.array(v, dtype=np.float64) for v in parts[0])
    for nb, mb, qb in parts[1:]:
        nb, mb, qb = (np.asarray(v, dtype=np.float64) for v in (nb, mb, qb))
        tot = n + nb
        safe = np.where(tot > 0, tot, 1.0)
        d = mb - m
        m = np.where(tot > 0, m + d * nb / safe, 0.0)
        q = q + qb + np.where(tot > 0, d * d * n * nb / safe, 0.0)
        n = tot
    return n, m, q


def rstd_of(count, M2, eps):
    """rstd = 1/sqrt(M2/count + eps), eps used at its fp32 value (as the library does)."""
    var = np.where(count > 0, M2 / np.where(count > 0, count, 1.0), 0.0)
    return 1.0 / np.sqrt(var + float(np.float32(eps)))


def relu(v):
    """F.relu on output values already rounded to the output type (as fp64):
    out = (v < 0) ? +0 : v -- the fused ReLU's forward, applied after the rounding."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape)
    _load().gn3d_oracle_relu(_ptr(v), v.size, _ptr(out))
    return out


def backward_relu(dy, x, out, mean, rstd, gamma, N, C, S, G, want_dx=True):
    """Backward of relu(GroupNorm(x)) at given statistics; `out` is the forward's
    result in x's dtype (float32, or uint16 bf16 bits)."""
    xr, dt = _raw(x)
    dyr, dt2 = _raw(dy)
    outr, dt3 = _raw(out)
    if not dt == dt2 == dt3:
        raise TypeError("dy, x and out must share a dtype")
    g = _params(gamma)
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    dx = np.empty(N * C * S) if want_dx else None
    dgamma, dbeta = np.empty(C), np.empty(C)
    _check(_load().gn3d_oracle_backward_relu(_ptr(dyr), _ptr(xr), _ptr(outr), dt, _ptr(mean), _ptr(rstd),
                                             _ptr(g), N, C, S, G, _ptr(dx), _ptr(dgamma), _ptr(dbeta)))
    return dx, dgamma, dbeta


def backward_relu_at(dy, x, out, mean, rstd, gamma, N, C, S, G, idx):
    xr, dt = _raw(x)
    dyr, _ = _raw(dy)
    outr, _ = _raw(out)
    g = _params(gamma)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    mean = np.ascontiguousarray(mean, dtype=np.float64)
    rstd = np.ascontiguousarray(rstd, dtype=np.float64)
    dx = np.empty(idx.size)
    dgamma, dbeta = np.empty(C), np.empty(C)
    _check(_load().gn3d_oracle_backward_relu_at(_ptr(dyr), _ptr(xr), _ptr(outr), dt, _ptr(mean), _ptr(rstd),
                                                _ptr(g), N, C, S, G, _ptr(idx), idx.size, _ptr(dx),
                                                _ptr(dgamma), _ptr(dbeta)))
    return dx, dgamma, dbeta


def round_bf16(v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().gn3d_oracle_round_bf16(_ptr(v), v.size, _ptr(out))
    return out


def round_f32(v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.float32)
    _load().gn3d_oracle_round_f32(_ptr(v), v.size, _ptr(out))
    return out


# ------------------------------------------------------- channels-last layout
# GroupNorm is defined on the logical tensor [N, C, D, H, W]; a channels-last
# (NDHWC) tensor is the same tensor stored position-major.  These adapters only
# move elements between the two storage orders and call the functions above.

def ndhwc_to_ncdhw(a, N, C, S):
    """Flat NDHWC storage -> flat NCDHW storage (same values, same dtype)."""
    return np.ascontiguousarray(np.asarray(a).reshape(N, S, C).transpose(0, 2, 1)).reshape(-1)


def ncdhw_to_ndhwc(a, N, C, S):
    """Flat NCDHW storage -> flat NDHWC storage."""
    return np.ascontiguousarray(np.asarray(a).reshape(N, C, S).transpose(0, 2, 1)).reshape(-1)


def ndhwc_index(idx, N, C, S):
    """NCDHW flat index of each NDHWC flat index: (n*S + s)*C + c -> (n*C + c)*S + s."""
    idx = np.asarray(idx, dtype=np.int64)
    c = idx % C
    ns = idx // C
    n, s_ = ns // S, ns % S
    return (n * C + c) * S + s_


def forward_ndhwc(x, gamma, beta, N, C, S, G, eps):
    """y64 (NDHWC), mean, rstd of GroupNorm of an NDHWC tensor."""
    y, mean, rstd = forward(ndhwc_to_ncdhw(x, N, C, S), gamma, beta, N, C, S, G, eps)
    return ncdhw_to_ndhwc(y, N, C, S), mean, rstd


def backward_ndhwc(dy, x, mean, rstd, gamma, N, C, S, G, want_dx=True):
    """dx64 (NDHWC), dgamma, dbeta of GroupNorm of an NDHWC tensor."""
    dx, dgamma, dbeta = backward(ndhwc_to_ncdhw(dy, N, C, S), ndhwc_to_ncdhw(x, N, C, S), mean, rstd, gamma, N,
                                 C, S, G, want_dx)
    return (ncdhw_to_ndhwc(dx, N, C, S) if want_dx else None), dgamma, dbeta


def backward_relu_ndhwc(dy, x, out, mean, rstd, gamma, N, C, S, G, want_dx=True):
    """Backward of relu(GroupNorm(x)) for NDHWC tensors (out: the forward's result, NDHWC)."""
    dx, dgamma, dbeta = backward_relu(ndhwc_to_ncdhw(dy, N, C, S), ndhwc_to_ncdhw(x, N, C, S),
                                      ndhwc_to_ncdhw(out, N, C, S), mean, rstd, gamma, N, C, S, G, want_dx)
    return (ncdhw_to_ndhwc(dx, N, C, S) if want_dx else None), dgamma, dbeta
