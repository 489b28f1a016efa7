"""Comparison rules between the CUDA path and the fp64 oracle (test helpers).

Rules (the readings of the stated tolerances; the GroupNorm pages fix fp32
statistics/compute with one rounding on the store):
  * bf16 outputs: within 1 bf16 ulp (ordinal distance <= 1) of the fp64 result
    rounded once; or, where the fp32 evaluation of a cancelling sum cannot
    resolve 1 ulp of a tiny result, |gpu - ref| <= ulp_bf16(ref) + 2^-21 * T,
    T = the sum of the magnitudes that enter the fp32 evaluation.  Elements
    that needed the second clause are counted and reported.
  * fp32 outputs (y, dx): |gpu - ref| <= 1e-5 * |ref| + 1e-6, per element.
  * reductions (dgamma, dbeta, mean): |gpu - ref| <= 1e-5 * |ref| + 1e-6 * L2
    with L2 the 2-norm of the summed terms; rstd: 1e-5 relative.
"""
from __future__ import annotations

import numpy as np

from bwd_gn3d_stats_gb300.synth import bits_to_f32


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def check_bf16(gpu_bits, ref64, terms, round_bf16):
    """Returns (ok_mask, n_second_clause)."""
    gpu_bits = np.asarray(gpu_bits, dtype=np.uint16)
    ref_bits = round_bf16(ref64)
    ok1 = np.abs(bf16_ordinal(gpu_bits) - bf16_ordinal(ref_bits)) <= 1
    g = bits_to_f32(gpu_bits).astype(np.float64)
    ok2 = np.abs(g - ref64) <= ulp_bf16(ref64) + 2.0 ** -21 * terms
    nan_ok = np.isnan(g) & np.isnan(ref64)
    ok = ok1 | ok2 | nan_ok
    return ok, int(np.count_nonzero(~ok1 & ok2))


def check_f32(gpu, ref64, rel=1e-5, abs_=1e-6):
    g = np.asarray(gpu, dtype=np.float64)
    ok = np.abs(g - ref64) <= rel * np.abs(ref64) + abs_
    return ok | (np.isnan(g) & np.isnan(ref64))


def check_reduction(gpu, ref64, l2, rel=1e-5, abs_=1e-6):
    g = np.asarray(gpu, dtype=np.float64)
    return np.abs(g - ref64) <= rel * np.abs(ref64) + abs_ * l2


def y_terms(xv, mean, rstd, gamma, beta, N, C, S, G):
    """Magnitudes entering y = (x - mean) * (rstd*gamma) + beta, per element."""
    Cg = C // G
    ng = (np.arange(N * C) // Cg)
    c = np.arange(N * C) % C
    gm = np.ones(C) if gamma is None else np.abs(gamma.astype(np.float64))
    bt = np.zeros(C) if beta is None else np.abs(beta.astype(np.float64))
    sc = np.repeat(np.abs(rstd[ng]) * gm[c], S)
    return (np.abs(xv) + np.repeat(np.abs(mean[ng]), S)) * sc + np.repeat(bt[c], S)


def dx_terms(dyv, xv, mean, rstd, gamma, a, b, N, C, S, G):
    """Magnitudes entering dx = rstd*((dy*gamma - a) - xhat*b), per element."""
    Cg = C // G
    ng = (np.arange(N * C) // Cg)
    c = np.arange(N * C) % C
    gm = np.ones(C) if gamma is None else np.abs(gamma.astype(np.float64))
    r = np.repeat(np.abs(rstd[ng]), S)
    xh = (np.abs(xv) + np.repeat(np.abs(mean[ng]), S)) * r
    return r * (np.abs(dyv) * np.repeat(gm[c], S) + np.repeat(np.abs(a[ng]), S) + xh * np.repeat(np.abs(b[ng]), S))


def group_ab(dyv, xv, mean, rstd, gamma, N, C, S, G):
    """fp64 a = mean(dy*gamma), b = mean(dy*gamma*xhat) per group (for the error scale only)."""
    Cg = C // G
    gm = np.ones(C) if gamma is None else gamma.astype(np.float64)
    g = dyv.reshape(N, C, S) * gm[None, :, None]
    xh = (xv.reshape(N, G, Cg * S) - mean.reshape(N, G, 1)) * rstd.reshape(N, G, 1)
    g = g.reshape(N, G, Cg * S)
    return g.mean(2).reshape(-1), (g * xh).mean(2).reshape(-1)
