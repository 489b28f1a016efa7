"""The fused ReLU (gn3d_forward_relu / gn3d_backward_relu).

Bit for bit: the fused forward is the plain forward followed by torch.relu,
and the fused backward is the plain backward on threshold_backward's gated dy
(the GroupNorm pages' claim: bit-exact against unfused + F.relu, NaN and both
infinities included).  Against the fp64 oracle: the parity rules of the plain
path, with the gate taken from the forward's result as the oracle's is.
"""
import numpy as np
import pytest

import oracle
from bwd_gn3d_stats_gb300 import synth

from . import parity
from .gpu_util import (device_inputs, run_backward, run_backward_relu, run_forward, run_forward_relu, to_np,
                       torch)
from .test_gpu_parity import check_out, param_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bwd_gn3d_stats_gb300 import build

    build.build()
    oracle.build()


def same(u, v):
    """Bit for bit, except that any two NaNs match (their payloads are not part of the contract)."""
    a, b = to_np(u), to_np(v)
    fa = synth.bits_to_f32(a) if a.dtype == np.uint16 else a
    fb = synth.bits_to_f32(b) if b.dtype == np.uint16 else b
    na, nb = np.isnan(fa), np.isnan(fb)
    return np.array_equal(na, nb) and np.array_equal(a[~na], b[~nb])


SHAPES = [
    (2, 16, 16, 16, 16, 4, synth.BF16, synth.BF16),
    (2, 16, 16, 16, 16, 4, synth.F32, synth.F32),
    (2, 8, 5, 6, 7, 4, synth.BF16, synth.BF16),     # ragged rows
    (1, 8, 24, 24, 24, 2, synth.BF16, synth.F32),   # bf16 in, fp32 out
    (1, 8, 24, 24, 24, 2, synth.F32, synth.BF16),   # fp32 in, bf16 out
    (2, 6, 1, 1, 1, 6, synth.BF16, synth.BF16),     # single-element groups
    (1, 32, 32, 32, 32, 8, synth.BF16, synth.BF16),  # full units
]


def special_inputs(site, seed):
    """Synthetic inputs with +-inf betas on two channels and a NaN in the last group."""
    inp = synth.make_inputs(site, seed=seed)
    beta = inp["beta"].copy()
    beta[0] = np.inf
    if site.C > 1:
        beta[1] = -np.inf
    inp["beta"] = beta
    x = inp["x"].copy()
    nan = np.array([np.nan], dtype=np.float32)
    x[-1] = nan.view(np.uint32).astype(np.uint32)[0] >> 16 if site.dtype == synth.BF16 else nan[0]
    inp["x"] = x
    return inp


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:6])) + f"_{s[6]}_{s[7]}")
@pytest.mark.parametrize("special", [False, True])
def test_fused_relu_is_relu_of_forward_and_gated_backward(shape, special):
    N, C, D, H, W, G, dt, out_dt = shape
    site = synth.Site(N, C, D, H, W, G, dt)
    inp = special_inputs(site, 40) if special else synth.make_inputs(site, seed=40)
    d = device_inputs(inp)
    t = torch()
    y, m, r = run_forward(site, d["x"], d["gamma"], d["beta"], out_dt)
    yr, mr, rr = run_forward_relu(site, d["x"], d["gamma"], d["beta"], out_dt)
    assert same(yr, t.relu(y)), "fused forward != relu(forward)"
    assert same(mr, m) and same(rr, r)
    if out_dt != dt:
        return  # the fused backward takes the forward's result in x's dtype
    gated = t.ops.aten.threshold_backward(d["dy"], yr, 0)
    dx0, dg0, db0 = run_backward(site, gated, d["x"], mr, rr, d["gamma"])
    dx1, dg1, db1 = run_backward_relu(site, d["dy"], d["x"], yr, mr, rr, d["gamma"])
    for a, b, what in ((dx1, dx0, "dx"), (dg1, dg0, "dgamma"), (db1, db0, "dbeta")):
        assert same(a, b), f"fused backward {what} != backward on the gated dy"


@pytest.mark.parametrize("shape", SHAPES[:3] + SHAPES[5:6], ids=lambda s: "x".join(map(str, s[:6])) + f"_{s[6]}")
def test_fused_relu_parity_with_oracle(shape):
    N, C, D, H, W, G, dt, out_dt = shape
    site = synth.Site(N, C, D, H, W, G, dt)
    inp = synth.make_inputs(site, seed=41)
    S = site.S
    d = device_inputs(inp)
    yr, mr, rr = run_forward_relu(site, d["x"], d["gamma"], d["beta"], out_dt)
    dx, dgamma, dbeta = run_backward_relu(site, d["dy"], d["x"], yr, mr, rr, d["gamma"])
    torch().cuda.synchronize()
    yg, mg, rg = to_np(yr), to_np(mr).astype(np.float64), to_np(rr).astype(np.float64)
    y64, m64, r64 = oracle.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    # the oracle's fused output: F.relu of its output rounded once
    if out_dt == synth.BF16:
        ref = oracle.relu(synth.bits_to_f32(oracle.round_bf16(y64)).astype(np.float64))
    else:
        ref = oracle.relu(oracle.round_f32(y64).astype(np.float64))
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64)
    dyv = synth.bits_to_f32(inp["dy"]).astype(np.float64)
    # a result that is an exact rounding of y64 differs from y64 by at most half an
    # ulp, inside the same per-element rules
    check_out(out_dt, yg, ref, parity.y_terms(xv, m64, r64, inp["gamma"], inp["beta"], N, C, S, G), "relu(y)")
    # backward at the GPU's statistics, gated by the GPU's forward result
    dx64, dg64, db64 = oracle.backward_relu(inp["dy"], inp["x"], yg, mg, rg, inp["gamma"], N, C, S, G)
    out_v = synth.bits_to_f32(yg).astype(np.float64) if dt == synth.BF16 else yg.astype(np.float64)
    gv = np.where(out_v <= 0, 0.0, dyv)
    a, b = parity.group_ab(gv, xv, mg, rg, inp["gamma"], N, C, S, G)
    check_out(dt, to_np(dx), dx64, parity.dx_terms(gv, xv, mg, rg, inp["gamma"], a, b, N, C, S, G), "dx")
    l2g, l2b = param_l2(gv, xv, mg, rg, N, C, S, G)
    assert np.all(parity.check_reduction(to_np(dgamma).astype(np.float64), dg64, l2g))
    assert np.all(parity.check_reduction(to_np(dbeta).astype(np.float64), db64, l2b))


def test_fused_relu_rejects_missing_result():
    import bwd_gn3d_stats_gb300 as gn

    site = synth.Site(1, 4, 4, 4, 4, 2, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=42))
    y, m, r = run_forward_relu(site, d["x"], d["gamma"], d["beta"])
    t = torch()
    dx = t.empty_like(d["x"])
    with pytest.raises(gn.GN3DError):
        gn.gn3d_backward_relu(d["dy"].data_ptr(), d["x"].data_ptr(), None, m.data_ptr(), r.data_ptr(), None,
                              site.N, site.C, site.D, site.H, site.W, site.G, gn.BF16, dx.data_ptr(), None, None,
                              t.cuda.current_stream().cuda_stream)
