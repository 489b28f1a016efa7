"""Channels-last (NDHWC) entry points against the fp64 oracle.

The oracle computes GroupNorm of the logical [N, C, D, H, W] tensor; the GPU
gets the same tensor stored channels-last, and its outputs are moved back to
NCDHW order (a permutation, no arithmetic) before the element-by-element
comparison under the same rules as the NCDHW parity tests.
"""
import numpy as np
import pytest

import oracle
from bwd_gn3d_stats_gb300 import synth

from . import parity
from .gpu_util import device_inputs, run_backward_ndhwc, run_forward_ndhwc, to_dev, to_np, torch
from .test_gpu_parity import check_out, param_l2, stats_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bwd_gn3d_stats_gb300 import build

    build.build()
    oracle.build()


def cl(a, site):
    return oracle.ncdhw_to_ndhwc(a, site.N, site.C, site.S)


def nc(a, site):
    return oracle.ndhwc_to_ncdhw(a, site.N, site.C, site.S)


def cl_inputs(site, inp):
    """Device copies of the inputs with x and dy stored channels-last."""
    d = device_inputs({k: v for k, v in inp.items() if k not in ("x", "dy")})
    d["x"] = to_dev(cl(inp["x"], site))
    d["dy"] = to_dev(cl(inp["dy"], site))
    return d


def run_cl(site, inp, out_dtype=None, affine=True, relu=False):
    d = cl_inputs(site, inp)
    gam = d["gamma"] if affine else None
    bet = d["beta"] if affine else None
    y, mean, rstd = run_forward_ndhwc(site, d["x"], gam, bet, out_dtype, relu=relu)
    dx, dg, db = run_backward_ndhwc(site, d["dy"], d["x"], mean, rstd, gam, out=y if relu else None)
    torch().cuda.synchronize()
    return [to_np(t) for t in (y, mean, rstd, dx, dg, db)]


def full_parity_cl(site, inp, out_dtype=None, affine=True):
    out_dtype = out_dtype or site.dtype
    N, C, S, G = site.N, site.C, site.S, site.G
    y, mg, rg, dx, dgg, dbg = run_cl(site, inp, out_dtype, affine)
    mg, rg, dgg, dbg = (a.astype(np.float64) for a in (mg, rg, dgg, dbg))
    gamma = inp["gamma"] if affine else None
    beta = inp["beta"] if affine else None
    m64, r64 = stats_check(site, inp, mg, rg)
    y64, _, _ = oracle.forward(inp["x"], gamma, beta, N, C, S, G, site.eps)
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64)
    dyv = synth.bits_to_f32(inp["dy"]).astype(np.float64)
    check_out(out_dtype, nc(y, site), y64, parity.y_terms(xv, m64, r64, gamma, beta, N, C, S, G), "y")
    dx64, dg64, db64 = oracle.backward(inp["dy"], inp["x"], mg, rg, gamma, N, C, S, G)
    a, b = parity.group_ab(dyv, xv, mg, rg, gamma, N, C, S, G)
    check_out(site.dtype, nc(dx, site), dx64, parity.dx_terms(dyv, xv, mg, rg, gamma, a, b, N, C, S, G), "dx")
    l2g, l2b = param_l2(dyv, xv, mg, rg, N, C, S, G)
    assert np.all(parity.check_reduction(dgg, dg64, l2g)), f"dgamma {np.max(np.abs(dgg - dg64))}"
    assert np.all(parity.check_reduction(dbg, db64, l2b)), f"dbeta {np.max(np.abs(dbg - db64))}"
    return dict(y=y, dx=dx, mean=mg, rstd=rg)


# Shapes chosen to reach every branch of the channels-last plan: channel ranges
# of 1 to 32 vectors (C = 8 .. 256, one warp step spanning 1 to 32 positions),
# ranges that do not fill the warp (C = 24, 48: 30 of 32 lanes), several ranges
# (C = 264, 512, 768), groups narrower than a vector (Cg = 2, 4, 6), groups
# straddling ranges (Cg = 96 at C = 768), ragged last units and blocks.
SHAPES = [
    (2, 16, 16, 16, 16, 4, synth.F32),    # the small fp32 workload, channels-last
    (1, 32, 16, 16, 16, 8, synth.BF16),   # the UNet's first site in miniature: 32 short units of 128 positions
    (1, 48, 13, 11, 7, 8, synth.BF16),    # C = 48: 6 vectors, 5 positions per step; Cg = 6; odd S
    (2, 64, 8, 9, 10, 32, synth.F32),     # 2 channels per group
    (1, 8, 20, 20, 20, 1, synth.BF16),    # one vector per position, one group
    (3, 24, 5, 5, 5, 3, synth.BF16),      # 3 vectors per position
    (1, 264, 3, 3, 3, 33, synth.F32),     # two ranges, the second one vector wide
    (1, 512, 4, 4, 5, 8, synth.BF16),     # two full ranges, 80 positions
    (1, 768, 2, 2, 3, 8, synth.BF16),     # groups of 96 channels across range boundaries
    (2, 16, 1, 1, 1, 16, synth.F32),      # single-element groups
    (1, 32, 40, 40, 40, 8, synth.BF16),   # 500 short units of 128 positions, ragged last unit
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_ndhwc_parity(shape):
    site = synth.Site(*shape)
    inp = synth.make_inputs(site, seed=11)
    full_parity_cl(site, inp)


@pytest.mark.parametrize("pair", [(synth.BF16, synth.F32), (synth.F32, synth.BF16)])
def test_ndhwc_mixed_out_dtype(pair):
    site = synth.Site(2, 32, 5, 6, 7, 4, pair[0])
    full_parity_cl(site, synth.make_inputs(site, seed=12), out_dtype=pair[1])


def test_ndhwc_no_affine():
    site = synth.Site(2, 16, 8, 8, 9, 2, synth.BF16)
    full_parity_cl(site, synth.make_inputs(site, seed=13), affine=False)


def test_ndhwc_single_element_groups_exact():
    site = synth.Site(3, 8, 1, 1, 1, 8, synth.F32)
    inp = synth.make_inputs(site, seed=14)
    r = full_parity_cl(site, inp)
    assert np.all(np.round(r["rstd"]) == 316)
    assert np.all(r["dx"] == 0.0)


def test_ndhwc_deterministic():
    """Repeated calls are bit-identical."""
    site = synth.Site(1, 64, 24, 24, 24, 8, synth.BF16)
    inp = synth.make_inputs(site, seed=15)
    outs = [run_cl(site, inp) for _ in range(5)]
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("shape", [(1, 32, 12, 12, 12, 8, synth.BF16), (2, 16, 6, 7, 8, 4, synth.F32),
                                   (1, 512, 4, 4, 5, 8, synth.BF16)],
                         ids=["bf16_ring", "f32_ring", "bf16_two_ranges"])
def test_ndhwc_relu_is_relu_of_forward(shape):
    """The fused ReLU forward is bit for bit F.relu of the plain forward; its
    backward matches the oracle's backward of relu(GroupNorm) at the saved statistics."""
    site = synth.Site(*shape)
    inp = synth.make_inputs(site, seed=16)
    t = torch()
    d = cl_inputs(site, inp)
    y, m, r = run_forward_ndhwc(site, d["x"], d["gamma"], d["beta"])
    yr, mr, rr = run_forward_ndhwc(site, d["x"], d["gamma"], d["beta"], relu=True)
    iv = t.int16 if site.dtype == synth.BF16 else t.int32
    assert t.equal(t.nn.functional.relu(y).view(iv), yr.view(iv))
    assert t.equal(m, mr) and t.equal(r, rr)
    dx, dg, db = run_backward_ndhwc(site, d["dy"], d["x"], mr, rr, d["gamma"], out=yr)
    t.cuda.synchronize()
    N, C, S, G = site.N, site.C, site.S, site.G
    mg, rg = to_np(mr).astype(np.float64), to_np(rr).astype(np.float64)
    out_nc = nc(to_np(yr), site)
    dx64, dg64, db64 = oracle.backward_relu(inp["dy"], inp["x"], out_nc, mg, rg, inp["gamma"], N, C, S, G)
    dyv = synth.bits_to_f32(inp["dy"]).astype(np.float64) * (synth.bits_to_f32(out_nc) > 0)
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64)
    a, b = parity.group_ab(dyv, xv, mg, rg, inp["gamma"], N, C, S, G)
    check_out(site.dtype, nc(to_np(dx), site), dx64, parity.dx_terms(dyv, xv, mg, rg, inp["gamma"], a, b, N, C, S,
                                                                    G), "dx")
    l2g, l2b = param_l2(dyv, xv, mg, rg, N, C, S, G)
    assert np.all(parity.check_reduction(to_np(dg).astype(np.float64), dg64, l2g))
    assert np.all(parity.check_reduction(to_np(db).astype(np.float64), db64, l2b))


def test_ndhwc_agrees_with_ncdhw():
    """The two layouts compute the same GroupNorm: statistics within fp32
    rounding, bf16 outputs within one ulp of each other."""
    from .gpu_util import run_backward, run_forward

    site = synth.Site(1, 32, 20, 20, 20, 8, synth.BF16)
    inp = synth.make_inputs(site, seed=17)
    y_cl, m_cl, r_cl, dx_cl, dg_cl, db_cl = run_cl(site, inp)
    d = device_inputs(inp)
    y, m, r = run_forward(site, d["x"], d["gamma"], d["beta"])
    dx, dg, db = run_backward(site, d["dy"], d["x"], m, r, d["gamma"])
    torch().cuda.synchronize()
    assert np.allclose(m_cl, to_np(m), rtol=1e-5, atol=1e-6)
    assert np.allclose(r_cl, to_np(r), rtol=1e-5)
    for a, b in ((nc(y_cl, site), to_np(y)), (nc(dx_cl, site), to_np(dx))):
        assert np.max(np.abs(parity.bf16_ordinal(a) - parity.bf16_ordinal(b))) <= 1
    assert np.allclose(dg_cl, to_np(dg), rtol=1e-4, atol=1e-3)
    assert np.allclose(db_cl, to_np(db), rtol=1e-4, atol=1e-3)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["bf16_1x32x128^3_G8", "bf16_2x64x96^3_G32", "bf16_2x64x96^3_G32_offset1e3",
                                  "bf16_1x32x256^3_G8"])
def test_ndhwc_full_size_sampled(name):
    """The bench volumes stored channels-last (including the 1e3 mean-offset
    cancellation probe): complete statistics and parameter gradients, and a
    seeded sample of y and dx, against the oracle."""
    site = synth.WORKLOADS[name].sites[0]
    inp = synth.make_inputs(site, seed=0)
    N, C, S, G = site.N, site.C, site.S, site.G
    d = cl_inputs(site, inp)
    y, mean, rstd = run_forward_ndhwc(site, d["x"], d["gamma"], d["beta"])
    dx, dgamma, dbeta = run_backward_ndhwc(site, d["dy"], d["x"], mean, rstd, d["gamma"])
    torch().cuda.synchronize()
    mg, rg = to_np(mean).astype(np.float64), to_np(rstd).astype(np.float64)
    m64, r64 = stats_check(site, inp, mg, rg)
    rng = np.random.default_rng(8)
    icl = np.unique(np.concatenate([rng.integers(0, site.numel, 200_000), np.arange(64),
                                    site.numel - 1 - np.arange(64)]))
    inc = oracle.ndhwc_index(icl, N, C, S)
    y64 = oracle.forward_at(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, m64, r64, inc)
    xv = synth.bits_to_f32(inp["x"])[inc].astype(np.float64)
    dyv = synth.bits_to_f32(inp["dy"])[inc].astype(np.float64)
    ng = (inc // S) // (C // G)
    c = (inc // S) % C
    tg = (np.abs(xv) + np.abs(m64[ng])) * r64[ng] * np.abs(inp["gamma"][c]) + np.abs(inp["beta"][c])
    check_out(site.dtype, to_np(y)[icl], y64, tg, "y(sampled)")
    dx64, dg64, db64 = oracle.backward_at(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G, inc)
    td = rg[ng] * (np.abs(dyv) * np.abs(inp["gamma"][c]) + 1.0 + (np.abs(xv) + np.abs(mg[ng])) * rg[ng])
    check_out(site.dtype, to_np(dx)[icl], dx64, td, "dx(sampled)")
    l2 = np.sqrt(N * S * 1.0) * np.ones(C)
    assert np.all(parity.check_reduction(to_np(dgamma).astype(np.float64), dg64, l2))
    assert np.all(parity.check_reduction(to_np(dbeta).astype(np.float64), db64, l2))


def test_ndhwc_bounded_wait_timeout_reports_and_recovers(testing_build):
    """The channels-last statistics kernel's bounded wait: a forced wait on a
    word nothing sets gives up, the kernel drains its bulk copies and exits,
    gn3d_stream_status reports GN3D_ERR_TIMEOUT once, and the next calls are
    correct again."""
    gn = testing_build
    site = synth.Site(1, 32, 16, 16, 16, 8, synth.BF16)
    inp = synth.make_inputs(site, seed=18)
    ref = run_cl(site, inp)
    d = cl_inputs(site, inp)
    st = torch().cuda.current_stream().cuda_stream
    L = gn.lib()
    try:
        gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 20000)
        gn.gn3d_debug_set(gn.DEBUG_FORCE_TIMEOUT, 1)
        run_forward_ndhwc(site, d["x"], d["gamma"], d["beta"])
        assert L.gn3d_stream_status(st) == gn.ERR_TIMEOUT
        assert L.gn3d_stream_status(st) == gn.OK  # read and cleared
    finally:
        gn.gn3d_debug_set(gn.DEBUG_FORCE_TIMEOUT, 0)
        gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 0)
    again = run_cl(site, inp)
    for a, b in zip(ref, again):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_ndhwc_plans_differ_by_direction():
    """1x32x86^3: 1243 units of 64 steps for the forward, and 2485 units of 32
    steps for the backward (which halves its units below 2432), so the two
    directions run different plans. The backward at the forward's statistics,
    and everything else, element by element against the oracle."""
    site = synth.Site(1, 32, 86, 86, 86, 8, synth.BF16)
    full_parity_cl(site, synth.make_inputs(site, seed=20))


def test_ndhwc_two_level_finalize_sampled():
    """A shape whose rows hold more than one finalize chunk (256 channels: units
    of 64 positions, 66^3 positions -> 4493 units per row, two chunks), so both
    finalize kernels take their two-level path: complete statistics and
    parameter gradients, and a seeded sample of y and dx, against the oracle."""
    site = synth.Site(1, 256, 66, 66, 66, 8, synth.BF16)
    inp = synth.make_inputs(site, seed=19)
    N, C, S, G = site.N, site.C, site.S, site.G
    d = cl_inputs(site, inp)
    y, mean, rstd = run_forward_ndhwc(site, d["x"], d["gamma"], d["beta"])
    dx, dgamma, dbeta = run_backward_ndhwc(site, d["dy"], d["x"], mean, rstd, d["gamma"])
    torch().cuda.synchronize()
    mg, rg = to_np(mean).astype(np.float64), to_np(rstd).astype(np.float64)
    m64, r64 = stats_check(site, inp, mg, rg)
    rng = np.random.default_rng(9)
    icl = np.unique(np.concatenate([rng.integers(0, site.numel, 100_000), np.arange(64),
                                    site.numel - 1 - np.arange(64)]))
    inc = oracle.ndhwc_index(icl, N, C, S)
    y64 = oracle.forward_at(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, m64, r64, inc)
    xv = synth.bits_to_f32(inp["x"])[inc].astype(np.float64)
    dyv = synth.bits_to_f32(inp["dy"])[inc].astype(np.float64)
    ng = (inc // S) // (C // G)
    c = (inc // S) % C
    tg = (np.abs(xv) + np.abs(m64[ng])) * r64[ng] * np.abs(inp["gamma"][c]) + np.abs(inp["beta"][c])
    check_out(site.dtype, to_np(y)[icl], y64, tg, "y(sampled)")
    dx64, dg64, db64 = oracle.backward_at(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G, inc)
    td = rg[ng] * (np.abs(dyv) * np.abs(inp["gamma"][c]) + 1.0 + (np.abs(xv) + np.abs(mg[ng])) * rg[ng])
    check_out(site.dtype, to_np(dx)[icl], dx64, td, "dx(sampled)")
    xf = synth.bits_to_f32(inp["x"]).astype(np.float64)
    dyf = synth.bits_to_f32(inp["dy"]).astype(np.float64)
    l2g, l2b = param_l2(dyf, xf, mg, rg, N, C, S, G)
    assert np.all(parity.check_reduction(to_np(dgamma).astype(np.float64), dg64, l2g))
    assert np.all(parity.check_reduction(to_np(dbeta).astype(np.float64), db64, l2b))
