"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small and medium shapes are compared element by element over the whole tensor;
the full-size volumes are compared on the complete statistics and dgamma/dbeta
and on a seeded sample of y and dx elements computed one by one by the oracle.
"""
import numpy as np
import pytest

import oracle
from bwd_gn3d_stats_gb300 import synth

from . import parity
from .gpu_util import device_inputs, run_backward, run_forward, to_np, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bwd_gn3d_stats_gb300 import build

    build.build()
    oracle.build()


def stats_check(site, inp, mean_g, rstd_g):
    N, C, S, G = site.N, site.C, site.S, site.G
    m64, v64, r64 = oracle.stats(inp["x"], N, C, S, G, site.eps)
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64).reshape(N * G, -1)
    l2 = np.sqrt((xv * xv).sum(1)) / max(xv.shape[1], 1)
    assert np.all(parity.check_reduction(mean_g, m64, l2)), f"mean: {np.max(np.abs(mean_g - m64))}"
    assert np.all(np.abs(rstd_g - r64) <= 1e-5 * r64), f"rstd rel: {np.max(np.abs(rstd_g / r64 - 1))}"
    return m64, r64


def check_out(dtype, gpu, ref, terms, what):
    if dtype == synth.BF16:
        ok, n2 = parity.check_bf16(gpu, ref, terms, oracle.round_bf16)
        assert ok.all(), f"{what}: {np.count_nonzero(~ok)} bf16 elements off, first at {np.argmax(~ok)}"
        assert n2 <= max(10, 1e-4 * ref.size), f"{what}: {n2} elements needed the cancellation clause"
        return n2
    ok = parity.check_f32(gpu, ref)
    i = np.argmax(~ok)
    assert ok.all(), f"{what}: {np.count_nonzero(~ok)} fp32 elements off, e.g. {gpu[i]} vs {ref[i]}"
    return 0


def param_l2(dyv, xv, mean, rstd, N, C, S, G):
    Cg = C // G
    xh = (xv.reshape(N, G, Cg, S) - mean.reshape(N, G, 1, 1)) * rstd.reshape(N, G, 1, 1)
    d = dyv.reshape(N, G, Cg, S)
    l2g = np.sqrt(((d * xh) ** 2).sum((0, 3))).reshape(C)
    l2b = np.sqrt((d ** 2).sum((0, 3))).reshape(C)
    return l2g, l2b


def full_parity(site, inp, out_dtype=None, affine=True):
    out_dtype = out_dtype or site.dtype
    N, C, S, G = site.N, site.C, site.S, site.G
    d = device_inputs(inp)
    gam = d["gamma"] if affine else None
    bet = d["beta"] if affine else None
    y, mean, rstd = run_forward(site, d["x"], gam, bet, out_dtype)
    dx, dgamma, dbeta = run_backward(site, d["dy"], d["x"], mean, rstd, gam)
    torch().cuda.synchronize()
    yg, mg, rg = to_np(y), to_np(mean).astype(np.float64), to_np(rstd).astype(np.float64)
    dxg, dgg, dbg = to_np(dx), to_np(dgamma).astype(np.float64), to_np(dbeta).astype(np.float64)
    gamma = inp["gamma"] if affine else None
    beta = inp["beta"] if affine else None
    m64, r64 = stats_check(site, inp, mg, rg)
    y64, _, _ = oracle.forward(inp["x"], gamma, beta, N, C, S, G, site.eps)
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64)
    dyv = synth.bits_to_f32(inp["dy"]).astype(np.float64)
    n2y = check_out(out_dtype, yg, y64, parity.y_terms(xv, m64, r64, gamma, beta, N, C, S, G), "y")
    # backward at the GPU's own saved statistics (isolates the backward's error)
    dx64, dg64, db64 = oracle.backward(inp["dy"], inp["x"], mg, rg, gamma, N, C, S, G)
    a, b = parity.group_ab(dyv, xv, mg, rg, gamma, N, C, S, G)
    n2dx = check_out(site.dtype, dxg, dx64, parity.dx_terms(dyv, xv, mg, rg, gamma, a, b, N, C, S, G), "dx")
    l2g, l2b = param_l2(dyv, xv, mg, rg, N, C, S, G)
    assert np.all(parity.check_reduction(dgg, dg64, l2g)), f"dgamma {np.max(np.abs(dgg - dg64))}"
    assert np.all(parity.check_reduction(dbg, db64, l2b)), f"dbeta {np.max(np.abs(dbg - db64))}"
    return dict(y=yg, mean=mg, rstd=rg, dx=dxg, dgamma=dgg, dbeta=dbg, n2y=n2y, n2dx=n2dx)


SMALL = [
    (2, 16, 16, 16, 16, 4, synth.F32),   # the small fp32 parity workload
    (2, 16, 16, 16, 16, 4, synth.BF16),
    (2, 8, 5, 6, 7, 4, synth.BF16),       # rows of 210 elements: unaligned heads/tails
    (1, 48, 9, 9, 9, 8, synth.BF16),      # odd spatial size (the 97^3 site in miniature)
    (1, 8, 24, 24, 24, 2, synth.BF16),    # 13824-element rows: two units per row, ragged second
    (1, 8, 24, 24, 24, 2, synth.F32),
    (3, 6, 2, 3, 1, 3, synth.BF16),       # 6-element rows, no aligned body at all
    (2, 4, 1, 1, 3, 2, synth.F32),
    (2, 6, 1, 1, 1, 6, synth.BF16),       # single-element groups
    (1, 64, 4, 4, 4, 32, synth.BF16),     # many small groups
    (2, 3, 17, 1, 29, 1, synth.F32),      # one group (LayerNorm over C,D,H,W)
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_parity_small(shape):
    site = synth.Site(*shape)
    inp = synth.make_inputs(site, seed=0)
    full_parity(site, inp)


@pytest.mark.parametrize("pair", [(synth.BF16, synth.F32), (synth.F32, synth.BF16)])
def test_parity_mixed_out_dtype(pair):
    site = synth.Site(2, 8, 5, 6, 7, 4, pair[0])
    inp = synth.make_inputs(site, seed=1)
    full_parity(site, inp, out_dtype=pair[1])


def test_parity_no_affine():
    site = synth.Site(2, 8, 8, 8, 9, 2, synth.BF16)
    full_parity(site, synth.make_inputs(site, seed=2), affine=False)


def test_single_element_groups_exact():
    """rstd = 1/sqrt(eps) (316 at eps = 1e-5) and dx exactly 0 when every group has one element."""
    site = synth.Site(3, 8, 1, 1, 1, 8, synth.F32)
    inp = synth.make_inputs(site, seed=3)
    r = full_parity(site, inp)
    assert np.all(np.round(r["rstd"]) == 316)
    assert np.all(r["dx"] == 0.0)
    assert np.array_equal(r["y"], np.tile(inp["beta"], site.N))


def test_nan_stays_in_its_group():
    site = synth.Site(1, 8, 4, 4, 4, 4, synth.F32)
    inp = synth.make_inputs(site, seed=4)
    inp["x"][5] = np.nan  # group 0
    d = device_inputs(inp)
    y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
    yg = to_np(y).reshape(site.G, -1)
    assert np.all(np.isnan(yg[0])) and not np.any(np.isnan(yg[1:]))


def test_determinism_and_dtype_independence():
    """10 repeated calls are bit-identical; fp32 and bf16 inputs holding the same
    values give bit-identical mean, rstd, dgamma, dbeta, and y/dx that round alike."""
    site = synth.Site(1, 16, 40, 40, 40, 4, synth.BF16)
    inp = synth.make_inputs(site, seed=5)
    d = device_inputs(inp)
    outs = []
    for _ in range(10):
        y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
        dx, dg, db = run_backward(site, d["dy"], d["x"], mean, rstd, d["gamma"])
        outs.append([to_np(t) for t in (y, mean, rstd, dx, dg, db)])
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    s32 = synth.Site(1, 16, 40, 40, 40, 4, synth.F32)
    x32 = {k: (synth.bits_to_f32(v) if k in ("x", "dy") else v) for k, v in inp.items()}
    d32 = device_inputs(x32)
    y32, m32, r32 = run_forward(s32, d32["x"], d32["gamma"], d32["beta"], synth.F32)
    dx32, dg32, db32 = run_backward(s32, d32["dy"], d32["x"], m32, r32, d32["gamma"])
    t = torch()
    for a, b in ((m32, outs[0][1]), (r32, outs[0][2]), (dg32, outs[0][4]), (db32, outs[0][5])):
        assert np.array_equal(to_np(a).view(np.uint32), b.view(np.uint32))
    assert np.array_equal(to_np(y32.to(t.bfloat16)), outs[0][0])
    assert np.array_equal(to_np(dx32.to(t.bfloat16)), outs[0][3])


@pytest.mark.parametrize("path", ["streaming", "fused", "resident", "cluster"])
@pytest.mark.parametrize("shape", [(2, 16, 16, 16, 16, 4, synth.F32), (1, 8, 24, 24, 24, 2, synth.BF16),
                                   (1, 32, 16, 16, 32, 8, synth.BF16), (2, 6, 1, 1, 1, 6, synth.BF16),
                                   (1, 128, 16, 16, 16, 8, synth.BF16), (1, 512, 16, 16, 16, 8, synth.BF16)],
                         ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_parity_other_launch_forms(path, shape, testing_build):
    """Each launch form against the oracle directly (not only against the
    streaming form): streaming, persistent, group-wave and cluster kernels;
    shapes a form does not take run on the streaming kernels under its setting."""
    gn = testing_build
    site = synth.Site(*shape)
    gn.gn3d_debug_set(gn.DEBUG_PATH, {"streaming": gn.PATH_STREAMING, "fused": gn.PATH_FUSED,
                                      "resident": gn.PATH_RESIDENT, "cluster": gn.PATH_CLUSTER}[path])
    full_parity(site, synth.make_inputs(site, seed=6))


# ------------------------------------------------------- full-size volumes

def sampled_parity(site, inp, k=200_000, seed=7):
    N, C, S, G = site.N, site.C, site.S, site.G
    d = device_inputs(inp)
    y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
    dx, dgamma, dbeta = run_backward(site, d["dy"], d["x"], mean, rstd, d["gamma"])
    torch().cuda.synchronize()
    mg, rg = to_np(mean).astype(np.float64), to_np(rstd).astype(np.float64)
    m64, r64 = stats_check(site, inp, mg, rg)
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([rng.integers(0, site.numel, k), np.arange(64),
                                    site.numel - 1 - np.arange(64)]))
    ys = to_np(y)[idx]
    y64 = oracle.forward_at(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, m64, r64, idx)
    xv = synth.bits_to_f32(inp["x"])[idx].astype(np.float64)
    dyv = synth.bits_to_f32(inp["dy"])[idx].astype(np.float64)
    ng = (idx // S) // (C // G)
    c = (idx // S) % C
    tg = (np.abs(xv) + np.abs(m64[ng])) * r64[ng] * np.abs(inp["gamma"][c]) + np.abs(inp["beta"][c])
    check_out(site.dtype, ys, y64, tg, "y(sampled)")
    dx64, dg64, db64 = oracle.backward_at(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G, idx)
    dxs = to_np(dx)[idx]
    # the magnitudes entering dx = rstd*((dy*gamma - a) - xhat*b), with the
    # group's a and b from the oracle's sums at the same statistics
    a, b, _, _ = oracle.backward_sums(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G)
    td = rg[ng] * (np.abs(dyv) * np.abs(inp["gamma"][c]) + np.abs(a[ng])
                   + (np.abs(xv) + np.abs(mg[ng])) * rg[ng] * np.abs(b[ng]))
    check_out(site.dtype, dxs, dx64, td, "dx(sampled)")
    dgg, dbg = to_np(dgamma).astype(np.float64), to_np(dbeta).astype(np.float64)
    # L2 of summed terms, from a sample of each channel's terms scaled to the full count
    l2b = np.sqrt(N * S * 1.0) * np.ones(C)
    l2g = l2b.copy()
    assert np.all(parity.check_reduction(dgg, dg64, l2g)), f"dgamma {np.max(np.abs(dgg - dg64))}"
    assert np.all(parity.check_reduction(dbg, db64, l2b)), f"dbeta {np.max(np.abs(dbg - db64))}"


FULL = ["bf16_1x32x128^3_G8", "bf16_2x64x96^3_G32", "bf16_2x64x96^3_G32_offset1e3", "bf16_1x32x256^3_G8"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    site = synth.WORKLOADS[name].sites[0]
    inp = synth.make_inputs(site, seed=0)
    sampled_parity(site, inp)


@pytest.mark.slow
def test_full_size_128_complete():
    """Every element of the 128^3 volume against the oracle."""
    site = synth.WORKLOADS["bf16_1x32x128^3_G8"].sites[0]
    full_parity(site, synth.make_inputs(site, seed=0))


@pytest.mark.slow
def test_unet_odd_site_complete():
    """The odd-shaped UNet site (48 channels of 97^3): unaligned rows everywhere."""
    site = synth.WORKLOADS["bf16_unet_stack_G8"].sites[-1]
    full_parity(site, synth.make_inputs(site, seed=0))
