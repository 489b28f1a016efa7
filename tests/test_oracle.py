"""Pins of the fp64 oracle against facts fixed outside it (CPU only).

Each test checks the oracle against something that is not the oracle's own
formula: values the GroupNorm pages state, closed forms and invariants of the
definition, finite differences, textbook special cases, and torch's float64
CPU GroupNorm / InstanceNorm / LayerNorm and autograd (independent library
code, run, not copied).
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from bwd_gn3d_stats_gb300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))
EPS32 = float(np.float32(1e-5))


def rand_case(rng, N, C, S, G, scale=1.0, offset=0.0):
    x = (offset + scale * rng.standard_normal(N * C * S)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = (0.1 * rng.standard_normal(C)).astype(np.float32)
    dy = rng.standard_normal(N * C * S).astype(np.float32)
    return x, gamma, beta, dy


def torch_gn(x, gamma, beta, N, C, S, G, eps=EPS32):
    xt = torch.from_numpy(x.astype(np.float64)).reshape(N, C, S)
    g = None if gamma is None else torch.from_numpy(gamma.astype(np.float64))
    b = None if beta is None else torch.from_numpy(beta.astype(np.float64))
    return F.group_norm(xt, G, g, b, eps).reshape(-1).numpy()


# ------------------------------------------------------------ page facts

def test_single_element_group_rstd_is_316(orc):
    f = GOLD["single_element_group_rstd"]
    rng = np.random.default_rng(1)
    N, C, S, G = 2, 4, 1, 4
    x, gamma, beta, dy = rand_case(rng, N, C, S, G)
    y, mean, rstd = orc.forward(x, gamma, beta, N, C, S, G, f["eps"])
    assert np.all(np.round(rstd) == f["rstd"])
    assert np.allclose(rstd, 1.0 / np.sqrt(EPS32), rtol=1e-15)
    # a zero-variance group maps to beta exactly
    assert np.array_equal(y, np.tile(beta.astype(np.float64), N))


def test_single_element_group_dx_is_exactly_zero(orc):
    rng = np.random.default_rng(2)
    N, C, S, G = 3, 6, 1, 6
    x, gamma, beta, dy = rand_case(rng, N, C, S, G)
    _, mean, rstd = orc.forward(x, gamma, beta, N, C, S, G, 1e-5)
    dx, dgamma, dbeta = orc.backward(dy, x, mean, rstd, gamma, N, C, S, G)
    assert GOLD["single_element_group_dx"]["dx"] == 0.0
    assert np.all(dx == 0.0)
    # dbeta is the plain sum of dy over n; dgamma is 0 since xhat = 0
    assert np.allclose(dbeta, dy.reshape(N, C).astype(np.float64).sum(0), rtol=1e-15, atol=0)
    assert np.all(dgamma == 0.0)


def test_degenerate_shape_matches_stock_raise():
    f = GOLD["degenerate_input_raises"]
    with pytest.raises(Exception):
        F.group_norm(torch.zeros(*f["shape"], dtype=torch.float64), f["G"])


# ------------------------------------------------------ closed forms

def test_two_point_group(orc):
    x = np.array([0.0, 2.0, 0.0, 2.0], dtype=np.float32)
    y, mean, rstd = orc.forward(x, None, None, 1, 2, 2, 2, 1e-5)
    _, var, _ = orc.stats(x, 1, 2, 2, 2, 1e-5)
    assert np.all(mean == 1.0) and np.all(var == 1.0)
    assert np.all(rstd == 1.0 / np.sqrt(1.0 + EPS32))
    r = 1.0 / np.sqrt(1.0 + EPS32)
    assert np.allclose(y, [-r, r, -r, r], rtol=1e-15)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_normalized_mean_zero_and_closed_form_variance(orc, dtype):
    site = synth.Site(2, 8, 6, 5, 7, 4, dtype)
    inp = synth.make_inputs(site, seed=3, with_dy=False)
    N, C, S, G = site.N, site.C, site.S, site.G
    y, mean, rstd = orc.forward(inp["x"], None, None, N, C, S, G, site.eps)
    _, var, _ = orc.stats(inp["x"], N, C, S, G, site.eps)
    yg = y.reshape(N * G, -1)
    assert np.max(np.abs(yg.mean(1))) < 1e-13
    assert np.allclose(yg.var(1), var / (var + EPS32), rtol=1e-12)
    # and var itself is the biased variance of the widened input values
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64).reshape(N * G, -1)
    assert np.allclose(var, xv.var(1), rtol=1e-12)
    assert np.allclose(mean, xv.mean(1), rtol=1e-13, atol=1e-15)


def test_affine_invariance_exact_with_scaled_eps(orc):
    # x on a coarse grid and power-of-two scales so a*x+b is exact in fp32
    rng = np.random.default_rng(4)
    N, C, S, G = 2, 6, 10, 3
    x = (rng.integers(-64, 64, N * C * S) / 16.0).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = (0.1 * rng.standard_normal(C)).astype(np.float32)
    y0, _, _ = orc.forward(x, gamma, beta, N, C, S, G, EPS32)
    M = (C // G) * S
    a = np.repeat(np.array([4.0, 0.5, 2.0, 8.0, 0.25, 1.0]), M)  # per group, > 0
    b = np.repeat(np.array([3.0, -7.0, 100.0, -0.5, 2.0, 0.0]), M)
    for grp_scale in (4.0,):
        xs = (x * grp_scale + 5.0).astype(np.float32)
        ys, _, _ = orc.forward(xs, gamma, beta, N, C, S, G, EPS32 * grp_scale ** 2)
        assert np.allclose(ys, y0, rtol=1e-13, atol=1e-13)
    # per-group a, b: each group normalised independently
    xg = (x * a + b).astype(np.float32)
    assert np.array_equal(xg.astype(np.float64), x.astype(np.float64) * a + b)
    # with eps scaled per group, compare group by group
    for k in range(N * G):
        n, g = divmod(k, G)
        sl = slice(k * M, (k + 1) * M)
        ak = a[k * M]
        yk, _, _ = orc.forward(xg[sl].copy(), gamma[g * (C // G):(g + 1) * (C // G)],
                               beta[g * (C // G):(g + 1) * (C // G)], 1, C // G, S, 1, EPS32 * ak * ak)
        assert np.allclose(yk, y0[sl], rtol=1e-13, atol=1e-13)
    # negative scale flips the normalised value: y(-x) - beta = -(y(x) - beta)
    yn, _, _ = orc.forward((-x).astype(np.float32), gamma, beta, N, C, S, G, EPS32)
    bb = np.repeat(np.tile(beta.astype(np.float64), N), S)
    assert np.allclose(yn - bb, -(y0 - bb), rtol=1e-13, atol=1e-13)


def test_affine_invariance_plain_eps_within_eps_over_var(orc):
    rng = np.random.default_rng(5)
    N, C, S, G = 1, 4, 64, 2
    x, gamma, beta, _ = rand_case(rng, N, C, S, G)
    y0, _, _ = orc.forward(x, gamma, beta, N, C, S, G, 1e-5)
    _, var, _ = orc.stats(x, N, C, S, G, 1e-5)
    a, b = np.float32(3.0), np.float32(-11.0)
    xs = (x * a + b).astype(np.float32)
    ys, _, _ = orc.forward(xs, gamma, beta, N, C, S, G, 1e-5)
    # only the eps/var term (and fp32 rounding of a*x+b) separates them
    assert np.max(np.abs(ys - y0)) < 20 * (1e-5 / var.min() + 1e-6)


# ------------------------------------------------ library special cases

def test_group_equals_channels_is_instance_norm(orc):
    rng = np.random.default_rng(6)
    N, C, S = 2, 5, 27
    x, gamma, beta, _ = rand_case(rng, N, C, S, C, scale=2.0, offset=0.5)
    y, _, _ = orc.forward(x, gamma, beta, N, C, S, C, EPS32)
    xt = torch.from_numpy(x.astype(np.float64)).reshape(N, C, 3, 3, 3)
    ref = F.instance_norm(xt, weight=torch.from_numpy(gamma.astype(np.float64)),
                          bias=torch.from_numpy(beta.astype(np.float64)), eps=EPS32).reshape(-1).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_one_group_is_layer_norm(orc):
    rng = np.random.default_rng(7)
    N, C, S = 3, 4, 8
    x, _, _, _ = rand_case(rng, N, C, S, 1, scale=3.0, offset=-1.0)
    y, _, _ = orc.forward(x, None, None, N, C, S, 1, EPS32)
    xt = torch.from_numpy(x.astype(np.float64)).reshape(N, C, 2, 2, 2)
    ref = F.layer_norm(xt, (C, 2, 2, 2), eps=EPS32).reshape(-1).numpy()
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 16, 4, 4, 4, 4), (1, 6, 3, 5, 2, 3), (3, 8, 1, 1, 1, 2)])
def test_forward_matches_torch_float64(orc, dtype, shape):
    N, C, D, H, W, G = shape
    site = synth.Site(N, C, D, H, W, G, dtype)
    inp = synth.make_inputs(site, seed=8, with_dy=False)
    y, mean, rstd = orc.forward(inp["x"], inp["gamma"], inp["beta"], N, C, site.S, G, site.eps)
    xv = synth.bits_to_f32(inp["x"])
    ref = torch_gn(xv, inp["gamma"], inp["beta"], N, C, site.S, G)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_large_mean_statistics_exact(orc):
    # mu/sigma = 1e5: the naive E[x^2]-E[x]^2 form loses the variance entirely
    # (ScaFFold PR #93, channels-last kernel commit); the oracle must not.
    rng = np.random.default_rng(9)
    base = np.float32(65536.0)
    k = rng.integers(-8, 8, 4096)
    x = (base + k.astype(np.float32) * np.float32(1.0 / 16)).astype(np.float32)
    _, var, _ = orc.stats(x, 1, 1, 4096, 1, 1e-5)
    exact = np.var(k.astype(np.float64) / 16.0)  # shift-invariant, exact in fp64
    assert abs(var[0] - exact) <= 1e-12 * exact


# -------------------------------------------------------------- backward

def _loss_grad_fd(orc, x, gamma, beta, w, N, C, S, G, eps, h):
    """Central differences of L = sum(w * y) w.r.t. every x, gamma and beta entry."""
    def L(xx, gg, bb):
        y, _, _ = orc.forward(xx, gg, bb, N, C, S, G, eps)
        return float(np.dot(w, y))
    gx = np.empty(x.size)
    for i in range(x.size):
        xp, xm = x.copy(), x.copy()
        xp[i] += np.float32(h)
        xm[i] -= np.float32(h)
        gx[i] = (L(xp, gamma, beta) - L(xm, gamma, beta)) / (2 * h)
    gg = np.empty(C)
    gb = np.empty(C)
    for c in range(C):
        p, m = gamma.copy(), gamma.copy()
        p[c] += np.float32(h)
        m[c] -= np.float32(h)
        gg[c] = (L(x, p, beta) - L(x, m, beta)) / (2 * h)
        p, m = beta.copy(), beta.copy()
        p[c] += np.float32(h)
        m[c] -= np.float32(h)
        gb[c] = (L(x, gamma, p) - L(x, gamma, m)) / (2 * h)
    return gx, gg, gb


@pytest.mark.parametrize("shape", [(1, 4, 8, 2), (2, 8, 64, 4)])
def test_backward_matches_finite_differences(orc, shape):
    N, C, S, G = shape
    rng = np.random.default_rng(10)
    h = 2.0 ** -14
    # values on a 2^-8 grid so x +- h, gamma +- h, beta +- h are exact in fp32
    x = (rng.integers(-512, 512, N * C * S) / 256.0).astype(np.float32)
    gamma = (rng.integers(128, 384, C) / 256.0).astype(np.float32)
    beta = (rng.integers(-32, 32, C) / 256.0).astype(np.float32)
    w = rng.standard_normal(N * C * S)
    eps = 1e-3
    _, mean, rstd = orc.forward(x, gamma, beta, N, C, S, G, eps)
    # dy = dL/dy = w, passed as fp32 bytes: use w rounded to fp32 for both sides
    w32 = w.astype(np.float32)
    dx, dgamma, dbeta = orc.backward(w32, x, mean, rstd, gamma, N, C, S, G)
    gx, gg, gb = _loss_grad_fd(orc, x, gamma, beta, w32.astype(np.float64), N, C, S, G, eps, h)
    scale = np.max(np.abs(gx))
    assert np.max(np.abs(dx - gx)) <= 1e-7 * scale
    assert np.allclose(dgamma, gg, rtol=1e-7, atol=1e-7 * np.max(np.abs(gg)))
    assert np.allclose(dbeta, gb, rtol=1e-7, atol=1e-7 * np.max(np.abs(gb)))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_matches_torch_autograd(orc, dtype):
    site = synth.Site(2, 12, 3, 4, 5, 3, dtype)
    inp = synth.make_inputs(site, seed=11)
    N, C, S, G = site.N, site.C, site.S, site.G
    _, mean, rstd = orc.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    dx, dgamma, dbeta = orc.backward(inp["dy"], inp["x"], mean, rstd, inp["gamma"], N, C, S, G)
    xt = torch.from_numpy(synth.bits_to_f32(inp["x"]).astype(np.float64)).reshape(N, C, S).requires_grad_()
    gt = torch.from_numpy(inp["gamma"].astype(np.float64)).requires_grad_()
    bt = torch.from_numpy(inp["beta"].astype(np.float64)).requires_grad_()
    y = F.group_norm(xt, G, gt, bt, EPS32)
    dyt = torch.from_numpy(synth.bits_to_f32(inp["dy"]).astype(np.float64)).reshape(N, C, S)
    y.backward(dyt)
    assert np.allclose(dx, xt.grad.reshape(-1).numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dgamma, gt.grad.numpy(), rtol=1e-10, atol=1e-10)
    assert np.allclose(dbeta, bt.grad.numpy(), rtol=1e-10, atol=1e-10)


def test_backward_group_invariants(orc):
    rng = np.random.default_rng(12)
    N, C, S, G = 2, 6, 50, 3
    x, gamma, beta, dy = rand_case(rng, N, C, S, G, scale=1.7, offset=0.3)
    _, mean, rstd = orc.forward(x, gamma, beta, N, C, S, G, 1e-2)
    _, var, _ = orc.stats(x, N, C, S, G, 1e-2)
    dx, _, _ = orc.backward(dy, x, mean, rstd, gamma, N, C, S, G)
    M = (C // G) * S
    dxg = dx.reshape(N * G, M)
    xh = (x.astype(np.float64).reshape(N * G, M) - mean[:, None]) * rstd[:, None]
    # sum of dx over a group is 0 for any gamma (sum of xhat is 0)
    assert np.max(np.abs(dxg.sum(1))) <= 1e-12 * np.abs(dxg).sum(1).max()
    # sum dx*xhat = rstd*M*b*eps/(var+eps), b = mean(dy*gamma*xhat)
    gam = np.repeat(gamma.astype(np.float64).reshape(1, G, C // G), N, 0).reshape(N * G, C // G)
    gfull = dy.astype(np.float64).reshape(N * G, C // G, S) * gam[:, :, None]
    b = (gfull.reshape(N * G, M) * xh).mean(1)
    eps = float(np.float32(1e-2))
    want = rstd * M * b * eps / (var + eps)
    got = (dxg * xh).sum(1)
    assert np.allclose(got, want, rtol=1e-9, atol=1e-12 * np.abs(dxg).sum())


def test_backward_at_matches_full(orc):
    site = synth.Site(2, 8, 4, 4, 4, 4, "bf16")
    inp = synth.make_inputs(site, seed=13)
    N, C, S, G = site.N, site.C, site.S, site.G
    _, mean, rstd = orc.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    dx, dg, db = orc.backward(inp["dy"], inp["x"], mean, rstd, inp["gamma"], N, C, S, G)
    idx = np.array([0, 5, 63, 64, 511, site.numel - 1])
    dxk, dgk, dbk = orc.backward_at(inp["dy"], inp["x"], mean, rstd, inp["gamma"], N, C, S, G, idx)
    assert np.array_equal(dxk, dx[idx]) and np.array_equal(dgk, dg) and np.array_equal(dbk, db)
    y, _, _ = orc.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    yk = orc.forward_at(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, mean, rstd, idx)
    assert np.array_equal(yk, y[idx])


# --------------------------------------------------------- output rounding

def test_round_bf16_ties_and_double_rounding(orc):
    one = 1.0
    cases = [
        (one + 2 ** -8, 0x3F80),            # halfway between 1 and 1+2^-7: ties to even (1.0)
        (one + 3 * 2 ** -8, 0x3F82),        # halfway between 1+2^-7 and 1+2^-6: ties to even
        (one + 2 ** -8 + 2 ** -40, 0x3F81),  # just above halfway: up (fp32 first would give 1.0)
        (-(one + 2 ** -8 + 2 ** -40), 0xBF81),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),              # smallest bf16 subnormal
        (2.0 ** -134, 0x0000),              # half of it: ties to even (zero)
        (1.5 * 2.0 ** -134, 0x0001),
        (3.3895313892515355e38, 0x7F7F),    # largest finite bf16
        (3.4e38, 0x7F80),                   # rounds past the largest finite: infinity
        (float("inf"), 0x7F80),
        (float("-inf"), 0xFF80),
    ]
    v = np.array([c[0] for c in cases])
    got = orc.round_bf16(v)
    assert [hex(g) for g in got] == [hex(c[1]) for c in cases]
    assert np.isnan(synth.bits_to_f32(orc.round_bf16(np.array([np.nan])))[0])


def test_round_bf16_agrees_with_torch_on_fp32_values(orc):
    rng = np.random.default_rng(14)
    v32 = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                          (rng.standard_normal(1000) * 1e-39).astype(np.float32)])
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.round_bf16(v32.astype(np.float64)), ref)


def test_round_f32(orc):
    v = np.array([1.0 + 2 ** -24, 1.0 + 3 * 2 ** -24, 0.1])
    assert np.array_equal(orc.round_f32(v), np.array([1.0, 1.0 + 2 ** -22, 0.1], dtype=np.float32))


# ------------------------------------------------------------ fused ReLU

def _vals(strs):
    return np.array([float(s) for s in strs])


def test_relu_special_values_are_the_pages(orc):
    f = GOLD["fused_relu_forward_special_values"]
    out, want = orc.relu(_vals(f["in"])), _vals(f["out"])
    assert np.array_equal(np.isnan(out), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(out[ok], want[ok])
    assert np.array_equal(np.signbit(out[ok]), np.signbit(want[ok]))  # -0.0 stays -0.0, -inf -> +0


def test_relu_matches_torch_relu_bitwise(orc):
    rng = np.random.default_rng(30)
    v = np.concatenate([_vals(["nan", "inf", "-inf", "-0.0", "0.0", "5e-324", "-5e-324"]),
                        rng.standard_normal(1000), -np.abs(rng.standard_normal(100)) * 1e-30])
    want = torch.relu(torch.from_numpy(v)).numpy()
    assert np.array_equal(orc.relu(v).view(np.uint64), want.view(np.uint64))


def test_backward_relu_gate_is_the_pages(orc):
    f = GOLD["fused_relu_backward_gate"]
    N, C, S, G = 1, 2, 3, 1
    rng = np.random.default_rng(31)
    x = rng.standard_normal(N * C * S).astype(np.float32)
    gamma = np.array([1.25, 0.75], dtype=np.float32)
    dy = rng.standard_normal(N * C * S).astype(np.float32)
    out = _vals(f["result"]).astype(np.float32)
    _, mean, rstd = orc.forward(x, gamma, None, N, C, S, G, 1e-5)
    got = orc.backward_relu(dy, x, out, mean, rstd, gamma, N, C, S, G)
    gated = np.where(np.array(f["passes"]), dy, np.float32(0)).astype(np.float32)
    want = orc.backward(gated, x, mean, rstd, gamma, N, C, S, G)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)


def test_backward_relu_matches_torch_autograd(orc):
    site = synth.Site(2, 12, 3, 4, 5, 3, synth.F32)
    inp = synth.make_inputs(site, seed=32)
    N, C, S, G = site.N, site.C, site.S, site.G
    y64, mean, rstd = orc.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    out = orc.relu(orc.round_f32(y64).astype(np.float64)).astype(np.float32)
    dx, dgamma, dbeta = orc.backward_relu(inp["dy"], inp["x"], out, mean, rstd, inp["gamma"], N, C, S, G)
    xt = torch.from_numpy(inp["x"].astype(np.float64)).reshape(N, C, S).requires_grad_()
    gt = torch.from_numpy(inp["gamma"].astype(np.float64)).requires_grad_()
    bt = torch.from_numpy(inp["beta"].astype(np.float64)).requires_grad_()
    yt = F.relu(F.group_norm(xt, G, gt, bt, EPS32))
    assert np.allclose(out, yt.detach().reshape(-1).numpy(), rtol=1e-6, atol=1e-7)
    yt.backward(torch.from_numpy(inp["dy"].astype(np.float64)).reshape(N, C, S))
    assert np.allclose(dx, xt.grad.reshape(-1).numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dgamma, gt.grad.numpy(), rtol=1e-10, atol=1e-10)
    assert np.allclose(dbeta, bt.grad.numpy(), rtol=1e-10, atol=1e-10)


def test_backward_relu_matches_finite_differences(orc):
    N, C, S, G = 1, 4, 8, 2
    rng = np.random.default_rng(33)
    h = 2.0 ** -14
    x = (rng.integers(-512, 512, N * C * S) / 256.0).astype(np.float32)
    gamma = (rng.integers(128, 384, C) / 256.0).astype(np.float32)
    beta = (rng.integers(-32, 32, C) / 256.0).astype(np.float32)
    w = rng.standard_normal(N * C * S).astype(np.float32)
    eps = 1e-3
    y64, mean, rstd = orc.forward(x, gamma, beta, N, C, S, G, eps)
    assert np.min(np.abs(y64)) > 1e-3  # ~10x what a step of h moves y: each difference sees one side of the kink
    out = orc.relu(orc.round_f32(y64).astype(np.float64)).astype(np.float32)
    dx, _, _ = orc.backward_relu(w, x, out, mean, rstd, gamma, N, C, S, G)

    def L(xx):
        yy, _, _ = orc.forward(xx, gamma, beta, N, C, S, G, eps)
        return float(np.dot(w.astype(np.float64), orc.relu(yy)))
    gx = np.empty(x.size)
    for i in range(x.size):
        xp, xm = x.copy(), x.copy()
        xp[i] += np.float32(h)
        xm[i] -= np.float32(h)
        gx[i] = (L(xp) - L(xm)) / (2 * h)
    assert np.max(np.abs(dx - gx)) <= 1e-7 * np.max(np.abs(gx))


# ------------------------------------------------------ channels-last layout

def test_ndhwc_layout_brute_force(orc):
    """The NDHWC adapters read element (n, c, s) at flat index (n*S + s)*C + c:
    group statistics and y recomputed here by loops over that index formula
    (a transposed reading would mix positions into channels and fail)."""
    rng = np.random.default_rng(30)
    N, C, S, G = 2, 6, 5, 3
    Cg = C // G
    xcl = (rng.standard_normal(N * S * C) + np.arange(N * S * C) % C).astype(np.float32)  # channel-dependent means
    gamma = rng.uniform(0.5, 1.5, C).astype(np.float32)
    beta = rng.standard_normal(C).astype(np.float32)
    y, mean, rstd = orc.forward_ndhwc(xcl, gamma, beta, N, C, S, G, 1e-5)
    for n in range(N):
        for g in range(G):
            vals = [float(xcl[(n * S + s) * C + c]) for s in range(S) for c in range(g * Cg, (g + 1) * Cg)]
            mu = sum(vals) / len(vals)
            var = sum((v - mu) ** 2 for v in vals) / len(vals)
            assert abs(mean[n * G + g] - mu) < 1e-12
            assert abs(rstd[n * G + g] - 1.0 / np.sqrt(var + EPS32)) < 1e-10
            for s in range(S):
                for c in range(g * Cg, (g + 1) * Cg):
                    i = (n * S + s) * C + c
                    ref = (float(xcl[i]) - mu) / np.sqrt(var + EPS32) * float(gamma[c]) + float(beta[c])
                    assert abs(y[i] - ref) < 1e-10


def test_ndhwc_matches_torch_channels_last_float64(orc):
    """Forward and backward against torch's float64 CPU GroupNorm run on a
    channels_last_3d tensor (torch's own channels-last kernel) and its autograd."""
    rng = np.random.default_rng(31)
    N, C, D, H, W, G = 2, 16, 3, 4, 5, 4
    S = D * H * W
    x, gamma, beta, dy = rand_case(rng, N, C, S, G, scale=2.0, offset=0.5)
    xt = torch.from_numpy(x.astype(np.float64)).reshape(N, C, D, H, W).contiguous(
        memory_format=torch.channels_last_3d).requires_grad_(True)
    gt = torch.from_numpy(gamma.astype(np.float64)).requires_grad_(True)
    bt = torch.from_numpy(beta.astype(np.float64)).requires_grad_(True)
    yt = F.group_norm(xt, G, gt, bt, EPS32)
    dyt = torch.from_numpy(dy.astype(np.float64)).reshape(N, C, D, H, W).contiguous(
        memory_format=torch.channels_last_3d)
    yt.backward(dyt)
    # channels-last storage of everything (torch keeps the memory format)
    xcl = orc.ncdhw_to_ndhwc(x, N, C, S)
    dycl = orc.ncdhw_to_ndhwc(dy, N, C, S)
    y, mean, rstd = orc.forward_ndhwc(xcl, gamma, beta, N, C, S, G, EPS32)
    ycl_t = yt.detach().permute(0, 2, 3, 4, 1).reshape(-1).numpy()
    assert np.allclose(y, ycl_t, rtol=1e-12, atol=1e-12)
    dx, dgamma, dbeta = orc.backward_ndhwc(dycl, xcl, mean, rstd, gamma, N, C, S, G)
    assert np.allclose(dx, xt.grad.permute(0, 2, 3, 4, 1).reshape(-1).numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dgamma, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dbeta, bt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_ndhwc_index_and_permutations_agree(orc):
    rng = np.random.default_rng(32)
    N, C, S = 3, 8, 7
    a = rng.standard_normal(N * C * S)
    cl = orc.ncdhw_to_ndhwc(a, N, C, S)
    assert np.array_equal(orc.ndhwc_to_ncdhw(cl, N, C, S), a)
    idx = np.arange(N * C * S)
    assert np.array_equal(a[orc.ndhwc_index(idx, N, C, S)], cl)


# ------------------------------------------- the backward's sums, the ReLU at indices

@pytest.mark.parametrize("dtype", [synth.F32, synth.BF16])
@pytest.mark.parametrize("gated", [False, True])
def test_backward_sums_closed_forms(orc, dtype, gated):
    """a = mean(dy*gamma) and b = mean(dy*gamma*xhat) per group, s1 = sum dy and
    s2 = sum dy*xhat per row, written out here with numpy on the widened inputs
    (behind the ReLU: dy zeroed where the forward's result is <= 0)."""
    site = synth.Site(2, 6, 3, 4, 5, 3, dtype)
    inp = synth.make_inputs(site, seed=41)
    N, C, S, G = site.N, site.C, site.S, site.G
    y64, mean, rstd = orc.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    out = None
    dyv = synth.bits_to_f32(inp["dy"]).astype(np.float64)
    if gated:
        if dtype == synth.BF16:
            out = orc.round_bf16(orc.relu(y64))
        else:
            out = orc.relu(orc.round_f32(y64).astype(np.float64)).astype(np.float32)
        dyv = np.where(synth.bits_to_f32(out).astype(np.float64) <= 0.0, 0.0, dyv)
    a, b, s1, s2 = orc.backward_sums(inp["dy"], inp["x"], mean, rstd, inp["gamma"], N, C, S, G, out=out)
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64).reshape(N, G, C // G, S)
    xh = (xv - mean.reshape(N, G, 1, 1)) * rstd.reshape(N, G, 1, 1)
    d = dyv.reshape(N, G, C // G, S)
    gm = inp["gamma"].astype(np.float64).reshape(1, G, C // G, 1)
    assert np.allclose(a, (d * gm).mean((2, 3)).reshape(-1), rtol=1e-12, atol=1e-14)
    assert np.allclose(b, (d * gm * xh).mean((2, 3)).reshape(-1), rtol=1e-12, atol=1e-14)
    assert np.allclose(s1, d.sum(3).reshape(-1), rtol=1e-12, atol=1e-12)
    assert np.allclose(s2, (d * xh).sum(3).reshape(-1), rtol=1e-12, atol=1e-12)


def test_backward_relu_at_matches_full(orc):
    """dx at chosen indices and the full dgamma/dbeta behind the ReLU equal the
    full backward behind the ReLU (itself pinned to torch autograd above)."""
    site = synth.Site(2, 8, 4, 4, 4, 4, synth.BF16)
    inp = synth.make_inputs(site, seed=42)
    N, C, S, G = site.N, site.C, site.S, site.G
    y64, mean, rstd = orc.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    out = orc.round_bf16(orc.relu(y64))
    assert 0.2 < np.mean(synth.bits_to_f32(out) <= 0) < 0.8  # both sides of the gate are exercised
    dx, dg, db = orc.backward_relu(inp["dy"], inp["x"], out, mean, rstd, inp["gamma"], N, C, S, G)
    idx = np.array([0, 3, 17, 63, 64, 300, 511, site.numel - 1])
    dxk, dgk, dbk = orc.backward_relu_at(inp["dy"], inp["x"], out, mean, rstd, inp["gamma"], N, C, S, G, idx)
    assert np.array_equal(dxk, dx[idx]) and np.array_equal(dgk, dg) and np.array_equal(dbk, db)


def test_backward_relu_ndhwc_matches_torch_channels_last(orc):
    """The channels-last backward behind the ReLU against torch's float64
    channels-last relu(group_norm) and its autograd."""
    rng = np.random.default_rng(43)
    N, C, D, H, W, G = 2, 8, 2, 3, 4, 2
    S = D * H * W
    x, gamma, beta, dy = rand_case(rng, N, C, S, G, scale=1.5)
    xt = torch.from_numpy(x.astype(np.float64)).reshape(N, C, D, H, W).contiguous(
        memory_format=torch.channels_last_3d).requires_grad_(True)
    gt = torch.from_numpy(gamma.astype(np.float64)).requires_grad_(True)
    bt = torch.from_numpy(beta.astype(np.float64)).requires_grad_(True)
    yt = F.relu(F.group_norm(xt, G, gt, bt, EPS32))
    yt.backward(torch.from_numpy(dy.astype(np.float64)).reshape(N, C, D, H, W).contiguous(
        memory_format=torch.channels_last_3d))
    xcl, dycl = orc.ncdhw_to_ndhwc(x, N, C, S), orc.ncdhw_to_ndhwc(dy, N, C, S)
    y, mean, rstd = orc.forward_ndhwc(xcl, gamma, beta, N, C, S, G, EPS32)
    out = orc.relu(orc.round_f32(y).astype(np.float64)).astype(np.float32)
    dx, dgamma, dbeta = orc.backward_relu_ndhwc(dycl, xcl, out, mean, rstd, gamma, N, C, S, G)
    assert np.allclose(dx, xt.grad.permute(0, 2, 3, 4, 1).reshape(-1).numpy(), rtol=1e-9, atol=1e-11)
    assert np.allclose(dgamma, gt.grad.numpy(), rtol=1e-9, atol=1e-10)
    assert np.allclose(dbeta, bt.grad.numpy(), rtol=1e-9, atol=1e-10)


# ------------------------------------------------------- sharded statistics

def test_combine_moments_textbook(orc):
    """Two sets {1, 2, 3} and {10, 20}: the combined moments are those of the
    union, {1, 2, 3, 10, 20} (mean 36/5, M2 = sum of squared deviations)."""
    a = (np.array([3.0]), np.array([2.0]), np.array([2.0]))
    b = (np.array([2.0]), np.array([15.0]), np.array([50.0]))
    n, m, q = orc.combine_moments([a, b])
    u = np.array([1.0, 2.0, 3.0, 10.0, 20.0])
    assert n[0] == 5 and abs(m[0] - u.mean()) < 1e-15 and abs(q[0] - ((u - u.mean()) ** 2).sum()) < 1e-12
    n1, m1, q1 = orc.combine_moments([a])
    assert n1[0] == 3 and m1[0] == 2.0 and q1[0] == 2.0


@pytest.mark.parametrize("cuts", [[4], [2, 2], [1, 2, 1], [3, 1]])
def test_sharded_moments_combine_to_the_whole(orc, cuts):
    """A volume cut along D into slabs (each slab its own contiguous tensor):
    the slabs' moments combined in rank order give the whole volume's count,
    mean and M2 -- and so its rstd -- to fp64 rounding."""
    rng = np.random.default_rng(44)
    N, C, D, H, W, G = 2, 6, sum(cuts), 3, 5, 3
    x = (3.0 + rng.standard_normal((N, C, D, H, W))).astype(np.float32)
    mean, var, rstd = orc.stats(x.reshape(-1), N, C, D * H * W, G, EPS32)
    parts, d0 = [], 0
    for dk in cuts:
        slab = np.ascontiguousarray(x[:, :, d0:d0 + dk]).reshape(-1)
        parts.append(orc.moments(slab, N, C, dk * H * W, G))
        d0 += dk
    n, m, q = orc.combine_moments(parts)
    M = (C // G) * D * H * W
    assert np.all(n == M)
    assert np.allclose(m, mean, rtol=1e-13, atol=1e-14)
    assert np.allclose(q / M, var, rtol=1e-12, atol=1e-14)
    assert np.allclose(orc.rstd_of(n, q, 1e-5), rstd, rtol=1e-12)


def test_sharded_backward_sums_add_up(orc):
    """At the whole volume's statistics, the slabs' per-row sums s1, s2 added in
    rank order are the whole volume's; a and b formed from them (A = sum_c
    gamma_c s1_c, B = sum_c gamma_c s2_c, over the group's M elements) are the
    whole volume's a and b, and rstd*(dy*gamma - a - xhat*b) is its dx."""
    rng = np.random.default_rng(45)
    N, C, D, H, W, G = 2, 6, 5, 2, 3, 2
    S = D * H * W
    x, gamma, beta, dy = rand_case(rng, N, C, S, G, scale=2.0, offset=1.0)
    _, mean, rstd = orc.forward(x, gamma, beta, N, C, S, G, EPS32)
    a, b, s1, s2 = orc.backward_sums(dy, x, mean, rstd, gamma, N, C, S, G)
    dx, dgamma, dbeta = orc.backward(dy, x, mean, rstd, gamma, N, C, S, G)
    x5, dy5 = x.reshape(N, C, D, H, W), dy.reshape(N, C, D, H, W)
    t1, t2, d0 = np.zeros(N * C), np.zeros(N * C), 0
    for dk in (2, 1, 2):
        xs = np.ascontiguousarray(x5[:, :, d0:d0 + dk]).reshape(-1)
        ds = np.ascontiguousarray(dy5[:, :, d0:d0 + dk]).reshape(-1)
        _, _, p1, p2 = orc.backward_sums(ds, xs, mean, rstd, gamma, N, C, dk * H * W, G)
        t1, t2 = t1 + p1, t2 + p2
        d0 += dk
    assert np.allclose(t1, s1, rtol=1e-12, atol=1e-12) and np.allclose(t2, s2, rtol=1e-12, atol=1e-12)
    Cg, M = C // G, (C // G) * S
    gm = gamma.astype(np.float64).reshape(G, Cg)
    A = (t1.reshape(N, G, Cg) * gm).sum(2).reshape(-1)
    B = (t2.reshape(N, G, Cg) * gm).sum(2).reshape(-1)
    assert np.allclose(A / M, a, rtol=1e-12, atol=1e-14) and np.allclose(B / M, b, rtol=1e-12, atol=1e-14)
    xh = (x.astype(np.float64).reshape(N, G, Cg * S) - mean.reshape(N, G, 1)) * rstd.reshape(N, G, 1)
    g = (dy.astype(np.float64).reshape(N, G, Cg, S) * gm.reshape(1, G, Cg, 1)).reshape(N, G, Cg * S)
    want = rstd.reshape(N, G, 1) * (g - (A / M).reshape(N, G, 1) - xh * (B / M).reshape(N, G, 1))
    assert np.allclose(dx, want.reshape(-1), rtol=1e-10, atol=1e-12)
    assert np.allclose(dbeta, t1.reshape(N, C).sum(0), rtol=1e-12, atol=1e-12)
    assert np.allclose(dgamma, t2.reshape(N, C).sum(0), rtol=1e-12, atol=1e-12)
