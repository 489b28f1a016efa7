"""Global statistics under spatial sharding, and dx from given sums, on one GPU.

A volume is cut along D into slabs, each its own contiguous tensor, as ranks
would hold it; the slabs' moments and row sums are combined in slab (rank)
order exactly as bwd_gn3d_stats_gb300.shard would combine them after an
all-gather, and the reassembled outputs are compared with the fp64 oracle on
the whole, unsharded volume.  With one slab every combine is the identity and
the results equal gn3d_forward / gn3d_backward bit for bit."""
import numpy as np
import pytest

import oracle
from bwd_gn3d_stats_gb300 import shard, synth

from . import parity
from .gpu_util import device_inputs, run_backward, run_forward, to_np, torch
from .test_gpu_parity import check_out, param_l2, stats_check

pytestmark = pytest.mark.gpu


def _slabs(t, site, cuts):
    """The D-slabs of a flat NCDHW tensor, each a contiguous [N, C, Dk, H, W]."""
    v = t.reshape(site.N, site.C, site.D, site.H, site.W)
    out, d0 = [], 0
    for dk in cuts:
        out.append(v[:, :, d0:d0 + dk].contiguous())
        d0 += dk
    return out


def _sharded_step(site, d, cuts):
    """Forward and backward of the whole volume through its slabs."""
    t = torch()
    xs, dys = _slabs(d["x"], site, cuts), _slabs(d["dy"], site, cuts)
    m = shard.combine_moments(t.stack([shard.moments(x, site.G) for x in xs]))
    fw = [shard.forward_apply(x, d["gamma"], d["beta"], site.G, m, site.eps) for x in xs]
    mean, rstd = fw[0][1], fw[0][2]
    count = int(shard.moment_counts(m)[0].item())
    sums = shard.combine_sums(t.stack([shard.backward_sums(dy, x, mean, rstd, site.G) for dy, x in zip(dys, xs)]))
    bw = [shard.backward_dx_from_sums(dy, x, mean, rstd, d["gamma"], site.G, sums, count)
          for dy, x in zip(dys, xs)]
    y = t.cat([f[0] for f in fw], dim=2).reshape(-1)
    dx = t.cat([b[0] for b in bw], dim=2).reshape(-1)
    t.cuda.synchronize()
    # every slab got the same statistics and parameter gradients
    for f in fw[1:]:
        assert t.equal(f[1], mean) and t.equal(f[2], rstd)
    for b in bw[1:]:
        assert t.equal(b[1], bw[0][1]) and t.equal(b[2], bw[0][2])
    return y, mean.reshape(-1), rstd.reshape(-1), dx, bw[0][1], bw[0][2], count


@pytest.mark.parametrize("shape", [(1, 48, 9, 9, 9, 8, synth.BF16), (2, 16, 16, 16, 16, 4, synth.F32),
                                   (1, 32, 32, 32, 32, 8, synth.BF16)],
                         ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_one_shard_is_the_plain_call_bit_for_bit(shape):
    site = synth.Site(*shape)
    d = device_inputs(synth.make_inputs(site, seed=81))
    y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
    dx, dg, db = run_backward(site, d["dy"], d["x"], mean, rstd, d["gamma"])
    got = _sharded_step(site, d, [site.D])
    for a, b in zip((y, mean, rstd, dx, dg, db), got[:6]):
        assert np.array_equal(to_np(a).view(np.uint8), to_np(b).view(np.uint8))
    assert got[6] == (site.C // site.G) * site.S


@pytest.mark.parametrize("shape,cuts", [((1, 48, 9, 9, 9, 8, synth.BF16), [4, 5]),
                                        ((2, 16, 12, 10, 8, 4, synth.F32), [3, 3, 6]),
                                        ((1, 32, 32, 32, 32, 8, synth.BF16), [8, 8, 8, 8]),
                                        ((2, 8, 5, 6, 7, 4, synth.BF16), [1, 2, 2]),
                                        ((1, 16, 64, 32, 32, 2, synth.BF16), [13, 51])],
                         ids=["97mini_2", "f32_3", "32cube_4", "ragged_3", "uneven_2"])
def test_sharded_volume_matches_the_oracle_on_the_whole(shape, cuts):
    """The slabs' y, mean, rstd, dx, dgamma and dbeta against the oracle on the
    unsharded volume, under the parity rules of the unsharded tests."""
    site = synth.Site(*shape)
    inp = synth.make_inputs(site, seed=82)
    d = device_inputs(inp)
    y, mean, rstd, dx, dg, db, count = _sharded_step(site, d, cuts)
    N, C, S, G = site.N, site.C, site.S, site.G
    assert count == (C // G) * S
    mg, rg = to_np(mean).astype(np.float64), to_np(rstd).astype(np.float64)
    m64, r64 = stats_check(site, inp, mg, rg)
    y64, _, _ = oracle.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, site.eps)
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64)
    dyv = synth.bits_to_f32(inp["dy"]).astype(np.float64)
    check_out(site.dtype, to_np(y), y64, parity.y_terms(xv, m64, r64, inp["gamma"], inp["beta"], N, C, S, G), "y")
    dx64, dg64, db64 = oracle.backward(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G)
    a, b, _, _ = oracle.backward_sums(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G)
    check_out(site.dtype, to_np(dx), dx64, parity.dx_terms(dyv, xv, mg, rg, inp["gamma"], a, b, N, C, S, G), "dx")
    l2g, l2b = param_l2(dyv, xv, mg, rg, N, C, S, G)
    assert np.all(parity.check_reduction(to_np(dg).astype(np.float64), dg64, l2g))
    assert np.all(parity.check_reduction(to_np(db).astype(np.float64), db64, l2b))


def test_dx_from_sums_made_elsewhere():
    """A producer of dy that forms the backward's sums itself: the dx pass from
    externally computed row sums (fp64 here, rounded to fp32) against the
    oracle, with no reduction pass in the library."""
    t = torch()
    site = synth.Site(2, 12, 8, 9, 10, 3, synth.BF16)
    inp = synth.make_inputs(site, seed=83)
    d = device_inputs(inp)
    N, C, S, G = site.N, site.C, site.S, site.G
    y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
    mg, rg = to_np(mean).astype(np.float64), to_np(rstd).astype(np.float64)
    xv = synth.bits_to_f32(inp["x"]).astype(np.float64).reshape(N, C, S)
    dyv = synth.bits_to_f32(inp["dy"]).astype(np.float64).reshape(N, C, S)
    mu = np.repeat(mg.reshape(N, G), C // G, axis=1)[:, :, None]
    sums = np.stack([dyv.sum(2), (dyv * (xv - mu)).sum(2)], axis=2).reshape(-1).astype(np.float32)
    dx, dg, db = shard.backward_dx_from_sums(d["dy"].reshape(N, C, site.D, site.H, site.W),
                                             d["x"].reshape(N, C, site.D, site.H, site.W), mean, rstd, d["gamma"],
                                             G, t.from_numpy(sums).cuda(), (C // G) * S)
    t.cuda.synchronize()
    dx64, dg64, db64 = oracle.backward(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G)
    a, b, _, _ = oracle.backward_sums(inp["dy"], inp["x"], mg, rg, inp["gamma"], N, C, S, G)
    check_out(site.dtype, to_np(dx), dx64, parity.dx_terms(dyv.reshape(-1), xv.reshape(-1), mg, rg, inp["gamma"], a,
                                                           b, N, C, S, G), "dx")
    l2g, l2b = param_l2(dyv.reshape(-1), xv.reshape(-1), mg, rg, N, C, S, G)
    assert np.all(parity.check_reduction(to_np(dg).astype(np.float64), dg64, l2g))
    assert np.all(parity.check_reduction(to_np(db).astype(np.float64), db64, l2b))


def test_shard_argument_checks():
    import bwd_gn3d_stats_gb300 as gn

    L = gn.lib()
    st = torch().cuda.current_stream().cuda_stream
    m = torch().zeros(4 * shard.MOMENT_BYTES, dtype=torch().uint8, device="cuda")
    assert L.gn3d_moments_combine(m.data_ptr(), 0, 4, m.data_ptr(), st) == gn.ERR_INVALID_ARG
    s = torch().zeros(8, device="cuda")
    assert L.gn3d_backward_dx_from_sums(None, None, s.data_ptr(), s.data_ptr(), None, s.data_ptr(), 0, 1, 4, 1, 1, 1,
                                        2, gn.F32, None, None, None, st) == gn.ERR_INVALID_ARG
    h = np.zeros(8, dtype=np.float32)
    assert L.gn3d_sums_combine(h.ctypes.data, 1, 4, s.data_ptr(), st) == gn.ERR_DEVICE
