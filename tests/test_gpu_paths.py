"""The launch forms (streaming, persistent, group-wave and cluster kernels) and every
tuning setting give bit-identical results; the bounded-wait failure path
reports GN3D_ERR_TIMEOUT and leaves the library usable.  (Run on the testing
build of the library, which carries the hooks.)"""
import numpy as np
import pytest

import bwd_gn3d_stats_gb300 as gn
from bwd_gn3d_stats_gb300 import synth

from .gpu_util import (device_inputs, run_backward, run_backward_relu, run_forward, run_forward_relu, to_np,
                       torch)

pytestmark = pytest.mark.gpu

@pytest.fixture(autouse=True)
def _testing(testing_build):
    """Every test here sets hooks of the testing build and runs on it."""
    yield


def run_all(site, d):
    y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
    dx, dg, db = run_backward(site, d["dy"], d["x"], mean, rstd, d["gamma"])
    torch().cuda.synchronize()
    return [to_np(t) for t in (y, mean, rstd, dx, dg, db)]


def same(a, b):
    return all(np.array_equal(u.view(np.uint8), v.view(np.uint8)) for u, v in zip(a, b))


SHAPES = [
    (1, 32, 40, 40, 40, 8, synth.BF16),
    (2, 8, 5, 6, 7, 4, synth.BF16),
    (1, 48, 13, 11, 9, 8, synth.BF16),
    (2, 6, 1, 1, 1, 6, synth.F32),
    (1, 16, 24, 24, 24, 2, synth.F32),
    (1, 512, 8, 8, 8, 8, synth.BF16),
    # rows of whole 4096-element units: the streaming kernels' full-unit variants
    # against the persistent kernels' general path
    (1, 16, 16, 16, 32, 4, synth.BF16),
    (2, 8, 16, 16, 16, 2, synth.F32),
    # odd rows of many units, each with head and tail scalars: the reduction
    # kernels' scalars loaded a unit ahead, across blocks and rows
    (1, 24, 33, 31, 29, 8, synth.BF16),
    (1, 12, 37, 35, 33, 4, synth.F32),
]

# the streaming kernels in unit shares by default (shares of 2 merge blocks or
# more): equal runs of units per warp, blocks cut between warps
LARGE = [
    (1, 40, 160, 160, 160, 8, synth.BF16),
    (1, 30, 181, 181, 181, 6, synth.BF16),
]


@pytest.mark.parametrize("shape", SHAPES + LARGE, ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_fused_and_streaming_bit_identical(shape):
    site = synth.Site(*shape)
    d = device_inputs(synth.make_inputs(site, seed=11))
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_FUSED)
    a = run_all(site, d)
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_STREAMING)
    b = run_all(site, d)
    assert same(a, b)


@pytest.mark.parametrize("knob,values", [(gn.DEBUG_LAG, [0, 1]), (gn.DEBUG_SLOTS, [1, 2, 3, 9])])
def test_tuning_does_not_move_a_bit(knob, values):
    site = synth.Site(1, 32, 36, 36, 36, 8, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=12))
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_FUSED)  # lag and slots shape the persistent kernels
    ref = run_all(site, d)
    for v in values:
        gn.gn3d_debug_set(knob, v)
        assert same(ref, run_all(site, d)), f"setting {knob}={v} changed the result"


def test_bounded_wait_timeout_reports_and_recovers():
    site = synth.Site(1, 8, 24, 24, 24, 4, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=13))
    ref = run_all(site, d)
    st = torch().cuda.current_stream().cuda_stream
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_FUSED)  # the forced wait is in the persistent kernels
    gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 20000)
    gn.gn3d_debug_set(gn.DEBUG_FORCE_TIMEOUT, 1)
    run_forward(site, d["x"], d["gamma"], d["beta"])
    L = gn.lib()
    assert L.gn3d_stream_status(st) == gn.ERR_TIMEOUT
    assert L.gn3d_stream_status(st) == gn.OK  # read-and-clear
    gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 0)
    assert same(ref, run_all(site, d))


@pytest.mark.parametrize("path,launches", [(gn.PATH_AUTO, 2), (gn.PATH_STREAMING, 4), (gn.PATH_FUSED, 2),
                                          (gn.PATH_CLUSTER, 2)])
def test_launch_count(path, launches):
    site = synth.Site(1, 8, 16, 16, 16, 4, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=14))
    gn.gn3d_debug_set(gn.DEBUG_PATH, path)
    n0 = gn.gn3d_launch_count()
    run_all(site, d)
    assert gn.gn3d_launch_count() - n0 == launches


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_block_and_unit_shares_bit_identical(shape):
    """Strided blocks (whole merge blocks dealt out to the warps in turn) and
    unit shares (equal contiguous runs of units, blocks cut between warps and
    merged by the warp completing them) place work differently and compute the
    same bits, with and without the fused ReLU."""
    site = synth.Site(*shape)
    d = device_inputs(synth.make_inputs(site, seed=13))
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_STREAMING)
    out = {}
    for mode in (0, 1):
        gn.gn3d_debug_set(gn.DEBUG_SHARES, mode)
        out[mode] = run_all(site, d)
        y, mean, rstd = run_forward_relu(site, d["x"], d["gamma"], d["beta"])
        dx, dg, db = run_backward_relu(site, d["dy"], d["x"], y, mean, rstd, d["gamma"])
        torch().cuda.synchronize()
        out[mode] += [to_np(t) for t in (y, mean, rstd, dx, dg, db)]
    assert same(out[0], out[1])


# rows of whole 4096-element units: the group-wave kernels' domain (several
# shares per group, groups smaller than the SM count, N > 1, fp32, one group)
RESIDENT = [
    (1, 32, 32, 32, 32, 8, synth.BF16),
    (2, 64, 32, 32, 48, 32, synth.BF16),
    (1, 512, 16, 16, 16, 8, synth.BF16),
    (1, 32, 128, 128, 128, 8, synth.BF16),
    (2, 16, 16, 16, 16, 4, synth.F32),
    (1, 16, 64, 64, 64, 1, synth.F32),
    (3, 12, 16, 32, 40, 3, synth.BF16),
]


@pytest.mark.parametrize("shape", RESIDENT, ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_group_wave_and_streaming_bit_identical(shape):
    """The group-wave kernels (each CTA a share of every group, the group merged
    from its unit partials by every CTA) and the streaming kernels give the same
    bits: the same units, merge blocks and group merges, placed differently."""
    site = synth.Site(*shape)
    d = device_inputs(synth.make_inputs(site, seed=21))
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_STREAMING)
    a = run_all(site, d)
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_RESIDENT)
    b = run_all(site, d)
    gn.gn3d_stream_status(torch().cuda.current_stream().cuda_stream)
    assert same(a, b)


@pytest.mark.parametrize("held,passes,window", [(0, 8, -1), (3, 4, -1), (20, 4, -1), (5, 4, 30), (10, 12, 200)])
def test_group_wave_ring_settings_do_not_move_a_bit(held, passes, window):
    """Held units per share, pass-ring slots and the producer's lead decide what
    stays on chip and what is read again from L2, never a value."""
    site = synth.Site(1, 24, 48, 48, 64, 6, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=22))
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_STREAMING)
    ref = run_all(site, d)
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_RESIDENT)
    gn.gn3d_debug_set(gn.DEBUG_RES_HELD, held)
    gn.gn3d_debug_set(gn.DEBUG_RES_PASS, passes)
    gn.gn3d_debug_set(gn.DEBUG_RES_WINDOW, window)
    assert same(ref, run_all(site, d))


def test_group_wave_mixed_dtypes_and_relu():
    """bf16 -> fp32 and fp32 -> bf16 forwards and the fused ReLU forward on the
    group-wave kernel match the streaming kernels bit for bit."""
    site = synth.Site(1, 16, 32, 32, 32, 4, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=23))
    outs = {}
    for path in (gn.PATH_STREAMING, gn.PATH_RESIDENT):
        gn.gn3d_debug_set(gn.DEBUG_PATH, path)
        r = [to_np(t) for t in run_forward(site, d["x"], d["gamma"], d["beta"], out_dtype=synth.F32)]
        r += [to_np(t) for t in run_forward_relu(site, d["x"], d["gamma"], d["beta"])]
        torch().cuda.synchronize()
        outs[path] = r
    assert same(outs[gn.PATH_STREAMING], outs[gn.PATH_RESIDENT])


def test_group_wave_timeout_reports_and_recovers():
    site = synth.Site(1, 8, 32, 32, 32, 4, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=24))
    ref = run_all(site, d)
    st = torch().cuda.current_stream().cuda_stream
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_RESIDENT)
    gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 20000)
    gn.gn3d_debug_set(gn.DEBUG_FORCE_TIMEOUT, 1)
    run_forward(site, d["x"], d["gamma"], d["beta"])
    L = gn.lib()
    assert L.gn3d_stream_status(st) == gn.ERR_TIMEOUT
    assert L.gn3d_stream_status(st) == gn.OK
    gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 0)
    assert same(ref, run_all(site, d))


# The cluster kernels (one cluster per group, the group held in the cluster's
# shared memory): groups of 1 .. 64 rows, rows of 1, 3, 8, 17 (a second block
# of one unit) units, 1 .. 16 CTAs per cluster, N > 1 (the parameter gradients
# across clusters), fp32; the backward of the 17-unit rows holds too many units
# per CTA and stays on the streaming kernels.
CLUSTER = [
    (1, 512, 16, 16, 16, 8, synth.BF16),
    (1, 64, 16, 16, 16, 8, synth.BF16),
    (2, 32, 32, 32, 32, 8, synth.BF16),
    (1, 8, 17, 64, 64, 2, synth.BF16),
    (1, 16, 16, 16, 16, 16, synth.BF16),
    (3, 24, 8, 32, 48, 6, synth.BF16),
    (2, 16, 16, 16, 16, 4, synth.F32),
    (1, 12, 3, 64, 64, 3, synth.F32),
]


def _launches(site, d):
    """Kernel launches of one forward and of one backward."""
    n0 = gn.gn3d_launch_count()
    y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
    n1 = gn.gn3d_launch_count()
    run_backward(site, d["dy"], d["x"], mean, rstd, d["gamma"])
    torch().cuda.synchronize()
    return n1 - n0, gn.gn3d_launch_count() - n1


@pytest.mark.parametrize("shape", CLUSTER, ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_cluster_and_streaming_bit_identical(shape):
    """The cluster kernels and the streaming kernels give the same bits: the
    same units, merge blocks and group merges, the block results gathered in
    distributed shared memory instead of global memory.  The cluster forward is
    one launch; so is the backward where its units fit."""
    site = synth.Site(*shape)
    d = device_inputs(synth.make_inputs(site, seed=25))
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_STREAMING)
    a = run_all(site, d)
    assert _launches(site, d) == (2, 2)
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_CLUSTER)
    b = run_all(site, d)
    gn.gn3d_stream_status(torch().cuda.current_stream().cuda_stream)
    assert same(a, b)
    fwd, bwd = _launches(site, d)
    assert fwd == 1
    assert bwd == (2 if shape[2:5] == (17, 64, 64) else 1)
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_AUTO)  # the automatic choice takes them too
    assert _launches(site, d) == (fwd, bwd)


def test_cluster_mixed_dtypes_relu_and_no_affine():
    """bf16 -> fp32 and fp32 -> bf16 forwards, the fused ReLU forward, and no
    affine parameters, on the cluster kernels, match the streaming kernels bit
    for bit (the fused ReLU's backward stays on the streaming kernels)."""
    site = synth.Site(1, 64, 16, 16, 16, 8, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=26))
    outs = {}
    for path in (gn.PATH_STREAMING, gn.PATH_CLUSTER):
        gn.gn3d_debug_set(gn.DEBUG_PATH, path)
        r = [to_np(t) for t in run_forward(site, d["x"], d["gamma"], d["beta"], out_dtype=synth.F32)]
        r += [to_np(t) for t in run_forward_relu(site, d["x"], d["gamma"], d["beta"])]
        y, mean, rstd = run_forward(site, d["x"], None, None)
        r += [to_np(t) for t in (y, mean, rstd)]
        r += [to_np(t) for t in run_backward(site, d["dy"], d["x"], mean, rstd, None)]
        torch().cuda.synchronize()
        outs[path] = r
    assert same(outs[gn.PATH_STREAMING], outs[gn.PATH_CLUSTER])


def test_cluster_timeout_reports_and_recovers():
    site = synth.Site(1, 64, 16, 16, 16, 8, synth.BF16)
    d = device_inputs(synth.make_inputs(site, seed=27))
    ref = run_all(site, d)
    st = torch().cuda.current_stream().cuda_stream
    L = gn.lib()
    gn.gn3d_debug_set(gn.DEBUG_PATH, gn.PATH_CLUSTER)
    gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 20000)
    for direction in ("forward", "backward"):
        y, mean, rstd = run_forward(site, d["x"], d["gamma"], d["beta"])
        torch().cuda.synchronize()
        gn.gn3d_debug_set(gn.DEBUG_FORCE_TIMEOUT, 1)
        if direction == "forward":
            run_forward(site, d["x"], d["gamma"], d["beta"])
        else:
            run_backward(site, d["dy"], d["x"], mean, rstd, d["gamma"])
        assert L.gn3d_stream_status(st) == gn.ERR_TIMEOUT
        assert L.gn3d_stream_status(st) == gn.OK
    gn.gn3d_debug_set(gn.DEBUG_SPIN_LIMIT, 0)
    assert same(ref, run_all(site, d))
