"""gn3d_forward_noalloc: the forward for callers that must not allocate device
memory during a call (fixed memory budgets, code inside another allocator's
critical section).  It runs the same kernel as gn3d_forward with its scratch in
the library's static device area, so its results must match gn3d_forward's.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process (the
first call on the device then does the one-time set-up).
"""
import numpy as np
import pytest

import bwd_gn3d_stats_gb300 as gn
from bwd_gn3d_stats_gb300 import synth

from .gpu_util import code, device_inputs, run_forward, to_np, torch

pytestmark = pytest.mark.gpu


def forward_noalloc(site, x, gamma, beta):
    t = torch()
    y = t.empty(site.numel, dtype=t.bfloat16 if site.dtype == synth.BF16 else t.float32, device=x.device)
    mean = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    rstd = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    gn.gn3d_forward_noalloc(x.data_ptr(), gamma.data_ptr(), beta.data_ptr(), site.N, site.C, site.D, site.H,
                            site.W, site.G, site.eps, code(site.dtype), code(site.dtype), y.data_ptr(),
                            mean.data_ptr(), rstd.data_ptr(), t.cuda.current_stream().cuda_stream)
    return y, mean, rstd


def same_bytes(a, b):
    return all(np.array_equal(to_np(u).view(np.uint8), to_np(v).view(np.uint8)) for u, v in zip(a, b))


@pytest.mark.parametrize("shape", [(1, 32, 40, 40, 40, 8, synth.BF16), (2, 8, 5, 6, 7, 4, synth.F32),
                                   (1, 32, 128, 128, 128, 8, synth.BF16)],
                         ids=["bf16_40^3", "f32_ragged", "bf16_128^3"])
def test_noalloc_matches_forward_twice_in_a_row(shape):
    """Bit for bit the same y, mean and rstd as gn3d_forward (the same units,
    merge blocks and group merges), on two calls in a row with different data:
    the shared area is reused and its counters are cleared by each call."""
    site = synth.Site(*shape)
    for seed in (21, 22):
        d = device_inputs(synth.make_inputs(site, seed=seed))
        ref = run_forward(site, d["x"], d["gamma"], d["beta"])
        got = forward_noalloc(site, d["x"], d["gamma"], d["beta"])
        torch().cuda.synchronize()
        assert same_bytes(got, ref)


def _scratch_fits(C):
    """Whether the area takes shape (1, C, 1, 1, 8) with G = 1, before any pointer
    is looked at: True if the shape's scratch fits (the call then fails on the
    missing pointers instead), False if it is rejected for its scratch."""
    try:
        gn.gn3d_forward_noalloc(None, None, None, 1, C, 1, 1, 8, 1, 1e-5, gn.BF16, gn.BF16, None, None, None,
                                torch().cuda.current_stream().cuda_stream)
    except gn.GN3DError as e:
        assert e.status == gn.ERR_INVALID_ARG
        return "bytes of scratch" not in str(e)
    raise AssertionError("a call without pointers was accepted")


def test_noalloc_at_the_edge_of_its_area():
    """Rows of 8 elements (one unit each): the largest C whose scratch fits runs
    and matches gn3d_forward bit for bit; one more channel is rejected with a
    message naming the bytes needed."""
    lo, hi = 1, 1 << 22
    assert _scratch_fits(lo) and not _scratch_fits(hi)
    while hi - lo > 1:  # largest C that fits
        mid = (lo + hi) // 2
        if _scratch_fits(mid):
            lo = mid
        else:
            hi = mid
    assert 100_000 < lo < 1 << 20  # about 17 B per unit plus per-block words in 8 MiB
    site = synth.Site(1, lo, 1, 1, 8, 1, synth.BF16)
    t = torch()
    g = t.Generator(device="cuda").manual_seed(3)
    x = (t.randn(site.numel, generator=g, device="cuda") * 3 + 1).to(t.bfloat16)
    gamma = t.rand(site.C, generator=g, device="cuda") + 0.5
    beta = t.randn(site.C, generator=g, device="cuda") * 0.1
    ref = run_forward(site, x, gamma, beta)
    got = forward_noalloc(site, x, gamma, beta)
    t.cuda.synchronize()
    assert same_bytes(got, ref)
    with pytest.raises(gn.GN3DError) as e:
        xs = t.empty(16, dtype=t.bfloat16, device="cuda")
        gn.gn3d_forward_noalloc(xs.data_ptr(), None, None, 1, lo + 1, 1, 1, 8, 1, 1e-5, gn.BF16, gn.BF16,
                                xs.data_ptr(), None, None, t.cuda.current_stream().cuda_stream)
    assert e.value.status == gn.ERR_INVALID_ARG and "bytes of scratch" in str(e.value)


def test_noalloc_rejects_shapes_beyond_its_area():
    t = torch()
    x = t.empty(16, dtype=t.bfloat16, device="cuda")
    with pytest.raises(gn.GN3DError) as e:
        # 2**20 rows of 8 elements: one unit per row, far more scratch than the static area holds
        gn.gn3d_forward_noalloc(x.data_ptr(), None, None, 1, 1 << 20, 1, 1, 8, 1, 1e-5, gn.BF16, gn.BF16,
                                x.data_ptr(), None, None, t.cuda.current_stream().cuda_stream)
    assert e.value.status == gn.ERR_INVALID_ARG
    assert "bytes of scratch" in str(e.value)
