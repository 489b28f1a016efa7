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

from . import parity
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


def close(site, a, b):
    """Within the tests' tolerance: bf16 outputs within 1 ulp, fp32 within 1e-5 rel + 1e-6 abs."""
    ya, yb = to_np(a[0]), to_np(b[0])
    if site.dtype == synth.BF16:
        ok = np.abs(parity.bf16_ordinal(ya) - parity.bf16_ordinal(yb)) <= 1
    else:
        ok = parity.check_f32(ya, yb.astype(np.float64))
    ms = [to_np(t).astype(np.float64) for t in (a[1], a[2], b[1], b[2])]
    return bool(ok.all() and np.allclose(ms[0], ms[2], rtol=1e-5, atol=1e-6)
                and np.allclose(ms[1], ms[3], rtol=1e-5))


@pytest.mark.parametrize("shape", [(1, 32, 40, 40, 40, 8, synth.BF16), (2, 8, 5, 6, 7, 4, synth.F32)],
                         ids=["bf16_40^3", "f32_ragged"])
def test_noalloc_matches_forward_twice_in_a_row(shape):
    site = synth.Site(*shape)
    for seed in (21, 22):  # two calls in a row on different data: the shared area is reused
        d = device_inputs(synth.make_inputs(site, seed=seed))
        ref = run_forward(site, d["x"], d["gamma"], d["beta"])
        got = forward_noalloc(site, d["x"], d["gamma"], d["beta"])
        torch().cuda.synchronize()
        assert close(site, got, ref)


def test_noalloc_rejects_shapes_beyond_its_area():
    t = torch()
    x = t.empty(16, dtype=t.bfloat16, device="cuda")
    with pytest.raises(gn.GN3DError) as e:
        # 2**20 rows of 8 elements: one unit per row, far more scratch than the static area holds
        gn.gn3d_forward_noalloc(x.data_ptr(), None, None, 1, 1 << 20, 1, 1, 8, 1, 1e-5, gn.BF16, gn.BF16,
                                x.data_ptr(), None, None, t.cuda.current_stream().cuda_stream)
    assert e.value.status == gn.ERR_INVALID_ARG
    assert "bytes of scratch" in str(e.value)
