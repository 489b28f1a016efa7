"""Guard bands around every output: no entry point writes outside its buffers.

compute-sanitizer is not available for these runs, so each output (y, mean,
rstd, dx, dgamma, dbeta) is placed in the middle of a larger allocation whose
64 KiB on either side hold a byte pattern; after the calls the pattern must be
intact.  The shapes reach the kernels' edge cases: ragged rows (the 48x97^3
site in miniature), fp32, single-element groups, channels-last with 264 and
768 channels, the fused ReLU, the allocation-free forward and the other launch
forms."""
import numpy as np
import pytest

import bwd_gn3d_stats_gb300 as gn
from bwd_gn3d_stats_gb300 import synth

from .gpu_util import code, device_inputs, to_dev, torch

pytestmark = pytest.mark.gpu
GUARD = 64 * 1024
PATTERN = 0xA5


class Guarded:
    """numel elements of dtype in the middle of a pattern-filled allocation."""

    def __init__(self, numel, dtype):
        t = torch()
        self.es = t.empty((), dtype=dtype).element_size()
        self.buf = t.full((2 * GUARD + max(numel, 1) * self.es,), PATTERN, dtype=t.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + numel * self.es].view(dtype)

    def ptr(self):
        return self.t.data_ptr()

    def intact(self):
        head = self.buf[:GUARD].cpu().numpy()
        tail = self.buf[-GUARD:].cpu().numpy()
        return bool(np.all(head == PATTERN) and np.all(tail == PATTERN))


def _dt(dtype):
    t = torch()
    return t.bfloat16 if dtype == synth.BF16 else t.float32


def run_guarded(site, d, relu=False, ndhwc=False, noalloc=False):
    """Forward then backward writing into guarded outputs; returns them."""
    t = torch()
    st = t.cuda.current_stream().cuda_stream
    y = Guarded(site.numel, _dt(site.dtype))
    mean, rstd = Guarded(site.N * site.G, t.float32), Guarded(site.N * site.G, t.float32)
    dx = Guarded(site.numel, _dt(site.dtype))
    dg, db = Guarded(site.C, t.float32), Guarded(site.C, t.float32)
    c = code(site.dtype)
    shape = (site.N, site.C, site.D, site.H, site.W, site.G)
    if noalloc:
        fwd = gn.gn3d_forward_noalloc
    elif ndhwc:
        fwd = gn.gn3d_forward_ndhwc_relu if relu else gn.gn3d_forward_ndhwc
    else:
        fwd = gn.gn3d_forward_relu if relu else gn.gn3d_forward
    fwd(d["x"].data_ptr(), d["gamma"].data_ptr(), d["beta"].data_ptr(), *shape, site.eps, c, c, y.ptr(),
        mean.ptr(), rstd.ptr(), st)
    args = (d["gamma"].data_ptr(), *shape, c, dx.ptr(), dg.ptr(), db.ptr(), st)
    if relu:
        bwd = gn.gn3d_backward_ndhwc_relu if ndhwc else gn.gn3d_backward_relu
        bwd(d["dy"].data_ptr(), d["x"].data_ptr(), y.ptr(), mean.ptr(), rstd.ptr(), *args)
    else:
        bwd = gn.gn3d_backward_ndhwc if ndhwc else gn.gn3d_backward
        bwd(d["dy"].data_ptr(), d["x"].data_ptr(), mean.ptr(), rstd.ptr(), *args)
    gn.gn3d_stream_status(st)
    return [y, mean, rstd, dx, dg, db]


CASES = [
    ("ragged_97_mini", (1, 48, 9, 9, 9, 8, synth.BF16), {}),
    ("ragged_f32", (2, 8, 5, 6, 7, 4, synth.F32), {}),
    ("single_element_groups", (3, 8, 1, 1, 1, 8, synth.F32), {}),
    ("whole_units", (1, 16, 16, 16, 32, 4, synth.BF16), {}),
    ("relu_ragged", (1, 24, 13, 11, 9, 8, synth.BF16), {"relu": True}),
    ("ndhwc_264", (1, 264, 5, 6, 7, 8, synth.BF16), {"ndhwc": True}),
    ("ndhwc_768", (1, 768, 3, 4, 5, 8, synth.BF16), {"ndhwc": True}),
    ("ndhwc_f32_relu", (2, 32, 4, 5, 6, 4, synth.F32), {"ndhwc": True, "relu": True}),
    ("noalloc_ragged", (1, 48, 9, 9, 9, 8, synth.BF16), {"noalloc": True}),
]


@pytest.mark.parametrize("name,shape,kw", CASES, ids=[c[0] for c in CASES])
def test_outputs_stay_inside_their_buffers(name, shape, kw):
    site = synth.Site(*shape)
    inp = synth.make_inputs(site, seed=51)
    d = device_inputs(inp)
    if kw.get("ndhwc"):
        import oracle

        for k in ("x", "dy"):
            d[k] = to_dev(oracle.ncdhw_to_ndhwc(inp[k], site.N, site.C, site.S))
    outs = run_guarded(site, d, **kw)
    torch().cuda.synchronize()
    for what, g in zip(("y", "mean", "rstd", "dx", "dgamma", "dbeta"), outs):
        assert g.intact(), f"{name}: a guard band around {what} was written"


@pytest.mark.parametrize("path", ["streaming", "fused", "resident", "cluster"])
@pytest.mark.parametrize("shape", [(1, 48, 9, 9, 9, 8, synth.BF16), (2, 16, 16, 16, 16, 4, synth.F32),
                                   (1, 32, 32, 32, 32, 8, synth.BF16), (1, 512, 16, 16, 16, 8, synth.BF16)],
                         ids=lambda s: "x".join(map(str, s[:6])) + "_" + s[6])
def test_other_launch_forms_stay_inside(path, shape, testing_build):
    testing_build.gn3d_debug_set(testing_build.DEBUG_PATH,
                                 {"streaming": 1, "fused": 2, "resident": 3, "cluster": 4}[path])
    site = synth.Site(*shape)
    d = device_inputs(synth.make_inputs(site, seed=52))
    outs = run_guarded(site, d)
    torch().cuda.synchronize()
    assert all(g.intact() for g in outs)
