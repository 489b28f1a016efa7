"""Host-side fault injection (testing build): a failed scratch allocation or a
failed first kernel launch makes the call return GN3D_ERR_CUDA with nothing
left behind -- its scratch is freed (the pool's used bytes return to where they
were) -- and the next call gives the same bits as before.  Nothing faults on
the GPU: the failure is made on the host, at the allocation or launch call."""
import numpy as np
import pytest

from bwd_gn3d_stats_gb300 import synth

from .gpu_util import (device_inputs, run_backward, run_backward_ndhwc, run_forward, run_forward_ndhwc, to_dev,
                       to_np, torch)

pytestmark = pytest.mark.gpu


def _ndhwc(site, inp):
    import oracle

    d = device_inputs(inp)
    for k in ("x", "dy"):
        d[k] = to_dev(oracle.ncdhw_to_ndhwc(inp[k], site.N, site.C, site.S))
    return d


ENTRIES = {
    # entry -> (shape, launch form, layout)
    "forward": ((1, 24, 13, 11, 9, 8, synth.BF16), 0, "ncdhw"),
    "backward": ((1, 24, 13, 11, 9, 8, synth.BF16), 0, "ncdhw"),
    "forward_ndhwc": ((1, 32, 6, 7, 8, 8, synth.BF16), 0, "ndhwc"),
    "backward_ndhwc": ((1, 32, 6, 7, 8, 8, synth.BF16), 0, "ndhwc"),
    "forward_group_wave": ((1, 16, 16, 16, 32, 4, synth.BF16), 3, "ncdhw"),
    "backward_group_wave": ((1, 16, 16, 16, 32, 4, synth.BF16), 3, "ncdhw"),
    "forward_persistent": ((2, 8, 5, 6, 7, 4, synth.F32), 2, "ncdhw"),
    "forward_cluster": ((1, 64, 16, 16, 16, 8, synth.BF16), 4, "ncdhw"),
    "backward_cluster": ((1, 64, 16, 16, 16, 8, synth.BF16), 4, "ncdhw"),
}


@pytest.mark.parametrize("fail", ["alloc", "launch"])
@pytest.mark.parametrize("entry", sorted(ENTRIES))
def test_injected_failure_leaves_nothing_behind(entry, fail, testing_build):
    if entry == "forward_cluster" and fail == "alloc":
        pytest.skip("the cluster forward allocates nothing")
    gn = testing_build
    shape, path, layout = ENTRIES[entry]
    gn.gn3d_debug_set(gn.DEBUG_PATH, path)
    site = synth.Site(*shape)
    inp = synth.make_inputs(site, seed=61)
    d = _ndhwc(site, inp) if layout == "ndhwc" else device_inputs(inp)
    fwd, bwd = (run_forward_ndhwc, run_backward_ndhwc) if layout == "ndhwc" else (run_forward, run_backward)
    t = torch()

    def call():
        y, mean, rstd = fwd(site, d["x"], d["gamma"], d["beta"])
        if entry.startswith("forward"):
            return [y, mean, rstd]
        return list(bwd(site, d["dy"], d["x"], mean, rstd, d["gamma"]))

    ref = [to_np(v) for v in call()]
    t.cuda.synchronize()
    used = gn.gn3d_debug_get(gn.DEBUG_POOL_USED)
    if entry.startswith("backward"):  # the forward must succeed, the backward fail
        y, mean, rstd = fwd(site, d["x"], d["gamma"], d["beta"])
        t.cuda.synchronize()
    gn.gn3d_debug_set(gn.DEBUG_FAIL_NEXT, gn.FAIL_ALLOC if fail == "alloc" else gn.FAIL_LAUNCH)
    with pytest.raises(gn.GN3DError) as e:
        if entry.startswith("backward"):
            bwd(site, d["dy"], d["x"], mean, rstd, d["gamma"])
        else:
            fwd(site, d["x"], d["gamma"], d["beta"])
    assert e.value.status == gn.ERR_CUDA
    assert ("scratch allocation" if fail == "alloc" else "launch") in str(e.value)
    t.cuda.synchronize()
    assert gn.gn3d_debug_get(gn.DEBUG_POOL_USED) == used  # the failed call's scratch is back in the pool
    assert gn.lib().gn3d_stream_status(t.cuda.current_stream().cuda_stream) == gn.OK
    again = [to_np(v) for v in call()]
    t.cuda.synchronize()
    for a, b in zip(ref, again):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
