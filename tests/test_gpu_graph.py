"""CUDA graph capture: a fwd+bwd step through the C ABI (NCDHW and NDHWC) is
captured once into a CUDA graph and replayed on new inputs; the replays give
bit for bit the results of eager calls on the same inputs."""
import pytest

from .gpu_util import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("layout", ["ncdhw", "ndhwc"])
def test_graph_capture_and_replay(layout):
    import bwd_gn3d_stats_gb300 as gn
    from bwd_gn3d_stats_gb300 import build

    build.build()
    t = torch()
    cl = layout == "ndhwc"
    fmt = t.channels_last_3d if cl else t.contiguous_format
    N, C, D, H, W, G = 2, 32, 12, 13, 14, 8
    gen = t.Generator(device="cuda").manual_seed(11)

    def fresh():
        x = t.randn(N, C, D, H, W, device="cuda", generator=gen).to(t.bfloat16).contiguous(memory_format=fmt)
        dy = t.randn(N, C, D, H, W, device="cuda", generator=gen).to(t.bfloat16).contiguous(memory_format=fmt)
        return x, dy

    gamma = t.rand(C, device="cuda", generator=gen) + 0.5
    beta = t.randn(C, device="cuda", generator=gen)
    fwd = gn.forward_ndhwc if cl else gn.forward
    bwd = gn.backward_ndhwc if cl else gn.backward
    x_static, dy_static = fresh()
    # warm up on a side stream (first calls set up per-device state), then capture
    s = t.cuda.Stream()
    s.wait_stream(t.cuda.current_stream())
    with t.cuda.stream(s):
        for _ in range(2):
            y, m, r = fwd(x_static, gamma, beta, G)
            bwd(dy_static, x_static, m, r, gamma, G)
    t.cuda.current_stream().wait_stream(s)
    t.cuda.synchronize()
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g):
        y_g, m_g, r_g = fwd(x_static, gamma, beta, G)
        dx_g, dg_g, db_g = bwd(dy_static, x_static, m_g, r_g, gamma, G)
    for _ in range(3):
        x_new, dy_new = fresh()
        x_static.copy_(x_new)
        dy_static.copy_(dy_new)
        g.replay()
        y_e, m_e, r_e = fwd(x_new, gamma, beta, G)
        dx_e, dg_e, db_e = bwd(dy_new, x_new, m_e, r_e, gamma, G)
        t.cuda.synchronize()
        assert t.equal(y_g.view(t.int16), y_e.view(t.int16))
        assert t.equal(dx_g.view(t.int16), dx_e.view(t.int16))
        for a, b in ((m_g, m_e), (r_g, r_e), (dg_g, dg_e), (db_g, db_e)):
            assert t.equal(a.view(t.int32), b.view(t.int32))
