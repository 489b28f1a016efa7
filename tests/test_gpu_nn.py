"""The torch front end on the GPU: the module and its autograd give exactly the
C ABI's results, load nn.GroupNorm's state dict, and agree with torch's own
fp32 GroupNorm (and ReLU) within fp32 rounding."""
import numpy as np
import pytest

import bwd_gn3d_stats_gb300 as gn

from .gpu_util import to_np, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bwd_gn3d_stats_gb300 import build

    build.build()


def same(u, v):
    return np.array_equal(to_np(u), to_np(v))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("affine", [True, False])
@pytest.mark.parametrize("relu", [False, True])
def test_module_is_the_c_abi(dtype, affine, relu):
    from bwd_gn3d_stats_gb300.nn import GroupNorm3d

    t = torch()
    tdt = t.bfloat16 if dtype == "bf16" else t.float32
    gen = t.Generator(device="cuda").manual_seed(5)
    N, C, D, H, W, G = 2, 16, 9, 10, 11, 4
    x = t.randn(N, C, D, H, W, device="cuda", generator=gen).to(tdt)
    dy = t.randn(N, C, D, H, W, device="cuda", generator=gen).to(tdt)
    m = GroupNorm3d(G, C, affine=affine, activation="relu" if relu else None).cuda()
    if affine:
        with t.no_grad():
            m.weight.uniform_(0.5, 1.5, generator=gen)
            m.bias.normal_(0, 0.3, generator=gen)
    xr = x.clone().requires_grad_()
    y = m(xr)
    y.backward(dy)
    w = m.weight.detach() if affine else None
    b = m.bias.detach() if affine else None
    y0, mean, rstd = gn.forward(x, w, b, G, 1e-5, relu=relu)
    dx0, dg0, db0 = gn.backward(dy, x, mean, rstd, w, G, out=y0 if relu else None)
    assert y.dtype == tdt and same(y, y0)
    assert same(xr.grad, dx0)
    if affine:
        assert same(m.weight.grad, dg0) and same(m.bias.grad, db0)


def test_module_loads_nn_groupnorm_and_matches_it():
    from bwd_gn3d_stats_gb300.nn import GroupNorm3d

    t = torch()
    gen = t.Generator(device="cuda").manual_seed(6)
    ref = t.nn.GroupNorm(8, 32).cuda()
    with t.no_grad():
        ref.weight.uniform_(0.5, 1.5, generator=gen)
        ref.bias.normal_(0, 0.3, generator=gen)
    ours = GroupNorm3d(8, 32, activation="relu").cuda()
    ours.load_state_dict(ref.state_dict())
    x = t.randn(2, 32, 12, 12, 12, device="cuda", generator=gen)
    dy = t.randn(2, 32, 12, 12, 12, device="cuda", generator=gen)
    x1, x2 = x.clone().requires_grad_(), x.clone().requires_grad_()
    y1 = ours(x1)
    y2 = t.relu(ref(x2))
    y1.backward(dy)
    y2.backward(dy)
    assert t.allclose(y1, y2, rtol=1e-5, atol=1e-5)
    assert t.allclose(x1.grad, x2.grad, rtol=1e-4, atol=1e-5)
    assert t.allclose(ours.weight.grad, ref.weight.grad, rtol=1e-4, atol=1e-3)
    assert t.allclose(ours.bias.grad, ref.bias.grad, rtol=1e-4, atol=1e-3)


def test_relu_needs_matching_out_dtype():
    from bwd_gn3d_stats_gb300.nn import group_norm_3d

    t = torch()
    x = t.randn(1, 8, 4, 4, 4, device="cuda").to(t.bfloat16)
    with pytest.raises(ValueError):
        group_norm_3d(x, 4, out_dtype=t.float32, relu=True)
    y = group_norm_3d(x, 4, out_dtype=t.float32)  # without the ReLU any pair is allowed
    assert y.dtype == t.float32


@pytest.mark.parametrize("relu", [False, True])
def test_channels_last_module_runs_ndhwc(relu):
    """A channels_last_3d input runs the NDHWC kernels (bit for bit the C ABI's
    NDHWC entry points), keeps its memory format in y and dx, and agrees with
    the NCDHW path to rounding."""
    from bwd_gn3d_stats_gb300.nn import GroupNorm3d

    t = torch()
    cl = t.channels_last_3d
    gen = t.Generator(device="cuda").manual_seed(7)
    N, C, D, H, W, G = 2, 32, 10, 11, 12, 8
    x = t.randn(N, C, D, H, W, device="cuda", generator=gen).to(t.bfloat16).contiguous(memory_format=cl)
    dy = t.randn(N, C, D, H, W, device="cuda", generator=gen).to(t.bfloat16).contiguous(memory_format=cl)
    m = GroupNorm3d(G, C, activation="relu" if relu else None).cuda()
    with t.no_grad():
        m.weight.uniform_(0.5, 1.5, generator=gen)
        m.bias.normal_(0, 0.3, generator=gen)
    xr = x.clone().requires_grad_()
    y = m(xr)
    y.backward(dy)
    assert y.is_contiguous(memory_format=cl) and not y.is_contiguous()
    assert xr.grad.is_contiguous(memory_format=cl)
    w, b = m.weight.detach(), m.bias.detach()
    n0 = gn.gn3d_launch_count()
    y0, mean, rstd = gn.forward_ndhwc(x, w, b, G, 1e-5, relu=relu)
    dx0, dg0, db0 = gn.backward_ndhwc(dy, x, mean, rstd, w, G, out=y0 if relu else None)
    assert gn.gn3d_launch_count() - n0 == 6  # three kernels per direction
    assert t.equal(y.view(t.int16), y0.view(t.int16)) and t.equal(xr.grad.view(t.int16), dx0.view(t.int16))
    assert t.equal(m.weight.grad, dg0) and t.equal(m.bias.grad, db0)
    # the NCDHW path on the same logical tensor
    m2 = GroupNorm3d(G, C, activation="relu" if relu else None).cuda()
    m2.load_state_dict(m.state_dict())
    x2 = x.contiguous().requires_grad_()
    y2 = m2(x2)
    y2.backward(dy.contiguous())
    d = (y.float() - y2.float()).abs().max().item()
    assert d <= 2 ** -6 * max(1.0, y2.float().abs().max().item())
    assert t.allclose(m.weight.grad, m2.weight.grad, rtol=1e-4, atol=1e-3)


def test_channels_last_with_c_not_multiple_of_8_takes_ncdhw():
    from bwd_gn3d_stats_gb300.nn import GroupNorm3d

    t = torch()
    gen = t.Generator(device="cuda").manual_seed(8)
    x = t.randn(1, 12, 6, 6, 6, device="cuda", generator=gen).contiguous(memory_format=t.channels_last_3d)
    m = GroupNorm3d(3, 12).cuda()
    y = m(x)
    ref = t.nn.functional.group_norm(x.contiguous(), 3, m.weight, m.bias, 1e-5)
    assert t.allclose(y, ref, rtol=1e-5, atol=1e-5)


def test_misaligned_views_are_handled():
    """Views whose storage offset breaks 16-byte alignment (the C ABI rejects
    those pointers) still run: the front end copies them to an aligned buffer."""
    from bwd_gn3d_stats_gb300.nn import group_norm_3d

    t = torch()
    gen = t.Generator(device="cuda").manual_seed(9)
    base = t.randn(1 + 2 * 16 * 6 * 6 * 6, device="cuda", generator=gen).to(t.bfloat16)
    x = base[1:].view(2, 16, 6, 6, 6)  # 2-byte offset
    assert x.data_ptr() % 16 != 0
    w = t.rand(16, device="cuda", generator=gen) + 0.5
    b = t.randn(16, device="cuda", generator=gen)
    y = group_norm_3d(x, 4, w, b)
    y_ref = group_norm_3d(x.clone(), 4, w, b)
    assert t.equal(y.view(t.int16), y_ref.view(t.int16))
    dyb = t.randn(1 + y.numel(), device="cuda", generator=gen).to(t.bfloat16)
    dy = dyb[1:].view_as(y)
    xr2 = x.clone().requires_grad_()
    group_norm_3d(xr2, 4, w, b).backward(dy)
    xr3 = x.clone().requires_grad_()
    group_norm_3d(xr3, 4, w, b).backward(dy.clone())
    assert t.equal(xr2.grad.view(t.int16), xr3.grad.view(t.int16))


@pytest.mark.parametrize("channels_last", [False, True])
def test_fp32_gradient_of_bf16_input_is_not_narrowed(channels_last):
    """out_dtype=float32 on a bf16 input: the fp32 gradient reaches the backward
    unrounded (the backward runs on x widened exactly to fp32), and dx is
    rounded once to bf16 -- not the backward of the gradient rounded to bf16."""
    from bwd_gn3d_stats_gb300.nn import GroupNorm3d

    t = torch()
    g = t.Generator(device="cuda").manual_seed(9)
    x = (t.randn((2, 16, 6, 7, 8), generator=g, device="cuda") * 2 + 1).to(t.bfloat16)
    if channels_last:
        x = x.contiguous(memory_format=t.channels_last_3d)
    dy = t.randn((2, 16, 6, 7, 8), generator=g, device="cuda") * (1 + 2 ** -12)  # not bf16 values
    m = GroupNorm3d(4, 16, out_dtype=t.float32).cuda()
    with t.no_grad():
        m.weight.uniform_(0.5, 1.5)
        m.bias.normal_(0, 0.1)
    xr = x.detach().requires_grad_(True)
    y = m(xr)
    assert y.dtype == t.float32
    y.backward(dy)
    # the same backward through the C ABI on the widened input and the fp32 gradient
    xf = x.float().contiguous(memory_format=t.channels_last_3d if channels_last else t.contiguous_format)
    _, mean, rstd = (gn.forward_ndhwc if channels_last else gn.forward)(x, m.weight.detach(), m.bias.detach(), 4,
                                                                       1e-5, t.float32)
    fn = gn.backward_ndhwc if channels_last else gn.backward
    mf = t.channels_last_3d if channels_last else t.contiguous_format
    dx32, dg32, db32 = fn(dy.contiguous(memory_format=mf), xf, mean, rstd, m.weight.detach(), 4)
    assert same(xr.grad, dx32.to(t.bfloat16)) and same(m.weight.grad, dg32) and same(m.bias.grad, db32)
    # and it differs from the backward of the gradient narrowed to bf16
    _, dgn, _ = fn(dy.to(t.bfloat16).contiguous(memory_format=mf), x, mean, rstd, m.weight.detach(), 4)
    assert not same(m.weight.grad, dgn)
