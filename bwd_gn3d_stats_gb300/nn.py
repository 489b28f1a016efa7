"""torch front end of libgn3d: an autograd Function and a drop-in module for
nn.GroupNorm over contiguous NCDHW volumes.

ScaFFold PR #93 "Optimize GroupNorm" keeps nn.GroupNorm's weight and bias, so
GroupNorm3d has the same parameters and state-dict keys; PR #105 "Preserve
GroupNorm dtype" fixes the output dtype policy (the input's dtype unless asked
otherwise); the GroupNorm pages' FastGroupNorm takes an activation argument
that fuses the following ReLU (gn3d_forward_relu / gn3d_backward_relu).

Memory format: a channels_last_3d input (as channels-last convolutions
produce it) runs the NDHWC entry points and gives a channels_last_3d output,
with no layout conversion; any other input runs the NCDHW entry points on its
contiguous form.  The NDHWC kernels need C % 8 == 0; other channel counts take
the NCDHW path.

Gradient dtype: the backward runs in x's dtype when the incoming gradient has
it (or is narrower: a bf16 gradient of an fp32 input widens exactly).  With
out_dtype=float32 on a bf16 input the incoming gradient is fp32; it is not
narrowed -- the backward then runs on fp32 copies of x (exact) and of the
gradient, and dx is rounded once to bf16, so no gradient precision is lost
before the backward's sums (PR #105 "Preserve GroupNorm dtype": compute in
fp32, round once on the store).

Every computation runs in libgn3d's kernels: this file only allocates outputs,
saves what the backward needs and converts the incoming gradient to the
backward's dtype and layout.  There is no CPU path -- a CPU tensor raises.
"""
from __future__ import annotations

import torch

from . import backward as _backward
from . import backward_ndhwc as _backward_ndhwc
from . import forward as _forward
from . import forward_ndhwc as _forward_ndhwc
from . import is_ndhwc as _is_ndhwc


def _aligned(t: torch.Tensor, memory_format=torch.contiguous_format) -> torch.Tensor:
    """t in the given memory format, starting on a 16-byte boundary (the C ABI's
    vector loads need it; a view with an odd storage offset is copied)."""
    t = t.contiguous(memory_format=memory_format)
    if t.data_ptr() % 16:
        t = t.clone(memory_format=memory_format)
    return t


def _check_input(x: torch.Tensor):
    if not x.is_cuda:
        raise RuntimeError("libgn3d runs on CUDA tensors only (there is no CPU path)")
    if x.dim() != 5:
        raise ValueError(f"expected an NCDHW tensor, got {x.dim()} dimensions")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError(f"libgn3d supports bfloat16 and float32 inputs, got {x.dtype}")


class GroupNorm3dFunction(torch.autograd.Function):
    """y = GroupNorm(x) (then ReLU when relu is set), with libgn3d's backward."""

    @staticmethod
    def forward(ctx, x, weight, bias, num_groups: int, eps: float, out_dtype, relu: bool):
        _check_input(x)
        out_dtype = x.dtype if out_dtype is None else out_dtype
        if relu and out_dtype != x.dtype:
            raise ValueError("the fused ReLU's backward gates on the forward's result in x's dtype: "
                             "out_dtype must equal x.dtype when relu is set")
        ndhwc = _is_ndhwc(x) and x.shape[1] % 8 == 0
        x = _aligned(x, torch.channels_last_3d if ndhwc else torch.contiguous_format)
        w = None if weight is None else weight.detach().float().contiguous()
        b = None if bias is None else bias.detach().float().contiguous()
        fwd = _forward_ndhwc if ndhwc else _forward
        y, mean, rstd = fwd(x, w, b, num_groups, eps, out_dtype, relu)
        ctx.num_groups = num_groups
        ctx.relu = relu
        ctx.ndhwc = ndhwc
        ctx.weight_dtype = None if weight is None else weight.dtype
        ctx.bias_dtype = None if bias is None else bias.dtype
        ctx.save_for_backward(x, w, mean, rstd, y if relu else None)
        return y

    @staticmethod
    def backward(ctx, dy):
        x, w, mean, rstd, y = ctx.saved_tensors
        xb = x
        if dy.dtype == torch.float32 and x.dtype == torch.bfloat16:
            # an fp32 gradient of a bf16 input (out_dtype=float32): keep it; the
            # backward runs on x widened to fp32 (exact) and dx is rounded once
            xb = x.float()
        mf = torch.channels_last_3d if ctx.ndhwc else torch.contiguous_format
        dy = _aligned(dy.to(xb.dtype), mf)
        xb = _aligned(xb, mf)
        if ctx.ndhwc:
            dx, dgamma, dbeta = _backward_ndhwc(dy, xb, mean, rstd, w, ctx.num_groups, out=y if ctx.relu else None)
        else:
            dx, dgamma, dbeta = _backward(dy, xb, mean, rstd, w, ctx.num_groups, out=y if ctx.relu else None)
        dx = dx.to(x.dtype)
        gw = dgamma.to(ctx.weight_dtype) if ctx.weight_dtype is not None and ctx.needs_input_grad[1] else None
        gb = dbeta.to(ctx.bias_dtype) if ctx.bias_dtype is not None and ctx.needs_input_grad[2] else None
        return dx, gw, gb, None, None, None, None


def group_norm_3d(x, num_groups: int, weight=None, bias=None, eps: float = 1e-5, out_dtype=None,
                  relu: bool = False):
    """Functional form: GroupNorm over an [N, C, D, H, W] CUDA tensor, NCDHW or
    channels_last_3d (then ReLU when relu is set)."""
    return GroupNorm3dFunction.apply(x, weight, bias, num_groups, eps, out_dtype, relu)


class GroupNorm3d(torch.nn.Module):
    """Drop-in for torch.nn.GroupNorm on [N, C, D, H, W] volumes (NCDHW or
    channels_last_3d), computed by libgn3d.

    Same constructor arguments, parameters ("weight", "bias") and state-dict keys
    as nn.GroupNorm, plus:
      activation  None or "relu": the ReLU that follows GroupNorm, fused.
      out_dtype   output dtype (default: the input's).
    """

    def __init__(self, num_groups: int, num_channels: int, eps: float = 1e-5, affine: bool = True,
                 activation: str | None = None, out_dtype=None, device=None, dtype=None):
        super().__init__()
        if num_channels % num_groups != 0:
            raise ValueError("num_channels must be divisible by num_groups")
        if activation not in (None, "relu"):
            raise ValueError(f"unsupported activation {activation!r} (None or 'relu')")
        self.num_groups = num_groups
        self.num_channels = num_channels
        self.eps = eps
        self.affine = affine
        self.activation = activation
        self.out_dtype = out_dtype
        if affine:
            kw = {"device": device, "dtype": dtype}
            self.weight = torch.nn.Parameter(torch.ones(num_channels, **kw))
            self.bias = torch.nn.Parameter(torch.zeros(num_channels, **kw))
        else:
            self.register_parameter("weight", None)
            self.register_parameter("bias", None)

    def forward(self, x):
        if x.dim() == 5 and x.shape[1] != self.num_channels:
            raise ValueError(f"expected {self.num_channels} channels, got {x.shape[1]}")
        return GroupNorm3dFunction.apply(x, self.weight, self.bias, self.num_groups, self.eps, self.out_dtype,
                                         self.activation == "relu")

    def extra_repr(self):
        return (f"{self.num_groups}, {self.num_channels}, eps={self.eps}, affine={self.affine}, "
                f"activation={self.activation}")
