"""Helpers for the GPU tests: run libgn3d through its C ABI on numpy inputs."""
from __future__ import annotations

import numpy as np

import bwd_gn3d_stats_gb300 as gn
from bwd_gn3d_stats_gb300 import synth


def torch():
    import torch as t

    return t


def to_dev(a: np.ndarray, dev="cuda"):
    t = torch()
    if a.dtype == np.uint16:
        return t.from_numpy(a.view(np.int16)).to(dev).view(t.bfloat16)
    return t.from_numpy(a).to(dev)


def to_np(t_):
    t = torch()
    t_ = t_.detach().contiguous().cpu()
    if t_.dtype == t.bfloat16:
        return t_.view(t.int16).numpy().view(np.uint16).reshape(-1).copy()
    return t_.numpy().reshape(-1).copy()


def code(dtype: str) -> int:
    return gn.BF16 if dtype == synth.BF16 else gn.F32


def run_forward(site: synth.Site, x, gamma, beta, out_dtype: str | None = None, eps=None):
    """x, gamma, beta: device tensors. Returns device (y, mean, rstd)."""
    t = torch()
    out_dtype = out_dtype or site.dtype
    y = t.empty(site.numel, dtype=t.bfloat16 if out_dtype == synth.BF16 else t.float32, device=x.device)
    mean = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    rstd = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    gn.gn3d_forward(x.data_ptr(), None if gamma is None else gamma.data_ptr(),
                    None if beta is None else beta.data_ptr(), site.N, site.C, site.D, site.H, site.W, site.G,
                    site.eps if eps is None else eps, code(site.dtype), code(out_dtype), y.data_ptr(),
                    mean.data_ptr(), rstd.data_ptr(), t.cuda.current_stream().cuda_stream)
    return y, mean, rstd


def run_backward(site: synth.Site, dy, x, mean, rstd, gamma):
    t = torch()
    dx = t.empty_like(x)
    dgamma = t.empty(site.C, dtype=t.float32, device=x.device)
    dbeta = t.empty(site.C, dtype=t.float32, device=x.device)
    gn.gn3d_backward(dy.data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                     None if gamma is None else gamma.data_ptr(), site.N, site.C, site.D, site.H, site.W,
                     site.G, code(site.dtype), dx.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(),
                     t.cuda.current_stream().cuda_stream)
    return dx, dgamma, dbeta


def device_inputs(inp):
    return {k: to_dev(v) for k, v in inp.items()}


def run_forward_relu(site: synth.Site, x, gamma, beta, out_dtype: str | None = None):
    """The fused GroupNorm + ReLU forward (C entry point gn3d_forward_relu)."""
    t = torch()
    out_dtype = out_dtype or site.dtype
    y = t.empty(site.numel, dtype=t.bfloat16 if out_dtype == synth.BF16 else t.float32, device=x.device)
    mean = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    rstd = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    gn.gn3d_forward_relu(x.data_ptr(), None if gamma is None else gamma.data_ptr(),
                         None if beta is None else beta.data_ptr(), site.N, site.C, site.D, site.H, site.W, site.G,
                         site.eps, code(site.dtype), code(out_dtype), y.data_ptr(), mean.data_ptr(),
                         rstd.data_ptr(), t.cuda.current_stream().cuda_stream)
    return y, mean, rstd


def run_backward_relu(site: synth.Site, dy, x, out, mean, rstd, gamma):
    t = torch()
    dx = t.empty_like(x)
    dgamma = t.empty(site.C, dtype=t.float32, device=x.device)
    dbeta = t.empty(site.C, dtype=t.float32, device=x.device)
    gn.gn3d_backward_relu(dy.data_ptr(), x.data_ptr(), out.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                          None if gamma is None else gamma.data_ptr(), site.N, site.C, site.D, site.H, site.W,
                          site.G, code(site.dtype), dx.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(),
                          t.cuda.current_stream().cuda_stream)
    return dx, dgamma, dbeta


# ------------------------------------------------ channels-last (NDHWC) runs
# Inputs and outputs are flat NDHWC storage (element (n, c, s) at (n*S + s)*C + c).

def run_forward_ndhwc(site: synth.Site, x, gamma, beta, out_dtype: str | None = None, relu: bool = False):
    t = torch()
    out_dtype = out_dtype or site.dtype
    y = t.empty(site.numel, dtype=t.bfloat16 if out_dtype == synth.BF16 else t.float32, device=x.device)
    mean = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    rstd = t.empty(site.N * site.G, dtype=t.float32, device=x.device)
    fn = gn.gn3d_forward_ndhwc_relu if relu else gn.gn3d_forward_ndhwc
    fn(x.data_ptr(), None if gamma is None else gamma.data_ptr(), None if beta is None else beta.data_ptr(),
       site.N, site.C, site.D, site.H, site.W, site.G, site.eps, code(site.dtype), code(out_dtype), y.data_ptr(),
       mean.data_ptr(), rstd.data_ptr(), t.cuda.current_stream().cuda_stream)
    return y, mean, rstd


def run_backward_ndhwc(site: synth.Site, dy, x, mean, rstd, gamma, out=None):
    t = torch()
    dx = t.empty_like(x)
    dgamma = t.empty(site.C, dtype=t.float32, device=x.device)
    dbeta = t.empty(site.C, dtype=t.float32, device=x.device)
    g = None if gamma is None else gamma.data_ptr()
    st = t.cuda.current_stream().cuda_stream
    args = (site.N, site.C, site.D, site.H, site.W, site.G, code(site.dtype), dx.data_ptr(), dgamma.data_ptr(),
            dbeta.data_ptr(), st)
    if out is None:
        gn.gn3d_backward_ndhwc(dy.data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), g, *args)
    else:
        gn.gn3d_backward_ndhwc_relu(dy.data_ptr(), x.data_ptr(), out.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                                    g, *args)
    return dx, dgamma, dbeta
