"""libgn3d: GroupNorm-3D forward/backward for GB300 (sm_103a) behind a C ABI.

Python binding.  It only marshals arguments: every step of the GroupNorm runs
in the library's CUDA kernels.  There is no CPU or PyTorch fallback -- if the
library is missing or fails to load, every call raises.

Two levels:
  * ``gn3d_forward`` / ``gn3d_backward`` / ``gn3d_stream_status`` mirror the C
    entry points one to one (integer pointers, sizes, dtype codes, stream
    handle) and raise ``GN3DError`` on a non-zero status.
  * ``forward`` / ``backward`` take torch CUDA tensors, allocate the outputs
    with torch and pass torch's current stream.  torch is used for device
    memory and streams only.  ``forward_ndhwc`` / ``backward_ndhwc`` do the same
    for channels_last_3d tensors (the C entry points ``gn3d_*_ndhwc*``).
"""
from __future__ import annotations

import ctypes
import os
import threading

F32, BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_DEVICE, ERR_CUDA, ERR_TIMEOUT = 0, 1, 2, 3, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_libs = {}
_current = "product"


class GN3DError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"gn3d status {status}: {msg}")
        self.status = status


def library_path(kind: str = "product") -> str:
    """The in-tree build of libgn3d: "product" (the shipped library) or "testing"
    (the same sources compiled with the testing and tuning hooks)."""
    from . import build as _b

    return {"product": _b.LIB, "testing": _b.TESTING_LIB}[kind]


def use_library(kind: str) -> str:
    """Route every call of this module to the product or the testing build;
    returns the previous choice.  The tests that set debug hooks run all their
    calls on the testing build (each library keeps its own settings)."""
    global _current
    if kind not in ("product", "testing"):
        raise ValueError("library kind: 'product' or 'testing'")
    prev, _current = _current, kind
    return prev


def lib():
    """The library calls go to (the product build unless use_library('testing'))."""
    return _load(_current)


def _load(kind: str):
    with _lock:
        if kind not in _libs:
            path = library_path(kind)
            if not os.path.exists(path):
                raise RuntimeError(f"libgn3d is not built ({path} missing): run "
                                   "python -m bwd_gn3d_stats_gb300.build")
            L = ctypes.CDLL(path)
            i64, vp, dbl, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
            L.gn3d_forward.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, dbl, ci, ci, vp, vp, vp, vp]
            L.gn3d_forward.restype = ci
            L.gn3d_backward.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ci, vp, vp, vp, vp]
            L.gn3d_backward.restype = ci
            L.gn3d_forward_relu.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, dbl, ci, ci, vp, vp, vp, vp]
            L.gn3d_forward_relu.restype = ci
            L.gn3d_backward_relu.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ci, vp, vp, vp,
                                             vp]
            L.gn3d_backward_relu.restype = ci
            for name in ("gn3d_forward_ndhwc", "gn3d_forward_ndhwc_relu", "gn3d_forward_noalloc"):
                getattr(L, name).argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, dbl, ci, ci, vp, vp, vp, vp]
                getattr(L, name).restype = ci
            L.gn3d_backward_ndhwc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ci, vp, vp, vp, vp]
            L.gn3d_backward_ndhwc.restype = ci
            L.gn3d_backward_ndhwc_relu.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ci, vp, vp,
                                                   vp, vp]
            L.gn3d_backward_ndhwc_relu.restype = ci
            L.gn3d_stream_status.argtypes = [vp]
            L.gn3d_stream_status.restype = ci
            L.gn3d_error_string.argtypes = [ci]
            L.gn3d_error_string.restype = ctypes.c_char_p
            L.gn3d_launch_count.argtypes = []
            L.gn3d_launch_count.restype = ctypes.c_uint64
            L.gn3d_version.argtypes = []
            L.gn3d_version.restype = ctypes.c_char_p
            L.gn3d_forward_moments.argtypes = [vp, i64, i64, i64, i64, i64, i64, ci, vp, vp]
            L.gn3d_moments_combine.argtypes = [vp, i64, i64, vp, vp]
            L.gn3d_forward_apply.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, dbl, ci, ci, vp, vp, vp, vp,
                                             vp]
            L.gn3d_backward_sums.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ci, vp, vp]
            L.gn3d_sums_combine.argtypes = [vp, i64, i64, vp, vp]
            L.gn3d_backward_dx_from_sums.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i64, ci,
                                                     vp, vp, vp, vp]
            for name in ("gn3d_forward_moments", "gn3d_moments_combine", "gn3d_forward_apply", "gn3d_backward_sums",
                         "gn3d_sums_combine", "gn3d_backward_dx_from_sums"):
                getattr(L, name).restype = ci
            L.gn3d_timing.argtypes = [ci]
            L.gn3d_timing.restype = ci
            L.gn3d_kernel_time.argtypes = [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_uint64)]
            L.gn3d_kernel_time.restype = ci
            if kind == "testing":
                L.gn3d_debug_set.argtypes = [ci, ctypes.c_longlong]
                L.gn3d_debug_set.restype = ci
                L.gn3d_debug_get.argtypes = [ci, ctypes.POINTER(ctypes.c_longlong)]
                L.gn3d_debug_get.restype = ci
            _libs[kind] = L
    return _libs[kind]


def _check(status: int):
    if status != OK:
        raise GN3DError(status, lib().gn3d_error_string(status).decode())


# ------------------------------------------------------------ C-ABI mirrors

def gn3d_forward(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd, stream):
    _check(lib().gn3d_forward(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd,
                              stream))


def gn3d_backward(dy, x, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream):
    _check(lib().gn3d_backward(dy, x, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream))


def gn3d_forward_relu(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, out, mean, rstd, stream):
    _check(lib().gn3d_forward_relu(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, out, mean, rstd,
                                   stream))


def gn3d_backward_relu(dy, x, out, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream):
    _check(lib().gn3d_backward_relu(dy, x, out, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta,
                                    stream))


def gn3d_forward_ndhwc(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd, stream):
    _check(lib().gn3d_forward_ndhwc(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd,
                                    stream))


def gn3d_forward_ndhwc_relu(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, out, mean, rstd, stream):
    _check(lib().gn3d_forward_ndhwc_relu(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, out, mean,
                                         rstd, stream))


def gn3d_backward_ndhwc(dy, x, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream):
    _check(lib().gn3d_backward_ndhwc(dy, x, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream))


def gn3d_backward_ndhwc_relu(dy, x, out, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma, dbeta, stream):
    _check(lib().gn3d_backward_ndhwc_relu(dy, x, out, mean, rstd, gamma, N, C, D, H, W, G, dtype, dx, dgamma,
                                          dbeta, stream))


def gn3d_forward_moments(x, N, C, D, H, W, G, in_dtype, moments, stream):
    _check(lib().gn3d_forward_moments(x, N, C, D, H, W, G, in_dtype, moments, stream))


def gn3d_moments_combine(shards, K, NG, combined, stream):
    _check(lib().gn3d_moments_combine(shards, K, NG, combined, stream))


def gn3d_forward_apply(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, moments, y, mean, rstd, stream):
    _check(lib().gn3d_forward_apply(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, moments, y, mean,
                                    rstd, stream))


def gn3d_backward_sums(dy, x, mean, rstd, N, C, D, H, W, G, dtype, sums, stream):
    _check(lib().gn3d_backward_sums(dy, x, mean, rstd, N, C, D, H, W, G, dtype, sums, stream))


def gn3d_sums_combine(shards, K, NC, total, stream):
    _check(lib().gn3d_sums_combine(shards, K, NC, total, stream))


def gn3d_backward_dx_from_sums(dy, x, mean, rstd, gamma, sums, group_count, N, C, D, H, W, G, dtype, dx, dgamma,
                               dbeta, stream):
    _check(lib().gn3d_backward_dx_from_sums(dy, x, mean, rstd, gamma, sums, group_count, N, C, D, H, W, G, dtype,
                                            dx, dgamma, dbeta, stream))


def gn3d_stream_status(stream):
    _check(lib().gn3d_stream_status(stream))


def gn3d_launch_count() -> int:
    return int(lib().gn3d_launch_count())


def gn3d_version() -> str:
    return lib().gn3d_version().decode()


# ------------------------------------------------------------ torch level

def _dtype_code(t):
    import torch

    if t == torch.bfloat16:
        return BF16
    if t == torch.float32:
        return F32
    raise TypeError(f"libgn3d supports bfloat16 and float32, got {t}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _shape5(x):
    if x.dim() != 5:
        raise ValueError("expected an NCDHW tensor")
    if not x.is_contiguous():
        raise ValueError("libgn3d takes contiguous NCDHW tensors")
    return tuple(int(s) for s in x.shape)


def _shape5_cl(x):
    import torch

    if x.dim() != 5:
        raise ValueError("expected an [N, C, D, H, W] tensor")
    if not x.is_contiguous(memory_format=torch.channels_last_3d):
        raise ValueError("the NDHWC entry points take channels_last_3d tensors")
    return tuple(int(s) for s in x.shape)


def is_ndhwc(x) -> bool:
    """x is stored channels-last (channels_last_3d) and not plain NCDHW-contiguous."""
    import torch

    return x.dim() == 5 and not x.is_contiguous() and x.is_contiguous(memory_format=torch.channels_last_3d)


def forward_ndhwc(x, gamma, beta, G: int, eps: float = 1e-5, out_dtype=None, relu: bool = False):
    """forward() for a channels_last_3d x: y (channels_last_3d), mean, rstd."""
    import torch

    N, C, D, H, W = _shape5_cl(x)
    out_dtype = x.dtype if out_dtype is None else out_dtype
    y = torch.empty((N, C, D, H, W), dtype=out_dtype, device=x.device, memory_format=torch.channels_last_3d)
    mean = torch.empty((N, G), dtype=torch.float32, device=x.device)
    rstd = torch.empty((N, G), dtype=torch.float32, device=x.device)
    fn = gn3d_forward_ndhwc_relu if relu else gn3d_forward_ndhwc
    fn(x.data_ptr(), _ptr(gamma), _ptr(beta), N, C, D, H, W, G, float(eps), _dtype_code(x.dtype),
       _dtype_code(out_dtype), y.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
       torch.cuda.current_stream(x.device).cuda_stream)
    return y, mean, rstd


def backward_ndhwc(dy, x, mean, rstd, gamma, G: int, out=None):
    """backward() for channels_last_3d tensors: dx (channels_last_3d), dgamma, dbeta."""
    import torch

    N, C, D, H, W = _shape5_cl(x)
    if dy.shape != x.shape or dy.dtype != x.dtype:
        raise ValueError("dy must match x in shape and dtype")
    if out is not None and (out.shape != x.shape or out.dtype != x.dtype):
        raise ValueError("out must match x in shape and dtype")
    cl = torch.channels_last_3d
    dy = dy.contiguous(memory_format=cl)
    dx = torch.empty((N, C, D, H, W), dtype=x.dtype, device=x.device, memory_format=cl)
    dgamma = torch.empty((C,), dtype=torch.float32, device=x.device)
    dbeta = torch.empty((C,), dtype=torch.float32, device=x.device)
    st = torch.cuda.current_stream(x.device).cuda_stream
    if out is None:
        gn3d_backward_ndhwc(dy.data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), _ptr(gamma), N, C, D, H,
                            W, G, _dtype_code(x.dtype), dx.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(), st)
    else:
        out = out.contiguous(memory_format=cl)
        gn3d_backward_ndhwc_relu(dy.data_ptr(), x.data_ptr(), out.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                                 _ptr(gamma), N, C, D, H, W, G, _dtype_code(x.dtype), dx.data_ptr(),
                                 dgamma.data_ptr(), dbeta.data_ptr(), st)
    return dx, dgamma, dbeta


def forward(x, gamma, beta, G: int, eps: float = 1e-5, out_dtype=None, relu: bool = False):
    """y, mean, rstd = GroupNorm(x) on x's device -- followed by the fused ReLU
    when relu is set; y has out_dtype (default x.dtype)."""
    import torch

    N, C, D, H, W = _shape5(x)
    out_dtype = x.dtype if out_dtype is None else out_dtype
    y = torch.empty((N, C, D, H, W), dtype=out_dtype, device=x.device)
    mean = torch.empty((N, G), dtype=torch.float32, device=x.device)
    rstd = torch.empty((N, G), dtype=torch.float32, device=x.device)
    fn = gn3d_forward_relu if relu else gn3d_forward
    fn(x.data_ptr(), _ptr(gamma), _ptr(beta), N, C, D, H, W, G, float(eps), _dtype_code(x.dtype),
       _dtype_code(out_dtype), y.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
       torch.cuda.current_stream(x.device).cuda_stream)
    return y, mean, rstd


def backward(dy, x, mean, rstd, gamma, G: int, out=None):
    """dx, dgamma, dbeta of GroupNorm at the saved (mean, rstd); with `out` (the
    fused ReLU forward's result, x's dtype) the backward of relu(GroupNorm(x))."""
    import torch

    N, C, D, H, W = _shape5(x)
    if dy.shape != x.shape or dy.dtype != x.dtype:
        raise ValueError("dy must match x in shape and dtype")
    if out is not None and (out.shape != x.shape or out.dtype != x.dtype):
        raise ValueError("out must match x in shape and dtype")
    dy = dy.contiguous()
    dx = torch.empty_like(x)
    dgamma = torch.empty((C,), dtype=torch.float32, device=x.device)
    dbeta = torch.empty((C,), dtype=torch.float32, device=x.device)
    st = torch.cuda.current_stream(x.device).cuda_stream
    if out is None:
        gn3d_backward(dy.data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), _ptr(gamma), N, C, D, H, W, G,
                      _dtype_code(x.dtype), dx.data_ptr(), dgamma.data_ptr(), dbeta.data_ptr(), st)
    else:
        out = out.contiguous()
        gn3d_backward_relu(dy.data_ptr(), x.data_ptr(), out.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                           _ptr(gamma), N, C, D, H, W, G, _dtype_code(x.dtype), dx.data_ptr(), dgamma.data_ptr(),
                           dbeta.data_ptr(), st)
    return dx, dgamma, dbeta


# ------------------------------------------------------------ testing hooks
# Present in the testing build only (use_library("testing")).

(DEBUG_PATH, DEBUG_SPIN_LIMIT, DEBUG_FORCE_TIMEOUT, DEBUG_LAG, DEBUG_SLOTS) = range(5)
(DEBUG_SHARES, DEBUG_RES_HELD, DEBUG_RES_WINDOW, DEBUG_RES_PASS, DEBUG_FAIL_NEXT) = range(6, 11)
PATH_AUTO, PATH_STREAMING, PATH_FUSED, PATH_RESIDENT, PATH_CLUSTER = 0, 1, 2, 3, 4
FAIL_NONE, FAIL_ALLOC, FAIL_LAUNCH = 0, 1, 2
DEBUG_POOL_USED = 0


def _testing():
    if _current != "testing":
        raise RuntimeError("the debug settings exist in the testing build only: call use_library('testing') first")
    return lib()


def gn3d_debug_set(what: int, value: int):
    L = _testing()
    _check(L.gn3d_debug_set(what, value))


def gn3d_debug_get(what: int) -> int:
    L = _testing()
    v = ctypes.c_longlong(0)
    _check(L.gn3d_debug_get(what, ctypes.byref(v)))
    return int(v.value)


KERNELS = ("k_fwd_fused", "k_bwd_fused", "k_fwd_stats", "k_fwd_norm", "k_bwd_reduce", "k_bwd_dx",
           "k_ndhwc_stats", "k_ndhwc_stats_final", "k_ndhwc_norm", "k_ndhwc_reduce", "k_ndhwc_reduce_final",
           "k_ndhwc_dx", "k_fwd_resident", "k_bwd_resident", "k_fwd_cluster", "k_bwd_cluster")


def gn3d_timing(on: bool):
    """Start (clearing earlier records) or stop per-kernel timing (C entry point gn3d_timing)."""
    _check(lib().gn3d_timing(1 if on else 0))


def gn3d_kernel_time(name: str):
    """(total milliseconds, launches) of one kernel since gn3d_timing(True)
    (C entry point gn3d_kernel_time)."""
    ms, n = ctypes.c_double(0.0), ctypes.c_uint64(0)
    _check(lib().gn3d_kernel_time(name.encode(), ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, n.value


def gn3d_forward_noalloc(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd, stream):
    """The allocation-free forward (C entry point gn3d_forward_noalloc)."""
    _check(lib().gn3d_forward_noalloc(x, gamma, beta, N, C, D, H, W, G, eps, in_dtype, out_dtype, y, mean, rstd,
                                      stream))
