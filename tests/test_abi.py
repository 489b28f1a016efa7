"""The C ABI: the library builds, loads and exports what include/gn3d.h declares;
argument checks return the documented status codes."""
import os
import re
import subprocess

import numpy as np
import pytest

import bwd_gn3d_stats_gb300 as gn
from bwd_gn3d_stats_gb300 import build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gn3d.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return gn.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gn3d_\w+)\s*\(", src)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("gn3d_forward", "gn3d_backward", "gn3d_stream_status", "gn3d_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    # the testing build exports everything the header declares (the hooks are
    # declared under GN3D_TESTING); the shipped one everything but the hooks
    testing = gn._load("testing")
    exported = set(re.findall(r"\bT (gn3d_\w+)", subprocess.run(
        ["nm", "-D", "--defined-only", build.TESTING_LIB], capture_output=True, text=True, check=True).stdout))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(testing, n)
        if n not in ("gn3d_debug_set", "gn3d_debug_get"):
            assert hasattr(L, n)


@pytest.mark.parametrize("testing", [False, True])
def test_header_compiles_as_c(tmp_path, testing):
    src = tmp_path / "t.c"
    src.write_text('#include "gn3d.h"\nint (*f)(void*) = gn3d_stream_status;\n'
                   'int main(void){ return f == 0; }\n')
    flags = ["-DGN3D_TESTING"] if testing else []
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror"] + flags + ["-I", os.path.join(ROOT, "include"), "-c",
                    str(src), "-o", str(tmp_path / "t.o")], check=True)


def test_version(L):
    assert gn.gn3d_version().startswith("gn3d ")


# Argument checks that fail before any CUDA call (no GPU needed).
BAD_SHAPES = [
    dict(N=1, C=8, D=4, H=4, W=4, G=3),      # C % G != 0
    dict(N=1, C=8, D=4, H=4, W=4, G=0),      # G < 1
    dict(N=-1, C=8, D=4, H=4, W=4, G=2),     # negative dimension
    dict(N=1, C=4, D=1, H=1, W=1, G=4),      # one value per group: stock GroupNorm raises
]


@pytest.mark.parametrize("shape", BAD_SHAPES)
def test_invalid_shapes_rejected(L, shape):
    s = shape
    rc = L.gn3d_forward(None, None, None, s["N"], s["C"], s["D"], s["H"], s["W"], s["G"], 1e-5, gn.BF16, gn.BF16,
                        None, None, None, None)
    assert rc == gn.ERR_INVALID_ARG
    assert L.gn3d_error_string(rc).decode().startswith("invalid argument")
    rc = L.gn3d_backward(None, None, None, None, None, s["N"], s["C"], s["D"], s["H"], s["W"], s["G"], gn.BF16,
                         None, None, None, None)
    assert rc == gn.ERR_INVALID_ARG


@pytest.mark.parametrize("shape", BAD_SHAPES)
def test_invalid_shapes_rejected_ndhwc(L, shape):
    s = shape
    rc = L.gn3d_forward_ndhwc(None, None, None, s["N"], s["C"], s["D"], s["H"], s["W"], s["G"], 1e-5, gn.BF16,
                              gn.BF16, None, None, None, None)
    assert rc == gn.ERR_INVALID_ARG
    rc = L.gn3d_backward_ndhwc(None, None, None, None, None, s["N"], s["C"], s["D"], s["H"], s["W"], s["G"], gn.BF16,
                               None, None, None, None)
    assert rc == gn.ERR_INVALID_ARG


def test_ndhwc_needs_channels_multiple_of_8(L):
    rc = L.gn3d_forward_ndhwc(None, None, None, 1, 12, 2, 2, 2, 4, 1e-5, gn.BF16, gn.BF16, None, None, None, None)
    assert rc == gn.ERR_INVALID_ARG
    assert "C % 8" in L.gn3d_error_string(rc).decode()
    rc = L.gn3d_forward_ndhwc_relu(None, None, None, 1, 12, 2, 2, 2, 4, 1e-5, gn.BF16, gn.BF16, None, None, None,
                                   None)
    assert rc == gn.ERR_INVALID_ARG
    rc = L.gn3d_backward_ndhwc(None, None, None, None, None, 1, 20, 2, 2, 2, 5, gn.F32, None, None, None, None)
    assert rc == gn.ERR_INVALID_ARG
    rc = L.gn3d_backward_ndhwc_relu(None, None, None, None, None, None, 1, 20, 2, 2, 2, 5, gn.F32, None, None, None,
                                    None)
    assert rc == gn.ERR_INVALID_ARG


def test_invalid_dtype_and_eps_rejected(L):
    assert L.gn3d_forward(None, None, None, 1, 4, 2, 2, 2, 2, 1e-5, 7, gn.BF16, None, None, None, None) == 1
    assert L.gn3d_forward(None, None, None, 1, 4, 2, 2, 2, 2, -1.0, gn.BF16, gn.BF16, None, None, None, None) == 1
    assert L.gn3d_forward(None, None, None, 1, 4, 2, 2, 2, 2, float("nan"), gn.BF16, gn.BF16, None, None, None,
                          None) == 1
    assert L.gn3d_backward(None, None, None, None, None, 1, 4, 2, 2, 2, 2, 9, None, None, None, None) == 1


def test_python_raises_gn3derror(L):
    with pytest.raises(gn.GN3DError) as e:
        gn.gn3d_forward(None, None, None, 1, 6, 1, 1, 1, 4, 1e-5, gn.BF16, gn.BF16, None, None, None, None)
    assert e.value.status == gn.ERR_INVALID_ARG


# ----------------------------------------------------------- on the GPU

@pytest.mark.gpu
def test_gpu_pointer_checks(L):
    import torch

    x = torch.zeros(64 * 4, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    st = torch.cuda.current_stream().cuda_stream
    # misaligned x (2-byte offset)
    rc = L.gn3d_forward(x.data_ptr() + 2, None, None, 1, 4, 1, 1, 63, 2, 1e-5, gn.BF16, gn.BF16, y.data_ptr(),
                        None, None, st)
    assert rc == gn.ERR_INVALID_ARG
    # host memory for y
    h = np.zeros(64 * 4, dtype=np.uint16)
    rc = L.gn3d_forward(x.data_ptr(), None, None, 1, 4, 1, 1, 64, 2, 1e-5, gn.BF16, gn.BF16, h.ctypes.data, None,
                        None, st)
    assert rc == gn.ERR_DEVICE
    # pinned host memory is not device memory either
    hp = torch.zeros(64 * 4, dtype=torch.bfloat16).pin_memory()
    rc = L.gn3d_forward(x.data_ptr(), None, None, 1, 4, 1, 1, 64, 2, 1e-5, gn.BF16, gn.BF16, hp.data_ptr(), None,
                        None, st)
    assert rc == gn.ERR_DEVICE
    assert L.gn3d_stream_status(st) == gn.OK


@pytest.mark.gpu
def test_gpu_empty_tensors(L):
    import torch

    st = torch.cuda.current_stream().cuda_stream
    mean = torch.full((2 * 4,), 7.0, device="cuda")
    rstd = torch.full((2 * 4,), 7.0, device="cuda")
    x = torch.empty(0, device="cuda")
    rc = L.gn3d_forward(x.data_ptr(), None, None, 2, 8, 0, 5, 5, 4, 1e-5, gn.F32, gn.F32, x.data_ptr(),
                        mean.data_ptr(), rstd.data_ptr(), st)
    assert rc == gn.OK
    assert torch.all(mean == 0) and torch.allclose(rstd, torch.full_like(rstd, 1e-5 ** -0.5))
    dg = torch.full((8,), 3.0, device="cuda")
    db = torch.full((8,), 3.0, device="cuda")
    rc = L.gn3d_backward(x.data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), None, 2, 8, 0, 5, 5, 4,
                         gn.F32, x.data_ptr(), dg.data_ptr(), db.data_ptr(), st)
    assert rc == gn.OK
    assert torch.all(dg == 0) and torch.all(db == 0)
    # N = 0: nothing to do at all
    rc = L.gn3d_forward(None, None, None, 0, 8, 4, 4, 4, 4, 1e-5, gn.BF16, gn.BF16, None, None, None, st)
    assert rc == gn.OK
    assert L.gn3d_stream_status(st) == gn.OK


@pytest.mark.gpu
def test_gpu_torch_level_wrappers():
    import torch

    site = synth.Site(1, 8, 6, 6, 6, 4, synth.BF16)
    inp = synth.make_inputs(site, seed=0)
    x = torch.from_numpy(inp["x"].view(np.int16)).cuda().view(torch.bfloat16).reshape(1, 8, 6, 6, 6)
    g = torch.from_numpy(inp["gamma"]).cuda()
    b = torch.from_numpy(inp["beta"]).cuda()
    y, mean, rstd = gn.forward(x, g, b, 4)
    assert y.dtype == torch.bfloat16 and mean.shape == (1, 4)
    y32, _, _ = gn.forward(x, g, b, 4, out_dtype=torch.float32)
    assert y32.dtype == torch.float32
    assert torch.equal(y32.to(torch.bfloat16), y)
    dx, dg, db = gn.backward(torch.ones_like(x), x, mean, rstd, g, 4)
    assert dx.dtype == torch.bfloat16 and dg.shape == (8,)


def test_kernel_timing_without_launches(L):
    # starting a timing window clears it; nothing launched -> zero time, zero launches
    gn.gn3d_timing(True)
    try:
        for name in gn.KERNELS:
            assert gn.gn3d_kernel_time(name) == (0.0, 0)
        with pytest.raises(gn.GN3DError):
            gn.gn3d_kernel_time("k_not_a_kernel")
        assert L.gn3d_timing(2) == gn.ERR_INVALID_ARG
    finally:
        gn.gn3d_timing(False)


def _exports(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    return set(re.findall(r"\bT (gn3d_\w+)", out))


def test_shipped_library_carries_no_test_hooks(L):
    """The testing and tuning hooks exist in the testing build only; the shipped
    library exports the GroupNorm entry points and diagnostics."""
    product, testing = _exports(build.LIB), _exports(build.TESTING_LIB)
    assert "gn3d_debug_set" not in product and "gn3d_debug_get" not in product
    assert {"gn3d_debug_set", "gn3d_debug_get"} <= testing
    assert product == testing - {"gn3d_debug_set", "gn3d_debug_get"}
    with pytest.raises(RuntimeError):
        gn.gn3d_debug_set(gn.DEBUG_PATH, 0)  # the product build is the current one


def test_debug_settings_ranges(testing_build):
    # every hook accepts its documented range and rejects the rest; none needs a GPU
    ok = {gn.DEBUG_PATH: (0, 1, 2, 3, 4), gn.DEBUG_LAG: (-1, 0, 8), gn.DEBUG_SLOTS: (-1, 1, 32),
          gn.DEBUG_SHARES: (-1, 0, 1), gn.DEBUG_SPIN_LIMIT: (0, 1 << 20), gn.DEBUG_RES_HELD: (-1, 0, 7),
          gn.DEBUG_RES_WINDOW: (-1, 1, 500), gn.DEBUG_RES_PASS: (-1, 1, 12), gn.DEBUG_FAIL_NEXT: (0, 1, 2)}
    bad = {gn.DEBUG_PATH: (-1, 5), gn.DEBUG_LAG: (-2, 9), gn.DEBUG_SLOTS: (0, -2, 33),
           gn.DEBUG_SHARES: (-2, 2), gn.DEBUG_SPIN_LIMIT: (-1,), gn.DEBUG_RES_HELD: (-2,),
           gn.DEBUG_RES_WINDOW: (-2, 0), gn.DEBUG_RES_PASS: (-2, 0), gn.DEBUG_FAIL_NEXT: (-1, 3)}
    for what, values in ok.items():
        for v in values:
            gn.gn3d_debug_set(what, v)
    for what, values in bad.items():
        for v in values:
            with pytest.raises(gn.GN3DError):
                gn.gn3d_debug_set(what, v)
    with pytest.raises(gn.GN3DError):
        gn.gn3d_debug_set(99, 0)
    with pytest.raises(gn.GN3DError):
        gn.gn3d_debug_get(7)


@pytest.mark.gpu
def test_gpu_ndhwc_empty_tensors_and_pointer_checks(L):
    """The channels-last entry points share the argument checks and the empty-
    tensor results: zero-size volumes give mean 0, rstd 1/sqrt(eps) and zero
    parameter gradients; misaligned or host pointers are rejected."""
    import torch

    st = torch.cuda.current_stream().cuda_stream
    mean = torch.full((2 * 4,), 7.0, device="cuda")
    rstd = torch.full((2 * 4,), 7.0, device="cuda")
    x = torch.empty(0, device="cuda")
    rc = L.gn3d_forward_ndhwc(x.data_ptr(), None, None, 2, 8, 0, 5, 5, 4, 1e-5, gn.F32, gn.F32, x.data_ptr(),
                              mean.data_ptr(), rstd.data_ptr(), st)
    assert rc == gn.OK
    assert torch.all(mean == 0) and torch.allclose(rstd, torch.full_like(rstd, 1e-5 ** -0.5))
    dg = torch.full((8,), 3.0, device="cuda")
    db = torch.full((8,), 3.0, device="cuda")
    rc = L.gn3d_backward_ndhwc(x.data_ptr(), x.data_ptr(), mean.data_ptr(), rstd.data_ptr(), None, 2, 8, 0, 5, 5, 4,
                               gn.F32, x.data_ptr(), dg.data_ptr(), db.data_ptr(), st)
    assert rc == gn.OK
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)
    xb = torch.zeros(64 * 8, dtype=torch.bfloat16, device="cuda")
    yb = torch.empty_like(xb)
    rc = L.gn3d_forward_ndhwc(xb.data_ptr() + 2, None, None, 1, 8, 1, 1, 63, 2, 1e-5, gn.BF16, gn.BF16,
                              yb.data_ptr(), None, None, st)
    assert rc == gn.ERR_INVALID_ARG
    h = np.zeros(64 * 8, dtype=np.uint16)
    rc = L.gn3d_forward_ndhwc(xb.data_ptr(), None, None, 1, 8, 1, 1, 64, 2, 1e-5, gn.BF16, gn.BF16, h.ctypes.data,
                              None, None, st)
    assert rc == gn.ERR_DEVICE
    assert L.gn3d_stream_status(st) == gn.OK
