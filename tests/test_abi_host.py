"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

The library must build, load on a machine without a GPU driver, export every
entry point the public header declares, and reject bad arguments
synchronously with the documented status codes before touching CUDA.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from conftest import ROOT

import ternary_weight_linear_02_gb300 as tl

TL_OK, TL_ERR_NULL, TL_ERR_SHAPE, TL_ERR_DTYPE, TL_ERR_ALIGN = 0, 1, 2, 3, 4
TL_ERR_CUDA, TL_ERR_UNSUPPORTED = 6, 8
A, B, C, D = 0x10000, 0x20000, 0x30000, 0x40000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    tl.build()
    return tl.load()


def header_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(ternary_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_hot_path(lib):
    names = header_functions()
    for want in ("ternary_pack", "ternary_unpack", "ternary_linear", "ternary_status_string"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", tl.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\b(ternary_\w+)\b", out))
    assert set(header_functions()) <= exported


def test_library_has_no_driver_link(lib):
    out = subprocess.run(["readelf", "-d", tl.library_path()], capture_output=True, text=True,
                         check=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    for s in range(0, 9):
        assert lib.ternary_status_string(s)
    assert b"unknown" in lib.ternary_status_string(99)
    # the accepted group sizes are named
    assert b"(0, 32, 64, 128, 256)" in lib.ternary_status_string(TL_ERR_DTYPE)
    assert lib.ternary_version() >= 100


def lin(lib, x=A, xdt=0, packed=B, scale=C, gs=0, out=D, odt=2, M=4, N=8, K=128, path=0,
        flags=0):
    return lib.ternary_linear_ex(ctypes.c_void_p(x), xdt, ctypes.c_void_p(packed),
                                 ctypes.c_void_p(scale), gs, ctypes.c_void_p(out), odt, M, N,
                                 K, path, flags, None)


def test_linear_argument_errors(lib):
    assert lin(lib, xdt=2) == TL_ERR_DTYPE          # fp32 x not supported
    assert lin(lib, xdt=-1) == TL_ERR_DTYPE
    assert lin(lib, odt=5) == TL_ERR_DTYPE
    assert lin(lib, gs=16) == TL_ERR_DTYPE          # group sizes: 0, 32, 64, 128, 256
    assert lin(lib, gs=48) == TL_ERR_DTYPE
    assert lin(lib, gs=512) == TL_ERR_DTYPE
    assert lin(lib, path=7) == TL_ERR_DTYPE
    assert lin(lib, flags=2) == TL_ERR_DTYPE
    assert lin(lib, M=-1) == TL_ERR_SHAPE
    assert lin(lib, N=-2) == TL_ERR_SHAPE
    assert lin(lib, K=-3) == TL_ERR_SHAPE
    assert lin(lib, gs=128, K=192) == TL_ERR_SHAPE   # K % 128 in group mode
    assert lin(lib, gs=64, K=96) == TL_ERR_SHAPE     # K % 64 in 64-wide group mode
    assert lin(lib, gs=256, K=384) == TL_ERR_SHAPE   # K % 256 in 256-wide group mode
    assert lin(lib, gs=32, K=48) == TL_ERR_SHAPE     # K % 32 in 32-wide group mode
    assert lin(lib, M=1 << 31) == TL_ERR_SHAPE
    assert lin(lib, out=0) == TL_ERR_NULL
    assert lin(lib, x=0) == TL_ERR_NULL
    assert lin(lib, packed=0) == TL_ERR_NULL
    assert lin(lib, scale=0) == TL_ERR_NULL
    assert lin(lib, x=A + 8) == TL_ERR_ALIGN
    assert lin(lib, out=D + 2) == TL_ERR_ALIGN
    assert lin(lib, scale=C + 4) == TL_ERR_ALIGN
    assert lin(lib, packed=B + 1) == TL_ERR_ALIGN


def test_linear_empty_is_noop(lib):
    # M == 0 or N == 0: nothing to do, even with NULL buffers
    assert lin(lib, M=0, x=0, out=0) == TL_OK
    assert lin(lib, N=0, packed=0, scale=0, out=0) == TL_OK


def silu(lib, x=A, xdt=1, packed=B, scale=C, gs=0, out=D, odt=2, M=4, N=8, K=128, flags=0):
    lib.ternary_linear_silu_mul.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                            ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p]
    return lib.ternary_linear_silu_mul(ctypes.c_void_p(x), xdt, ctypes.c_void_p(packed),
                                       ctypes.c_void_p(scale), gs, ctypes.c_void_p(out), odt,
                                       M, N, K, flags, None)


def test_silu_mul_argument_errors(lib):
    # checked on the host before any device work
    assert silu(lib, gs=16) == TL_ERR_DTYPE
    assert silu(lib, gs=32, K=48) == TL_ERR_SHAPE
    assert silu(lib, flags=4) == TL_ERR_DTYPE
    assert silu(lib, N=-1) == TL_ERR_SHAPE
    assert silu(lib, gs=64, K=130) == TL_ERR_SHAPE   # K % 64 in 64-wide group mode
    assert silu(lib, gs=256, K=384) == TL_ERR_SHAPE
    assert silu(lib, out=0) == TL_ERR_NULL
    assert silu(lib, packed=B + 1) == TL_ERR_ALIGN
    assert silu(lib, M=0, x=0, out=0) == TL_OK         # empty: no-op
    assert silu(lib, N=0, packed=0, scale=0, out=0) == TL_OK


def test_packing_argument_errors(lib):
    p = ctypes.c_void_p
    assert lib.ternary_pack(p(A), p(B), 4, -6, None, None) == TL_ERR_SHAPE
    assert lib.ternary_pack(p(A), p(B), -1, 8, None, None) == TL_ERR_SHAPE
    assert lib.ternary_unpack(p(B), p(A), 4, -10, None, None) == TL_ERR_SHAPE
    # K % 4 != 0 is a padded row, not an error: the checks pass up to the device query
    assert lib.ternary_pack(p(A), p(B), 4, 6, None, None) != TL_ERR_SHAPE
    assert lib.ternary_unpack(p(B), p(A), 4, 10, None, None) != TL_ERR_SHAPE
    assert lib.ternary_pack(None, p(B), 4, 8, None, None) == TL_ERR_NULL
    assert lib.ternary_unpack(p(B), None, 4, 8, None, None) == TL_ERR_NULL
    assert lib.ternary_pack(p(A + 1), p(B), 4, 8, None, None) == TL_ERR_ALIGN
    assert lib.ternary_unpack(p(B), p(A), 4, 8, p(C + 4), None) == TL_ERR_ALIGN
    # N * K beyond 2^48 elements: rejected before any product can overflow
    assert lib.ternary_pack(p(A), p(B), (1 << 39), (1 << 20), None, None) == TL_ERR_SHAPE
    assert lib.ternary_unpack(p(B), p(A), (1 << 30), (1 << 30), None, None) == TL_ERR_SHAPE


def test_injected_launch_failure_reported_before_cuda(lib):
    lib.ternary_test_inject_launch_failures(2)
    assert lin(lib) == TL_ERR_CUDA
    assert lib.ternary_unpack(ctypes.c_void_p(B), ctypes.c_void_p(A), 4, 8, None,
                              None) == TL_ERR_CUDA
    lib.ternary_test_inject_launch_failures(0)


def test_binding_raises_with_status(lib):
    lib.ternary_test_inject_launch_failures(1)
    try:
        with pytest.raises(tl.TernaryError) as ei:
            tl._check(lin(lib), "ternary_linear")
        assert ei.value.status == TL_ERR_CUDA
        assert "TL_ERR_CUDA" in str(ei.value)
    finally:
        lib.ternary_test_inject_launch_failures(0)


def test_binding_refuses_cpu_tensors(lib):
    x = torch.zeros(2, 128, dtype=torch.float16)
    p = torch.zeros(4, 32, dtype=torch.uint8)
    s = torch.ones(4, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        tl.linear(x, p, s)
    with pytest.raises(ValueError, match="CUDA"):
        tl.unpack(p)


def test_fused_shard_sizes_checked(lib):
    x = torch.zeros(2, 128, dtype=torch.float16)
    p = torch.zeros(4, 32, dtype=torch.uint8)
    s = torch.ones(4, dtype=torch.float16)
    with pytest.raises(ValueError, match="shard"):
        tl.linear_fused(x, p, s, [3, 2])


def test_block_mask_host_checks(lib):
    p = ctypes.c_void_p
    assert lib.ternary_block_mask_words(300, 4160) == 3 * 3
    assert lib.ternary_block_mask_words(0, 64) == 0
    assert lib.ternary_block_mask_words(4, 6) == 1     # K % 4 != 0: padded rows
    assert lib.ternary_block_mask_words(4, -6) == -1
    assert lib.ternary_block_mask(p(B), 4, -6, p(A), None, None) == TL_ERR_SHAPE
    assert lib.ternary_block_mask(None, 4, 8, p(A), None, None) == TL_ERR_NULL
    assert lib.ternary_block_mask(p(B), 4, 8, p(A + 2), None, None) == TL_ERR_ALIGN
    assert lib.ternary_block_mask(p(B), 4, 8, p(A), p(C + 4), None) == TL_ERR_ALIGN


def test_masked_linear_host_checks(lib):
    v = ctypes.c_void_p
    # NULL map with work to do; misaligned map; argument errors as the plain call
    assert lib.ternary_linear_masked(v(A), 0, v(B), v(C), 0, None, v(D), 2, 4, 8, 128, 0,
                                     None) == TL_ERR_NULL
    assert lib.ternary_linear_masked(v(A), 0, v(B), v(C), 0, v(A + 2), v(D), 2, 4, 8, 128, 0,
                                     None) == TL_ERR_ALIGN
    assert lib.ternary_linear_masked(v(A), 0, v(B), v(C), 128, v(A), v(D), 2, 4, 8, 130, 0,
                                     None) == TL_ERR_SHAPE
    assert lib.ternary_linear_silu_mul_masked(v(A), 0, v(B), v(C), 16, v(A), v(D), 2, 4, 8, 128,
                                              0, None) == TL_ERR_DTYPE
