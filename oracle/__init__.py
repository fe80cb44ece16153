"""CPU oracle for the ternary-weight linear layer -- TEST INFRASTRUCTURE ONLY.

This package is the independent reference the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import it; the product package never does.  It shares no
code with the CUDA path: the arithmetic lives in ``ternary_oracle.c`` (plain C,
fp64), and this module only converts fp16 / bf16 bit patterns to fp64 exactly
and marshals numpy arrays.

Sources: "三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战"
(trdm.cn/news/729035) §1.1, §3.1, §4.2, and the Qwen2.5-7B ternary-in-vLLM
write-up (m.nxbn.cn/news/169761) §2.2, §2.3, §3.2, §4.2.  Each C function names the
passage it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ternary_oracle.c")
_LIB = os.path.join(_HERE, "libternary_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: builds on x86-64 and aarch64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_trit.argtypes = [ctypes.c_uint]
        lib.oracle_trit.restype = ctypes.c_int
        lib.oracle_unpack.argtypes = [p, p, i64, i64, p]
        lib.oracle_unpack.restype = None
        lib.oracle_pack.argtypes = [p, p, i64, i64]
        lib.oracle_pack.restype = i64
        lib.oracle_linear_f64.argtypes = [p, p, p, i64, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_linear_f64.restype = ctypes.c_int
        lib.oracle_silu_mul_f64.argtypes = [p, p, p, i64, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_silu_mul_f64.restype = ctypes.c_int
        lib.oracle_block_mask.argtypes = [p, i64, i64, p]
        lib.oracle_block_mask.restype = i64
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- conversions
def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns (uint16) -> exact float64."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 (bf16 is the top half of binary32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f16_bits_to_f64(bits)
    if dtype == "bf16":
        return bf16_bits_to_f64(bits)
    raise ValueError(f"unknown 16-bit dtype {dtype!r}")


# ------------------------------------------------------------------ the oracle
def trit(code: int) -> int:
    """Value of one 2-bit code (00->0, 01->+1, 10->-1, 11->0)."""
    return int(_load().oracle_trit(int(code)))


def _row_bytes(K: int) -> int:
    return (K + 3) // 4


def unpack(packed: np.ndarray, K: int | None = None) -> tuple[np.ndarray, int]:
    """packed [N, ceil(K/4)] uint8 -> (t [N, K] int8, number of reserved 11 fields
    among the K weights of each row).  K defaults to 4 * bytes per row; a smaller
    K leaves the last byte's high fields as padding."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N, Kq = packed.shape
    K = 4 * Kq if K is None else int(K)
    if _row_bytes(K) != Kq:
        raise ValueError(f"packed rows of {Kq} bytes do not hold K = {K}")
    t = np.empty((N, K), dtype=np.int8)
    cnt = ctypes.c_int64(0)
    _load().oracle_unpack(_ptr(packed), _ptr(t), N, K, ctypes.byref(cnt))
    return t, int(cnt.value)


def pack(t: np.ndarray) -> tuple[np.ndarray, int]:
    """t [N, K] int8 -> (packed [N, ceil(K/4)] uint8, number of entries outside
    {-1,0,1}); padding fields are 00."""
    t = np.ascontiguousarray(t, dtype=np.int8)
    N, K = t.shape
    packed = np.empty((N, _row_bytes(K)), dtype=np.uint8)
    invalid = _load().oracle_pack(_ptr(t), _ptr(packed), N, K)
    return packed, int(invalid)


def linear_f64(x: np.ndarray, packed: np.ndarray, scale: np.ndarray, group_size: int,
               nthreads: int = 1) -> np.ndarray:
    """y[M,N] = per-channel or per-group scaled ternary product, all in fp64.

    x: [M,K] float64; packed: [N, ceil(K/4)] uint8; scale: [N] (group_size 0)
    or [N, K/group_size] float64.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float64)
    M, K = x.shape
    N = packed.shape[0]
    if packed.shape[1] != _row_bytes(K):
        raise ValueError("packed must be [N, ceil(K/4)]")
    want = (N,) if group_size == 0 else (N, K // group_size)
    if scale.shape != want:
        raise ValueError(f"scale shape {scale.shape} != {want}")
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_linear_f64(_ptr(x), _ptr(packed), _ptr(scale), int(group_size),
                                   _ptr(y), M, N, K, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_linear_f64 rejected its arguments")
    return y


def linear_from_bits(x_bits: np.ndarray, x_dtype: str, packed: np.ndarray,
                     scale_bits: np.ndarray, group_size: int, nthreads: int = 1) -> np.ndarray:
    """Same as linear_f64, taking x and the fp16 scale as raw 16-bit patterns."""
    return linear_f64(bits_to_f64(x_bits, x_dtype), packed, f16_bits_to_f64(scale_bits),
                      group_size, nthreads)


def silu_mul_f64(x: np.ndarray, packed: np.ndarray, scale: np.ndarray, group_size: int,
                 nthreads: int = 1) -> np.ndarray:
    """h[M,N] = silu(g) * u for a stacked gate/up layer (packed [2N, K/4], scale
    [2N] or [2N, K/G]; gate rows first), in fp64."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float64)
    M, K = x.shape
    N2 = packed.shape[0]
    if N2 % 2 or packed.shape[1] != _row_bytes(K):
        raise ValueError("packed must be [2N, ceil(K/4)]")
    want = (N2,) if group_size == 0 else (N2, K // group_size)
    if scale.shape != want:
        raise ValueError(f"scale shape {scale.shape} != {want}")
    h = np.empty((M, N2 // 2), dtype=np.float64)
    rc = _load().oracle_silu_mul_f64(_ptr(x), _ptr(packed), _ptr(scale), int(group_size),
                                     _ptr(h), M, N2 // 2, K, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_silu_mul_f64 rejected its arguments")
    return h


def silu_mul_from_bits(x_bits: np.ndarray, x_dtype: str, packed: np.ndarray,
                       scale_bits: np.ndarray, group_size: int, nthreads: int = 1) -> np.ndarray:
    """Same as silu_mul_f64, taking x and the fp16 scale as raw 16-bit patterns."""
    return silu_mul_f64(bits_to_f64(x_bits, x_dtype), packed, f16_bits_to_f64(scale_bits),
                        group_size, nthreads)


def block_mask(packed: np.ndarray, K: int | None = None) -> tuple[np.ndarray, int]:
    """Zero-block map of packed [N, ceil(K/4)]: uint32 [ceil(N/128), ceil(K/64/32)],
    bit kb of row block rb set when rows [128 rb, +128) x k [64 kb, +64) hold a
    non-zero weight; and the number of zero blocks.  K defaults to 4 * bytes per row."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N, Kq = packed.shape
    K = 4 * Kq if K is None else int(K)
    if _row_bytes(K) != Kq:
        raise ValueError(f"packed rows of {Kq} bytes do not hold K = {K}")
    RB, KB = (N + 127) // 128, (K + 63) // 64
    mask = np.empty((RB, (KB + 31) // 32), dtype=np.uint32)
    zero = _load().oracle_block_mask(_ptr(packed), N, K, _ptr(mask))
    return mask, int(zero)
