"""Ternary-weight linear layer for GB300 (sm_103a): thin Python binding.

Every step of the computation runs in the CUDA kernels of
``libternary_gb300.so`` (C ABI in ``include/ternary_linear.h``).  This module
only marshals torch tensors (device memory, shapes, the current CUDA stream)
into that ABI; there is no Python or CPU fallback, and a missing library is an
error.

Format: W[N,K] in {-1,0,+1} packed as uint8 [N, K/4], code table 00->0, 01->+1,
10->-1, 11->0 (reserved), first weight in the low bits
("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战", trdm.cn/news/729035, §3.1).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "TernaryError", "build", "library_path", "load", "pack", "unpack", "block_mask", "linear",
    "row_bytes",
    "linear_fused",
    "linear_silu_mul",
    "device_status", "device_status_async", "status_string", "skinny_max_m", "PATHS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libternary_gb300.so")
_lib = None

TL_F16, TL_BF16, TL_F32 = 0, 1, 2
PATHS = {"auto": 0, "skinny": 1, "tile": 2, "generic": 3}
FLAG_STATIC_WEIGHTS = 1
_DT = {torch.float16: TL_F16, torch.bfloat16: TL_BF16, torch.float32: TL_F32}


class TernaryError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {status_string(status)}")


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force, verbose=verbose)


def load():
    """Load libternary_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with ternary_weight_linear_02_gb300.build() "
            "(needs nvcc); there is no fallback implementation")
    lib = ctypes.CDLL(_LIB_PATH)
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.ternary_pack.argtypes = [p, p, i64, i64, p, p]
    lib.ternary_unpack.argtypes = [p, p, i64, i64, p, p]
    lib.ternary_linear.argtypes = [p, i32, p, p, i32, p, i32, i64, i64, i64, p]
    lib.ternary_linear_ex.argtypes = [p, i32, p, p, i32, p, i32, i64, i64, i64, i32,
                                      ctypes.c_uint32, p]
    lib.ternary_linear_silu_mul.argtypes = [p, i32, p, p, i32, p, i32, i64, i64, i64,
                                            ctypes.c_uint32, p]
    for f in (lib.ternary_pack, lib.ternary_unpack, lib.ternary_linear, lib.ternary_linear_ex,
              lib.ternary_linear_silu_mul):
        f.restype = ctypes.c_int
    lib.ternary_device_status.argtypes = [ctypes.POINTER(ctypes.c_int32), i32]
    lib.ternary_device_status.restype = ctypes.c_int
    lib.ternary_status_string.argtypes = [i32]
    lib.ternary_status_string.restype = ctypes.c_char_p
    lib.ternary_skinny_max_m.restype = i32
    lib.ternary_version.restype = i32
    lib.ternary_test_inject_launch_failures.argtypes = [i32]
    lib.ternary_test_inject_launch_failures.restype = None
    lib.ternary_test_set_wait_limit.argtypes = [i64, i32]
    lib.ternary_test_set_wait_limit.restype = None
    lib.ternary_test_set_tile_mode.argtypes = [i32]
    lib.ternary_test_set_tile_mode.restype = None
    lib.ternary_device_status_async.argtypes = [p, i32, p]
    lib.ternary_device_status_async.restype = ctypes.c_int
    lib.ternary_block_mask_words.argtypes = [i64, i64]
    lib.ternary_block_mask_words.restype = i64
    lib.ternary_block_mask.argtypes = [p, i64, i64, p, p, p]
    lib.ternary_block_mask.restype = ctypes.c_int
    lib.ternary_linear_masked.argtypes = [p, i32, p, p, i32, p, p, i32, i64, i64, i64,
                                          ctypes.c_uint32, p]
    lib.ternary_linear_masked.restype = ctypes.c_int
    lib.ternary_linear_silu_mul_masked.argtypes = [p, i32, p, p, i32, p, p, i32, i64, i64, i64,
                                                   ctypes.c_uint32, p]
    lib.ternary_linear_silu_mul_masked.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().ternary_status_string(int(status)).decode()
    except Exception:  # library missing: still produce a message
        return f"status {status}"


def skinny_max_m() -> int:
    return int(load().ternary_skinny_max_m())


def _ptr(t: torch.Tensor | None):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(rc: int, what: str):
    if rc != 0:
        raise TernaryError(rc, what)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device (no CPU path)")


def row_bytes(K: int) -> int:
    """Bytes per packed row of K weights: ceil(K/4) (a K % 4 != 0 row ends in
    padding fields)."""
    return (int(K) + 3) // 4


def pack(t: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """t [N,K] int8 in {-1,0,1} -> (packed [N, ceil(K/4)] uint8, invalid-entry count
    (device int64)); padding fields of a K % 4 != 0 row are written 00."""
    _need_cuda(t)
    if t.dtype != torch.int8 or t.dim() != 2:
        raise ValueError("t must be a 2-D int8 tensor")
    t = t.contiguous()
    N, K = t.shape
    packed = torch.empty((N, row_bytes(K)), dtype=torch.uint8, device=t.device)
    cnt = torch.empty((), dtype=torch.int64, device=t.device)
    _check(load().ternary_pack(_ptr(t), _ptr(packed), N, K, _ptr(cnt), _stream(t.device)),
           "ternary_pack")
    return packed, cnt


def _row_width(packed: torch.Tensor, K: int | None) -> int:
    Kq = packed.shape[1]
    K = 4 * Kq if K is None else int(K)
    if row_bytes(K) != Kq:
        raise ValueError(f"packed rows of {Kq} bytes do not hold K = {K}")
    return K


def unpack(packed: torch.Tensor, K: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """packed [N, ceil(K/4)] uint8 -> (t [N,K] int8, reserved-code count (device
    int64)).  K defaults to 4 * bytes per row; a smaller K drops the padding fields."""
    _need_cuda(packed)
    if packed.dtype != torch.uint8 or packed.dim() != 2:
        raise ValueError("packed must be a 2-D uint8 tensor")
    packed = packed.contiguous()
    N = packed.shape[0]
    K = _row_width(packed, K)
    t = torch.empty((N, K), dtype=torch.int8, device=packed.device)
    cnt = torch.empty((), dtype=torch.int64, device=packed.device)
    _check(load().ternary_unpack(_ptr(packed), _ptr(t), N, K, _ptr(cnt),
                                 _stream(packed.device)), "ternary_unpack")
    return t, cnt


def block_mask(packed: torch.Tensor, K: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """Zero-block map of packed [N, ceil(K/4)]: (mask uint32 [ceil(N/128), W], number
    of zero blocks (device int64)); bit kb of row block rb is set when rows
    [128 rb, +128) x k [64 kb, +64) hold a non-zero weight.  K defaults to
    4 * bytes per row."""
    _need_cuda(packed)
    if packed.dtype != torch.uint8 or packed.dim() != 2:
        raise ValueError("packed must be a 2-D uint8 tensor")
    packed = packed.contiguous()
    N = packed.shape[0]
    K = _row_width(packed, K)
    lib = load()
    words = int(lib.ternary_block_mask_words(N, K))
    rb = (N + 127) // 128
    mask = torch.empty((rb, words // max(rb, 1) if rb else 0), dtype=torch.int32,
                       device=packed.device)
    cnt = torch.empty((), dtype=torch.int64, device=packed.device)
    _check(lib.ternary_block_mask(_ptr(packed), N, K, _ptr(mask), _ptr(cnt),
                                  _stream(packed.device)), "ternary_block_mask")
    return mask, cnt


def linear(x: torch.Tensor, packed: torch.Tensor, scale: torch.Tensor,
           group_size: int | None = None, out_dtype: torch.dtype | None = None,
           out: torch.Tensor | None = None, path: str = "auto",
           static_weights: bool = False, mask: torch.Tensor | None = None) -> torch.Tensor:
    """out[..., N] = x[..., K] @ (t * scale)^T with t decoded from ``packed``.

    ``scale`` is fp16 [N] (per channel) or [N, K/G] (per G-wide K group, G in
    32, 64, 128, 256); ``group_size`` defaults from its shape.  ``path`` is
    "auto", "skinny", "tile" or "generic" (the CUDA-core kernel that "auto"
    takes when K % 64 != 0).  Leading dimensions of ``x`` are
    flattened into M (the kernel takes a dense 2-D [M, K]).
    ``static_weights=True`` promises that ``packed`` / ``scale`` are not being
    written by work still running on the stream (TL_FLAG_STATIC_WEIGHTS), which
    lets consecutive layers overlap.  ``mask`` (from ``block_mask(packed)``)
    makes the kernel skip all-zero weight blocks (automatic path only).
    """
    _need_cuda(x, packed, scale, out)
    if x.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("x must be fp16 or bf16")
    if scale.dtype != torch.float16:
        raise ValueError("scale must be fp16")
    if packed.dtype != torch.uint8 or packed.dim() != 2:
        raise ValueError("packed must be a 2-D uint8 tensor [N, K/4]")
    K = x.shape[-1]
    lead = x.shape[:-1]
    M = 1
    for d in lead:
        M *= int(d)
    x2 = x.reshape(M, K).contiguous()
    N = packed.shape[0]
    if packed.shape[1] != row_bytes(K):
        raise ValueError(f"packed is [N, {packed.shape[1]}] but ceil(K/4) = {row_bytes(K)}")
    if group_size is None:
        group_size = 0 if scale.dim() == 1 else K // max(scale.shape[-1], 1)
    want = (N,) if group_size == 0 else (N, K // group_size if group_size else 0)
    if tuple(scale.shape) != want:
        raise ValueError(f"scale shape {tuple(scale.shape)} != {want}")
    odt = out_dtype or x.dtype
    if out is None:
        out = torch.empty((M, N), dtype=odt, device=x.device)
    elif out.shape != (M, N) or not out.is_contiguous() or out.dtype != odt:
        raise ValueError("out must be a contiguous [M, N] tensor of out_dtype")
    packed = packed.contiguous()
    scale = scale.contiguous()
    lib = load()
    if mask is not None:
        if path != "auto":
            raise ValueError("a zero-block mask runs on the automatic path only")
        _need_cuda(mask)
        rc = lib.ternary_linear_masked(_ptr(x2), _DT[x.dtype], _ptr(packed), _ptr(scale),
                                       int(group_size), _ptr(mask.contiguous()), _ptr(out),
                                       _DT[odt], M, N, K,
                                       FLAG_STATIC_WEIGHTS if static_weights else 0,
                                       _stream(x.device))
        _check(rc, "ternary_linear_masked")
        return out.reshape(*lead, N)
    rc = lib.ternary_linear_ex(_ptr(x2), _DT[x.dtype], _ptr(packed), _ptr(scale),
                               int(group_size), _ptr(out), _DT[odt], M, N, K, PATHS[path],
                               FLAG_STATIC_WEIGHTS if static_weights else 0, _stream(x.device))
    _check(rc, "ternary_linear")
    return out.reshape(*lead, N)


def linear_fused(x: torch.Tensor, packed: torch.Tensor, scale: torch.Tensor,
                 shard_sizes: list[int], **kw) -> list[torch.Tensor]:
    """One call over a fused layer (e.g. QKV, gate/up): rows of the shards are
    stacked in ``packed`` and ``scale`` at the same offsets; returns each
    shard's output as a column view of the fused output."""
    if sum(shard_sizes) != packed.shape[0] or scale.shape[0] != packed.shape[0]:
        raise ValueError("shard sizes must add up to the rows of packed and of scale")
    y = linear(x, packed, scale, **kw)
    outs, off = [], 0
    for n in shard_sizes:
        outs.append(y[..., off:off + n])
        off += n
    return outs


def device_status(clear: bool = True) -> int:
    """Read the current device's status word (0 = OK, TL_ERR_TIMEOUT after a
    bounded device wait gave up).  Synchronous."""
    code = ctypes.c_int32(0)
    _check(load().ternary_device_status(ctypes.byref(code), int(clear)), "ternary_device_status")
    return int(code.value)


def device_status_async(dst: torch.Tensor, clear: bool = True) -> torch.Tensor:
    """Enqueue a copy of the status word into ``dst`` (an int32 tensor of one
    element on the device, or pinned on the host) on the current stream."""
    if dst.dtype != torch.int32 or dst.numel() != 1:
        raise ValueError("dst must be a one-element int32 tensor")
    dev = dst.device if dst.is_cuda else torch.device("cuda", torch.cuda.current_device())
    _check(load().ternary_device_status_async(_ptr(dst), int(clear), _stream(dev)),
           "ternary_device_status_async")
    return dst


def linear_silu_mul(x: torch.Tensor, packed: torch.Tensor, scale: torch.Tensor,
                    group_size: int | None = None, out_dtype: torch.dtype | None = None,
                    out: torch.Tensor | None = None,
                    static_weights: bool = False, mask: torch.Tensor | None = None) -> torch.Tensor:
    """silu(g) * u for a fused gate/up layer, in one kernel.

    ``packed`` [2N, K/4] and ``scale`` ([2N] or [2N, K/G]) stack the gate rows
    then the up rows; g = x @ gate^T, u = x @ up^T; returns [..., N].
    """
    _need_cuda(x, packed, scale, out)
    if x.dtype not in (torch.float16, torch.bfloat16):
        raise ValueError("x must be fp16 or bf16")
    if scale.dtype != torch.float16:
        raise ValueError("scale must be fp16")
    if packed.dtype != torch.uint8 or packed.dim() != 2 or packed.shape[0] % 2:
        raise ValueError("packed must be a 2-D uint8 tensor [2N, K/4]")
    K = x.shape[-1]
    lead = x.shape[:-1]
    M = 1
    for d in lead:
        M *= int(d)
    x2 = x.reshape(M, K).contiguous()
    N2 = packed.shape[0]
    N = N2 // 2
    if packed.shape[1] != row_bytes(K):
        raise ValueError(f"packed is [2N, {packed.shape[1]}] but ceil(K/4) = {row_bytes(K)}")
    if group_size is None:
        group_size = 0 if scale.dim() == 1 else K // max(scale.shape[-1], 1)
    want = (N2,) if group_size == 0 else (N2, K // group_size if group_size else 0)
    if tuple(scale.shape) != want:
        raise ValueError(f"scale shape {tuple(scale.shape)} != {want}")
    odt = out_dtype or x.dtype
    if out is None:
        out = torch.empty((M, N), dtype=odt, device=x.device)
    elif out.shape != (M, N) or not out.is_contiguous() or out.dtype != odt:
        raise ValueError("out must be a contiguous [M, N] tensor of out_dtype")
    packed = packed.contiguous()
    scale = scale.contiguous()
    if mask is not None:
        _need_cuda(mask)
        rc = load().ternary_linear_silu_mul_masked(_ptr(x2), _DT[x.dtype], _ptr(packed),
                                                   _ptr(scale), int(group_size),
                                                   _ptr(mask.contiguous()), _ptr(out), _DT[odt],
                                                   M, N, K,
                                                   FLAG_STATIC_WEIGHTS if static_weights else 0,
                                                   _stream(x.device))
        _check(rc, "ternary_linear_silu_mul_masked")
        return out.reshape(*lead, N)
    rc = load().ternary_linear_silu_mul(_ptr(x2), _DT[x.dtype], _ptr(packed), _ptr(scale),
                                        int(group_size), _ptr(out), _DT[odt], M, N, K,
                                        FLAG_STATIC_WEIGHTS if static_weights else 0,
                                        _stream(x.device))
    _check(rc, "ternary_linear_silu_mul")
    return out.reshape(*lead, N)
