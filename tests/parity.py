"""Shared helpers for the GPU parity tests: run the CUDA path through the
binding and compare with the CPU oracle under the stated tolerance."""
import numpy as np
import torch

import oracle

# Tolerance (fp32 accumulation): relative L2 <= 1e-4 and per element
# |err| <= 2e-3 * s_max(n) * sum_k |x[m,k]|.  A 16-bit output adds its own
# rounding: half an ulp of the reference per element and the unit roundoff
# to the relative L2 bound.
REL_L2 = 1e-4
PER_ELEM = 2e-3
UNIT_ROUNDOFF = {torch.float32: 0.0, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def x_dtype_name(dt: torch.dtype) -> str:
    return {torch.float16: "f16", torch.bfloat16: "bf16"}[dt]


def ulp(y: np.ndarray, dt: torch.dtype) -> np.ndarray:
    if dt == torch.float32:
        return np.zeros_like(y)
    mant, emin = (10, -14) if dt == torch.float16 else (7, -126)
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** emin)))
    return 2.0 ** (e - mant)


def oracle_ref(x: torch.Tensor, packed: torch.Tensor, scale: torch.Tensor, group_size: int,
               rows=None, nthreads: int = 8) -> np.ndarray:
    """Oracle output, optionally for a subset of output rows n (columns of y)."""
    p = packed.detach().cpu().numpy()
    s = bits(scale)
    if rows is not None:
        p = p[rows]
        s = s[rows]
    return oracle.linear_from_bits(bits(x), x_dtype_name(x.dtype), p, s, group_size, nthreads)


def round_to(y: np.ndarray, dt: torch.dtype) -> np.ndarray:
    """Round-to-nearest-even of fp64 values to the 16-bit output type (via torch's
    exact float64 -> 16-bit conversion), back in fp64."""
    return torch.from_numpy(np.ascontiguousarray(y)).to(dt).double().numpy()


def check(y_gpu: torch.Tensor, y_ref: np.ndarray, x: torch.Tensor, scale: torch.Tensor,
          rows=None, what=""):
    """Assert the documented tolerance; returns (rel_l2, max_ratio).

    A 16-bit output must also be the round-to-nearest-even image of a value
    within the per-element bound E of the exact result: rounding is monotonic, so
    RNE(y_ref - E) <= y_gpu <= RNE(y_ref + E).  (The fp32 accumulation itself is
    held to relative L2 <= 1e-4 by the fp32-output cases of every kernel path.)"""
    g = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == y_ref.shape, (g.shape, y_ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    s = scale.detach().float().cpu().numpy().astype(np.float64)
    if rows is not None:
        s = s[rows]
    smax = np.abs(s).reshape(s.shape[0], -1).max(axis=1)            # [N]
    xabs = np.abs(x.detach().float().cpu().numpy().astype(np.float64)).sum(axis=1)  # [M]
    E = PER_ELEM * xabs[:, None] * smax[None, :]
    bound = E + 0.5 * ulp(y_ref, y_gpu.dtype)
    if y_gpu.dtype != torch.float32:
        lo, hi = round_to(y_ref - E, y_gpu.dtype), round_to(y_ref + E, y_gpu.dtype)
        bad = (g < lo) | (g > hi)
        assert not bad.any(), f"{what}: {int(bad.sum())} outputs outside the rounded bracket"
    err = np.abs(g - y_ref)
    ratio = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    assert np.all(err <= bound), f"{what}: per-element bound exceeded (max ratio {ratio:.3g})"
    den = float(np.linalg.norm(y_ref))
    rel = float(np.linalg.norm(g - y_ref)) / den if den > 0 else float(np.linalg.norm(g))
    lim = REL_L2 + UNIT_ROUNDOFF[y_gpu.dtype]
    assert rel <= lim, f"{what}: relative L2 {rel:.3g} > {lim:.3g}"
    return rel, ratio


def silu_refs(x: torch.Tensor, packed: torch.Tensor, scale: torch.Tensor, group_size: int,
              nthreads: int = 8):
    """Oracle h = silu(g) * u and the oracle's g, u (fp64) for a stacked gate/up layer."""
    p = packed.detach().cpu().numpy()
    sb = bits(scale)
    xb = bits(x)
    h = oracle.silu_mul_from_bits(xb, x_dtype_name(x.dtype), p, sb, group_size, nthreads)
    y = oracle.linear_from_bits(xb, x_dtype_name(x.dtype), p, sb, group_size, nthreads)
    n = p.shape[0] // 2
    return h, y[:, :n], y[:, n:]


def check_silu(h_gpu: torch.Tensor, h_ref: np.ndarray, g_ref: np.ndarray, u_ref: np.ndarray,
               x: torch.Tensor, scale: torch.Tensor, what=""):
    """Tolerance of the gated product, propagated from the linear's: with E the
    per-element bound of g and u (2e-3 * s_max * sum|x|) and |silu'| <= 1.1,
    |dh| <= 1.1 E |u| + |silu(g)| E + 1.1 E^2, plus 1e-5 |h| for the fp32
    exp / divide / multiply and half an ulp of a 16-bit output; relative L2
    <= 1e-4 (+ unit roundoff of the output dtype)."""
    h = h_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert h.shape == h_ref.shape, (h.shape, h_ref.shape)
    assert np.all(np.isfinite(h)), f"{what}: non-finite output"
    s = scale.detach().float().cpu().numpy().astype(np.float64)
    smax = np.abs(s).reshape(s.shape[0], -1).max(axis=1)
    n = g_ref.shape[1]
    sm = np.maximum(smax[:n], smax[n:])
    xabs = np.abs(x.detach().float().cpu().numpy().astype(np.float64)).sum(axis=1)
    E = PER_ELEM * xabs[:, None] * sm[None, :]
    silu_g = g_ref / (1.0 + np.exp(-g_ref))
    bound = (1.1 * E * np.abs(u_ref) + np.abs(silu_g) * E + 1.1 * E * E + 1e-5 * np.abs(h_ref)
             + 0.5 * ulp(h_ref, h_gpu.dtype))
    err = np.abs(h - h_ref)
    ratio = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    assert np.all(err <= bound), f"{what}: per-element bound exceeded (max ratio {ratio:.3g})"
    den = float(np.linalg.norm(h_ref))
    rel = float(np.linalg.norm(h - h_ref)) / den if den > 0 else float(np.linalg.norm(h))
    lim = REL_L2 + UNIT_ROUNDOFF[h_gpu.dtype]
    assert rel <= lim, f"{what}: relative L2 {rel:.3g} > {lim:.3g}"
    return rel, ratio
