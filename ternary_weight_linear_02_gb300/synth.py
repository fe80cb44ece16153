"""Seeded synthetic inputs for the ternary linear layer.

This module only draws random inputs.  It holds none of the layer's
arithmetic: it never maps a code to a value and never computes a product.  It
writes four independently drawn 2-bit codes into each byte at the storage
positions the format fixes (field j of a byte at bits [2j+1:2j]), which is
needed to give the bytes the stated code distribution.  Both the CUDA path and
the CPU oracle are fed the tensors it returns.

The workloads of the pages are layer shapes of real checkpoints (a ~0.6B
embedding model, a 7B- and a 27B-class model); no checkpoint is available, so
the shapes are reproduced with these draws:

* codes iid per weight: P(00)=0.4, P(01)=0.3, P(10)=0.3 (the code table's
  three legal codes; the ±1 codes are equally likely, so which of 01 / 10 is
  +1 does not matter here).  Optionally, with probability ``p_reserved`` per
  byte, one uniformly chosen field of that byte is overwritten with the
  reserved code 11.
* activations x ~ N(0,1), rounded to fp16 or bf16 (round-to-nearest-even).
* fp16 scales ~ U[lo, hi].
"""
from __future__ import annotations

import hashlib

import torch

CODE_P = (0.4, 0.3, 0.3)  # P(00), P(01), P(10)


def seed_for(*keys) -> int:
    """A 63-bit seed derived from a tuple of keys (config name, shape, tensor id...)."""
    h = hashlib.sha256(repr(keys).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def packed_codes(N: int, K: int, seed: int, device="cpu", p_reserved: float = 0.0,
                 chunk_rows: int | None = None) -> torch.Tensor:
    """Random packed weights [N, ceil(K/4)] uint8 with the code distribution above.
    When K % 4 != 0 the last byte's padding fields are drawn like the rest (any
    code, 11 included), so a reader that took them for weights would be seen."""
    dev = torch.device(device)
    Kq = (K + 3) // 4
    out = torch.empty((N, Kq), dtype=torch.uint8, device=dev)
    g = _gen(seed, dev)
    if chunk_rows is None:
        chunk_rows = max(1, (1 << 26) // max(K, 1))
    lo, hi = CODE_P[0], CODE_P[0] + CODE_P[1]
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        u = torch.rand((r1 - r0, Kq, 4), generator=g, device=dev)
        codes = torch.zeros_like(u, dtype=torch.uint8)
        codes[(u >= lo) & (u < hi)] = 1
        codes[u >= hi] = 2
        if p_reserved > 0.0:
            hit = torch.rand((r1 - r0, Kq), generator=g, device=dev) < p_reserved
            field = torch.randint(0, 4, (r1 - r0, Kq), generator=g, device=dev)
            sel = torch.nn.functional.one_hot(field, 4).to(torch.bool) & hit.unsqueeze(-1)
            codes[sel] = 3
        byte = (codes[..., 0] | (codes[..., 1] << 2) | (codes[..., 2] << 4)
                | (codes[..., 3] << 6))
        out[r0:r1] = byte
        del u, codes, byte
    return out


def block_sparse(packed: torch.Tensor, p_zero: float, seed: int, rows: int = 128,
                 cols: int = 64) -> torch.Tensor:
    """A copy of packed [N, K/4] in which each block of `rows` weight rows x `cols`
    weights is, with probability p_zero, overwritten with zero codes (00, or 11 in
    a random half of the zeroed blocks) -- block-sparse weights for the
    zero-block map.  Returns the copy; the drawn pattern is not returned."""
    out = packed.clone()
    N, Kq = out.shape
    g = _gen(seed, "cpu")
    RB, KB = (N + rows - 1) // rows, (4 * Kq + cols - 1) // cols
    zero = torch.rand((RB, KB), generator=g) < p_zero
    fill = torch.randint(0, 2, (RB, KB), generator=g)
    for rb, kb in zero.nonzero().tolist():
        out[rb * rows:(rb + 1) * rows, kb * cols // 4:(kb + 1) * cols // 4] = 0xFF if fill[rb, kb] else 0
    return out


def activations(M: int, K: int, dtype: torch.dtype, seed: int, device="cpu") -> torch.Tensor:
    """x [M, K] ~ N(0,1) rounded to fp16 / bf16."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    return torch.randn((M, K), generator=g, device=dev, dtype=torch.float32).to(dtype)


def scales(N: int, groups: int, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    """fp16 scales ~ U[lo, hi]: shape [N] if groups == 0 else [N, groups]."""
    dev = torch.device(device)
    g = _gen(seed, dev)
    shape = (N,) if groups == 0 else (N, groups)
    u = torch.rand(shape, generator=g, device=dev, dtype=torch.float32)
    return (lo + (hi - lo) * u).to(torch.float16)


def layer(M: int, N: int, K: int, x_dtype: torch.dtype, group_size: int, s_lo: float,
          s_hi: float, keys: tuple, device="cpu", p_reserved: float = 0.0):
    """(x, packed, scale) for one layer, every tensor seeded from ``keys``."""
    groups = 0 if group_size == 0 else K // group_size
    x = activations(M, K, x_dtype, seed_for(*keys, "x", M), device)
    packed = packed_codes(N, K, seed_for(*keys, "w"), device, p_reserved)
    s = scales(N, groups, s_lo, s_hi, seed_for(*keys, "s"), device)
    return x, packed, s
