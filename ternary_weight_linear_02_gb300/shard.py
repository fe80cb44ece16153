"""Tensor-parallel sharding of a packed ternary layer.

A layer is packed [N, ceil(K/4)] uint8 plus an fp16 scale [N] (per output
channel) or [N, K/G] (per G-wide K group, G in 32, 64, 128, 256).  The two ways
to split it across ranks ("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战",
trdm.cn/news/729035, §3.2, §5.1):

* column parallel (split N): packed rows and scale rows are cut at the same
  offsets; each rank computes its output columns, an all-gather (or just the
  concatenation) rebuilds out[M, N].  No arithmetic changes.
* row parallel (split K): each rank takes a contiguous K range; a per-channel
  scale is kept whole on every rank, a group scale is cut by groups.  Each
  rank's output is a partial sum already multiplied by its scales; summing the
  partials (an all-reduce) rebuilds out[M, N].

Where a K cut does not fall on a byte boundary (k0 % 4 != 0), the packed codes
of the range cannot be sliced out as bytes: the same page (§3.2) has the rows
unpacked to integers, cut on the original shape and packed again.  That is done
here with the library's own unpack / pack kernels (CUDA tensors only); the
resulting shard has K_i weights per row in ceil(K_i/4) bytes.  With a group
scale, a cut inside a group would leave that group's scale to two shards whose
groups no longer start at their own k = 0, so group-mode cuts must be whole
groups (always byte-aligned, since G % 4 == 0).  Cuts on multiples of 64 keep
every shard on the TMA-fed kernels; other shards run on the generic kernel.
"""
from __future__ import annotations

import torch

FAST_ALIGN = 64    # k per 16-byte packed row segment: shards stay on the TMA-fed kernels


def row_bytes(K: int) -> int:
    return (int(K) + 3) // 4


def even_cuts(total: int, parts: int, align: int) -> list[int]:
    """Split `total` into `parts` contiguous sizes, each a multiple of `align`
    (the last one takes the remainder), as even as the alignment allows."""
    if parts < 1:
        raise ValueError("parts must be >= 1")
    if total % align:
        raise ValueError(f"total {total} is not a multiple of {align}")
    units = total // align
    if units < parts:
        raise ValueError(f"cannot cut {total} into {parts} parts of multiples of {align}")
    base, extra = divmod(units, parts)
    return [(base + (1 if i < extra else 0)) * align for i in range(parts)]


def split_n(packed: torch.Tensor, scale: torch.Tensor, sizes: list[int]):
    """Column-parallel shards: [(packed_i [N_i, ceil(K/4)], scale_i [N_i] or [N_i, K/G])]."""
    if sum(sizes) != packed.shape[0] or scale.shape[0] != packed.shape[0]:
        raise ValueError("shard sizes must add up to the rows of packed and of scale")
    out, off = [], 0
    for n in sizes:
        out.append((packed[off:off + n].contiguous(), scale[off:off + n].contiguous()))
        off += n
    return out


def _group_size(scale: torch.Tensor, K: int, group_size: int | None) -> int:
    if scale.dim() == 1:
        return 0
    G = group_size if group_size is not None else K // max(scale.shape[1], 1)
    if G <= 0 or K % G or scale.shape[1] != K // G:
        raise ValueError(f"scale {tuple(scale.shape)} is not a [N, K/G] group scale for K = {K}")
    return G


def _repack_range(packed: torch.Tensor, K: int, k0: int, k: int) -> torch.Tensor:
    """Weights [k0, k0 + k) of every row as a packed [N, ceil(k/4)] matrix:
    unpack on the device, cut, pack again (padding fields written 00)."""
    if not packed.is_cuda:
        raise ValueError(f"a K cut at {k0} is not on a byte boundary: unpacking and "
                         "repacking runs on the device, move packed to CUDA first")
    from . import pack, unpack  # the library's kernels
    t, _ = unpack(packed, K)
    p, bad = pack(t[:, k0:k0 + k].contiguous())
    if int(bad.item()) != 0:
        raise RuntimeError("repacking produced invalid codes")
    return p


def split_k(packed: torch.Tensor, scale: torch.Tensor, sizes: list[int],
            group_size: int | None = None, K: int | None = None):
    """Row-parallel shards: [(packed_i [N, ceil(K_i/4)], scale_i, k_offset_i)].

    `sizes` are the K extents of the shards (sum = K; K defaults to 4 * bytes per
    row).  A per-channel scale [N] is shared by all shards; a group scale
    [N, K/G] is cut by groups, and every cut must then be a multiple of G.
    Cuts off byte boundaries are unpacked and repacked (CUDA tensors)."""
    K = 4 * packed.shape[1] if K is None else int(K)
    if row_bytes(K) != packed.shape[1]:
        raise ValueError(f"packed rows of {packed.shape[1]} bytes do not hold K = {K}")
    if sum(sizes) != K or any(k <= 0 for k in sizes):
        raise ValueError(f"shard K sizes {sizes} must be positive and add up to K = {K}")
    G = _group_size(scale, K, group_size)
    out, k0 = [], 0
    for k in sizes:
        if G and (k % G or k0 % G):
            raise ValueError(f"K cut at {k0}+{k} splits a {G}-wide scale group")
        if k0 % 4 == 0 and (k % 4 == 0 or k0 + k == K):
            p = packed[:, k0 // 4:row_bytes(k0 + k)].contiguous()  # whole bytes: a plain slice
        else:
            p = _repack_range(packed, K, k0, k)
        s = scale[:, k0 // G:(k0 + k) // G].contiguous() if G else scale
        out.append((p, s, k0))
        k0 += k
    return out
