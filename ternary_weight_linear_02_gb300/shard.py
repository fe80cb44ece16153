"""Tensor-parallel sharding of a packed ternary layer (host-side slicing only).

A layer is packed [N, K/4] uint8 plus an fp16 scale [N] (per output channel) or
[N, K/128] (per 128-wide K group).  The two ways to split it across ranks
("三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战", trdm.cn/news/729035,
§3.2, §5.1):

* column parallel (split N): packed rows and scale rows are cut at the same
  offsets; each rank computes its output columns, an all-gather (or just the
  concatenation) rebuilds out[M, N].  No arithmetic changes.
* row parallel (split K): packed columns are cut at byte offsets and the group
  scale columns at group offsets; a per-channel scale is kept whole on every
  rank.  Each rank's output is a partial sum already multiplied by its scales;
  summing the partials (an all-reduce) rebuilds out[M, N].  The cuts must land
  on multiples of 64 k (16-byte packed rows, the kernel's K alignment) and, with
  a group scale, of 128 k (whole groups).

Nothing here reads the codes: slicing is exact, and a cut that would split a
group or a 16-byte row is rejected rather than repacked.
"""
from __future__ import annotations

import torch

K_ALIGN = 64       # k per 16-byte packed row segment (kernel requirement)
GROUP = 128        # k per scale group


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
    """Column-parallel shards: [(packed_i [N_i, K/4], scale_i [N_i] or [N_i, G])]."""
    if sum(sizes) != packed.shape[0] or scale.shape[0] != packed.shape[0]:
        raise ValueError("shard sizes must add up to the rows of packed and of scale")
    out, off = [], 0
    for n in sizes:
        out.append((packed[off:off + n].contiguous(), scale[off:off + n].contiguous()))
        off += n
    return out


def split_k(packed: torch.Tensor, scale: torch.Tensor, sizes: list[int]):
    """Row-parallel shards: [(packed_i [N, K_i/4], scale_i, k_offset_i)].

    `sizes` are the K extents of the shards (sum = K).  A per-channel scale [N]
    is shared by all shards; a group scale [N, K/128] is cut by groups."""
    K = packed.shape[1] * 4
    if sum(sizes) != K:
        raise ValueError(f"shard K sizes add up to {sum(sizes)}, not K = {K}")
    group = scale.dim() == 2
    align = GROUP if group else K_ALIGN
    out, k0 = [], 0
    for k in sizes:
        if k % align or k0 % align:
            raise ValueError(f"K cut at {k0}+{k} is not a multiple of {align}")
        p = packed[:, k0 // 4:(k0 + k) // 4].contiguous()
        s = scale[:, k0 // GROUP:(k0 + k) // GROUP].contiguous() if group else scale
        out.append((p, s, k0))
        k0 += k
    return out
