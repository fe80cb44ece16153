"""Host-side tensor-parallel slicing (no GPU): per-shard oracle results must
reassemble the whole layer's oracle result -- exactly for a column split (each
output row is computed from the same codes, scales and x), and up to fp64
summation order for a K split (partial sums added across shards)."""
import numpy as np
import pytest
import torch

import oracle
from ternary_weight_linear_02_gb300 import shard, synth
from parity import oracle_ref


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_even_cuts():
    assert shard.even_cuts(4096, 4, 64) == [1024] * 4
    cuts = shard.even_cuts(11008, 3, 128)
    assert sum(cuts) == 11008 and all(c % 128 == 0 for c in cuts)
    assert max(cuts) - min(cuts) <= 128
    with pytest.raises(ValueError):
        shard.even_cuts(4096 + 64, 2, 128)
    with pytest.raises(ValueError):
        shard.even_cuts(128, 3, 64)


@pytest.mark.parametrize("gs", [0, 128])
def test_split_n_reassembles_exactly(gs):
    M, N, K = 3, 300, 512
    x, p, s = synth.layer(M, N, K, torch.bfloat16, gs, 0.005, 0.05, ("shard-n", gs), "cpu", 0.01)
    full = oracle_ref(x, p, s, gs)
    parts = shard.split_n(p, s, [100, 72, 128])
    got = np.concatenate([oracle_ref(x, pi, si, gs) for pi, si in parts], axis=1)
    assert np.array_equal(got, full)


@pytest.mark.parametrize("gs", [0, 128])
def test_split_k_sums_to_full(gs):
    M, N, K = 4, 96, 1536
    x, p, s = synth.layer(M, N, K, torch.float16, gs, 0.005, 0.05, ("shard-k", gs), "cpu", 0.01)
    full = oracle_ref(x, p, s, gs)
    sizes = shard.even_cuts(K, 3, 128 if gs else 64)
    total = np.zeros_like(full)
    for pi, si, k0 in shard.split_k(p, s, sizes):
        total += oracle_ref(x[:, k0:k0 + pi.shape[1] * 4].contiguous(), pi, si, gs)
    np.testing.assert_allclose(total, full, rtol=1e-12, atol=1e-12)


def test_split_k_rejects_misaligned_cuts():
    _, p, s = synth.layer(1, 8, 512, torch.float16, 128, 0.005, 0.05, ("shard-bad",), "cpu")
    with pytest.raises(ValueError):
        shard.split_k(p, s, [192, 320])          # 192 splits a 128-wide group
    _, p32, s32 = synth.layer(1, 8, 512, torch.float16, 32, 0.005, 0.05, ("shard-32",), "cpu")
    shard.split_k(p32, s32, [96, 416])           # whole 32-wide groups
    with pytest.raises(ValueError):
        shard.split_k(p32, s32, [100, 412])
    _, p0, s0 = synth.layer(1, 8, 512, torch.float16, 0, 0.005, 0.05, ("shard-bad0",), "cpu")
    shard.split_k(p0, s0, [192, 320])            # per channel: any byte boundary slices
    shard.split_k(p0, s0, [96, 416])
    with pytest.raises(ValueError, match="device"):
        shard.split_k(p0, s0, [97, 415])         # off a byte boundary: repacked on the device only
    with pytest.raises(ValueError):
        shard.split_k(p0, s0, [0, 512])
    with pytest.raises(ValueError):
        shard.split_n(p0, s0, [4, 3])


@pytest.mark.parametrize("gs,sizes", [(0, [96, 4, 412]), (32, [160, 352]), (64, [64, 448])])
def test_split_k_byte_aligned_cuts_sum_to_full(gs, sizes):
    """Byte-aligned cuts off the 64-k grid are plain slices; the shards' oracle
    results add up to the whole layer's."""
    M, N, K = 3, 40, 512
    x, p, s = synth.layer(M, N, K, torch.bfloat16, gs, 0.005, 0.05, ("shard-byte", gs), "cpu", 0.01)
    full = oracle_ref(x, p, s, gs)
    total = np.zeros_like(full)
    for (pi, si, k0), k in zip(shard.split_k(p, s, sizes), sizes):
        assert pi.shape == (N, (k + 3) // 4)
        total += oracle_ref(x[:, k0:k0 + k].contiguous(), pi, si, gs)
    np.testing.assert_allclose(total, full, rtol=1e-12, atol=1e-12)


def test_split_k_last_shard_keeps_padding():
    """K % 4 != 0: a last shard that starts on a byte boundary is a plain slice
    whose last byte carries the layer's padding fields."""
    M, N, K = 2, 16, 103
    x, p, s = synth.layer(M, N, K, torch.float16, 0, 0.005, 0.05, ("shard-pad",), "cpu", 0.01)
    parts = shard.split_k(p, s, [64, 39], K=K)
    assert parts[1][0].shape == (N, 10)
    full = oracle_ref(x, p, s, 0)
    total = sum(oracle_ref(x[:, k0:k0 + k].contiguous(), pi, si, 0)
                for (pi, si, k0), k in zip(parts, [64, 39]))
    np.testing.assert_allclose(total, full, rtol=1e-12, atol=1e-12)
