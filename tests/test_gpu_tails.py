"""K tails and 32-wide groups against the oracle.

K % 64 != 0: packed rows are ceil(K/4) bytes, not 16-byte pitched, so the
TMA-fed kernels cannot take them and the automatic path runs the generic
CUDA-core kernel.  K % 4 != 0 rows end in padding fields (the Qwen2.5-7B
ternary-in-vLLM write-up §2.3: an export pads rows to whole bytes, and the
padding is cut off after unpacking); the synthetic weights put random codes
there, 11 included, so any reader that took them for weights is caught.

32-wide groups ("第13章 量化：精度与速度的工程平衡" §13.3.3) run on the tile
kernel at every M when K % 64 == 0 (two scales per 64-k chunk), on the generic
kernel otherwise.  The generic kernel is
also checked at K % 64 == 0 through path="generic", against the oracle and
against the other kernels.
"""
import numpy as np
import pytest
import torch

import oracle
import ternary_weight_linear_02_gb300 as tl
from ternary_weight_linear_02_gb300 import synth

from parity import check, check_silu, oracle_ref, silu_refs

pytestmark = pytest.mark.gpu

DEV = "cuda"
F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tl.build()
    oracle.build()
    tl.load()


def inputs(M, N, K, xdt, gs, seed, p_reserved=0.01):
    x, p, s = synth.layer(M, N, K, xdt, gs, 0.005, 0.05, ("tails", seed, M, N, K, str(xdt), gs),
                          "cpu", p_reserved)
    return x.to(DEV), p.to(DEV), s.to(DEV)


TAIL_CASES = [
    # M, N, K, x dtype, group size, out dtype
    (1, 1, 4, BF16, 0, F32),           # one packed byte
    (1, 33, 12, F16, 0, F32),
    (1, 300, 100, BF16, 0, F32),
    (1, 4096, 4100, BF16, 0, F32),     # a 7B-sized row with a 4-wide tail
    (5, 7, 4, F16, 0, F16),
    (5, 129, 12, BF16, 0, BF16),
    (5, 300, 100, F16, 0, F32),
    (5, 513, 4100, BF16, 0, F32),
    (40, 33, 100, BF16, 0, F32),       # several token blocks
    (40, 300, 4100, F16, 0, F32),
    (300, 65, 12, BF16, 0, F32),
    (300, 129, 4100, BF16, 0, BF16),
    (1, 64, 32, BF16, 32, F32),        # one 32-wide group
    (3, 200, 96, F16, 32, F32),
    (17, 300, 160, BF16, 32, F32),
    (9, 257, 4128, BF16, 32, F32),     # 129 groups of 32
    (64, 100, 4128, F16, 32, F16),
    # K % 4 != 0: per channel only (a group size divides K)
    (1, 1, 1, BF16, 0, F32),
    (1, 300, 3, F16, 0, F32),
    (5, 129, 5, BF16, 0, F32),
    (5, 200, 7, F16, 0, F16),
    (9, 300, 101, BF16, 0, F32),
    (40, 513, 4099, BF16, 0, F32),
    (300, 65, 2, F16, 0, BF16),
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", TAIL_CASES)
def test_k_tail_against_oracle(M, N, K, xdt, gs, odt):
    assert K % 64 != 0
    x, p, s = inputs(M, N, K, xdt, gs, 1)
    y = tl.linear(x, p, s, gs, out_dtype=odt)
    torch.cuda.synchronize()
    check(y, oracle_ref(x, p, s, gs), x, s, what=f"tail {M}x{N}x{K} g{gs}")


G32_CASES = [
    # K % 64 == 0: the tile kernel folds two scales per 64-k chunk
    (1, 300, 64, BF16, F32),
    (1, 4096, 4096, BF16, F32),
    (8, 129, 1024, F16, F32),
    (16, 300, 3584, BF16, BF16),
    (17, 513, 2048, BF16, F32),
    (64, 257, 4096, F16, F32),
    (300, 200, 1536, BF16, F16),
]


@pytest.mark.parametrize("M,N,K,xdt,odt", G32_CASES)
def test_group32_tile_against_oracle(M, N, K, xdt, odt):
    x, p, s = inputs(M, N, K, xdt, 32, 2)
    y = tl.linear(x, p, s, 32, out_dtype=odt)
    torch.cuda.synchronize()
    if N * K > 2048 * 2048:
        rows = np.unique(np.concatenate([np.arange(0, N, max(1, N // 97)), [N - 1]]))
        check(y[:, rows], oracle_ref(x, p, s, 32, rows=rows), x, s, rows=rows,
              what=f"g32 {M}x{N}x{K}")
    else:
        check(y, oracle_ref(x, p, s, 32), x, s, what=f"g32 {M}x{N}x{K}")


def test_group32_scales_are_per_half_chunk():
    """Every weight +1, x = 1, s[n, g] = g + 1: y[m, n] = 32 * sum_g (g + 1), exact.
    A kernel that applied one scale per 64-k chunk would give 64 * sum of the
    even-indexed (or odd-indexed) scales instead."""
    M, N, K = 3, 128, 256
    p = torch.full((N, K // 4), 0x55, dtype=torch.uint8)  # 01 01 01 01: four +1
    x = torch.ones((M, K), dtype=BF16)
    s = (torch.arange(K // 32, dtype=torch.float32) + 1).repeat(N, 1).to(F16)
    want = 32.0 * sum(range(1, K // 32 + 1))
    for path in ("auto", "tile", "generic"):
        y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), 32, out_dtype=F32, path=path)
        assert torch.all(y.cpu() == want), path


GENERIC_CASES = [
    # K % 64 == 0 through the generic kernel: every scale mode
    (1, 300, 256, BF16, 0),
    (5, 129, 1024, F16, 64),
    (17, 200, 2048, BF16, 128),
    (40, 65, 4096, BF16, 256),
    (9, 100, 192, F16, 32),
]


@pytest.mark.parametrize("M,N,K,xdt,gs", GENERIC_CASES)
def test_generic_path_matches_oracle_and_auto(M, N, K, xdt, gs):
    x, p, s = inputs(M, N, K, xdt, gs, 3)
    g = tl.linear(x, p, s, gs, out_dtype=F32, path="generic")
    a = tl.linear(x, p, s, gs, out_dtype=F32)
    torch.cuda.synchronize()
    check(g, oracle_ref(x, p, s, gs), x, s, what=f"generic {M}x{N}x{K} g{gs}")
    check(a, oracle_ref(x, p, s, gs), x, s, what=f"auto {M}x{N}x{K} g{gs}")


def test_generic_every_byte_exact():
    """Row n holds byte n in its last four weights (a tail byte at K = 100);
    x = (1, 3, 9, 27) there, s = 1: y[0, n] is the balanced-ternary value of the
    byte, an exact integer that identifies all four decoded weights."""
    K = 100
    p = torch.zeros((256, K // 4), dtype=torch.uint8)
    p[:, -1] = torch.arange(256, dtype=torch.uint8)
    x = torch.zeros((2, K), dtype=torch.float32)
    x[0, -4:] = torch.tensor([1.0, 3.0, 9.0, 27.0])
    x[1, -4:] = torch.tensor([27.0, -9.0, 3.0, -1.0])
    x = x.to(F16)
    s = torch.ones(256, dtype=F16)
    want = oracle_ref(x, p, s, 0)
    y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), 0, out_dtype=F32)
    assert np.array_equal(y.cpu().double().numpy(), want)


SILU_CASES = [
    # M, N (gate rows = up rows = output columns), K, x dtype, group size, out dtype
    (1, 100, 100, BF16, 0, F32),       # generic kernel
    (5, 129, 103, F16, 0, F32),        # padded rows
    (9, 300, 4100, F16, 0, F32),
    (40, 65, 96, BF16, 32, BF16),
    (3, 200, 1024, BF16, 32, F32),     # tile kernel, 32-wide groups
    (64, 129, 4096, F16, 32, F32),
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", SILU_CASES)
def test_silu_mul_tails_and_group32(M, N, K, xdt, gs, odt):
    x, p, s = inputs(M, 2 * N, K, xdt, gs, 4, p_reserved=0.001)
    h = tl.linear_silu_mul(x, p, s, gs, out_dtype=odt)
    torch.cuda.synchronize()
    h_ref, g_ref, u_ref = silu_refs(x, p, s, gs)
    check_silu(h, h_ref, g_ref, u_ref, x, s, what=f"silu {M}x{N}x{K} g{gs}")


def test_forced_tma_paths_refuse_k_tails():
    x, p, s = inputs(4, 64, 100, BF16, 0, 5)
    for path in ("skinny", "tile"):
        with pytest.raises(tl.TernaryError, match="UNSUPPORTED"):
            tl.linear(x, p, s, 0, path=path)


@pytest.mark.parametrize("K", [4100, 4099])
def test_masked_call_with_k_tail_equals_unmasked(K):
    x, p, s = inputs(4, 300, K, BF16, 0, 6)
    mask, _ = tl.block_mask(p, K)
    a = tl.linear(x, p, s, 0, out_dtype=F32)
    b = tl.linear(x, p, s, 0, out_dtype=F32, mask=mask)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("N,K", [(1, 1), (7, 2), (129, 3), (300, 5), (64, 4099), (513, 201)])
def test_pack_unpack_padded_rows_bit_exact(N, K):
    """Unpack drops the padding fields (whatever codes they hold) and counts
    reserved codes among the K weights only; pack writes padding as 00 and
    round-trips the weights -- all bit for bit against the oracle."""
    p = synth.packed_codes(N, K, synth.seed_for("tails-pack", N, K), "cpu", 0.05)
    t_ref, r_ref = oracle.unpack(p.numpy(), K)
    t, r = tl.unpack(p.to(DEV), K)
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), t_ref) and int(r.item()) == r_ref
    p_ref, bad_ref = oracle.pack(t_ref)
    q, bad = tl.pack(t)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), p_ref) and int(bad.item()) == bad_ref == 0


@pytest.mark.parametrize("N,K", [(300, 4099), (129, 61), (256, 131), (1, 3)])
def test_block_mask_padded_rows_against_oracle(N, K):
    """Padding fields never light a block: weights zeroed everywhere except a
    few rows, padding filled with 01 / 10 codes."""
    p = torch.zeros((N, tl.row_bytes(K)), dtype=torch.uint8)
    pad = 4 * p.shape[1] - K
    if pad:
        p[:, -1] = sum(1 << (2 * j) for j in range(4 - pad, 4))  # padding fields = 01
    p[N // 2, 0] |= 0x02                                          # one -1 weight at k = 0
    m_ref, z_ref = oracle.block_mask(p.numpy(), K)
    m, z = tl.block_mask(p.to(DEV), K)
    torch.cuda.synchronize()
    assert np.array_equal(m.cpu().numpy().view(np.uint32), m_ref) and int(z.item()) == z_ref


@pytest.mark.parametrize("gs,K,sizes", [(0, 4096, [1001, 2047, 1048]),   # off byte boundaries
                                        (0, 4099, [2050, 2049]),
                                        (32, 4096, [1056, 3040])])        # whole 32-wide groups
def test_split_k_repacked_shards(gs, K, sizes):
    """Row-parallel shards cut off byte boundaries are unpacked, cut and packed
    again on the device: each shard's bytes equal the oracle's pack of the
    oracle's unpacked range, and the shards' outputs add up to the layer's."""
    from ternary_weight_linear_02_gb300 import shard
    M, N = 5, 300
    x, p, s = inputs(M, N, K, BF16, gs, 7)
    t_ref, _ = oracle.unpack(p.cpu().numpy(), K)
    total = torch.zeros((M, N), dtype=F32, device=DEV)
    for (pi, si, k0), k in zip(shard.split_k(p, s, sizes, K=K), sizes):
        want, _ = oracle.pack(t_ref[:, k0:k0 + k])
        if k0 % 4 or k % 4:
            assert np.array_equal(pi.cpu().numpy(), want), (k0, k)
        total += tl.linear(x[:, k0:k0 + k].contiguous(), pi, si, gs, out_dtype=F32)
    torch.cuda.synchronize()
    check(total, oracle_ref(x, p, s, gs), x, s, what=f"split-K shards {sizes}")
