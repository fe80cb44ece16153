"""Split K on the tile kernel against the oracle.

When ceil(N/128) * ceil(M/BN) output tiles alone would leave SMs idle, a cluster
of up to 8 CTAs shares one tile: each multiplies its own K range, the partial
tiles are exchanged through cluster shared memory (each CTA owns BN/sk token
columns) and added in rank order.  The shapes below have few row blocks and long
K, so the planner splits; they cover every scale mode (per channel, fp16 folded
group scales, bf16 split group scales, 32- to 256-wide groups), ragged N and M
(slices past the last token), every output dtype, the zero-block map, and
bit-for-bit repeatability of the rank-ordered sum.
"""
import numpy as np
import pytest
import torch

import oracle
import ternary_weight_linear_02_gb300 as tl
from ternary_weight_linear_02_gb300 import synth

from parity import check, oracle_ref

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


def inputs(M, N, K, xdt, gs, seed):
    x, p, s = synth.layer(M, N, K, xdt, gs, 0.005, 0.05, ("tile-split", seed, M, N, K, str(xdt), gs),
                          "cpu", 0.01)
    return x.to(DEV), p.to(DEV), s.to(DEV)


CASES = [
    # M, N, K, x dtype, group size, out dtype  (BN = 64 / 128 / 256 by M)
    (17, 128, 8192, BF16, 0, F32),
    (33, 300, 4096, F16, 0, F32),
    (37, 129, 18944, BF16, 0, BF16),     # ragged M: the last slices hold no token
    (64, 128, 3584, BF16, 0, F32),
    (64, 200, 4096, BF16, 128, F32),     # bf16 x, split group scales
    (64, 257, 4096, F16, 128, F16),      # fp16 x, folded group scales
    (90, 100, 2048, BF16, 64, F32),
    (100, 64, 4096, F16, 32, F32),
    (128, 300, 8192, BF16, 256, F32),
    (200, 129, 4096, BF16, 0, F32),
    (256, 384, 3584, F16, 0, F32),
    (300, 100, 18944, BF16, 0, F16),
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", CASES)
def test_tile_split_against_oracle(M, N, K, xdt, gs, odt):
    x, p, s = inputs(M, N, K, xdt, gs, 1)
    y = tl.linear(x, p, s, gs, out_dtype=odt, path="tile")
    torch.cuda.synchronize()
    check(y, oracle_ref(x, p, s, gs), x, s, what=f"tile split {M}x{N}x{K} g{gs}")


@pytest.mark.parametrize("M,N,K,gs", [(64, 300, 18944, 0), (256, 200, 8192, 128)])
def test_tile_split_repeatable(M, N, K, gs):
    x, p, s = inputs(M, N, K, BF16, gs, 2)
    a = tl.linear(x, p, s, gs, out_dtype=F32, path="tile")
    b = tl.linear(x, p, s, gs, out_dtype=F32, path="tile")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_tile_split_every_byte_exact():
    """Row n holds byte n at k = 8000 (inside the last CTA's K range when split):
    token 0 is x = (1, 3, 9, 27) there, s = 1, so y[0, n] is the byte's
    balanced-ternary value, exact; the other tokens are zero."""
    M, K = 64, 8192
    p = torch.zeros((256, K // 4), dtype=torch.uint8)
    p[:, 2000] = torch.arange(256, dtype=torch.uint8)
    x = torch.zeros((M, K), dtype=F32)
    x[0, 8000:8004] = torch.tensor([1.0, 3.0, 9.0, 27.0])
    x = x.to(BF16)
    s = torch.ones(256, dtype=F16)
    want = oracle_ref(x, p, s, 0)
    y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), 0, out_dtype=F32, path="tile")
    assert np.array_equal(y.cpu().double().numpy(), want)


def test_tile_split_with_zero_block_map():
    M, N, K = 64, 384, 8192
    x, p, s = inputs(M, N, K, BF16, 0, 3)
    p = synth.block_sparse(p.cpu(), 0.5, 77).to(DEV)
    mask, _ = tl.block_mask(p)
    a = tl.linear(x, p, s, 0, out_dtype=F32)
    b = tl.linear(x, p, s, 0, out_dtype=F32, mask=mask)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    check(b, oracle_ref(x, p, s, 0), x, s, what="tile split, masked")
