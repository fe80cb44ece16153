"""Zero-block skipping against the oracle: the map built on the GPU is the
oracle's map bit for bit, and a masked call -- which neither loads nor
multiplies zero blocks -- equals the unmasked call bit for bit and meets the
oracle's tolerance, on block-sparse weights (about 30% zero blocks), on the
decode kernel, the tcgen05 skinny kernel (per-channel scales) and the tile
kernel, including row blocks with no live block at all."""
import numpy as np
import pytest
import torch

import oracle
import ternary_weight_linear_02_gb300 as tl
from ternary_weight_linear_02_gb300 import synth

from parity import check, check_silu, oracle_ref, silu_refs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tl.build()
    oracle.build()
    tl.load()


def sparse_inputs(M, N, K, xdt, gs, seed, p_zero=0.3):
    x, p, s = synth.layer(M, N, K, xdt, gs, 0.005, 0.05, ("mask", seed, M, N, K, gs), "cpu")
    p = synth.block_sparse(p, p_zero, synth.seed_for("mask", seed, N, K) & 0xFFFFFFFF)
    return x.to(DEV), p.to(DEV), s.to(DEV)


@pytest.mark.parametrize("N,K", [(1, 64), (300, 4160), (1000, 2048), (129, 100), (256, 12)])
def test_block_mask_matches_oracle(N, K):
    p = synth.packed_codes(N, K, synth.seed_for("maskmap", N, K), "cpu", p_reserved=0.05)
    p = synth.block_sparse(p, 0.4, N * 7 + K)
    want, zero = oracle.block_mask(p.numpy())
    got, cnt = tl.block_mask(p.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy().view(np.uint32).reshape(want.shape), want)
    assert int(cnt.item()) == zero


CASES = [
    # M, N, K, x dtype, group size
    (1, 4096, 4096, torch.bfloat16, 0),     # decode kernel, split K
    (4, 1000, 2048, torch.float16, 128),
    (9, 300, 8192, torch.bfloat16, 0),
    (16, 3584, 3584, torch.bfloat16, 0),
    (16, 512, 1024, torch.float16, 64),
    (24, 700, 3072, torch.bfloat16, 0),      # tcgen05 skinny kernel, 32-token tile
    (24, 300, 2048, torch.bfloat16, 128),    # group scales: tile kernel when masked
    (33, 640, 1024, torch.bfloat16, 0),      # tile kernel from here on
    (100, 300, 2048, torch.float16, 128),
    (300, 512, 1536, torch.bfloat16, 0),
]


def same_kernel(M, N, gs, gated=False):
    """Whether the unmasked call runs on the kernel the masked call runs on.
    Per-channel scales and 64-wide groups: always.  128- and 256-wide groups:
    the tcgen05 skinny kernel reads no map with group scales, so masked calls
    run on the decode kernel (M <= 16) or the tile kernel (17 <= M <= 32) where
    the unmasked call may run on the skinny kernel (M > 8, or plain layers of
    2049..4608 rows, at M <= 16; every M of 17..32)."""
    if gs in (0, 64) or M > 32:
        return True
    if M > 16:
        return False
    if gated:
        return M <= 8
    return M <= 8 and not (2048 < N <= 4608)


@pytest.mark.parametrize("M,N,K,xdt,gs", CASES)
def test_masked_linear_equals_unmasked(M, N, K, xdt, gs):
    x, p, s = sparse_inputs(M, N, K, xdt, gs, 1)
    mask, zero = tl.block_mask(p)
    dense = tl.linear(x, p, s, gs, out_dtype=torch.float32)
    skip = tl.linear(x, p, s, gs, out_dtype=torch.float32, mask=mask)
    torch.cuda.synchronize()
    assert int(zero.item()) > 0
    if same_kernel(M, N, gs):
        assert torch.equal(dense, skip)
    else:
        check(dense, oracle_ref(x, p, s, gs), x, s, what=f"unmasked {M}x{N}x{K}")
    if N * K > 2048 * 2048:
        rows = np.unique(np.concatenate([np.arange(0, N, max(1, N // 83)), [N - 1]]))
        check(skip[:, rows], oracle_ref(x, p, s, gs, rows=rows), x, s, rows=rows,
              what=f"masked {M}x{N}x{K}")
    else:
        check(skip, oracle_ref(x, p, s, gs), x, s, what=f"masked {M}x{N}x{K}")


@pytest.mark.parametrize("M", [2, 12, 24, 40])
def test_masked_all_zero_rows_give_zero(M):
    """Whole CTAs whose every block is zero still write their (zero) outputs."""
    N, K = 512, 2048
    x = synth.activations(M, K, torch.bfloat16, 5, DEV)
    p = synth.packed_codes(N, K, 3, "cpu")
    p[128:384] = 0           # two 128-row blocks of zero codes
    p[384:448] = 0xFF        # half a block of reserved codes: still zero weights
    p = p.to(DEV)
    s = synth.scales(N, 0, 0.005, 0.05, 4, DEV)
    mask, _ = tl.block_mask(p)
    out = torch.full((M, N), 7.0, dtype=torch.float32, device=DEV)
    tl.linear(x, p, s, 0, out=out, out_dtype=torch.float32, mask=mask)
    dense = tl.linear(x, p, s, 0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out, dense)
    assert torch.all(out[:, 128:448] == 0)


@pytest.mark.parametrize("M,N,K,gs", [(1, 1000, 2048, 0), (8, 300, 4096, 128), (16, 700, 2048, 0),
                                      (24, 200, 1024, 0), (64, 384, 1024, 0)])
def test_masked_silu_mul_equals_unmasked(M, N, K, gs):
    x, p, s = sparse_inputs(M, 2 * N, K, torch.bfloat16, gs, 2)
    mask, _ = tl.block_mask(p)
    dense = tl.linear_silu_mul(x, p, s, gs, out_dtype=torch.float32)
    skip = tl.linear_silu_mul(x, p, s, gs, out_dtype=torch.float32, mask=mask)
    torch.cuda.synchronize()
    assert same_kernel(M, N, gs, gated=True) and torch.equal(dense, skip)
    h_ref, g_ref, u_ref = silu_refs(x, p, s, gs)
    check_silu(skip, h_ref, g_ref, u_ref, x, s, what=f"masked silu {M}x{N}x{K}")
