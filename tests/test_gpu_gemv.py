"""Decode shapes (M <= 16 tokens, path "skinny") against the oracle.

The automatic dispatch serves them with the register-fed decode kernel
(gemv.cuh) or, for M > 8 and for plain layers of 2049..4608 rows, with the
tcgen05 skinny kernel; 64-wide groups always run on the decode kernel, so its
two-token-tile form (M = 9..16) is covered by the group-64 cases here and by
the masked calls of test_gpu_mask.py.  Covers every scale mode (per channel,
64-, 128- and 256-wide groups), K ranges that end inside a 256-k stage or hold
fewer than one column per warp, ragged row counts, split K over 1..8 cluster
CTAs, every output dtype (fp32 for each mode and token-tile width: the
relative-L2 <= 1e-4 check of the accumulation), and the SiLU-gated gate/up
variant.
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
    x, p, s = synth.layer(M, N, K, xdt, gs, 0.005, 0.05, ("gemv", seed, M, N, K, str(xdt), gs),
                          "cpu", p_reserved)
    return x.to(DEV), p.to(DEV), s.to(DEV)


CASES = [
    # M, N, K, x dtype, group size, out dtype
    (1, 1, 64, BF16, 0, F32),          # one row, one 64-k column
    (1, 7, 128, F16, 64, F32),
    (1, 200, 192, BF16, 64, F32),      # three columns: some warps idle
    (1, 4096, 4096, BF16, 0, F32),     # q/o-shaped
    (1, 300, 18944, BF16, 0, F32),     # long K, split K over the cluster
    (1, 129, 1088, F16, 64, F32),      # 4.25 stages: the last stage holds one column
    (2, 64, 8192, BF16, 256, F32),     # one row block, split K 8
    (2, 1000, 2048, F16, 0, F16),
    (3, 33, 384, BF16, 128, BF16),
    (4, 11008, 4096, BF16, 0, F32),    # gate/up-shaped
    (4, 513, 1024, F16, 256, F32),
    (5, 300, 3584, BF16, 128, F32),
    (7, 257, 2816, F16, 256, F16),
    (8, 4608, 3584, BF16, 0, BF16),    # fused QKV-shaped
    (8, 96, 640, F16, 64, F32),
    (9, 200, 1024, BF16, 0, F32),      # two token tiles from here on
    (9, 31, 256, F16, 64, F32),
    (12, 129, 4096, BF16, 128, F32),
    (12, 3584, 3584, F16, 256, F32),
    (16, 4096, 11008, BF16, 0, F32),   # down-shaped
    (16, 75, 1536, BF16, 64, BF16),
    (16, 300, 2048, F16, 128, F16),
    (16, 64, 16384, BF16, 256, F32),   # split K 8 with two token tiles
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", CASES)
def test_gemv_against_oracle(M, N, K, xdt, gs, odt):
    x, p, s = inputs(M, N, K, xdt, gs, 1)
    y = tl.linear(x, p, s, gs, out_dtype=odt, path="skinny")
    torch.cuda.synchronize()
    if N * K > 4096 * 4096:  # large layers: sampled output columns
        rows = np.unique(np.concatenate([np.arange(0, N, max(1, N // 97)), [N - 1]]))
        check(y[:, rows], oracle_ref(x, p, s, gs, rows=rows), x, s, rows=rows,
              what=f"gemv {M}x{N}x{K} g{gs}")
    else:
        check(y, oracle_ref(x, p, s, gs), x, s, what=f"gemv {M}x{N}x{K} g{gs}")


@pytest.mark.parametrize("M", [1, 4, 8, 9, 16])
@pytest.mark.parametrize("gs", [0, 64, 128])
def test_gemv_every_byte_exact(M, gs):
    """Row n holds byte n in its first four weights; token 0 is x = (1, 3, 9, 27),
    s = 1, so y[0, n] is the balanced-ternary value of the byte: an exact
    integer that identifies all four decoded weights."""
    K = 256
    p = torch.zeros((256, K // 4), dtype=torch.uint8)
    p[:, 0] = torch.arange(256, dtype=torch.uint8)
    x = torch.zeros((M, K), dtype=torch.float32)
    x[0, :4] = torch.tensor([1.0, 3.0, 9.0, 27.0])
    if M > 1:
        x[M - 1, :4] = torch.tensor([27.0, -9.0, 3.0, -1.0])
    x = x.to(BF16)
    s = torch.ones((256,) if gs == 0 else (256, K // gs), dtype=F16)
    want = oracle_ref(x, p, s, gs)
    y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), gs, out_dtype=F32, path="skinny")
    assert np.array_equal(y.cpu().double().numpy(), want)


def test_gemv_deterministic_split_k():
    x, p, s = inputs(6, 200, 16384, BF16, 128, 2)
    a = tl.linear(x, p, s, 128, out_dtype=F32)
    b = tl.linear(x, p, s, 128, out_dtype=F32)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_gemv_token_rows_independent():
    """Rows of x are independent: a call on rows 0..8 equals those rows of a call
    on 16 tokens (different token tiles, same columns)."""
    x, p, s = inputs(16, 300, 2048, BF16, 0, 3)
    full = tl.linear(x, p, s, 0, out_dtype=F32)
    part = tl.linear(x[:9].contiguous(), p, s, 0, out_dtype=F32)
    torch.cuda.synchronize()
    torch.testing.assert_close(part, full[:9], rtol=0, atol=0)


SILU_CASES = [
    # M, N (gate rows = up rows = output columns), K, x dtype, group size, out dtype
    (1, 100, 1024, BF16, 0, F32),
    (1, 18944, 3584, BF16, 0, F32),    # the 7B gate/up
    (3, 64, 640, F16, 64, F32),
    (4, 1000, 2048, F16, 128, F32),
    (7, 100, 8192, BF16, 256, F32),    # split K
    (8, 300, 1024, BF16, 0, BF16),
    (9, 129, 2048, BF16, 128, F32),
    (16, 5632, 2048, BF16, 0, F32),
    (16, 77, 4096, F16, 64, F16),
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", SILU_CASES)
def test_gemv_silu_mul(M, N, K, xdt, gs, odt):
    x, p, s = inputs(M, 2 * N, K, xdt, gs, 4, p_reserved=0.001)
    h = tl.linear_silu_mul(x, p, s, gs, out_dtype=odt)
    torch.cuda.synchronize()
    if N > 2048:
        J = np.unique(np.concatenate([np.arange(0, N, max(1, N // 61)), [N - 1]]))
        idx = torch.as_tensor(np.concatenate([J, N + J]), device=DEV)
        ps, ss = p[idx].contiguous(), s[idx].contiguous()
        h_ref, g_ref, u_ref = silu_refs(x, ps, ss, gs)
        check_silu(h[:, torch.as_tensor(J, device=DEV)], h_ref, g_ref, u_ref, x, ss,
                   what=f"gemv silu {M}x{N}x{K} g{gs}")
    else:
        h_ref, g_ref, u_ref = silu_refs(x, p, s, gs)
        check_silu(h, h_ref, g_ref, u_ref, x, s, what=f"gemv silu {M}x{N}x{K} g{gs}")


def test_device_status_async_reads_zero():
    x, p, s = inputs(4, 256, 1024, BF16, 0, 5)
    tl.linear(x, p, s, 0)
    dst = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    tl.device_status_async(dst)
    torch.cuda.synchronize()
    assert int(dst.item()) == 0
