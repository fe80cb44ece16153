"""The persistent form of the tile kernel against the oracle.

One CTA per SM walks a list of tiles: 128 rows x 192 tokens with two TMEM
accumulators, the epilogue of one tile overlapping the main loop of the next
(tile mode 2), or 128 rows x 256 tokens with one accumulator (tile mode 3,
per-channel scales; group scales fall back to 192).  The module runs once per
mode; ternary_test_set_tile_mode makes every tile-kernel call use that form,
whatever its shape, so the cases cover: one tile and many tiles per CTA,
ragged M (partial last token tile) and N (partial last row block), every scale
mode (per channel; fp16 x with folded group scales; bf16 x with split group
scales; 32- to 256-wide groups), every output dtype, the SiLU-gated variant
(exchange through shared memory, 32 tokens at a time), the zero-block map, a
chained graph under programmatic dependent launch, and repeatability.
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


@pytest.fixture(scope="module", autouse=True, params=[2, 3], ids=["tiles192", "tiles256"])
def _persistent(request):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tl.build()
    oracle.build()
    lib = tl.load()
    lib.ternary_test_set_tile_mode(request.param)
    yield request.param
    lib.ternary_test_set_tile_mode(0)


def inputs(M, N, K, xdt, gs, seed, p_reserved=0.01):
    x, p, s = synth.layer(M, N, K, xdt, gs, 0.005, 0.05, ("persist", seed, M, N, K, str(xdt), gs),
                          "cpu", p_reserved)
    return x.to(DEV), p.to(DEV), s.to(DEV)


def sampled(N, k=61):
    return np.unique(np.concatenate([np.arange(0, N, max(1, N // k)), [N - 1]]))


CASES = [
    # M, N, K, x dtype, group size, out dtype
    (33, 128, 1024, BF16, 0, F32),        # one tile
    (192, 300, 2048, F16, 0, F32),        # exactly one token tile, ragged N
    (193, 129, 4096, BF16, 0, BF16),      # a second 192-token tile holding one token
    (256, 300, 2048, BF16, 0, F32),       # exactly one 256-token tile
    (257, 129, 2048, F16, 0, BF16),       # a second 256-token tile holding one token
    (400, 1000, 1024, BF16, 128, F32),    # bf16 x, split group scales
    (400, 1000, 1024, F16, 128, F16),     # fp16 x, folded group scales
    (300, 513, 2048, BF16, 32, F32),      # 32-wide groups
    (300, 513, 2048, F16, 64, F32),
    (600, 384, 4096, BF16, 256, F32),
    (1024, 8192, 1024, BF16, 0, BF16),    # 384 tiles: two or three per CTA
    (2048, 3584, 3584, BF16, 0, F32),     # the 7B o projection at M = 2048
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", CASES)
def test_persist_against_oracle(M, N, K, xdt, gs, odt):
    x, p, s = inputs(M, N, K, xdt, gs, 1)
    y = tl.linear(x, p, s, gs, out_dtype=odt, path="tile")
    torch.cuda.synchronize()
    if M * N * K > 2 ** 31:
        rows = sampled(N)
        check(y[:, rows], oracle_ref(x, p, s, gs, rows=rows), x, s, rows=rows,
              what=f"persist {M}x{N}x{K} g{gs}")
    else:
        check(y, oracle_ref(x, p, s, gs), x, s, what=f"persist {M}x{N}x{K} g{gs}")


SILU_CASES = [
    # M, N (gate rows = up rows = outputs), K, x dtype, group size, out dtype
    (40, 100, 1024, BF16, 0, F32),
    (193, 300, 2048, BF16, 0, BF16),
    (400, 129, 2048, F16, 128, F32),
    (300, 200, 1024, BF16, 32, F32),
    (2048, 18944, 3584, BF16, 0, BF16),   # the 7B gate/up at M = 2048 (sampled)
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", SILU_CASES)
def test_persist_silu_mul(M, N, K, xdt, gs, odt):
    x, p, s = inputs(M, 2 * N, K, xdt, gs, 2, p_reserved=0.001)
    h = tl.linear_silu_mul(x, p, s, gs, out_dtype=odt)
    torch.cuda.synchronize()
    if N > 2048:
        J = sampled(N, 29)
        idx = torch.as_tensor(np.concatenate([J, N + J]), device=DEV)
        ps, ss = p[idx].contiguous(), s[idx].contiguous()
        h_ref, g_ref, u_ref = silu_refs(x, ps, ss, gs)
        check_silu(h[:, torch.as_tensor(J, device=DEV)], h_ref, g_ref, u_ref, x, ss,
                   what=f"persist silu {M}x{N}x{K}")
    else:
        h_ref, g_ref, u_ref = silu_refs(x, p, s, gs)
        check_silu(h, h_ref, g_ref, u_ref, x, s, what=f"persist silu {M}x{N}x{K} g{gs}")


def test_persist_every_byte_exact():
    """Row n holds byte n at k = 1000..1003; token m = 200 (second token tile) has
    x = (1, 3, 9, 27) there, s = 1: y[200, n] is the byte's balanced-ternary value."""
    M, K = 300, 2048
    p = torch.zeros((256, K // 4), dtype=torch.uint8)
    p[:, 250] = torch.arange(256, dtype=torch.uint8)
    x = torch.zeros((M, K), dtype=F32)
    x[200, 1000:1004] = torch.tensor([1.0, 3.0, 9.0, 27.0])
    x = x.to(BF16)
    s = torch.ones(256, dtype=F16)
    want = oracle_ref(x, p, s, 0)
    y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), 0, out_dtype=F32, path="tile")
    assert np.array_equal(y.cpu().double().numpy(), want)


def test_persist_repeatable_and_one_tile_per_cta_form(_persistent):
    """Bit-identical across calls; the one-tile-per-CTA form (here with split K)
    meets the same bound against the oracle."""
    lib = tl.load()
    x, p, s = inputs(700, 1500, 2048, BF16, 0, 3)
    a = tl.linear(x, p, s, 0, out_dtype=F32, path="tile")
    b = tl.linear(x, p, s, 0, out_dtype=F32, path="tile")
    lib.ternary_test_set_tile_mode(1)
    try:
        c = tl.linear(x, p, s, 0, out_dtype=F32, path="tile")
        torch.cuda.synchronize()
    finally:
        lib.ternary_test_set_tile_mode(_persistent)
    assert torch.equal(a, b)
    want = oracle_ref(x, p, s, 0)
    check(a, want, x, s, what="persistent")
    check(c, want, x, s, what="one tile per CTA")


def test_persist_with_zero_block_map():
    x, p, s = inputs(500, 640, 4096, BF16, 0, 4)
    p = synth.block_sparse(p.cpu(), 0.5, 91).to(DEV)
    mask, _ = tl.block_mask(p)
    a = tl.linear(x, p, s, 0, out_dtype=F32)
    b = tl.linear(x, p, s, 0, out_dtype=F32, mask=mask)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    check(b, oracle_ref(x, p, s, 0), x, s, what="persist, masked")


def test_persist_chained_graph():
    """Persistent calls back to back in a PDL-chained static-weights graph, each
    reading its predecessor's output: o -> gate/up (gated) -> down -> o, M = 300."""
    M, H, F = 300, 1024, 2816
    dt = BF16
    w_o = (synth.packed_codes(H, H, 11, DEV), synth.scales(H, 0, 0.005, 0.05, 12, DEV))
    w_gu = (synth.packed_codes(2 * F, H, 13, DEV), synth.scales(2 * F, 0, 0.005, 0.05, 14, DEV))
    w_dn = (synth.packed_codes(H, F, 15, DEV), synth.scales(H, 0, 0.005, 0.05, 16, DEV))
    x0 = synth.activations(M, H, dt, 17, DEV)
    y_o = torch.empty((M, H), dtype=dt, device=DEV)
    h = torch.empty((M, F), dtype=dt, device=DEV)
    y_dn = torch.empty((M, H), dtype=dt, device=DEV)
    y_o2 = torch.empty((M, H), dtype=dt, device=DEV)

    def chain():
        tl.linear(x0, *w_o, 0, out=y_o, static_weights=True)
        tl.linear_silu_mul(y_o, *w_gu, 0, out=h, static_weights=True)
        tl.linear(h, *w_dn, 0, out=y_dn, static_weights=True)
        tl.linear(y_dn, *w_o, 0, out=y_o2, static_weights=True)

    chain()
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            chain()
    for t in (y_o, h, y_dn, y_o2):
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert tl.device_status(clear=True) == 0
    check(y_o, oracle_ref(x0, *w_o, 0), x0, w_o[1], what="chain o")
    h_ref, g_ref, u_ref = silu_refs(y_o, *w_gu, 0)
    check_silu(h, h_ref, g_ref, u_ref, y_o, w_gu[1], what="chain gate/up")
    check(y_dn, oracle_ref(h, *w_dn, 0), h, w_dn[1], what="chain down")
    check(y_o2, oracle_ref(y_dn, *w_o, 0), y_dn, w_o[1], what="chain o again")
