"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer work (unpack, pack, counts) must be bit-exact; the linear layer must
stay within the tolerance in tests/parity.py.  Inputs come from the seeded
generator in ternary_weight_linear_02_gb300.synth; no expected value is
produced by the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle
import ternary_weight_linear_02_gb300 as tl
from ternary_weight_linear_02_gb300 import synth
from ternary_weight_linear_02_gb300.workloads import CONFIGS

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


def layer_inputs(M, N, K, xdt, gs, seed, p_reserved=0.0, s_lo=0.005, s_hi=0.05):
    x, p, s = synth.layer(M, N, K, xdt, gs, s_lo, s_hi, ("parity", seed, M, N, K, str(xdt), gs),
                          "cpu", p_reserved)
    return x.to(DEV), p.to(DEV), s.to(DEV)


# ------------------------------------------------------------------ unpack / pack
@pytest.mark.parametrize("N,K", [(1, 4), (3, 12), (7, 64), (33, 100), (256, 1024), (129, 4100),
                                 (1000, 3584)])
def test_unpack_bit_exact(N, K):
    p = synth.packed_codes(N, K, synth.seed_for("unpack", N, K), "cpu", p_reserved=0.05)
    t_ref, res_ref = oracle.unpack(p.numpy())
    t, cnt = tl.unpack(p.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy(), t_ref)
    assert int(cnt.item()) == res_ref


def test_unpack_all_bytes():
    p = torch.arange(256, dtype=torch.uint8).reshape(64, 4)
    t_ref, res_ref = oracle.unpack(p.numpy())
    t, cnt = tl.unpack(p.to(DEV))
    assert np.array_equal(t.cpu().numpy(), t_ref)
    assert int(cnt.item()) == res_ref == 256


@pytest.mark.parametrize("N,K", [(1, 4), (5, 24), (64, 256), (129, 4100), (1000, 3584)])
def test_pack_bit_exact_and_invalid_count(N, K):
    g = torch.Generator().manual_seed(N * 131 + K)
    t = torch.randint(-1, 2, (N, K), dtype=torch.int8, generator=g)
    bad = torch.rand((N, K), generator=g) < 0.01
    t[bad] = torch.randint(2, 100, (int(bad.sum()),), generator=g, dtype=torch.int8)
    p_ref, inv_ref = oracle.pack(t.numpy())
    p, cnt = tl.pack(t.to(DEV))
    assert np.array_equal(p.cpu().numpy(), p_ref)
    assert int(cnt.item()) == inv_ref == int(bad.sum())


def test_pack_unpack_roundtrip():
    g = torch.Generator().manual_seed(3)
    t = torch.randint(-1, 2, (300, 640), dtype=torch.int8, generator=g).to(DEV)
    p, _ = tl.pack(t)
    back, res = tl.unpack(p)
    assert torch.equal(back, t)
    assert int(res.item()) == 0


# ------------------------------------------------------------------ linear, small
SMALL = [
    # M, N, K, x dtype, group size, out dtype
    (1, 64, 128, torch.float16, 128, torch.float32),
    (1, 70, 1152, torch.bfloat16, 0, torch.float32),
    (1, 200, 64, torch.float16, 0, torch.float32),
    (1, 1, 384, torch.bfloat16, 128, torch.float32),
    (3, 129, 384, torch.bfloat16, 128, torch.bfloat16),
    (4, 257, 192, torch.float16, 0, torch.float16),
    (8, 96, 1024, torch.bfloat16, 0, torch.float32),
    (9, 200, 640, torch.float16, 128, torch.float32),
    (16, 131, 2048, torch.bfloat16, 128, torch.bfloat16),
    (16, 64, 320, torch.bfloat16, 0, torch.float32),
    (17, 100, 256, torch.float16, 0, torch.float16),
    (24, 75, 1536, torch.bfloat16, 0, torch.float32),
    (32, 300, 1024, torch.float16, 128, torch.float32),
    (32, 64, 4096, torch.bfloat16, 128, torch.bfloat16),
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", SMALL)
def test_linear_skinny_small(M, N, K, xdt, gs, odt):
    x, p, s = layer_inputs(M, N, K, xdt, gs, 1, p_reserved=0.01)
    y = tl.linear(x, p, s, gs, out_dtype=odt, path="skinny")
    torch.cuda.synchronize()
    check(y, oracle_ref(x, p, s, gs), x, s, what=f"skinny {M}x{N}x{K}")


@pytest.mark.parametrize("gs", [0, 128])
@pytest.mark.parametrize("xdt", [torch.float16, torch.bfloat16])
def test_linear_every_byte_exact(xdt, gs):
    """Row n carries byte n in its first 4 weights (the rest 00); token 0 is
    x = (1, 3, 9, 27, 0, ...), s = 1: y[0, n] is the balanced-ternary value of
    the byte's four weights, an exact small integer."""
    K = 128
    p = torch.zeros((256, K // 4), dtype=torch.uint8)
    p[:, 0] = torch.arange(256, dtype=torch.uint8)
    x = torch.zeros((3, K), dtype=torch.float32)
    x[0, :4] = torch.tensor([1.0, 3.0, 9.0, 27.0])
    x[1, :4] = torch.tensor([-1.0, 0.5, 2.0, -4.0])
    x[2] = torch.randn(K, generator=torch.Generator().manual_seed(0))
    x = x.to(xdt)
    s = torch.ones((256,) if gs == 0 else (256, K // 128), dtype=torch.float16)
    want = oracle_ref(x, p, s, gs)
    y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), gs, out_dtype=torch.float32, path="skinny")
    y = y.cpu().double().numpy()
    assert np.array_equal(y[:2], want[:2])
    np.testing.assert_allclose(y[2], want[2], rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("gs", [0, 128])
def test_linear_closed_forms(gs):
    M, K = 5, 512
    rows = [0x55, 0xAA, 0x00, 0xFF]  # all +1, all -1, all 0, all reserved
    p = torch.tensor([[r] * (K // 4) for r in rows], dtype=torch.uint8)
    x = synth.activations(M, K, torch.bfloat16, 9)
    s = torch.full((4,) if gs == 0 else (4, K // 128), 0.03125, dtype=torch.float16)
    y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), gs, out_dtype=torch.float32, path="skinny")
    y = y.cpu().double()
    xs = x.double().sum(1)
    torch.testing.assert_close(y[:, 0], 0.03125 * xs, rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(y[:, 1], -0.03125 * xs, rtol=1e-5, atol=1e-6)
    assert torch.all(y[:, 2] == 0) and torch.all(y[:, 3] == 0)


def test_linear_three_d_input_and_k_zero():
    x, p, s = layer_inputs(6, 40, 256, torch.bfloat16, 0, 2)
    y = tl.linear(x.reshape(2, 3, 256), p, s)
    assert y.shape == (2, 3, 40)
    check(y.reshape(6, 40), oracle_ref(x, p, s, 0), x, s)
    z = tl.linear(torch.empty((4, 0), dtype=torch.float16, device=DEV),
                  torch.empty((8, 0), dtype=torch.uint8, device=DEV),
                  torch.ones(8, dtype=torch.float16, device=DEV))
    assert torch.count_nonzero(z) == 0


@pytest.mark.parametrize("M", [1, 12])
def test_linear_static_weights_flag(M):
    """TL_FLAG_STATIC_WEIGHTS only changes when weights are read, not results."""
    x, p, s = layer_inputs(M, 4096, 4096, torch.bfloat16, 0, 6)
    a = tl.linear(x, p, s, 0, out_dtype=torch.float32, static_weights=True)
    b = tl.linear(x, p, s, 0, out_dtype=torch.float32)
    assert torch.equal(a, b)
    check(a, oracle_ref(x, p, s, 0), x, s)


def test_linear_deterministic():
    x, p, s = layer_inputs(7, 3000, 4096, torch.bfloat16, 128, 4)
    a = tl.linear(x, p, s, 128, out_dtype=torch.float32)
    b = tl.linear(x, p, s, 128, out_dtype=torch.float32)
    assert torch.equal(a, b)


def test_linear_fused_shards_match_standalone():
    M, K = 4, 3584
    shards = [512, 128, 128]
    parts = [layer_inputs(M, n, K, torch.bfloat16, 0, 10 + i) for i, n in enumerate(shards)]
    x = parts[0][0]
    p = torch.cat([q[1] for q in parts])
    s = torch.cat([q[2] for q in parts])
    ys = tl.linear_fused(x, p, s, shards, out_dtype=torch.float32)
    for (xq, pq, sq), y in zip(parts, ys):
        alone = tl.linear(x, pq, sq, out_dtype=torch.float32)
        torch.testing.assert_close(y, alone, rtol=1e-5, atol=1e-6)


def test_linear_graph_capture():
    x, p, s = layer_inputs(4, 1024, 2048, torch.float16, 128, 5)
    tl.linear(x, p, s, 128)  # first call on the device outside capture
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        out = torch.empty((4, 1024), dtype=torch.float16, device=DEV)
        with torch.cuda.graph(g, stream=st):
            tl.linear(x, p, s, 128, out=out)
    g.replay()
    torch.cuda.synchronize()
    check(out, oracle_ref(x, p, s, 128), x, s)


TILE = [
    # M, N, K, x dtype, group size, out dtype
    (64, 128, 64, torch.bfloat16, 0, torch.float32),
    (64, 256, 256, torch.bfloat16, 0, torch.bfloat16),
    (100, 200, 320, torch.bfloat16, 0, torch.float32),
    (128, 384, 512, torch.float16, 0, torch.float16),
    (256, 128, 1024, torch.float16, 128, torch.float32),
    (300, 300, 768, torch.bfloat16, 128, torch.float32),
    (70, 130, 384, torch.float16, 128, torch.float16),
    (512, 256, 2048, torch.bfloat16, 0, torch.float32),
    (33, 129, 128, torch.bfloat16, 128, torch.bfloat16),
    (1, 64, 128, torch.float16, 0, torch.float32),
]


@pytest.mark.parametrize("M,N,K,xdt,gs,odt", TILE)
def test_linear_tile_small(M, N, K, xdt, gs, odt):
    x, p, s = layer_inputs(M, N, K, xdt, gs, 2, p_reserved=0.01)
    y = tl.linear(x, p, s, gs, out_dtype=odt, path="tile")
    torch.cuda.synchronize()
    check(y, oracle_ref(x, p, s, gs), x, s, what=f"tile {M}x{N}x{K}")
    assert tl.device_status() == 0


@pytest.mark.parametrize("gs", [0, 128])
def test_linear_tile_every_byte_exact(gs):
    K = 128
    p = torch.zeros((256, K // 4), dtype=torch.uint8)
    p[:, 0] = torch.arange(256, dtype=torch.uint8)
    x = torch.zeros((64, K), dtype=torch.float32)
    x[0, :4] = torch.tensor([1.0, 3.0, 9.0, 27.0])
    x = x.to(torch.float16)
    s = torch.ones((256,) if gs == 0 else (256, 1), dtype=torch.float16)
    want = oracle_ref(x, p, s, gs)
    y = tl.linear(x.to(DEV), p.to(DEV), s.to(DEV), gs, out_dtype=torch.float32, path="tile")
    assert np.array_equal(y.cpu().double().numpy(), want)


# ------------------------------------------------------------------ full-size configs
def sampled_rows(N, seed, k=48):
    g = np.random.default_rng(seed)
    rows = set(g.choice(N, size=min(k, N), replace=False).tolist())
    rows |= {0, N - 1, N // 2}
    return np.array(sorted(rows))


SKINNY_FULL = [(c.key, l, M) for c in CONFIGS.values() for l in c.layers for M in c.Ms if M <= 32]
TILE_FULL = [(c.key, l, M) for c in CONFIGS.values() for l in c.layers for M in c.Ms if M > 32]


@pytest.mark.parametrize("key,layer,M", SKINNY_FULL,
                         ids=[f"{k}-{l.name}-M{M}" for k, l, M in SKINNY_FULL])
def test_full_size_skinny_sampled(key, layer, M):
    cfg = CONFIGS[key]
    x, p, s = synth.layer(M, layer.N, layer.K, cfg.x_dtype, cfg.group_size, cfg.s_lo, cfg.s_hi,
                          (key, layer.name, 0), DEV, cfg.p_reserved)
    y = tl.linear(x, p, s, cfg.group_size, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = sampled_rows(layer.N, synth.seed_for(key, layer.name, M) & 0xFFFF)
    ref = oracle_ref(x, p, s, cfg.group_size, rows=rows)
    check(y[:, rows], ref, x, s, rows=rows, what=f"{key} {layer.name} M={M}")


@pytest.mark.parametrize("key,layer,M", TILE_FULL,
                         ids=[f"{k}-{l.name}-M{M}" for k, l, M in TILE_FULL])
def test_full_size_tile_sampled(key, layer, M):
    cfg = CONFIGS[key]
    x, p, s = synth.layer(M, layer.N, layer.K, cfg.x_dtype, cfg.group_size, cfg.s_lo, cfg.s_hi,
                          (key, layer.name, 0), DEV, cfg.p_reserved)
    y = tl.linear(x, p, s, cfg.group_size, out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = sampled_rows(layer.N, synth.seed_for(key, layer.name, M) & 0xFFFF, k=24)
    ref = oracle_ref(x, p, s, cfg.group_size, rows=rows)
    check(y[:, rows], ref, x, s, rows=rows, what=f"{key} {layer.name} M={M}")
    assert tl.device_status() == 0


# ------------------------------------------------------------------ tensor-parallel shards
@pytest.mark.parametrize("gs", [0, 128])
def test_tp_shards_reassemble(gs):
    """Per-shard calls rebuild the whole layer: a column split (rows of packed and
    scale cut together) concatenates; a K split's fp32 partials add up."""
    from ternary_weight_linear_02_gb300 import shard
    M, N, K = 8, 512, 2048
    x, p, s = layer_inputs(M, N, K, torch.bfloat16, gs, 7, p_reserved=0.01)
    ref = oracle_ref(x, p, s, gs)
    ys = [tl.linear(x, pi, si, gs, out_dtype=torch.float32)
          for pi, si in shard.split_n(p, s, [128, 256, 128])]
    check(torch.cat(ys, dim=1), ref, x, s, what="column shards")
    tot = None
    for pi, si, k0 in shard.split_k(p, s, shard.even_cuts(K, 4, 128 if gs else 64)):
        xs = x[:, k0:k0 + pi.shape[1] * 4].contiguous()
        part = tl.linear(xs, pi, si, gs, out_dtype=torch.float32)
        tot = part if tot is None else tot + part
    check(tot, ref, x, s, what="K shards")


# ------------------------------------------------------------------ 64-wide scale groups
G64 = [
    # M, N, K, x dtype, out dtype
    (1, 200, 512, torch.bfloat16, torch.float32),
    (4, 129, 1088, torch.float16, torch.float32),
    (16, 300, 4096, torch.bfloat16, torch.bfloat16),
    (33, 256, 640, torch.float16, torch.float16),
    (300, 384, 2048, torch.bfloat16, torch.float32),
]


@pytest.mark.parametrize("M,N,K,xdt,odt", G64)
def test_linear_group64(M, N, K, xdt, odt):
    x, p, s = layer_inputs(M, N, K, xdt, 64, 3, p_reserved=0.01)
    assert s.shape == (N, K // 64)
    y = tl.linear(x, p, s, 64, out_dtype=odt)
    torch.cuda.synchronize()
    check(y, oracle_ref(x, p, s, 64), x, s, what=f"g64 {M}x{N}x{K}")
    assert tl.device_status() == 0


# ------------------------------------------------------------------ 256-wide scale groups
G256 = [
    # M, N, K, x dtype, out dtype: mma.sync skinny (M <= 2), tcgen05 skinny (3..32),
    # tile (> 32); K = 2816 = 11 groups, so split-K ranges of 384 k end mid-group
    (1, 300, 2816, torch.bfloat16, torch.float32),
    (2, 4096, 2816, torch.float16, torch.float32),
    (4, 4096, 2816, torch.bfloat16, torch.float32),
    (16, 129, 1024, torch.float16, torch.bfloat16),
    (32, 256, 4096, torch.bfloat16, torch.float32),
    (33, 256, 768, torch.float16, torch.float16),
    (300, 384, 2048, torch.bfloat16, torch.float32),
]


@pytest.mark.parametrize("M,N,K,xdt,odt", G256)
def test_linear_group256(M, N, K, xdt, odt):
    x, p, s = layer_inputs(M, N, K, xdt, 256, 5, p_reserved=0.01)
    assert s.shape == (N, K // 256)
    y = tl.linear(x, p, s, 256, out_dtype=odt)
    torch.cuda.synchronize()
    check(y, oracle_ref(x, p, s, 256), x, s, what=f"g256 {M}x{N}x{K}")
    assert tl.device_status() == 0


# ------------------------------------------------------------------ SiLU-gated gate/up
SILU = [
    # M, N (output columns = gate rows = up rows), K, x dtype, out dtype, group size
    (1, 300, 1024, torch.bfloat16, torch.float32, 0),      # split K over 8 CTAs
    (2, 4096, 4096, torch.bfloat16, torch.float32, 0),     # M = 2 on the tcgen05 kernel
    (3, 64, 640, torch.float16, torch.float16, 0),         # split K 5: uneven pair slices
    (4, 1000, 2048, torch.float16, torch.float32, 128),
    (7, 100, 8192, torch.bfloat16, torch.float32, 128),    # ragged last pair tile
    (16, 11008, 4096, torch.bfloat16, torch.bfloat16, 0),  # 7B gate/up, no split K
    (32, 256, 4096, torch.bfloat16, torch.float32, 256),   # 32 tokens, 256-wide groups
    (4, 320, 1024, torch.float16, torch.float32, 64),      # 64-wide groups: tile kernel
    (33, 300, 1024, torch.bfloat16, torch.float32, 0),     # tile kernel from here on
    (100, 1000, 2048, torch.float16, torch.float16, 128),
    (300, 384, 2048, torch.bfloat16, torch.float32, 128),
    (1024, 512, 1024, torch.bfloat16, torch.bfloat16, 0),  # BN = 256 tiles
]


@pytest.mark.parametrize("M,N,K,xdt,odt,gs", SILU)
def test_linear_silu_mul(M, N, K, xdt, odt, gs):
    x, p, s = layer_inputs(M, 2 * N, K, xdt, gs, 6, p_reserved=0.001)
    h = tl.linear_silu_mul(x, p, s, gs, out_dtype=odt, static_weights=True)
    torch.cuda.synchronize()
    h_ref, g_ref, u_ref = silu_refs(x, p, s, gs)
    check_silu(h, h_ref, g_ref, u_ref, x, s, what=f"silu {M}x{N}x{K} g{gs}")
    assert tl.device_status() == 0


@pytest.mark.parametrize("M", [m for m in CONFIGS["stack7b"].Ms], ids=lambda m: f"stack7b-gate_up-M{m}")
def test_silu_mul_full_size_sampled(M):
    """The 7B gate/up layer (2 x 18944 rows, K = 3584) at every M of the stack:
    decode kernel for M <= 32, tile kernel above; output column j needs only
    rows j and 18944 + j, so the oracle runs on sampled pairs."""
    cfg = CONFIGS["stack7b"]
    layer = [l for l in cfg.layers if l.name == "gate_up"][0]
    n = layer.N // 2
    x, p, s = synth.layer(M, layer.N, layer.K, cfg.x_dtype, cfg.group_size, cfg.s_lo, cfg.s_hi,
                          ("stack7b", "gate_up_silu", 0), DEV, cfg.p_reserved)
    h = tl.linear_silu_mul(x, p, s, cfg.group_size, out_dtype=torch.float32)
    torch.cuda.synchronize()
    J = sampled_rows(n, synth.seed_for("stack7b", "silu", M) & 0xFFFF, k=24)
    idx = torch.as_tensor(np.concatenate([J, n + J]), device=DEV)
    ps, ss = p[idx].contiguous(), s[idx].contiguous()
    h_ref, g_ref, u_ref = silu_refs(x, ps, ss, cfg.group_size)
    check_silu(h[:, torch.as_tensor(J, device=DEV)], h_ref, g_ref, u_ref, x, ss,
               what=f"stack7b gate_up silu M={M}")
    assert tl.device_status() == 0


def test_silu_mul_matches_unfused_calls():
    """The fused call equals silu(g) * u formed from the plain kernel's fp32 g and u."""
    M, N, K = 5, 640, 3072
    x, p, s = layer_inputs(M, 2 * N, K, torch.bfloat16, 128, 7)
    h = tl.linear_silu_mul(x, p, s, 128, out_dtype=torch.float32)
    y = tl.linear(x, p, s, 128, out_dtype=torch.float32)
    g, u = y[:, :N], y[:, N:]
    want = torch.nn.functional.silu(g) * u
    torch.cuda.synchronize()
    assert torch.allclose(h, want, rtol=1e-5, atol=1e-6 * float(want.abs().max()))


def test_silu_mul_tile_matches_unfused_calls():
    M, N, K = 200, 384, 2048
    x, p, s = layer_inputs(M, 2 * N, K, torch.float16, 0, 9)
    h = tl.linear_silu_mul(x, p, s, 0, out_dtype=torch.float32)
    y = tl.linear(x, p, s, 0, out_dtype=torch.float32)
    want = torch.nn.functional.silu(y[:, :N]) * y[:, N:]
    torch.cuda.synchronize()
    assert torch.allclose(h, want, rtol=1e-5, atol=1e-6 * float(want.abs().max()))


def test_group64_skinny_path_refused_above_16_tokens():
    """64-wide groups run on the decode kernel up to M = 16; the tcgen05 skinny
    kernel (17..32 tokens) folds scales per 128 k and refuses them."""
    x, p, s = layer_inputs(20, 64, 256, torch.bfloat16, 64, 4)
    with pytest.raises(tl.TernaryError) as e:
        tl.linear(x, p, s, 64, path="skinny")
    assert e.value.status == 8  # TL_ERR_UNSUPPORTED
