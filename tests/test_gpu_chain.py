"""The mode the benchmark times, checked against the oracle.

The benchmark captures a whole stack of calls in one CUDA graph with
TL_FLAG_STATIC_WEIGHTS, so consecutive kernels overlap under programmatic
dependent launch: a kernel reads its weights before its predecessor has
finished and only waits for it before reading x and writing out.  Here a
4-layer chain in the same fused layout -- QKV, o, gate/up with the SiLU-gated
product, down reading that product, the next layer's o reading down's output --
is captured, replayed twice, and every call's output is compared with the
oracle evaluated on that call's actual input.  The shapes need split K and more
CTAs than one per SM, so CTAs of neighbouring kernels share SMs.  M = 1, 4, 16
run the decode kernel, M = 24 the tcgen05 skinny kernel, M = 64 and 300 the
tile kernel with split-K clusters.
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
DEPTH = 4
K_HID, N_QKV, N_FF = 2048, 3072, 5632   # hidden, fused QKV rows, gate (= up) rows


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tl.build()
    oracle.build()
    tl.load()


def weights(d, name, N, K, gs):
    p = synth.packed_codes(N, K, synth.seed_for("chain", d, name, "w"), DEV)
    s = synth.scales(N, 0 if gs == 0 else K // gs, 0.005, 0.05, synth.seed_for("chain", d, name, "s"),
                     DEV)
    return p, s


@pytest.mark.parametrize("gs", [0, 128])
@pytest.mark.parametrize("M", [1, 4, 16, 24, 64, 300])
def test_static_weight_chain_graph(M, gs):
    dt = torch.bfloat16
    W = [{"qkv": weights(d, "qkv", N_QKV, K_HID, gs), "o": weights(d, "o", K_HID, K_HID, gs),
          "gu": weights(d, "gu", 2 * N_FF, K_HID, gs), "down": weights(d, "down", K_HID, N_FF, gs)}
         for d in range(DEPTH)]
    x_qkv = [synth.activations(M, K_HID, dt, synth.seed_for("chain", d, "xq", M), DEV)
             for d in range(DEPTH)]
    x0 = synth.activations(M, K_HID, dt, synth.seed_for("chain", "x0", M), DEV)
    y_qkv = [torch.empty((M, N_QKV), dtype=dt, device=DEV) for _ in range(DEPTH)]
    y_o = [torch.empty((M, K_HID), dtype=dt, device=DEV) for _ in range(DEPTH)]
    h = [torch.empty((M, N_FF), dtype=dt, device=DEV) for _ in range(DEPTH)]
    y_dn = [torch.empty((M, K_HID), dtype=dt, device=DEV) for _ in range(DEPTH)]

    def chain():
        for d in range(DEPTH):
            w = W[d]
            tl.linear(x_qkv[d], *w["qkv"], gs, out=y_qkv[d], static_weights=True)
            tl.linear(x0 if d == 0 else y_dn[d - 1], *w["o"], gs, out=y_o[d], static_weights=True)
            tl.linear_silu_mul(y_o[d], *w["gu"], gs, out=h[d], static_weights=True)
            tl.linear(h[d], *w["down"], gs, out=y_dn[d], static_weights=True)

    chain()  # first calls outside capture
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            chain()
    for t in y_qkv + y_o + h + y_dn:
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    first = [t.clone() for t in y_qkv + y_o + h + y_dn]
    g.replay()
    torch.cuda.synchronize()
    assert tl.device_status(clear=True) == 0
    # the replays are deterministic
    for a, b in zip(first, y_qkv + y_o + h + y_dn):
        assert torch.equal(a, b)
    for d in range(DEPTH):
        w = W[d]
        check(y_qkv[d], oracle_ref(x_qkv[d], *w["qkv"], gs), x_qkv[d], w["qkv"][1],
              what=f"chain M={M} layer {d} qkv")
        xo = x0 if d == 0 else y_dn[d - 1]
        check(y_o[d], oracle_ref(xo, *w["o"], gs), xo, w["o"][1], what=f"chain M={M} layer {d} o")
        h_ref, g_ref, u_ref = silu_refs(y_o[d], *w["gu"], gs)
        check_silu(h[d], h_ref, g_ref, u_ref, y_o[d], w["gu"][1], what=f"chain M={M} layer {d} gate/up")
        check(y_dn[d], oracle_ref(h[d], *w["down"], gs), h[d], w["down"][1],
              what=f"chain M={M} layer {d} down")
        assert np.isfinite(y_dn[d].float().cpu().numpy()).all()
