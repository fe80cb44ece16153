"""Host-side logic of bench.py (no GPU): workload byte / flop counts and the
fused-layout stack built from the same weights."""
import dataclasses

import torch

import bench
from ternary_weight_linear_02_gb300.workloads import (CONFIGS, algorithmic_bytes, flops,
                                                      packed_bytes, scale_bytes)


def test_decode7b_byte_counts():
    cfg = CONFIGS["decode7b"]
    per_layer = 4 * 4096 * 4096 // 4 + 2 * 11008 * 4096 // 4 + 4096 * 11008 // 4
    assert packed_bytes(cfg) == 32 * per_layer
    assert scale_bytes(cfg) == 32 * 2 * (4 * 4096 + 2 * 11008 + 4096)
    M = 4
    xo = sum(2 * M * l.K + 2 * M * l.N for l in cfg.layers) * 32
    assert algorithmic_bytes(cfg, M) == packed_bytes(cfg) + scale_bytes(cfg) + xo
    assert flops(cfg, 1) == 8 * packed_bytes(cfg)  # 2*N*K per token = 8 * packed bytes


class _RecordingTL:
    """Stands in for the binding: checks shapes and records the calls."""

    def __init__(self):
        self.calls = []

    def linear(self, x, p, s, gs, out=None, static_weights=False):
        assert x.shape[1] == p.shape[1] * 4 and out.shape == (x.shape[0], p.shape[0])
        assert s.shape[0] == p.shape[0] and static_weights
        self.calls.append(("linear", p.shape[0], p.shape[1] * 4))

    def linear_silu_mul(self, x, p, s, gs, out=None, static_weights=False):
        assert x.shape[1] == p.shape[1] * 4 and out.shape == (x.shape[0], p.shape[0] // 2)
        assert s.shape[0] == p.shape[0] and static_weights
        self.calls.append(("silu", p.shape[0], p.shape[1] * 4))


def test_fused_layout_reuses_the_same_weights():
    cfg = dataclasses.replace(CONFIGS["decode7b"], depth=2)
    st = bench.Stack(cfg, (2,), torch.device("cpu"))
    fs = bench.FusedStack(st)
    assert fs.ok and fs.calls_per_layer() == 4
    ix = {l.name: i for i, l in enumerate(cfg.layers)}
    for d in range(cfg.depth):
        (qkv, o, gu, dn) = fs.w[d]
        w = st.w[d]
        assert torch.equal(qkv[0], torch.cat([w[ix[n]][0] for n in "qkv"]))
        assert torch.equal(gu[0], torch.cat([w[ix["gate"]][0], w[ix["up"]][0]]))
        assert torch.equal(gu[1], torch.cat([w[ix["gate"]][1], w[ix["up"]][1]]))
        assert o[0] is w[ix["o"]][0] and dn[0] is w[ix["down"]][0]
        # same packed bytes as the 7-call layer
        assert sum(t[0].numel() for t in fs.w[d]) == sum(p.numel() for p, _ in w)
    tl = _RecordingTL()
    fs.run_m(tl, 2)
    assert tl.calls == [("linear", 12288, 4096), ("linear", 4096, 4096), ("silu", 22016, 4096),
                        ("linear", 4096, 11008)] * cfg.depth


def test_fused_layout_needs_all_projections():
    cfg = dataclasses.replace(CONFIGS["layers27b"], depth=1)
    st = bench.Stack(cfg, (1,), torch.device("cpu"))
    assert not bench.FusedStack(st).ok
