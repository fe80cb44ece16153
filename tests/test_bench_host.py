"""Host-side logic of bench.py (no GPU): workload byte / flop counts, the call
layouts and the stack built from them."""
import dataclasses

import torch

import bench
from ternary_weight_linear_02_gb300.workloads import (CONFIGS, algorithmic_bytes, flops,
                                                      layer_calls, packed_bytes, scale_bytes)


def test_decode7b_byte_counts():
    cfg = CONFIGS["decode7b"]
    per_layer = 4 * 4096 * 4096 // 4 + 2 * 11008 * 4096 // 4 + 4096 * 11008 // 4
    assert packed_bytes(cfg) == 32 * per_layer
    assert scale_bytes(cfg) == 32 * 2 * (4 * 4096 + 2 * 11008 + 4096)
    M = 4
    xo = sum(2 * M * l.K + 2 * M * l.N for l in cfg.layers) * 32
    assert algorithmic_bytes(cfg, M) == packed_bytes(cfg) + scale_bytes(cfg) + xo
    assert flops(cfg, 1) == 8 * packed_bytes(cfg)  # 2*N*K per token = 8 * packed bytes


def test_stack7b_byte_counts():
    """The fused layout: QKV, o, gate/up (its gated output is [M, 18944]), down."""
    cfg = CONFIGS["stack7b"]
    per_layer = (4608 * 3584 + 3584 * 3584 + 37888 * 3584 + 3584 * 18944) // 4
    assert packed_bytes(cfg) == 28 * per_layer == 1631322112
    M = 16
    xo = 2 * M * (3584 + 4608 + 3584 + 3584 + 3584 + 18944 + 18944 + 3584)
    assert algorithmic_bytes(cfg, M) == packed_bytes(cfg) + scale_bytes(cfg) + 28 * xo
    assert [c.kind for c in layer_calls(cfg)] == ["linear", "linear", "silu_mul", "linear"]
    assert layer_calls(cfg)[3].src == 2


def test_rotation_exceeds_twice_l2():
    l2 = 129e6
    for key in CONFIGS:
        cfg = bench.bench_config(key)
        assert packed_bytes(cfg) >= 2 * l2, key


class _RecordingTL:
    """Stands in for the binding: checks shapes and records the calls."""

    def __init__(self):
        self.calls = []

    def linear(self, x, p, s, gs, out=None, static_weights=False):
        assert x.shape[1] == p.shape[1] * 4 and out.shape == (x.shape[0], p.shape[0])
        assert s.shape[0] == p.shape[0] and static_weights
        self.calls.append(("linear", p.shape[0], p.shape[1] * 4, x.data_ptr(), out.data_ptr()))

    def linear_silu_mul(self, x, p, s, gs, out=None, static_weights=False):
        assert x.shape[1] == p.shape[1] * 4 and out.shape == (x.shape[0], p.shape[0] // 2)
        assert s.shape[0] == p.shape[0] and static_weights
        self.calls.append(("silu", p.shape[0], p.shape[1] * 4, x.data_ptr(), out.data_ptr()))


def small_stack7b(depth=2):
    layers = (CONFIGS["stack7b"].layers[0].__class__("qkv", 192, 128, (128, 32, 32)),
              CONFIGS["stack7b"].layers[0].__class__("o", 128, 128),
              CONFIGS["stack7b"].layers[0].__class__("gate_up", 512, 128, (256, 256)),
              CONFIGS["stack7b"].layers[0].__class__("down", 128, 256))
    return dataclasses.replace(CONFIGS["stack7b"], layers=layers, depth=depth)


def test_fused_layout_chains_gated_product_into_down():
    cfg = small_stack7b()
    wl = bench.Workload(cfg, (2, 3), torch.device("cpu"))
    tl = _RecordingTL()
    wl.run(tl, 3)
    kinds = [(k, n, kk) for k, n, kk, _, _ in tl.calls]
    assert kinds == [("linear", 192, 128), ("linear", 128, 128), ("silu", 512, 128),
                     ("linear", 128, 256)] * cfg.depth
    for d in range(cfg.depth):
        gate_up, down = tl.calls[4 * d + 2], tl.calls[4 * d + 3]
        assert down[3] == gate_up[4]  # down reads the gated product
    # independent inputs live in one flat buffer per M, outputs in another
    xs = [c[3] for c in tl.calls if c[0] != "linear" or c[2] != 256]
    base = wl.xflat[3].data_ptr()
    assert all(base <= p < base + wl.xflat[3].numel() * 2 for p in xs)
    assert wl.calls_per_pass() == 4 * cfg.depth


def test_plain_layout_has_independent_inputs():
    cfg = dataclasses.replace(CONFIGS["layers27b"], depth=1,
                              layers=tuple(dataclasses.replace(l, N=64, K=128)
                                           for l in CONFIGS["layers27b"].layers))
    wl = bench.Workload(cfg, (1,), torch.device("cpu"))
    tl = _RecordingTL()
    wl.run(tl, 1)
    assert len(tl.calls) == 3 and len({c[3] for c in tl.calls}) == 3
