"""The layer shapes of the pages' workloads, reproduced as synthetic configs.

No checkpoint is available; each config fixes only shapes, dtypes, the scale
mode and the input distributions (see ``synth``):

``linear1k``: one linear, M=1, N=K=1024, fp16 x, per-128-group scales U[0.01,0.05]
   (the ~0.6B embedding model of "三元量化模型接入vLLM：从逆向加载到Kernel优化的完整实战").
``decode7b``: 7B-shaped decode set: (N,K) = (4096,4096) q/k/v/o, (11008,4096) gate/up,
   (4096,11008) down; M in {1,4,8,16}; bf16 x; per-channel scales
   U[0.005,0.05] (the Qwen2.5-7B ternary-in-vLLM write-up, §1.1, §1.3).
   As a decode step it runs through a 32-layer stack (a 7B model's depth),
   every layer with its own weights, so each step streams 1.62 GB of packed
   weights -- far more than the 129 MB L2.
``embed06b``: ~0.6B embedding model: hidden 1024, intermediate 3072, 28 layers of
   q/k/v/o (1024x1024), gate/up (3072x1024), down (1024x3072); M in
   {64,256,1024}; fp16 x; per-128-group scales U[0.005,0.05]; about 0.1% of
   bytes carry one reserved 11 field.
``layers27b``: 27B-class layers: (5120,5120), (17408,5120), (5120,17408); M in {1,8,32};
   bf16 x; per-128-group scales U[0.005,0.05].
``stack7b``: 7B-shaped decode / prefill stack: 28 layers of fused QKV (N=3584+512+512,
   K=3584), o (3584x3584), fused gate/up (N=2*18944, K=3584), down
   (N=3584, K=18944); M in {1,16,64,256,2048}; bf16 x; per-channel scales
   U[0.005,0.05].
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Layer:
    name: str
    N: int
    K: int
    shards: tuple = ()      # fused layer: row counts of the shards, in order


@dataclass(frozen=True)
class Config:
    key: str
    title: str
    layers: tuple           # one model layer (a list of projections)
    depth: int              # number of model layers in a step
    Ms: tuple
    x_dtype: torch.dtype
    group_size: int         # 0 = per channel, 128 = per group
    s_lo: float
    s_hi: float
    p_reserved: float = 0.0
    layout: str = "plain"   # "plain": one call per projection, each on its own input;
                            # "fused_mlp": QKV and o as plain calls, gate/up with the
                            # SiLU-gated product fused, down reading that product
    rotate: int = 1         # weight sets cycled by the benchmark so a pass exceeds 2x L2


@dataclass(frozen=True)
class Call:
    """One kernel call of a model layer.  kind: "linear" or "silu_mul";
    layer: index into Config.layers; src: -1 for an input of its own, else the
    index of the call (same model layer) whose output it reads."""
    kind: str
    layer: int
    src: int = -1


def layer_calls(cfg: "Config") -> tuple:
    """The calls of one model layer in the config's layout."""
    if cfg.layout == "fused_mlp":
        ix = {l.name: i for i, l in enumerate(cfg.layers)}
        return (Call("linear", ix["qkv"]), Call("linear", ix["o"]),
                Call("silu_mul", ix["gate_up"]), Call("linear", ix["down"], src=2))
    return tuple(Call("linear", i) for i in range(len(cfg.layers)))


def out_cols(cfg: "Config", c: Call) -> int:
    n = cfg.layers[c.layer].N
    return n // 2 if c.kind == "silu_mul" else n


CONFIGS = {
    "linear1k": Config(
        "linear1k", "single ternary linear M=1 K=N=1024 fp16 g128",
        (Layer("linear", 1024, 1024),), 1, (1,), torch.float16, 128, 0.01, 0.05, rotate=1024),
    "decode7b": Config(
        "decode7b", "7B-shaped decode set (4096/11008), per-channel, bf16",
        (Layer("q", 4096, 4096), Layer("k", 4096, 4096), Layer("v", 4096, 4096),
         Layer("o", 4096, 4096), Layer("gate", 11008, 4096),
         Layer("up", 11008, 4096), Layer("down", 4096, 11008)),
        32, (1, 4, 8, 16), torch.bfloat16, 0, 0.005, 0.05),
    "embed06b": Config(
        "embed06b", "0.6B embedding model batch, 28 layers, fp16 g128, reserved codes",
        (Layer("q", 1024, 1024), Layer("k", 1024, 1024), Layer("v", 1024, 1024),
         Layer("o", 1024, 1024), Layer("gate", 3072, 1024), Layer("up", 3072, 1024),
         Layer("down", 1024, 3072)),
        28, (64, 256, 1024), torch.float16, 128, 0.005, 0.05, 0.001, rotate=3),
    "layers27b": Config(
        "layers27b", "27B-class layers (5120/17408), bf16 g128",
        (Layer("attn", 5120, 5120), Layer("up", 17408, 5120),
         Layer("down", 5120, 17408)),
        1, (1, 8, 32), torch.bfloat16, 128, 0.005, 0.05, rotate=6),
    "stack7b": Config(
        "stack7b", "7B-shaped 28-layer stack, fused QKV and gate/up, per-channel, bf16",
        (Layer("qkv", 4608, 3584, (3584, 512, 512)), Layer("o", 3584, 3584),
         Layer("gate_up", 37888, 3584, (18944, 18944)), Layer("down", 3584, 18944)),
        28, (1, 16, 64, 256, 2048), torch.bfloat16, 0, 0.005, 0.05, layout="fused_mlp"),
}


def packed_bytes(cfg: Config) -> int:
    """Packed-weight bytes of one pass over the config's stack (one M)."""
    return cfg.depth * sum(cfg.layers[c.layer].N * cfg.layers[c.layer].K // 4
                           for c in layer_calls(cfg))


def scale_bytes(cfg: Config) -> int:
    def per(l):
        return 2 * l.N if cfg.group_size == 0 else 2 * l.N * l.K // cfg.group_size
    return cfg.depth * sum(per(cfg.layers[c.layer]) for c in layer_calls(cfg))


def call_bytes(cfg: Config, c: Call, M: int) -> int:
    """Algorithmic bytes of one call: packed + scales + x + out."""
    l = cfg.layers[c.layer]
    sc = 2 * l.N if cfg.group_size == 0 else 2 * l.N * l.K // cfg.group_size
    return l.N * l.K // 4 + sc + 2 * M * l.K + 2 * M * out_cols(cfg, c)


def algorithmic_bytes(cfg: Config, M: int) -> int:
    """Bytes one pass must move at minimum: packed + scales + x + out."""
    return cfg.depth * sum(call_bytes(cfg, c, M) for c in layer_calls(cfg))


def flops(cfg: Config, M: int) -> int:
    """Effective 2*M*N*K flops of one pass (N = every stacked weight row)."""
    return cfg.depth * sum(2 * M * cfg.layers[c.layer].N * cfg.layers[c.layer].K
                           for c in layer_calls(cfg))
