"""Seeded synthetic inputs for the two-stage MoE expert computation.

This module only draws random numbers (torch generators) and shapes them into
the workloads the aiter pages measure: bf16 activations, top-k routing and
fp32 expert weights. It holds none of the method's arithmetic: no format
encoding, no quantisation, no GEMM, no activation function. Both the CUDA
path's tests/bench and the CPU oracle take their inputs from here; weights are
quantised to MXFP4 by whichever side needs them.

Recipe (each draw from its own seeded torch.Generator):
  x            ~ N(0, 1), rounded to bf16, shape [T, H]
  routing      "softmax_topk": logits ~ N(0,1) [T,E] -> softmax -> top-k
                 (ties: lower expert id first) -> weights renormalised over k
               "uniform": K distinct experts per token, uniformly without
                 replacement; weights = softmax of K N(0,1) logits
               "zipf": expert popularity p_e ~ rank_e^-s with ranks a seeded
                 permutation of 1..E; K distinct experts per token by
                 Gumbel-top-k on log p_e; weights = softmax of K N(0,1) logits
  w13[e]       ~ N(0, 1/sqrt(H)), fp32 [2I, H]  (rows 0..I-1 gate, I..2I-1 up)
  w2[e]        ~ N(0, 1/sqrt(I)), fp32 [H, I]
Every expert's weights come from a generator seeded by (seed, expert), so any
subset of experts can be drawn on its own.
"""
from dataclasses import dataclass, field
from typing import List

import torch

_MIX = 0x9E3779B97F4A7C15


def sub_seed(seed: int, stream: int, index: int = 0) -> int:
    """Deterministic seed of one random stream (x, routing, w13[e], w2[e])."""
    v = (seed * _MIX + stream * 0xBF58476D1CE4E5B9 + index * 0x94D049BB133111EB) & ((1 << 64) - 1)
    v ^= v >> 31
    return v & ((1 << 62) - 1)


def _gen(seed: int, stream: int, index: int = 0, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, stream, index))
    return g


STREAM_X, STREAM_ROUTING, STREAM_W13, STREAM_W2, STREAM_ROUTING_W = 1, 2, 3, 4, 5


@dataclass
class MoEConfig:
    name: str
    tokens: List[int]
    hidden: int
    inter: int
    experts: int
    topk: int
    a_dtype: str            # "bf16" | "fp8" | "fp4"
    acts: List[str]         # activations the workload runs
    routing: str            # "softmax_topk" | "uniform" | "zipf"
    seed: int
    beta: float = 4.0
    linear_beta: float = 25.0
    zipf_s: float = 1.1
    notes: str = field(default="")


CONFIGS = {
    "tiny": MoEConfig("tiny", [16], 256, 128, 8, 2, "bf16", ["situv2"], "softmax_topk", 0,
                      notes="tiny a16w4 parity case"),
    "tp8_decode": MoEConfig("tp8_decode", [1, 4, 16, 64], 3584, 384, 896, 16, "bf16", ["situv2"],
                            "uniform", 123, notes="Kimi-K3 TP8-shard decode a16w4"),
    "tp8_a8": MoEConfig("tp8_a8", [256, 1024, 4096], 3584, 384, 896, 16, "fp8", ["situv2"],
                        "uniform", 123, notes="TP8 shape a8w4"),
    "ep_wide": MoEConfig("ep_wide", [1, 128, 2048, 8192], 3584, 3072, 112, 16, "fp8", ["situv2"],
                         "uniform", 7, notes="EP-shard wide-inter a8w4"),
    "tp8_a4_zipf": MoEConfig("tp8_a4_zipf", [8192, 16384, 32768], 3584, 384, 896, 16, "fp4",
                             ["silu", "situv2"], "zipf", 42, notes="TP8 a4w4 prefill, Zipf(1.1) routing"),
}


def make_x(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, STREAM_X, 0, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_router_logits(T: int, E: int, seed: int, device="cpu") -> torch.Tensor:
    """Router logits ~ N(0, 1), fp32 [T, E]: the draw the "softmax_topk" routing starts from."""
    g = _gen(seed, STREAM_ROUTING, 0, device)
    return torch.randn(T, E, generator=g, device=device, dtype=torch.float32)


def make_routing(T: int, E: int, K: int, kind: str, seed: int, zipf_s: float = 1.1, device="cpu"):
    """Returns (topk_ids int32 [T,K], topk_weights fp32 [T,K])."""
    if kind == "softmax_topk":
        logits = make_router_logits(T, E, seed, device)
        probs = torch.softmax(logits, dim=-1)
        order = torch.sort(-probs, dim=-1, stable=True).indices[:, :K]
        w = torch.gather(probs, 1, order)
        w = w / w.sum(dim=-1, keepdim=True)
        return order.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()
    g = _gen(seed, STREAM_ROUTING, 0, device)
    if kind == "uniform":
        keys = torch.rand(T, E, generator=g, device=device)
        ids = torch.sort(keys, dim=-1, stable=True).indices[:, :K]
    elif kind == "zipf":
        ranks = torch.randperm(E, generator=g, device=device).to(torch.float64) + 1.0
        logp = -zipf_s * torch.log(ranks)
        u = torch.rand(T, E, generator=g, device=device, dtype=torch.float64)
        gumbel = -torch.log(-torch.log(u))
        scores = logp.unsqueeze(0) + gumbel
        ids = torch.sort(-scores, dim=-1, stable=True).indices[:, :K]
    else:
        raise ValueError(kind)
    gw = _gen(seed, STREAM_ROUTING_W, 0, device)
    w = torch.softmax(torch.randn(T, K, generator=gw, device=device, dtype=torch.float32), dim=-1)
    return ids.to(torch.int32).contiguous(), w.contiguous()


def expert_w13(e: int, H: int, I: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, STREAM_W13, e, device)
    return torch.randn(2 * I, H, generator=g, device=device, dtype=torch.float32) * (H ** -0.5)


def expert_w2(e: int, H: int, I: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, STREAM_W2, e, device)
    return torch.randn(H, I, generator=g, device=device, dtype=torch.float32) * (I ** -0.5)
