"""Seeded synthetic inputs for one sparse Mixture-of-Experts layer forward.

This module only draws random numbers. It holds none of the layer's arithmetic
(no routing, no capacity rule, no FFN), so that both the CUDA path and the CPU
oracle can consume exactly the same stored tensors without sharing any code.

Recipe (the same for every workload):
  * ``torch.Generator('cpu')`` seeded with ``seed`` (0 unless stated), drawing
    float32 standard normals in the fixed order x, W_g, W1, b1, W2, b2;
  * x ~ N(0, 1); W_g and W1 ~ N(0, 1/d); W2 ~ N(0, 1/d_ff) (fan-in scaling);
    b1 and b2 ~ N(0, 0.01), i.e. standard deviation 0.1;
  * the draws are then cast to the workload's storage dtype (fp32 or bf16);
  * an optional router logit bias is a closed form, not a draw: the "zipf"
    bias is b_e = 2*log(1/(e+1)) in float32 (natural log, e counted from 0).

Weights follow the nn.Linear [out, in] layout: W_g [N, d], W1 [N, d_ff, d],
b1 [N, d_ff], W2 [N, d, d_ff], b2 [N, d]; x is [T, d] row-major.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    """Shape and input law of one MoE-layer forward."""

    name: str
    dtype: str  # "f32" or "bf16": storage type of x and all weights
    T: int  # tokens in the batch
    d: int  # model width
    N: int  # experts
    k: int  # experts per token
    d_ff: int  # expert hidden width
    capacity_factor: float  # math.inf: no capacity limit
    router_bias: str = "none"  # "none" or "zipf"
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _wl(name, dtype, T, d, N, k, d_ff, cf, router_bias="none"):
    return Workload(name, dtype, T, d, N, k, d_ff, cf, router_bias)


# The five published workloads, named by what they are.
WORKLOADS = {
    w.name: w
    for w in (
        _wl("f32_T256_d64_N4_k1_dff256_cf1.25", "f32", 256, 64, 4, 1, 256, 1.25),
        _wl("bf16_T4096_d1024_N8_k2_dff4096_cf1.25", "bf16", 4096, 1024, 8, 2, 4096, 1.25),
        _wl("bf16_T16384_d4096_N8_k2_dff14336_nocap", "bf16", 16384, 4096, 8, 2, 14336, math.inf),
        _wl("bf16_T8192_d2048_N64_k2_dff1408_cf1.0_zipf", "bf16", 8192, 2048, 64, 2, 1408, 1.0, "zipf"),
        _wl("bf16_T64_d4096_N8_k2_dff14336_nocap", "bf16", 64, 4096, 8, 2, 14336, math.inf),
    )
}
SMALL_FP32 = "f32_T256_d64_N4_k1_dff256_cf1.25"
HEADLINE = "bf16_T4096_d1024_N8_k2_dff4096_cf1.25"
PREFILL = "bf16_T16384_d4096_N8_k2_dff14336_nocap"
SKEWED = "bf16_T8192_d2048_N64_k2_dff1408_cf1.0_zipf"
DECODE = "bf16_T64_d4096_N8_k2_dff14336_nocap"


def custom(T, d, d_ff, N, k, capacity_factor, dtype="bf16", router_bias="none", seed=0) -> Workload:
    """A workload of any shape with the same input law (used by parity tests).
    Argument order follows the C config: T, d, d_ff, N, k."""
    name = f"{dtype}_T{T}_d{d}_N{N}_k{k}_dff{d_ff}_cf{capacity_factor}_{router_bias}_s{seed}"
    return Workload(name, dtype, T, d, N, k, d_ff, capacity_factor, router_bias, seed)


def router_bias_values(kind: str, N: int):
    """Closed-form router logit bias (float32 [N]) or None."""
    if kind == "none":
        return None
    if kind == "zipf":
        return torch.tensor([2.0 * math.log(1.0 / (e + 1)) for e in range(N)], dtype=torch.float32)
    if kind.startswith("const:"):
        # "const:<e>:<v>": add v to expert e only (forces skewed routing in tests)
        _, e, v = kind.split(":")
        b = torch.zeros(N, dtype=torch.float32)
        b[int(e)] = float(v)
        return b
    raise ValueError(f"unknown router bias kind {kind!r}")


def draw(w: Workload, draw_x: bool = True) -> dict:
    """Draw the inputs of ``w`` as CPU tensors in the workload's dtype.

    Returns a dict with x, w_g, w1, b1, w2, b2 (storage dtype) and router_bias
    (float32 or None).  With ``draw_x=False`` x is still drawn (to keep the
    stream of draws identical) but discarded.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    dt = DTYPES[w.dtype]

    def normal(shape, std):
        t = torch.randn(*shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(dt)

    x = normal((w.T, w.d), 1.0)
    out = {
        "x": x if draw_x else None,
        "w_g": normal((w.N, w.d), 1.0 / math.sqrt(w.d)),
        "w1": normal((w.N, w.d_ff, w.d), 1.0 / math.sqrt(w.d)),
        "b1": normal((w.N, w.d_ff), 0.1),
        "w2": normal((w.N, w.d, w.d_ff), 1.0 / math.sqrt(w.d_ff)),
        "b2": normal((w.N, w.d), 0.1),
        "router_bias": router_bias_values(w.router_bias, w.N),
    }
    return out


def draw_shared(w: Workload, seed: int = 1) -> dict:
    """Weights of a shared (always-on) expert with the routed experts' shapes
    and laws: sw1 [d_ff, d], sb1 [d_ff], sw2 [d, d_ff], sb2 [d], from their own
    seeded generator (drawn in that order)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    dt = DTYPES[w.dtype]

    def normal(shape, std):
        return (torch.randn(*shape, generator=g, dtype=torch.float32) * std).to(dt)

    return {"sw1": normal((w.d_ff, w.d), 1.0 / math.sqrt(w.d)), "sb1": normal((w.d_ff,), 0.1),
            "sw2": normal((w.d, w.d_ff), 1.0 / math.sqrt(w.d_ff)), "sb2": normal((w.d,), 0.1)}


def draw_x_only(w: Workload, seed: int) -> torch.Tensor:
    """A fresh token batch of the workload's shape from another seed."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn(w.T, w.d, generator=g, dtype=torch.float32).to(DTYPES[w.dtype])


def as_f32_numpy(t):
    """Exact float32 copy of a stored tensor (bf16 and fp32 values are exact in fp32)."""
    if t is None:
        return None
    return t.to(torch.float32).contiguous().numpy()
