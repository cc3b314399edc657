"""Seeded synthetic inputs for the TP-MLP block and the TP self-attention block.

This module holds no arithmetic of the method: it only draws Gaussian tensors.
It is the one module that both the CUDA path (tests, benchmark) and the CPU
oracle take their inputs from, so that both see bit-identical values.

Recipe: a CPU ``torch.Generator`` seeded with ``seed``; fp32 normals drawn in the
fixed order X, A, a, B, b, dZ, each as one ``torch.randn(shape) * std``; then
rounded to the workload dtype (round-to-nearest-even for bf16).  The attention
block draws X, Wqkv, bqkv, Wo, bo, dZ in that order the same way.
"""
from __future__ import annotations

import torch

ORDER = ("X", "A", "a", "B", "b", "dZ")

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DT[name]


def shapes(tokens: int, hidden: int, ffn: int) -> dict:
    return {"X": (tokens, hidden), "A": (hidden, ffn), "a": (ffn,),
            "B": (ffn, hidden), "b": (hidden,), "dZ": (tokens, hidden)}


def make(tokens: int, hidden: int, ffn: int, dtype: str = "bf16", seed: int = 0,
         std: dict | None = None) -> dict:
    """Draw X, A, a, B, b, dZ on the CPU in the given dtype.

    ``std`` maps a tensor name to its standard deviation (default 1 for X and dZ,
    0.02 for A and B, 0 for the biases)."""
    s = {"X": 1.0, "A": 0.02, "a": 0.0, "B": 0.02, "b": 0.0, "dZ": 1.0}
    if std:
        s.update(std)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {}
    for name, shape in shapes(tokens, hidden, ffn).items():
        v = torch.randn(shape, generator=g, dtype=torch.float32)
        if s[name] != 1.0:
            v.mul_(s[name])
        out[name] = v.to(_DT[dtype])
    return out


def for_workload(w, seed: int = 0, tokens: int | None = None) -> dict:
    """Inputs of a :class:`~.workloads.Workload` (optionally with fewer tokens)."""
    return make(tokens if tokens is not None else w.tokens, w.hidden, w.ffn, w.dtype, seed,
                {"X": w.std_X, "A": w.std_A, "a": w.std_a, "B": w.std_B, "b": w.std_b,
                 "dZ": w.std_dZ})


ATTN_ORDER = ("X", "Wqkv", "bqkv", "Wo", "bo", "dZ")


def attn_shapes(tokens: int, hidden: int) -> dict:
    return {"X": (tokens, hidden), "Wqkv": (hidden, 3 * hidden), "bqkv": (3 * hidden,),
            "Wo": (hidden, hidden), "bo": (hidden,), "dZ": (tokens, hidden)}


def make_attn(tokens: int, hidden: int, seed: int = 0, std: dict | None = None) -> dict:
    """Draw X, Wqkv, bqkv, Wo, bo, dZ on the CPU in bf16 (default std 1 for X and
    dZ, 0.02 for the weights, 0 for the biases)."""
    s = {"X": 1.0, "Wqkv": 0.02, "bqkv": 0.0, "Wo": 0.02, "bo": 0.0, "dZ": 1.0}
    if std:
        s.update(std)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {}
    for name, shape in attn_shapes(tokens, hidden).items():
        v = torch.randn(shape, generator=g, dtype=torch.float32)
        if s[name] != 1.0:
            v.mul_(s[name])
        out[name] = v.to(torch.bfloat16)
    return out
