"""Seeded random shapes and unit counts against the oracle (GPU).

The tile schedules depend on the shape and on the number of units the GEMMs
run on: wide tiles and their split last wave, odd waves walking K downwards,
the M-walk tile order, and the complementary M-tile pairs of the causal
per-head products.  Each case draws a ragged shape within the library's rules
(h and F multiples of 8, shards of F on 64-element k-blocks) and a unit count
from 1 to 9 (TPMLP_MAX_UNITS), so that many waves, split tails, odd and even
unit counts and partial double rounds occur, and compares every output in
full with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import TOL_BF16, compare_full, rel, run_gpu, to_np
from tensor_transformer_mlp_tma_gb300 import inputs

pytestmark = pytest.mark.gpu

STD = {"X": 1.0, "A": 0.05, "a": 0.1, "B": 0.05, "b": 0.1, "dZ": 1.0}


def mlp_case(i):
    r = np.random.default_rng(1000 + i)
    t = int(r.choice([1, 2, 3, 4, 8]))
    F = t * 64 * int(r.integers(1, 6)) if t > 1 else 8 * int(r.integers(8, 160))
    h = 8 * int(r.integers(8, 100))
    T = int(r.integers(1, 700))
    units = int(r.integers(1, 10))
    return T, h, F, t, units


@pytest.mark.parametrize("i", range(10))
def test_random_mlp_shapes(i, monkeypatch):
    T, h, F, t, units = mlp_case(i)
    monkeypatch.setenv("TPMLP_MAX_UNITS", str(units))
    inp = inputs.make(T, h, F, "bf16", seed=i, std=STD)
    out, _ = run_gpu(inp, t)
    ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
    compare_full(out, ref, TOL_BF16)


ATTN_TOL = {"QKV": 1e-2, "O": 2e-2, "Z": 2e-2, "dX": 3e-2, "dWqkv": 3e-2, "dbqkv": 3e-2, "dWo": 3e-2,
            "dbo": 3e-2}


def attn_case(i):
    r = np.random.default_rng(2000 + i)
    d = int(r.choice([64, 128]))
    t = int(r.choice([1, 2, 4]))
    heads = t * int(r.integers(1, 3))
    nb = int(r.integers(1, 3))
    S = 8 * int(r.integers(16, 160))
    units = int(r.integers(1, 10))
    return nb, S, heads * d, heads, t, units


@pytest.mark.parametrize("i", range(6))
def test_random_attention_shapes(i, monkeypatch):
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    nb, S, h, heads, t, units = attn_case(i)
    monkeypatch.setenv("TPMLP_MAX_UNITS", str(units))
    inp = inputs.make_attn(nb * S, h, 50 + i, {"X": 1.0, "Wqkv": 0.05, "bqkv": 0.1, "Wo": 0.04, "bo": 0.1,
                                               "dZ": 1.0})
    d = {k: v.cuda() for k, v in inp.items()}
    ctx = tpmlp.AttnContext(nb, S, h, heads, t)
    Z = tpmlp.attn_forward(ctx, d["X"], d["Wqkv"], d["bqkv"], d["Wo"], d["bo"])
    g = tpmlp.attn_backward(ctx, d["dZ"])
    torch.cuda.synchronize()
    assert tpmlp.check_device_status(ctx) == tpmlp.OK
    out = {"QKV": ctx.QKV, "O": ctx.O, "Z": Z}
    out.update(g)
    f = {k: v.double().numpy() for k, v in inp.items()}
    ref = oracle.attn_forward_backward(f["X"], f["Wqkv"], f["bqkv"], f["Wo"], f["bo"], f["dZ"], nb, heads, t)
    errs = {k: rel(to_np(out[k]), ref[k].reshape(to_np(out[k]).shape)) for k in ATTN_TOL}
    assert all(v <= ATTN_TOL[k] for k, v in errs.items()), errs
