"""The seeded input recipe (CPU only): one CPU generator, fp32 normals drawn in
the fixed order X, A, a, B, b, dZ (attention: X, Wqkv, bqkv, Wo, bo, dZ), each
scaled by its standard deviation, then rounded to the workload dtype.  The CUDA
path and the oracle take their inputs from this one module, so the recipe is
pinned here by drawing the same stream by hand."""
import torch

from tensor_transformer_mlp_tma_gb300 import inputs
from tensor_transformer_mlp_tma_gb300.workloads import WORKLOADS


def _by_hand(shapes, stds, seed, dtype):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return {k: (torch.randn(shp, generator=g) * stds[k]).to(dtype) for k, shp in shapes}


def test_mlp_recipe():
    T, h, F = 5, 8, 32
    std = {"X": 1.0, "A": 0.02, "a": 0.3, "B": 0.05, "b": 0.1, "dZ": 2.0}
    got = inputs.make(T, h, F, "bf16", seed=7, std=std)
    want = _by_hand([("X", (T, h)), ("A", (h, F)), ("a", (F,)), ("B", (F, h)), ("b", (h,)), ("dZ", (T, h))],
                    std, 7, torch.bfloat16)
    assert list(got) == list(inputs.ORDER)
    for k in want:
        assert got[k].dtype == torch.bfloat16 and torch.equal(got[k], want[k]), k
    f32 = inputs.make(T, h, F, "f32", seed=7, std=std)
    assert all(f32[k].dtype == torch.float32 for k in f32)
    # bf16 values are the fp32 draws rounded to nearest even
    assert torch.equal(f32["A"].to(torch.bfloat16), got["A"])


def test_attention_recipe():
    T, h = 6, 8
    std = {"X": 1.0, "Wqkv": 0.02, "bqkv": 0.1, "Wo": 0.04, "bo": 0.2, "dZ": 1.0}
    got = inputs.make_attn(T, h, seed=3, std=std)
    want = _by_hand([("X", (T, h)), ("Wqkv", (h, 3 * h)), ("bqkv", (3 * h,)), ("Wo", (h, h)), ("bo", (h,)),
                     ("dZ", (T, h))], std, 3, torch.bfloat16)
    assert list(got) == list(inputs.ATTN_ORDER)
    for k in want:
        assert torch.equal(got[k], want[k]), k


def test_workload_defaults_and_zero_biases():
    w = WORKLOADS["h2048"]
    inp = inputs.for_workload(w, tokens=4)
    assert inp["X"].shape == (4, w.hidden) and inp["A"].shape == (w.hidden, w.ffn)
    # biases have std 0: drawn (the stream is unchanged) but all zero
    assert torch.count_nonzero(inp["a"]) == 0 and torch.count_nonzero(inp["b"]) == 0
    # same seed, same values; another seed, other values
    assert torch.equal(inputs.for_workload(w, tokens=4)["A"], inp["A"])
    assert not torch.equal(inputs.for_workload(w, seed=1, tokens=4)["A"], inp["A"])
