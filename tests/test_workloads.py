"""The named workloads and the FLOP counts every reported TFLOP/s divides by
(CPU only).

The MLP counts two GEMMs of 2*T*h*F per forward and three times that for
forward + backward; biases, GeLU and column sums are not counted.  The
attention counts the QKV and output projections and, per head, the two
products over the causal lower triangle only.  Both are checked here against
figures worked out independently: the tabulated per-workload counts, and a
brute-force count of the multiply-adds of a causal product on small shapes."""
import math

import pytest

from tensor_transformer_mlp_tma_gb300.workloads import ATTN_WORKLOADS, HEADLINE, WORKLOADS

# (T, h, F, shard counts, dtype, fwd+bwd FLOP to three significant figures)
TABLE = {
    "tiny-fp32": (128, 256, 1024, (2,), "f32", 4.03e8),
    "h2048": (2048, 2048, 8192, (1, 2, 4), "bf16", 4.12e11),
    "h4096": (8192, 4096, 16384, (8,), "bf16", 6.60e12),
    "h8192": (4096, 8192, 32768, (8,), "bf16", 1.32e13),
    "h12288-b1": (2048, 12288, 49152, (8,), "bf16", 1.48e13),
}


@pytest.mark.parametrize("name", sorted(TABLE))
def test_mlp_workloads(name):
    T, h, F, shards, dtype, flops = TABLE[name]
    w = WORKLOADS[name]
    assert (w.tokens, w.hidden, w.ffn, w.shards, w.dtype) == (T, h, F, shards, dtype)
    assert F == 4 * h
    assert w.flops_fwd == 2 * (2 * T * h * F)
    assert math.isclose(w.flops_fwd_bwd, flops, rel_tol=5e-3)
    for t in shards:  # shard boundaries on whole 64-wide k-blocks (bf16 tensor-core path)
        assert F % t == 0 and (dtype == "f32" or (F // t) % 64 == 0)


def test_sweep_scales_with_the_microbatch():
    base = WORKLOADS["h12288-b1"].flops_fwd_bwd
    for b in (2, 4, 8):
        assert WORKLOADS["h12288-b%d" % b].flops_fwd_bwd == b * base


def test_headline_distributions():
    w = WORKLOADS[HEADLINE]
    assert HEADLINE == "h8192"
    assert (w.std_X, w.std_A, w.std_a, w.std_b, w.std_dZ) == (1.0, 0.02, 0.0, 0.0, 1.0)
    assert math.isclose(w.std_B, 0.02 / math.sqrt(192))
    tiny = WORKLOADS["tiny-fp32"]
    assert (tiny.std_a, tiny.std_b) == (0.01, 0.01)


def _causal_products_brute(nb, S, h, heads):
    """FLOP of Q K^T and P V over the causal lower triangle, one multiply-add
    at a time: query r of every head meets keys 0..r, each a d-long dot product
    for the score and d multiply-adds for the output."""
    d = h // heads
    macs = 0
    for _ in range(nb * heads):
        for r in range(S):
            macs += (r + 1) * d * 2
    return 2 * macs


@pytest.mark.parametrize("nb,S,h,heads", [(1, 1, 64, 1), (2, 5, 128, 2), (3, 16, 256, 4)])
def test_attention_flops_against_a_brute_force_count(nb, S, h, heads):
    import dataclasses
    w = dataclasses.replace(ATTN_WORKLOADS["attn-h4096"], batch=nb, seq=S, hidden=h, heads=heads)
    T = nb * S
    projections = 2 * T * h * (3 * h) + 2 * T * h * h
    assert w.flops_fwd == projections + _causal_products_brute(nb, S, h, heads)
    assert w.flops_fwd_bwd == 3 * w.flops_fwd


def test_attention_workloads():
    for name, (nb, S, h, heads, t) in {"attn-h4096": (4, 2048, 4096, 32, 8),
                                       "attn-h8192": (2, 2048, 8192, 64, 8)}.items():
        w = ATTN_WORKLOADS[name]
        assert (w.batch, w.seq, w.hidden, w.heads, w.t) == (nb, S, h, heads, t)
        assert h // heads == 128 and heads % t == 0
    assert math.isclose(ATTN_WORKLOADS["attn-h8192"].flops_fwd_bwd, 7.0096e12, rel_tol=1e-4)
