"""The sequence-parallel block on the GPU (LayerNorm in front of the TP-MLP, the
report's section 4.3) against the fp64 oracle: LayerNorm alone, the whole block
forward and backward, repeatability, and full-size rows at h8192."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import TOL_BF16, compare_full, compare_slices, rel, sample_indices, to_np
from tensor_transformer_mlp_tma_gb300 import inputs
from tensor_transformer_mlp_tma_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

STD = {"X": 1.0, "A": 0.05, "a": 0.1, "B": 0.05, "b": 0.1, "dZ": 1.0}
EPS = 1e-5
TOL = dict(TOL_BF16, Xn=1e-2, dX_in=2e-2, dgamma=2e-2, dbeta=2e-2)


def _ln_params(h, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    gamma = (1.0 + 0.2 * torch.randn(h, generator=g)).to(dtype)
    beta = (0.1 * torch.randn(h, generator=g)).to(dtype)
    return gamma, beta


def run_sp(inp, gamma, beta, t, algo=None, recompute=False):
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    algo = tpmlp.ALGO_DEFAULT if algo is None else algo
    d = {k: v.cuda() for k, v in inp.items()}
    T, h = d["X"].shape
    F = d["A"].shape[1]
    ctx = tpmlp.Context(T, h, F, t, d["X"].dtype, algo, layernorm=True, eps=EPS, recompute=recompute)
    Z = tpmlp.sp_forward(ctx, d["X"], gamma.cuda(), beta.cuda(), d["A"], d["a"], d["B"], d["b"])
    g = tpmlp.sp_backward(ctx, d["dZ"])
    torch.cuda.synchronize()
    assert tpmlp.check_device_status(ctx) == tpmlp.OK
    out = {"Xn": ctx.Xn, "H": ctx.H, "Y": ctx.Y.clone(), "Z": Z, "dY": ctx.dY.clone(), "dX": ctx.dXn.clone()}
    out.update(g)
    return out, ctx


@pytest.mark.parametrize("algo", ["tc", "simt"])
@pytest.mark.parametrize("T,h,F,t", [(300, 384, 1280, 2), (130, 264, 576, 3)])
def test_sp_block_matches_oracle(T, h, F, t, algo):
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    inp = inputs.make(T, h, F, "bf16", seed=T + 17 * t, std=STD)
    gamma, beta = _ln_params(h, 7)
    out, _ = run_sp(inp, gamma, beta, t, algo=tpmlp.ALGO_SIMT if algo == "simt" else None)
    ref = oracle.sp_forward_backward(inp["X"], gamma, beta, EPS, inp["A"], inp["a"], inp["B"], inp["b"],
                                     inp["dZ"], t)
    compare_full(out, ref, TOL)


# (T, h, dtype): every LayerNorm kernel path.  bf16 rows of 8-element chunks take
# the block-per-row kernels with 1 (h = 200), 2 (3000), 4 (8192) or 8 (12288)
# chunks per thread; longer rows (20000) the warp-per-row vector kernels; rows
# that are not whole 16-byte chunks (203) the scalar ones.  fp32 rows of
# 4-element chunks: 1 chunk (1000) and 8 chunks (8100).
LN_CASES = [(257, 8192, "bf16"), (33, 200, "bf16"), (9, 3000, "bf16"), (5, 12288, "bf16"), (3, 20000, "bf16"),
            (7, 203, "bf16"), (11, 1000, "f32"), (4, 8100, "f32")]


@pytest.mark.parametrize("T,h,dt", LN_CASES)
def test_layernorm_alone_matches_oracle(T, h, dt):
    """LayerNorm forward and backward on rows with a large common offset."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    tol_y, tol_g = (1e-2, 2e-2) if dt == "bf16" else (1e-5, 1e-5)
    g = torch.Generator().manual_seed(h)
    X = (torch.randn(T, h, generator=g) * 2 + 3).to(dtype)
    dXn = torch.randn(T, h, generator=g).to(dtype)
    gamma, beta = _ln_params(h, 11, dtype)
    ctx = tpmlp.Context(T, h, 64, 1, dtype, tpmlp.ALGO_SIMT, layernorm=True, eps=EPS)
    tpmlp.ln_forward(ctx, X.cuda(), gamma.cuda(), beta.cuda())
    bw = tpmlp.ln_backward(ctx, dXn.cuda())
    torch.cuda.synchronize()
    fw_ref = oracle.layernorm_forward(X, gamma, beta, EPS)
    bw_ref = oracle.layernorm_backward(dXn, X, gamma, EPS)
    assert rel(to_np(ctx.Xn), fw_ref["Y"]) <= tol_y
    assert rel(to_np(ctx.mean), fw_ref["mean"]) <= 1e-5
    assert rel(to_np(ctx.rstd), fw_ref["rstd"]) <= 1e-5
    for k in ("dX_in", "dgamma", "dbeta"):
        ref = bw_ref["dX" if k == "dX_in" else k]
        assert rel(to_np(bw[k]), ref) <= tol_g, k


@pytest.mark.parametrize("algo", ["tc", "simt"])
def test_sp_block_with_recompute(algo):
    """Recomputation (only H kept) with the LayerNorm in front: against the
    oracle, and bit-identical to the plain sequence-parallel block in every
    output but dB, which uses Y rebuilt from the stored bf16 H."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    a = tpmlp.ALGO_SIMT if algo == "simt" else None
    inp = inputs.make(300, 384, 1280, "bf16", seed=41, std=STD)
    gamma, beta = _ln_params(384, 13)
    rec, ctx = run_sp(inp, gamma, beta, 2, algo=a, recompute=True)
    assert tpmlp.saved_bytes(ctx.shape) == 300 * 1280 * 2
    ref = oracle.sp_forward_backward(inp["X"], gamma, beta, EPS, inp["A"], inp["a"], inp["B"], inp["b"],
                                     inp["dZ"], 2)
    compare_full(rec, ref, TOL)
    plain, _ = run_sp(inp, gamma, beta, 2, algo=a)
    for k in ("Xn", "Z", "H", "dY", "dX", "dX_in", "dgamma", "dbeta", "dA", "da", "db"):
        assert torch.equal(rec[k].view(torch.int16), plain[k].view(torch.int16)), k
    compare_full({"dB": rec["dB"]}, {"dB": to_np(plain["dB"])}, {"dB": 2e-2})


def test_sp_block_repeatable():
    inp = inputs.make(300, 384, 1280, "bf16", seed=5, std=STD)
    gamma, beta = _ln_params(384, 3)
    first, _ = run_sp(inp, gamma, beta, 2)
    for _ in range(4):
        again, _ = run_sp(inp, gamma, beta, 2)
        for k in ("Xn", "Z", "dX_in", "dgamma", "dbeta", "dA", "dB"):
            assert torch.equal(first[k].view(torch.int16), again[k].view(torch.int16)), k


def test_sp_full_size_rows_h8192():
    """h8192 workload with LayerNorm in front: Z and dX_in on sampled token rows,
    the MLP gradients on sampled ffn columns, against the exact slice oracle on
    the oracle's own normalised rows."""
    w = WORKLOADS["h8192"]
    t = 8
    inp = inputs.for_workload(w)
    gamma, beta = _ln_params(w.hidden, 9)
    out, _ = run_sp(inp, gamma, beta, t)
    ln = oracle.layernorm_forward(inp["X"], gamma, beta, EPS)
    T, F = w.tokens, w.ffn
    R = sample_indices(T, 24, seed=5, must=(0, T - 1))
    J = sample_indices(F, 64, seed=6, must=[0, F - 1])
    ref = oracle.slice_(ln["Y"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t, R, J)
    compare_slices(out, ref, R, J, TOL_BF16)
    dxin = oracle.layernorm_backward(ref["dXr"], oracle._f64(inp["X"])[R], gamma, EPS)["dX"]
    Rt = torch.as_tensor(R, device="cuda")
    assert rel(to_np(out["dX_in"][Rt]), dxin) <= 2e-2
    assert rel(to_np(out["Xn"][Rt]), ln["Y"][R]) <= 1e-2
