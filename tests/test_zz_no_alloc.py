"""The column-sum entry point that allocates nothing (tpmlp_colsum_noalloc).

It serves callers that cannot call cudaMalloc -- a runtime whose device memory
is one arena owned by someone else, or a latency-critical path where an
allocation's implicit synchronisation or its failure is not acceptable -- by
keeping its fp32 partial sums in a fixed array inside the library instead of a
caller workspace.

What is checked, on two shapes run larger first (so the smaller call finds the
larger call's extra partials still in the shared array) and each called twice in
a row:
- the column sums of dZ and of dY against the oracle's db = 1^T dZ and
  da = 1^T dY, within the bias-gradient tolerance;
- the two calls on the same input give the same bits;
- the same bits as the bias gradients of tpmlp_backward on the FFMA path, which
  runs the same two-pass column sum with a caller workspace.

This file sorts last so that a failure here cannot hide a failure elsewhere; it
also passes when run alone in a fresh process (the first call does the set-up).
"""
import ctypes

import pytest
import torch

import oracle
from gpu_cases import TOL_BF16, rel, run_gpu, to_np
from tensor_transformer_mlp_tma_gb300 import inputs

pytestmark = pytest.mark.gpu

STD = {"X": 1.0, "A": 0.05, "a": 0.1, "B": 0.05, "b": 0.1, "dZ": 1.0}


def _fn(tp):
    f = tp.lib.tpmlp_colsum_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p]
    return f


def _noalloc(tp, x):
    """Column sums of the 2-D device tensor x through the C ABI; a fresh output
    filled with NaN first, so an unwritten entry cannot pass."""
    out = torch.full((x.shape[1],), float("nan"), dtype=x.dtype, device=x.device)
    dt = tp.BF16 if x.dtype == torch.bfloat16 else tp.F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = _fn(tp)(dt, x.data_ptr(), x.shape[0], x.shape[1], out.data_ptr(), stream)
    assert st == tp.OK, tp.last_error()
    return out


def _bits(x):
    return x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)


def test_noalloc_colsum_against_oracle_and_ffma_backward():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    for T, h, F, t in [(1000, 1024, 4096, 4), (300, 384, 1280, 2)]:  # larger first
        inp = inputs.make(T, h, F, "bf16", seed=T + F, std=STD)
        ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
        simt, ctx = run_gpu(inp, t, algo=tpmlp.ALGO_SIMT)  # db, da by the two-pass column sum
        dZ = inp["dZ"].cuda()
        dY = ctx.dY  # the FFMA path's dY, whose column sums are its da
        db1, da1 = _noalloc(tpmlp, dZ), _noalloc(tpmlp, dY)
        db2, da2 = _noalloc(tpmlp, dZ), _noalloc(tpmlp, dY)
        torch.cuda.synchronize()
        assert rel(to_np(db1), ref["db"]) <= TOL_BF16["db"]
        assert rel(to_np(da1), ref["da"]) <= TOL_BF16["da"]
        assert torch.equal(_bits(db1), _bits(db2)) and torch.equal(_bits(da1), _bits(da2))
        assert torch.equal(_bits(db1), _bits(simt["db"]))
        assert torch.equal(_bits(da1), _bits(simt["da"]))


def test_noalloc_colsum_fp32_exact_small_integers():
    """fp32 columns of small integers: every partial and total is exact, so the
    sums equal the integer column sums whatever the chunking."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    g = torch.Generator().manual_seed(5)
    x = torch.randint(-8, 9, (777, 300), generator=g).float()
    got = _noalloc(tpmlp, x.cuda())
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), x.sum(0))


def test_noalloc_colsum_rejects_sizes_beyond_its_scratch():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    before = tpmlp.launch_count()
    x = torch.zeros((1, 1), dtype=torch.float32, device="cuda")
    # 2^21 columns need more fp32 partials than the fixed 2^20-float array holds;
    # the call is rejected before any pointer is touched.
    st = _fn(tpmlp)(tpmlp.F32, x.data_ptr(), 16, 1 << 21, x.data_ptr(), None)
    assert st == tpmlp.ERR_UNSUPPORTED
    assert "scratch" in tpmlp.last_error()
    assert tpmlp.launch_count() == before
