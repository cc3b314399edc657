"""The column-sum entry point that allocates nothing (tpmlp_colsum_noalloc).

It serves callers that cannot call cudaMalloc -- a runtime whose device memory
is one arena owned by someone else, or a latency-critical path where an
allocation's implicit synchronisation or its failure is not acceptable -- by
keeping its fp32 partial sums in a fixed array inside the library instead of a
caller workspace.  Its results must match the bias gradients the regular entry
point (tpmlp_backward) computes with the same kernel, on two calls in a row (the
second call finds the first call's partials still in the shared array).

This file sorts last so that a failure here cannot hide a failure elsewhere; it
also passes when run alone in a fresh process (the first call does the set-up).
"""
import ctypes

import pytest
import torch

from gpu_cases import TOL_BF16, rel, run_gpu, to_np
from tensor_transformer_mlp_tma_gb300 import inputs

pytestmark = pytest.mark.gpu

STD = {"X": 1.0, "A": 0.05, "a": 0.1, "B": 0.05, "b": 0.1, "dZ": 1.0}


def _noalloc(tp, x, out):
    f = tp.lib.tpmlp_colsum_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p]
    dt = tp.BF16 if x.dtype == torch.bfloat16 else tp.F32
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(dt, x.data_ptr(), x.shape[0], x.shape[1], out.data_ptr(), stream)


def test_noalloc_colsum_matches_backward_bias_gradients():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    for T, h, F, t in [(300, 384, 1280, 2), (1000, 1024, 4096, 4)]:  # two calls in a row
        inp = inputs.make(T, h, F, "bf16", seed=T + F, std=STD)
        ref, ctx = run_gpu(inp, t)  # the regular entry point: db = 1^T dZ, da = 1^T dY
        dZ = inp["dZ"].cuda()
        db = torch.full((h,), float("nan"), dtype=torch.bfloat16, device="cuda")
        da = torch.full((F,), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(tpmlp, dZ, db) == tpmlp.OK, tpmlp.last_error()
        assert _noalloc(tpmlp, ctx.dY, da) == tpmlp.OK, tpmlp.last_error()
        torch.cuda.synchronize()
        assert rel(to_np(db), to_np(ref["db"])) <= TOL_BF16["db"]
        assert rel(to_np(da), to_np(ref["da"])) <= TOL_BF16["da"]


def test_noalloc_colsum_rejects_sizes_beyond_its_scratch():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    before = tpmlp.launch_count()
    x = torch.zeros((1, 1), dtype=torch.float32, device="cuda")
    f = tpmlp.lib.tpmlp_colsum_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p]
    # 2^21 columns need more fp32 partials than the fixed 2^20-float array holds;
    # the call is rejected before any pointer is touched.
    st = f(tpmlp.F32, x.data_ptr(), 16, 1 << 21, x.data_ptr(), None)
    assert st == tpmlp.ERR_UNSUPPORTED
    assert "scratch" in tpmlp.last_error()
    assert tpmlp.launch_count() == before
