"""Repeated runs are bit-identical (fixed-order shard folds and column sums), and
the bounded-wait error path reports a timeout without hurting the context."""
import pytest
import torch

from gpu_cases import run_gpu
from tensor_transformer_mlp_tma_gb300 import inputs

pytestmark = pytest.mark.gpu

STD = {"X": 1.0, "A": 0.05, "a": 0.1, "B": 0.05, "b": 0.1, "dZ": 1.0}


def _bits(x):
    return x.contiguous().view(torch.int16) if x.dtype == torch.bfloat16 else x.contiguous().view(torch.int32)


@pytest.mark.parametrize("T,h,F,t", [(512, 1024, 4096, 4), (300, 384, 1280, 2)])
def test_ten_runs_bit_identical(T, h, F, t):
    inp = inputs.make(T, h, F, "bf16", seed=9, std=STD)
    first, _ = run_gpu(inp, t)
    for _ in range(9):
        again, _ = run_gpu(inp, t)
        for k in ("H", "Y", "Z", "dY", "dX", "dA", "da", "dB", "db"):
            assert torch.equal(_bits(first[k]), _bits(again[k])), k


@pytest.mark.parametrize("name,t", [("h8192", 8), ("h2048", 4)])
def test_full_size_runs_bit_identical(name, t):
    """The headline workload at full size (and the small h2048 one), in the
    benchmark's launch configuration: two runs on fresh buffers give the same
    bits in every output and intermediate, so the t-shard folds and the bias
    gradient sums have one fixed order per shape."""
    from tensor_transformer_mlp_tma_gb300.workloads import WORKLOADS
    inp = inputs.for_workload(WORKLOADS[name])
    first, _ = run_gpu(inp, t)
    first = {k: _bits(first[k]).cpu() for k in ("H", "Y", "Z", "dY", "dX", "dA", "da", "dB", "db")}
    torch.cuda.empty_cache()
    again, _ = run_gpu(inp, t)
    for k, v in first.items():
        assert torch.equal(v, _bits(again[k]).cpu()), k


def test_timeout_probe_reports_and_context_survives():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    assert tpmlp.debug_timeout_probe(ws, 2_000_000) == tpmlp.OK  # 2 ms limit
    assert tpmlp.check_device_status(ws) == tpmlp.ERR_TIMEOUT
    assert tpmlp.check_device_status(ws) == tpmlp.OK  # read-and-clear
    # the context still works: a normal call after the timeout succeeds
    out, _ = run_gpu(inputs.make(128, 256, 512, "bf16", seed=1, std=STD), 2)
    assert torch.isfinite(out["Z"].float()).all()
