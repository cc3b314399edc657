"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes are compared element by element on every output; they span several
256x256 (CTA pair) and 128x256 (single CTA) tiles and leave ragged tails in
every dimension.  The named workloads
are run at full size in the same launch configuration as the benchmark and
compared on seeded rows and ffn columns against the exact slice oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import TOL_BF16, TOL_F32, compare_full, compare_slices, run_gpu, sample_indices, to_np
from tensor_transformer_mlp_tma_gb300 import inputs
from tensor_transformer_mlp_tma_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

STD = {"X": 1.0, "A": 0.05, "a": 0.1, "B": 0.05, "b": 0.1, "dZ": 1.0}

# (T, h, F, t): ragged M, N and K tails, t = 1..16 including a non power of two
SMALL = [
    (300, 384, 1280, 2),   # M = 2 tiles + 44 rows; Z is 1.5 N tiles; shards of 640
    (128, 256, 512, 1),    # exactly one tile, no shards
    (200, 200, 520, 1),    # K = h = 200: ragged k-block; N = F = 520 ragged
    (257, 512, 1024, 4),   # one row past two tiles; shards of 256
    (64, 256, 2048, 8),    # fewer tokens than one tile
    (130, 264, 576, 3),    # t = 3 (shards of 192); h = 264 ragged
    (1, 128, 1024, 16),    # one token, 16 shards of 64
]


@pytest.mark.parametrize("T,h,F,t", SMALL)
def test_tensor_core_path_matches_oracle(T, h, F, t):
    inp = inputs.make(T, h, F, "bf16", seed=T + h + F + t, std=STD)
    out, _ = run_gpu(inp, t)
    ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
    compare_full(out, ref, TOL_BF16)


@pytest.mark.parametrize("env", [{"TPMLP_CTA_PAIR": "0"}, {"TPMLP_MN4": "0"}, {"TPMLP_RASTER": "n:3"},
                                 {"TPMLP_RASTER": "m:1", "TPMLP_CTA_PAIR": "0"}, {"TPMLP_PDL": "0"},
                                 {"TPMLP_WIDE": "0"}, {"TPMLP_WIDE_TAIL": "0"}, {"TPMLP_MAX_UNITS": "4"},
                                 {"TPMLP_SERPENTINE": "0"}, {"TPMLP_MAX_UNITS": "3"},
                                 {"TPMLP_MAX_UNITS": "3", "TPMLP_RASTER": "n:2"},
                                 {"TPMLP_MAX_UNITS": "2", "TPMLP_WIDE_TAIL": "0", "TPMLP_MN4": "0"}])
@pytest.mark.parametrize("T,h,F,t", [(300, 384, 1280, 2), (257, 512, 1024, 4)])
def test_tuning_knobs_keep_parity(T, h, F, t, env, monkeypatch):
    """The library's tuning knobs (single-CTA 128 x 256 tiles, per-block maps
    for MN-major operands, forced tile orders, launches without programmatic
    dependence, 256 x 256 instead of 256 x 512 tiles, the wide tiles' last wave
    kept whole, few persistent units so that each runs several wide tiles and
    split half-width tiles in one launch) change the schedule, not the result."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    inp = inputs.make(T, h, F, "bf16", seed=T + h + len(env), std=STD)
    out, _ = run_gpu(inp, t)
    ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
    compare_full(out, ref, TOL_BF16)


@pytest.mark.parametrize("T,h,F,t", [(300, 384, 1280, 2), (1000, 1024, 4096, 4)])
def test_wide_and_square_tiles_agree(T, h, F, t, monkeypatch):
    """256 x 512 tiles (default) against 256 x 256 tiles (TPMLP_WIDE=0): all
    within tolerance of the oracle, and within bf16 rounding of each other.
    With every wave walking K upwards (TPMLP_SERPENTINE=0) the two accumulate
    every output element over k in the same order with the same MMA shape, so
    they are expected to agree bit for bit; the test reports whether they do
    but requires only the tolerance."""
    inp = inputs.make(T, h, F, "bf16", seed=T + 5 * t, std=STD)
    ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
    default, _ = run_gpu(inp, t)
    compare_full(default, ref, TOL_BF16)
    monkeypatch.setenv("TPMLP_SERPENTINE", "0")
    wide, _ = run_gpu(inp, t)
    compare_full(wide, ref, TOL_BF16)
    monkeypatch.setenv("TPMLP_WIDE", "0")
    square, _ = run_gpu(inp, t)
    compare_full(square, ref, TOL_BF16)
    same = {k: bool(torch.equal(wide[k].view(torch.int16), square[k].view(torch.int16)))
            for k in ("H", "Y", "Z", "dY", "dX", "dA", "da", "dB", "db")}
    print("wide vs 256 x 256 bit-identical:", same)
    compare_full(wide, {k: to_np(v) for k, v in square.items() if k in TOL_BF16}, TOL_BF16)


def test_fp32_workload_matches_oracle():
    w = WORKLOADS["tiny-fp32"]
    for t in w.shards:
        inp = inputs.for_workload(w)
        out, _ = run_gpu(inp, t)
        ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
        compare_full(out, ref, TOL_F32)


@pytest.mark.parametrize("T,h,F,t", [(300, 384, 1280, 2), (129, 136, 192, 2)])
def test_simt_path_matches_oracle(T, h, F, t):
    """The FFMA kernels on bf16 inputs (no 64-element shard rule: F/t = 96 works)."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    inp = inputs.make(T, h, F, "bf16", seed=7, std=STD)
    out, _ = run_gpu(inp, t, algo=tpmlp.ALGO_SIMT)
    ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
    compare_full(out, ref, TOL_BF16)


def test_tensor_core_matches_simt_mid_size():
    """Full-tensor cross-check of the two GPU paths at a size with many tiles."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    inp = inputs.make(1000, 1024, 4096, "bf16", seed=3, std=STD)
    tc, _ = run_gpu(inp, 4)
    si, _ = run_gpu(inp, 4, algo=tpmlp.ALGO_SIMT)
    compare_full(tc, {k: to_np(v) for k, v in si.items()}, TOL_BF16)


def test_special_cases_exact():
    """X = 0 gives dA = 0 exactly; A = 0, a = 0 give H = Y = 0, Z = b, dX = dB = 0 exactly."""
    T, h, F, t = 200, 256, 1024, 2
    inp = inputs.make(T, h, F, "bf16", seed=11, std=STD)
    x0 = dict(inp, X=torch.zeros_like(inp["X"]))
    out, _ = run_gpu(x0, t)
    assert torch.count_nonzero(out["dA"]).item() == 0
    ref = oracle.forward_backward(x0["X"], x0["A"], x0["a"], x0["B"], x0["b"], x0["dZ"], t)
    compare_full(out, ref, TOL_BF16)
    a0 = dict(inp, A=torch.zeros_like(inp["A"]), a=torch.zeros_like(inp["a"]))
    out, _ = run_gpu(a0, t)
    assert torch.count_nonzero(out["H"]).item() == 0
    assert torch.count_nonzero(out["Y"]).item() == 0
    assert torch.equal(out["Z"].cpu(), inp["b"].expand(T, h))
    assert torch.count_nonzero(out["dX"]).item() == 0
    assert torch.count_nonzero(out["dB"]).item() == 0


def test_empty_batch():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    h, F, t = 256, 1024, 2
    inp = inputs.make(0, h, F, "bf16", seed=1, std=STD)
    d = {k: v.cuda() for k, v in inp.items()}
    ctx = tpmlp.Context(0, h, F, t, torch.bfloat16)
    Z = tpmlp.forward(ctx, d["X"], d["A"], d["a"], d["B"], d["b"])
    assert Z.shape == (0, h)
    outs = {n: torch.full(s, float("nan"), dtype=torch.bfloat16, device="cuda")
            for n, s in (("dA", (h, F)), ("da", (F,)), ("dB", (F, h)), ("db", (h,)))}
    dX = torch.empty((0, h), dtype=torch.bfloat16, device="cuda")
    g = tpmlp.backward(ctx, d["dZ"], dX=dX, **outs)
    torch.cuda.synchronize()
    for n in outs:
        assert torch.count_nonzero(g[n]).item() == 0


def test_unsupported_shard_size_is_rejected_without_launch():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    inp = inputs.make(64, 128, 192, "bf16", seed=1, std=STD)
    d = {k: v.cuda() for k, v in inp.items()}
    ctx = tpmlp.Context(64, 128, 192, 2, torch.bfloat16)
    before = tpmlp.launch_count()
    with pytest.raises(tpmlp.TpmlpError) as e:
        tpmlp.forward(ctx, d["X"], d["A"], d["a"], d["B"], d["b"])
    assert e.value.status == tpmlp.ERR_UNSUPPORTED
    assert tpmlp.launch_count() == before


def test_misaligned_pointer_is_rejected():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    T, h, F = 64, 128, 256
    inp = inputs.make(T, h, F, "bf16", seed=1, std=STD)
    d = {k: v.cuda() for k, v in inp.items()}
    big = torch.zeros(T * h + 1, dtype=torch.bfloat16, device="cuda")
    Xoff = big[1:].view(T, h)  # 2-byte offset
    ctx = tpmlp.Context(T, h, F, 1, torch.bfloat16)
    with pytest.raises(tpmlp.TpmlpError) as e:
        tpmlp.forward(ctx, Xoff, d["A"], d["a"], d["B"], d["b"])
    assert e.value.status == tpmlp.ERR_UNSUPPORTED


def test_golden_worked_example_fp32():
    """The hand-worked two-shard example of tests/golden/worked_example_t2.txt on
    the fp32 FFMA path: every output matches the hand-derived values to fp32
    rounding (they are small integers and halves)."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    from oracle_pins import read_golden
    g = read_golden("worked_example_t2.txt")
    d = {k: torch.tensor(g[k], dtype=torch.float32, device="cuda") for k in ("X", "A", "B", "dZ")}
    a = torch.tensor(g["a"].ravel(), dtype=torch.float32, device="cuda")
    b = torch.tensor(g["b"].ravel(), dtype=torch.float32, device="cuda")
    ctx = tpmlp.Context(g["T"], g["h"], g["F"], g["t"], torch.float32)
    Z = tpmlp.forward(ctx, d["X"], d["A"], a, d["B"], b)
    out = tpmlp.backward(ctx, d["dZ"])
    torch.cuda.synchronize()
    assert tpmlp.check_device_status(ctx) == tpmlp.OK
    got = {"H": ctx.H, "Y": ctx.Y, "Z": Z, "dY": ctx.dY, "dA": out["dA"], "dB": out["dB"], "dX": out["dX"],
           "da": out["da"][None, :], "db": out["db"][None, :]}
    for k, v in got.items():
        assert np.allclose(to_np(v), g[k], rtol=0, atol=1e-5), (k, to_np(v), g[k])


def test_inference_forward_without_saved():
    """tpmlp_forward with saved == NULL: Z is bit-identical to the training
    forward, and Y is left in the workspace's dY region."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    T, h, F, t = 300, 384, 1280, 2
    inp = inputs.make(T, h, F, "bf16", seed=77, std=STD)
    d = {k: v.cuda() for k, v in inp.items()}
    ctx = tpmlp.Context(T, h, F, t, torch.bfloat16)
    Z_train = tpmlp.forward(ctx, d["X"], d["A"], d["a"], d["B"], d["b"]).clone()
    Y_train = ctx.Y.clone()
    ctx2 = tpmlp.Context(T, h, F, t, torch.bfloat16)
    Z_inf = tpmlp.forward(ctx2, d["X"], d["A"], d["a"], d["B"], d["b"], inference=True)
    torch.cuda.synchronize()
    assert tpmlp.check_device_status(ctx2) == tpmlp.OK
    assert torch.equal(Z_inf, Z_train)
    assert torch.equal(ctx2.dY, Y_train)


def test_inference_forward_without_H():
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    T, h, F, t = 300, 384, 1280, 2
    inp = inputs.make(T, h, F, "bf16", seed=5, std=STD)
    d = {k: v.cuda() for k, v in inp.items()}
    ctx = tpmlp.Context(T, h, F, t, torch.bfloat16, keep_H=False)
    Z = tpmlp.forward(ctx, d["X"], d["A"], d["a"], d["B"], d["b"])
    torch.cuda.synchronize()
    ref = oracle.forward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], t)
    compare_full({"Z": Z, "Y": ctx.Y}, ref, {"Z": 1e-2, "Y": 1e-2})


@pytest.mark.parametrize("algo", ["tc", "simt"])
@pytest.mark.parametrize("T,h,F,t", [(300, 384, 1280, 2), (257, 512, 1024, 4)])
def test_recompute_matches_oracle_and_plain_mode(T, h, F, t, algo):
    """Activation recomputation (only H kept between the passes, Y rebuilt from H
    in the backward GeLU' epilogue) against the oracle, and against the plain
    mode.  The forward computes Y as GeLU of H as stored, which is exactly what
    the recomputation rebuilds, so every output, dB included, must be
    bit-identical to the plain mode."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    a = tpmlp.ALGO_SIMT if algo == "simt" else tpmlp.ALGO_DEFAULT
    inp = inputs.make(T, h, F, "bf16", seed=T * 3 + t, std=STD)
    rec, ctx = run_gpu(inp, t, algo=a, recompute=True)
    assert tpmlp.saved_bytes(ctx.shape) == T * F * 2
    ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
    compare_full(rec, ref, TOL_BF16)
    plain, _ = run_gpu(inp, t, algo=a)
    for k in ("Z", "H", "Y", "dY", "dX", "dA", "da", "db", "dB"):
        assert torch.equal(rec[k].view(torch.int16), plain[k].view(torch.int16)), k


FULL = [("h2048", 1), ("h2048", 2), ("h2048", 4), ("h4096", 8), ("h8192", 8), ("h12288-b1", 8),
        ("h12288-b2", 8), ("h12288-b4", 8), ("h12288-b8", 8)]


@pytest.mark.parametrize("name,t", [("h8192", 8)])
def test_full_size_recompute_slices(name, t):
    w = WORKLOADS[name]
    inp = inputs.for_workload(w)
    out, _ = run_gpu(inp, t, recompute=True)
    T, F = w.tokens, w.ffn
    R = sample_indices(T, 32, seed=3, must=(0, T - 1))
    J = sample_indices(F, 96, seed=4, must=[0, F - 1] + [i * (F // t) for i in range(t)])
    ref = oracle.slice_(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t, R, J)
    errs = compare_slices(out, ref, R, J, TOL_BF16)
    print("%s t=%d slice errors: %s" % (name, t, " ".join("%s=%.2e" % kv for kv in sorted(errs.items()))))


@pytest.mark.parametrize("name,t", FULL)
def test_full_size_workload_slices(name, t):
    w = WORKLOADS[name]
    if name.startswith("h12288"):
        import os
        mem = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
        if mem < 64 * 2 ** 30:
            pytest.skip("the slice oracle holds A and B in fp64 (about 10 GB)")
    inp = inputs.for_workload(w)
    out, _ = run_gpu(inp, t)
    T, F = w.tokens, w.ffn
    Fs = F // t
    R = sample_indices(T, 48, seed=1, must=(0, 127, 128, T - 1))
    J = sample_indices(F, 192, seed=2, must=[0, 255, 256, F - 1] + [i * Fs for i in range(t)])
    ref = oracle.slice_(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t, R, J)
    errs = compare_slices(out, ref, R, J, TOL_BF16)
    print("%s t=%d slice errors: %s" % (name, t, " ".join("%s=%.2e" % kv for kv in sorted(errs.items()))))
