"""Helpers shared by the GPU tests: run the CUDA path through the C ABI on seeded
inputs, compare with the oracle by the relative max-error metric."""
from __future__ import annotations

import numpy as np
import torch

# max|out - ref| / max|ref| bounds: bf16 inputs with fp32 accumulation, and fp32.
TOL_BF16 = {"H": 1e-2, "Y": 1e-2, "Z": 1e-2, "dY": 2e-2, "dX": 2e-2, "dA": 2e-2, "da": 2e-2,
            "dB": 2e-2, "db": 2e-2}
TOL_F32 = {k: 1e-5 for k in TOL_BF16}


def rel(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    return num / den if den > 0 else num


def to_np(x: torch.Tensor) -> np.ndarray:
    return x.detach().double().cpu().numpy()


def run_gpu(inp: dict, t: int, algo=None, device="cuda", keep=False, recompute=False):
    """Forward + backward on the GPU; returns (outputs as GPU tensors, context)."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    algo = tpmlp.ALGO_DEFAULT if algo is None else algo
    d = {k: v.to(device) for k, v in inp.items()}
    T, h = d["X"].shape
    F = d["A"].shape[1]
    ctx = tpmlp.Context(T, h, F, t, d["X"].dtype, algo, device, recompute=recompute)
    Z = tpmlp.forward(ctx, d["X"], d["A"], d["a"], d["B"], d["b"])
    g = tpmlp.backward(ctx, d["dZ"])
    torch.cuda.synchronize()
    st = tpmlp.check_device_status(ctx)
    assert st == tpmlp.OK, "device status: %s" % tpmlp.status_string(st)
    out = {"H": ctx.H, "Y": ctx.Y.clone(), "Z": Z, "dY": ctx.dY.clone()}
    out.update(g)
    if keep:
        out["_dev_inputs"] = d
    return out, ctx


def compare_full(out: dict, ref: dict, tol: dict) -> dict:
    errs = {}
    for k in tol:
        if k in ref:
            errs[k] = rel(to_np(out[k]), ref[k])
    bad = {k: v for k, v in errs.items() if not (v <= tol[k])}
    assert not bad, "outside tolerance: %s (all: %s)" % (bad, errs)
    return errs


def sample_indices(n: int, k: int, seed: int, must=()) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(int(i) for i in must if 0 <= i < n)
    pick.update(int(i) for i in rng.choice(n, size=min(n, k), replace=False))
    return np.array(sorted(pick), dtype=np.int64)


def compare_slices(out: dict, ref: dict, R, J, tol: dict) -> dict:
    """Compare GPU outputs on rows R / ffn columns J with the exact slice oracle."""
    Rt = torch.as_tensor(R, device=out["Z"].device)
    Jt = torch.as_tensor(J, device=out["Z"].device)
    pairs = {
        "Z": (out["Z"][Rt], ref["Zr"]), "dX": (out["dX"][Rt], ref["dXr"]),
        "H": (torch.cat([out["H"][Rt].flatten(), out["H"][:, Jt].flatten()]),
              np.concatenate([ref["Hr"].ravel(), ref["Hc"].ravel()])),
        "Y": (torch.cat([out["Y"][Rt].flatten(), out["Y"][:, Jt].flatten()]),
              np.concatenate([ref["Yr"].ravel(), ref["Yc"].ravel()])),
        "dY": (torch.cat([out["dY"][Rt].flatten(), out["dY"][:, Jt].flatten()]),
               np.concatenate([ref["dYr"].ravel(), ref["dYc"].ravel()])),
        "dA": (out["dA"][:, Jt], ref["dAc"]), "da": (out["da"][Jt], ref["daJ"]),
        "dB": (out["dB"][Jt], ref["dBr"]), "db": (out["db"], ref["db"]),
    }
    errs = {k: rel(to_np(g), r) for k, (g, r) in pairs.items()}
    bad = {k: v for k, v in errs.items() if not (v <= tol[k])}
    assert not bad, "outside tolerance: %s (all: %s)" % (bad, errs)
    return errs
