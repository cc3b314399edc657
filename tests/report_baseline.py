"""Per-workload report on a GB300: the CUDA path against the fp64 oracle.

For every named workload (and its shard counts) it prints one JSON line with:
- max |out - ref| / max |ref| for Z and the largest over the gradients. The
  small workloads are compared with the full oracle; the large ones with the
  exact slice oracle on sampled token rows and ffn columns;
- whether three repeated runs are bit-identical;
- the oracle's fp64 wall time on this host: measured in full for the small
  workloads; for the large ones, measured on a `--tokens`-token instance of the
  workload (its recipe with fewer tokens, full-size weights) and
  scaled to the full token count (marked "extrapolated": the oracle's work is
  linear in the tokens at a fixed h and F).

  python tests/report_baseline.py [--workloads tiny-fp32,h2048,...] [--tokens 32]
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from gpu_cases import rel, run_gpu, sample_indices, to_np  # noqa: E402
from tensor_transformer_mlp_tma_gb300 import inputs  # noqa: E402
from tensor_transformer_mlp_tma_gb300.workloads import WORKLOADS  # noqa: E402

FULL_ORACLE = {"tiny-fp32", "h2048"}
GRADS = ("dX", "dA", "da", "dB", "db")


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def report(name: str, t: int, tokens: int) -> dict:
    w = WORKLOADS[name]
    inp = inputs.for_workload(w)
    out, _ = run_gpu(inp, t)
    torch.cuda.synchronize()
    line = {"workload": name, "t": t, "tokens": w.tokens, "hidden": w.hidden, "ffn": w.ffn, "dtype": w.dtype}
    if name in FULL_ORACLE:
        t0 = time.perf_counter()
        ref = oracle.forward_backward(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t)
        secs = time.perf_counter() - t0
        err_z = rel(to_np(out["Z"]), ref["Z"])
        err_g = max(rel(to_np(out[k]), ref[k]) for k in GRADS)
        line.update(compare="full oracle", oracle_s=secs, oracle_timing="measured")
    else:
        T, F = w.tokens, w.ffn
        R = sample_indices(T, 64, seed=1, must=(0, T - 1))
        J = sample_indices(F, 256, seed=2, must=[0, F - 1] + [i * (F // t) for i in range(t)])
        ref = oracle.slice_(inp["X"], inp["A"], inp["a"], inp["B"], inp["b"], inp["dZ"], t, R, J)
        Rt = torch.as_tensor(R, device="cuda")
        Jt = torch.as_tensor(J, device="cuda")
        err_z = rel(to_np(out["Z"][Rt]), ref["Zr"])
        err_g = max(rel(to_np(out["dX"][Rt]), ref["dXr"]), rel(to_np(out["dA"][:, Jt]), ref["dAc"]),
                    rel(to_np(out["da"][Jt]), ref["daJ"]), rel(to_np(out["dB"][Jt]), ref["dBr"]),
                    rel(to_np(out["db"]), ref["db"]))
        sub = inputs.for_workload(w, tokens=tokens)
        t0 = time.perf_counter()
        oracle.forward_backward(sub["X"], sub["A"], sub["a"], sub["B"], sub["b"], sub["dZ"], t)
        secs = (time.perf_counter() - t0) * w.tokens / tokens
        line.update(compare="slice oracle (%d rows, %d ffn columns)" % (len(R), len(J)), oracle_s=secs,
                    oracle_timing="extrapolated from the first %d token rows" % tokens)
    runs = [{k: v.clone() for k, v in out.items() if isinstance(v, torch.Tensor)}]
    for _ in range(2):
        o, _ = run_gpu(inp, t)
        runs.append({k: v.clone() for k, v in o.items() if isinstance(v, torch.Tensor)})
    torch.cuda.synchronize()
    same = all(torch.equal(runs[0][k], r[k]) for r in runs[1:] for k in runs[0])
    line.update(max_rel_err_Z=err_z, max_rel_err_grads=err_g, bit_identical_3_runs=same,
                oracle_gflops=w.flops_fwd_bwd / line["oracle_s"] / 1e9, oracle_threads=oracle.num_threads(),
                cpu=cpu_model(), nproc=os.cpu_count())
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", default="tiny-fp32,h2048,h4096,h8192,h12288-b1,h12288-b2,h12288-b4,h12288-b8")
    ap.add_argument("--tokens", type=int, default=32)
    args = ap.parse_args()
    for name in args.workloads.split(","):
        for t in WORKLOADS[name].shards:
            print(json.dumps(report(name, t, args.tokens)), flush=True)


if __name__ == "__main__":
    main()
