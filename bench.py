#!/usr/bin/env python
"""Throughput of the TP-MLP block (forward + backward) on GB300.

One step = tpmlp_forward + tpmlp_backward over one batch of the workload
(default: h8192 -- T=4096 tokens, h=8192, F=32768, t=8 shards, bf16), inputs
resident in HBM.  FLOPs per step: 3 x (2 GEMMs x 2*T*h*F) = 12*T*h*F.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload (the path has no cross-GPU step here): weak scaling.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on a token sample
  python bench.py --sweep                # microbatch sweep, one line per b
  python bench.py --attn                 # the tensor-parallel self-attention block
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from tensor_transformer_mlp_tma_gb300 import inputs  # noqa: E402
from tensor_transformer_mlp_tma_gb300.workloads import HEADLINE, WORKLOADS  # noqa: E402

METRIC = "TP-MLP fwd+bwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 peak"
UNIT = "TFLOP/s"
REF_BUDGET_S = 150.0  # wall-time target of the reference arm's warm-up + timed steps
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) per launch of each tensor-core GEMM, from one ncu
# capture, with the hash of the kernel and launch sources they were taken at
# (kernel_source_hash).  After a change to either, traffic is reported null.
NCU_TRAFFIC = {  # profiles/dram_traffic_h8192_gemms.md (h8192 workload, one kernel per capture)
    "fc1_bias_gelu": (1.343788e9 + 0.520588e9, "20c49dd1ab49"),
    "fc2_shard_fold": (2.323672e9 + 0.095526e9, "20c49dd1ab49"),
    "bwd_dY_dgelu": (1.780639e9 + 0.278026e9, "20c49dd1ab49"),
    "bwd_dB": (0.931116e9 + 0.515468e9, "20c49dd1ab49"),
    "bwd_dA": (0.983755e9 + 0.514475e9, "20c49dd1ab49"),
    "bwd_dX_shard_fold": (2.323205e9 + 0.083362e9, "20c49dd1ab49"),
}


def kernel_source_hash() -> str:
    """sha256 prefix of the GEMM kernel source followed by the launch code (which
    picks the tile order, and so the DRAM traffic)."""
    h = hashlib.sha256()
    for name in ("tc_gemm.cu", "api.cu"):
        h.update(open(os.path.join(ROOT, "tensor_transformer_mlp_tma_gb300", "csrc", name), "rb").read())
    return h.hexdigest()[:12]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ distributed
def bf16_peak(peaks, peak_src):
    """The bf16 denominator of every fraction of peak: the measured burst figure
    (cuBLAS bf16 8192^3, best of 10 calls), the one for kernels timed in runs of
    well under a second.  The sustained figure (the same GEMM looped for seconds
    under the power cap, at a lower median clock) is reported beside it, never
    in its place."""
    return peaks["bf16_tflops"], "%s bf16_tflops (burst)" % peak_src


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.idx = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def host_cpu() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


# ------------------------------------------------------------------ oracle leg
def oracle_sample(w, tokens: int):
    """Time the fp64 oracle on a `tokens`-token instance of the workload: its
    recipe with fewer token rows (same h, F, t and value distributions, weights
    of full size, drawn after the smaller X); returns (seconds, flops, threads)."""
    import oracle
    inp = inputs.for_workload(w, tokens=tokens)
    lib = oracle.load()
    f64 = {k: oracle._f64(v) for k, v in inp.items()}
    t0 = time.perf_counter()
    oracle.forward_backward(f64["X"], f64["A"], f64["a"], f64["B"], f64["b"], f64["dZ"], w.shards[-1], lib=lib)
    dt = time.perf_counter() - t0
    return dt, 12.0 * tokens * w.hidden * w.ffn, oracle.num_threads(lib)


def attn_oracle_sample(w, tokens: int, seed: int):
    """Time the fp64 attention oracle on one sequence of `tokens` tokens with the
    workload's h, heads and t (full weights); returns (seconds, flops, threads)."""
    import dataclasses
    import oracle
    sw = dataclasses.replace(w, batch=1, seq=tokens)
    inp = inputs.make_attn(tokens, w.hidden, seed, {"Wqkv": w.std_W, "Wo": w.std_W, "bqkv": w.std_b, "bo": w.std_b})
    lib = oracle.load()
    f64 = {k: oracle._f64(v) for k, v in inp.items()}
    t0 = time.perf_counter()
    oracle.attn_forward_backward(f64["X"], f64["Wqkv"], f64["bqkv"], f64["Wo"], f64["bo"], f64["dZ"], 1, w.heads,
                                 w.t, lib=lib)
    dt = time.perf_counter() - t0
    return dt, sw.flops_fwd_bwd, oracle.num_threads(lib)


def run_reference(args, rank, world):
    """The reference arm: the fp64 CPU oracle as it stands, on host cores."""
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    import oracle
    lib = oracle.load()
    t = w.shards[-1]
    # Size the per-step token sample so that warm-up + timed steps take about
    # REF_BUDGET_S seconds: one calibration step on the requested sample first.
    tokens = args.oracle_tokens
    inp = inputs.for_workload(w, tokens=tokens)
    f64 = {k: oracle._f64(v) for k, v in inp.items()}
    c0 = time.perf_counter()
    oracle.forward_backward(f64["X"], f64["A"], f64["a"], f64["B"], f64["b"], f64["dZ"], t, lib=lib)
    per_step = time.perf_counter() - c0
    n = args.steps + args.warmup
    if n * per_step > REF_BUDGET_S and tokens > 1:
        tokens = max(1, int(tokens * REF_BUDGET_S / (n * per_step)))
        inp = inputs.for_workload(w, tokens=tokens)
        f64 = {k: oracle._f64(v) for k, v in inp.items()}
    args.oracle_tokens = tokens

    def step():
        oracle.forward_backward(f64["X"], f64["A"], f64["a"], f64["B"], f64["b"], f64["dZ"], t, lib=lib)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    flops = 12.0 * args.oracle_tokens * w.hidden * w.ffn
    val = flops / dt / 1e12
    sample = ("%d of %d token rows of %s per step (the workload's recipe with fewer tokens; full-size weights), "
              "fp64" % (args.oracle_tokens, w.tokens, w.name))
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, t, world),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": oracle.num_threads(lib), "kind": "oracle",
                             "sample": sample, "cpu": host_cpu()},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, t, world, fwd_only=False, recompute=False, sp=False):
    return {"workload": w.name, "tokens": w.tokens, "hidden": w.hidden, "ffn": w.ffn, "t": t,
            "pass": "forward" if fwd_only else "forward+backward",
            "activations_kept": "H only (recompute Y)" if recompute else "H and Y",
            "layernorm_in_front": bool(sp),
            "dtype": w.dtype, "parallelism": "replicas x%d" % world if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (A, B 537 MB each; ~3.2 GB touched per step)"
            if w.name == "h8192" else "per-step working set larger than L2"}


# ------------------------------------------------------------------ end to end
def gpu_local_cpus(dev):
    """The host cores the system lists as local to the GPU (its PCI device's
    local_cpulist), or None where that is not known."""
    try:
        p = torch.cuda.get_device_properties(dev)
        bdf = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bdf) as f:
            text = f.read().strip()
        cpus = set()
        for part in text.split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        return cpus or None
    except (AttributeError, OSError, ValueError):
        return None


def overlapped_e2e(dev, stream, world, steps, warmup, host_in, dev_out, copy_out, fwd, bwd):
    """Times `steps` steps end to end: every step copies `host_in` (pinned host
    tensors) to the device, runs fwd (and bwd, if given) on `stream`, and copies
    the `copy_out` outputs back to pinned host memory.  The copies run on their
    own streams, overlapped with compute: step i+1's inputs are copied in while
    step i computes, and step i's results are copied out while step i+1
    computes (device inputs and outputs double-buffered).  The timed region
    opens before the first step's input copy and closes after the last step's
    results have reached host memory.

    dev_out: name -> (shape, dtype) of the device outputs; copy_out: (names
    copied after the forward, names copied after the backward); fwd(ins, outs)
    and bwd(ins, outs) launch one step's work.  Returns (max over ranks of the
    ms per step, host-to-device bytes per step, device-to-host bytes per step,
    a note on the host cores used, the measured copy rates).

    While the pinned buffers are made and the steps run, the calling thread is
    held to the host cores local to the GPU (where the system names them and the
    process may use them): a pinned page is placed in the memory of the core
    that first touches it, and copies from a far memory node cross one more
    link."""
    allowed = os.sched_getaffinity(0)
    local = gpu_local_cpus(dev)
    near = (local & allowed) if local else set()
    if near and near != allowed:
        os.sched_setaffinity(0, near)
        note = "calling thread on the %d of %d allowed host cores local to the GPU" % (len(near), len(allowed))
    elif near:
        note = "all %d allowed host cores are local to the GPU" % len(allowed)
    else:
        note = "GPU-local host cores not known or not allowed; %d cores, affinity unchanged" % len(allowed)
    try:
        ems, h2d, d2h, rates = overlapped_e2e_run(dev, stream, world, steps, warmup, host_in, dev_out, copy_out,
                                                  fwd, bwd)
        return ems, h2d, d2h, note, rates
    finally:
        os.sched_setaffinity(0, allowed)


def overlapped_e2e_run(dev, stream, world, steps, warmup, host_in, dev_out, copy_out, fwd, bwd):
    hin = {k: v.pin_memory() for k, v in host_in.items()}
    din = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in hin.items()} for _ in range(2)]
    dout = [{k: torch.empty(shape, dtype=dt, device=dev) for k, (shape, dt) in dev_out.items()} for _ in range(2)]
    out_fwd, out_bwd = copy_out
    hout = [{k: torch.empty(dout[0][k].shape, dtype=dout[0][k].dtype).pin_memory() for k in out_fwd + out_bwd}
            for _ in range(2)]
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    fwd_done = [torch.cuda.Event() for _ in range(2)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    pend = {"done": [False, False], "out": [False, False]}

    def copy_in(b):
        if pend["done"][b]:  # the step that last read buffer b has finished
            s_in.wait_event(step_done[b])
        with torch.cuda.stream(s_in):
            for k, v in hin.items():
                din[b][k].copy_(v, non_blocking=True)
        in_ready[b].record(s_in)

    def copy_out(b):
        # results of the step that used buffer b, each copy gated on the event that
        # makes it ready
        s_out.wait_event(fwd_done[b])
        with torch.cuda.stream(s_out):
            for k in out_fwd:
                hout[b][k].copy_(dout[b][k], non_blocking=True)
        if out_bwd:
            s_out.wait_event(step_done[b])
            with torch.cuda.stream(s_out):
                for k in out_bwd:
                    hout[b][k].copy_(dout[b][k], non_blocking=True)
        out_done[b].record(s_out)
        pend["out"][b] = True

    def one_step(i, last):
        # Host order: this step's kernels first, then the copies of the previous
        # step's results and of the next step's inputs, so that a copy call that
        # returns late cannot hold back the kernels queued behind it.
        b = i % 2
        stream.wait_event(in_ready[b])
        if pend["out"][b]:  # results of step i-2 have left buffer b
            stream.wait_event(out_done[b])
        fwd(din[b], dout[b])
        fwd_done[b].record(stream)
        if bwd is not None:
            bwd(din[b], dout[b])
        step_done[b].record(stream)
        pend["done"][b] = True
        if i > 0:
            copy_out(b ^ 1)
        if not last:
            copy_in(b ^ 1)
        else:
            copy_out(b)

    def run_steps(n, start_event=None, end_event=None):
        if start_event is not None:
            start_event.record(stream)
            s_in.wait_event(start_event)
        copy_in(0)
        for i in range(n):
            one_step(i, i == n - 1)
        for b in range(2):
            if pend["out"][b]:
                stream.wait_event(out_done[b])
        if end_event is not None:
            end_event.record(stream)
        torch.cuda.synchronize(dev)
        pend["done"] = [False, False]
        pend["out"] = [False, False]

    run_steps(max(1, warmup))
    barrier(world)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    run_steps(steps, f0, f1)
    barrier(world)
    ems = max_over_ranks(f0.elapsed_time(f1) / steps, world)
    h2d = sum(v.numel() * v.element_size() for v in hin.values())
    d2h = sum(v.numel() * v.element_size() for v in hout[0].values())
    # The copy rates alone, outside the timed region: one step's inputs in and
    # results out, each timed on its copy stream with nothing else running (best
    # of three).  A step cannot run faster end to end than its copies allow.
    rates = {}
    for name, cs, pairs in (("h2d_gbs", s_in, [(din[0][k], v) for k, v in hin.items()]),
                            ("d2h_gbs", s_out, [(hout[0][k], dout[0][k]) for k in hout[0]])):
        best_ms, best_enq = None, None
        for _ in range(3):
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(cs)
            h0 = time.perf_counter()
            with torch.cuda.stream(cs):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            # host time to enqueue them: near zero when the copies run asynchronously
            enq = (time.perf_counter() - h0) * 1e3
            c1.record(cs)
            torch.cuda.synchronize(dev)
            ms = c0.elapsed_time(c1)
            best_ms = ms if best_ms is None else min(best_ms, ms)
            best_enq = enq if best_enq is None else min(best_enq, enq)
        nbytes = sum(dst.numel() * dst.element_size() for dst, _ in pairs)
        rates[name] = nbytes / (best_ms * 1e-3) / 1e9 if nbytes else None
        rates[name.replace("gbs", "enqueue_ms")] = best_enq
    return ems, h2d, d2h, rates


# ------------------------------------------------------------------ timed passes
def timed_passes(tpmlp, step, steps, stream, dev, world):
    """Two passes of `steps` steps each on `stream`, inputs resident in HBM.

    1. The headline pass: nothing but the steps between two CUDA events, with
       nvidia-smi sampling the clocks meanwhile.  Its time is the line's value.
    2. The per-kernel pass: the same steps with the library's per-launch event
       pairs switched on (every launch bracketed by two events on its own
       stream); it gives each kernel's mean duration and share, from which the
       roofline's `achieved` is computed.

    Returns (ms per step of pass 1 (max over ranks), clock summary of pass 1,
    launches of pass 1, {kernel: (launches, total ms)} of pass 2, ms per step of
    pass 2, clock summary of pass 2)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    launches0 = tpmlp.launch_count()
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clocks:
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    launches = tpmlp.launch_count() - launches0
    ms_max = max_over_ranks(e0.elapsed_time(e1) / steps, world)

    tpmlp.profile_reset()
    tpmlp.profile_enable(True)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clocks2:
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    tpmlp.profile_enable(False)
    kernels = tpmlp.profile_collect()
    return ms_max, clocks.summary(), launches, kernels, e0.elapsed_time(e1) / steps, clocks2.summary()


# ------------------------------------------------------------------ GPU leg
def run_ours(args, rank, world, local, w=None, quiet=False):
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    w = w or WORKLOADS[args.workload]
    t = args.t or w.shards[-1]
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dt = inputs.torch_dtype(w.dtype)
    host = inputs.for_workload(w, seed=args.seed + rank)
    d = {k: v.to(dev) for k, v in host.items()}
    T, h, F = w.tokens, w.hidden, w.ffn
    ctx = tpmlp.Context(T, h, F, t, dt, device=dev, recompute=args.recompute, layernorm=args.sp)
    if args.sp:  # LayerNorm parameters of the sequence-parallel block
        gamma = torch.ones((h,), dtype=dt, device=dev)
        beta = torch.zeros((h,), dtype=dt, device=dev)
    Z = torch.empty((T, h), dtype=dt, device=dev)
    g = {"dX": torch.empty((T, h), dtype=dt, device=dev), "dA": torch.empty((h, F), dtype=dt, device=dev),
         "da": torch.empty((F,), dtype=dt, device=dev), "dB": torch.empty((F, h), dtype=dt, device=dev),
         "db": torch.empty((h,), dtype=dt, device=dev)}
    stream = torch.cuda.Stream(device=dev)

    def step():
        if args.sp:
            tpmlp.sp_forward(ctx, d["X"], gamma, beta, d["A"], d["a"], d["B"], d["b"], Z=Z, stream=stream)
            if not args.fwd_only:
                tpmlp.sp_backward(ctx, d["dZ"], stream=stream, dX_in=g["dX"], dgamma=sp_dg, dbeta=sp_db,
                                  dA=g["dA"], da=g["da"], dB=g["dB"], db=g["db"])
            return
        tpmlp.forward(ctx, d["X"], d["A"], d["a"], d["B"], d["b"], Z=Z, stream=stream)
        if not args.fwd_only:
            tpmlp.backward(ctx, d["dZ"], stream=stream, **g)

    if args.sp:
        sp_dg = torch.empty((h,), dtype=dt, device=dev)
        sp_db = torch.empty((h,), dtype=dt, device=dev)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    st = tpmlp.check_device_status(ctx, stream)
    if st != tpmlp.OK:
        raise RuntimeError("device status after warm-up: %s" % tpmlp.status_string(st))

    # ---- timed region: inputs resident in HBM (headline pass, then the
    # per-kernel pass)
    ms_max, clk, launches, kernels, ms_prof, clk_prof = timed_passes(tpmlp, step, args.steps, stream, dev, world)
    st = tpmlp.check_device_status(ctx, stream)
    if st != tpmlp.OK:
        raise RuntimeError("device status after timed region: %s" % tpmlp.status_string(st))
    flops = (4.0 if args.fwd_only else 12.0) * T * h * F
    value = flops * world / (ms_max * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    peak_bf16, peak_bf16_src = bf16_peak(peaks, peak_src)
    # dominant kernel: largest share of the timed region
    name, (n, tot) = max(kernels.items(), key=lambda kv: kv[1][1])
    per_launch_ms = tot / n
    gemm_flops = {"fc1_bias_gelu": 2.0 * T * h * F, "fc2_shard_fold": 2.0 * T * h * F,
                  "bwd_dY_dgelu": 2.0 * T * h * F, "bwd_dB": 2.0 * T * h * F, "bwd_dA": 2.0 * T * h * F,
                  "bwd_dX_shard_fold": 2.0 * T * h * F}
    if name in gemm_flops:
        achieved = gemm_flops[name] / (per_launch_ms * 1e-3) / 1e12
        tr = NCU_TRAFFIC.get(name) if w.name == "h8192" else None
        traffic = tr[0] if tr and tr[1] == kernel_source_hash() else None
        roof = {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak_bf16, "unit": UNIT,
                "frac": achieved / peak_bf16, "traffic": traffic, "peak_source": peak_bf16_src,
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "sm_mhz_median": clk_prof["sm_mhz"],
                "timing": "mean launch duration from the per-kernel pass (%d steps after the headline "
                          "pass, %.3f ms per step with the per-launch events)" % (args.steps, ms_prof)}
    else:  # a column sum: HBM bound
        roof = {"bound": "hbm", "kernel": name, "achieved": None, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": None, "traffic": None}

    # ---- end to end: pinned host inputs in, results out, every step, on copy
    # streams overlapped with the neighbouring steps' compute.
    e2e = None
    if not args.no_e2e:
        host_in = {"X": host["X"]} if args.fwd_only else {"X": host["X"], "dZ": host["dZ"]}
        dev_out = {"Z": ((T, h), dt)}
        if not args.fwd_only:
            dev_out.update({k: (tuple(v.shape), v.dtype) for k, v in g.items()})

        def fwd(ins, outs):
            if args.sp:
                tpmlp.sp_forward(ctx, ins["X"], gamma, beta, d["A"], d["a"], d["B"], d["b"], Z=outs["Z"],
                                 stream=stream)
            else:
                tpmlp.forward(ctx, ins["X"], d["A"], d["a"], d["B"], d["b"], Z=outs["Z"], stream=stream)

        def bwd(ins, outs):
            if args.sp:
                tpmlp.sp_backward(ctx, ins["dZ"], stream=stream, dX_in=outs["dX"], dgamma=sp_dg, dbeta=sp_db,
                                  dA=outs["dA"], da=outs["da"], dB=outs["dB"], db=outs["db"])
            else:
                tpmlp.backward(ctx, ins["dZ"], stream=stream, **{k: outs[k] for k in g})

        ems, h2d, d2h, host_note, rates = overlapped_e2e(dev, stream, world, args.steps, args.warmup, host_in,
                                                         dev_out,
                                       (["Z"], [] if args.fwd_only else ["dX", "da", "db"]), fwd,
                                       None if args.fwd_only else bwd)
        e2e = {"value": flops * world / (ems * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "what": "X and dZ copied in from pinned host memory, Z, dX, da, db copied out, every "
                       "step, on copy streams overlapped with the neighbouring steps' compute; weights "
                       "and weight gradients stay resident", "host": host_note,
               "copy_rates_gbs": rates}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": config_of(w, t, world, args.fwd_only, args.recompute, args.sp),
            "frac_of_peak": value / world / peak_bf16,
            "peak_tflops": peak_bf16, "peak_source": peak_bf16_src,
            "frac_of_sustained_peak": value / world / peaks["bf16_tflops_sustained"],
            "roofline": roof, "e2e": e2e, "gpu_launches": int(sum_over_ranks(launches, world)),
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
            "kernels": {k: {"launches": n, "ms_per_launch": tot / n, "share": tot / sum(v[1] for v in kernels.values())}
                        for k, (n, tot) in kernels.items()}}
    return line


# ------------------------------------------------------------------ attention leg
def run_attn_bench(args, rank, world, local):
    """Forward + backward of the tensor-parallel self-attention block (heads split
    among t shards; the projections and per-head products on the tensor-core
    GEMMs).  One step = tpmlp_attn_forward + tpmlp_attn_backward."""
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    from tensor_transformer_mlp_tma_gb300.workloads import ATTN_WORKLOADS
    w = ATTN_WORKLOADS[args.attn_workload]
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    host = inputs.make_attn(w.tokens, w.hidden, args.seed + rank,
                            {"Wqkv": w.std_W, "Wo": w.std_W, "bqkv": w.std_b, "bo": w.std_b})
    d = {k: v.to(dev) for k, v in host.items()}
    T, h, S = w.tokens, w.hidden, w.seq
    ctx = tpmlp.AttnContext(w.batch, S, h, w.heads, w.t, device=dev)
    Z = torch.empty((T, h), dtype=torch.bfloat16, device=dev)
    g = {"dX": torch.empty((T, h), dtype=torch.bfloat16, device=dev),
         "dWqkv": torch.empty((h, 3 * h), dtype=torch.bfloat16, device=dev),
         "dbqkv": torch.empty((3 * h,), dtype=torch.bfloat16, device=dev),
         "dWo": torch.empty((h, h), dtype=torch.bfloat16, device=dev),
         "dbo": torch.empty((h,), dtype=torch.bfloat16, device=dev)}
    stream = torch.cuda.Stream(device=dev)

    def step():
        tpmlp.attn_forward(ctx, d["X"], d["Wqkv"], d["bqkv"], d["Wo"], d["bo"], Z=Z, stream=stream)
        tpmlp.attn_backward(ctx, d["dZ"], stream=stream, **g)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize(dev)
    if tpmlp.check_device_status(ctx, stream) != tpmlp.OK:
        raise RuntimeError("device status after warm-up")
    ms_max, clk, launches, kernels, ms_prof, clk_prof = timed_passes(tpmlp, step, args.steps, stream, dev, world)
    if tpmlp.check_device_status(ctx, stream) != tpmlp.OK:
        raise RuntimeError("device status after timed region")
    value = w.flops_fwd_bwd * world / (ms_max * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    # per-head products over the causal lower triangle (the work the path needs)
    proj, head = 2.0 * T * h * h, 1.0 * T * (S + 1) * h
    gemm_flops = {"attn_qkv_proj": 3 * proj, "attn_out_proj_fold": proj, "attn_scores": head, "attn_pv": head,
                  "attn_bwd_dO": proj, "attn_bwd_dWo": proj, "attn_bwd_dV": head, "attn_bwd_dS": head,
                  "attn_bwd_dQ": head, "attn_bwd_dK": head, "attn_bwd_dWqkv": 3 * proj,
                  "attn_bwd_dX_shard_fold": 3 * proj}
    name, (n, tot) = max(kernels.items(), key=lambda kv: kv[1][1])
    achieved = gemm_flops[name] / (tot / n * 1e-3) / 1e12 if name in gemm_flops else None
    peak, peak_bf16_src = bf16_peak(peaks, peak_src)
    roof = {"bound": "tensor", "kernel": name, "achieved": achieved, "peak": peak, "unit": UNIT,
            "frac": achieved / peak if achieved else None, "traffic": None, "peak_source": peak_bf16_src,
            "sm_mhz_median": clk_prof["sm_mhz"],
            "timing": "mean launch duration from the per-kernel pass (%d steps after the headline "
                      "pass, %.3f ms per step with the per-launch events)" % (args.steps, ms_prof)}
    total = sum(v[1] for v in kernels.values())

    e2e = None
    if not args.no_e2e:
        dev_out = {"Z": ((T, h), torch.bfloat16)}
        dev_out.update({k: (tuple(v.shape), v.dtype) for k, v in g.items()})

        def fwd(ins, outs):
            tpmlp.attn_forward(ctx, ins["X"], d["Wqkv"], d["bqkv"], d["Wo"], d["bo"], Z=outs["Z"], stream=stream)

        def bwd(ins, outs):
            tpmlp.attn_backward(ctx, ins["dZ"], stream=stream, **{k: outs[k] for k in g})

        ems, h2d, d2h, host_note, rates = overlapped_e2e(dev, stream, world, args.steps, args.warmup,
                                       {"X": host["X"], "dZ": host["dZ"]}, dev_out,
                                       (["Z"], ["dX", "dbqkv", "dbo"]), fwd, bwd)
        e2e = {"value": w.flops_fwd_bwd * world / (ems * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "what": "X and dZ copied in from pinned host memory, Z, dX, dbqkv, dbo copied out, every "
                       "step, on copy streams overlapped with the neighbouring steps' compute; weights "
                       "and weight gradients stay resident", "host": host_note,
               "copy_rates_gbs": rates}
    return {"metric": "TP self-attention fwd+bwd TFLOP/s (bf16, 1×GB300)", "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "seq": S, "hidden": h, "heads": w.heads, "t": w.t,
                       "causal": True, "pass": "forward+backward",
                       "flops_per_step": w.flops_fwd_bwd,
                       "flops_note": "projections 24*T*h^2 + per-head products 6*T*h*(seq+1) (the causal "
                                     "lower triangle only; tiles above the diagonal are skipped)",
                       "l2": "per-step working set larger than L2"},
            "frac_of_peak": value / world / peak, "roofline": roof, "e2e": e2e,
            "gpu_launches": int(sum_over_ranks(launches, world)),
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
            "kernels": {k: {"launches": n, "ms_per_launch": t_ / n, "share": t_ / total,
                            "tflops": (gemm_flops[k] / (t_ / n * 1e-3) / 1e12) if k in gemm_flops else None}
                        for k, (n, t_) in kernels.items()}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--t", type=int, default=0, help="shard count (default: the workload's)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sweep", action="store_true", help="microbatch sweep h12288-b{1,2,4,8}")
    ap.add_argument("--fwd-only", action="store_true",
                    help="time tpmlp_forward alone (4*T*h*F FLOP per step)")
    ap.add_argument("--recompute", action="store_true",
                    help="activation recomputation: keep only H between forward and backward")
    ap.add_argument("--sp", action="store_true",
                    help="sequence-parallel block: LayerNorm in front of the MLP")
    ap.add_argument("--attn", action="store_true",
                    help="the tensor-parallel self-attention block (its own line, not the headline)")
    ap.add_argument("--attn-workload", default="attn-h8192", choices=["attn-h4096", "attn-h8192"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-tokens", type=int, default=256,
                    help="token rows of the oracle's bounded sample (about 13 s of fp64 work at h8192 on "
                         "16 cores; the reference arm shrinks it to fit its time budget)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.attn:
        line = run_attn_bench(args, rank, world, local)
        if rank == 0:
            if not args.no_cpu_baseline:
                from tensor_transformer_mlp_tma_gb300.workloads import ATTN_WORKLOADS
                w = ATTN_WORKLOADS[args.attn_workload]
                secs, fl, cores = attn_oracle_sample(w, args.oracle_tokens, args.seed)
                line["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                                        "cpu": host_cpu(),
                                        "sample": "one sequence of %d tokens with the full weights of %s "
                                                  "(h %d, %d heads, t %d), fp64 (%.1f s)"
                                                  % (args.oracle_tokens, w.name, w.hidden, w.heads, w.t, secs)}
            print(json.dumps(line), flush=True)
        return
    if args.sweep:
        for b in (1, 2, 4, 8):
            line = run_ours(args, rank, world, local, w=WORKLOADS["h12288-b%d" % b])
            if rank == 0:
                print(json.dumps(line), flush=True)
        return
    line = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            w = WORKLOADS[args.workload]
            secs, fl, cores = oracle_sample(w, args.oracle_tokens)
            line["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                                    "cpu": host_cpu(),
                                    "sample": "%d of %d token rows of %s (the workload's recipe with fewer "
                                              "tokens; full-size weights), fp64 (%.1f s)"
                                              % (args.oracle_tokens, w.tokens, w.name, secs)}
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
