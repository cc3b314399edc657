"""The bounds-checked build (libtpmlp_debug.so, TPMLP_LIBRARY=debug) on the GPU.

Compute-sanitizer cannot run on this machine, so the debug build stands in for
it: its tensor-core GEMM checks, before every TMA copy, MMA, TMEM load and
store, that tile coordinates, k-block ranges, shared-memory addresses and TMEM
columns lie inside what the launch set up, and reports a failed check as
TPMLP_ERR_DEVICE in the status word instead of making the access.  Here the
ragged-shape parity tests (every tile kind: pair, single-CTA, wide and split
half-width tiles, every tile order knob) and the attention parity tests run in a
child process on that build.  Each of them reads the status word after its run
and compares every output with the oracle, so a passing run means that no check
failed and the results are unchanged.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_debug(args):
    env = dict(os.environ, TPMLP_LIBRARY="debug")
    cmd = [sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider"] + args
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    return r.returncode, r.stdout[-3000:] + r.stderr[-2000:]


def test_debug_build_is_the_one_loaded():
    env = dict(os.environ, TPMLP_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", "from tensor_transformer_mlp_tma_gb300 import tpmlp; print(tpmlp.LIB_PATH)"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("libtpmlp_debug.so")


def test_mlp_parity_under_bounds_checks():
    rc, out = _run_debug(["tests/test_gpu_parity.py", "-k",
                          "tensor_core_path_matches_oracle or tuning_knobs or wide_and_square or special_cases"])
    assert rc == 0, out


def test_attention_parity_under_bounds_checks():
    rc, out = _run_debug(["tests/test_gpu_attn.py", "-k", "not full_size"])
    assert rc == 0, out
