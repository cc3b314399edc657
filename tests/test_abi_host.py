"""The C ABI without a GPU: the library builds, loads and exports every symbol
include/tpmlp.h declares; size queries and host-side validation return the
documented values.  Only argument checks that fail before any CUDA call are
exercised here (no pointer is ever dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tp():
    from tensor_transformer_mlp_tma_gb300 import build
    build.build()
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    return tpmlp


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tpmlp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tpmlp_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tpmlp_forward", "tpmlp_backward", "tpmlp_saved_bytes", "tpmlp_workspace_bytes",
              "tpmlp_check_device_status", "tpmlp_status_string"):
        assert n in names


def test_binding_constants_match_the_header(tp):
    """Every enumerator the header declares has the same value in the binding
    (TPMLP_X in C is X in Python), so the two cannot drift apart."""
    src = open(os.path.join(ROOT, "include", "tpmlp.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    enums = dict((k, int(v)) for k, v in re.findall(r"\bTPMLP_([A-Z0-9_]+)\s*=\s*(-?\d+)", src))
    assert len(enums) >= 18, enums  # status, dtype, algo, flags, workspace regions, attention flags
    for name, value in enums.items():
        assert getattr(tp, name) == value, name


def test_every_declared_symbol_is_exported(tp):
    lib = ctypes.CDLL(tp.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_debug_build_exports_the_same_symbols(tp):
    """libtpmlp_debug.so (the bounds-checked build, TPMLP_LIBRARY=debug) is built
    beside the library and exports every declared entry point too."""
    from tensor_transformer_mlp_tma_gb300 import build
    assert os.path.exists(build.LIB_DEBUG)
    lib = ctypes.CDLL(build.LIB_DEBUG)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(tp):
    for s in range(6):
        assert tp.status_string(s)
    assert tp.status_string(0) == "ok"
    assert tp.status_string(99) == "unknown status"


def test_size_queries(tp):
    s = tp.make_shape(4096, 8192, 32768, 8, tp.BF16)
    assert tp.saved_bytes(s) == 2 * 4096 * 32768 * 2
    ws = tp.workspace_bytes(s)
    off = tp.workspace_offset(s, tp.WS_DY)
    assert off % 1024 == 0 and off >= 1024
    assert ws >= off + 4096 * 32768 * 2
    assert tp.workspace_offset(s, tp.WS_STATUS) == 0
    assert tp.workspace_offset(s, 7) == ctypes.c_size_t(-1).value
    f32 = tp.make_shape(128, 256, 1024, 2, tp.F32)
    assert tp.saved_bytes(f32) == 2 * 128 * 1024 * 4
    # invalid shapes: 0
    for bad in (tp.make_shape(128, 256, 1000, 3, tp.BF16),   # F % t != 0
                tp.make_shape(128, 0, 1024, 2, tp.BF16),     # h = 0
                tp.make_shape(-1, 256, 1024, 2, tp.BF16),    # T < 0
                tp.make_shape(128, 256, 1024, 17, tp.BF16),  # t > 16
                tp.make_shape(128, 256, 1024, 0, tp.BF16),   # t < 1
                tp.Shape(128, 256, 1024, 2, 7, 0, 0),        # dtype
                tp.Shape(128, 256, 1024, 2, 1, 5, 0),        # algo
                tp.Shape(128, 256, 1024, 2, 1, 0, 4)):       # unknown flag
        assert tp.saved_bytes(bad) == 0
        assert tp.workspace_bytes(bad) == 0
    # every dimension within its limit, but more output tiles than the kernels'
    # 32-bit tile counter holds
    huge = tp.make_shape(1 << 30, 256, 1 << 30, 1, tp.BF16)
    assert tp.saved_bytes(huge) == 0 and tp.workspace_bytes(huge) == 0
    # recomputation keeps H only and moves Y into the workspace
    rec = tp.make_shape(4096, 8192, 32768, 8, tp.BF16, flags=tp.FLAG_RECOMPUTE)
    assert tp.saved_bytes(rec) == 4096 * 32768 * 2
    # Y follows dY; the workspace grows by exactly Y (the 8 KiB block of ones for
    # the bias-gradient tiles stays at the end)
    assert tp.workspace_offset(rec, tp.WS_Y) == tp.workspace_offset(s, tp.WS_DY) + 4096 * 32768 * 2
    assert tp.workspace_bytes(rec) == tp.workspace_bytes(s) + 4096 * 32768 * 2
    # an empty batch is valid
    assert tp.workspace_bytes(tp.make_shape(0, 256, 1024, 2, tp.BF16)) > 0


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fwd(tp, shape, ptrs=None, saved=None, ws=FAKE):
    p = ptrs or [FAKE] * 6
    sv = saved if saved is not None else tp.Saved(None, None, None, FAKE, FAKE)
    return tp.lib.tpmlp_forward(ctypes.byref(shape) if shape is not None else None, *p,
                                ctypes.byref(sv), ws, None)


def _fwd_inference(tp, shape, ptrs=None, ws=FAKE):
    p = ptrs or [FAKE] * 6
    return tp.lib.tpmlp_forward(ctypes.byref(shape), *p, None, ws, None)


def test_forward_inference_validation(tp):
    """saved == NULL (inference) is accepted by validation; the inputs are still checked."""
    good = tp.make_shape(256, 256, 1024, 2, tp.BF16)
    for i in range(6):
        p = [FAKE] * 6
        p[i] = None
        assert _fwd_inference(tp, good, ptrs=p) == tp.ERR_INVALID_ARG
    p = [FAKE] * 6
    p[0] = FAKE + 2
    assert _fwd_inference(tp, good, ptrs=p) == tp.ERR_UNSUPPORTED
    assert _fwd_inference(tp, good, ws=None) == tp.ERR_INVALID_ARG


def _bwd(tp, shape, ptrs=None, saved=None, ws=FAKE):
    p = ptrs or [FAKE] * 6
    sv = saved if saved is not None else tp.Saved(FAKE, FAKE, FAKE, FAKE, FAKE)
    return tp.lib.tpmlp_backward(ctypes.byref(shape), p[0], ctypes.byref(sv), *p[1:], ws, None)


def test_forward_invalid_arguments(tp):
    good = tp.make_shape(256, 256, 1024, 2, tp.BF16)
    assert _fwd(tp, None) == tp.ERR_INVALID_ARG
    assert _fwd(tp, tp.make_shape(256, 256, 1000, 3, tp.BF16)) == tp.ERR_INVALID_ARG
    assert _fwd(tp, tp.make_shape(256, 256, 1024, 17, tp.BF16)) == tp.ERR_INVALID_ARG
    for i in range(6):  # each required pointer NULL in turn
        p = [FAKE] * 6
        p[i] = None
        assert _fwd(tp, good, ptrs=p) == tp.ERR_INVALID_ARG
    assert _fwd(tp, good, saved=tp.Saved(None, None, None, FAKE, None)) == tp.ERR_INVALID_ARG
    assert _fwd(tp, good, ws=None) == tp.ERR_INVALID_ARG
    # under recomputation H is required (it is the saved activation)
    rec = tp.make_shape(256, 256, 1024, 2, tp.BF16, flags=tp.FLAG_RECOMPUTE)
    assert _fwd(tp, rec, saved=tp.Saved(None, None, None, None, FAKE)) == tp.ERR_INVALID_ARG


def test_forward_unsupported(tp):
    good = tp.make_shape(256, 256, 1024, 2, tp.BF16)
    p = [FAKE] * 6
    p[1] = FAKE + 2  # bf16-aligned but not 16-byte aligned: TMA cannot take it
    assert _fwd(tp, good, ptrs=p) == tp.ERR_UNSUPPORTED
    p = [FAKE] * 6
    p[0] = FAKE + 1  # not even element-aligned
    assert _fwd(tp, good, ptrs=p) == tp.ERR_UNSUPPORTED
    # shard size F/t = 96 is not a multiple of the 64-wide k-block
    assert _fwd(tp, tp.make_shape(256, 256, 192, 2, tp.BF16)) == tp.ERR_UNSUPPORTED
    # hidden size whose row pitch is not 16-byte aligned
    assert _fwd(tp, tp.make_shape(256, 260, 1024, 2, tp.BF16)) == tp.ERR_UNSUPPORTED
    # optional H misaligned
    assert _fwd(tp, good, saved=tp.Saved(None, None, None, FAKE + 2, FAKE)) == tp.ERR_UNSUPPORTED
    assert _fwd(tp, good, ws=FAKE + 8) == tp.ERR_UNSUPPORTED


def test_backward_invalid_arguments(tp):
    good = tp.make_shape(256, 256, 1024, 2, tp.BF16)
    for i in range(6):
        p = [FAKE] * 6
        p[i] = None
        assert _bwd(tp, good, ptrs=p) == tp.ERR_INVALID_ARG
    for field in ("X", "A", "B", "H", "Y"):
        sv = tp.Saved(FAKE, FAKE, FAKE, FAKE, FAKE)
        setattr(sv, field, None)
        assert _bwd(tp, good, saved=sv) == tp.ERR_INVALID_ARG
    assert _bwd(tp, tp.make_shape(256, 256, 192, 2, tp.BF16)) == tp.ERR_UNSUPPORTED


def test_debug_probe_rejects_bad_arguments(tp):
    assert tp.lib.tpmlp_debug_timeout_probe(None, 1000, None) == tp.ERR_INVALID_ARG
    assert tp.lib.tpmlp_debug_timeout_probe(FAKE, 20_000_000_000, None) == tp.ERR_INVALID_ARG


def test_profile_table_starts_empty(tp):
    tp.profile_reset()
    assert tp.lib.tpmlp_profile_count() == 0
    assert tp.lib.tpmlp_profile_entry(0, None, 0, None, None) == -1


def _attn_fwd(tp, shape, ptrs=None, saved=None, ws=FAKE):
    p = ptrs or [FAKE] * 6
    sv = saved if saved is not None else tp.AttnSaved(None, None, None, FAKE, FAKE, FAKE)
    return tp.lib.tpmlp_attn_forward(ctypes.byref(shape) if shape is not None else None, *p,
                                     ctypes.byref(sv) if sv is not False else None, ws, None)


def _attn_bwd(tp, shape, ptrs=None, saved=None, ws=FAKE):
    p = ptrs or [FAKE] * 6
    sv = saved if saved is not None else tp.AttnSaved(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    return tp.lib.tpmlp_attn_backward(ctypes.byref(shape), p[0], ctypes.byref(sv), *p[1:], ws, None)


def test_attention_size_queries(tp):
    s = tp.AttnShape(2, 2048, 8192, 64, 8, tp.BF16, 0)
    T, h, S, nz = 4096, 8192, 2048, 128
    assert tp.lib.tpmlp_attn_saved_bytes(ctypes.byref(s)) == 2 * (T * 3 * h + T * h + nz * S * S)
    ws = tp.lib.tpmlp_attn_workspace_bytes(ctypes.byref(s))
    # token-major dO and dQKV, fp16 scores (the per-head operands are views)
    assert ws >= 4 * T * h * 2 + nz * S * S * 2
    assert ws < 5 * T * h * 2 + nz * S * S * 2
    assert ws % 1024 == 0
    assert tp.attn_saved_bytes(2, 2048, 8192, 64, 8) == tp.lib.tpmlp_attn_saved_bytes(ctypes.byref(s))
    for bad in (tp.AttnShape(1, 64, 256, 3, 1, tp.BF16, 0),    # h % heads != 0
                tp.AttnShape(1, 64, 256, 2, 4, tp.BF16, 0),    # heads % t != 0
                tp.AttnShape(1, 64, 256, 2, 0, tp.BF16, 0),    # t < 1
                tp.AttnShape(1, 0, 256, 2, 1, tp.BF16, 0),     # seq = 0
                tp.AttnShape(-1, 64, 256, 2, 1, tp.BF16, 0),   # batch < 0
                tp.AttnShape(1, 64, 256, 2, 1, tp.BF16, 2),    # unknown flag
                tp.AttnShape(1, 64, 256, 2, 1, tp.BF16, -1),   # unknown flags
                tp.AttnShape(1 << 10, 1 << 20, 1024, 8, 1, tp.BF16, 0)):  # scores past 2^48 elements
        assert tp.lib.tpmlp_attn_saved_bytes(ctypes.byref(bad)) == 0
        assert tp.lib.tpmlp_attn_workspace_bytes(ctypes.byref(bad)) == 0
    assert tp.lib.tpmlp_attn_workspace_bytes(ctypes.byref(tp.AttnShape(0, 64, 256, 2, 2, tp.BF16, 0))) > 0
    # TPMLP_ATTN_P_UPPER_ZERO changes which tiles of P are written, not any size
    up = tp.AttnShape(1, 64, 256, 2, 1, tp.BF16, tp.ATTN_P_UPPER_ZERO)
    plain = tp.AttnShape(1, 64, 256, 2, 1, tp.BF16, 0)
    assert tp.lib.tpmlp_attn_saved_bytes(ctypes.byref(up)) == tp.lib.tpmlp_attn_saved_bytes(ctypes.byref(plain)) > 0
    assert tp.lib.tpmlp_attn_workspace_bytes(ctypes.byref(up)) == tp.lib.tpmlp_attn_workspace_bytes(ctypes.byref(plain)) > 0


def test_attention_invalid_and_unsupported_arguments(tp):
    good = tp.AttnShape(2, 128, 256, 2, 2, tp.BF16, 0)
    assert _attn_fwd(tp, None) == tp.ERR_INVALID_ARG
    assert _attn_fwd(tp, good, saved=False) == tp.ERR_INVALID_ARG
    assert _attn_fwd(tp, good, ws=None) == tp.ERR_INVALID_ARG
    for i in range(6):
        p = [FAKE] * 6
        p[i] = None
        assert _attn_fwd(tp, good, ptrs=p) == tp.ERR_INVALID_ARG
        assert _attn_bwd(tp, good, ptrs=p) == tp.ERR_INVALID_ARG
    for field in ("X", "Wqkv", "Wo", "QKV", "P", "O"):
        sv = tp.AttnSaved(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
        setattr(sv, field, None)
        assert _attn_bwd(tp, good, saved=sv) == tp.ERR_INVALID_ARG
    # fp32, head size 32, seq not a multiple of 8, misaligned pointer: unsupported
    assert _attn_fwd(tp, tp.AttnShape(2, 128, 256, 2, 2, tp.F32, 0)) == tp.ERR_UNSUPPORTED
    assert _attn_fwd(tp, tp.AttnShape(2, 128, 256, 8, 2, tp.BF16, 0)) == tp.ERR_UNSUPPORTED
    assert _attn_fwd(tp, tp.AttnShape(2, 100, 256, 2, 2, tp.BF16, 0)) == tp.ERR_UNSUPPORTED
    p = [FAKE] * 6
    p[1] = FAKE + 2
    assert _attn_fwd(tp, good, ptrs=p) == tp.ERR_UNSUPPORTED
    assert _attn_bwd(tp, good, ws=FAKE + 8) == tp.ERR_UNSUPPORTED
