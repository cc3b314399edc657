"""ctypes binding of libtpmlp.so (C ABI in include/tpmlp.h): argument marshalling
only.  Every step of the forward and backward pass runs in the library's CUDA
kernels; PyTorch supplies device memory and the current stream.

Importing this module loads the compiled library and raises if it is missing:
there is no fallback implementation.  TPMLP_LIBRARY=debug (read at import)
loads libtpmlp_debug.so instead, the build whose GEMM kernels bounds-check every
tile access and report a failed check as ERR_DEVICE in the status word.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtpmlp_debug.so" if os.environ.get("TPMLP_LIBRARY") == "debug"
                        else "libtpmlp.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(6)
F32, BF16 = 0, 1
ALGO_DEFAULT, ALGO_SIMT = 0, 1
WS_STATUS, WS_PARTIALS, WS_DY, WS_Y, WS_DXN = 0, 1, 2, 3, 4
FLAG_RECOMPUTE, FLAG_LAYERNORM = 1, 2
ATTN_P_UPPER_ZERO = 1

_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}


class Shape(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("t", ctypes.c_int32), ("dtype", ctypes.c_int32), ("algo", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class Saved(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("H", ctypes.c_void_p), ("Y", ctypes.c_void_p)]


class LayerNorm(ctypes.Structure):
    _fields_ = [("X_in", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("Xn", ctypes.c_void_p), ("mean", ctypes.c_void_p), ("rstd", ctypes.c_void_p),
                ("eps", ctypes.c_float)]


class AttnShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seq", ctypes.c_int64), ("hidden", ctypes.c_int64),
                ("heads", ctypes.c_int32), ("t", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class AttnSaved(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("Wqkv", ctypes.c_void_p), ("Wo", ctypes.c_void_p),
                ("QKV", ctypes.c_void_p), ("P", ctypes.c_void_p), ("O", ctypes.c_void_p)]


class TpmlpError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = last_error()
        super().__init__("%s: %s (status %d)%s" % (what, status_string(status), status,
                                                    (": " + detail) if detail else ""))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("%s is not built (expected at %s); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`"
                          % (os.path.basename(LIB_PATH), LIB_PATH))
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32, i64, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64
    SP = ctypes.POINTER(Shape)
    decl = {
        "tpmlp_status_string": (ctypes.c_char_p, [i32]),
        "tpmlp_version": (i32, []),
        "tpmlp_last_error": (ctypes.c_char_p, []),
        "tpmlp_saved_bytes": (sz, [SP]),
        "tpmlp_workspace_bytes": (sz, [SP]),
        "tpmlp_workspace_offset": (sz, [SP, i32]),
        "tpmlp_forward": (i32, [SP, vp, vp, vp, vp, vp, vp, ctypes.POINTER(Saved), vp, vp]),
        "tpmlp_backward": (i32, [SP, vp, ctypes.POINTER(Saved), vp, vp, vp, vp, vp, vp, vp]),
        "tpmlp_ln_forward": (i32, [SP, ctypes.POINTER(LayerNorm), vp]),
        "tpmlp_ln_backward": (i32, [SP, ctypes.POINTER(LayerNorm), vp, vp, vp, vp, vp, vp]),
        "tpmlp_sp_forward": (i32, [SP, ctypes.POINTER(LayerNorm), vp, vp, vp, vp, vp, ctypes.POINTER(Saved),
                                   vp, vp]),
        "tpmlp_sp_backward": (i32, [SP, ctypes.POINTER(LayerNorm), vp, ctypes.POINTER(Saved)] + [vp] * 9),
        "tpmlp_attn_saved_bytes": (sz, [ctypes.POINTER(AttnShape)]),
        "tpmlp_attn_workspace_bytes": (sz, [ctypes.POINTER(AttnShape)]),
        "tpmlp_attn_forward": (i32, [ctypes.POINTER(AttnShape)] + [vp] * 6 + [ctypes.POINTER(AttnSaved), vp, vp]),
        "tpmlp_attn_backward": (i32, [ctypes.POINTER(AttnShape), vp, ctypes.POINTER(AttnSaved)] + [vp] * 7),
        "tpmlp_check_device_status": (i32, [vp, vp]),
        "tpmlp_set_wait_limit_ns": (None, [u64]),
        "tpmlp_debug_timeout_probe": (i32, [vp, u64, vp]),
        "tpmlp_launch_count": (u64, []),
        "tpmlp_profile_enable": (None, [i32]),
        "tpmlp_profile_reset": (None, []),
        "tpmlp_profile_collect": (i32, []),
        "tpmlp_profile_count": (i32, []),
        "tpmlp_profile_entry": (i32, [i32, ctypes.c_char_p, i32, ctypes.POINTER(i64),
                                      ctypes.POINTER(ctypes.c_double)]),
    }
    for name, (res, args) in decl.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.tpmlp_status_string(int(status)).decode()


def last_error() -> str:
    return lib.tpmlp_last_error().decode(errors="replace")


def make_shape(tokens: int, hidden: int, ffn: int, t: int, dtype, algo: int = ALGO_DEFAULT,
               flags: int = 0) -> Shape:
    if isinstance(dtype, torch.dtype):
        dtype = _DTYPES[dtype]
    return Shape(int(tokens), int(hidden), int(ffn), int(t), int(dtype), int(algo), int(flags))


def saved_bytes(shape: Shape) -> int:
    return int(lib.tpmlp_saved_bytes(ctypes.byref(shape)))


def workspace_bytes(shape: Shape) -> int:
    return int(lib.tpmlp_workspace_bytes(ctypes.byref(shape)))


def workspace_offset(shape: Shape, region: int) -> int:
    return int(lib.tpmlp_workspace_offset(ctypes.byref(shape), int(region)))


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, what: str):
    if status != OK:
        raise TpmlpError(status, what)


def _need(x, name, dtype, shape):
    if not (x.is_cuda and x.is_contiguous()):
        raise ValueError("%s must be a contiguous CUDA tensor" % name)
    if x.dtype != dtype:
        raise ValueError("%s has dtype %s, expected %s" % (name, x.dtype, dtype))
    if tuple(x.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(x.shape), tuple(shape)))


def new_workspace(shape: Shape, device=None) -> torch.Tensor:
    """A zeroed workspace of the size the library asks for (uint8, 256-byte aligned)."""
    n = workspace_bytes(shape)
    if n == 0:
        raise ValueError("invalid shape")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


class Context:
    """The buffers one layer needs between forward and backward: H, Y and the
    workspace, plus the ctypes shape and saved-activation records."""

    def __init__(self, tokens, hidden, ffn, t, dtype, algo=ALGO_DEFAULT, device=None, keep_H=True,
                 recompute=False, layernorm=False, eps=1e-5):
        """recompute=True keeps only H between the passes (TPMLP_FLAG_RECOMPUTE):
        Y then lives in the workspace and is rebuilt by the backward pass.
        layernorm=True adds the LayerNorm in front (the sequence-parallel block,
        TPMLP_FLAG_LAYERNORM): Xn, mean and rstd buffers are allocated here."""
        flags = (FLAG_RECOMPUTE if recompute else 0) | (FLAG_LAYERNORM if layernorm else 0)
        self.shape = make_shape(tokens, hidden, ffn, t, dtype, algo, flags)
        if saved_bytes(self.shape) == 0 and tokens > 0:
            raise ValueError("invalid shape (tokens=%d hidden=%d ffn=%d t=%d)" % (tokens, hidden, ffn, t))
        self.dtype = dtype
        self.recompute = recompute
        dev = device or "cuda"
        self.H = torch.empty((tokens, ffn), dtype=dtype, device=dev) if (keep_H or recompute) else None
        self._Y = None if recompute else torch.empty((tokens, ffn), dtype=dtype, device=dev)
        self.workspace = new_workspace(self.shape, dev)
        self.saved = Saved(None, None, None, _ptr(self.H), _ptr(self._Y))
        self._keep = []
        if layernorm:
            self.Xn = torch.empty((tokens, hidden), dtype=dtype, device=dev)
            self.mean = torch.empty((tokens,), dtype=torch.float32, device=dev)
            self.rstd = torch.empty((tokens,), dtype=torch.float32, device=dev)
            self.ln = LayerNorm(None, None, None, _ptr(self.Xn), _ptr(self.mean), _ptr(self.rstd), float(eps))

    def _ws_view(self, region, cols=None):
        T = self.shape.tokens
        C = self.shape.ffn if cols is None else cols
        off = workspace_offset(self.shape, region)
        esz = 2 if self.dtype == torch.bfloat16 else 4
        return self.workspace[off:off + T * C * esz].view(self.dtype).view(T, C)

    @property
    def dXn(self) -> torch.Tensor:
        """The MLP's input gradient of the last sequence-parallel backward (the
        LayerNorm's output gradient; a view into the workspace)."""
        return self._ws_view(WS_DXN, self.shape.hidden)

    @property
    def Y(self) -> torch.Tensor:
        """GeLU(H): the caller-owned buffer, or under recomputation the workspace
        copy (written by forward, rebuilt by backward)."""
        return self._ws_view(WS_Y) if self.recompute else self._Y

    @property
    def dY(self) -> torch.Tensor:
        """The dY intermediate of the last backward (a view into the workspace)."""
        return self._ws_view(WS_DY)


def forward(ctx: Context, X, A, a, B, b, Z=None, stream=None, inference=False):
    """Z = GeLU(X A + a) B + b with the t-shard fold; fills ctx.H, ctx.Y.
    inference=True passes no saved record: nothing is kept for backward (Y goes
    to the workspace's dY region, H is not stored)."""
    s = ctx.shape
    T, h, F = s.tokens, s.hidden, s.ffn
    for x, n, shp in ((X, "X", (T, h)), (A, "A", (h, F)), (a, "a", (F,)), (B, "B", (F, h)), (b, "b", (h,))):
        _need(x, n, ctx.dtype, shp)
    if Z is None:
        Z = torch.empty((T, h), dtype=ctx.dtype, device=X.device)
    _need(Z, "Z", ctx.dtype, (T, h))
    ctx._keep = [X, A, B]
    st = lib.tpmlp_forward(ctypes.byref(s), _ptr(X), _ptr(A), _ptr(a), _ptr(B), _ptr(b), _ptr(Z),
                           None if inference else ctypes.byref(ctx.saved), _ptr(ctx.workspace), _stream(stream))
    _check(st, "tpmlp_forward")
    return Z


def backward(ctx: Context, dZ, dX=None, dA=None, da=None, dB=None, db=None, stream=None):
    """dX, dA, da, dB, db for L = sum(dZ * Z), using what forward saved in ctx."""
    s = ctx.shape
    T, h, F = s.tokens, s.hidden, s.ffn
    dev = dZ.device
    _need(dZ, "dZ", ctx.dtype, (T, h))
    out = {}
    for name, val, shp in (("dX", dX, (T, h)), ("dA", dA, (h, F)), ("da", da, (F,)),
                           ("dB", dB, (F, h)), ("db", db, (h,))):
        if val is None:
            val = torch.empty(shp, dtype=ctx.dtype, device=dev)
        _need(val, name, ctx.dtype, shp)
        out[name] = val
    st = lib.tpmlp_backward(ctypes.byref(s), _ptr(dZ), ctypes.byref(ctx.saved), _ptr(out["dX"]),
                            _ptr(out["dA"]), _ptr(out["da"]), _ptr(out["dB"]), _ptr(out["db"]),
                            _ptr(ctx.workspace), _stream(stream))
    _check(st, "tpmlp_backward")
    return out


def sp_forward(ctx: Context, X_in, gamma, beta, A, a, B, b, Z=None, stream=None):
    """Sequence-parallel block forward: Xn = LayerNorm(X_in), then the MLP on Xn."""
    s = ctx.shape
    T, h, F = s.tokens, s.hidden, s.ffn
    for x, n, shp in ((X_in, "X_in", (T, h)), (gamma, "gamma", (h,)), (beta, "beta", (h,)), (A, "A", (h, F)),
                      (a, "a", (F,)), (B, "B", (F, h)), (b, "b", (h,))):
        _need(x, n, ctx.dtype, shp)
    if Z is None:
        Z = torch.empty((T, h), dtype=ctx.dtype, device=X_in.device)
    _need(Z, "Z", ctx.dtype, (T, h))
    ctx.ln.X_in, ctx.ln.gamma, ctx.ln.beta = _ptr(X_in), _ptr(gamma), _ptr(beta)
    ctx._keep = [X_in, gamma, beta, A, B]
    st = lib.tpmlp_sp_forward(ctypes.byref(s), ctypes.byref(ctx.ln), _ptr(A), _ptr(a), _ptr(B), _ptr(b), _ptr(Z),
                              ctypes.byref(ctx.saved), _ptr(ctx.workspace), _stream(stream))
    _check(st, "tpmlp_sp_forward")
    return Z


def sp_backward(ctx: Context, dZ, stream=None, **outs):
    """Sequence-parallel block backward: dX_in, dgamma, dbeta and the MLP's
    weight and bias gradients."""
    s = ctx.shape
    T, h, F = s.tokens, s.hidden, s.ffn
    _need(dZ, "dZ", ctx.dtype, (T, h))
    out = {}
    for name, shp in (("dX_in", (T, h)), ("dgamma", (h,)), ("dbeta", (h,)), ("dA", (h, F)), ("da", (F,)),
                      ("dB", (F, h)), ("db", (h,))):
        val = outs.get(name)
        if val is None:
            val = torch.empty(shp, dtype=ctx.dtype, device=dZ.device)
        _need(val, name, ctx.dtype, shp)
        out[name] = val
    st = lib.tpmlp_sp_backward(ctypes.byref(s), ctypes.byref(ctx.ln), _ptr(dZ), ctypes.byref(ctx.saved),
                               *(_ptr(out[k]) for k in ("dX_in", "dgamma", "dbeta", "dA", "da", "dB", "db")),
                               _ptr(ctx.workspace), _stream(stream))
    _check(st, "tpmlp_sp_backward")
    return out


def ln_forward(ctx: Context, X_in, gamma, beta, stream=None):
    """LayerNorm alone (the block's first step): fills ctx.Xn, ctx.mean, ctx.rstd."""
    ctx.ln.X_in, ctx.ln.gamma, ctx.ln.beta = _ptr(X_in), _ptr(gamma), _ptr(beta)
    ctx._keep = [X_in, gamma, beta]
    _check(lib.tpmlp_ln_forward(ctypes.byref(ctx.shape), ctypes.byref(ctx.ln), _stream(stream)), "tpmlp_ln_forward")
    return ctx.Xn


def ln_backward(ctx: Context, dXn, stream=None):
    """LayerNorm backward alone for the gradient dXn of its output."""
    T, h = ctx.shape.tokens, ctx.shape.hidden
    dX_in = torch.empty((T, h), dtype=ctx.dtype, device=dXn.device)
    dg = torch.empty((h,), dtype=ctx.dtype, device=dXn.device)
    dbt = torch.empty((h,), dtype=ctx.dtype, device=dXn.device)
    st = lib.tpmlp_ln_backward(ctypes.byref(ctx.shape), ctypes.byref(ctx.ln), _ptr(dXn), _ptr(dX_in), _ptr(dg),
                               _ptr(dbt), _ptr(ctx.workspace), _stream(stream))
    _check(st, "tpmlp_ln_backward")
    return {"dX_in": dX_in, "dgamma": dg, "dbeta": dbt}


class AttnContext:
    """Buffers of one tensor-parallel self-attention layer between forward and
    backward: the saved QKV [T,3h], P [batch*heads, seq, seq], O [T,h] and the
    workspace (bf16 only).

    p_upper_zero=True (the default) allocates P zeroed and sets
    ATTN_P_UPPER_ZERO: the tiles of P wholly above the diagonal keep those
    zeros and the forward does not rewrite them.  False: P is allocated
    uninitialised and every row is written in full."""

    def __init__(self, batch, seq, hidden, heads, t, device=None, p_upper_zero=True):
        flags = ATTN_P_UPPER_ZERO if p_upper_zero else 0
        self.shape = AttnShape(int(batch), int(seq), int(hidden), int(heads), int(t), BF16, flags)
        n = int(lib.tpmlp_attn_workspace_bytes(ctypes.byref(self.shape)))
        if n == 0:
            raise ValueError("invalid attention shape (batch=%d seq=%d hidden=%d heads=%d t=%d)"
                             % (batch, seq, hidden, heads, t))
        dev = device or "cuda"
        T, h = batch * seq, hidden
        self.dtype = torch.bfloat16
        self.QKV = torch.empty((T, 3 * h), dtype=self.dtype, device=dev)
        alloc = torch.zeros if p_upper_zero else torch.empty
        self.P = alloc((batch * heads, seq, seq), dtype=self.dtype, device=dev)
        self.O = torch.empty((T, h), dtype=self.dtype, device=dev)
        self.workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
        self.saved = AttnSaved(None, None, None, _ptr(self.QKV), _ptr(self.P), _ptr(self.O))
        self._keep = []

    @property
    def tokens(self) -> int:
        return self.shape.batch * self.shape.seq


def attn_saved_bytes(batch, seq, hidden, heads, t) -> int:
    s = AttnShape(int(batch), int(seq), int(hidden), int(heads), int(t), BF16, 0)
    return int(lib.tpmlp_attn_saved_bytes(ctypes.byref(s)))


def attn_forward(ctx: AttnContext, X, Wqkv, bqkv, Wo, bo, Z=None, stream=None):
    """Z = bo + sum_i O_i Wo_i with per-head causal attention over X Wqkv + bqkv."""
    s = ctx.shape
    T, h = ctx.tokens, s.hidden
    for x, n, shp in ((X, "X", (T, h)), (Wqkv, "Wqkv", (h, 3 * h)), (bqkv, "bqkv", (3 * h,)),
                      (Wo, "Wo", (h, h)), (bo, "bo", (h,))):
        _need(x, n, ctx.dtype, shp)
    if Z is None:
        Z = torch.empty((T, h), dtype=ctx.dtype, device=X.device)
    _need(Z, "Z", ctx.dtype, (T, h))
    ctx._keep = [X, Wqkv, Wo]
    st = lib.tpmlp_attn_forward(ctypes.byref(s), _ptr(X), _ptr(Wqkv), _ptr(bqkv), _ptr(Wo), _ptr(bo), _ptr(Z),
                                ctypes.byref(ctx.saved), _ptr(ctx.workspace), _stream(stream))
    _check(st, "tpmlp_attn_forward")
    return Z


def attn_backward(ctx: AttnContext, dZ, stream=None, **outs):
    """dX, dWqkv, dbqkv, dWo, dbo for L = sum(dZ * Z), from what attn_forward saved."""
    s = ctx.shape
    T, h = ctx.tokens, s.hidden
    _need(dZ, "dZ", ctx.dtype, (T, h))
    out = {}
    for name, shp in (("dX", (T, h)), ("dWqkv", (h, 3 * h)), ("dbqkv", (3 * h,)), ("dWo", (h, h)),
                      ("dbo", (h,))):
        val = outs.get(name)
        if val is None:
            val = torch.empty(shp, dtype=ctx.dtype, device=dZ.device)
        _need(val, name, ctx.dtype, shp)
        out[name] = val
    st = lib.tpmlp_attn_backward(ctypes.byref(s), _ptr(dZ), ctypes.byref(ctx.saved),
                                 *(_ptr(out[k]) for k in ("dX", "dWqkv", "dbqkv", "dWo", "dbo")),
                                 _ptr(ctx.workspace), _stream(stream))
    _check(st, "tpmlp_attn_backward")
    return out


def check_device_status(ctx_or_ws, stream=None) -> int:
    ws = ctx_or_ws.workspace if isinstance(ctx_or_ws, (Context, AttnContext)) else ctx_or_ws
    return int(lib.tpmlp_check_device_status(_ptr(ws), _stream(stream)))


def set_wait_limit_ns(ns: int):
    lib.tpmlp_set_wait_limit_ns(int(ns))


def debug_timeout_probe(workspace, wait_ns: int, stream=None) -> int:
    return int(lib.tpmlp_debug_timeout_probe(_ptr(workspace), int(wait_ns), _stream(stream)))


def launch_count() -> int:
    return int(lib.tpmlp_launch_count())


def profile_enable(on: bool = True):
    lib.tpmlp_profile_enable(1 if on else 0)


def profile_reset():
    lib.tpmlp_profile_reset()


def profile_collect() -> dict:
    """{kernel name: (launches, total ms)} of the launches timed since the reset."""
    _check(lib.tpmlp_profile_collect(), "tpmlp_profile_collect")
    out = {}
    buf = ctypes.create_string_buffer(128)
    for i in range(lib.tpmlp_profile_count()):
        n = ctypes.c_int64()
        ms = ctypes.c_double()
        if lib.tpmlp_profile_entry(i, buf, 128, ctypes.byref(n), ctypes.byref(ms)) == 0:
            out[buf.value.decode()] = (int(n.value), float(ms.value))
    return out
