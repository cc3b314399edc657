"""Oracle for the tensor-parallel Transformer MLP block -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is a plain fp64 CPU implementation
(``oracle.c``, compiled with gcc + OpenMP) of what the CUDA library computes; the
two share no code.  The library never imports or calls anything here.

What it computes (the method, stated in the "Megatron-LM" industry report,
section 4.1, for the MLP block Y = f(XA)B with A split by columns and B by rows):

    H = X A + a,  Y = gelu(H),  Z_i = Y[:, S_i] B[S_i, :],  Z = b + sum_i Z_i
    db = 1^T dZ,  dY = (dZ B^T) * gelu'(H),  da = 1^T dY,
    dB = Y^T dZ,  dA = X^T dY,  dX = sum_i dY[:, S_i] A[:, S_i]^T

with shard i owning the ffn columns [i*F/t, (i+1)*F/t).  Every function here is
pinned by ``tests/test_oracle_pins.py`` (pins in ``tests/oracle_pins.py``):
closed forms and identities (GeLU's odd-part identity and asymptotes, the
sharded sum equal to the unsharded product, X = 0 and A = 0), numpy matmuls in
the special case t = 1 and per shard block, examples worked by hand (two
shards and attention under ``tests/golden/``, LayerNorm in the pins), central finite
differences of the loss for every gradient, and 24 planted one-line mistakes
that the pins must catch (``tests/test_oracle_mutants.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (-O2, OpenMP)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_DP = ctypes.POINTER(ctypes.c_double)
_LP = ctypes.POINTER(ctypes.c_int64)


def load(path: str | None = None):
    """Load (building first if needed) the oracle library and declare its ABI."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        lib.oracle_gelu.restype = ctypes.c_double
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu_prime.restype = ctypes.c_double
        lib.oracle_gelu_prime.argtypes = [ctypes.c_double]
        lib.oracle_gelu_vec.restype = None
        lib.oracle_gelu_vec.argtypes = [_DP, _DP, _DP, _I64]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [_I64, _I64, _I64, _I32] + [_DP] * 9
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [_I64, _I64, _I64, _I32] + [_DP] * 13
        lib.oracle_slice.restype = ctypes.c_int
        lib.oracle_slice.argtypes = ([_I64, _I64, _I64, _I32] + [_DP] * 6 +
                                     [_I64, _LP, _I64, _LP] + [_DP] * 12)
        lib.oracle_layernorm_forward.restype = None
        lib.oracle_layernorm_forward.argtypes = [_I64, _I64, _DP, _DP, _DP, ctypes.c_double, _DP, _DP, _DP]
        lib.oracle_layernorm_backward.restype = ctypes.c_int
        lib.oracle_layernorm_backward.argtypes = [_I64, _I64, _DP, _DP, _DP, ctypes.c_double, _DP, _DP, _DP]
        lib.oracle_attn_forward.restype = ctypes.c_int
        lib.oracle_attn_forward.argtypes = [_I64, _I64, _I64, _I64, _I32] + [_DP] * 9
        lib.oracle_attn_backward.restype = ctypes.c_int
        lib.oracle_attn_backward.argtypes = [_I64, _I64, _I64, _I64, _I32] + [_DP] * 12
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        if path is None:
            _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    """Exact conversion to a C-contiguous float64 array (bf16/fp32 widen exactly)."""
    if hasattr(x, "detach"):  # a torch tensor on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(x):
    return None if x is None else x.ctypes.data_as(_DP)


def gelu(x, lib=None) -> np.ndarray:
    lib = lib or load()
    x = _f64(x)
    y = np.empty_like(x)
    lib.oracle_gelu_vec(_p(x), _p(y), None, x.size)
    return y


def gelu_prime(x, lib=None) -> np.ndarray:
    lib = lib or load()
    x = _f64(x)
    dy = np.empty_like(x)
    lib.oracle_gelu_vec(_p(x), None, _p(dy), x.size)
    return dy


def forward(X, A, a, B, b, t: int, parts: bool = False, lib=None) -> dict:
    """H, Y, Z (and the t partial products Z_i if ``parts``) in fp64."""
    lib = lib or load()
    X, A, a, B, b = (_f64(v) for v in (X, A, a, B, b))
    T, h = X.shape
    F = A.shape[1]
    H = np.empty((T, F))
    Y = np.empty((T, F))
    Z = np.empty((T, h))
    Zp = np.empty((t, T, h)) if parts else None
    rc = lib.oracle_forward(T, h, F, t, _p(X), _p(A), _p(a), _p(B), _p(b),
                            _p(H), _p(Y), _p(Zp), _p(Z))
    if rc != 0:
        raise ValueError("oracle_forward rejected the shape (rc=%d)" % rc)
    out = {"H": H, "Y": Y, "Z": Z}
    if parts:
        out["Zpart"] = Zp
    return out


def backward(X, A, B, H, Y, dZ, t: int, parts: bool = False, lib=None) -> dict:
    """dY, dX, dA, da, dB, db (and the t dX partials if ``parts``) in fp64."""
    lib = lib or load()
    X, A, B, H, Y, dZ = (_f64(v) for v in (X, A, B, H, Y, dZ))
    T, h = X.shape
    F = A.shape[1]
    dY = np.empty((T, F))
    dX = np.empty((T, h))
    dA = np.empty((h, F))
    da = np.empty(F)
    dB = np.empty((F, h))
    db = np.empty(h)
    dXp = np.empty((t, T, h)) if parts else None
    rc = lib.oracle_backward(T, h, F, t, _p(X), _p(A), _p(B), _p(H), _p(Y), _p(dZ),
                             _p(dY), _p(dX), _p(dXp), _p(dA), _p(da), _p(dB), _p(db))
    if rc != 0:
        raise ValueError("oracle_backward rejected the shape (rc=%d)" % rc)
    out = {"dY": dY, "dX": dX, "dA": dA, "da": da, "dB": dB, "db": db}
    if parts:
        out["dXpart"] = dXp
    return out


def forward_backward(X, A, a, B, b, dZ, t: int, lib=None) -> dict:
    fw = forward(X, A, a, B, b, t, lib=lib)
    bw = backward(X, A, B, fw["H"], fw["Y"], dZ, t, lib=lib)
    fw.update(bw)
    return fw


def slice_(X, A, a, B, b, dZ, t: int, rows, cols, lib=None) -> dict:
    """Exact values on token rows ``rows`` and ffn columns ``cols``.

    Returns Hr, Yr, dYr ([len(rows), F]), Zr, dXr ([len(rows), h]),
    Hc, Yc, dYc ([T, len(cols)]), dAc ([h, len(cols)]), daJ ([len(cols)]),
    dBr ([len(cols), h]) and db ([h]).
    """
    lib = lib or load()
    X, A, a, B, b, dZ = (_f64(v) for v in (X, A, a, B, b, dZ))
    T, h = X.shape
    F = A.shape[1]
    R = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    J = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    nR, nJ = R.size, J.size
    out = {
        "Hr": np.empty((nR, F)), "Yr": np.empty((nR, F)), "dYr": np.empty((nR, F)),
        "Zr": np.empty((nR, h)), "dXr": np.empty((nR, h)),
        "Hc": np.empty((T, nJ)), "Yc": np.empty((T, nJ)), "dYc": np.empty((T, nJ)),
        "dAc": np.empty((h, nJ)), "daJ": np.empty(nJ), "dBr": np.empty((nJ, h)),
        "db": np.empty(h),
    }
    rc = lib.oracle_slice(T, h, F, t, _p(X), _p(A), _p(a), _p(B), _p(b), _p(dZ),
                          nR, R.ctypes.data_as(_LP), nJ, J.ctypes.data_as(_LP),
                          *(_p(out[k]) for k in ("Hr", "Yr", "dYr", "Zr", "dXr", "Hc", "Yc",
                                                 "dYc", "dAc", "daJ", "dBr", "db")))
    if rc != 0:
        raise ValueError("oracle_slice rejected the arguments (rc=%d)" % rc)
    return out


def layernorm_forward(X, gamma, beta, eps: float, lib=None) -> dict:
    """LayerNorm of every row: Y, and the row mean and 1/std (fp64)."""
    lib = lib or load()
    X, gamma, beta = (_f64(v) for v in (X, gamma, beta))
    T, h = X.shape
    Y = np.empty((T, h))
    mean = np.empty(T)
    rstd = np.empty(T)
    lib.oracle_layernorm_forward(T, h, _p(X), _p(gamma), _p(beta), float(eps), _p(Y), _p(mean), _p(rstd))
    return {"Y": Y, "mean": mean, "rstd": rstd}


def layernorm_backward(dY, X, gamma, eps: float, lib=None) -> dict:
    """dX, dgamma, dbeta of LayerNorm for the upstream gradient dY (fp64)."""
    lib = lib or load()
    dY, X, gamma = (_f64(v) for v in (dY, X, gamma))
    T, h = X.shape
    dX = np.empty((T, h))
    dg = np.empty(h)
    db = np.empty(h)
    rc = lib.oracle_layernorm_backward(T, h, _p(dY), _p(X), _p(gamma), float(eps), _p(dX), _p(dg), _p(db))
    if rc != 0:
        raise MemoryError("oracle_layernorm_backward")
    return {"dX": dX, "dgamma": dg, "dbeta": db}


def sp_forward_backward(X_in, gamma, beta, eps, A, a, B, b, dZ, t: int, lib=None) -> dict:
    """The sequence-parallel MLP block: LayerNorm of the input rows, then the
    tensor-parallel MLP, and the backward pass through both.  Token shards only
    change where rows live, not any value, so the whole batch is processed at
    once.  Returns the MLP outputs plus Xn (normalised input), mean, rstd,
    dX_in, dgamma, dbeta."""
    ln = layernorm_forward(X_in, gamma, beta, eps, lib=lib)
    out = forward_backward(ln["Y"], A, a, B, b, dZ, t, lib=lib)
    lb = layernorm_backward(out["dX"], X_in, gamma, eps, lib=lib)
    out.update({"Xn": ln["Y"], "mean": ln["mean"], "rstd": ln["rstd"], "dX_in": lb["dX"],
                "dgamma": lb["dgamma"], "dbeta": lb["dbeta"]})
    return out


def attn_forward(X, Wqkv, bqkv, Wo, bo, nb: int, heads: int, t: int, lib=None) -> dict:
    """Tensor-parallel causal self-attention forward in fp64: QKV [T,3h] (shard-
    major columns [Q_i | K_i | V_i]), P [nb, heads, S, S], O [T,h], Z [T,h]."""
    lib = lib or load()
    X, Wqkv, bqkv, Wo, bo = (_f64(v) for v in (X, Wqkv, bqkv, Wo, bo))
    T, h = X.shape
    S = T // nb
    QKV = np.empty((T, 3 * h))
    P = np.empty((nb, heads, S, S))
    O = np.empty((T, h))
    Z = np.empty((T, h))
    rc = lib.oracle_attn_forward(nb, S, h, heads, t, _p(X), _p(Wqkv), _p(bqkv), _p(Wo), _p(bo),
                                 _p(QKV), _p(P), _p(O), _p(Z))
    if rc != 0:
        raise ValueError("oracle_attn_forward rejected the shape (rc=%d)" % rc)
    return {"QKV": QKV, "P": P, "O": O, "Z": Z}


def attn_backward(X, Wqkv, Wo, QKV, P, O, dZ, nb: int, heads: int, t: int, lib=None) -> dict:
    """dX, dWqkv, dbqkv, dWo, dbo of the attention block in fp64."""
    lib = lib or load()
    X, Wqkv, Wo, QKV, P, O, dZ = (_f64(v) for v in (X, Wqkv, Wo, QKV, P, O, dZ))
    T, h = X.shape
    S = T // nb
    out = {"dX": np.empty((T, h)), "dWqkv": np.empty((h, 3 * h)), "dbqkv": np.empty(3 * h),
           "dWo": np.empty((h, h)), "dbo": np.empty(h)}
    rc = lib.oracle_attn_backward(nb, S, h, heads, t, _p(X), _p(Wqkv), _p(Wo), _p(QKV), _p(P), _p(O), _p(dZ),
                                  *(_p(out[k]) for k in ("dX", "dWqkv", "dbqkv", "dWo", "dbo")))
    if rc != 0:
        raise ValueError("oracle_attn_backward failed (rc=%d)" % rc)
    return out


def attn_forward_backward(X, Wqkv, bqkv, Wo, bo, dZ, nb: int, heads: int, t: int, lib=None) -> dict:
    fw = attn_forward(X, Wqkv, bqkv, Wo, bo, nb, heads, t, lib=lib)
    fw.update(attn_backward(X, Wqkv, Wo, fw["QKV"], fw["P"], fw["O"], dZ, nb, heads, t, lib=lib))
    return fw


def num_threads(lib=None) -> int:
    return int((lib or load()).oracle_num_threads())
