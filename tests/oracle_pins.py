"""Pins for the oracle: checks against what the pages and mathematics fix.

Each ``check_*`` takes a loaded oracle library and returns a list of failure
strings (empty = pass), so that the same checks serve the normal test run and the
planted-mistake run (tests/test_oracle_mutants.py), which must see every planted
mistake caught by at least one of them.

What pins what:
  * GeLU      -- the tanh form stays within its published error of the exact
                 x*Phi(x) (max |diff| ~4.73e-4, Hendrycks & Gimpel 2016); the
                 algebraic identity gelu(x) - gelu(-x) = x; gelu(0) = 0;
                 gelu'(0) = 1/2; the asymptotes; gelu' against central
                 differences of gelu.
  * forward   -- t = 1 reduces to the textbook MLP, built here from numpy
                 matmuls; for t = 2, 4, 8 the sum of the shard partials plus b
                 equals the unsharded result and each partial is the column /
                 row block product of the "Megatron-LM" report, section 4.1
                 (Z = Y_1 B_1 + Y_2 B_2 for t = 2).
  * backward  -- central finite differences of L = sum(dZ * Z) for every element
                 of X, A, a, B and b; the dX shard partials against numpy.
  * worked example -- tests/golden/worked_example_t2.txt: the two-shard split of
                 section 4.1 with pre-activations of exactly 10, -10 and 0, every
                 forward, backward and shard-partial value worked by hand.
  * closed forms -- X = 0 gives Z = gelu(a) B + b and dA = 0; A = 0, a = 0 give
                 Z = b, dY = dZ B^T / 2, dX = 0; db is the column sum of dZ.
  * slices    -- the exact row/column slices equal the full result.
  * LayerNorm -- numpy's population mean/variance definition; normalised rows
                 have mean 0 and variance 1; invariance to a positive scale and a
                 shift of a row; dX orthogonal to 1 and xhat; central finite
                 differences for dX, dgamma, dbeta, and for the whole
                 sequence-parallel block (LayerNorm, then the sharded MLP).
  * attention -- numpy einsum/softmax on the canonical [Q|K|V] layout; the same
                 outputs for t = 1, 2, 4 after the shard-major column permutation
                 (the head split of section 4.1); rows of P sum to 1 and put no
                 weight on later tokens; a token changes only its own and later
                 outputs of its own sequence; central finite differences for dX,
                 dWqkv, dbqkv, dWo, dbo.
"""
from __future__ import annotations

import math

import os

import numpy as np

import oracle


def _rel(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(x - ref)) if ref.size else 0.0
    return num / den if den > 0 else num


def _rand(rng, shape, std=1.0):
    return rng.standard_normal(shape) * std


def _case(T, h, F, seed, stds=(1.0, 0.5, 0.5, 0.5, 0.5, 1.0)):
    rng = np.random.default_rng(seed)
    sX, sA, sa, sB, sb, sdZ = stds
    return (_rand(rng, (T, h), sX), _rand(rng, (h, F), sA), _rand(rng, (F,), sa),
            _rand(rng, (F, h), sB), _rand(rng, (h,), sb), _rand(rng, (T, h), sdZ))


def check_gelu_vs_erf(lib):
    x = np.linspace(-8.0, 8.0, 160001)
    exact = 0.5 * x * (1.0 + np.vectorize(math.erf)(x / math.sqrt(2.0)))
    err = np.max(np.abs(oracle.gelu(x, lib=lib) - exact))
    # the tanh form's largest deviation from x*Phi(x) is 4.73e-4 (near |x| = 2.7);
    # a wrong constant (0.04 or 0.05 for 0.044715, or sqrt(pi/2) for
    # sqrt(2/pi)) moves it to >= 2.8e-3.
    return [] if err <= 5.0e-4 else ["gelu deviates from x*Phi(x) by %.3e" % err]


def check_gelu_identities(lib):
    f = []
    x = np.linspace(-6.0, 6.0, 1201)
    d = oracle.gelu(x, lib=lib) - oracle.gelu(-x, lib=lib) - x
    if np.max(np.abs(d)) > 1e-14:
        f.append("gelu(x) - gelu(-x) != x (%.3e)" % np.max(np.abs(d)))
    if lib.oracle_gelu(0.0) != 0.0:
        f.append("gelu(0) != 0")
    if abs(lib.oracle_gelu_prime(0.0) - 0.5) > 1e-15:
        f.append("gelu'(0) != 1/2")
    if abs(lib.oracle_gelu(30.0) - 30.0) > 1e-12 or abs(lib.oracle_gelu(-30.0)) > 1e-12:
        f.append("gelu asymptotes wrong")
    if abs(lib.oracle_gelu_prime(30.0) - 1.0) > 1e-12 or abs(lib.oracle_gelu_prime(-30.0)) > 1e-12:
        f.append("gelu' asymptotes wrong")
    return f


def check_gelu_prime_fd(lib):
    x = np.linspace(-6.0, 6.0, 2401)
    eps = 1e-5
    fd = (oracle.gelu(x + eps, lib=lib) - oracle.gelu(x - eps, lib=lib)) / (2 * eps)
    err = np.max(np.abs(fd - oracle.gelu_prime(x, lib=lib)))
    return [] if err <= 1e-9 else ["gelu' disagrees with central differences by %.3e" % err]


def _numpy_forward(X, A, a, B, b, lib):
    H = X @ A + a
    Y = oracle.gelu(H, lib=lib)
    return H, Y, Y @ B + b


def check_forward_numpy(lib):
    f = []
    for (T, h, F), t, seed in [((5, 7, 16), 1, 1), ((6, 8, 16), 2, 2), ((9, 12, 32), 4, 3),
                               ((4, 16, 64), 8, 4), ((1, 3, 8), 8, 5)]:
        X, A, a, B, b, _ = _case(T, h, F, seed)
        out = oracle.forward(X, A, a, B, b, t, parts=True, lib=lib)
        H, Y, Z = _numpy_forward(X, A, a, B, b, lib)
        for name, got, ref in (("H", out["H"], H), ("Y", out["Y"], Y), ("Z", out["Z"], Z)):
            if _rel(got, ref) > 1e-12:
                f.append("forward %s t=%d rel %.3e vs numpy" % (name, t, _rel(got, ref)))
        Fs = F // t
        for i in range(t):
            S = slice(i * Fs, (i + 1) * Fs)
            ref = Y[:, S] @ B[S, :]
            if _rel(out["Zpart"][i], ref) > 1e-12:
                f.append("Z partial %d of t=%d wrong" % (i, t))
        if _rel(out["Zpart"].sum(axis=0) + b, out["Z"]) > 1e-12:
            f.append("sum of partials + b != Z for t=%d" % t)
    return f


def check_worked_example_t2(lib):
    """Two shards exactly as the report's section 4.1 writes them:
    Y_1 = f(X W_{1,1}), Y_2 = f(X W_{1,2}), Z = Y_1 W_{2,1} + Y_2 W_{2,2} (+ b)."""
    X, A, a, B, b, _ = _case(4, 6, 10, 11)
    A1, A2 = A[:, :5], A[:, 5:]
    a1, a2 = a[:5], a[5:]
    B1, B2 = B[:5, :], B[5:, :]
    Y1 = oracle.gelu(X @ A1 + a1, lib=lib)
    Y2 = oracle.gelu(X @ A2 + a2, lib=lib)
    Zref = Y1 @ B1 + Y2 @ B2 + b
    out = oracle.forward(X, A, a, B, b, 2, parts=True, lib=lib)
    f = []
    if _rel(out["Z"], Zref) > 1e-12:
        f.append("t=2 worked example: Z differs (%.3e)" % _rel(out["Z"], Zref))
    if _rel(out["Zpart"][0], Y1 @ B1) > 1e-12 or _rel(out["Zpart"][1], Y2 @ B2) > 1e-12:
        f.append("t=2 worked example: partials differ")
    if _rel(out["Y"], np.concatenate([Y1, Y2], axis=1)) > 1e-12:
        f.append("t=2 worked example: Y is not [Y_1, Y_2]")
    return f


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    """A tests/golden fixture: scalars as 'name value', matrices as 'name rows
    cols' followed by the rows; '#' starts a comment line."""
    out, lines = {}, [ln.split() for ln in open(os.path.join(GOLDEN, name))
                      if ln.strip() and not ln.lstrip().startswith("#")]
    i = 0
    while i < len(lines):
        f = lines[i]
        if len(f) == 2:
            out[f[0]] = int(f[1])
            i += 1
        else:
            r, c = int(f[1]), int(f[2])
            out[f[0]] = np.array([[float(x) for x in lines[i + 1 + k]] for k in range(r)]).reshape(r, c)
            i += 1 + r
    return out


def check_golden_worked_example_t2(lib):
    """The hand-worked two-shard example of tests/golden/worked_example_t2.txt
    (report section 4.1's two-GPU split, pre-activations of exactly 10, -10 and
    0): forward, backward and both sets of shard partials."""
    g = read_golden("worked_example_t2.txt")
    t = g["t"]
    fw = oracle.forward(g["X"], g["A"], g["a"].ravel(), g["B"], g["b"].ravel(), t, parts=True, lib=lib)
    bw = oracle.backward(g["X"], g["A"], g["B"], fw["H"], fw["Y"], g["dZ"], t, parts=True, lib=lib)
    got = {"H": fw["H"], "Y": fw["Y"], "Z": fw["Z"], "Z1": fw["Zpart"][0], "Z2": fw["Zpart"][1],
           "dY": bw["dY"], "da": bw["da"][None, :], "db": bw["db"][None, :], "dB": bw["dB"], "dA": bw["dA"],
           "dX": bw["dX"], "dX1": bw["dXpart"][0], "dX2": bw["dXpart"][1]}
    f = []
    for k, v in got.items():
        err = float(np.max(np.abs(v - g[k])))
        if err > 1e-12 * max(1.0, float(np.max(np.abs(g[k])))):
            f.append("golden t=2 example: %s differs by %.3e" % (k, err))
    return f


def _loss(lib, X, A, a, B, b, dZ, t):
    return float(np.sum(dZ * oracle.forward(X, A, a, B, b, t, lib=lib)["Z"]))


def check_backward_fd(lib, shapes=((3, 4, 8),), ts=(1, 2, 4), eps=1e-6, tol=1e-6):
    f = []
    for (T, h, F) in shapes:
        for t in ts:
            X, A, a, B, b, dZ = _case(T, h, F, 100 + t)
            fw = oracle.forward(X, A, a, B, b, t, lib=lib)
            bw = oracle.backward(X, A, B, fw["H"], fw["Y"], dZ, t, lib=lib)
            params = {"X": X, "A": A, "a": a, "B": B, "b": b}
            grads = {"X": bw["dX"], "A": bw["dA"], "a": bw["da"], "B": bw["dB"], "b": bw["db"]}
            for name, p in params.items():
                fd = np.empty_like(p)
                flat = p.reshape(-1)
                for idx in range(flat.size):
                    old = flat[idx]
                    flat[idx] = old + eps
                    lp = _loss(lib, X, A, a, B, b, dZ, t)
                    flat[idx] = old - eps
                    lm = _loss(lib, X, A, a, B, b, dZ, t)
                    flat[idx] = old
                    fd.reshape(-1)[idx] = (lp - lm) / (2 * eps)
                r = _rel(grads[name], fd)
                if r > tol:
                    f.append("d%s (T=%d h=%d F=%d t=%d) vs finite differences: rel %.3e"
                             % (name, T, h, F, t, r))
    return f


def check_backward_partials(lib):
    f = []
    for t in (1, 2, 4):
        X, A, a, B, b, dZ = _case(6, 8, 16, 200 + t)
        fw = oracle.forward(X, A, a, B, b, t, lib=lib)
        bw = oracle.backward(X, A, B, fw["H"], fw["Y"], dZ, t, parts=True, lib=lib)
        Fs = 16 // t
        for i in range(t):
            S = slice(i * Fs, (i + 1) * Fs)
            if _rel(bw["dXpart"][i], bw["dY"][:, S] @ A[:, S].T) > 1e-12:
                f.append("dX partial %d of t=%d wrong" % (i, t))
        if _rel(bw["dXpart"].sum(axis=0), bw["dX"]) > 1e-12:
            f.append("sum of dX partials != dX for t=%d" % t)
    return f


def check_closed_forms(lib):
    f = []
    T, h, F, t = 5, 6, 12, 3
    X, A, a, B, b, dZ = _case(T, h, F, 300)
    # X = 0: H = a in every row, so Z = gelu(a) B + b and dA = X^T dY = 0
    Z0 = np.zeros_like(X)
    fw = oracle.forward(Z0, A, a, B, b, t, lib=lib)
    bw = oracle.backward(Z0, A, B, fw["H"], fw["Y"], dZ, t, lib=lib)
    zref = np.tile(oracle.gelu(a, lib=lib) @ B + b, (T, 1))
    if _rel(fw["Z"], zref) > 1e-12:
        f.append("X = 0: Z != gelu(a) B + b")
    if np.max(np.abs(bw["dA"])) != 0.0:
        f.append("X = 0: dA != 0")
    # A = 0, a = 0: H = 0, Y = 0, Z = b, dY = dZ B^T * gelu'(0) = dZ B^T / 2, dX = 0
    A0 = np.zeros_like(A)
    a0 = np.zeros_like(a)
    fw = oracle.forward(X, A0, a0, B, b, t, lib=lib)
    bw = oracle.backward(X, A0, B, fw["H"], fw["Y"], dZ, t, lib=lib)
    if _rel(fw["Z"], np.tile(b, (T, 1))) > 0:
        f.append("A = 0, a = 0: Z != b")
    if _rel(bw["dY"], 0.5 * dZ @ B.T) > 1e-12:
        f.append("A = 0, a = 0: dY != dZ B^T / 2")
    if np.max(np.abs(bw["dX"])) != 0.0:
        f.append("A = 0, a = 0: dX != 0")
    if np.max(np.abs(bw["dB"])) != 0.0:
        f.append("A = 0, a = 0: dB != 0 (Y = 0)")
    # db is the column sum of dZ whatever the weights
    if _rel(bw["db"], dZ.sum(axis=0)) > 1e-13:
        f.append("db != column sum of dZ")
    return f


def check_slice_vs_full(lib):
    f = []
    for (T, h, F), t, seed in [((13, 10, 24), 2, 400), ((128, 32, 64), 4, 401), ((7, 5, 16), 1, 402)]:
        X, A, a, B, b, dZ = _case(T, h, F, seed)
        full = oracle.forward_backward(X, A, a, B, b, dZ, t, lib=lib)
        rng = np.random.default_rng(seed)
        R = np.sort(rng.choice(T, size=min(T, 5), replace=False))
        J = np.sort(rng.choice(F, size=min(F, 7), replace=False))
        s = oracle.slice_(X, A, a, B, b, dZ, t, R, J, lib=lib)
        pairs = [("Hr", full["H"][R]), ("Yr", full["Y"][R]), ("dYr", full["dY"][R]),
                 ("Zr", full["Z"][R]), ("dXr", full["dX"][R]),
                 ("Hc", full["H"][:, J]), ("Yc", full["Y"][:, J]), ("dYc", full["dY"][:, J]),
                 ("dAc", full["dA"][:, J]), ("daJ", full["da"][J]), ("dBr", full["dB"][J]),
                 ("db", full["db"])]
        for k, ref in pairs:
            if _rel(s[k], ref) > 1e-12:
                f.append("slice %s differs from the full oracle (T=%d t=%d): %.3e"
                         % (k, T, t, _rel(s[k], ref)))
    return f


def check_layernorm_numpy(lib):
    """LayerNorm against numpy's population mean and variance (the textbook
    definition, Ba et al. 2016)."""
    f = []
    rng = np.random.default_rng(500)
    for T, h, eps in ((4, 16, 1e-5), (7, 33, 1e-6), (1, 8192, 1e-5)):
        X = rng.standard_normal((T, h)) * 3 + 1.5
        g = rng.standard_normal(h)
        b = rng.standard_normal(h)
        out = oracle.layernorm_forward(X, g, b, eps, lib=lib)
        mu = X.mean(axis=1, keepdims=True)
        var = X.var(axis=1, keepdims=True)
        ref = (X - mu) / np.sqrt(var + eps) * g + b
        if _rel(out["Y"], ref) > 1e-12:
            f.append("layernorm h=%d differs from numpy (%.3e)" % (h, _rel(out["Y"], ref)))
        if _rel(out["mean"], mu[:, 0]) > 1e-14 or _rel(out["rstd"], 1 / np.sqrt(var[:, 0] + eps)) > 1e-12:
            f.append("layernorm statistics differ from numpy")
    return f


def check_layernorm_invariants(lib):
    f = []
    rng = np.random.default_rng(501)
    T, h = 5, 64
    X = rng.standard_normal((T, h))
    one, zero = np.ones(h), np.zeros(h)
    y = oracle.layernorm_forward(X, one, zero, 0.0, lib=lib)["Y"]
    if np.max(np.abs(y.mean(axis=1))) > 1e-14 or np.max(np.abs(y.var(axis=1) - 1)) > 1e-13:
        f.append("normalised rows do not have mean 0 and variance 1")
    y2 = oracle.layernorm_forward(3.7 * X - 2.0, one, zero, 0.0, lib=lib)["Y"]
    if _rel(y2, y) > 1e-12:
        f.append("layernorm is not invariant to a positive scale and a shift of the row")
    # dX is orthogonal to the all-ones and to xhat directions (LN is invariant to both)
    dY = rng.standard_normal((T, h))
    bw = oracle.layernorm_backward(dY, X, one, 0.0, lib=lib)
    xh = y
    if np.max(np.abs(bw["dX"].sum(axis=1))) > 1e-12 or np.max(np.abs((bw["dX"] * xh).sum(axis=1))) > 1e-11:
        f.append("layernorm dX is not orthogonal to 1 and xhat")
    if _rel(bw["dbeta"], dY.sum(axis=0)) > 1e-13:
        f.append("dbeta != column sum of dY")
    return f


def check_layernorm_backward_fd(lib, eps_fd=1e-6, tol=1e-6):
    f = []
    rng = np.random.default_rng(502)
    T, h, eps = 3, 5, 1e-5
    X = rng.standard_normal((T, h)) * 2
    g = rng.standard_normal(h)
    b = rng.standard_normal(h)
    dY = rng.standard_normal((T, h))

    def loss():
        return float(np.sum(dY * oracle.layernorm_forward(X, g, b, eps, lib=lib)["Y"]))

    bw = oracle.layernorm_backward(dY, X, g, eps, lib=lib)
    for name, p, grad in (("X", X, bw["dX"]), ("gamma", g, bw["dgamma"]), ("beta", b, bw["dbeta"])):
        fd = np.empty_like(p)
        flat = p.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps_fd
            lp = loss()
            flat[i] = old - eps_fd
            lm = loss()
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * eps_fd)
        if _rel(grad, fd) > tol:
            f.append("layernorm d%s vs finite differences: rel %.3e" % (name, _rel(grad, fd)))
    return f


def check_sp_composition_fd(lib, eps_fd=1e-6, tol=1e-6):
    """The sequence-parallel block (LayerNorm, then the sharded MLP) as one
    function: finite differences of L = sum(dZ * Z) w.r.t. its input rows and the
    LayerNorm parameters."""
    f = []
    rng = np.random.default_rng(503)
    T, h, F, t, eps = 3, 4, 8, 2, 1e-5
    Xi = rng.standard_normal((T, h)) * 2
    g = rng.standard_normal(h)
    be = rng.standard_normal(h)
    _, A, a, B, b, dZ = _case(T, h, F, 504)

    def loss():
        xn = oracle.layernorm_forward(Xi, g, be, eps, lib=lib)["Y"]
        return float(np.sum(dZ * oracle.forward(xn, A, a, B, b, t, lib=lib)["Z"]))

    out = oracle.sp_forward_backward(Xi, g, be, eps, A, a, B, b, dZ, t, lib=lib)
    for name, p, grad in (("X_in", Xi, out["dX_in"]), ("gamma", g, out["dgamma"]), ("beta", be, out["dbeta"])):
        fd = np.empty_like(p)
        flat = p.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps_fd
            lp = loss()
            flat[i] = old - eps_fd
            lm = loss()
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * eps_fd)
        if _rel(grad, fd) > tol:
            f.append("sequence-parallel block d%s vs finite differences: rel %.3e" % (name, _rel(grad, fd)))
    return f


def _attn_perm(h, heads, t):
    """Column permutation from the canonical [Q | K | V] layout (heads in order)
    to the shard-major layout [Q_0 | K_0 | V_0 | Q_1 | ...] of t shards."""
    d, hpt, hs = h // heads, heads // t, h // t
    perm = []
    for i in range(t):
        for which in range(3):
            for j in range(hpt):
                g = i * hpt + j
                perm.extend(range(which * h + g * d, which * h + (g + 1) * d))
    return np.array(perm)


def _attn_case(nb, S, h, seed):
    rng = np.random.default_rng(seed)
    T = nb * S
    return (rng.standard_normal((T, h)), rng.standard_normal((h, 3 * h)) * 0.5,
            rng.standard_normal(3 * h) * 0.3, rng.standard_normal((h, h)) * 0.5,
            rng.standard_normal(h) * 0.3, rng.standard_normal((T, h)))


def _numpy_attention(X, Wc, bc, Wo, bo, nb, heads):
    """Causal multi-head attention from numpy primitives, canonical [Q|K|V] layout."""
    T, h = X.shape
    S, d = T // nb, h // heads
    qkv = X @ Wc + bc
    q = qkv[:, :h].reshape(nb, S, heads, d).transpose(0, 2, 1, 3)
    k = qkv[:, h:2 * h].reshape(nb, S, heads, d).transpose(0, 2, 1, 3)
    v = qkv[:, 2 * h:].reshape(nb, S, heads, d).transpose(0, 2, 1, 3)
    sc = np.einsum("bgrd,bgcd->bgrc", q, k) / np.sqrt(d)
    sc = np.where(np.tril(np.ones((S, S), dtype=bool)), sc, -np.inf)
    sc = sc - sc.max(axis=-1, keepdims=True)
    p = np.exp(sc)
    p /= p.sum(axis=-1, keepdims=True)
    o = np.einsum("bgrc,bgcd->bgrd", p, v).transpose(0, 2, 1, 3).reshape(T, h)
    return p, o, o @ Wo + bo


def check_attn_numpy(lib):
    f = []
    nb, S, h, heads = 2, 5, 8, 2
    X, Wc, bc, Wo, bo, _ = _attn_case(nb, S, h, 600)
    p_ref, o_ref, z_ref = _numpy_attention(X, Wc, bc, Wo, bo, nb, heads)
    for t in (1, 2):
        perm = _attn_perm(h, heads, t)
        out = oracle.attn_forward(X, Wc[:, perm], bc[perm], Wo, bo, nb, heads, t, lib=lib)
        for name, got, ref in (("P", out["P"], p_ref), ("O", out["O"], o_ref), ("Z", out["Z"], z_ref)):
            if _rel(got, ref) > 1e-12:
                f.append("attention %s (t=%d) differs from numpy: %.3e" % (name, t, _rel(got, ref)))
    return f


def check_attn_sharding(lib):
    """Z is the same for t = 1, 2, 4 once Wqkv's columns are laid out shard-major,
    i.e. the head split of the report's section 4.1 does not change the result."""
    f = []
    nb, S, h, heads = 2, 4, 16, 4
    X, Wc, bc, Wo, bo, dZ = _attn_case(nb, S, h, 601)
    ref = None
    for t in (1, 2, 4):
        perm = _attn_perm(h, heads, t)
        fw = oracle.attn_forward(X, Wc[:, perm], bc[perm], Wo, bo, nb, heads, t, lib=lib)
        bw = oracle.attn_backward(X, Wc[:, perm], Wo, fw["QKV"], fw["P"], fw["O"], dZ, nb, heads, t, lib=lib)
        inv = np.argsort(perm)
        got = {"Z": fw["Z"], "dX": bw["dX"], "dWo": bw["dWo"], "dWqkv": bw["dWqkv"][:, inv]}
        if ref is None:
            ref = got
        for k in got:
            if _rel(got[k], ref[k]) > 1e-12:
                f.append("attention %s for t=%d differs from t=1" % (k, t))
    return f


def check_attn_causal(lib):
    f = []
    nb, S, h, heads, t = 2, 6, 8, 2, 2
    X, Wc, bc, Wo, bo, _ = _attn_case(nb, S, h, 602)
    out = oracle.attn_forward(X, Wc, bc, Wo, bo, nb, heads, t, lib=lib)
    P = out["P"]
    if np.max(np.abs(P.sum(axis=-1) - 1)) > 1e-14:
        f.append("attention rows do not sum to 1")
    if np.max(np.abs(np.triu(P, 1))) != 0.0:
        f.append("attention puts weight on later positions")
    X2 = X.copy()
    X2[S + 3] += 1.0  # token 3 of sequence 1
    Z2 = oracle.attn_forward(X2, Wc, bc, Wo, bo, nb, heads, t, lib=lib)["Z"]
    dz = np.abs(Z2 - out["Z"]).max(axis=1)
    if dz[:S + 3].max() != 0.0 or dz[S + 3:].min() == 0.0:
        f.append("a token changes outputs of earlier tokens or of another sequence")
    return f


def check_attn_fd(lib, eps_fd=1e-6, tol=1e-6):
    f = []
    nb, S, h, heads, t = 2, 3, 4, 2, 2
    X, Wc, bc, Wo, bo, dZ = _attn_case(nb, S, h, 603)

    def loss():
        return float(np.sum(dZ * oracle.attn_forward(X, Wc, bc, Wo, bo, nb, heads, t, lib=lib)["Z"]))

    out = oracle.attn_forward_backward(X, Wc, bc, Wo, bo, dZ, nb, heads, t, lib=lib)
    for name, p, grad in (("X", X, out["dX"]), ("Wqkv", Wc, out["dWqkv"]), ("bqkv", bc, out["dbqkv"]),
                          ("Wo", Wo, out["dWo"]), ("bo", bo, out["dbo"])):
        fd = np.empty_like(p)
        flat = p.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps_fd
            lp = loss()
            flat[i] = old - eps_fd
            lm = loss()
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * eps_fd)
        if _rel(grad, fd) > tol:
            f.append("attention d%s vs finite differences: rel %.3e" % (name, _rel(grad, fd)))
    return f


def check_layernorm_worked_example(lib):
    """LayerNorm worked by hand (the sequence-parallel block's first step), eps = 0:
      x = [1, 3, 1, 3]: mean 2, population variance 1, rstd 1, xhat = [-1, 1, -1, 1]
      x = [0, 0, 4, 4]: mean 2, variance 4, rstd 1/2, xhat = [-1, -1, 1, 1]
    With gamma = [1, 2, 1/2, -1], beta = [0, 1, -1, 1/2]: y = gamma xhat + beta.
    Backward for dY = [[1, 0, 2, -1], [0, 1, 1, 2]]: g = dY gamma,
      dx = rstd (g - mean(g) - xhat mean(g xhat)),  dgamma = sum dY xhat,
      dbeta = sum dY."""
    X = np.array([[1.0, 3, 1, 3], [0, 0, 4, 4]])
    gamma = np.array([1.0, 2, 0.5, -1])
    beta = np.array([0.0, 1, -1, 0.5])
    dY = np.array([[1.0, 0, 2, -1], [0, 1, 1, 2]])
    want = {"Y": [[-1, 3, -1.5, -0.5], [-1, -1, -0.5, -0.5]], "mean": [2, 2], "rstd": [1, 0.5],
            "dX": [[0, -0.5, 0, 0.5], [-0.5, 0.5, 0.625, -0.625]], "dgamma": [-1, -1, -1, 1],
            "dbeta": [1, 1, 3, 1]}
    fw = oracle.layernorm_forward(X, gamma, beta, 0.0, lib=lib)
    bw = oracle.layernorm_backward(dY, X, gamma, 0.0, lib=lib)
    got = dict(fw, **bw)
    f = []
    for k, v in want.items():
        err = float(np.max(np.abs(np.asarray(got[k]) - np.asarray(v))))
        if err > 1e-14:
            f.append("LayerNorm worked example: %s differs by %.3e" % (k, err))
    return f


def check_golden_attention_worked_example(lib):
    """The hand-worked attention example of tests/golden/attention_worked_example.txt
    (one sequence of two tokens, one head of d = 4, equal keys so that the second
    row's probabilities are exactly 1/2): forward and every gradient.  Equal
    logits make the softmax blind to the 1/sqrt(d) scale of the scores; the
    numpy and finite-difference pins cover that."""
    g = read_golden("attention_worked_example.txt")
    nb, heads, t = g["nb"], g["heads"], g["t"]
    fw = oracle.attn_forward(g["X"], g["Wqkv"], g["bqkv"].ravel(), g["Wo"], g["bo"].ravel(), nb, heads, t, lib=lib)
    bw = oracle.attn_backward(g["X"], g["Wqkv"], g["Wo"], fw["QKV"], fw["P"], fw["O"], g["dZ"], nb, heads, t,
                              lib=lib)
    got = {"QKV": fw["QKV"], "P": fw["P"].reshape(g["P"].shape), "O": fw["O"], "Z": fw["Z"],
           "dbo": bw["dbo"][None, :], "dWo": bw["dWo"], "dWqkv": bw["dWqkv"], "dbqkv": bw["dbqkv"][None, :],
           "dX": bw["dX"]}
    f = []
    for k, v in got.items():
        err = float(np.max(np.abs(v - g[k])))
        if err > 1e-12 * max(1.0, float(np.max(np.abs(g[k])))):
            f.append("golden attention example: %s differs by %.3e" % (k, err))
    return f


ALL = [check_gelu_vs_erf, check_gelu_identities, check_gelu_prime_fd, check_forward_numpy,
       check_worked_example_t2, check_golden_worked_example_t2, check_backward_fd, check_backward_partials,
       check_closed_forms, check_slice_vs_full, check_layernorm_numpy, check_layernorm_invariants,
       check_layernorm_backward_fd, check_sp_composition_fd, check_attn_numpy, check_attn_sharding,
       check_attn_causal, check_attn_fd, check_golden_attention_worked_example, check_layernorm_worked_example]


def run_all(lib) -> list:
    out = []
    for c in ALL:
        try:
            out += ["%s: %s" % (c.__name__, m) for m in c(lib)]
        except Exception as e:  # a planted mistake may also make a check raise
            out.append("%s raised %r" % (c.__name__, e))
    return out
