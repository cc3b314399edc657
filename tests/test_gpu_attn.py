"""Tensor-parallel self-attention block on the GPU against the fp64 oracle.

Heads are split among the t shards: the QKV projection is column-parallel, the
output projection row-parallel with the fixed-order shard fold ("Megatron-LM"
industry report, section 4.1).  Every case runs the tensor-core path through the
C ABI and compares, element by element, the saved activations (QKV, P, O), the
output Z and every gradient with the oracle on the same seeded bf16 inputs.
Shapes span several 256-wide tiles of the per-head products (whose causal
tile skipping and K ranges depend on the tile row), ragged sequence tails, every
softmax row-length class, head sizes 64 and 128, t = 1..4, and the empty batch.
"""
import numpy as np
import pytest
import torch

from gpu_cases import rel, to_np

pytestmark = pytest.mark.gpu

# max|out - ref| / max|ref|.  QKV comes out of one fp32-accumulated GEMM and is
# stored in bf16: 1e-2 as for the MLP's outputs.  Everything downstream of the
# logits carries two bf16 roundings in a row: Q and K are stored in bf16 (unit
# roundoff u = 2^-9), which moves a logit s by up to about 2u|s| (|s| reaches 10
# and more when the logit std is about 3, as at h = 8192 with weights of std
# 0.02), and P is rounded to bf16 again before P V.  Observed errors there are
# about 1.1e-2 at that logit scale: P, O and Z are held to 2e-2, the gradients
# (through dO, dS and dQKV, also stored in bf16) to 3e-2.
TOL = {"QKV": 1e-2, "P": 2e-2, "O": 2e-2, "Z": 2e-2,
       "dX": 3e-2, "dWqkv": 3e-2, "dbqkv": 3e-2, "dWo": 3e-2, "dbo": 3e-2}

# Weights large enough that the softmax is far from uniform: at h = 512 the
# logits have a standard deviation of about 1.3.
STD = {"X": 1.0, "Wqkv": 0.05, "bqkv": 0.1, "Wo": 0.04, "bo": 0.1, "dZ": 1.0}

# Peaky logits (std about 3.3, as in the h = 8192 workload).
STD_PEAKY = dict(STD, Wqkv=0.08)


@pytest.fixture(scope="module")
def tp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from tensor_transformer_mlp_tma_gb300 import tpmlp
    return tpmlp


def run_attn(tp, nb, S, h, heads, t, seed, std=STD, perm=None):
    """perm, if given, reorders the columns of Wqkv and bqkv (a layout change)."""
    from tensor_transformer_mlp_tma_gb300 import inputs
    inp = inputs.make_attn(nb * S, h, seed, std)
    if perm is not None:
        pt = torch.as_tensor(perm)
        inp = dict(inp, Wqkv=inp["Wqkv"][:, pt].contiguous(), bqkv=inp["bqkv"][pt].contiguous())
    d = {k: v.cuda() for k, v in inp.items()}
    ctx = tp.AttnContext(nb, S, h, heads, t)
    Z = tp.attn_forward(ctx, d["X"], d["Wqkv"], d["bqkv"], d["Wo"], d["bo"])
    g = tp.attn_backward(ctx, d["dZ"])
    torch.cuda.synchronize()
    assert tp.check_device_status(ctx) == tp.OK
    out = {"QKV": ctx.QKV, "P": ctx.P.view(nb, heads, S, S), "O": ctx.O, "Z": Z}
    out.update(g)
    return inp, out, ctx


def shard_major(h, heads, t):
    """Column permutation from the [Q | K | V] layout (heads in order) to the
    shard-major layout [Q_1 | K_1 | V_1 | Q_2 | ...] the library takes."""
    d, hpt = h // heads, heads // t
    perm = []
    for i in range(t):
        for which in range(3):
            for j in range(hpt):
                g = i * hpt + j
                perm.extend(range(which * h + g * d, which * h + (g + 1) * d))
    return np.array(perm)


def oracle_ref(inp, nb, heads, t):
    import oracle
    f = {k: v.double().numpy() for k, v in inp.items()}
    return oracle.attn_forward_backward(f["X"], f["Wqkv"], f["bqkv"], f["Wo"], f["bo"], f["dZ"], nb, heads, t)


CASES = [
    # nb, S, h, heads, t
    (2, 256, 512, 4, 2),     # d = 128, one 256 x 256 score tile per head
    (1, 520, 512, 8, 4),     # d = 64, three score tiles with a ragged tail of 8
    (3, 136, 384, 3, 3),     # ragged single tile, t = 3
    (2, 384, 256, 2, 1),     # t = 1
    (2, 256, 1024, 16, 8),   # t = 8 shards of two heads (d = 64), as in the bench's shard count
    (1, 2056, 256, 2, 2),    # rows past 2048 columns (widest register softmax)
    (1, 4104, 128, 1, 1),    # rows past 4096 columns (multi-pass softmax)
]


@pytest.mark.parametrize("nb,S,h,heads,t", CASES)
def test_attention_matches_oracle(tp, nb, S, h, heads, t):
    inp, out, _ = run_attn(tp, nb, S, h, heads, t, seed=11 + S)
    ref = oracle_ref(inp, nb, heads, t)
    errs = {k: rel(to_np(out[k]), ref[k]) for k in TOL}
    print("attention %s errors:" % ((nb, S, h, heads, t),), {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not (v <= TOL[k])}
    assert not bad, "outside tolerance: %s (all: %s)" % (bad, errs)


def test_attention_peaky_logits_match_oracle(tp):
    nb, S, h, heads, t = 1, 520, 512, 8, 4
    inp, out, _ = run_attn(tp, nb, S, h, heads, t, seed=7, std=STD_PEAKY)
    ref = oracle_ref(inp, nb, heads, t)
    errs = {k: rel(to_np(out[k]), ref[k]) for k in TOL}
    print("attention, peaky logits, errors:", {k: "%.2e" % v for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not (v <= TOL[k])}
    assert not bad, "outside tolerance: %s (all: %s)" % (bad, errs)


def test_causal_probabilities_are_exact_zero_above_diagonal(tp):
    nb, S, h, heads, t = 1, 264, 256, 2, 2
    _, out, _ = run_attn(tp, nb, S, h, heads, t, seed=5)
    P = out["P"].float()
    upper = torch.triu(torch.ones(S, S, dtype=torch.bool, device=P.device), diagonal=1)
    assert torch.all(P[..., upper] == 0)
    # each row is a distribution (bf16 rounding of up to S terms)
    rs = P.sum(-1)
    assert torch.all((rs - 1).abs() < 2e-2)


def test_huge_logits_saturate_and_stay_finite(tp):
    """The scores are kept in fp16, whose largest finite value is 65504.  With
    weights large enough that the scaled logits reach far beyond it, the score
    epilogue saturates them instead of producing infinities, so the softmax sees
    no inf - inf: P and every output stay finite, P's rows still sum to one, its
    upper triangle stays exactly zero, and each row's largest probability sits
    where the oracle's largest logit is (rows whose two largest logits, in the
    oracle, both exceed the fp16 range are skipped)."""
    import oracle
    nb, S, h, heads, t = 1, 136, 256, 2, 1
    std = dict(STD, Wqkv=11.0)  # logit std ~ 256 * 11^2 = 3e4: a few percent past 65504
    inp, out, _ = run_attn(tp, nb, S, h, heads, t, seed=21, std=std)
    for k, v in out.items():
        assert torch.isfinite(v.float()).all(), k
    P = out["P"].float()
    upper = torch.triu(torch.ones(S, S, dtype=torch.bool, device=P.device), diagonal=1)
    assert torch.all(P[..., upper] == 0)
    assert torch.all((P.sum(-1) - 1).abs() < 2e-2)
    # the oracle's logits, from the same QKV the GPU computed (bf16, in place)
    q = out["QKV"].double().cpu().numpy()
    d = h // heads
    for g in range(heads):
        Q, K = q[:, g * d:(g + 1) * d], q[:, h + g * d:h + (g + 1) * d]
        s = (Q @ K.T) / np.sqrt(d)
        s[np.triu_indices(S, 1)] = -np.inf
        top2 = np.sort(s, axis=1)[:, -2:]
        ok = ~(top2[:, 0] > 65504.0)          # at most one logit past the fp16 range
        ok &= (top2[:, 1] - top2[:, 0]) > 1.0  # a clear winner
        got = P[0, g].argmax(-1).cpu().numpy()
        want = s.argmax(1)
        assert (top2[:, 1] > 65504.0).any()   # some rows do saturate
        assert ok.sum() >= 10
        assert np.array_equal(got[ok], want[ok])


def test_attention_is_bit_identical_across_runs(tp):
    nb, S, h, heads, t = 2, 256, 512, 4, 4
    _, a, _ = run_attn(tp, nb, S, h, heads, t, seed=3)
    a = {k: v.clone() for k, v in a.items()}
    _, b, _ = run_attn(tp, nb, S, h, heads, t, seed=3)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_sharding_does_not_change_the_math(tp):
    """One model, its Wqkv columns laid out for t = 1 and for t = 4: the results
    agree within the bf16 tolerance (the head split and the shard fold only
    regroup fp32 sums; dWqkv comes back in each run's own column layout)."""
    nb, S, h, heads = 1, 256, 512, 8
    runs = {}
    for t in (1, 4):
        perm = shard_major(h, heads, t)
        _, out, _ = run_attn(tp, nb, S, h, heads, t, seed=21, perm=perm)
        out = dict(out, dWqkv=out["dWqkv"][:, torch.as_tensor(np.argsort(perm), device="cuda")])
        runs[t] = out
    for k in ("Z", "dX", "dWqkv", "dWo", "dbo"):
        assert rel(to_np(runs[4][k]), to_np(runs[1][k])) < 1e-2, k


def test_empty_batch(tp):
    ctx = tp.AttnContext(0, 64, 256, 2, 2)
    z = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    W = torch.randn(256, 768, device="cuda").bfloat16()
    Wo = torch.randn(256, 256, device="cuda").bfloat16()
    bq = torch.zeros(768, device="cuda").bfloat16()
    bo = torch.zeros(256, device="cuda").bfloat16()
    Z = tp.attn_forward(ctx, z, W, bq, Wo, bo)
    assert Z.shape == (0, 256)
    g = tp.attn_backward(ctx, z)
    torch.cuda.synchronize()
    for k in ("dWqkv", "dbqkv", "dWo", "dbo"):
        assert torch.count_nonzero(g[k]) == 0, k


def test_rejects_unsupported_shapes(tp):
    # head size 32 (not a multiple of 64) and seq not a multiple of 8
    for args in ((1, 64, 256, 8, 2), (1, 60, 256, 2, 2)):
        ctx = tp.AttnContext(*args)
        nb, S, h = args[0], args[1], args[2]
        X = torch.zeros((nb * S, h), dtype=torch.bfloat16, device="cuda")
        W = torch.zeros((h, 3 * h), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(tp.TpmlpError) as e:
            tp.attn_forward(ctx, X, W, torch.zeros(3 * h, dtype=torch.bfloat16, device="cuda"),
                            torch.zeros((h, h), dtype=torch.bfloat16, device="cuda"),
                            torch.zeros(h, dtype=torch.bfloat16, device="cuda"))
        assert e.value.status == tp.ERR_UNSUPPORTED


def test_full_size_prefix_matches_oracle(tp):
    """At the benchmark's size (h = 8192, 64 heads of 128, t = 8, two sequences of
    2048) the causal mask makes the first rows of each sequence depend only on
    the rows before them: the oracle runs on a 64-token prefix of each sequence
    and must match those rows of QKV, O and Z and the prefix block of P."""
    from tensor_transformer_mlp_tma_gb300 import inputs
    from tensor_transformer_mlp_tma_gb300.workloads import ATTN_WORKLOADS
    import oracle
    w = ATTN_WORKLOADS["attn-h8192"]
    inp = inputs.make_attn(w.tokens, w.hidden, 0, {"Wqkv": w.std_W, "Wo": w.std_W, "bqkv": w.std_b,
                                                  "bo": w.std_b})
    d = {k: v.cuda() for k, v in inp.items() if k != "dZ"}
    ctx = tp.AttnContext(w.batch, w.seq, w.hidden, w.heads, w.t)
    Z = tp.attn_forward(ctx, d["X"], d["Wqkv"], d["bqkv"], d["Wo"], d["bo"])
    torch.cuda.synchronize()
    assert tp.check_device_status(ctx) == tp.OK
    pre = 64
    P = ctx.P.view(w.batch, w.heads, w.seq, w.seq)
    f = {k: v.double().numpy() for k, v in inp.items()}
    for b in range(w.batch):
        rows = slice(b * w.seq, b * w.seq + pre)
        ref = oracle.attn_forward(f["X"][rows], f["Wqkv"], f["bqkv"], f["Wo"], f["bo"], 1, w.heads, w.t)
        got = {"QKV": ctx.QKV[rows], "O": ctx.O[rows], "Z": Z[rows], "P": P[b, :, :pre, :pre]}
        for k, v in got.items():
            e = rel(to_np(v), ref[k].reshape(to_np(v).shape))
            print("attn-h8192 prefix, sequence %d, %s error %.2e" % (b, k, e))
            assert e <= TOL[k], (b, k, e)
        # probabilities past the prefix are zero on the prefix rows
        assert torch.count_nonzero(P[b, :, :pre, pre:]) == 0


def test_attention_single_cta_tiles_match_oracle(tp, monkeypatch):
    """128-row tiles on single CTAs: the causal tile skipping and K ranges follow
    the tile height."""
    monkeypatch.setenv("TPMLP_CTA_PAIR", "0")
    nb, S, h, heads, t = 1, 520, 512, 8, 4
    inp, out, _ = run_attn(tp, nb, S, h, heads, t, seed=9)
    ref = oracle_ref(inp, nb, heads, t)
    errs = {k: rel(to_np(out[k]), ref[k]) for k in TOL}
    bad = {k: v for k, v in errs.items() if not (v <= TOL[k])}
    assert not bad, "outside tolerance: %s (all: %s)" % (bad, errs)


def test_tile_order_does_not_change_results(tp, monkeypatch):
    """The causal per-head products walk odd problems' M-tiles backwards (load
    balance); each output element is still made by one tile with the same K
    order, so both orders give bit-identical results."""
    nb, S, h, heads, t = 2, 520, 512, 8, 4
    _, fwd, _ = run_attn(tp, nb, S, h, heads, t, seed=21)
    monkeypatch.setenv("TPMLP_FLIP_ODD", "0")
    _, inorder, _ = run_attn(tp, nb, S, h, heads, t, seed=21)
    for k in TOL:
        assert torch.equal(fwd[k], inorder[k]), k


def test_wide_tiles_match_oracle(tp, monkeypatch):
    """The per-head products with N = d take 256 x 128 tiles by default;
    TPMLP_NARROW=0 runs them on the 256 x 256 tiles, with the same results."""
    monkeypatch.setenv("TPMLP_NARROW", "0")
    nb, S, h, heads, t = 1, 520, 512, 8, 4
    inp, out, _ = run_attn(tp, nb, S, h, heads, t, seed=10)
    ref = oracle_ref(inp, nb, heads, t)
    errs = {k: rel(to_np(out[k]), ref[k]) for k in TOL}
    bad = {k: v for k, v in errs.items() if not (v <= TOL[k])}
    assert not bad, "outside tolerance: %s (all: %s)" % (bad, errs)


def test_projections_on_square_tiles_match_wide(tp, monkeypatch):
    """The QKV projection (bias, no activation), dO = dZ Wo^T (two K-major
    operands), dWo and dWqkv run on 256 x 512 tiles by default; TPMLP_WIDE=0
    runs them on 256 x 256 tiles.  All match the oracle, and with every wave
    walking K upwards (TPMLP_SERPENTINE=0) each output element is accumulated
    over k in the same order by the same MMA shape, so the two give the same
    bits."""
    nb, S, h, heads, t = 2, 264, 1024, 8, 4
    inp, default, _ = run_attn(tp, nb, S, h, heads, t, seed=31)
    ref = oracle_ref(inp, nb, heads, t)
    monkeypatch.setenv("TPMLP_SERPENTINE", "0")
    _, wide, _ = run_attn(tp, nb, S, h, heads, t, seed=31)
    for out in (default, wide):
        errs = {k: rel(to_np(out[k]), ref[k]) for k in TOL}
        assert all(v <= TOL[k] for k, v in errs.items()), errs
    monkeypatch.setenv("TPMLP_WIDE", "0")
    _, square, _ = run_attn(tp, nb, S, h, heads, t, seed=31)
    for k in TOL:
        assert torch.equal(wide[k], square[k]), k


@pytest.mark.parametrize("pair", ["1", "0"])
def test_p_upper_tiles_flag(tp, pair, monkeypatch):
    """TPMLP_ATTN_P_UPPER_ZERO leaves the 256 x 256 tiles of P wholly above the
    diagonal as they were and writes everything else as without the flag; no
    later kernel reads those tiles (CTA-pair 256-row or single-CTA 128-row
    tiles), so every output is bit-identical.  Without the flag every row of P
    is written in full (sentinel values overwritten)."""
    from tensor_transformer_mlp_tma_gb300 import inputs
    monkeypatch.setenv("TPMLP_CTA_PAIR", pair)
    nb, S, h, heads, t = 2, 520, 512, 4, 2   # 3 tile rows of 256, ragged last
    inp = inputs.make_attn(nb * S, h, 31, STD)
    d = {k: v.cuda() for k, v in inp.items()}
    res = {}
    for flag in (False, True):
        ctx = tp.AttnContext(nb, S, h, heads, t, p_upper_zero=flag)
        ctx.P.fill_(7.0)  # a sentinel in every entry
        Z = tp.attn_forward(ctx, d["X"], d["Wqkv"], d["bqkv"], d["Wo"], d["bo"])
        g = tp.attn_backward(ctx, d["dZ"])
        torch.cuda.synchronize()
        assert tp.check_device_status(ctx) == tp.OK
        res[flag] = dict(g, Z=Z, P=ctx.P.clone(), O=ctx.O.clone(), QKV=ctx.QKV.clone())
    s = torch.arange(S, device="cuda")
    upper = (s[None, :] // 256) > (s[:, None] // 256)  # [S, S]: tile column past the tile row
    P0, P1 = res[False]["P"], res[True]["P"]
    assert torch.count_nonzero(P0[:, upper]) == 0                   # written as zeros
    assert bool((P1[:, upper] == 7.0).all())                        # left as they were
    assert torch.equal(P0[:, ~upper], P1[:, ~upper])
    for k in ("Z", "O", "QKV", "dX", "dWqkv", "dbqkv", "dWo", "dbo"):
        assert torch.equal(res[False][k], res[True][k]), k


@pytest.mark.parametrize("units", [None, "5", "3"])
def test_pair_order_gives_the_same_bits(tp, units, monkeypatch):
    """The causal products against P and dS hand each unit complementary pairs
    of M-tiles (TPMLP_PAIR_ORDER, default) instead of reversing odd problems.
    Only the unit that computes a tile changes, so every output is bit-identical
    to the other order, and matches the oracle; small unit counts exercise the
    full double rounds and the leftover slots on a small shape."""
    if units:
        monkeypatch.setenv("TPMLP_MAX_UNITS", units)
    nb, S, h, heads, t = 2, 1024, 512, 4, 2   # 4 M-tiles of 256 per head, 8 problems
    inp, paired, _ = run_attn(tp, nb, S, h, heads, t, seed=47)
    ref = oracle_ref(inp, nb, heads, t)
    errs = {k: rel(to_np(paired[k]), ref[k]) for k in TOL}
    assert all(v <= TOL[k] for k, v in errs.items()), errs
    monkeypatch.setenv("TPMLP_PAIR_ORDER", "0")
    _, flipped, _ = run_attn(tp, nb, S, h, heads, t, seed=47)
    for k in TOL:
        assert torch.equal(paired[k], flipped[k]), k
