"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is a one-line edit of ``oracle/oracle.c`` compiled into a temporary
library on the CPU; the shipped oracle is never touched.  A mutant that no pin
catches would mean the pins leave that part of the oracle unchecked.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins

MUTANTS = {
    # the bias b added once per shard instead of once after the all-reduce
    "bias_per_shard": ("Z[r * h + j] = b[j] + sum[j];", "Z[r * h + j] = t * b[j] + sum[j];"),
    # wrong cubic coefficient in the tanh argument of GeLU
    "gelu_constant": ("    double u = c * (x + 0.044715 * x * x * x);\n    return",
                      "    double u = c * (x + 0.05 * x * x * x);\n    return"),
    # derivative of tanh(u) without the inner derivative du/dx
    "gelu_prime_chain": ("0.5 * x * (1.0 - th * th) * du;", "0.5 * x * (1.0 - th * th);"),
    # sign error in dY
    "dY_sign": ("dY[r * F + f] = g * oracle_gelu_prime", "dY[r * F + f] = -g * oracle_gelu_prime"),
    # transposed / misindexed operand in dA = X^T dY
    "dA_index": ("for (int64_t f = 0; f < F; ++f) dAk[f] += x * dYr[f];",
                 "for (int64_t f = 0; f < F; ++f) dAk[f] += x * dYr[F - 1 - f];"),
    # the backward all-reduce drops the last shard
    "dX_drop_shard": ("                if (dXpart) dXpart[((int64_t)i * T + r) * h + k] = p;\n"
                      "                sum += p;",
                      "                if (dXpart) dXpart[((int64_t)i * T + r) * h + k] = p;\n"
                      "                if (i + 1 < t || t == 1) sum += p;"),
    # da summed over the wrong column
    "da_column": ("for (int64_t r = 0; r < T; ++r) s += dY[r * F + f];",
                  "for (int64_t r = 0; r < T; ++r) s += dY[r * F + (f + 1) % F];"),
    # the forward uses the wrong shard range for the row-parallel GEMM
    "shard_range": ("for (int64_t f = i * Fs; f < (i + 1) * Fs; ++f) {\n                    const double yf = Yr[f];",
                    "for (int64_t f = i * Fs; f < (i + 1) * Fs - 1; ++f) {\n                    const double yf = Yr[f];"),
    # the slice oracle reads the wrong token row
    "slice_row": ("const int64_t r = R[q];", "const int64_t r = (R[q] + 1) % T;"),
    # LayerNorm with the sample variance (h - 1) instead of the population variance
    "ln_sample_var": ("        v /= (double)h;\n        const double rs = 1.0 / sqrt(v + eps);\n        for (int64_t j = 0; j < h; ++j) Y[",
                      "        v /= (double)(h - 1);\n        const double rs = 1.0 / sqrt(v + eps);\n        for (int64_t j = 0; j < h; ++j) Y["),
    # LayerNorm backward without the projection onto xhat
    "ln_bwd_drop_term": ("dX[r * h + j] = rstd * (dy[j] * gamma[j] - mg - xh * mgx);",
                         "dX[r * h + j] = rstd * (dy[j] * gamma[j] - mg);"),
    # dgamma without xhat
    "ln_dgamma": ("sg += dY[r * h + j] * (X[r * h + j] - mu[r]) * rs[r];", "sg += dY[r * h + j];"),
    # LayerNorm forward: eps added outside the square root
    "ln_eps_outside": ("const double rs = 1.0 / sqrt(v + eps);", "const double rs = 1.0 / sqrt(v) + eps;"),
    # LayerNorm forward: beta added before the gamma scale
    "ln_beta_inside": ("Y[r * h + j] = (x[j] - mu) * rs * gamma[j] + beta[j];",
                       "Y[r * h + j] = ((x[j] - mu) * rs + beta[j]) * gamma[j];"),
    # attention without the causal mask on the scores
    "attn_no_mask": ("const int64_t last = r; /* causal", "const int64_t last = S - 1; /* causal"),
    # scores without the 1/sqrt(d) scale
    "attn_no_scale": ("Pg[r * S + c] = sc * scale;", "Pg[r * S + c] = sc;"),
    # softmax backward without the row term D
    "attn_ds_no_D": ("const double ds = Pg[r * S + c] * (dP[c] - D) * scale;",
                     "const double ds = Pg[r * S + c] * dP[c] * scale;"),
    # dK built from K instead of Q
    "attn_dk_operand": ("dk[e] += ds * qr[e];", "dk[e] += ds * kr[e];"),
    # dV from the transposed probability (P[c][r] instead of P[r][c])
    "attn_dv_transposed_p": ("dv[e] += Pg[r * S + c] * dor[e];", "dv[e] += Pg[c * S + r] * dor[e];"),
    # dQ built from Q instead of K
    "attn_dq_operand": ("dq[e] += ds * kr[e];", "dq[e] += ds * qr[e];"),
    # dbqkv summed over the wrong column
    "attn_dbqkv_column": ("for (int64_t r = 0; r < T; ++r) sb += dQKV[r * H3 + c];",
                          "for (int64_t r = 0; r < T; ++r) sb += dQKV[r * H3 + (c + 1) % H3];"),
    # the softmax row term D = rowsum(dP * P) without the P
    "attn_D_without_p": ("D += s * Pg[r * S + c];", "D += s;"),
    # dO read at the head's offset within its shard instead of its global offset
    "attn_head_offset": ("const double *dor = dO + (b * S + r) * h + g * d;",
                         "const double *dor = dO + (b * S + r) * h + (g % hpt) * d;"),
    # output projection: a shard's partial added twice
    "attn_fold": ("                for (int64_t c = 0; c < h; ++c) Z[r * h + c] += part[c];\n            }\n            for (int64_t c = 0; c < h; ++c) Z[r * h + c] += bo[c];",
                  "                for (int64_t c = 0; c < h; ++c) Z[r * h + c] += (i == 0 ? 2.0 : 1.0) * part[c];\n            }\n            for (int64_t c = 0; c < h; ++c) Z[r * h + c] += bo[c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, "mutation site for %s not found exactly once" % name
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mutant.c")
        so = os.path.join(d, "libmutant.so")
        with open(c, "w") as fh:
            fh.write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-fopenmp", "-std=c11", "-shared", "-fPIC", c, "-o", so, "-lm"],
                       check=True)
        lib = oracle.load(so)
        failures = oracle_pins.run_all(lib)
    assert failures, "planted mistake %r passed every pin" % name
