/*
 * Oracle for the tensor-parallel Transformer MLP block.  TEST INFRASTRUCTURE:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load this code.  It shares nothing with the CUDA library and the CUDA library
 * never calls it.
 *
 * Plain, slow, obviously correct fp64 C, parallelised over independent output
 * rows/columns with OpenMP.  Every output element is produced by one thread in a
 * fixed summation order, so results do not depend on the thread count.
 *
 * Sources (the pages describe the method; no code is taken from them):
 *  - "Megatron-LM" (compassingai.com industry report), section 4.1 (basic
 *    principle of tensor parallelism): the MLP is Y = f(XA)B; the first weight is
 *    split by columns [W_{1,1}, W_{1,2}], the second by rows; the input X is
 *    replicated; shard i computes Y_i = f(X W_{1,i}) and Z_i = Y_i W_{2,i}; an
 *    all-reduce sums the partial Z_i into the full output.
 *  - same report, section 4.2: the tensor-parallel exchange happens in both the
 *    forward and the backward direction.
 *  - "In-Depth Analysis of Distributed Training Frameworks for Large Models ...
 *    Megatron-LM" (oreateai.com), section 2.2: the activation f is GeLU.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - biases: a is split with A's columns; b is added once, after the sum.
 *  - f is the tanh form of GeLU: 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3))).
 *  - backward is the plain chain rule for the scalar loss L = sum(dZ * Z).
 *  - the all-reduce is the fixed-order sum ((Z_0 + Z_1) + ...) + Z_{t-1}.
 *
 * Layout: every matrix is row-major and contiguous.  X[T,h], A[h,F], a[F],
 * B[F,h], b[h], Z[T,h]; H, Y, dY are [T,F].  Shard i (0-based) owns the columns
 * [i*Fs, (i+1)*Fs) of A and a and the same rows of B, Fs = F / t.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PI 3.14159265358979323846

/* ---- activation ------------------------------------------------------------
 * GeLU in its tanh approximation (Hendrycks & Gimpel, "Gaussian Error Linear
 * Units", 2016), the form the workloads name "tanh-GeLU". */
double oracle_gelu(double x) {
    const double c = sqrt(2.0 / ORACLE_PI);
    double u = c * (x + 0.044715 * x * x * x);
    return 0.5 * x * (1.0 + tanh(u));
}

/* d/dx of oracle_gelu, by the product and chain rules:
 *   0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) du/dx,  du/dx = c (1 + 3*0.044715 x^2). */
double oracle_gelu_prime(double x) {
    const double c = sqrt(2.0 / ORACLE_PI);
    double u = c * (x + 0.044715 * x * x * x);
    double th = tanh(u);
    double du = c * (1.0 + 3.0 * 0.044715 * x * x);
    return 0.5 * (1.0 + th) + 0.5 * x * (1.0 - th * th) * du;
}

void oracle_gelu_vec(const double *x, double *y, double *dy, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        if (y) y[i] = oracle_gelu(x[i]);
        if (dy) dy[i] = oracle_gelu_prime(x[i]);
    }
}

static int bad_shape(int64_t T, int64_t h, int64_t F, int32_t t) {
    return T < 0 || h <= 0 || F <= 0 || t < 1 || F % t != 0;
}

/* ---- forward ----------------------------------------------------------------
 * H = X A + a;  Y = gelu(H);  Z_i = Y[:, S_i] B[S_i, :];  Z = b + sum_i Z_i
 * (report section 4.1).  Zpart, when not NULL, receives the t partial products
 * as [t][T][h]; Z receives the fixed-order sum plus the bias. */
int oracle_forward(int64_t T, int64_t h, int64_t F, int32_t t,
                   const double *X, const double *A, const double *a,
                   const double *B, const double *b,
                   double *H, double *Y, double *Zpart, double *Z) {
    if (bad_shape(T, h, F, t)) return -1;
    const int64_t Fs = F / t;
    int failed = 0;
#pragma omp parallel
    {
        double *part = (double *)malloc(sizeof(double) * (size_t)h);
        double *sum = (double *)malloc(sizeof(double) * (size_t)h);
        if (!part || !sum) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < T; ++r) {
            if (!part || !sum) continue;
            double *Hr = H + r * F;
            double *Yr = Y + r * F;
            /* column-parallel GEMM: all shards at once, they are disjoint columns */
            for (int64_t f = 0; f < F; ++f) Hr[f] = a[f];
            for (int64_t k = 0; k < h; ++k) {
                const double xk = X[r * h + k];
                const double *Ak = A + k * F;
                for (int64_t f = 0; f < F; ++f) Hr[f] += xk * Ak[f];
            }
            for (int64_t f = 0; f < F; ++f) Yr[f] = oracle_gelu(Hr[f]);
            /* row-parallel GEMM, one shard at a time, then the all-reduce */
            for (int64_t j = 0; j < h; ++j) sum[j] = 0.0;
            for (int32_t i = 0; i < t; ++i) {
                for (int64_t j = 0; j < h; ++j) part[j] = 0.0;
                for (int64_t f = i * Fs; f < (i + 1) * Fs; ++f) {
                    const double yf = Yr[f];
                    const double *Bf = B + f * h;
                    for (int64_t j = 0; j < h; ++j) part[j] += yf * Bf[j];
                }
                if (Zpart) memcpy(Zpart + ((int64_t)i * T + r) * h, part, sizeof(double) * (size_t)h);
                for (int64_t j = 0; j < h; ++j) sum[j] += part[j];
            }
            for (int64_t j = 0; j < h; ++j) Z[r * h + j] = b[j] + sum[j];
        }
        free(part);
        free(sum);
    }
    return failed ? -2 : 0;
}

/* ---- backward ---------------------------------------------------------------
 * Chain rule for L = sum(dZ * Z) (the pages state only that the exchange runs in
 * both directions, report section 4.2):
 *   db = 1^T dZ;  G = dZ B^T;  dY = G * gelu'(H);  da = 1^T dY;
 *   dB = Y^T dZ;  dA = X^T dY;  dX = sum_i dY[:, S_i] A[:, S_i]^T.
 * The sum over shards in dX is the backward all-reduce; dXpart (optional)
 * receives its t terms as [t][T][h]. */
int oracle_backward(int64_t T, int64_t h, int64_t F, int32_t t,
                    const double *X, const double *A, const double *B,
                    const double *H, const double *Y, const double *dZ,
                    double *dY, double *dX, double *dXpart,
                    double *dA, double *da, double *dB, double *db) {
    if (bad_shape(T, h, F, t)) return -1;
    const int64_t Fs = F / t;

    /* db: column sums of dZ, rows in ascending order */
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < h; ++j) {
        double s = 0.0;
        for (int64_t r = 0; r < T; ++r) s += dZ[r * h + j];
        db[j] = s;
    }

    /* dY = (dZ B^T) * gelu'(H) */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < T; ++r) {
        const double *dZr = dZ + r * h;
        for (int64_t f = 0; f < F; ++f) {
            const double *Bf = B + f * h;
            double g = 0.0;
            for (int64_t j = 0; j < h; ++j) g += dZr[j] * Bf[j];
            dY[r * F + f] = g * oracle_gelu_prime(H[r * F + f]);
        }
    }

    /* da: column sums of dY */
#pragma omp parallel for schedule(static)
    for (int64_t f = 0; f < F; ++f) {
        double s = 0.0;
        for (int64_t r = 0; r < T; ++r) s += dY[r * F + f];
        da[f] = s;
    }

    /* dB = Y^T dZ, one row of dB (one ffn index) per iteration */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t f = 0; f < F; ++f) {
        double *dBf = dB + f * h;
        for (int64_t j = 0; j < h; ++j) dBf[j] = 0.0;
        for (int64_t r = 0; r < T; ++r) {
            const double y = Y[r * F + f];
            const double *dZr = dZ + r * h;
            for (int64_t j = 0; j < h; ++j) dBf[j] += y * dZr[j];
        }
    }

    /* dA = X^T dY, one row of dA (one hidden index) per iteration */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t k = 0; k < h; ++k) {
        double *dAk = dA + k * F;
        for (int64_t f = 0; f < F; ++f) dAk[f] = 0.0;
        for (int64_t r = 0; r < T; ++r) {
            const double x = X[r * h + k];
            const double *dYr = dY + r * F;
            for (int64_t f = 0; f < F; ++f) dAk[f] += x * dYr[f];
        }
    }

    /* dX = sum over shards of dY_i A_i^T, shards summed in ascending order */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < T; ++r) {
        const double *dYr = dY + r * F;
        for (int64_t k = 0; k < h; ++k) {
            const double *Ak = A + k * F;
            double sum = 0.0;
            for (int32_t i = 0; i < t; ++i) {
                double p = 0.0;
                for (int64_t f = i * Fs; f < (i + 1) * Fs; ++f) p += dYr[f] * Ak[f];
                if (dXpart) dXpart[((int64_t)i * T + r) * h + k] = p;
                sum += p;
            }
            dX[r * h + k] = sum;
        }
    }
    return 0;
}

/* ---- exact slices ------------------------------------------------------------
 * The same definitions restricted to a set R of token rows and a set J of ffn
 * columns.  Rows of Z and dX are independent of one another; column j of H, Y,
 * dY, dA and da and row j of dB depend only on column j of A (with a_j and row j
 * of B).  So these entries are exact, not sampled estimates, at a cost of
 * O((|R| F + T |J|) h) instead of O(T h F).
 *
 * Row outputs ([nR][F] or [nR][h]):  Hr, Yr, dYr, Zr, dXr.
 * Column outputs: Hc, Yc, dYc as [T][nJ]; dAc as [h][nJ]; daJ[nJ]; dBr[nJ][h].
 * db[h] is a full column sum (cheap).  Any output pointer may be NULL except
 * those a later step needs (none: each part is recomputed locally). */
int oracle_slice(int64_t T, int64_t h, int64_t F, int32_t t,
                 const double *X, const double *A, const double *a,
                 const double *B, const double *b, const double *dZ,
                 int64_t nR, const int64_t *R, int64_t nJ, const int64_t *J,
                 double *Hr, double *Yr, double *dYr, double *Zr, double *dXr,
                 double *Hc, double *Yc, double *dYc, double *dAc, double *daJ,
                 double *dBr, double *db) {
    if (bad_shape(T, h, F, t)) return -1;
    for (int64_t q = 0; q < nR; ++q)
        if (R[q] < 0 || R[q] >= T) return -1;
    for (int64_t q = 0; q < nJ; ++q)
        if (J[q] < 0 || J[q] >= F) return -1;
    const int64_t Fs = F / t;
    int failed = 0;

    /* token rows: row r of H, Y, dY, Z and dX needs only row r of X and dZ */
#pragma omp parallel
    {
        double *hrow = (double *)malloc(sizeof(double) * (size_t)F);
        double *dyrow = (double *)malloc(sizeof(double) * (size_t)F);
        double *part = (double *)malloc(sizeof(double) * (size_t)h);
        double *sum = (double *)malloc(sizeof(double) * (size_t)h);
        const int ok = hrow && dyrow && part && sum;
        if (!ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nR; ++q) {
            if (!ok) continue;
            const int64_t r = R[q];
            const double *Xr = X + r * h;
            const double *dZr = dZ + r * h;
            for (int64_t f = 0; f < F; ++f) hrow[f] = a[f];
            for (int64_t k = 0; k < h; ++k) {
                const double xk = Xr[k];
                const double *Ak = A + k * F;
                for (int64_t f = 0; f < F; ++f) hrow[f] += xk * Ak[f];
            }
            for (int64_t f = 0; f < F; ++f) {
                const double *Bf = B + f * h;
                double g = 0.0;
                for (int64_t j = 0; j < h; ++j) g += dZr[j] * Bf[j];
                dyrow[f] = g * oracle_gelu_prime(hrow[f]);
                if (Hr) Hr[q * F + f] = hrow[f];
                if (Yr) Yr[q * F + f] = oracle_gelu(hrow[f]);
                if (dYr) dYr[q * F + f] = dyrow[f];
            }
            if (Zr) {
                for (int64_t j = 0; j < h; ++j) sum[j] = 0.0;
                for (int32_t i = 0; i < t; ++i) {
                    for (int64_t j = 0; j < h; ++j) part[j] = 0.0;
                    for (int64_t f = i * Fs; f < (i + 1) * Fs; ++f) {
                        const double yf = oracle_gelu(hrow[f]);
                        const double *Bf = B + f * h;
                        for (int64_t j = 0; j < h; ++j) part[j] += yf * Bf[j];
                    }
                    for (int64_t j = 0; j < h; ++j) sum[j] += part[j];
                }
                for (int64_t j = 0; j < h; ++j) Zr[q * h + j] = b[j] + sum[j];
            }
            if (dXr) {
                for (int64_t k = 0; k < h; ++k) {
                    const double *Ak = A + k * F;
                    double s = 0.0;
                    for (int32_t i = 0; i < t; ++i) {
                        double p = 0.0;
                        for (int64_t f = i * Fs; f < (i + 1) * Fs; ++f) p += dyrow[f] * Ak[f];
                        s += p;
                    }
                    dXr[q * h + k] = s;
                }
            }
        }
        free(hrow);
        free(dyrow);
        free(part);
        free(sum);
    }
    if (failed) return -2;

    /* ffn columns: column j of H, Y, dY, dA and row j of dB need only column j
     * of A, a_j and row j of B (plus all of X and dZ) */
#pragma omp parallel
    {
        double *acol = (double *)malloc(sizeof(double) * (size_t)h);
        double *ycol = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double *dycol = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)h);
        const int ok = acol && ycol && dycol && acc;
        if (!ok) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < nJ; ++q) {
            if (!ok) continue;
            const int64_t j = J[q];
            const double *Bj = B + j * h;
            for (int64_t k = 0; k < h; ++k) acol[k] = A[k * F + j];
            double dasum = 0.0;
            for (int64_t r = 0; r < T; ++r) {
                const double *Xr = X + r * h;
                const double *dZr = dZ + r * h;
                double s = a[j];
                double g = 0.0;
                for (int64_t k = 0; k < h; ++k) s += Xr[k] * acol[k];
                for (int64_t k = 0; k < h; ++k) g += dZr[k] * Bj[k];
                ycol[r] = oracle_gelu(s);
                dycol[r] = g * oracle_gelu_prime(s);
                dasum += dycol[r];
                if (Hc) Hc[r * nJ + q] = s;
                if (Yc) Yc[r * nJ + q] = ycol[r];
                if (dYc) dYc[r * nJ + q] = dycol[r];
            }
            if (daJ) daJ[q] = dasum;
            if (dAc) {
                for (int64_t k = 0; k < h; ++k) acc[k] = 0.0;
                for (int64_t r = 0; r < T; ++r) {
                    const double d = dycol[r];
                    const double *Xr = X + r * h;
                    for (int64_t k = 0; k < h; ++k) acc[k] += d * Xr[k];
                }
                for (int64_t k = 0; k < h; ++k) dAc[k * nJ + q] = acc[k];
            }
            if (dBr) {
                for (int64_t k = 0; k < h; ++k) acc[k] = 0.0;
                for (int64_t r = 0; r < T; ++r) {
                    const double y = ycol[r];
                    const double *dZr = dZ + r * h;
                    for (int64_t k = 0; k < h; ++k) acc[k] += y * dZr[k];
                }
                for (int64_t k = 0; k < h; ++k) dBr[q * h + k] = acc[k];
            }
        }
        free(acol);
        free(ycol);
        free(dycol);
        free(acc);
    }
    if (failed) return -2;

    if (db) {
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < h; ++j) {
            double s = 0.0;
            for (int64_t r = 0; r < T; ++r) s += dZ[r * h + j];
            db[j] = s;
        }
    }
    return 0;
}

/* ---- LayerNorm (sequence-parallel MLP) ----------------------------------------
 * The report's section 4.3 runs LayerNorm locally on each token shard in front
 * of the tensor-parallel MLP (sequence parallelism); LayerNorm itself is the
 * textbook per-row normalisation (Ba, Kiros & Hinton, 2016):
 *   mu_r = mean_j x[r,j],  var_r = mean_j (x[r,j] - mu_r)^2,  rstd_r = 1/sqrt(var_r + eps),
 *   y[r,j] = (x[r,j] - mu_r) * rstd_r * gamma[j] + beta[j].
 * Rows are independent, so token shards need no exchange. */
void oracle_layernorm_forward(int64_t T, int64_t h, const double *X, const double *gamma,
                              const double *beta, double eps, double *Y, double *mean,
                              double *rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        const double *x = X + r * h;
        double s = 0.0;
        for (int64_t j = 0; j < h; ++j) s += x[j];
        const double mu = s / (double)h;
        double v = 0.0;
        for (int64_t j = 0; j < h; ++j) v += (x[j] - mu) * (x[j] - mu);
        v /= (double)h;
        const double rs = 1.0 / sqrt(v + eps);
        for (int64_t j = 0; j < h; ++j) Y[r * h + j] = (x[j] - mu) * rs * gamma[j] + beta[j];
        if (mean) mean[r] = mu;
        if (rstd) rstd[r] = rs;
    }
}

/* Backward of the above for an upstream gradient dY (chain rule through mu and
 * var):  xhat = (x - mu) rstd,  g = dY * gamma,
 *   dX[r,j] = rstd_r (g[r,j] - mean_j g[r,.] - xhat[r,j] mean_j (g[r,.] xhat[r,.])),
 *   dgamma = sum_r dY * xhat,  dbeta = sum_r dY.  mean and rstd are recomputed. */
int oracle_layernorm_backward(int64_t T, int64_t h, const double *dY, const double *X,
                              const double *gamma, double eps, double *dX, double *dgamma,
                              double *dbeta) {
    double *mu = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *rs = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    if (!mu || !rs) {
        free(mu);
        free(rs);
        return -2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        const double *x = X + r * h;
        const double *dy = dY + r * h;
        double s = 0.0;
        for (int64_t j = 0; j < h; ++j) s += x[j];
        const double m = s / (double)h;
        double v = 0.0;
        for (int64_t j = 0; j < h; ++j) v += (x[j] - m) * (x[j] - m);
        v /= (double)h;
        const double rstd = 1.0 / sqrt(v + eps);
        mu[r] = m;
        rs[r] = rstd;
        double mg = 0.0, mgx = 0.0;
        for (int64_t j = 0; j < h; ++j) {
            const double g = dy[j] * gamma[j];
            mg += g;
            mgx += g * (x[j] - m) * rstd;
        }
        mg /= (double)h;
        mgx /= (double)h;
        for (int64_t j = 0; j < h; ++j) {
            const double xh = (x[j] - m) * rstd;
            dX[r * h + j] = rstd * (dy[j] * gamma[j] - mg - xh * mgx);
        }
    }
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < h; ++j) {
        double sg = 0.0, sb = 0.0;
        for (int64_t r = 0; r < T; ++r) {
            sg += dY[r * h + j] * (X[r * h + j] - mu[r]) * rs[r];
            sb += dY[r * h + j];
        }
        dgamma[j] = sg;
        dbeta[j] = sb;
    }
    free(mu);
    free(rs);
    return 0;
}

/* ---- tensor-parallel self-attention ---------------------------------------------
 * The report's section 4.1 splits self-attention the same way as the MLP: the
 * heads are divided among the t shards, the QKV projection is split by columns
 * (each shard computes the Q, K and V of its own heads from the replicated
 * input) and the output projection by rows, whose t partial products are summed
 * (the all-reduce).  The attention of each head is the textbook causal scaled
 * dot-product attention (Vaswani et al., 2017):
 *   S = Q K^T / sqrt(d) (row r attends to positions c <= r),  P = softmax_row(S),
 *   O = P V.
 * Layout.  X[T,h] with T = nb*S tokens (nb sequences of S); heads of width
 * d = h/heads; hpt = heads/t heads per shard.  QKV = X Wqkv + bqkv is [T,3h]
 * with shard-major columns: shard i owns [i*3h/t, (i+1)*3h/t) = [Q_i | K_i | V_i],
 * each h/t wide, head j of the shard at offset j*d inside each.  Global head
 * g = i*hpt + j writes O columns [g*d, (g+1)*d), so shard i's heads are O's
 * columns [i*h/t, (i+1)*h/t), which are the rows of Wo[h,h] the shard owns.
 * P is [nb, heads, S, S]. */
static int64_t qkv_col(int64_t h, int32_t t, int64_t d, int64_t hpt, int64_t g, int which) {
    const int64_t i = g / hpt, j = g % hpt;
    return i * (3 * h / t) + (int64_t)which * (h / t) + j * d;
}

static int bad_attn(int64_t nb, int64_t S, int64_t h, int64_t heads, int32_t t) {
    return nb < 0 || S <= 0 || h <= 0 || heads <= 0 || t < 1 || h % heads != 0 || heads % t != 0;
}

int oracle_attn_forward(int64_t nb, int64_t S, int64_t h, int64_t heads, int32_t t,
                        const double *X, const double *Wqkv, const double *bqkv,
                        const double *Wo, const double *bo,
                        double *QKV, double *P, double *O, double *Z) {
    if (bad_attn(nb, S, h, heads, t)) return -1;
    const int64_t T = nb * S, d = h / heads, hpt = heads / t, H3 = 3 * h, hs = h / t;
    /* column-parallel QKV projection of all shards */
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r) {
        double *q = QKV + r * H3;
        for (int64_t c = 0; c < H3; ++c) q[c] = bqkv[c];
        for (int64_t k = 0; k < h; ++k) {
            const double x = X[r * h + k];
            const double *w = Wqkv + k * H3;
            for (int64_t c = 0; c < H3; ++c) q[c] += x * w[c];
        }
    }
    /* causal attention of every head of every sequence */
    const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < nb; ++b)
        for (int64_t g = 0; g < heads; ++g) {
            const int64_t qc = qkv_col(h, t, d, hpt, g, 0), kc = qkv_col(h, t, d, hpt, g, 1),
                          vc = qkv_col(h, t, d, hpt, g, 2);
            double *Pg = P + (b * heads + g) * S * S;
            for (int64_t r = 0; r < S; ++r) {
                const double *qr = QKV + (b * S + r) * H3 + qc;
                const int64_t last = r; /* causal: row r sees positions 0..r */
                double mx = -INFINITY;
                for (int64_t c = 0; c <= last; ++c) {
                    const double *kr = QKV + (b * S + c) * H3 + kc;
                    double sc = 0.0;
                    for (int64_t e = 0; e < d; ++e) sc += qr[e] * kr[e];
                    Pg[r * S + c] = sc * scale;
                    if (Pg[r * S + c] > mx) mx = Pg[r * S + c];
                }
                double den = 0.0;
                for (int64_t c = 0; c <= last; ++c) {
                    Pg[r * S + c] = exp(Pg[r * S + c] - mx);
                    den += Pg[r * S + c];
                }
                for (int64_t c = 0; c <= last; ++c) Pg[r * S + c] /= den;
                for (int64_t c = last + 1; c < S; ++c) Pg[r * S + c] = 0.0;
                double *orow = O + (b * S + r) * h + g * d;
                for (int64_t e = 0; e < d; ++e) orow[e] = 0.0;
                for (int64_t c = 0; c <= last; ++c) {
                    const double pc = Pg[r * S + c];
                    const double *vr = QKV + (b * S + c) * H3 + vc;
                    for (int64_t e = 0; e < d; ++e) orow[e] += pc * vr[e];
                }
            }
        }
    /* row-parallel output projection, shard partials summed in order, + bo */
#pragma omp parallel
    {
        double *part = (double *)malloc(sizeof(double) * (size_t)h);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < T; ++r) {
            if (!part) continue;
            for (int64_t c = 0; c < h; ++c) Z[r * h + c] = 0.0;
            for (int32_t i = 0; i < t; ++i) {
                for (int64_t c = 0; c < h; ++c) part[c] = 0.0;
                for (int64_t k = i * hs; k < (i + 1) * hs; ++k) {
                    const double o = O[r * h + k];
                    const double *w = Wo + k * h;
                    for (int64_t c = 0; c < h; ++c) part[c] += o * w[c];
                }
                for (int64_t c = 0; c < h; ++c) Z[r * h + c] += part[c];
            }
            for (int64_t c = 0; c < h; ++c) Z[r * h + c] += bo[c];
        }
        free(part);
    }
    return 0;
}

/* Backward for L = sum(dZ * Z): the chain rule through the output projection,
 * the attention of each head and the QKV projection:
 *   dbo = 1^T dZ, dO = dZ Wo^T, dWo = O^T dZ;
 *   per head: dV = P^T dO, dP = dO V^T, dS = P * (dP - rowsum(dP * P)),
 *             dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d);
 *   dbqkv = 1^T dQKV, dWqkv = X^T dQKV, dX = sum_i dQKV[:, shard i] Wqkv[:, shard i]^T. */
int oracle_attn_backward(int64_t nb, int64_t S, int64_t h, int64_t heads, int32_t t,
                         const double *X, const double *Wqkv, const double *Wo,
                         const double *QKV, const double *P, const double *O, const double *dZ,
                         double *dX, double *dWqkv, double *dbqkv, double *dWo, double *dbo) {
    if (bad_attn(nb, S, h, heads, t)) return -1;
    const int64_t T = nb * S, d = h / heads, hpt = heads / t, H3 = 3 * h, hs3 = H3 / t;
    double *dO = (double *)malloc(sizeof(double) * (size_t)(T * h + 1));
    double *dQKV = (double *)calloc((size_t)(T * H3 + 1), sizeof(double));
    if (!dO || !dQKV) {
        free(dO);
        free(dQKV);
        return -2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < h; ++c) {
        double sb = 0.0;
        for (int64_t r = 0; r < T; ++r) sb += dZ[r * h + c];
        dbo[c] = sb;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r)
        for (int64_t k = 0; k < h; ++k) {
            double s = 0.0;
            for (int64_t c = 0; c < h; ++c) s += dZ[r * h + c] * Wo[k * h + c];
            dO[r * h + k] = s;
        }
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < h; ++k)
        for (int64_t c = 0; c < h; ++c) {
            double s = 0.0;
            for (int64_t r = 0; r < T; ++r) s += O[r * h + k] * dZ[r * h + c];
            dWo[k * h + c] = s;
        }
    const double scale = 1.0 / sqrt((double)d);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < nb; ++b)
        for (int64_t g = 0; g < heads; ++g) {
            const int64_t qc = qkv_col(h, t, d, hpt, g, 0), kc = qkv_col(h, t, d, hpt, g, 1),
                          vc = qkv_col(h, t, d, hpt, g, 2);
            const double *Pg = P + (b * heads + g) * S * S;
            double *dP = (double *)malloc(sizeof(double) * (size_t)S);
            if (!dP) continue;
            for (int64_t r = 0; r < S; ++r) {
                const double *dor = dO + (b * S + r) * h + g * d;
                double D = 0.0;
                for (int64_t c = 0; c <= r; ++c) {
                    const double *vr = QKV + (b * S + c) * H3 + vc;
                    double s = 0.0;
                    for (int64_t e = 0; e < d; ++e) s += dor[e] * vr[e];
                    dP[c] = s;
                    D += s * Pg[r * S + c];
                }
                for (int64_t c = 0; c <= r; ++c) {
                    const double ds = Pg[r * S + c] * (dP[c] - D) * scale;
                    const double *qr = QKV + (b * S + r) * H3 + qc;
                    const double *kr = QKV + (b * S + c) * H3 + kc;
                    double *dq = dQKV + (b * S + r) * H3 + qc;
                    double *dk = dQKV + (b * S + c) * H3 + kc;
                    double *dv = dQKV + (b * S + c) * H3 + vc;
                    for (int64_t e = 0; e < d; ++e) {
                        dq[e] += ds * kr[e];
                        dk[e] += ds * qr[e];
                        dv[e] += Pg[r * S + c] * dor[e];
                    }
                }
            }
            free(dP);
        }
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < H3; ++c) {
        double sb = 0.0;
        for (int64_t r = 0; r < T; ++r) sb += dQKV[r * H3 + c];
        dbqkv[c] = sb;
    }
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < h; ++k)
        for (int64_t c = 0; c < H3; ++c) {
            double s = 0.0;
            for (int64_t r = 0; r < T; ++r) s += X[r * h + k] * dQKV[r * H3 + c];
            dWqkv[k * H3 + c] = s;
        }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < T; ++r)
        for (int64_t k = 0; k < h; ++k) {
            double sum = 0.0;
            for (int32_t i = 0; i < t; ++i) {
                double p = 0.0;
                for (int64_t c = i * hs3; c < (i + 1) * hs3; ++c) p += dQKV[r * H3 + c] * Wqkv[k * H3 + c];
                sum += p;
            }
            dX[r * h + k] = sum;
        }
    free(dO);
    free(dQKV);
    return 0;
}

/* Number of OpenMP threads a parallel region of this library will use. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
