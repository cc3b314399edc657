// Host-side launchers of the kernels behind the C ABI (internal to libtpmlp.so).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tpmlp {

// Epilogues of the GEMM kernels.  Each names the step of the MLP it finishes.
enum Epi : int {
    EPI_BIAS_GELU = 0,  // H = acc + a (optional store), Y = GeLU(H) (optional) -- column-parallel GEMM
    EPI_FOLD_BIAS = 1,  // Z = b + ((Z_1 + Z_2) + ...)                      -- row-parallel GEMM
    EPI_DGELU = 2,      // dY = acc * GeLU'(H)                              -- dZ B^T
    EPI_STORE = 3,      // out = acc                                       -- dB, dA
    EPI_FOLD = 4,       // dX = ((P_1 + P_2) + ...)                        -- dY A^T
    EPI_ATTN_SCORE = 5, // S = scale * acc, -inf above the diagonal (causal), fp16 out -- Q K^T
    EPI_ATTN_DS = 6,    // dS = P * (acc - D[row]) * scale                  -- dO V^T -> dS
};

// A per-head operand or output read or written in place inside a token-major
// array (rank 4 or 5), instead of a contiguous [batch][rows][cols] block (rank 3).
// Element (e, s) of problem z = b * heads + g, head g = i * hpt + j:
//   rank 4 (O, dO [T, h]):           base[(b*S + s) * ld + g * d + e]
//   rank 5 (Q, K, V inside QKV or dQKV [T, 3h], base at the Q/K/V column offset):
//                                     base[(b*S + s) * ld + i * coli + j * d + e]
struct HeadView {
    int rank;  // 3 (plain block), 4 or 5
    int64_t S, nb, heads, hpt, d, ld, coli;
};

// One GEMM  out[M,N] = sum_k opA(m,k) opB(k,n)  over row-major operands.
//   A operand: K-major ([M,K] row-major, a_mn = false) or MN-major ([K,M], a_mn = true)
//   B operand: K-major ([N,K] row-major, b_mn = false) or MN-major ([K,N], b_mn = true)
// The K range is split into `nshards` consecutive ranges of `kshard` elements;
// each range is accumulated on its own and, for the FOLD epilogues, the range
// partials are summed in ascending order.  For the other epilogues nshards = 1.
struct GemmArgs {
    const void *a;
    bool a_mn;
    const void *b;
    bool b_mn;
    int64_t M, N, K;
    int nshards;
    int64_t kshard;
    void *out0;        // H / Z / dY / dB / dA / dX
    void *out1;        // Y for EPI_BIAS_GELU (null: no activation); Y rebuilt from H for EPI_DGELU (optional)
    const void *aux;   // H for EPI_DGELU
    const void *bias;  // a for EPI_BIAS_GELU, b for EPI_FOLD_BIAS
    uint32_t *status;  // device status word
    uint64_t wait_ns;
    int group;         // raster: tiles walk `group` M-tiles (N-tiles if raster_n) fastest
    bool raster_n;
    bool cta_pair;     // tensor-core path: 256 x 256 tiles on CTA pairs (tcgen05 cta_group::2)
    float *colsum_part;  // EPI_DGELU on tensor cores: fp32 column sums per 32-row block [ceil(M/32), N]
    // Batched GEMMs: `batch` independent problems whose operands and outputs are
    // contiguous [batch][rows][cols] arrays (attention heads).  1 = plain GEMM.
    int64_t batch;
    float scale;          // EPI_ATTN_SCORE, EPI_ATTN_DS
    bool causal;          // EPI_ATTN_SCORE: mask columns past the row
    const float *rowvec;  // EPI_ATTN_DS: D, one fp32 per output row, [batch][M]
    // Causal per-head products (tensor-core path, square M = K, one shard): only
    // the k range the zero pattern leaves, in whole tiles.  1: k below the end of
    // the M-tile (P V, dS K); 2: k from the start of the M-tile on (P^T dO, dS^T Q).
    int causal_k;
    bool skip_upper;  // skip tiles wholly above the diagonal (scores, dS)
    // EPI_STORE with an MN-major A on tensor cores: also write bias_grad[n] =
    // sum_k B(k, n) (bf16), computed by the MMA from an extra M-tile whose A is
    // `ones`, a 64 x 64 bf16 block of ones (8 KiB, 16-byte aligned).
    const void *ones;
    void *bias_grad;
    // Per-head GEMMs addressing their operands and output in place (tensor-core
    // path; EPI_ATTN_SCORE, EPI_ATTN_DS, EPI_STORE): a rank of 0 or 3 is the
    // plain [batch][rows][cols] block.
    bool heads_layout;
    HeadView a_view, b_view, o_view;
};

// Tensor-core path: bf16 operands, fp32 accumulation in TMEM (tcgen05).
cudaError_t launch_tc_gemm(Epi epi, const GemmArgs &g, int num_sms, cudaStream_t st);

// Whether launch_tc_gemm runs this product on 256 x 512 tiles (CTA pairs; the
// store (both operands MN-major or both K-major), bias + GeLU and GeLU'
// epilogues of one shard on plain operands) rather than 256 x 256.  TPMLP_WIDE=0 keeps 256 x 256 (a tuning knob, read per call).
bool tc_wide_tile(Epi epi, const GemmArgs &g);

// FFMA path: element type fp32 (is_bf16 = false) or bf16, fp32 accumulation.
cudaError_t launch_simt_gemm(Epi epi, bool is_bf16, const GemmArgs &g, cudaStream_t st);

// Deterministic column sums out[c] = sum_r x[r,c] in two launches (per-chunk fp32
// partials into `partials`, then an in-order sum of the chunks).
int64_t colsum_chunks(int64_t rows, int64_t cols);
cudaError_t launch_colsum(bool is_bf16, const void *x, int64_t rows, int64_t cols, float *partials,
                          void *out, cudaStream_t st, int *launches);

// Second pass alone: out[c] = sum over `chunks` rows of partials[k, c], in order.
// `ones` (optional): an 8 KiB block the kernel also fills with bf16 ones.
cudaError_t launch_colsum_final(bool is_bf16, const float *partials, int64_t chunks, int64_t cols, void *out,
                                cudaStream_t st, void *ones = nullptr);

// A kernel that waits on a barrier nothing arrives on and reports the timeout.
cudaError_t launch_timeout_probe(uint32_t *status, uint64_t wait_ns, cudaStream_t st);

// LayerNorm over the rows of a row-major [rows, h] matrix (fp32 statistics).
struct LnArgs {
    int64_t rows, h;
    float eps;
    const void *x;      // input rows
    const void *gamma;  // [h]
    const void *beta;   // [h] (forward)
    void *y;            // forward output
    float *mean;        // [rows]
    float *rstd;        // [rows]
    const void *dy;     // backward: gradient w.r.t. the output
    void *dx;           // backward: gradient w.r.t. the input
    void *dgamma;       // [h]
    void *dbeta;        // [h]
    float *partials;    // backward: ln_partial_floats(rows, h) floats of scratch
};
int64_t ln_partial_floats(int64_t rows, int64_t h);
cudaError_t launch_ln_forward(bool is_bf16, const LnArgs &a, cudaStream_t st);
cudaError_t launch_ln_backward(bool is_bf16, const LnArgs &a, cudaStream_t st, int *launches);

// Attention support.  Problem z = b*heads + g over `nb` sequences of S tokens;
// token-major O and dO are [T, h] with head g at columns [g*d, (g+1)*d).
struct HeadLayout {
    int64_t nb, S, h, heads, d;
};
// wtile > 0: each row writes P only up to the end of its wtile-wide column tile.
cudaError_t launch_softmax(const void *S, void *P, int64_t rows, int64_t cols, bool causal, int64_t wtile,
                           cudaStream_t st);
// D[z*S + s] = row dot of dO and O over head g's columns of token b*S + s (token-major inputs).
// `ones` (optional): an 8 KiB block the kernel also fills with bf16 ones.
cudaError_t launch_rowdot(const HeadLayout &L, const void *dO, const void *O, float *D, cudaStream_t st,
                          void *ones = nullptr);

// Records a description of the last failure of this host thread (read back by
// tpmlp_last_error()).
void set_last_error(const char *fmt, ...);

// Adds to the count reported by tpmlp_launch_count().
void add_launches(uint64_t n);

}  // namespace tpmlp
