/*
 * tpmlp -- the tensor-parallel Transformer MLP block on one GB300 (sm_103a).
 *
 *     Z = GeLU(X A + a) B + b
 *
 * The method ("Megatron-LM" industry report, section 4.1, basic principle of
 * tensor parallelism): the first weight A is split by columns into t shards
 * [A_1 .. A_t] (with its bias a), the second weight B by rows into [B_1 .. B_t];
 * the input X is replicated; shard i computes Y_i = GeLU(X A_i + a_i) and the
 * partial product Z_i = Y_i B_i; an all-reduce sums the Z_i.  Section 4.2 of the
 * same report adds that the exchange runs in both directions, i.e. the backward
 * pass sums the shard contributions to dX.  Here all t shards live on one GPU:
 * the column-parallel GEMM of every shard is one launch (the shards are disjoint
 * column blocks) and each all-reduce is a fixed-order fp32 sum of the t shard
 * partials, Z = b + (((Z_1 + Z_2) + Z_3) + ... + Z_t), done on chip (the tiles
 * that the tensor-core schedule walks down K sum the same partials in the
 * opposite order, b + (((Z_t + Z_t-1) + ...) + Z_1)).  Repeated
 * calls with the same inputs give bit-identical outputs.  The tensor-core GEMMs
 * accumulate over k in an order that depends on their tile schedule, and so on
 * the number of SMs they run on: a GPU with another SM count (or the
 * TPMLP_MAX_UNITS / TPMLP_SERPENTINE knobs) may round differently, within the
 * same tolerances.
 *
 * Layout.  Every tensor is row-major, contiguous and in device memory:
 *   X[T,h]  A[h,F]  a[F]  B[F,h]  b[h]  Z[T,h]  H,Y[T,F]  (T tokens, h hidden,
 *   F ffn).  Shard i (0-based) owns columns [i*F/t, (i+1)*F/t) of A and a and
 *   the same rows of B.  Weights are in the math layout X.A, not in the
 *   [out, in] layout of a PyTorch Linear.
 *
 * Types.  Every input and output of one call has the shape's dtype (fp32 or
 * bf16).  bf16 runs on the tensor cores (tcgen05, fp32 accumulation, fp32
 * epilogue math, round-to-nearest-even on store); fp32 runs on plain FFMA
 * kernels (no TF32).
 *
 * Ownership.  The caller owns all memory.  The library allocates no device
 * memory; it keeps only host-side caches (device properties, kernel attributes).
 *
 * Streams and errors.  Calls are asynchronous on the given CUDA stream (a
 * cudaStream_t passed as void*, NULL = the legacy default stream).  The return
 * value covers host-side validation and launch errors only.  Errors found on the
 * device (a bounded wait that ran out) are recorded in the status word at the
 * start of the workspace and read by tpmlp_check_device_status().
 *
 * Thread safety.  Calls may be made from several host threads; each call only
 * reads its arguments and the shared caches are locked.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TPMLP_OK = 0,
    TPMLP_ERR_INVALID_ARG = 1, /* a NULL pointer, a size <= 0, t out of [1,16], F % t != 0 */
    TPMLP_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels take (alignment, F/t % 64) */
    TPMLP_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    TPMLP_ERR_TIMEOUT = 4,     /* a bounded device-side wait ran out (device status word) */
    TPMLP_ERR_DEVICE = 5       /* no usable sm_100-family device */
} tpmlp_status;

typedef enum { TPMLP_F32 = 0, TPMLP_BF16 = 1 } tpmlp_dtype;

/* Kernel family.  DEFAULT: tensor cores for bf16, FFMA for fp32.  SIMT: FFMA
 * kernels for either dtype (a second, independent GPU path used to cross-check
 * the tensor-core kernels). */
typedef enum { TPMLP_ALGO_DEFAULT = 0, TPMLP_ALGO_SIMT = 1 } tpmlp_algo;

typedef struct {
    int64_t tokens; /* T >= 0 (T = 0 is an empty batch) */
    int64_t hidden; /* h > 0 */
    int64_t ffn;    /* F > 0, F % t == 0 */
    int32_t t;      /* number of tensor-parallel shards, 1..16 */
    int32_t dtype;  /* tpmlp_dtype */
    int32_t algo;   /* tpmlp_algo */
    int32_t flags;  /* tpmlp_flags, 0 for the plain pass */
} tpmlp_shape;

/* TPMLP_FLAG_RECOMPUTE: activation recomputation (the "activation checkpointing"
 * of the oreateai page, section 2.2; "selective recomputation" in the report's
 * section 6.4).  The forward pass keeps only the pre-activation H for the
 * backward pass; Y = GeLU(H) goes to the workspace (TPMLP_WS_Y) for the
 * row-parallel GEMM and is rebuilt from H by the backward pass's GeLU'
 * epilogue, which reads H anyway.  Activation memory kept between the passes is
 * T*F elements instead of 2*T*F.  saved->Y may then be NULL; saved->H is
 * required. */
/* TPMLP_FLAG_LAYERNORM: the block has LayerNorm in front, the sequence-parallel
 * MLP of the report's section 4.3 (see tpmlp_sp_forward).  The workspace then
 * also holds the MLP's input gradient (TPMLP_WS_DXN) for the LayerNorm backward. */
typedef enum { TPMLP_FLAG_RECOMPUTE = 1, TPMLP_FLAG_LAYERNORM = 2 } tpmlp_flags;

/* The LayerNorm in front of the sequence-parallel block.  All buffers are the
 * caller's: X_in [T,h] (the token shards' rows side by side), gamma and beta [h],
 * Xn [T,h] (the normalised rows, which the MLP takes as its X), mean and rstd [T]
 * in fp32 (row statistics kept for the backward pass). */
typedef struct {
    const void *X_in;
    const void *gamma;
    const void *beta;
    void *Xn;
    float *mean;
    float *rstd;
    float eps;
} tpmlp_layernorm;

/* What the forward pass keeps for the backward pass.  The caller allocates H and
 * Y (T*F elements each, tpmlp_saved_bytes() in total); tpmlp_forward() fills in
 * X, A and B with the pointers it was given.  H may be NULL in a forward-only
 * (inference) call, in which case the pre-activation is not stored; Y is always
 * needed because the row-parallel GEMM reads it. */
typedef struct {
    const void *X;
    const void *A;
    const void *B;
    void *H; /* pre-activation X A + a, [T,F] */
    void *Y; /* GeLU(H), [T,F] */
} tpmlp_saved;

/* Offsets into the workspace, for callers that want the intermediates. */
typedef enum {
    TPMLP_WS_STATUS = 0,  /* uint32 status word (tpmlp_status), then a uint32 detail word */
    TPMLP_WS_PARTIALS = 1, /* fp32 column-sum partials */
    TPMLP_WS_DY = 2,       /* dY = (dZ B^T) * GeLU'(H), [T,F] in the shape's dtype */
    TPMLP_WS_Y = 3,        /* Y under TPMLP_FLAG_RECOMPUTE, [T,F]; absent (size 0) otherwise */
    TPMLP_WS_DXN = 4       /* dXn, the MLP's input gradient, under TPMLP_FLAG_LAYERNORM, [T,h] */
} tpmlp_ws_region;

/* Human-readable name of a status code (static storage). */
const char *tpmlp_status_string(tpmlp_status s);

/* Library version, major*10000 + minor*100 + patch. */
int tpmlp_version(void);

/* Description of the most recent failure of a call made from this host thread
 * (empty after a call that succeeded from the start).  Static, per-thread storage. */
const char *tpmlp_last_error(void);

/* Bytes the caller must allocate for the saved activations: H and Y together
 * (2*T*F elements), or H alone (T*F) under TPMLP_FLAG_RECOMPUTE; 0 when the shape
 * is invalid. */
size_t tpmlp_saved_bytes(const tpmlp_shape *shape);

/* Bytes of device workspace forward and backward need: the status word, the
 * column-sum partials, the dY intermediate (plus Y or dXn under the flags) and an
 * 8 KiB block the backward fills with bf16 ones.  A 256-byte aligned buffer of at
 * least this size, whose first 8 bytes are zero before first use, is required.
 * 0 when the shape is invalid. */
size_t tpmlp_workspace_bytes(const tpmlp_shape *shape);

/* Byte offset of a region inside the workspace (see tpmlp_ws_region);
 * (size_t)-1 when the shape or region is invalid. */
size_t tpmlp_workspace_offset(const tpmlp_shape *shape, int region);

/* Forward pass ("Megatron-LM" report, section 4.1):
 *   H = X A + a,  Y = GeLU(H)   -- the column-parallel GEMM of all t shards,
 *                                  bias and GeLU fused in its epilogue;
 *   Z = b + sum_{i=1..t} Y_i B_i -- the row-parallel GEMM; the t shard partials
 *                                  are summed in order on chip, then b is added.
 * X[T,h], A[h,F], a[F], B[F,h], b[h] are inputs; Z[T,h] is the output; saved->Y
 * (and saved->H unless NULL) receive the activations.  saved == NULL is
 * inference: H is not stored and Y goes to the workspace's dY region (which
 * only the backward pass uses), so nothing is kept for a backward pass.  GeLU is the tanh form
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 * Errors: INVALID_ARG for NULL shape/pointers (saved and saved->H excepted), bad sizes;
 * UNSUPPORTED on the tensor-core path when a pointer is not 16-byte aligned,
 * h or F is not a multiple of 8, or t > 1 and F/t is not a multiple of 64;
 * CUDA when a launch fails.  Nothing is launched when an error is returned. */
tpmlp_status tpmlp_forward(const tpmlp_shape *shape, const void *X, const void *A, const void *a,
                           const void *B, const void *b, void *Z, tpmlp_saved *saved,
                           void *workspace, void *stream);

/* Backward pass for the scalar loss L = sum(dZ * Z) (the chain rule; the report
 * states only that the exchange also runs backward, section 4.2):
 *   db = 1^T dZ,  dY = (dZ B^T) * GeLU'(H),  da = 1^T dY,
 *   dB = Y^T dZ,  dA = X^T dY,  dX = sum_{i=1..t} dY_i A_i^T  (fixed-order sum).
 * dZ[T,h] and the saved activations are inputs; dX[T,h], dA[h,F], da[F],
 * dB[F,h], db[h] are outputs.  dY is left in the workspace (TPMLP_WS_DY).
 * On the tensor-core path da comes from the dY GEMM's epilogue (fixed-order
 * per-32-row block sums) and db from the dB GEMM itself: one extra M-tile whose
 * A operand is a block of ones yields 1^T dZ in fp32 (bf16 at the end).  The
 * FFMA path computes both as two-pass column sums.
 * With T = 0 the weight and bias gradients are set to zero.
 * Errors: as tpmlp_forward; saved->H, saved->Y, X, A, B must all be set. */
tpmlp_status tpmlp_backward(const tpmlp_shape *shape, const void *dZ, const tpmlp_saved *saved,
                            void *dX, void *dA, void *da, void *dB, void *db,
                            void *workspace, void *stream);

/* LayerNorm of every row of ln->X_in into ln->Xn, keeping ln->mean and ln->rstd
 * (the per-token-shard LayerNorm of the report's section 4.3; rows are
 * independent, so all shards are one launch):
 *   mu = mean_j x, var = mean_j (x - mu)^2, rstd = 1/sqrt(var + eps),
 *   xn = (x - mu) * rstd * gamma + beta.
 * Uses shape->tokens, hidden and dtype.  Errors: INVALID_ARG for a bad shape or
 * a NULL pointer, or eps < 0; CUDA when a launch fails. */
tpmlp_status tpmlp_ln_forward(const tpmlp_shape *shape, tpmlp_layernorm *ln, void *stream);

/* Backward of tpmlp_ln_forward for the gradient dXn of its output:
 *   dX_in = rstd * (g - mean_j g - xhat * mean_j(g * xhat)),  g = dXn * gamma,
 *   dgamma = sum_rows dXn * xhat,  dbeta = sum_rows dXn   (fixed-order sums).
 * The workspace is a tpmlp_workspace_bytes() buffer of a shape with
 * TPMLP_FLAG_LAYERNORM (its column-sum partials are used). */
tpmlp_status tpmlp_ln_backward(const tpmlp_shape *shape, const tpmlp_layernorm *ln, const void *dXn, void *dX_in,
                               void *dgamma, void *dbeta, void *workspace, void *stream);

/* The sequence-parallel MLP block (report section 4.3): LayerNorm of the input
 * rows, then tpmlp_forward on the normalised rows.  Across t GPUs the
 * normalised token shards would be all-gathered before the column-parallel GEMM
 * and the output partials reduce-scattered back to token shards; with every
 * shard on one GPU the gathered input is the Xn buffer itself and the shard fold
 * already produces every output row.  shape->flags must include
 * TPMLP_FLAG_LAYERNORM.  saved->X is set to ln->Xn. */
tpmlp_status tpmlp_sp_forward(const tpmlp_shape *shape, tpmlp_layernorm *ln, const void *A, const void *a,
                              const void *B, const void *b, void *Z, tpmlp_saved *saved, void *workspace,
                              void *stream);

/* Backward of tpmlp_sp_forward: tpmlp_backward into the workspace's dXn, then
 * tpmlp_ln_backward.  Outputs dX_in [T,h], dgamma, dbeta [h] and the MLP's
 * weight and bias gradients. */
tpmlp_status tpmlp_sp_backward(const tpmlp_shape *shape, const tpmlp_layernorm *ln, const void *dZ,
                               const tpmlp_saved *saved, void *dX_in, void *dgamma, void *dbeta, void *dA,
                               void *da, void *dB, void *db, void *workspace, void *stream);

/* ---- tensor-parallel self-attention block (report section 4.1) ---------------
 * The report splits self-attention like the MLP: the heads are divided among
 * the t shards; the QKV projection is column-parallel (each shard projects the
 * replicated input onto the Q, K and V of its own heads) and the output
 * projection row-parallel (each shard multiplies its heads' columns of O by its
 * rows of Wo; the t partial products are summed, the all-reduce).  Each head is
 * causal scaled dot-product attention:
 *   S = Q K^T / sqrt(d) (row r sees positions <= r),  P = softmax_row(S),  O = P V,
 *   Z = bo + sum_i O_i Wo_i   (fixed shard order).
 * Layout: X, Z, O [T,h] with T = batch*seq tokens (batch sequences of seq
 * tokens); Wqkv [h,3h], bqkv [3h] with shard-major columns: shard i owns columns
 * [i*3h/t, (i+1)*3h/t) = [Q_i | K_i | V_i], each h/t wide, head j of the shard at
 * offset j*d (d = h/heads); global head g = i*heads/t + j owns O's columns
 * [g*d, (g+1)*d); Wo [h,h], bo [h].  bf16 only (tensor cores). */
typedef struct {
    int64_t batch;  /* sequences (>= 0) */
    int64_t seq;    /* tokens per sequence, a multiple of 8 */
    int64_t hidden; /* h */
    int32_t heads;  /* h % heads == 0, heads % t == 0, d = h/heads a multiple of 64 */
    int32_t t;      /* shards, 1..16 */
    int32_t dtype;  /* TPMLP_BF16 */
    int32_t flags;  /* tpmlp_attn_flags, 0 for the plain pass */
} tpmlp_attn_shape;

/* TPMLP_ATTN_P_UPPER_ZERO: the caller's P buffer already holds zeros in every
 * 256 x 256 tile that lies wholly above the diagonal (each key of the tile past
 * each query), so the forward does not write those tiles: row s of a head
 * writes columns [0, min(seq, (s/256 + 1)*256)).  No kernel reads them.  A
 * caller that keeps one P buffer across steps and zeroes it once can set it; the
 * values of P are then the same as without it.  Without the flag every row of P
 * is written in full. */
typedef enum { TPMLP_ATTN_P_UPPER_ZERO = 1 } tpmlp_attn_flags;

/* What the forward pass keeps for the backward pass (caller-owned except the
 * weights, which tpmlp_attn_forward records): QKV [T,3h], P [batch*heads, seq,
 * seq] (bf16 probabilities of every head; with TPMLP_ATTN_P_UPPER_ZERO the tiles
 * wholly above the diagonal are left as the caller holds them), O [T,h]. */
typedef struct {
    const void *X;
    const void *Wqkv;
    const void *Wo;
    void *QKV;
    void *P;
    void *O;
} tpmlp_attn_saved;

/* Bytes of QKV + P + O; 0 for an invalid shape. */
size_t tpmlp_attn_saved_bytes(const tpmlp_attn_shape *shape);
/* Bytes of device workspace for forward and backward (status word, the row terms,
 * token-major dO and dQKV, the fp16 scores reused for dS, and an 8 KiB block of
 * ones; the per-head GEMMs address Q, K, V, O, dO, dQ, dK, dV in place inside the
 * token-major arrays); 256-byte aligned, first 8 bytes zero before first use. */
size_t tpmlp_attn_workspace_bytes(const tpmlp_attn_shape *shape);

/* Forward: QKV = X Wqkv + bqkv (one column-parallel GEMM for all shards), per
 * head P = softmax(causal Q K^T / sqrt(d)) and O = P V (batched over heads),
 * Z = bo + fixed-order sum of the t row-parallel partials.  The scaled scores
 * are computed in fp32 and kept in fp16 (11 significant bits) between the score
 * GEMM and the fp32 softmax; P is stored in bf16.
 * Errors: INVALID_ARG for a bad shape or NULL pointer; UNSUPPORTED for a non-bf16
 * dtype, misaligned pointers, d % 64 != 0, seq % 8 != 0, or h/t or 3h/t not a
 * multiple of 64 when t > 1; CUDA when a launch fails. */
tpmlp_status tpmlp_attn_forward(const tpmlp_attn_shape *shape, const void *X, const void *Wqkv,
                                const void *bqkv, const void *Wo, const void *bo, void *Z,
                                tpmlp_attn_saved *saved, void *workspace, void *stream);

/* Backward for L = sum(dZ * Z): dbo = 1^T dZ, dO = dZ Wo^T, dWo = O^T dZ; per head
 * dV = P^T dO, dS = P * (dO V^T - rowsum(dO * O)) / sqrt(d), dQ = dS K, dK = dS^T Q;
 * dbqkv = 1^T dQKV, dWqkv = X^T dQKV, dX = fixed-order sum over shards of
 * dQKV_i Wqkv_i^T (the backward all-reduce).  dbo and dbqkv come from extra
 * ones tiles of the dWo and dWqkv GEMMs.  Errors as the forward. */
tpmlp_status tpmlp_attn_backward(const tpmlp_attn_shape *shape, const void *dZ, const tpmlp_attn_saved *saved,
                                 void *dX, void *dWqkv, void *dbqkv, void *dWo, void *dbo, void *workspace,
                                 void *stream);

/* Synchronises the stream, reads the workspace status word, clears it and
 * returns it (TPMLP_OK when no device-side error was recorded). */
tpmlp_status tpmlp_check_device_status(void *workspace, void *stream);

/* Upper limit, in nanoseconds, of every device-side wait of later launches
 * (default 2e9).  A wait that runs out records TPMLP_ERR_TIMEOUT and the kernel
 * returns after releasing what it holds. */
void tpmlp_set_wait_limit_ns(uint64_t ns);

/* Launches one small kernel that waits on a barrier nothing arrives on, for at
 * most wait_ns, then records TPMLP_ERR_TIMEOUT in the workspace status word and
 * returns (after freeing the tensor memory it allocated).  It exercises the
 * error path of the bounded waits without faulting or hanging the GPU. */
tpmlp_status tpmlp_debug_timeout_probe(void *workspace, uint64_t wait_ns, void *stream);

/* Column sums out[c] = sum_r x[r, c] of a row-major [rows, cols] device matrix
 * of the given dtype, for callers that cannot allocate device memory.  It runs
 * the two-pass column-sum kernels that tpmlp_backward's FFMA path (fp32, or
 * TPMLP_ALGO_SIMT) uses for db = 1^T dZ and da = 1^T dY, and gives the same bits
 * as that path.  tpmlp_backward's tensor-core path sums in other orders (db in
 * the dB GEMM's ones tile, da in per-32-row block sums of the dY epilogue), so
 * against it the results agree to within bf16 rounding, not bit for bit.  The
 * pages have no counterpart to this entry point; it exists for the caller, not
 * the method.
 *
 * Who needs it: code that must not call cudaMalloc, e.g. a runtime whose device
 * memory is one pre-reserved arena owned by another component, or a caller on a
 * latency-critical path where cudaMalloc's implicit synchronisation or its
 * failure under memory pressure is not acceptable.  tpmlp_backward needs a
 * caller workspace; this entry point takes only the input and the output.
 *
 * Scratch: the fp32 partial sums go to a fixed 4 MiB array inside the library
 * (1,048,576 floats), which every GPU that loads the library holds until the
 * process exits.  A call needs chunks*cols floats, where chunks depends only on
 * (rows, cols) and is at most ceil(1024 / ceil(cols/256)); requests that need
 * more (for instance cols > 1,048,576) return TPMLP_ERR_UNSUPPORTED with the
 * reason in tpmlp_last_error().  The first call on a device (and the first call
 * after that device's context has been destroyed and recreated, e.g. by
 * cudaDeviceReset) looks up the array's device address in the current context
 * (cudaGetSymbolAddress); make that call before any stream capture.  Every call
 * uses the same array and leaves its partials there; pass 1 writes every
 * partial that pass 2 reads, so nothing in it needs to start at zero.  Calls
 * that can overlap on the GPU (other streams, other host threads) race on the
 * array: serialise them.  rows = 0 writes zeros.
 * Errors: INVALID_ARG for an unknown dtype, rows < 0, cols <= 0 or a NULL
 * pointer; UNSUPPORTED beyond the scratch limit; CUDA when a launch fails. */
tpmlp_status tpmlp_colsum_noalloc(int32_t dtype, const void *x, int64_t rows, int64_t cols, void *out,
                                  void *stream);

/* Number of kernels this library has launched since it was loaded. */
uint64_t tpmlp_launch_count(void);

/* Per-kernel timing.  While enabled, every launch is bracketed by CUDA events
 * on its own stream; tpmlp_profile_collect() waits for them and adds their
 * durations to a per-kernel table (name, launches, total milliseconds). */
void tpmlp_profile_enable(int on);
void tpmlp_profile_reset(void);
tpmlp_status tpmlp_profile_collect(void);
int tpmlp_profile_count(void);
int tpmlp_profile_entry(int i, char *name, int name_len, int64_t *launches, double *total_ms);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
