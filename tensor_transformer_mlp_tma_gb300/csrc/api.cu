// The C ABI of libtpmlp.so (declared in include/tpmlp.h): argument validation,
// workspace layout, the launch sequence of the forward and backward passes, the
// device status word and per-kernel timing.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"
#include "tpmlp.h"

namespace tpmlp {

thread_local char g_last_error[512] = "";

void set_last_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

}  // namespace tpmlp

namespace {
std::atomic<uint64_t> g_launches{0};
}

void tpmlp::add_launches(uint64_t n) { g_launches.fetch_add(n); }

namespace {

using tpmlp::Epi;
using tpmlp::GemmArgs;

std::atomic<uint64_t> g_wait_ns{2000000000ull};

// ---- per-kernel timing --------------------------------------------------------
struct PendingTiming {
    std::string name;
    cudaEvent_t e0, e1;
};
struct TimingTotal {
    int64_t launches = 0;
    double ms = 0.0;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<PendingTiming> g_pending;
std::vector<cudaEvent_t> g_event_pool;
std::vector<std::pair<std::string, TimingTotal>> g_totals;

cudaEvent_t get_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Brackets one launch with events on its stream when timing is on.
struct Timed {
    const char *name;
    cudaStream_t st;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    Timed(const char *n, cudaStream_t s) : name(n), st(s) {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        if (!g_prof_on) return;
        e0 = get_event();
        e1 = get_event();
        if (e0 && e1) cudaEventRecord(e0, st);
    }
    ~Timed() {
        if (!e0 || !e1) return;
        cudaEventRecord(e1, st);
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_pending.push_back({name, e0, e1});
    }
};

// ---- device properties -----------------------------------------------------------
int num_sms_current() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev] == 0) {
        int n = 0, major = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
        int minor = 0;
        if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return 0;
        cache[dev] = (major == 10 && minor == 3) ? n : -1;  // the kernels are built for sm_103a only
    }
    return cache[dev];
}

// ---- shapes and workspace --------------------------------------------------------------
bool shape_valid(const tpmlp_shape *s) {
    if (!s) return false;
    if (s->tokens < 0 || s->hidden <= 0 || s->ffn <= 0) return false;
    if (s->t < 1 || s->t > 16 || s->ffn % s->t != 0) return false;
    if (s->dtype != TPMLP_F32 && s->dtype != TPMLP_BF16) return false;
    if (s->algo != TPMLP_ALGO_DEFAULT && s->algo != TPMLP_ALGO_SIMT) return false;
    if ((s->flags & ~(TPMLP_FLAG_RECOMPUTE | TPMLP_FLAG_LAYERNORM)) != 0) return false;
    // int32 tile and grid arithmetic inside the kernels
    if (s->tokens > (1LL << 30) || s->hidden > (1LL << 30) || s->ffn > (1LL << 30)) return false;
    return true;
}

size_t elt(const tpmlp_shape *s) { return s->dtype == TPMLP_BF16 ? 2 : 4; }

bool use_tc(const tpmlp_shape *s) { return s->dtype == TPMLP_BF16 && s->algo == TPMLP_ALGO_DEFAULT; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t STATUS_BYTES = 1024;

// fp32 column-sum partials: the two-pass column sums of db (and of da on the
// FFMA path), or the per-32-row-block da partials written by the tensor-core
// GeLU' epilogue.  They are used one after the other, so they share one region.
size_t partials_bytes(const tpmlp_shape *s) {
    const int64_t T = s->tokens, h = s->hidden, F = s->ffn;
    int64_t n = tpmlp::colsum_chunks(T, h) * h;
    const int64_t p2 = tpmlp::colsum_chunks(T, F) * F;
    const int64_t p3 = (T + 31) / 32 * F;
    const int64_t p4 = (s->flags & TPMLP_FLAG_LAYERNORM) ? tpmlp::ln_partial_floats(T, h) : 0;
    n = n > p2 ? n : p2;
    n = n > p3 ? n : p3;
    n = n > p4 ? n : p4;
    return align_up(static_cast<size_t>(n) * sizeof(float), 1024);
}

size_t dy_offset(const tpmlp_shape *s) { return STATUS_BYTES + partials_bytes(s); }

size_t dy_bytes(const tpmlp_shape *s) {
    return align_up(static_cast<size_t>(s->tokens) * static_cast<size_t>(s->ffn) * elt(s), 1024);
}

bool recompute(const tpmlp_shape *s) { return (s->flags & TPMLP_FLAG_RECOMPUTE) != 0; }

size_t y_offset(const tpmlp_shape *s) { return dy_offset(s) + dy_bytes(s); }

size_t y_bytes(const tpmlp_shape *s) { return recompute(s) ? dy_bytes(s) : 0; }

bool layernorm(const tpmlp_shape *s) { return (s->flags & TPMLP_FLAG_LAYERNORM) != 0; }

size_t dxn_offset(const tpmlp_shape *s) { return y_offset(s) + y_bytes(s); }

size_t dxn_bytes(const tpmlp_shape *s) {
    return layernorm(s) ? align_up(static_cast<size_t>(s->tokens) * static_cast<size_t>(s->hidden) * elt(s), 1024)
                        : 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_elt(const void *p, size_t e) { return (reinterpret_cast<uintptr_t>(p) % e) == 0; }

// Checks common to forward and backward.  Returns OK, INVALID_ARG or UNSUPPORTED.
tpmlp_status check_ptrs(const tpmlp_shape *s, std::initializer_list<const void *> required,
                        std::initializer_list<const void *> optional) {
    for (const void *p : required)
        if (!p) return TPMLP_ERR_INVALID_ARG;
    const size_t e = elt(s);
    for (const void *p : required)
        if (!aligned_elt(p, e)) return TPMLP_ERR_UNSUPPORTED;
    for (const void *p : optional)
        if (p && !aligned_elt(p, e)) return TPMLP_ERR_UNSUPPORTED;
    if (use_tc(s)) {
        // TMA: 16-byte aligned bases and row pitches; shard boundaries on 64-element k-blocks.
        for (const void *p : required)
            if (!aligned16(p)) return TPMLP_ERR_UNSUPPORTED;
        for (const void *p : optional)
            if (p && !aligned16(p)) return TPMLP_ERR_UNSUPPORTED;
        if (s->hidden % 8 != 0 || s->ffn % 8 != 0) return TPMLP_ERR_UNSUPPORTED;
        if (s->t > 1 && (s->ffn / s->t) % 64 != 0) return TPMLP_ERR_UNSUPPORTED;
    }
    return TPMLP_OK;
}

tpmlp_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return TPMLP_OK;
    if (tpmlp::g_last_error[0] == '\0') tpmlp::set_last_error("%s", cudaGetErrorString(e));
    return TPMLP_ERR_CUDA;
}

tpmlp_status invalid(const char *why) {
    tpmlp::set_last_error("%s", why);
    return TPMLP_ERR_INVALID_ARG;
}

// One GEMM launch on the selected path.
cudaError_t gemm(const tpmlp_shape *s, const char *name, Epi epi, const GemmArgs &g, int sms,
                 cudaStream_t st) {
    Timed timed(name, st);
    cudaError_t e;
    if (use_tc(s))
        e = tpmlp::launch_tc_gemm(epi, g, sms, st);
    else
        e = tpmlp::launch_simt_gemm(epi, s->dtype == TPMLP_BF16, g, st);
    if (e == cudaSuccess && g.M > 0 && g.N > 0) g_launches.fetch_add(1);
    return e;
}

cudaError_t colsum(const tpmlp_shape *s, const char *name, const void *x, int64_t rows, int64_t cols,
                   float *partials, void *out, cudaStream_t st) {
    Timed timed(name, st);
    int n = 0;
    cudaError_t e = tpmlp::launch_colsum(s->dtype == TPMLP_BF16, x, rows, cols, partials, out, st, &n);
    g_launches.fetch_add(static_cast<uint64_t>(n));
    return e;
}

GemmArgs base_args(uint32_t *status) {
    GemmArgs g;
    std::memset(&g, 0, sizeof(g));
    g.nshards = 1;
    g.status = status;
    g.wait_ns = g_wait_ns.load();
    g.group = 1;
    g.raster_n = false;
    // CTA pairs (256 x 256 tiles) by default; TPMLP_CTA_PAIR=0 selects single-CTA
    // 128 x 256 tiles (a tuning knob, read per call).
    const char *pair = std::getenv("TPMLP_CTA_PAIR");
    g.cta_pair = !(pair && pair[0] == '0');
    return g;
}

// Raster order of the tensor-core GEMM tiles (128 x 256).  Tiles are walked in
// super-rows of G tiles along M (or N); the G operand panels of the grouped
// dimension (each spans all of K) are re-read while the super-row lasts, so
// they should stay in L2, and each panel of the other operand is read once per
// super-row.  DRAM traffic is about  A + B * ceil(m_tiles / G)  (groups along M)
// or  B + A * ceil(n_tiles / G)  (along N); G is the largest group whose panels
// fit in the L2 budget, and the cheaper direction wins.
// TPMLP_RASTER=m:G or n:G overrides the choice (a tuning knob, read per call).
void pick_raster(GemmArgs &g) {
    const int64_t tile_m = g.cta_pair ? 256 : 128;
    const int64_t m_tiles = (g.M + tile_m - 1) / tile_m, n_tiles = (g.N + 255) / 256;
    const char *env = std::getenv("TPMLP_RASTER");
    if (env && (env[0] == 'm' || env[0] == 'n') && env[1] == ':') {
        g.raster_n = env[0] == 'n';
        g.group = std::atoi(env + 2);
        return;
    }
    const char *bud = std::getenv("TPMLP_L2_PANEL_MB");
    const double budget = (bud ? std::atof(bud) : 24.0) * 1048576.0;
    const double a_panel = static_cast<double>(tile_m) * g.K * 2, b_panel = 256.0 * g.K * 2;
    const double a_total = static_cast<double>(g.M) * g.K * 2, b_total = static_cast<double>(g.N) * g.K * 2;
    int64_t gm = static_cast<int64_t>(budget / a_panel), gn = static_cast<int64_t>(budget / b_panel);
    // Very long K makes panels too big for the budget; tiles that run in the same
    // wave still share panels while they walk K together, so keep the wave
    // roughly square: G between 8 and 24 tiles (measured best on GB300).
    gm = gm < 8 ? 8 : (gm > 24 ? 24 : gm);
    gn = gn < 8 ? 8 : (gn > 24 ? 24 : gn);
    gm = gm > m_tiles ? m_tiles : gm;
    gn = gn > n_tiles ? n_tiles : gn;
    const double tm = a_total + b_total * static_cast<double>((m_tiles + gm - 1) / gm);
    const double tn = b_total + a_total * static_cast<double>((n_tiles + gn - 1) / gn);
    g.raster_n = tn < tm;
    g.group = static_cast<int>(g.raster_n ? gn : gm);
}

}  // namespace

extern "C" {

const char *tpmlp_status_string(tpmlp_status s) {
    switch (s) {
        case TPMLP_OK: return "ok";
        case TPMLP_ERR_INVALID_ARG: return "invalid argument";
        case TPMLP_ERR_UNSUPPORTED: return "unsupported argument (alignment or shard size)";
        case TPMLP_ERR_CUDA: return "CUDA error";
        case TPMLP_ERR_TIMEOUT: return "device-side wait timed out";
        case TPMLP_ERR_DEVICE: return "no usable sm_100-family device";
    }
    return "unknown status";
}

int tpmlp_version(void) { return 100; }

const char *tpmlp_last_error(void) { return tpmlp::g_last_error; }

size_t tpmlp_saved_bytes(const tpmlp_shape *s) {
    if (!shape_valid(s)) return 0;
    return (recompute(s) ? 1 : 2) * static_cast<size_t>(s->tokens) * static_cast<size_t>(s->ffn) * elt(s);
}

size_t tpmlp_workspace_bytes(const tpmlp_shape *s) {
    if (!shape_valid(s)) return 0;
    return dxn_offset(s) + dxn_bytes(s);
}

size_t tpmlp_workspace_offset(const tpmlp_shape *s, int region) {
    if (!shape_valid(s)) return static_cast<size_t>(-1);
    switch (region) {
        case TPMLP_WS_STATUS: return 0;
        case TPMLP_WS_PARTIALS: return STATUS_BYTES;
        case TPMLP_WS_DY: return dy_offset(s);
        case TPMLP_WS_Y: return y_offset(s);
        case TPMLP_WS_DXN: return dxn_offset(s);
    }
    return static_cast<size_t>(-1);
}

}  // extern "C"

namespace {

tpmlp_status validate_forward(const tpmlp_shape *s, const void *X, const void *A, const void *a, const void *B,
                              const void *b, const void *Z, const tpmlp_saved *saved, const void *workspace) {
    if (!shape_valid(s)) return invalid("tpmlp_forward: invalid shape");
    if (!saved || !workspace) return invalid("tpmlp_forward: saved or workspace is NULL");
    if (!aligned16(workspace)) return TPMLP_ERR_UNSUPPORTED;
    // With no tokens the [T, .] tensors are empty and may have NULL data pointers.
    // Under recomputation H is the saved activation and Y lives in the workspace.
    const bool rec = recompute(s);
    return s->tokens == 0 ? check_ptrs(s, {A, a, B, b}, {X, Z, saved->Y, saved->H})
           : rec          ? check_ptrs(s, {X, A, a, B, b, Z, saved->H}, {saved->Y})
                          : check_ptrs(s, {X, A, a, B, b, Z, saved->Y}, {saved->H});
}

tpmlp_status validate_backward(const tpmlp_shape *s, const void *dZ, const tpmlp_saved *saved, const void *dX,
                               const void *dA, const void *da, const void *dB, const void *db,
                               const void *workspace) {
    if (!shape_valid(s)) return invalid("tpmlp_backward: invalid shape");
    if (!saved || !workspace) return invalid("tpmlp_backward: saved or workspace is NULL");
    if (!aligned16(workspace)) return TPMLP_ERR_UNSUPPORTED;
    const bool rec = recompute(s);
    return s->tokens == 0
               ? check_ptrs(s, {saved->A, saved->B, dA, da, dB, db}, {dZ, saved->X, saved->H, saved->Y, dX})
           : rec ? check_ptrs(s, {dZ, saved->X, saved->A, saved->B, saved->H, dX, dA, da, dB, db}, {saved->Y})
                 : check_ptrs(s, {dZ, saved->X, saved->A, saved->B, saved->H, saved->Y, dX, dA, da, dB, db}, {});
}

}  // namespace

extern "C" {

tpmlp_status tpmlp_forward(const tpmlp_shape *s, const void *X, const void *A, const void *a,
                           const void *B, const void *b, void *Z, tpmlp_saved *saved,
                           void *workspace, void *stream) {
    tpmlp::g_last_error[0] = '\0';
    tpmlp_status rc = validate_forward(s, X, A, a, B, b, Z, saved, workspace);
    if (rc != TPMLP_OK) return rc;
    const bool rec = recompute(s);
    saved->X = X;
    saved->A = A;
    saved->B = B;
    const int64_t T = s->tokens, h = s->hidden, F = s->ffn;
    if (T == 0) return TPMLP_OK;
    const int sms = num_sms_current();
    if (sms == 0) return TPMLP_ERR_CUDA;
    if (use_tc(s) && sms < 0) return TPMLP_ERR_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t *status = static_cast<uint32_t *>(workspace);
    void *Y = rec ? static_cast<void *>(static_cast<uint8_t *>(workspace) + y_offset(s)) : saved->Y;

    // Column-parallel GEMM of all shards, bias and GeLU fused: H = X A + a, Y = GeLU(H).
    GemmArgs g1 = base_args(status);
    g1.a = X, g1.a_mn = false;  // X[T,h]: K-major
    g1.b = A, g1.b_mn = true;   // A[h,F]: N contiguous, MN-major
    g1.M = T, g1.N = F, g1.K = h, g1.kshard = h;
    g1.out0 = saved->H, g1.out1 = Y, g1.bias = a;
    pick_raster(g1);
    cudaError_t e = gemm(s, "fc1_bias_gelu", tpmlp::EPI_BIAS_GELU, g1, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // Row-parallel GEMM, one accumulation per shard, shard partials folded in order, + b.
    GemmArgs g2 = base_args(status);
    g2.a = Y, g2.a_mn = false;  // Y[T,F]: K-major
    g2.b = B, g2.b_mn = true;          // B[F,h]: MN-major
    g2.M = T, g2.N = h, g2.K = F;
    g2.nshards = s->t, g2.kshard = F / s->t;
    g2.out0 = Z, g2.bias = b;
    pick_raster(g2);
    e = gemm(s, "fc2_shard_fold", tpmlp::EPI_FOLD_BIAS, g2, sms, st);
    return from_cuda(e);
}

tpmlp_status tpmlp_backward(const tpmlp_shape *s, const void *dZ, const tpmlp_saved *saved, void *dX,
                            void *dA, void *da, void *dB, void *db, void *workspace, void *stream) {
    tpmlp::g_last_error[0] = '\0';
    tpmlp_status rc = validate_backward(s, dZ, saved, dX, dA, da, dB, db, workspace);
    if (rc != TPMLP_OK) return rc;
    const bool rec = recompute(s);
    const int64_t T = s->tokens, h = s->hidden, F = s->ffn;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // Empty batch: the weight and bias gradients are sums over no tokens.
        cudaError_t e = cudaMemsetAsync(dA, 0, static_cast<size_t>(h) * F * elt(s), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dB, 0, static_cast<size_t>(F) * h * elt(s), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(da, 0, static_cast<size_t>(F) * elt(s), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(db, 0, static_cast<size_t>(h) * elt(s), st);
        return from_cuda(e);
    }
    const int sms = num_sms_current();
    if (sms == 0) return TPMLP_ERR_CUDA;
    if (use_tc(s) && sms < 0) return TPMLP_ERR_DEVICE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    float *partials = reinterpret_cast<float *>(ws + STATUS_BYTES);
    void *dY = ws + dy_offset(s);
    // Under recomputation the GeLU' epilogue rebuilds Y = GeLU(H) into the workspace.
    void *Y = rec ? static_cast<void *>(ws + y_offset(s)) : saved->Y;

    // db = column sums of dZ
    cudaError_t e = colsum(s, "colsum_db", dZ, T, h, partials, db, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dY = (dZ B^T) * GeLU'(H)
    GemmArgs g3 = base_args(status);
    g3.a = dZ, g3.a_mn = false;        // dZ[T,h]: K-major
    g3.b = saved->B, g3.b_mn = false;  // B[F,h] as [N=F, K=h]: K-major
    g3.M = T, g3.N = F, g3.K = h, g3.kshard = h;
    g3.out0 = dY, g3.aux = saved->H;
    g3.out1 = rec ? Y : nullptr;
    // On tensor cores the epilogue also sums dY's columns per 32-row block.
    g3.colsum_part = use_tc(s) ? partials : nullptr;
    pick_raster(g3);
    e = gemm(s, "bwd_dY_dgelu", tpmlp::EPI_DGELU, g3, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // da = column sums of dY: the in-order sum of those block partials, or a
    // two-pass column sum of dY on the FFMA path.
    if (use_tc(s)) {
        Timed timed("da_block_sum", st);
        e = tpmlp::launch_colsum_final(true, partials, (T + 31) / 32, F, da, st);
        if (e == cudaSuccess) g_launches.fetch_add(1);
    } else {
        e = colsum(s, "colsum_da", dY, T, F, partials, da, st);
    }
    if (e != cudaSuccess) return from_cuda(e);

    // dB = Y^T dZ
    GemmArgs g4 = base_args(status);
    g4.a = Y, g4.a_mn = true;  // Y[T,F] as [K=T, M=F]: MN-major
    g4.b = dZ, g4.b_mn = true;        // dZ[T,h] as [K=T, N=h]: MN-major
    g4.M = F, g4.N = h, g4.K = T, g4.kshard = T;
    g4.out0 = dB;
    pick_raster(g4);
    e = gemm(s, "bwd_dB", tpmlp::EPI_STORE, g4, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dA = X^T dY
    GemmArgs g5 = base_args(status);
    g5.a = saved->X, g5.a_mn = true;  // X[T,h] as [K=T, M=h]: MN-major
    g5.b = dY, g5.b_mn = true;        // dY[T,F] as [K=T, N=F]: MN-major
    g5.M = h, g5.N = F, g5.K = T, g5.kshard = T;
    g5.out0 = dA;
    pick_raster(g5);
    e = gemm(s, "bwd_dA", tpmlp::EPI_STORE, g5, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dX = sum_i dY_i A_i^T, shard partials folded in order (the backward all-reduce)
    GemmArgs g6 = base_args(status);
    g6.a = dY, g6.a_mn = false;        // dY[T,F]: K-major
    g6.b = saved->A, g6.b_mn = false;  // A[h,F] as [N=h, K=F]: K-major
    g6.M = T, g6.N = h, g6.K = F;
    g6.nshards = s->t, g6.kshard = F / s->t;
    g6.out0 = dX;
    pick_raster(g6);
    e = gemm(s, "bwd_dX_shard_fold", tpmlp::EPI_FOLD, g6, sms, st);
    return from_cuda(e);
}

tpmlp_status tpmlp_ln_forward(const tpmlp_shape *s, tpmlp_layernorm *ln, void *stream) {
    tpmlp::g_last_error[0] = '\0';
    if (!shape_valid(s) || !ln) return invalid("tpmlp_ln_forward: invalid shape or NULL layernorm");
    if (!(ln->eps >= 0.0f)) return invalid("tpmlp_ln_forward: eps must be >= 0");
    const int64_t T = s->tokens;
    tpmlp_status rc = T > 0 ? check_ptrs(s, {ln->X_in, ln->gamma, ln->beta, ln->Xn}, {})
                            : check_ptrs(s, {ln->gamma, ln->beta}, {ln->X_in, ln->Xn});
    if (rc != TPMLP_OK) return rc;
    if (T > 0 && (!ln->mean || !ln->rstd)) return invalid("tpmlp_ln_forward: NULL mean or rstd");
    if (T == 0) return TPMLP_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    tpmlp::LnArgs a;
    std::memset(&a, 0, sizeof(a));
    a.rows = T, a.h = s->hidden, a.eps = ln->eps;
    a.x = ln->X_in, a.gamma = ln->gamma, a.beta = ln->beta, a.y = ln->Xn, a.mean = ln->mean, a.rstd = ln->rstd;
    Timed timed("ln_forward", st);
    cudaError_t e = tpmlp::launch_ln_forward(s->dtype == TPMLP_BF16, a, st);
    if (e == cudaSuccess) g_launches.fetch_add(1);
    return from_cuda(e);
}

tpmlp_status tpmlp_ln_backward(const tpmlp_shape *s, const tpmlp_layernorm *ln, const void *dXn, void *dX_in,
                               void *dgamma, void *dbeta, void *workspace, void *stream) {
    tpmlp::g_last_error[0] = '\0';
    if (!shape_valid(s) || !ln || !workspace) return invalid("tpmlp_ln_backward: invalid shape or NULL argument");
    if (!layernorm(s)) return invalid("tpmlp_ln_backward: the shape needs TPMLP_FLAG_LAYERNORM (workspace size)");
    const int64_t T = s->tokens;
    tpmlp_status rc = T > 0 ? check_ptrs(s, {dXn, ln->X_in, ln->gamma, dX_in, dgamma, dbeta}, {})
                            : check_ptrs(s, {ln->gamma, dgamma, dbeta}, {dXn, ln->X_in, dX_in});
    if (rc != TPMLP_OK) return rc;
    if (T > 0 && (!ln->mean || !ln->rstd)) return invalid("tpmlp_ln_backward: NULL mean or rstd");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    tpmlp::LnArgs a;
    std::memset(&a, 0, sizeof(a));
    a.rows = T, a.h = s->hidden, a.eps = ln->eps;
    a.x = ln->X_in, a.gamma = ln->gamma, a.mean = ln->mean, a.rstd = ln->rstd;
    a.dy = dXn, a.dx = dX_in, a.dgamma = dgamma, a.dbeta = dbeta;
    a.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + STATUS_BYTES);
    Timed timed("ln_backward", st);
    int n = 0;
    cudaError_t e = tpmlp::launch_ln_backward(s->dtype == TPMLP_BF16, a, st, &n);
    g_launches.fetch_add(static_cast<uint64_t>(n));
    return from_cuda(e);
}

tpmlp_status tpmlp_sp_forward(const tpmlp_shape *s, tpmlp_layernorm *ln, const void *A, const void *a,
                              const void *B, const void *b, void *Z, tpmlp_saved *saved, void *workspace,
                              void *stream) {
    if (!shape_valid(s) || !ln) return invalid("tpmlp_sp_forward: invalid shape or NULL layernorm");
    if (!layernorm(s)) return invalid("tpmlp_sp_forward: the shape needs TPMLP_FLAG_LAYERNORM");
    // Validate the whole call before the first launch.
    tpmlp_status rc = validate_forward(s, ln->Xn, A, a, B, b, Z, saved, workspace);
    if (rc != TPMLP_OK) return rc;
    if (s->tokens > 0 && (!ln->X_in || !ln->mean || !ln->rstd)) return invalid("tpmlp_sp_forward: NULL layernorm buffer");
    rc = tpmlp_ln_forward(s, ln, stream);
    if (rc != TPMLP_OK) return rc;
    return tpmlp_forward(s, ln->Xn, A, a, B, b, Z, saved, workspace, stream);
}

tpmlp_status tpmlp_sp_backward(const tpmlp_shape *s, const tpmlp_layernorm *ln, const void *dZ,
                               const tpmlp_saved *saved, void *dX_in, void *dgamma, void *dbeta, void *dA,
                               void *da, void *dB, void *db, void *workspace, void *stream) {
    if (!shape_valid(s) || !ln || !workspace) return invalid("tpmlp_sp_backward: invalid shape or NULL argument");
    if (!layernorm(s)) return invalid("tpmlp_sp_backward: the shape needs TPMLP_FLAG_LAYERNORM");
    void *dXn = static_cast<uint8_t *>(workspace) + dxn_offset(s);
    void *dXn_or_null = s->tokens > 0 ? dXn : nullptr;
    // Validate the whole call before the first launch.
    tpmlp_status rc = validate_backward(s, dZ, saved, dXn_or_null, dA, da, dB, db, workspace);
    if (rc != TPMLP_OK) return rc;
    rc = s->tokens > 0 ? check_ptrs(s, {ln->X_in, ln->gamma, dX_in, dgamma, dbeta}, {})
                       : check_ptrs(s, {ln->gamma, dgamma, dbeta}, {ln->X_in, dX_in});
    if (rc != TPMLP_OK) return rc;
    if (s->tokens > 0 && (!ln->mean || !ln->rstd)) return invalid("tpmlp_sp_backward: NULL mean or rstd");
    rc = tpmlp_backward(s, dZ, saved, dXn_or_null, dA, da, dB, db, workspace, stream);
    if (rc != TPMLP_OK) return rc;
    return tpmlp_ln_backward(s, ln, dXn, dX_in, dgamma, dbeta, workspace, stream);
}

tpmlp_status tpmlp_check_device_status(void *workspace, void *stream) {
    if (!workspace) return TPMLP_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t words[2] = {0, 0};
    cudaError_t e = cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return TPMLP_ERR_CUDA;
    if (words[0] != 0) {
        e = cudaMemsetAsync(workspace, 0, sizeof(words), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return TPMLP_ERR_CUDA;
    }
    if (words[0] > TPMLP_ERR_DEVICE) return TPMLP_ERR_DEVICE;
    return static_cast<tpmlp_status>(words[0]);
}

void tpmlp_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns == 0 ? 1 : ns); }

tpmlp_status tpmlp_debug_timeout_probe(void *workspace, uint64_t wait_ns, void *stream) {
    if (!workspace) return TPMLP_ERR_INVALID_ARG;
    if (wait_ns > 10000000000ull) return TPMLP_ERR_INVALID_ARG;  // at most 10 s
    const int sms = num_sms_current();
    if (sms == 0) return TPMLP_ERR_CUDA;
    if (sms < 0) return TPMLP_ERR_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Timed timed("timeout_probe", st);
    cudaError_t e = tpmlp::launch_timeout_probe(static_cast<uint32_t *>(workspace), wait_ns, st);
    if (e == cudaSuccess) g_launches.fetch_add(1);
    return from_cuda(e);
}

uint64_t tpmlp_launch_count(void) { return g_launches.load(); }

void tpmlp_profile_enable(int on) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = on != 0;
}

void tpmlp_profile_reset(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    for (auto &p : g_pending) {
        g_event_pool.push_back(p.e0);
        g_event_pool.push_back(p.e1);
    }
    g_pending.clear();
    g_totals.clear();
}

tpmlp_status tpmlp_profile_collect(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    tpmlp_status rc = TPMLP_OK;
    for (auto &p : g_pending) {
        float ms = 0.0f;
        if (cudaEventSynchronize(p.e1) != cudaSuccess || cudaEventElapsedTime(&ms, p.e0, p.e1) != cudaSuccess) {
            rc = TPMLP_ERR_CUDA;
        } else {
            bool found = false;
            for (auto &t : g_totals)
                if (t.first == p.name) {
                    t.second.launches += 1;
                    t.second.ms += ms;
                    found = true;
                    break;
                }
            if (!found) {
                TimingTotal tt;
                tt.launches = 1;
                tt.ms = ms;
                g_totals.emplace_back(p.name, tt);
            }
        }
        g_event_pool.push_back(p.e0);
        g_event_pool.push_back(p.e1);
    }
    g_pending.clear();
    return rc;
}

int tpmlp_profile_count(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    return static_cast<int>(g_totals.size());
}

int tpmlp_profile_entry(int i, char *name, int name_len, int64_t *launches, double *total_ms) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (i < 0 || i >= static_cast<int>(g_totals.size())) return -1;
    const auto &t = g_totals[static_cast<size_t>(i)];
    if (name && name_len > 0) {
        std::strncpy(name, t.first.c_str(), static_cast<size_t>(name_len - 1));
        name[name_len - 1] = '\0';
    }
    if (launches) *launches = t.second.launches;
    if (total_ms) *total_ms = t.second.ms;
    return 0;
}

}  // extern "C"
