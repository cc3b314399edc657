// The C ABI of libtpmlp.so (declared in include/tpmlp.h): argument validation,
// workspace layout, the launch sequence of the forward and backward passes, the
// device status word and per-kernel timing.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
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
// The GEMM kernels count output tiles (128 x 256 at the smallest, times the
// problem count) in 32-bit integers.
bool tiles_fit(int64_t M, int64_t N, int64_t batch = 1) {
    const int64_t t = ((M + 127) / 128) * ((N + 255) / 256);
    return t <= (int64_t{1} << 31) / 2 && batch <= (int64_t{1} << 31) / 2 / (t > 0 ? t : 1);
}

bool shape_valid(const tpmlp_shape *s) {
    if (!s) return false;
    if (s->tokens < 0 || s->hidden <= 0 || s->ffn <= 0) return false;
    if (s->t < 1 || s->t > 16 || s->ffn % s->t != 0) return false;
    if (s->dtype != TPMLP_F32 && s->dtype != TPMLP_BF16) return false;
    if (s->algo != TPMLP_ALGO_DEFAULT && s->algo != TPMLP_ALGO_SIMT) return false;
    if ((s->flags & ~(TPMLP_FLAG_RECOMPUTE | TPMLP_FLAG_LAYERNORM)) != 0) return false;
    // int32 tile and grid arithmetic inside the kernels
    if (s->tokens > (1LL << 30) || s->hidden > (1LL << 30) || s->ffn > (1LL << 30)) return false;
    const int64_t T = s->tokens, h = s->hidden, F = s->ffn;
    // the six GEMMs: T x F (fc1, dY), T x h (fc2, dX), F x h (dB), h x F (dA)
    if (!tiles_fit(T, F) || !tiles_fit(T, h) || !tiles_fit(F + 256, h) || !tiles_fit(h, F)) return false;
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

// 64 x 64 bf16 ones: the A operand of the bias-gradient tile of dB = Y^T dZ.
constexpr size_t ONES_BYTES = 64 * 64 * 2;

size_t ones_offset(const tpmlp_shape *s) { return dxn_offset(s) + dxn_bytes(s); }

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

// Raster order of the tensor-core GEMM tiles (256 x 256, 256 x 512 or 128 x 256).  Tiles are walked in
// super-rows of G tiles along M (or N); the G operand panels of the grouped
// dimension (each spans all of K) are re-read while the super-row lasts, so
// they should stay in L2, and each panel of the other operand is read once per
// super-row.  DRAM traffic is about  A + B * ceil(m_tiles / G)  (groups along M)
// or  B + A * ceil(n_tiles / G)  (along N); G is the largest group whose panels
// fit in the L2 budget, and the cheaper direction wins.
// TPMLP_RASTER=m:G or n:G overrides the choice (a tuning knob, read per call).
void pick_raster(GemmArgs &g, Epi epi = tpmlp::EPI_FOLD) {
    const int64_t tile_m = g.cta_pair ? 256 : 128;
    const int64_t tile_n = tpmlp::tc_wide_tile(epi, g) ? 512 : 256;
    const int64_t m_tiles = (g.M + tile_m - 1) / tile_m, n_tiles = (g.N + tile_n - 1) / tile_n;
    const char *env = std::getenv("TPMLP_RASTER");
    if (env && (env[0] == 'm' || env[0] == 'n') && env[1] == ':') {
        g.raster_n = env[0] == 'n';
        g.group = std::atoi(env + 2);
        return;
    }
    // At most 32 M-tiles (M is the token count or the hidden size in every GEMM
    // of the MLP and attention blocks at these sizes): walk up to 16 of them,
    // all where there are 16 or fewer, down each group of N columns.  Per GEMM
    // at h8192 (ncu, one kernel per capture) this order read 8-25% fewer DRAM
    // bytes than the panel-budget rule below and ran up to 2% faster alone.
    if (g.batch <= 1 && m_tiles <= 32) {
        g.raster_n = false;
        g.group = static_cast<int>(m_tiles < 16 ? m_tiles : 16);
        return;
    }
    const char *bud = std::getenv("TPMLP_L2_PANEL_MB");
    const double budget = (bud ? std::atof(bud) : 24.0) * 1048576.0;
    const double a_panel = static_cast<double>(tile_m) * g.K * 2, b_panel = static_cast<double>(tile_n) * g.K * 2;
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
    return ones_offset(s) + ONES_BYTES;
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
    if (!workspace) return invalid("tpmlp_forward: workspace is NULL");
    if (!aligned16(workspace)) return TPMLP_ERR_UNSUPPORTED;
    // Inference (saved == NULL): nothing is kept; Y goes to the workspace.
    if (!saved)
        return s->tokens == 0 ? check_ptrs(s, {A, a, B, b}, {X, Z}) : check_ptrs(s, {X, A, a, B, b, Z}, {});
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
    if (saved) {
        saved->X = X;
        saved->A = A;
        saved->B = B;
    }
    const int64_t T = s->tokens, h = s->hidden, F = s->ffn;
    if (T == 0) return TPMLP_OK;
    const int sms = num_sms_current();
    if (sms == 0) return TPMLP_ERR_CUDA;
    if (use_tc(s) && sms < 0) return TPMLP_ERR_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t *status = static_cast<uint32_t *>(workspace);
    // Y: the caller's buffer; under recomputation the workspace's Y region; for
    // inference (saved == NULL) the workspace's dY region, which only the
    // backward pass uses.
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *Y = !saved ? static_cast<void *>(ws + dy_offset(s)) : (rec ? static_cast<void *>(ws + y_offset(s)) : saved->Y);

    // Column-parallel GEMM of all shards, bias and GeLU fused: H = X A + a, Y = GeLU(H).
    GemmArgs g1 = base_args(status);
    g1.a = X, g1.a_mn = false;  // X[T,h]: K-major
    g1.b = A, g1.b_mn = true;   // A[h,F]: N contiguous, MN-major
    g1.M = T, g1.N = F, g1.K = h, g1.kshard = h;
    g1.out0 = saved ? saved->H : nullptr, g1.out1 = Y, g1.bias = a;
    pick_raster(g1, tpmlp::EPI_BIAS_GELU);
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

    // db = column sums of dZ: on tensor cores from the dB GEMM's ones tile (below,
    // its block of ones is filled by the da pass), on the FFMA path a two-pass
    // column sum.
    void *ones = ws + ones_offset(s);
    cudaError_t e = cudaSuccess;
    if (!use_tc(s)) {
        e = colsum(s, "colsum_db", dZ, T, h, partials, db, st);
        if (e != cudaSuccess) return from_cuda(e);
    }

    // dY = (dZ B^T) * GeLU'(H)
    GemmArgs g3 = base_args(status);
    g3.a = dZ, g3.a_mn = false;        // dZ[T,h]: K-major
    g3.b = saved->B, g3.b_mn = false;  // B[F,h] as [N=F, K=h]: K-major
    g3.M = T, g3.N = F, g3.K = h, g3.kshard = h;
    g3.out0 = dY, g3.aux = saved->H;
    g3.out1 = rec ? Y : nullptr;
    // On tensor cores the epilogue also sums dY's columns per 32-row block.
    g3.colsum_part = use_tc(s) ? partials : nullptr;
    pick_raster(g3, tpmlp::EPI_DGELU);
    e = gemm(s, "bwd_dY_dgelu", tpmlp::EPI_DGELU, g3, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // da = column sums of dY: the in-order sum of those block partials, or a
    // two-pass column sum of dY on the FFMA path.
    if (use_tc(s)) {
        Timed timed("da_block_sum", st);
        e = tpmlp::launch_colsum_final(true, partials, (T + 31) / 32, F, da, st, ones);
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
    if (use_tc(s)) g4.ones = ones, g4.bias_grad = db;  // db = 1^T dZ from an extra ones tile
    pick_raster(g4, tpmlp::EPI_STORE);
    e = gemm(s, "bwd_dB", tpmlp::EPI_STORE, g4, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dA = X^T dY
    GemmArgs g5 = base_args(status);
    g5.a = saved->X, g5.a_mn = true;  // X[T,h] as [K=T, M=h]: MN-major
    g5.b = dY, g5.b_mn = true;        // dY[T,F] as [K=T, N=F]: MN-major
    g5.M = h, g5.N = F, g5.K = T, g5.kshard = T;
    g5.out0 = dA;
    pick_raster(g5, tpmlp::EPI_STORE);
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

// ---- tensor-parallel self-attention block ------------------------------------------------
namespace {

bool attn_shape_valid(const tpmlp_attn_shape *s) {
    if (!s) return false;
    if (s->batch < 0 || s->seq <= 0 || s->hidden <= 0 || s->heads <= 0) return false;
    if (s->t < 1 || s->t > 16 || s->heads % s->t != 0 || s->hidden % s->heads != 0) return false;
    if ((s->flags & ~TPMLP_ATTN_P_UPPER_ZERO) != 0) return false;
    // int32 tile and grid arithmetic inside the kernels
    if (s->hidden > (1LL << 28) || s->seq > (1LL << 20) || s->batch * s->seq > (1LL << 30)) return false;
    if (static_cast<int64_t>(s->batch) * s->heads > (1LL << 24)) return false;
    // tile counts of the projections and the per-head products; the scores
    // ([batch*heads][seq][seq]) must be addressable
    const int64_t T = s->batch * s->seq, h = s->hidden, nz = s->batch * s->heads;
    if (!tiles_fit(T, 3 * h) || !tiles_fit(h + 256, 3 * h) || !tiles_fit(s->seq, s->seq, nz)) return false;
    if (static_cast<double>(nz) * s->seq * s->seq > static_cast<double>(1LL << 48)) return false;
    return true;
}

// Device workspace of the attention block, 1 KB-aligned regions:
//   status | D [batch*heads*seq] fp32 | dO [T,h] bf16 | dQKV [T,3h] bf16 |
//   scores [batch*heads][seq][seq] fp16 (the backward reuses it for dS in bf16) |
//   a 64 x 64 bf16 block of ones (bias-gradient tiles).
// The per-head GEMMs address Q, K, V, O, dO, dQ, dK, dV in place inside the
// token-major QKV, O, dO and dQKV arrays (4-D and 5-D tensor maps).
struct AttnLayout {
    size_t D, dO, dQKV, scores, ones, total;
};

AttnLayout attn_layout(const tpmlp_attn_shape *s) {
    const int64_t T = s->batch * s->seq, h = s->hidden;
    AttnLayout L;
    size_t off = STATUS_BYTES;
    L.D = off;
    off += align_up(static_cast<size_t>(T) * s->heads * 4, 1024);
    const size_t th = align_up(static_cast<size_t>(T) * h * 2, 1024);
    L.dO = off;
    off += th;
    L.dQKV = off;
    off += 3 * th;
    L.scores = off;
    off += align_up(static_cast<size_t>(s->batch) * s->heads * s->seq * s->seq * 2, 1024);
    L.ones = off;
    off += ONES_BYTES;
    L.total = off;
    return L;
}

// The MLP shape that routes the attention GEMMs and column sums to the bf16
// tensor-core path.
tpmlp_shape attn_route(const tpmlp_attn_shape *s) {
    tpmlp_shape m;
    std::memset(&m, 0, sizeof(m));
    m.tokens = s->batch * s->seq;
    m.hidden = s->hidden;
    m.ffn = 3 * s->hidden;
    m.t = s->t;
    m.dtype = TPMLP_BF16;
    m.algo = TPMLP_ALGO_DEFAULT;
    return m;
}

tpmlp::HeadLayout head_layout(const tpmlp_attn_shape *s) {
    tpmlp::HeadLayout L;
    L.nb = s->batch;
    L.S = s->seq;
    L.h = s->hidden;
    L.heads = s->heads;
    L.d = s->hidden / s->heads;
    return L;
}

// Head g's Q (which = 0), K (1) or V (2) columns inside a token-major [T, 3h]
// array with shard-major columns (QKV, dQKV), as a rank-5 view; its base is the
// array plus which * h/t elements.
tpmlp::HeadView qkv_view(const tpmlp_attn_shape *s) {
    tpmlp::HeadView v;
    v.rank = 5;
    v.S = s->seq;
    v.nb = s->batch;
    v.heads = s->heads;
    v.hpt = s->heads / s->t;
    v.d = s->hidden / s->heads;
    v.ld = 3 * s->hidden;
    v.coli = 3 * s->hidden / s->t;
    return v;
}

// Head g's columns [g*d, (g+1)*d) of a token-major [T, h] array (O, dO), rank 4.
tpmlp::HeadView tok_view(const tpmlp_attn_shape *s) {
    tpmlp::HeadView v;
    v.rank = 4;
    v.S = s->seq;
    v.nb = s->batch;
    v.heads = s->heads;
    v.hpt = s->heads / s->t;
    v.d = s->hidden / s->heads;
    v.ld = s->hidden;
    v.coli = 0;
    return v;
}

const void *qkv_part(const void *base, const tpmlp_attn_shape *s, int which) {
    return static_cast<const uint8_t *>(base) + static_cast<size_t>(which) * (s->hidden / s->t) * 2;
}

tpmlp_status attn_check(const tpmlp_attn_shape *s, const char *who, std::initializer_list<const void *> required,
                        std::initializer_list<const void *> token_ptrs, const void *workspace) {
    if (!attn_shape_valid(s)) {
        tpmlp::set_last_error("%s: invalid shape", who);
        return TPMLP_ERR_INVALID_ARG;
    }
    if (!workspace) {
        tpmlp::set_last_error("%s: workspace is NULL", who);
        return TPMLP_ERR_INVALID_ARG;
    }
    const bool empty = s->batch == 0;
    for (const void *p : required)
        if (!p) {
            tpmlp::set_last_error("%s: NULL pointer", who);
            return TPMLP_ERR_INVALID_ARG;
        }
    for (const void *p : token_ptrs)
        if (!p && !empty) {
            tpmlp::set_last_error("%s: NULL pointer", who);
            return TPMLP_ERR_INVALID_ARG;
        }
    if (s->dtype != TPMLP_BF16) {
        tpmlp::set_last_error("%s: the attention block runs in bf16 only", who);
        return TPMLP_ERR_UNSUPPORTED;
    }
    const int64_t d = s->hidden / s->heads;
    if (d % 64 != 0 || s->seq % 8 != 0) {
        tpmlp::set_last_error("%s: head size %lld must be a multiple of 64 and seq %lld of 8", who,
                              static_cast<long long>(d), static_cast<long long>(s->seq));
        return TPMLP_ERR_UNSUPPORTED;
    }
    if (!aligned16(workspace)) return TPMLP_ERR_UNSUPPORTED;
    for (const void *p : required)
        if (!aligned16(p)) return TPMLP_ERR_UNSUPPORTED;
    for (const void *p : token_ptrs)
        if (p && !aligned16(p)) return TPMLP_ERR_UNSUPPORTED;
    return TPMLP_OK;
}

// One batched GEMM of the per-head products.
GemmArgs head_gemm(uint32_t *status, const void *a, bool a_mn, const void *b, bool b_mn, int64_t M, int64_t N,
                   int64_t K, int64_t batch, void *out) {
    GemmArgs g = base_args(status);
    g.a = a, g.a_mn = a_mn;
    g.b = b, g.b_mn = b_mn;
    g.M = M, g.N = N, g.K = K, g.kshard = K;
    g.batch = batch;
    g.out0 = out;
    pick_raster(g);
    return g;
}

}  // namespace

extern "C" {

size_t tpmlp_attn_saved_bytes(const tpmlp_attn_shape *s) {
    if (!attn_shape_valid(s)) return 0;
    const size_t T = static_cast<size_t>(s->batch * s->seq), h = static_cast<size_t>(s->hidden);
    return 2 * (T * 3 * h + T * h + static_cast<size_t>(s->batch) * s->heads * s->seq * s->seq);
}

size_t tpmlp_attn_workspace_bytes(const tpmlp_attn_shape *s) {
    if (!attn_shape_valid(s)) return 0;
    return attn_layout(s).total;
}

tpmlp_status tpmlp_attn_forward(const tpmlp_attn_shape *s, const void *X, const void *Wqkv, const void *bqkv,
                                const void *Wo, const void *bo, void *Z, tpmlp_attn_saved *saved, void *workspace,
                                void *stream) {
    tpmlp::g_last_error[0] = '\0';
    if (!saved) return invalid("tpmlp_attn_forward: saved is NULL");
    tpmlp_status rc = attn_check(s, "tpmlp_attn_forward", {Wqkv, bqkv, Wo, bo},
                                 {X, Z, saved->QKV, saved->P, saved->O}, workspace);
    if (rc != TPMLP_OK) return rc;
    saved->X = X;
    saved->Wqkv = Wqkv;
    saved->Wo = Wo;
    if (s->batch == 0) return TPMLP_OK;
    const int sms = num_sms_current();
    if (sms == 0) return TPMLP_ERR_CUDA;
    if (sms < 0) return TPMLP_ERR_DEVICE;
    const tpmlp_shape ms = attn_route(s);
    const AttnLayout L = attn_layout(s);
    const int64_t T = s->batch * s->seq, h = s->hidden, S = s->seq, d = h / s->heads;
    const int64_t nz = s->batch * s->heads;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    void *scores = ws + L.scores;
    const tpmlp::HeadView qv = qkv_view(s), tv = tok_view(s);
    const void *Qp = qkv_part(saved->QKV, s, 0), *Kp = qkv_part(saved->QKV, s, 1), *Vp = qkv_part(saved->QKV, s, 2);

    // Column-parallel projection of all shards: QKV = X Wqkv + bqkv (the bias
    // epilogue without an activation, on 256 x 512 tiles).
    GemmArgs g1 = base_args(status);
    g1.a = X, g1.a_mn = false;     // X[T,h]: K-major
    g1.b = Wqkv, g1.b_mn = true;   // Wqkv[h,3h]: MN-major
    g1.M = T, g1.N = 3 * h, g1.K = h, g1.kshard = h;
    g1.out0 = saved->QKV, g1.out1 = nullptr, g1.bias = bqkv;
    pick_raster(g1, tpmlp::EPI_BIAS_GELU);
    cudaError_t e = gemm(&ms, "attn_qkv_proj", tpmlp::EPI_BIAS_GELU, g1, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // Scores of every head: scale * Q K^T, causal; Q and K read in place in QKV.
    GemmArgs g2 = head_gemm(status, Qp, false, Kp, false, S, S, d, nz, scores);
    g2.heads_layout = true, g2.a_view = qv, g2.b_view = qv;
    g2.scale = 1.0f / std::sqrt(static_cast<float>(d));
    g2.causal = true;
    g2.skip_upper = true;  // never read: the softmax stops at the diagonal
    e = gemm(&ms, "attn_scores", tpmlp::EPI_ATTN_SCORE, g2, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    {
        Timed timed("attn_softmax", st);
        // With TPMLP_ATTN_P_UPPER_ZERO the 256 x 256 tiles of P wholly above the
        // diagonal (never read: P V and dS K stop at the tile's keys, P^T dO starts
        // at its queries, dS skips them) already hold zeros and are not written.
        const int64_t wtile = (s->flags & TPMLP_ATTN_P_UPPER_ZERO) ? 256 : 0;
        e = tpmlp::launch_softmax(scores, saved->P, nz * S, S, true, wtile, st);
        if (e != cudaSuccess) return from_cuda(e);
        g_launches.fetch_add(1);
    }

    // O_head = P V, V read in place in QKV, O_head written in place in O[T,h].
    GemmArgs g3 = head_gemm(status, saved->P, false, Vp, true, S, d, S, nz, saved->O);
    g3.causal_k = 1;  // P is zero past each row's last key
    g3.heads_layout = true, g3.b_view = qv, g3.o_view = tv;
    e = gemm(&ms, "attn_pv", tpmlp::EPI_STORE, g3, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // Row-parallel output projection: shard partials O_i Wo_i folded in order, + bo.
    GemmArgs g4 = base_args(status);
    g4.a = saved->O, g4.a_mn = false;  // O[T,h]: K-major
    g4.b = Wo, g4.b_mn = true;         // Wo[h,h]: MN-major
    g4.M = T, g4.N = h, g4.K = h;
    g4.nshards = s->t, g4.kshard = h / s->t;
    g4.out0 = Z, g4.bias = bo;
    pick_raster(g4);
    e = gemm(&ms, "attn_out_proj_fold", tpmlp::EPI_FOLD_BIAS, g4, sms, st);
    return from_cuda(e);
}

tpmlp_status tpmlp_attn_backward(const tpmlp_attn_shape *s, const void *dZ, const tpmlp_attn_saved *saved,
                                 void *dX, void *dWqkv, void *dbqkv, void *dWo, void *dbo, void *workspace,
                                 void *stream) {
    tpmlp::g_last_error[0] = '\0';
    if (!saved) return invalid("tpmlp_attn_backward: saved is NULL");
    tpmlp_status rc = attn_check(s, "tpmlp_attn_backward", {saved->Wqkv, saved->Wo, dWqkv, dbqkv, dWo, dbo},
                                 {dZ, saved->X, saved->QKV, saved->P, saved->O, dX}, workspace);
    if (rc != TPMLP_OK) return rc;
    const int64_t T = s->batch * s->seq, h = s->hidden, S = s->seq, d = h / s->heads;
    const int64_t nz = s->batch * s->heads;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // Empty batch: the weight and bias gradients are sums over no tokens.
        cudaError_t e = cudaMemsetAsync(dWqkv, 0, static_cast<size_t>(h) * 3 * h * 2, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dbqkv, 0, static_cast<size_t>(3 * h) * 2, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dWo, 0, static_cast<size_t>(h) * h * 2, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(dbo, 0, static_cast<size_t>(h) * 2, st);
        return from_cuda(e);
    }
    const int sms = num_sms_current();
    if (sms == 0) return TPMLP_ERR_CUDA;
    if (sms < 0) return TPMLP_ERR_DEVICE;
    const tpmlp_shape ms = attn_route(s);
    const AttnLayout L = attn_layout(s);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws);
    float *D = reinterpret_cast<float *>(ws + L.D);
    void *dO = ws + L.dO, *dQKV = ws + L.dQKV;
    // Per-head Q, K, V (in the saved QKV), dO (in dO[T,h]) and dQ, dK, dV (in
    // dQKV) are addressed in place through rank-5 and rank-4 views.
    const tpmlp::HeadView qv = qkv_view(s), tv = tok_view(s);
    const void *Qp = qkv_part(saved->QKV, s, 0), *Kp = qkv_part(saved->QKV, s, 1), *Vp = qkv_part(saved->QKV, s, 2);
    void *dQp = const_cast<void *>(qkv_part(dQKV, s, 0)), *dKp = const_cast<void *>(qkv_part(dQKV, s, 1)),
         *dVp = const_cast<void *>(qkv_part(dQKV, s, 2));
    void *dS = ws + L.scores;  // bf16 [nz][S][S] over the dead fp16 scores
    const float scale = 1.0f / std::sqrt(static_cast<float>(d));

    // dbo = 1^T dZ and dbqkv = 1^T dQKV come from the ones tiles of the dWo and
    // dWqkv GEMMs; the row-dot pass, which runs before both, fills the ones.
    void *ones = ws + L.ones;
    cudaError_t e;

    // dO = dZ Wo^T (every shard's columns at once; no fold needed)
    GemmArgs g1 = base_args(status);
    g1.a = dZ, g1.a_mn = false;         // dZ[T,h]: K-major
    g1.b = saved->Wo, g1.b_mn = false;  // Wo[h,h] as [N, K]: K-major
    g1.M = T, g1.N = h, g1.K = h, g1.kshard = h;
    g1.out0 = dO;
    pick_raster(g1, tpmlp::EPI_STORE);
    e = gemm(&ms, "attn_bwd_dO", tpmlp::EPI_STORE, g1, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // D = rowsum(dO * O) per head (and the block of ones)
    {
        Timed timed("attn_bwd_rowdot", st);
        e = tpmlp::launch_rowdot(head_layout(s), dO, saved->O, D, st, ones);
        if (e != cudaSuccess) return from_cuda(e);
        g_launches.fetch_add(1);
    }

    // dWo = O^T dZ
    GemmArgs g2 = base_args(status);
    g2.a = saved->O, g2.a_mn = true;  // O[T,h] as [K=T, M=h]: MN-major
    g2.b = dZ, g2.b_mn = true;        // dZ[T,h] as [K=T, N=h]: MN-major
    g2.M = h, g2.N = h, g2.K = T, g2.kshard = T;
    g2.out0 = dWo;
    g2.ones = ones, g2.bias_grad = dbo;
    pick_raster(g2, tpmlp::EPI_STORE);
    e = gemm(&ms, "attn_bwd_dWo", tpmlp::EPI_STORE, g2, sms, st);
    if (e != cudaSuccess) return from_cuda(e);


    // dV_head = P^T dO_head
    GemmArgs g3 = head_gemm(status, saved->P, true, dO, true, S, d, S, nz, dVp);
    g3.causal_k = 2;  // key j only gets gradient from queries i >= j
    g3.heads_layout = true, g3.b_view = tv, g3.o_view = qv;
    e = gemm(&ms, "attn_bwd_dV", tpmlp::EPI_STORE, g3, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dS = P * (dO V^T - D) * scale
    GemmArgs g4 = head_gemm(status, dO, false, Vp, false, S, S, d, nz, dS);
    g4.heads_layout = true, g4.a_view = tv, g4.b_view = qv;
    g4.aux = saved->P;
    g4.rowvec = D;
    g4.scale = scale;
    g4.skip_upper = true;  // dS is zero above the diagonal; dQ and dK below never read those tiles
    e = gemm(&ms, "attn_bwd_dS", tpmlp::EPI_ATTN_DS, g4, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dQ_head = dS K_head,  dK_head = dS^T Q_head
    GemmArgs g5 = head_gemm(status, dS, false, Kp, true, S, d, S, nz, dQp);
    g5.causal_k = 1;
    g5.heads_layout = true, g5.b_view = qv, g5.o_view = qv;
    e = gemm(&ms, "attn_bwd_dQ", tpmlp::EPI_STORE, g5, sms, st);
    if (e != cudaSuccess) return from_cuda(e);
    GemmArgs g6 = head_gemm(status, dS, true, Qp, true, S, d, S, nz, dKp);
    g6.causal_k = 2;
    g6.heads_layout = true, g6.b_view = qv, g6.o_view = qv;
    e = gemm(&ms, "attn_bwd_dK", tpmlp::EPI_STORE, g6, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dWqkv = X^T dQKV
    GemmArgs g7 = base_args(status);
    g7.a = saved->X, g7.a_mn = true;  // X[T,h] as [K=T, M=h]: MN-major
    g7.b = dQKV, g7.b_mn = true;      // dQKV[T,3h] as [K=T, N=3h]: MN-major
    g7.M = h, g7.N = 3 * h, g7.K = T, g7.kshard = T;
    g7.out0 = dWqkv;
    g7.ones = ones, g7.bias_grad = dbqkv;
    pick_raster(g7, tpmlp::EPI_STORE);
    e = gemm(&ms, "attn_bwd_dWqkv", tpmlp::EPI_STORE, g7, sms, st);
    if (e != cudaSuccess) return from_cuda(e);

    // dX = sum_i dQKV_i Wqkv_i^T, shard partials folded in order (the backward all-reduce)
    GemmArgs g8 = base_args(status);
    g8.a = dQKV, g8.a_mn = false;         // dQKV[T,3h]: K-major
    g8.b = saved->Wqkv, g8.b_mn = false;  // Wqkv[h,3h] as [N=h, K=3h]: K-major
    g8.M = T, g8.N = h, g8.K = 3 * h;
    g8.nshards = s->t, g8.kshard = 3 * h / s->t;
    g8.out0 = dX;
    pick_raster(g8);
    e = gemm(&ms, "attn_bwd_dX_shard_fold", tpmlp::EPI_FOLD, g8, sms, st);
    return from_cuda(e);
}

}  // extern "C"
