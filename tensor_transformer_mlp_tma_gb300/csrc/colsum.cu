// Bias gradients db = 1^T dZ and da = 1^T dY: deterministic column sums of a
// row-major [rows, cols] matrix, memory bound.
//
// Pass 1: a (32 x 8)-thread block owns 32*VEC consecutive columns (one 16-byte
// vector per thread and row, so a warp reads 512 contiguous bytes per row) and
// one chunk of rows; the 8 row-interleaved partial sums are combined in fixed
// order and written to an fp32 partials array [chunks, cols].
// Pass 2: one thread per column adds the chunk partials in ascending order
// (16 loads in flight per thread).
// Every sum has a fixed order for a given shape, so results are bit-identical
// from run to run.
//
// Also here: the timeout probe, a kernel whose only job is to run a bounded wait
// to its limit and report it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tpmlp.h"

namespace tpmlp {
namespace colsum {

constexpr int BX = 32, BY = 8;

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int N = 4;
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
};

template <typename T>
__device__ __forceinline__ void load_vec(const T *p, float *v);
template <>
__device__ __forceinline__ void load_vec<float>(const float *p, float *v) {
    const float4 w = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = w.x;
    v[1] = w.y;
    v[2] = w.z;
    v[3] = w.w;
}
template <>
__device__ __forceinline__ void load_vec<__nv_bfloat16>(const __nv_bfloat16 *p, float *v) {
    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u[i]);
        v[2 * i] = __low2float(b);
        v[2 * i + 1] = __high2float(b);
    }
}

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

// VEC > 1: vector loads (cols % VEC == 0 and x 16-byte aligned); VEC == 1: scalar.
template <typename T, int VEC>
__global__ void __launch_bounds__(BX *BY) partial_kernel(const T *__restrict__ x, int64_t rows,
                                                         int64_t cols, int64_t rows_per_chunk,
                                                         float *__restrict__ part) {
    __shared__ float red[BY][BX * VEC];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t col = (static_cast<int64_t>(blockIdx.x) * BX + tx) * VEC;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_chunk;
    const int64_t r1 = min(rows, r0 + rows_per_chunk);
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.0f;
    if (col < cols) {
        for (int64_t r = r0 + ty; r < r1; r += BY) {
            float v[VEC];
            if constexpr (VEC > 1) {
                load_vec<T>(x + r * cols + col, v);
            } else {
                v[0] = to_f<T>(x[r * cols + col]);
            }
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] += v[i];
        }
    }
#pragma unroll
    for (int v = 0; v < VEC; ++v) red[ty][tx * VEC + v] = acc[v];
    __syncthreads();
    // BX*VEC columns, BX*BY threads: each thread finishes up to VEC/BY... use a
    // strided loop so any VEC works.
    for (int c = ty * BX + tx; c < BX * VEC; c += BX * BY) {
        float s = red[0][c];
#pragma unroll
        for (int y = 1; y < BY; ++y) s += red[y][c];
        const int64_t gc = static_cast<int64_t>(blockIdx.x) * BX * VEC + c;
        if (gc < cols) part[static_cast<int64_t>(blockIdx.y) * cols + gc] = s;
    }
}

template <typename T>
__device__ __forceinline__ void store_out(T *p, int64_t i, float v);
template <>
__device__ __forceinline__ void store_out<float>(float *p, int64_t i, float v) {
    p[i] = v;
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16 *p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

// The chunk partials of a column are added in ascending order.  They are loaded
// 16 at a time before being added (same order), so a thread keeps 16 loads in
// flight instead of waiting one memory round trip per chunk.
//
// `ones` (optional, 8 KiB, 16-byte aligned): block 0 also fills it with bf16 ones
// (the A operand of the bias-gradient tile of the GEMM that follows), which
// saves that GEMM's input its own launch.  Launched with programmatic stream
// serialisation it waits for the previous kernel's grid before reading, and lets
// the next kernel start its set-up at once.
template <typename T>
__global__ void __launch_bounds__(256) final_kernel(const float *__restrict__ part, int64_t chunks,
                                                    int64_t cols, T *__restrict__ out, uint4 *__restrict__ ones) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
    if (ones && blockIdx.x == 0) {
        const uint32_t two = 0x3F803F80u;  // two bf16 ones
        for (int i = threadIdx.x; i < 64 * 64 * 2 / 16; i += blockDim.x) ones[i] = make_uint4(two, two, two, two);
    }
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    constexpr int U = 16;
    float s = 0.0f;
    int64_t k = 0;
    for (; k + U <= chunks; k += U) {
        float a[U];
#pragma unroll
        for (int u = 0; u < U; ++u) a[u] = __ldg(part + (k + u) * cols + c);
#pragma unroll
        for (int u = 0; u < U; ++u) s += a[u];
    }
    for (; k < chunks; ++k) s += __ldg(part + k * cols + c);
    store_out<T>(out, c, s);
}

template <typename T>
static cudaError_t launch_t(const T *x, int64_t rows, int64_t cols, float *part, T *out,
                            cudaStream_t st, int *launches) {
    const int64_t chunks = colsum_chunks(rows, cols);
    const int64_t rpc = (rows + chunks - 1) / chunks;
    constexpr int V = Vec<T>::N;
    const bool vec = (cols % V == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0);
    const int64_t per_block = vec ? BX * V : BX;
    const dim3 grid(static_cast<unsigned>((cols + per_block - 1) / per_block), static_cast<unsigned>(chunks));
    if (vec)
        partial_kernel<T, V><<<grid, dim3(BX, BY), 0, st>>>(x, rows, cols, rpc, part);
    else
        partial_kernel<T, 1><<<grid, dim3(BX, BY), 0, st>>>(x, rows, cols, rpc, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    final_kernel<T><<<static_cast<unsigned>((cols + 255) / 256), 256, 0, st>>>(part, chunks, cols, out, nullptr);
    if (launches) *launches += 2;
    return cudaGetLastError();
}

}  // namespace colsum

// Chunks of rows for pass 1: enough blocks to cover the GPU (about 1024 in total),
// at least 16 rows per chunk.  Depends only on the shape, so the partials buffer
// size and the summation order are fixed per shape.
int64_t colsum_chunks(int64_t rows, int64_t cols) {
    const int64_t col_blocks = (cols + 255) / 256;
    int64_t chunks = (1024 + col_blocks - 1) / col_blocks;
    const int64_t max_chunks = (rows + 15) / 16;
    if (chunks > max_chunks) chunks = max_chunks;
    return chunks < 1 ? 1 : chunks;
}

cudaError_t launch_colsum(bool is_bf16, const void *x, int64_t rows, int64_t cols, float *partials,
                          void *out, cudaStream_t st, int *launches) {
    if (cols <= 0) return cudaSuccess;
    if (is_bf16)
        return colsum::launch_t<__nv_bfloat16>(static_cast<const __nv_bfloat16 *>(x), rows, cols, partials,
                                               static_cast<__nv_bfloat16 *>(out), st, launches);
    return colsum::launch_t<float>(static_cast<const float *>(x), rows, cols, partials,
                                   static_cast<float *>(out), st, launches);
}

cudaError_t launch_colsum_final(bool is_bf16, const float *partials, int64_t chunks, int64_t cols, void *out,
                                cudaStream_t st, void *ones) {
    if (cols <= 0) return cudaSuccess;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((cols + 255) / 256), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    const char *pdl_env = std::getenv("TPMLP_PDL");
    if (!(pdl_env && pdl_env[0] == '0')) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    uint4 *o = static_cast<uint4 *>(ones);
    if (is_bf16)
        return cudaLaunchKernelEx(&cfg, colsum::final_kernel<__nv_bfloat16>, partials, chunks, cols,
                                  static_cast<__nv_bfloat16 *>(out), o);
    return cudaLaunchKernelEx(&cfg, colsum::final_kernel<float>, partials, chunks, cols, static_cast<float *>(out), o);
}

// ---------------------------------------------------------------- timeout probe
// One warp allocates 32 TMEM columns (so the release path is exercised too),
// waits on a barrier that never completes for at most wait_ns, records the
// timeout in the status word, frees the TMEM and returns.
__global__ void __launch_bounds__(32) timeout_probe_kernel(uint32_t *status, unsigned long long wait_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_sh;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::fence_mbar_init();
    }
    ptx::tmem_alloc(ptx::smem_u32(&tmem_sh), 32);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
    __syncwarp();
    ptx::tc_fence_after();
    const uint32_t taddr = tmem_sh;
    bool ok = true;
    if (threadIdx.x == 0) ok = ptx::mbar_wait(ptx::smem_u32(&bar), 0, wait_ns, nullptr);
    if (threadIdx.x == 0 && !ok) {
        if (atomicCAS(status, 0u, 4u) == 0u) atomicExch(status + 1, 100u);
    }
    __syncwarp();
    ptx::tmem_dealloc(taddr, 32);
}

cudaError_t launch_timeout_probe(uint32_t *status, uint64_t wait_ns, cudaStream_t st) {
    timeout_probe_kernel<<<1, 32, 0, st>>>(status, wait_ns);
    return cudaGetLastError();
}

}  // namespace tpmlp

// ---------------------------------------------------------------- no-allocation variant
// Column sums whose fp32 partials live in a fixed device array of this library
// instead of a caller workspace, for callers that cannot allocate device memory.
// The array is part of the module image: every GPU that loads the library holds
// it (4 MiB) until the process exits.  Pass 1 writes every partial that pass 2
// reads, so nothing in it has to start at zero; a call simply overwrites what the
// previous call left there.
namespace tpmlp {
namespace noalloc {

constexpr int64_t SCRATCH_FLOATS = int64_t(1) << 20;  // 4 MiB of fp32 partials
static __device__ __align__(256) float g_scratch[SCRATCH_FLOATS];

// Identifier of the current CUDA context, 0 when it cannot be read.  An address
// looked up with cudaGetSymbolAddress belongs to the context it was looked up in;
// after cudaDeviceReset the device's primary context is a new one.
static unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_scratch on the current device, looked up once per device
// and context (again if the context has changed since, or cannot be identified).
// Host code must not use the symbol itself: on the host it is only a stand-in.
static cudaError_t scratch_ptr(float **out) {
    static std::mutex mu;
    static float *ptrs[64] = {};
    static unsigned long long ctx_ids[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    const unsigned long long id = current_context_id();
    if (!ptrs[dev] || id == 0 || id != ctx_ids[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        ptrs[dev] = static_cast<float *>(p);
        ctx_ids[dev] = current_context_id();
    }
    *out = ptrs[dev];
    return cudaSuccess;
}

}  // namespace noalloc
}  // namespace tpmlp

extern "C" tpmlp_status tpmlp_colsum_noalloc(int32_t dtype, const void *x, int64_t rows, int64_t cols,
                                             void *out, void *stream) {
    using namespace tpmlp;
    set_last_error("%s", "");
    if (dtype != TPMLP_F32 && dtype != TPMLP_BF16) {
        set_last_error("tpmlp_colsum_noalloc: unknown dtype %d", dtype);
        return TPMLP_ERR_INVALID_ARG;
    }
    if (rows < 0 || cols <= 0 || !out || (rows > 0 && !x)) {
        set_last_error("tpmlp_colsum_noalloc: invalid sizes or NULL pointer");
        return TPMLP_ERR_INVALID_ARG;
    }
    const int64_t need = colsum_chunks(rows, cols) * cols;
    if (need > noalloc::SCRATCH_FLOATS) {
        set_last_error("tpmlp_colsum_noalloc: %lld columns need %lld fp32 partials, more than the %lld "
                       "of the library's fixed scratch array",
                       static_cast<long long>(cols), static_cast<long long>(need),
                       static_cast<long long>(noalloc::SCRATCH_FLOATS));
        return TPMLP_ERR_UNSUPPORTED;
    }
    float *scratch = nullptr;
    cudaError_t e = noalloc::scratch_ptr(&scratch);
    if (e != cudaSuccess) {
        set_last_error("tpmlp_colsum_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    // rows == 0 needs no special case: pass 1 then sums over no rows and writes zeros.
    int launches = 0;
    e = launch_colsum(dtype == TPMLP_BF16, x, rows, cols, scratch, out, static_cast<cudaStream_t>(stream),
                      &launches);
    add_launches(static_cast<uint64_t>(launches));
    if (e != cudaSuccess) {
        set_last_error("tpmlp_colsum_noalloc: launch failed: %s", cudaGetErrorString(e));
        return TPMLP_ERR_CUDA;
    }
    return TPMLP_OK;
}

