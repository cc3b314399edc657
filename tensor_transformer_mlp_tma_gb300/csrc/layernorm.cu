// LayerNorm in front of the MLP: the sequence-parallel block of the
// "Megatron-LM" report (section 4.3), where each token shard normalises its own
// rows before the tensor-parallel MLP.  Rows are independent, so on one GPU the
// token shards are simply row ranges of one launch.  Memory bound: one block per
// row with the row held in registers (one read of x, dy), 16-byte vector loads,
// fp32 statistics, fixed-order reductions; one warp per row (three passes over
// the row) when the row is too long for the registers or not 16-byte aligned.
//
//   forward : mu = mean(x), var = mean((x - mu)^2), rstd = 1/sqrt(var + eps),
//             y = (x - mu) * rstd * gamma + beta          (mu, rstd kept)
//   backward: xhat = (x - mu) rstd, g = dy * gamma,
//             dx = rstd * (g - mean(g) - xhat * mean(g * xhat))
//   params  : dgamma = sum_rows dy * xhat, dbeta = sum_rows dy (two-pass, in order)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace tpmlp {
namespace ln {

constexpr int ROWS_PER_BLOCK = 8;  // one warp per row

template <typename T>
struct V;
template <>
struct V<float> {
    static constexpr int N = 4;
};
template <>
struct V<__nv_bfloat16> {
    static constexpr int N = 8;
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float v, float &o) { o = v; }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16 &o) { o = __float2bfloat16_rn(v); }

// Loads VEC consecutive elements (vector load when VEC > 1).
template <typename T, int VEC>
__device__ __forceinline__ void ldv(const T *p, float *v) {
    if constexpr (VEC == 1) {
        v[0] = to_f(p[0]);
    } else if constexpr (sizeof(T) == 4) {
        const float4 w = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = w.x, v[1] = w.y, v[2] = w.z, v[3] = w.w;
    } else {
        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u[i]);
            v[2 * i] = __low2float(b);
            v[2 * i + 1] = __high2float(b);
        }
    }
}

template <typename T, int VEC>
__device__ __forceinline__ void stv(T *p, const float *v) {
    if constexpr (VEC == 1) {
        from_f(v[0], p[0]);
    } else if constexpr (sizeof(T) == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            u[i] = *reinterpret_cast<uint32_t *>(&b);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(u[0], u[1], u[2], u[3]);
    }
}

// Fixed butterfly: every lane ends with the same total, summed in the same tree.
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---- one block per row: each thread holds up to MAXC 16-byte chunks of the row
constexpr int ROW_THREADS = 256;

// 16 bytes as VEC floats (8 bf16 or 4 fp32).
template <typename T>
__device__ __forceinline__ void unpack(const uint4 w, float *v) {
    if constexpr (sizeof(T) == 4) {
        v[0] = __uint_as_float(w.x), v[1] = __uint_as_float(w.y), v[2] = __uint_as_float(w.z),
        v[3] = __uint_as_float(w.w);
    } else {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u[i]);
            v[2 * i] = __low2float(b);
            v[2 * i + 1] = __high2float(b);
        }
    }
}

// Sum over the block, every thread gets the same total: warp butterflies, then
// the warps' sums added in warp order.
__device__ __forceinline__ float2 block_sum2(float2 x, float2 *red) {
    x.x = warp_sum(x.x);
    x.y = warp_sum(x.y);
    __syncthreads();  // a previous call's readers are done with red
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    float2 t = red[0];
#pragma unroll
    for (int w = 1; w < ROW_THREADS / 32; ++w) t.x += red[w].x, t.y += red[w].y;
    return t;
}

template <typename T, int MAXC>
__global__ void __launch_bounds__(ROW_THREADS)
    forward_row_kernel(const T *__restrict__ x, const T *__restrict__ gamma, const T *__restrict__ beta, float eps,
                       int64_t h, T *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd) {
    constexpr int VEC = V<T>::N;
    __shared__ float2 red[ROW_THREADS / 32];
    const int64_t r = blockIdx.x;
    const int nch = static_cast<int>(h / VEC);
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + r * h);
    uint4 xw[MAXC];
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        const int j = static_cast<int>(threadIdx.x) + c * ROW_THREADS;
        xw[c] = j < nch ? __ldg(xr + j) : make_uint4(0u, 0u, 0u, 0u);  // zeros add nothing to the sum
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        float v[VEC];
        unpack<T>(xw[c], v);
#pragma unroll
        for (int i = 0; i < VEC; ++i) s += v[i];
    }
    const float mu = block_sum2(make_float2(s, 0.0f), red).x / static_cast<float>(h);
    float q = 0.0f;
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        if (static_cast<int>(threadIdx.x) + c * ROW_THREADS >= nch) break;
        float v[VEC];
        unpack<T>(xw[c], v);
#pragma unroll
        for (int i = 0; i < VEC; ++i) q += (v[i] - mu) * (v[i] - mu);
    }
    const float var = block_sum2(make_float2(q, 0.0f), red).x / static_cast<float>(h);
    const float rs = 1.0f / sqrtf(var + eps);
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        const int j = static_cast<int>(threadIdx.x) + c * ROW_THREADS;
        if (j >= nch) break;
        float v[VEC], g[VEC], b[VEC], o[VEC];
        unpack<T>(xw[c], v);
        ldv<T, VEC>(gamma + static_cast<int64_t>(j) * VEC, g);
        ldv<T, VEC>(beta + static_cast<int64_t>(j) * VEC, b);
#pragma unroll
        for (int i = 0; i < VEC; ++i) o[i] = (v[i] - mu) * rs * g[i] + b[i];
        stv<T, VEC>(y + r * h + static_cast<int64_t>(j) * VEC, o);
    }
    if (threadIdx.x == 0) {
        mean[r] = mu;
        rstd[r] = rs;
    }
}

template <typename T, int MAXC>
__global__ void __launch_bounds__(ROW_THREADS)
    backward_row_kernel(const T *__restrict__ dy, const T *__restrict__ x, const T *__restrict__ gamma,
                        const float *__restrict__ mean, const float *__restrict__ rstd, int64_t h,
                        T *__restrict__ dx) {
    constexpr int VEC = V<T>::N;
    __shared__ float2 red[ROW_THREADS / 32];
    const int64_t r = blockIdx.x;
    const int nch = static_cast<int>(h / VEC);
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + r * h);
    const uint4 *dyr = reinterpret_cast<const uint4 *>(dy + r * h);
    // gamma (one row for all rows, L2-resident) is read in both passes
    const uint4 *gr = reinterpret_cast<const uint4 *>(gamma);
    uint4 xw[MAXC], dw[MAXC];
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        const int j = static_cast<int>(threadIdx.x) + c * ROW_THREADS;
        xw[c] = dw[c] = make_uint4(0u, 0u, 0u, 0u);  // zeros add nothing to the sums
        if (j < nch) {
            xw[c] = __ldg(xr + j);
            dw[c] = __ldg(dyr + j);
        }
    }
    const float mu = mean[r], rs = rstd[r];
    float sg = 0.0f, sgx = 0.0f;
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        const int j = static_cast<int>(threadIdx.x) + c * ROW_THREADS;
        if (j >= nch) break;
        float v[VEC], d[VEC], g[VEC];
        unpack<T>(xw[c], v);
        unpack<T>(dw[c], d);
        unpack<T>(__ldg(gr + j), g);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const float gg = d[i] * g[i];
            sg += gg;
            sgx += gg * (v[i] - mu) * rs;
        }
    }
    const float2 t = block_sum2(make_float2(sg, sgx), red);
    const float mg = t.x / static_cast<float>(h), mgx = t.y / static_cast<float>(h);
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
        const int j = static_cast<int>(threadIdx.x) + c * ROW_THREADS;
        if (j >= nch) break;
        float v[VEC], d[VEC], g[VEC], o[VEC];
        unpack<T>(xw[c], v);
        unpack<T>(dw[c], d);
        unpack<T>(__ldg(gr + j), g);
#pragma unroll
        for (int i = 0; i < VEC; ++i) o[i] = rs * (d[i] * g[i] - mg - (v[i] - mu) * rs * mgx);
        stv<T, VEC>(dx + r * h + static_cast<int64_t>(j) * VEC, o);
    }
}

// Chunks of 16 bytes per thread for a row of h elements: the smallest of 1, 2,
// 4, 8 that covers the row, or 0 when the row does not fit (warp kernels).
template <typename T>
static int row_chunks(int64_t h) {
    const int64_t nch = h / V<T>::N;
    for (int c = 1; c <= 8; c *= 2)
        if (nch <= static_cast<int64_t>(c) * ROW_THREADS) return c;
    return 0;
}

// ---- one warp per row (rows too long for the block kernels, or unaligned)
template <typename T, int VEC>
__global__ void __launch_bounds__(32 * ROWS_PER_BLOCK)
    forward_kernel(const T *__restrict__ x, const T *__restrict__ gamma, const T *__restrict__ beta, float eps,
                   int64_t rows, int64_t h, T *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * ROWS_PER_BLOCK + (threadIdx.x >> 5);
    if (r >= rows) return;
    const T *xr = x + r * h;
    float s = 0.0f;
    for (int64_t j = static_cast<int64_t>(lane) * VEC; j < h; j += 32 * VEC) {
        float v[VEC];
        ldv<T, VEC>(xr + j, v);
#pragma unroll
        for (int i = 0; i < VEC; ++i) s += v[i];
    }
    const float mu = warp_sum(s) / static_cast<float>(h);
    float q = 0.0f;
    for (int64_t j = static_cast<int64_t>(lane) * VEC; j < h; j += 32 * VEC) {
        float v[VEC];
        ldv<T, VEC>(xr + j, v);
#pragma unroll
        for (int i = 0; i < VEC; ++i) q += (v[i] - mu) * (v[i] - mu);
    }
    const float var = warp_sum(q) / static_cast<float>(h);
    const float rs = 1.0f / sqrtf(var + eps);
    T *yr = y + r * h;
    for (int64_t j = static_cast<int64_t>(lane) * VEC; j < h; j += 32 * VEC) {
        float v[VEC], g[VEC], b[VEC], o[VEC];
        ldv<T, VEC>(xr + j, v);
        ldv<T, VEC>(gamma + j, g);
        ldv<T, VEC>(beta + j, b);
#pragma unroll
        for (int i = 0; i < VEC; ++i) o[i] = (v[i] - mu) * rs * g[i] + b[i];
        stv<T, VEC>(yr + j, o);
    }
    if (lane == 0) {
        mean[r] = mu;
        rstd[r] = rs;
    }
}

template <typename T, int VEC>
__global__ void __launch_bounds__(32 * ROWS_PER_BLOCK)
    backward_kernel(const T *__restrict__ dy, const T *__restrict__ x, const T *__restrict__ gamma,
                    const float *__restrict__ mean, const float *__restrict__ rstd, int64_t rows, int64_t h,
                    T *__restrict__ dx) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * ROWS_PER_BLOCK + (threadIdx.x >> 5);
    if (r >= rows) return;
    const T *xr = x + r * h;
    const T *dyr = dy + r * h;
    const float mu = mean[r], rs = rstd[r];
    float sg = 0.0f, sgx = 0.0f;
    for (int64_t j = static_cast<int64_t>(lane) * VEC; j < h; j += 32 * VEC) {
        float v[VEC], d[VEC], g[VEC];
        ldv<T, VEC>(xr + j, v);
        ldv<T, VEC>(dyr + j, d);
        ldv<T, VEC>(gamma + j, g);
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const float gg = d[i] * g[i];
            sg += gg;
            sgx += gg * (v[i] - mu) * rs;
        }
    }
    const float mg = warp_sum(sg) / static_cast<float>(h);
    const float mgx = warp_sum(sgx) / static_cast<float>(h);
    T *dxr = dx + r * h;
    for (int64_t j = static_cast<int64_t>(lane) * VEC; j < h; j += 32 * VEC) {
        float v[VEC], d[VEC], g[VEC], o[VEC];
        ldv<T, VEC>(xr + j, v);
        ldv<T, VEC>(dyr + j, d);
        ldv<T, VEC>(gamma + j, g);
#pragma unroll
        for (int i = 0; i < VEC; ++i) o[i] = rs * (d[i] * g[i] - mg - (v[i] - mu) * rs * mgx);
        stv<T, VEC>(dxr + j, o);
    }
}

// Pass 1 of dgamma and dbeta: a (32 x 8)-thread block owns 32*VEC columns and a
// chunk of rows; partial sums of dy * xhat and dy go to [chunks, h] arrays.
template <typename T, int VEC>
__global__ void __launch_bounds__(256)
    param_partial_kernel(const T *__restrict__ dy, const T *__restrict__ x, const float *__restrict__ mean,
                         const float *__restrict__ rstd, int64_t rows, int64_t h, int64_t rows_per_chunk,
                         float *__restrict__ pg, float *__restrict__ pb) {
    __shared__ float rg[8][32 * VEC];
    __shared__ float rb[8][32 * VEC];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int64_t col = (static_cast<int64_t>(blockIdx.x) * 32 + tx) * VEC;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_chunk;
    const int64_t r1 = min(rows, r0 + rows_per_chunk);
    float ag[VEC], ab[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) ag[i] = ab[i] = 0.0f;
    if (col < h) {
#pragma unroll 4
        for (int64_t r = r0 + ty; r < r1; r += 8) {
            float v[VEC], d[VEC];
            ldv<T, VEC>(x + r * h + col, v);
            ldv<T, VEC>(dy + r * h + col, d);
            const float mu = mean[r], rs = rstd[r];
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                ag[i] += d[i] * (v[i] - mu) * rs;
                ab[i] += d[i];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        rg[ty][tx * VEC + i] = ag[i];
        rb[ty][tx * VEC + i] = ab[i];
    }
    __syncthreads();
    for (int c = ty * 32 + tx; c < 32 * VEC; c += 256) {
        float sg = rg[0][c], sb = rb[0][c];
#pragma unroll
        for (int y = 1; y < 8; ++y) {
            sg += rg[y][c];
            sb += rb[y][c];
        }
        const int64_t gc = static_cast<int64_t>(blockIdx.x) * 32 * VEC + c;
        if (gc < h) {
            pg[static_cast<int64_t>(blockIdx.y) * h + gc] = sg;
            pb[static_cast<int64_t>(blockIdx.y) * h + gc] = sb;
        }
    }
}

template <typename T>
static bool vec_ok(const void *p, int64_t h) {
    return h % V<T>::N == 0 && reinterpret_cast<uintptr_t>(p) % 16 == 0;
}

template <typename T>
static cudaError_t fwd_t(const LnArgs &a, cudaStream_t st) {
    const dim3 grid(static_cast<unsigned>((a.rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK));
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *b = static_cast<const T *>(a.beta);
    T *y = static_cast<T *>(a.y);
    const bool v = vec_ok<T>(a.x, a.h) && vec_ok<T>(a.gamma, a.h) && vec_ok<T>(a.beta, a.h) && vec_ok<T>(a.y, a.h);
    const int rc = v ? row_chunks<T>(a.h) : 0;
    const dim3 rgrid(static_cast<unsigned>(a.rows));
    if (rc == 1)
        forward_row_kernel<T, 1><<<rgrid, ROW_THREADS, 0, st>>>(x, g, b, a.eps, a.h, y, a.mean, a.rstd);
    else if (rc == 2)
        forward_row_kernel<T, 2><<<rgrid, ROW_THREADS, 0, st>>>(x, g, b, a.eps, a.h, y, a.mean, a.rstd);
    else if (rc == 4)
        forward_row_kernel<T, 4><<<rgrid, ROW_THREADS, 0, st>>>(x, g, b, a.eps, a.h, y, a.mean, a.rstd);
    else if (rc == 8)
        forward_row_kernel<T, 8><<<rgrid, ROW_THREADS, 0, st>>>(x, g, b, a.eps, a.h, y, a.mean, a.rstd);
    else if (v)
        forward_kernel<T, V<T>::N><<<grid, 32 * ROWS_PER_BLOCK, 0, st>>>(x, g, b, a.eps, a.rows, a.h, y, a.mean,
                                                                          a.rstd);
    else
        forward_kernel<T, 1><<<grid, 32 * ROWS_PER_BLOCK, 0, st>>>(x, g, b, a.eps, a.rows, a.h, y, a.mean, a.rstd);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t bwd_t(const LnArgs &a, cudaStream_t st, int *launches) {
    const T *dy = static_cast<const T *>(a.dy);
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    T *dx = static_cast<T *>(a.dx);
    const bool v = vec_ok<T>(a.dy, a.h) && vec_ok<T>(a.x, a.h) && vec_ok<T>(a.gamma, a.h) && vec_ok<T>(a.dx, a.h);
    if (a.rows > 0) {
        const dim3 grid(static_cast<unsigned>((a.rows + ROWS_PER_BLOCK - 1) / ROWS_PER_BLOCK));
        const int rc = v ? row_chunks<T>(a.h) : 0;
        const dim3 rgrid(static_cast<unsigned>(a.rows));
        if (rc == 1)
            backward_row_kernel<T, 1><<<rgrid, ROW_THREADS, 0, st>>>(dy, x, g, a.mean, a.rstd, a.h, dx);
        else if (rc == 2)
            backward_row_kernel<T, 2><<<rgrid, ROW_THREADS, 0, st>>>(dy, x, g, a.mean, a.rstd, a.h, dx);
        else if (rc == 4)
            backward_row_kernel<T, 4><<<rgrid, ROW_THREADS, 0, st>>>(dy, x, g, a.mean, a.rstd, a.h, dx);
        else if (rc == 8)
            backward_row_kernel<T, 8><<<rgrid, ROW_THREADS, 0, st>>>(dy, x, g, a.mean, a.rstd, a.h, dx);
        else if (v)
            backward_kernel<T, V<T>::N><<<grid, 32 * ROWS_PER_BLOCK, 0, st>>>(dy, x, g, a.mean, a.rstd, a.rows, a.h,
                                                                               dx);
        else
            backward_kernel<T, 1><<<grid, 32 * ROWS_PER_BLOCK, 0, st>>>(dy, x, g, a.mean, a.rstd, a.rows, a.h, dx);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (launches) *launches += 1;
    }
    // dgamma, dbeta: pass 1 into [chunks, h] partials, then in-order sums.
    const int64_t chunks = colsum_chunks(a.rows, a.h);
    const int64_t rpc = (a.rows + chunks - 1) / chunks;
    float *pg = a.partials, *pb = a.partials + chunks * a.h;
    const bool vp = vec_ok<T>(a.dy, a.h) && vec_ok<T>(a.x, a.h);
    const int64_t per_block = vp ? 32 * V<T>::N : 32;
    const dim3 grid(static_cast<unsigned>((a.h + per_block - 1) / per_block), static_cast<unsigned>(chunks));
    if (vp)
        param_partial_kernel<T, V<T>::N><<<grid, dim3(32, 8), 0, st>>>(dy, x, a.mean, a.rstd, a.rows, a.h, rpc, pg, pb);
    else
        param_partial_kernel<T, 1><<<grid, dim3(32, 8), 0, st>>>(dy, x, a.mean, a.rstd, a.rows, a.h, rpc, pg, pb);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const bool bf = sizeof(T) == 2;
    e = launch_colsum_final(bf, pg, chunks, a.h, a.dgamma, st);
    if (e == cudaSuccess) e = launch_colsum_final(bf, pb, chunks, a.h, a.dbeta, st);
    if (launches) *launches += 3;
    return e;
}

}  // namespace ln

int64_t ln_partial_floats(int64_t rows, int64_t h) { return 2 * colsum_chunks(rows, h) * h; }

cudaError_t launch_ln_forward(bool is_bf16, const LnArgs &a, cudaStream_t st) {
    if (a.rows <= 0) return cudaSuccess;
    return is_bf16 ? ln::fwd_t<__nv_bfloat16>(a, st) : ln::fwd_t<float>(a, st);
}

cudaError_t launch_ln_backward(bool is_bf16, const LnArgs &a, cudaStream_t st, int *launches) {
    return is_bf16 ? ln::bwd_t<__nv_bfloat16>(a, st, launches) : ln::bwd_t<float>(a, st, launches);
}

}  // namespace tpmlp
