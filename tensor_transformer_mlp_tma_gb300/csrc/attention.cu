// Support kernels of the tensor-parallel self-attention block ("Megatron-LM"
// report, section 4.1: heads divided among the t shards).  The projections and
// the per-head products run on the tensor-core GEMMs, which read and write each
// head's Q, K, V, O, dO, dQ, dK, dV in place in the token-major arrays; these
// memory-bound kernels compute the row-wise parts of the attention:
//   - causal softmax of fp16 scores [nb*heads*S][S] (computed in fp32) into bf16 P;
//   - D[z, s] = sum_e dO[token, head cols] * O[token, head cols], the row term of
//     the softmax backward.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace tpmlp {
namespace attn {

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Columns of P that row r of a head (r = row % S) writes: all S, or with
// wtile > 0 only up to the end of the row's wtile-wide tile (the tiles wholly
// above the diagonal, which no later kernel reads, are left as they are).
__device__ __forceinline__ int64_t write_end(int64_t row, int64_t S, int64_t wtile) {
    return wtile > 0 ? min(S, (row % S / wtile + 1) * wtile) : S;
}

// One score row, held in U float4 registers per lane: row r of a head (r = row %
// S) sees columns 0..last; the others are written as exact zeros (up to wend).
// Max-subtracted exponentials (the fast __expf), fp32 sum.  The row is read once,
// four fp16 scores (8 bytes) per lane at a time; only the columns up to the
// diagonal are read.
template <int U>
__device__ __forceinline__ void softmax_row(const uint2 *__restrict__ in, uint2 *__restrict__ out, int64_t last,
                                            int64_t wend, int lane) {
    float4 x[U];
    float mx = -INFINITY;
#pragma unroll
    for (int v = 0; v < U; ++v) {
        const int64_t c = 4 * (lane + 32 * v);
        if (c <= last) {
            const uint2 u = __ldcs(in + lane + 32 * v);  // streamed: read once
            const float2 lo = __half22float2(*reinterpret_cast<const __half2 *>(&u.x));
            const float2 hi = __half22float2(*reinterpret_cast<const __half2 *>(&u.y));
            x[v] = make_float4(lo.x, lo.y, hi.x, hi.y);
            if (c + 1 > last) x[v].y = -INFINITY;
            if (c + 2 > last) x[v].z = -INFINITY;
            if (c + 3 > last) x[v].w = -INFINITY;
        } else {
            x[v] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        mx = fmaxf(mx, fmaxf(fmaxf(x[v].x, x[v].y), fmaxf(x[v].z, x[v].w)));
    }
    mx = warp_max(mx);
    float sum = 0.0f;
#pragma unroll
    for (int v = 0; v < U; ++v) {
        // the fast exponential (its error is far below P's bf16 rounding);
        // exp(-inf) = 0 for the masked columns
        x[v].x = __expf(x[v].x - mx);
        x[v].y = __expf(x[v].y - mx);
        x[v].z = __expf(x[v].z - mx);
        x[v].w = __expf(x[v].w - mx);
        sum += (x[v].x + x[v].y) + (x[v].z + x[v].w);
    }
    sum = warp_sum(sum);
    const float inv = 1.0f / sum;
#pragma unroll
    for (int v = 0; v < U; ++v) {
        const int64_t c = 4 * (lane + 32 * v);
        if (c < wend) {  // wend is a multiple of 4
            __nv_bfloat162 lo = __floats2bfloat162_rn(x[v].x * inv, x[v].y * inv);
            __nv_bfloat162 hi = __floats2bfloat162_rn(x[v].z * inv, x[v].w * inv);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t *>(&lo);
            w.y = *reinterpret_cast<uint32_t *>(&hi);
            out[lane + 32 * v] = w;
        }
    }
    // columns past the U slots, all past the diagonal, up to wend: zeros
    for (int64_t c = 4 * (lane + 32 * U); c < wend; c += 128) out[c / 4] = make_uint2(0u, 0u);
}

// One warp per score row, for rows of up to 128 V columns.  A causal row r needs
// only its first r + 1 columns, so each warp runs the smallest of four unrolled
// bodies (V/4, V/2, 3V/4 or V float4 registers per lane) that covers them: the
// choice is uniform over the warp, and the slots it leaves out would only have
// added exp(-inf) = +0.0 to the sum and -inf to the max, so P is the same, bit
// for bit.  On average it halves the exponentials and the arithmetic of a causal
// softmax.
template <int V>
__global__ void __launch_bounds__(256, V <= 16 ? 3 : 1)  // 24 warps per SM up to 2048 columns
    softmax_reg_kernel(const __half *__restrict__ S_, __nv_bfloat16 *__restrict__ P, int64_t rows, int64_t S,
                       bool causal, int64_t wtile) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int64_t last = causal ? row % S : S - 1;
    const int64_t wend = write_end(row, S, wtile);
    const uint2 *in = reinterpret_cast<const uint2 *>(S_ + row * S);
    uint2 *out = reinterpret_cast<uint2 *>(P + row * S);
    const int64_t need = last / 128 + 1;  // 4-score slots per lane up to the diagonal
    constexpr int V1 = V / 4 > 0 ? V / 4 : 1, V2 = V / 2 > V1 ? V / 2 : V1, V3 = 3 * V / 4 > V2 ? 3 * V / 4 : V2;
    if (need <= V1)
        softmax_row<V1>(in, out, last, wend, lane);
    else if (need <= V2)
        softmax_row<V2>(in, out, last, wend, lane);
    else if (need <= V3)
        softmax_row<V3>(in, out, last, wend, lane);
    else
        softmax_row<V>(in, out, last, wend, lane);
}

// Rows longer than the register version holds: the same arithmetic with three
// passes over the row (max, sum, write).
__global__ void __launch_bounds__(256)
    softmax_kernel(const __half *__restrict__ S_, __nv_bfloat16 *__restrict__ P, int64_t rows, int64_t S,
                   bool causal, int64_t wtile) {
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int64_t last = causal ? row % S : S - 1;
    const __half *in = S_ + row * S;
    __nv_bfloat16 *out = P + row * S;
    float mx = -INFINITY;
    for (int64_t c = lane; c <= last; c += 32) mx = fmaxf(mx, __half2float(in[c]));
    mx = warp_max(mx);
    float sum = 0.0f;
    for (int64_t c = lane; c <= last; c += 32) sum += __expf(__half2float(in[c]) - mx);
    sum = warp_sum(sum);
    const float inv = 1.0f / sum;
    const int64_t wend = write_end(row, S, wtile);
    for (int64_t c = lane; c < wend; c += 32)
        out[c] = __float2bfloat16_rn(c <= last ? __expf(__half2float(in[c]) - mx) * inv : 0.0f);
}

// D[z*S + s] = sum_e dO[r, g*d + e] * O[r, g*d + e] over the token-major [T, h]
// arrays, written in per-head order (z = b*heads + g, r = b*S + s).  d is a
// multiple of 8; a lane takes 8 consecutive elements (one 16-byte load of each
// array) and its dot product is 4 fused pairs in element order.
__device__ __forceinline__ float dot8(const uint4 va, const uint4 vb) {
    const uint32_t ua[4] = {va.x, va.y, va.z, va.w}, ub[4] = {vb.x, vb.y, vb.z, vb.w};
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&ua[i]);
        const __nv_bfloat162 y = *reinterpret_cast<const __nv_bfloat162 *>(&ub[i]);
        s += __low2float(x) * __low2float(y) + __high2float(x) * __high2float(y);
    }
    return s;
}

// One block of ROWDOT_THREADS per token row, for d / 8 a power of two up to 32:
// thread j takes the row's 8-element chunks j, j + ROWDOT_THREADS, ..., two of
// them in flight at once, and the d / 8 lanes that hold one head's chunks add
// them by shuffles (butterfly).  40 registers: 12 blocks (8 KB of loads in
// flight each) stay resident per SM.
constexpr int ROWDOT_THREADS = 128;
constexpr int ROWDOT_UNROLL = 2;
__device__ __forceinline__ void fill_ones_block(uint4 *ones) {
    // the 64 x 64 bf16 ones (8 KiB) that the dWo and dWqkv GEMMs' bias-gradient
    // tiles read, written by block 0 so that they need no launch of their own
    if (ones && blockIdx.x == 0)
        for (int i = threadIdx.x; i < 64 * 64 * 2 / 16; i += blockDim.x)
            ones[i] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
}

__global__ void __launch_bounds__(ROWDOT_THREADS)
    rowdot_row_kernel(const HeadLayout L, const __nv_bfloat16 *__restrict__ a, const __nv_bfloat16 *__restrict__ b,
                      float *__restrict__ D, uint4 *__restrict__ ones) {
    fill_ones_block(ones);
    const int r = static_cast<int>(blockIdx.x), S = static_cast<int>(L.S);
    const int chunks = static_cast<int>(L.h / 8);
    const int G = static_cast<int>(L.d / 8);
    const uint4 *pa = reinterpret_cast<const uint4 *>(a + static_cast<int64_t>(r) * L.h);
    const uint4 *pb = reinterpret_cast<const uint4 *>(b + static_cast<int64_t>(r) * L.h);
    float *out = D + static_cast<int64_t>(r / S) * L.heads * S + r % S;  // + head * S
    for (int j0 = 0; j0 < chunks; j0 += ROWDOT_THREADS * ROWDOT_UNROLL) {
        uint4 va[ROWDOT_UNROLL], vb[ROWDOT_UNROLL];
#pragma unroll
        for (int u = 0; u < ROWDOT_UNROLL; ++u) {
            const int j = j0 + u * ROWDOT_THREADS + static_cast<int>(threadIdx.x);
            va[u] = vb[u] = make_uint4(0u, 0u, 0u, 0u);
            if (j < chunks) {
                va[u] = __ldg(pa + j);
                vb[u] = __ldg(pb + j);
            }
        }
#pragma unroll
        for (int u = 0; u < ROWDOT_UNROLL; ++u) {
            float v = dot8(va[u], vb[u]);
            for (int off = G / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            const int j = j0 + u * ROWDOT_THREADS + static_cast<int>(threadIdx.x);
            if (j < chunks && threadIdx.x % G == 0) out[static_cast<int64_t>(j / G) * S] = v;
        }
    }
}

// One warp per (token r, head g), for any d that is a multiple of 8.
__global__ void __launch_bounds__(256)
    rowdot_kernel(const HeadLayout L, const __nv_bfloat16 *__restrict__ a, const __nv_bfloat16 *__restrict__ b,
                  float *__restrict__ D, uint4 *__restrict__ ones) {
    fill_ones_block(ones);
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= L.nb * L.S * L.heads) return;
    const int64_t r = row / L.heads, g = row % L.heads;
    const int64_t base = r * L.h + g * L.d;
    float s = 0.0f;
    for (int64_t e = static_cast<int64_t>(lane) * 8; e < L.d; e += 256)
        s += dot8(__ldg(reinterpret_cast<const uint4 *>(a + base + e)), __ldg(reinterpret_cast<const uint4 *>(b + base + e)));
    s = warp_sum(s);
    if (lane == 0) D[((r / L.S) * L.heads + g) * L.S + r % L.S] = s;
}

}  // namespace attn

cudaError_t launch_softmax(const void *S_, void *P, int64_t rows, int64_t cols, bool causal, int64_t wtile,
                           cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    const __half *S = static_cast<const __half *>(S_);
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(P);
    // 8-byte row starts (cols a multiple of 4) for the vector loads
    if (cols % 4 != 0 || cols > 128 * 32)
        attn::softmax_kernel<<<grid, 256, 0, st>>>(S, out, rows, cols, causal, wtile);
    else if (cols <= 128 * 4)
        attn::softmax_reg_kernel<4><<<grid, 256, 0, st>>>(S, out, rows, cols, causal, wtile);
    else if (cols <= 128 * 8)
        attn::softmax_reg_kernel<8><<<grid, 256, 0, st>>>(S, out, rows, cols, causal, wtile);
    else if (cols <= 128 * 16)
        attn::softmax_reg_kernel<16><<<grid, 256, 0, st>>>(S, out, rows, cols, causal, wtile);
    else
        attn::softmax_reg_kernel<32><<<grid, 256, 0, st>>>(S, out, rows, cols, causal, wtile);
    return cudaGetLastError();
}

cudaError_t launch_rowdot(const HeadLayout &L, const void *a, const void *b, float *D, cudaStream_t st, void *ones) {
    const int64_t rows = L.nb * L.S * L.heads;
    if (rows <= 0) return cudaSuccess;
    const int64_t G = L.d / 8;
    if (G >= 1 && G <= 32 && (G & (G - 1)) == 0) {
        attn::rowdot_row_kernel<<<static_cast<unsigned>(L.nb * L.S), attn::ROWDOT_THREADS, 0, st>>>(
            L, static_cast<const __nv_bfloat16 *>(a), static_cast<const __nv_bfloat16 *>(b), D,
            static_cast<uint4 *>(ones));
        return cudaGetLastError();
    }
    attn::rowdot_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
        L, static_cast<const __nv_bfloat16 *>(a), static_cast<const __nv_bfloat16 *>(b), D,
        static_cast<uint4 *>(ones));
    return cudaGetLastError();
}

}  // namespace tpmlp
