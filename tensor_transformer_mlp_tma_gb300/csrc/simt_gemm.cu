// FFMA GEMMs (no tensor cores) for the fp32 workloads and as an independent GPU
// cross-check of the tensor-core kernels on bf16 inputs.  Same six products and
// the same fused epilogues as the tensor-core path, with exact GeLU (tanhf):
// fp32 accumulation, one FMA per k in ascending order, shard partials summed in
// ascending shard order.  64x64 output tile per 256-thread block, 4x4 per thread.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace tpmlp {
namespace simt {

constexpr int TM = 64, TN = 64, TK = 16;

template <typename T>
__device__ __forceinline__ float ld(const T *p, int64_t i);
template <>
__device__ __forceinline__ float ld<float>(const float *p, int64_t i) {
    return p[i];
}
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16 *p, int64_t i) {
    return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st(T *p, int64_t i, float v);
template <>
__device__ __forceinline__ void st<float>(float *p, int64_t i, float v) {
    p[i] = v;
}
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16 *p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

// v rounded to T and back (round to nearest even), i.e. the value stored as T.
template <typename T>
__device__ __forceinline__ float rounded(float v);
template <>
__device__ __forceinline__ float rounded<float>(float v) {
    return v;
}
template <>
__device__ __forceinline__ float rounded<__nv_bfloat16>(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ float gelu_exact_tanh(float x) {
    const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
    return 0.5f * x * (1.0f + tanhf(u));
}

__device__ __forceinline__ float gelu_prime_exact_tanh(float x) {
    const float u = 0.7978845608028654f * (x + 0.044715f * x * x * x);
    const float th = tanhf(u);
    const float du = 0.7978845608028654f * (1.0f + 3.0f * 0.044715f * x * x);
    return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * du;
}

struct Params {
    const void *a;
    const void *b;
    int64_t M, N, K, kshard;
    int nshards;
    // element (m,k) of op(A) is a[m*sam + k*sak]; element (k,n) of op(B) is b[k*sbk + n*sbn]
    int64_t sam, sak, sbk, sbn;
    void *out0;
    void *out1;
    const void *aux;
    const void *bias;
};

template <typename T, int EPI>
__global__ void __launch_bounds__(256) gemm_kernel(const Params p) {
    __shared__ float As[TK][TM + 4];
    __shared__ float Bs[TK][TN + 4];
    const T *A = static_cast<const T *>(p.a);
    const T *B = static_cast<const T *>(p.b);
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * TN;
    const bool a_kcontig = p.sak == 1;
    const bool b_ncontig = p.sbn == 1;

    float sum[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sum[i][j] = 0.0f;

    for (int s = 0; s < p.nshards; ++s) {
        const int64_t kbeg = s * p.kshard;
        const int64_t kend = min(kbeg + p.kshard, p.K);
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
        for (int64_t k0 = kbeg; k0 < kend; k0 += TK) {
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
                const int e = tid + 256 * e4;
                int mm, kk;
                if (a_kcontig) {
                    kk = e % TK;
                    mm = e / TK;
                } else {
                    mm = e % TM;
                    kk = e / TM;
                }
                const int64_t gm = m0 + mm, gk = k0 + kk;
                As[kk][mm] = (gm < p.M && gk < kend) ? ld<T>(A, gm * p.sam + gk * p.sak) : 0.0f;
                int nn, kb;
                if (b_ncontig) {
                    nn = e % TN;
                    kb = e / TN;
                } else {
                    kb = e % TK;
                    nn = e / TK;
                }
                const int64_t gn = n0 + nn, gkb = k0 + kb;
                Bs[kb][nn] = (gn < p.N && gkb < kend) ? ld<T>(B, gkb * p.sbk + gn * p.sbn) : 0.0f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < TK; ++kk) {
                float av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = As[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) sum[i][j] = (s == 0) ? acc[i][j] : sum[i][j] + acc[i][j];
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty + 16 * i;
        if (m >= p.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx + 16 * j;
            if (n >= p.N) continue;
            const int64_t o = m * p.N + n;
            float v = sum[i][j];
            if constexpr (EPI == EPI_BIAS_GELU) {
                // Y is GeLU of H as stored (rounded to T), the value the
                // backward's recomputation rebuilds from the saved H
                v += ld<T>(static_cast<const T *>(p.bias), n);
                const float h = rounded<T>(v);
                if (p.out0) st<T>(static_cast<T *>(p.out0), o, h);
                if (p.out1) st<T>(static_cast<T *>(p.out1), o, gelu_exact_tanh(h));
            } else if constexpr (EPI == EPI_FOLD_BIAS) {
                st<T>(static_cast<T *>(p.out0), o, v + ld<T>(static_cast<const T *>(p.bias), n));
            } else if constexpr (EPI == EPI_DGELU) {
                const float hv = ld<T>(static_cast<const T *>(p.aux), o);
                st<T>(static_cast<T *>(p.out0), o, v * gelu_prime_exact_tanh(hv));
                if (p.out1) st<T>(static_cast<T *>(p.out1), o, gelu_exact_tanh(hv));  // Y rebuilt from H
            } else {
                st<T>(static_cast<T *>(p.out0), o, v);
            }
        }
    }
}

template <typename T>
static cudaError_t launch_t(Epi epi, const Params &p, cudaStream_t st) {
    const dim3 grid(static_cast<unsigned>((p.N + TN - 1) / TN), static_cast<unsigned>((p.M + TM - 1) / TM));
    switch (epi) {
        case EPI_BIAS_GELU: gemm_kernel<T, EPI_BIAS_GELU><<<grid, 256, 0, st>>>(p); break;
        case EPI_FOLD_BIAS: gemm_kernel<T, EPI_FOLD_BIAS><<<grid, 256, 0, st>>>(p); break;
        case EPI_DGELU: gemm_kernel<T, EPI_DGELU><<<grid, 256, 0, st>>>(p); break;
        case EPI_STORE: gemm_kernel<T, EPI_STORE><<<grid, 256, 0, st>>>(p); break;
        case EPI_FOLD: gemm_kernel<T, EPI_FOLD><<<grid, 256, 0, st>>>(p); break;
        default: return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace simt

cudaError_t launch_simt_gemm(Epi epi, bool is_bf16, const GemmArgs &g, cudaStream_t st) {
    if (g.M <= 0 || g.N <= 0) return cudaSuccess;
    if (g.M > 65535LL * simt::TM) return cudaErrorInvalidValue;
    simt::Params p;
    p.a = g.a;
    p.b = g.b;
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.kshard = g.kshard;
    p.nshards = g.nshards;
    // K-major A is [M,K]; MN-major A is [K,M].  K-major B is [N,K]; MN-major B is [K,N].
    if (g.a_mn) {
        p.sam = 1;
        p.sak = g.M;
    } else {
        p.sam = g.K;
        p.sak = 1;
    }
    if (g.b_mn) {
        p.sbk = g.N;
        p.sbn = 1;
    } else {
        p.sbk = 1;
        p.sbn = g.K;
    }
    p.out0 = g.out0;
    p.out1 = g.out1;
    p.aux = g.aux;
    p.bias = g.bias;
    return is_bf16 ? simt::launch_t<__nv_bfloat16>(epi, p, st) : simt::launch_t<float>(epi, p, st);
}

}  // namespace tpmlp
