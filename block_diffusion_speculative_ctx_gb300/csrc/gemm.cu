// CUDA-core GEMM C[M, N] (=|+=) A[M, K] . W[N, K]^T with fp32 accumulation.
//
// This is the fp32 path (FP32 FMA, no TF32); bf16 operands go to the tcgen05
// kernel in gemm_tc.cu.  Each output element is one dot product reduced in
// a fixed k order that does not depend on M, so a row's result is the same
// whether it is computed alone or with other rows.
#include "launch.h"

namespace dfl {

namespace {

__device__ __forceinline__ void load8(const float* p, float* o) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16* p, float* o) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = __uint_as_float(w[i] << 16);
        o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <typename T, int BM, int BN, int BK, int TM, int TN>
__global__ void __launch_bounds__((BM / TM) * (BN / TN))
    gemm_cc_kernel(const T* __restrict__ A, int lda, const T* __restrict__ W, float* __restrict__ C, int ldc, int M,
                   int N, int K, int accumulate) {
    pdl_wait();
    pdl_trigger();
    constexpr int NTX = BN / TN, NTY = BM / TM, NT = NTX * NTY;
    __shared__ __align__(16) float As[BK][BM + 4];
    __shared__ __align__(16) float Ws[BK][BN + 4];
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int tid = threadIdx.x, tx = tid % NTX, ty = tid / NTX;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int v = tid; v < BM * BK / 8; v += NT) {
            const int m = v / (BK / 8), kk = (v % (BK / 8)) * 8;
            float t[8];
            if (m0 + m < M && k0 + kk < K) load8(A + (size_t)(m0 + m) * lda + k0 + kk, t);
            else {
#pragma unroll
                for (int e = 0; e < 8; ++e) t[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) As[kk + e][m] = t[e];
        }
        for (int v = tid; v < BN * BK / 8; v += NT) {
            const int n = v / (BK / 8), kk = (v % (BK / 8)) * 8;
            float t[8];
            if (n0 + n < N && k0 + kk < K) load8(W + (size_t)(n0 + n) * K + k0 + kk, t);
            else {
#pragma unroll
                for (int e = 0; e < 8; ++e) t[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) Ws[kk + e][n] = t[e];
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < BK; ++k) {
            float a[TM], w[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = As[k][ty * TM + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) w[j] = Ws[k][tx * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = m0 + ty * TM + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int n = n0 + tx * TN + j;
            if (n >= N) continue;
            float* c = C + (size_t)m * ldc + n;
            *c = accumulate ? (*c + acc[i][j]) : acc[i][j];
        }
    }
}

}  // namespace

template <typename T>
void gemm_cc(const Launch& L, const T* A, int lda, const T* W, int M, int N, int K, float* C, int ldc, bool accumulate) {
    if (M <= 0 || N <= 0) return;
    if (M <= 16) {
        constexpr int BM = 16, BN = 128;
        dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
        launch_k(L, gemm_cc_kernel<T, BM, BN, 32, 2, 4>, grid, dim3(256), 0, 1, A, lda, W, C, ldc, M, N, K,
                 (int)accumulate);
    } else {
        constexpr int BM = 64, BN = 64;
        dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
        launch_k(L, gemm_cc_kernel<T, BM, BN, 32, 4, 4>, grid, dim3(256), 0, 1, A, lda, W, C, ldc, M, N, K,
                 (int)accumulate);
    }
}

template <>
void gemm<float>(const Launch& L, const float* A, int lda, const float* W, int M, int N, int K, float* C, int ldc,
                 bool accumulate) {
    gemm_cc<float>(L, A, lda, W, M, N, K, C, ldc, accumulate);
}

template <>
void gemm<bf16>(const Launch& L, const bf16* A, int lda, const bf16* W, int M, int N, int K, float* C, int ldc,
                bool accumulate) {
    if (M <= 0 || N <= 0) return;
    if (!gemm_tc(L, A, lda, M, W, M, N, K, C, ldc, accumulate)) L.fail();
}

}  // namespace dfl
