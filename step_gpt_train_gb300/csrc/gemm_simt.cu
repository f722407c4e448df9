// fp32 matmul for the exact-parity mode (true fp32 FMA, no TF32), and the
// matmul entry that routes bf16 to the tensor-core kernel.
#include "common.cuh"
#include "launch.h"

size_t matmul_tc_scratch(int M, int N, int K, int d_fp32, int accumulate);
int launch_matmul_tc(void* D, int d_fp32, const void* A, int a_mn, const void* B, int b_mn, const void* bias, int M,
                     int N, int K, void* scratch, int* status, cudaStream_t s, int accumulate);

// 64 x 64 output tile, 16-deep k slices through shared memory, 256 threads,
// 4 x 4 outputs per thread. A(m,k) = A[m*K+k] or A[k*M+m]; B likewise. With
// accumulate the result is added to D.
template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(256) gemm_f32_kernel(float* __restrict__ D, const float* __restrict__ A,
                                                       const float* __restrict__ B, const float* __restrict__ bias,
                                                       int M, int N, int K, int accumulate) {
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int idx = tid + e * 256;
            int mm, kk;
            if (A_MN) { kk = idx / 64; mm = idx % 64; }
            else { mm = idx / 16; kk = idx % 16; }
            const int gm = m0 + mm, gk = k0 + kk;
            float v = 0.f;
            if (gm < M && gk < K) v = A_MN ? A[(int64_t)gk * M + gm] : A[(int64_t)gm * K + gk];
            As[kk][mm] = v;
            int nn;
            if (B_MN) { kk = idx / 64; nn = idx % 64; }
            else { nn = idx / 16; kk = idx % 16; }
            const int gn = n0 + nn, gk2 = k0 + kk;
            float w = 0.f;
            if (gn < N && gk2 < K) w = B_MN ? B[(int64_t)gk2 * N + gn] : B[(int64_t)gn * K + gk2];
            Bs[kk][nn] = w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; kk++) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; i++) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int n = n0 + tx * 4 + j;
            if (n < N) {
                const float v = acc[i][j] + (bias ? bias[n] : 0.f);
                D[(int64_t)m * N + n] = accumulate ? D[(int64_t)m * N + n] + v : v;
            }
        }
    }
}

size_t matmul_scratch(int dtype, int M, int N, int K, int d_fp32, int accumulate) {
    if (dtype == GPT2_MODE_BF16) return matmul_tc_scratch(M, N, K, d_fp32, accumulate);
    return 0;
}

int launch_matmul(int dtype, void* D, int d_fp32, const void* A, int a_mn, const void* B, int b_mn, const void* bias,
                  int M, int N, int K, void* scratch, int* status, cudaStream_t s, int accumulate) {
    if (M == 0 || N == 0) return 0;
    if (dtype == GPT2_MODE_BF16)
        return launch_matmul_tc(D, d_fp32, A, a_mn, B, b_mn, bias, M, N, K, scratch, status, s, accumulate);
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    float* d = (float*)D;
    const float* a = (const float*)A;
    const float* b = (const float*)B;
    const float* bb = (const float*)bias;
    if (!a_mn && !b_mn) gemm_f32_kernel<false, false><<<grid, 256, 0, s>>>(d, a, b, bb, M, N, K, accumulate);
    else if (!a_mn && b_mn) gemm_f32_kernel<false, true><<<grid, 256, 0, s>>>(d, a, b, bb, M, N, K, accumulate);
    else if (a_mn && !b_mn) gemm_f32_kernel<true, false><<<grid, 256, 0, s>>>(d, a, b, bb, M, N, K, accumulate);
    else gemm_f32_kernel<true, true><<<grid, 256, 0, s>>>(d, a, b, bb, M, N, K, accumulate);
    return 1;
}
