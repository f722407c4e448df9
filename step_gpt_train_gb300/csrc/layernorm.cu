// LayerNorm forward and backward: one warp per row, the row held in
// registers (16-byte vector loads), statistics by warp shuffles.
#include "common.cuh"
#include "launch.h"

#define LN_EPS 1e-5f
#define LN_FWD_WARPS 8
#define LN_BWD_WARPS 8
#define LN_BWD_MAX_BLOCKS 608  // four resident blocks on each of 152 SMs

// y = (x - mean) * rstd * gamma + beta, biased variance, eps 1e-5.
// VPL = 8-element vectors per lane (C <= 256 * VPL).
template <typename T, int VPL>
__global__ void __launch_bounds__(LN_FWD_WARPS * 32) ln_fwd_kernel(T* __restrict__ y, float* __restrict__ mean,
                                                                   float* __restrict__ rstd, const T* __restrict__ x,
                                                                   const T* __restrict__ gamma,
                                                                   const T* __restrict__ beta, int N, int C) {
    const int row = blockIdx.x * LN_FWD_WARPS + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= N) return;
    const int cv = C / 8;
    const T* xr = x + (int64_t)row * C;
    float v[VPL][8];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int idx = lane + 32 * i;
        if (idx < cv) {
            load8_stream(xr + idx * 8, v[i]);
#pragma unroll
            for (int j = 0; j < 8; j++) s += v[i][j];
        }
    }
    const float mu = warp_sum(s) / (float)C;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        if (lane + 32 * i < cv) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float d = v[i][j] - mu;
                ss += d * d;
            }
        }
    }
    const float rs = 1.0f / sqrtf(warp_sum(ss) / (float)C + LN_EPS);
    T* yr = y + (int64_t)row * C;
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int idx = lane + 32 * i;
        if (idx < cv) {
            float g[8], b[8], o[8];
            load8(gamma + idx * 8, g);
            load8(beta + idx * 8, b);
#pragma unroll
            for (int j = 0; j < 8; j++) o[j] = (v[i][j] - mu) * rs * g[j] + b[j];
            store8(yr + idx * 8, o);
        }
    }
    if (lane == 0) {
        mean[row] = mu;
        rstd[row] = rs;
    }
}

// dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat)), dxhat = dy gamma.
// Warp per row, rows strided over a fixed grid; the next row's x and dy are
// loaded (raw) before the current row is computed. Each warp accumulates
// dy*xhat and dy for its lane's columns in its own shared-memory rows (no two
// threads touch the same word; column idx*8+j at word j*(C/8)+idx, so a
// warp's accesses hit 32 distinct banks). The block then sums its warps in
// order into partial[block][0..2C); a column reduce finishes dgamma, dbeta.
template <typename T, int VPL>
__global__ void __launch_bounds__(LN_BWD_WARPS * 32, VPL <= 3 ? 2 : 1) ln_bwd_kernel(T* __restrict__ dx, float* __restrict__ partial,
                                                                   const T* __restrict__ dy, const T* __restrict__ x,
                                                                   const T* __restrict__ gamma,
                                                                   const float* __restrict__ mean,
                                                                   const float* __restrict__ rstd, int N, int C) {
    extern __shared__ float sh[];  // [LN_BWD_WARPS][2][C]
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cv = C / 8;
    float* acc_g = sh + (size_t)w * 2 * C;
    float* acc_b = acc_g + C;
    for (int c = lane; c < C; c += 32) {
        acc_g[c] = 0.f;
        acc_b[c] = 0.f;
    }
    __syncwarp();
    const int stride = gridDim.x * LN_BWD_WARPS;
    int row = blockIdx.x * LN_BWD_WARPS + w;
    Raw8<T> rx[VPL], rd[VPL];
    if (row < N) {
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                raw_load(rx[i], x + (int64_t)row * C + idx * 8);
                raw_load(rd[i], dy + (int64_t)row * C + idx * 8);
            }
        }
    }
    while (row < N) {
        const int next = row + stride;
        Raw8<T> nx[VPL], nd[VPL];
        if (next < N) {
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int idx = lane + 32 * i;
                if (idx < cv) {
                    raw_load(nx[i], x + (int64_t)next * C + idx * 8);
                    raw_load(nd[i], dy + (int64_t)next * C + idx * 8);
                }
            }
        }
        const float mu = mean[row], rs = rstd[row];
        float xh[VPL][8], dh[VPL][8];
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                float g[8];
                raw_unpack(rx[i], xh[i]);
                raw_unpack(rd[i], dh[i]);
                load8(gamma + idx * 8, g);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    xh[i][j] = (xh[i][j] - mu) * rs;
                    const int a = j * cv + idx;
                    acc_g[a] += dh[i][j] * xh[i][j];
                    acc_b[a] += dh[i][j];
                    dh[i][j] *= g[j];
                    s1 += dh[i][j];
                    s2 += dh[i][j] * xh[i][j];
                }
            }
        }
        const float m1 = warp_sum(s1) / (float)C;
        const float m2 = warp_sum(s2) / (float)C;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                float o[8];
#pragma unroll
                for (int j = 0; j < 8; j++) o[j] = rs * (dh[i][j] - m1 - xh[i][j] * m2);
                store8(dx + (int64_t)row * C + idx * 8, o);
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            rx[i] = nx[i];
            rd[i] = nd[i];
        }
        row = next;
    }
    __syncthreads();
    for (int a = threadIdx.x; a < C; a += blockDim.x) {
        float sg = 0.f, sb = 0.f;
#pragma unroll
        for (int k = 0; k < LN_BWD_WARPS; k++) {
            sg += sh[(size_t)k * 2 * C + a];
            sb += sh[(size_t)k * 2 * C + C + a];
        }
        const int c = (a % cv) * 8 + a / cv;
        partial[(size_t)blockIdx.x * 2 * C + c] = sg;
        partial[(size_t)blockIdx.x * 2 * C + C + c] = sb;
    }
}

static int ln_vpl(int C) { return (C / 8 + 31) / 32; }

#define LN_DISPATCH(VPLV, CALL) \
    switch (VPLV) {             \
        case 1: CALL(1); break; \
        case 2: CALL(2); break; \
        case 3: CALL(3); break; \
        case 4: CALL(4); break; \
        case 5: CALL(5); break; \
        case 6: CALL(6); break; \
        case 7: CALL(7); break; \
        default: CALL(8); break; \
    }

int launch_layernorm_forward(int dtype, void* y, float* mean, float* rstd, const void* x, const void* gamma,
                             const void* beta, int N, int C, cudaStream_t s) {
    const int blocks = (N + LN_FWD_WARPS - 1) / LN_FWD_WARPS;
    if (blocks == 0) return 0;
#define LN_FWD_CALL(V)                                                                                       \
    if (dtype == GPT2_MODE_BF16)                                                                             \
        ln_fwd_kernel<bf16, V><<<blocks, LN_FWD_WARPS * 32, 0, s>>>((bf16*)y, mean, rstd, (const bf16*)x,    \
                                                                    (const bf16*)gamma, (const bf16*)beta, N, \
                                                                    C);                                      \
    else                                                                                                     \
        ln_fwd_kernel<float, V><<<blocks, LN_FWD_WARPS * 32, 0, s>>>((float*)y, mean, rstd, (const float*)x, \
                                                                     (const float*)gamma, (const float*)beta, \
                                                                     N, C);
    LN_DISPATCH(ln_vpl(C), LN_FWD_CALL)
#undef LN_FWD_CALL
    return 1;
}

static int ln_bwd_blocks(int N) {
    int b = (N + LN_BWD_WARPS - 1) / LN_BWD_WARPS;
    return b < LN_BWD_MAX_BLOCKS ? (b < 1 ? 1 : b) : LN_BWD_MAX_BLOCKS;
}

size_t layernorm_backward_scratch(int N, int C) { return (size_t)ln_bwd_blocks(N) * 2 * C * 4; }

template <typename T, int VPL>
static void ln_bwd_launch(int blocks, size_t smem, void* dx, float* partial, const void* dy, const void* x,
                          const void* gamma, const float* mean, const float* rstd, int N, int C, cudaStream_t s) {
    static bool configured = false;  // per instantiation: allow > 48 KB dynamic smem once
    if (!configured) {
        cudaFuncSetAttribute(ln_bwd_kernel<T, VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             LN_BWD_WARPS * 2 * 2048 * 4);
        configured = true;
    }
    ln_bwd_kernel<T, VPL><<<blocks, LN_BWD_WARPS * 32, smem, s>>>((T*)dx, partial, (const T*)dy, (const T*)x,
                                                                  (const T*)gamma, mean, rstd, N, C);
}

int launch_layernorm_backward(int dtype, void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                              const void* gamma, const float* mean, const float* rstd, int N, int C, void* scratch,
                              cudaStream_t s) {
    const int blocks = ln_bwd_blocks(N);
    const size_t smem = (size_t)LN_BWD_WARPS * 2 * C * 4;
    float* partial = (float*)scratch;
#define LN_BWD_CALL(V)                                                                                     \
    if (dtype == GPT2_MODE_BF16)                                                                           \
        ln_bwd_launch<bf16, V>(blocks, smem, dx, partial, dy, x, gamma, mean, rstd, N, C, s);             \
    else                                                                                                   \
        ln_bwd_launch<float, V>(blocks, smem, dx, partial, dy, x, gamma, mean, rstd, N, C, s);
    LN_DISPATCH(ln_vpl(C), LN_BWD_CALL)
#undef LN_BWD_CALL
    launch_colsum(dgamma, dbeta, C, partial, blocks, 2 * C, s);
    return 2;
}
