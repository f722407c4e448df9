// Per-tensor FP8 quantization for the FP8 linear layers (the modded-nanogpt
// project page, "NanoGPT (124M) in 90 seconds", "How it works": FP8 for the
// MLP, the QKV projections and the head), to e4m3 (largest finite value 448,
// for weights and activations) or e5m2 (largest finite value 57344, the wider
// range for gradients), both as in the OCP 8-bit floating point format.
//   amax_partial_kernel  each of FP8_BLOCKS blocks takes the largest |x| of a
//                        fixed contiguous range (a maximum does not depend on
//                        the order, so the result is exact);
//   amax_scale_kernel    one block: amax, scale = fmax / amax, 1 / scale as
//                        amax / fmax (both 1 when amax is 0);
//   quantize_fp8_kernel  q = fp8(x * scale), the product rounded to fp32 and
//                        converted with round-to-nearest-even and saturation
//                        at +-fmax (cvt.rn.satfinite), 8 values per thread;
//   quantize_fp8_t_kernel the same codes for a [R][C] matrix written
//                        transposed, [C][R] (and optionally also [R][C]): the
//                        K-major operands of the weight-gradient and
//                        input-gradient products, 64 x 64 tiles through
//                        shared memory.
// NaN inputs do not enter amax (fmaxf ignores them) and quantize to NaN.
#include "common.cuh"
#include "launch.h"

#define FP8_BLOCKS 1024

namespace {

__global__ void __launch_bounds__(256) amax_partial_kernel(float* __restrict__ partial, const bf16* __restrict__ x,
                                                           int64_t n) {
    __shared__ float sh[8];
    const int64_t per = ((n + FP8_BLOCKS - 1) / FP8_BLOCKS + 7) / 8 * 8;  // whole 8-value vectors
    const int64_t lo = (int64_t)blockIdx.x * per;
    const int64_t hi = lo + per < n ? lo + per : n;
    float m = 0.f;
    for (int64_t i = lo + 8 * (int64_t)threadIdx.x; i < hi; i += 8 * 256) {
        if (i + 8 <= hi) {
            float v[8];
            load8(x + i, v);
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[j]));
        } else {
            for (int64_t k = i; k < hi; k++) m = fmaxf(m, fabsf(__bfloat162float(x[k])));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (threadIdx.x % 32 == 0) sh[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; w++) t = fmaxf(t, sh[w]);
        partial[blockIdx.x] = t;
    }
}

__global__ void __launch_bounds__(FP8_BLOCKS) amax_scale_kernel(float* __restrict__ scales,
                                                                const float* __restrict__ partial, float fmax) {
    __shared__ float sh[32];
    float m = partial[threadIdx.x];
#pragma unroll
    for (int off = 16; off > 0; off /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (threadIdx.x % 32 == 0) sh[threadIdx.x / 32] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < FP8_BLOCKS / 32; w++) t = fmaxf(t, sh[w]);
        scales[0] = t > 0.f ? fmax / t : 1.f;
        scales[1] = t > 0.f ? t / fmax : 1.f;
    }
}

// Two fp32 values to two codes of format FMT (0: e4m3, 1: e5m2), lo in the low byte.
template <int FMT>
__device__ __forceinline__ uint16_t fp8x2(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == 0)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int FMT>
__global__ void __launch_bounds__(256) quantize_fp8_kernel(uint8_t* __restrict__ q, const bf16* __restrict__ x,
                                                           int64_t n, const float* __restrict__ scales) {
    const float s = scales[0];
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i >= n) return;
    if (i + 8 <= n) {
        float v[8];
        load8(x + i, v);
        uint2 w;
        w.x = (uint32_t)fp8x2<FMT>(v[0] * s, v[1] * s) | ((uint32_t)fp8x2<FMT>(v[2] * s, v[3] * s) << 16);
        w.y = (uint32_t)fp8x2<FMT>(v[4] * s, v[5] * s) | ((uint32_t)fp8x2<FMT>(v[6] * s, v[7] * s) << 16);
        *reinterpret_cast<uint2*>(q + i) = w;
    } else {
        for (int64_t k = i; k < n; k++) q[k] = (uint8_t)(fp8x2<FMT>(__bfloat162float(x[k]) * s, 0.f) & 0xFF);
    }
}

// 64 x 64 tile of x [R][C] (bf16) -> codes, written transposed to qt [C][R]
// and, when q is given, as they are to q [R][C]. 256 threads: each converts
// two 8-column pieces of the tile (rows r, r + 32), stores the codes to a
// transposed shared tile, then writes 16 consecutive codes of one output row.
// Parts of the tile outside the matrix are skipped; R and C need not be
// multiples of 64, but rows of qt and q are written 16 bytes at a time only
// where R (resp. C) is a multiple of 16 and the piece is whole.
template <int FMT>
__global__ void __launch_bounds__(256) quantize_fp8_t_kernel(uint8_t* __restrict__ qt, uint8_t* __restrict__ q,
                                                             const bf16* __restrict__ x, int R, int C,
                                                             const float* __restrict__ scales) {
    __shared__ __align__(16) uint8_t tile[64][64 + 16];  // [column][row]
    const float s = scales[0];
    const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
    const int t = threadIdx.x;
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const int rl = t / 8 + 32 * h, cl = (t % 8) * 8;  // row and first column within the tile
        const int r = r0 + rl, c = c0 + cl;
        uint8_t code[8];
        if (r < R && c + 8 <= C) {
            float v[8];
            load8(x + (int64_t)r * C + c, v);
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const uint16_t w = fp8x2<FMT>(v[j] * s, v[j + 1] * s);
                code[j] = (uint8_t)(w & 0xFF);
                code[j + 1] = (uint8_t)(w >> 8);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++)
                code[j] = (r < R && c + j < C)
                              ? (uint8_t)(fp8x2<FMT>(__bfloat162float(x[(int64_t)r * C + c + j]) * s, 0.f) & 0xFF)
                              : 0;
        }
#pragma unroll
        for (int j = 0; j < 8; j++) tile[cl + j][rl] = code[j];
        if (q && r < R) {
            if (c + 8 <= C && C % 8 == 0) {
                uint2 w;
                w.x = code[0] | (code[1] << 8) | (code[2] << 16) | ((uint32_t)code[3] << 24);
                w.y = code[4] | (code[5] << 8) | (code[6] << 16) | ((uint32_t)code[7] << 24);
                *reinterpret_cast<uint2*>(q + (int64_t)r * C + c) = w;
            } else {
                for (int j = 0; j < 8 && c + j < C; j++) q[(int64_t)r * C + c + j] = code[j];
            }
        }
    }
    __syncthreads();
    const int cl = t / 4, rl = (t % 4) * 16;  // output row (a column of x) and its first code
    const int c = c0 + cl, r = r0 + rl;
    if (c < C) {
        uint8_t* dst = qt + (int64_t)c * R + r;
        if (r + 16 <= R && R % 16 == 0) {
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(&tile[cl][rl]);
        } else {
            for (int j = 0; j < 16 && r + j < R; j++) dst[j] = tile[cl][rl + j];
        }
    }
}

}  // namespace

size_t fp8_quantize_scratch() { return FP8_BLOCKS * 4; }

int launch_fp8_amax_scale(float* scales, const bf16* x, int64_t n, int fmt, float* partial, cudaStream_t s) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return GPT2_ERR_ARG;
    amax_partial_kernel<<<FP8_BLOCKS, 256, 0, s>>>(partial, x, n);
    amax_scale_kernel<<<1, FP8_BLOCKS, 0, s>>>(scales, partial, fmt == FP8_E4M3 ? 448.f : 57344.f);
    return 2;
}

int launch_quantize_fp8_rows(uint8_t* q, const float* scales, const bf16* x, int64_t n, int fmt, cudaStream_t s) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return GPT2_ERR_ARG;
    if (n <= 0) return 0;
    const int64_t threads = (n + 7) / 8;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    if (fmt == FP8_E4M3) quantize_fp8_kernel<FP8_E4M3><<<blocks, 256, 0, s>>>(q, x, n, scales);
    else quantize_fp8_kernel<FP8_E5M2><<<blocks, 256, 0, s>>>(q, x, n, scales);
    return 1;
}

int launch_quantize_fp8_t(uint8_t* qt, uint8_t* q, const float* scales, const bf16* x, int R, int C, int fmt,
                          cudaStream_t s) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return GPT2_ERR_ARG;
    if (R <= 0 || C <= 0) return 0;
    if ((C % 8) != 0) return GPT2_ERR_ARG;  // 16-byte vector reads of x rows
    const dim3 grid((unsigned)((C + 63) / 64), (unsigned)((R + 63) / 64));
    if (grid.y > 65535) return GPT2_ERR_ARG;
    if (fmt == FP8_E4M3) quantize_fp8_t_kernel<FP8_E4M3><<<grid, 256, 0, s>>>(qt, q, x, R, C, scales);
    else quantize_fp8_t_kernel<FP8_E5M2><<<grid, 256, 0, s>>>(qt, q, x, R, C, scales);
    return 1;
}

int launch_quantize_fp8(uint8_t* q, float* scales, const bf16* x, int64_t n, int fmt, float* partial,
                        cudaStream_t s) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return GPT2_ERR_ARG;
    if (n <= 0) return 0;
    const int a = launch_fp8_amax_scale(scales, x, n, fmt, partial, s);
    return a + launch_quantize_fp8_rows(q, scales, x, n, fmt, s);
}
