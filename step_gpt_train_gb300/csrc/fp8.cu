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
//                        input-gradient products, 128 x 64 tiles through
//                        shared memory, 16-byte loads.
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
    constexpr int64_t STEP = 8 * 256;
    float m = 0.f;
    int64_t i = lo + 8 * (int64_t)threadIdx.x;
    // four vectors per thread in flight, then the rest one at a time
    for (; i + 3 * STEP + 8 <= hi; i += 4 * STEP) {
        float v[4][8];
#pragma unroll
        for (int u = 0; u < 4; u++) load8(x + i + u * STEP, v[u]);
#pragma unroll
        for (int u = 0; u < 4; u++)
#pragma unroll
            for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(v[u][j]));
    }
    for (; i < hi; i += STEP) {
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

// x [R][C] (bf16) -> codes, written transposed to qt [C][R] and, when q is
// given, as they are to q [R][C]. A block takes 128 rows (r0) and 64 columns
// (c0); warp w rows r0 + 32w .. + 31. Lane l reads 16 bytes (8 columns,
// 8 (l % 8) ..) of 8 consecutive rows, 8 (l / 8) .., so each load of the warp
// covers four whole 128-byte row pieces; it writes the row-layout codes 8
// at a time, and the 8 codes of each of its columns (8 consecutive rows) to a
// shared tile [64 columns][128 rows] as two 4-byte words (a 132-byte tile
// row keeps the 8 lanes of a row group on distinct banks but for pairs);
// the block then writes 16-byte pieces of qt's rows from the tile (byte by
// byte at a ragged edge or where R % 16 != 0).
constexpr int QT_ROWS = 128, QT_STRIDE = 132;
// With amax (the tensor's largest |value| as float bits, taken by the kernel
// that wrote x) the scale pair is formed here as amax_scale_kernel forms it,
// block (0, 0) writing it to scales; else scales holds it already.
template <int FMT>
__global__ void __launch_bounds__(128) quantize_fp8_t_kernel(uint8_t* __restrict__ qt, uint8_t* __restrict__ q,
                                                             const bf16* __restrict__ x, int R, int C,
                                                             float* __restrict__ scales,
                                                             const unsigned* __restrict__ amax, float fmax) {
    __shared__ __align__(16) uint8_t tile[64 * QT_STRIDE];
    float s;
    if (amax) {
        const float t = __uint_as_float(*amax);
        s = t > 0.f ? fmax / t : 1.f;
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
            scales[0] = s;
            scales[1] = t > 0.f ? t / fmax : 1.f;
        }
    } else {
        s = scales[0];
    }
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int r0 = blockIdx.y * QT_ROWS, c0 = blockIdx.x * 64;
    const int cl = 8 * (lane % 8);               // first of this lane's 8 columns within the tile
    const int rl = 32 * w + 8 * (lane / 8);      // first of its 8 rows within the tile
    const int c = c0 + cl;
    if (c < C) {  // C % 8 == 0: the 8 columns are all inside
        uint32_t col[8][2];  // codes of column cl + j, rows rl .. rl + 7, four to a word
#pragma unroll
        for (int j = 0; j < 8; j++) col[j][0] = col[j][1] = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int r = r0 + rl + i;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < R) v = *reinterpret_cast<const uint4*>(x + (int64_t)r * C + c);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
            uint32_t rowc[2];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const uint16_t cc =
                    fp8x2<FMT>(__uint_as_float(u[k] << 16) * s, __uint_as_float(u[k] & 0xFFFF0000u) * s);
                col[2 * k][i / 4] |= (uint32_t)(cc & 0xFF) << (8 * (i % 4));
                col[2 * k + 1][i / 4] |= (uint32_t)(cc >> 8) << (8 * (i % 4));
                if (k % 2 == 0) rowc[k / 2] = cc;
                else rowc[k / 2] |= (uint32_t)cc << 16;
            }
            if (q && r < R) *reinterpret_cast<uint2*>(q + (int64_t)r * C + c) = make_uint2(rowc[0], rowc[1]);
        }
#pragma unroll
        for (int j = 0; j < 8; j++) {
            uint32_t* t = reinterpret_cast<uint32_t*>(tile + (cl + j) * QT_STRIDE + rl);
            t[0] = col[j][0];
            t[1] = col[j][1];
        }
    }
    __syncthreads();
    const int nrows = min(QT_ROWS, R - r0);  // rows of this block inside the matrix
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int idx = threadIdx.x + 128 * i;   // 64 qt rows x 8 pieces of 16 bytes
        const int row = idx / 8, piece = idx % 8;
        const int cc = c0 + row;
        const int rr = 16 * piece;
        if (cc >= C || rr >= nrows) continue;
        uint8_t* dst = qt + (int64_t)cc * R + r0 + rr;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(tile + row * QT_STRIDE + rr);
        if (rr + 16 <= nrows && R % 16 == 0) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(src[0], src[1], src[2], src[3]);
        } else {
            const uint8_t* sb = tile + row * QT_STRIDE + rr;
            for (int j = 0; j < 16 && rr + j < nrows; j++) dst[j] = sb[j];
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
                          cudaStream_t s, const unsigned* amax) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return GPT2_ERR_ARG;
    if (R <= 0 || C <= 0) return 0;
    if ((C % 8) != 0) return GPT2_ERR_ARG;  // 16-byte vector reads of x rows
    const dim3 grid((unsigned)((C + 63) / 64), (unsigned)((R + QT_ROWS - 1) / QT_ROWS));
    if (grid.y > 65535) return GPT2_ERR_ARG;
    const float fmax = fmt == FP8_E4M3 ? 448.f : 57344.f;
    float* sc = const_cast<float*>(scales);  // written only when amax is given
    if (fmt == FP8_E4M3) quantize_fp8_t_kernel<FP8_E4M3><<<grid, 128, 0, s>>>(qt, q, x, R, C, sc, amax, fmax);
    else quantize_fp8_t_kernel<FP8_E5M2><<<grid, 128, 0, s>>>(qt, q, x, R, C, sc, amax, fmax);
    return 1;
}

int launch_quantize_fp8(uint8_t* q, float* scales, const bf16* x, int64_t n, int fmt, float* partial,
                        cudaStream_t s) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return GPT2_ERR_ARG;
    if (n <= 0) return 0;
    const int a = launch_fp8_amax_scale(scales, x, n, fmt, partial, s);
    return a + launch_quantize_fp8_rows(q, scales, x, n, fmt, s);
}
