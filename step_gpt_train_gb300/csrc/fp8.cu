// Per-tensor FP8 quantization for the FP8 linear layer (the modded-nanogpt
// project page, "NanoGPT (124M) in 90 seconds", "How it works": FP8 for the
// MLP, the QKV projections and the head), to e4m3 (largest finite value 448,
// for weights and activations) or e5m2 (largest finite value 57344, the wider
// range for gradients), both as in the OCP 8-bit floating point format.
// Three launches:
//   amax_partial_kernel  each of FP8_BLOCKS blocks takes the largest |x| of a
//                        fixed contiguous range (a maximum does not depend on
//                        the order, so the result is exact);
//   amax_scale_kernel    one block: amax, scale = fmax / amax, 1 / scale as
//                        amax / fmax (both 1 when amax is 0);
//   quantize_fp8_kernel  q = fp8(x * scale), the product rounded to fp32 and
//                        converted with round-to-nearest-even and saturation
//                        at +-fmax (cvt.rn.satfinite), 8 values per thread.
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

}  // namespace

size_t fp8_quantize_scratch() { return FP8_BLOCKS * 4; }

int launch_quantize_fp8(uint8_t* q, float* scales, const bf16* x, int64_t n, int fmt, float* partial,
                        cudaStream_t s) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return GPT2_ERR_ARG;
    if (n <= 0) return 0;
    amax_partial_kernel<<<FP8_BLOCKS, 256, 0, s>>>(partial, x, n);
    amax_scale_kernel<<<1, FP8_BLOCKS, 0, s>>>(scales, partial, fmt == FP8_E4M3 ? 448.f : 57344.f);
    const int64_t threads = (n + 7) / 8;
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    if (fmt == FP8_E4M3) quantize_fp8_kernel<FP8_E4M3><<<blocks, 256, 0, s>>>(q, x, n, scales);
    else quantize_fp8_kernel<FP8_E5M2><<<blocks, 256, 0, s>>>(q, x, n, scales);
    return 3;
}
