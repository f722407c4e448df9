// Shared device helpers for the GPT-2 step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

#include "../../include/gpt2.h"
#include "../../include/gpt2_ops.h"

typedef __nv_bfloat16 bf16;

// Bits OR-ed into a device status word; never a trap.
#define GPT2_FLAG_TOKEN_RANGE 1
#define GPT2_FLAG_TIMEOUT 2
#define GPT2_FLAG_TARGET_RANGE 4

// Bounded spin: a wait gives up after this many clock cycles (~2 s at 2 GHz).
#define GPT2_WAIT_LIMIT_CYCLES (4000000000LL)

__device__ __forceinline__ void set_status(int* status, int bit) {
    if (status) atomicOr(status, bit);
}

// The largest |value| of what a warp stored as bf16 (m: this lane's largest
// |value| before the rounding, which is monotone, so rounding the maximum
// gives the maximum of the rounded values), merged into *amax: the bits of a
// non-negative float order as unsigned integers, so atomicMax on them is the
// float maximum, whatever the order of the merges. Every lane of the warp
// calls it. The amax of an FP8 operand, taken by the kernel that writes it.
__device__ __forceinline__ void amax_merge(unsigned* amax, float m) {
    m = __bfloat162float(__float2bfloat16_rn(m));
#pragma unroll
    for (int off = 16; off > 0; off /= 2) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) atomicMax(amax, __float_as_uint(m));
}

// Allow `bytes` of dynamic shared memory for `kernel` on the current device,
// once per (kernel, device): thread-safe, and a failed attempt is not
// remembered (the next launch tries again, and a launch that still lacks
// the attribute fails with an error the caller reports).
inline cudaError_t smem_attr(const void* kernel, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kernel, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({kernel, dev});
    return e;
}

// ---- 8-element vector access: one 16-byte access for bf16, two for fp32 ----

__device__ __forceinline__ void load8(const bf16* p, float (&f)[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 v = __bfloat1622float2(h[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}
__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
    float4 a = reinterpret_cast<const float4*>(p)[0];
    float4 b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
// Streaming (evict-first) variants for data read exactly once.
__device__ __forceinline__ void load8_stream(const bf16* p, float (&f)[8]) {
    uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 v = __bfloat1622float2(h[i]);
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
    }
}
__device__ __forceinline__ void load8_stream(const float* p, float (&f)[8]) {
    float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void store8(bf16* p, const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// Raw 8-element vectors, loaded now and converted later (prefetch into registers).
template <typename T> struct Raw8;
template <> struct Raw8<bf16> { uint4 v; };
template <> struct Raw8<float> { float4 a, b; };
__device__ __forceinline__ void raw_load(Raw8<bf16>& r, const bf16* p) { r.v = *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ void raw_load(Raw8<float>& r, const float* p) {
    r.a = reinterpret_cast<const float4*>(p)[0];
    r.b = reinterpret_cast<const float4*>(p)[1];
}
__device__ __forceinline__ void raw_unpack(const Raw8<bf16>& r, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r.v);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ void raw_unpack(const Raw8<float>& r, float (&f)[8]) {
    f[0] = r.a.x; f[1] = r.a.y; f[2] = r.a.z; f[3] = r.a.w;
    f[4] = r.b.x; f[5] = r.b.y; f[6] = r.b.z; f[7] = r.b.w;
}

// ---- per-thread asynchronous global -> shared copies (cp.async groups) ----

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still pending.
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_float<bf16>(float x) { return __float2bfloat16_rn(x); }

// ---- warp / block reductions (fixed shuffle order: deterministic) ----

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---- hardware approximate transcendental instructions (PTX, MUFU) ----

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GELU tanh-form constants: sqrt(2/pi) and the cubic coefficient.
#define GELU_K 0.7978845608028654f
#define GELU_A 0.044715f

// GELU's 0.5 (1 + tanh(y)) evaluated as the logistic function of 2y,
// 1 / (1 + exp(-2y)) (the same quantity, since tanh y = 2 sigmoid(2y) - 1).
// This form keeps full relative accuracy on the negative tail, where
// 1 + tanh(y) cancels. bf16 activations use the hardware exp2 and a fast
// divide; the fp32 parity mode uses expf and an IEEE divide.
template <typename T> __device__ __forceinline__ float gelu_sigmoid(float y);
template <> __device__ __forceinline__ float gelu_sigmoid<bf16>(float y) {
    const float z = fminf(-2.f * 1.4426950408889634f * y, 126.f);  // exp(-2y) = 2^z, capped below overflow
    return __fdividef(1.f, 1.f + ex2_approx(z));
}
template <> __device__ __forceinline__ float gelu_sigmoid<float>(float y) { return 1.f / (1.f + expf(-2.f * y)); }

// g = u s and g' = s + 2 u s (1 - s) sqrt(2/pi) (1 + 3*0.044715 u^2), with
// s = 0.5 (1 + tanh(y)), y = sqrt(2/pi) (u + 0.044715 u^3); the derivative uses
// 1 - tanh(y)^2 = 4 s (1 - s).
template <typename T>
__device__ __forceinline__ float gelu_fwd_f(float u) {
    const float y = GELU_K * (u + GELU_A * u * u * u);
    return u * gelu_sigmoid<T>(y);
}
template <typename T>
__device__ __forceinline__ float gelu_grad_f(float u) {
    const float y = GELU_K * (u + GELU_A * u * u * u);
    const float s = gelu_sigmoid<T>(y);
    return s + 2.f * u * s * (1.f - s) * GELU_K * (1.f + 3.f * GELU_A * u * u);
}
// Both at once (one sigmoid): g = gelu(u), d = gelu'(u).
template <typename T>
__device__ __forceinline__ void gelu_both_f(float u, float& g, float& d) {
    const float y = GELU_K * (u + GELU_A * u * u * u);
    const float s = gelu_sigmoid<T>(y);
    g = u * s;
    d = s + 2.f * u * s * (1.f - s) * GELU_K * (1.f + 3.f * GELU_A * u * u);
}

// ---- host-side helpers ----

static inline int grid_for(int64_t work_items, int threads, int max_blocks) {
    int64_t b = (work_items + threads - 1) / threads;
    if (b < 1) b = 1;
    if (b > max_blocks) b = max_blocks;
    return (int)b;
}

// Number of SMs on the current device (cached per process).
int gpt2_num_sms();
