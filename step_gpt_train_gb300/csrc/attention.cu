// Causal multi-head attention: the fp32 path (the exact-parity mode, head
// size <= 64; one thread per query for the forward and dQ, per key for dK and
// dV; fp32 FMA and expf) and the launchers. The bf16 path runs on the tcgen05
// tensor cores (attention_tc.cu); its backward starts here with
// D = rowsum(dO * O). Both backwards recompute P from the saved log-sum-exp
// and give every output element a single writer: no atomics, deterministic.
#include "common.cuh"
#include "launch.h"

#include <cfloat>

#define ATT_LOG2E 1.4426950408889634f
#define ATT_LN2 0.6931471805599453f

// ============================================================ backward: D = rowsum(dO * O)

// One 8-element vector of dO and of O per thread; the PARTS = hd/8 threads
// of a (row, head) pair are adjacent lanes and add their partial dot products
// by a shuffle tree (PARTS is 1, 2, 4 or 8). All loads of a warp are
// contiguous. Indices are 32-bit (the launcher checks B*T*H*PARTS < 2^31):
// with 64-bit divisions the kernel was bound by integer arithmetic.
template <typename T, int PARTS>
__global__ void attn_bwd_dot_kernel(float* __restrict__ D, const T* __restrict__ dout, const T* __restrict__ o,
                                    int B, int Tlen, int C, int H) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;  // ((b, t, h), part)
    const int pair = i / PARTS, part = i % PARTS;
    const bool valid = pair < B * Tlen * H;
    const int bt = valid ? pair / H : 0, h = pair - bt * H;
    float s = 0.f;
    if (valid) {
        float x[8], y[8];
        const int64_t off = (int64_t)bt * C + h * (8 * PARTS) + part * 8;
        load8(dout + off, x);
        load8(o + off, y);
#pragma unroll
        for (int j = 0; j < 8; j++) s += x[j] * y[j];
    }
#pragma unroll
    for (int off = PARTS / 2; off > 0; off /= 2) s += __shfl_xor_sync(0xffffffffu, s, off, PARTS);
    if (valid && part == 0) {
        const int b = bt / Tlen, t = bt - b * Tlen;
        D[(b * H + h) * Tlen + t] = s;
    }
}

template <typename T>
void launch_dot(float* D, const T* dout, const T* o, int B, int T_, int C, int H, cudaStream_t s) {
    const int parts = C / H / 8;
    const int blocks = (int)(((int64_t)B * T_ * H * parts + 255) / 256);
    switch (parts) {
        case 1: attn_bwd_dot_kernel<T, 1><<<blocks, 256, 0, s>>>(D, dout, o, B, T_, C, H); break;
        case 2: attn_bwd_dot_kernel<T, 2><<<blocks, 256, 0, s>>>(D, dout, o, B, T_, C, H); break;
        case 4: attn_bwd_dot_kernel<T, 4><<<blocks, 256, 0, s>>>(D, dout, o, B, T_, C, H); break;
        default: attn_bwd_dot_kernel<T, 8><<<blocks, 256, 0, s>>>(D, dout, o, B, T_, C, H); break;
    }
}

// ============================================================ fp32 path

template <int HD>
__global__ void attn_fwd_f32_kernel(float* __restrict__ o, float* __restrict__ lse, const float* __restrict__ qkv,
                                    int B, int T, int C, int H, float scale) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (b, h, t)
    if (i >= (int64_t)B * H * T) return;
    const int t = (int)(i % T);
    const int h = (int)((i / T) % H);
    const int b = (int)(i / ((int64_t)T * H));
    const int ld = 3 * C;
    const float* base = qkv + (int64_t)b * T * ld + h * HD;
    float q[HD], acc[HD];
#pragma unroll
    for (int d = 0; d < HD; d++) {
        q[d] = base[(int64_t)t * ld + d];
        acc[d] = 0.f;
    }
    float m = -FLT_MAX, l = 0.f;
    for (int s = 0; s <= t; s++) {
        const float* k = base + (int64_t)s * ld + C;
        const float* v = base + (int64_t)s * ld + 2 * C;
        float x = 0.f;
#pragma unroll
        for (int d = 0; d < HD; d++) x += q[d] * k[d];
        x *= scale;
        if (x > m) {
            const float a = expf(m - x);
            l *= a;
#pragma unroll
            for (int d = 0; d < HD; d++) acc[d] *= a;
            m = x;
        }
        const float p = expf(x - m);
        l += p;
#pragma unroll
        for (int d = 0; d < HD; d++) acc[d] += p * v[d];
    }
    float* out = o + ((int64_t)b * T + t) * C + h * HD;
#pragma unroll
    for (int d = 0; d < HD; d++) out[d] = acc[d] / l;
    lse[((int64_t)b * H + h) * T + t] = m + logf(l);
}

template <int HD>
__global__ void attn_bwd_dq_f32_kernel(float* __restrict__ dqkv, const float* __restrict__ dout,
                                       const float* __restrict__ qkv, const float* __restrict__ lse,
                                       const float* __restrict__ Dg, int B, int T, int C, int H, float scale) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * H * T) return;
    const int t = (int)(i % T);
    const int h = (int)((i / T) % H);
    const int b = (int)(i / ((int64_t)T * H));
    const int ld = 3 * C;
    const float* base = qkv + (int64_t)b * T * ld + h * HD;
    const float* dorow = dout + ((int64_t)b * T + t) * C + h * HD;
    float q[HD], dov[HD], dq[HD];
#pragma unroll
    for (int d = 0; d < HD; d++) {
        q[d] = base[(int64_t)t * ld + d];
        dov[d] = dorow[d];
        dq[d] = 0.f;
    }
    const float L = lse[((int64_t)b * H + h) * T + t];
    const float Dt = Dg[((int64_t)b * H + h) * T + t];
    for (int s = 0; s <= t; s++) {
        const float* k = base + (int64_t)s * ld + C;
        const float* v = base + (int64_t)s * ld + 2 * C;
        float x = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < HD; d++) {
            x += q[d] * k[d];
            dp += dov[d] * v[d];
        }
        const float p = expf(x * scale - L);
        const float ds = p * (dp - Dt);
#pragma unroll
        for (int d = 0; d < HD; d++) dq[d] += ds * k[d];
    }
    float* out = dqkv + ((int64_t)b * T + t) * ld + h * HD;
#pragma unroll
    for (int d = 0; d < HD; d++) out[d] = dq[d] * scale;
}

template <int HD>
__global__ void attn_bwd_dkdv_f32_kernel(float* __restrict__ dqkv, const float* __restrict__ dout,
                                         const float* __restrict__ qkv, const float* __restrict__ lse,
                                         const float* __restrict__ Dg, int B, int T, int C, int H, float scale) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * H * T) return;
    const int s = (int)(i % T);
    const int h = (int)((i / T) % H);
    const int b = (int)(i / ((int64_t)T * H));
    const int ld = 3 * C;
    const float* base = qkv + (int64_t)b * T * ld + h * HD;
    float k[HD], v[HD], dk[HD], dv[HD];
#pragma unroll
    for (int d = 0; d < HD; d++) {
        k[d] = base[(int64_t)s * ld + C + d];
        v[d] = base[(int64_t)s * ld + 2 * C + d];
        dk[d] = 0.f;
        dv[d] = 0.f;
    }
    const float* lrow = lse + ((int64_t)b * H + h) * T;
    const float* drow = Dg + ((int64_t)b * H + h) * T;
    for (int t = s; t < T; t++) {
        const float* q = base + (int64_t)t * ld;
        const float* dov = dout + ((int64_t)b * T + t) * C + h * HD;
        float x = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < HD; d++) {
            x += q[d] * k[d];
            dp += dov[d] * v[d];
        }
        const float p = expf(x * scale - lrow[t]);
        const float ds = p * (dp - drow[t]);
#pragma unroll
        for (int d = 0; d < HD; d++) {
            dv[d] += p * dov[d];
            dk[d] += ds * q[d];
        }
    }
    float* out = dqkv + ((int64_t)b * T + s) * ld + h * HD;
#pragma unroll
    for (int d = 0; d < HD; d++) {
        out[C + d] = dk[d] * scale;
        out[2 * C + d] = dv[d];
    }
}

// ============================================================ launchers

int launch_attention_forward(int dtype, void* o, float* lse, const void* qkv, int B, int T, int C, int H,
                             int* status, cudaStream_t s) {
    const int hd = C / H;
    if (B * T == 0) return 0;
    if (dtype == GPT2_MODE_BF16) {
        if (hd != 64) return GPT2_ERR_ARG;
        return launch_attention_forward_tc((bf16*)o, lse, (const bf16*)qkv, B, T, C, H, status, s);
    }
    const int64_t n = (int64_t)B * H * T;
    const int blocks = (int)((n + 127) / 128);
    const float scale = 1.0f / sqrtf((float)hd);
    switch (hd) {
        case 8: attn_fwd_f32_kernel<8><<<blocks, 128, 0, s>>>((float*)o, lse, (const float*)qkv, B, T, C, H, scale); break;
        case 16: attn_fwd_f32_kernel<16><<<blocks, 128, 0, s>>>((float*)o, lse, (const float*)qkv, B, T, C, H, scale); break;
        case 32: attn_fwd_f32_kernel<32><<<blocks, 128, 0, s>>>((float*)o, lse, (const float*)qkv, B, T, C, H, scale); break;
        case 64: attn_fwd_f32_kernel<64><<<blocks, 128, 0, s>>>((float*)o, lse, (const float*)qkv, B, T, C, H, scale); break;
        default: return GPT2_ERR_ARG;
    }
    return 1;
}

size_t attention_backward_scratch(int B, int T, int H) { return (size_t)B * H * T * 4; }

int launch_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv, const void* o,
                              const float* lse, int B, int T, int C, int H, void* scratch, int* status,
                              cudaStream_t s) {
    const int hd = C / H;
    if (hd != 8 && hd != 16 && hd != 32 && hd != 64) return GPT2_ERR_ARG;  // the head sizes built
    if (B * T == 0) return 0;
    if ((int64_t)B * T * H * (hd / 8) + 255 >= ((int64_t)1 << 31)) return GPT2_ERR_ARG;  // 32-bit indices below
    float* D = (float*)scratch;
    const float scale = 1.0f / sqrtf((float)hd);
    if (dtype == GPT2_MODE_BF16) {
        if (hd != 64) return GPT2_ERR_ARG;
        return launch_attention_backward_tc((bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv, (const bf16*)o, lse, D,
                                            B, T, C, H, status, s);
    }
    launch_dot(D, (const float*)dout, (const float*)o, B, T, C, H, s);
    const int64_t n = (int64_t)B * H * T;
    const int blocks = (int)((n + 127) / 128);
#define ATT_BWD_F32(HDV)                                                                                          \
    attn_bwd_dq_f32_kernel<HDV><<<blocks, 128, 0, s>>>((float*)dqkv, (const float*)dout, (const float*)qkv, lse, \
                                                       D, B, T, C, H, scale);                                     \
    attn_bwd_dkdv_f32_kernel<HDV><<<blocks, 128, 0, s>>>((float*)dqkv, (const float*)dout, (const float*)qkv,    \
                                                         lse, D, B, T, C, H, scale);                              \
    break;
    switch (hd) {
        case 8: ATT_BWD_F32(8)
        case 16: ATT_BWD_F32(16)
        case 32: ATT_BWD_F32(32)
        case 64: ATT_BWD_F32(64)
        default: return GPT2_ERR_ARG;
    }
#undef ATT_BWD_F32
    return 3;
}
