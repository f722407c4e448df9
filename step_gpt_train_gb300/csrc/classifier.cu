// Fused softmax cross-entropy classifier and the mean-loss reduction.
//
// Each row of logits is read from HBM once, reduced to (max, sum of exp)
// over the real vocabulary columns, and the gradient is written back in place
// over the logits. The normalised probabilities are never stored. Columns
// V..Vp-1 (padding) get 0. Two forms:
//   classifier_stream_kernel  bf16 rows wider than 4096 (the GPT-2 step): a
//                             persistent kernel, two CTAs per SM, each row
//                             copied whole into shared memory by one bulk
//                             copy and processed from there;
//   classifier_kernel         fp32 rows and narrow bf16 rows: one block per
//                             row, the row held in registers (raw 16-byte
//                             vectors).
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

#include <cfloat>

#define LOG2E 1.4426950408889634f

// exp(x - m) for the two modes: ex2.approx for bf16 activations (its error is
// far below bf16 resolution), the accurate expf for the fp32 parity mode.
template <typename T> __device__ __forceinline__ float exp_shift(float x, float m);
template <> __device__ __forceinline__ float exp_shift<bf16>(float x, float m) { return ex2_approx((x - m) * LOG2E); }
template <> __device__ __forceinline__ float exp_shift<float>(float x, float m) { return expf(x - m); }

template <typename T> struct RawVec;
template <> struct RawVec<bf16> { uint4 r; };
template <> struct RawVec<float> { float4 a, b; };

__device__ __forceinline__ void raw_load(RawVec<bf16>& v, const bf16* p) { v.r = __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void raw_load(RawVec<float>& v, const float* p) {
    v.a = __ldcs(reinterpret_cast<const float4*>(p));
    v.b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
}
__device__ __forceinline__ void raw_unpack(const RawVec<bf16>& v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v.r);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ void raw_unpack(const RawVec<float>& v, float (&f)[8]) {
    f[0] = v.a.x; f[1] = v.a.y; f[2] = v.a.z; f[3] = v.a.w;
    f[4] = v.b.x; f[5] = v.b.y; f[6] = v.b.z; f[7] = v.b.w;
}

template <int NT>
__device__ __forceinline__ float block_reduce(float v, bool is_max, float* sh) {
    const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
    v = is_max ? warp_max(v) : warp_sum(v);
    __syncthreads();  // sh may still be read from a previous reduction
    if (lane == 0) sh[w] = v;
    __syncthreads();
    float r = is_max ? -FLT_MAX : 0.f;
    if (threadIdx.x < 32) {
        float x = threadIdx.x < NT / 32 ? sh[threadIdx.x] : (is_max ? -FLT_MAX : 0.f);
        r = is_max ? warp_max(x) : warp_sum(x);
        if (threadIdx.x == 0) sh[32] = r;
    }
    __syncthreads();
    return sh[32];
}

// NT threads per row, VPT 8-element vectors per thread (Vp <= 8 * NT * VPT).
// amax (both classifier kernels; or null): the largest |dlogit| as stored is
// merged into it (float bits), the scale of an FP8 operand.
template <typename T, int NT, int VPT>
__global__ void __launch_bounds__(NT) classifier_kernel(T* __restrict__ logits, float* __restrict__ losses,
                                                        const int32_t* __restrict__ targets, int V, int Vp,
                                                        float dloss, int* status, unsigned* __restrict__ amax) {
    __shared__ float sh[33];
    const int row = blockIdx.x;
    T* z = logits + (int64_t)row * Vp;
    const int nv = Vp / 8;
    RawVec<T> cache[VPT];
#pragma unroll
    for (int i = 0; i < VPT; i++) {
        const int idx = threadIdx.x + i * NT;
        if (idx < nv) raw_load(cache[i], z + idx * 8);
    }
    int tgt = targets[row];
    if (tgt < 0 || tgt >= V) {
        if (threadIdx.x == 0) set_status(status, GPT2_FLAG_TARGET_RANGE);
        tgt = 0;
    }
    // Only the vector that straddles V (and vectors past it) need a column
    // test; every other vector is handled without per-element checks.
    const int full_nv = V / 8;  // vectors wholly inside the real vocabulary
    float m = -FLT_MAX;
#pragma unroll
    for (int i = 0; i < VPT; i++) {
        const int idx = threadIdx.x + i * NT;
        if (idx < nv) {
            float f[8];
            raw_unpack(cache[i], f);
            if (idx < full_nv) {
#pragma unroll
                for (int j = 0; j < 8; j++) m = fmaxf(m, f[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (idx * 8 + j < V) m = fmaxf(m, f[j]);
            }
        }
    }
    m = block_reduce<NT>(m, true, sh);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; i++) {
        const int idx = threadIdx.x + i * NT;
        if (idx < nv) {
            float f[8];
            raw_unpack(cache[i], f);
            if (idx < full_nv) {
#pragma unroll
                for (int j = 0; j < 8; j++) s += exp_shift<T>(f[j], m);
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (idx * 8 + j < V) s += exp_shift<T>(f[j], m);
            }
        }
    }
    s = block_reduce<NT>(s, false, sh);
    const float scale = dloss / s;
    const int tvec = tgt / 8;
    float am = 0.f;  // this thread's largest |dlogit| (amax)
#pragma unroll
    for (int i = 0; i < VPT; i++) {
        const int idx = threadIdx.x + i * NT;
        if (idx < nv) {
            float f[8];
            raw_unpack(cache[i], f);
            if (idx == tvec) {
                // the thread holding the target column reports the loss: lse - z_t
                const int jt = tgt % 8;
                float zt = f[0];
#pragma unroll
                for (int j = 1; j < 8; j++)
                    if (j == jt) zt = f[j];
                losses[row] = m + logf(s) - zt;
            }
            if (idx < full_nv) {
#pragma unroll
                for (int j = 0; j < 8; j++) f[j] = exp_shift<T>(f[j], m) * scale;
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++) f[j] = idx * 8 + j < V ? exp_shift<T>(f[j], m) * scale : 0.f;
            }
            if (idx == tvec) {
                const int jt = tgt % 8;
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (j == jt) f[j] -= dloss;
            }
            store8(z + idx * 8, f);
            if (amax) {
#pragma unroll
                for (int j = 0; j < 8; j++) am = fmaxf(am, fabsf(f[j]));
            }
        }
    }
    if (amax) amax_merge(amax, am);
}

// The bf16 classifier as a persistent kernel: a CTA walks rows row0, row0 + G,
// ... (G = grid size), each copied whole into shared memory by the bulk-copy
// engine, reduced there and written back in place. With NBUF = 2 the next
// row is copied into the other buffer while this one is processed; with
// NBUF = 1 two CTAs share an SM and overlap each other's copies.
template <int NT, int NBUF>
__global__ void __launch_bounds__(NT, 2 / NBUF) classifier_stream_kernel(bf16* __restrict__ logits, float* __restrict__ losses,
                                                                  const int32_t* __restrict__ targets, int N, int V,
                                                                  int Vp, float dloss, int* status,
                                                                  unsigned* __restrict__ amax) {
    float am = 0.f;  // this thread's largest |dlogit| (amax)
    extern __shared__ __align__(128) uint8_t cls_smem[];  // NBUF rows of Vp bf16
    __shared__ float sh[33];
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;
    const uint32_t row_bytes = (uint32_t)Vp * 2;
    const bf16* bufs[2] = {reinterpret_cast<const bf16*>(cls_smem),
                           reinterpret_cast<const bf16*>(cls_smem) + (NBUF == 2 ? Vp : 0)};
    const uint32_t bar[2] = {tc::smem_addr(&bars[0]), tc::smem_addr(&bars[1])};
    if (threadIdx.x == 0) {
        tc::mbar_init(bar[0], 1);
        tc::mbar_init(bar[1], 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    int issued[2] = {-1, -1};  // thread 0: phase parity of the last copy into each buffer
    auto issue = [&](int row, int slot, int k) {
        tc::mbar_expect_tx(bar[slot], row_bytes);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(logits + (int64_t)row * Vp);
        const uint32_t dst = tc::smem_addr(bufs[slot]);
        for (uint32_t off = 0; off < row_bytes; off += 32768u)
            tc::bulk_load_1d(dst + off, src + off, row_bytes - off < 32768u ? row_bytes - off : 32768u, bar[slot]);
        issued[slot] = (k >> 1) & 1;
    };
    const int nv = Vp / 8;
    const int full_nv = V / 8;  // vectors wholly inside the real vocabulary
    if (threadIdx.x == 0 && (int)blockIdx.x < N) issue(blockIdx.x, 0, 0);
    int k = 0;
    for (int row = blockIdx.x; row < N; row += gridDim.x, k++) {
        const int slot = NBUF == 2 ? (k & 1) : 0;
        const int next = row + gridDim.x;
        // the other buffer was released by the barrier that ended the previous row
        if (NBUF == 2 && threadIdx.x == 0 && next < N) issue(next, slot ^ 1, k + 1);
        const bool ok = tc::mbar_wait(bar[slot], NBUF == 2 ? (k >> 1) & 1 : k & 1, &abort_flag, status);
        if (__syncthreads_or(!ok)) break;  // one outcome for the whole block
        const bf16* z = bufs[slot];
        int tgt = targets[row];
        if (tgt < 0 || tgt >= V) {
            if (threadIdx.x == 0) set_status(status, GPT2_FLAG_TARGET_RANGE);
            tgt = 0;
        }
        float m = -FLT_MAX;
        for (int idx = threadIdx.x; idx < nv; idx += NT) {
            float f[8];
            load8(z + idx * 8, f);
            if (idx < full_nv) {
#pragma unroll
                for (int j = 0; j < 8; j++) m = fmaxf(m, f[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (idx * 8 + j < V) m = fmaxf(m, f[j]);
            }
        }
        m = block_reduce<NT>(m, true, sh);
        float s = 0.f;
        for (int idx = threadIdx.x; idx < nv; idx += NT) {
            float f[8];
            load8(z + idx * 8, f);
            if (idx < full_nv) {
#pragma unroll
                for (int j = 0; j < 8; j++) s += exp_shift<bf16>(f[j], m);
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (idx * 8 + j < V) s += exp_shift<bf16>(f[j], m);
            }
        }
        s = block_reduce<NT>(s, false, sh);
        const float scale = dloss / s;
        const int tvec = tgt / 8;
        bf16* zg = logits + (int64_t)row * Vp;
        for (int idx = threadIdx.x; idx < nv; idx += NT) {
            float f[8];
            load8(z + idx * 8, f);
            if (idx == tvec) {
                const int jt = tgt % 8;
                float zt = f[0];
#pragma unroll
                for (int j = 1; j < 8; j++)
                    if (j == jt) zt = f[j];
                losses[row] = m + logf(s) - zt;
            }
            if (idx < full_nv) {
#pragma unroll
                for (int j = 0; j < 8; j++) f[j] = exp_shift<bf16>(f[j], m) * scale;
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++) f[j] = idx * 8 + j < V ? exp_shift<bf16>(f[j], m) * scale : 0.f;
            }
            if (idx == tvec) {
                const int jt = tgt % 8;
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (j == jt) f[j] -= dloss;
            }
            store8(zg + idx * 8, f);
            if (amax) {
#pragma unroll
                for (int j = 0; j < 8; j++) am = fmaxf(am, fabsf(f[j]));
            }
        }
        __syncthreads();  // every thread is done with this buffer before it is refilled
        if (NBUF == 1 && threadIdx.x == 0 && next < N) issue(next, 0, 2 * (k + 1));
    }
    if (amax) amax_merge(amax, am);
    // copies still in flight after an early exit
    if (threadIdx.x == 0)
        for (int b = 0; b < 2; b++)
            if (issued[b] >= 0) tc::mbar_drain(bar[b], (uint32_t)issued[b], status);
}

#define CLS_STREAM_MAX_SMEM (220 * 1024)  // two rows per SM

template <typename T, int NT>
static int classifier_dispatch(void* logits, float* losses, const int32_t* targets, int N, int V, int Vp,
                               float dloss, int* status, cudaStream_t s, unsigned* amax) {
    const int nv = Vp / 8;
    const int vpt = (nv + NT - 1) / NT;
#define CLS_CALL(K)                                                                                                \
    classifier_kernel<T, NT, K><<<N, NT, 0, s>>>((T*)logits, losses, targets, V, Vp, dloss, status, amax); \
    return 1;
    switch (vpt) {
        case 1: CLS_CALL(1)
        case 2: CLS_CALL(2)
        case 3: CLS_CALL(3)
        case 4: CLS_CALL(4)
        case 5: CLS_CALL(5)
        case 6: CLS_CALL(6)
        case 7: CLS_CALL(7)
        case 8: CLS_CALL(8)
        default: return GPT2_ERR_ARG;
    }
#undef CLS_CALL
}

int classifier_set_wait_limit(long long cycles) { return tc::set_wait_limit(cycles); }

int launch_classifier(int dtype, void* logits, float* losses, const int32_t* targets, int N, int V, int Vp,
                      float dloss, int* status, cudaStream_t s, unsigned* amax) {
    if (N == 0) return 0;
    if (dtype == GPT2_MODE_BF16) {
        const size_t smem = (size_t)Vp * 2 * 2;  // two rows per SM either way
        if (Vp > 8 * 256 * 2 && smem <= CLS_STREAM_MAX_SMEM) {
            smem_attr((const void*)classifier_stream_kernel<512, 1>, CLS_STREAM_MAX_SMEM / 2);
            const int grid = N < 2 * gpt2_num_sms() ? N : 2 * gpt2_num_sms();
            classifier_stream_kernel<512, 1><<<grid, 512, smem / 2, s>>>((bf16*)logits, losses, targets, N, V, Vp, dloss,
                                                                         status, amax);
            return 1;
        }
        if (Vp <= 8 * 256 * 2)
            return classifier_dispatch<bf16, 256>(logits, losses, targets, N, V, Vp, dloss, status, s, amax);
        return classifier_dispatch<bf16, 1024>(logits, losses, targets, N, V, Vp, dloss, status, s, amax);
    }
    if (Vp <= 8 * 256 * 2)
        return classifier_dispatch<float, 256>(logits, losses, targets, N, V, Vp, dloss, status, s, amax);
    return classifier_dispatch<float, 1024>(logits, losses, targets, N, V, Vp, dloss, status, s, amax);
}

// Mean of N losses: each of 1024 threads sums a fixed strided subset in
// order, then a fixed shuffle tree; deterministic.
__global__ void __launch_bounds__(1024) mean_loss_kernel(float* out, const float* __restrict__ losses, int N) {
    __shared__ float sh[33];
    float s = 0.f;
    for (int i = threadIdx.x; i < N; i += 1024) s += losses[i];
    s = block_reduce<1024>(s, false, sh);
    if (threadIdx.x == 0) *out = s / (float)N;
}

int launch_mean_loss(float* out, const float* losses, int N, cudaStream_t s) {
    mean_loss_kernel<<<1, 1024, 0, s>>>(out, losses, N);
    return 1;
}
