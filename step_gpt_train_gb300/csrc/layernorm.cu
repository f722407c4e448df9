// LayerNorm forward and backward: one warp per row, the row held in
// registers (16-byte vector loads), statistics by warp shuffles.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

#define LN_EPS 1e-5f
#define LN_FWD_WARPS 8
#define LN_BWD_WARPS 8
#define LN_BWD_MAX_BLOCKS 608  // four resident blocks on each of 152 SMs
#define LN_STAGES 3                    // row slots per warp in the staged kernels
#define LN_STAGED_MAX_ROW_BYTES 2048  // rows of up to 1024 bf16 or 512 fp32 values

// y = (x - mean) * rstd * gamma + beta, biased variance, eps 1e-5.
// With r != null the row normalised is the residual sum x + r, rounded to T
// and stored to xsum first (the residual join followed by the next block's
// LayerNorm, in one pass over the row).
// VPL = 8-element vectors per lane (C <= 256 * VPL). amax (or null): the
// largest |y| as stored is merged into it (an FP8 operand's scale).
template <typename T, int VPL>
__global__ void __launch_bounds__(LN_FWD_WARPS * 32) ln_fwd_kernel(T* __restrict__ y, float* __restrict__ mean,
                                                                   float* __restrict__ rstd, T* __restrict__ xsum,
                                                                   const T* __restrict__ x, const T* __restrict__ r,
                                                                   const T* __restrict__ gamma,
                                                                   const T* __restrict__ beta, int N, int C,
                                                                   unsigned* __restrict__ amax) {
    const int row = blockIdx.x * LN_FWD_WARPS + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= N) return;  // the whole warp
    const int cv = C / 8;
    const T* xr = x + (int64_t)row * C;
    float v[VPL][8];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int idx = lane + 32 * i;
        if (idx < cv) {
            load8_stream(xr + idx * 8, v[i]);
            if (r) {
                float u[8];
                load8_stream(r + (int64_t)row * C + idx * 8, u);
#pragma unroll
                for (int j = 0; j < 8; j++) v[i][j] = to_float(from_float<T>(v[i][j] + u[j]));
                store8(xsum + (int64_t)row * C + idx * 8, v[i]);
            }
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
    float am = 0.f;
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
            if (amax) {
#pragma unroll
                for (int j = 0; j < 8; j++) am = fmaxf(am, fabsf(o[j]));
            }
        }
    }
    if (lane == 0) {
        mean[row] = mu;
        rstd[row] = rs;
    }
    if (amax) amax_merge(amax, am);
}

// The same forward arranged like the staged backward: a persistent grid,
// warps striding over rows, each with a ring of LN_STAGES row slots in shared
// memory (x, and r when given) that cp.async fills LN_STAGES - 1 rows ahead,
// so that loads stay in flight while rows are normalised. A lane copies and
// reads only its own 16-byte pieces. Same arithmetic as ln_fwd_kernel.
#define LN_FWD_STAGED_WARPS 8
template <typename T, int VPL>
__global__ void __launch_bounds__(LN_FWD_STAGED_WARPS * 32)
    ln_fwd_staged_kernel(T* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd, T* __restrict__ xsum,
                         const T* __restrict__ x, const T* __restrict__ r, const T* __restrict__ gamma,
                         const T* __restrict__ beta, int N, int C, unsigned* __restrict__ amax) {
    extern __shared__ __align__(16) uint8_t sm_raw[];
    constexpr int PIECES = (int)sizeof(T) / 2;  // 16-byte copies per 8-element vector
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cv = C / 8;
    const size_t row_bytes = (size_t)C * sizeof(T);
    const size_t slot_bytes = 2 * row_bytes;  // x | r
    uint8_t* ring = sm_raw + (size_t)w * LN_STAGES * slot_bytes;
    const int stride = gridDim.x * LN_FWD_STAGED_WARPS;
    const int row0 = blockIdx.x * LN_FWD_STAGED_WARPS + w;
    auto issue = [&](int row, int slot) {
        if (row < N) {
            uint8_t* sb = ring + (size_t)slot * slot_bytes;
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int idx = lane + 32 * i;
                if (idx < cv) {
#pragma unroll
                    for (int p = 0; p < PIECES; p++) {
                        const size_t off = (size_t)idx * 8 * sizeof(T) + p * 16;
                        const size_t goff = ((size_t)row * C + idx * 8) * sizeof(T) + p * 16;
                        cp_async16(sb + off, (const uint8_t*)x + goff);
                        if (r) cp_async16(sb + row_bytes + off, (const uint8_t*)r + goff);
                    }
                }
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < LN_STAGES - 1; k++) issue(row0 + k * stride, k);
    int slot = 0;
    float am = 0.f;  // largest |y| of this lane (amax)
    for (int row = row0; row < N; row += stride) {
        __syncwarp();
        issue(row + (LN_STAGES - 1) * stride, (slot + LN_STAGES - 1) % LN_STAGES);
        cp_async_wait<LN_STAGES - 1>();  // this lane's pieces of the row have landed
        const uint8_t* sb = ring + (size_t)slot * slot_bytes;
        const T* sx = reinterpret_cast<const T*>(sb);
        const T* sr = reinterpret_cast<const T*>(sb + row_bytes);
        float v[VPL][8];
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                load8(sx + idx * 8, v[i]);
                if (r) {
                    float u[8];
                    load8(sr + idx * 8, u);
#pragma unroll
                    for (int j = 0; j < 8; j++) v[i][j] = to_float(from_float<T>(v[i][j] + u[j]));
                    store8(xsum + (int64_t)row * C + idx * 8, v[i]);
                }
#pragma unroll
                for (int j = 0; j < 8; j++) sum += v[i][j];
            }
        }
        const float mu = warp_sum(sum) / (float)C;
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
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                float g[8], b[8], o[8];
                load8(gamma + idx * 8, g);
                load8(beta + idx * 8, b);
#pragma unroll
                for (int j = 0; j < 8; j++) o[j] = (v[i][j] - mu) * rs * g[j] + b[j];
                store8(y + (int64_t)row * C + idx * 8, o);
                if (amax) {
#pragma unroll
                    for (int j = 0; j < 8; j++) am = fmaxf(am, fabsf(o[j]));
                }
            }
        }
        if (lane == 0) {
            mean[row] = mu;
            rstd[row] = rs;
        }
        slot = (slot + 1) % LN_STAGES;
    }
    cp_async_wait<0>();
    if (amax) amax_merge(amax, am);
}

// dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat)), dxhat = dy gamma.
// Warp per row, rows strided over a fixed grid; the next row's x and dy are
// loaded (raw) before the current row is computed. Each warp accumulates
// dy*xhat and dy (and, with np == 3, the values it writes) for its lane's
// columns in its own shared-memory rows (no two threads touch the same word;
// column idx*8+j at word j*(C/8)+idx, so a warp's accesses hit 32 distinct
// banks). The block then sums its warps in order into
// partial[block][0..np*C); a column reduce finishes dgamma, dbeta (and the
// column sums of the output, which are the bias gradient of the linear layer
// that reads this gradient next).
// Output: with res == null, out = dx; otherwise res += dx in place (the
// residual join of the backward pass), and out = res.
template <typename T, int VPL>
__global__ void __launch_bounds__(LN_BWD_WARPS * 32, VPL <= 3 ? 2 : 1)
    ln_bwd_kernel(T* __restrict__ out, bool accumulate, float* __restrict__ partial, int np,
                  const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
                  const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C,
                  unsigned* __restrict__ amax) {
    float am = 0.f;  // largest |out| of this lane (amax)
    extern __shared__ float sh[];  // [LN_BWD_WARPS][np][C]
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cv = C / 8;
    float* acc_g = sh + (size_t)w * np * C;
    float* acc_b = acc_g + C;
    float* acc_o = acc_b + C;  // used when np == 3
    for (int c = lane; c < np * C; c += 32) acc_g[c] = 0.f;
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
                if (accumulate) {  // the residual gradient this row's result is added to
                    float rv[8];
                    load8(out + (int64_t)row * C + idx * 8, rv);
#pragma unroll
                    for (int j = 0; j < 8; j++) o[j] += rv[j];
                }
                store8(out + (int64_t)row * C + idx * 8, o);
                if (np == 3) {
#pragma unroll
                    for (int j = 0; j < 8; j++) acc_o[j * cv + idx] += to_float(from_float<T>(o[j]));
                }
                if (amax) {
#pragma unroll
                    for (int j = 0; j < 8; j++) am = fmaxf(am, fabsf(o[j]));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            rx[i] = nx[i];
            rd[i] = nd[i];
        }
        row = next;
    }
    if (amax) amax_merge(amax, am);
    __syncthreads();
    for (int a = threadIdx.x; a < np * C; a += blockDim.x) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < LN_BWD_WARPS; k++) sum += sh[(size_t)k * np * C + a];
        const int q = a / C, e = a % C;  // which array; element within it
        const int c = (e % cv) * 8 + e / cv;
        partial[(size_t)blockIdx.x * np * C + (size_t)q * C + c] = sum;
    }
}

// The same backward for C <= 1024 (VPL <= 4), arranged for memory-level
// parallelism: each warp keeps a ring of LN_STAGES row slots in shared memory
// that cp.async fills (x, dy, the residual gradient when accumulating, mean,
// rstd), LN_STAGES - 1 rows ahead of the row it computes. A lane copies and
// reads only its own 16-byte pieces of a row (plus lane 0's mean and rstd,
// read after a warp barrier). The per-column sums are register accumulators
// of the lane that owns the column; at the end the warps' sums go through
// shared memory and are added in warp order into partial[block].

template <typename T, int VPL>
__global__ void __launch_bounds__(LN_BWD_WARPS * 32, 2)
    ln_bwd_staged_kernel(T* __restrict__ out, bool accumulate, float* __restrict__ partial, int np,
                         const T* __restrict__ dy, const T* __restrict__ x, const T* __restrict__ gamma,
                         const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C) {
    extern __shared__ __align__(16) uint8_t sm_raw[];
    constexpr int PIECES = (int)sizeof(T) / 2;  // 16-byte copies per 8-element vector
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cv = C / 8;
    const size_t row_bytes = (size_t)C * sizeof(T);
    const size_t slot_bytes = 3 * row_bytes + 16;  // x | dy | residual gradient | mean, rstd
    uint8_t* ring = sm_raw + (size_t)w * LN_STAGES * slot_bytes;
    const int stride = gridDim.x * LN_BWD_WARPS;
    const int row0 = blockIdx.x * LN_BWD_WARPS + w;

    auto issue = [&](int row, int slot) {
        if (row < N) {
            uint8_t* sb = ring + (size_t)slot * slot_bytes;
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int idx = lane + 32 * i;
                if (idx < cv) {
#pragma unroll
                    for (int p = 0; p < PIECES; p++) {
                        const size_t off = (size_t)idx * 8 * sizeof(T) + p * 16;
                        const size_t goff = ((size_t)row * C + idx * 8) * sizeof(T) + p * 16;
                        cp_async16(sb + off, (const uint8_t*)x + goff);
                        cp_async16(sb + row_bytes + off, (const uint8_t*)dy + goff);
                        if (accumulate) cp_async16(sb + 2 * row_bytes + off, (const uint8_t*)out + goff);
                    }
                }
            }
            if (lane == 0) {
                cp_async4(sb + 3 * row_bytes, mean + row);
                cp_async4(sb + 3 * row_bytes + 4, rstd + row);
            }
        }
        cp_async_commit();  // one group per row slot, empty past the end
    };

    float ag[VPL][8], ab[VPL][8], ao[VPL][8];
#pragma unroll
    for (int i = 0; i < VPL; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) ag[i][j] = ab[i][j] = ao[i][j] = 0.f;

#pragma unroll
    for (int k = 0; k < LN_STAGES - 1; k++) issue(row0 + k * stride, k);
    int slot = 0;
    for (int row = row0; row < N; row += stride) {
        // refill the slot read in the previous iteration (all lanes are done with it)
        __syncwarp();
        issue(row + (LN_STAGES - 1) * stride, (slot + LN_STAGES - 1) % LN_STAGES);
        cp_async_wait<LN_STAGES - 1>();  // this row's group has landed
        __syncwarp();                     // ... for every lane (mean and rstd come from lane 0)
        const uint8_t* sb = ring + (size_t)slot * slot_bytes;
        const T* sx = reinterpret_cast<const T*>(sb);
        const T* sdy = reinterpret_cast<const T*>(sb + row_bytes);
        const T* sres = reinterpret_cast<const T*>(sb + 2 * row_bytes);
        const float mu = reinterpret_cast<const float*>(sb + 3 * row_bytes)[0];
        const float rs = reinterpret_cast<const float*>(sb + 3 * row_bytes)[1];
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                float xv[8], dv[8], g[8];
                load8(sx + idx * 8, xv);
                load8(sdy + idx * 8, dv);
                load8(gamma + idx * 8, g);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float xh = (xv[j] - mu) * rs;
                    ag[i][j] += dv[j] * xh;
                    ab[i][j] += dv[j];
                    const float dh = dv[j] * g[j];
                    s1 += dh;
                    s2 += dh * xh;
                }
            }
        }
        const float m1 = warp_sum(s1) / (float)C;
        const float m2 = warp_sum(s2) / (float)C;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                float xv[8], dv[8], g[8], o[8];
                load8(sx + idx * 8, xv);
                load8(sdy + idx * 8, dv);
                load8(gamma + idx * 8, g);
#pragma unroll
                for (int j = 0; j < 8; j++) o[j] = rs * (dv[j] * g[j] - m1 - (xv[j] - mu) * rs * m2);
                if (accumulate) {
                    float rv[8];
                    load8(sres + idx * 8, rv);
#pragma unroll
                    for (int j = 0; j < 8; j++) o[j] += rv[j];
                }
                store8(out + (int64_t)row * C + idx * 8, o);
                if (np == 3) {
#pragma unroll
                    for (int j = 0; j < 8; j++) ao[i][j] += to_float(from_float<T>(o[j]));
                }
            }
        }
        slot = (slot + 1) % LN_STAGES;
    }
    cp_async_wait<0>();
    __syncthreads();
    // the warps' column sums, [warp][np][C] over the ring's memory, then summed in warp order
    float* red = reinterpret_cast<float*>(sm_raw);
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int idx = lane + 32 * i;
        if (idx < cv) {
#pragma unroll
            for (int j = 0; j < 8; j++) {
                float* r = red + (size_t)w * np * C + idx * 8 + j;
                r[0] = ag[i][j];
                r[C] = ab[i][j];
                if (np == 3) r[2 * C] = ao[i][j];
            }
        }
    }
    __syncthreads();
    for (int a = threadIdx.x; a < np * C; a += blockDim.x) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < LN_BWD_WARPS; k++) sum += red[(size_t)k * np * C + a];
        partial[(size_t)blockIdx.x * np * C + a] = sum;
    }
}

// bf16 pair (element 0 in the low half) to an fp32 pair.
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) { return tc::f2_pack(w << 16, w & 0xffff0000u); }

// The bf16 staged backward with paired fp32 arithmetic (f32x2): the same ring
// and the same per-element formulas as ln_bwd_staged_kernel, two columns per
// instruction; gamma is held in shared memory as fp32 for the block. Column
// pairs (2p, 2p+1) of a lane's 8-vector sit in one 64-bit accumulator.
template <int VPL, int STG = LN_STAGES>
__global__ void __launch_bounds__(LN_BWD_WARPS * 32, 2)
    ln_bwd_bf16_kernel(bf16* __restrict__ out, bool accumulate, float* __restrict__ partial, int np,
                       const bf16* __restrict__ dy, const bf16* __restrict__ x, const bf16* __restrict__ gamma,
                       const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C,
                       unsigned* __restrict__ amax) {
    float am = 0.f;  // largest |out| of this lane (amax)
    using namespace tc;
    extern __shared__ __align__(16) uint8_t sm_raw[];
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int cv = C / 8;
    const size_t g_bytes = ((size_t)C * 4 + 15) & ~(size_t)15;
    float* sg = reinterpret_cast<float*>(sm_raw);  // gamma, fp32
    const size_t row_bytes = (size_t)C * 2;
    const size_t slot_bytes = 3 * row_bytes + 16;  // x | dy | residual gradient | mean, rstd
    uint8_t* ring = sm_raw + g_bytes + (size_t)w * STG * slot_bytes;
    const int stride = gridDim.x * LN_BWD_WARPS;
    const int row0 = blockIdx.x * LN_BWD_WARPS + w;
    for (int c = threadIdx.x; c < C; c += blockDim.x) sg[c] = __bfloat162float(gamma[c]);

    auto issue = [&](int row, int slot) {
        if (row < N) {
            uint8_t* sb = ring + (size_t)slot * slot_bytes;
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int idx = lane + 32 * i;
                if (idx < cv) {
                    const size_t off = (size_t)idx * 16, goff = ((size_t)row * C + idx * 8) * 2;
                    cp_async16(sb + off, (const uint8_t*)x + goff);
                    cp_async16(sb + row_bytes + off, (const uint8_t*)dy + goff);
                    if (accumulate) cp_async16(sb + 2 * row_bytes + off, (const uint8_t*)out + goff);
                }
            }
            if (lane == 0) {
                cp_async4(sb + 3 * row_bytes, mean + row);
                cp_async4(sb + 3 * row_bytes + 4, rstd + row);
            }
        }
        cp_async_commit();
    };

    uint64_t ag[VPL][4], ab[VPL][4], ao[VPL][4];
#pragma unroll
    for (int i = 0; i < VPL; i++)
#pragma unroll
        for (int p = 0; p < 4; p++) ag[i][p] = ab[i][p] = ao[i][p] = 0;
    __syncthreads();  // gamma staged

#pragma unroll
    for (int k = 0; k < STG - 1; k++) issue(row0 + k * stride, k);
    int slot = 0;
    for (int row = row0; row < N; row += stride) {
        __syncwarp();
        issue(row + (STG - 1) * stride, (slot + STG - 1) % STG);
        cp_async_wait<STG - 1>();
        __syncwarp();
        const uint8_t* sb = ring + (size_t)slot * slot_bytes;
        const float mu = reinterpret_cast<const float*>(sb + 3 * row_bytes)[0];
        const float rs = reinterpret_cast<const float*>(sb + 3 * row_bytes)[1];
        const uint64_t rs2 = f2_pack(rs, rs), nmr2 = f2_pack(-mu * rs, -mu * rs);
        uint64_t s1 = 0, s2 = 0;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                const uint4 xr = *reinterpret_cast<const uint4*>(sb + idx * 16);
                const uint4 dr = *reinterpret_cast<const uint4*>(sb + row_bytes + idx * 16);
                const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w}, dw[4] = {dr.x, dr.y, dr.z, dr.w};
                const uint64_t* g2 = reinterpret_cast<const uint64_t*>(sg + idx * 8);
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    const uint64_t x2 = bf2_to_f2(xw[p]), d2 = bf2_to_f2(dw[p]);
                    const uint64_t xh = f2_fma(x2, rs2, nmr2);
                    ag[i][p] = f2_fma(d2, xh, ag[i][p]);
                    ab[i][p] = f2_add(ab[i][p], d2);
                    const uint64_t dh = f2_mul(d2, g2[p]);
                    s1 = f2_add(s1, dh);
                    s2 = f2_fma(dh, xh, s2);
                }
            }
        }
        float a0, a1, b0, b1;
        f2_unpack(s1, a0, a1);
        f2_unpack(s2, b0, b1);
        const float m1 = warp_sum(a0 + a1) / (float)C;
        const float m2 = warp_sum(b0 + b1) / (float)C;
        const uint64_t m1_2 = f2_pack(m1, m1), m2_2 = f2_pack(m2, m2);
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                const uint4 xr = *reinterpret_cast<const uint4*>(sb + idx * 16);
                const uint4 dr = *reinterpret_cast<const uint4*>(sb + row_bytes + idx * 16);
                uint4 rr = make_uint4(0, 0, 0, 0);
                if (accumulate) rr = *reinterpret_cast<const uint4*>(sb + 2 * row_bytes + idx * 16);
                const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w}, dw[4] = {dr.x, dr.y, dr.z, dr.w};
                const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
                const uint64_t* g2 = reinterpret_cast<const uint64_t*>(sg + idx * 8);
                uint32_t ow[4];
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    const uint64_t xh = f2_fma(bf2_to_f2(xw[p]), rs2, nmr2);
                    const uint64_t dh = f2_mul(bf2_to_f2(dw[p]), g2[p]);
                    // rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat))
                    uint64_t o = f2_mul(rs2, f2_sub(dh, f2_fma(xh, m2_2, m1_2)));
                    if (accumulate) o = f2_add(o, bf2_to_f2(rw[p]));
                    float o0, o1;
                    f2_unpack(o, o0, o1);
                    if (amax) am = fmaxf(am, fmaxf(fabsf(o0), fabsf(o1)));
                    __nv_bfloat162 h = __floats2bfloat162_rn(o0, o1);
                    ow[p] = *reinterpret_cast<uint32_t*>(&h);
                    if (np == 3) ao[i][p] = f2_add(ao[i][p], bf2_to_f2(ow[p]));
                }
                *reinterpret_cast<uint4*>(out + (int64_t)row * C + idx * 8) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
        }
        slot = (slot + 1) % STG;
    }
    if (amax) amax_merge(amax, am);
    cp_async_wait<0>();
    __syncthreads();
    float* red = reinterpret_cast<float*>(sm_raw + g_bytes);  // [warp][np][C] over the rings
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int idx = lane + 32 * i;
        if (idx < cv) {
#pragma unroll
            for (int p = 0; p < 4; p++) {
                float* r = red + (size_t)w * np * C + idx * 8 + 2 * p;
                f2_unpack(ag[i][p], r[0], r[1]);
                f2_unpack(ab[i][p], r[C], r[C + 1]);
                if (np == 3) f2_unpack(ao[i][p], r[2 * C], r[2 * C + 1]);
            }
        }
    }
    __syncthreads();
    for (int a = threadIdx.x; a < np * C; a += blockDim.x) {
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < LN_BWD_WARPS; k++) sum += red[(size_t)k * np * C + a];
        partial[(size_t)blockIdx.x * np * C + a] = sum;
    }
}

// Wide rows (bf16, C from 1032 to 2048 values, beyond the staged forms: the
// 1.5B model's 1600), where a warp per row leaves each lane 40 or more columns
// of accumulators: a block of LN_WIDE_THREADS threads takes a group of rows at a
// time, and thread t owns the 8 columns of vector t of every row, so its
// column sums stay in registers and no block merges them across warps. A
// group's row sums go through one block reduction per quantity: warp
// shuffles, then the warps' values from shared memory added in warp order
// (double-buffered by group, so one barrier a reduction suffices). Each
// thread copies its own 16-byte pieces of the rows LN_WIDE_S - 1 groups ahead
// into a ring in shared memory (cp.async) and reads only those, so the ring
// needs no barrier and loads stay in flight through the reductions. Same
// formulas as the other forms; a row's sums are added in a different order,
// so results differ from them in the last bits.
#define LN_WIDE_THREADS 256
#define LN_WIDE_WARPS (LN_WIDE_THREADS / 32)
#define LN_WIDE_R 4      // rows a group, forward
#define LN_WIDE_R_BWD 2  // rows a group, backward
#define LN_WIDE_S 3      // groups in a block's ring
// ring bytes of a block: LN_WIDE_S groups x rows x pieces (forward: x, r;
// backward: x, dy, the residual gradient, mean and rstd) x threads x 16
#define LN_WIDE_FWD_SMEM (LN_WIDE_S * LN_WIDE_R * 2 * LN_WIDE_THREADS * 16)
#define LN_WIDE_BWD_SMEM (LN_WIDE_S * LN_WIDE_R_BWD * 4 * LN_WIDE_THREADS * 16)

// The R sums of this thread, summed over the block, into v[] (every thread
// gets them). red: this call's [LN_WIDE_WARPS][R] buffer, not written again
// before the block's next barrier.
template <int R>
__device__ __forceinline__ void ln_wide_block_sum(float (&v)[R], float* red) {
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
#pragma unroll
    for (int k = 0; k < R; k++) v[k] = warp_sum(v[k]);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < R; k++) red[w * R + k] = v[k];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < R; k++) {
        float t = 0.f;
#pragma unroll
        for (int ww = 0; ww < LN_WIDE_WARPS; ww++) t += red[ww * R + k];
        v[k] = t;
    }
}

__global__ void __launch_bounds__(LN_WIDE_THREADS, 2)
    ln_fwd_wide_kernel(bf16* __restrict__ y, float* __restrict__ mean, float* __restrict__ rstd,
                       bf16* __restrict__ xsum, const bf16* __restrict__ x, const bf16* __restrict__ r,
                       const bf16* __restrict__ gamma, const bf16* __restrict__ beta, int N, int C,
                       unsigned* __restrict__ amax) {
    constexpr int R = LN_WIDE_R, S = LN_WIDE_S;
    extern __shared__ __align__(16) uint8_t wring[];  // [S][R][x | r][threads][16 B]
    __shared__ float red[4][LN_WIDE_WARPS * R];       // two reductions a group, double-buffered by group
    const int t = threadIdx.x;
    const bool own = t < C / 8;                       // this thread's vector is inside the row
    auto piece = [&](int slot, int q, int a) { return wring + ((size_t)((slot * R + q) * 2 + a) * LN_WIDE_THREADS + t) * 16; };
    const int gstride = gridDim.x * R;
    auto issue = [&](int r0, int slot) {
        if (own) {
#pragma unroll
            for (int q = 0; q < R; q++) {
                const int row = r0 + q;
                if (row < N) {
                    cp_async16(piece(slot, q, 0), x + (int64_t)row * C + t * 8);
                    if (r) cp_async16(piece(slot, q, 1), r + (int64_t)row * C + t * 8);
                }
            }
        }
        cp_async_commit();
    };
    float g[8], b[8];
    if (own) {
        load8(gamma + t * 8, g);
        load8(beta + t * 8, b);
    }
    const int g0 = blockIdx.x * R;
#pragma unroll
    for (int k = 0; k < S - 1; k++) issue(g0 + k * gstride, k);
    float am = 0.f;  // largest |y| of this thread (amax)
    int slot = 0, it = 0;
    for (int r0 = g0; r0 < N; r0 += gstride, it ^= 1) {
        issue(r0 + (S - 1) * gstride, (slot + S - 1) % S);
        cp_async_wait<S - 1>();  // this thread's pieces of the group have landed
        float v[R][8];
#pragma unroll
        for (int q = 0; q < R; q++) {
            const int row = r0 + q;
            if (own && row < N) {
                load8(reinterpret_cast<const bf16*>(piece(slot, q, 0)), v[q]);
                if (r) {
                    float u[8];
                    load8(reinterpret_cast<const bf16*>(piece(slot, q, 1)), u);
#pragma unroll
                    for (int j = 0; j < 8; j++) v[q][j] = to_float(from_float<bf16>(v[q][j] + u[j]));
                    store8(xsum + (int64_t)row * C + t * 8, v[q]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++) v[q][j] = 0.f;
            }
        }
        float mu[R];
#pragma unroll
        for (int q = 0; q < R; q++) {
            float sum = 0.f;
#pragma unroll
            for (int j = 0; j < 8; j++) sum += v[q][j];
            mu[q] = sum;
        }
        ln_wide_block_sum<R>(mu, red[2 * it]);
        float rs[R];
#pragma unroll
        for (int q = 0; q < R; q++) {
            mu[q] /= (float)C;
            float ss = 0.f;
            if (own) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float d = v[q][j] - mu[q];
                    ss += d * d;
                }
            }
            rs[q] = ss;
        }
        ln_wide_block_sum<R>(rs, red[2 * it + 1]);
#pragma unroll
        for (int q = 0; q < R; q++) {
            const int row = r0 + q;
            rs[q] = 1.0f / sqrtf(rs[q] / (float)C + LN_EPS);
            if (row >= N) continue;
            if (own) {
                float o[8];
#pragma unroll
                for (int j = 0; j < 8; j++) o[j] = (v[q][j] - mu[q]) * rs[q] * g[j] + b[j];
                store8(y + (int64_t)row * C + t * 8, o);
                if (amax) {
#pragma unroll
                    for (int j = 0; j < 8; j++) am = fmaxf(am, fabsf(o[j]));
                }
            }
            if (t == 0) {
                mean[row] = mu[q];
                rstd[row] = rs[q];
            }
        }
        slot = (slot + 1) % S;
    }
    cp_async_wait<0>();
    if (amax) amax_merge(amax, am);
}

__global__ void __launch_bounds__(LN_WIDE_THREADS, 2)
    ln_bwd_wide_kernel(bf16* __restrict__ out, bool accumulate, float* __restrict__ partial, int np,
                       const bf16* __restrict__ dy, const bf16* __restrict__ x, const bf16* __restrict__ gamma,
                       const float* __restrict__ mean, const float* __restrict__ rstd, int N, int C,
                       unsigned* __restrict__ amax) {
    using namespace tc;
    constexpr int R = LN_WIDE_R_BWD, S = LN_WIDE_S;
    extern __shared__ __align__(16) uint8_t wring[];  // [S][R][x | dy | residual gradient | mean, rstd][threads][16 B]
    __shared__ float red[2][LN_WIDE_WARPS * 2 * R];   // one reduction a group, double-buffered by group
    const int t = threadIdx.x;
    const bool own = t < C / 8;
    auto piece = [&](int slot, int q, int a) { return wring + ((size_t)((slot * R + q) * 4 + a) * LN_WIDE_THREADS + t) * 16; };
    const int gstride = gridDim.x * R;
    auto issue = [&](int r0, int slot) {
        if (own) {
#pragma unroll
            for (int q = 0; q < R; q++) {
                const int row = r0 + q;
                if (row < N) {
                    const int64_t off = (int64_t)row * C + t * 8;
                    cp_async16(piece(slot, q, 0), x + off);
                    cp_async16(piece(slot, q, 1), dy + off);
                    if (accumulate) cp_async16(piece(slot, q, 2), out + off);
                    cp_async4(piece(slot, q, 3), mean + row);
                    cp_async4(piece(slot, q, 3) + 4, rstd + row);
                }
            }
        }
        cp_async_commit();
    };
    uint64_t g2[4], ag[4], ab[4], ao[4];
    {
        uint4 gr = make_uint4(0, 0, 0, 0);
        if (own) gr = *reinterpret_cast<const uint4*>(gamma + t * 8);
        const uint32_t gw[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
        for (int p = 0; p < 4; p++) {
            g2[p] = bf2_to_f2(gw[p]);
            ag[p] = ab[p] = ao[p] = 0;
        }
    }
    const int g0 = blockIdx.x * R;
#pragma unroll
    for (int k = 0; k < S - 1; k++) issue(g0 + k * gstride, k);
    float am = 0.f;  // largest |out| of this thread (amax)
    int slot = 0, it = 0;
    for (int r0 = g0; r0 < N; r0 += gstride, it ^= 1) {
        issue(r0 + (S - 1) * gstride, (slot + S - 1) % S);
        cp_async_wait<S - 1>();
        // the row sums of dxhat = dy gamma and of dxhat xhat
        float s[2 * R];
#pragma unroll
        for (int q = 0; q < R; q++) {
            s[2 * q] = s[2 * q + 1] = 0.f;
            if (own && r0 + q < N) {
                const float* mr = reinterpret_cast<const float*>(piece(slot, q, 3));
                const float mu = mr[0], rs = mr[1];
                const uint64_t rs2 = f2_pack(rs, rs), nmr2 = f2_pack(-mu * rs, -mu * rs);
                const uint4 xr = *reinterpret_cast<const uint4*>(piece(slot, q, 0));
                const uint4 dr = *reinterpret_cast<const uint4*>(piece(slot, q, 1));
                const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w}, dw[4] = {dr.x, dr.y, dr.z, dr.w};
                uint64_t s1 = 0, s2 = 0;
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    const uint64_t xh = f2_fma(bf2_to_f2(xw[p]), rs2, nmr2);
                    const uint64_t dh = f2_mul(bf2_to_f2(dw[p]), g2[p]);
                    s1 = f2_add(s1, dh);
                    s2 = f2_fma(dh, xh, s2);
                }
                float a0, a1, b0, b1;
                f2_unpack(s1, a0, a1);
                f2_unpack(s2, b0, b1);
                s[2 * q] = a0 + a1;
                s[2 * q + 1] = b0 + b1;
            }
        }
        ln_wide_block_sum<2 * R>(s, red[it]);
#pragma unroll
        for (int q = 0; q < R; q++) {
            const int row = r0 + q;
            if (!own || row >= N) continue;
            const float m1 = s[2 * q] / (float)C, m2 = s[2 * q + 1] / (float)C;
            const float* mr = reinterpret_cast<const float*>(piece(slot, q, 3));
            const float mu = mr[0], rs = mr[1];
            const uint64_t rs2 = f2_pack(rs, rs), nmr2 = f2_pack(-mu * rs, -mu * rs);
            const uint64_t m1_2 = f2_pack(m1, m1), m2_2 = f2_pack(m2, m2);
            const uint4 xr = *reinterpret_cast<const uint4*>(piece(slot, q, 0));
            const uint4 dr = *reinterpret_cast<const uint4*>(piece(slot, q, 1));
            uint4 rr = make_uint4(0, 0, 0, 0);
            if (accumulate) rr = *reinterpret_cast<const uint4*>(piece(slot, q, 2));
            const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w}, dw[4] = {dr.x, dr.y, dr.z, dr.w};
            const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
            uint32_t ow[4];
#pragma unroll
            for (int p = 0; p < 4; p++) {
                const uint64_t d2 = bf2_to_f2(dw[p]);
                const uint64_t xh = f2_fma(bf2_to_f2(xw[p]), rs2, nmr2);
                ag[p] = f2_fma(d2, xh, ag[p]);
                ab[p] = f2_add(ab[p], d2);
                const uint64_t dh = f2_mul(d2, g2[p]);
                // rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat))
                uint64_t o = f2_mul(rs2, f2_sub(dh, f2_fma(xh, m2_2, m1_2)));
                if (accumulate) o = f2_add(o, bf2_to_f2(rw[p]));
                float o0, o1;
                f2_unpack(o, o0, o1);
                if (amax) am = fmaxf(am, fmaxf(fabsf(o0), fabsf(o1)));
                __nv_bfloat162 h = __floats2bfloat162_rn(o0, o1);
                ow[p] = *reinterpret_cast<uint32_t*>(&h);
                if (np == 3) ao[p] = f2_add(ao[p], bf2_to_f2(ow[p]));
            }
            *reinterpret_cast<uint4*>(out + (int64_t)row * C + t * 8) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        }
        slot = (slot + 1) % S;
    }
    cp_async_wait<0>();
    if (amax) amax_merge(amax, am);
    // this thread's column sums: partial[block][q * C + column]
    if (own) {
        float* pb = partial + (size_t)blockIdx.x * np * C;
        float vg[8], vb[8], vo[8];
#pragma unroll
        for (int p = 0; p < 4; p++) {
            f2_unpack(ag[p], vg[2 * p], vg[2 * p + 1]);
            f2_unpack(ab[p], vb[2 * p], vb[2 * p + 1]);
            f2_unpack(ao[p], vo[2 * p], vo[2 * p + 1]);
        }
        store8(pb + t * 8, vg);
        store8(pb + C + t * 8, vb);
        if (np == 3) store8(pb + 2 * C + t * 8, vo);
    }
}

// The wide-row forms (bf16, rows of LN_WIDE_MIN_C to 8 * LN_WIDE_THREADS
// values): two resident blocks per SM. At C = 1024 the staged forms measured
// faster (forward 1.52 against 1.99 ms per step of the 350M model at B = 16,
// backward equal); at C = 1600 the wide ones (1.5B at B = 8: forward 2.74
// against 3.25 ms, backward 3.60 against 9.59).
#define LN_WIDE_MIN_C 1025
static bool ln_wide(int dtype, int C) {
    return dtype == GPT2_MODE_BF16 && C >= LN_WIDE_MIN_C && C <= 8 * LN_WIDE_THREADS;
}
static int ln_wide_blocks(int N, int rows = LN_WIDE_R) {
    const int cap = 2 * gpt2_num_sms();
    const int b = (N + rows - 1) / rows;
    return b < cap ? (b < 1 ? 1 : b) : cap;
}

static size_t ln_staged_smem(int dtype, int C) {
    const size_t es = dtype == GPT2_MODE_BF16 ? 2 : 4;
    return (size_t)LN_BWD_WARPS * LN_STAGES * (3 * C * es + 16);
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

template <typename T, int VPL>
static void ln_fwd_staged_launch(int blocks, size_t smem, void* y, float* mean, float* rstd, void* xsum,
                                 const void* x, const void* r, const void* gamma, const void* beta, int N, int C,
                                 cudaStream_t s, unsigned* amax) {
    smem_attr((const void*)ln_fwd_staged_kernel<T, VPL>,
              LN_FWD_STAGED_WARPS * LN_STAGES * 2 * LN_STAGED_MAX_ROW_BYTES);
    ln_fwd_staged_kernel<T, VPL><<<blocks, LN_FWD_STAGED_WARPS * 32, smem, s>>>(
        (T*)y, mean, rstd, (T*)xsum, (const T*)x, (const T*)r, (const T*)gamma, (const T*)beta, N, C, amax);
}

static int ln_forward(int dtype, void* y, float* mean, float* rstd, void* xsum, const void* x, const void* r,
                      const void* gamma, const void* beta, int N, int C, cudaStream_t s, unsigned* amax) {
    const int blocks = (N + LN_FWD_WARPS - 1) / LN_FWD_WARPS;
    if (blocks == 0) return 0;
    if (ln_wide(dtype, C)) {
        smem_attr((const void*)ln_fwd_wide_kernel, LN_WIDE_FWD_SMEM);
        ln_fwd_wide_kernel<<<ln_wide_blocks(N), LN_WIDE_THREADS, LN_WIDE_FWD_SMEM, s>>>(
            (bf16*)y, mean, rstd, (bf16*)xsum, (const bf16*)x, (const bf16*)r, (const bf16*)gamma, (const bf16*)beta,
            N, C, amax);
        return 1;
    }
    const size_t es = dtype == GPT2_MODE_BF16 ? 2 : 4;
    if ((size_t)C * es <= LN_STAGED_MAX_ROW_BYTES) {
        // three blocks of 8 warps per SM (74 KB of ring each at C = 768 bf16)
        const size_t smem = (size_t)LN_FWD_STAGED_WARPS * LN_STAGES * 2 * C * es;
        int sblocks = 3 * gpt2_num_sms();
        const int need = (N + LN_FWD_STAGED_WARPS - 1) / LN_FWD_STAGED_WARPS;
        if (sblocks > need) sblocks = need;
#define LN_FWD_STAGED_CALL(V)                                                                                     \
    if (dtype == GPT2_MODE_BF16)                                                                                  \
        ln_fwd_staged_launch<bf16, V>(sblocks, smem, y, mean, rstd, xsum, x, r, gamma, beta, N, C, s, amax);     \
    else                                                                                                          \
        ln_fwd_staged_launch<float, V>(sblocks, smem, y, mean, rstd, xsum, x, r, gamma, beta, N, C, s, amax);
        switch (ln_vpl(C)) {
            case 1: LN_FWD_STAGED_CALL(1); break;
            case 2: LN_FWD_STAGED_CALL(2); break;
            case 3: LN_FWD_STAGED_CALL(3); break;
            default: LN_FWD_STAGED_CALL(4); break;
        }
#undef LN_FWD_STAGED_CALL
        return 1;
    }
#define LN_FWD_CALL(V)                                                                                            \
    if (dtype == GPT2_MODE_BF16)                                                                                  \
        ln_fwd_kernel<bf16, V><<<blocks, LN_FWD_WARPS * 32, 0, s>>>((bf16*)y, mean, rstd, (bf16*)xsum,            \
                                                                    (const bf16*)x, (const bf16*)r,               \
                                                                    (const bf16*)gamma, (const bf16*)beta, N, C,  \
                                                                    amax);                                        \
    else                                                                                                          \
        ln_fwd_kernel<float, V><<<blocks, LN_FWD_WARPS * 32, 0, s>>>((float*)y, mean, rstd, (float*)xsum,         \
                                                                     (const float*)x, (const float*)r,            \
                                                                     (const float*)gamma, (const float*)beta, N,  \
                                                                     C, amax);
    LN_DISPATCH(ln_vpl(C), LN_FWD_CALL)
#undef LN_FWD_CALL
    return 1;
}

int launch_layernorm_forward(int dtype, void* y, float* mean, float* rstd, const void* x, const void* gamma,
                             const void* beta, int N, int C, cudaStream_t s, unsigned* amax) {
    return ln_forward(dtype, y, mean, rstd, nullptr, x, nullptr, gamma, beta, N, C, s, amax);
}

int launch_residual_layernorm_forward(int dtype, void* y, float* mean, float* rstd, void* xsum, const void* x,
                                      const void* r, const void* gamma, const void* beta, int N, int C,
                                      cudaStream_t s, unsigned* amax) {
    return ln_forward(dtype, y, mean, rstd, xsum, x, r, gamma, beta, N, C, s, amax);
}

static int ln_bwd_blocks(int N) {
    int b = (N + LN_BWD_WARPS - 1) / LN_BWD_WARPS;
    return b < LN_BWD_MAX_BLOCKS ? (b < 1 ? 1 : b) : LN_BWD_MAX_BLOCKS;
}

// The staged kernel: two resident blocks per SM, every row of a block's
// stride handled in one pass of the grid.
static int ln_bwd_staged_blocks(int N) {
    const int cap = 2 * gpt2_num_sms();
    int b = (N + LN_BWD_WARPS - 1) / LN_BWD_WARPS;
    return b < cap ? (b < 1 ? 1 : b) : cap;
}

size_t layernorm_backward_scratch(int N, int C) {
    int b = ln_bwd_blocks(N) > ln_bwd_staged_blocks(N) ? ln_bwd_blocks(N) : ln_bwd_staged_blocks(N);
    if (ln_wide_blocks(N, LN_WIDE_R_BWD) > b) b = ln_wide_blocks(N, LN_WIDE_R_BWD);
    return (size_t)b * 3 * C * 4;
}

template <typename T, int VPL>
static void ln_bwd_launch(int blocks, size_t smem, void* out, bool accumulate, float* partial, int np, const void* dy,
                          const void* x, const void* gamma, const float* mean, const float* rstd, int N, int C,
                          cudaStream_t s, unsigned* amax) {
    smem_attr((const void*)ln_bwd_kernel<T, VPL>, LN_BWD_WARPS * 3 * 2048 * 4);
    ln_bwd_kernel<T, VPL><<<blocks, LN_BWD_WARPS * 32, smem, s>>>((T*)out, accumulate, partial, np, (const T*)dy,
                                                                  (const T*)x, (const T*)gamma, mean, rstd, N, C,
                                                                  amax);
}

template <typename T, int VPL>
static void ln_bwd_staged_launch(int blocks, size_t smem, void* out, bool accumulate, float* partial, int np,
                                 const void* dy, const void* x, const void* gamma, const float* mean,
                                 const float* rstd, int N, int C, cudaStream_t s) {
    smem_attr((const void*)ln_bwd_staged_kernel<T, VPL>,
              LN_BWD_WARPS * LN_STAGES * (3 * LN_STAGED_MAX_ROW_BYTES + 16));
    ln_bwd_staged_kernel<T, VPL><<<blocks, LN_BWD_WARPS * 32, smem, s>>>(
        (T*)out, accumulate, partial, np, (const T*)dy, (const T*)x, (const T*)gamma, mean, rstd, N, C);
}

template <int VPL, int STG>
static void ln_bwd_bf16_launch(int blocks, size_t smem, void* out, bool accumulate, float* partial, int np,
                               const void* dy, const void* x, const void* gamma, const float* mean,
                               const float* rstd, int N, int C, cudaStream_t s, unsigned* amax) {
    smem_attr((const void*)ln_bwd_bf16_kernel<VPL, STG>,
              LN_BWD_WARPS * STG * (3 * LN_STAGED_MAX_ROW_BYTES + 16) + 1024 * 4);
    ln_bwd_bf16_kernel<VPL, STG><<<blocks, LN_BWD_WARPS * 32, smem, s>>>((bf16*)out, accumulate, partial, np,
                                                                          (const bf16*)dy, (const bf16*)x,
                                                                          (const bf16*)gamma, mean, rstd, N, C,
                                                                          amax);
}

// Shared memory of an SM of the current device, and the part reserved per block.
static int sm_smem_bytes() {
    static const int v = [] {
        int d = 0, x = 0;
        cudaGetDevice(&d);
        if (cudaDeviceGetAttribute(&x, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d) != cudaSuccess) x = 0;
        cudaGetLastError();
        return x;
    }();
    return v;
}

// The row pass of the backward: out (+)= dx and the per-block column sums
// partial [blocks][np * C] (dy * xhat | dy | the values written, np == 3).
// Returns the number of blocks (the partial rows). amax (bf16 only): see
// launch_layernorm_forward.
static int ln_backward_rows(int dtype, void* out, bool accumulate, float* partial_s, int np, const void* dy,
                            const void* x, const void* gamma, const float* mean, const float* rstd, int N, int C,
                            cudaStream_t s, unsigned* amax = nullptr) {
    if (ln_wide(dtype, C)) {
        const int blocks = ln_wide_blocks(N, LN_WIDE_R_BWD);
        smem_attr((const void*)ln_bwd_wide_kernel, LN_WIDE_BWD_SMEM);
        ln_bwd_wide_kernel<<<blocks, LN_WIDE_THREADS, LN_WIDE_BWD_SMEM, s>>>(
            (bf16*)out, accumulate, partial_s, np, (const bf16*)dy, (const bf16*)x, (const bf16*)gamma, mean, rstd, N,
            C, amax);
        return blocks;
    }
    if ((size_t)C * (dtype == GPT2_MODE_BF16 ? 2 : 4) <= LN_STAGED_MAX_ROW_BYTES) {
        // bf16: 111 KB of ring per block at C = 768, two blocks per SM; where
        // two blocks of three slots a warp do not fit (C = 1024: 148 KB each),
        // two slots a warp (100 KB), so that two blocks do
        const int blocks = ln_bwd_staged_blocks(N);
        const size_t smem = ln_staged_smem(dtype, C);
        const size_t gbytes = ((size_t)C * 4 + 15) & ~(size_t)15;
        const size_t smem2 = (size_t)LN_BWD_WARPS * 2 * (3 * (size_t)C * 2 + 16) + gbytes;
        const bool two = 2 * (smem + gbytes + 1024) > (size_t)sm_smem_bytes();
#define LN_BWD_STAGED_CALL(V)                                                                                   \
    if (dtype == GPT2_MODE_BF16 && two)                                                                         \
        ln_bwd_bf16_launch<V, 2>(blocks, smem2, out, accumulate, partial_s, np, dy, x, gamma, mean, rstd, N, C, \
                                 s, amax);                                                                      \
    else if (dtype == GPT2_MODE_BF16)                                                                           \
        ln_bwd_bf16_launch<V, LN_STAGES>(blocks, smem + gbytes, out, accumulate, partial_s, np, dy, x, gamma,   \
                                         mean, rstd, N, C, s, amax);                                            \
    else                                                                                                        \
        ln_bwd_staged_launch<float, V>(blocks, smem, out, accumulate, partial_s, np, dy, x, gamma, mean, rstd,  \
                                       N, C, s);
        switch (ln_vpl(C)) {
            case 1: LN_BWD_STAGED_CALL(1); break;
            case 2: LN_BWD_STAGED_CALL(2); break;
            case 3: LN_BWD_STAGED_CALL(3); break;
            default: LN_BWD_STAGED_CALL(4); break;
        }
#undef LN_BWD_STAGED_CALL
        return blocks;
    }
    const int blocks = ln_bwd_blocks(N);
    const size_t smem = (size_t)LN_BWD_WARPS * np * C * 4;
    float* partial = partial_s;
#define LN_BWD_CALL(V)                                                                                           \
    if (dtype == GPT2_MODE_BF16)                                                                                 \
        ln_bwd_launch<bf16, V>(blocks, smem, out, accumulate, partial, np, dy, x, gamma, mean, rstd, N, C, s,   \
                               amax);                                                                            \
    else                                                                                                         \
        ln_bwd_launch<float, V>(blocks, smem, out, accumulate, partial, np, dy, x, gamma, mean, rstd, N, C, s,  \
                                amax);
    LN_DISPATCH(ln_vpl(C), LN_BWD_CALL)
#undef LN_BWD_CALL
    return blocks;
}

static int ln_backward(int dtype, void* out, bool accumulate, float* dgamma, float* dbeta, float* dout_colsum,
                       const void* dy, const void* x, const void* gamma, const float* mean, const float* rstd, int N,
                       int C, void* scratch, cudaStream_t s, int grad_accumulate = 0) {
    const int np = dout_colsum ? 3 : 2;
    const int blocks =
        ln_backward_rows(dtype, out, accumulate, (float*)scratch, np, dy, x, gamma, mean, rstd, N, C, s);
    launch_colsum3(dgamma, dbeta, dout_colsum, C, (const float*)scratch, blocks, np * C, s, grad_accumulate);
    return 2;
}

int launch_layernorm_backward_residual_rows(int dtype, void* dres, int accumulate, float* partial, int np,
                                            const void* dy, const void* x, const void* gamma, const float* mean,
                                            const float* rstd, int N, int C, cudaStream_t s, int* rows,
                                            unsigned* amax) {
    *rows = ln_backward_rows(dtype, dres, accumulate != 0, partial, np, dy, x, gamma, mean, rstd, N, C, s, amax);
    return 1;
}

int launch_layernorm_backward(int dtype, void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                              const void* gamma, const float* mean, const float* rstd, int N, int C, void* scratch,
                              cudaStream_t s) {
    return ln_backward(dtype, dx, false, dgamma, dbeta, nullptr, dy, x, gamma, mean, rstd, N, C, scratch, s);
}

int launch_layernorm_backward_residual(int dtype, void* dres, int accumulate, float* dgamma, float* dbeta,
                                       float* dres_colsum, const void* dy, const void* x, const void* gamma,
                                       const float* mean, const float* rstd, int N, int C, void* scratch,
                                       cudaStream_t s, int grad_accumulate) {
    return ln_backward(dtype, dres, accumulate != 0, dgamma, dbeta, dres_colsum, dy, x, gamma, mean, rstd, N, C,
                       scratch, s, grad_accumulate);
}
