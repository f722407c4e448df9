// Causal multi-head attention backward (and the fp32 forward), flash-style:
// the T x T score matrix exists only tile by tile in registers. The bf16
// forward is the tcgen05 kernel of attention_tc.cu.
//
// bf16 backward (head size 64): 64 x 64 tiles, four warps of 16 rows, bf16
// tensor-core MMAs (m16n8k16, fp32 accumulate), K/V/Q/dO tiles in
// XOR-swizzled shared memory by cp.async.
// The backward recomputes P from the saved log-sum-exp and runs two kernels,
// one per key block (dK, dV) and one per query block (dQ), so that every
// output element has a single writer: no atomics, deterministic.
//
// fp32 path (the exact-parity mode, head size <= 64): one thread per query
// (forward, dQ) or per key (dK, dV), fp32 FMA, expf.
#include "common.cuh"
#include "launch.h"

#include <cfloat>

#define ATT_LOG2E 1.4426950408889634f
#define ATT_LN2 0.6931471805599453f

// ============================================================ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
    const int n = pred ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// d += a * b, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// A 64 x 64 bf16 tile in shared memory: row r is 128 bytes (8 chunks of 16);
// chunk c of row r is stored at chunk position c ^ (r & 7), so the 8 rows an
// ldmatrix phase reads fall in 8 different bank groups.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int col) {
    return base + r * 128 + ((((col >> 3) ^ (r & 7))) << 4) + ((col & 7) << 1);
}

// Load rows [row0, row0+64) of one 64-column head slice into a tile; rows at
// or past T are zero-filled. 128 threads, 4 chunks each.
__device__ __forceinline__ void load_tile64(uint32_t tile, const bf16* g, int row0, int T, int ld, int tid) {
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int id = tid + k * 128;
        const int r = id >> 3, c = id & 7;
        const int row = row0 + r;
        const bool ok = row < T;
        const bf16* src = g + (int64_t)(ok ? row : 0) * ld + c * 8;
        cp_async16(tile + r * 128 + ((c ^ (r & 7)) << 4), src, ok);
    }
}

// A-operand fragment (16 x 16) at (row0, col0) of a tile.
__device__ __forceinline__ void frag_a(uint32_t (&a)[4], uint32_t tile, int row0, int col0, int lane) {
    const int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = col0 + (lane >> 4) * 8;
    ldsm_x4(a, tile_addr(tile, r, c));
}
// B fragments for n-tiles n0 and n0+8, k-block k0, from a tile stored [n][k].
__device__ __forceinline__ void frag_b_nk(uint32_t (&b)[4], uint32_t tile, int n0, int k0, int lane) {
    const int r = n0 + (lane & 7) + (lane >> 4) * 8;
    const int c = k0 + ((lane >> 3) & 1) * 8;
    ldsm_x4(b, tile_addr(tile, r, c));
}
// B fragments for n-tiles n0 and n0+8, k-block k0, from a tile stored [k][n].
__device__ __forceinline__ void frag_b_kn(uint32_t (&b)[4], uint32_t tile, int k0, int n0, int lane) {
    const int r = k0 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = n0 + (lane >> 4) * 8;
    ldsm_x4_t(b, tile_addr(tile, r, c));
}

// acc[16 x 64] += A[16 x 64 (k)] * B, B from a [n][k] tile (S = Q K^T form).
__device__ __forceinline__ void mma_rows_x_tileT(float (&acc)[8][4], const uint32_t (&a)[4][4], uint32_t tile,
                                                 int lane) {
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
#pragma unroll
        for (int np = 0; np < 4; np++) {
            uint32_t b[4];
            frag_b_nk(b, tile, np * 16, kk * 16, lane);
            mma16816(acc[2 * np], a[kk], b[0], b[1]);
            mma16816(acc[2 * np + 1], a[kk], b[2], b[3]);
        }
    }
}
// acc[16 x 64] += P[16 x 64 (k)] * B, P given as fp32 accumulator fragments,
// B from a [k][n] tile (O = P V form).
__device__ __forceinline__ void mma_p_x_tile(float (&acc)[8][4], const float (&p)[8][4], uint32_t tile, int lane) {
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
        uint32_t a[4];
        a[0] = pack_bf16(p[2 * kk][0], p[2 * kk][1]);
        a[1] = pack_bf16(p[2 * kk][2], p[2 * kk][3]);
        a[2] = pack_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1]);
        a[3] = pack_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3]);
#pragma unroll
        for (int dp = 0; dp < 4; dp++) {
            uint32_t b[4];
            frag_b_kn(b, tile, kk * 16, dp * 16, lane);
            mma16816(acc[2 * dp], a, b[0], b[1]);
            mma16816(acc[2 * dp + 1], a, b[2], b[3]);
        }
    }
}

__device__ __forceinline__ void zero_acc(float (&a)[8][4]) {
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) a[i][j] = 0.f;
}

// Write a warp's 16 x 64 fp32 accumulator, times `scale`, as bf16 into rows
// row0 .. row0+15 (rows >= T skipped) of a [*, ld] matrix at column col0.
__device__ __forceinline__ void store_rows_bf16(bf16* g, const float (&acc)[8][4], float scale, int row0, int T,
                                                int ld, int col0, int lane) {
    const int gq = lane >> 2, tq = lane & 3;
    const int r0 = row0 + gq, r1 = r0 + 8;
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
        const int c = col0 + nt * 8 + 2 * tq;
        if (r0 < T)
            *reinterpret_cast<uint32_t*>(g + (int64_t)r0 * ld + c) = pack_bf16(acc[nt][0] * scale, acc[nt][1] * scale);
        if (r1 < T)
            *reinterpret_cast<uint32_t*>(g + (int64_t)r1 * ld + c) = pack_bf16(acc[nt][2] * scale, acc[nt][3] * scale);
    }
}

// ============================================================ backward: D = rowsum(dO * O)

template <typename T>
__global__ void attn_bwd_dot_kernel(float* __restrict__ D, const T* __restrict__ dout, const T* __restrict__ o,
                                    int B, int Tlen, int C, int H) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (b, t, h)
    if (i >= (int64_t)B * Tlen * H) return;
    const int h = (int)(i % H);
    const int64_t bt = i / H;
    const int hd = C / H;
    const T* a = dout + bt * C + h * hd;
    const T* c = o + bt * C + h * hd;
    float s = 0.f;
    for (int d = 0; d < hd; d += 8) {
        float x[8], y[8];
        load8(a + d, x);
        load8(c + d, y);
#pragma unroll
        for (int j = 0; j < 8; j++) s += x[j] * y[j];
    }
    const int b = (int)(bt / Tlen), t = (int)(bt % Tlen);
    D[((int64_t)b * H + h) * Tlen + t] = s;
}

// ============================================================ bf16 backward: dK, dV per key block

__global__ void __launch_bounds__(128) attn_bwd_dkdv_bf16_kernel(bf16* __restrict__ dqkv, const bf16* __restrict__ dout,
                                                                 const bf16* __restrict__ qkv,
                                                                 const float* __restrict__ lse,
                                                                 const float* __restrict__ Dg, int T, int C, int H,
                                                                 float scale_log2, float scale) {
    __shared__ __align__(1024) bf16 sQ[2][64 * 64];
    __shared__ __align__(1024) bf16 sO[2][64 * 64];  // dO tiles
    __shared__ __align__(1024) bf16 sKV[64 * 64];    // K, then V, for the fragments
    __shared__ float sL[2][64], sD[2][64];
    const int kb = blockIdx.x;
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int ld = 3 * C;
    const bf16* base = qkv + (int64_t)b * T * ld + h * 64;
    const bf16* dob = dout + (int64_t)b * T * C + h * 64;
    const float* lrow = lse + ((int64_t)b * H + h) * T;
    const float* drow = Dg + ((int64_t)b * H + h) * T;
    const uint32_t tkv = smem_u32(sKV);
    const uint32_t tqs[2] = {smem_u32(sQ[0]), smem_u32(sQ[1])};
    const uint32_t tos[2] = {smem_u32(sO[0]), smem_u32(sO[1])};

    uint32_t kf[4][4], vf[4][4];
    load_tile64(tkv, base + C, kb * 64, T, ld, tid);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 4; kk++) frag_a(kf[kk], tkv, w * 16, kk * 16, lane);
    __syncthreads();
    load_tile64(tkv, base + 2 * C, kb * 64, T, ld, tid);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 4; kk++) frag_a(vf[kk], tkv, w * 16, kk * 16, lane);

    float dk[8][4], dv[8][4];
    zero_acc(dk);
    zero_acc(dv);
    const int gq = lane >> 2, tq4 = lane & 3;
    const int key0 = kb * 64 + w * 16 + gq;  // this thread's keys: key0, key0 + 8
    const int nqb = (T + 63) / 64;
    auto load_q = [&](int qb, int buf) {
        load_tile64(tqs[buf], base, qb * 64, T, ld, tid);
        load_tile64(tos[buf], dob, qb * 64, T, C, tid);
        if (tid < 64) {
            const int q = qb * 64 + tid;
            sL[buf][tid] = q < T ? lrow[q] * ATT_LOG2E : 0.f;
            sD[buf][tid] = q < T ? drow[q] : 0.f;
        }
    };
    load_q(kb, 0);
    cp_async_commit();
    for (int qb = kb; qb < nqb; qb++) {
        const int buf = (qb - kb) & 1;
        cp_async_wait<0>();
        __syncthreads();
        if (qb + 1 < nqb) load_q(qb + 1, buf ^ 1);
        cp_async_commit();
        // S^T = K Q^T, P^T = exp2(S^T scale_log2 - lse2[q])
        float p[8][4];
        zero_acc(p);
        mma_rows_x_tileT(p, kf, tqs[buf], lane);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int ql = nt * 8 + 2 * tq4 + (e & 1);
                const int q = qb * 64 + ql;
                const int key = key0 + (e >> 1) * 8;
                const float x = p[nt][e] * scale_log2 - sL[buf][ql];
                p[nt][e] = (q < key || q >= T) ? 0.f : ex2_approx(x);
            }
        }
        // dV += P^T dO
        mma_p_x_tile(dv, p, tos[buf], lane);
        // dP^T = V dO^T, dS^T = P^T (dP^T - D[q])
        float ds[8][4];
        zero_acc(ds);
        mma_rows_x_tileT(ds, vf, tos[buf], lane);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int ql = nt * 8 + 2 * tq4 + (e & 1);
                ds[nt][e] = p[nt][e] * (ds[nt][e] - sD[buf][ql]);
            }
        }
        // dK += dS^T Q
        mma_p_x_tile(dk, ds, tqs[buf], lane);
    }
    cp_async_wait<0>();
    bf16* out = dqkv + (int64_t)b * T * ld;
    store_rows_bf16(out, dk, scale, kb * 64 + w * 16, T, ld, C + h * 64, lane);
    store_rows_bf16(out, dv, 1.f, kb * 64 + w * 16, T, ld, 2 * C + h * 64, lane);
}

// ============================================================ bf16 backward: dQ per query block

__global__ void __launch_bounds__(128) attn_bwd_dq_bf16_kernel(bf16* __restrict__ dqkv, const bf16* __restrict__ dout,
                                                               const bf16* __restrict__ qkv,
                                                               const float* __restrict__ lse,
                                                               const float* __restrict__ Dg, int T, int C, int H,
                                                               float scale_log2, float scale) {
    __shared__ __align__(1024) bf16 sK[2][64 * 64];
    __shared__ __align__(1024) bf16 sV[2][64 * 64];
    __shared__ __align__(1024) bf16 sQ[64 * 64];
    const int qb = gridDim.x - 1 - blockIdx.x;
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int ld = 3 * C;
    const bf16* base = qkv + (int64_t)b * T * ld + h * 64;
    const bf16* dob = dout + (int64_t)b * T * C + h * 64;
    const uint32_t tq = smem_u32(sQ);
    const uint32_t tk[2] = {smem_u32(sK[0]), smem_u32(sK[1])};
    const uint32_t tv[2] = {smem_u32(sV[0]), smem_u32(sV[1])};

    uint32_t qf[4][4], of[4][4];
    load_tile64(tq, base, qb * 64, T, ld, tid);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 4; kk++) frag_a(qf[kk], tq, w * 16, kk * 16, lane);
    __syncthreads();
    load_tile64(tq, dob, qb * 64, T, C, tid);
    load_tile64(tk[0], base + C, 0, T, ld, tid);
    load_tile64(tv[0], base + 2 * C, 0, T, ld, tid);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 4; kk++) frag_a(of[kk], tq, w * 16, kk * 16, lane);

    const int gq = lane >> 2, tq4 = lane & 3;
    const int row0 = qb * 64 + w * 16 + gq;
    float l2[2], dd[2];
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int row = row0 + r * 8;
        const int rr = row < T ? row : 0;
        l2[r] = lse[((int64_t)b * H + h) * T + rr] * ATT_LOG2E;
        dd[r] = Dg[((int64_t)b * H + h) * T + rr];
    }
    float dq[8][4];
    zero_acc(dq);
    const int nkb = qb + 1;
    for (int kb = 0; kb < nkb; kb++) {
        const int buf = kb & 1;
        if (kb + 1 < nkb) {
            load_tile64(tk[buf ^ 1], base + C, (kb + 1) * 64, T, ld, tid);
            load_tile64(tv[buf ^ 1], base + 2 * C, (kb + 1) * 64, T, ld, tid);
        }
        cp_async_commit();
        float p[8][4];
        zero_acc(p);
        mma_rows_x_tileT(p, qf, tk[buf], lane);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int key = kb * 64 + nt * 8 + 2 * tq4 + (e & 1);
                const int row = row0 + (e >> 1) * 8;
                const float x = p[nt][e] * scale_log2 - l2[e >> 1];
                p[nt][e] = (key > row || key >= T) ? 0.f : ex2_approx(x);
            }
        }
        float ds[8][4];
        zero_acc(ds);
        mma_rows_x_tileT(ds, of, tv[buf], lane);  // dP = dO V^T
#pragma unroll
        for (int nt = 0; nt < 8; nt++)
#pragma unroll
            for (int e = 0; e < 4; e++) ds[nt][e] = p[nt][e] * (ds[nt][e] - dd[e >> 1]);
        mma_p_x_tile(dq, ds, tk[buf], lane);  // dQ += dS K
        cp_async_wait<0>();
        __syncthreads();
    }
    store_rows_bf16(dqkv + (int64_t)b * T * ld, dq, scale, qb * 64 + w * 16, T, ld, h * 64, lane);
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
                              const float* lse, int B, int T, int C, int H, void* scratch, cudaStream_t s) {
    const int hd = C / H;
    if (B * T == 0) return 0;
    float* D = (float*)scratch;
    const int64_t nrows = (int64_t)B * T * H;
    const int dblocks = (int)((nrows + 255) / 256);
    const float scale = 1.0f / sqrtf((float)hd);
    if (dtype == GPT2_MODE_BF16) {
        if (hd != 64) return GPT2_ERR_ARG;
        attn_bwd_dot_kernel<bf16><<<dblocks, 256, 0, s>>>(D, (const bf16*)dout, (const bf16*)o, B, T, C, H);
        dim3 grid((T + 63) / 64, B * H);
        attn_bwd_dkdv_bf16_kernel<<<grid, 128, 0, s>>>((bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv, lse, D, T,
                                                       C, H, scale * ATT_LOG2E, scale);
        attn_bwd_dq_bf16_kernel<<<grid, 128, 0, s>>>((bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv, lse, D, T, C,
                                                     H, scale * ATT_LOG2E, scale);
        return 3;
    }
    attn_bwd_dot_kernel<float><<<dblocks, 256, 0, s>>>(D, (const float*)dout, (const float*)o, B, T, C, H);
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
