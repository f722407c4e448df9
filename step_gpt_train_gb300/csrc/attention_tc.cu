// Causal attention forward on the tcgen05 tensor cores (bf16, head size 64).
//
// One CTA per (128-query tile, batch, head); two CTAs share an SM. The T x T
// score matrix exists only as 128 x 128 fp32 tiles in tensor memory (TMEM).
// Per key block j (causal: j <= query tile):
//   S = Q K_j^T           tcgen05.mma M=128 N=128 K=64, into TMEM;
//   softmax threads       (thread = query row = TMEM lane) load their S row,
//                         hand the S buffer back, and form
//                         P = exp2(S log2(e)/sqrt(hd) - m) with a per-row
//                         reference m, accumulating the row sum l;
//                         P goes to shared memory as bf16 in the MMA's
//                         K-major 128-byte swizzled layout;
//   O += P V_j            tcgen05.mma M=128 N=64 K=128, into a TMEM accumulator.
// The reference m moves only when a row's maximum grows by more than 8 (log2
// units), so P <= 256; when it moves, the row's O (in TMEM) and l are scaled
// by exp2(m_old - m_new) before the next PV MMA. Finally O / l and the
// log-sum-exp m + log l are written.
//
// Warps: 0 TMA producer (Q once; K per block into a two-stage ring, V into
// one buffer), 1 TMEM allocation and MMA issue (one thread; it issues S for
// block j+1 before PV for block j), 2..5 softmax. Every wait is bounded.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

#include <cfloat>

namespace {

using namespace tc;

constexpr int AT_M = 128;                  // queries per CTA
constexpr int AT_N = 128;                  // keys per block
constexpr int AT_HD = 64;                  // head size
constexpr int AT_TILE = AT_M * AT_HD * 2;  // 16 KB: 128 rows of 64 bf16
constexpr int AT_THREADS = 192;
// shared memory: Q | K stage 0 | K stage 1 | V | P (two 64-key chunks) | barriers
constexpr int AT_SMEM = 6 * AT_TILE + 256 + 1024;  // Q | K0 | K1 | V | P (2 chunks) | barriers
constexpr uint32_t AT_TMEM_COLS = 256;     // S [0,128), O [128,192)
constexpr float AT_LN2 = 0.6931471805599453f;
constexpr float AT_RESCALE = 8.f;          // log2 of the largest P before the reference max moves

struct FwdArgs {
    bf16* o;       // [B*T, C]
    float* lse;    // [B, H, T]
    int* status;
    int T, C, H;
    float scale_log2;  // log2(e) / sqrt(hd)
};

__global__ void __launch_bounds__(AT_THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base;
    auto sK = [&](int st) { return base + (1 + st) * AT_TILE; };
    const uint32_t sV = base + 3 * AT_TILE;
    const uint32_t sP = base + 4 * AT_TILE;
    uint8_t* gP = gbase + 4 * AT_TILE;
    const uint32_t bars = base + 6 * AT_TILE;
    uint8_t* bar_area = gbase + 6 * AT_TILE;
    // barriers: q_full, k_full[2], k_empty[2], v_full, v_empty, s_full, s_free, p_full, p_free, o_done, drain
    const uint32_t q_full = bars;
    auto k_full = [&](int i) { return bars + 8u * (1 + i); };
    auto k_empty = [&](int i) { return bars + 8u * (3 + i); };
    const uint32_t v_full = bars + 8u * 5, v_empty = bars + 8u * 6;
    const uint32_t s_full = bars + 8u * 7, s_free = bars + 8u * 8;
    const uint32_t p_full = bars + 8u * 9, p_free = bars + 8u * 10;
    const uint32_t o_done = bars + 8u * 11, drain = bars + 8u * 12;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * 13);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * 13 + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = gridDim.x - 1 - blockIdx.x;  // longest rows first
    const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
    const int nkb = qt + 1;                     // causal: key blocks 0..qt

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; i++) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
        }
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(p_free, 1);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_addr((const void*)tmem_slot), AT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------------- TMA producer
            int k_issued[2] = {-1, -1}, v_issued = -1;
            mbar_expect_tx(q_full, AT_TILE);
            tma_load_3d(sQ, &tm_qkv, q_full, h * AT_HD, qt * AT_M, b);
            for (int j = 0; j < nkb; j++) {
                const int st = j & 1;
                const uint32_t ph = (j >> 1) & 1;
                if (!mbar_wait(k_empty(st), ph ^ 1u, abort_flag, a.status)) break;
                mbar_expect_tx(k_full(st), AT_TILE);
                tma_load_3d(sK(st), &tm_qkv, k_full(st), a.C + h * AT_HD, j * AT_N, b);
                k_issued[st] = (int)ph;
                // V(j) once PV(j-1) has read the buffer
                if (!mbar_wait(v_empty, (j & 1) ^ 1u, abort_flag, a.status)) break;
                mbar_expect_tx(v_full, AT_TILE);
                tma_load_3d(sV, &tm_qkv, v_full, 2 * a.C + h * AT_HD, j * AT_N, b);
                v_issued = j & 1;
            }
            mbar_drain(q_full, 0, a.status);
            for (int st = 0; st < 2; st++)
                if (k_issued[st] >= 0) mbar_drain(k_full(st), (uint32_t)k_issued[st], a.status);
            if (v_issued >= 0) mbar_drain(v_full, (uint32_t)v_issued, a.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // -------------------------------------------------- MMA issuer
            constexpr uint32_t idesc_s = make_idesc(AT_M, AT_N, false, false);
            constexpr uint32_t idesc_o = make_idesc(AT_M, AT_HD, false, true);
            bool ok = mbar_wait(q_full, 0, abort_flag, a.status);
            // S(j) = Q K(j)^T; the K stage is free once these MMAs finish
            auto issue_s = [&](int j) -> bool {
                const int st = j & 1;
                if (!mbar_wait(k_full(st), (j >> 1) & 1, abort_flag, a.status)) return false;
                if (!mbar_wait(s_free, (j & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < AT_HD / 16; k++)
                    tc_mma(tmem, sw128_desc(sQ + k * 32, 16, 1024), sw128_desc(sK(st) + k * 32, 16, 1024), idesc_s,
                           k > 0 ? 1u : 0u);
                tc_commit(s_full);
                tc_commit(k_empty(st));
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < nkb; j++) {
                if (j + 1 < nkb && !(ok = issue_s(j + 1))) break;
                // O += P(j) V(j)
                if (!(ok = mbar_wait(p_full, j & 1, abort_flag, a.status))) break;
                if (!(ok = mbar_wait(v_full, j & 1, abort_flag, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < AT_N / 16; kk++)
                    tc_mma(tmem + 128u, sw128_desc(sP + (kk >> 2) * AT_TILE + (kk & 3) * 32, 16, 1024),
                           sw128_desc(sV + kk * 2048, 8192, 1024), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(p_free);
                tc_commit(v_empty);
            }
            if (ok) tc_commit(o_done);
            tc_commit(drain);
            mbar_drain(drain, 0, a.status);
        }
    } else {
        // ------------------------------------------------------ softmax (warps 2..5)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row in the tile = TMEM lane
        const int q = qt * AT_M + r;     // query position
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        float m = -FLT_MAX, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkb; j++) {
            uint32_t v[4][32];
            if (!(ok = warp_wait(s_full, j & 1, abort_flag, a.status))) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 4; c++) tc_ld32_issue(trow + (uint32_t)(c * 32), v[c]);
#pragma unroll
            for (int c = 0; c < 4; c++) tc_ld_wait(v[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);  // the MMA may now write S(j+1)
            // scaled scores, masked on the diagonal block
            const bool diag = j == qt;
            float mx = -FLT_MAX;
#pragma unroll
            for (int c = 0; c < 4; c++)
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    float x = __uint_as_float(v[c][i]) * a.scale_log2;
                    if (diag && j * AT_N + c * 32 + i > q) x = -FLT_MAX;
                    v[c][i] = __float_as_uint(x);
                    mx = fmaxf(mx, x);
                }
            // move the reference max only when it grew by more than AT_RESCALE
            float factor = 1.f;
            const bool move = mx > m + AT_RESCALE;
            if (move) {
                factor = ex2_approx(m - mx);  // 0 on the first block (m = -FLT_MAX)
                m = mx;
                l *= factor;
            }
            // P as packed bf16 pairs: pk[c*16 + i/2] holds keys c*32+i, c*32+i+1
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 4; c++)
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const float x0 = __uint_as_float(v[c][i]), x1 = __uint_as_float(v[c][i + 1]);
                    const float p0 = x0 == -FLT_MAX ? 0.f : ex2_approx(x0 - m);
                    const float p1 = x1 == -FLT_MAX ? 0.f : ex2_approx(x1 - m);
                    l += p0 + p1;
                    __nv_bfloat162 hh = __floats2bfloat162_rn(p0, p1);
                    pk[c * 16 + i / 2] = *reinterpret_cast<uint32_t*>(&hh);
                }
            // PV(j-1) has finished with the P buffer and with O
            if (!(ok = warp_wait(p_free, (j & 1) ^ 1u, abort_flag, a.status))) break;
            if (j > 0 && __any_sync(0xffffffffu, move)) {
                tc_fence_after();
#pragma unroll
                for (int half = 0; half < 2; half++) {
                    uint32_t ov[32];
                    tc_ld32_issue(trow + 128u + half * 32, ov);
                    tc_ld_wait(ov);
#pragma unroll
                    for (int i = 0; i < 32; i++) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * factor);
                    tc_st32(trow + 128u + half * 32, ov);
                }
                tc_st_wait();
                tc_fence_before();
            }
            uint8_t* prow = gP + r * 128;
#pragma unroll
            for (int u = 0; u < 16; u++) {  // 16-byte units: keys 8u .. 8u+7
                const uint4 w = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                const int kc = u >> 3, uu = u & 7;  // 64-key chunk, unit within the 128-byte row
                *reinterpret_cast<uint4*>(prow + kc * AT_TILE + ((uu ^ (r & 7)) << 4)) = w;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        // O / l, log-sum-exp
        if (ok && warp_wait(o_done, 0, abort_flag, a.status)) {
            tc_fence_after();
            uint32_t ov[2][32];
            tc_ld32_issue(trow + 128u, ov[0]);
            tc_ld32_issue(trow + 160u, ov[1]);
            tc_ld_wait(ov[0]);
            tc_ld_wait(ov[1]);
            if (q < a.T) {
                const float inv = 1.f / l;
                bf16* orow = a.o + ((int64_t)b * a.T + q) * a.C + h * AT_HD;
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) f[e] = __uint_as_float(ov[u / 4][(u % 4) * 8 + e]) * inv;
                    store8(orow + u * 8, f);
                }
                a.lse[((int64_t)b * a.H + h) * a.T + q] = (m + log2f(l)) * AT_LN2;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, AT_TMEM_COLS);
    }
}

// 3-D map over qkv viewed as [B][T][3C] bf16, box = 128 rows x 64 columns of
// one batch; rows at or past T read as zero.
bool make_qkv_map(CUtensorMap* map, const void* qkv, int B, int T, int C) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)3 * C, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)3 * C * 2, (cuuint64_t)T * 3 * C * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// bf16 forward, head size 64 (the attention.cu launcher routes here).
int launch_attention_forward_tc(bf16* o, float* lse, const bf16* qkv, int B, int T, int C, int H, int* status,
                                cudaStream_t s) {
    CUtensorMap map;
    if (!make_qkv_map(&map, qkv, B, T, C)) return GPT2_ERR_CUDA;
    static bool configured = false;
    if (!configured) {
        cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, AT_SMEM);
        configured = true;
    }
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.status = status;
    a.T = T;
    a.C = C;
    a.H = H;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)(C / H));
    dim3 grid((T + AT_M - 1) / AT_M, B * H);
    attn_fwd_tc_kernel<<<grid, AT_THREADS, AT_SMEM, s>>>(map, a);
    return 1;
}

// =============================================================================
// Attention backward on tcgen05 (bf16, head size 64), two deterministic
// kernels: one per 128-key tile (dK, dV) and one per 128-query tile (dQ).
// Every output element has one writer; no atomics.
//
// dK/dV kernel, for each 128-query block i at or after the key tile:
//   S^T  = K Q_i^T,  dP^T = V dO_i^T        (M=128 keys, N=128 queries, K=64)
//   P^T  = exp2(S^T log2(e)/sqrt(hd) - lse_i log2(e)), 0 where query < key
//   dS^T = P^T (dP^T - D_i),  D = rowsum(dO * O)
//   dV  += P^T dO_i,  dK += dS^T Q_i          (M=128 keys, N=64, K=128)
// dQ kernel, for each 128-key block j at or before the query tile:
//   S = Q K_j^T, dP = dO V_j^T, P, dS as above (rows = queries),
//   dQ += dS K_j;  dK and dQ are scaled by 1/sqrt(hd) at the end.
// P^T and dS^T (dS) are written to shared memory as bf16 in the MMA's K-major
// 128-byte swizzled layout; the accumulators stay in TMEM until the end.
//
// Warps: 0 TMA producer (lane 0) and, in the dK/dV kernel, all lanes stage
// each block's log-sum-exp and D into shared memory; 1 MMA issuer; 2..9
// elementwise (warp w serves TMEM lanes 32*(w%4).. and half of the 128
// columns). One CTA per SM (512 TMEM columns).
// =============================================================================

namespace {

constexpr int BW_THREADS = 320;
constexpr int BW_EW = 8;     // elementwise warps
constexpr int DKDV_ST = 3;   // Q/dO (and lse/D) stages of the dK/dV kernel
constexpr int DQ_ST = 4;     // K/V stages of the dQ kernel

struct BwdArgs {
    bf16* dqkv;          // [B*T, 3C]
    const float* lse;    // [B, H, T]
    const float* D;      // [B, H, T]
    int* status;
    int T, C, H;
    float scale_log2;    // log2(e) / sqrt(hd)
    float scale;         // 1 / sqrt(hd)
};

// Store 32 fp32 values (times s) as bf16 to global (64 bytes).
__device__ __forceinline__ void store32_bf16(bf16* dst, const uint32_t (&v)[32], float s) {
#pragma unroll
    for (int u = 0; u < 4; u++) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; e++) f[e] = __uint_as_float(v[u * 8 + e]) * s;
        store8(dst + u * 8, f);
    }
}

// Write this thread's 64 bf16 values (row r, columns half*64 .. +63) into a
// [128][128] K-major operand buffer (two 64-column chunks of 16 KB, 128-byte
// swizzle: 16-byte unit u of row r at position u ^ (r & 7)).
__device__ __forceinline__ void write_row64(uint8_t* buf, int r, int half, const uint32_t (&pk)[32]) {
    uint8_t* row = buf + half * AT_TILE + r * 128;
#pragma unroll
    for (int u = 0; u < 8; u++)
        *reinterpret_cast<uint4*>(row + ((u ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// -------------------------------------------------------------------------- dK, dV
__global__ void __launch_bounds__(BW_THREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                            BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    // K | V | DKDV_ST x (Q, dO) | P^T (2 chunks) | dS^T (2 chunks) | lse/D slots | barriers
    constexpr int NS = DKDV_ST;
    const uint32_t sK = base, sV = base + AT_TILE;
    auto sQ = [&](int st) { return base + (2 + 2 * st) * AT_TILE; };
    auto sO = [&](int st) { return base + (3 + 2 * st) * AT_TILE; };
    const uint32_t sP = base + (2 + 2 * NS) * AT_TILE, sS = base + (4 + 2 * NS) * AT_TILE;
    uint8_t* gP = gbase + (2 + 2 * NS) * AT_TILE;
    uint8_t* gS = gbase + (4 + 2 * NS) * AT_TILE;
    float* ldslot = reinterpret_cast<float*>(gbase + (6 + 2 * NS) * AT_TILE);  // [NS][256]: lse2[128], D[128]
    const uint32_t bars = base + (6 + 2 * NS) * AT_TILE + NS * 1024;
    uint8_t* bar_area = gbase + (6 + 2 * NS) * AT_TILE + NS * 1024;
    const uint32_t kv_full = bars;
    auto qd_full = [&](int i) { return bars + 8u * (1 + i); };
    auto qd_empty = [&](int i) { return bars + 8u * (1 + NS + i); };
    auto ld_full = [&](int i) { return bars + 8u * (1 + 2 * NS + i); };
    auto ld_empty = [&](int i) { return bars + 8u * (1 + 3 * NS + i); };
    const uint32_t bx = bars + 8u * (1 + 4 * NS);
    const uint32_t s_full = bx, s_free = bx + 8u;
    const uint32_t dp_full = bx + 16u, dp_free = bx + 24u;
    const uint32_t p_full = bx + 32u, p_free = bx + 40u;
    const uint32_t ds_full = bx + 48u, ds_free = bx + 56u;
    const uint32_t o_done = bx + 64u, drain = bx + 72u;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * (1 + 4 * NS) + 80);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (1 + 4 * NS) + 84);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int kt = blockIdx.x;  // key tile; the first tiles have the most query blocks
    const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
    const int nqt = (a.T + AT_M - 1) / AT_M;
    const int nblk = nqt - kt;  // query blocks kt .. nqt-1

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < NS; i++) {
            mbar_init(qd_full(i), 1);
            mbar_init(qd_empty(i), 1);
            mbar_init(ld_full(i), 1);
            mbar_init(ld_empty(i), BW_EW);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, BW_EW);
        mbar_init(dp_full, 1);
        mbar_init(dp_free, BW_EW);
        mbar_init(p_full, BW_EW);
        mbar_init(p_free, 1);
        mbar_init(ds_full, BW_EW);
        mbar_init(ds_free, 1);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_addr((const void*)tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;  // S^T [0,128) dP^T [128,256) dV [256,320) dK [320,384)

    if (warp == 0) {
        // ------------------------------------------------------ producer
        int qd_issued[NS];
        for (int i = 0; i < NS; i++) qd_issued[i] = -1;
        if (lane == 0) {
            mbar_expect_tx(kv_full, 2 * AT_TILE);
            tma_load_3d(sK, &tm_qkv, kv_full, a.C + h * AT_HD, kt * AT_N, b);
            tma_load_3d(sV, &tm_qkv, kv_full, 2 * a.C + h * AT_HD, kt * AT_N, b);
        }
        const float* lrow = a.lse + ((int64_t)b * a.H + h) * a.T;
        const float* drow = a.D + ((int64_t)b * a.H + h) * a.T;
        for (int n = 0; n < nblk; n++) {
            const int st = n % NS;
            const uint32_t ph = (n / NS) & 1;
            const int q0 = (kt + n) * AT_M;
            int ok = 1;
            if (lane == 0) {
                ok = mbar_wait(qd_empty(st), ph ^ 1u, abort_flag, a.status);
                if (ok) {
                    mbar_expect_tx(qd_full(st), 2 * AT_TILE);
                    tma_load_3d(sQ(st), &tm_qkv, qd_full(st), h * AT_HD, q0, b);
                    tma_load_3d(sO(st), &tm_do, qd_full(st), h * AT_HD, q0, b);
                    qd_issued[st] = (int)ph;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok || !warp_wait(ld_empty(st), ph ^ 1u, abort_flag, a.status)) break;
            float* slot = ldslot + st * 256;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int c = lane * 4 + e, q = q0 + c;
                slot[c] = q < a.T ? lrow[q] * 1.4426950408889634f : 0.f;
                slot[128 + c] = q < a.T ? drow[q] : 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ld_full(st));
        }
        if (lane == 0) {
            mbar_drain(kv_full, 0, a.status);
            for (int st = 0; st < NS; st++)
                if (qd_issued[st] >= 0) mbar_drain(qd_full(st), (uint32_t)qd_issued[st], a.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // -------------------------------------------------- MMA issuer
            constexpr uint32_t idesc_s = make_idesc(AT_M, AT_N, false, false);  // K-major x K-major
            constexpr uint32_t idesc_o = make_idesc(AT_M, AT_HD, false, true);  // K-major x MN-major
            bool ok = mbar_wait(kv_full, 0, abort_flag, a.status);
            auto issue_sdp = [&](int n) -> bool {  // S^T(n)
                const int st = n % NS;
                if (!mbar_wait(qd_full(st), (n / NS) & 1, abort_flag, a.status)) return false;
                if (!mbar_wait(s_free, (n & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; k++)
                    tc_mma(tmem, sw128_desc(sK + k * 32, 16, 1024), sw128_desc(sQ(st) + k * 32, 16, 1024), idesc_s,
                           k > 0 ? 1u : 0u);
                tc_commit(s_full);
                return true;
            };
            auto issue_dp = [&](int n) -> bool {
                const int st = n % NS;
                if (!mbar_wait(dp_free, (n & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; k++)
                    tc_mma(tmem + 128u, sw128_desc(sV + k * 32, 16, 1024), sw128_desc(sO(st) + k * 32, 16, 1024),
                           idesc_s, k > 0 ? 1u : 0u);
                tc_commit(dp_full);
                return true;
            };
            if (ok) ok = issue_sdp(0) && issue_dp(0);
            for (int n = 0; ok && n < nblk; n++) {
                const int st = n % NS;
                if (n + 1 < nblk && !(ok = issue_sdp(n + 1))) break;
                // dV += P^T dO
                if (!(ok = mbar_wait(p_full, n & 1, abort_flag, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; kk++)
                    tc_mma(tmem + 256u, sw128_desc(sP + (kk >> 2) * AT_TILE + (kk & 3) * 32, 16, 1024),
                           sw128_desc(sO(st) + kk * 2048, 8192, 1024), idesc_o, (n > 0 || kk > 0) ? 1u : 0u);
                tc_commit(p_free);
                if (n + 1 < nblk && !(ok = issue_dp(n + 1))) break;
                // dK += dS^T Q
                if (!(ok = mbar_wait(ds_full, n & 1, abort_flag, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; kk++)
                    tc_mma(tmem + 320u, sw128_desc(sS + (kk >> 2) * AT_TILE + (kk & 3) * 32, 16, 1024),
                           sw128_desc(sQ(st) + kk * 2048, 8192, 1024), idesc_o, (n > 0 || kk > 0) ? 1u : 0u);
                tc_commit(ds_free);
                tc_commit(qd_empty(st));
            }
            if (ok) tc_commit(o_done);
            tc_commit(drain);
            mbar_drain(drain, 0, a.status);
        }
    } else {
        // ------------------------------------------------------ elementwise (warps 2..9)
        const int ew = warp - 2;
        const int quad = warp & 3, half = ew >> 2;
        const int r = quad * 32 + lane;      // key row = TMEM lane
        const int key = kt * AT_N + r;
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        bool ok = true;
        for (int n = 0; n < nblk; n++) {
            const int st = n % NS;
            const int q0 = (kt + n) * AT_M + half * 64;  // first query of this thread's columns
            const bool diag = n == 0;
            uint32_t sv[2][32];
            if (!(ok = warp_wait(s_full, n & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + (uint32_t)(half * 64), sv[0]);
            tc_ld32_issue(trow + (uint32_t)(half * 64 + 32), sv[1]);
            tc_ld_wait(sv[0]);
            tc_ld_wait(sv[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            if (!(ok = warp_wait(ld_full(st), (n / NS) & 1, abort_flag, a.status))) break;
            const float* slot = ldslot + st * 256 + half * 64;
            float p[64];
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                float pp[2];
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const int cc = c + e, q = q0 + cc;
                    const float x = __uint_as_float(sv[cc >> 5][cc & 31]) * a.scale_log2 - slot[cc];
                    pp[e] = ((diag && q < key) || q >= a.T) ? 0.f : ex2_approx(x);
                    p[cc] = pp[e];
                }
                pk[c / 2] = pack2(pp[0], pp[1]);
            }
            if (!(ok = warp_wait(p_free, (n & 1) ^ 1u, abort_flag, a.status))) break;
            write_row64(gP, r, half, pk);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            // dS^T = P^T (dP^T - D)
            if (!(ok = warp_wait(dp_full, n & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + 128u + (uint32_t)(half * 64), sv[0]);
            tc_ld32_issue(trow + 128u + (uint32_t)(half * 64 + 32), sv[1]);
            tc_ld_wait(sv[0]);
            tc_ld_wait(sv[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_free);
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float d0 = p[c] * (__uint_as_float(sv[c >> 5][c & 31]) - slot[128 + c]);
                const float d1 = p[c + 1] * (__uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]) - slot[128 + c + 1]);
                pk[c / 2] = pack2(d0, d1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ld_empty(st));  // lse and D of this block are no longer read
            if (!(ok = warp_wait(ds_free, (n & 1) ^ 1u, abort_flag, a.status))) break;
            write_row64(gS, r, half, pk);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
        }
        if (ok && warp_wait(o_done, 0, abort_flag, a.status)) {
            tc_fence_after();
            uint32_t dv[32], dk[32];
            tc_ld32_issue(trow + 256u + (uint32_t)(half * 32), dv);
            tc_ld32_issue(trow + 320u + (uint32_t)(half * 32), dk);
            tc_ld_wait(dv);
            tc_ld_wait(dk);
            if (key < a.T) {
                bf16* out = a.dqkv + ((int64_t)b * a.T + key) * 3 * a.C + h * AT_HD + half * 32;
                store32_bf16(out + a.C, dk, a.scale);
                store32_bf16(out + 2 * a.C, dv, 1.f);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

// -------------------------------------------------------------------------- dQ
__global__ void __launch_bounds__(BW_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                          BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    // Q | dO | DQ_ST x (K, V) | dS (2 chunks) | barriers
    constexpr int NS = DQ_ST;
    const uint32_t sQ = base, sO = base + AT_TILE;
    auto sK = [&](int st) { return base + (2 + 2 * st) * AT_TILE; };
    auto sV = [&](int st) { return base + (3 + 2 * st) * AT_TILE; };
    const uint32_t sS = base + (2 + 2 * NS) * AT_TILE;
    uint8_t* gS = gbase + (2 + 2 * NS) * AT_TILE;
    const uint32_t bars = base + (4 + 2 * NS) * AT_TILE;
    uint8_t* bar_area = gbase + (4 + 2 * NS) * AT_TILE;
    const uint32_t qo_full = bars;
    auto kv_full = [&](int i) { return bars + 8u * (1 + i); };
    auto kv_empty = [&](int i) { return bars + 8u * (1 + NS + i); };
    const uint32_t bx = bars + 8u * (1 + 2 * NS);
    const uint32_t s_full = bx, s_free = bx + 8u;
    const uint32_t dp_full = bx + 16u, dp_free = bx + 24u;
    const uint32_t ds_full = bx + 32u, ds_free = bx + 40u;
    const uint32_t o_done = bx + 48u, drain = bx + 56u;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * (1 + 2 * NS) + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (1 + 2 * NS) + 68);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = gridDim.x - 1 - blockIdx.x;  // longest rows first
    const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
    const int nkb = qt + 1;

    if (threadIdx.x == 0) {
        mbar_init(qo_full, 1);
        for (int i = 0; i < NS; i++) {
            mbar_init(kv_full(i), 1);
            mbar_init(kv_empty(i), 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, BW_EW);
        mbar_init(dp_full, 1);
        mbar_init(dp_free, BW_EW);
        mbar_init(ds_full, BW_EW);
        mbar_init(ds_free, 1);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_addr((const void*)tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;  // S [0,128) dP [128,256) dQ [256,320)

    if (warp == 0) {
        if (lane == 0) {
            int kv_issued[NS];
            for (int i = 0; i < NS; i++) kv_issued[i] = -1;
            mbar_expect_tx(qo_full, 2 * AT_TILE);
            tma_load_3d(sQ, &tm_qkv, qo_full, h * AT_HD, qt * AT_M, b);
            tma_load_3d(sO, &tm_do, qo_full, h * AT_HD, qt * AT_M, b);
            for (int j = 0; j < nkb; j++) {
                const int st = j % NS;
                const uint32_t ph = (j / NS) & 1;
                if (!mbar_wait(kv_empty(st), ph ^ 1u, abort_flag, a.status)) break;
                mbar_expect_tx(kv_full(st), 2 * AT_TILE);
                tma_load_3d(sK(st), &tm_qkv, kv_full(st), a.C + h * AT_HD, j * AT_N, b);
                tma_load_3d(sV(st), &tm_qkv, kv_full(st), 2 * a.C + h * AT_HD, j * AT_N, b);
                kv_issued[st] = (int)ph;
            }
            mbar_drain(qo_full, 0, a.status);
            for (int st = 0; st < NS; st++)
                if (kv_issued[st] >= 0) mbar_drain(kv_full(st), (uint32_t)kv_issued[st], a.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = make_idesc(AT_M, AT_N, false, false);
            constexpr uint32_t idesc_o = make_idesc(AT_M, AT_HD, false, true);
            bool ok = mbar_wait(qo_full, 0, abort_flag, a.status);
            auto issue_s = [&](int j) -> bool {
                const int st = j % NS;
                if (!mbar_wait(kv_full(st), (j / NS) & 1, abort_flag, a.status)) return false;
                if (!mbar_wait(s_free, (j & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; k++)
                    tc_mma(tmem, sw128_desc(sQ + k * 32, 16, 1024), sw128_desc(sK(st) + k * 32, 16, 1024), idesc_s,
                           k > 0 ? 1u : 0u);
                tc_commit(s_full);
                return true;
            };
            auto issue_dp = [&](int j) -> bool {
                const int st = j % NS;
                if (!mbar_wait(dp_free, (j & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; k++)
                    tc_mma(tmem + 128u, sw128_desc(sO + k * 32, 16, 1024), sw128_desc(sV(st) + k * 32, 16, 1024),
                           idesc_s, k > 0 ? 1u : 0u);
                tc_commit(dp_full);
                return true;
            };
            if (ok) ok = issue_s(0) && issue_dp(0);
            for (int j = 0; ok && j < nkb; j++) {
                const int st = j % NS;
                if (j + 1 < nkb && !(ok = issue_s(j + 1) && issue_dp(j + 1))) break;
                // dQ += dS K
                if (!(ok = mbar_wait(ds_full, j & 1, abort_flag, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; kk++)
                    tc_mma(tmem + 256u, sw128_desc(sS + (kk >> 2) * AT_TILE + (kk & 3) * 32, 16, 1024),
                           sw128_desc(sK(st) + kk * 2048, 8192, 1024), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(ds_free);
                tc_commit(kv_empty(st));
            }
            if (ok) tc_commit(o_done);
            tc_commit(drain);
            mbar_drain(drain, 0, a.status);
        }
    } else {
        const int ew = warp - 2;
        const int quad = warp & 3, half = ew >> 2;
        const int r = quad * 32 + lane;  // query row = TMEM lane
        const int q = qt * AT_M + r;
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        const int qc = q < a.T ? q : 0;
        const float lse2 = a.lse[((int64_t)b * a.H + h) * a.T + qc] * 1.4426950408889634f;
        const float Dq = a.D[((int64_t)b * a.H + h) * a.T + qc];
        bool ok = true;
        for (int j = 0; j < nkb; j++) {
            const int k0 = j * AT_N + half * 64;  // first key of this thread's columns
            const bool diag = j == qt;
            uint32_t sv[2][32];
            if (!(ok = warp_wait(s_full, j & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + (uint32_t)(half * 64), sv[0]);
            tc_ld32_issue(trow + (uint32_t)(half * 64 + 32), sv[1]);
            tc_ld_wait(sv[0]);
            tc_ld_wait(sv[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            float p[64];
#pragma unroll
            for (int c = 0; c < 64; c++) {
                const int kk = k0 + c;
                const float x = __uint_as_float(sv[c >> 5][c & 31]) * a.scale_log2 - lse2;
                p[c] = ((diag && kk > q) || kk >= a.T) ? 0.f : ex2_approx(x);
            }
            if (!(ok = warp_wait(dp_full, j & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + 128u + (uint32_t)(half * 64), sv[0]);
            tc_ld32_issue(trow + 128u + (uint32_t)(half * 64 + 32), sv[1]);
            tc_ld_wait(sv[0]);
            tc_ld_wait(sv[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_free);
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 64; c += 2)
                pk[c / 2] = pack2(p[c] * (__uint_as_float(sv[c >> 5][c & 31]) - Dq),
                                  p[c + 1] * (__uint_as_float(sv[(c + 1) >> 5][(c + 1) & 31]) - Dq));
            if (!(ok = warp_wait(ds_free, (j & 1) ^ 1u, abort_flag, a.status))) break;
            write_row64(gS, r, half, pk);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
        }
        if (ok && warp_wait(o_done, 0, abort_flag, a.status)) {
            tc_fence_after();
            uint32_t dq[32];
            tc_ld32_issue(trow + 256u + (uint32_t)(half * 32), dq);
            tc_ld_wait(dq);
            if (q < a.T) store32_bf16(a.dqkv + ((int64_t)b * a.T + q) * 3 * a.C + h * AT_HD + half * 32, dq, a.scale);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

// 3-D map over dO viewed as [B][T][C] bf16, box = 128 rows x 64 columns.
bool make_do_map(CUtensorMap* map, const void* dout, int B, int T, int C) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)C * 2, (cuuint64_t)T * C * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(dout), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int DKDV_SMEM = (6 + 2 * DKDV_ST) * AT_TILE + DKDV_ST * 1024 + 256 + 1024;
constexpr int DQ_SMEM = (4 + 2 * DQ_ST) * AT_TILE + 256 + 1024;
static_assert(DKDV_SMEM <= 232448 && DQ_SMEM <= 232448, "shared memory per CTA");

}  // namespace

// bf16 backward after D = rowsum(dO * O) is in D (the attention.cu launcher
// computes it and routes here).
int launch_attention_backward_tc(bf16* dqkv, const bf16* dout, const bf16* qkv, const float* lse, const float* D,
                                 int B, int T, int C, int H, int* status, cudaStream_t s) {
    CUtensorMap mq, mo;
    if (!make_qkv_map(&mq, qkv, B, T, C) || !make_do_map(&mo, dout, B, T, C)) return GPT2_ERR_CUDA;
    static bool configured = false;
    if (!configured) {
        cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DKDV_SMEM);
        cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
        configured = true;
    }
    BwdArgs a;
    a.dqkv = dqkv;
    a.lse = lse;
    a.D = D;
    a.status = status;
    a.T = T;
    a.C = C;
    a.H = H;
    a.scale = 1.0f / sqrtf((float)(C / H));
    a.scale_log2 = 1.4426950408889634f * a.scale;
    dim3 grid((T + AT_M - 1) / AT_M, B * H);
    attn_bwd_dkdv_tc_kernel<<<grid, BW_THREADS, DKDV_SMEM, s>>>(mq, mo, a);
    attn_bwd_dq_tc_kernel<<<grid, BW_THREADS, DQ_SMEM, s>>>(mq, mo, a);
    return 2;
}
