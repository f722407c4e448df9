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
            if (!(ok = mbar_wait(s_full, j & 1, abort_flag, a.status))) break;
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
            if (!(ok = mbar_wait(p_free, (j & 1) ^ 1u, abort_flag, a.status))) break;
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
        if (ok && mbar_wait(o_done, 0, abort_flag, a.status)) {
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
