// Causal attention forward on the tcgen05 tensor cores (bf16, head size 64).
//
// Persistent: two CTAs per SM walk a list of (128-query tile, batch-head)
// work items ordered longest first (CTA c takes items c, c + G, c + 2G, ...
// of G CTAs), so the operand rings, the TMEM hand-offs and the next item's
// loads carry on across items instead of every tile paying a cold start.
// The T x T score matrix exists only as 128 x 128 fp32 tiles in tensor
// memory (TMEM). Per key block j (causal: j <= query tile):
//   S = Q K_j^T           tcgen05.mma M=128 N=128 K=64, into TMEM;
//   softmax threads       (thread = query row = TMEM lane) load their S row,
//                         hand the S buffer back, and form
//                         P = exp2(S log2(e)/sqrt(hd) - m) in fp32 with a
//                         per-row reference m, accumulating the row sum l;
//                         P goes back to TMEM as bf16 pairs (tcgen05.st),
//                         32 keys at a time;
//   O += P V_j            tcgen05.mma M=128 N=64 K=128 with P read from TMEM
//                         as the A operand, into a TMEM accumulator.
// The reference m moves only when a row's maximum grows by more than 8 (log2
// units), so P <= 256; when it moves, the row's O (in TMEM) and l are scaled
// by exp2(m_old - m_new) before the next PV MMA. At the end of an item the
// softmax threads read O, hand the accumulator back (the next item's first
// PV may start) and write O / l and the log-sum-exp m + log l.
//
// Warps: 0 TMA producer (Q double-buffered across items, the next item's Q
// loaded while the current one runs; K and V per block, each into a two-stage
// ring, so that K(j+1) never waits for PV(j-1)), 1 TMEM allocation and the
// MMA schedule (run by the whole warp, one elected lane issuing; S of the
// next step is issued before PV of the current one, across item boundaries),
// 2..5 softmax. Every wait is bounded.
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
// shared memory: Q stage 0, 1 | K stage 0, 1 | V stage 0, 1 | barriers
constexpr int AT_OSTG = 2048;             // per softmax warp: 16 rows of O (bf16) on their way out
constexpr int AT_SMEM = 6 * AT_TILE + 4 * AT_OSTG + 256 + 1024;
constexpr uint32_t AT_TMEM_COLS = 256;     // S [0,128), O [128,192), P [192,256) (bf16 pairs)
constexpr float AT_LN2 = 0.6931471805599453f;
constexpr float AT_RESCALE = 8.f;          // log2 of the largest P before the reference max moves

// Work schedule of the persistent attention kernels, over the nqt tiles of
// each of BH batch-heads, where a tile's work (its key or query blocks)
// depends on its rank u: rank 0 is the longest tile, rank nqt-1 the shortest,
// and ranks u and nqt-1-u together make nqt+1 blocks. CTA c of G takes:
//   first R pair rounds: in round r the pair r*G + c, i.e. batch-head
//     (r*G + c) / (nqt/2) and ranks p and nqt-1-p with p = (r*G + c) % (nqt/2),
//     the long one first: every CTA gets the same work, and the CTAs that run
//     at the same time cover all tiles of G/(nqt/2) batch-heads, so the K/V
//     (Q/dO) blocks they share are read while they are still in L2;
//   then the tiles of the remaining batch-heads bh >= bh0, longest first
//     (rank-major), round robin: t = j*G + c is rank t / NB of batch-head
//     bh0 + t % NB (NB = BH - bh0).
// The host chooses R one round short of all the pairs (R = 0 when nqt is odd
// or there are fewer pairs than CTAs), which leaves the tail enough items to
// even out.
struct Sched {
    int BH, nqt, R, bh0;
};

__host__ __device__ inline Sched make_sched(int BH, int nqt, int G) {
    Sched s;
    s.BH = BH;
    s.nqt = nqt;
    s.R = 0;
    if (nqt % 2 == 0) {
        const int np = nqt / 2;
        const int rmax = (int)(((int64_t)BH * np) / G);
        const int r = rmax >= 1 ? rmax - 1 : 0;
        if (r > 0 && ((int64_t)r * G) % np == 0) s.R = r;
    }
    s.bh0 = s.nqt % 2 == 0 && s.R ? (int)(((int64_t)s.R * G) / (s.nqt / 2)) : 0;
    return s;
}

// Item i of this CTA: the tile's rank u (0 = longest) and batch-head, or false.
__device__ __forceinline__ bool sched_item(const Sched& s, int i, int& u, int& bh) {
    const int G = gridDim.x, c = blockIdx.x;
    if (i < 2 * s.R) {
        const int np = s.nqt / 2;
        const int pair = (i >> 1) * G + c;
        bh = pair / np;
        const int p = pair % np;
        u = (i & 1) ? s.nqt - 1 - p : p;
        return true;
    }
    const int NB = s.BH - s.bh0;
    const int t = (i - 2 * s.R) * G + c;
    if (t >= NB * s.nqt) return false;
    u = t / NB;
    bh = s.bh0 + t % NB;
    return true;
}

struct FwdArgs {
    bf16* o;       // [B*T, C]
    float* lse;    // [B, H, T]
    int* status;
    int T, C, H;
    int nqt;       // 128-query tiles per sequence
    Sched sched;
    float scale_log2;  // log2(e) / sqrt(hd)
};

// Work item i of this CTA: query tile (rank u is tile nqt-1-u: the last
// query tile has the most key blocks) and batch-head.
struct FItem {
    int qt, bh;
};
__device__ __forceinline__ bool fwd_item(const FwdArgs& a, int i, FItem& it) {
    int u;
    if (!sched_item(a.sched, i, u, it.bh)) return false;
    it.qt = a.nqt - 1 - u;
    return true;
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// (lo, hi) rounded to a packed bf16 pair, lo in the low half.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
// A packed bf16 pair as a packed fp32 pair (low half first).
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t p) { return f2_pack(p << 16, p & 0xFFFF0000u); }


__global__ void __launch_bounds__(AT_THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, FwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    auto sQ = [&](int st) { return base + st * AT_TILE; };
    auto sK = [&](int st) { return base + (2 + st) * AT_TILE; };
    auto sV = [&](int st) { return base + (4 + st) * AT_TILE; };
    uint8_t* ostg = gbase + 6 * AT_TILE;  // [4 softmax warps][AT_OSTG]
    const uint32_t bars = base + 6 * AT_TILE + 4 * AT_OSTG;
    uint8_t* bar_area = gbase + 6 * AT_TILE + 4 * AT_OSTG;
    // barriers: q_full[2], q_empty[2], k_full[2], k_empty[2], v_full[2], v_empty[2], s_full, s_free,
    // p_full, p_free, o_done, o_free, drain
    auto q_full = [&](int i) { return bars + 8u * (0 + i); };
    auto q_empty = [&](int i) { return bars + 8u * (2 + i); };
    auto k_full = [&](int i) { return bars + 8u * (4 + i); };
    auto k_empty = [&](int i) { return bars + 8u * (6 + i); };
    auto v_full = [&](int i) { return bars + 8u * (8 + i); };
    auto v_empty = [&](int i) { return bars + 8u * (10 + i); };
    const uint32_t s_full = bars + 8u * 12, s_free = bars + 8u * 13;
    const uint32_t p_full = bars + 8u * 14, p_free = bars + 8u * 15;
    const uint32_t o_done = bars + 8u * 16, o_free = bars + 8u * 17, drain = bars + 8u * 18;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * 19);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * 19 + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; i++) {
            mbar_init(q_full(i), 1);
            mbar_init(q_empty(i), 1);
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(p_free, 1);
        mbar_init(o_done, 1);
        mbar_init(o_free, 4);
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
            // Q of item i into stage i & 1 once item i - 2 has finished with
            // it; K and V of the g-th block (over all items) into stage g & 1.
            int q_issued[2] = {-1, -1}, k_issued[2] = {-1, -1}, v_issued[2] = {-1, -1};
            auto load_q = [&](int i, const FItem& it) -> bool {
                const int st = i & 1;
                const uint32_t ph = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(q_empty(st), ph ^ 1u, abort_flag, a.status)) return false;
                mbar_expect_tx(q_full(st), AT_TILE);
                tma_load_3d(sQ(st), &tm_qkv, q_full(st), (it.bh % a.H) * AT_HD, it.qt * AT_M, it.bh / a.H);
                q_issued[st] = (int)ph;
                return true;
            };
            FItem it;
            bool ok = !fwd_item(a, 0, it) || load_q(0, it);
            int g = 0;
            for (int i = 0; ok && fwd_item(a, i, it); i++) {
                const int b = it.bh / a.H, h = it.bh % a.H;
                for (int j = 0; j <= it.qt; j++, g++) {
                    const int st = g & 1;
                    const uint32_t ph = (uint32_t)(g >> 1) & 1u;
                    if (!(ok = mbar_wait(k_empty(st), ph ^ 1u, abort_flag, a.status))) break;
                    mbar_expect_tx(k_full(st), AT_TILE);
                    tma_load_3d(sK(st), &tm_qkv, k_full(st), a.C + h * AT_HD, j * AT_N, b);
                    k_issued[st] = (int)ph;
                    // V(g) once PV(g-2) has read the stage
                    if (!(ok = mbar_wait(v_empty(st), ph ^ 1u, abort_flag, a.status))) break;
                    mbar_expect_tx(v_full(st), AT_TILE);
                    tma_load_3d(sV(st), &tm_qkv, v_full(st), 2 * a.C + h * AT_HD, j * AT_N, b);
                    v_issued[st] = (int)ph;
                    // the next item's Q after this item's first K/V block
                    FItem nit;
                    if (j == 0 && fwd_item(a, i + 1, nit) && !(ok = load_q(i + 1, nit))) break;
                }
            }
            for (int st = 0; st < 2; st++) {
                if (q_issued[st] >= 0) mbar_drain(q_full(st), (uint32_t)q_issued[st], a.status);
                if (k_issued[st] >= 0) mbar_drain(k_full(st), (uint32_t)k_issued[st], a.status);
                if (v_issued[st] >= 0) mbar_drain(v_full(st), (uint32_t)v_issued[st], a.status);
            }
        }
    } else if (warp == 1) {
        {
            // -------------------------------------------------- MMA issuer: the
            // whole warp runs the schedule (warp-uniform operands), one elected
            // lane issues the MMAs and commits
            const bool leader = elect_one();
            constexpr uint32_t idesc_s = make_idesc(AT_M, AT_N, false, false);
            constexpr uint32_t idesc_o = make_idesc(AT_M, AT_HD, false, true);
            // S(g) = Q(i) K(g)^T for block j of item i; the K stage is free once
            // these MMAs finish, the Q stage after the item's last block
            auto issue_s = [&](int i, int j, int last, int g) -> bool {
                const int st = g & 1;
                if (j == 0 && !warp_wait(q_full(i & 1), (i >> 1) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(k_full(st), (g >> 1) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(s_free, (g & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint32_t q = sQ(i & 1);
                if (leader) {
#pragma unroll
                    for (int k = 0; k < AT_HD / 16; k++)
                        tc_mma(tmem, sw128_desc(q + k * 32, 16, 1024), sw128_desc(sK(st) + k * 32, 16, 1024), idesc_s,
                               k > 0 ? 1u : 0u);
                }
                if (leader) tc_commit(s_full);
                if (leader) tc_commit(k_empty(st));
                if (leader && j == last) tc_commit(q_empty(i & 1));
                return true;
            };
            FItem it;
            bool ok = fwd_item(a, 0, it);
            int i = 0, j = 0, g = 0;
            if (ok) ok = issue_s(0, 0, it.qt, 0);
            while (ok) {
                // the step after (i, j): S for it is issued before PV(i, j)
                int ni = i, nj = j + 1;
                FItem nit = it;
                bool more = true;
                if (nj > it.qt) {
                    ni = i + 1;
                    nj = 0;
                    more = fwd_item(a, ni, nit);
                }
                if (more && !(ok = issue_s(ni, nj, nit.qt, g + 1))) break;
                // O += P(g) V(g); an item's first PV waits for the previous item's O to be read
                if (!(ok = warp_wait(p_full, g & 1, abort_flag, a.status))) break;
                if (!(ok = warp_wait(v_full(g & 1), (g >> 1) & 1, abort_flag, a.status))) break;
                if (j == 0 && i > 0 && !(ok = warp_wait(o_free, (i - 1) & 1, abort_flag, a.status))) break;
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < AT_N / 16; kk++)
                        tc_mma_ts(tmem + 128u, tmem + 192u + kk * 8, sw128_desc(sV(g & 1) + kk * 2048, 8192, 1024),
                                  idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                }
                if (leader) tc_commit(p_free);
                if (leader) tc_commit(v_empty(g & 1));
                if (leader && j == it.qt) tc_commit(o_done);
                if (!more) break;
                i = ni;
                j = nj;
                it = nit;
                g++;
            }
            if (leader) tc_commit(drain);
            mbar_drain(drain, 0, a.status);
        }
    } else {
        // ------------------------------------------------------ softmax (warps 2..5)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;  // row in the tile = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        const uint64_t scale2 = f2_pack(a.scale_log2, a.scale_log2);
        bool ok = true;
        FItem it;
        int g = 0;
        for (int i = 0; ok && fwd_item(a, i, it); i++) {
            const int q = it.qt * AT_M + r;  // query position
            float m = -FLT_MAX, l = 0.f;
            for (int j = 0; j <= it.qt; j++, g++) {
                uint32_t v[4][32];
                if (!(ok = warp_wait(s_full, g & 1, abort_flag, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 4; c++) tc_ld32_issue(trow + (uint32_t)(c * 32), v[c]);
#pragma unroll
                for (int c = 0; c < 4; c++) tc_ld_wait(v[c]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);  // the MMA may now write the next S
                // The row maximum of the raw scores (the scale is positive), with
                // the keys after the query masked to -FLT_MAX on the diagonal block;
                // four independent three-input maxima keep the chains short.
                if (j == it.qt) {
#pragma unroll
                    for (int c = 0; c < 4; c++)
#pragma unroll
                        for (int e = 0; e < 32; e++)
                            if (j * AT_N + c * 32 + e > q) v[c][e] = __float_as_uint(-FLT_MAX);
                }
                float m4[4] = {-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX};
#pragma unroll
                for (int c = 0; c < 4; c++)
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(v[c][e]), __uint_as_float(v[c][e + 1]));
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * a.scale_log2;
                // move the reference max only when it grew by more than AT_RESCALE
                float factor = 1.f;
                const bool move = mx > m + AT_RESCALE;
                if (move) {
                    factor = ex2_approx(m - mx);  // 0 on the first block (m = -FLT_MAX)
                    m = mx;
                    l *= factor;
                }
                // PV of the previous step has finished with the P buffer and O
                if (!(ok = warp_wait(p_free, (g & 1) ^ 1u, abort_flag, a.status))) break;
                tc_fence_after();
                // P = exp2(s scale - m), 32 keys at a time into TMEM as bf16
                // pairs (pk[e/2] holds keys c*32+e, c*32+e+1), the row sum in
                // four paired fp32 accumulators
                const uint64_t nm2 = f2_pack(-m, -m);
                uint64_t l2[4] = {0, 0, 0, 0};
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(v[c][e], v[c][e + 1]), scale2, nm2), x0, x1);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        l2[(e >> 1) & 3] = f2_add(l2[(e >> 1) & 3], f2_pack(p0, p1));
                        pk[e / 2] = cvt_bf16x2(p0, p1);
                    }
                    tc_st16(trow + 192u + (uint32_t)(c * 16), pk);
                }
                {
                    float s0, s1, s2, s3, s4, s5, s6, s7;
                    f2_unpack(l2[0], s0, s1);
                    f2_unpack(l2[1], s2, s3);
                    f2_unpack(l2[2], s4, s5);
                    f2_unpack(l2[3], s6, s7);
                    l += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
                }
                // O rescaled (once the scores' registers are free) before PV reads it
                if (j > 0 && __any_sync(0xffffffffu, move)) {
#pragma unroll
                    for (int half = 0; half < 2; half++) {
                        uint32_t ov[32];
                        tc_ld32_issue(trow + 128u + half * 32, ov);
                        tc_ld_wait(ov);
#pragma unroll
                        for (int e = 0; e < 32; e++) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
                        tc_st32(trow + 128u + half * 32, ov);
                    }
                }
                tc_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
            if (!ok) break;
            // O / l, log-sum-exp; O is handed back once it is in registers
            if (!(ok = warp_wait(o_done, i & 1, abort_flag, a.status))) break;
            tc_fence_after();
            uint32_t ov[2][32];
            tc_ld32_issue(trow + 128u, ov[0]);
            tc_ld32_issue(trow + 160u, ov[1]);
            tc_ld_wait(ov[0]);
            tc_ld_wait(ov[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            {
                // O / l as bf16 pairs (pk[u]: columns 2u, 2u + 1), out through
                // this warp's staging buffer 16 rows at a time (chunk c of
                // staged row s at (c ^ (s & 7)) * 16: conflict-free both ways),
                // so that each global store covers four whole 128-byte rows
                const int b = it.bh / a.H, h = it.bh % a.H;
                const float inv = 1.f / l;
                uint32_t pk[32];
#pragma unroll
                for (int u = 0; u < 32; u++)
                    pk[u] = cvt_bf16x2(__uint_as_float(ov[u >> 4][(u & 15) * 2]) * inv,
                                       __uint_as_float(ov[u >> 4][(u & 15) * 2 + 1]) * inv);
                uint8_t* st = ostg + (warp - 2) * AT_OSTG;
                bf16* obase = a.o + (int64_t)b * a.T * a.C + h * AT_HD;
                const int q0 = it.qt * AT_M + quad * 32;  // the warp's first row
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    __syncwarp();  // the previous rows have been read out
                    if ((lane >> 4) == hh) {
                        const int sr = lane & 15;
#pragma unroll
                        for (int c = 0; c < 8; c++)
                            *reinterpret_cast<uint4*>(st + sr * 128 + ((c ^ (sr & 7)) << 4)) =
                                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int sr = i * 4 + (lane >> 3), c = lane & 7;
                        const int qr = q0 + 16 * hh + sr;
                        const uint4 v = *reinterpret_cast<const uint4*>(st + sr * 128 + ((c ^ (sr & 7)) << 4));
                        if (qr < a.T) *reinterpret_cast<uint4*>(obase + (int64_t)qr * a.C + c * 8) = v;
                    }
                }
                if (q < a.T) a.lse[(int64_t)it.bh * a.T + q] = (m + log2f(l)) * AT_LN2;
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

int attention_tc_set_wait_limit(long long cycles) { return set_wait_limit(cycles); }

// bf16 forward, head size 64 (the attention.cu launcher routes here).
int launch_attention_forward_tc(bf16* o, float* lse, const bf16* qkv, int B, int T, int C, int H, int* status,
                                cudaStream_t s) {
    CUtensorMap map;
    if (!make_qkv_map(&map, qkv, B, T, C)) return GPT2_ERR_CUDA;
    smem_attr((const void*)attn_fwd_tc_kernel, AT_SMEM);
    FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.status = status;
    a.T = T;
    a.C = C;
    a.H = H;
    a.nqt = (T + AT_M - 1) / AT_M;
    const int items = a.nqt * B * H;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)(C / H));
    const int grid = items < 2 * gpt2_num_sms() ? items : 2 * gpt2_num_sms();  // persistent: two CTAs per SM
    a.sched = make_sched(B * H, a.nqt, grid);
    attn_fwd_tc_kernel<<<grid, AT_THREADS, AT_SMEM, s>>>(map, a);
    return 1;
}

// =============================================================================
// Attention backward on tcgen05 (bf16, head size 64), two deterministic
// kernels: dK, dV with a 128-key tile as the work item, and dQ with a
// 128-query tile.
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
// P^T and dS^T (dS) go back into tensor memory as bf16 pairs (tcgen05.st),
// and the dV, dK and dQ products read them from there as their A operand, so
// the only shared-memory operands are the Q, dO, K and V tiles the TMA loads.
//
// Both are persistent (one CTA per SM walking a list of (tile, batch-head)
// items, longest first), so the operand rings and the MMA / elementwise
// hand-offs carry on across items; an item's accumulators go from TMEM to
// global memory while the next item's first products are computed.
// Warps: 0 TMA producer (lane 0; an item's K/V (dQ kernel: Q/dO) tiles are
// loaded while the item before it runs); 1 MMA issuer (the whole warp, one
// elected lane issuing); 2..17 elementwise (warp w serves TMEM lanes 32*(w%4)..
// and one quarter, 32, of the 128 columns: four warps per scheduler, so that
// the exp / multiply chains of one warp hide the latencies of the others);
// 18 sends an item's accumulators, which the elementwise warps stage in shared
// memory as bf16, to global memory with TMA stores. One CTA per SM (512 TMEM
// columns).
// =============================================================================

namespace {

constexpr int BW_EW = 16;                        // elementwise warps
constexpr int BW_STORE_WARP = 2 + BW_EW;          // issues the TMA stores of the accumulators
constexpr int BW_THREADS = 32 * (BW_STORE_WARP + 1);  // + producer, MMA and store warps
constexpr int EW_COLS = 32;                 // columns of a 128-wide tile per elementwise thread
constexpr int DKDV_ST = 3;   // Q/dO stages of the dK/dV kernel
constexpr int DQ_ST = 4;     // K/V stages of the dQ kernel
// TMEM columns. dK/dV kernel: S^T, dP^T (fp32), dV, dK (fp32), P^T, dS^T
// (bf16 pairs: 128 queries in 64 columns).
constexpr uint32_t KV_S = 0, KV_DP = 128, KV_DV = 256, KV_DK = 320, KV_P = 384, KV_DS = 448;
// dQ kernel: S, dP (fp32), dQ (fp32), dS (bf16 pairs).
constexpr uint32_t Q_S = 0, Q_DP = 128, Q_DQ = 256, Q_DS = 320;

struct BwdArgs {
    bf16* dqkv;          // [B*T, 3C]
    const float* lse;    // [B, H, T]
    const float* D;      // [B, H, T]: read by the dK/dV kernel
    float* Dw;           // the same buffer: written by the dQ kernel
    int* status;
    int B, T, C, H;
    int nqt;             // 128-row tiles per sequence
    Sched sched;
    float scale_log2;    // log2(e) / sqrt(hd)
    float scale;         // 1 / sqrt(hd)
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// A warp's 32 x 32 block of an accumulator (lane = row, 32 fp32 columns, as a
// 32x32b TMEM load leaves it), times s, as bf16 into row `row`, 16-byte units
// 4 * half .. 4 * half + 3, of a 128-row x 128-byte tile laid out with the
// 128-byte swizzle (unit u of row r at u ^ (r & 7)): the layout a tensor map
// with SWIZZLE_128B stores from.
__device__ __forceinline__ void stage_block_sw128(uint8_t* tile, int row, int half, const uint32_t (&v)[32],
                                                  float s) {
#pragma unroll
    for (int u = 0; u < 4; u++) {
        uint4 w;
        w.x = pack2(__uint_as_float(v[8 * u + 0]) * s, __uint_as_float(v[8 * u + 1]) * s);
        w.y = pack2(__uint_as_float(v[8 * u + 2]) * s, __uint_as_float(v[8 * u + 3]) * s);
        w.z = pack2(__uint_as_float(v[8 * u + 4]) * s, __uint_as_float(v[8 * u + 5]) * s);
        w.w = pack2(__uint_as_float(v[8 * u + 6]) * s, __uint_as_float(v[8 * u + 7]) * s);
        *reinterpret_cast<uint4*>(tile + row * 128 + (((half * 4 + u) ^ (row & 7)) << 4)) = w;
    }
}

// -------------------------------------------------------------------------- schedule
// Both kernels are persistent: CTA c takes its work items from the schedule
// of sched_item (pairs of a long and a short tile of one batch-head, then a
// longest-first tail), and its producer, MMA and elementwise roles walk the
// same sequence of (item, block) steps, so the operand rings run on across
// item boundaries instead of starting cold.
struct Item {
    int tile, bh, nblk;  // dK/dV: key tile, blocks tile..nqt-1; dQ: query tile, blocks 0..tile
};

template <bool DQ> __device__ __forceinline__ bool get_item(const BwdArgs& a, int i, Item& it) {
    int u;
    if (!sched_item(a.sched, i, u, it.bh)) return false;
    if (DQ) {
        it.tile = a.nqt - 1 - u;  // the last query tile has the most key blocks
        it.nblk = it.tile + 1;
    } else {
        it.tile = u;  // the first key tile has the most query blocks
        it.nblk = a.nqt - it.tile;
    }
    return true;
}

// Position in a CTA's step sequence: item i, block n of it, step counter g.
struct Cur {
    int i, n, g;
    bool valid;
    Item it;
};
template <bool DQ> __device__ __forceinline__ Cur cur_first(const BwdArgs& a) {
    Cur c;
    c.i = 0;
    c.n = 0;
    c.g = 0;
    c.valid = get_item<DQ>(a, 0, c.it);
    return c;
}
template <bool DQ> __device__ __forceinline__ Cur cur_next(const BwdArgs& a, Cur c) {
    c.g++;
    if (++c.n >= c.it.nblk) {
        c.i++;
        c.n = 0;
        c.valid = get_item<DQ>(a, c.i, c.it);
    }
    return c;
}

// -------------------------------------------------------------------------- dK, dV
// Shared memory: 2 x (K, V) (an item's tile and the next one's) | DKDV_ST x
// (Q, dO) | dV, dK staging tiles for the TMA stores | per elementwise warp 64
// floats (its columns' lse and D) | barriers.
__global__ void __launch_bounds__(BW_THREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                            const __grid_constant__ CUtensorMap tm_dqkv, BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    constexpr int NS = DKDV_ST;
    // item i uses K/V buffer i & 1 (its (i >> 1)-th use)
    auto sK = [&](int b) { return base + (2 * b) * AT_TILE; };
    auto sV = [&](int b) { return base + (2 * b + 1) * AT_TILE; };
    auto sQ = [&](int st) { return base + (4 + 2 * st) * AT_TILE; };
    auto sO = [&](int st) { return base + (5 + 2 * st) * AT_TILE; };
    uint8_t* stg = gbase + (4 + 2 * NS) * AT_TILE;  // dV tile, then the dK tile
    const uint32_t stg_addr = base + (4 + 2 * NS) * AT_TILE;
    float* ldslots = reinterpret_cast<float*>(gbase + (6 + 2 * NS) * AT_TILE);  // [BW_EW][64]
    const uint32_t bars = base + (6 + 2 * NS) * AT_TILE + BW_EW * 256;
    uint8_t* bar_area = gbase + (6 + 2 * NS) * AT_TILE + BW_EW * 256;
    auto k_full = [&](int b) { return bars + 8u * b; };
    auto k_empty = [&](int b) { return bars + 8u * (2 + b); };
    auto v_full = [&](int b) { return bars + 8u * (4 + b); };
    auto v_empty = [&](int b) { return bars + 8u * (6 + b); };
    auto qd_full = [&](int i) { return bars + 8u * (8 + i); };
    auto qd_empty = [&](int i) { return bars + 8u * (8 + NS + i); };
    const uint32_t bx = bars + 8u * (8 + 2 * NS);
    const uint32_t s_full = bx, s_free = bx + 8u;
    const uint32_t dp_full = bx + 16u, dp_free = bx + 24u;
    const uint32_t p_full = bx + 32u;
    const uint32_t ds_full = bx + 48u, ds_free = bx + 56u;
    const uint32_t acc_full = bx + 64u, acc_empty = bx + 72u, drain = bx + 80u;
    const uint32_t stg_free = bx + 88u, stg_full = bx + 96u;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * (8 + 2 * NS) + 104);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (8 + 2 * NS) + 108);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; b++) {
            mbar_init(k_full(b), 1);
            mbar_init(k_empty(b), 1);
            mbar_init(v_full(b), 1);
            mbar_init(v_empty(b), 1);
        }
        for (int i = 0; i < NS; i++) {
            mbar_init(qd_full(i), 1);
            mbar_init(qd_empty(i), 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, BW_EW);
        mbar_init(dp_full, 1);
        mbar_init(dp_free, BW_EW);
        mbar_init(p_full, BW_EW);
        mbar_init(ds_full, BW_EW);
        mbar_init(ds_free, 1);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, BW_EW);
        mbar_init(drain, 1);
        mbar_init(stg_free, 1);
        mbar_init(stg_full, BW_EW);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_addr((const void*)tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;  // columns KV_*

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------------- TMA producer
            int qd_issued[NS], kv_issued[2] = {-1, -1};  // parity of each buffer's last load (final drain)
            for (int i = 0; i < NS; i++) qd_issued[i] = -1;
            int g = 0;
            // K and V of item i into buffer i & 1, once the item before last has
            // finished with it
            auto load_kv = [&](int i, const Item& it) -> bool {
                const int b = it.bh / a.H, h = it.bh % a.H;
                const int kb = i & 1;
                const uint32_t kph = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(k_empty(kb), kph ^ 1u, abort_flag, a.status)) return false;
                mbar_expect_tx(k_full(kb), AT_TILE);
                tma_load_3d(sK(kb), &tm_qkv, k_full(kb), a.C + h * AT_HD, it.tile * AT_N, b);
                if (!mbar_wait(v_empty(kb), kph ^ 1u, abort_flag, a.status)) return false;
                mbar_expect_tx(v_full(kb), AT_TILE);
                tma_load_3d(sV(kb), &tm_qkv, v_full(kb), 2 * a.C + h * AT_HD, it.tile * AT_N, b);
                kv_issued[kb] = (int)kph;
                return true;
            };
            Item it0;
            bool ok = !get_item<false>(a, 0, it0) || load_kv(0, it0);
            for (int i = 0; ok; i++) {
                Item it;
                if (!get_item<false>(a, i, it)) break;
                const int b = it.bh / a.H, h = it.bh % a.H;
                auto load_qd = [&](int n) -> bool {
                    const int st = g % NS;
                    const uint32_t ph = (g / NS) & 1;
                    if (!mbar_wait(qd_empty(st), ph ^ 1u, abort_flag, a.status)) return false;
                    mbar_expect_tx(qd_full(st), 2 * AT_TILE);
                    tma_load_3d(sQ(st), &tm_qkv, qd_full(st), h * AT_HD, (it.tile + n) * AT_M, b);
                    tma_load_3d(sO(st), &tm_do, qd_full(st), h * AT_HD, (it.tile + n) * AT_M, b);
                    qd_issued[st] = (int)ph;
                    g++;
                    return true;
                };
                // the item's first Q/dO block, then the next item's K and V (a
                // whole item ahead of their first use), then the other blocks
                if (!(ok = load_qd(0))) break;
                Item nit;
                if (get_item<false>(a, i + 1, nit) && !(ok = load_kv(i + 1, nit))) break;
                for (int n = 1; ok && n < it.nblk; n++) ok = load_qd(n);
            }
            for (int kb = 0; kb < 2; kb++)
                if (kv_issued[kb] >= 0) {
                    mbar_drain(k_full(kb), (uint32_t)kv_issued[kb], a.status);
                    mbar_drain(v_full(kb), (uint32_t)kv_issued[kb], a.status);
                }
            for (int st = 0; st < NS; st++)
                if (qd_issued[st] >= 0) mbar_drain(qd_full(st), (uint32_t)qd_issued[st], a.status);
        }
    } else if (warp == 1) {
        {
            // -------------------------------------------------- MMA issuer: the
            // whole warp runs the schedule (warp-uniform operands), one elected
            // lane issues the MMAs and commits
            const bool leader = elect_one();
            constexpr uint32_t idesc_s = make_idesc(AT_M, AT_N, false, false);  // K-major x K-major
            constexpr uint32_t idesc_o = make_idesc(AT_M, AT_HD, false, true);  // K-major x MN-major
            auto issue_s = [&](const Cur& x) -> bool {  // S^T = K Q^T
                const int st = x.g % NS, kb = x.i & 1;
                if (x.n == 0 && !warp_wait(k_full(kb), (x.i >> 1) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(qd_full(st), (x.g / NS) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(s_free, (x.g & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
                // one 16-wide k step = 32 bytes = 2 units of the descriptors' address field
                const uint64_t da = sw128_desc(sK(kb), 16, 1024), db = sw128_desc(sQ(st), 16, 1024);
                if (leader) {
#pragma unroll
                    for (int k = 0; k < 4; k++) tc_mma(tmem + KV_S, da + 2 * k, db + 2 * k, idesc_s, k > 0 ? 1u : 0u);
                }
                if (leader) tc_commit(s_full);
                if (leader && x.n == x.it.nblk - 1) tc_commit(k_empty(kb));  // the item's last read of K
                return true;
            };
            auto issue_dp = [&](const Cur& x) -> bool {  // dP^T = V dO^T
                const int st = x.g % NS, kb = x.i & 1;
                if (x.n == 0 && !warp_wait(v_full(kb), (x.i >> 1) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(dp_free, (x.g & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint64_t da = sw128_desc(sV(kb), 16, 1024), db = sw128_desc(sO(st), 16, 1024);
                if (leader) {
#pragma unroll
                    for (int k = 0; k < 4; k++) tc_mma(tmem + KV_DP, da + 2 * k, db + 2 * k, idesc_s, k > 0 ? 1u : 0u);
                }
                if (leader) tc_commit(dp_full);
                if (leader && x.n == x.it.nblk - 1) tc_commit(v_empty(kb));  // the item's last read of V
                return true;
            };
            Cur c = cur_first<false>(a);
            bool ok = !c.valid || (issue_s(c) && issue_dp(c));
            while (ok && c.valid) {
                const Cur nx = cur_next<false>(a, c);
                const int st = c.g % NS;
                if (nx.valid && !(ok = issue_s(nx))) break;
                // dV += P^T dO (the first block of an item starts the accumulator
                // once the elementwise warps have stored the previous item's)
                if (!(ok = warp_wait(p_full, c.g & 1, abort_flag, a.status))) break;
                if (c.n == 0 && c.i > 0 && !(ok = warp_wait(acc_empty, (c.i - 1) & 1, abort_flag, a.status))) break;
                tc_fence_after();
                // MN-major B: one 16-row k step = 2048 bytes = 128 units of the address field
                const uint64_t dbo = sw128_desc(sO(st), 8192, 1024);
                const uint32_t acc0 = c.n > 0 ? 1u : 0u;
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)
                        tc_mma_ts(tmem + KV_DV, tmem + KV_P + kk * 8, dbo + 128 * kk, idesc_o, kk > 0 ? 1u : acc0);
                }
                if (nx.valid && !(ok = issue_dp(nx))) break;
                // dK += dS^T Q
                if (!(ok = warp_wait(ds_full, c.g & 1, abort_flag, a.status))) break;
                tc_fence_after();
                const uint64_t dbq = sw128_desc(sQ(st), 8192, 1024);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)
                        tc_mma_ts(tmem + KV_DK, tmem + KV_DS + kk * 8, dbq + 128 * kk, idesc_o, kk > 0 ? 1u : acc0);
                }
                if (leader) tc_commit(ds_free);
                if (leader) tc_commit(qd_empty(st));
                if (leader && c.n == c.it.nblk - 1) tc_commit(acc_full);  // the item's dV and dK are complete
                c = nx;
            }
            if (leader) tc_commit(drain);
            mbar_drain(drain, 0, a.status);
        }
    } else if (warp == BW_STORE_WARP) {
        // ------------------------------------------------------ accumulator stores
        // item f's dV and dK tiles, once the elementwise warps have staged them
        Item it;
        for (int f = 0; get_item<false>(a, f, it); f++) {
            if (!warp_wait(stg_full, f & 1, abort_flag, a.status)) break;
            if (lane == 0) {
                const int b = it.bh / a.H, h = it.bh % a.H;
                tma_store_3d(&tm_dqkv, stg_addr, 2 * a.C + h * AT_HD, it.tile * AT_N, b);        // dV
                tma_store_3d(&tm_dqkv, stg_addr + AT_TILE, a.C + h * AT_HD, it.tile * AT_N, b);  // dK
                bulk_wait_read_all();  // the tiles may be written again
                mbar_arrive(stg_free);
            }
            __syncwarp();
        }
        if (lane == 0) bulk_wait_all();  // the stores are complete before the CTA ends
    } else {
        // ------------------------------------------------------ elementwise (warps 2..17)
        const int ew = warp - 2;
        const int quad = warp & 3, part = ew >> 2;
        const int r = quad * 32 + lane;  // key row within the tile = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        float* slot = ldslots + ew * 64;  // [0,32): -lse * log2(e), [32,64): D of this warp's 32 queries
        // lse and D of query column part*32 + lane of a step's block, loaded a
        // step ahead and used as they are (no arithmetic waits on the loads
        // until the step they belong to); `in` says whether the query is < T
        auto load_ld = [&](const Cur& x, float& l, float& d, bool& in) {
            const int q = (x.it.tile + x.n) * AT_M + part * EW_COLS + lane;
            in = q < a.T;
            const int64_t o = (int64_t)x.it.bh * a.T + (in ? q : 0);
            l = a.lse[o];
            d = a.D[o];
        };
        const uint64_t scale2 = f2_pack(a.scale_log2, a.scale_log2);
        // An item's dV and dK leave TMEM during the next item's first step,
        // once its exponentials are done, so the last dK product of the item
        // runs while they are computed. Parts 0, 1 hold dV columns part*32..,
        // parts 2, 3 dK columns (part-2)*32..; each warp hands TMEM back and
        // writes its block into the staging tiles (once the store warp has sent
        // the previous item's out), and the store warp sends both tiles out.
        int pend_i = -1, nflush = 0;
        auto flush = [&]() -> bool {
            if (!warp_wait(acc_full, pend_i & 1, abort_flag, a.status)) return false;
            tc_fence_after();
            const bool is_dk = part >= 2;
            const int half = part & 1;
            uint32_t acc[32];
            tc_ld32_issue(trow + (is_dk ? KV_DK : KV_DV) + (uint32_t)(half * 32), acc);
            tc_ld_wait(acc);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            if (!warp_wait(stg_free, (nflush & 1) ^ 1u, abort_flag, a.status)) return false;
            stage_block_sw128(stg + (is_dk ? AT_TILE : 0), r, half, acc, is_dk ? a.scale : 1.f);
            fence_proxy_async_smem();  // the writes, visible to the TMA
            __syncwarp();
            if (lane == 0) mbar_arrive(stg_full);
            nflush++;
            pend_i = -1;
            return true;
        };
        Cur c = cur_first<false>(a);
        float l_nx = 0.f, d_nx = 0.f;
        bool in_nx = false;
        if (c.valid) load_ld(c, l_nx, d_nx, in_nx);
        bool ok = true;
        while (c.valid) {
            const Cur nx = cur_next<false>(a, c);
            const int g = c.g;
            const int key = c.it.tile * AT_N + r;
            const int q0 = (c.it.tile + c.n) * AT_M + part * EW_COLS;  // first query of this thread's columns
            const bool diag = c.n == 0;
            __syncwarp();  // every lane is done with the previous step's slot
            slot[lane] = in_nx ? -l_nx * 1.4426950408889634f : 0.f;  // 0 past the sequence end
            slot[32 + lane] = in_nx ? d_nx : 0.f;
            __syncwarp();
            if (nx.valid) load_ld(nx, l_nx, d_nx, in_nx);  // the next step's, in flight meanwhile
            uint32_t sv[32];
            if (!(ok = warp_wait(s_full, g & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + KV_S + (uint32_t)(part * EW_COLS), sv);
            tc_ld_wait(sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            // P^T = exp2(S^T scale - lse); the mask is needed only on the
            // diagonal block (query < key) and past the sequence end
            float p[EW_COLS];
            uint32_t pk[EW_COLS / 2];
            const uint64_t* nl2 = reinterpret_cast<const uint64_t*>(slot);
            if (diag || q0 + EW_COLS > a.T) {
                const int lo = diag ? key - q0 : 0, hi = a.T - q0;  // valid columns [lo, hi)
#pragma unroll
                for (int cc = 0; cc < EW_COLS; cc += 2) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(sv[cc], sv[cc + 1]), scale2, nl2[cc / 2]), x0, x1);
                    p[cc] = (cc >= lo && cc < hi) ? ex2_approx(x0) : 0.f;
                    p[cc + 1] = (cc + 1 >= lo && cc + 1 < hi) ? ex2_approx(x1) : 0.f;
                    pk[cc / 2] = cvt_bf16x2(p[cc], p[cc + 1]);
                }
            } else {
#pragma unroll
                for (int cc = 0; cc < EW_COLS; cc += 2) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(sv[cc], sv[cc + 1]), scale2, nl2[cc / 2]), x0, x1);
                    p[cc] = ex2_approx(x0);
                    p[cc + 1] = ex2_approx(x1);
                    pk[cc / 2] = cvt_bf16x2(p[cc], p[cc + 1]);
                }
            }
            // the previous step's P^T and dS^T have been read: its dK product,
            // issued after its dV product, is complete (one wait covers both stores)
            if (!(ok = warp_wait(ds_free, (g & 1) ^ 1u, abort_flag, a.status))) break;
            tc_st16(trow + KV_P + (uint32_t)(part * EW_COLS / 2), pk);
            tc_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            if (pend_i >= 0 && !(ok = flush())) break;
            // dS^T = P^T (dP^T - D)
            if (!(ok = warp_wait(dp_full, g & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + KV_DP + (uint32_t)(part * EW_COLS), sv);
            tc_ld_wait(sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_free);
            const uint64_t* d2 = reinterpret_cast<const uint64_t*>(slot + 32);
            uint32_t dk[EW_COLS / 2];
#pragma unroll
            for (int cc = 0; cc < EW_COLS; cc += 2) {
                float d0, d1;
                f2_unpack(f2_mul(f2_pack(p[cc], p[cc + 1]), f2_sub(f2_pack(sv[cc], sv[cc + 1]), d2[cc / 2])), d0, d1);
                dk[cc / 2] = cvt_bf16x2(d0, d1);
            }
            tc_st16(trow + KV_DS + (uint32_t)(part * EW_COLS / 2), dk);
            tc_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
            if (c.n == c.it.nblk - 1) pend_i = c.i;
            c = nx;
        }
        if (ok && pend_i >= 0) flush();
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
// Shared memory: 2 x (Q, dO) (an item's tile and the next one's) | DQ_ST x
// (K, V) | dQ staging tile for the TMA store | the forward's output O tile of
// an item | D of two items (128 floats each) | barriers.
// This kernel runs first and also forms D = rowsum(dO * O) of every query
// (its store warp, from the dO and O tiles, one item ahead), which it uses
// itself and writes for the dK/dV kernel.
__global__ void __launch_bounds__(BW_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                          const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_dqkv,
                          BwdArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    constexpr int NS = DQ_ST;
    // item i uses Q/dO buffer i & 1 (its (i >> 1)-th use)
    auto sQ = [&](int b) { return base + (2 * b) * AT_TILE; };
    auto sO = [&](int b) { return base + (2 * b + 1) * AT_TILE; };
    auto sK = [&](int st) { return base + (4 + 2 * st) * AT_TILE; };
    auto sV = [&](int st) { return base + (5 + 2 * st) * AT_TILE; };
    uint8_t* stg = gbase + (4 + 2 * NS) * AT_TILE;
    const uint32_t stg_addr = base + (4 + 2 * NS) * AT_TILE;
    const uint32_t sX = base + (5 + 2 * NS) * AT_TILE;  // O of the forward
    const uint8_t* xtile = gbase + (5 + 2 * NS) * AT_TILE;
    float* dslot = reinterpret_cast<float*>(gbase + (6 + 2 * NS) * AT_TILE);  // [2][128]
    const uint32_t bars = base + (6 + 2 * NS) * AT_TILE + 1024;
    uint8_t* bar_area = gbase + (6 + 2 * NS) * AT_TILE + 1024;
    auto q_full = [&](int b) { return bars + 8u * b; };
    auto q_empty = [&](int b) { return bars + 8u * (2 + b); };
    auto o_full = [&](int b) { return bars + 8u * (4 + b); };
    auto o_empty = [&](int b) { return bars + 8u * (6 + b); };
    auto kv_full = [&](int i) { return bars + 8u * (8 + i); };
    auto kv_empty = [&](int i) { return bars + 8u * (8 + NS + i); };
    const uint32_t bx = bars + 8u * (8 + 2 * NS);
    const uint32_t s_full = bx, s_free = bx + 8u;
    const uint32_t dp_full = bx + 16u, dp_free = bx + 24u;
    const uint32_t ds_full = bx + 32u, ds_free = bx + 40u;
    const uint32_t acc_full = bx + 48u, acc_empty = bx + 56u, drain = bx + 64u;
    const uint32_t stg_free = bx + 72u, stg_full = bx + 80u;
    const uint32_t x_full = bx + 88u, x_empty = bx + 96u;
    auto d_full = [&](int sl) { return bx + 104u + 8u * sl; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * (8 + 2 * NS) + 120);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (8 + 2 * NS) + 124);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; b++) {
            mbar_init(q_full(b), 1);
            mbar_init(q_empty(b), 1);
            mbar_init(o_full(b), 1);
            mbar_init(o_empty(b), 1);
        }
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
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, BW_EW);
        mbar_init(drain, 1);
        mbar_init(stg_free, 1);
        mbar_init(stg_full, BW_EW);
        mbar_init(x_full, 1);
        mbar_init(x_empty, 1);
        mbar_init(d_full(0), 1);
        mbar_init(d_full(1), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_addr((const void*)tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;  // columns Q_*

    if (warp == 0) {
        if (lane == 0) {
            // -------------------------------------------------- TMA producer
            int kv_issued[NS], qo_issued[2] = {-1, -1};  // parity of each buffer's last load (final drain)
            int x_issued = -1;
            for (int i = 0; i < NS; i++) kv_issued[i] = -1;
            int g = 0;
            // Q, dO and O of item i: Q and dO into buffer i & 1, once the item
            // before last has finished with it, O into the one O tile; all three
            // once D of the previous item is formed (which also means the store
            // warp is done with the dO tile of the item before last)
            auto load_qo = [&](int i, const Item& it) -> bool {
                const int b = it.bh / a.H, h = it.bh % a.H;
                const int qb = i & 1;
                const uint32_t qph = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(x_empty, (uint32_t)(i & 1) ^ 1u, abort_flag, a.status)) return false;
                mbar_expect_tx(x_full, AT_TILE);
                tma_load_3d(sX, &tm_o, x_full, h * AT_HD, it.tile * AT_M, b);
                x_issued = i & 1;
                if (!mbar_wait(q_empty(qb), qph ^ 1u, abort_flag, a.status)) return false;
                mbar_expect_tx(q_full(qb), AT_TILE);
                tma_load_3d(sQ(qb), &tm_qkv, q_full(qb), h * AT_HD, it.tile * AT_M, b);
                if (!mbar_wait(o_empty(qb), qph ^ 1u, abort_flag, a.status)) return false;
                mbar_expect_tx(o_full(qb), AT_TILE);
                tma_load_3d(sO(qb), &tm_do, o_full(qb), h * AT_HD, it.tile * AT_M, b);
                qo_issued[qb] = (int)qph;
                return true;
            };
            Item it0;
            bool ok = !get_item<true>(a, 0, it0) || load_qo(0, it0);
            for (int i = 0; ok; i++) {
                Item it;
                if (!get_item<true>(a, i, it)) break;
                const int b = it.bh / a.H, h = it.bh % a.H;
                auto load_kv = [&](int j) -> bool {
                    const int st = g % NS;
                    const uint32_t ph = (g / NS) & 1;
                    if (!mbar_wait(kv_empty(st), ph ^ 1u, abort_flag, a.status)) return false;
                    mbar_expect_tx(kv_full(st), 2 * AT_TILE);
                    tma_load_3d(sK(st), &tm_qkv, kv_full(st), a.C + h * AT_HD, j * AT_N, b);
                    tma_load_3d(sV(st), &tm_qkv, kv_full(st), 2 * a.C + h * AT_HD, j * AT_N, b);
                    kv_issued[st] = (int)ph;
                    g++;
                    return true;
                };
                // the item's first K/V block, then the next item's Q and dO (a
                // whole item ahead of their first use), then the other blocks
                if (!(ok = load_kv(0))) break;
                Item nit;
                if (get_item<true>(a, i + 1, nit) && !(ok = load_qo(i + 1, nit))) break;
                for (int j = 1; ok && j < it.nblk; j++) ok = load_kv(j);
            }
            for (int qb = 0; qb < 2; qb++)
                if (qo_issued[qb] >= 0) {
                    mbar_drain(q_full(qb), (uint32_t)qo_issued[qb], a.status);
                    mbar_drain(o_full(qb), (uint32_t)qo_issued[qb], a.status);
                }
            if (x_issued >= 0) mbar_drain(x_full, (uint32_t)x_issued, a.status);
            for (int st = 0; st < NS; st++)
                if (kv_issued[st] >= 0) mbar_drain(kv_full(st), (uint32_t)kv_issued[st], a.status);
        }
    } else if (warp == 1) {
        {
            // -------------------------------------------------- MMA issuer: the
            // whole warp runs the schedule (warp-uniform operands), one elected
            // lane issues the MMAs and commits
            const bool leader = elect_one();
            constexpr uint32_t idesc_s = make_idesc(AT_M, AT_N, false, false);
            constexpr uint32_t idesc_o = make_idesc(AT_M, AT_HD, false, true);
            auto issue_s = [&](const Cur& x) -> bool {  // S = Q K^T
                const int st = x.g % NS, qb = x.i & 1;
                if (x.n == 0 && !warp_wait(q_full(qb), (x.i >> 1) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(kv_full(st), (x.g / NS) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(s_free, (x.g & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
                // one 16-wide k step = 32 bytes = 2 units of the descriptors' address field
                const uint64_t da = sw128_desc(sQ(qb), 16, 1024), db = sw128_desc(sK(st), 16, 1024);
                if (leader) {
#pragma unroll
                    for (int k = 0; k < 4; k++) tc_mma(tmem + Q_S, da + 2 * k, db + 2 * k, idesc_s, k > 0 ? 1u : 0u);
                }
                if (leader) tc_commit(s_full);
                if (leader && x.n == x.it.nblk - 1) tc_commit(q_empty(qb));  // the item's last read of Q
                return true;
            };
            auto issue_dp = [&](const Cur& x) -> bool {  // dP = dO V^T
                const int st = x.g % NS, qb = x.i & 1;
                if (x.n == 0 && !warp_wait(o_full(qb), (x.i >> 1) & 1, abort_flag, a.status)) return false;
                if (!warp_wait(dp_free, (x.g & 1) ^ 1u, abort_flag, a.status)) return false;
                tc_fence_after();
                const uint64_t da = sw128_desc(sO(qb), 16, 1024), db = sw128_desc(sV(st), 16, 1024);
                if (leader) {
#pragma unroll
                    for (int k = 0; k < 4; k++) tc_mma(tmem + Q_DP, da + 2 * k, db + 2 * k, idesc_s, k > 0 ? 1u : 0u);
                }
                if (leader) tc_commit(dp_full);
                if (leader && x.n == x.it.nblk - 1) tc_commit(o_empty(qb));  // the item's last read of dO
                return true;
            };
            Cur c = cur_first<true>(a);
            bool ok = !c.valid || (issue_s(c) && issue_dp(c));
            while (ok && c.valid) {
                const Cur nx = cur_next<true>(a, c);
                const int st = c.g % NS;
                if (nx.valid && !(ok = issue_s(nx) && issue_dp(nx))) break;
                // dQ += dS K
                if (!(ok = warp_wait(ds_full, c.g & 1, abort_flag, a.status))) break;
                if (c.n == 0 && c.i > 0 && !(ok = warp_wait(acc_empty, (c.i - 1) & 1, abort_flag, a.status))) break;
                tc_fence_after();
                // MN-major B: one 16-row k step = 2048 bytes = 128 units of the address field
                const uint64_t dbk = sw128_desc(sK(st), 8192, 1024);
                const uint32_t acc0 = c.n > 0 ? 1u : 0u;
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < 8; kk++)
                        tc_mma_ts(tmem + Q_DQ, tmem + Q_DS + kk * 8, dbk + 128 * kk, idesc_o, kk > 0 ? 1u : acc0);
                }
                if (leader) tc_commit(ds_free);
                if (leader) tc_commit(kv_empty(st));
                if (leader && c.n == c.it.nblk - 1) tc_commit(acc_full);
                c = nx;
            }
            if (leader) tc_commit(drain);
            mbar_drain(drain, 0, a.status);
        }
    } else if (warp == BW_STORE_WARP) {
        // ------------------------------------------------------ D and the accumulator stores
        // D of item i (rows lane, lane + 32, ...: each lane sums the 64 products
        // of its row in a fixed order) from the item's dO tile (buffer i & 1) and
        // O tile, into D slot i & 1 and to global memory for the dK/dV kernel.
        auto form_d = [&](int i, const Item& it) -> bool {
            if (!warp_wait(x_full, i & 1, abort_flag, a.status)) return false;
            if (!warp_wait(o_full(i & 1), (i >> 1) & 1, abort_flag, a.status)) return false;
            const uint8_t* dot = gbase + (2 * (i & 1) + 1) * AT_TILE;
            float* dst = dslot + (i & 1) * 128;
#pragma unroll 1
            for (int k = 0; k < 4; k++) {
                const int row = lane + 32 * k;
                uint64_t acc2 = 0;
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int off = row * 128 + ((u ^ (row & 7)) << 4);  // 128-byte swizzle
                    const uint4 x = *reinterpret_cast<const uint4*>(dot + off);
                    const uint4 y = *reinterpret_cast<const uint4*>(xtile + off);
                    acc2 = f2_fma(bf16x2_to_f2(x.x), bf16x2_to_f2(y.x), acc2);
                    acc2 = f2_fma(bf16x2_to_f2(x.y), bf16x2_to_f2(y.y), acc2);
                    acc2 = f2_fma(bf16x2_to_f2(x.z), bf16x2_to_f2(y.z), acc2);
                    acc2 = f2_fma(bf16x2_to_f2(x.w), bf16x2_to_f2(y.w), acc2);
                }
                float d0, d1;
                f2_unpack(acc2, d0, d1);
                const float d = d0 + d1;
                dst[row] = d;
                const int q = it.tile * AT_M + row;
                if (q < a.T) a.Dw[(int64_t)it.bh * a.T + q] = d;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(x_empty);   // the O tile may be loaded again
                mbar_arrive(d_full(i & 1));
            }
            return true;
        };
        // D of the first two items, then per item f: its dQ tile out, once the
        // elementwise warps have staged it (after they read D(f + 1)), then
        // D(f + 2) into the slot D(f) used
        Item it, it2;
        bool ok = true;
        for (int i = 0; ok && i < 2 && get_item<true>(a, i, it2); i++) ok = form_d(i, it2);
        for (int f = 0; ok && get_item<true>(a, f, it); f++) {
            if (!warp_wait(stg_full, f & 1, abort_flag, a.status)) break;
            if (lane == 0) {
                const int b = it.bh / a.H, h = it.bh % a.H;
                tma_store_3d(&tm_dqkv, stg_addr, h * AT_HD, it.tile * AT_M, b);
                bulk_wait_read_all();  // the tile may be written again
                mbar_arrive(stg_free);
            }
            __syncwarp();
            if (get_item<true>(a, f + 2, it2)) ok = form_d(f + 2, it2);
        }
        if (lane == 0) bulk_wait_all();  // the stores are complete before the CTA ends
    } else {
        const int ew = warp - 2;
        const int quad = warp & 3, part = ew >> 2;
        const int r = quad * 32 + lane;  // query row within the tile = TMEM lane
        const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
        // this row's lse for an item; the next item's is loaded ahead and used as
        // it is (converted to log2 units when its item starts); D comes from the
        // store warp's slot
        auto load_row = [&](const Item& it, float& l) {
            const int q = it.tile * AT_M + r;
            l = a.lse[(int64_t)it.bh * a.T + (q < a.T ? q : 0)];
        };
        // An item's dQ leaves TMEM during the next item's first step, once its
        // exponentials are done, so the item's last dQ product runs meanwhile:
        // Parts 0, 1 hold dQ columns part*32..: they write their blocks into the
        // staging tile (once the store warp has sent the previous item's out),
        // every warp hands TMEM back, and the store warp sends the tile out.
        int pend_i = -1, nflush = 0;
        auto flush = [&]() -> bool {
            if (!warp_wait(acc_full, pend_i & 1, abort_flag, a.status)) return false;
            tc_fence_after();
            uint32_t dq[32];  // parts p and p + 2 read the same columns; p + 2 does not stage them
            tc_ld32_issue(trow + Q_DQ + (uint32_t)((part & 1) * 32), dq);
            tc_ld_wait(dq);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            if (!warp_wait(stg_free, (nflush & 1) ^ 1u, abort_flag, a.status)) return false;
            if (part < 2) {
                stage_block_sw128(stg, r, part, dq, a.scale);
                fence_proxy_async_smem();  // the writes, visible to the TMA
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(stg_full);
            nflush++;
            pend_i = -1;
            return true;
        };
        Cur c = cur_first<true>(a);
        float l_nx = 0.f, lse2 = 0.f, Dq = 0.f;
        if (c.valid) load_row(c.it, l_nx);
        bool ok = true;
        while (c.valid) {
            const Cur nx = cur_next<true>(a, c);
            const int g = c.g;
            const int q = c.it.tile * AT_M + r;
            if (c.n == 0) {
                lse2 = l_nx * 1.4426950408889634f;
                Item it2;
                if (get_item<true>(a, c.i + 1, it2)) load_row(it2, l_nx);
                if (!(ok = warp_wait(d_full(c.i & 1), (c.i >> 1) & 1, abort_flag, a.status))) break;
                Dq = dslot[(c.i & 1) * 128 + r];
            }
            const int k0 = c.n * AT_N + part * EW_COLS;  // first key of this thread's columns
            const bool diag = c.n == c.it.tile;
            uint32_t sv[32];
            if (!(ok = warp_wait(s_full, g & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + Q_S + (uint32_t)(part * EW_COLS), sv);
            tc_ld_wait(sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            // P = exp2(S scale - lse); masked only on the diagonal block (key >
            // query) and past the sequence end
            float p[EW_COLS];
            const uint64_t scale2 = f2_pack(a.scale_log2, a.scale_log2), nl2 = f2_pack(-lse2, -lse2);
            if (diag || k0 + EW_COLS > a.T) {
                const int hi = min(diag ? q - k0 + 1 : EW_COLS, a.T - k0);  // valid columns [0, hi)
#pragma unroll
                for (int cc = 0; cc < EW_COLS; cc += 2) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(sv[cc], sv[cc + 1]), scale2, nl2), x0, x1);
                    p[cc] = cc < hi ? ex2_approx(x0) : 0.f;
                    p[cc + 1] = cc + 1 < hi ? ex2_approx(x1) : 0.f;
                }
            } else {
#pragma unroll
                for (int cc = 0; cc < EW_COLS; cc += 2) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(sv[cc], sv[cc + 1]), scale2, nl2), x0, x1);
                    p[cc] = ex2_approx(x0);
                    p[cc + 1] = ex2_approx(x1);
                }
            }
            if (pend_i >= 0 && !(ok = flush())) break;
            if (!(ok = warp_wait(dp_full, g & 1, abort_flag, a.status))) break;
            tc_fence_after();
            tc_ld32_issue(trow + Q_DP + (uint32_t)(part * EW_COLS), sv);
            tc_ld_wait(sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_free);
            uint32_t pk[EW_COLS / 2];
            const uint64_t dq2 = f2_pack(Dq, Dq);
#pragma unroll
            for (int cc = 0; cc < EW_COLS; cc += 2) {
                float d0, d1;
                f2_unpack(f2_mul(f2_pack(p[cc], p[cc + 1]), f2_sub(f2_pack(sv[cc], sv[cc + 1]), dq2)), d0, d1);
                pk[cc / 2] = cvt_bf16x2(d0, d1);
            }
            if (!(ok = warp_wait(ds_free, (g & 1) ^ 1u, abort_flag, a.status))) break;
            tc_st16(trow + Q_DS + (uint32_t)(part * EW_COLS / 2), pk);
            tc_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
            if (c.n == c.it.nblk - 1) pend_i = c.i;
            c = cur_next<true>(a, c);
        }
        if (ok && pend_i >= 0) flush();
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

constexpr int DKDV_SMEM = (6 + 2 * DKDV_ST) * AT_TILE + BW_EW * 256 + 256 + 1024;
constexpr int DQ_SMEM = (6 + 2 * DQ_ST) * AT_TILE + 1024 + 256 + 1024;
static_assert(DKDV_SMEM <= 232448 && DQ_SMEM <= 232448, "shared memory per CTA");

}  // namespace

// bf16 backward (the attention.cu launcher routes here). D = rowsum(dO * O)
// is formed by the dQ kernel, which runs first, into D ([B, H, T] scratch),
// and read from there by the dK/dV kernel.
int launch_attention_backward_tc(bf16* dqkv, const bf16* dout, const bf16* qkv, const bf16* o, const float* lse,
                                 float* D, int B, int T, int C, int H, int* status, cudaStream_t s) {
    CUtensorMap mq, mo, mx, md;  // md: the same view of dqkv, for the TMA stores of dQ, dK, dV
    if (!make_qkv_map(&mq, qkv, B, T, C) || !make_do_map(&mo, dout, B, T, C) || !make_do_map(&mx, o, B, T, C) ||
        !make_qkv_map(&md, dqkv, B, T, C))
        return GPT2_ERR_CUDA;
    smem_attr((const void*)attn_bwd_dkdv_tc_kernel, DKDV_SMEM);
    smem_attr((const void*)attn_bwd_dq_tc_kernel, DQ_SMEM);
    BwdArgs a;
    a.dqkv = dqkv;
    a.lse = lse;
    a.D = D;
    a.Dw = D;
    a.status = status;
    a.B = B;
    a.T = T;
    a.C = C;
    a.H = H;
    a.nqt = (T + AT_M - 1) / AT_M;
    a.scale = 1.0f / sqrtf((float)(C / H));
    a.scale_log2 = 1.4426950408889634f * a.scale;
    const int items = a.nqt * B * H;
    const int grid = items < gpt2_num_sms() ? items : gpt2_num_sms();  // persistent: one CTA per SM
    a.sched = make_sched(B * H, a.nqt, grid);
    attn_bwd_dq_tc_kernel<<<grid, BW_THREADS, DQ_SMEM, s>>>(mq, mo, mx, md, a);
    attn_bwd_dkdv_tc_kernel<<<grid, BW_THREADS, DKDV_SMEM, s>>>(mq, mo, md, a);
    return 2;
}
