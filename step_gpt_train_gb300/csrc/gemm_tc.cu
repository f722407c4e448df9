// bf16 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// D[M,N] = sum_k A(m,k) B(n,k) (+ bias[n]), bf16 operands, fp32 accumulation
// in tensor memory (TMEM). These are the matmuls of the GPT-2 step: the
// linear forwards (A = activations, K-major; B = weight [N,K], K-major), the
// input gradients dX = dY W (B = W read MN-major) and the weight gradients
// dW = dY^T X (both operands MN-major, fp32 output, long K = B*T).
//
// Structure: a persistent kernel, one CTA per SM, 10 warps.
//   warp 0      TMA producer: 128x64 A and BNx64 B tiles (128-byte swizzle)
//               into a ring of shared-memory stages, completion on mbarriers.
//   warp 1      allocates TMEM (two BN-column fp32 accumulators) and runs
//               the MMA schedule warp-uniformly: one elected lane issues
//               tcgen05.mma (M=128, N=BN, K=16; kind::f8f6f4 with K=32 for
//               FP8 operands) from shared-memory descriptors, and
//               tcgen05.commit frees each stage and signals a finished
//               accumulator.
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..+31 = tile rows; two warps per lane quarter,
//               each owning half of the tile's columns), + bias (each warp
//               stages its own slice in shared memory once per tile, so only
//               warp-level syncs are needed), convert, then each 32-row chunk
//               goes through a 2 KB swizzled shared-memory buffer to a TMA
//               bulk-tensor store (coalesced, asynchronous; TMA clips rows and
//               columns outside the matrix). The next chunk's TMEM load is in
//               flight while the current one is stored.
// Two accumulators let the epilogue of one tile overlap the MMAs of the next.
// Work is a round robin of units over the CTAs. A unit is a whole 128 x BN
// tile or, for weight gradients with few tiles and a long K, one of S equal
// k-ranges of a tile (split-K). Units are numbered tile-major, so the CTAs
// that run at the same time read the same k-blocks of A and B in lockstep and
// share them through L2. A split unit stores an fp32 partial tile; a reduce
// kernel adds the S partials of each tile in split order (deterministic).
// Every mbarrier wait is bounded: on timeout the kernel sets a status bit,
// stops, waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

#include <cuda.h>

namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;               // 64 bf16 = 128 bytes = one swizzle row
constexpr int NUM_THREADS = 320;     // 10 warps
constexpr int EPI_WARP0 = 2;
constexpr int EPI_WARPS = 8;

// NB: output staging buffers per epilogue warp (two for the GELU epilogue's
// two outputs, paid for with one operand stage).
template <int BN, int NB = 1> struct TileCfg {
    static constexpr int STAGES = (BN == 256 ? 4 : (BN == 192 ? 5 : 6)) - (NB == 2 ? 1 : 0);
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // power of two >= two accumulators
    static constexpr int OUT_STAGE_BYTES = 2048;                        // per epilogue warp: 32 rows x 64 B
    static constexpr int OUT_BYTES = EPI_WARPS * NB * OUT_STAGE_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int BIAS_BYTES = EPI_WARPS * (BN / 2) * 4;         // per warp: its half of the tile (fp32)
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 /*align*/ + BAR_BYTES + BIAS_BYTES;
};

// Epilogue operations fused into the bf16-output GEMM.
constexpr int EPI_NONE = 0;
constexpr int EPI_GELU = 1;  // u = bf16(x); D = gelu'(u), D2 = gelu(u): the MLP's first linear and its GELU
constexpr int EPI_MUL = 2;   // D = bf16(x) * aux: the input gradient through that GELU, aux = gelu'(u)

struct GemmArgs {
    const void* bias;    // bf16 [N] or null
    const bf16* aux;     // EPI_MUL: the factor [M][N]
    float* colsum;       // EPI_MUL, or null: column sums of the stored D per 32-row slice, [4 * m_tiles][N]
    unsigned* amax;      // or null: the largest |output| as stored merged in (EPI_GELU: gelu(u); EPI_MUL: D)
    int* status;
    int M, N, K;
    int d_fp32;
    int splits;          // k-ranges per tile
    int partials;        // 1: store fp32 partial tiles for the reduce kernel (split-K or accumulation)
    int kbs;             // k-blocks per split
    int n_tiles;         // ceil(N / BN)
    int units;           // m_tiles * n_tiles * splits
    int num_kb;          // ceil(K / k-block width): 64 bf16 or 128 e4m3 values (128 bytes either way)
    int m_tiles;         // ceil(M / 128)
    int group_n;         // tile raster: column tiles per group (n_tiles: plain row-major order)
    const float* a_scale;  // FP8 operands: device scalars by which the codes of A and of B are
    const float* b_scale;  // multiplied back (the product scales the accumulator)
    int a_fmt, b_fmt;      // FP8 operands: their formats (0 e4m3, 1 e5m2)
};

// One unit of a CTA's work: k-blocks [kb0, kb1) of tile (mt, nt); z = partial slot.
struct Work {
    int tile, mt, nt, kb0, kb1, z;
};

// The idx-th unit of this CTA, or false when there is none. Tile t is the
// t-th of a grouped raster: groups of group_n column tiles, each walked row
// by row, so the CTAs at work at one time share a few B tiles through L2
// instead of streaming all of B for every row of tiles (with group_n =
// n_tiles this is the plain row-major order; units with partial tiles use it).
__device__ __forceinline__ bool get_work(const GemmArgs& g, int idx, Work& w) {
    const int u = blockIdx.x + idx * gridDim.x;
    if (u >= g.units) return false;
    const int sp = u % g.splits;
    w.tile = u / g.splits;
    const int per_group = g.m_tiles * g.group_n;
    const int gi = w.tile / per_group, r = w.tile - gi * per_group;
    const int gw = min(g.group_n, g.n_tiles - gi * g.group_n);
    w.mt = r / gw;
    w.nt = gi * g.group_n + r % gw;
    w.kb0 = sp * g.kbs;
    w.kb1 = min(g.num_kb, w.kb0 + g.kbs);
    w.z = u;
    return true;
}

// A warp's output staging: NB buffers of 2 KB (32 rows x 64 bytes) used in
// turn, each TMA store from the next one. A buffer is written once the store
// that last used it has read it: with one buffer that is the store before,
// with two the one before that (the store before may still be reading the
// other buffer), so consecutive stores overlap.
template <int NB>
struct Stager {
    uint8_t* base;
    uint32_t base_addr;
    int sel;
    __device__ __forceinline__ uint8_t* buf() const { return base + sel * 2048; }
    __device__ __forceinline__ uint32_t addr() const { return base_addr + (uint32_t)sel * 2048u; }
    __device__ __forceinline__ void wait_free(int lane) const {
        if (lane == 0) {
            if (NB == 2) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            else bulk_wait_read_all();
        }
        __syncwarp();
    }
    __device__ __forceinline__ void advance() {
        if (NB == 2) sel ^= 1;
    }
};

// Stage 32 bf16 values of this lane's row (64 bytes) in the stager's next
// buffer, then store the 32 x 32 box at (x, y, z); returns the buffer written.
// am2 (or null): a running maximum of the stored values' magnitudes, as a
// bf16 pair (NaN-ignoring, as fmaxf).
template <int NB>
__device__ __forceinline__ uint8_t* stage_store_bf16(const float (&f)[32], Stager<NB>& st, const CUtensorMap* map,
                                                     int x, int y, int z, int lane, __nv_bfloat162* am2 = nullptr) {
    st.wait_free(lane);
    uint8_t* stage = st.buf();
#pragma unroll
    for (int q = 0; q < 4; q++) {
        uint4 v;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) h[i] = __floats2bfloat162_rn(f[q * 8 + 2 * i], f[q * 8 + 2 * i + 1]);
        if (am2) {
#pragma unroll
            for (int i = 0; i < 4; i++) *am2 = __hmax2(*am2, __habs2(h[i]));
        }
        stage16(stage, lane, q, v);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tma_store_3d(map, st.addr(), x, y, z);
    st.advance();
    return stage;
}

// One 32-column chunk of this warp's 32 rows: + bias, the epilogue op,
// convert, stage, TMA store. fp32 output goes out as two 16-column halves.
// ncols_valid = columns of the chunk inside the matrix (> 0). aux holds this
// lane's 32 factors (EPI_MUL). EPI_MUL with csum_dst: csum_dst[j] (j <
// ncols_valid) also receives the sum of column j of the stored (bf16) values
// over the first nrows of the warp's 32 rows, read back from the staging buffer.
// am2 (EPI_GELU, EPI_MUL; or null): this lane's running maximum of |gelu(u)|
// (resp. |D|) as stored. Only rows inside the matrix may pass it (outside,
// a GELU row is gelu(bias)); columns outside hold 0 in both forms (B's rows
// and the bias read as 0 there, and the factor of EPI_MUL is 0).
template <int EPI, bool F8 = false, int NB = 1>
__device__ __forceinline__ void epi_chunk(const uint32_t (&r)[32], const float* bias_s, bool fp32_out,
                                          Stager<NB>& st, const CUtensorMap* mapD,
                                          const CUtensorMap* mapD2, const uint4 (&aux)[4], int x, int y, int z,
                                          int ncols_valid, int lane, float alpha = 1.f, float* csum_dst = nullptr,
                                          int nrows = 32, __nv_bfloat162* am2 = nullptr) {
    float f[32];
    if (!F8 && bias_s) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {  // + bias, in pairs
            const uint64_t v = f2_add(f2_pack(r[j], r[j + 1]), *reinterpret_cast<const uint64_t*>(bias_s + j));
            f2_unpack(v, f[j], f[j + 1]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; j++)
            f[j] = (F8 ? __uint_as_float(r[j]) * alpha : __uint_as_float(r[j])) + (bias_s ? bias_s[j] : 0.f);
    }
    if (EPI == EPI_MUL) {
        // the linear output rounded to bf16 (as a separate pass would read it),
        // times gelu'(u): the product of two bf16 values is exact in fp32 and
        // rounds once when staged
#pragma unroll
        for (int j = 0; j < 32; j++) f[j] = __bfloat162float(__float2bfloat16_rn(f[j]));
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&aux[q]);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                f[q * 8 + 2 * i] *= __low2float(h[i]);
                f[q * 8 + 2 * i + 1] *= __high2float(h[i]);
            }
        }
        const uint8_t* stage = stage_store_bf16(f, st, mapD, x, y, z, lane, am2);
        if (csum_dst) {
            // the staged rows (the TMA store only reads them too; they are
            // written again only after this warp's next sync)
            int col;
            const float sum = staged_colsum32(
                [&](int r, int q) { return stage + r * 64 + ((q ^ ((r >> 1) & 3)) << 4); }, nrows, lane, col);
            if (col < ncols_valid) csum_dst[col] = sum;
        }
    } else if (EPI == EPI_GELU) {
        // u = the linear output rounded to bf16, then its GELU and GELU'
        float gd[32];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            uint32_t ub;
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(ub) : "f"(f[j + 1]), "f"(f[j]));
            gelu_pair(__uint_as_float(ub << 16), __uint_as_float(ub & 0xFFFF0000u), f[j], f[j + 1], gd[j], gd[j + 1]);
        }
        stage_store_bf16(gd, st, mapD, x, y, z, lane);  // gelu'(u), kept for the backward
        stage_store_bf16(f, st, mapD2, x, y, z, lane, am2);  // gelu(u)
    } else if (!fp32_out) {
        stage_store_bf16(f, st, mapD, x, y, z, lane);
    } else {
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
            if (hh * 16 >= ncols_valid) break;  // uniform across the warp
            st.wait_free(lane);
            uint8_t* stage = st.buf();
#pragma unroll
            for (int q = 0; q < 4; q++)
                stage16(stage, lane, q,
                        make_uint4(__float_as_uint(f[hh * 16 + q * 4]), __float_as_uint(f[hh * 16 + q * 4 + 1]),
                                   __float_as_uint(f[hh * 16 + q * 4 + 2]), __float_as_uint(f[hh * 16 + q * 4 + 3])));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tma_store_3d(mapD, st.addr(), x + hh * 16, y, z);
            st.advance();
        }
    }
}

// ---------------------------------------------------------------- kernel

// Failure-path test switch (off unless gemm_tc_stall_for_test() sets it on
// the current device): the MMA warp first waits on a barrier that nothing
// arrives at, so its bounded wait runs out and the kernel takes its abort
// path (status bit, abort flag, bounded drain of the copies in flight, TMEM
// freed, return) on otherwise normal inputs.
static __device__ int stall_for_test = 0;

// F8: FP8 operands, e4m3 or e5m2 each (K-major only): a k-block is 128 values,
// four K = 32 MMAs of kind::f8f6f4, and the epilogue scales the accumulator by
// a_scale * b_scale before its bias and operation.
template <int BN, bool A_MN, bool B_MN, int EPI, bool F8 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                   const GemmArgs g) {
    static_assert(!F8 || (!A_MN && !B_MN), "FP8 operands: K-major");
    constexpr int KE = F8 ? 128 : BK;  // values of a k-block (128 bytes of each row either way)
    constexpr int NB = EPI != EPI_NONE ? 2 : 1;  // output staging buffers per epilogue warp
    using Cfg = TileCfg<BN, NB>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned operand ring (the 128-byte swizzle pattern repeats every 1024 B).
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t a_stage0 = base;
    const uint32_t b_stage0 = base + S * Cfg::A_BYTES;
    uint8_t* out_stage = gbase + S * Cfg::STAGE_BYTES;  // [EPI_WARPS][NB][2 KB], 1024-aligned
    uint8_t* bar_area = out_stage + Cfg::OUT_BYTES;
    const uint32_t bars = base + S * Cfg::STAGE_BYTES + Cfg::OUT_BYTES;
    // barrier layout: full[S], empty[S], tmem_full[2], tmem_empty[2], drain
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * S + 4);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * (2 * S + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (2 * S + 5) + 4);
    const uint32_t stall_bar = bars + 8u * (2 * S + 6);  // never arrived at (failure-path test)

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr((const void*)tmem_slot)),
                     "r"(Cfg::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;


    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[S];
            for (int s = 0; s < S; s++) issued_phase[s] = -1;
            bool ok = true;
            Work w;
            for (int idx = 0; ok && get_work(g, idx, w); idx++) {
                const int m0 = w.mt * BM, n0 = w.nt * BN;
                for (int kb = w.kb0; kb < w.kb1; kb++) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, g.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(full_bar(stage), Cfg::STAGE_BYTES);
                    const uint32_t sa = a_stage0 + stage * Cfg::A_BYTES;
                    const uint32_t sb = b_stage0 + stage * Cfg::B_BYTES;
                    if (!A_MN) {
                        tma_load_2d(sa, &tmA, full_bar(stage), kb * KE, m0);
                    } else {
                        tma_load_2d(sa, &tmA, full_bar(stage), m0, kb * BK);
                        tma_load_2d(sa + 64 * 128, &tmA, full_bar(stage), m0 + 64, kb * BK);
                    }
                    if (!B_MN) {
                        tma_load_2d(sb, &tmB, full_bar(stage), kb * KE, n0);
                    } else {
#pragma unroll
                        for (int c = 0; c < BN / 64; c++)
                            tma_load_2d(sb + c * 64 * 128, &tmB, full_bar(stage), n0 + 64 * c, kb * BK);
                    }
                    issued_phase[stage] = (int)phase;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // make sure no copy into this CTA's shared memory is still in flight
            for (int s = 0; s < S; s++)
                if (issued_phase[s] >= 0) mbar_drain(full_bar(s), (uint32_t)issued_phase[s], g.status);
        }
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer: the
            // whole warp runs the schedule (warp-uniform operands), one elected
            // lane issues the MMAs and commits
            const bool leader = elect_one();
            const uint32_t idesc = F8 ? make_idesc_f8(BM, BN, g.a_fmt, g.b_fmt) : make_idesc(BM, BN, A_MN, B_MN);
            constexpr uint32_t a_kstep = A_MN ? 16 * 128 : 32;  // bytes per 16-wide k step
            constexpr uint32_t b_kstep = B_MN ? 16 * 128 : 32;
            constexpr uint32_t a_lbo = A_MN ? 64 * 128 : 16;
            constexpr uint32_t b_lbo = B_MN ? 64 * 128 : 16;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            if (*(volatile int*)&stall_for_test) ok = warp_wait(stall_bar, 0, abort_flag, g.status);
            Work w;
            for (int idx = 0; ok && get_work(g, idx, w); idx++) {
                const int kb0 = w.kb0, kb1 = w.kb1;
                if (!warp_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, g.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; kb++) {
                    if (!warp_wait(full_bar(stage), phase, abort_flag, g.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = a_stage0 + stage * Cfg::A_BYTES;
                    const uint32_t sb = b_stage0 + stage * Cfg::B_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; k++) {
                        const uint64_t ad = sw128_desc(sa + k * a_kstep, a_lbo, 1024);
                        const uint64_t bd = sw128_desc(sb + k * b_kstep, b_lbo, 1024);
                        if (leader) {
                            if (F8) tc_mma_f8(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                            else tc_mma(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                    }
                    if (leader) tc_commit(empty_bar(stage));  // stage reusable once these MMAs finish
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (leader) tc_commit(tfull_bar(acc));  // accumulator complete
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // all MMAs issued by this thread must finish before TMEM is freed
            if (leader) tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, g.status);
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2..9)
        const int ew = warp - EPI_WARP0;         // 0..7
        const int quad = warp & 3;               // TMEM lanes 32*quad .. 32*quad+31
        const int half = ew >> 2;                // which half of the tile's columns
        constexpr int CHUNKS = BN / 64;          // 32-column chunks per warp
        const int row_in_tile = quad * 32 + lane;
        // this warp's bias slice [BN/2 columns] and output staging buffer
        float* bias_s = reinterpret_cast<float*>(bar_area + Cfg::BAR_BYTES) + ew * (BN / 2);
        uint8_t* stage = out_stage + ew * NB * Cfg::OUT_STAGE_BYTES;
        Stager<NB> stg{stage, smem_addr(stage), 0};
        const bool use_bias = g.bias != nullptr && !g.partials;
        const float alpha = F8 ? *g.a_scale * *g.b_scale : 1.f;
        // EPI_MUL column sums: each warp writes the sums of its 32 rows of a
        // tile, row 4 * mt + quad of g.colsum
        const bool want_csum = EPI == EPI_MUL && g.colsum != nullptr;
        // (the FP8 step's operands only: the bf16 kernels carry none of it)
        const bool want_amax = F8 && (EPI == EPI_GELU || EPI == EPI_MUL) && g.amax != nullptr;
        __nv_bfloat162 am2 = __floats2bfloat162_rn(0.f, 0.f);  // this lane's largest |output| (amax)
        int acc = 0;
        uint32_t acc_phase = 0;
        Work w;
        for (int idx = 0; get_work(g, idx, w); idx++) {
            const int m0 = w.mt * BM, n0 = w.nt * BN;
            const int cfirst = half * CHUNKS;
            if (use_bias) {
                // the bias of this warp's half of the tile; the buffer's only
                // reader is this same warp, done with the previous tile
                const bf16* bp = reinterpret_cast<const bf16*>(g.bias);
                const int nb = n0 + cfirst * 32;
                __syncwarp();
                for (int i = lane; i < BN / 2; i += 32) bias_s[i] = nb + i < g.N ? __bfloat162float(bp[nb + i]) : 0.f;
                __syncwarp();
            }
            // EPI_MUL: this lane's factors, a ring of two chunks; the
            // first two load while the tile's MMAs run, and each slot is
            // refilled with the chunk after next once its chunk is done
            uint4 aux[2][4];
            auto load_aux = [&](int c, uint4 (&dst)[4]) {
                const int row = m0 + row_in_tile;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int col = n0 + (cfirst + c) * 32 + q * 8;
                    dst[q] = (row < g.M && col < g.N) ? *reinterpret_cast<const uint4*>(g.aux + (int64_t)row * g.N + col)
                                                      : make_uint4(0, 0, 0, 0);
                }
            };
            if (EPI == EPI_MUL) {
                load_aux(0, aux[0]);
                if (CHUNKS > 1) load_aux(1, aux[1]);
            }
            if (!warp_wait(tfull_bar(acc), acc_phase, abort_flag, g.status)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
            const int y = m0 + quad * 32;
            int nchunks = 0;  // chunks of this warp with a valid row and column (uniform across the warp)
            if (y < g.M) {
#pragma unroll
                for (int c = 0; c < CHUNKS; c++)
                    if (n0 + (cfirst + c) * 32 < g.N) nchunks = c + 1;
            }
            const bool split = g.partials != 0;
            const bool fp32_out = split || g.d_fp32 != 0;
            // split partials are stored tile-local: [unit][128 rows][BN columns]
            const int z = split ? w.z : 0;
            const int ys = split ? quad * 32 : y;
            auto xcol = [&](int c) { return (split ? 0 : n0) + (cfirst + c) * 32; };
            auto ncols = [&](int c) { return g.N - (n0 + (cfirst + c) * 32); };
            auto bias_at = [&](int c) -> const float* { return use_bias ? bias_s + c * 32 : nullptr; };
            float* csum_row = want_csum ? g.colsum + (int64_t)(w.mt * 4 + quad) * g.N + n0 + cfirst * 32 : nullptr;
            auto csum_at = [&](int c) -> float* { return want_csum ? csum_row + c * 32 : nullptr; };
            const int nrows = max(0, min(32, g.M - y));  // this warp's rows inside the matrix
            uint32_t ra[32], rb[32];
            if (nchunks > 0) {
                tc_ld32_issue(tbase + (uint32_t)(cfirst * 32), ra);
                tc_ld_wait(ra);
            }
            for (int c = 0; c < nchunks; c += 2) {
                // ra holds chunk c; chunk c+1 is loaded into rb while ra is stored
                const bool more = c + 1 < nchunks;
                if (more) tc_ld32_issue(tbase + (uint32_t)((cfirst + c + 1) * 32), rb);
                epi_chunk<EPI, F8>(ra, bias_at(c), fp32_out, stg, &tmD, &tmD2, aux[0], xcol(c), ys, z,
                                   ncols(c), lane, alpha, csum_at(c), nrows,
                                   want_amax && m0 + row_in_tile < g.M ? &am2 : nullptr);
                if (EPI == EPI_MUL && c + 2 < CHUNKS) load_aux(c + 2, aux[0]);
                __syncwarp();  // reconverge before the warp-collective TMEM ops
                if (!more) break;
                tc_ld_wait(rb);
                const bool more2 = c + 2 < nchunks;
                if (more2) tc_ld32_issue(tbase + (uint32_t)((cfirst + c + 2) * 32), ra);
                epi_chunk<EPI, F8>(rb, bias_at(c + 1), fp32_out, stg, &tmD, &tmD2, aux[1], xcol(c + 1),
                                   ys, z, ncols(c + 1), lane, alpha, csum_at(c + 1), nrows,
                                   want_amax && m0 + row_in_tile < g.M ? &am2 : nullptr);
                if (EPI == EPI_MUL && c + 3 < CHUNKS) load_aux(c + 3, aux[1]);
                __syncwarp();
                if (more2) tc_ld_wait(ra);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (want_csum) {  // rows outside the matrix: zero sums for the columns inside it
                for (int c = nchunks; c < CHUNKS; c++)
                    if (n0 + (cfirst + c) * 32 + lane < g.N) csum_row[c * 32 + lane] = 0.f;
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (want_amax) amax_merge(g.amax, fmaxf(__low2float(am2), __high2float(am2)));
        if (lane == 0) bulk_wait_all();  // this warp's stores are complete
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(Cfg::TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- CTA-pair kernel
//
// The same GEMM with the MMAs of two CTAs (a cluster of two on neighbouring
// SMs) fused into one M = 256 product per instruction (tcgen05.mma
// .cta_group::2): each CTA holds 128 rows of A and half of the tile's PN (256
// or 192) columns of B in its shared memory, the pair's 256 x PN tile is
// computed by the even CTA's MMA warp, and each CTA's tensor memory receives
// its own 128 rows. Per SM and k-block the operand traffic at PN = 256 is
// 16 KB of A and 16 KB of B for the work that takes 16 KB of A and 32 KB of B
// in the one-CTA kernel.
// Cross-CTA hand-offs (no multicast): both CTAs' operand copies complete on
// the even CTA's full barriers (TMA .cta_group::2 with a cluster address);
// the even CTA's MMA warp commits each stage's release and each accumulator's
// completion twice, to its own barrier and to the odd CTA's (one commit per
// barrier, by its cluster address), so the odd CTA's producer and epilogue
// wait on barriers of their own; the odd CTA's epilogue warps arrive remotely
// on the even CTA's accumulator-empty barriers. (A relay warp that waited on
// the even CTA's barriers and arrived on the odd CTA's halved the rate: the
// odd CTA's refills started a relay hop late.) Both CTAs allocate and free
// tensor memory together (.cta_group::2), and leave only after a cluster
// barrier, once the even CTA's MMAs, which read the odd CTA's shared memory
// and write its tensor memory, are complete. Every mbarrier wait is bounded
// (cluster-scope acquire where the arrival comes from the other CTA) and uses
// try_wait, so a waiting producer or MMA warp takes no issue slots from the
// epilogue warps on its scheduler (spinning on test_wait measured 1% slower
// on the GELU epilogues).
// EPI_MUL's column sums: each warp's 32 rows, as in the one-CTA kernel (row
// 4 * (128-row tile) + quad of the partials).
constexpr int PBM = 256;                    // pair tile: 256 rows x PN (256, or 192 for N = 768 outputs)
constexpr int P_NBUF = 1;                   // output staging buffers per epilogue warp
constexpr int P_A_BYTES = 128 * BK * 2;     // this CTA's A rows
constexpr int P_NACC = 2;                   // accumulators in TMEM: a tile's epilogue overlaps the next tile's MMAs
constexpr int P_TMEM_COLS = 512;
constexpr int P_THREADS = 320;              // 10 warps: TMA, MMA, 8 epilogue
constexpr int P_OUT_BYTES = EPI_WARPS * P_NBUF * 2048;
constexpr int P_BAR_BYTES = 512;
template <int PN> struct PairCfg {
    static constexpr int B_BYTES = (PN / 2) * BK * 2;  // this CTA's half of B
    static constexpr int STAGE_BYTES = P_A_BYTES + B_BYTES;
    static constexpr int STAGES = PN == 256 ? 6 : 7;
    static constexpr int BIAS_BYTES = EPI_WARPS * (PN / 2) * 4;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + P_OUT_BYTES + 1024 + P_BAR_BYTES + BIAS_BYTES;
};
constexpr int P_SMEM_MAX = PairCfg<256>::SMEM_BYTES > PairCfg<192>::SMEM_BYTES ? PairCfg<256>::SMEM_BYTES
                                                                                : PairCfg<192>::SMEM_BYTES;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Arrive on the barrier at the same shared-memory offset in CTA `rank` of the
// cluster, with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
__device__ __forceinline__ bool mbar_try_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait, cluster-scope acquire (as mbar_wait otherwise).
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    if (mbar_try_cl(bar, parity)) return true;
    const long long t0 = clock64();
    const long long limit = *(volatile long long*)&wait_limit_cycles;
    for (uint32_t it = 1;; it++) {
        if (mbar_try_cl(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                set_status(status, GPT2_FLAG_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool warp_wait_cl(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    const bool ok = mbar_wait_cl(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// Commit of the pair's MMAs issued so far to the barrier at offset `bar` in
// both CTAs of the pair: this CTA's, then the odd CTA's (by its cluster
// address). Each commit arrives once its MMAs are complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 1;" : "=r"(remote) : "r"(bar));
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(remote)
                 : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on a
// barrier of the CTA pair's even CTA (cluster address), .cta_group::2.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}

// The idx-th unit of this CTA pair: pair tile (mt over 256-row tiles, nt) and k-range.
__device__ __forceinline__ bool get_work_pair(const GemmArgs& g, int idx, Work& w) {
    const int u = (blockIdx.x >> 1) + idx * (gridDim.x >> 1);
    if (u >= g.units) return false;
    const int sp = u % g.splits;
    w.tile = u / g.splits;
    const int per_group = g.m_tiles * g.group_n;
    const int gi = w.tile / per_group, r = w.tile - gi * per_group;
    const int gw = min(g.group_n, g.n_tiles - gi * g.group_n);
    w.mt = r / gw;
    w.nt = gi * g.group_n + r % gw;
    w.kb0 = sp * g.kbs;
    w.kb1 = min(g.num_kb, w.kb0 + g.kbs);
    w.z = u;
    return true;
}

template <bool A_MN, bool B_MN, int EPI, int PN>
__global__ void __launch_bounds__(P_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                     const GemmArgs g) {
    static_assert(PN == 256 || PN == 192, "pair tile width");
    // 192-wide tiles with MN-major B: a CTA's 96 columns of B as three 32-column
    // atoms of the 64-byte swizzle (the 128-byte swizzle's atoms are 64 columns)
    constexpr bool B_SW64 = B_MN && PN == 192;
    using PC = PairCfg<PN>;
    constexpr int PBN = PN;
    constexpr int S = PC::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t a_stage0 = base;
    const uint32_t b_stage0 = base + S * P_A_BYTES;
    uint8_t* out_stage = gbase + S * PC::STAGE_BYTES;
    uint8_t* bar_area = out_stage + P_OUT_BYTES;
    const uint32_t bars = base + S * PC::STAGE_BYTES + P_OUT_BYTES;
    // barriers: full[S], empty[S], pfull[S], tmem_full[NACC], tmem_empty[NACC], drain
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
    auto pfull_bar = [&](int s) { return bars + 8u * (2 * S + s); };
    auto tfull_bar = [&](int a) { return bars + 8u * (3 * S + a); };
    auto tempty_bar = [&](int a) { return bars + 8u * (3 * S + P_NACC + a); };
    const uint32_t drain_bar = bars + 8u * (3 * S + 2 * P_NACC);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bar_area + 8 * (3 * S + 2 * P_NACC + 1));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_area + 8 * (3 * S + 2 * P_NACC + 1) + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();  // 0: issues the pair's MMAs
    const uint32_t peer = rank ^ 1u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            mbar_init(pfull_bar(s), 1);
        }
        for (int a = 0; a < P_NACC; a++) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * EPI_WARPS);  // both CTAs' epilogue warps
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr((const void*)tmem_slot)),
                     "r"(P_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    // both CTAs' barriers are initialised before either arrives on the other's
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[S];
            for (int s = 0; s < S; s++) issued_phase[s] = -1;
            bool ok = true;
            Work w;
            for (int idx = 0; ok && get_work_pair(g, idx, w); idx++) {
                const int m0 = w.mt * PBM + (int)rank * 128, n0 = w.nt * PBN + (int)rank * (PBN / 2);
                for (int kb = w.kb0; kb < w.kb1; kb++) {
                    if (!mbar_wait_cl(empty_bar(stage), phase ^ 1u, abort_flag, g.status)) {
                        ok = false;
                        break;
                    }
                    // both CTAs' loads complete on the even CTA's full barrier,
                    // which expects the pair's bytes
                    if (rank == 0) mbar_expect_tx(full_bar(stage), 2 * PC::STAGE_BYTES);
                    uint32_t fb;
                    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(fb) : "r"(full_bar(stage)));
                    const uint32_t sa = a_stage0 + stage * P_A_BYTES;
                    const uint32_t sb = b_stage0 + stage * PC::B_BYTES;
                    if (!A_MN) {
                        tma_load_2d_pair(sa, &tmA, fb, kb * BK, m0);
                    } else {
                        tma_load_2d_pair(sa, &tmA, fb, m0, kb * BK);
                        tma_load_2d_pair(sa + 64 * 128, &tmA, fb, m0 + 64, kb * BK);
                    }
                    if (!B_MN) {
                        tma_load_2d_pair(sb, &tmB, fb, kb * BK, n0);
                    } else if (B_SW64) {
#pragma unroll
                        for (int i = 0; i < 3; i++) tma_load_2d_pair(sb + i * 4096, &tmB, fb, n0 + 32 * i, kb * BK);
                    } else {
                        tma_load_2d_pair(sb, &tmB, fb, n0, kb * BK);
                        tma_load_2d_pair(sb + 64 * 128, &tmB, fb, n0 + 64, kb * BK);
                    }
                    issued_phase[stage] = (int)phase;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the even CTA's full barriers count both CTAs' copies: it waits for them
            // all (the odd CTA stays until the cluster barrier at the end)
            if (rank == 0)
                for (int s = 0; s < S; s++)
                    if (issued_phase[s] >= 0) mbar_drain(full_bar(s), (uint32_t)issued_phase[s], g.status);
        }
    } else if (warp == 1) {
        if (rank == 0) {
            // ------------------------------------------------ MMA issuer (even CTA)
            const bool leader = elect_one();
            const uint32_t idesc = make_idesc(PBM, PBN, A_MN, B_MN);
            constexpr uint32_t a_kstep = A_MN ? 16 * 128 : 32;
            constexpr uint32_t b_kstep = B_MN ? 16 * 128 : 32;
            constexpr uint32_t a_lbo = A_MN ? 64 * 128 : 16;
            constexpr uint32_t b_lbo = B_MN ? 64 * 128 : 16;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            Work w;
            for (int idx = 0; ok && get_work_pair(g, idx, w); idx++) {
                const int kb0 = w.kb0, kb1 = w.kb1;
                if (!warp_wait_cl(tempty_bar(acc), acc_phase ^ 1u, abort_flag, g.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * PBN);
                for (int kb = kb0; kb < kb1; kb++) {
                    // both CTAs' operands (their copies complete on this CTA's barrier)
                    if (!warp_wait_cl(full_bar(stage), phase, abort_flag, g.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = a_stage0 + stage * P_A_BYTES;
                    const uint32_t sb = b_stage0 + stage * PC::B_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; k++) {
                        const uint64_t ad = sw128_desc(sa + k * a_kstep, a_lbo, 1024);
                        // (64-byte swizzle: a 16-row k step is 1024 bytes, atoms 4096 apart along N)
                        const uint64_t bd = B_SW64 ? sw64_desc(sb + k * 1024, 4096, 512)
                                                   : sw128_desc(sb + k * b_kstep, b_lbo, 1024);
                        if (leader)
                            asm volatile(
                                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                                " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                                ::"r"(d_tmem), "l"(ad), "l"(bd), "r"(idesc), "r"((kb > kb0 || k > 0) ? 1u : 0u)
                                : "memory");
                    }
                    if (leader) tc_commit_pair(empty_bar(stage));  // the stage may be refilled in both CTAs
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (leader) tc_commit_pair(tfull_bar(acc));  // both CTAs' accumulator rows are complete
                if (++acc == P_NACC) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (leader)
                asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 drain_bar)
                             : "memory");
            mbar_drain(drain_bar, 0, g.status);
        }
    } else {
        // ---------------------------------------------------- epilogue (warps 2..9, both CTAs)
        const int ew = warp - EPI_WARP0;
        const int quad = warp & 3;
        const int half = ew >> 2;
        constexpr int CHUNKS = PBN / 64;
        const int row_in_tile = (int)rank * 128 + quad * 32 + lane;  // row in the pair tile
        float* bias_s = reinterpret_cast<float*>(bar_area + P_BAR_BYTES) + ew * (PBN / 2);
        uint8_t* stage = out_stage + ew * P_NBUF * 2048;
        Stager<P_NBUF> stg{stage, smem_addr(stage), 0};
        const bool use_bias = g.bias != nullptr && !g.partials;
        const bool want_csum = EPI == EPI_MUL && g.colsum != nullptr;
        int acc = 0;
        uint32_t acc_phase = 0;
        Work w;
        for (int idx = 0; get_work_pair(g, idx, w); idx++) {
            const int m0 = w.mt * PBM, n0 = w.nt * PBN;
            const int cfirst = half * CHUNKS;
            if (use_bias) {
                const bf16* bp = reinterpret_cast<const bf16*>(g.bias);
                const int nb = n0 + cfirst * 32;
                __syncwarp();
                for (int i = lane; i < PBN / 2; i += 32) bias_s[i] = nb + i < g.N ? __bfloat162float(bp[nb + i]) : 0.f;
                __syncwarp();
            }
            uint4 aux[2][4];
            auto load_aux = [&](int c, uint4 (&dst)[4]) {
                const int row = m0 + row_in_tile;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int col = n0 + (cfirst + c) * 32 + q * 8;
                    dst[q] = (row < g.M && col < g.N) ? *reinterpret_cast<const uint4*>(g.aux + (int64_t)row * g.N + col)
                                                      : make_uint4(0, 0, 0, 0);
                }
            };
            if (EPI == EPI_MUL) {
                load_aux(0, aux[0]);
                load_aux(1, aux[1]);
            }
            if (!warp_wait_cl(tfull_bar(acc), acc_phase, abort_flag, g.status)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * PBN);
            const int y = m0 + (int)rank * 128 + quad * 32;
            int nchunks = 0;
            if (y < g.M) {
#pragma unroll
                for (int c = 0; c < CHUNKS; c++)
                    if (n0 + (cfirst + c) * 32 < g.N) nchunks = c + 1;
            }
            const bool split = g.partials != 0;
            const bool fp32_out = split || g.d_fp32 != 0;
            // split partials are stored pair-tile-local: [unit][256 rows][256 columns]
            const int z = split ? w.z : 0;
            const int ys = split ? (int)rank * 128 + quad * 32 : y;
            auto xcol = [&](int c) { return (split ? 0 : n0) + (cfirst + c) * 32; };
            auto ncols = [&](int c) { return g.N - (n0 + (cfirst + c) * 32); };
            auto bias_at = [&](int c) -> const float* { return use_bias ? bias_s + c * 32 : nullptr; };
            // EPI_MUL column sums of this warp's 32 rows: row 4 * (128-row tile) + quad
            float* csum_row =
                want_csum ? g.colsum + (int64_t)((2 * w.mt + (int)rank) * 4 + quad) * g.N + n0 + cfirst * 32 : nullptr;
            auto csum_at = [&](int c) -> float* { return want_csum ? csum_row + c * 32 : nullptr; };
            const int nrows = max(0, min(32, g.M - y));  // this warp's rows inside the matrix
            uint32_t ra[32], rb[32];
            if (nchunks > 0) {
                tc_ld32_issue(tbase + (uint32_t)(cfirst * 32), ra);
                tc_ld_wait(ra);
            }
            for (int c = 0; c < nchunks; c += 2) {
                const bool more = c + 1 < nchunks;
                if (more) tc_ld32_issue(tbase + (uint32_t)((cfirst + c + 1) * 32), rb);
                epi_chunk<EPI>(ra, bias_at(c), fp32_out, stg, &tmD, &tmD2, aux[0], xcol(c), ys, z,
                               ncols(c), lane, 1.f, csum_at(c), nrows);
                if (EPI == EPI_MUL && c + 2 < CHUNKS) load_aux(c + 2, aux[0]);
                __syncwarp();
                if (!more) break;
                tc_ld_wait(rb);
                const bool more2 = c + 2 < nchunks;
                if (more2) tc_ld32_issue(tbase + (uint32_t)((cfirst + c + 2) * 32), ra);
                epi_chunk<EPI>(rb, bias_at(c + 1), fp32_out, stg, &tmD, &tmD2, aux[1], xcol(c + 1), ys,
                               z, ncols(c + 1), lane, 1.f, csum_at(c + 1), nrows);
                if (EPI == EPI_MUL && c + 3 < CHUNKS) load_aux(c + 3, aux[1]);
                __syncwarp();
                if (more2) tc_ld_wait(ra);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(tempty_bar(acc));
                else mbar_arrive_cta(tempty_bar(acc), 0);
            }
            if (want_csum && m0 + (int)rank * 128 < g.M) {
                // rows outside the matrix in a 128-row tile that has rows inside it (the
                // partials hold 4 rows per such tile): zero sums for the columns inside it
                for (int c = nchunks; c < CHUNKS; c++)
                    if (n0 + (cfirst + c) * 32 + lane < g.N) csum_row[c * 32 + lane] = 0.f;
            }
            if (++acc == P_NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // the pair's MMAs (which read both CTAs' shared memory and write both
    // tensor memories) are complete before either CTA frees or leaves
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(P_TMEM_COLS)
                     : "memory");
    }
}

// Split-K reduce: D[m][n] (fp32) = bias[n] (if any) + the partial tiles of
// the tile of (m, n), added in split order; with accumulate, added to D's
// current value. 8 consecutive columns per thread (N and BN are multiples of 8).
__global__ void __launch_bounds__(256) split_reduce_kernel(float* __restrict__ D, const float* __restrict__ partial,
                                                           const bf16* __restrict__ bias, int M, int N, int BN,
                                                           int n_tiles, int splits, int accumulate) {
    // 32-bit element index (the launcher keeps M * N < 2^31)
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i >= M * N) return;
    const int m = i / N, n = i - m * N;
    const int64_t tile = (int64_t)(m / BM) * n_tiles + n / BN;
    const int64_t tile_elems = (int64_t)BM * BN;
    const float* p = partial + tile * splits * tile_elems + (int64_t)(m % BM) * BN + n % BN;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (bias) load8(bias + n, acc);
    if (accumulate) {
        float d[8];
        load8(D + i, d);
#pragma unroll
        for (int j = 0; j < 8; j++) acc[j] += d[j];
    }
    for (int sp = 0; sp < splits; sp++) {
        float v[8];
        load8(p + sp * tile_elems, v);
#pragma unroll
        for (int j = 0; j < 8; j++) acc[j] += v[j];
    }
    store8(D + i, acc);
}

// ---------------------------------------------------------------- host side

// 2-D bf16 tensor map over a row-major [outer, inner] matrix, box
// [box_outer, 64] (64 inner elements = 128 bytes), 128-byte swizzle,
// out-of-bounds elements read as zero.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {64, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over a row-major [outer, inner] bf16 matrix, box [64, 32] (64 bytes
// of the inner dimension), 64-byte swizzle: the MN-major B of 192-wide pair
// tiles, in 32-column atoms.
bool make_map_sw64(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {32, 64};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over a row-major [outer, inner] matrix of bytes (e4m3 codes), box
// [box_outer, 128] (128 bytes), 128-byte swizzle, out-of-bounds bytes read as zero.
bool make_map_u8(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {128, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D tensor map over an output [Z][M][N] (bf16 or fp32): box of 32 rows by
// 64 bytes of columns, 64-byte swizzle; stores outside [0,N) x [0,M) are clipped.
bool make_out_map(CUtensorMap* map, const void* ptr, bool fp32, uint64_t N, uint64_t M, uint64_t Z) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const uint64_t es = fp32 ? 4 : 2;
    cuuint64_t dims[3] = {N, M, Z};
    cuuint64_t strides[2] = {N * es, M * N * es};
    cuuint32_t box[3] = {(cuuint32_t)(64 / es), 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct Plan {
    int bn, n_tiles, m_tiles, tiles, num_kb, splits, kbs, units, grid, group_n;
};

// HBM bytes moved in the time one SM takes for one 128 x 256 x 64 k-block of
// MMAs (about 0.32 us at 13 TFLOP/s per SM and 6.8 TB/s): the exchange rate
// between partial-sum traffic and MMA time in the split-K cost model.
constexpr double KB_HBM_BYTES = 2.0e6;

Plan make_plan(int M, int N, int K, int d_fp32) {
    Plan p;
    const int sms = gpt2_num_sms();
    p.m_tiles = (M + BM - 1) / BM;
    p.num_kb = (K + BK - 1) / BK;
    // tile width: 256, or 192 where that cuts (tile waves x width) by more
    // than 10% (e.g. N = 768: 1024 tiles in 7 waves instead of 768 in 6);
    // 128 only for narrow matrices
    const long long t256 = (long long)p.m_tiles * ((N + 255) / 256);
    const long long t192 = (long long)p.m_tiles * ((N + 191) / 192);
    const long long c256 = (t256 + sms - 1) / sms * 256, c192 = (t192 + sms - 1) / sms * 192;
    p.bn = N <= 128 ? 128 : (c192 * 10 < c256 * 9 ? 192 : 256);
    p.splits = 1;
    if (d_fp32) {
        // Weight gradients: cost(S) = waves x k-blocks per unit (the busiest
        // SM's MMA time, in 128x256 k-block units) + the fp32 partials written
        // and read back. S = 1 keeps the chosen width; S > 1 uses 256.
        auto waves = [&](long long units) { return (double)((units + sms - 1) / sms); };
        const long long t1 = (long long)p.m_tiles * ((N + p.bn - 1) / p.bn);
        double best = waves(t1) * p.num_kb * (p.bn / 256.0);
        const int bn_split = N <= 128 ? 128 : 256;
        const long long ts = (long long)p.m_tiles * ((N + bn_split - 1) / bn_split);
        for (int sp = 2; sp <= 64 && sp * 4 <= p.num_kb; sp++) {
            const int kbs = (p.num_kb + sp - 1) / sp;
            const double cost = waves(ts * sp) * kbs * (bn_split / 256.0) + (double)sp * M * N * 8 / KB_HBM_BYTES;
            if (cost < best) {
                best = cost;
                p.splits = sp;
            }
        }
        if (p.splits > 1) p.bn = bn_split;
    }
    p.n_tiles = (N + p.bn - 1) / p.bn;
    p.tiles = p.m_tiles * p.n_tiles;
    p.kbs = (p.num_kb + p.splits - 1) / p.splits;
    p.splits = (p.num_kb + p.kbs - 1) / p.kbs;  // no empty split
    p.units = p.tiles * p.splits;
    p.grid = p.units < sms ? p.units : sms;
    // raster: wide outputs (the LM head: 197 column tiles) in groups of 32
    // column tiles (12.6 MB of B at K = 768), so B is read from DRAM about once
    // and A once per group instead of B once per row of tiles
    p.group_n = p.n_tiles > 32 ? 32 : p.n_tiles;
    return p;
}

template <int BN, bool A_MN, bool B_MN, int EPI, bool F8 = false>
void launch_tc(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md, const CUtensorMap& md2,
               const GemmArgs& args, int grid, cudaStream_t s) {
    using Cfg = TileCfg<BN, EPI != EPI_NONE ? 2 : 1>;
    constexpr int smem = Cfg::SMEM_BYTES;
    static_assert(smem <= 232448, "shared memory per CTA");
    smem_attr((const void*)gemm_tc_kernel<BN, A_MN, B_MN, EPI, F8>, smem);
    gemm_tc_kernel<BN, A_MN, B_MN, EPI, F8><<<grid, NUM_THREADS, smem, s>>>(ma, mb, md, md2, args);
}

// The operand layouts, and the fused epilogues only where the step uses them:
// GELU after a linear forward (A, B K-major), its gradient after an input
// gradient (B MN-major).
template <int BN>
bool launch_tc_layout(int epi, int a_mn, int b_mn, const CUtensorMap& ma, const CUtensorMap& mb,
                      const CUtensorMap& md, const CUtensorMap& md2, const GemmArgs& args, int grid, cudaStream_t s) {
    if (epi == EPI_GELU) {
        if (a_mn || b_mn) return false;
        launch_tc<BN, false, false, EPI_GELU>(ma, mb, md, md2, args, grid, s);
    } else if (epi == EPI_MUL) {
        if (a_mn || !b_mn) return false;
        launch_tc<BN, false, true, EPI_MUL>(ma, mb, md, md2, args, grid, s);
    } else if (!a_mn && !b_mn) {
        launch_tc<BN, false, false, EPI_NONE>(ma, mb, md, md2, args, grid, s);
    } else if (!a_mn && b_mn) {
        launch_tc<BN, false, true, EPI_NONE>(ma, mb, md, md2, args, grid, s);
    } else if (a_mn && !b_mn) {
        launch_tc<BN, true, false, EPI_NONE>(ma, mb, md, md2, args, grid, s);
    } else {
        launch_tc<BN, true, true, EPI_NONE>(ma, mb, md, md2, args, grid, s);
    }
    return true;
}

// FP8 operands (K-major): the plain, GELU-forward and GELU-backward epilogues.
template <int BN>
bool launch_tc_layout_f8(int epi, const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                         const CUtensorMap& md2, const GemmArgs& args, int grid, cudaStream_t s) {
    if (epi == EPI_GELU) launch_tc<BN, false, false, EPI_GELU, true>(ma, mb, md, md2, args, grid, s);
    else if (epi == EPI_MUL) launch_tc<BN, false, false, EPI_MUL, true>(ma, mb, md, md2, args, grid, s);
    else launch_tc<BN, false, false, EPI_NONE, true>(ma, mb, md, md2, args, grid, s);
    return true;
}

// CTA-pair kernel: the layouts and epilogues the step uses (as launch_tc_layout),
// launched in clusters of two.
template <bool A_MN, bool B_MN, int EPI, int PN = 256>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md, const CUtensorMap& md2,
                        const GemmArgs& args, int pairs, cudaStream_t s) {
    constexpr int smem = PairCfg<PN>::SMEM_BYTES;
    static_assert(smem <= 232448, "shared memory per CTA");
    smem_attr((const void*)gemm_pair_kernel<A_MN, B_MN, EPI, PN>, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(P_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<A_MN, B_MN, EPI, PN>, ma, mb, md, md2, args);
}

// Clusters of two CTA-pair kernel CTAs that can be resident at once on the
// current device (one CTA per SM; looked up once per process, else #SMs / 2).
int pair_clusters() {
    static const int n = [] {
        int v = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * 256, 1, 1);
        cfg.blockDim = dim3(P_THREADS, 1, 1);
        cfg.dynamicSmemBytes = P_SMEM_MAX;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaFuncSetAttribute(gemm_pair_kernel<false, false, EPI_NONE, 256>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_MAX);
        if (cudaOccupancyMaxActiveClusters(&v, gemm_pair_kernel<false, false, EPI_NONE, 256>, &cfg) != cudaSuccess ||
            v < 1)
            v = gpt2_num_sms() / 2;
        cudaGetLastError();
        return v;
    }();
    return n;
}

// The pair kernel takes plain bf16 products (no epilogue op) with one
// k-range per tile (no partials) and at least two 256-row tiles, in 256-wide
// tiles of a wide output (N >= 1024), or 192-wide tiles of a 384 to 960-wide
// output with K from 2048 to 16384 (four column tiles a row of tiles at
// N = 768; a CTA holds 96 rows or columns of B). At 32768 x 768: K = 3072,
// B K-major 92 us against 99.5 (one CTA), MN-major 98.6 against 100.0;
// K = 2304 76.1 against 78.5; but K = 768 36 against 34 and the LM head's
// K = 50304 1521 against 1460 (gemm_tc_use_pair(0) turns it all off); the
// rest runs on the one-CTA kernel. Measured at 32768 rows: K = 768, N = 2304 78 us
// against 84 (one CTA), N = 50304 1419 us against 1579; the GELU and
// GELU-gradient epilogues, which bound their products, ran 7% slower in the
// pair kernel (152 against 142 us, 172 against 160), so those stay on the
// one-CTA kernel (gemm_tc_use_pair(2...) routes them too, for measurements).
bool g_use_pair = true;
bool g_pair_epi = false;  // also the GELU and GELU-gradient epilogues
bool g_pair_mn192 = true;  // 192-wide tiles also with MN-major B
int g_pair_override = 0;  // > 0: the number of clusters to launch instead of the resident count
// The pair tile width for this product, or 0 for the one-CTA kernel.
int use_pair(int M, int N, int K, bool partials, int epi, int b_mn) {
    if (!g_use_pair || (epi != EPI_NONE && !g_pair_epi) || partials || M < 512) return 0;
    if (N >= 1024) return 256;
    return epi == EPI_NONE && (!b_mn || g_pair_mn192) && N >= 384 && N % 192 == 0 && K >= 2048 && K <= 16384
               ? 192
               : 0;
}

}  // namespace

int gemm_tc_set_wait_limit(long long cycles) { return set_wait_limit(cycles); }

int gemm_tc_use_pair(int on) {
    g_use_pair = on != 0;
    g_pair_epi = on > 1;
    g_pair_override = on > 2 ? on : 0;
    return on ? (g_pair_override ? g_pair_override : pair_clusters()) : 0;
}

int gemm_tc_stall_for_test(int on) {
    const int v = on ? 1 : 0;
    return cudaMemcpyToSymbol(stall_for_test, &v, sizeof(v)) == cudaSuccess ? 0 : -1;
}

size_t matmul_tc_scratch(int M, int N, int K, int d_fp32, int accumulate) {
    Plan p = make_plan(M, N, K, d_fp32);
    return p.splits > 1 || (d_fp32 && accumulate) ? (size_t)p.units * BM * p.bn * 4 : 0;
}

// FP8 operands: a k-block holds 128 values (the bytes and MMA time of a 64-value
// bf16 k-block), so the plan is the one of a bf16 product with K / 2.
size_t matmul_f8_scratch(int M, int N, int K, int d_fp32, int accumulate) {
    return matmul_tc_scratch(M, N, (K + 1) / 2, d_fp32, accumulate);
}


namespace {

// D (and D2) = the epilogue op of A B^T (+ bias); see launch_matmul_tc.
int matmul_tc(int epi, void* D, void* D2, const bf16* aux, int d_fp32, const void* A, int a_mn, const void* B,
              int b_mn, const void* bias, int M, int N, int K, void* scratch, int* status, cudaStream_t s,
              int accumulate = 0, float* colsum = nullptr, const F8Args* f8 = nullptr, unsigned* amax = nullptr) {
    if (f8 && (a_mn || b_mn || K % 16 || N % 8)) return GPT2_ERR_ARG;
    Plan p = make_plan(M, N, f8 ? (K + 1) / 2 : K, epi == EPI_NONE ? d_fp32 : 0);
    // partial tiles for the reduce kernel: split-K, or an fp32 result added to D
    const bool partials = p.splits > 1 || (accumulate && d_fp32 && epi == EPI_NONE);
    if (partials && (int64_t)M * N + 2048 >= ((int64_t)1 << 31)) return GPT2_ERR_ARG;  // the reduce uses 32-bit indices
    const int pn = f8 || amax ? 0 : use_pair(M, N, K, partials, epi, b_mn);
    if (pn) {
        // 256 x pn pair tiles, each CTA loading 128 rows of A and pn / 2 columns of B
        const int m_tiles = (M + PBM - 1) / PBM, n_tiles = (N + pn - 1) / pn;
        CUtensorMap ma, mb, md, md2;
        bool ok = a_mn ? make_map(&ma, A, (uint64_t)M, (uint64_t)K, 64) : make_map(&ma, A, (uint64_t)K, (uint64_t)M, 128);
        ok = ok && (b_mn ? (pn == 192 ? make_map_sw64(&mb, B, (uint64_t)N, (uint64_t)K)
                                      : make_map(&mb, B, (uint64_t)N, (uint64_t)K, 64))
                         : make_map(&mb, B, (uint64_t)K, (uint64_t)N, (uint32_t)(pn / 2)));
        ok = ok && make_out_map(&md, D, d_fp32 != 0, (uint64_t)N, (uint64_t)M, 1);
        if (epi == EPI_GELU) ok = ok && make_out_map(&md2, D2, false, (uint64_t)N, (uint64_t)M, 1);
        else md2 = md;
        if (!ok) return GPT2_ERR_CUDA;
        GemmArgs g = {};
        g.a_scale = g.b_scale = nullptr;
        g.a_fmt = g.b_fmt = 0;
        g.bias = bias;
        g.aux = aux;
        g.colsum = colsum;
        g.amax = nullptr;
        g.status = status;
        g.M = M;
        g.N = N;
        g.K = K;
        g.d_fp32 = d_fp32;
        g.splits = 1;
        g.partials = 0;
        g.num_kb = (K + BK - 1) / BK;
        g.kbs = g.num_kb;
        g.n_tiles = n_tiles;
        g.m_tiles = m_tiles;
        g.units = m_tiles * n_tiles;
        g.group_n = n_tiles > 32 ? 32 : n_tiles;
        const int resident = g_pair_override ? g_pair_override : pair_clusters();
        const int pairs = g.units < resident ? g.units : resident;
        cudaError_t e;
        if (pn == 192) {
            if (epi != EPI_NONE) return GPT2_ERR_ARG;
            if (!b_mn)
                e = a_mn ? launch_pair<true, false, EPI_NONE, 192>(ma, mb, md, md2, g, pairs, s)
                         : launch_pair<false, false, EPI_NONE, 192>(ma, mb, md, md2, g, pairs, s);
            else
                e = a_mn ? launch_pair<true, true, EPI_NONE, 192>(ma, mb, md, md2, g, pairs, s)
                         : launch_pair<false, true, EPI_NONE, 192>(ma, mb, md, md2, g, pairs, s);
        } else if (epi == EPI_GELU) {
            if (a_mn || b_mn) return GPT2_ERR_ARG;
            e = launch_pair<false, false, EPI_GELU>(ma, mb, md, md2, g, pairs, s);
        } else if (epi == EPI_MUL) {
            if (a_mn || !b_mn) return GPT2_ERR_ARG;
            e = launch_pair<false, true, EPI_MUL>(ma, mb, md, md2, g, pairs, s);
        } else if (!a_mn && !b_mn) {
            e = launch_pair<false, false, EPI_NONE>(ma, mb, md, md2, g, pairs, s);
        } else if (!a_mn && b_mn) {
            e = launch_pair<false, true, EPI_NONE>(ma, mb, md, md2, g, pairs, s);
        } else if (a_mn && !b_mn) {
            e = launch_pair<true, false, EPI_NONE>(ma, mb, md, md2, g, pairs, s);
        } else {
            e = launch_pair<true, true, EPI_NONE>(ma, mb, md, md2, g, pairs, s);
        }
        return e == cudaSuccess ? 1 : GPT2_ERR_CUDA;
    }
    CUtensorMap ma, mb;
    bool ok;
    if (f8) {
        ok = make_map_u8(&ma, A, (uint64_t)K, (uint64_t)M, BM) && make_map_u8(&mb, B, (uint64_t)K, (uint64_t)N, p.bn);
    } else {
        ok = a_mn ? make_map(&ma, A, (uint64_t)M, (uint64_t)K, 64) : make_map(&ma, A, (uint64_t)K, (uint64_t)M, BM);
        ok = ok && (b_mn ? make_map(&mb, B, (uint64_t)N, (uint64_t)K, 64)
                         : make_map(&mb, B, (uint64_t)K, (uint64_t)N, (uint32_t)p.bn));
    }
    CUtensorMap md, md2;
    if (partials) ok = ok && make_out_map(&md, scratch, true, (uint64_t)p.bn, BM, (uint64_t)p.units);
    else ok = ok && make_out_map(&md, D, d_fp32 != 0, (uint64_t)N, (uint64_t)M, 1);
    if (epi == EPI_GELU) ok = ok && make_out_map(&md2, D2, false, (uint64_t)N, (uint64_t)M, 1);
    else md2 = md;
    if (!ok) return GPT2_ERR_CUDA;
    GemmArgs g = {};
    g.a_scale = g.b_scale = nullptr;
    g.a_fmt = g.b_fmt = 0;
    g.bias = partials ? nullptr : bias;
    g.aux = aux;
    g.colsum = epi == EPI_MUL ? colsum : nullptr;
    g.amax = epi == EPI_GELU || epi == EPI_MUL ? amax : nullptr;
    g.status = status;
    g.M = M;
    g.N = N;
    g.K = K;
    g.d_fp32 = d_fp32;
    g.splits = p.splits;
    g.partials = partials ? 1 : 0;
    g.kbs = p.kbs;
    g.n_tiles = p.n_tiles;
    g.units = p.units;
    g.num_kb = p.num_kb;
    g.m_tiles = p.m_tiles;
    g.group_n = partials ? p.n_tiles : p.group_n;  // the reduce kernel finds partials in row-major order
    if (f8) {
        g.a_scale = f8->a_scale;
        g.b_scale = f8->b_scale;
        g.a_fmt = f8->a_fmt;
        g.b_fmt = f8->b_fmt;
    }
    bool launched;
    if (f8) {
        if (p.bn == 128) launched = launch_tc_layout_f8<128>(epi, ma, mb, md, md2, g, p.grid, s);
        else if (p.bn == 192) launched = launch_tc_layout_f8<192>(epi, ma, mb, md, md2, g, p.grid, s);
        else launched = launch_tc_layout_f8<256>(epi, ma, mb, md, md2, g, p.grid, s);
    } else if (p.bn == 128) launched = launch_tc_layout<128>(epi, a_mn, b_mn, ma, mb, md, md2, g, p.grid, s);
    else if (p.bn == 192) launched = launch_tc_layout<192>(epi, a_mn, b_mn, ma, mb, md, md2, g, p.grid, s);
    else launched = launch_tc_layout<256>(epi, a_mn, b_mn, ma, mb, md, md2, g, p.grid, s);
    if (!launched) return GPT2_ERR_ARG;
    if (partials) {
        const int64_t MN = (int64_t)M * N;
        const int blocks = (int)((MN / 8 + 255) / 256);
        split_reduce_kernel<<<blocks, 256, 0, s>>>((float*)D, (const float*)scratch, (const bf16*)bias, M, N, p.bn,
                                                   p.n_tiles, p.splits, accumulate && d_fp32 ? 1 : 0);
        return 2;
    }
    return 1;
}

}  // namespace

int launch_matmul_fp8(bf16* D, const uint8_t* A, int a_fmt, const float* a_scale, const uint8_t* B, int b_fmt,
                      const float* b_scale, const bf16* bias, int M, int N, int K, int* status, cudaStream_t s) {
    if (!D || !A || !B || !a_scale || !b_scale || M < 1 || N < 1 || K < 1) return GPT2_ERR_ARG;
    if ((a_fmt != FP8_E4M3 && a_fmt != FP8_E5M2) || (b_fmt != FP8_E4M3 && b_fmt != FP8_E5M2)) return GPT2_ERR_ARG;
    const F8Args f8 = {a_fmt, b_fmt, a_scale, b_scale};
    return matmul_tc(EPI_NONE, D, nullptr, nullptr, 0, A, 0, B, 0, bias, M, N, K, nullptr, status, s, 0, nullptr, &f8);
}

int launch_matmul_f8(void* D, int d_fp32, const uint8_t* A, const uint8_t* B, const F8Args& f8, const void* bias,
                     int M, int N, int K, void* scratch, int* status, cudaStream_t s, int accumulate) {
    if (M == 0 || N == 0) return 0;
    return matmul_tc(EPI_NONE, D, nullptr, nullptr, d_fp32, A, 0, B, 0, bias, M, N, K, scratch, status, s, accumulate,
                     nullptr, &f8);
}

int launch_matmul_gelu_f8(void* dgelu, void* out, const uint8_t* A, const uint8_t* W, const F8Args& f8,
                          const void* bias, int M, int N, int K, int* status, cudaStream_t s, unsigned* amax) {
    if (M == 0 || N == 0) return 0;
    return matmul_tc(EPI_GELU, dgelu, out, nullptr, 0, A, 0, W, 0, bias, M, N, K, nullptr, status, s, 0, nullptr,
                     &f8, amax);
}

int launch_matmul_gelu_backward_f8(void* du, const uint8_t* dY, const uint8_t* WT, const F8Args& f8,
                                   const void* dgelu, int M, int N, int K, int* status, cudaStream_t s,
                                   float* du_colsum, unsigned* amax) {
    if (M == 0 || N == 0) return 0;
    return matmul_tc(EPI_MUL, du, nullptr, (const bf16*)dgelu, 0, dY, 0, WT, 0, nullptr, M, N, K, nullptr, status, s,
                     0, du_colsum, &f8, amax);
}

int launch_matmul_tc(void* D, int d_fp32, const void* A, int a_mn, const void* B, int b_mn, const void* bias, int M,
                     int N, int K, void* scratch, int* status, cudaStream_t s, int accumulate) {
    return matmul_tc(EPI_NONE, D, nullptr, nullptr, d_fp32, A, a_mn, B, b_mn, bias, M, N, K, scratch, status, s,
                     accumulate);
}

int launch_matmul_gelu(void* dgelu, void* out, const void* A, const void* W, const void* bias, int M, int N, int K,
                       int* status, cudaStream_t s, unsigned* amax) {
    if (M == 0 || N == 0) return 0;
    return matmul_tc(EPI_GELU, dgelu, out, nullptr, 0, A, 0, W, 0, bias, M, N, K, nullptr, status, s, 0, nullptr,
                     nullptr, amax);
}

int launch_matmul_gelu_backward(void* du, const void* dY, const void* W, const void* dgelu, int M, int N, int K,
                                int* status, cudaStream_t s, float* du_colsum, unsigned* amax) {
    if (M == 0 || N == 0) return 0;
    return matmul_tc(EPI_MUL, du, nullptr, (const bf16*)dgelu, 0, dY, 0, W, 1, nullptr, M, N, K, nullptr, status,
                     s, 0, du_colsum, nullptr, amax);
}
