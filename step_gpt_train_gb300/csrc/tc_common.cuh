// tcgen05 / TMA / mbarrier building blocks shared by the tensor-core kernels
// (GEMM and attention) of sm_103a. Inline PTX only.
#pragma once

#include "common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace tc {

// The bound of every wait below, in clock cycles: GPT2_WAIT_LIMIT_CYCLES
// (about 2 s) unless a caller lowers it for the current device with
// set_wait_limit() (the failure-path test does, for one call). Each
// translation unit that includes this header has its own copy.
static __device__ long long wait_limit_cycles = GPT2_WAIT_LIMIT_CYCLES;

// Host side: sets this translation unit's bound on the current device
// (cycles <= 0: the default). Returns 0 or -1 on a CUDA error.
[[maybe_unused]] static int set_wait_limit(long long cycles) {
    const long long v = cycles > 0 ? cycles : GPT2_WAIT_LIMIT_CYCLES;
    return cudaMemcpyToSymbol(wait_limit_cycles, &v, sizeof(v)) == cudaSuccess ? 0 : -1;
}


__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity. Returns false (after
// flagging) on timeout or when another role has already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    const long long limit = *(volatile long long*)&wait_limit_cycles;
    for (uint32_t it = 1;; it++) {
        if (mbar_try(bar, parity)) return true;
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
// Non-blocking probe of the phase with the given parity (test_wait returns at
// once; try_wait may suspend the thread for a while before it re-checks).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, "
        "p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait by spinning on test_wait (as mbar_wait otherwise), for waits on
// events that come from another role at a steady rate, where a suspended
// thread would notice the phase change late. CL: cluster-scope acquire.
template <bool CL = false>
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    if (CL ? mbar_test_cl(bar, parity) : mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    const long long limit = *(volatile long long*)&wait_limit_cycles;
    for (uint32_t it = 1;; it++) {
        if (CL ? mbar_test_cl(bar, parity) : mbar_test(bar, parity)) return true;
        if ((it & 255) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
                set_status(status, GPT2_FLAG_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}
template <bool CL = false>
__device__ __forceinline__ bool warp_spin(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    const bool ok = mbar_spin<CL>(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// One lane of a fully active warp (the lowest), for work that a single
// thread issues on the warp's behalf.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n" : "=r"(pred));
    return pred != 0;
}
// Bounded wait by every lane of a warp, with one outcome for the whole warp:
// if any lane gave up, all give up, so no lane goes on alone into a warp-wide
// operation (a shuffle, __syncwarp or a .sync.aligned TMEM access).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    const bool ok = mbar_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}
// Bounded wait used while shutting down (ignores the abort flag).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, int* status) {
    const long long t0 = clock64();
    const long long limit = *(volatile long long*)&wait_limit_cycles;
    while (!mbar_try(bar, parity)) {
        if (clock64() - t0 > limit) {
            set_status(status, GPT2_FLAG_TIMEOUT);
            return;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0),
// completing bytes of transaction on the mbarrier.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// D(tmem) (+)= A(smem) * B(smem), kind::f16 (bf16 operands), fp32 accumulate.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(smem) * B(smem), kind::f8f6f4 (e4m3 or e5m2 operands), fp32
// accumulate; one instruction is K = 32 (32 bytes of each row).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem), kind::f16. A is M lanes (rows) by K
// 16-bit values, two per 32-bit column: element k of a row in column k/2,
// the even k in the low half. One instruction reads K = 16, 8 columns.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Packed pairs of fp32 (one 64-bit register pair, element 0 in the low half)
// and the paired fp32 arithmetic of sm_100 and later.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) { return f2_pack(__float_as_uint(lo), __float_as_uint(hi)); }
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// GELU (tanh form, through the logistic of 2y as gelu_both_f<bf16>) of a pair
// of values with paired fp32 arithmetic: g = gelu(u), d = gelu'(u), where
// s = 1 / (1 + 2^z), z = -2 log2(e) y, y = sqrt(2/pi) (u + 0.044715 u^3),
// g = u s and d = s + u s (1 - s) 2 sqrt(2/pi) (1 + 3 * 0.044715 u^2).
// The exponential and the reciprocal are the hardware approximations. Used by
// every bf16 GELU (the GEMM epilogues and the elementwise kernel), so fused
// and separate passes give the same bits.
__device__ __forceinline__ void gelu_pair(float u0, float u1, float& g0, float& g1, float& d0, float& d1) {
    constexpr float kz = (float)(-2.0 * 1.4426950408889634 * 0.7978845608028654);
    constexpr float kza = (float)(-2.0 * 1.4426950408889634 * 0.7978845608028654 * 0.044715);
    constexpr float kw = (float)(2.0 * 0.7978845608028654);
    constexpr float kwa = (float)(2.0 * 0.7978845608028654 * 3.0 * 0.044715);
    const uint64_t u = f2_pack(u0, u1);
    const uint64_t uu = f2_mul(u, u);
    const uint64_t z = f2_mul(u, f2_fma(uu, f2_pack(kza, kza), f2_pack(kz, kz)));
    float z0, z1;
    f2_unpack(z, z0, z1);
    const uint64_t one = f2_pack(1.f, 1.f);
    float e0, e1;
    f2_unpack(f2_add(f2_pack(ex2_approx(z0), ex2_approx(z1)), one), e0, e1);
    const uint64_t sv = f2_pack(__fdividef(1.f, e0), __fdividef(1.f, e1));
    const uint64_t g = f2_mul(u, sv);
    const uint64_t w = f2_fma(uu, f2_pack(kwa, kwa), f2_pack(kw, kw));
    const uint64_t d = f2_fma(f2_mul(g, w), f2_sub(one, sv), sv);
    f2_unpack(g, g0, g1);
    f2_unpack(d, d0, d1);
}

// Column sums of a warp's 32-row x 32-column bf16 block in shared memory held
// as four 16-byte units per row (unit q: columns 8q .. 8q+7) at
// unit_addr(r, q). Lane L loads unit L & 3 of rows L/4 + 8i (i < 4; rows >=
// nrows count as 0) and adds them in fp32 in that order; then the eight lanes
// that share a unit combine their sums in three halving exchanges (partners
// across lane bits 4, 3, 2: a lane keeps half of its columns and adds its
// partner's values of them). Afterwards lane L holds the sum of column
//   8 (L & 3) + 4 ((L >> 4) & 1) + 2 ((L >> 3) & 1) + ((L >> 2) & 1),
// which is returned in col. The order of the additions is fixed.
template <typename UnitAddr>
__device__ __forceinline__ float staged_colsum32(UnitAddr unit_addr, int nrows, int lane, int& col) {
    const int q = lane & 3, r0 = lane >> 2;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; j++) v[j] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int r = r0 + 8 * i;
        if (r < nrows) {
            const uint4 w = *reinterpret_cast<const uint4*>(unit_addr(r, q));
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                v[2 * k] += __uint_as_float(u[k] << 16);
                v[2 * k + 1] += __uint_as_float(u[k] & 0xFFFF0000u);
            }
        }
    }
#pragma unroll
    for (int w = 4, m = 16; w >= 1; w /= 2, m /= 2) {
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int i = 0; i < w; i++) {
            const float keep = up ? v[i + w] : v[i];
            const float send = up ? v[i] : v[i + w];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    col = 8 * q + 4 * ((lane >> 4) & 1) + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
    return v[0];
}

// Issue a load of 32 consecutive fp32 accumulator columns of this thread's
// TMEM lane; the registers are valid only after tc_ld_wait on them.
__device__ __forceinline__ void tc_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// Store 32 consecutive fp32 columns of this thread's TMEM lane; complete
// after tc_st_wait.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// Store 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tc_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Wait for this thread's outstanding TMEM loads. The registers are listed as
// read-write operands so that no use of them is scheduled before the wait.
__device__ __forceinline__ void tc_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// TMA store of a [1, 32, box_x] box from shared memory (3-D map: columns,
// rows, split), tracked by this thread's bulk-async group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Write 16 bytes (chunk q of 4) of this lane's 64-byte row into a buffer laid
// out with the 64-byte swizzle: 16-byte chunk q of row r sits at chunk
// position q ^ ((r >> 1) & 3), so the 32 lanes of a warp spread over all banks.
__device__ __forceinline__ void stage16(uint8_t* buf, int row, int q, uint4 v) {
    *reinterpret_cast<uint4*>(buf + row * 64 + ((q ^ ((row >> 1) & 3)) << 4)) = v;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// TMEM allocation by one full warp; the base address is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(ncols) : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format):
// start address >> 4 in bits 0-13, leading-dimension byte offset >> 4 in
// 16-29, stride-dimension byte offset >> 4 in 32-45, descriptor version 1 in
// 46-47, layout type 2 (128-byte swizzle) in 61-63.
// K-major operand (rows of 64 k-values = 128 B, 8-row groups of 1024 B):
//   SBO = 1024 (next 8 rows), LBO unused.
// MN-major operand (rows of 64 m- or n-values at one k, 8-k-row groups of
//   1024 B, 64-wide MN chunks one after another): LBO = chunk stride,
//   SBO = 1024 (next 8 k-rows).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// The same with the 64-byte swizzle (swizzle field 4): atoms of 8 rows of 64
// bytes, 512 bytes each.
__device__ __forceinline__ uint64_t sw64_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)4 << 61;
    return d;
}

// Instruction descriptor, kind::f8f6f4: fp32 accumulator (bits 4-5 = 1), the
// formats of A and B in bits 7-9 and 10-12 (0 = e4m3, 1 = e5m2), both K-major,
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc_f8(int M, int N, int a_fmt, int b_fmt) {
    return (1u << 4) | ((uint32_t)(a_fmt & 7) << 7) | ((uint32_t)(b_fmt & 7) << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B
// bf16 (bits 7-9 and 10-12 = 1), A/B major-ness (bits 15, 16: 1 = MN-major),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// cuTensorMapEncodeTiled from the driver, looked up once at run time (so the
// library does not link the driver library).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    }();
    return fn;
}

}  // namespace tc
