// Elementwise and reduction kernels of the GPT-2 step: encoder forward and
// backward, GELU, residual, bias gradient, AdamW. All loads and stores are
// 16-byte vectors (8 bf16 or 2 x 4 fp32), so every warp access is a
// coalesced 512-byte span.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

#include <algorithm>
#include <cmath>

// ===================================================================== encoder

// x0[r,:] = wte[tok[r],:] + wpe[r % T,:]. Thread per 8-element vector.
template <typename T>
__global__ void __launch_bounds__(256) encoder_fwd_kernel(T* __restrict__ x0, const int32_t* __restrict__ tokens,
                                                          const T* __restrict__ wte, const T* __restrict__ wpe,
                                                          int BT, int Tlen, int C, int V, int* status) {
    const int cv = C / 8;
    const int64_t total = (int64_t)BT * cv;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int r = (int)(i / cv);
    const int c = (int)(i % cv) * 8;
    int tok = tokens[r];
    if (tok < 0 || tok >= V) {
        set_status(status, GPT2_FLAG_TOKEN_RANGE);
        tok = 0;
    }
    float a[8], b[8];
    load8(wte + (int64_t)tok * C + c, a);
    load8(wpe + (int64_t)(r % Tlen) * C + c, b);
#pragma unroll
    for (int j = 0; j < 8; j++) a[j] += b[j];
    store8(x0 + (int64_t)r * C + c, a);
}

int launch_encoder_forward(int dtype, void* x0, const int32_t* tokens, const void* wte, const void* wpe, int B,
                           int T, int C, int V, int* status, cudaStream_t s) {
    const int64_t total = (int64_t)B * T * (C / 8);
    const int blocks = (int)((total + 255) / 256);
    if (dtype == GPT2_MODE_BF16)
        encoder_fwd_kernel<bf16><<<blocks, 256, 0, s>>>((bf16*)x0, tokens, (const bf16*)wte, (const bf16*)wpe, B * T,
                                                        T, C, V, status);
    else
        encoder_fwd_kernel<float><<<blocks, 256, 0, s>>>((float*)x0, tokens, (const float*)wte, (const float*)wpe,
                                                         B * T, T, C, V, status);
    return 1;
}

// ---- encoder backward ----
// dwpe[t,:] = sum over b (in order) of dx0[b*T+t,:]: thread per (t, vector).
template <typename T>
__global__ void __launch_bounds__(256) encoder_bwd_wpe_kernel(float* __restrict__ dwpe, const T* __restrict__ dx0,
                                                              int B, int Tlen, int C, int accumulate) {
    const int cv = C / 8;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)Tlen * cv) return;
    const int t = (int)(i / cv);
    const int c = (int)(i % cv) * 8;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int b = 0; b < B; b++) {
        float v[8];
        load8(dx0 + ((int64_t)b * Tlen + t) * C + c, v);
#pragma unroll
        for (int j = 0; j < 8; j++) acc[j] += v[j];
    }
    if (accumulate) {
        float d[8];
        load8(dwpe + (int64_t)t * C + c, d);
#pragma unroll
        for (int j = 0; j < 8; j++) acc[j] = d[j] + acc[j];
    }
    store8(dwpe + (int64_t)t * C + c, acc);
}

// dwte: the positions are sorted by token id with a stable two-pass LSD radix
// sort (8-bit digits, ids < 65536); then each token's rows are summed in
// ascending position order, split into 32-entry chunks of the sorted list so
// that a very frequent id is summed by many warps, and the chunk pieces of a
// long run are combined in a fixed order (enc_combine_kernel). Every token
// row of dwte has exactly one writer, so the result is deterministic.

#define ENC_TILE 1024  // sorted elements per block in the radix passes
#define ENC_CHUNK 32   // sorted entries per warp in the summation

// Pass setup: keys = token ids, values = positions.
__global__ void enc_init_kernel(uint32_t* keys, int32_t* vals, const int32_t* tokens, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        keys[i] = (uint32_t)tokens[i];
        vals[i] = i;
    }
}

// hist[d * nblk + blk] = count of digit d in tile blk.
__global__ void __launch_bounds__(ENC_TILE) enc_hist_kernel(int32_t* hist, const uint32_t* keys, int n, int shift) {
    __shared__ int h[256];
    if (threadIdx.x < 256) h[threadIdx.x] = 0;
    __syncthreads();
    int i = blockIdx.x * ENC_TILE + threadIdx.x;
    if (i < n) atomicAdd(&h[(keys[i] >> shift) & 255], 1);
    __syncthreads();
    if (threadIdx.x < 256) hist[threadIdx.x * gridDim.x + blockIdx.x] = h[threadIdx.x];
}

// Exclusive scan of hist in (digit, block) order, single block.
__global__ void __launch_bounds__(1024) enc_scan_kernel(int32_t* hist, int total) {
    __shared__ int partial[1024];
    const int per = (total + 1023) / 1024;
    const int lo = threadIdx.x * per;
    const int hi = min(total, lo + per);
    int s = 0;
    for (int i = lo; i < hi; i++) s += hist[i];
    partial[threadIdx.x] = s;
    __syncthreads();
    // Hillis-Steele inclusive scan over 1024 partial sums.
    for (int off = 1; off < 1024; off <<= 1) {
        int v = threadIdx.x >= off ? partial[threadIdx.x - off] : 0;
        __syncthreads();
        partial[threadIdx.x] += v;
        __syncthreads();
    }
    int run = threadIdx.x == 0 ? 0 : partial[threadIdx.x - 1];
    for (int i = lo; i < hi; i++) {
        int c = hist[i];
        hist[i] = run;
        run += c;
    }
}

// Stable scatter of one tile: rank within a warp from __match_any_sync,
// across warps from a per-warp digit-count table.
__global__ void __launch_bounds__(ENC_TILE) enc_scatter_kernel(uint32_t* keys_out, int32_t* vals_out,
                                                               const uint32_t* keys, const int32_t* vals,
                                                               const int32_t* offsets, int n, int shift) {
    __shared__ int cnt[ENC_TILE / 32][256];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    for (int i = threadIdx.x; i < (ENC_TILE / 32) * 256; i += blockDim.x) (&cnt[0][0])[i] = 0;
    __syncthreads();
    const int i = blockIdx.x * ENC_TILE + threadIdx.x;
    const bool valid = i < n;
    const uint32_t key = valid ? keys[i] : 0xffffffffu;
    const int d = valid ? (int)((key >> shift) & 255) : 256;
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const int rank = __popc(peers & ((1u << lane) - 1));
    if (valid && rank == 0) cnt[warp][d] = __popc(peers);
    __syncthreads();
    if (threadIdx.x < 256) {  // exclusive prefix over warps for digit threadIdx.x
        int run = 0;
        for (int w = 0; w < ENC_TILE / 32; w++) {
            int c = cnt[w][threadIdx.x];
            cnt[w][threadIdx.x] = run;
            run += c;
        }
    }
    __syncthreads();
    if (valid) {
        const int dst = offsets[d * gridDim.x + blockIdx.x] + cnt[warp][d] + rank;
        keys_out[dst] = key;
        vals_out[dst] = vals[i];
    }
}

__device__ __forceinline__ bool enc_is_head(const uint32_t* skey, int j) {
    return j == 0 || skey[j] != skey[j - 1];
}

// Sum of rows [lo, hi) of the sorted list into acc (lane's vectors).
template <typename T, int VPL>
__device__ __forceinline__ void enc_sum_rows(float (&acc)[VPL][8], const T* dx0, const int32_t* spos, int lo, int hi,
                                             int C, int lane) {
    const int cv = C / 8;
    // U rows in flight at a time, added in row order (the sums are those of
    // one row at a time)
    constexpr int U = VPL <= 3 ? 4 : 2;
    int j = lo;
    for (; j + U <= hi; j += U) {
        float v[U][VPL][8];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const T* row = dx0 + (int64_t)spos[j + u] * C;
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int idx = lane + 32 * i;
                if (idx < cv) load8(row + idx * 8, v[u][i]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; u++)
#pragma unroll
            for (int i = 0; i < VPL; i++)
                if (lane + 32 * i < cv) {
#pragma unroll
                    for (int k = 0; k < 8; k++) acc[i][k] += v[u][i][k];
                }
    }
    for (; j < hi; j++) {
        const T* row = dx0 + (int64_t)spos[j] * C;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            int idx = lane + 32 * i;
            if (idx < cv) {
                float v[8];
                load8(row + idx * 8, v);
#pragma unroll
                for (int k = 0; k < 8; k++) acc[i][k] += v[k];
            }
        }
    }
}

template <int VPL>
__device__ __forceinline__ void enc_flush(float (&acc)[VPL][8], float* dst, bool accumulate, int C, int lane) {
    const int cv = C / 8;
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        int idx = lane + 32 * i;
        if (idx < cv) {
            float* p = dst + idx * 8;
            if (accumulate) {
                float o[8];
                load8(p, o);
#pragma unroll
                for (int k = 0; k < 8; k++) acc[i][k] += o[k];
            }
            store8(p, acc[i]);
        }
#pragma unroll
        for (int k = 0; k < 8; k++) acc[i][k] = 0.f;
    }
}

// One warp per 32-entry chunk of the sorted list. A run of equal ids that
// lies wholly inside the chunk is added to dwte here. A run that crosses the
// chunk's end and starts inside it goes to tail[chunk]; the piece at the
// chunk's start that continues a run from an earlier chunk goes to head[chunk].
template <typename T, int VPL>
__global__ void __launch_bounds__(256) enc_piece_kernel(float* dwte, float* head, float* tail, const T* dx0,
                                                        const uint32_t* skey, const int32_t* spos, int n, int C) {
    const int chunk = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    const int lo = chunk * ENC_CHUNK;
    if (lo >= n) return;
    const int hi = min(n, lo + ENC_CHUNK);
    float acc[VPL][8];
#pragma unroll
    for (int i = 0; i < VPL; i++)
#pragma unroll
        for (int k = 0; k < 8; k++) acc[i][k] = 0.f;
    const int cv = C / 8;
    int ps = lo;
    while (ps < hi) {
        int pe = ps + 1;
        while (pe < hi && skey[pe] == skey[ps]) pe++;
        const bool starts = enc_is_head(skey, ps);
        const bool ends = (pe == n) || skey[pe] != skey[ps];
        if (starts && ends) {
            // the dwte row is loaded first, so its latency overlaps the row sums
            float* dst = dwte + (int64_t)skey[ps] * C;
            float pre[VPL][8];
#pragma unroll
            for (int i = 0; i < VPL; i++)
                if (lane + 32 * i < cv) load8(dst + (lane + 32 * i) * 8, pre[i]);
            enc_sum_rows<T, VPL>(acc, dx0, spos, ps, pe, C, lane);
#pragma unroll
            for (int i = 0; i < VPL; i++)
                if (lane + 32 * i < cv) {
#pragma unroll
                    for (int k = 0; k < 8; k++) acc[i][k] += pre[i][k];
                }
            enc_flush<VPL>(acc, dst, false, C, lane);
            ps = pe;
            continue;
        }
        enc_sum_rows<T, VPL>(acc, dx0, spos, ps, pe, C, lane);
        if (!starts)
            enc_flush<VPL>(acc, head + (int64_t)chunk * C, false, C, lane);
        else
            enc_flush<VPL>(acc, tail + (int64_t)chunk * C, false, C, lane);
        ps = pe;
    }
}

// One block of ENC_COMBINE_WARPS warps per chunk whose last run starts inside
// it and continues into later chunks (the other blocks return at once): the
// run's total is tail[chunk] + head[chunk+1] + ... + head[last chunk of the
// run]. Warp w sums the heads of the chunks chunk+1+w, chunk+1+w+W, ... in
// increasing order, two loads in flight; the block then adds tail[chunk] and
// the warps' partial sums in warp order and adds the total to dwte. The
// order of the additions is fixed, so the result is deterministic.
#define ENC_COMBINE_WARPS 4
template <int VPL>
__global__ void __launch_bounds__(32 * ENC_COMBINE_WARPS) enc_combine_kernel(float* dwte, const float* head,
                                                                              const float* tail,
                                                                              const uint32_t* skey, int n, int C) {
    __shared__ float part[ENC_COMBINE_WARPS - 1][2048];  // warps 1.. leave their sums here (C <= 2048)
    const int chunk = blockIdx.x;
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int lo = chunk * ENC_CHUNK;
    const int hi = min(n, lo + ENC_CHUNK);
    if (hi == n || skey[hi] != skey[hi - 1]) return;  // last run ends in this chunk
    int start = hi - 1;
    while (start > lo && skey[start - 1] == skey[hi - 1]) start--;
    if (!enc_is_head(skey, start)) return;  // run began in an earlier chunk
    const uint32_t key = skey[hi - 1];
    // the last chunk of the run: the first later chunk that does not run on
    // into the next; each lane tests one chunk, 32 chunks per step
    int last = chunk + 1;
    for (;;) {
        const int cc = last + lane;
        const int chi = min(n, (cc + 1) * ENC_CHUNK);
        const bool stop = chi == n || skey[chi] != key || skey[chi - 1] != key;
        const unsigned m = __ballot_sync(0xffffffffu, stop);
        if (m) {
            last += __ffs(m) - 1;
            break;
        }
        last += 32;
    }
    const int cv = C / 8;
    float acc[VPL][8];
#pragma unroll
    for (int i = 0; i < VPL; i++)
#pragma unroll
        for (int k = 0; k < 8; k++) acc[i][k] = 0.f;
    int c = chunk + 1 + w;
    for (; c + ENC_COMBINE_WARPS <= last; c += 2 * ENC_COMBINE_WARPS) {
        float v0[VPL][8], v1[VPL][8];
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                load8(head + (int64_t)c * C + idx * 8, v0[i]);
                load8(head + (int64_t)(c + ENC_COMBINE_WARPS) * C + idx * 8, v1[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < VPL; i++)
            if (lane + 32 * i < cv) {
#pragma unroll
                for (int k = 0; k < 8; k++) acc[i][k] += v0[i][k];
#pragma unroll
                for (int k = 0; k < 8; k++) acc[i][k] += v1[i][k];
            }
    }
    if (c <= last) {
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                float v[8];
                load8(head + (int64_t)c * C + idx * 8, v);
#pragma unroll
                for (int k = 0; k < 8; k++) acc[i][k] += v[k];
            }
        }
    }
    if (w > 0) {
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv)
#pragma unroll
                for (int k = 0; k < 8; k++) part[w - 1][idx * 8 + k] = acc[i][k];
        }
    }
    __syncthreads();
    if (w == 0) {
        float tot[VPL][8];
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            const int idx = lane + 32 * i;
            if (idx < cv) {
                load8(tail + (int64_t)chunk * C + idx * 8, tot[i]);
#pragma unroll
                for (int k = 0; k < 8; k++) tot[i][k] += acc[i][k];
                for (int ww = 1; ww < ENC_COMBINE_WARPS; ww++)
#pragma unroll
                    for (int k = 0; k < 8; k++) tot[i][k] += part[ww - 1][idx * 8 + k];
            }
        }
        enc_flush<VPL>(tot, dwte + (int64_t)key * C, true, C, lane);
    }
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t encoder_backward_scratch(int B, int T, int C) {
    const size_t n = (size_t)B * T;
    const size_t nblk = (n + ENC_TILE - 1) / ENC_TILE;
    const size_t nchunk = (n + ENC_CHUNK - 1) / ENC_CHUNK;
    return 4 * align256(n * 4) + align256(256 * nblk * 4) + 2 * align256(nchunk * C * 4);
}

template <typename T, int VPL>
static void enc_sum_launch(float* dwte, float* head, float* tail, const void* dx0, const uint32_t* skey,
                           const int32_t* spos, int n, int C, cudaStream_t s) {
    const int nchunk = (n + ENC_CHUNK - 1) / ENC_CHUNK;
    const int blocks = (nchunk * 32 + 255) / 256;
    enc_piece_kernel<T, VPL><<<blocks, 256, 0, s>>>(dwte, head, tail, (const T*)dx0, skey, spos, n, C);
    enc_combine_kernel<VPL><<<nchunk, 32 * ENC_COMBINE_WARPS, 0, s>>>(dwte, head, tail, skey, n, C);
}

template <typename T>
static void enc_sum_dispatch(float* dwte, float* head, float* tail, const void* dx0, const uint32_t* skey,
                             const int32_t* spos, int n, int C, cudaStream_t s) {
    const int vpl = (C / 8 + 31) / 32;
    switch (vpl) {
        case 1: enc_sum_launch<T, 1>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
        case 2: enc_sum_launch<T, 2>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
        case 3: enc_sum_launch<T, 3>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
        case 4: enc_sum_launch<T, 4>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
        case 5: enc_sum_launch<T, 5>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
        case 6: enc_sum_launch<T, 6>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
        case 7: enc_sum_launch<T, 7>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
        default: enc_sum_launch<T, 8>(dwte, head, tail, dx0, skey, spos, n, C, s); break;
    }
}

int launch_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dx0, const int32_t* tokens, int B, int T,
                            int C, void* scratch, cudaStream_t s, int accumulate) {
    const int n = B * T;
    const int nblk = (n + ENC_TILE - 1) / ENC_TILE;
    const int nchunk = (n + ENC_CHUNK - 1) / ENC_CHUNK;
    char* p = (char*)scratch;
    uint32_t* ka = (uint32_t*)p; p += align256((size_t)n * 4);
    int32_t* va = (int32_t*)p; p += align256((size_t)n * 4);
    uint32_t* kb = (uint32_t*)p; p += align256((size_t)n * 4);
    int32_t* vb = (int32_t*)p; p += align256((size_t)n * 4);
    int32_t* hist = (int32_t*)p; p += align256((size_t)256 * nblk * 4);
    float* head = (float*)p; p += align256((size_t)nchunk * C * 4);
    float* tail = (float*)p;
    int launches = 0;
    {
        const int blocks = (T * (C / 8) + 255) / 256;
        if (dtype == GPT2_MODE_BF16)
            encoder_bwd_wpe_kernel<bf16><<<blocks, 256, 0, s>>>(dwpe, (const bf16*)dx0, B, T, C, accumulate);
        else
            encoder_bwd_wpe_kernel<float><<<blocks, 256, 0, s>>>(dwpe, (const float*)dx0, B, T, C, accumulate);
        launches++;
    }
    enc_init_kernel<<<(n + 255) / 256, 256, 0, s>>>(ka, va, tokens, n);
    launches++;
    for (int pass = 0; pass < 2; pass++) {
        const int shift = pass * 8;
        uint32_t* kin = pass == 0 ? ka : kb;
        int32_t* vin = pass == 0 ? va : vb;
        uint32_t* kout = pass == 0 ? kb : ka;
        int32_t* vout = pass == 0 ? vb : va;
        enc_hist_kernel<<<nblk, ENC_TILE, 0, s>>>(hist, kin, n, shift);
        enc_scan_kernel<<<1, 1024, 0, s>>>(hist, 256 * nblk);
        enc_scatter_kernel<<<nblk, ENC_TILE, 0, s>>>(kout, vout, kin, vin, hist, n, shift);
        launches += 3;
    }
    // After two passes the sorted list is back in (ka, va).
    if (dtype == GPT2_MODE_BF16)
        enc_sum_dispatch<bf16>(dwte, head, tail, dx0, ka, va, n, C, s);
    else
        enc_sum_dispatch<float>(dwte, head, tail, dx0, ka, va, n, C, s);
    launches += 2;
    return launches;
}

// ===================================================================== GELU, residual

#define EW_UNROLL 4
#define EW_THREADS 256

// op 0: out = gelu(a); op 1: out = b * gelu'(a); op 2: out = a + b; op 3:
// out = a * b; op 4: out = gelu(a) and b = gelu'(a) (b may alias a).
template <typename T, int OP>
__global__ void __launch_bounds__(EW_THREADS) ew_kernel(T* out, const T* a, T* b, int64_t n8) {
    // No __restrict__: out may alias a (in-place GELU and residual accumulate).
    // Each thread loads all its inputs before its first store.
    const int64_t base = (int64_t)blockIdx.x * (EW_THREADS * EW_UNROLL) + threadIdx.x;
    float va[EW_UNROLL][8], vb[EW_UNROLL][8];
#pragma unroll
    for (int u = 0; u < EW_UNROLL; u++) {
        const int64_t i = base + (int64_t)u * EW_THREADS;
        if (i < n8) {
            load8_stream(a + i * 8, va[u]);
            if (OP != 0 && OP != 4) load8_stream(b + i * 8, vb[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < EW_UNROLL; u++) {
        const int64_t i = base + (int64_t)u * EW_THREADS;
        if (i < n8) {
            float r[8], r2[8];
            if (sizeof(T) == 2 && (OP == 0 || OP == 1 || OP == 4)) {
                // bf16: the paired GELU the GEMM epilogues use (same bits)
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    float g0, g1, d0, d1;
                    tc::gelu_pair(va[u][j], va[u][j + 1], g0, g1, d0, d1);
                    if (OP == 1) {
                        r[j] = vb[u][j] * d0;
                        r[j + 1] = vb[u][j + 1] * d1;
                    } else {
                        r[j] = g0;
                        r[j + 1] = g1;
                        r2[j] = d0;
                        r2[j + 1] = d1;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    if (OP == 0) r[j] = gelu_fwd_f<T>(va[u][j]);
                    else if (OP == 1) r[j] = vb[u][j] * gelu_grad_f<T>(va[u][j]);
                    else if (OP == 2) r[j] = va[u][j] + vb[u][j];
                    else if (OP == 3) r[j] = va[u][j] * vb[u][j];
                    else gelu_both_f<T>(va[u][j], r[j], r2[j]);
                }
            }
            store8(out + i * 8, r);
            if (OP == 4) store8(b + i * 8, r2);
        }
    }
}

template <int OP>
static int ew_launch(int dtype, void* out, const void* a, void* b, int64_t n, cudaStream_t s) {
    const int64_t n8 = n / 8;
    const int64_t per_block = EW_THREADS * EW_UNROLL;
    const int blocks = (int)((n8 + per_block - 1) / per_block);
    if (blocks == 0) return 0;
    if (dtype == GPT2_MODE_BF16)
        ew_kernel<bf16, OP><<<blocks, EW_THREADS, 0, s>>>((bf16*)out, (const bf16*)a, (bf16*)b, n8);
    else
        ew_kernel<float, OP><<<blocks, EW_THREADS, 0, s>>>((float*)out, (const float*)a, (float*)b, n8);
    return 1;
}

int launch_gelu_forward(int dtype, void* g, const void* u, int64_t n, cudaStream_t s) {
    return ew_launch<0>(dtype, g, u, nullptr, n, s);
}
int launch_gelu_backward(int dtype, void* du, const void* u, const void* dg, int64_t n, cudaStream_t s) {
    return ew_launch<1>(dtype, du, u, const_cast<void*>(dg), n, s);
}
int launch_residual_forward(int dtype, void* out, const void* a, const void* b, int64_t n, cudaStream_t s) {
    return ew_launch<2>(dtype, out, a, const_cast<void*>(b), n, s);
}
int launch_residual_backward(int dtype, void* dres, const void* dbranch, int64_t n, cudaStream_t s) {
    return ew_launch<2>(dtype, dres, dres, const_cast<void*>(dbranch), n, s);
}
int launch_mul(int dtype, void* out, const void* a, const void* b, int64_t n, cudaStream_t s) {
    return ew_launch<3>(dtype, out, a, const_cast<void*>(b), n, s);
}
int launch_gelu_both(int dtype, void* out, void* dgelu, const void* u, int64_t n, cudaStream_t s) {
    return ew_launch<4>(dtype, out, u, dgelu, n, s);
}

// ===================================================================== bias gradient

#define BIAS_ROWS_PER_CHUNK 128

// Stage 1: block (32 column vectors) x (8 row lanes) sums one chunk of rows
// for 256 columns into partial[chunk][c]; the blocks of one column slab
// step over the chunks by gridDim.y (at most 65535 of them per launch).
template <typename T>
__global__ void __launch_bounds__(256) bias_partial_kernel(float* __restrict__ partial, const T* __restrict__ dy,
                                                           int N, int C, int chunks) {
    __shared__ float sm[8][256 + 8];
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
    const int c = (blockIdx.x * 32 + tx) * 8;
    for (int chunk = blockIdx.y; chunk < chunks; chunk += gridDim.y) {
        const int r0 = chunk * BIAS_ROWS_PER_CHUNK;
        const int r1 = min(N, r0 + BIAS_ROWS_PER_CHUNK);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (c < C) {
#pragma unroll 4
            for (int r = r0 + ty; r < r1; r += 8) {
                float v[8];
                load8_stream(dy + (int64_t)r * C + c, v);
#pragma unroll
                for (int j = 0; j < 8; j++) acc[j] += v[j];
            }
        }
        __syncthreads();  // the previous chunk's sums have been read
#pragma unroll
        for (int j = 0; j < 8; j++) sm[ty][tx * 8 + j] = acc[j];
        __syncthreads();
        const int col = threadIdx.x;  // 0..255 within this block's slab
        const int gc = blockIdx.x * 256 + col;
        if (gc < C) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < 8; k++) s += sm[k][col];
            partial[(int64_t)chunk * C + gc] = s;
        }
    }
}

// Deterministic column sums of an fp32 [R, ncols] matrix (row stride ncols):
// out[c] = sum over r of in[r][c], r in ascending order within each of 32
// row lanes, then the 32 lane sums in lane order. Block = 32 columns x 32 row
// lanes; a warp reads 32 consecutive floats of one row (coalesced). Columns
// c >= split go to out2[c - split] (two outputs that share one pass).
// out_q[c] = column sums of in [R, ncols] for column q * seg + c: the ncols
// columns are up to three consecutive segments of seg columns, each going to
// its own output. Fixed order (deterministic).
struct ColsumOut {
    float* p[3];
};

__global__ void __launch_bounds__(1024) colsum_kernel(ColsumOut outs, int seg, const float* __restrict__ in, int R,
                                                      int ncols, int accumulate) {
    __shared__ float sm[32][33];
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
    const int c = blockIdx.x * 32 + tx;
    float s = 0.f;
    if (c < ncols) {
#pragma unroll 4
        for (int r = ty; r < R; r += 32) s += in[(int64_t)r * ncols + c];
    }
    sm[ty][tx] = s;
    __syncthreads();
    if (ty == 0 && c < ncols) {
        float t = 0.f;
        for (int k = 0; k < 32; k++) t += sm[k][tx];
        const int q = c / seg;
        if (q < 3 && outs.p[q]) {
            float* o = outs.p[q] + (c - q * seg);
            *o = accumulate ? *o + t : t;
        }
    }
}

int launch_colsum3(float* out0, float* out1, float* out2, int seg, const float* in, int R, int ncols,
                   cudaStream_t s, int accumulate) {
    ColsumOut o = {{out0, out1, out2}};
    colsum_kernel<<<(ncols + 31) / 32, 1024, 0, s>>>(o, seg, in, R, ncols, accumulate);
    return 1;
}

int launch_colsum(float* out, float* out2, int split, const float* in, int R, int ncols, cudaStream_t s) {
    return launch_colsum3(out, out2, nullptr, split, in, R, ncols, s);
}

// Many column sums in one launch: block b serves 32 columns of the job whose
// block range holds b, with the arithmetic of colsum_kernel (so a job gives
// the bits colsum_kernel gives for it).
constexpr int COLSUM_MAX_JOBS = 32;
struct ColsumBatch {
    ColsumJob job[COLSUM_MAX_JOBS];
    int block0[COLSUM_MAX_JOBS + 1];
    int n;
};

__global__ void __launch_bounds__(1024) colsum_jobs_kernel(const __grid_constant__ ColsumBatch b) {
    __shared__ float sm[32][33];
    int k = 0;
    while (k + 1 < b.n && (int)blockIdx.x >= b.block0[k + 1]) k++;
    const ColsumJob& j = b.job[k];
    const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
    const int c = ((int)blockIdx.x - b.block0[k]) * 32 + tx;
    float s = 0.f;
    if (c < j.ncols) {
#pragma unroll 4
        for (int r = ty; r < j.R; r += 32) s += j.in[(int64_t)r * j.ncols + c];
    }
    sm[ty][tx] = s;
    __syncthreads();
    if (ty == 0 && c < j.ncols) {
        float t = 0.f;
        for (int q = 0; q < 32; q++) t += sm[q][tx];
        const int q = c / j.seg;
        if (q < 3 && j.out[q]) {
            float* o = j.out[q] + (c - q * j.seg);
            *o = j.accumulate ? *o + t : t;
        }
    }
}

int launch_colsum_jobs(const ColsumJob* jobs, int n, cudaStream_t s) {
    int launches = 0;
    for (int i0 = 0; i0 < n; i0 += COLSUM_MAX_JOBS) {
        ColsumBatch b;
        b.n = n - i0 < COLSUM_MAX_JOBS ? n - i0 : COLSUM_MAX_JOBS;
        int blocks = 0;
        for (int k = 0; k < b.n; k++) {
            b.job[k] = jobs[i0 + k];
            b.block0[k] = blocks;
            blocks += b.job[k].R > 0 ? (b.job[k].ncols + 31) / 32 : 0;
        }
        b.block0[b.n] = blocks;
        if (blocks == 0) continue;
        colsum_jobs_kernel<<<blocks, 1024, 0, s>>>(b);
        launches++;
    }
    return launches;
}

size_t bias_backward_scratch(int N, int C) {
    const size_t chunks = ((size_t)N + BIAS_ROWS_PER_CHUNK - 1) / BIAS_ROWS_PER_CHUNK;
    return chunks * C * 4;
}

int launch_bias_partials(int dtype, float* partial, const void* dy, int N, int C, cudaStream_t s, int* rows) {
    const int chunks = (int)(((int64_t)N + BIAS_ROWS_PER_CHUNK - 1) / BIAS_ROWS_PER_CHUNK);
    *rows = chunks;
    if (chunks == 0) return 0;
    dim3 grid((C + 255) / 256, chunks < 65535 ? chunks : 65535);
    if (dtype == GPT2_MODE_BF16)
        bias_partial_kernel<bf16><<<grid, 256, 0, s>>>(partial, (const bf16*)dy, N, C, chunks);
    else
        bias_partial_kernel<float><<<grid, 256, 0, s>>>(partial, (const float*)dy, N, C, chunks);
    return 1;
}

int launch_bias_backward(int dtype, float* dbias, const void* dy, int N, int C, void* scratch, cudaStream_t s,
                         int accumulate) {
    int chunks = 0;
    launch_bias_partials(dtype, (float*)scratch, dy, N, C, s, &chunks);
    launch_colsum3(dbias, nullptr, nullptr, C, (const float*)scratch, chunks, C, s, accumulate);
    return 2;
}

// ===================================================================== AdamW

#define ADAM_UNROLL 2

// Thread per 4 consecutive parameters (float4), ADAM_UNROLL groups per thread.
// The gradient enters as g * grad_scale * clip, clip = min(1, max_norm /
// (||g|| grad_scale + 1e-6)) when gnorm (the device-held ||g||) is given and
// max_norm > 0; weight decay applies to the 64-element chunks whose bit is set
// in decay_bits (every chunk when decay_bits is null).
__global__ void __launch_bounds__(256) adamw_kernel(float* __restrict__ theta, bf16* __restrict__ pbf,
                                                    const float* __restrict__ grad, float* __restrict__ m,
                                                    float* __restrict__ v, int64_t n4, float lr, float b1, float b2,
                                                    float eps, float wd, float inv_bc1, float inv_bc2,
                                                    float grad_scale, const float* __restrict__ gnorm, float max_norm,
                                                    const uint32_t* __restrict__ decay_bits,
                                                    const float* __restrict__ hp) {
    if (hp) {
        // the step's values from device memory (a captured step graph reads
        // the values written before each launch)
        lr = hp[0];
        b1 = hp[1];
        b2 = hp[2];
        eps = hp[3];
        wd = hp[4];
        inv_bc1 = hp[5];
        inv_bc2 = hp[6];
        grad_scale = hp[7];
    }
    const int64_t base = (int64_t)blockIdx.x * (256 * ADAM_UNROLL) + threadIdx.x;
    float gs = grad_scale;
    if (gnorm && max_norm > 0.f) gs *= fminf(1.f, max_norm / (*gnorm * grad_scale + 1e-6f));
    float4 th[ADAM_UNROLL], g[ADAM_UNROLL], mm[ADAM_UNROLL], vv[ADAM_UNROLL];
#pragma unroll
    for (int u = 0; u < ADAM_UNROLL; u++) {
        const int64_t i = base + u * 256;
        if (i < n4) {
            th[u] = __ldcs(reinterpret_cast<const float4*>(theta) + i);
            g[u] = __ldcs(reinterpret_cast<const float4*>(grad) + i);
            mm[u] = __ldcs(reinterpret_cast<const float4*>(m) + i);
            vv[u] = __ldcs(reinterpret_cast<const float4*>(v) + i);
        }
    }
#pragma unroll
    for (int u = 0; u < ADAM_UNROLL; u++) {
        const int64_t i = base + u * 256;
        if (i >= n4) continue;
        float* pt = &th[u].x;
        const float* pg = &g[u].x;
        float* pm = &mm[u].x;
        float* pv = &vv[u].x;
        // float4 i holds elements 4i..4i+3, in 64-element chunk i / 16
        const float wdu = decay_bits && !((decay_bits[i >> 9] >> ((i >> 4) & 31)) & 1u) ? 0.f : wd;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float gj = pg[j] * gs;
            pm[j] = b1 * pm[j] + (1.f - b1) * gj;
            pv[j] = b2 * pv[j] + (1.f - b2) * gj * gj;
            const float mhat = pm[j] * inv_bc1;
            const float vhat = pv[j] * inv_bc2;
            pt[j] = pt[j] - lr * (mhat / (sqrtf(vhat) + eps) + wdu * pt[j]);
        }
        __stcs(reinterpret_cast<float4*>(theta) + i, th[u]);
        __stcs(reinterpret_cast<float4*>(m) + i, mm[u]);
        __stcs(reinterpret_cast<float4*>(v) + i, vv[u]);
        if (pbf) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(pt[0], pt[1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(pt[2], pt[3]);
            uint2 w;
            w.x = *reinterpret_cast<uint32_t*>(&lo);
            w.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(pbf)[i] = w;
        }
    }
}

// hp, when given: a device block {lr, beta1, beta2, eps, weight_decay,
// 1/(1-beta1^t), 1/(1-beta2^t), grad_scale} read in place of those arguments.
int launch_adamw(float* master, void* pbf, const float* grad, float* m, float* v, int64_t n, float lr, float b1,
                 float b2, float eps, float wd, int t, cudaStream_t s, float grad_scale, const float* gnorm,
                 float max_norm, const uint32_t* decay_bits, const float* hp) {
    const int64_t n4 = n / 4;
    const double bc1 = 1.0 - pow((double)b1, (double)t);
    const double bc2 = 1.0 - pow((double)b2, (double)t);
    const int64_t per_block = 256 * ADAM_UNROLL;
    const int blocks = (int)((n4 + per_block - 1) / per_block);
    if (blocks == 0) return 0;
    adamw_kernel<<<blocks, 256, 0, s>>>(master, (bf16*)pbf, grad, m, v, n4, lr, b1, b2, eps, wd,
                                        (float)(1.0 / bc1), (float)(1.0 / bc2), grad_scale, gnorm, max_norm,
                                        decay_bits, hp);
    return 1;
}

// ===================================================================== gradient norm

// ||g||_2 over n fp32 values (n % 4 == 0), deterministic: block b sums its
// fixed contiguous range of float4s (thread t takes every 256th from t, then a
// fixed shuffle tree), one block adds the GN_BLOCKS partial sums in order.
#define GN_BLOCKS 1024

__global__ void __launch_bounds__(256) grad_sumsq_kernel(float* __restrict__ partial, const float* __restrict__ g,
                                                         int64_t n4) {
    __shared__ float sh[8];
    const int64_t per = (n4 + GN_BLOCKS - 1) / GN_BLOCKS;
    const int64_t lo = (int64_t)blockIdx.x * per;
    const int64_t hi = lo + per < n4 ? lo + per : n4;
    float acc = 0.f;
    for (int64_t i = lo + threadIdx.x; i < hi; i += 256) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(g) + i);
        acc += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    acc = warp_sum(acc);
    if (threadIdx.x % 32 == 0) sh[threadIdx.x / 32] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; w++) t += sh[w];
        partial[blockIdx.x] = t;
    }
}

__global__ void __launch_bounds__(1024) grad_norm_final_kernel(float* __restrict__ out,
                                                               const float* __restrict__ partial, int root) {
    __shared__ float sh[32];
    float v = partial[threadIdx.x];  // GN_BLOCKS == blockDim.x
    v = warp_sum(v);
    if (threadIdx.x % 32 == 0) sh[threadIdx.x / 32] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 32; w++) t += sh[w];
        *out = root ? sqrtf(t) : t;
    }
}

size_t grad_norm_scratch() { return GN_BLOCKS * 4; }

int launch_grad_norm(float* norm_out, float* partial, const float* g, int64_t n, cudaStream_t s, int root) {
    grad_sumsq_kernel<<<GN_BLOCKS, 256, 0, s>>>(partial, g, n / 4);
    grad_norm_final_kernel<<<1, GN_BLOCKS, 0, s>>>(norm_out, partial, root);
    return 2;
}
