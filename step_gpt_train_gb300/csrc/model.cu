// GPT-2 training step: workspace plan, init, and the forward / backward /
// AdamW launch sequences behind the C ABI of gpt2.h.
//
// The sequence follows the kernel table of llm.c "State of the Union
// [May 3, 2024]" ("Runtime, DRAM traffic, instructions"): per step one
// encoder forward, 2L+1 layernorm forwards, 4 matmuls per layer plus the LM
// head, L attention forwards, 2L residuals, L GELUs, the fused classifier;
// then the mirrored backward and one AdamW over every parameter. Around it:
// gradient accumulation, the global gradient norm and clipping, the decay
// mask, gpt2_step (the whole step captured once and replayed as a CUDA
// graph) and the sharded (ZeRO-1 style) AdamW over ranges of the flat layout.
#include "common.cuh"
#include "launch.h"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

int gpt2_num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    }
    return n;
}

namespace {

constexpr size_t WS_ALIGN = 1024;
constexpr int64_t PARAM_ALIGN = 64;  // elements; keeps every tensor 128-byte aligned in bf16

enum InitKind { INIT_NORMAL = 0, INIT_ZERO = 1, INIT_ONE = 2 };

struct TensorSpec {
    std::string name;
    int64_t rows, cols;
    int64_t offset;  // element offset in the flat parameter buffers
    int init;
    double std;
};

struct LayerBufs {
    void *x, *ln1, *qkv, *atty, *x1, *ln2, *fch, *fchg;
    float *mean1, *rstd1, *lse, *mean2, *rstd2;
};

}  // namespace

struct gpt2 {
    gpt2_config cfg;
    int L, C, H, V, Vp, maxT, maxB, mode, dtype;
    size_t act;  // bytes per activation element
    cudaStream_t stream;
    uint8_t* ws;
    size_t ws_bytes;
    std::vector<TensorSpec> tensors;
    int64_t np;  // flat parameter count (with alignment gaps)
    float *master, *grads, *adam_m, *adam_v;
    void* params;  // compute copy: bf16 (bf16 mode) or the master itself
    int* status;
    float* loss_dev;
    int32_t* tokens;
    int32_t* targets;  // gpt2_step's copy of the step's targets (a fixed address for its graph)
    float* hp_dev;     // gpt2_step: the AdamW values of the step, read by the captured AdamW
    std::vector<LayerBufs> layers;
    void *xL, *lnf, *logits, *fwd_tmp;
    float *meanf, *rstdf, *losses;
    void *dres, *dtmp, *dbig, *dqkv;
    void* scratch;
    size_t scratch_bytes;
    // The backward's parameter-gradient column sums (LayerNorm scale and
    // shift, the four biases of a block): their partial sums go to regions of
    // this pool as they are formed, and one deferred launch at the end of the
    // backward reduces them all.
    float* cs_pool;
    size_t cs_pool_bytes, cs_used;
    std::vector<ColsumJob> cs_jobs;
    // FP8 linear layers (gpt2_set_fp8): which ones, and the codes they read,
    // in the caller's second workspace
    int fp8 = 0;
    uint8_t *f8_x = nullptr, *f8_w = nullptr, *f8_wT = nullptr, *f8_dy = nullptr, *f8_dyT = nullptr;
    std::vector<uint8_t*> f8_xT;  // per FP8 linear (slot): the forward's transposed codes of its input x
    float* f8_scales = nullptr;   // per FP8 linear: (scale, 1/scale) of x, W and dy
    unsigned* f8_amax = nullptr;  // per FP8 linear: amax of x and of dy (float bits) from the kernels that write them
    float* f8_partial = nullptr;  // amax partials
    void* f8_scratch = nullptr;   // split-K partial tiles of the FP8 weight gradients
    size_t f8_scratch_bytes = 0;
    int B, T;
    int state;  // 0: none, 1: forward with targets done, 2: backward done
    int grad_accum;          // backward adds into the gradients instead of overwriting them
    float* gnorm;            // device: ||g||_2 of the last gpt2_grad_norm / clipped AdamW step
    float* gnorm_partial;    // device: its per-block partial sums
    uint32_t* decay_bits;    // device: one bit per 64-element chunk, set for the 2-D tensors
    int64_t launches;
    int64_t fam_calls[GPT2_K_COUNT], fam_launches[GPT2_K_COUNT];
    double fam_work[GPT2_K_COUNT], fam_ms[GPT2_K_COUNT];
    bool timing;
    struct Pending { int fam; cudaEvent_t a, b; };
    std::vector<Pending> pending;
    std::vector<cudaEvent_t> pool;
    // gpt2_step: the captured step and what it was captured for
    struct StepKey {
        int B, T, grad_accum, clip, decay_mask, fp8;
        float max_grad_norm;
        bool operator==(const StepKey& o) const {
            return B == o.B && T == o.T && grad_accum == o.grad_accum && clip == o.clip &&
                   decay_mask == o.decay_mask && fp8 == o.fp8 && max_grad_norm == o.max_grad_norm;
        }
    };
    StepKey step_key{};
    bool step_warm = false;                // one eager step ran with step_key
    cudaGraphExec_t step_exec = nullptr;   // the captured step for step_key
    cudaStream_t capture_stream = nullptr;  // the graph is captured here (the caller's may be the legacy stream)
    int64_t step_launches = 0;             // kernel launches in one replay
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool config_ok(const gpt2_config* c) {
    if (!c) return false;
    if (c->n_layer < 1 || c->n_embd < 8 || c->n_head < 1 || c->vocab < 1 || c->max_T < 1 || c->max_B < 1) return false;
    if (c->n_embd % 8 || c->n_embd % c->n_head || c->n_embd > 2048) return false;
    if (c->vocab_padded < c->vocab || c->vocab_padded % 8 || c->vocab_padded > 65536) return false;
    const int hd = c->n_embd / c->n_head;
    if (c->mode == GPT2_MODE_BF16) return hd == 64;
    if (c->mode == GPT2_MODE_FP32) return hd == 8 || hd == 16 || hd == 32 || hd == 64;
    return false;
}

std::vector<TensorSpec> make_specs(const gpt2_config* c, int64_t* np_out) {
    const int64_t C = c->n_embd, L = c->n_layer;
    const double std_w = 0.02, std_res = 0.02 / std::sqrt(2.0 * (double)L);
    std::vector<TensorSpec> t;
    auto add = [&](const std::string& n, int64_t r, int64_t cc, int init, double sd) {
        t.push_back({n, r, cc, 0, init, sd});
    };
    add("wte", c->vocab_padded, C, INIT_NORMAL, std_w);
    add("wpe", c->max_T, C, INIT_NORMAL, std_w);
    for (int l = 0; l < L; l++) {
        const std::string p = "h" + std::to_string(l) + ".";
        add(p + "ln1.g", C, 1, INIT_ONE, 0);
        add(p + "ln1.b", C, 1, INIT_ZERO, 0);
        add(p + "qkv.w", 3 * C, C, INIT_NORMAL, std_w);
        add(p + "qkv.b", 3 * C, 1, INIT_ZERO, 0);
        add(p + "proj.w", C, C, INIT_NORMAL, std_res);
        add(p + "proj.b", C, 1, INIT_ZERO, 0);
        add(p + "ln2.g", C, 1, INIT_ONE, 0);
        add(p + "ln2.b", C, 1, INIT_ZERO, 0);
        add(p + "fc.w", 4 * C, C, INIT_NORMAL, std_w);
        add(p + "fc.b", 4 * C, 1, INIT_ZERO, 0);
        add(p + "fcproj.w", C, 4 * C, INIT_NORMAL, std_res);
        add(p + "fcproj.b", C, 1, INIT_ZERO, 0);
    }
    add("lnf.g", C, 1, INIT_ONE, 0);
    add("lnf.b", C, 1, INIT_ZERO, 0);
    int64_t off = 0;
    for (auto& s : t) {
        s.offset = off;
        off += (s.rows * s.cols + PARAM_ALIGN - 1) / PARAM_ALIGN * PARAM_ALIGN;
    }
    *np_out = off;
    return t;
}

enum { T_WTE = 0, T_WPE = 1 };
inline int tidx(int l, int k) { return 2 + 12 * l + k; }  // k: 0 ln1.g 1 ln1.b 2 qkv.w 3 qkv.b 4 proj.w 5 proj.b
                                                          //    6 ln2.g 7 ln2.b 8 fc.w 9 fc.b 10 fcproj.w 11 fcproj.b
inline int tlnf(int L, int k) { return 2 + 12 * L + k; }

// Carve the workspace. With m == nullptr only the total size is computed.
size_t plan(const gpt2_config* c, gpt2* m) {
    int64_t np = 0;
    make_specs(c, &np);
    const size_t act = c->mode == GPT2_MODE_BF16 ? 2 : 4;
    const size_t BT = (size_t)c->max_B * c->max_T;
    const size_t C = c->n_embd, L = c->n_layer, Vp = c->vocab_padded, H = c->n_head;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        off = align_up(off, WS_ALIGN);
        size_t r = off;
        off += bytes;
        return r;
    };
    const size_t o_status = take(256);
    const size_t o_tokens = take(BT * 4);
    const size_t o_targets = take(BT * 4);
    const size_t o_master = take((size_t)np * 4);
    const size_t o_params = c->mode == GPT2_MODE_BF16 ? take((size_t)np * 2) : o_master;
    const size_t o_grads = take((size_t)np * 4);
    const size_t o_m = take((size_t)np * 4);
    const size_t o_v = take((size_t)np * 4);
    const size_t o_gnp = take(grad_norm_scratch());
    const size_t o_decay = take((((size_t)np / 64 + 1) + 31) / 32 * 4);
    std::vector<size_t> lo(13 * L);
    for (size_t l = 0; l < L; l++) {
        size_t* p = &lo[13 * l];
        p[0] = take(BT * C * act);      // x (layer input)
        p[1] = take(BT * C * act);      // ln1
        p[2] = take(BT * 3 * C * act);  // qkv
        p[3] = take(BT * C * act);      // atty
        p[4] = take(BT * C * act);      // x1
        p[5] = take(BT * C * act);      // ln2
        p[6] = take(BT * 4 * C * act);  // fch
        p[7] = take(BT * 4 * C * act);  // fchg
        p[8] = take(BT * 4);            // mean1
        p[9] = take(BT * 4);            // rstd1
        p[10] = take(BT * H * 4);       // lse
        p[11] = take(BT * 4);           // mean2
        p[12] = take(BT * 4);           // rstd2
    }
    const size_t o_xL = take(BT * C * act);
    const size_t o_lnf = take(BT * C * act);
    const size_t o_meanf = take(BT * 4);
    const size_t o_rstdf = take(BT * 4);
    const size_t o_logits = take(BT * Vp * act);
    const size_t o_losses = take(BT * 4);
    const size_t o_fwd_tmp = take(BT * C * act);
    const size_t o_dres = take(BT * C * act);
    const size_t o_dtmp = take(BT * C * act);
    const size_t o_dbig = take(BT * 4 * C * act);
    const size_t o_dqkv = take(BT * 3 * C * act);
    // scratch: the largest need of any scratch-using op of the backward
    const int dt = c->mode;
    const int iBT = (int)BT, iC = (int)C, iVp = (int)Vp;
    size_t sc = 256;
    auto need = [&](size_t b) { sc = b > sc ? b : sc; };
    const int outs[4] = {3 * iC, iC, 4 * iC, iC};
    const int ins[4] = {iC, iC, iC, 4 * iC};
    for (int k = 0; k < 4; k++) {
        need(matmul_scratch(dt, outs[k], ins[k], iBT, 1, 1));    // dW (also when accumulating)
        need(matmul_scratch(dt, iBT, ins[k], outs[k], 0));       // dX
        need(bias_backward_scratch(iBT, outs[k]));
    }
    need(matmul_scratch(dt, iVp, iC, iBT, 1, 1));
    need(matmul_scratch(dt, iBT, iC, iVp, 0));
    need(layernorm_backward_scratch(iBT, iC));
    need(attention_backward_scratch(c->max_B, c->max_T, (int)H));
    need(encoder_backward_scratch(c->max_B, c->max_T, iC));
    const size_t o_scratch = take(sc);
    // the column-sum partials of one backward: per block two LayerNorms, the
    // MLP's first bias (from the GELU-gradient matmul, or the bias pass) and
    // the QKV bias (the bias pass); the final LayerNorm (each region rounded
    // up to WS_ALIGN)
    const size_t ln_part = align_up(layernorm_backward_scratch(iBT, iC), WS_ALIGN);
    const size_t fc_mm = (size_t)matmul_gelu_backward_colsum_rows(iBT) * 4 * C * 4;
    const size_t fc_part = align_up(std::max(bias_backward_scratch(iBT, 4 * iC), fc_mm), WS_ALIGN);
    const size_t qkv_part = align_up(bias_backward_scratch(iBT, 3 * iC), WS_ALIGN);
    const size_t cs_bytes = L * (2 * ln_part + fc_part + qkv_part) + ln_part;
    const size_t o_cs = take(cs_bytes);
    const size_t total = align_up(off, WS_ALIGN);
    if (m) {
        uint8_t* w = m->ws;
        m->np = np;
        m->status = (int*)(w + o_status);
        m->loss_dev = (float*)(w + o_status + 64);
        m->tokens = (int32_t*)(w + o_tokens);
        m->targets = (int32_t*)(w + o_targets);
        m->hp_dev = (float*)(w + o_status + 192);
        m->master = (float*)(w + o_master);
        m->params = w + o_params;
        m->grads = (float*)(w + o_grads);
        m->adam_m = (float*)(w + o_m);
        m->adam_v = (float*)(w + o_v);
        m->gnorm = (float*)(w + o_status + 128);
        m->gnorm_partial = (float*)(w + o_gnp);
        m->decay_bits = (uint32_t*)(w + o_decay);
        m->layers.resize(L);
        for (size_t l = 0; l < L; l++) {
            size_t* p = &lo[13 * l];
            LayerBufs& b = m->layers[l];
            b.x = w + p[0]; b.ln1 = w + p[1]; b.qkv = w + p[2]; b.atty = w + p[3]; b.x1 = w + p[4];
            b.ln2 = w + p[5]; b.fch = w + p[6]; b.fchg = w + p[7];
            b.mean1 = (float*)(w + p[8]); b.rstd1 = (float*)(w + p[9]); b.lse = (float*)(w + p[10]);
            b.mean2 = (float*)(w + p[11]); b.rstd2 = (float*)(w + p[12]);
        }
        m->xL = w + o_xL;
        m->lnf = w + o_lnf;
        m->meanf = (float*)(w + o_meanf);
        m->rstdf = (float*)(w + o_rstdf);
        m->logits = w + o_logits;
        m->losses = (float*)(w + o_losses);
        m->fwd_tmp = w + o_fwd_tmp;
        m->dres = w + o_dres;
        m->dtmp = w + o_dtmp;
        m->dbig = w + o_dbig;
        m->dqkv = w + o_dqkv;
        m->scratch = w + o_scratch;
        m->scratch_bytes = sc;
        m->cs_pool = (float*)(w + o_cs);
        m->cs_pool_bytes = cs_bytes;
        m->cs_used = 0;
    }
    return total;
}

// ---- counter-based init (splitmix64 + Box-Muller, both published) ----

inline uint64_t splitmix64_next(uint64_t& s) {
    s += 0x9E3779B97F4A7C15ULL;
    uint64_t z = s;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

// Element i of tensor k: counter k*2^40 + i; state seed ^ (counter * golden);
// two splitmix64 outputs give u1 in (0,1], u2 in [0,1); z = sqrt(-2 ln u1) cos(2 pi u2).
inline float init_draw(uint64_t seed, uint64_t k, uint64_t i, double sd) {
    uint64_t s = seed ^ (((k << 40) + i) * 0x9E3779B97F4A7C15ULL);
    const uint64_t r1 = splitmix64_next(s);
    const uint64_t r2 = splitmix64_next(s);
    const double u1 = ((double)(r1 >> 11) + 1.0) * 0x1p-53;
    const double u2 = (double)(r2 >> 11) * 0x1p-53;
    const double z = std::sqrt(-2.0 * std::log(u1)) * std::cos(2.0 * 3.141592653589793 * u2);
    return (float)(sd * z);
}

void init_host(const gpt2_config* c, uint64_t seed, const std::vector<TensorSpec>& specs, float* out) {
    unsigned nth = std::thread::hardware_concurrency();
    if (nth == 0) nth = 4;
    if (nth > 32) nth = 32;
    std::vector<std::thread> th;
    for (unsigned w = 0; w < nth; w++) {
        th.emplace_back([&, w] {
            for (size_t k = 0; k < specs.size(); k++) {
                const TensorSpec& s = specs[k];
                const int64_t n = s.rows * s.cols;
                const int64_t per = (n + nth - 1) / nth;
                const int64_t lo = (int64_t)w * per, hi = std::min<int64_t>(n, lo + per);
                for (int64_t i = lo; i < hi; i++) {
                    float v;
                    if (s.init == INIT_ZERO) v = 0.f;
                    else if (s.init == INIT_ONE) v = 1.f;
                    else v = init_draw(seed, (uint64_t)k, (uint64_t)i, s.std);
                    if (k == T_WTE && i / s.cols >= c->vocab) v = 0.f;  // padded vocab rows
                    out[s.offset + i] = v;
                }
            }
        });
    }
    for (auto& t : th) t.join();
}

__global__ void f32_to_bf16_kernel(bf16* __restrict__ out, const float* __restrict__ in, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = __float2bfloat16_rn(in[i]);
}

// ---- op accounting ----

struct Op {
    gpt2* m;
    int fam;
    cudaEvent_t a = nullptr;
    Op(gpt2* mm, int f) : m(mm), fam(f) {
        if (m->timing) {
            if (m->pool.empty()) {
                cudaEvent_t e;
                cudaEventCreate(&e);
                m->pool.push_back(e);
            }
            a = m->pool.back();
            m->pool.pop_back();
            cudaEventRecord(a, m->stream);
        }
    }
    // Record the op's launches and work; returns GPT2_OK or an error.
    int done(int launches, double work) {
        if (launches < 0) return launches;
        m->launches += launches;
        m->fam_calls[fam] += 1;
        m->fam_launches[fam] += launches;
        m->fam_work[fam] += work;
        if (a) {
            cudaEvent_t b;
            if (m->pool.empty()) cudaEventCreate(&b);
            else { b = m->pool.back(); m->pool.pop_back(); }
            cudaEventRecord(b, m->stream);
            m->pending.push_back({fam, a, b});
            a = nullptr;
        }
        return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
    }
};

#define TRY(x)                     \
    do {                           \
        int _r = (x);              \
        if (_r != GPT2_OK) return _r; \
    } while (0)

inline void* P(gpt2* m, int i) { return (uint8_t*)m->params + (size_t)m->tensors[i].offset * m->act; }
inline float* G(gpt2* m, int i) { return m->grads + m->tensors[i].offset; }

// A region of the column-sum pool for rows x ncols fp32 partials (null when
// the pool is exhausted, which plan() rules out for the configured sizes).
float* cs_take(gpt2* m, int rows, int ncols) {
    const size_t bytes = align_up((size_t)rows * ncols * 4, WS_ALIGN);
    if (m->cs_used + bytes > m->cs_pool_bytes) return nullptr;
    float* p = (float*)((uint8_t*)m->cs_pool + m->cs_used);
    m->cs_used += bytes;
    return p;
}

// Defer out_q[c] (+)= column sums of partial [rows][ncols], q < 3.
void cs_defer(gpt2* m, const float* partial, int rows, int ncols, int seg, float* o0, float* o1, float* o2) {
    ColsumJob j;
    j.in = partial;
    j.out[0] = o0;
    j.out[1] = o1;
    j.out[2] = o2;
    j.R = rows;
    j.ncols = ncols;
    j.seg = seg;
    j.accumulate = m->grad_accum;
    m->cs_jobs.push_back(j);
}

// ---- FP8 linear layers ----
// Per-tensor current scaling: each operand's codes use the scale of its own
// amax, taken just before the product (the forward writes x's codes in both
// layouts and keeps the transposed ones for the weight gradient; W's scale
// serves the backward's transposed codes of the same, unchanged weight).
// Activations and weights in e4m3, output gradients in e5m2.

// The FP8 linears as (in, out) sizes: qkv, fc, fcproj, head.
struct F8Lin {
    int mask_bit, in, out;
};
std::vector<F8Lin> f8_linears(const gpt2_config* c, int mask) {
    const int C = c->n_embd;
    std::vector<F8Lin> v;
    if (mask & GPT2_FP8_QKV) v.push_back({GPT2_FP8_QKV, C, 3 * C});
    if (mask & GPT2_FP8_MLP) {
        v.push_back({GPT2_FP8_MLP, C, 4 * C});
        v.push_back({GPT2_FP8_MLP, 4 * C, C});
    }
    if (mask & GPT2_FP8_HEAD) v.push_back({GPT2_FP8_HEAD, C, c->vocab_padded});
    return v;
}

// The FP8 linear in slot 3l + k (k: F8_QKV, F8_FC, F8_FCPROJ) or 3L (the head):
// whether mask selects it, and its input width.
inline bool f8_slot_on(const gpt2_config* c, int mask, int slot, int* in) {
    const int C = c->n_embd;
    if (slot == 3 * c->n_layer) {
        *in = C;
        return mask & GPT2_FP8_HEAD;
    }
    const int k = slot % 3;
    *in = k == 2 ? 4 * C : C;
    return mask & (k == 0 ? GPT2_FP8_QKV : GPT2_FP8_MLP);
}

// Carve the FP8 workspace (m == nullptr: the size only).
size_t fp8_plan(const gpt2_config* c, int mask, gpt2* m, uint8_t* w) {
    const size_t BT = (size_t)c->max_B * c->max_T;
    size_t max_in = 0, max_out = 0, max_w = 0, scr = 0;
    for (const F8Lin& f : f8_linears(c, mask)) {
        max_in = std::max(max_in, (size_t)f.in);
        max_out = std::max(max_out, (size_t)f.out);
        max_w = std::max(max_w, (size_t)f.in * f.out);
        scr = std::max(scr, matmul_f8_scratch(f.out, f.in, (int)BT, 1, 1));
    }
    size_t off = 0;
    auto take = [&](size_t bytes) {
        off = align_up(off, WS_ALIGN);
        const size_t r = off;
        off += bytes;
        return r;
    };
    const size_t o_x = take(BT * max_in), o_w = take(max_w), o_wT = take(max_w);
    const int slots = 3 * c->n_layer + 1;
    std::vector<size_t> o_xT(slots, 0);
    for (int sl = 0; sl < slots; sl++) {
        int in = 0;
        if (f8_slot_on(c, mask, sl, &in)) o_xT[sl] = take(BT * in);
    }
    const size_t o_dy = take(BT * max_out), o_dyT = take(BT * max_out);
    const size_t o_sc = take((size_t)(3 * c->n_layer + 1) * 8 * 4), o_part = take(fp8_quantize_scratch());
    const size_t o_amax = take((size_t)(3 * c->n_layer + 1) * 2 * 4);
    const size_t o_scr = take(std::max(scr, (size_t)256));
    if (m) {
        m->f8_x = w + o_x;
        m->f8_xT.assign(slots, nullptr);
        for (int sl = 0; sl < slots; sl++) {
            int in = 0;
            if (f8_slot_on(c, mask, sl, &in)) m->f8_xT[sl] = w + o_xT[sl];
        }
        m->f8_w = w + o_w;
        m->f8_wT = w + o_wT;
        m->f8_dy = w + o_dy;
        m->f8_dyT = w + o_dyT;
        m->f8_scales = (float*)(w + o_sc);
        m->f8_amax = (unsigned*)(w + o_amax);
        m->f8_partial = (float*)(w + o_part);
        m->f8_scratch = w + o_scr;
        m->f8_scratch_bytes = std::max(scr, (size_t)256);
    }
    return align_up(off, WS_ALIGN);
}

enum { F8_QKV = 0, F8_FC = 1, F8_FCPROJ = 2 };
inline float* f8_sc(gpt2* m, int slot) { return m->f8_scales + (size_t)slot * 8; }
// The amax word of slot's input x (which = 0) or output gradient dy (which = 1),
// or null when that linear is not FP8 (what the producing kernel is given).
inline unsigned* f8_am(gpt2* m, bool on, int slot, int which) {
    return on ? m->f8_amax + (size_t)slot * 2 + which : nullptr;
}

// y = x W^T + b with FP8 operands (y2: the GELU form, y = gelu'(u), y2 = gelu(u)).
// x's amax comes from the kernel that wrote x (f8_am(slot, 0)); y2 passes the
// amax of gelu(u) on to the next FP8 linear (y2_amax).
int f8_linear_fwd(gpt2* m, int slot, void* y, void* y2, const void* x, int wi, int bi, int BT, int in, int out,
                  unsigned* y2_amax = nullptr) {
    float* sc = f8_sc(m, slot);
    const bf16* xb = (const bf16*)x;
    const bf16* wb = (const bf16*)P(m, wi);
    {
        Op op(m, GPT2_K_FP8_QUANT);
        int n = 0, r;
        const int64_t nx = (int64_t)BT * in, nw = (int64_t)out * in;
        // x's codes in both layouts, under the scale of the amax its producer
        // took: rows for this product, transposed (kept until the backward)
        // for the weight gradient
        if ((r = launch_quantize_fp8_t(m->f8_xT[slot], m->f8_x, sc, xb, BT, in, FP8_E4M3, m->stream,
                                       f8_am(m, true, slot, 0))) < 0)
            return r;
        n += r;
        if ((r = launch_fp8_amax_scale(sc + 2, wb, nw, FP8_E4M3, m->f8_partial, m->stream)) < 0) return r;
        n += r;
        if ((r = launch_quantize_fp8_rows(m->f8_w, sc + 2, wb, nw, FP8_E4M3, m->stream)) < 0) return r;
        TRY(op.done(n + r, 4.0 * (double)nx + 5.0 * (double)nw));
    }
    const F8Args f8 = {FP8_E4M3, FP8_E4M3, sc + 1, sc + 3};
    const void* bias = bi >= 0 ? P(m, bi) : nullptr;
    Op op(m, GPT2_K_MATMUL);
    const double flops = 2.0 * BT * out * in;
    if (y2)
        return op.done(launch_matmul_gelu_f8(y, y2, m->f8_x, m->f8_w, f8, bias, BT, out, in, m->status, m->stream,
                                             y2_amax),
                       flops);
    return op.done(launch_matmul_f8(y, 0, m->f8_x, m->f8_w, f8, bias, BT, out, in, nullptr, m->status, m->stream), flops);
}

// dx = dy W and dW (+)= dy^T x with FP8 operands (dy in e5m2, its codes in
// both layouts; W transposed under its forward scale; x's transposed codes
// as the forward wrote them); the bias
// gradient from dy as stored (bf16), deferred. aux: dx is the gradient
// through the GELU, bf16(dy W) * aux, with its column sums to colsum.
// dy's amax comes from the kernel that wrote dy (f8_am(slot, 1)), or, with
// dy_pass, from a pass of its own over dy (the QKV projection's: taking it in
// the attention backward's accumulator stores measured no cheaper); with aux,
// dx_amax takes the amax of the gradient through the GELU for the next FP8
// linear down.
int f8_linear_bwd(gpt2* m, int slot, void* dx, const void* dy, const void* x, int wi, int bi, int BT, int in,
                  int out, const void* aux, float* colsum, unsigned* dx_amax = nullptr, bool dy_pass = false) {
    float* sc = f8_sc(m, slot);
    const bf16* dyb = (const bf16*)dy;
    {
        Op op(m, GPT2_K_FP8_QUANT);
        int n = 0, r;
        const int64_t ny = (int64_t)BT * out;
        // dy's codes in both layouts under the scale of its amax
        if (dy_pass && (r = launch_fp8_amax_scale(sc + 4, dyb, ny, FP8_E5M2, m->f8_partial, m->stream)) < 0) return r;
        n += dy_pass ? r : 0;
        if ((r = launch_quantize_fp8_t(m->f8_dyT, m->f8_dy, sc + 4, dyb, BT, out, FP8_E5M2, m->stream,
                                       dy_pass ? nullptr : f8_am(m, true, slot, 1))) < 0)
            return r;
        n += r;
        if ((r = launch_quantize_fp8_t(m->f8_wT, nullptr, sc + 2, (const bf16*)P(m, wi), out, in, FP8_E4M3,
                                       m->stream)) < 0)
            return r;
        TRY(op.done(n + r, (dy_pass ? 6.0 : 4.0) * ny + 3.0 * (double)out * in));
        (void)x;  // its transposed codes were written by the forward
    }
    const double flops = 2.0 * BT * in * out;
    {
        const F8Args f8 = {FP8_E5M2, FP8_E4M3, sc + 5, sc + 3};
        Op op(m, GPT2_K_MATMUL);
        const int r = aux ? launch_matmul_gelu_backward_f8(dx, m->f8_dy, m->f8_wT, f8, aux, BT, in, out, m->status,
                                                           m->stream, colsum, dx_amax)
                          : launch_matmul_f8(dx, 0, m->f8_dy, m->f8_wT, f8, nullptr, BT, in, out, nullptr, m->status,
                                             m->stream);
        TRY(op.done(r, flops));
    }
    {
        const F8Args f8 = {FP8_E5M2, FP8_E4M3, sc + 5, sc + 1};
        Op op(m, GPT2_K_MATMUL);
        TRY(op.done(launch_matmul_f8(G(m, wi), 1, m->f8_dyT, m->f8_xT[slot], f8, nullptr, out, in, BT, m->f8_scratch,
                                     m->status, m->stream, m->grad_accum),
                    flops));
    }
    if (bi >= 0) {
        float* part = cs_take(m, (int)((BT + 127) / 128), out);
        if (!part) return GPT2_ERR_WORKSPACE;
        Op op(m, GPT2_K_BIAS_BWD);
        int rows = 0;
        TRY(op.done(launch_bias_partials(m->dtype, part, dy, BT, out, m->stream, &rows), (double)BT * out * m->act));
        cs_defer(m, part, rows, out, out, G(m, bi), nullptr, nullptr);
    }
    return GPT2_OK;
}

int op_matmul(gpt2* m, void* D, int d_fp32, const void* A, int a_mn, const void* B, int b_mn, const void* bias, int M,
              int N, int K, int accumulate = 0) {
    Op op(m, GPT2_K_MATMUL);
    return op.done(launch_matmul(m->dtype, D, d_fp32, A, a_mn, B, b_mn, bias, M, N, K, m->scratch, m->status,
                                 m->stream, accumulate),
                   2.0 * M * N * K);
}

// y = x W^T + b for x [BT, in], W [out, in].
int linear_fwd(gpt2* m, void* y, const void* x, int wi, int bi, int BT, int in, int out) {
    return op_matmul(m, y, 0, x, 0, P(m, wi), 0, bi >= 0 ? P(m, bi) : nullptr, BT, out, in);
}

// dx = dy W, dW = dy^T x, db = column sums of dy (partials now, reduced at
// the end of the backward).
int linear_bwd(gpt2* m, void* dx, const void* dy, const void* x, int wi, int bi, int BT, int in, int out) {
    TRY(op_matmul(m, dx, 0, dy, 0, P(m, wi), 1, nullptr, BT, in, out));
    TRY(op_matmul(m, G(m, wi), 1, dy, 1, x, 1, nullptr, out, in, BT, m->grad_accum));
    if (bi >= 0) {
        float* part = cs_take(m, (int)((BT + 127) / 128), out);
        if (!part) return GPT2_ERR_WORKSPACE;
        Op op(m, GPT2_K_BIAS_BWD);
        int rows = 0;
        TRY(op.done(launch_bias_partials(m->dtype, part, dy, BT, out, m->stream, &rows), (double)BT * out * m->act));
        cs_defer(m, part, rows, out, out, G(m, bi), nullptr, nullptr);
    }
    return GPT2_OK;
}

int ln_fwd(gpt2* m, void* y, float* mean, float* rstd, const void* x, int gi, int BT, unsigned* amax = nullptr) {
    Op op(m, GPT2_K_LAYERNORM_FWD);
    return op.done(launch_layernorm_forward(m->dtype, y, mean, rstd, x, P(m, gi), P(m, gi + 1), BT, m->C, m->stream,
                                            amax),
                   (double)BT * (2.0 * m->C * m->act + 8));
}

// Residual join then LayerNorm: xsum = x + r; y = LN(xsum) with the norm at gi.
// amax (or null): the largest |y| is merged into it (an FP8 linear's input).
int res_ln_fwd(gpt2* m, void* y, float* mean, float* rstd, void* xsum, const void* x, const void* r, int gi, int BT,
               unsigned* amax = nullptr) {
    Op op(m, GPT2_K_LAYERNORM_FWD);
    return op.done(launch_residual_layernorm_forward(m->dtype, y, mean, rstd, xsum, x, r, P(m, gi), P(m, gi + 1), BT,
                                                     m->C, m->stream, amax),
                   (double)BT * (4.0 * m->C * m->act + 8));
}

// LayerNorm backward into the residual gradient: dres (+)= dx; the column sums
// of the new dres go to the bias gradient bi (when bi >= 0): the bias of the
// linear layer whose output joins the residual stream at this point.
int ln_bwd_res(gpt2* m, int accumulate, const void* dy, const void* x, int gi, const float* mean, const float* rstd,
               int bi, int BT, unsigned* amax = nullptr) {
    const int np = bi >= 0 ? 3 : 2;
    float* part = (float*)cs_take(m, 1, (int)(layernorm_backward_scratch(BT, m->C) / 4));
    if (!part) return GPT2_ERR_WORKSPACE;
    Op op(m, GPT2_K_LAYERNORM_BWD);
    int rows = 0;
    TRY(op.done(launch_layernorm_backward_residual_rows(m->dtype, m->dres, accumulate, part, np, dy, x, P(m, gi),
                                                        mean, rstd, BT, m->C, m->stream, &rows, amax),
                (double)BT * ((3.0 + accumulate) * m->C * m->act + 8)));
    cs_defer(m, part, rows, np * m->C, m->C, G(m, gi), G(m, gi + 1), bi >= 0 ? G(m, bi) : nullptr);
    return GPT2_OK;
}

double attn_fwd_flops(int B, int T, int C) { return 2.0 * 2.0 * B * C * (double)T * (T + 1) / 2.0; }

int forward_impl(gpt2* m, const int32_t* targets, int B, int T) {
    const int BT = B * T, C = m->C, L = m->L;
    if (m->fp8 && BT % 16) return GPT2_ERR_ARG;  // the FP8 weight gradients contract over B*T in 16-byte rows
    const bool f8_qkv = m->fp8 & GPT2_FP8_QKV, f8_mlp = m->fp8 & GPT2_FP8_MLP, f8_head = m->fp8 & GPT2_FP8_HEAD;
    // the FP8 operands' amax words, filled by the kernels that write the operands
    if (m->fp8 && cudaMemsetAsync(m->f8_amax, 0, (size_t)(3 * L + 1) * 2 * 4, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    {
        Op op(m, GPT2_K_ENCODER_FWD);
        TRY(op.done(launch_encoder_forward(m->dtype, m->layers[0].x, m->tokens, P(m, T_WTE), P(m, T_WPE), B, T, C,
                                           m->V, m->status, m->stream),
                    (double)BT * (3.0 * C * m->act + 4)));
    }
    // each residual join is fused with the LayerNorm that reads its result
    TRY(ln_fwd(m, m->layers[0].ln1, m->layers[0].mean1, m->layers[0].rstd1, m->layers[0].x, tidx(0, 0), BT,
               f8_am(m, f8_qkv, F8_QKV, 0)));
    for (int l = 0; l < L; l++) {
        LayerBufs& b = m->layers[l];
        if (f8_qkv) TRY(f8_linear_fwd(m, 3 * l + F8_QKV, b.qkv, nullptr, b.ln1, tidx(l, 2), tidx(l, 3), BT, C, 3 * C));
        else TRY(linear_fwd(m, b.qkv, b.ln1, tidx(l, 2), tidx(l, 3), BT, C, 3 * C));
        {
            Op op(m, GPT2_K_ATTENTION_FWD);
            TRY(op.done(launch_attention_forward(m->dtype, b.atty, b.lse, b.qkv, B, T, C, m->H, m->status, m->stream),
                        attn_fwd_flops(B, T, C)));
        }
        TRY(linear_fwd(m, m->fwd_tmp, b.atty, tidx(l, 4), tidx(l, 5), BT, C, C));
        TRY(res_ln_fwd(m, b.ln2, b.mean2, b.rstd2, b.x1, b.x, m->fwd_tmp, tidx(l, 6), BT,
                       f8_am(m, f8_mlp, 3 * l + F8_FC, 0)));
        if (f8_mlp) {
            TRY(f8_linear_fwd(m, 3 * l + F8_FC, b.fch, b.fchg, b.ln2, tidx(l, 8), tidx(l, 9), BT, C, 4 * C,
                              f8_am(m, true, 3 * l + F8_FCPROJ, 0)));
        } else if (m->dtype == GPT2_MODE_BF16) {
            // the GELU runs in the epilogue of its linear, which keeps gelu'
            // (in fch) for the backward instead of the GELU input
            Op op(m, GPT2_K_MATMUL);
            TRY(op.done(launch_matmul_gelu(b.fch, b.fchg, b.ln2, P(m, tidx(l, 8)), P(m, tidx(l, 9)), BT, 4 * C, C,
                                           m->status, m->stream),
                        2.0 * BT * 4 * C * C));
        } else {
            TRY(linear_fwd(m, b.fch, b.ln2, tidx(l, 8), tidx(l, 9), BT, C, 4 * C));
            Op op(m, GPT2_K_GELU_FWD);
            TRY(op.done(launch_gelu_forward(m->dtype, b.fchg, b.fch, (int64_t)BT * 4 * C, m->stream),
                        2.0 * BT * 4 * C * m->act));
        }
        if (f8_mlp)
            TRY(f8_linear_fwd(m, 3 * l + F8_FCPROJ, m->fwd_tmp, nullptr, b.fchg, tidx(l, 10), tidx(l, 11), BT, 4 * C, C));
        else TRY(linear_fwd(m, m->fwd_tmp, b.fchg, tidx(l, 10), tidx(l, 11), BT, 4 * C, C));
        if (l + 1 < L) {
            LayerBufs& n = m->layers[l + 1];
            TRY(res_ln_fwd(m, n.ln1, n.mean1, n.rstd1, n.x, b.x1, m->fwd_tmp, tidx(l + 1, 0), BT,
                           f8_am(m, f8_qkv, 3 * (l + 1) + F8_QKV, 0)));
        } else {
            TRY(res_ln_fwd(m, m->lnf, m->meanf, m->rstdf, m->xL, b.x1, m->fwd_tmp, tlnf(L, 0), BT,
                           f8_am(m, f8_head, 3 * L, 0)));
        }
    }
    if (f8_head) TRY(f8_linear_fwd(m, 3 * L, m->logits, nullptr, m->lnf, T_WTE, -1, BT, C, m->Vp));
    else TRY(op_matmul(m, m->logits, 0, m->lnf, 0, P(m, T_WTE), 0, nullptr, BT, m->Vp, C));
    if (targets) {
        {
            Op op(m, GPT2_K_CLASSIFIER);
            TRY(op.done(launch_classifier(m->dtype, m->logits, m->losses, targets, BT, m->V, m->Vp, 1.0f / BT,
                                          m->status, m->stream, f8_am(m, f8_head, 3 * L, 1)),
                        (double)BT * (2.0 * m->Vp * m->act + 8)));
        }
        Op op(m, GPT2_K_LOSS_MEAN);
        TRY(op.done(launch_mean_loss(m->loss_dev, m->losses, BT, m->stream), BT * 4.0));
    }
    return GPT2_OK;
}

int backward_impl(gpt2* m) {
    const int B = m->B, T = m->T, BT = B * T, C = m->C, L = m->L;
    m->cs_used = 0;
    m->cs_jobs.clear();
    const bool f8_qkv = m->fp8 & GPT2_FP8_QKV, f8_mlp = m->fp8 & GPT2_FP8_MLP, f8_head = m->fp8 & GPT2_FP8_HEAD;
    // LM head (tied with wte): dlnf = dlogits wte; dwte = dlogits^T lnf (overwrites dwte)
    if (f8_head) {
        TRY(f8_linear_bwd(m, 3 * L, m->dtmp, m->logits, m->lnf, T_WTE, -1, BT, C, m->Vp, nullptr, nullptr));
    } else {
        TRY(op_matmul(m, m->dtmp, 0, m->logits, 0, P(m, T_WTE), 1, nullptr, BT, C, m->Vp));
        TRY(op_matmul(m, G(m, T_WTE), 1, m->logits, 1, m->lnf, 1, nullptr, m->Vp, C, BT, m->grad_accum));
    }
    // the LayerNorm backwards write the residual gradient dres and, on the
    // way, the bias gradient of the projection whose output joins there
    TRY(ln_bwd_res(m, 0, m->dtmp, m->xL, tlnf(L, 0), m->meanf, m->rstdf, tidx(L - 1, 11), BT,
                   f8_am(m, f8_mlp, 3 * (L - 1) + F8_FCPROJ, 1)));
    for (int l = L - 1; l >= 0; l--) {
        LayerBufs& b = m->layers[l];
        // MLP branch
        if (f8_mlp) {
            // the projection's input gradient through the GELU, with the first
            // linear's bias-gradient partials, and its weight gradient
            const int rows = matmul_gelu_backward_colsum_rows(BT);
            float* part = cs_take(m, rows, 4 * C);
            if (!part) return GPT2_ERR_WORKSPACE;
            TRY(f8_linear_bwd(m, 3 * l + F8_FCPROJ, m->dbig, m->dres, b.fchg, tidx(l, 10), -1, BT, 4 * C, C, b.fch,
                              part, f8_am(m, true, 3 * l + F8_FC, 1)));
            cs_defer(m, part, rows, 4 * C, 4 * C, G(m, tidx(l, 9)), nullptr, nullptr);
        } else if (m->dtype == GPT2_MODE_BF16) {
            // dW of the MLP projection, then its input gradient times the
            // GELU's derivative (kept in fch by the forward), in the GEMM epilogue
            // (and the column sums of that gradient per 32-row slice: the
            // partials of the first linear's bias gradient)
            TRY(op_matmul(m, G(m, tidx(l, 10)), 1, m->dres, 1, b.fchg, 1, nullptr, C, 4 * C, BT, m->grad_accum));
            const int rows = matmul_gelu_backward_colsum_rows(BT);
            float* part = cs_take(m, rows, 4 * C);
            if (!part) return GPT2_ERR_WORKSPACE;
            Op op(m, GPT2_K_MATMUL);
            TRY(op.done(launch_matmul_gelu_backward(m->dbig, m->dres, P(m, tidx(l, 10)), b.fch, BT, 4 * C, C,
                                                    m->status, m->stream, part),
                        2.0 * BT * 4 * C * C));
            cs_defer(m, part, rows, 4 * C, 4 * C, G(m, tidx(l, 9)), nullptr, nullptr);
        } else {
            TRY(linear_bwd(m, m->dbig, m->dres, b.fchg, tidx(l, 10), -1, BT, 4 * C, C));
            Op op(m, GPT2_K_GELU_BWD);
            TRY(op.done(launch_gelu_backward(m->dtype, m->dbig, b.fch, m->dbig, (int64_t)BT * 4 * C, m->stream),
                        3.0 * BT * 4 * C * m->act));
        }
        if (f8_mlp) TRY(f8_linear_bwd(m, 3 * l + F8_FC, m->dtmp, m->dbig, b.ln2, tidx(l, 8), -1, BT, C, 4 * C, nullptr, nullptr));
        else TRY(linear_bwd(m, m->dtmp, m->dbig, b.ln2, tidx(l, 8), m->dtype == GPT2_MODE_BF16 ? -1 : tidx(l, 9), BT, C,
                            4 * C));
        TRY(ln_bwd_res(m, 1, m->dtmp, b.x1, tidx(l, 6), b.mean2, b.rstd2, tidx(l, 5), BT));
        // attention branch
        TRY(linear_bwd(m, m->dtmp, m->dres, b.atty, tidx(l, 4), -1, BT, C, C));
        {
            Op op(m, GPT2_K_ATTENTION_BWD);
            TRY(op.done(launch_attention_backward(m->dtype, m->dqkv, m->dtmp, b.qkv, b.atty, b.lse, B, T, C, m->H,
                                                  m->scratch, m->status, m->stream),
                        2.5 * attn_fwd_flops(B, T, C)));
        }
        if (f8_qkv)
            TRY(f8_linear_bwd(m, 3 * l + F8_QKV, m->dtmp, m->dqkv, b.ln1, tidx(l, 2), tidx(l, 3), BT, C, 3 * C, nullptr,
                              nullptr, nullptr, true));
        else TRY(linear_bwd(m, m->dtmp, m->dqkv, b.ln1, tidx(l, 2), tidx(l, 3), BT, C, 3 * C));
        TRY(ln_bwd_res(m, 1, m->dtmp, b.x, tidx(l, 0), b.mean1, b.rstd1, l > 0 ? tidx(l - 1, 11) : -1, BT,
                       l > 0 ? f8_am(m, f8_mlp, 3 * (l - 1) + F8_FCPROJ, 1) : nullptr));
    }
    {
        // every deferred column sum of this backward, in ceil(jobs / 32) launches
        double bytes = 0;
        for (const ColsumJob& j : m->cs_jobs) bytes += (double)j.R * j.ncols * 4 + (double)j.ncols * 4;
        Op op(m, GPT2_K_GRAD_COLSUM);
        TRY(op.done(launch_colsum_jobs(m->cs_jobs.data(), (int)m->cs_jobs.size(), m->stream), bytes));
    }
    if (T < m->maxT && !m->grad_accum &&
        cudaMemsetAsync(G(m, T_WPE) + (size_t)T * C, 0, (size_t)(m->maxT - T) * C * 4, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;  // positions >= T get a zero gradient (kept as they are when accumulating)
    Op op(m, GPT2_K_ENCODER_BWD);
    return op.done(launch_encoder_backward(m->dtype, G(m, T_WTE), G(m, T_WPE), m->dres, m->tokens, B, T, C,
                                           m->scratch, m->stream, m->grad_accum),
                   (double)BT * (C * m->act + 4) * 2 + (double)BT * C * 8);
}

int cuda_ok(cudaError_t e) { return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA; }

int refresh_compute_copy(gpt2* m, int64_t off, int64_t n) {
    if (m->mode != GPT2_MODE_BF16 || n == 0) return GPT2_OK;
    f32_to_bf16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, m->stream>>>((bf16*)m->params + off, m->master + off, n);
    m->launches++;
    return cuda_ok(cudaGetLastError());
}

int read_status(gpt2* m) {
    int st = 0;
    if (cudaMemcpyAsync(&st, m->status, sizeof(int), cudaMemcpyDeviceToHost, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    if (cudaStreamSynchronize(m->stream) != cudaSuccess) return GPT2_ERR_CUDA;
    if (st & GPT2_FLAG_TIMEOUT) return GPT2_ERR_TIMEOUT;
    if (st & (GPT2_FLAG_TOKEN_RANGE | GPT2_FLAG_TARGET_RANGE)) return GPT2_ERR_TOKEN_RANGE;
    return GPT2_OK;
}

}  // namespace

// =============================================================== C ABI

extern "C" {

int gpt2_workspace_bytes(const gpt2_config* cfg, size_t* bytes_out) {
    if (!config_ok(cfg) || !bytes_out) return GPT2_ERR_ARG;
    *bytes_out = plan(cfg, nullptr);
    return GPT2_OK;
}

int gpt2_init(gpt2_t** out, const gpt2_config* cfg, uint64_t seed, void* d_workspace, size_t workspace_bytes,
              void* cuda_stream) {
    if (!out || !config_ok(cfg) || !d_workspace) return GPT2_ERR_ARG;
    *out = nullptr;
    if (((uintptr_t)d_workspace) % WS_ALIGN) return GPT2_ERR_WORKSPACE;
    const size_t need = plan(cfg, nullptr);
    if (workspace_bytes < need) return GPT2_ERR_WORKSPACE;
    gpt2* m = new gpt2();
    m->cfg = *cfg;
    m->L = cfg->n_layer; m->C = cfg->n_embd; m->H = cfg->n_head; m->V = cfg->vocab; m->Vp = cfg->vocab_padded;
    m->maxT = cfg->max_T; m->maxB = cfg->max_B; m->mode = cfg->mode; m->dtype = cfg->mode;
    m->act = cfg->mode == GPT2_MODE_BF16 ? 2 : 4;
    m->stream = (cudaStream_t)cuda_stream;
    m->ws = (uint8_t*)d_workspace;
    m->ws_bytes = workspace_bytes;
    int64_t np = 0;
    m->tensors = make_specs(cfg, &np);
    plan(cfg, m);
    m->B = m->T = 0;
    m->state = 0;
    m->launches = 0;
    for (int f = 0; f < GPT2_K_COUNT; f++) {
        m->fam_calls[f] = m->fam_launches[f] = 0;
        m->fam_work[f] = m->fam_ms[f] = 0;
    }
    m->timing = false;
    m->grad_accum = 0;
    // weight decay on the 2-D tensors (wte, wpe, the weight matrices), not on
    // biases and LayerNorm parameters; every tensor starts on a 64-element boundary
    std::vector<uint32_t> bits(((size_t)m->np / 64 + 1 + 31) / 32, 0u);
    for (const auto& t : m->tensors) {
        if (t.cols <= 1) continue;
        const int64_t c0 = t.offset / 64, c1 = (t.offset + t.rows * t.cols + 63) / 64;
        for (int64_t c = c0; c < c1; c++) bits[(size_t)c / 32] |= 1u << (c % 32);
    }
    std::vector<float> host((size_t)m->np, 0.f);
    init_host(cfg, seed, m->tensors, host.data());
    int r = GPT2_OK;
    if (cudaMemsetAsync(m->status, 0, 256, m->stream) != cudaSuccess ||
        cudaMemcpyAsync(m->master, host.data(), (size_t)m->np * 4, cudaMemcpyHostToDevice, m->stream) != cudaSuccess ||
        cudaMemsetAsync(m->grads, 0, (size_t)m->np * 4, m->stream) != cudaSuccess ||
        cudaMemsetAsync(m->adam_m, 0, (size_t)m->np * 4, m->stream) != cudaSuccess ||
        cudaMemsetAsync(m->adam_v, 0, (size_t)m->np * 4, m->stream) != cudaSuccess ||
        cudaMemcpyAsync(m->decay_bits, bits.data(), bits.size() * 4, cudaMemcpyHostToDevice, m->stream) != cudaSuccess)
        r = GPT2_ERR_CUDA;
    if (r == GPT2_OK) r = refresh_compute_copy(m, 0, m->np);
    if (r == GPT2_OK) r = cuda_ok(cudaStreamSynchronize(m->stream));
    if (r != GPT2_OK) {
        delete m;
        return r;
    }
    *out = m;
    return GPT2_OK;
}

int gpt2_forward(gpt2_t* m, const int32_t* d_tokens, const int32_t* d_targets, int B, int T, float* loss_out) {
    if (!m || !d_tokens || B < 1 || T < 1 || B > m->maxB || T > m->maxT) return GPT2_ERR_ARG;
    if (d_targets && !loss_out) return GPT2_ERR_ARG;
    m->state = 0;
    m->B = B;
    m->T = T;
    if (cudaMemsetAsync(m->status, 0, sizeof(int), m->stream) != cudaSuccess ||
        cudaMemcpyAsync(m->tokens, d_tokens, (size_t)B * T * 4, cudaMemcpyDeviceToDevice, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    TRY(forward_impl(m, d_targets, B, T));
    if (!d_targets) return GPT2_OK;
    float loss = 0.f;
    if (cudaMemcpyAsync(&loss, m->loss_dev, sizeof(float), cudaMemcpyDeviceToHost, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    TRY(read_status(m));  // synchronises the stream
    *loss_out = loss;
    if (!std::isfinite(loss)) return GPT2_ERR_NONFINITE;
    m->state = 1;
    return GPT2_OK;
}

int gpt2_backward(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    if (m->state != 1) return GPT2_ERR_STATE;
    TRY(backward_impl(m));
    m->state = 2;
    return GPT2_OK;
}

int gpt2_adamw_step(gpt2_t* m, float lr, float beta1, float beta2, float eps, float weight_decay, int t) {
    if (!m) return GPT2_ERR_ARG;
    if (t < 1 || !(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) || !(eps >= 0.f) ||
        !std::isfinite(lr) || !std::isfinite(weight_decay))
        return GPT2_ERR_ARG;
    if (m->state != 2) return GPT2_ERR_STATE;
    Op op(m, GPT2_K_ADAMW);
    TRY(op.done(launch_adamw(m->master, m->mode == GPT2_MODE_BF16 ? m->params : nullptr, m->grads, m->adam_m,
                             m->adam_v, m->np, lr, beta1, beta2, eps, weight_decay, t, m->stream),
                (double)m->np * (m->mode == GPT2_MODE_BF16 ? 30.0 : 28.0)));
    m->state = 3;
    return GPT2_OK;
}

int gpt2_fp8_workspace_bytes(const gpt2_config* cfg, int mask, size_t* bytes_out) {
    if (!config_ok(cfg) || !bytes_out || mask < 0 || mask > GPT2_FP8_ALL) return GPT2_ERR_ARG;
    if (mask && cfg->mode != GPT2_MODE_BF16) return GPT2_ERR_ARG;
    *bytes_out = mask ? fp8_plan(cfg, mask, nullptr, nullptr) : 0;
    return GPT2_OK;
}

int gpt2_set_fp8(gpt2_t* m, int mask, void* d_workspace, size_t workspace_bytes) {
    if (!m || mask < 0 || mask > GPT2_FP8_ALL) return GPT2_ERR_ARG;
    if (mask && m->mode != GPT2_MODE_BF16) return GPT2_ERR_ARG;
    if (mask) {
        if (!d_workspace || ((uintptr_t)d_workspace) % WS_ALIGN) return GPT2_ERR_WORKSPACE;
        if (workspace_bytes < fp8_plan(&m->cfg, mask, nullptr, nullptr)) return GPT2_ERR_WORKSPACE;
        fp8_plan(&m->cfg, mask, m, (uint8_t*)d_workspace);
    }
    m->fp8 = mask;
    m->state = 0;  // a forward with the new layers comes first
    return GPT2_OK;
}

int gpt2_set_grad_accumulation(gpt2_t* m, int accumulate) {
    if (!m || (accumulate != 0 && accumulate != 1)) return GPT2_ERR_ARG;
    m->grad_accum = accumulate;
    return GPT2_OK;
}

int gpt2_zero_grad(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    return cuda_ok(cudaMemsetAsync(m->grads, 0, (size_t)m->np * 4, m->stream));
}

int gpt2_grad_norm(gpt2_t* m, float* norm_out) {
    if (!m) return GPT2_ERR_ARG;
    if (launch_grad_norm(m->gnorm, m->gnorm_partial, m->grads, m->np, m->stream) < 0) return GPT2_ERR_CUDA;
    m->launches += 2;
    if (cudaGetLastError() != cudaSuccess) return GPT2_ERR_CUDA;
    if (!norm_out) return GPT2_OK;
    float v = 0.f;
    if (cudaMemcpyAsync(&v, m->gnorm, sizeof(float), cudaMemcpyDeviceToHost, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    TRY(cuda_ok(cudaStreamSynchronize(m->stream)));
    *norm_out = v;
    return GPT2_OK;
}

int gpt2_adamw_step_ex(gpt2_t* m, const gpt2_adamw_config* c) {
    if (!m || !c) return GPT2_ERR_ARG;
    if (c->t < 1 || !(c->beta1 >= 0.f && c->beta1 < 1.f) || !(c->beta2 >= 0.f && c->beta2 < 1.f) || !(c->eps >= 0.f) ||
        !std::isfinite(c->lr) || !std::isfinite(c->weight_decay) || !(c->grad_scale > 0.f) ||
        !std::isfinite(c->grad_scale) || !(c->max_grad_norm >= 0.f) || (c->decay_mask != 0 && c->decay_mask != 1))
        return GPT2_ERR_ARG;
    if (m->state != 2) return GPT2_ERR_STATE;
    if (c->max_grad_norm > 0.f) {
        // the norm stays on the device: the clip factor is formed inside AdamW
        if (launch_grad_norm(m->gnorm, m->gnorm_partial, m->grads, m->np, m->stream) < 0) return GPT2_ERR_CUDA;
        m->launches += 2;
    }
    Op op(m, GPT2_K_ADAMW);
    TRY(op.done(launch_adamw(m->master, m->mode == GPT2_MODE_BF16 ? m->params : nullptr, m->grads, m->adam_m,
                             m->adam_v, m->np, c->lr, c->beta1, c->beta2, c->eps, c->weight_decay, c->t, m->stream,
                             c->grad_scale, c->max_grad_norm > 0.f ? m->gnorm : nullptr, c->max_grad_norm,
                             c->decay_mask ? m->decay_bits : nullptr),
                (double)m->np * (m->mode == GPT2_MODE_BF16 ? 30.0 : 28.0)));
    m->state = 3;
    return GPT2_OK;
}

int64_t gpt2_flat_params(const gpt2_t* m) { return m ? m->np : GPT2_ERR_ARG; }

namespace {

// Everything of one training step after its inputs are in place: forward to
// the mean loss, backward, the device-side clip norm when asked, and AdamW
// with its values read from hp_dev.
int step_body(gpt2* m, int B, int T, const gpt2_adamw_config* c) {
    TRY(forward_impl(m, m->targets, B, T));
    TRY(backward_impl(m));
    if (c->max_grad_norm > 0.f) {
        if (launch_grad_norm(m->gnorm, m->gnorm_partial, m->grads, m->np, m->stream) < 0) return GPT2_ERR_CUDA;
        m->launches += 2;
    }
    Op op(m, GPT2_K_ADAMW);
    return op.done(launch_adamw(m->master, m->mode == GPT2_MODE_BF16 ? m->params : nullptr, m->grads, m->adam_m,
                                m->adam_v, m->np, c->lr, c->beta1, c->beta2, c->eps, c->weight_decay, c->t,
                                m->stream, c->grad_scale, c->max_grad_norm > 0.f ? m->gnorm : nullptr,
                                c->max_grad_norm, c->decay_mask ? m->decay_bits : nullptr, m->hp_dev),
                   (double)m->np * (m->mode == GPT2_MODE_BF16 ? 30.0 : 28.0));
}

}  // namespace

namespace {

// gpt2_step with the token and target batches read from device memory
// (cudaMemcpyDeviceToDevice) or host memory (cudaMemcpyHostToDevice).
int step_impl(gpt2_t* m, const int32_t* d_tokens, const int32_t* d_targets, int B, int T, const gpt2_adamw_config* c,
              float* loss_out, cudaMemcpyKind kind);

}  // namespace

int gpt2_step(gpt2_t* m, const int32_t* d_tokens, const int32_t* d_targets, int B, int T, const gpt2_adamw_config* c,
              float* loss_out) {
    return step_impl(m, d_tokens, d_targets, B, T, c, loss_out, cudaMemcpyDeviceToDevice);
}

int gpt2_step_host(gpt2_t* m, const int32_t* h_tokens, const int32_t* h_targets, int B, int T,
                   const gpt2_adamw_config* c, float* loss_out) {
    return step_impl(m, h_tokens, h_targets, B, T, c, loss_out, cudaMemcpyHostToDevice);
}

namespace {

int step_impl(gpt2_t* m, const int32_t* d_tokens, const int32_t* d_targets, int B, int T, const gpt2_adamw_config* c,
              float* loss_out, cudaMemcpyKind kind) {
    if (!m || !d_tokens || !d_targets || !loss_out || !c || B < 1 || T < 1 || B > m->maxB || T > m->maxT)
        return GPT2_ERR_ARG;
    if (c->t < 1 || !(c->beta1 >= 0.f && c->beta1 < 1.f) || !(c->beta2 >= 0.f && c->beta2 < 1.f) || !(c->eps >= 0.f) ||
        !std::isfinite(c->lr) || !std::isfinite(c->weight_decay) || !(c->grad_scale > 0.f) ||
        !std::isfinite(c->grad_scale) || !(c->max_grad_norm >= 0.f) || (c->decay_mask != 0 && c->decay_mask != 1))
        return GPT2_ERR_ARG;
    m->state = 0;
    m->B = B;
    m->T = T;
    // the step's AdamW values, computed as launch_adamw computes its arguments
    const float hp[8] = {c->lr, c->beta1, c->beta2, c->eps, c->weight_decay,
                         (float)(1.0 / (1.0 - std::pow((double)c->beta1, (double)c->t))),
                         (float)(1.0 / (1.0 - std::pow((double)c->beta2, (double)c->t))), c->grad_scale};
    const size_t bt = (size_t)B * T * 4;
    if (cudaMemcpyAsync(m->hp_dev, hp, sizeof(hp), cudaMemcpyHostToDevice, m->stream) != cudaSuccess ||
        cudaMemsetAsync(m->status, 0, sizeof(int), m->stream) != cudaSuccess ||
        cudaMemcpyAsync(m->tokens, d_tokens, bt, kind, m->stream) != cudaSuccess ||
        cudaMemcpyAsync(m->targets, d_targets, bt, kind, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    const gpt2::StepKey key{B, T, m->grad_accum, c->max_grad_norm > 0.f ? 1 : 0, c->decay_mask, m->fp8,
                            c->max_grad_norm};
    if (!(key == m->step_key)) {
        if (m->step_exec) cudaGraphExecDestroy(m->step_exec);
        m->step_exec = nullptr;
        m->step_warm = false;
        m->step_key = key;
    }
    if (m->timing || !m->step_warm) {
        // eagerly: with per-op timing on, and the first time for these sizes
        // and options, so that every lazy setup of the kernels runs outside a capture
        TRY(step_body(m, B, T, c));
        m->step_warm = !m->timing;
    } else {
        if (!m->step_exec) {
            // capturing enqueues nothing: the per-family counters are put back after it
            const int64_t before = m->launches;
            int64_t calls[GPT2_K_COUNT], launches[GPT2_K_COUNT];
            double work[GPT2_K_COUNT];
            std::copy(m->fam_calls, m->fam_calls + GPT2_K_COUNT, calls);
            std::copy(m->fam_launches, m->fam_launches + GPT2_K_COUNT, launches);
            std::copy(m->fam_work, m->fam_work + GPT2_K_COUNT, work);
            cudaGraph_t graph = nullptr;
            // capture on a stream of the library's own (the legacy default
            // stream cannot be captured); the work is launched below on the
            // caller's stream, so capturing enqueues nothing anywhere
            if (!m->capture_stream && cudaStreamCreateWithFlags(&m->capture_stream, cudaStreamNonBlocking) != cudaSuccess)
                return GPT2_ERR_CUDA;
            const cudaStream_t user_stream = m->stream;
            if (cudaStreamBeginCapture(m->capture_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
                return GPT2_ERR_CUDA;
            m->stream = m->capture_stream;
            const int r = step_body(m, B, T, c);
            m->stream = user_stream;
            const cudaError_t e = cudaStreamEndCapture(m->capture_stream, &graph);
            if (r != GPT2_OK || e != cudaSuccess) {
                if (graph) cudaGraphDestroy(graph);
                return r != GPT2_OK ? r : GPT2_ERR_CUDA;
            }
            const cudaError_t ie = cudaGraphInstantiate(&m->step_exec, graph, 0);
            cudaGraphDestroy(graph);
            if (ie != cudaSuccess) {
                m->step_exec = nullptr;
                return GPT2_ERR_CUDA;
            }
            m->step_launches = m->launches - before;
            m->launches = before;
            std::copy(calls, calls + GPT2_K_COUNT, m->fam_calls);
            std::copy(launches, launches + GPT2_K_COUNT, m->fam_launches);
            std::copy(work, work + GPT2_K_COUNT, m->fam_work);
        }
        if (cudaGraphLaunch(m->step_exec, m->stream) != cudaSuccess) return GPT2_ERR_CUDA;
        m->launches += m->step_launches;
    }
    float loss = 0.f;
    if (cudaMemcpyAsync(&loss, m->loss_dev, sizeof(float), cudaMemcpyDeviceToHost, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    TRY(read_status(m));  // synchronises the stream
    *loss_out = loss;
    if (!std::isfinite(loss)) return GPT2_ERR_NONFINITE;
    m->state = 3;
    return GPT2_OK;
}

}  // namespace

int gpt2_grad_sumsq_range(gpt2_t* m, int64_t begin, int64_t count, float* out) {
    if (!m || !out || begin < 0 || count < 4 || count % 4 != 0 || begin % 4 != 0 || begin + count > m->np)
        return GPT2_ERR_ARG;
    if (launch_grad_norm(m->gnorm, m->gnorm_partial, m->grads + begin, count, m->stream, 0) < 0) return GPT2_ERR_CUDA;
    m->launches += 2;
    if (cudaGetLastError() != cudaSuccess) return GPT2_ERR_CUDA;
    float v = 0.f;
    if (cudaMemcpyAsync(&v, m->gnorm, sizeof(float), cudaMemcpyDeviceToHost, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    TRY(cuda_ok(cudaStreamSynchronize(m->stream)));
    *out = v;
    return GPT2_OK;
}

int gpt2_adamw_step_shard(gpt2_t* m, const gpt2_adamw_config* c, int64_t begin, int64_t count) {
    if (!m || !c) return GPT2_ERR_ARG;
    if (c->t < 1 || !(c->beta1 >= 0.f && c->beta1 < 1.f) || !(c->beta2 >= 0.f && c->beta2 < 1.f) || !(c->eps >= 0.f) ||
        !std::isfinite(c->lr) || !std::isfinite(c->weight_decay) || !(c->grad_scale > 0.f) ||
        !std::isfinite(c->grad_scale) || c->max_grad_norm != 0.f || (c->decay_mask != 0 && c->decay_mask != 1))
        return GPT2_ERR_ARG;
    // a shard starts on a 2048-element boundary (one 32-bit word of the
    // decay mask, one bit per 64 elements) and holds whole float4s
    if (begin < 0 || count < 4 || begin % 2048 != 0 || count % 4 != 0 || begin + count > m->np) return GPT2_ERR_ARG;
    if (m->state != 2 && m->state != 4) return GPT2_ERR_STATE;
    Op op(m, GPT2_K_ADAMW);
    TRY(op.done(launch_adamw(m->master + begin,
                             m->mode == GPT2_MODE_BF16 ? (void*)((bf16*)m->params + begin) : nullptr,
                             m->grads + begin, m->adam_m + begin, m->adam_v + begin, count, c->lr, c->beta1,
                             c->beta2, c->eps, c->weight_decay, c->t, m->stream, c->grad_scale, nullptr, 0.f,
                             c->decay_mask ? m->decay_bits + begin / 2048 : nullptr),
                (double)count * (m->mode == GPT2_MODE_BF16 ? 30.0 : 28.0)));
    m->state = 4;
    return GPT2_OK;
}

float gpt2_lr_cosine(int t, int warmup, int total, float lr_max, float lr_min) {
    if (t < 1) return 0.f;
    if (warmup > 0 && t <= warmup) return lr_max * (float)t / (float)warmup;
    if (t >= total) return lr_min;
    const double frac = (double)(t - warmup) / (double)(total - warmup);  // in (0, 1)
    return (float)(lr_min + 0.5 * (lr_max - lr_min) * (1.0 + std::cos(3.14159265358979323846 * frac)));
}

int gpt2_destroy(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    cudaStreamSynchronize(m->stream);
    if (m->step_exec) cudaGraphExecDestroy(m->step_exec);
    if (m->capture_stream) cudaStreamDestroy(m->capture_stream);
    for (auto& p : m->pending) {
        cudaEventDestroy(p.a);
        cudaEventDestroy(p.b);
    }
    for (auto e : m->pool) cudaEventDestroy(e);
    delete m;
    return GPT2_OK;
}

const char* gpt2_strerror(int s) {
    switch (s) {
        case GPT2_OK: return "ok";
        case GPT2_ERR_ARG: return "invalid argument";
        case GPT2_ERR_STATE: return "call out of order";
        case GPT2_ERR_TOKEN_RANGE: return "token or target id out of range";
        case GPT2_ERR_NONFINITE: return "loss is not finite";
        case GPT2_ERR_TIMEOUT: return "device wait timed out";
        case GPT2_ERR_CUDA: return "CUDA runtime error";
        case GPT2_ERR_WORKSPACE: return "workspace too small or misaligned";
        default: return "unknown status";
    }
}

int gpt2_num_tensors(const gpt2_t* m) { return m ? (int)m->tensors.size() : GPT2_ERR_ARG; }

int gpt2_tensor_info(const gpt2_t* m, int i, const char** name, int64_t shape[2]) {
    if (!m || i < 0 || i >= (int)m->tensors.size()) return GPT2_ERR_ARG;
    if (name) *name = m->tensors[i].name.c_str();
    if (shape) {
        shape[0] = m->tensors[i].rows;
        shape[1] = m->tensors[i].cols;
    }
    return GPT2_OK;
}

int gpt2_copy_tensor(gpt2_t* m, int i, int kind, float* host_dst) {
    if (!m || !host_dst || i < 0 || i >= (int)m->tensors.size()) return GPT2_ERR_ARG;
    const TensorSpec& s = m->tensors[i];
    const int64_t n = s.rows * s.cols;
    const float* src = nullptr;
    switch (kind) {
        case GPT2_TENSOR_MASTER: src = m->master; break;
        case GPT2_TENSOR_GRAD: src = m->grads; break;
        case GPT2_TENSOR_ADAM_M: src = m->adam_m; break;
        case GPT2_TENSOR_ADAM_V: src = m->adam_v; break;
        case GPT2_TENSOR_PARAM:
            if (m->mode != GPT2_MODE_BF16) {
                src = m->master;
                break;
            } else {
                std::vector<uint16_t> tmp((size_t)n);
                if (cudaMemcpyAsync(tmp.data(), (bf16*)m->params + s.offset, (size_t)n * 2, cudaMemcpyDeviceToHost,
                                    m->stream) != cudaSuccess ||
                    cudaStreamSynchronize(m->stream) != cudaSuccess)
                    return GPT2_ERR_CUDA;
                for (int64_t k = 0; k < n; k++) {
                    const uint32_t bits = (uint32_t)tmp[(size_t)k] << 16;
                    std::memcpy(&host_dst[k], &bits, 4);
                }
                return GPT2_OK;
            }
        default: return GPT2_ERR_ARG;
    }
    if (cudaMemcpyAsync(host_dst, src + s.offset, (size_t)n * 4, cudaMemcpyDeviceToHost, m->stream) != cudaSuccess)
        return GPT2_ERR_CUDA;
    return cuda_ok(cudaStreamSynchronize(m->stream));
}

int gpt2_load_tensor(gpt2_t* m, int i, const float* host_src) {
    if (!m || !host_src || i < 0 || i >= (int)m->tensors.size()) return GPT2_ERR_ARG;
    const TensorSpec& s = m->tensors[i];
    const int64_t n = s.rows * s.cols;
    if (cudaMemcpyAsync(m->master + s.offset, host_src, (size_t)n * 4, cudaMemcpyHostToDevice, m->stream) !=
        cudaSuccess)
        return GPT2_ERR_CUDA;
    TRY(refresh_compute_copy(m, s.offset, n));
    return cuda_ok(cudaStreamSynchronize(m->stream));
}

int gpt2_copy_losses(gpt2_t* m, float* host_dst) {
    if (!m || !host_dst) return GPT2_ERR_ARG;
    if (m->state < 1) return GPT2_ERR_STATE;
    if (cudaMemcpyAsync(host_dst, m->losses, (size_t)m->B * m->T * 4, cudaMemcpyDeviceToHost, m->stream) !=
        cudaSuccess)
        return GPT2_ERR_CUDA;
    return cuda_ok(cudaStreamSynchronize(m->stream));
}

int64_t gpt2_num_params(const gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    int64_t n = 0;
    for (auto& s : m->tensors) n += s.rows * s.cols;
    return n;
}

int64_t gpt2_launch_count(const gpt2_t* m) { return m ? m->launches : GPT2_ERR_ARG; }

int gpt2_family_stats(const gpt2_t* m, int family, int64_t* calls, int64_t* launches, double* work) {
    if (!m || family < 0 || family >= GPT2_K_COUNT) return GPT2_ERR_ARG;
    if (calls) *calls = m->fam_calls[family];
    if (launches) *launches = m->fam_launches[family];
    if (work) *work = m->fam_work[family];
    return GPT2_OK;
}

int gpt2_set_timing(gpt2_t* m, int enable) {
    if (!m) return GPT2_ERR_ARG;
    m->timing = enable != 0;
    return GPT2_OK;
}

int gpt2_family_time(gpt2_t* m, int family, double* ms) {
    if (!m || family < 0 || family >= GPT2_K_COUNT || !ms) return GPT2_ERR_ARG;
    if (cudaStreamSynchronize(m->stream) != cudaSuccess) return GPT2_ERR_CUDA;
    for (auto& p : m->pending) {
        float t = 0.f;
        cudaEventElapsedTime(&t, p.a, p.b);
        m->fam_ms[p.fam] += t;
        m->pool.push_back(p.a);
        m->pool.push_back(p.b);
    }
    m->pending.clear();
    *ms = m->fam_ms[family];
    return GPT2_OK;
}

int gpt2_reset_stats(gpt2_t* m) {
    if (!m) return GPT2_ERR_ARG;
    if (cudaStreamSynchronize(m->stream) != cudaSuccess) return GPT2_ERR_CUDA;
    for (auto& p : m->pending) {
        m->pool.push_back(p.a);
        m->pool.push_back(p.b);
    }
    m->pending.clear();
    m->launches = 0;
    for (int f = 0; f < GPT2_K_COUNT; f++) {
        m->fam_calls[f] = m->fam_launches[f] = 0;
        m->fam_work[f] = m->fam_ms[f] = 0;
    }
    return GPT2_OK;
}

}  // extern "C"
