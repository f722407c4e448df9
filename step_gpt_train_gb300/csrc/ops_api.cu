// C entry points of gpt2_ops.h: argument checks, then the kernel launchers.
#include "common.cuh"
#include "launch.h"

namespace {

inline bool dt_ok(int dtype) { return dtype == GPT2_MODE_FP32 || dtype == GPT2_MODE_BF16; }
inline bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline int finish(int launches) {
    if (launches < 0) return launches;
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}
inline cudaStream_t st(void* s) { return (cudaStream_t)s; }

}  // namespace

extern "C" {

int gpt2_op_encoder_forward(int dtype, void* x0, const int32_t* tokens, const void* wte, const void* wpe, int B,
                            int T, int C, int V, int* d_status, void* stream) {
    if (!dt_ok(dtype) || !x0 || !tokens || !wte || !wpe || B < 0 || T < 0 || C <= 0 || C % 8 || V < 1)
        return GPT2_ERR_ARG;
    if (!al16(x0) || !al16(wte) || !al16(wpe)) return GPT2_ERR_ARG;
    if ((int64_t)B * T == 0) return GPT2_OK;
    return finish(launch_encoder_forward(dtype, x0, tokens, wte, wpe, B, T, C, V, d_status, st(stream)));
}

size_t gpt2_op_encoder_backward_scratch(int B, int T, int C) {
    if (B < 0 || T < 0 || C < 0) return 0;
    return encoder_backward_scratch(B, T, C);
}

int gpt2_op_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dx0, const int32_t* tokens, int B,
                             int T, int C, int Vp, void* scratch, size_t scratch_bytes, void* stream) {
    if (!dt_ok(dtype) || !dwte || !dwpe || !dx0 || !tokens || B < 0 || T < 0 || C <= 0 || C % 8 || Vp < 1 ||
        Vp > 65536)
        return GPT2_ERR_ARG;
    if ((int64_t)B * T == 0) {
        // no rows: dwte gains nothing; dwpe[0, T) is the empty sum (zero) when only B is 0
        if (T > 0 && cudaMemsetAsync(dwpe, 0, (size_t)T * C * 4, st(stream)) != cudaSuccess) return GPT2_ERR_CUDA;
        return GPT2_OK;
    }
    if (!scratch || scratch_bytes < encoder_backward_scratch(B, T, C)) return GPT2_ERR_WORKSPACE;
    if (!al16(dwte) || !al16(dwpe) || !al16(dx0)) return GPT2_ERR_ARG;
    return finish(launch_encoder_backward(dtype, dwte, dwpe, dx0, tokens, B, T, C, scratch, st(stream)));
}

int gpt2_op_layernorm_forward(int dtype, void* y, float* mean, float* rstd, const void* x, const void* gamma,
                              const void* beta, int N, int C, void* stream) {
    if (!dt_ok(dtype) || !y || !mean || !rstd || !x || !gamma || !beta || N < 0 || C <= 0 || C % 8 || C > 2048)
        return GPT2_ERR_ARG;
    if (!al16(y) || !al16(x) || !al16(gamma) || !al16(beta)) return GPT2_ERR_ARG;
    return finish(launch_layernorm_forward(dtype, y, mean, rstd, x, gamma, beta, N, C, st(stream)));
}

size_t gpt2_op_layernorm_backward_scratch(int N, int C) {
    if (N < 0 || C < 0) return 0;
    return layernorm_backward_scratch(N, C);
}

int gpt2_op_layernorm_backward(int dtype, void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                               const void* gamma, const float* mean, const float* rstd, int N, int C, void* scratch,
                               size_t scratch_bytes, void* stream) {
    if (!dt_ok(dtype) || !dx || !dgamma || !dbeta || !dy || !x || !gamma || !mean || !rstd || N < 0 || C <= 0 ||
        C % 8 || C > 2048)
        return GPT2_ERR_ARG;
    if (!scratch || scratch_bytes < layernorm_backward_scratch(N, C)) return GPT2_ERR_WORKSPACE;
    if (!al16(dx) || !al16(dy) || !al16(x) || !al16(gamma)) return GPT2_ERR_ARG;
    return finish(launch_layernorm_backward(dtype, dx, dgamma, dbeta, dy, x, gamma, mean, rstd, N, C, scratch,
                                            st(stream)));
}

int gpt2_op_residual_layernorm_forward(int dtype, void* y, float* mean, float* rstd, void* xsum, const void* x,
                                       const void* r, const void* gamma, const void* beta, int N, int C,
                                       void* stream) {
    if (!dt_ok(dtype) || !y || !mean || !rstd || !xsum || !x || !r || !gamma || !beta || N < 0 || C <= 0 ||
        C % 8 || C > 2048)
        return GPT2_ERR_ARG;
    if (!al16(y) || !al16(xsum) || !al16(x) || !al16(r) || !al16(gamma) || !al16(beta)) return GPT2_ERR_ARG;
    return finish(launch_residual_layernorm_forward(dtype, y, mean, rstd, xsum, x, r, gamma, beta, N, C, st(stream)));
}

int gpt2_op_layernorm_backward_residual(int dtype, void* dres, int accumulate, float* dgamma, float* dbeta,
                                        float* dres_colsum, const void* dy, const void* x, const void* gamma,
                                        const float* mean, const float* rstd, int N, int C, void* scratch,
                                        size_t scratch_bytes, void* stream) {
    if (!dt_ok(dtype) || !dres || !dgamma || !dbeta || !dy || !x || !gamma || !mean || !rstd || N < 0 || C <= 0 ||
        C % 8 || C > 2048 || (accumulate != 0 && accumulate != 1))
        return GPT2_ERR_ARG;
    if (!scratch || scratch_bytes < layernorm_backward_scratch(N, C)) return GPT2_ERR_WORKSPACE;
    if (!al16(dres) || !al16(dy) || !al16(x) || !al16(gamma)) return GPT2_ERR_ARG;
    return finish(launch_layernorm_backward_residual(dtype, dres, accumulate, dgamma, dbeta, dres_colsum, dy, x, gamma,
                                                     mean, rstd, N, C, scratch, st(stream)));
}

size_t gpt2_op_matmul_scratch(int dtype, int M, int N, int K, int d_fp32) {
    if (!dt_ok(dtype) || M < 0 || N < 0 || K < 0) return 0;
    return matmul_scratch(dtype, M, N, K, d_fp32);
}

int gpt2_op_matmul(int dtype, void* D, int d_fp32, const void* A, int a_mn_major, const void* B, int b_mn_major,
                   const void* bias, int M, int N, int K, void* scratch, size_t scratch_bytes, int* d_status,
                   void* stream) {
    if (!dt_ok(dtype) || !D || !A || !B || M < 0 || N < 0 || K < 1) return GPT2_ERR_ARG;
    if (dtype == GPT2_MODE_BF16) {
        if (K % 8 || N % 8 || (a_mn_major && M % 8)) return GPT2_ERR_ARG;
        if (!al16(D) || !al16(A) || !al16(B) || (bias && !al16(bias))) return GPT2_ERR_ARG;
    }
    if ((int64_t)M * N == 0) return GPT2_OK;
    const size_t need = matmul_scratch(dtype, M, N, K, d_fp32);
    if (need && (!scratch || scratch_bytes < need)) return GPT2_ERR_WORKSPACE;
    return finish(launch_matmul(dtype, D, d_fp32, A, a_mn_major, B, b_mn_major, bias, M, N, K, scratch, d_status,
                                st(stream)));
}

size_t gpt2_op_quantize_fp8_scratch(void) { return fp8_quantize_scratch(); }

static bool fp8_format_ok(int f) { return f == GPT2_FP8_E4M3 || f == GPT2_FP8_E5M2; }
static_assert(GPT2_FP8_E4M3 == FP8_E4M3 && GPT2_FP8_E5M2 == FP8_E5M2, "FP8 format codes");

int gpt2_op_quantize_fp8(void* q, float* scales, const void* x, int64_t n, int format, void* scratch,
                         size_t scratch_bytes, void* stream) {
    if (!q || !scales || !x || n < 0 || !fp8_format_ok(format)) return GPT2_ERR_ARG;
    if (((uintptr_t)q % 8) || !al16(x)) return GPT2_ERR_ARG;
    if (n == 0) return GPT2_OK;
    if (!scratch || scratch_bytes < fp8_quantize_scratch()) return GPT2_ERR_WORKSPACE;
    return finish(launch_quantize_fp8((uint8_t*)q, scales, (const bf16*)x, n, format, (float*)scratch, st(stream)));
}

int gpt2_op_matmul_fp8(void* D, const void* A, int a_format, const float* a_scales, const void* B, int b_format,
                       const float* b_scales, const void* bias, int M, int N, int K, int* d_status, void* stream) {
    if (!D || !A || !B || !a_scales || !b_scales || M < 0 || N < 0 || K < 1) return GPT2_ERR_ARG;
    if (!fp8_format_ok(a_format) || !fp8_format_ok(b_format)) return GPT2_ERR_ARG;
    if (K % 16 || N % 8) return GPT2_ERR_ARG;
    if (!al16(D) || !al16(A) || !al16(B) || (bias && !al16(bias))) return GPT2_ERR_ARG;
    if ((int64_t)M * N == 0) return GPT2_OK;
    return finish(launch_matmul_fp8((bf16*)D, (const uint8_t*)A, a_format, a_scales + 1, (const uint8_t*)B, b_format,
                                    b_scales + 1, (const bf16*)bias, M, N, K, d_status, st(stream)));
}

int gpt2_op_quantize_fp8_transpose(void* qt, void* q, const float* scales, const void* x, int R, int C, int format,
                                   void* stream) {
    if (!qt || !scales || !x || R < 0 || C < 0 || C % 8 || !fp8_format_ok(format) || !al16(x)) return GPT2_ERR_ARG;
    if ((int64_t)R * C == 0) return GPT2_OK;
    if ((int64_t)R * C >= ((int64_t)1 << 40) || (R + 127) / 128 > 65535) return GPT2_ERR_ARG;
    return finish(launch_quantize_fp8_t((uint8_t*)qt, (uint8_t*)q, scales, (const bf16*)x, R, C, format, st(stream)));
}

size_t gpt2_op_matmul_fp8_scratch(int M, int N, int K, int d_fp32, int accumulate) {
    if (M < 0 || N < 0 || K < 1) return 0;
    return matmul_f8_scratch(M, N, K, d_fp32, accumulate);
}

int gpt2_op_matmul_fp8_ex(int epi, void* D, void* D2, const void* aux, int d_fp32, int accumulate, const void* A,
                          int a_format, const float* a_scales, const void* B, int b_format, const float* b_scales,
                          const void* bias, int M, int N, int K, void* scratch, size_t scratch_bytes, int* d_status,
                          void* stream) {
    if (!D || !A || !B || !a_scales || !b_scales || M < 0 || N < 0 || K < 1 || epi < 0 || epi > 2) return GPT2_ERR_ARG;
    if (!fp8_format_ok(a_format) || !fp8_format_ok(b_format) || K % 16 || N % 8) return GPT2_ERR_ARG;
    if (!al16(D) || !al16(A) || !al16(B) || (bias && !al16(bias))) return GPT2_ERR_ARG;
    if (epi == 1 && (!D2 || !al16(D2) || D2 == D || d_fp32)) return GPT2_ERR_ARG;
    if (epi == 2 && (!aux || !al16(aux) || aux == D || d_fp32 || bias)) return GPT2_ERR_ARG;
    if (accumulate && (!d_fp32 || epi)) return GPT2_ERR_ARG;
    if ((int64_t)M * N == 0) return GPT2_OK;
    if (scratch_bytes < matmul_f8_scratch(M, N, K, d_fp32, accumulate) || (scratch_bytes && !scratch))
        return GPT2_ERR_WORKSPACE;
    const F8Args f8 = {a_format, b_format, a_scales + 1, b_scales + 1};
    const uint8_t* a8 = (const uint8_t*)A;
    const uint8_t* b8 = (const uint8_t*)B;
    if (epi == 1) return finish(launch_matmul_gelu_f8(D, D2, a8, b8, f8, bias, M, N, K, d_status, st(stream)));
    if (epi == 2) return finish(launch_matmul_gelu_backward_f8(D, a8, b8, f8, aux, M, N, K, d_status, st(stream)));
    return finish(launch_matmul_f8(D, d_fp32, a8, b8, f8, bias, M, N, K, scratch, d_status, st(stream), accumulate));
}

int gpt2_op_matmul_gelu(int dtype, void* dgelu, void* out, const void* A, const void* W, const void* bias, int M,
                        int N, int K, int* d_status, void* stream) {
    if (!dt_ok(dtype) || !dgelu || !out || !A || !W || M < 0 || N < 0 || K < 1 || dgelu == out) return GPT2_ERR_ARG;
    if (dtype != GPT2_MODE_BF16 && ((int64_t)M * N) % 8) return GPT2_ERR_ARG;  // the GELU pass works on 8-vectors
    if (dtype == GPT2_MODE_BF16) {
        if (K % 8 || N % 8) return GPT2_ERR_ARG;
        if (!al16(dgelu) || !al16(out) || !al16(A) || !al16(W) || (bias && !al16(bias))) return GPT2_ERR_ARG;
    }
    if ((int64_t)M * N == 0) return GPT2_OK;
    if (dtype == GPT2_MODE_BF16)
        return finish(launch_matmul_gelu(dgelu, out, A, W, bias, M, N, K, d_status, st(stream)));
    const int r = launch_matmul(dtype, dgelu, 0, A, 0, W, 0, bias, M, N, K, nullptr, d_status, st(stream));
    if (r < 0) return r;
    return finish(launch_gelu_both(dtype, out, dgelu, dgelu, (int64_t)M * N, st(stream)));
}

int gpt2_op_matmul_gelu_backward(int dtype, void* du, const void* dY, const void* W, const void* dgelu, int M, int N,
                                 int K, int* d_status, void* stream) {
    if (!dt_ok(dtype) || !du || !dY || !W || !dgelu || M < 0 || N < 0 || K < 1 || du == dgelu) return GPT2_ERR_ARG;
    if (dtype != GPT2_MODE_BF16 && ((int64_t)M * N) % 8) return GPT2_ERR_ARG;  // the multiply works on 8-vectors
    if (dtype == GPT2_MODE_BF16) {
        if (K % 8 || N % 8) return GPT2_ERR_ARG;
        if (!al16(du) || !al16(dY) || !al16(W) || !al16(dgelu)) return GPT2_ERR_ARG;
    }
    if ((int64_t)M * N == 0) return GPT2_OK;
    if (dtype == GPT2_MODE_BF16)
        return finish(launch_matmul_gelu_backward(du, dY, W, dgelu, M, N, K, d_status, st(stream)));
    const int r = launch_matmul(dtype, du, 0, dY, 0, W, 1, nullptr, M, N, K, nullptr, d_status, st(stream));
    if (r < 0) return r;
    return finish(launch_mul(dtype, du, du, dgelu, (int64_t)M * N, st(stream)));
}

size_t gpt2_op_matmul_gelu_backward_bias_scratch(int M, int N) {
    if (M < 0 || N < 0) return 0;
    const size_t fused = (size_t)matmul_gelu_backward_colsum_rows(M) * N * 4;  // bf16: per 32-row slice
    const size_t pass = bias_backward_scratch(M, N);                           // fp32: per 128 rows
    return fused > pass ? fused : pass;
}

int gpt2_op_matmul_gelu_backward_bias(int dtype, void* du, float* dbias, const void* dY, const void* W,
                                      const void* dgelu, int M, int N, int K, void* scratch, size_t scratch_bytes,
                                      int* d_status, void* stream) {
    if (!dbias) return GPT2_ERR_ARG;
    if (!scratch || scratch_bytes < gpt2_op_matmul_gelu_backward_bias_scratch(M, N)) return GPT2_ERR_WORKSPACE;
    if (dtype != GPT2_MODE_BF16 || (int64_t)M * N == 0) {
        const int r = gpt2_op_matmul_gelu_backward(dtype, du, dY, W, dgelu, M, N, K, d_status, stream);
        if (r != GPT2_OK) return r;
        if (N > 0) return finish(launch_bias_backward(dtype, dbias, du, M, N, scratch, st(stream)));
        return GPT2_OK;
    }
    if (!du || !dY || !W || !dgelu || K < 1 || du == dgelu || K % 8 || N % 8 || M < 0 || N < 0) return GPT2_ERR_ARG;
    if (!al16(du) || !al16(dY) || !al16(W) || !al16(dgelu)) return GPT2_ERR_ARG;
    const int r = launch_matmul_gelu_backward(du, dY, W, dgelu, M, N, K, d_status, st(stream), (float*)scratch);
    if (r < 0) return r;
    return finish(launch_colsum3(dbias, nullptr, nullptr, N, (const float*)scratch,
                                 matmul_gelu_backward_colsum_rows(M), N, st(stream)));
}

int gpt2_op_attention_forward(int dtype, void* o, float* lse, const void* qkv, int B, int T, int C, int H,
                              void* stream) {
    if (!dt_ok(dtype) || !o || !lse || !qkv || B < 0 || T < 0 || C <= 0 || H <= 0 || C % H || C % 8)
        return GPT2_ERR_ARG;
    if (!al16(o) || !al16(qkv)) return GPT2_ERR_ARG;
    return finish(launch_attention_forward(dtype, o, lse, qkv, B, T, C, H, nullptr, st(stream)));
}

size_t gpt2_op_attention_backward_scratch(int B, int T, int H) {
    if (B < 0 || T < 0 || H < 0) return 0;
    return attention_backward_scratch(B, T, H);
}

int gpt2_op_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv, const void* o,
                               const float* lse, int B, int T, int C, int H, void* scratch, size_t scratch_bytes,
                               void* stream) {
    if (!dt_ok(dtype) || !dqkv || !dout || !qkv || !o || !lse || B < 0 || T < 0 || C <= 0 || H <= 0 || C % H ||
        C % 8)
        return GPT2_ERR_ARG;
    if (!scratch || scratch_bytes < attention_backward_scratch(B, T, H)) return GPT2_ERR_WORKSPACE;
    if (!al16(dqkv) || !al16(dout) || !al16(qkv) || !al16(o)) return GPT2_ERR_ARG;
    return finish(launch_attention_backward(dtype, dqkv, dout, qkv, o, lse, B, T, C, H, scratch, nullptr, st(stream)));
}

int gpt2_op_gelu_forward(int dtype, void* g, const void* u, int64_t n, void* stream) {
    if (!dt_ok(dtype) || !g || !u || n < 0 || n % 8 || !al16(g) || !al16(u)) return GPT2_ERR_ARG;
    return finish(launch_gelu_forward(dtype, g, u, n, st(stream)));
}

int gpt2_op_gelu_backward(int dtype, void* du, const void* u, const void* dg, int64_t n, void* stream) {
    if (!dt_ok(dtype) || !du || !u || !dg || n < 0 || n % 8 || !al16(du) || !al16(u) || !al16(dg))
        return GPT2_ERR_ARG;
    return finish(launch_gelu_backward(dtype, du, u, dg, n, st(stream)));
}

int gpt2_op_residual_forward(int dtype, void* out, const void* a, const void* b, int64_t n, void* stream) {
    if (!dt_ok(dtype) || !out || !a || !b || n < 0 || n % 8 || !al16(out) || !al16(a) || !al16(b))
        return GPT2_ERR_ARG;
    return finish(launch_residual_forward(dtype, out, a, b, n, st(stream)));
}

int gpt2_op_residual_backward(int dtype, void* dres, const void* dbranch, int64_t n, void* stream) {
    if (!dt_ok(dtype) || !dres || !dbranch || n < 0 || n % 8 || !al16(dres) || !al16(dbranch)) return GPT2_ERR_ARG;
    return finish(launch_residual_backward(dtype, dres, dbranch, n, st(stream)));
}

size_t gpt2_op_bias_backward_scratch(int N, int C) {
    if (N < 0 || C < 0) return 0;
    return bias_backward_scratch(N, C);
}

int gpt2_op_bias_backward(int dtype, float* dbias, const void* dy, int N, int C, void* scratch, size_t scratch_bytes,
                          void* stream) {
    if (!dt_ok(dtype) || !dbias || !dy || N < 0 || C <= 0 || C % 8 || !al16(dy)) return GPT2_ERR_ARG;
    if (N == 0) return cudaMemsetAsync(dbias, 0, (size_t)C * 4, st(stream)) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
    if (!scratch || scratch_bytes < bias_backward_scratch(N, C)) return GPT2_ERR_WORKSPACE;
    return finish(launch_bias_backward(dtype, dbias, dy, N, C, scratch, st(stream)));
}

int gpt2_op_classifier(int dtype, void* logits, float* losses, const int32_t* targets, int N, int V, int Vp,
                       float dloss, int* d_status, void* stream) {
    if (!dt_ok(dtype) || !logits || !losses || !targets || N < 0 || V < 1 || Vp < V || Vp % 8 || !al16(logits))
        return GPT2_ERR_ARG;
    return finish(launch_classifier(dtype, logits, losses, targets, N, V, Vp, dloss, d_status, st(stream)));
}

int gpt2_op_mean_loss(float* out, const float* losses, int N, void* stream) {
    if (!out || !losses || N < 1) return GPT2_ERR_ARG;
    return finish(launch_mean_loss(out, losses, N, st(stream)));
}

int gpt2_op_adamw(float* master, void* param_bf16, const float* grad, float* m, float* v, int64_t n, float lr,
                  float beta1, float beta2, float eps, float weight_decay, int t, void* stream) {
    if (!master || !grad || !m || !v || n < 0 || n % 4 || t < 1) return GPT2_ERR_ARG;
    if (!al16(master) || !al16(grad) || !al16(m) || !al16(v) || (param_bf16 && ((uintptr_t)param_bf16 & 7u)))
        return GPT2_ERR_ARG;
    return finish(launch_adamw(master, param_bf16, grad, m, v, n, lr, beta1, beta2, eps, weight_decay, t,
                               st(stream)));
}

int gpt2_debug_set_wait_limit(int64_t cycles) {
    const long long c = cycles > 0 ? (long long)cycles : 0;
    if (gemm_tc_set_wait_limit(c) || attention_tc_set_wait_limit(c) || classifier_set_wait_limit(c))
        return GPT2_ERR_CUDA;
    return GPT2_OK;
}

int gpt2_debug_stall_matmul(int on) { return gemm_tc_stall_for_test(on) ? GPT2_ERR_CUDA : GPT2_OK; }

int gpt2_debug_matmul_pair(int on) { return gemm_tc_use_pair(on); }

}  // extern "C"
