// Host-side launchers of the step's kernels. Each enqueues its kernels on
// stream s and returns the number of kernel launches it made (>= 0), or a
// negative gpt2_status for an unsupported shape. Arguments are already
// validated by the caller.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

int launch_encoder_forward(int dtype, void* x0, const int32_t* tokens, const void* wte, const void* wpe, int B,
                           int T, int C, int V, int* status, cudaStream_t s);
size_t encoder_backward_scratch(int B, int T, int C);
// dwte rows of the ids += the embedding gradient (dwte holds the LM head's
// part); dwpe[t] = (or +=, with accumulate) the column sums over the batch.
int launch_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dx0, const int32_t* tokens, int B, int T,
                            int C, void* scratch, cudaStream_t s, int accumulate = 0);

// amax (optional, every LayerNorm forward and backward below): the largest |output| as
// stored is merged into it (float bits; the caller zeroes it), the scale of an FP8 operand.
int launch_layernorm_forward(int dtype, void* y, float* mean, float* rstd, const void* x, const void* gamma,
                             const void* beta, int N, int C, cudaStream_t s, unsigned* amax = nullptr);
size_t layernorm_backward_scratch(int N, int C);
int launch_layernorm_backward(int dtype, void* dx, float* dgamma, float* dbeta, const void* dy, const void* x,
                              const void* gamma, const float* mean, const float* rstd, int N, int C, void* scratch,
                              cudaStream_t s);

// The residual join followed by LayerNorm: xsum = x + r (rounded to dtype),
// y = LayerNorm(xsum).
int launch_residual_layernorm_forward(int dtype, void* y, float* mean, float* rstd, void* xsum, const void* x,
                                      const void* r, const void* gamma, const void* beta, int N, int C,
                                      cudaStream_t s, unsigned* amax = nullptr);
// LayerNorm backward into the residual gradient: dres = dx (accumulate == 0)
// or dres += dx; dres_colsum (optional) = column sums of the resulting dres.
// grad_accumulate: dgamma, dbeta and dres_colsum are added to instead of overwritten.
int launch_layernorm_backward_residual(int dtype, void* dres, int accumulate, float* dgamma, float* dbeta,
                                       float* dres_colsum, const void* dy, const void* x, const void* gamma,
                                       const float* mean, const float* rstd, int N, int C, void* scratch,
                                       cudaStream_t s, int grad_accumulate = 0);
// Its row pass alone: dres (+)= dx and partial [*rows][np * C] (np 2: dgamma,
// dbeta parts; 3: and the column sums of dres), for a deferred ColsumJob.
// partial: layernorm_backward_scratch(N, C) bytes.
int launch_layernorm_backward_residual_rows(int dtype, void* dres, int accumulate, float* partial, int np,
                                            const void* dy, const void* x, const void* gamma, const float* mean,
                                            const float* rstd, int N, int C, cudaStream_t s, int* rows,
                                            unsigned* amax = nullptr);

int launch_gelu_forward(int dtype, void* g, const void* u, int64_t n, cudaStream_t s);
int launch_gelu_backward(int dtype, void* du, const void* u, const void* dg, int64_t n, cudaStream_t s);
int launch_residual_forward(int dtype, void* out, const void* a, const void* b, int64_t n, cudaStream_t s);
int launch_residual_backward(int dtype, void* dres, const void* dbranch, int64_t n, cudaStream_t s);

// out[c] (c < split) / out2[c - split] (c >= split) = column sums of in [R, ncols], deterministic.
int launch_colsum(float* out, float* out2, int split, const float* in, int R, int ncols, cudaStream_t s);
// out_q[c] = column sums of column q * seg + c of in [R, ncols], q < 3 (null outputs skipped).
int launch_colsum3(float* out0, float* out1, float* out2, int seg, const float* in, int R, int ncols,
                   cudaStream_t s, int accumulate = 0);

// A column sum whose launch is deferred (the parameter-gradient reductions of
// a backward pass, gathered into one launch at its end): out[q][c] (+)= the
// sum over r of in[r][q * seg + c], q < 3 (null outputs skipped).
struct ColsumJob {
    const float* in;
    float* out[3];
    int R, ncols, seg, accumulate;
};
// All the jobs, in ceil(n / 32) launches; each job's result has the bits
// launch_colsum3 gives for it. Returns the launches.
int launch_colsum_jobs(const ColsumJob* jobs, int n, cudaStream_t s);

size_t bias_backward_scratch(int N, int C);
int launch_bias_backward(int dtype, float* dbias, const void* dy, int N, int C, void* scratch, cudaStream_t s,
                         int accumulate = 0);
// The first pass of launch_bias_backward alone: partial [rows][C] of column
// sums over 128-row chunks of dy; *rows = ceil(N / 128).
int launch_bias_partials(int dtype, float* partial, const void* dy, int N, int C, cudaStream_t s, int* rows);

// amax (optional): the largest |dlogit| as stored is merged into it (float bits).
int launch_classifier(int dtype, void* logits, float* losses, const int32_t* targets, int N, int V, int Vp,
                      float dloss, int* status, cudaStream_t s, unsigned* amax = nullptr);
int launch_mean_loss(float* out, const float* losses, int N, cudaStream_t s);

// grad_scale multiplies the gradient; with gnorm (device ||g||) and max_norm > 0
// the gradient is also clipped to max_norm; decay_bits (one bit per 64-element
// chunk, null = all) selects where weight decay applies.
int launch_adamw(float* master, void* pbf, const float* grad, float* m, float* v, int64_t n, float lr, float b1,
                 float b2, float eps, float wd, int t, cudaStream_t s, float grad_scale = 1.f,
                 const float* gnorm = nullptr, float max_norm = 0.f, const uint32_t* decay_bits = nullptr,
                 const float* hp = nullptr);
// *norm_out = ||g||_2 over n fp32 values (n % 4 == 0), deterministic; partial: grad_norm_scratch() bytes.
size_t grad_norm_scratch();
int launch_grad_norm(float* norm_out, float* partial, const float* g, int64_t n, cudaStream_t s, int root = 1);

int launch_attention_forward(int dtype, void* o, float* lse, const void* qkv, int B, int T, int C, int H,
                             int* status, cudaStream_t s);
// bf16 backward; D ([B, H, T] fp32 scratch) receives rowsum(dO * O).
int launch_attention_backward_tc(__nv_bfloat16* dqkv, const __nv_bfloat16* dout, const __nv_bfloat16* qkv,
                                 const __nv_bfloat16* o, const float* lse, float* D, int B, int T, int C, int H,
                                 int* status, cudaStream_t s);
int launch_attention_forward_tc(__nv_bfloat16* o, float* lse, const __nv_bfloat16* qkv, int B, int T, int C, int H,
                                int* status, cudaStream_t s);
size_t attention_backward_scratch(int B, int T, int H);
int launch_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv, const void* o,
                              const float* lse, int B, int T, int C, int H, void* scratch, int* status,
                              cudaStream_t s);

// bf16 linear forward with the GELU fused into its epilogue: u = A W^T + bias
// (A [M,K], W [N,K], both K-major) rounded to bf16, out = gelu(u), dgelu =
// gelu'(u) (kept for the backward); see gpt2_op_matmul_gelu.
// amax (optional, here and in the GELU backward): the largest |gelu(u)| (resp. |du|) as
// stored is merged into it (float bits; the caller zeroes it), the scale of an FP8 operand.
int launch_matmul_gelu(void* dgelu, void* out, const void* A, const void* W, const void* bias, int M, int N, int K,
                       int* status, cudaStream_t s, unsigned* amax = nullptr);
// bf16 input gradient through that GELU: du = bf16(dY W) * dgelu, dY [M,K], W [K,N];
// du_colsum (or null): column sums of the stored du per 32-row slice, [4 ceil(M/128)][N]
// (matmul_gelu_backward_colsum_rows).
inline int matmul_gelu_backward_colsum_rows(int M) { return 4 * ((M + 127) / 128); }
int launch_matmul_gelu_backward(void* du, const void* dY, const void* W, const void* dgelu, int M, int N, int K,
                                int* status, cudaStream_t s, float* du_colsum = nullptr, unsigned* amax = nullptr);
// out = gelu(u) and dgelu = gelu'(u) (dgelu may be u itself); n % 8 == 0.
int launch_gelu_both(int dtype, void* out, void* dgelu, const void* u, int64_t n, cudaStream_t s);
// out = a * b elementwise; n % 8 == 0.
int launch_mul(int dtype, void* out, const void* a, const void* b, int64_t n, cudaStream_t s);

// FP8 formats (OCP 8-bit floating point): e4m3 (largest finite 448), e5m2 (57344).
enum { FP8_E4M3 = 0, FP8_E5M2 = 1 };
// D (bf16 [M,N]) = (A B^T) * (*a_scale) * (*b_scale) (+ bias) on the tensor cores, A [M,K] and B
// [N,K] FP8 codes (K-major) in formats a_fmt and b_fmt, fp32 accumulation; K % 16 == 0, N % 8 == 0.
int launch_matmul_fp8(bf16* D, const uint8_t* A, int a_fmt, const float* a_scale, const uint8_t* B, int b_fmt,
                      const float* b_scale, const bf16* bias, int M, int N, int K, int* status, cudaStream_t s);
// Per-tensor FP8 quantization of n bf16 values to format fmt (largest finite value fmax):
// scales[0] = fmax / amax and scales[1] = amax / fmax (1 and 1 when amax is 0),
// q = fp8(x * scales[0]), round to nearest even, saturated; partial: fp8_quantize_scratch() bytes.
size_t fp8_quantize_scratch();
int launch_quantize_fp8(uint8_t* q, float* scales, const bf16* x, int64_t n, int fmt, float* partial, cudaStream_t s);
// Its two passes alone: the scales of n values (2 launches), and the codes of n
// values under given scales.
int launch_fp8_amax_scale(float* scales, const bf16* x, int64_t n, int fmt, float* partial, cudaStream_t s);
int launch_quantize_fp8_rows(uint8_t* q, const float* scales, const bf16* x, int64_t n, int fmt, cudaStream_t s);
// The codes of x [R][C] (C % 8 == 0) under given scales written transposed,
// qt [C][R], and (q non-null) also as they are, q [R][C]. With amax (x's
// largest |value| as float bits, from the kernel that wrote x) the scales are
// formed from it first and written to scales.
int launch_quantize_fp8_t(uint8_t* qt, uint8_t* q, const float* scales, const bf16* x, int R, int C, int fmt,
                          cudaStream_t s, const unsigned* amax = nullptr);

// FP8 operands of the general matmul (K-major codes, scale_inv device scalars).
struct F8Args {
    int a_fmt, b_fmt;
    const float* a_scale;  // amax / fmax of A's codes (the factor that maps them back)
    const float* b_scale;
};
// The matmul, its GELU-forward and GELU-backward epilogue forms with FP8
// operands: as launch_matmul_tc, launch_matmul_gelu and
// launch_matmul_gelu_backward, A [M,K] and B [N,K] FP8 codes (both K-major;
// the input gradient takes the weight's transposed codes), the accumulator
// scaled by *a_scale * *b_scale. K % 16 == 0, N % 8 == 0.
int launch_matmul_f8(void* D, int d_fp32, const uint8_t* A, const uint8_t* B, const F8Args& f8, const void* bias,
                     int M, int N, int K, void* scratch, int* status, cudaStream_t s, int accumulate = 0);
int launch_matmul_gelu_f8(void* dgelu, void* out, const uint8_t* A, const uint8_t* W, const F8Args& f8,
                          const void* bias, int M, int N, int K, int* status, cudaStream_t s,
                          unsigned* amax = nullptr);
int launch_matmul_gelu_backward_f8(void* du, const uint8_t* dY, const uint8_t* WT, const F8Args& f8,
                                   const void* dgelu, int M, int N, int K, int* status, cudaStream_t s,
                                   float* du_colsum = nullptr, unsigned* amax = nullptr);
// Scratch of launch_matmul_f8 (split-K partial tiles of an fp32 output).
size_t matmul_f8_scratch(int M, int N, int K, int d_fp32, int accumulate = 0);

// Matmul: D[M,N] = sum_k A(m,k) B(n,k) (+ bias), see gpt2_op_matmul.
// accumulate (fp32 D only): D += the product instead of D = it; the scratch
// size then covers the partial tiles that route through the reduce kernel.
size_t matmul_scratch(int dtype, int M, int N, int K, int d_fp32, int accumulate = 0);
int launch_matmul(int dtype, void* D, int d_fp32, const void* A, int a_mn, const void* B, int b_mn, const void* bias,
                  int M, int N, int K, void* scratch, int* status, cudaStream_t s, int accumulate = 0);

// Failure-path test hooks (current device): each translation unit with
// bounded tcgen05 / bulk-copy waits sets its own wait bound (cycles <= 0:
// the default); the GEMM's stall switch makes its MMA warp wait on a barrier
// nothing arrives at. 0 or -1 on a CUDA error.
int gemm_tc_set_wait_limit(long long cycles);
int attention_tc_set_wait_limit(long long cycles);
int classifier_set_wait_limit(long long cycles);
int gemm_tc_stall_for_test(int on);
// The CTA-pair GEMM for the wide matmuls (on != 0) or the one-CTA kernel only
// (0, the default); returns the pair kernel's resident clusters when on.
int gemm_tc_use_pair(int on);
