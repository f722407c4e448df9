/*
 * gpt2_ops.h - the kernels of the GPT-2 training step, one entry point each.
 *
 * These are the same kernels gpt2_forward/gpt2_backward/gpt2_adamw_step run,
 * exposed on caller-owned device buffers so that each can be checked alone.
 * The kernel list is the one of llm.c "State of the Union [May 3, 2024]",
 * kernel table under "Runtime, DRAM traffic, instructions": encoder forward
 * and backward, layernorm forward and backward, the bf16 matmuls, attention
 * forward and backward, GELU forward and backward, residual, the fused
 * classifier, the bias-gradient reduction and AdamW.
 *
 * Conventions:
 *   - dtype: GPT2_MODE_FP32 (0) for fp32 activations, GPT2_MODE_BF16 (1) for
 *     bf16 activations. Arithmetic inside a kernel is fp32 in both.
 *   - Every pointer is a device pointer unless stated. All tensors are
 *     dense and row-major. Activation buffers need 16-byte alignment.
 *   - stream is a cudaStream_t (NULL = legacy default stream). Calls only
 *     enqueue work; they never synchronise, allocate or free.
 *   - scratch: caller-owned device memory of at least the size the matching
 *     *_scratch_bytes() call returns (256-byte aligned); its contents on
 *     entry do not matter. Two calls that share a scratch buffer must not
 *     overlap on the device.
 *   - d_status: optional device int; kernels OR an error bit into it
 *     (1 = token id out of range, 2 = bounded wait timed out, 4 = target id
 *     out of range) and never trap.
 *   - Return GPT2_OK or a negative gpt2_status (see gpt2.h) for bad
 *     arguments or a failed launch.
 */
#ifndef GPT2_OPS_H
#define GPT2_OPS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* x0[b,t,:] = wte[tokens[b,t],:] + wpe[t,:] (section "Single GPU training":
 * GPT-2's token plus learned position embedding; kernel "encoder_forward").
 * x0 [B*T, C], wte [>=V, C], wpe [>=T, C] in dtype. An id outside [0,V) sets
 * bit 1 of *d_status and reads row 0 instead. */
int gpt2_op_encoder_forward(int dtype, void* x0, const int32_t* tokens, const void* wte,
                            const void* wpe, int B, int T, int C, int V, int* d_status,
                            void* stream);

/* Embedding backward ("encoder_backward"): dwte[v,:] += sum of dx0 rows
 * whose token is v, summed in ascending position order (deterministic);
 * dwpe[t,:] = sum_b dx0[b,t,:] for t < T (rows t >= T untouched).
 * dwte [Vp, C] fp32 (accumulated into), dwpe [>=T, C] fp32 (overwritten),
 * dx0 [B*T, C] dtype, tokens in [0, Vp). */
size_t gpt2_op_encoder_backward_scratch(int B, int T, int C);
int gpt2_op_encoder_backward(int dtype, float* dwte, float* dwpe, const void* dx0,
                             const int32_t* tokens, int B, int T, int C, int Vp,
                             void* scratch, size_t scratch_bytes, void* stream);

/* LayerNorm forward ("layernorm_forward"): per row of x [N, C],
 * y = (x - mean) * rstd * gamma + beta, rstd = 1/sqrt(biased var + 1e-5);
 * mean and rstd [N] fp32 are saved for the backward. C % 8 == 0, C <= 2048. */
int gpt2_op_layernorm_forward(int dtype, void* y, float* mean, float* rstd, const void* x,
                              const void* gamma, const void* beta, int N, int C, void* stream);

/* LayerNorm backward ("layernorm_backward"): with xhat = (x-mean)*rstd and
 * dxhat = dy*gamma, dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat))
 * (dtype, overwritten); dgamma = sum_rows dy xhat, dbeta = sum_rows dy (fp32,
 * overwritten, deterministic two-stage reduction through scratch). */
size_t gpt2_op_layernorm_backward_scratch(int N, int C);
int gpt2_op_layernorm_backward(int dtype, void* dx, float* dgamma, float* dbeta, const void* dy,
                               const void* x, const void* gamma, const float* mean,
                               const float* rstd, int N, int C, void* scratch,
                               size_t scratch_bytes, void* stream);

/* Residual join followed by LayerNorm, one pass: xsum = x + r (rounded to
 * dtype, stored), then y, mean, rstd = LayerNorm of xsum exactly as
 * gpt2_op_layernorm_forward computes it. In the GPT-2 block every residual
 * sum ("residual_forward") is read next by a LayerNorm ("layernorm_forward";
 * llm.c "State of the Union", section "Runtime, DRAM traffic,
 * instructions"). xsum must not overlap x, r or y. Limits as for
 * gpt2_op_layernorm_forward. */
int gpt2_op_residual_layernorm_forward(int dtype, void* y, float* mean, float* rstd, void* xsum,
                                       const void* x, const void* r, const void* gamma,
                                       const void* beta, int N, int C, void* stream);

/* LayerNorm backward into the residual-stream gradient: with dx as in
 * gpt2_op_layernorm_backward, dres = dx (accumulate = 0) or dres += dx
 * (accumulate = 1, the residual join of the backward pass; dres is read and
 * written in place). dgamma, dbeta as in gpt2_op_layernorm_backward; if
 * dres_colsum is not null it receives the column sums of the resulting dres
 * (as stored, in dtype), fp32 [C], overwritten: the bias gradient
 * ("matmul_backward_bias") of the projection whose output joined the
 * residual stream at this point. Scratch: gpt2_op_layernorm_backward_scratch. */
int gpt2_op_layernorm_backward_residual(int dtype, void* dres, int accumulate, float* dgamma,
                                        float* dbeta, float* dres_colsum, const void* dy,
                                        const void* x, const void* gamma, const float* mean,
                                        const float* rstd, int N, int C, void* scratch,
                                        size_t scratch_bytes, void* stream);

/* Matmul (the bf16 GEMMs of the kernel table, "ampere_bf16" and
 * "cutlass::Kernel2"): D[M,N] = sum_k A(m,k) B(n,k) (+ bias[n]).
 * A(m,k) is A[m*K + k] (a_mn_major = 0) or A[k*M + m] (a_mn_major = 1);
 * B(n,k) is B[n*K + k] (b_mn_major = 0) or B[k*N + n] (b_mn_major = 1).
 * So the linear forward is (0,0) with B = W [N,K]; the input gradient
 * dX = dY W is (0,1); the weight gradient dW = dY^T X is (1,1).
 * A, B and bias (optional, length N, dtype) are in dtype; D is fp32 if
 * d_fp32 else dtype, overwritten. bf16: tcgen05 tensor cores (TMA-fed,
 * fp32 accumulate in tensor memory); fp32: fp32 FMA. Needs K % 8 == 0 and
 * N % 8 == 0 (and M % 8 == 0 when a_mn_major); 16-byte aligned buffers.
 * K >= 1 (K = 0 is GPT2_ERR_ARG); M = 0 or N = 0 launches nothing.
 * Scratch holds split-K partial sums (fp32 D only). */
size_t gpt2_op_matmul_scratch(int dtype, int M, int N, int K, int d_fp32);
int gpt2_op_matmul(int dtype, void* D, int d_fp32, const void* A, int a_mn_major, const void* B,
                   int b_mn_major, const void* bias, int M, int N, int K, void* scratch,
                   size_t scratch_bytes, int* d_status, void* stream);

/* FP8 linear layer (the modded-nanogpt project page, "NanoGPT (124M) in 90
 * seconds", "How it works": FP8 for the MLP, the QKV projections and the
 * head), with per-tensor scaling to one of two 8-bit floating-point formats
 * (OCP 8-bit floating point):
 *   GPT2_FP8_E4M3  1 sign, 4 exponent bits (bias 7), 3 mantissa bits, largest
 *                  finite value fmax = 448 (weights and activations);
 *   GPT2_FP8_E5M2  1 sign, 5 exponent bits (bias 15), 2 mantissa bits,
 *                  largest finite value fmax = 57344 (gradients).
 *
 * gpt2_op_quantize_fp8: q[i] = fp8(x[i] * scales[0]) for n bf16 values x in
 * the given format, with scales[0] = fmax / amax and scales[1] = amax / fmax
 * written on the device (both 1 when amax = max |x| is 0); the product is
 * rounded to fp32, then to the nearest value of the format (ties to even),
 * saturating at +-fmax; a NaN stays NaN and does not enter amax. q: n bytes
 * (8-byte aligned), x 16-byte aligned, scales: 2 floats; scratch:
 * gpt2_op_quantize_fp8_scratch() bytes. An unknown format is GPT2_ERR_ARG.
 *
 * gpt2_op_matmul_fp8: D[M,N] (bf16, overwritten) = (A B^T)[m,n] *
 * a_scales[1] * b_scales[1] (+ bias[n], bf16, optional), A [M,K] and B [N,K]
 * FP8 codes row-major (B is the [out, in] weight), each in its own format
 * (an e5m2 gradient times an e4m3 weight, for instance), the scale arrays as
 * written by gpt2_op_quantize_fp8 (read on the device). tcgen05 tensor cores
 * (kind::f8f6f4, TMA-fed, fp32 accumulation in tensor memory). Needs K % 16
 * == 0 and N % 8 == 0, 16-byte aligned A, B, D and bias; an unknown format is
 * GPT2_ERR_ARG. */
#define GPT2_FP8_E4M3 0
#define GPT2_FP8_E5M2 1
size_t gpt2_op_quantize_fp8_scratch(void);
int gpt2_op_quantize_fp8(void* q, float* scales, const void* x, int64_t n, int format, void* scratch,
                         size_t scratch_bytes, void* stream);
int gpt2_op_matmul_fp8(void* D, const void* A, int a_format, const float* a_scales, const void* B, int b_format,
                       const float* b_scales, const void* bias, int M, int N, int K, int* d_status, void* stream);

/* The codes of x [R][C] (bf16, row-major, C % 8 == 0, 16-byte aligned) under
 * the scales of an earlier gpt2_op_quantize_fp8 of the same values (scales[0]
 * multiplies, as there), written transposed to qt [C][R] and, when q is not
 * null, also as they are to q [R][C]: the same codes gpt2_op_quantize_fp8
 * gives, in the K-major layout the weight-gradient and input-gradient
 * products of an FP8 linear layer read. */
int gpt2_op_quantize_fp8_transpose(void* qt, void* q, const float* scales, const void* x, int R, int C,
                                   int format, void* stream);

/* The general FP8 product: epi 0: D[M,N] = (A B^T) a_scales[1] b_scales[1]
 * (+ bias), in bf16 or (d_fp32) fp32, accumulate (fp32 only): D += instead;
 * epi 1 (the MLP's first linear and its GELU): u = that product + bias
 * rounded to bf16, D = gelu'(u), D2 = gelu(u) (bf16); epi 2 (the input
 * gradient through the GELU): D = bf16(A B^T scales) * aux[m,n] (aux bf16
 * [M,N]). A [M,K], B [N,K] FP8 codes, K-major, K % 16 == 0, N % 8 == 0;
 * scratch: gpt2_op_matmul_fp8_scratch(M, N, K, d_fp32, accumulate) bytes
 * (split-K partial tiles of an fp32 product). */
size_t gpt2_op_matmul_fp8_scratch(int M, int N, int K, int d_fp32, int accumulate);
int gpt2_op_matmul_fp8_ex(int epi, void* D, void* D2, const void* aux, int d_fp32, int accumulate, const void* A,
                          int a_format, const float* a_scales, const void* B, int b_format, const float* b_scales,
                          const void* bias, int M, int N, int K, void* scratch, size_t scratch_bytes, int* d_status,
                          void* stream);

/* Linear forward with the GELU after it fused into the GEMM epilogue (the
 * MLP's first linear, "matmul_forward", followed by "gelu_forward" in the
 * kernel table): u = A W^T + bias (A [M,K], W [N,K] row-major, bias [N]
 * optional), rounded to dtype; out = gelu(u) with the tanh-approximation
 * GELU of gpt2_op_gelu_forward, and dgelu = gelu'(u), the factor the
 * backward needs (the backward of the step uses nothing else of u). Both
 * outputs [M,N] in dtype, overwritten, not overlapping. bf16: one
 * tensor-core GEMM whose epilogue writes both; fp32: the fp32 GEMM (into
 * dgelu) then one elementwise pass. Same shape and alignment rules as
 * gpt2_op_matmul. */
int gpt2_op_matmul_gelu(int dtype, void* dgelu, void* out, const void* A, const void* W,
                        const void* bias, int M, int N, int K, int* d_status, void* stream);

/* The input gradient of that GELU's input, fused ("gelu_backward" of the
 * kernel table folded into the preceding "matmul_backward"): du[M,N] =
 * (dY W)[m,n] * dgelu[m,n] with dY [M,K], W [K,N] row-major (the weight of
 * the linear that read gelu(u)) and dgelu from gpt2_op_matmul_gelu; the
 * product dY W is rounded to dtype before the multiply. du overwritten, in
 * dtype; it may not overlap dgelu. */
int gpt2_op_matmul_gelu_backward(int dtype, void* du, const void* dY, const void* W,
                                 const void* dgelu, int M, int N, int K, int* d_status,
                                 void* stream);

/* The same, and the bias gradient of the linear whose output gradient du is
 * ("matmul_backward"'s bias part): dbias[n] = sum over m of du[m,n], fp32
 * [N], overwritten, summed from the values as stored in du. bf16: the sums
 * of each 32-row slice are formed in the matmul's epilogue and reduced by a
 * second launch; fp32: a separate column-sum pass over du. scratch: at least
 * gpt2_op_matmul_gelu_backward_bias_scratch(M, N) bytes (else
 * GPT2_ERR_WORKSPACE). */
size_t gpt2_op_matmul_gelu_backward_bias_scratch(int M, int N);
int gpt2_op_matmul_gelu_backward_bias(int dtype, void* du, float* dbias, const void* dY,
                                      const void* W, const void* dgelu, int M, int N, int K,
                                      void* scratch, size_t scratch_bytes, int* d_status,
                                      void* stream);

/* Causal multi-head attention forward ("flash attention", section "Single
 * GPU training"; kernel "cudnn_generated_fort_native_sdpa"): qkv [B*T, 3C]
 * holds q | k | v column blocks, head h at columns h*hd..h*hd+hd-1 of each.
 * o [B*T, C] (dtype) = softmax(q k^T / sqrt(hd), causal) v per head; lse
 * [B, H, T] fp32 = log-sum-exp of each scaled score row. The T x T score
 * matrix is never stored. hd == 64 for bf16; hd <= 64 for fp32. */
int gpt2_op_attention_forward(int dtype, void* o, float* lse, const void* qkv, int B, int T,
                              int C, int H, void* stream);

/* Attention backward (kernels "compute_dot_do_o", the SDPA backward and
 * "rearrange_n_convert_dq" of the table): D = rowsum(dO * O) into scratch,
 * then with P recomputed from lse: dV = P^T dO, dS = P (dO V^T - D),
 * dQ = dS K / sqrt(hd), dK = dS^T Q / sqrt(hd), written to dqkv [B*T, 3C]
 * (dtype, overwritten) in the q | k | v layout. Deterministic (no atomics). */
size_t gpt2_op_attention_backward_scratch(int B, int T, int H);
int gpt2_op_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv,
                               const void* o, const float* lse, int B, int T, int C, int H,
                               void* scratch, size_t scratch_bytes, void* stream);

/* GELU, tanh form ("gelu_forward"): g = 0.5 u (1 + tanh(sqrt(2/pi)(u + 0.044715 u^3))).
 * n % 8 == 0. In place (g == u) is allowed. */
int gpt2_op_gelu_forward(int dtype, void* g, const void* u, int64_t n, void* stream);

/* GELU backward ("gelu_backward"): du = dg * g'(u). In place (du == dg) allowed. */
int gpt2_op_gelu_backward(int dtype, void* du, const void* u, const void* dg, int64_t n,
                          void* stream);

/* Residual forward ("residual_forward"): out = a + b, n % 8 == 0. */
int gpt2_op_residual_forward(int dtype, void* out, const void* a, const void* b, int64_t n,
                             void* stream);

/* Residual backward: the gradient reaching a residual join from the
 * branch is added to the stream gradient, dres += dbranch, n % 8 == 0.
 * llm.c's kernel table has no row of its own for it (the step folds it into
 * the LayerNorm backward, gpt2_op_layernorm_backward_residual). */
int gpt2_op_residual_backward(int dtype, void* dres, const void* dbranch, int64_t n,
                              void* stream);

/* Bias gradient ("matmul_backward_bias"): dbias[c] = sum_rows dy[r, c]
 * (fp32, overwritten), dy [N, C] dtype; deterministic two-stage reduction. */
size_t gpt2_op_bias_backward_scratch(int N, int C);
int gpt2_op_bias_backward(int dtype, float* dbias, const void* dy, int N, int C, void* scratch,
                          size_t scratch_bytes, void* stream);

/* Bias gradient without caller scratch (no counterpart on the pages; in
 * place of a citation: an addition of this library). It serves callers that
 * cannot allocate or lend device memory (for example a program whose device memory is wholly owned by
 * another runtime's allocator or a fixed pool, or code that must not call
 * cudaMalloc because it can synchronise the device). It computes exactly
 * what gpt2_op_bias_backward computes, dbias[c] = sum_rows dy[r, c] (fp32,
 * overwritten), but its partial sums go to a fixed 4 MiB array inside the
 * library instead of caller scratch. It calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *   - Limit: ceil(N/128) * C <= 1,048,576 (e.g. N = 32768 rows with
 *     C <= 4096). Larger sizes return GPT2_ERR_WORKSPACE and launch nothing.
 *   - The array is held by every GPU that loads the library until the
 *     process exits. The first call on each device looks up its device
 *     address (cudaGetSymbolAddress) with that device current; make that
 *     first call before any stream capture.
 *   - All calls share the one array. Calls that overlap on the GPU (on
 *     different streams, or from several threads) race and give wrong
 *     results; order them on one stream. Nothing in the array needs to
 *     start at zero: each call writes every partial it reads.
 * Arguments as gpt2_op_bias_backward, without the scratch. */
int gpt2_op_bias_backward_noalloc(int dtype, float* dbias, const void* dy, int N, int C,
                                  void* stream);

/* Fused classifier ("fused_classifier", section "Single GPU training" and
 * "Fine print"): per row i of logits [N, Vp] (dtype), over columns j < V only:
 * lse_i = log sum exp z_ij, losses[i] = lse_i - z_i,targets[i] (fp32), and in
 * place z_ij <- dloss * (exp(z_ij - lse_i) - [j == target_i]) for j < V,
 * 0 for V <= j < Vp. Normalised logits are never stored. dloss is the
 * gradient of the loss w.r.t. each row's loss (1/N for a mean).
 * A target outside [0,V) sets bit 4 of *d_status and is treated as 0. */
int gpt2_op_classifier(int dtype, void* logits, float* losses, const int32_t* targets, int N,
                       int V, int Vp, float dloss, int* d_status, void* stream);

/* Mean of losses [N] into *out (device fp32): fixed-order tree, deterministic.
 * The mean loss of the forward with targets (llm.c "State of the Union",
 * "Single GPU training"). */
int gpt2_op_mean_loss(float* out, const float* losses, int N, void* stream);

/* AdamW ("adamw_kernel"): over n fp32 elements, m = b1 m + (1-b1) g;
 * v = b2 v + (1-b2) g^2; theta -= lr (m/(1-b1^t) / (sqrt(v/(1-b2^t)) + eps)
 * + wd theta); if param_bf16 != NULL also writes bf16(theta) (round to
 * nearest even) there. n % 4 == 0. */
int gpt2_op_adamw(float* master, void* param_bf16, const float* grad, float* m, float* v,
                  int64_t n, float lr, float beta1, float beta2, float eps, float weight_decay,
                  int t, void* stream);

/* Failure-path testing of the bounded device waits (the design's failure
 * detection: a wait that runs out sets a status bit and the kernel returns;
 * nothing traps or hangs).
 * gpt2_debug_set_wait_limit: the bound, in SM clock cycles, of every
 * mbarrier wait of the tensor-core GEMM, the attention kernels and the
 * classifier on the current device; cycles <= 0 restores the default
 * (about 2 s). Takes effect for kernels launched after it returns; must not
 * be called while such kernels run.
 * gpt2_debug_stall_matmul: on != 0 makes every tensor-core GEMM launched
 * afterwards on the current device wait, before its first product, on a
 * barrier that nothing arrives at. The wait runs out after the bound above;
 * the kernel then sets the timeout bit (2) of its status word, stops its
 * other warps, waits (bounded) for its copies in flight, frees its tensor
 * memory and returns, leaving its output unwritten; the model's calls
 * report GPT2_ERR_TIMEOUT. on = 0 restores normal operation.
 * Both return GPT2_OK or GPT2_ERR_CUDA. Test hooks, not for the hot path. */
int gpt2_debug_set_wait_limit(int64_t cycles);
int gpt2_debug_stall_matmul(int on);

/* gpt2_debug_matmul_pair: on = 1 (the default) routes the plain bf16
 * matmuls with M >= 512 and one k-range per tile (no GELU epilogue) to the
 * CTA-pair kernel when N >= 1024, or when N is 384 to 960, a multiple of 192,
 * and K is 2048 to 16384 (192-wide pair tiles); the pair kernel issues one M = 256
 * tensor-core product for two neighbouring SMs (tcgen05 .cta_group::2) so
 * that each SM loads half of the B tile; on = 2 routes the GELU and GELU-gradient matmuls of that size there
 * too; 0 keeps every matmul on the one-CTA kernel. Process-wide; takes effect
 * for matmuls launched after it returns (a captured step graph keeps the
 * kernels it was captured with); on > 2 also sets the number of two-CTA
 * clusters launched (else the number the device keeps resident). Returns
 * the number of clusters the pair kernel launches (on != 0) or 0. A switch
 * for measurements and tests, not needed in normal use. */
int gpt2_debug_matmul_pair(int on);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_OPS_H */
