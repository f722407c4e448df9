/*
 * gpt2.h - one GPT-2 training step (forward, backward, AdamW) on one GPU.
 *
 * The step is the one llm.c's "State of the Union [May 3, 2024]" describes
 * under "Single GPU training": GPT-2 trained in bfloat16 with a master copy
 * of the parameters kept in fp32, a fused classifier that takes the loss
 * only at the label's index and never stores normalised logits, flash-style
 * attention, and a vocabulary padded from 50257 to 50304 whose padded
 * columns are masked to -inf ("Fine print"). The kernel list it runs is the
 * one in that page's kernel table ("Runtime, DRAM traffic, instructions").
 *
 * Conventions for every call:
 *   - Returns GPT2_OK (0) or a negative gpt2_status. Nothing aborts, traps
 *     or prints; gpt2_strerror() names the status.
 *   - Device pointers are CUDA device addresses on the current device.
 *     Host pointers are ordinary process memory.
 *   - The caller owns the workspace (one device allocation of
 *     gpt2_workspace_bytes()), the token and target buffers and the CUDA
 *     stream. The library never allocates or frees device memory; the
 *     handle (host memory) is freed by gpt2_destroy().
 *   - All device work is enqueued on the stream given to gpt2_init().
 *     gpt2_forward() synchronises that stream once, to return the loss.
 */
#ifndef GPT2_H
#define GPT2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Model shape and arithmetic mode.
 *   n_layer L, n_embd C, n_head H (head size C/H), vocab V (real ids
 *   0..V-1), vocab_padded Vp >= V (rows V..Vp-1 of the embedding table are
 *   padding: initialised to 0, masked out of the softmax), max_T and max_B
 *   (largest sequence length and batch a forward may use), mode.
 * Constraints: C % 8 == 0, C % H == 0, Vp % 8 == 0; in bf16 mode the head
 * size is 64; in fp32 mode it is at most 64. */
typedef struct gpt2_config {
    int32_t n_layer;
    int32_t n_embd;
    int32_t n_head;
    int32_t vocab;
    int32_t vocab_padded;
    int32_t max_T;
    int32_t max_B;
    int32_t mode;
} gpt2_config;

/* mode: GPT2_MODE_BF16 = bf16 activations and GEMM operands, fp32
 * accumulation, fp32 master weights, gradients and moments (the pages'
 * mixed precision). GPT2_MODE_FP32 = every tensor fp32 with true fp32 FMA
 * (no TF32): the exact-parity mode. */
enum { GPT2_MODE_FP32 = 0, GPT2_MODE_BF16 = 1 };

typedef enum gpt2_status {
    GPT2_OK = 0,
    GPT2_ERR_ARG = -1,          /* bad config, size, pointer or hyper-parameter */
    GPT2_ERR_STATE = -2,        /* calls out of order (e.g. backward before forward) */
    GPT2_ERR_TOKEN_RANGE = -3,  /* a token or target id outside [0, V): found on the device */
    GPT2_ERR_NONFINITE = -4,    /* the mean loss is NaN or Inf */
    GPT2_ERR_TIMEOUT = -5,      /* a bounded device-side wait gave up */
    GPT2_ERR_CUDA = -6,         /* a CUDA runtime call failed */
    GPT2_ERR_WORKSPACE = -7     /* workspace too small or misaligned (needs 1024-byte alignment) */
} gpt2_status;

/* Which copy gpt2_copy_tensor() reads. */
enum {
    GPT2_TENSOR_PARAM = 0,  /* the compute copy: bf16 in bf16 mode (returned widened to fp32), else the master */
    GPT2_TENSOR_MASTER = 1, /* fp32 master weights */
    GPT2_TENSOR_GRAD = 2,   /* fp32 gradient of the last backward */
    GPT2_TENSOR_ADAM_M = 3, /* fp32 first moment */
    GPT2_TENSOR_ADAM_V = 4  /* fp32 second moment */
};

typedef struct gpt2 gpt2_t;

/* Bytes of device workspace a model of this config needs (parameters,
 * gradients, AdamW moments, saved activations for max_B x max_T, backward
 * scratch). Host-only; touches no device. */
int gpt2_workspace_bytes(const gpt2_config* cfg, size_t* bytes_out);

/* Create a model in the caller's workspace and initialise it from `seed`:
 * wte, wpe and every weight matrix ~ N(0, 0.02); the two residual
 * projections of each layer ~ N(0, 0.02/sqrt(2L)); biases 0; LayerNorm gain
 * 1 and bias 0; padded wte rows 0 ("init from random weights direct in C",
 * section "Functional"). Draws are counter-based (splitmix64 + Box-Muller,
 * element i of tensor k from counter k*2^40 + i), made on the host and
 * copied once. AdamW moments start at 0.
 * d_workspace: device, >= gpt2_workspace_bytes, 1024-byte aligned; it must
 * stay valid until gpt2_destroy(). cuda_stream: a cudaStream_t (NULL = the
 * legacy default stream). */
int gpt2_init(gpt2_t** out, const gpt2_config* cfg, uint64_t seed, void* d_workspace,
              size_t workspace_bytes, void* cuda_stream);

/* Forward pass on tokens [B, T] (device int32, row-major): the forward rows
 * of llm.c's kernel table ("State of the Union", "Runtime, DRAM traffic,
 * instructions": encoder_forward, layernorm_forward, the matmuls, attention,
 * gelu_forward, residual_forward, fused_classifier). With targets
 * (device int32 [B, T]) it also runs the fused classifier: per-position
 * loss at the label index, dlogits written in place over the logits, and
 * writes the mean loss over the B*T positions to *loss_out (host float) after
 * one stream synchronisation. targets == NULL computes only the logits
 * (loss_out may then be NULL) and does not synchronise.
 * 1 <= B <= max_B, 1 <= T <= max_T. Ids outside [0, V) give
 * GPT2_ERR_TOKEN_RANGE (the kernels clamp them, so no memory is touched
 * out of bounds). */
int gpt2_forward(gpt2_t* m, const int32_t* d_tokens, const int32_t* d_targets, int B, int T,
                 float* loss_out);

/* Backward pass of the last forward (which must have had targets): the
 * backward rows of the same kernel table (matmul and bias backward,
 * gelu_backward, layernorm_backward, attention backward,
 * encoder_backward).
 * Overwrites every parameter gradient, or adds to them after
 * gpt2_set_grad_accumulation(m, 1). */
int gpt2_backward(gpt2_t* m);

/* One AdamW step on every parameter tensor from the last backward's
 * gradients (the kernel table's adamw row; "Single GPU training": the
 * parameter master copy kept in fp32): m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
 * theta -= lr (m/(1-b1^t) / (sqrt(v/(1-b2^t)) + eps) + weight_decay theta),
 * then the bf16 copy is refreshed (bf16 mode). t >= 1 is the 1-based step.
 * Weight decay applies to every tensor. */
int gpt2_adamw_step(gpt2_t* m, float lr, float beta1, float beta2, float eps,
                    float weight_decay, int t);

/* ---- the training loop around the step (gradient accumulation, clipping,
 * decay mask, learning-rate schedule) ---- */

/* accumulate = 1: every following gpt2_backward adds its gradients to the ones
 * held (each micro-batch contributes the gradient of its own mean loss);
 * accumulate = 0 (the default): each backward overwrites them. Start an
 * accumulation with gpt2_zero_grad(). Host-only; takes effect at the next
 * backward. */
int gpt2_set_grad_accumulation(gpt2_t* m, int accumulate);

/* Set every parameter gradient to 0 (enqueued on the model's stream). */
int gpt2_zero_grad(gpt2_t* m);

/* ---- FP8 linear layers (the modded-nanogpt project page, "NanoGPT (124M)
 * in 90 seconds", "How it works": FP8 for the MLP forward and backward
 * passes, the QKV projections and the head) ----
 *
 * mask: GPT2_FP8_QKV (the QKV projection), GPT2_FP8_MLP (both MLP linears),
 * GPT2_FP8_HEAD (the tied LM head), OR-ed; 0 (the default) keeps every
 * matmul in bf16. In a selected linear all three products (output, input
 * gradient, weight gradient) take FP8 operands on the tensor cores
 * (tcgen05 kind::f8f6f4, fp32 accumulation): activations and weights in
 * e4m3, the output gradient in e5m2, each tensor with its own per-tensor
 * scale fmax / amax taken just before the product (the forward's codes of x
 * and scale of W also serve the backward, whose operands are the same
 * tensors). The workspace keeps each selected linear's transposed input
 * codes from the forward to the backward (B*T x its input width bytes).
 * Outputs stay bf16 (fp32 for weight gradients), biases, GELU and the bias
 * gradients as in the bf16 step. bf16 mode only (else GPT2_ERR_ARG); B*T
 * must then be a multiple of 16 (gpt2_forward returns GPT2_ERR_ARG
 * otherwise).
 *
 * gpt2_fp8_workspace_bytes: the size of the second device workspace the
 * FP8 codes need (0 for mask 0); gpt2_set_fp8 takes it (1024-byte aligned,
 * owned by the caller, not needed with mask 0) and the mask. The next
 * gpt2_forward starts a new step; gpt2_step recaptures its graph. */
#define GPT2_FP8_QKV 1
#define GPT2_FP8_MLP 2
#define GPT2_FP8_HEAD 4
#define GPT2_FP8_ALL 7
int gpt2_fp8_workspace_bytes(const gpt2_config* cfg, int mask, size_t* bytes_out);
int gpt2_set_fp8(gpt2_t* m, int mask, void* d_workspace, size_t workspace_bytes);

/* ||g||_2 over all parameter gradients (fp32, deterministic two-stage sum),
 * kept on the device; if norm_out is not NULL it is also written there after
 * one stream synchronisation. */
int gpt2_grad_norm(gpt2_t* m, float* norm_out);

/* AdamW with the usual training-loop options. lr ... t as for
 * gpt2_adamw_step. grad_scale > 0 multiplies every gradient first (e.g. 1/n
 * after accumulating n micro-batches). max_grad_norm > 0 clips by the global
 * norm: g *= min(1, max_grad_norm / (||g grad_scale|| + 1e-6)), the norm
 * computed on the device (no host synchronisation); 0 disables clipping.
 * decay_mask = 1 applies weight_decay only to the 2-D tensors (wte, wpe and
 * the weight matrices) and not to biases and LayerNorm parameters; 0 applies
 * it to every tensor. With grad_scale 1, max_grad_norm 0 and decay_mask 0 this
 * is gpt2_adamw_step. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int t;
    float grad_scale;
    float max_grad_norm;
    int decay_mask;
} gpt2_adamw_config;
int gpt2_adamw_step_ex(gpt2_t* m, const gpt2_adamw_config* cfg);

/* One whole training step (the step above: llm.c "State of the Union",
 * "Single GPU training"), replayed as a CUDA graph (the modded-nanogpt
 * project page, "How it works", lists CUDA-graph capture among its systems
 * techniques): tokens and targets
 * (device, int32 [B,T]) are copied into the library's own buffers, then the
 * forward to the mean loss, the backward, the global-norm clip when
 * cfg->max_grad_norm > 0 and AdamW run as one captured graph; the loss comes
 * back in *loss_out (the stream is synchronised once). The values of cfg
 * (lr, t, ...) are read by the device each step, so one graph serves every
 * step; it is captured again when B, T, gradient accumulation, the decay mask
 * or max_grad_norm change. The first step with new such settings, and every
 * step while per-op timing is on, run eagerly. The results equal
 * gpt2_forward, gpt2_backward and gpt2_adamw_step_ex bit for bit. Errors as
 * for those calls; on success the state is that after gpt2_adamw_step_ex. */
int gpt2_step(gpt2_t* m, const int32_t* d_tokens, const int32_t* d_targets, int B, int T,
              const gpt2_adamw_config* cfg, float* loss_out);

/* gpt2_step with the batch in HOST memory: h_tokens and h_targets (int32
 * [B,T], row-major, contiguous, owned by the caller) are copied to the
 * device by the call itself (cudaMemcpyAsync host to device on the model's
 * stream, before the step's graph), so a caller with data on the host makes
 * one call per step: 2*B*T*4 bytes go in, the 4-byte loss comes back. Page-
 * locked (pinned) host buffers make the copies asynchronous; pageable ones
 * work but are staged by the driver. The buffers may be reused once the call
 * returns. Same results, errors and state as gpt2_step. */
int gpt2_step_host(gpt2_t* m, const int32_t* h_tokens, const int32_t* h_targets, int B, int T,
                   const gpt2_adamw_config* cfg, float* loss_out);

/* ZeRO-1 style sharded update (llm.c "State of the Union", "Multi-GPU
 * training": optimizer state split over data-parallel ranks). AdamW as in
 * gpt2_adamw_step_ex, applied only to the elements [begin, begin + count) of
 * the flat parameter layout (master, moments, compute copy and gradient of
 * that range; gpt2_flat_params elements: the tensors in canonical order, each
 * starting on a 64-element boundary, the gaps zero and left zero by AdamW);
 * a rank that owns a shard calls it for its range, and calls over ranges that
 * tile [0, n) give, element for element, the values of one
 * gpt2_adamw_step_ex (the update is elementwise). begin is a multiple of
 * 2048, count a positive multiple of 4, begin + count <= n. Clipping needs the norm of
 * every shard's gradient: max_grad_norm must be 0 here, and a caller that
 * clips combines the shards' gpt2_grad_sumsq_range values into the clip
 * factor and passes it in grad_scale. Allowed after gpt2_backward and after
 * another shard call of the same step; GPT2_ERR_ARG / GPT2_ERR_STATE
 * otherwise. */
int gpt2_adamw_step_shard(gpt2_t* m, const gpt2_adamw_config* cfg, int64_t begin, int64_t count);

/* Length n of the flat parameter layout (with the alignment gaps). */
int64_t gpt2_flat_params(const gpt2_t* m);

/* Sum of squares of the gradient elements [begin, begin + count) (fp32,
 * deterministic order), written to *out (host); synchronises the stream.
 * begin and count multiples of 4, count >= 4, begin + count <= n. */
int gpt2_grad_sumsq_range(gpt2_t* m, int64_t begin, int64_t count, float* out);

/* Learning rate of step t (1-based): linear warmup to lr_max over `warmup`
 * steps, then a half-cosine from lr_max down to lr_min at step `total`, and
 * lr_min after it. Host-only. */
float gpt2_lr_cosine(int t, int warmup, int total, float lr_max, float lr_min);

/* Free the handle (not the workspace, which the caller owns). */
int gpt2_destroy(gpt2_t* m);

/* Static text for a status code. */
const char* gpt2_strerror(int status);

/* ---- inspection (tests, checkpointing); not on the training hot path ---- */

/* Number of parameter tensors, in canonical order: wte [Vp,C], wpe
 * [max_T,C]; per layer ln1.g, ln1.b, qkv.w [3C,C], qkv.b, proj.w [C,C],
 * proj.b, ln2.g, ln2.b, fc.w [4C,C], fc.b, fcproj.w [C,4C], fcproj.b; then
 * lnf.g, lnf.b. Weights use the [out, in] layout. */
int gpt2_num_tensors(const gpt2_t* m);

/* Name (static string owned by the handle) and shape of tensor i; a
 * vector has shape[1] == 1. */
int gpt2_tensor_info(const gpt2_t* m, int i, const char** name, int64_t shape[2]);

/* Copy one copy (GPT2_TENSOR_*) of tensor i to host_dst as fp32
 * (shape[0]*shape[1] floats). Synchronises the stream. */
int gpt2_copy_tensor(gpt2_t* m, int i, int kind, float* host_dst);

/* Overwrite the fp32 master of tensor i from host fp32 data and refresh
 * its compute copy. Synchronises the stream. */
int gpt2_load_tensor(gpt2_t* m, int i, const float* host_src);

/* Per-position losses [B*T] (fp32) of the last forward with targets.
 * Synchronises the stream. */
int gpt2_copy_losses(gpt2_t* m, float* host_dst);

/* Number of parameters (sum of tensor sizes, padded vocab rows included). */
int64_t gpt2_num_params(const gpt2_t* m);

/* ---- launch accounting and timing ---- */

/* Kernel families, for per-family launch counts and times. */
enum {
    GPT2_K_ENCODER_FWD = 0, GPT2_K_LAYERNORM_FWD, GPT2_K_MATMUL, GPT2_K_ATTENTION_FWD,
    GPT2_K_RESIDUAL_FWD, GPT2_K_GELU_FWD, GPT2_K_CLASSIFIER, GPT2_K_LOSS_MEAN,
    GPT2_K_LAYERNORM_BWD, GPT2_K_GELU_BWD, GPT2_K_BIAS_BWD, GPT2_K_ATTENTION_BWD,
    GPT2_K_RESIDUAL_BWD, GPT2_K_ENCODER_BWD, GPT2_K_ADAMW,
    GPT2_K_GRAD_COLSUM, /* the deferred column sums of the LayerNorm and bias gradients */
    GPT2_K_FP8_QUANT,   /* FP8 quantization of the FP8 linear layers' operands */
    GPT2_K_COUNT
};

/* Kernels launched by this handle so far (every launch, all families). */
int64_t gpt2_launch_count(const gpt2_t* m);

/* Per-family counters: op calls (one matmul or one LayerNorm backward is
 * one call, however many kernels it takes), kernel launches, and the
 * algorithmic work those calls did (FLOPs for matmul and attention, bytes
 * for the rest). Host-side, always on. */
int gpt2_family_stats(const gpt2_t* m, int family, int64_t* calls, int64_t* launches,
                      double* work);

/* Enable (1) or disable (0) CUDA-event timing of every op on the model's
 * stream. While enabled each op is bracketed by two events. */
int gpt2_set_timing(gpt2_t* m, int enable);

/* Synchronise the stream and return the summed device time (ms) of the
 * timed ops of one family since timing was enabled or last reset. */
int gpt2_family_time(gpt2_t* m, int family, double* ms);

/* Reset counters and accumulated times. */
int gpt2_reset_stats(gpt2_t* m);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_H */
