// Bias-gradient reduction that allocates nothing: its scratch is a
// file-scope device array instead of caller-provided memory.
//
// Some callers cannot hand this library a scratch buffer: for example a host
// program whose device memory is owned entirely by another runtime (a
// framework's caching allocator or a fixed memory pool that forbids side
// allocations), or code that must not call cudaMalloc because that call can
// synchronise the whole device. gpt2_op_bias_backward_noalloc serves them: the
// caller passes only the input and the output.
//
// The scratch below lives in every GPU that loads this library, from load
// until process exit. In host code the symbol is only a host-side stand-in,
// so its device address is fetched once per device with cudaGetSymbolAddress
// (on the first call made while that device is current) and passed to the
// kernels; host code never hands the symbol itself to a kernel.
#include "common.cuh"
#include "launch.h"

#include <mutex>

// 4 MiB: enough for ceil(N/128) * C <= 1,048,576 (e.g. N = 32768 rows with
// C <= 4096 columns).
#define NOALLOC_BIAS_SCRATCH_FLOATS (1 << 20)
#define NOALLOC_MAX_DEVICES 64

static __device__ __align__(256) float g_bias_scratch[NOALLOC_BIAS_SCRATCH_FLOATS];

namespace {

std::mutex g_mu;
float* g_scratch_addr[NOALLOC_MAX_DEVICES] = {};

// Device address of g_bias_scratch on the current device (looked up once).
int scratch_on_current_device(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GPT2_ERR_CUDA;
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return GPT2_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bias_scratch) != cudaSuccess || !p) return GPT2_ERR_CUDA;
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_addr[dev];
    return GPT2_OK;
}

}  // namespace

extern "C" int gpt2_op_bias_backward_noalloc(int dtype, float* dbias, const void* dy, int N, int C, void* stream) {
    if ((dtype != GPT2_MODE_FP32 && dtype != GPT2_MODE_BF16) || !dbias || !dy || N < 0 || C <= 0 || C % 8 ||
        ((uintptr_t)dy & 15u))
        return GPT2_ERR_ARG;
    const size_t need = bias_backward_scratch(N, C);
    if (need > sizeof(g_bias_scratch)) return GPT2_ERR_WORKSPACE;  // larger than the fixed scratch
    cudaStream_t s = (cudaStream_t)stream;
    if (N == 0) return cudaMemsetAsync(dbias, 0, (size_t)C * 4, s) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
    float* scratch = nullptr;
    const int r = scratch_on_current_device(&scratch);
    if (r != GPT2_OK) return r;
    // Every partial sum the reduction reads is written first by the same
    // call, so nothing in the scratch has to start at zero.
    const int launches = launch_bias_backward(dtype, dbias, dy, N, C, scratch, s);
    if (launches < 0) return launches;
    return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}
