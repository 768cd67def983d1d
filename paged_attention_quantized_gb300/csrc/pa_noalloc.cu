// pa_attention_noalloc: the whole attention (plan, split-KV run, combine) for
// callers that cannot allocate device memory -- for example a plugin whose
// host application hands it only its input and output buffers and owns every
// allocation itself.  The
// scratch that pa_attention keeps in a caller-owned workspace (plan records,
// split partials, the device error word) lives here instead in one static
// device array, reserved on every GPU that loads this library until the
// process exits.
#include <mutex>

#include "pa.h"
#include "pa_common.cuh"

namespace {

// Largest workspace this entry point can serve.
constexpr size_t NOALLOC_SCRATCH_BYTES = 32u << 20;  // 32 MiB

// The scratch itself.  In host code `pa_noalloc_scratch` is only a host-side
// stand-in for the symbol, never a device address: kernels get the address
// from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t pa_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_lock;
void *g_scratch[MAX_DEVICES] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and kept for the life of the process; a
// cudaDeviceReset makes the kept address stale (the header says so).
pa_status scratch_address(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_lock);
    if (g_scratch[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, pa_noalloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        g_scratch[dev] = p;
    }
    *ptr = g_scratch[dev];
    return PA_OK;
}

}  // namespace

extern "C" PA_API pa_status pa_attention_noalloc(const pa_problem *p, const void *q, const void *k_pool,
                                                 const void *v_pool, const int32_t *block_table,
                                                 const int32_t *context_lens, const float *k_scale,
                                                 const float *v_scale, void *out, float *lse,
                                                 pa_stream_t stream) {
    size_t need = 0;
    pa_status st = pa_workspace_size(p, &need);
    if (st != PA_OK) return st;
    if (need > NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((st = scratch_address(&scratch)) != PA_OK) return st;
    // Nothing in the scratch has to start at zero: pa_plan rewrites the header
    // (error word included) and every record that pa_run and pa_combine read.
    return pa_attention(p, q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale, scratch,
                        NOALLOC_SCRATCH_BYTES, out, lse, stream);
}
