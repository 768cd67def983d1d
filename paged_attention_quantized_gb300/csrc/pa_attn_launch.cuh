// Launch helpers for the split-KV attention kernel (one instantiation per KV
// encoding and head dimension, compiled in separate translation units).
#pragma once

#include <algorithm>

#include "pa_attn.cuh"

namespace pa {

// dynamic shared memory of one CTA: alignment slack, the stage ring, the q'
// fragments, the merge buffer, row constants and the stage barriers
inline size_t attn_smem_bytes(int D, int stages, int stage_bytes) {
    const size_t misc = (sizeof(SmemMisc) + 15) & ~size_t(15);
    // the merge buffer [ROWS][D] fp32 lives in the ring after the last page
    const size_t ring = std::max((size_t)stages * stage_bytes, (size_t)ROWS * D * 4);
    return 1024 + ring + (size_t)(D / 16) * 512 + misc + 2 * MAX_STAGES * sizeof(uint64_t);
}

template <int KVT, int D>
cudaError_t launch_attn(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid, size_t smem,
                        cudaStream_t s);

#define PA_DEFINE_ATTN(KVT, D)                                                                                  \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, cudaStream_t s) {                                   \
        cudaError_t e = cudaFuncSetAttribute(pa_attn_kernel<KVT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                             (int)smem);                                                        \
        if (e != cudaSuccess) return e;                                                                         \
        pa_attn_kernel<KVT, D><<<grid, ATTN_THREADS, smem, s>>>(tk, tv, P);                                     \
        return cudaGetLastError();                                                                              \
    }

#define PA_DECLARE_ATTN(KVT, D)                                                                                 \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, cudaStream_t s);

PA_DECLARE_ATTN(PA_F16, 64) PA_DECLARE_ATTN(PA_F16, 128) PA_DECLARE_ATTN(PA_F16, 256)
PA_DECLARE_ATTN(PA_BF16, 64) PA_DECLARE_ATTN(PA_BF16, 128) PA_DECLARE_ATTN(PA_BF16, 256)
PA_DECLARE_ATTN(PA_E4M3, 64) PA_DECLARE_ATTN(PA_E4M3, 128) PA_DECLARE_ATTN(PA_E4M3, 256)
PA_DECLARE_ATTN(PA_INT8, 64) PA_DECLARE_ATTN(PA_INT8, 128) PA_DECLARE_ATTN(PA_INT8, 256)
PA_DECLARE_ATTN(PA_INT4, 128) PA_DECLARE_ATTN(PA_INT4, 256)

}  // namespace pa
