// Launch helpers for the split-KV attention kernel (one instantiation per KV
// encoding and head dimension, compiled in separate translation units).
#pragma once

#include <algorithm>

#include "pa_attn.cuh"

namespace pa {

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
