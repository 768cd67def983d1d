// Launch helpers for the split-KV attention kernel (one pair of instantiations
// -- rows or tokens on the MMA M axis -- per KV encoding and head dimension,
// compiled in separate translation units).
#pragma once

#include <algorithm>

#include "pa_attn.cuh"

namespace pa {

template <int KVT, int D>
cudaError_t launch_attn(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid, size_t smem,
                        bool tokens_as_m, cudaStream_t s);

template <int KVT, int D, bool TOKM>
cudaError_t launch_attn_t(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid, size_t smem,
                          cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(pa_attn_kernel<KVT, D, TOKM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(pa_attn_kernel<KVT, D, TOKM>, grid, dim3(ATTN_THREADS), smem, s, tk, tv, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

#define PA_DEFINE_ATTN(KVT, D)                                                                                  \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s) {                 \
        return tokens_as_m ? launch_attn_t<KVT, D, true>(tk, tv, P, grid, smem, s)                              \
                           : launch_attn_t<KVT, D, false>(tk, tv, P, grid, smem, s);                            \
    }

#define PA_DECLARE_ATTN(KVT, D)                                                                                 \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s);

PA_DECLARE_ATTN(PA_F16, 64) PA_DECLARE_ATTN(PA_F16, 128) PA_DECLARE_ATTN(PA_F16, 256)
PA_DECLARE_ATTN(PA_BF16, 64) PA_DECLARE_ATTN(PA_BF16, 128) PA_DECLARE_ATTN(PA_BF16, 256)
PA_DECLARE_ATTN(PA_E4M3, 64) PA_DECLARE_ATTN(PA_E4M3, 128) PA_DECLARE_ATTN(PA_E4M3, 256)
PA_DECLARE_ATTN(PA_INT8, 64) PA_DECLARE_ATTN(PA_INT8, 128) PA_DECLARE_ATTN(PA_INT8, 256)
PA_DECLARE_ATTN(PA_INT4, 128) PA_DECLARE_ATTN(PA_INT4, 256)

}  // namespace pa
