// Launch helpers for the split-KV attention kernel: per KV encoding and head
// dimension, the instantiations with rows or tokens on the MMA M axis, for
// whole blocks (launch_attn) and for blocks handled as several work pages
// (launch_attn_split), compiled in separate translation units.
#pragma once

#include <algorithm>

#include "pa_attn.cuh"

namespace pa {

template <int KVT, int D>
cudaError_t launch_attn(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid, size_t smem,
                        bool tokens_as_m, cudaStream_t s);
template <int KVT, int D>
cudaError_t launch_attn_split(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid,
                              size_t smem, bool tokens_as_m, cudaStream_t s);

template <int KVT, int D, bool TOKM, bool SPLIT>
cudaError_t launch_attn_t(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid, size_t smem,
                          cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(pa_attn_kernel<KVT, D, TOKM, SPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(pa_attn_kernel<KVT, D, TOKM, SPLIT>, grid, dim3(ATTN_THREADS), smem, s, tk, tv, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

#define PA_DEFINE_ATTN(KVT, D)                                                                                  \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s) {                 \
        return tokens_as_m ? launch_attn_t<KVT, D, true, false>(tk, tv, P, grid, smem, s)                       \
                           : launch_attn_t<KVT, D, false, false>(tk, tv, P, grid, smem, s);                     \
    }

#define PA_DEFINE_ATTN_SPLIT(KVT, D)                                                                            \
    template <>                                                                                                 \
    cudaError_t launch_attn_split<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,    \
                                          dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s) {           \
        return tokens_as_m ? launch_attn_t<KVT, D, true, true>(tk, tv, P, grid, smem, s)                        \
                           : launch_attn_t<KVT, D, false, true>(tk, tv, P, grid, smem, s);                      \
    }

#define PA_DECLARE_ATTN(KVT, D)                                                                                 \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s);                  \
    template <>                                                                                                 \
    cudaError_t launch_attn_split<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,    \
                                          dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s);

PA_DECLARE_ATTN(PA_F16, 64) PA_DECLARE_ATTN(PA_F16, 128) PA_DECLARE_ATTN(PA_F16, 256)
PA_DECLARE_ATTN(PA_BF16, 64) PA_DECLARE_ATTN(PA_BF16, 128) PA_DECLARE_ATTN(PA_BF16, 256)
PA_DECLARE_ATTN(PA_E4M3, 64) PA_DECLARE_ATTN(PA_E4M3, 128) PA_DECLARE_ATTN(PA_E4M3, 256)
PA_DECLARE_ATTN(PA_INT8, 64) PA_DECLARE_ATTN(PA_INT8, 128) PA_DECLARE_ATTN(PA_INT8, 256)
PA_DECLARE_ATTN(PA_INT4, 128) PA_DECLARE_ATTN(PA_INT4, 256)

}  // namespace pa
