// Launch helpers for the split-KV attention kernel: per KV encoding and head
// dimension, the instantiations with rows or tokens on the MMA M axis, for
// whole blocks (launch_attn), for blocks handled as several work pages
// (launch_attn_split) and for work pages of several blocks (launch_attn_merged,
// for short rows only), compiled in separate translation units.
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
template <int KVT, int D>
cudaError_t launch_attn_merged(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid,
                               size_t smem, bool tokens_as_m, cudaStream_t s);

// Merged work pages are built for K/V rows of at most 64 bytes (INT4 at D=128,
// 8-bit codes at D=64): one swizzle line per row, and pages small enough that
// the per-page work dominates.  The host merges only these shapes.
__host__ __device__ constexpr bool merge_rows(int row_bytes) { return row_bytes <= 64; }

template <int KVT, int D, bool TOKM, int WM>
cudaError_t launch_attn_t(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid, size_t smem,
                          cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(pa_attn_kernel<KVT, D, TOKM, WM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(pa_attn_kernel<KVT, D, TOKM, WM>, grid, dim3(ATTN_THREADS), smem, s, tk, tv, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int KVT, int D, bool OK = merge_rows(Geo<KVT, D>::RB)>
struct MergedLaunch {
    static cudaError_t go(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P, dim3 grid, size_t smem,
                          bool tokens_as_m, cudaStream_t s) {
        return tokens_as_m ? launch_attn_t<KVT, D, true, WP_MERGED>(tk, tv, P, grid, smem, s)
                           : launch_attn_t<KVT, D, false, WP_MERGED>(tk, tv, P, grid, smem, s);
    }
};
template <int KVT, int D>
struct MergedLaunch<KVT, D, false> {  // never chosen by the host for these shapes
    static cudaError_t go(const CUtensorMap &, const CUtensorMap &, const AttnParams &, dim3, size_t, bool,
                          cudaStream_t) {
        return cudaErrorNotSupported;
    }
};

#define PA_DEFINE_ATTN(KVT, D)                                                                                  \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s) {                 \
        return tokens_as_m ? launch_attn_t<KVT, D, true, WP_WHOLE>(tk, tv, P, grid, smem, s)                    \
                           : launch_attn_t<KVT, D, false, WP_WHOLE>(tk, tv, P, grid, smem, s);                  \
    }

#define PA_DEFINE_ATTN_SPLIT(KVT, D)                                                                            \
    template <>                                                                                                 \
    cudaError_t launch_attn_split<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,    \
                                          dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s) {           \
        return tokens_as_m ? launch_attn_t<KVT, D, true, WP_PART>(tk, tv, P, grid, smem, s)                     \
                           : launch_attn_t<KVT, D, false, WP_PART>(tk, tv, P, grid, smem, s);                   \
    }

#define PA_DEFINE_ATTN_MERGED(KVT, D)                                                                           \
    template <>                                                                                                 \
    cudaError_t launch_attn_merged<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,   \
                                           dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s) {          \
        return MergedLaunch<KVT, D>::go(tk, tv, P, grid, smem, tokens_as_m, s);                                 \
    }

#define PA_DECLARE_ATTN(KVT, D)                                                                                 \
    template <>                                                                                                 \
    cudaError_t launch_attn<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,          \
                                    dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s);                  \
    template <>                                                                                                 \
    cudaError_t launch_attn_split<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,    \
                                          dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s);           \
    template <>                                                                                                 \
    cudaError_t launch_attn_merged<KVT, D>(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &P,   \
                                           dim3 grid, size_t smem, bool tokens_as_m, cudaStream_t s);

PA_DECLARE_ATTN(PA_F16, 64) PA_DECLARE_ATTN(PA_F16, 128) PA_DECLARE_ATTN(PA_F16, 256)
PA_DECLARE_ATTN(PA_BF16, 64) PA_DECLARE_ATTN(PA_BF16, 128) PA_DECLARE_ATTN(PA_BF16, 256)
PA_DECLARE_ATTN(PA_E4M3, 64) PA_DECLARE_ATTN(PA_E4M3, 128) PA_DECLARE_ATTN(PA_E4M3, 256)
PA_DECLARE_ATTN(PA_INT8, 64) PA_DECLARE_ATTN(PA_INT8, 128) PA_DECLARE_ATTN(PA_INT8, 256)
PA_DECLARE_ATTN(PA_INT4, 128) PA_DECLARE_ATTN(PA_INT4, 256)

}  // namespace pa
