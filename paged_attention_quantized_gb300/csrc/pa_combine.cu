// Split-KV merge for paged attention (sm_103a).
//
// Every segment (request, kv head, block of 16 -- or, for the latent kernel,
// 64 -- query rows) whose pages were shared by several workers (warps, or
// CTAs of the latent kernel) has one normalised partial output o_s and
// log-sum-exp lse_s per worker; they are merged in ascending position order:
//     M = max_s lse_s,  w_s = exp(lse_s - M),
//     out = (sum_s w_s o_s) / (sum_s w_s) * v_scale,   lse = M + ln(sum_s w_s)
// (the pages name split "partial" kernels -- 1Cat-vLLM PR #647, Fix -- and
// leave the merge to the standard log-sum-exp identity).  A NaN partial (a
// unit that found a contract violation) makes the row NaN.  The order is
// fixed, so the result is bitwise reproducible.
#include "pa_common.cuh"

namespace pa {

constexpr int COMBINE_THREADS = 256;

// first position of warp k's share of the n positions split over nw warps
__device__ __forceinline__ long long share_start(long long k, long long n, long long nw) { return k * n / nw; }

// the warp whose share holds position x (the last k with share_start <= x)
__device__ __forceinline__ long long share_owner(long long x, long long n, long long nw) {
    return ((x + 1) * nw + n - 1) / n - 1;
}

constexpr int MAX_CACHED_PIECES = 64;
constexpr int MAX_ROWS_SEG = 64;

// One CTA per segment (request, kv head, row block).  The pieces (non-empty
// warp shares) and the per-row weights w = exp(lse - M) / sum exp(lse - M) are
// worked out once; every output element is then one weighted sum.
__global__ void __launch_bounds__(COMBINE_THREADS) pa_combine_kernel(CombineParams P) {
    __shared__ long long s_piece[MAX_CACHED_PIECES];   // partial slots, ascending warp order
    __shared__ float s_w[MAX_CACHED_PIECES][MAX_ROWS_SEG];  // weight of piece k for row i
    __shared__ float s_M[MAX_ROWS_SEG], s_den[MAX_ROWS_SEG];
    __shared__ int s_np, s_nan[MAX_ROWS_SEG];
    grid_dependency_wait();  // the attention's partials are complete
    const int X = P.Hkv * P.RBLK;
    const int seg = blockIdx.x;
    const int b = seg / X, q = seg % X;
    const int kvh = q / P.RBLK, rblk = q % P.RBLK;
    // positions run over units of gs segments; worker groups share them
    const int GS = P.gs, U = X / GS, u = q / GS, gi = q % GS;
    const long long NG = P.nwarps / GS;
    const int4 Rq = P.req[b];
    const int Pb = Rq.y;
    const int RS = P.rows_seg;
    const int rows_here = min(RS, P.R - rblk * RS);
    const float NaN = __int_as_float(0x7fc00000);
    const float LOG2E_ = 1.4426950408889634f;
    const long long N = (long long)P.hdr[HDR_TOTAL_PAGES] * U;
    long long kf = 0, kl = -1;
    if (Pb > 0) {
        const long long x0 = (long long)Rq.z * U + (long long)u * Pb;
        const long long xl = x0 + Pb - 1;
        if (xl >= N) return;  // not a plan of this problem
        kf = share_owner(x0, N, NG);
        kl = share_owner(xl, N, NG);
        if (kf == kl) return;  // one piece: the attention kernel wrote the output
    }
    const long long slot0 = ((long long)b * U + u) * GS + gi;  // slot of group g: slot0 + g * GS
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // 1. the pieces: worker groups kf..kl with a non-empty share (empty shares
    //    only exist when there are fewer positions than groups)
    if (threadIdx.x == 0) {
        int np = 0;
        for (long long k = kf; k <= kl; ++k) {
            if (share_start(k, N, NG) == share_start(k + 1, N, NG)) continue;
            if (np < MAX_CACHED_PIECES) s_piece[np] = slot0 + k * GS;
            ++np;
        }
        s_np = np;
    }
    __syncthreads();
    const int np = s_np;
    const bool cached = np <= MAX_CACHED_PIECES;
    // slot of the n-th piece (recomputed when there are too many to cache)
    auto piece_slot = [&](int n) -> long long {
        if (cached) return s_piece[n];
        int seen = 0;
        for (long long k = kf; k <= kl; ++k) {
            if (share_start(k, N, NG) == share_start(k + 1, N, NG)) continue;
            if (seen++ == n) return slot0 + k * GS;
        }
        return slot0 + kf * GS;
    };
    // 2. per row: M = max lse, den = sum exp(lse - M), NaN if any piece is NaN
    if (Pb > 0) {
        for (int i = warp; i < rows_here; i += COMBINE_THREADS / 32) {
            float M = -INFINITY;
            int nan = 0;
            for (int n = lane; n < np; n += 32) {
                const float l = P.part_lse[piece_slot(n) * RS + i];
                nan |= (l != l);
                M = fmaxf(M, l);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                nan |= __shfl_xor_sync(0xffffffffu, nan, o);
            }
            float den = 0.f;
            if (M != -INFINITY && !nan) {
                for (int n = lane; n < np; n += 32) {
                    const float w = ex2((P.part_lse[piece_slot(n) * RS + i] - M) * LOG2E_);
                    if (cached) s_w[n][i] = w;
                    den += w;
                }
            }
            // fixed-order sum of the lane partials (bitwise reproducible)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
            if (lane == 0) {
                s_M[i] = M;
                s_den[i] = den;
                s_nan[i] = nan;
            }
        }
    }
    __syncthreads();
    // 3. every output element: one weighted sum in ascending piece order
    for (int idx = threadIdx.x; idx < rows_here * P.Dv; idx += COMBINE_THREADS) {
        const int i = idx / P.Dv, d = idx % P.Dv;
        const int r = rblk * RS + i;
        float y, lse_v;
        if (Pb == 0) {
            // no visible page: a flagged request is NaN, an empty one is 0
            y = Rq.w ? NaN : 0.f;
            lse_v = Rq.w ? NaN : -INFINITY;
        } else if (s_nan[i]) {
            y = lse_v = NaN;
        } else if (s_M[i] == -INFINITY) {
            y = 0.f;
            lse_v = -INFINITY;
        } else {
            const float M = s_M[i], den = s_den[i];
            float acc = 0.f;
            for (int n = 0; n < np; ++n) {
                const long long slot = piece_slot(n);
                const float w = cached ? s_w[n][i] : ex2((P.part_lse[slot * RS + i] - M) * LOG2E_);
                acc += w * P.part_o[(slot * RS + i) * P.Dv + d];
            }
            y = acc / den;
            lse_v = M + lg2(den) * 0.6931471805599453f;
        }
        float vsc = 1.0f;
        if (P.v_mode == PA_SCALE_TENSOR) vsc = P.v_scale[0];
        else if (P.v_mode == PA_SCALE_CHANNEL) vsc = P.v_scale[(size_t)kvh * P.Dv + d];
        y *= vsc;
        const int jq = r / P.G, h = kvh * P.G + (r % P.G);
        const size_t oi = (((size_t)b * P.n + jq) * P.Hq + h) * P.Dv + d;
        if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = y;
        else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(y);
        else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(y);
        if (P.lse != nullptr && d == 0) P.lse[((size_t)b * P.n + jq) * P.Hq + h] = lse_v;
    }
}

cudaError_t launch_combine(const CombineParams &P, cudaStream_t s) {
    if (P.B == 0) return cudaSuccess;
    if (P.rows_seg < 1 || P.rows_seg > MAX_ROWS_SEG || P.gs < 1 || (P.Hkv * P.RBLK) % P.gs != 0 ||
        P.nwarps % P.gs != 0)
        return cudaErrorInvalidValue;
    cudaError_t e = launch_pdl(pa_combine_kernel, dim3(P.B * P.Hkv * P.RBLK), dim3(COMBINE_THREADS), 0, s, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace pa
