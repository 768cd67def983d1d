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
constexpr int COMBINE_ROWS = 16;  // query rows of a segment handled by one CTA

// first position of warp k's share of the n positions split over nw warps
__device__ __forceinline__ long long share_start(long long k, long long n, long long nw) { return k * n / nw; }

// the warp whose share holds position x (the last k with share_start <= x)
__device__ __forceinline__ long long share_owner(long long x, long long n, long long nw) {
    return ((x + 1) * nw + n - 1) / n - 1;
}

constexpr int MAX_CACHED_PIECES = 64;
constexpr int MAX_ROWS_SEG = 64;

__device__ __forceinline__ void store4(const CombineParams &P, size_t oi, float4 y, bool vec) {
    if (P.out_dtype == PA_F32) {
        float *o = reinterpret_cast<float *>(P.out) + oi;
        if (vec) *reinterpret_cast<float4 *>(o) = y;
        else { o[0] = y.x; o[1] = y.y; o[2] = y.z; o[3] = y.w; }
    } else if (P.out_dtype == PA_F16) {
        __half *o = reinterpret_cast<__half *>(P.out) + oi;
        const __half2 a = __floats2half2_rn(y.x, y.y), b = __floats2half2_rn(y.z, y.w);
        if (vec) {
            uint2 u;
            memcpy(&u.x, &a, 4);
            memcpy(&u.y, &b, 4);
            *reinterpret_cast<uint2 *>(o) = u;
        } else { o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y; }
    } else {
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(P.out) + oi;
        const __nv_bfloat162 a = __floats2bfloat162_rn(y.x, y.y), b = __floats2bfloat162_rn(y.z, y.w);
        if (vec) {
            uint2 u;
            memcpy(&u.x, &a, 4);
            memcpy(&u.y, &b, 4);
            *reinterpret_cast<uint2 *>(o) = u;
        } else { o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y; }
    }
}

// One CTA per (segment, block of 16 query rows of it).  Every thread owns 4
// output channels of a row at a time and merges them on its own: the row's
// lse values (the same for the 32 threads of a row, so they come from L1),
// their maximum, the weights and their sum in ascending piece order, and the
// weighted float4 sum of the partials -- a single memory latency and no
// block barrier (except for listing the pieces when some shares are empty).
__global__ void __launch_bounds__(COMBINE_THREADS) pa_combine_kernel(CombineParams P) {
    __shared__ long long s_piece[MAX_CACHED_PIECES];  // partial slots, ascending worker order (some shares empty)
    __shared__ int s_np;
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
    const int i0 = blockIdx.y * COMBINE_ROWS;             // first row of this CTA within the segment
    const int rows_here = min(min(COMBINE_ROWS, RS - i0), P.R - rblk * RS - i0);
    if (rows_here <= 0) return;
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
    // 1. the pieces: worker groups kf..kl with a non-empty share.  With at
    //    least as many positions as groups every share is non-empty and the
    //    n-th piece is group kf + n; otherwise thread 0 lists them.
    if (threadIdx.x == 0 && N < NG) {
        int np = 0;
        for (long long k = kf; k <= kl; ++k) {
            if (share_start(k, N, NG) == share_start(k + 1, N, NG)) continue;
            if (np < MAX_CACHED_PIECES) s_piece[np] = slot0 + k * GS;
            ++np;
        }
        s_np = np;
    }
    if (N < NG) __syncthreads();  // uniform: the same N and NG in every thread
    const int np = (N >= NG) ? (int)min(kl - kf + 1, 0x7fffffffll) : s_np;
    const bool cached = np <= MAX_CACHED_PIECES;
    // slot of the n-th piece (recomputed when there are too many to cache)
    auto piece_slot = [&](int n) -> long long {
        if (N >= NG) return slot0 + (kf + n) * GS;
        if (cached) return s_piece[n];
        int seen = 0;
        for (long long k = kf; k <= kl; ++k) {
            if (share_start(k, N, NG) == share_start(k + 1, N, NG)) continue;
            if (seen++ == n) return slot0 + k * GS;
        }
        return slot0 + kf * GS;
    };
    // 2. every 4 output channels of a row: the row's M = max lse, the weights
    //    exp(lse - M) and their sum in ascending piece order, then one weighted
    //    float4 sum; the loads of a row's lse values and partials are all
    //    independent (a single memory latency, no block barrier)
    const int DV4 = P.Dv >> 2;
    const float4 *po = reinterpret_cast<const float4 *>(P.part_o);
    const bool vec = (reinterpret_cast<uintptr_t>(P.out) & 15) == 0;
    for (int idx = threadIdx.x; idx < rows_here * DV4; idx += COMBINE_THREADS) {
        const int ii = idx / DV4, d = (idx - ii * DV4) * 4;
        const int i = i0 + ii;
        const int r = rblk * RS + i;
        float4 y;
        float lse_v;
        if (Pb == 0) {
            // no visible page: a flagged request is NaN, an empty one is 0
            const float z = Rq.w ? NaN : 0.f;
            y = make_float4(z, z, z, z);
            lse_v = Rq.w ? NaN : -INFINITY;
        } else {
            float M = -INFINITY;
            bool nan = false;
            for (int n = 0; n < np; ++n) {
                const float l = P.part_lse[piece_slot(n) * RS + i];
                nan |= (l != l);
                M = fmaxf(M, l);
            }
            if (nan) {
                y = make_float4(NaN, NaN, NaN, NaN);
                lse_v = NaN;
            } else if (M == -INFINITY) {
                y = make_float4(0.f, 0.f, 0.f, 0.f);
                lse_v = -INFINITY;
            } else {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float den = 0.f;
                int n = 0;
                for (; n + 4 <= np; n += 4) {  // four pieces' loads in flight
                    float4 v[4];
                    float w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const long long slot = piece_slot(n + k);
                        w[k] = P.part_lse[slot * RS + i];
                        v[k] = po[(slot * RS + i) * DV4 + (d >> 2)];
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        w[k] = ex2((w[k] - M) * LOG2E_);
                        den += w[k];
                        acc.x += w[k] * v[k].x;
                        acc.y += w[k] * v[k].y;
                        acc.z += w[k] * v[k].z;
                        acc.w += w[k] * v[k].w;
                    }
                }
                for (; n < np; ++n) {
                    const long long slot = piece_slot(n);
                    const float w = ex2((P.part_lse[slot * RS + i] - M) * LOG2E_);
                    const float4 v = po[(slot * RS + i) * DV4 + (d >> 2)];
                    den += w;
                    acc.x += w * v.x;
                    acc.y += w * v.y;
                    acc.z += w * v.z;
                    acc.w += w * v.w;
                }
                const float inv = 1.0f / den;
                y = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                lse_v = M + lg2(den) * 0.6931471805599453f;
            }
        }
        if (P.v_mode == PA_SCALE_TENSOR) {
            const float sc = P.v_scale[0];
            y.x *= sc; y.y *= sc; y.z *= sc; y.w *= sc;
        } else if (P.v_mode == PA_SCALE_CHANNEL) {
            const float *vs = P.v_scale + (size_t)kvh * P.Dv + d;
            y.x *= vs[0]; y.y *= vs[1]; y.z *= vs[2]; y.w *= vs[3];
        }
        const int jq = r / P.G, h = kvh * P.G + (r % P.G);
        const size_t oi = (((size_t)b * P.n + jq) * P.Hq + h) * P.Dv + d;
        store4(P, oi, y, vec);
        if (P.lse != nullptr && d == 0) P.lse[((size_t)b * P.n + jq) * P.Hq + h] = lse_v;
    }
}

cudaError_t launch_combine(const CombineParams &P, cudaStream_t s) {
    if (P.B == 0) return cudaSuccess;
    if (P.rows_seg < 1 || P.rows_seg > MAX_ROWS_SEG || P.gs < 1 || (P.Hkv * P.RBLK) % P.gs != 0 ||
        P.nwarps % P.gs != 0 || (P.Dv & 3) != 0)
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(P.B * P.Hkv * P.RBLK), (unsigned)((P.rows_seg + COMBINE_ROWS - 1) / COMBINE_ROWS));
    cudaError_t e = launch_pdl(pa_combine_kernel, grid, dim3(COMBINE_THREADS), 0, s, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace pa
