// Device-side planning for paged attention (sm_103a).
//
//  * pa_max_abs_scale_kernel: one block reduces max |k_scale| over every
//    (kv head, channel) entry and stores it in the workspace header (1 when
//    the maximum is 0).  It runs on the device so a captured step stays free
//    of host synchronisation (onnxruntime PR #32520, "Normalize the
//    PER_CHANNEL K scale folded into Q for paged XQA", Approach and Cost).
//  * pa_plan_kernel: one block turns context_lens into work units.  The split
//    of each request's pages depends only on the lengths and fixed sizes --
//    never on block ids -- and units are emitted in logical order, so every
//    reduction order is independent of where pages live (1Cat-vLLM PR #494,
//    "Stabilize QSA page4 order under KV relocation", Summary).  A plan is
//    only valid for the lengths it saw (FlashInfer docs,
//    "flashinfer.fp4_paged_mqa_logits", schedule_meta); the attention kernel
//    compares them again.
//
// Rule (pages P_b = ceil(L_b / bs); W = sum P_b; T = target units per head):
//   C   = forced_pages > 0 ? forced_pages : max(min_pages, ceil(W / T))
//   S_b = max(1, ceil(P_b / C))
//   unit u = ofs_b * Hkv + h * S_b + s covers pages [s*C, min((s+1)*C, P_b)).
#include "pa_common.cuh"

namespace pa {

constexpr int PLAN_THREADS = 1024;

__global__ void __launch_bounds__(256) pa_max_abs_scale_kernel(const float *k_scale, int count, uint32_t *hdr) {
    __shared__ float red[8];
    float m = 0.f;
    for (int i = threadIdx.x; i < count; i += blockDim.x) m = fmaxf(m, fabsf(k_scale[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (threadIdx.x == 0) hdr[HDR_KMAX] = __float_as_uint(m == 0.f ? 1.0f : m);
    }
}

// pages of request b, or -1 when its length breaks the contract
__device__ __forceinline__ int req_pages(const PlanParams &P, int L) {
    if (L < 0 || L > P.max_ctx) return -1;
    const int pb = (L + P.bs - 1) / P.bs;
    return pb > P.mbps ? -1 : pb;
}

// exclusive block-wide prefix sum of v (PLAN_THREADS threads); *total gets the sum
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = (lane < PLAN_THREADS / 32) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
    if (threadIdx.x == 0) *total = warp_tot[PLAN_THREADS / 32 - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(PLAN_THREADS) pa_plan_kernel(PlanParams P) {
    __shared__ long long wsum[PLAN_THREADS / 32];
    __shared__ uint32_t werr[PLAN_THREADS / 32];
    __shared__ int warp_tot[32];
    __shared__ int s_total;
    __shared__ int s_C;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // 1. total pages and contract violations
    long long w = 0;
    uint32_t err = 0;
    for (int b = threadIdx.x; b < P.B; b += PLAN_THREADS) {
        const int pb = req_pages(P, P.context_lens[b]);
        if (pb < 0) err |= PA_DEV_ERR_CONTEXT_LEN;
        else w += pb;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        w += __shfl_xor_sync(0xffffffffu, w, o);
        err |= __shfl_xor_sync(0xffffffffu, err, o);
    }
    if (lane == 0) {
        wsum[warp] = w;
        werr[warp] = err;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        long long W = 0;
        uint32_t e = 0;
        for (int i = 0; i < PLAN_THREADS / 32; ++i) {
            W += wsum[i];
            e |= werr[i];
        }
        long long C = P.forced_pages > 0 ? P.forced_pages : (W + P.T - 1) / P.T;
        if (P.forced_pages <= 0 && C < P.min_pages) C = P.min_pages;
        if (C < 1) C = 1;
        if (C > 0x7fffffff) C = 0x7fffffff;
        s_C = (int)C;
        P.hdr[HDR_ERR] = e;  // a new plan starts with a clean error word
        P.hdr[HDR_CHUNK] = (uint32_t)C;
    }
    __syncthreads();
    const int C = s_C;

    // 2. splits, their prefix sums, and the unit records
    int carry = 0;
    for (int base = 0; base < P.B; base += PLAN_THREADS) {
        const int b = base + threadIdx.x;
        int L = 0, pb = 0, flags = 0, S = 0;
        if (b < P.B) {
            L = P.context_lens[b];
            pb = req_pages(P, L);
            if (pb < 0) { flags = 1; pb = 0; }
            S = max(1, (pb + C - 1) / C);
        }
        const int ofs = carry + block_exclusive_scan(S, warp_tot, &s_total);
        if (b < P.B) {
            P.req[b] = make_int4(L, S, ofs, flags);
            for (int h = 0; h < P.Hkv; ++h) {
                for (int s = 0; s < S; ++s) {
                    const long long u = (long long)ofs * P.Hkv + (long long)h * S + s;
                    if (u < P.max_units) {
                        const int pa = min(s * C, pb), pe = (int)min((long long)(s + 1) * C, (long long)pb);
                        P.units[u] = make_int4(b, (h << 16) | s, pa, pe);
                    }
                }
            }
        }
        carry += s_total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const long long nu = (long long)carry * P.Hkv;
        if (nu > P.max_units) {
            atomicOr(P.hdr + HDR_ERR, PA_DEV_ERR_PLAN_OVERFLOW);
            P.hdr[HDR_NUM_UNITS] = 0;  // run nothing rather than a partial plan
        } else {
            P.hdr[HDR_NUM_UNITS] = (uint32_t)nu;
        }
    }
}

cudaError_t launch_plan(const PlanParams &P, const float *k_scale, int k_count, cudaStream_t s) {
    if (k_scale != nullptr) {
        pa_max_abs_scale_kernel<<<1, 256, 0, s>>>(k_scale, k_count, P.hdr);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    pa_plan_kernel<<<1, PLAN_THREADS, 0, s>>>(P);
    return cudaGetLastError();
}

}  // namespace pa
