// Device-side planning for paged attention (sm_103a).
//
//  * pa_max_abs_scale_kernel: one block reduces max |k_scale| over every
//    (kv head, channel) entry and stores it in the workspace header (1 when
//    the maximum is 0).  It runs on the device so a captured step stays free
//    of host synchronisation (onnxruntime PR #32520, "Normalize the
//    PER_CHANNEL K scale folded into Q for paged XQA", Approach and Cost).
//  * pa_plan_kernel: one block turns context_lens into the work plan: pages
//    P_b = ceil(L_b / bs) of every request, bs the tokens of a work page (0 for
//    a request whose length breaks the contract, which is flagged) and their
//    exclusive prefix sums PS_b.  The
//    attention launch orders all pages as (request, kv head, row block, page)
//    -- logical positions only, never block ids -- and gives every warp an equal
//    contiguous share, so every reduction order is independent of where pages
//    live (1Cat-vLLM PR #494, "Stabilize QSA page4 order under KV relocation",
//    Summary).  A plan is only valid for the lengths it saw (FlashInfer docs,
//    "flashinfer.fp4_paged_mqa_logits", schedule_meta); the attention kernel
//    compares them again.
//
// Request record: {L_b as seen, P_b, PS_b, flags}; header word 1 = sum_b P_b.
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

// pages of request b, or -1 when its length breaks the contract (longer than
// max_context_len, or than the blocks its table row can name)
__device__ __forceinline__ int req_pages(const PlanParams &P, int L) {
    if (L < 0 || L > P.max_ctx || (long long)L > (long long)P.tbl * P.bsb) return -1;
    const int pb = (L + P.bs - 1) / P.bs;
    return pb > P.mbps ? -1 : pb;
}

// exclusive block-wide prefix sum of v (PLAN_THREADS threads); *total gets the sum
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long *warp_tot, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long t = (lane < PLAN_THREADS / 32) ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_tot[lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const long long before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
    if (threadIdx.x == 0) *total = warp_tot[PLAN_THREADS / 32 - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(PLAN_THREADS) pa_plan_kernel(PlanParams P) {
    // the attention launch may queue up behind this single block right away
    grid_dependents_launch();
    __shared__ long long warp_tot[32];
    __shared__ long long s_total;
    __shared__ uint32_t s_err;
    if (threadIdx.x == 0) s_err = 0;
    __syncthreads();
    long long carry = 0;
    for (int base = 0; base < P.B; base += PLAN_THREADS) {
        const int b = base + threadIdx.x;
        int L = 0, pb = 0, flags = 0;
        if (b < P.B) {
            L = P.context_lens[b];
            pb = req_pages(P, L);
            if (pb < 0) {
                flags = 1;
                pb = 0;
                atomicOr(&s_err, PA_DEV_ERR_CONTEXT_LEN);
            }
        }
        const long long ofs = carry + block_exclusive_scan(pb, warp_tot, &s_total);
        if (b < P.B) P.req[b] = make_int4(L, pb, (int)ofs, flags);
        carry += s_total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        uint32_t e = s_err;
        if (carry > 0x7fffffffll) {  // positions must fit 32 bits per request record
            e |= PA_DEV_ERR_PLAN_OVERFLOW;
            carry = 0;
        }
        P.hdr[HDR_ERR] = e;  // a new plan starts with a clean error word
        P.hdr[HDR_TOTAL_PAGES] = (uint32_t)carry;
        P.hdr[2] = 0;
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
