// Split-KV merge for paged attention (sm_103a).
//
// For every request with S_b > 1 splits and every row of one kv head, the
// normalised partial outputs o_s and log-sum-exps lse_s of the splits are
// merged in ascending split order:
//     M = max_s lse_s,  w_s = exp(lse_s - M),
//     out = (sum_s w_s o_s) / (sum_s w_s) * v_scale,   lse = M + ln(sum_s w_s)
// (the pages name split "partial" kernels -- 1Cat-vLLM PR #647, Fix -- and
// leave the merge to the standard log-sum-exp identity).  A NaN partial (a
// unit that found a contract violation) makes the row NaN.  The order is
// fixed, so the result is bitwise reproducible.
#include "pa_common.cuh"

namespace pa {

constexpr int COMBINE_THREADS = 256;

__global__ void __launch_bounds__(COMBINE_THREADS) pa_combine_kernel(CombineParams P) {
    const int b = blockIdx.x / P.Hkv, kvh = blockIdx.x % P.Hkv;
    const int4 Rq = P.req[b];
    const int S = Rq.y;
    if (S <= 1) return;
    const long long u0 = (long long)Rq.z * P.Hkv + (long long)kvh * S;
    if (Rq.z < 0 || u0 + S > P.max_units) return;  // not a plan of this problem
    const float LOG2E_ = 1.4426950408889634f;
    for (int idx = threadIdx.x; idx < P.R * P.Dv; idx += COMBINE_THREADS) {
        const int r = idx / P.Dv, d = idx % P.Dv;
        float M = -INFINITY;
        bool nan = false;
        for (int s = 0; s < S; ++s) {
            const float l = P.part_lse[(u0 + s) * P.R + r];
            nan |= (l != l);
            M = fmaxf(M, l);
        }
        float y, lse_v;
        if (nan) {
            y = lse_v = __int_as_float(0x7fc00000);
        } else if (M == -INFINITY) {
            y = 0.f;
            lse_v = -INFINITY;
        } else {
            float acc = 0.f, den = 0.f;
            for (int s = 0; s < S; ++s) {
                const float w = ex2((P.part_lse[(u0 + s) * P.R + r] - M) * LOG2E_);
                den += w;
                acc += w * P.part_o[((u0 + s) * P.R + r) * P.Dv + d];
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
    pa_combine_kernel<<<P.B * P.Hkv, COMBINE_THREADS, 0, s>>>(P);
    return cudaGetLastError();
}

}  // namespace pa
