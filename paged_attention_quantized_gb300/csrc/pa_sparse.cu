// Sparse (selected-token) paged attention: every query token attends only to
// the logical token positions its selection names.
//
// Sources (page title, section):
//  - 1Cat-vLLM PR #494, "[Bugfix][SM70] Stabilize QSA page4 order under KV
//    relocation", Summary / Contract and limits: sparse (QSA) attention over
//    per-query selected token ids, whose work is ordered by logical position
//    (physical ids are only payload), so results are bitwise identical when
//    pages are relocated and do not depend on how selections are listed.
//  - the same page, Upstream and duplicate-work check: unused selection
//    entries are skipped.
//
// Two kernels:
//  pa_sparse_plan_kernel  one CTA per query token: the selection's visible
//      positions are set in a shared-memory bitmap (duplicates collapse) and
//      compacted in ascending order into the workspace -- the token list is a
//      function of the selection as a set, never of its order or of physical
//      ids.
//  pa_sparse_attn_kernel  one CTA per (query token, kv head): its G heads
//      share the token list.  Four warps take contiguous quarters of the
//      list, in groups of 2 or 4 tokens: the list entries, block ids and K
//      and V rows of a group are loaded together (coalesced: lane i holds
//      channels [i*D/32, (i+1)*D/32)), so their latencies overlap; the rows
//      are dequantized in fp32, the G scores formed with shuffle reductions
//      and an fp32 online softmax updated once per head and group; the
//      quarters are merged in warp order.  All arithmetic is
//      fp32 (the per-channel K scale is applied to q in fp32, so no fold can
//      overflow), there are no waits, and every index is checked before use.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "pa.h"

namespace {

constexpr int PLAN_THREADS = 256;
constexpr int ATTN_THREADS = 128;
constexpr int ATTN_WARPS = ATTN_THREADS / 32;
constexpr size_t MAX_PLAN_SMEM = 227 * 1024;

struct SparseParams {
    const uint8_t *q;
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    const int32_t *block_table;
    const float *k_scale;
    const float *v_scale;
    const int32_t *counts;   // [B * n] selected visible tokens, -1 for a flagged request
    const int32_t *lists;    // [B * n][top_k] ascending logical positions
    uint32_t *hdr;           // workspace word 0: device error bits
    void *out;
    float *lse;
    long long k_block, v_block;  // bytes per block of each plane
    int row_bytes;               // code bytes of one token row
    int k_codes, v_codes;        // code bytes of a block (offset of its per-token scales)
    int B, n, Hq, Hkv, G, bs, mbps, num_blocks, top_k;
    int q_dtype, out_dtype, k_mode, v_mode;
    float softmax_scale;
};

// --------------------------------------------------------------- planning

__global__ void __launch_bounds__(PLAN_THREADS)
pa_sparse_plan_kernel(const int32_t *__restrict__ sel, const int32_t *__restrict__ context_lens,
                      int32_t *__restrict__ counts, int32_t *__restrict__ lists, uint32_t *hdr, int n, int top_k,
                      int causal, int max_ctx, int mbps, int bs) {
    extern __shared__ uint32_t bitmap[];
    __shared__ int warp_total[PLAN_THREADS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bj = blockIdx.x;
    const int b = bj / n, j = bj - b * n;
    const int L = context_lens[b];
    if (L < 0 || L > max_ctx || (L > 0 && (L - 1) / bs + 1 > mbps)) {
        if (tid == 0) {
            counts[bj] = -1;
            atomicOr(hdr, PA_DEV_ERR_CONTEXT_LEN);
        }
        return;
    }
    const int vis = max(0, causal ? L - (n - 1 - j) : L);
    const int words = (vis + 31) >> 5;  // <= ceil(max_ctx / 32): the bitmap's size
    for (int w = tid; w < words; w += PLAN_THREADS) bitmap[w] = 0u;
    __syncthreads();
    const int32_t *s = sel + (long long)bj * top_k;
    for (int k = tid; k < top_k; k += PLAN_THREADS) {
        const int t = s[k];
        if (t >= 0 && t < vis) atomicOr(&bitmap[t >> 5], 1u << (t & 31));
    }
    __syncthreads();
    // thread i compacts words [w0, w1): contiguous chunks in thread order, so
    // the list comes out ascending
    const int w0 = (int)((long long)words * tid / PLAN_THREADS);
    const int w1 = (int)((long long)words * (tid + 1) / PLAN_THREADS);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bitmap[w]);
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_total[warp] = x;
    __syncthreads();
    int base = 0;
    for (int i = 0; i < warp; ++i) base += warp_total[i];
    int off = base + x - c;  // distinct positions <= entries, so off < top_k
    int32_t *out = lists + (long long)bj * top_k;
    for (int w = w0; w < w1; ++w) {
        uint32_t bits = bitmap[w];
        while (bits) {
            const int bit = __ffs(bits) - 1;
            out[off++] = (w << 5) + bit;
            bits &= bits - 1;
        }
    }
    if (tid == PLAN_THREADS - 1) counts[bj] = base + x;
}

// -------------------------------------------------------------- attention

template <int KV>
struct Codes {
    static constexpr int BITS = (KV == PA_F16 || KV == PA_BF16) ? 16 : (KV == PA_INT4 ? 4 : 8);
};

// Load a lane's CPL channels of a code row (CPL * bits / 8 bytes, naturally aligned).
template <int KV, int CPL>
__device__ __forceinline__ void load_codes(const uint8_t *p, uint32_t (&w)[4]) {
    constexpr int LB = CPL * Codes<KV>::BITS / 8;
    w[0] = w[1] = w[2] = w[3] = 0u;
    if constexpr (LB == 16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (LB == 8) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
        w[0] = v.x; w[1] = v.y;
    } else if constexpr (LB == 4) {
        w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
    } else if constexpr (LB == 2) {
        w[0] = __ldg(reinterpret_cast<const unsigned short *>(p));
    } else {
        w[0] = __ldg(p);
    }
}

// Exact fp32 values of the CPL codes in w (channel order).
template <int KV, int CPL>
__device__ __forceinline__ void decode(const uint32_t (&w)[4], float (&x)[CPL]) {
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
        if constexpr (KV == PA_F16) {
            const uint16_t h = (uint16_t)(w[i >> 1] >> (16 * (i & 1)));
            x[i] = __half2float(__ushort_as_half(h));
        } else if constexpr (KV == PA_BF16) {
            x[i] = __uint_as_float((w[i >> 1] >> (16 * (i & 1))) << 16);
        } else if constexpr (KV == PA_E4M3) {
            const uint16_t c = (uint16_t)((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
            uint32_t r;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));  // the code lands in the low half
            x[i] = __half2float(__ushort_as_half((uint16_t)(r & 0xFFFFu)));
        } else if constexpr (KV == PA_INT8) {
            x[i] = (float)(int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
        } else {  // INT4: channel 2k in the low nibble of byte k
            const int v = (int)((w[i >> 3] >> (4 * (i & 7))) & 0xFu);
            x[i] = (float)(v >= 8 ? v - 16 : v);
        }
    }
}

__device__ __forceinline__ float load_q(const uint8_t *q, long long idx, int dtype) {
    const uint16_t h = reinterpret_cast<const uint16_t *>(q)[idx];
    return dtype == PA_BF16 ? __uint_as_float((uint32_t)h << 16) : __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ void store_out(void *out, long long idx, int dtype, float v) {
    if (dtype == PA_F32) reinterpret_cast<float *>(out)[idx] = v;
    else if (dtype == PA_F16) reinterpret_cast<__half *>(out)[idx] = __float2half_rn(v);
    else reinterpret_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

template <int KV, int D>
__global__ void __launch_bounds__(ATTN_THREADS) pa_sparse_attn_kernel(const SparseParams P) {
    constexpr int CPL = D / 32;                 // channels per lane
    constexpr int NH = (2048 / D) < 16 ? (2048 / D) : 16;  // heads per kv head at most
    constexpr int LB = CPL * Codes<KV>::BITS / 8;
    __shared__ float s_m[ATTN_WARPS][NH], s_l[ATTN_WARPS][NH];
    __shared__ float s_o[ATTN_WARPS][NH][D];
    __shared__ int s_bad;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.x % P.Hkv;
    const int bj = blockIdx.x / P.Hkv;  // request b, query token j: bj = b * n + j
    const int b = bj / P.n;
    const int G = P.G;
    if (threadIdx.x == 0) s_bad = 0;
    const int cnt = P.counts[bj];

    // q of this lane's channels for every head, with the softmax scale and
    // the K scale applied in fp32
    float qv[NH][CPL];
    const long long q0 = ((long long)bj * P.Hq + (long long)g * G) * D;
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            const int c = lane * CPL + i;
            float v = 0.f;
            if (h < G) {
                v = load_q(P.q, q0 + (long long)h * D + c, P.q_dtype) * P.softmax_scale;
                if (P.k_mode == PA_SCALE_CHANNEL) v *= __ldg(P.k_scale + (long long)g * D + c);
                else if (P.k_mode == PA_SCALE_TENSOR) v *= __ldg(P.k_scale);
            }
            qv[h][i] = v;
        }
    float m[NH], l[NH], o[NH][CPL];
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) o[h][i] = 0.f;
    }
    bool bad = cnt < 0;
    const int total = cnt < 0 ? 0 : cnt;
    const int lo = (int)((long long)total * warp / ATTN_WARPS);
    const int hi = (int)((long long)total * (warp + 1) / ATTN_WARPS);
    const int32_t *list = P.lists + (long long)bj * P.top_k;
    const int32_t *tab = P.block_table + (long long)b * P.mbps;
    // groups of TK tokens: the list entries, block ids and rows of a group are
    // loaded together, then one rescale per head and group
    constexpr int TK = NH >= 16 ? 2 : 4;
    for (int idx0 = lo; idx0 < hi; idx0 += TK) {
        int t[TK], blk[TK];
        bool ok[TK];
#pragma unroll
        for (int u = 0; u < TK; ++u) t[u] = idx0 + u < hi ? __ldg(list + idx0 + u) : -1;
#pragma unroll
        for (int u = 0; u < TK; ++u) {
            blk[u] = t[u] >= 0 ? __ldg(tab + t[u] / P.bs) : 0;  // t < L: the table holds its page
            ok[u] = t[u] >= 0 && blk[u] >= 1 && blk[u] < P.num_blocks;
            if (t[u] >= 0 && !ok[u]) bad = true;
        }
        uint32_t kw[TK][4], vw[TK][4];
        float ks[TK], vs[TK];
#pragma unroll
        for (int u = 0; u < TK; ++u) {
            ks[u] = vs[u] = 1.f;
            if (!ok[u]) {
                kw[u][0] = kw[u][1] = kw[u][2] = kw[u][3] = 0u;
                vw[u][0] = vw[u][1] = vw[u][2] = vw[u][3] = 0u;
                continue;
            }
            const int slot = t[u] - (t[u] / P.bs) * P.bs;
            const long long row_off = (long long)(g * P.bs + slot) * P.row_bytes + lane * LB;
            const uint8_t *kb = P.k_pool + (long long)blk[u] * P.k_block;
            const uint8_t *vb = P.v_pool + (long long)blk[u] * P.v_block;
            load_codes<KV, CPL>(kb + row_off, kw[u]);
            load_codes<KV, CPL>(vb + row_off, vw[u]);
            if (P.k_mode == PA_SCALE_TOKEN) ks[u] = __ldg(reinterpret_cast<const float *>(kb + P.k_codes) + g * P.bs + slot);
            if (P.v_mode == PA_SCALE_TOKEN) vs[u] = __ldg(reinterpret_cast<const float *>(vb + P.v_codes) + g * P.bs + slot);
        }
        float sc[TK][NH];
#pragma unroll
        for (int u = 0; u < TK; ++u) {
            float kx[CPL];
            decode<KV, CPL>(kw[u], kx);
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                sc[u][h] = -INFINITY;
                if (h >= G) continue;
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < CPL; ++i) s = fmaf(qv[h][i], kx[i], s);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                if (ok[u]) sc[u][h] = s * ks[u];
            }
        }
        float vx[TK][CPL];
#pragma unroll
        for (int u = 0; u < TK; ++u) decode<KV, CPL>(vw[u], vx[u]);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            if (h >= G) break;
            float gm = sc[0][h];
#pragma unroll
            for (int u = 1; u < TK; ++u) gm = fmaxf(gm, sc[u][h]);
            const float mn = fmaxf(m[h], gm);
            if (mn == -INFINITY) continue;               // nothing visible yet
            const float corr = expf(m[h] - mn);         // 0 while m = -inf
            l[h] *= corr;
#pragma unroll
            for (int i = 0; i < CPL; ++i) o[h][i] *= corr;
#pragma unroll
            for (int u = 0; u < TK; ++u) {
                const float p = expf(sc[u][h] - mn);    // 0 for a skipped token
                l[h] += p;
                const float pv = p * vs[u];
#pragma unroll
                for (int i = 0; i < CPL; ++i) o[h][i] = fmaf(pv, vx[u][i], o[h][i]);
            }
            m[h] = mn;
        }
    }
    __syncthreads();  // s_bad initialised
    if (bad && lane == 0) atomicOr(&s_bad, 1);
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        if (h >= G) break;
        if (lane == 0) {
            s_m[warp][h] = m[h];
            s_l[warp][h] = l[h];
        }
#pragma unroll
        for (int i = 0; i < CPL; ++i) s_o[warp][h][lane * CPL + i] = o[h][i];
    }
    __syncthreads();
    // merge the quarters in warp order, apply the V scale, write out and lse
    const bool flagged = s_bad != 0;
    for (int e = threadIdx.x; e < G * D; e += ATTN_THREADS) {
        const int h = e / D, d = e - h * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < ATTN_WARPS; ++w) M = fmaxf(M, s_m[w][h]);
        float val, ls;
        if (M == -INFINITY) {  // no token: 0 and -inf
            val = 0.f;
            ls = -INFINITY;
        } else {
            float Ls = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < ATTN_WARPS; ++w) {
                const float f = expf(s_m[w][h] - M);
                Ls += s_l[w][h] * f;
                O += s_o[w][h][d] * f;
            }
            val = O / Ls;
            if (P.v_mode == PA_SCALE_CHANNEL) val *= __ldg(P.v_scale + (long long)g * D + d);
            else if (P.v_mode == PA_SCALE_TENSOR) val *= __ldg(P.v_scale);
            ls = M + logf(Ls);
        }
        if (flagged) val = ls = NAN;
        const long long row = (long long)bj * P.Hq + (long long)g * G + h;
        store_out(P.out, row * D + d, P.out_dtype, val);
        if (d == 0 && P.lse != nullptr) P.lse[row] = ls;
    }
    if (threadIdx.x == 0 && flagged && cnt >= 0) atomicOr(P.hdr, PA_DEV_ERR_BLOCK_ID);
}

template <int KV, int D>
cudaError_t launch_attn(const SparseParams &P, unsigned ctas, cudaStream_t s) {
    pa_sparse_attn_kernel<KV, D><<<ctas, ATTN_THREADS, 0, s>>>(P);
    return cudaPeekAtLastError();
}

template <int D>
cudaError_t dispatch_kv(const SparseParams &P, int kv, unsigned ctas, cudaStream_t s) {
    switch (kv) {
        case PA_F16: return launch_attn<PA_F16, D>(P, ctas, s);
        case PA_BF16: return launch_attn<PA_BF16, D>(P, ctas, s);
        case PA_E4M3: return launch_attn<PA_E4M3, D>(P, ctas, s);
        case PA_INT8: return launch_attn<PA_INT8, D>(P, ctas, s);
        case PA_INT4: return launch_attn<PA_INT4, D>(P, ctas, s);
        default: return cudaErrorInvalidValue;
    }
}

int code_bits(int dt) {
    switch (dt) {
        case PA_F16: case PA_BF16: return 16;
        case PA_E4M3: case PA_INT8: return 8;
        case PA_INT4: return 4;
        default: return 0;
    }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

struct SparseLayout {
    size_t counts, lists, total;
};

pa_status sparse_layout(const pa_problem *p, int32_t top_k, SparseLayout *lo) {
    if (p == nullptr || lo == nullptr) return PA_ERR_INVALID_ARG;
    if (p->batch < 0 || p->next_n < 1 || top_k < 0) return PA_ERR_INVALID_ARG;
    const long long rows = (long long)p->batch * p->next_n;
    if (rows * (long long)std::max(top_k, 1) > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
    lo->counts = 256;
    lo->lists = align256(lo->counts + (size_t)rows * 4);
    lo->total = align256(lo->lists + (size_t)rows * top_k * 4);
    return PA_OK;
}

// the planner's bitmap: one bit per position up to max_context_len
size_t plan_smem(const pa_problem *p) { return (size_t)((p->max_context_len + 31) / 32) * 4; }

}  // namespace

extern "C" PA_API pa_status pa_sparse_workspace_size(const pa_problem *p, int32_t top_k, size_t *bytes) {
    if (bytes == nullptr) return PA_ERR_INVALID_ARG;
    SparseLayout lo;
    const pa_status st = sparse_layout(p, top_k, &lo);
    if (st != PA_OK) return st;
    *bytes = lo.total;
    return PA_OK;
}

extern "C" PA_API pa_status pa_sparse_attention(const pa_problem *p, int32_t top_k, const int32_t *sel, const void *q,
                                                const void *k_pool, const void *v_pool, const int32_t *block_table,
                                                const int32_t *context_lens, const float *k_scale,
                                                const float *v_scale, void *workspace, size_t workspace_bytes,
                                                void *out, float *lse, pa_stream_t stream) {
    SparseLayout lo;
    pa_status st = sparse_layout(p, top_k, &lo);
    if (st != PA_OK) return st;
    if (p->num_q_heads < 1 || p->num_kv_heads < 1 || p->num_q_heads % p->num_kv_heads != 0 || p->block_size < 1 ||
        p->num_blocks < 1 || p->max_blocks_per_seq < 1 || p->max_context_len < 0)
        return PA_ERR_INVALID_ARG;
    if ((p->q_dtype != PA_F16 && p->q_dtype != PA_BF16) ||
        (p->out_dtype != PA_F32 && p->out_dtype != PA_F16 && p->out_dtype != PA_BF16))
        return PA_ERR_INVALID_ARG;
    const int bits = code_bits(p->kv_dtype);
    if (bits == 0) return PA_ERR_INVALID_ARG;
    if (p->k_scale_mode < PA_SCALE_NONE || p->k_scale_mode > PA_SCALE_TOKEN || p->v_scale_mode < PA_SCALE_NONE ||
        p->v_scale_mode > PA_SCALE_TOKEN || (p->causal != 0 && p->causal != 1) || !std::isfinite(p->softmax_scale))
        return PA_ERR_INVALID_ARG;
    const int D = p->head_dim_k;
    if (p->v_is_k_prefix != 0 || p->head_dim_v != D || (D != 64 && D != 128 && D != 256)) return PA_ERR_UNSUPPORTED;
    const int G = p->num_q_heads / p->num_kv_heads;
    const int nh = std::min(16, 2048 / D);
    if (G > nh) return PA_ERR_UNSUPPORTED;
    if ((p->k_scale_mode == PA_SCALE_TOKEN || p->v_scale_mode == PA_SCALE_TOKEN) && p->kv_dtype != PA_E4M3)
        return PA_ERR_UNSUPPORTED;
    const size_t smem = plan_smem(p);
    if (smem > MAX_PLAN_SMEM) return PA_ERR_UNSUPPORTED;
    const int row_bytes = D * bits / 8;
    const long long codes = (long long)p->num_kv_heads * p->block_size * row_bytes;
    const long long kblk = codes + (p->k_scale_mode == PA_SCALE_TOKEN ? (long long)p->num_kv_heads * p->block_size * 4 : 0);
    const long long vblk = codes + (p->v_scale_mode == PA_SCALE_TOKEN ? (long long)p->num_kv_heads * p->block_size * 4 : 0);
    if (kblk % 16 != 0 || vblk % 16 != 0 || codes > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
    const long long rows = (long long)p->batch * p->next_n;
    if (rows * p->num_kv_heads > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
    if (workspace == nullptr || misaligned(workspace, 256) || workspace_bytes < lo.total) return PA_ERR_WORKSPACE;
    if (rows == 0) return PA_OK;
    if ((top_k > 0 && sel == nullptr) || q == nullptr || k_pool == nullptr || v_pool == nullptr ||
        block_table == nullptr || context_lens == nullptr || out == nullptr)
        return PA_ERR_INVALID_ARG;
    if (misaligned(k_pool, 16) || misaligned(v_pool, 16) || misaligned(q, 2) || misaligned(sel, 4) ||
        misaligned(out, p->out_dtype == PA_F32 ? 4 : 2) || misaligned(lse, 4))
        return PA_ERR_INVALID_ARG;
    if ((p->k_scale_mode == PA_SCALE_TENSOR || p->k_scale_mode == PA_SCALE_CHANNEL) && k_scale == nullptr)
        return PA_ERR_INVALID_ARG;
    if ((p->v_scale_mode == PA_SCALE_TENSOR || p->v_scale_mode == PA_SCALE_CHANNEL) && v_scale == nullptr)
        return PA_ERR_INVALID_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *hdr = reinterpret_cast<uint32_t *>(ws);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + lo.counts);
    int32_t *lists = reinterpret_cast<int32_t *>(ws + lo.lists);
    if (cudaMemsetAsync(hdr, 0, sizeof(uint32_t), s) != cudaSuccess) return PA_ERR_CUDA;
    if (smem > 48 * 1024 && cudaFuncSetAttribute(pa_sparse_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem) != cudaSuccess)
        return PA_ERR_CUDA;
    pa_sparse_plan_kernel<<<(unsigned)rows, PLAN_THREADS, smem, s>>>(sel, context_lens, counts, lists, hdr, p->next_n,
                                                                     top_k, p->causal, p->max_context_len,
                                                                     p->max_blocks_per_seq, p->block_size);
    if (cudaPeekAtLastError() != cudaSuccess) return PA_ERR_CUDA;

    SparseParams P;
    P.q = static_cast<const uint8_t *>(q);
    P.k_pool = static_cast<const uint8_t *>(k_pool);
    P.v_pool = static_cast<const uint8_t *>(v_pool);
    P.block_table = block_table;
    P.k_scale = k_scale;
    P.v_scale = v_scale;
    P.counts = counts;
    P.lists = lists;
    P.hdr = hdr;
    P.out = out;
    P.lse = lse;
    P.k_block = kblk;
    P.v_block = vblk;
    P.row_bytes = row_bytes;
    P.k_codes = (int)codes;
    P.v_codes = (int)codes;
    P.B = p->batch;
    P.n = p->next_n;
    P.Hq = p->num_q_heads;
    P.Hkv = p->num_kv_heads;
    P.G = G;
    P.bs = p->block_size;
    P.mbps = p->max_blocks_per_seq;
    P.num_blocks = p->num_blocks;
    P.top_k = top_k;
    P.q_dtype = p->q_dtype;
    P.out_dtype = p->out_dtype;
    P.k_mode = p->k_scale_mode;
    P.v_mode = p->v_scale_mode;
    P.softmax_scale = p->softmax_scale;
    const unsigned ctas = (unsigned)(rows * p->num_kv_heads);
    cudaError_t e;
    switch (D) {
        case 64: e = dispatch_kv<64>(P, p->kv_dtype, ctas, s); break;
        case 128: e = dispatch_kv<128>(P, p->kv_dtype, ctas, s); break;
        default: e = dispatch_kv<256>(P, p->kv_dtype, ctas, s); break;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
