// FP4 (MXFP4) paged MQA logits for sm_103a on the fifth-generation tensor
// cores (FlashInfer docs, "flashinfer.fp4_paged_mqa_logits", Parameters).
//
// For query row r = b * next_n + j (its H heads, E2M1 values with one UE8M0
// scale per 32 values) and every token t of request b (E2M1 codes and UE8M0
// scales in a kv_fused block: all tokens' packed values, then all tokens'
// scale words, in token or interleaved order):
//     logit[r, t] = sum_h w[r, h] * f(q^[h] . k^[t]),  f = identity or max(0, .)
// for t < vis (L_b, or L_b - next_n + 1 + j when causal), -inf for the other
// columns of the row up to max_context_len.
//
// Exact arithmetic without block-scaled MMAs: every row is rescaled by its own
// largest scale, q^[h, d] = e2m1 * 2^(s_hd - A_h) and k^[t, d] = e2m1 *
// 2^(s_td - B_t), which is an exact f16 (E2M1 has two significant bits) while a
// row's scales span at most 2^22; the dot products then run as f16 MMAs with
// fp32 accumulation (products of f16 are exact in fp32), and 2^A_h goes into
// the head weight, 2^B_t into the token's logit.
//
// Work: 128-token tiles in logical order (request, tile) -- never by block
// id -- shared evenly by persistent CTAs (one per SM).  Roles (10 warps):
//  (this kernel serves rectified heads and next_n > 4; the plain weighted sum
//  runs on pa_fp4_logits_sum_kernel below)
//  * warp 0 copies each tile's kv_fused blocks (whole blocks, one bulk copy
//    each; ids range-checked first) into a 4-slot ring;
//  * warps 6-9 (one token per thread) decode the token's 128 values into the
//    f16 A operand in tensor memory (lane = token, 2 values per column) and
//    its scale 2^B_t into shared memory; slots past L_b get zeros;
//  * warp 1 issues S^T = K^ Q^T: 8 MMAs of M = 128 tokens, N = next_n * H
//    rows, K = 16 channels, A from tensor memory, B (q^ of the request,
//    staged once per request) from shared memory;
//  * warps 2-5 (one token per thread) fold each row's head sum from S^T in
//    tensor memory and write the logits (coalesced across tokens).
// Every wait is bounded; a wait that runs out raises the CTA's abort word,
// sets PA_DEV_ERR_TIMEOUT and NaN-fills the columns the CTA still owned.
#include "pa_attn.cuh"
#include "pa_tc.cuh"

namespace pa {

struct Fp4Params {
    const uint8_t *q;           // [B][n][H][64] packed E2M1
    const int32_t *sf_q;        // [B][n][H] four UE8M0 bytes
    const uint8_t *kv;          // [num_blocks][bs * 68]
    const float *weights;       // [B * n][H]
    const int32_t *block_table; // [B][tbl]
    const int32_t *context_lens;
    uint32_t *hdr;
    const int4 *req;            // plan records over 128-token tiles
    float *qw;                  // [B][n][128] folded query rows (plain weighted sum)
    void *out;
    long long out_stride;       // elements per output row
    long long block_bytes;      // bs * 68
    int B, n, H, N, bs, bpt, num_blocks, tbl, mbps, max_ctx;
    int out_dtype, causal, rectify, interleaved;
};

namespace fp4 {

using namespace tc;

constexpr int ROWB = 68, TILE = 128, NSLOT = 4, MAX_N = 192;  // 128 channels: 64 packed bytes + 4 scale bytes
constexpr int SLOT_BYTES = TILE * ROWB;                // whole blocks of one tile, back to back
constexpr int NWARPS = 10, THREADS = NWARPS * 32;
constexpr int W_PROD = 0, W_MMA = 1, W_DQ = 6;  // warps 2-5 write the logits
constexpr int QB_OFF = 0;                              // q^ f16: 2 channel blocks x [MAX_N rows][128 B], SW128
constexpr int QB_BLK = MAX_N * 128;
constexpr int RING_OFF = QB_OFF + 2 * QB_BLK;
constexpr int W_OFF = RING_OFF + NSLOT * SLOT_BYTES;   // [MAX_N] w * 2^A
constexpr int TS_OFF = W_OFF + MAX_N * 4;              // [4][128] 2^B_t
constexpr int BAR_OFF = TS_OFF + 4 * TILE * 4;
enum {
    B_FULL = 0,                    // [NSLOT] tile copied
    B_SLOTFREE = B_FULL + NSLOT,   // [NSLOT] decoded by the four dequant warps
    B_AFULL = B_SLOTFREE + NSLOT,  // [2] A operand written
    B_AFREE = B_AFULL + 2,         // [2] its MMAs complete
    B_SFULL = B_AFREE + 2,         // [2] S^T complete
    B_SFREE = B_SFULL + 2,         // [2] S^T read out
    B_TSFULL = B_SFREE + 2,        // [4] token scales of the tile written
    B_QFULL = B_TSFULL + 4,        // q^ and weights of the request staged
    B_MDONE = B_QFULL + 1,         // every MMA of the CTA complete
    NBARS = B_MDONE + 1
};
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;          // [0] tmem base, [1] abort, [2 + s] slot s bad, [8] errors
constexpr int SMEM_USED = MISC_OFF + 64;
// at least half an SM's shared memory, so one CTA per SM holds all 512 columns
// of tensor memory without a neighbour waiting on its allocation
constexpr int SMEM_BYTES = (SMEM_USED + 1024) > 116 * 1024 ? (SMEM_USED + 1024) : 116 * 1024;
constexpr uint32_t TM_A = 0, TM_S = 128;               // A[2] x 64 columns, S^T[2] x N columns
static_assert(SMEM_USED + 1024 <= 227 * 1024, "fp4 logits kernel exceeds the shared memory of one CTA");
static_assert(QB_BLK % 1024 == 0 && RING_OFF % 1024 == 0, "operand tiles must stay 1 KB aligned");

// E2M1 pair (low nibble -> low half) to f16x2, exact
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte) {
    uint32_t r;
    const uint16_t v = static_cast<uint16_t>(byte & 0xFFu);
    asm("{\n\t.reg .b8 b;\n\tmov.b16 {b, _}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(r) : "h"(v));
    return r;
}

// f16x2 {2^-delta, 2^-delta} for 0 <= delta (0 when 2^-delta is below the f16 range)
__device__ __forceinline__ uint32_t f16_pow2_neg(int delta) {
    uint32_t h;
    if (delta <= 14) h = (uint32_t)(15 - delta) << 10;   // normal
    else if (delta <= 24) h = 1u << (24 - delta);        // subnormal
    else h = 0u;
    return h | (h << 16);
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// 64 packed bytes (128 E2M1 values) and their four UE8M0 bytes -> 64 f16x2
// words scaled by 2^(s_k - smax); returns smax
__device__ __forceinline__ int decode_row(const uint4 (&raw)[4], uint32_t sw, uint32_t (&wd)[64]) {
    const int s0 = sw & 0xFF, s1 = (sw >> 8) & 0xFF, s2 = (sw >> 16) & 0xFF, s3 = sw >> 24;
    const int smax = max(max(s0, s1), max(s2, s3));
    const uint32_t f[4] = {f16_pow2_neg(smax - s0), f16_pow2_neg(smax - s1), f16_pow2_neg(smax - s2),
                           f16_pow2_neg(smax - s3)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w4[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = 16 * c + 4 * e + k;  // byte i holds values 2i, 2i + 1
                wd[i] = hmul2_u(e2m1x2_f16x2(w4[e] >> (8 * k)), f[i >> 4]);
            }
    }
    return smax;
}

// UE8M0 byte -> 2^(e - 127) as fp32 (2^-127 is the subnormal 0x00400000); 0xFF is NaN
__device__ __forceinline__ float ue8m0_f32(int e) {
    return e == 255 ? __int_as_float(0x7fc00000) : (e == 0 ? __int_as_float(0x00400000) : __int_as_float(e << 23));
}

}  // namespace fp4

__global__ void __launch_bounds__(fp4::THREADS, 1) pa_fp4_logits_kernel(Fp4Params P) {
    using namespace fp4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    int *misc = reinterpret_cast<int *>(smem + MISC_OFF);
    volatile int *abort = misc + 1;
    float *wsm = reinterpret_cast<float *>(smem + W_OFF);
    float *tsm = reinterpret_cast<float *>(smem + TS_OFF);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float NaN = __int_as_float(0x7fc00000);

    const long long total = P.hdr[HDR_TOTAL_PAGES];
    if (total > (long long)P.B * P.mbps) {
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    const long long x0 = blockIdx.x * total / gridDim.x, x1 = (blockIdx.x + 1) * total / gridDim.x;
    if (x0 >= x1) return;
    const int npg = (int)(x1 - x0);
    const Cursor c0 = cursor_at(x0, P.req, P.B, 1, P.mbps);
    if (c0.b >= P.B) {
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < NBARS; ++i) {
            // barriers the four dequant or the four logit warps arrive on count 4
            const bool four = (i >= B_SLOTFREE && i < B_SLOTFREE + NSLOT) || (i >= B_AFULL && i < B_AFULL + 2) ||
                              (i >= B_SFREE && i < B_SFREE + 2) || (i >= B_TSFULL && i < B_TSFULL + 4) ||
                              i == B_QFULL;
            mbar_init(&bars[i], four ? 4u : 1u);
        }
        misc[1] = 0;
        misc[8] = 0;
        mbar_fence_init();
    }
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(sb + MISC_OFF)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)misc[0];
    uint32_t err = 0;

    if (warp == W_PROD) {
        // ================================================== copies
        Cursor ci = c0;
        int issued = 0;
        int idc_b = -1, idc_w0 = 0, idc = 0;  // block ids [idc_w0, idc_w0 + 32) of request idc_b, one per lane
#ifdef PA_FAULT_INJECT
        const unsigned fi_withhold = P.hdr[HDR_WITHHOLD];
#endif
        for (int j = 0; j < npg; ++j) {
            const int slot = j % NSLOT;
            if (j >= NSLOT && !warp_wait(&bars[B_SLOTFREE + slot], ((j / NSLOT) - 1) & 1, abort, err)) break;
#ifdef PA_FAULT_INJECT
            if (fi_withhold != 0 && x0 + j + 1 == (long long)fi_withhold && ci.b < P.B) {
                ++issued;
                cursor_next<true>(ci, P.req, P.B, 1, P.mbps);
                continue;  // no copy and no arrive: the waits on this slot run out
            }
#endif
            bool ok = false;
            int nb = 0, id = 0;
            if (ci.b < P.B) {
                const int nblk = min((ci.L + P.bs - 1) / P.bs, P.tbl);
                const int fb = ci.p * P.bpt;
                nb = min(P.bpt, nblk - fb);
                if (ci.b != idc_b || fb < idc_w0 || fb + nb > idc_w0 + 32) {
                    // 32 ids per load: the next tiles' ids are already here
                    idc_b = ci.b;
                    idc_w0 = fb;
                    idc = (fb + lane < nblk) ? P.block_table[(size_t)ci.b * P.tbl + fb + lane] : 1;
                }
                id = __shfl_sync(0xffffffffu, idc, (fb - idc_w0 + lane) & 31);
                if (lane >= nb) id = 1;
                ok = nb >= 1 && __all_sync(0xffffffffu, id >= 1 && id < P.num_blocks);
            }
            if (lane == 0) {
                misc[2 + slot] = ok ? 0 : 1;
                if (!ok) mbar_arrive(&bars[B_FULL + slot]);  // no copy: the tile is NaN-filled
                else mbar_arrive_expect_tx(&bars[B_FULL + slot], (uint32_t)(nb * P.block_bytes));
            }
            __syncwarp();
            if (ok) {
                for (int i = 0; i < nb; ++i) {
                    const int bi = __shfl_sync(0xffffffffu, id, i);
                    if (lane == 0)
                        bulk_load(smem + RING_OFF + slot * SLOT_BYTES + i * P.block_bytes,
                                  P.kv + (size_t)bi * P.block_bytes, (uint32_t)P.block_bytes, &bars[B_FULL + slot]);
                }
            }
            __syncwarp();
            ++issued;
            if (ci.b < P.B) cursor_next<true>(ci, P.req, P.B, 1, P.mbps);
        }
        if (*abort && lane == 0) {
            // let every copy still in flight land before the CTA exits
            for (int i = max(0, issued - NSLOT); i < issued; ++i)
                (void)mbar_wait_bounded(&bars[B_FULL + i % NSLOT], (i / NSLOT) & 1, nullptr);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ================================================== MMA issue
        const uint32_t ID = idesc(128, P.N, 0);
        Cursor cm = c0;
        int piece = -1, pb = -1;
        for (int j = 0; j < npg; ++j) {
            if (cm.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; break; }
            if (cm.b != pb) {
                ++piece;
                pb = cm.b;
                if (!warp_wait(&bars[B_QFULL], piece & 1, abort, err)) break;
            }
            if (!warp_wait(&bars[B_AFULL + (j & 1)], (j >> 1) & 1, abort, err)) break;
            if (j >= 2 && !warp_wait(&bars[B_SFREE + (j & 1)], ((j >> 1) - 1) & 1, abort, err)) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t dS = tmem + TM_S + (uint32_t)(P.N * (j & 1));
                const uint32_t aA = tmem + TM_A + 64u * (j & 1);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t bd = sdesc(sb + QB_OFF + (k >> 2) * QB_BLK + 32 * (k & 3), 16, 1024, 2);
                    mma_f16_ts(dS, aA + 8u * k, bd, ID, k > 0 ? 1u : 0u);
                }
                mma_commit(&bars[B_SFULL + (j & 1)]);
                mma_commit(&bars[B_AFREE + (j & 1)]);
            }
            __syncwarp();
            cursor_next<true>(cm, P.req, P.B, 1, P.mbps);
        }
        if (lane == 0) {
            mma_commit(&bars[B_MDONE]);
            (void)mbar_wait_bounded(&bars[B_MDONE], 0, nullptr);
        }
        __syncwarp();
    } else if (warp >= W_DQ) {
        // ================================================== FP4 -> f16 A operand
        const int qd = warp & 3;
        const int t = 32 * qd + lane;  // token of the tile = tensor-memory lane
        const int q4 = P.bs >> 2;
        Cursor cd = c0;
        for (int j = 0; j < npg; ++j) {
            if (cd.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; break; }
            const int slot = j % NSLOT;
            if (!warp_wait(&bars[B_FULL + slot], (j / NSLOT) & 1, abort, err)) break;
            const int ntok = min(TILE, cd.L - cd.p * TILE);
            const bool bad = misc[2 + slot] != 0;
            if (bad) err |= PA_DEV_ERR_BLOCK_ID;
            uint4 raw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                            make_uint4(0, 0, 0, 0)};
            uint32_t sw = 0x7F7F7F7Fu;  // scale bytes of 2^0 for unused slots (their values are zero)
            const bool live = !bad && t < ntok;
            if (live) {
                const uint8_t *blk = smem + RING_OFF + slot * SLOT_BYTES + (t / P.bs) * P.block_bytes;
                const int s = t % P.bs;
                const uint8_t *row = blk + s * 64;
                const int rot = (lane >> 1) & 3;  // spread the 16-byte loads of a warp over all banks
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int cc = (c + rot) & 3;
                    const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * cc);
                    if (cc == 0) raw[0] = v;
                    else if (cc == 1) raw[1] = v;
                    else if (cc == 2) raw[2] = v;
                    else raw[3] = v;
                }
                const int ws = P.interleaved ? 4 * (s % q4) + s / q4 : s;
                sw = *reinterpret_cast<const uint32_t *>(blk + P.bs * 64 + ws * 4);
            }
            warp_arrive(&bars[B_SLOTFREE + slot]);  // the ring slot is no longer read here
            uint32_t wd[64];
            const int smax = decode_row(raw, sw, wd);
            const float tsv = bad ? NaN : (live ? ue8m0_f32(smax) : 0.f);
            if (j >= 2 && !warp_wait(&bars[B_AFREE + (j & 1)], ((j >> 1) - 1) & 1, abort, err)) break;
            tc_fence_after();
            const uint32_t ta = tmem + TM_A + 64u * (j & 1) + ((uint32_t)(32 * qd) << 16);
            tmem_st32_u(ta, wd);
            tmem_st32_u(ta + 32u, wd + 32);
            tmem_st_wait();
            tsm[(j & 3) * TILE + t] = tsv;
            tc_fence_before();
            warp_arrive(&bars[B_AFULL + (j & 1)]);
            warp_arrive(&bars[B_TSFULL + (j & 3)]);
            cursor_next<true>(cd, P.req, P.B, 1, P.mbps);
        }
    } else {
        // ================================================== logits (warps 2-5)
        const int qd = warp & 3;
        const int t = 32 * qd + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
        Cursor ce = c0;
        int pb = -1, L = 0, qphase = 0;
        bool pbad = false;
        int j = 0;
        auto store = [&](int b, int p, float v0, int jq) {
            const long long col = (long long)p * TILE + t;
            if (col >= P.max_ctx) return;
            const size_t oi = (size_t)((long long)b * P.n + jq) * (size_t)P.out_stride + (size_t)col;
            if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = v0;
            else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(v0);
            else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(v0);
        };
        for (; j < npg; ++j) {
            if (ce.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; break; }
            if (ce.b != pb) {
                // a new request: stage its q^ rows and weights (every MMA that
                // read the previous q^ is complete: its last S^T was waited for)
                pb = ce.b;
                L = P.context_lens[pb];
                const int4 Rq = P.req[pb];
                pbad = false;
                if (Rq.w != 0) { pbad = true; err |= PA_DEV_ERR_CONTEXT_LEN; }
                if (L != Rq.x) { pbad = true; err |= PA_DEV_ERR_STALE_PLAN; }
                for (int r = t; r < P.N; r += TILE) {
                    const int jq = r / P.H, h = r - jq * P.H;
                    const size_t qi = ((size_t)pb * P.n + jq) * P.H + h;
                    const uint4 *src = reinterpret_cast<const uint4 *>(P.q + qi * 64);
                    const uint4 raw[4] = {src[0], src[1], src[2], src[3]};
                    uint32_t wd[64];
                    const int amax = decode_row(raw, (uint32_t)P.sf_q[qi], wd);
                    wsm[r] = P.weights[qi] * ue8m0_f32(amax);
#pragma unroll
                    for (int c = 0; c < 16; ++c) {  // 16-byte chunk c: channels 8c .. 8c + 7
                        const int cb = c >> 3, ch = c & 7;
                        *reinterpret_cast<uint4 *>(smem + QB_OFF + cb * QB_BLK + r * 128 + ((ch ^ (r & 7)) << 4)) =
                            make_uint4(wd[4 * c], wd[4 * c + 1], wd[4 * c + 2], wd[4 * c + 3]);
                    }
                }
                fence_proxy_async_smem();
                warp_arrive(&bars[B_QFULL]);
                // every row and weight is staged once all four warps arrived
                if (!warp_wait(&bars[B_QFULL], qphase & 1, abort, err)) break;
                ++qphase;
            }
            if (!warp_wait(&bars[B_SFULL + (j & 1)], (j >> 1) & 1, abort, err)) break;
            if (!warp_wait(&bars[B_TSFULL + (j & 3)], (j >> 2) & 1, abort, err)) break;
            tc_fence_after();
            const float tsv = tsm[(j & 3) * TILE + t];
            const int col = ce.p * TILE + t;
            for (int jq = 0; jq < P.n; ++jq) {
                float acc = 0.f;
                for (int c0 = 0; c0 < P.H; c0 += 64) {
                    // up to four 16-column loads in flight, one wait
                    uint32_t v[4][16];
                    const int cidx = jq * P.H + c0;
                    const int nch = min(4, (P.H - c0) >> 4);
                    const uint32_t ta = tl + TM_S + (uint32_t)(P.N * (j & 1) + cidx);
                    tmem_ld16_nowait(ta, v[0]);
                    if (nch > 1) tmem_ld16_nowait(ta + 16u, v[1]);
                    if (nch > 2) tmem_ld16_nowait(ta + 32u, v[2]);
                    if (nch > 3) tmem_ld16_nowait(ta + 48u, v[3]);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (k >= nch) break;
                        const float4 *w4 = reinterpret_cast<const float4 *>(wsm + cidx + 16 * k);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 wv = w4[i];
                            float s0 = __uint_as_float(v[k][4 * i]), s1 = __uint_as_float(v[k][4 * i + 1]);
                            float s2 = __uint_as_float(v[k][4 * i + 2]), s3 = __uint_as_float(v[k][4 * i + 3]);
                            if (P.rectify) {
                                s0 = fmaxf(s0, 0.f); s1 = fmaxf(s1, 0.f); s2 = fmaxf(s2, 0.f); s3 = fmaxf(s3, 0.f);
                            }
                            acc = fmaf(wv.x, s0, acc);
                            acc = fmaf(wv.y, s1, acc);
                            acc = fmaf(wv.z, s2, acc);
                            acc = fmaf(wv.w, s3, acc);
                        }
                    }
                }
                const int vis = P.causal ? L - (P.n - 1 - jq) : L;
                const float val = pbad ? NaN : (col < vis ? acc * tsv : -INFINITY);
                store(ce.b, ce.p, val, jq);
            }
            tc_fence_before();
            warp_arrive(&bars[B_SFREE + (j & 1)]);
            cursor_next<true>(ce, P.req, P.B, 1, P.mbps);
        }
        if (j < npg) {
            // a wait ran out: the columns this CTA still owned are NaN
            for (; j < npg && ce.b < P.B; ++j) {
                for (int jq = 0; jq < P.n; ++jq) store(ce.b, ce.p, NaN, jq);
                cursor_next<true>(ce, P.req, P.B, 1, P.mbps);
            }
        }
    }

    // ---- teardown: one error word per CTA, tensor memory released
    if (err) atomicOr(reinterpret_cast<unsigned *>(misc + 8), err);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    if (tid == 0) atomic_or_err(P.hdr, (uint32_t)misc[8]);
}

// Plain weighted sum (rectify = 0): the logit is linear in the heads, so it
// equals k^[t] . qw with qw = sum_h w[r, h] * q^[h] -- one 128-wide vector per
// query row, folded once per request in fp32.  Each token is then a dot
// product of its 128 decoded values with the row vectors: HBM-bound work for
// the CUDA cores (no dense contraction left for the tensor cores).  Tiles of
// 128 tokens in logical order are shared evenly by persistent CTAs of 128
// threads, one token per thread; a token's 64 packed bytes and its scale word
// are loaded straight from the pool (the warp reads 2 KB of consecutive rows
// of a block).  Scale groups are summed separately and scaled by
// 2^(s - 127) exactly.
namespace fp4 {
constexpr int SUM_THREADS = 128;
constexpr int SUM_MAX_N = 4;       // query rows per request this kernel folds (next_n; more use the MMA kernel)
constexpr int SUM_CTAS_PER_SM = 8; // persistent CTAs per SM of the launch
}  // namespace fp4

// qw[b][j][d] = sum_h w[b * n + j][h] * q^[b][j][h][d] in fp32, one CTA per
// query row, thread d per channel (heads in ascending order)
__global__ void __launch_bounds__(128) pa_fp4_fold_kernel(Fp4Params P) {
    const int r = blockIdx.x;  // b * n + j
    const int t = threadIdx.x;
    float acc = 0.f;
    for (int h = 0; h < P.H; ++h) {
        const size_t qi = (size_t)r * P.H + h;
        const uint32_t h2 = fp4::e2m1x2_f16x2(P.q[qi * 64 + (t >> 1)]);
        const float2 v = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
        const int sb = (int)(((uint32_t)P.sf_q[qi] >> (8 * (t >> 5))) & 0xFFu);
        acc = fmaf(P.weights[qi] * fp4::ue8m0_f32(sb), (t & 1) ? v.y : v.x, acc);
    }
    P.qw[(size_t)r * 128 + t] = acc;
}

template <int NQ>
__global__ void __launch_bounds__(fp4::SUM_THREADS) pa_fp4_logits_sum_kernel(Fp4Params P) {
    using namespace fp4;
    __shared__ __align__(16) float qw[NQ][128];  // folded query rows of the current request
    const int t = threadIdx.x;
    const float NaN = __int_as_float(0x7fc00000);
    const long long total = P.hdr[HDR_TOTAL_PAGES];
    if (total > (long long)P.B * P.mbps) {
        if (t == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    const long long x0 = blockIdx.x * total / gridDim.x, x1 = (blockIdx.x + 1) * total / gridDim.x;
    if (x0 >= x1) return;
    Cursor cu = cursor_at(x0, P.req, P.B, 1, P.mbps);
    if (cu.b >= P.B) {
        if (t == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    uint32_t err = 0;
    int pb = -1, L = 0, nblk = 0;
    bool pbad = false;
    const int q4 = P.bs >> 2;
    for (long long x = x0; x < x1; ++x) {
        if (cu.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; break; }
        if (cu.b != pb) {
            // the request's folded query rows (written by pa_fp4_fold_kernel)
            __syncthreads();  // the previous request's rows are no longer read
            pb = cu.b;
            L = P.context_lens[pb];
            const int4 Rq = P.req[pb];
            pbad = false;
            if (Rq.w != 0) { pbad = true; err |= PA_DEV_ERR_CONTEXT_LEN; }
            if (L != Rq.x) { pbad = true; err |= PA_DEV_ERR_STALE_PLAN; }
            nblk = min((L + P.bs - 1) / P.bs, P.tbl);
#pragma unroll
            for (int jq = 0; jq < NQ; ++jq) qw[jq][t] = P.qw[((size_t)pb * NQ + jq) * 128 + t];
            __syncthreads();
        }
        const int tok = cu.p * TILE + t;
        float lg[NQ];
#pragma unroll
        for (int jq = 0; jq < NQ; ++jq) lg[jq] = 0.f;
        bool bad = false;
        if (tok < L) {
            const int bi = tok / P.bs;
            const int blk = bi < nblk ? P.block_table[(size_t)pb * P.tbl + bi] : 0;
            if (blk < 1 || blk >= P.num_blocks) {
                bad = true;
                err |= PA_DEV_ERR_BLOCK_ID;
            } else {
                const uint8_t *base = P.kv + (size_t)blk * (size_t)P.block_bytes;
                const int s = tok - bi * P.bs;
                const uint4 *row = reinterpret_cast<const uint4 *>(base + s * 64);
                const int ws = P.interleaved ? 4 * (s % q4) + s / q4 : s;
                const uint32_t sw = *reinterpret_cast<const uint32_t *>(base + P.bs * 64 + ws * 4);
                uint4 raw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) raw[k] = row[k];
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // scale group k: values 32k .. 32k + 31 = bytes 16k .. 16k + 15
                    float gs[NQ];
#pragma unroll
                    for (int jq = 0; jq < NQ; ++jq) gs[jq] = 0.f;
                    const uint32_t w4[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // the 8 values of word e: channels 32k + 8e .. + 7
                        float v[8];
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb) {
                            const uint32_t h2 = e2m1x2_f16x2(w4[e] >> (8 * bb));
                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
                            v[2 * bb] = f.x;
                            v[2 * bb + 1] = f.y;
                        }
                        const int d = 32 * k + 8 * e;
#pragma unroll
                        for (int jq = 0; jq < NQ; ++jq) {
                            const float4 a = *reinterpret_cast<const float4 *>(&qw[jq][d]);
                            const float4 b = *reinterpret_cast<const float4 *>(&qw[jq][d + 4]);
                            float g = gs[jq];
                            g = fmaf(a.x, v[0], g); g = fmaf(a.y, v[1], g); g = fmaf(a.z, v[2], g); g = fmaf(a.w, v[3], g);
                            g = fmaf(b.x, v[4], g); g = fmaf(b.y, v[5], g); g = fmaf(b.z, v[6], g); g = fmaf(b.w, v[7], g);
                            gs[jq] = g;
                        }
                    }
                    const float sc = ue8m0_f32((int)((sw >> (8 * k)) & 0xFFu));
#pragma unroll
                    for (int jq = 0; jq < NQ; ++jq) lg[jq] = fmaf(sc, gs[jq], lg[jq]);
                }
            }
        }
        if (tok < P.max_ctx) {
#pragma unroll
            for (int jq = 0; jq < NQ; ++jq) {
                const int vis = P.causal ? L - (NQ - 1 - jq) : L;
                const float val = (pbad || bad) ? NaN : (tok < vis ? lg[jq] : -INFINITY);
                const size_t oi = (size_t)((long long)pb * NQ + jq) * (size_t)P.out_stride + (size_t)tok;
                if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = val;
                else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(val);
                else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(val);
            }
        }
        cursor_next<true>(cu, P.req, P.B, 1, P.mbps);
    }
    if (err) atomic_or_err(P.hdr, err);
}

// Columns no tile covers: -inf from the last tile of each request to
// max_context_len, NaN over the whole row of a request the plan flagged.
__global__ void __launch_bounds__(256) pa_fp4_fill_kernel(Fp4Params P) {
    const int r = blockIdx.x;  // query row b * n + j
    const int b = r / P.n;
    const int4 Rq = P.req[b];
    const long long c0 = Rq.w ? 0 : min((long long)Rq.y * fp4::TILE, (long long)P.max_ctx);
    const float v = Rq.w ? __int_as_float(0x7fc00000) : -INFINITY;
    for (long long c = c0 + threadIdx.x; c < P.max_ctx; c += blockDim.x) {
        const size_t oi = (size_t)r * (size_t)P.out_stride + (size_t)c;
        if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = v;
        else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(v);
        else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(v);
    }
}

cudaError_t launch_plan(const PlanParams &P, const float *k_scale, int k_count, cudaStream_t s);

cudaError_t launch_fp4_logits(const Fp4Params &P, int ctas, cudaStream_t s) {
    if (P.B == 0) return cudaSuccess;
    pa_fp4_fill_kernel<<<P.B * P.n, 256, 0, s>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!P.rectify && P.n <= fp4::SUM_MAX_N) {
        // the plain weighted sum: one folded query vector per row, CUDA cores
        pa_fp4_fold_kernel<<<P.B * P.n, 128, 0, s>>>(P);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const dim3 g((unsigned)(ctas * fp4::SUM_CTAS_PER_SM));
        switch (P.n) {
            case 1: pa_fp4_logits_sum_kernel<1><<<g, fp4::SUM_THREADS, 0, s>>>(P); break;
            case 2: pa_fp4_logits_sum_kernel<2><<<g, fp4::SUM_THREADS, 0, s>>>(P); break;
            case 3: pa_fp4_logits_sum_kernel<3><<<g, fp4::SUM_THREADS, 0, s>>>(P); break;
            default: pa_fp4_logits_sum_kernel<4><<<g, fp4::SUM_THREADS, 0, s>>>(P); break;
        }
        return cudaGetLastError();
    }
    e = cudaFuncSetAttribute(pa_fp4_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fp4::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    pa_fp4_logits_kernel<<<ctas, fp4::THREADS, fp4::SMEM_BYTES, s>>>(P);
    return cudaGetLastError();
}

}  // namespace pa

// ------------------------------------------------------------------ host side

namespace {

size_t fp4_align(size_t x) { return (x + 255) / 256 * 256; }

// tiles (128 tokens) a request can have at most: the table width in tokens
long long fp4_tiles_per_seq(const pa_fp4_problem *p) {
    return ((long long)p->max_blocks_per_seq * p->block_size + pa::fp4::TILE - 1) / pa::fp4::TILE;
}

pa_status fp4_check(const pa_fp4_problem *p) {
    if (p == nullptr) return PA_ERR_INVALID_ARG;
    if (p->batch < 0 || p->next_n < 1 || p->num_heads < 1 || p->num_blocks < 1 || p->max_blocks_per_seq < 1 ||
        p->max_context_len < 0 || p->num_sms < 0 || p->grid_ctas < 0 || p->grid_ctas > (1 << 20) ||
        p->out_stride < 0)
        return PA_ERR_INVALID_ARG;
    if (p->out_dtype != PA_F32 && p->out_dtype != PA_F16 && p->out_dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if ((p->causal != 0 && p->causal != 1) || (p->rectify != 0 && p->rectify != 1) ||
        (p->sf_interleaved != 0 && p->sf_interleaved != 1))
        return PA_ERR_INVALID_ARG;
    if (p->out_stride != 0 && p->out_stride < p->max_context_len) return PA_ERR_INVALID_ARG;
    if (p->head_dim != 128 || p->sf_vec_size != 32) return PA_ERR_UNSUPPORTED;
    if (p->block_size != 16 && p->block_size != 32 && p->block_size != 64 && p->block_size != 128)
        return PA_ERR_UNSUPPORTED;
    if (p->num_heads % 16 != 0 || (long long)p->next_n * p->num_heads > pa::fp4::MAX_N) return PA_ERR_UNSUPPORTED;
    if ((long long)p->batch * fp4_tiles_per_seq(p) > 0x7fffffffll) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// header (64 B), request records (16 B each), folded query rows (fp32 [B][n][128])
size_t fp4_ws_bytes(const pa_fp4_problem *p) {
    return fp4_align(64) + fp4_align((size_t)p->batch * 16) + fp4_align((size_t)p->batch * p->next_n * 128 * 4);
}

}  // namespace

extern "C" {

PA_API pa_status pa_fp4_logits_workspace_size(const pa_fp4_problem *p, size_t *bytes) {
    if (bytes == nullptr) return PA_ERR_INVALID_ARG;
    const pa_status st = fp4_check(p);
    if (st != PA_OK) return st;
    *bytes = fp4_ws_bytes(p);
    return PA_OK;
}

PA_API pa_status pa_fp4_logits(const pa_fp4_problem *p, const uint8_t *q, const int32_t *sf_q,
                               const uint8_t *kv_fused, const float *weights, const int32_t *context_lens,
                               const int32_t *block_table, void *workspace, size_t workspace_bytes, void *out,
                               pa_stream_t stream) {
    pa_status st = fp4_check(p);
    if (st != PA_OK) return st;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
        workspace_bytes < fp4_ws_bytes(p))
        return PA_ERR_WORKSPACE;
    if (p->batch == 0) return PA_OK;
    const size_t esz = p->out_dtype == PA_F32 ? 4 : 2;
    if (q == nullptr || sf_q == nullptr || kv_fused == nullptr || weights == nullptr || context_lens == nullptr ||
        block_table == nullptr || out == nullptr)
        return PA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(kv_fused) & 15) ||
        (reinterpret_cast<uintptr_t>(sf_q) & 3) || (reinterpret_cast<uintptr_t>(weights) & 3) ||
        (reinterpret_cast<uintptr_t>(out) & (esz - 1)))
        return PA_ERR_INVALID_ARG;
    int sms = p->num_sms;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            return PA_ERR_CUDA;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    pa::PlanParams pp;
    pp.context_lens = context_lens;
    pp.hdr = reinterpret_cast<uint32_t *>(ws);
    pp.req = reinterpret_cast<int4 *>(ws + fp4_align(64));
    pp.B = p->batch;
    pp.bs = pa::fp4::TILE;  // the plan's pages are 128-token tiles
    pp.max_ctx = p->max_context_len;
    pp.mbps = (int)fp4_tiles_per_seq(p);
    pp.bsb = p->block_size;
    pp.tbl = p->max_blocks_per_seq;
    cudaError_t e = pa::launch_plan(pp, nullptr, 0, s);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    pa::Fp4Params P;
    P.q = q;
    P.sf_q = sf_q;
    P.kv = kv_fused;
    P.weights = weights;
    P.block_table = block_table;
    P.context_lens = context_lens;
    P.hdr = pp.hdr;
    P.req = pp.req;
    P.qw = reinterpret_cast<float *>(ws + fp4_align(64) + fp4_align((size_t)p->batch * 16));
    P.out = out;
    P.out_stride = p->out_stride > 0 ? p->out_stride : p->max_context_len;
    P.block_bytes = (long long)p->block_size * pa::fp4::ROWB;
    P.B = p->batch;
    P.n = p->next_n;
    P.H = p->num_heads;
    P.N = p->next_n * p->num_heads;
    P.bs = p->block_size;
    P.bpt = pa::fp4::TILE / p->block_size;
    P.num_blocks = p->num_blocks;
    P.tbl = p->max_blocks_per_seq;
    P.mbps = pp.mbps;
    P.max_ctx = p->max_context_len;
    P.out_dtype = p->out_dtype;
    P.causal = p->causal;
    P.rectify = p->rectify;
    P.interleaved = p->sf_interleaved;
    const int ctas = p->grid_ctas > 0 ? p->grid_ctas : sms;
    e = pa::launch_fp4_logits(P, ctas, s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
