// Single-latent-KV MQA decode / verify attention for sm_103a, on the fifth-
// generation tensor cores (tcgen05: operands in shared memory, accumulators in
// tensor memory).
//
// K and V live in one E4M3 plane per kv head: a token row holds 576 channels,
// V is its first 512, and every block ends with one fp32 scale per token
// (the layout of a "data region then scale region" block, FlashInfer docs,
// "flashinfer.fp4_paged_mqa_logits", Parameters).  With 128 query heads on
// one kv head and two query rows per request there are 256 query rows per
// request, so S = q K^T (576 deep) and O = P V (512 wide) are dense
// contractions.
//
// Work split: pages in logical order -- (request, kv head, page), never by
// physical id (1Cat-vLLM PR #494, "Stabilize QSA page4 order under KV
// relocation", Summary) -- shared evenly over groups of R/64 CTAs of a
// persistent launch, one CTA per SM; CTA i of a group computes query rows
// 64i..64i+63 (row block i) of every page of the group's share, so the group
// reads each page at about the same time and all but the first read hit L2.
// A CTA's run of pages inside one (request, kv head) is a piece; a piece that
// covers all of them writes `out`, the others write a normalised partial and
// its log-sum-exp to slot ((b*Hkv + kv head) + group)*G + i for the combine.
//
// Roles (10 warps), hand-offs through mbarriers whose waits are all bounded:
//  * warp 0 (producer): block ids (32 per load, range-checked) and the bulk
//    tensor copies of each page -- the codes as four 128-byte and one 64-byte
//    swizzled column boxes, exactly the K-major operand layout the MMA reads
//    -- plus the 256-byte scale tail, into a 2-slot ring;
//  * warp 1 (MMA): S = q' K^T as E4M3 x E4M3 MMAs (M = 64 query rows, N = 64
//    tokens, K = 32 channels per step) straight from the ring, q' given as
//    two E4M3 terms hi + lo that add up to the bf16 query exactly (a bf16
//    significand has 8 bits, each E4M3 term carries 4), into one of two S
//    buffers in tensor memory; then O^T += V^T P'^T as f16 MMAs (M = 128
//    channels, N = 64 query rows, K = 16 tokens) for four channel tiles, V^T
//    read MN-major from the dequantized V tile.  S(j+1) is issued before
//    O(j), so the tensor pipe works while page j's softmax runs;
//  * warps 2-5 (softmax, one query row per lane 0-15 of each warp -- the
//    M = 64 accumulator layout): scores scaled in fp32 by softmax_scale, the
//    row's power-of-two factor and the token scale, masked (t >= vis), online
//    softmax in the exp2 domain with a lazy maximum (O is rescaled only when
//    a row maximum grows by more than 2^6, or when the page-scale exponent E
//    leaves its band); P' = p * scale_t * 2^-E stored as f16 for the MMA, the
//    row sum keeps p; at the end of a piece they read O^T back, normalise
//    and write `out` or the partial.  They also stage q' for each piece;
//  * warps 6-9 (dequant): V codes of each page -> f16 tile (exact), token
//    slots past L_b zeroed, so neither NaN codes nor NaN scales in padding
//    reach P.V (1Cat-vLLM PR #647, "Stop grouped-page4 null-block padding
//    from leaking E4M3 NaN", Fix).
#include "pa_attn.cuh"
#include "pa_tc.cuh"

namespace pa {
namespace lat {

using namespace tc;

constexpr int DK = 576, DV = 512, BS = 64, LROWS = 64, NSLOT = 2;
constexpr int NWARPS = 10, THREADS = NWARPS * 32;
constexpr int W_PROD = 0, W_MMA = 1, W_SM = 2, W_DQ = 6;
// shared memory (offsets from a 1 KB aligned base)
constexpr int QH_OFF = 0;                              // q' hi, E4M3 [64 rows]: 4 x SW128 [64][128 B] + SW64 [64][64 B]
constexpr int QL_OFF = 36864;                          // q' lo, same layout
constexpr int RING_OFF = 73728;                        // NSLOT pages as copied, same layout
constexpr int SLOT_BYTES = 36864;
constexpr int V_OFF = RING_OFF + NSLOT * SLOT_BYTES;   // V f16 [8 x 64 channels][64 tokens][128 B], SW128
constexpr int P_OFF = V_OFF + 65536;                   // P' f16 [2][64 rows][64 tokens], SW128
constexpr int TSRAW_OFF = P_OFF + 2 * 8192;            // [NSLOT][64] token scales as copied
constexpr int ALPHA_OFF = TSRAW_OFF + NSLOT * 256;     // [2][64] O rescale factors
constexpr int STAT_OFF = ALPHA_OFF + 2 * 256;          // [64] 2^E / l, [64] lse
constexpr int NEED_OFF = STAT_OFF + 512;               // [2][4] rescale votes of the softmax warps
constexpr int BAR_OFF = NEED_OFF + 32;
enum {
    B_FULL = 0,                     // [NSLOT] page copied (tx bytes)
    B_SLOTFREE = B_FULL + NSLOT,    // [NSLOT] S MMAs done + dequant and softmax done reading
    B_SFULL = B_SLOTFREE + NSLOT,   // [2] S(j) complete
    B_SFREE = B_SFULL + 2,          // [2] S(j) read out
    B_PFULL = B_SFREE + 2,          // [2] P'(j) written (and O^T rescaled)
    B_PVDONE = B_PFULL + 2,         // [2] O^T += V^T P'(j)^T complete
    B_VFULL = B_PVDONE + 2,         // V tile of page j written
    B_QFULL = B_VFULL + 1,          // q' of the piece staged
    B_OFREE = B_QFULL + 1,          // O^T of the previous piece read out
    B_WG = B_OFREE + 1,             // the four softmax warps
    B_MDONE = B_WG + 1,             // every MMA of the CTA complete
    NBARS = B_MDONE + 1
};
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;          // [0] tmem base, [1] abort, [2 + s] slot s bad, [4] errors
constexpr int SMEM_USED = MISC_OFF + 64;
constexpr int SMEM_BYTES = SMEM_USED + 1024;           // + alignment of the base to 1 KB
constexpr uint32_t PAGE_TX = SLOT_BYTES + BS * 4;
constexpr uint32_t TM_S = 0, TM_O = 256;               // tensor-memory columns: S[2] x 64, O^T[4] x 64
constexpr float ROW_SLACK = 6.0f;                      // lazy maximum: rescale when a row max grows by > 2^6
static_assert(SMEM_BYTES <= 227 * 1024, "latent kernel exceeds the shared memory of one CTA");
static_assert(NSLOT == 2, "barrier counts below assume two ring slots");

// two fp32 -> two E4M3 codes (RNE, saturating), lo in the low byte
__device__ __forceinline__ uint32_t f32x2_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float2 e4m3x2_f32x2(uint32_t two_codes) {
    const uint32_t h = e4m3x2_f16x2(two_codes);
    __half2 hh;
    memcpy(&hh, &h, 4);
    return __half22float2(hh);
}

// byte offset of the 16-byte chunk c (0..35, 16 E4M3 channels each) of row r
// in a [4 x SW128 [64][128 B] | SW64 [64][64 B]] tile (the copied page layout)
__device__ __forceinline__ uint32_t e4_off(int r, int c) {
    if (c < 32) return (uint32_t)((c >> 3) * (64 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    return (uint32_t)(4 * 64 * 128 + r * 64 + ((((c - 32) & 3) ^ ((r >> 1) & 3)) << 4));
}

// byte offset of the 16-byte chunk c (0..63, 8 f16 channels each) of token t
// in the V tile [8][64 tokens][128 B]
__device__ __forceinline__ uint32_t v_off(int t, int c) {
    return (uint32_t)((c >> 3) * (64 * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// two consecutive q values of a packed word (low half first)
__device__ __forceinline__ float2 q_pair(uint32_t u, int q_dtype) {
    if (q_dtype == PA_BF16) return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    return make_float2(__half2float(__ushort_as_half((uint16_t)(u & 0xFFFFu))),
                       __half2float(__ushort_as_half((uint16_t)(u >> 16))));
}

}  // namespace lat

// After a wait ran out (or the records ran short): every piece of this CTA's
// share of positions [x0, x0 + npg) is written as NaN, finished or not, with
// no access to tensor memory -- outputs, or partial log-sum-exps that the
// combine turns into NaN rows -- so no row keeps stale values.  Run by the
// 128 threads of the softmax warps (ti = 0..127); kept out of line so that
// the main loop's registers are not shaped by it.
__device__ __noinline__ void latent_nan_share(const LatentParams &P, long long x0, int npg, int U, int GS, long long kg,
                                              int rb, int ti) {
    using namespace lat;
    const float NaN = __int_as_float(0x7fc00000);
    auto nan_piece = [&](int b_, int q_, int p0_, int pl_) {
        const int Pb = planned_pages(P.req, b_, P.mbps);
        const bool complete = (p0_ == 0 && pl_ == Pb - 1);
        const long long slot_id = ((long long)b_ * U + q_ + kg) * GS + rb;
        for (int rr = 0; rr < LROWS; ++rr) {
            const int r = rb * LROWS + rr;
            if (r >= P.R) break;
            const int jq = r / P.G, h = q_ * P.G + r % P.G;
            if (complete) {
                const size_t row = (((size_t)b_ * P.n + jq) * P.Hq + h) * DV;
                for (int d = ti; d < DV; d += 128) {
                    if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[row + d] = NaN;
                    else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[row + d] = __float2half_rn(NaN);
                    else reinterpret_cast<__nv_bfloat16 *>(P.out)[row + d] = __float2bfloat16_rn(NaN);
                }
                if (ti == 0 && P.lse != nullptr) P.lse[((size_t)b_ * P.n + jq) * P.Hq + h] = NaN;
            } else if (ti == 0) {
                P.part_lse[(size_t)slot_id * LROWS + rr] = NaN;
            }
        }
    };
    Cursor cw = cursor_at(x0, P.req, P.B, U, P.mbps);
    int wb = -1, wq = -1, wp0 = 0, wl = 0;
    for (int j = 0; j < npg && cw.b < P.B; ++j) {
        if (cw.b != wb || cw.q != wq) {
            if (wb >= 0) nan_piece(wb, wq, wp0, wl);
            wb = cw.b;
            wq = cw.q;
            wp0 = cw.p;
        }
        wl = cw.p;
        cursor_next(cw, P.req, P.B, U, P.mbps);
    }
    if (wb >= 0) nan_piece(wb, wq, wp0, wl);
}

__global__ void __launch_bounds__(lat::THREADS, 1)
    pa_latent_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                     LatentParams P) {
    using namespace lat;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    int *misc = reinterpret_cast<int *>(smem + MISC_OFF);
    volatile int *abort = misc + 1;
    const float *tsraw = reinterpret_cast<const float *>(smem + TSRAW_OFF);
    float *alpha = reinterpret_cast<float *>(smem + ALPHA_OFF);
    float *stat_f = reinterpret_cast<float *>(smem + STAT_OFF);
    float *stat_lse = stat_f + 64;
    volatile int *need = reinterpret_cast<volatile int *>(smem + NEED_OFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int GS = P.RBLK;                 // CTAs per group: one per row block
    const int rb = (int)(blockIdx.x % GS);  // this CTA's row block
    const int U = P.Hkv;                   // units (kv heads) per request

    grid_dependency_wait();
    const long long total = P.hdr[HDR_TOTAL_PAGES];
    if (total > (long long)P.B * P.mbps) {
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    const long long Ntot = total * U;
    const long long NG = gridDim.x / GS;
    const long long kg = blockIdx.x / GS;  // this CTA's group
    if (kg >= NG) return;                  // the host launches whole groups
    const long long x0 = kg * Ntot / NG, x1 = (kg + 1) * Ntot / NG;
    if (x0 >= x1) return;
    const int npg = (int)(x1 - x0);
    const Cursor c0 = cursor_at(x0, P.req, P.B, U, P.mbps);
    if (c0.b >= P.B) {  // uniform: every thread computed the same cursor
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }

    // ---- setup: barriers, tensor memory (512 columns, one CTA per SM)
    if (tid == 0) {
        const uint32_t counts[NBARS] = {1, 1, 9, 9, 1, 1, 4, 4, 4, 4, 1, 1, 4, 4, 4, 4, 1};
        for (int i = 0; i < NBARS; ++i) mbar_init(&bars[i], counts[i]);
        misc[1] = 0;
        misc[4] = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tma);
        tma_prefetch_desc(&tmb);
    }
    if (warp == W_PROD) {
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
        // ================================================== producer
        Cursor ci = c0;
        int idc_b = -1, idc_w0 = 0, idc = 0, issued = 0;
#ifdef PA_FAULT_INJECT
        const unsigned fi_withhold = P.hdr[HDR_WITHHOLD];
#endif
        for (int j = 0; j < npg; ++j) {
            const int slot = j % NSLOT;
            if (j >= NSLOT && !warp_wait(&bars[B_SLOTFREE + slot], ((j / NSLOT) - 1) & 1, abort, err)) break;
#ifdef PA_FAULT_INJECT
            if (fi_withhold != 0 && x0 + j + 1 == (long long)fi_withhold && ci.b < P.B) {
                ++issued;
                cursor_next(ci, P.req, P.B, U, P.mbps);
                continue;  // no copy and no arrive: the waits on this slot run out
            }
#endif
            bool ok = false;
            int blk = 0;
            if (ci.b < P.B) {
                if (ci.b != idc_b || ci.p < idc_w0 || ci.p >= idc_w0 + 32) {
                    idc_b = ci.b;
                    idc_w0 = ci.p;
                    const int pg = idc_w0 + lane;
                    idc = (pg < ci.Pb) ? P.block_table[(size_t)ci.b * P.mbps + pg] : 0;
                }
                blk = __shfl_sync(0xffffffffu, idc, ci.p - idc_w0);
                ok = blk >= 1 && blk < P.num_blocks;
            }
            if (lane == 0) {
                misc[2 + slot] = ok ? 0 : 1;
                uint64_t *bar = &bars[B_FULL + slot];
                if (ok) {
                    const int kvh = ci.q;
                    uint8_t *dst = smem + RING_OFF + slot * SLOT_BYTES;
                    mbar_arrive_expect_tx(bar, PAGE_TX);
#pragma unroll
                    for (int sg = 0; sg < 4; ++sg) tma_load_4d(dst + sg * BS * 128, &tma, bar, sg * 128, 0, kvh, blk);
                    tma_load_4d(dst + 4 * BS * 128, &tmb, bar, 512, 0, kvh, blk);
                    const uint8_t *src = P.k_pool + (size_t)blk * P.block_stride + P.codes_bytes + (size_t)kvh * BS * 4;
                    bulk_load(smem + TSRAW_OFF + slot * BS * 4, src, BS * 4, bar);
                } else {
                    mbar_arrive(bar);  // no copy: the piece is NaN-filled
                }
            }
            __syncwarp();
            ++issued;
            if (ci.b < P.B) cursor_next(ci, P.req, P.B, U, P.mbps);
        }
        if (*abort && lane == 0) {
            // let every copy still in flight land before the CTA exits
            for (int i = max(0, issued - NSLOT); i < issued; ++i)
                (void)mbar_wait_bounded(&bars[B_FULL + i % NSLOT], (i / NSLOT) & 1, nullptr);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ================================================== MMA issue
        constexpr uint32_t ID_QK = idesc(64, 64, 0), ID_PV = idesc(128, 64, 1);
        Cursor cq = c0, cp = c0;
        const uint64_t qh128 = sdesc(sb + QH_OFF, 16, 1024, 2), qh64 = sdesc(sb + QH_OFF, 16, 512, 4);
        const uint64_t ql128 = sdesc(sb + QL_OFF, 16, 1024, 2), ql64 = sdesc(sb + QL_OFF, 16, 512, 4);
        int q_piece = -1, q_pb = -1, q_pq = -1;  // pieces seen by the S stream
        int p_piece = -1, p_pb = -1, p_pq = -1;  // pieces seen by the O stream
        auto issue_s = [&](int j) -> bool {
            if (cq.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; return false; }
            const int slot = j % NSLOT, sbuf = j & 1;
            if (cq.b != q_pb || cq.q != q_pq) {
                ++q_piece;
                q_pb = cq.b;
                q_pq = cq.q;
                if (!lane_wait(&bars[B_QFULL], q_piece & 1, abort, err)) return false;
            }
            if (!lane_wait(&bars[B_FULL + slot], (j / NSLOT) & 1, abort, err)) return false;
            if (j >= 2 && !lane_wait(&bars[B_SFREE + sbuf], ((j >> 1) - 1) & 1, abort, err)) return false;
            tc_fence_after();
            // descriptors of the step's operands: the tile base's descriptor plus
            // the step's offset in 16-byte units (no carry out of the 14-bit
            // address field: shared memory ends below 256 KB)
            const uint32_t ring = sb + RING_OFF + slot * SLOT_BYTES;
            const uint64_t r128 = sdesc(ring, 16, 1024, 2), r64 = sdesc(ring, 16, 512, 4);
            {
                const uint32_t dS = tmem + TM_S + 64u * sbuf;
                uint32_t acc = 0;
#pragma unroll
                for (int cb = 0; cb < 5; ++cb) {
#pragma unroll
                    for (int ks = 0; ks < (cb < 4 ? 4 : 2); ++ks) {
                        const uint64_t off = (uint64_t)(cb * 512 + 2 * ks);
                        const uint64_t bdesc = (cb < 4 ? r128 : r64) + off;
                        mma_f8(dS, (cb < 4 ? qh128 : qh64) + off, bdesc, ID_QK, acc);
                        acc = 1;
                        mma_f8(dS, (cb < 4 ? ql128 : ql64) + off, bdesc, ID_QK, 1);
                    }
                }
                mma_commit(&bars[B_SFULL + sbuf]);
                mma_commit(&bars[B_SLOTFREE + slot]);
            }
            cursor_next(cq, P.req, P.B, U, P.mbps);
            return true;
        };
        auto issue_o = [&](int j) -> bool {
            const int pbuf = j & 1;
            bool first = false;
            if (cp.b != p_pb || cp.q != p_pq) {
                ++p_piece;
                p_pb = cp.b;
                p_pq = cp.q;
                first = true;
                if (p_piece > 0 && !lane_wait(&bars[B_OFREE], (p_piece - 1) & 1, abort, err)) return false;
            }
            if (!lane_wait(&bars[B_PFULL + pbuf], (j >> 1) & 1, abort, err)) return false;
            if (!lane_wait(&bars[B_VFULL], j & 1, abort, err)) return false;
            tc_fence_after();
            const uint64_t vb = sdesc(sb + V_OFF, 8192, 1024, 2), pbd = sdesc(sb + P_OFF + pbuf * 8192, 16, 1024, 2);
            {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t dO = tmem + TM_O + 64u * i;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t adesc = vb + (uint64_t)(((2 * i) * (64 * 128) + 2048 * k) >> 4);
                        const uint64_t bdesc = pbd + (uint64_t)((32 * k) >> 4);
                        mma_f16(dO, adesc, bdesc, ID_PV, (first && k == 0) ? 0u : 1u);
                    }
                }
                mma_commit(&bars[B_PVDONE + pbuf]);
            }
            cursor_next(cp, P.req, P.B, U, P.mbps);
            return true;
        };
        // lane 0 runs this role alone (its waits need no broadcast); the other
        // lanes wait at the warp barrier below
        if (lane == 0) {
            if (issue_s(0)) {
                for (int j = 0; j < npg; ++j) {
                    if (j + 1 < npg && !issue_s(j + 1)) break;
                    if (!issue_o(j)) break;
                }
            }
            // every MMA issued so far is complete before tensor memory is released
            mma_commit(&bars[B_MDONE]);
            (void)mbar_wait_bounded(&bars[B_MDONE], 0, nullptr);
        }
        __syncwarp();
    } else if (warp >= W_SM && warp < W_SM + 4) {
        // ================================================== softmax, q staging, epilogue
        const int qd = warp & 3;                 // tensor-memory lane quarter
        const bool owner = lane < 16;            // lanes whose TMEM lane holds the row of S
        const int half = lane >> 4;              // tokens 32 * half .. of the row
        const int row = 16 * qd + (lane & 15);   // this lane's row
        const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
        Cursor cs = c0;
        int piece = -1, pb = -1, pq = -1, p0 = 0, last_p = 0, kvh = 0, rblk = 0, L = 0;
        int wg_phase = 0;
        float m = -INFINITY, lsum = 0.f, rowsc = 0.f;
        int vis = 0, E_run = 0;
        bool E_set = false, pbad = false;
        const float NaN = __int_as_float(0x7fc00000);

        // q' of segment (cs.b, kvh_n, rblk_n): row `row`, channel half (lane >> 4)
        auto stage_q = [&](int kvh_n, int rblk_n) -> float {
            const int r = rblk_n * LROWS + row;
            const bool rok = r < P.R;
            size_t qbase = 0;
            if (rok) {
                const int jq = r / P.G, h = kvh_n * P.G + r % P.G;
                qbase = (((size_t)cs.b * P.n + jq) * P.Hq + h) * DK;
            }
            const uint8_t *qrow = P.q + 2 * qbase;
            float mx = 0.f;
            if (rok) {
#pragma unroll 6
                for (int c = 18 * half; c < 18 * half + 18; ++c) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(qrow + 32 * c);
                    const uint4 w = *reinterpret_cast<const uint4 *>(qrow + 32 * c + 16);
                    const uint32_t u[8] = {v.x, v.y, v.z, v.w, w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 f = q_pair(u[e], P.q_dtype);
                        mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
                    }
                }
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            // q * 2^s has its largest magnitude in [128, 256): both E4M3 terms stay finite
            int ex = 0;
            const bool fin = mx > 0.f && mx < 3.0e38f;
            if (fin) frexpf(mx, &ex);
            const int s = fin ? 8 - ex : 0;
            const float up = pow2f(s);
#pragma unroll 3
            for (int c = 18 * half; c < 18 * half + 18; ++c) {
                uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
                if (rok) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(qrow + 32 * c);
                    const uint4 w = *reinterpret_cast<const uint4 *>(qrow + 32 * c + 16);
                    const uint32_t u[8] = {v.x, v.y, v.z, v.w, w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 f = q_pair(u[e], P.q_dtype);
                        const float a = f.x * up, b = f.y * up;
                        const uint32_t h2 = f32x2_e4m3x2(a, b);
                        const float2 hf = e4m3x2_f32x2(h2);
                        const uint32_t l2 = f32x2_e4m3x2(a - hf.x, b - hf.y);
                        hw[e >> 1] |= h2 << (16 * (e & 1));
                        lw[e >> 1] |= l2 << (16 * (e & 1));
                    }
                }
                *reinterpret_cast<uint4 *>(smem + QH_OFF + e4_off(row, c)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(smem + QL_OFF + e4_off(row, c)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            return rok ? P.softmax_scale * LOG2E * pow2f(-s) : 0.f;
        };

        // read O^T of the finished piece (last page jl), normalise, write out / partial
        auto epilogue = [&](int jl) -> bool {
            const int Pb = planned_pages(P.req, pb, P.mbps);
            const bool complete = (p0 == 0 && last_p == Pb - 1);
            const long long slot_id = ((long long)pb * U + pq + kg) * GS + rb;
            const int r0 = rblk * LROWS;
            const float lrow = lsum + __shfl_xor_sync(0xffffffffu, lsum, 16);
            if (owner) {
                const bool lok = lrow > 0.f;
                stat_f[row] = pbad ? NaN : (lok ? pow2f(E_run) / lrow : 0.f);
                float lse_v = lok ? (m + lg2(lrow)) * LN2 : -INFINITY;
                if (pbad) lse_v = NaN;
                stat_lse[row] = lse_v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_WG]);
            if (!warp_wait(&bars[B_WG], wg_phase & 1, abort, err)) return false;
            ++wg_phase;
            if (!warp_wait(&bars[B_PVDONE + (jl & 1)], (jl >> 1) & 1, abort, err)) return false;
            tc_fence_after();
            if (owner && r0 + row < P.R) {
                const int r = r0 + row, jq = r / P.G, h = kvh * P.G + r % P.G;
                if (complete) {
                    if (P.lse != nullptr) P.lse[((size_t)pb * P.n + jq) * P.Hq + h] = stat_lse[row];
                } else {
                    P.part_lse[(size_t)slot_id * LROWS + row] = stat_lse[row];
                }
            }
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const int d = 128 * i + 32 * qd + lane;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    float o[32];
                    tmem_ld32(tl + TM_O + 64u * i + 32u * half, o);
                    // row r = r0 + 32 half + k is query row jq, head kvh G + g: both
                    // advanced by one row at a time instead of a division per element
                    int jq = (r0 + 32 * half) / P.G, g = (r0 + 32 * half) % P.G;
#pragma unroll 4
                    for (int k = 0; k < 32; ++k, ++g) {
                        if (g == P.G) { g = 0; ++jq; }
                        const int rr = 32 * half + k;
                        const int r = r0 + rr;
                        if (r >= P.R) break;
                        const float y = o[k] * stat_f[rr];
                        if (complete) {
                            const int h = kvh * P.G + g;
                            const size_t oi = (((size_t)pb * P.n + jq) * P.Hq + h) * DV + d;
                            if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = y;
                            else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(y);
                            else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(y);
                        } else {
                            P.part_o[((size_t)slot_id * LROWS + rr) * DV + d] = y;
                        }
                    }
                }
            }
            tc_fence_before();
            warp_arrive(&bars[B_OFREE]);
            return true;
        };

        bool alive = true;
        int j = 0;
        for (; j < npg; ++j) {
            if (cs.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; alive = false; break; }
            const int slot = j % NSLOT, sbuf = j & 1;
            const bool first = (cs.b != pb || cs.q != pq);
            if (first) {
                // stage q' of the new piece first (its S MMAs wait for it), then
                // finish the previous piece (whose last O MMAs are already queued)
                const float rowsc_new = stage_q(cs.q, rb);
                fence_proxy_async_smem();
                warp_arrive(&bars[B_QFULL]);
                if (piece >= 0 && !epilogue(j - 1)) { alive = false; break; }
                ++piece;
                pb = cs.b;
                pq = cs.q;
                p0 = cs.p;
                kvh = cs.q;
                rblk = rb;
                const int4 Rq = P.req[cs.b];
                L = P.context_lens[cs.b];
                pbad = false;
                if (Rq.w != 0) { pbad = true; err |= PA_DEV_ERR_CONTEXT_LEN; }
                if (L != Rq.x) { pbad = true; err |= PA_DEV_ERR_STALE_PLAN; }
                const int r = rblk * LROWS + row;
                vis = (r < P.R && P.causal) ? L - (P.n - 1 - r / P.G) : L;
                rowsc = rowsc_new;
                {
                    // the next segment's q rows of this row block into L2, so that its
                    // q' staging reads L2 rather than DRAM
                    const int nb = pq + 1 < U ? pb : pb + 1, nq = pq + 1 < U ? pq + 1 : 0;
                    if (nb < P.B && r < P.R) {
                        const int jq = r / P.G, h = nq * P.G + r % P.G;
                        const uint8_t *qa = P.q + 2 * ((((size_t)nb * P.n + jq) * P.Hq + h) * DK) + 576 * half;
#pragma unroll
                        for (int k = 0; k < 5; ++k) asm volatile("prefetch.global.L2 [%0];" ::"l"(qa + 128 * k));
                    }
                }
                m = -INFINITY;
                lsum = 0.f;
                E_set = false;
            }
            // ---- scores of page j: lane l < 16 takes tokens 0..31 of row 16qd + l,
            // lane l + 16 tokens 32..63 of the same row
            if (!warp_wait(&bars[B_SFULL + sbuf], (j >> 1) & 1, abort, err)) { alive = false; break; }
            if (!warp_wait(&bars[B_FULL + slot], (j / NSLOT) & 1, abort, err)) { alive = false; break; }
            tc_fence_after();
            float x[32];
            {
                float xa[32], xb[32];
                tmem_ld32(tl + TM_S + 64u * sbuf, xa);
                tmem_ld32(tl + TM_S + 64u * sbuf + 32u, xb);
                tc_fence_before();
                warp_arrive(&bars[B_SFREE + sbuf]);
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float up = __shfl_up_sync(0xffffffffu, xb[k], 16);
                    x[k] = half ? up : xa[k];
                }
            }
            if (misc[2 + slot]) { pbad = true; err |= PA_DEV_ERR_BLOCK_ID; }
            const int nvalid = min(BS, max(0, L - cs.p * BS));
            float ts[32];
            {
                const float4 *tq = reinterpret_cast<const float4 *>(tsraw + slot * BS + 32 * half);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 v = tq[k];
                    ts[4 * k] = v.x; ts[4 * k + 1] = v.y; ts[4 * k + 2] = v.z; ts[4 * k + 3] = v.w;
                }
            }
            warp_arrive(&bars[B_SLOTFREE + slot]);  // the ring slot is no longer read here
            const int t0 = 32 * half;
            float sm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                ts[k] = (t0 + k < nvalid) ? ts[k] : 0.f;
                sm4[k & 3] = fmaxf(sm4[k & 3], fabsf(ts[k]));
            }
            // the page's scale exponent (the same in every thread)
            float smax = fmaxf(fmaxf(sm4[0], sm4[1]), fmaxf(sm4[2], sm4[3]));
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 16));
            float aE = 1.f;
            if (smax > 0.f && smax < 3.0e38f) {
                int e;
                frexpf(smax, &e);
                e = min(max(e, -120), 120);
                if (!E_set) {
                    E_run = e;
                    E_set = true;
                } else if (e > E_run + 4 || e < E_run - 8) {
                    aE = pow2f(E_run - e);
                    E_run = e;
                }
            }
            const float nE = pow2f(-E_run);
            const int tv = vis - cs.p * BS - t0;  // tokens of this half that are visible: k < tv
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                x[k] = (k < tv) ? x[k] * rowsc * ts[k] : -INFINITY;
                mx4[k & 3] = fmaxf(mx4[k & 3], x[k]);
            }
            float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            // alm rescales the row sum (p carries no token scale); O^T also takes aE
            float alm = 1.f;
            if (mx > m + ROW_SLACK) {  // also true for m = -inf and a finite maximum
                if (m != -INFINITY) alm = ex2(m - mx);
                m = mx;
            }
            const float base = (m == -INFINITY) ? 0.f : m;
            float al = alm * aE;
            if (first) al = 1.f;  // O^T is overwritten by the piece's first P.V
            const bool resc = (al != 1.f);
            float ps4[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pw[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                const float a = ex2(x[k] - base), b = ex2(x[k + 1] - base);
                ps4[(k >> 1) & 3] += a + b;
                pw[k >> 1] = pack_f16x2(a * ts[k] * nE, b * ts[k + 1] * nE);
            }
            lsum = lsum * alm + ((ps4[0] + ps4[1]) + (ps4[2] + ps4[3]));  // this half's share of the row sum
            // P'(j) goes into buffer sbuf: the O MMAs of page j-2 must be done with it
            if (j >= 2 && !warp_wait(&bars[B_PVDONE + sbuf], ((j >> 1) - 1) & 1, abort, err)) { alive = false; break; }
            {
                uint8_t *prow = smem + P_OFF + sbuf * 8192 + row * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(prow + (((4 * half + c) ^ (row & 7)) << 4)) =
                        make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                if (owner) alpha[sbuf * 64 + row] = al;
            }
            const int vote = __any_sync(0xffffffffu, resc) ? 1 : 0;
            if (lane == 0) need[sbuf * 4 + qd] = vote;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_WG]);
            if (!warp_wait(&bars[B_WG], wg_phase & 1, abort, err)) { alive = false; break; }
            ++wg_phase;
            if (need[sbuf * 4] | need[sbuf * 4 + 1] | need[sbuf * 4 + 2] | need[sbuf * 4 + 3]) {
                // rescale the O^T columns (query rows) of this lane quarter once page j-1's O is in
                if (!warp_wait(&bars[B_PVDONE + (sbuf ^ 1)], ((j - 1) >> 1) & 1, abort, err)) { alive = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        float o[32];
                        const uint32_t ta = tl + TM_O + 64u * i + 32u * half;
                        tmem_ld32(ta, o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] *= alpha[sbuf * 64 + 32 * half + k];
                        tmem_st32(ta, o);
                    }
                }
                tc_fence_before();
            }
            warp_arrive(&bars[B_PFULL + sbuf]);
            last_p = cs.p;
            cursor_next(cs, P.req, P.B, U, P.mbps);
        }
        if (alive && piece >= 0) (void)epilogue(npg - 1);
        if (!alive) latent_nan_share(P, x0, npg, U, GS, kg, rb, tid - 32 * W_SM);
    } else {
        // ================================================== V dequant
        const int dt = tid - 32 * W_DQ;  // 0..127
        Cursor cd = c0;
        int pb = -1, pq = -1, L = 0;
        for (int j = 0; j < npg; ++j) {
            if (cd.b >= P.B) break;
            const int slot = j % NSLOT;
            if (cd.b != pb || cd.q != pq) {
                pb = cd.b;
                pq = cd.q;
                L = P.context_lens[cd.b];
            }
            if (!warp_wait(&bars[B_FULL + slot], (j / NSLOT) & 1, abort, err)) break;
            const int nvalid = min(BS, max(0, L - cd.p * BS));
            const uint8_t *pg8 = smem + RING_OFF + slot * SLOT_BYTES;
            // the codes go to registers first, so the ring slot is released at once.
            // A warp instruction covers tokens t and t^5 (4 lanes each per 8-lane
            // phase): under the XOR swizzle their loads fall in different halves
            // and their stores in even / odd chunk slots, so neither conflicts.
            const int w4 = dt >> 5, ln = dt & 31;
            const int ph = ln >> 3, sub = (ln >> 2) & 1, q4 = ln & 3;
            uint4 cv[16];
#pragma unroll
            for (int it = 0; it < 16; ++it) {
                const int combo = it * 4 + w4;            // 32 token pairs x 2 channel halves
                const int pair = combo >> 1, hh = combo & 1;
                const int t = (8 * (pair >> 2) + (pair & 3)) ^ (sub ? 5 : 0);
                const int c16 = 16 * hh + 4 * ph + q4;
                cv[it] = (t < nvalid) ? *reinterpret_cast<const uint4 *>(pg8 + e4_off(t, c16)) : make_uint4(0u, 0u, 0u, 0u);
            }
            warp_arrive(&bars[B_SLOTFREE + slot]);
            if (j >= 1 && !warp_wait(&bars[B_PVDONE + ((j - 1) & 1)], ((j - 1) >> 1) & 1, abort, err)) break;
#pragma unroll
            for (int it = 0; it < 16; ++it) {
                const int combo = it * 4 + w4;
                const int pair = combo >> 1, hh = combo & 1;
                const int t = (8 * (pair >> 2) + (pair & 3)) ^ (sub ? 5 : 0);
                const int c16 = 16 * hh + 4 * ph + q4;
                const uint32_t w[4] = {cv[it].x, cv[it].y, cv[it].z, cv[it].w};
                uint32_t h[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    h[2 * e] = e4m3x2_f16x2(w[e]);
                    h[2 * e + 1] = e4m3x2_f16x2(w[e] >> 16);
                }
                *reinterpret_cast<uint4 *>(smem + V_OFF + v_off(t, 2 * c16)) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(smem + V_OFF + v_off(t, 2 * c16 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
            }
            fence_proxy_async_smem();
            warp_arrive(&bars[B_VFULL]);
            cursor_next(cd, P.req, P.B, U, P.mbps);
        }
    }

    // ---- teardown: one error word per CTA, tensor memory released
    grid_dependents_launch();
    if (err) atomicOr(reinterpret_cast<unsigned *>(misc + 4), err);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_PROD)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    if (tid == 0) atomic_or_err(P.hdr, (uint32_t)misc[4]);
}

cudaError_t launch_latent(const CUtensorMap &ta, const CUtensorMap &tb, const LatentParams &P, int ctas,
                          cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(pa_latent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lat::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = launch_pdl(pa_latent_kernel, dim3((unsigned)ctas), dim3(lat::THREADS), (size_t)lat::SMEM_BYTES, s, ta, tb, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace pa
