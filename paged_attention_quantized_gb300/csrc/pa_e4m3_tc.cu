// E4M3 paged decode / verify attention at head dim 256 with 16..64 query rows
// per kv head, on the fifth-generation tensor cores (tcgen05).
//
// The shapes of the FP8 verify batches (next_n query rows times the query
// heads of a kv head: 16 rows at next_n = 4, 64 rows at next_n = 16) are too
// few rows for rows-on-M MMAs and too many for the warp-level kernel's
// registers.  Here tokens are the MMA M axis and the rows its N axis:
//
//   S^T = K [q'_hi | q'_lo]^T   M = 128 tokens (one chunk), N = 2R, K = 256
//                     channels, E4M3 x E4M3 (kind::f8f6f4): K straight from
//                     the copied codes, q' as two E4M3 terms that add up to
//                     the query exactly (row scaled by a power of two first),
//                     side by side on N so that K is read once; the two halves
//                     of S^T are added in fp32;
//   O^T += V^T [P_0 | P_1 | P_2]^T   M = 128 channels (two tiles), N = 3R,
//                     K = 128 tokens, E4M3 x E4M3: V^T read channel-major
//                     straight from the copied V codes, P^T as three E4M3
//                     terms of 4 significant bits each (12 bits in all, more
//                     than the f16 P of the warp-level kernel), side by side
//                     on N; the three partial sums are added in the epilogue.
//
// Work split: chunks of 128 logical tokens of one (request, kv head) in
// logical order -- never by physical id (1Cat-vLLM PR #494, "Stabilize QSA
// page4 order under KV relocation", Summary) -- shared evenly by persistent
// CTAs, one per SM; a CTA's run of chunks inside one (request, kv head) is a
// piece, whole pieces write `out`, cut ones a normalised partial for the
// combine (one segment per kv head: all R rows).
//
// Roles (3 + 4 G warps, G = 2 softmax groups, 4 at 64 rows):
//  * warp 0 and the last warp copy K and V of each chunk into their own
//    rings (tensor copies of one block's 128-channel half, 128-byte swizzled:
//    the K-major operand layout), with an L2 evict-first policy since every
//    page is read once; K is released as soon as the chunk's S MMAs are
//    done, V after its O MMAs.  Blocks past the request's length and blocks
//    with an invalid id are not copied;
//  * lane 0 of warp 1 issues the MMAs: S(j+1) before O(j), so the tensor
//    pipe works while chunk j's softmax runs;
//  * warps 2 .. 4G+1, G groups of four (one token per thread: S^T has tokens
//    on the tensor-memory lanes; each group owns R/G rows) run the online
//    softmax in the exp2 domain with a lazy reference maximum (a chunk
//    reduces the maxima across the 128 tokens, and rescales O^T, only when
//    some score passes its row's reference by more than 0.75; the reference
//    then moves to one above the chunk's maximum), zero the V rows past the
//    request's length before the chunk's O MMAs (uncopied rows, or slots of
//    the last block that may hold NaN codes: 1Cat-vLLM PR #647, "Stop
//    grouped-page4 null-block padding from leaking E4M3 NaN", Fix), write
//    P^T (times 2^8, so small weights stay E4M3 normals; K-major, or MN-major
//    at 32 and 64 rows), stage q' at each piece (and fetch the next piece's record
//    and q rows ahead) and write the output at its end.
// Every wait is bounded (PA_DEV_ERR_TIMEOUT); after a timeout every piece of
// the CTA's share is written as NaN.
#include "pa_attn.cuh"
#include "pa_tc.cuh"

namespace pa {


namespace e4tc {

using namespace tc;

constexpr int D = 256, CH = 128;  // head dim, tokens per chunk
constexpr int W_KPROD = 0, W_MMA = 1, W_SM0 = 2;  // then the softmax groups of 4 warps, then the V producer
constexpr int TILE = 2 * CH * 128;                  // one K or V stage: [2 channel halves][128 tokens][128 B]
// lazy maximum (exp2 domain): the reference m is moved only when a score
// passes it by more than SLACK, and then to the chunk's maximum plus HEAD, so
// that p = 2^(s - m) stays below 2^SLACK and a new maximum must climb
// HEAD + SLACK before O^T is rescaled again; P^T is stored as p * 2^8 =
// 2^(s - m + 8) (at most 431 < 448) so that weights down to 2^-14 of the
// maximum are E4M3 normals in every term; the row sums carry the same 2^8
constexpr float SLACK = 0.75f, HEAD = 1.0f;
constexpr float PSHIFT = 8.0f;

template <int N>
struct Lay {
    static constexpr int NWG = (N >= 64) ? 4 : 2;   // softmax warpgroups, each owning NR rows
    static constexpr int NR = N / NWG;
    static constexpr int W_VPROD = W_SM0 + 4 * NWG;
    static constexpr int NWARPS = W_VPROD + 1, THREADS = NWARPS * 32;
    // tensor memory: SB buffers of S^T (2N columns: the hi and lo halves of
    // q'), then O^T as two channel tiles of 3N columns (one per P^T term)
    static constexpr int SB = (10 * N <= 512) ? 2 : 1;
    static constexpr int TM_O = SB * 2 * N;
    static constexpr int TM_COLS = (TM_O + 6 * N <= 256) ? 256 : 512;
    static_assert(TM_O + 6 * N <= 512, "tensor memory of one CTA exceeded");
    static constexpr int Q_OFF = 0;                  // q' [2 halves][N hi rows, N lo rows][128 B]
    static constexpr int Q_BYTES = 2 * 2 * N * 128;
    static constexpr int P_OFF = Q_OFF + Q_BYTES;    // P^T [2 buffers][3 terms x N rows][128 B]
    static constexpr int P_TERM = N * 128;
    static constexpr int P_BUF = 3 * P_TERM;
    // at 32 and 64 rows P^T is stored MN-major (each token's N row values of
    // a term contiguous, a 32- or 64-byte swizzle, one block of 128 N bytes
    // per term), so a softmax group writes its 16 rows of a term with one
    // 16-byte store
    static constexpr bool PMN = (N == 64 || N == 32);
    static constexpr uint32_t PMN_SWZ = (N == 64) ? 4u : 6u;  // descriptor swizzle: 64 B, 32 B
    static constexpr int NK = (N <= 48) ? 3 : 2;     // K stages
    static constexpr int NV = (N <= 16) ? 3 : 2;     // V stages
    static constexpr int K_OFF = P_OFF + 2 * P_BUF;
    static constexpr int V_OFF = K_OFF + NK * TILE;
    // per-row constants, double-buffered by piece parity: running maxima [2 pieces][2][64]
    // (flip-buffered within a piece), score scale [2][64], visible length [2][64]
    static constexpr int M_OFF = V_OFF + NV * TILE;
    static constexpr int RS_OFF = M_OFF + 4 * 64 * 4;
    static constexpr int VIS_OFF = RS_OFF + 2 * 64 * 4;
    static constexpr int RED_OFF = VIS_OFF + 2 * 64 * 4;     // [4][64] per-warp reductions
    static constexpr int NEED_OFF = RED_OFF + 4 * 64 * 4;    // [4 groups][2][4] votes
    static constexpr int ALPHA_OFF = NEED_OFF + 128;         // [64] O^T factors of a rescale
    static constexpr int VBAD_OFF = ALPHA_OFF + 256;           // [NV] the chunk in V stage s had an invalid block id
    static constexpr int BAR_OFF = VBAD_OFF + 64;
    enum {
        B_KFULL = 0,                     // [3] K of a chunk landed (tensor copies)
        B_KFREE = B_KFULL + 3,           // [3] its S MMAs complete
        B_VFULL = B_KFREE + 3,           // [3] V of a chunk landed
        B_VFREE = B_VFULL + 3,           // [3] its O MMAs complete
        B_SFULL = B_VFREE + 3,           // [2]
        B_SFREE = B_SFULL + 2,           // [2]
        B_PFULL = B_SFREE + 2,           // [2] P^T written, O^T rescaled, V padding zeroed
        B_ODONE = B_PFULL + 2,           // [2] O^T += V^T P^T complete
        B_QFULL = B_ODONE + 2,           // q' of the piece staged
        B_OFREE = B_QFULL + 1,           // O^T of the previous piece read out
        B_WG = B_OFREE + 1,              // [4] the four warps of a softmax group
        B_MDONE = B_WG + 4,
        NBARS = B_MDONE + 1
    };
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;     // [0] tmem, [1] abort, [4] errors
    static constexpr int SMEM = MISC_OFF + 64 + 1024;        // + alignment of the base
    static_assert(SMEM <= 227 * 1024, "e4m3 tensor-core kernel exceeds the shared memory of one CTA");
    static_assert(K_OFF % 1024 == 0 && P_OFF % 1024 == 0 && V_OFF % 1024 == 0,
                  "operand tiles must stay 1 KB aligned");
};

// two fp32 -> two E4M3 codes (RNE, saturating), lo in the low byte
__device__ __forceinline__ uint32_t f32x2_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float2 e4m3x2_f32x2(uint32_t two) {
    const uint32_t h = e4m3x2_f16x2(two);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Splits x >= 0 into a + r with a = x truncated to 4 significant bits (sign,
// exponent and the top 3 stored mantissa bits kept) and r = x - a, exact in
// fp32 (x and a share their exponent)
__device__ __forceinline__ float split4(float x, float &r) {
    const float a = __uint_as_float(__float_as_uint(x) & 0xFFF00000u);
    r = __fsub_rn(x, a);
    return a;
}

// two consecutive q values of a packed word (low half first)
__device__ __forceinline__ float2 q_pair2(uint32_t u, int q_dtype) {
    if (q_dtype == PA_BF16) return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
    return make_float2(__half2float(__ushort_as_half((uint16_t)(u & 0xFFFFu))),
                       __half2float(__ushort_as_half((uint16_t)(u >> 16))));
}

// byte offset of 16-byte chunk c (0..15) of token row t in a [2][128][128 B] SW128 tile
__device__ __forceinline__ uint32_t tile_off(int t, int c) {
    return (uint32_t)((c >> 3) * (CH * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

}  // namespace e4tc

// After a wait ran out: every piece of the CTA's share is NaN (outputs, or
// partial log-sum-exps the combine turns into NaN rows).
__device__ __noinline__ void e4tc_nan_share(const E4TcParams &P, long long x0, int npg, int ti, int nth) {
    using namespace e4tc;
    const float NaN = __int_as_float(0x7fc00000);
    const long long kw = blockIdx.x;
    auto nan_piece = [&](int b_, int u_, int p0_, int pl_) {
        const int Pb = planned_pages(P.req, b_, P.mbps);
        const bool complete = (p0_ == 0 && pl_ == Pb - 1);
        const long long slot_id = (long long)b_ * P.Hkv + u_ + kw;
        for (int r = 0; r < P.R; ++r) {
            const int jq = r / P.G, h = u_ * P.G + r % P.G;
            if (complete) {
                const size_t row = (((size_t)b_ * P.n + jq) * P.Hq + h) * D;
                for (int d = ti; d < D; d += nth) {
                    if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[row + d] = NaN;
                    else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[row + d] = __float2half_rn(NaN);
                    else reinterpret_cast<__nv_bfloat16 *>(P.out)[row + d] = __float2bfloat16_rn(NaN);
                }
                if (ti == 0 && P.lse != nullptr) P.lse[((size_t)b_ * P.n + jq) * P.Hq + h] = NaN;
            } else if (ti == 0) {
                P.part_lse[(size_t)slot_id * P.R + r] = NaN;
            }
        }
    };
    Cursor cw = cursor_at(x0, P.req, P.B, P.Hkv, P.mbps);
    int wb = -1, wq = -1, wp0 = 0, wl = 0;
    for (int j = 0; j < npg && cw.b < P.B; ++j) {
        if (cw.b != wb || cw.q != wq) {
            if (wb >= 0) nan_piece(wb, wq, wp0, wl);
            wb = cw.b;
            wq = cw.q;
            wp0 = cw.p;
        }
        wl = cw.p;
        cursor_next(cw, P.req, P.B, P.Hkv, P.mbps);
    }
    if (wb >= 0) nan_piece(wb, wq, wp0, wl);
}

template <int N>
__global__ void __launch_bounds__(e4tc::Lay<N>::THREADS, 1)
    pa_e4m3_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, E4TcParams P) {
    using namespace e4tc;
    using Y = Lay<N>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Y::BAR_OFF);
    int *misc = reinterpret_cast<int *>(smem + Y::MISC_OFF);
    volatile int *abort = misc + 1;
    volatile int *vbad = reinterpret_cast<volatile int *>(smem + Y::VBAD_OFF);
    float *m_s = reinterpret_cast<float *>(smem + Y::M_OFF);
    float *rs_s = reinterpret_cast<float *>(smem + Y::RS_OFF);
    int *vis_s = reinterpret_cast<int *>(smem + Y::VIS_OFF);
    float *red = reinterpret_cast<float *>(smem + Y::RED_OFF);
    volatile int *need = reinterpret_cast<volatile int *>(smem + Y::NEED_OFF);
    float *alpha_s = reinterpret_cast<float *>(smem + Y::ALPHA_OFF);
    constexpr int NK = Y::NK, NV = Y::NV, SB = Y::SB, NR = Y::NR;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float NaN = __int_as_float(0x7fc00000);
    const int U = P.Hkv;  // segments (kv heads) per request

    grid_dependency_wait();
    const long long total = P.hdr[HDR_TOTAL_PAGES];
    if (total > (long long)P.B * P.mbps) {
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    const long long Ntot = total * U;
    const long long x0 = blockIdx.x * Ntot / gridDim.x, x1 = (blockIdx.x + 1) * Ntot / gridDim.x;
    if (x0 >= x1) return;
    const int npg = (int)(x1 - x0);
    const Cursor c0 = cursor_at(x0, P.req, P.B, U, P.mbps);
    if (c0.b >= P.B) {
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    const long long kw = blockIdx.x;

    if (tid == 0) {
        for (int i = 0; i < Y::NBARS; ++i) {
            uint32_t c = 1;
            if ((i >= Y::B_SFREE && i < Y::B_SFREE + 2) || (i >= Y::B_PFULL && i < Y::B_PFULL + 2) ||
                i == Y::B_QFULL || i == Y::B_OFREE)
                c = 4 * Y::NWG;  // every softmax warp
            if (i >= Y::B_WG && i < Y::B_WG + 4) c = 4;
            mbar_init(&bars[i], c);
        }
        misc[1] = 0;
        misc[4] = 0;
        mbar_fence_init();
    }
    if (warp == W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sb + Y::MISC_OFF),
                     "r"(Y::TM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)misc[0];
    constexpr uint32_t TM_S = 0, TM_O = Y::TM_O;
    uint32_t err = 0;

    constexpr int W_VPROD = Y::W_VPROD, NWG = Y::NWG;
    if (warp == W_KPROD || warp == W_VPROD) {
        // ================================================== producers: K (warp 0) and V (warp 6)
        // of each chunk, one tensor copy per block and 128-channel half (the
        // 128-byte-swizzled operand layout); blocks past the request's length
        // and blocks with an invalid id are not copied
        const bool isv = warp == W_VPROD;
        const CUtensorMap *tm = isv ? &tv : &tk;
        uint64_t *full = &bars[isv ? Y::B_VFULL : Y::B_KFULL];
        uint64_t *freeb = &bars[isv ? Y::B_VFREE : Y::B_KFREE];
        const int NS = isv ? NV : NK;
        uint8_t *ring = smem + (isv ? Y::V_OFF : Y::K_OFF);
        const int mpb = CH / P.bs;  // blocks per chunk (at most 8)
        const uint64_t pol = l2_evict_first_policy();
        Cursor ci = c0;
        int issued = 0;
#ifdef PA_FAULT_INJECT
        const unsigned fi_withhold = P.hdr[HDR_WITHHOLD];
#endif
        for (int j = 0; j < npg; ++j) {
            const int slot = j % NS;
            if (j >= NS && !warp_wait_u(&freeb[slot], ((j / NS) - 1) & 1, abort, err)) break;
            if (ci.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; break; }
#ifdef PA_FAULT_INJECT
            if (fi_withhold != 0 && x0 + j + 1 == (long long)fi_withhold) {
                ++issued;
                cursor_next<true>(ci, P.req, P.B, U, P.mbps);
                continue;  // no copies and no arrives: the waits on this stage run out
            }
#endif
            const int nblk = min((ci.L + P.bs - 1) / P.bs, P.tbl);
            const int fb = ci.p * mpb;
            const bool live = lane < mpb && fb + lane < nblk;
            const int blk = live ? P.block_table[(size_t)ci.b * P.tbl + fb + lane] : 0;
            const bool ok = live && blk >= 1 && blk < P.num_blocks;
            const unsigned okm = __ballot_sync(0xffffffffu, ok);
            const bool anybad = __any_sync(0xffffffffu, live && !ok);
            if (lane == 0) {
                if (isv) vbad[slot] = anybad ? 1 : 0;  // published by the arrive
                mbar_arrive_expect_tx(&full[slot], (uint32_t)__popc(okm) * 2u * (uint32_t)P.bs * 128u);
            }
            __syncwarp();
            if (ok) {
                uint8_t *dst = ring + slot * TILE + lane * P.bs * 128;
                tma_load_4d_hint(dst, tm, &full[slot], 0, 0, ci.q, blk, pol);
                tma_load_4d_hint(dst + CH * 128, tm, &full[slot], 128, 0, ci.q, blk, pol);
            }
            ++issued;
            cursor_next<true>(ci, P.req, P.B, U, P.mbps);
        }
        if (*abort && lane == 0) {
            // let every copy still in flight land before the CTA exits
            for (int i = max(0, issued - NS); i < issued; ++i)
                (void)mbar_wait_bounded(&full[i % NS], (i / NS) & 1, nullptr);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ================================================== MMA issue
        // S^T = K [q'_hi | q'_lo]^T (N' = 2N), O^T += V^T [P_0 | P_1 | P_2]^T (N' = 3N)
        constexpr uint32_t ID_S = idesc(128, 2 * N, 0);
        // O^T: A = V^T read MN-major; B = P^T K-major, or MN-major (bit 16) at 64 rows
        constexpr uint32_t ID_O = idesc(128, 3 * N, 1) | (Y::PMN ? (1u << 16) : 0u);
        Cursor cq = c0, cp = c0;
        int q_piece = -1, q_pb = -1, q_pq = -1;
        int p_piece = -1, p_pb = -1, p_pq = -1;
        auto issue_s = [&](int j) -> bool {
            if (cq.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; return false; }
            const int kslot = j % NK, sbuf = j % SB;
            if (cq.b != q_pb || cq.q != q_pq) {
                ++q_piece;
                q_pb = cq.b;
                q_pq = cq.q;
                if (!lane_wait(&bars[Y::B_QFULL], q_piece & 1, abort, err)) return false;
            }
            if (!lane_wait(&bars[Y::B_KFULL + kslot], (j / NK) & 1, abort, err)) return false;
            if (j >= SB && !lane_wait(&bars[Y::B_SFREE + sbuf], ((j / SB) - 1) & 1, abort, err)) return false;
            tc_fence_after();
            {
                const uint32_t kst = sb + Y::K_OFF + kslot * TILE;
                const uint32_t dS = tmem + TM_S + (uint32_t)(2 * N * sbuf);
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // 32 channels per step
                    const uint64_t ad = sdesc(kst + (uint32_t)((k >> 2) * (CH * 128) + 32 * (k & 3)), 16, 1024, 2);
                    const uint64_t bd =
                        sdesc(sb + Y::Q_OFF + (uint32_t)((k >> 2) * (2 * N * 128) + 32 * (k & 3)), 16, 1024, 2);
                    mma_f8(dS, ad, bd, ID_S, k > 0 ? 1u : 0u);
                }
                mma_commit(&bars[Y::B_SFULL + sbuf]);
                mma_commit(&bars[Y::B_KFREE + kslot]);
            }
            cursor_next(cq, P.req, P.B, U, P.mbps);
            return true;
        };
        auto issue_o = [&](int j) -> bool {
            const int vslot = j % NV, pbuf = j & 1;
            bool first = false;
            if (cp.b != p_pb || cp.q != p_pq) {
                ++p_piece;
                p_pb = cp.b;
                p_pq = cp.q;
                first = true;
                if (p_piece > 0 && !lane_wait(&bars[Y::B_OFREE], (p_piece - 1) & 1, abort, err)) return false;
            }
            if (!lane_wait(&bars[Y::B_PFULL + pbuf], (j >> 1) & 1, abort, err)) return false;
            if (!lane_wait(&bars[Y::B_VFULL + vslot], (j / NV) & 1, abort, err)) return false;
            tc_fence_after();
            {
                const uint32_t vst = sb + Y::V_OFF + vslot * TILE;
                const uint32_t pst = sb + Y::P_OFF + pbuf * Y::P_BUF;
#pragma unroll
                for (int i = 0; i < 2; ++i) {  // channel tiles 0..127, 128..255
                    const uint32_t dO = tmem + TM_O + (uint32_t)(3 * N * i);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {  // 32 tokens per step
                        const uint64_t ad = sdesc(vst + (uint32_t)(i * (CH * 128) + k * 32 * 128), 16, 1024, 2);
                        // MN-major: 32 tokens x N bytes per step, terms CH * N bytes apart,
                        // 8-token groups 8 N bytes apart
                        const uint64_t bd = Y::PMN ? sdesc(pst + 32 * N * k, CH * N, 8 * N, Y::PMN_SWZ)
                                                   : sdesc(pst + 32 * k, 16, 1024, 2);
                        mma_f8(dO, ad, bd, ID_O, (first && k == 0) ? 0u : 1u);
                    }
                }
                mma_commit(&bars[Y::B_ODONE + pbuf]);
                mma_commit(&bars[Y::B_VFREE + vslot]);
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
            mma_commit(&bars[Y::B_MDONE]);
            (void)mbar_wait_bounded(&bars[Y::B_MDONE], 0, nullptr);
        }
        __syncwarp();
    } else {
        // ================================================== softmax, q' staging, epilogue
        // NWG warpgroups, each owning NR = N / NWG rows (S^T and O^T columns):
        // rows are independent in the softmax, so each group votes, rescales
        // and writes P^T for its own rows; one token per thread
        const int wg = (warp - W_SM0) >> 2;
        const int rb = wg * NR;                  // the group's first row
        const int qd = warp & 3;                 // tensor-memory lane quarter
        const int t = 32 * qd + lane;            // token of the chunk (S^T) / channel of a tile (O^T)
        const int ti = t;                        // 0..127 within the group
        const uint32_t tl = tmem + ((uint32_t)(32 * qd) << 16);
        uint64_t *bwg = &bars[Y::B_WG + wg];
        volatile int *needw = need + 8 * wg;
        const float ksc = (P.k_mode == PA_SCALE_TENSOR) ? P.k_scale[0] : 1.0f;
        const float vsc = (P.v_mode == PA_SCALE_TENSOR) ? P.v_scale[0] : 1.0f;
        Cursor cs = c0;
        int piece = -1, pb = -1, pq = -1, p0 = 0, last_p = 0, L = 0, vmin = 0, wg_phase = 0, pPb = 0;
        // the next segment's length and plan record, loaded one piece ahead
        int nx_b = c0.b, nx_L = P.context_lens[c0.b];
        int4 nx_R = P.req[c0.b];
        int pp = 0, mb = 0;  // buffer of the piece's row constants, running-maximum buffer
        bool pbad = false;
        float lsum[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) lsum[r] = 0.f;
        auto mrow = [&](int ppb, int mbb) -> float * { return m_s + (ppb * 2 + mbb) * 64; };
        auto wg_sync = [&]() -> bool {  // the group's four warps (bounded)
            __syncwarp();
            if (lane == 0) mbar_arrive(bwg);
            const bool ok = warp_wait_u(bwg, wg_phase & 1, abort, err);
            ++wg_phase;
            return ok;
        };

        // q' of the segment (b, kv head u) for the group's rows: TPR threads
        // per row load it together (one round trip), agree on its largest
        // magnitude, and write two exact E4M3 terms of q * 2^s_r (largest
        // magnitude in [128, 256)); the row's score scale and visible length
        // go to the buffers of parity ppb
        constexpr int TPR = (NR <= 8) ? 16 : (NR <= 16) ? 8 : 4;  // threads per q row
        constexpr int QW = 32 / TPR;                              // 16-byte words of the row per thread
        static_assert(NR * TPR <= 128, "one round of q rows");
        auto stage_q = [&](int b, int u, int Lb, int ppb) {
            const int r = rb + ti / TPR, part = ti % TPR;
            const bool rok = ti / TPR < NR && r < P.R;
            const int jq = rok ? r / P.G : 0, h = u * P.G + (rok ? r % P.G : 0);
            const uint4 *qrow =
                reinterpret_cast<const uint4 *>(P.q + 2 * ((((size_t)b * P.n + jq) * P.Hq + h) * D)) + part * QW;
            uint4 v[QW];
#pragma unroll
            for (int i = 0; i < QW; ++i) v[i] = rok ? qrow[i] : make_uint4(0u, 0u, 0u, 0u);
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < QW; ++i) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = q_pair2(w[e], P.q_dtype);
                    mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
            }
#pragma unroll
            for (int o = TPR / 2; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            int ex = 0;
            const bool fin = mx > 0.f && mx < 3.0e38f;
            if (fin) frexpf(mx, &ex);
            const int sh = fin ? 8 - ex : 0;
            const float up = pow2f(sh);
            if (rok) {
#pragma unroll
                for (int cc = 0; cc < QW / 2; ++cc) {  // 16 channels = 16 bytes of each term
                    const int c = part * (QW / 2) + cc;
                    const uint32_t w[8] = {v[2 * cc].x,     v[2 * cc].y,     v[2 * cc].z,     v[2 * cc].w,
                                           v[2 * cc + 1].x, v[2 * cc + 1].y, v[2 * cc + 1].z, v[2 * cc + 1].w};
                    uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 f = q_pair2(w[e], P.q_dtype);
                        const float a = f.x * up, bb = f.y * up;
                        const uint32_t h2 = f32x2_e4m3x2(a, bb);
                        const float2 hf = e4m3x2_f32x2(h2);
                        const uint32_t l2 = f32x2_e4m3x2(a - hf.x, bb - hf.y);
                        hw[e >> 1] |= h2 << (16 * (e & 1));
                        lw[e >> 1] |= l2 << (16 * (e & 1));
                    }
                    // hi in row r, lo in row N + r of the half's [2N][128 B] tile
                    const uint32_t off = (uint32_t)((c >> 3) * (2 * N * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
                    *reinterpret_cast<uint4 *>(smem + Y::Q_OFF + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(smem + Y::Q_OFF + N * 128 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            if (ti / TPR < NR && part == 0) {
                rs_s[ppb * 64 + r] = rok ? P.softmax_scale * ksc * LOG2E * pow2f(-sh) : 0.f;
                vis_s[ppb * 64 + r] = rok ? (P.causal ? Lb - (P.n - 1 - jq) : Lb) : 0;
                mrow(ppb, 0)[r] = -INFINITY;
                mrow(ppb, 1)[r] = -INFINITY;
            }
        };

        // the finished segment's output (or partial) for the group's rows from
        // the three O^T partial sums and the row sums; its row constants are in
        // the buffers of parity ppb, maxima in mbb
        auto epilogue = [&](int jl, int ppb, int mbb) -> bool {
#pragma unroll
            for (int k = 0; k < NR; ++k) {  // row sums over the 128 tokens
                float v = lsum[k];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) red[qd * 64 + rb + k] = v;
            }
            if (!wg_sync()) return false;
            if (!warp_wait_u(&bars[Y::B_ODONE + (jl & 1)], (jl >> 1) & 1, abort, err)) return false;
            tc_fence_after();
            const bool complete = (p0 == 0 && last_p == pPb - 1);
            const long long slot_id = (long long)pb * U + pq + kw;
            auto row_l = [&](int r) -> float { return (red[r] + red[64 + r]) + (red[128 + r] + red[192 + r]); };
            if (ti < NR && rb + ti < P.R) {
                const int r = rb + ti;
                const float l = row_l(r);
                float lse_v = l > 0.f ? (mrow(ppb, mbb)[r] + lg2(l) - PSHIFT) * LN2 : -INFINITY;
                if (pbad) lse_v = NaN;
                const int jq = r / P.G, h = pq * P.G + r % P.G;
                if (complete) {
                    if (P.lse != nullptr) P.lse[((size_t)pb * P.n + jq) * P.Hq + h] = lse_v;
                } else {
                    P.part_lse[(size_t)slot_id * P.R + r] = lse_v;
                }
            }
            // this path runs once per piece: kept as loops, not unrolled
#pragma unroll 1
            for (int i = 0; i < 2; ++i) {
                const int d = 128 * i + t;
#pragma unroll 1
                for (int g = 0; g < NR; g += 8) {
                    uint32_t a[8], b2[8], c2[8];
                    const uint32_t ta = tl + TM_O + (uint32_t)(3 * N * i + rb + g);
                    tmem_ld8_nowait(ta, a);
                    tmem_ld8_nowait(ta + N, b2);
                    tmem_ld8_nowait(ta + 2 * N, c2);
                    tmem_ld_wait();
                    // row r = rb + g + k is query row jq, head pq G + hg: advanced one
                    // row at a time instead of a division per element
                    int jq = (rb + g) / P.G, hg = (rb + g) % P.G;
#pragma unroll
                    for (int k = 0; k < 8; ++k, ++hg) {
                        if (hg == P.G) { hg = 0; ++jq; }
                        const int r = rb + g + k;
                        if (r >= P.R) break;
                        const float l = row_l(r);
                        const float o = (__uint_as_float(a[k]) + __uint_as_float(b2[k])) + __uint_as_float(c2[k]);
                        float y = o * (l > 0.f ? 1.0f / l : 0.f);
                        if (pbad) y = NaN;
                        if (complete) {
                            const int h = pq * P.G + hg;
                            const size_t oi = (((size_t)pb * P.n + jq) * P.Hq + h) * D + d;
                            const float z = y * vsc;
                            if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = z;
                            else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(z);
                            else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(z);
                        } else {
                            P.part_o[((size_t)slot_id * P.R + r) * D + d] = y;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[Y::B_OFREE]);
            return true;
        };

        bool alive = true;
        int j = 0;
        for (; j < npg; ++j) {
            if (cs.b >= P.B) { err |= PA_DEV_ERR_STALE_PLAN; alive = false; break; }
            const int vslot = j % NV, sbuf = j % SB, pbuf = j & 1;
            const bool first = (cs.b != pb || cs.q != pq);
            if (first) {
                // the previous piece's S MMAs are complete (its last S^T was read):
                // stage q' of the new piece first (its S MMAs wait for it), then
                // finish the previous piece (its last O MMAs are already queued)
                const int ppn = piece >= 0 ? (pp ^ 1) : 0;
                const bool hit = nx_b == cs.b;
                const int Ln = hit ? nx_L : P.context_lens[cs.b];
                const int4 Rq = hit ? nx_R : P.req[cs.b];
                stage_q(cs.b, cs.q, Ln, ppn);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[Y::B_QFULL]);
                if (piece >= 0 && !epilogue(j - 1, pp, mb)) { alive = false; break; }
                ++piece;
                pp = ppn;
                mb = 0;
                pb = cs.b;
                pq = cs.q;
                p0 = cs.p;
                pPb = cs.Pb;
                L = Ln;
                vmin = P.causal ? L - (P.n - 1) : L;
                pbad = false;
                if (Rq.w != 0) { pbad = true; err |= PA_DEV_ERR_CONTEXT_LEN; }
                if (L != Rq.x) { pbad = true; err |= PA_DEV_ERR_STALE_PLAN; }
#pragma unroll
                for (int k = 0; k < NR; ++k) lsum[k] = 0.f;
                {
                    // the segment after this one: its record now, its q rows into L2
                    const int nb = pq + 1 < U ? pb : pb + 1, nq = pq + 1 < U ? pq + 1 : 0;
                    if (nb < P.B) {
                        if (nb != nx_b) {
                            nx_b = nb;
                            nx_L = P.context_lens[nb];
                            nx_R = P.req[nb];
                        }
                        for (int i = ti; i < 4 * NR; i += 128) {
                            const int rr = rb + (i >> 2);
                            if (rr < P.R) {
                                const int jq = rr / P.G, h = nq * P.G + rr % P.G;
                                const uint8_t *qa = P.q + 2 * ((((size_t)nb * P.n + jq) * P.Hq + h) * D) + 128 * (i & 3);
                                asm volatile("prefetch.global.L2 [%0];" ::"l"(qa));
                            }
                        }
                    }
                }
                if (!wg_sync()) { alive = false; break; }  // the new row constants are visible
            }
            if (!warp_wait_u(&bars[Y::B_SFULL + sbuf], (j / SB) & 1, abort, err)) { alive = false; break; }
            tc_fence_after();
            float x[NR];
            {
                uint32_t hi[NR], lo[NR];
#pragma unroll
                for (int g = 0; g < NR; g += 8) {
                    const uint32_t ta = tl + TM_S + (uint32_t)(2 * N * sbuf + rb + g);
                    tmem_ld8_nowait(ta, hi + g);
                    tmem_ld8_nowait(ta + N, lo + g);
                }
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < NR; ++k) x[k] = __uint_as_float(hi[k]) + __uint_as_float(lo[k]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[Y::B_SFREE + sbuf]);
            const int tok = cs.p * CH + t;
            const float *mc = mrow(pp, mb) + rb;
            const float *rsp = rs_s + pp * 64 + rb;
            bool exceed = false;
            if (cs.p * CH + CH <= vmin) {  // every row sees every token of the chunk
#pragma unroll
                for (int k = 0; k < NR; ++k) {
                    x[k] *= rsp[k];
                    exceed |= x[k] > mc[k] + SLACK;  // also true for a finite score and m = -inf
                }
            } else {
                const int *vp = vis_s + pp * 64 + rb;
#pragma unroll
                for (int k = 0; k < NR; ++k) {
                    x[k] = (tok < vp[k]) ? x[k] * rsp[k] : -INFINITY;
                    exceed |= x[k] > mc[k] + SLACK;
                }
            }
            const int vote = __any_sync(0xffffffffu, exceed) ? 1 : 0;
            if (lane == 0) needw[pbuf * 4 + qd] = vote;
            if (!wg_sync()) { alive = false; break; }
            const bool resc = (needw[pbuf * 4] | needw[pbuf * 4 + 1] | needw[pbuf * 4 + 2] | needw[pbuf * 4 + 3]) != 0;
            if (resc) {
                // new row maxima over the chunk's 128 tokens, into the other buffer
#pragma unroll
                for (int k = 0; k < NR; ++k) {
                    float v = x[k];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    if (lane == 0) red[qd * 64 + rb + k] = v;
                }
                if (!wg_sync()) { alive = false; break; }
                float *mn_s = mrow(pp, mb ^ 1) + rb;
                float *al = alpha_s + rb;  // the factor of each row, exp2(m_old - m_new)
                if (ti < NR) {
                    const int r = rb + ti;
                    const float mo = mc[ti];
                    const float cm = fmaxf(fmaxf(red[r], red[64 + r]), fmaxf(red[128 + r], red[192 + r]));
                    const float mn = (mo == -INFINITY || cm > mo + SLACK) ? fmaxf(cm + HEAD, mo) : mo;
                    mn_s[ti] = mn;
                    al[ti] = (mn == mo) ? 1.f : ex2(mo - mn);
                }
                if (!wg_sync()) { alive = false; break; }
#pragma unroll
                for (int k = 0; k < NR; ++k) lsum[k] *= al[k];
                // O^T (channels on lanes, rows on columns, three partial sums per
                // tile) takes the same factors once the previous chunk's O MMAs
                // are in; the first chunk of a piece overwrites O^T
                if (!first) {
                    if (!warp_wait_u(&bars[Y::B_ODONE + (pbuf ^ 1)], ((j - 1) >> 1) & 1, abort, err)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int i = 0; i < 6; ++i) {  // (tile, term): the group's NR columns in one round trip
                        uint32_t w[NR];
                        const uint32_t ta = tl + TM_O + (uint32_t)(N * i + rb);
#pragma unroll
                        for (int g = 0; g < NR; g += 8) tmem_ld8_nowait(ta + g, w + g);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < NR; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * al[k]);
#pragma unroll
                        for (int g = 0; g < NR; g += 8) tmem_st8_u(ta + g, w + g);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                }
                mb ^= 1;  // every thread switches to the new maxima
            }
            // this chunk's P^T buffer is free once chunk j-2's O MMAs are done
            if (j >= 2 && !warp_wait_u(&bars[Y::B_ODONE + pbuf], ((j >> 1) - 1) & 1, abort, err)) {
                alive = false;
                break;
            }
            // V of the chunk has landed: flag invalid block ids, and zero the V
            // rows past the request's length (uncopied, or slots of the last
            // block that may hold NaN codes), so that 0 * NaN cannot reach O^T;
            // each group zeroes one 128-channel half of the row
            if (!warp_wait_u(&bars[Y::B_VFULL + vslot], (j / NV) & 1, abort, err)) { alive = false; break; }
            if (vbad[vslot]) { pbad = true; err |= PA_DEV_ERR_BLOCK_ID; }
            if (tok >= L) {
                uint8_t *vrow = smem + Y::V_OFF + vslot * TILE;
#pragma unroll
                for (int c = (16 / NWG) * wg; c < (16 / NWG) * (wg + 1); ++c)
                    *reinterpret_cast<uint4 *>(vrow + tile_off(t, c)) = make_uint4(0u, 0u, 0u, 0u);
            }
            // P^T = 2^(x - m + 8) as three E4M3 terms of 4 significant bits each
            // (rows in pairs, one conversion per pair and term); the row sums add
            // the same values
            uint8_t *pt = smem + Y::P_OFF + pbuf * Y::P_BUF;
            const float *mcur = mrow(pp, mb) + rb;
            uint32_t pw[3][NR / 4];  // MN-major: the group's bytes of each term, 4 rows per word
#pragma unroll
            for (int k = 0; k < NR; k += 2) {
                const int r = rb + k;
                const float ma = mcur[k], mb2 = mcur[k + 1];
                const float pa0 = ex2(x[k] - ((ma == -INFINITY) ? 0.f : ma - PSHIFT));
                const float pb0 = ex2(x[k + 1] - ((mb2 == -INFINITY) ? 0.f : mb2 - PSHIFT));
                lsum[k] += pa0;
                lsum[k + 1] += pb0;
                float ra, rb2, sa, sb2;
                const float ha = split4(pa0, ra), hb = split4(pb0, rb2);
                const float ma1 = split4(ra, sa), mb1 = split4(rb2, sb2);
                const uint32_t ch = f32x2_e4m3x2(ha, hb), cm = f32x2_e4m3x2(ma1, mb1), cl = f32x2_e4m3x2(sa, sb2);
                if constexpr (Y::PMN) {
                    const int wi = k >> 2, sh = 8 * (k & 3);  // rows k, k + 1 go to bytes k % 4 .. of word k / 4
                    if ((k & 3) == 0) { pw[0][wi] = 0u; pw[1][wi] = 0u; pw[2][wi] = 0u; }
                    pw[0][wi] |= ch << sh;
                    pw[1][wi] |= cm << sh;
                    pw[2][wi] |= cl << sh;
                } else {
                    // K-major, 128-byte swizzle: row r of 128 tokens, 16-byte chunk
                    // t / 16 lands at (t / 16) ^ (r & 7)
                    const uint32_t oa = (uint32_t)r * 128 + ((((t >> 4) ^ (r & 7)) << 4) | (t & 15));
                    const uint32_t ob = (uint32_t)(r + 1) * 128 + ((((t >> 4) ^ ((r + 1) & 7)) << 4) | (t & 15));
                    pt[oa] = (uint8_t)(ch & 0xFF);
                    pt[ob] = (uint8_t)(ch >> 8);
                    pt[Y::P_TERM + oa] = (uint8_t)(cm & 0xFF);
                    pt[Y::P_TERM + ob] = (uint8_t)(cm >> 8);
                    pt[2 * Y::P_TERM + oa] = (uint8_t)(cl & 0xFF);
                    pt[2 * Y::P_TERM + ob] = (uint8_t)(cl >> 8);
                }
            }
            if constexpr (Y::PMN) {
                // token t's row of a term: N bytes (rows 0..N-1), 16-byte chunk wg at
                // wg ^ ((t / 2) & 3) (64-byte swizzle, N = 64) or wg ^ ((t / 4) & 1)
                // (32-byte swizzle, N = 32); one block of 128 N bytes per term
                static_assert(NR == 16, "one 16-byte chunk per group and term");
                const uint32_t sw = (N == 64) ? (uint32_t)((t >> 1) & 3) : (uint32_t)((t >> 2) & 1);
                const uint32_t off = (uint32_t)t * N + ((uint32_t)wg ^ sw) * 16u;
#pragma unroll
                for (int tm = 0; tm < 3; ++tm)
                    *reinterpret_cast<uint4 *>(pt + tm * (CH * N) + off) =
                        make_uint4(pw[tm][0], pw[tm][1], pw[tm][2], pw[tm][3]);
            }

            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[Y::B_PFULL + pbuf]);
            last_p = cs.p;
            cursor_next(cs, P.req, P.B, U, P.mbps);
        }
        if (alive && piece >= 0 && !epilogue(npg - 1, pp, mb)) alive = false;
        if (!alive) e4tc_nan_share(P, x0, npg, wg * 128 + ti, 128 * NWG);
    }

    // ---- teardown
    grid_dependents_launch();
    if (err) atomicOr(reinterpret_cast<unsigned *>(misc + 4), err);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Y::TM_COLS) : "memory");
    if (tid == 0) atomic_or_err(P.hdr, (uint32_t)misc[4]);
}

template <int N>
cudaError_t launch_e4tc_n(const CUtensorMap &tk, const CUtensorMap &tv, const E4TcParams &P, int ctas,
                          cudaStream_t s) {
    using Y = e4tc::Lay<N>;
    cudaError_t e = cudaFuncSetAttribute(pa_e4m3_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, Y::SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(pa_e4m3_tc_kernel<N>, dim3((unsigned)ctas), dim3(Y::THREADS), (size_t)Y::SMEM, s, tk, tv, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_e4m3_tc(const CUtensorMap &tk, const CUtensorMap &tv, const E4TcParams &P, int ctas,
                           cudaStream_t s) {
    switch (P.R) {
        case 16: return launch_e4tc_n<16>(tk, tv, P, ctas, s);
        case 32: return launch_e4tc_n<32>(tk, tv, P, ctas, s);
        case 48: return launch_e4tc_n<48>(tk, tv, P, ctas, s);
        case 64: return launch_e4tc_n<64>(tk, tv, P, ctas, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
