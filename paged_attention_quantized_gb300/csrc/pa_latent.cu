// Single-latent-KV MQA decode / verify attention for sm_103a.
//
// K and V live in one E4M3 plane per kv head: a token row holds 576 channels,
// V is its first 512, and every block ends with one fp32 scale per token
// (the layout of a "data region then scale region" block, FlashInfer docs,
// "flashinfer.fp4_paged_mqa_logits", Parameters).  With 128 query heads on
// one kv head and two query rows per request there are 256 query rows per
// request, so both S = q K^T (576 deep) and O = P V (512 wide) are dense
// contractions; the MMA tiles are the point of this kernel.
//
// Work split: the same global page order as the grouped kernel -- (request,
// kv head, block of 64 query rows = "segment", page), logical positions only
// (1Cat-vLLM PR #494, "Stabilize QSA page4 order under KV relocation",
// Summary) -- shared evenly over the CTAs of a persistent launch, one CTA
// per SM.  A CTA's run of pages inside one segment is a piece; a piece that
// is a whole segment writes `out`, the others write a normalised partial and
// its log-sum-exp to slot (segment + CTA index) for the combine kernel.
//
// Per page (64 tokens), the CTA's eight warps:
//  1. wait for the page's bulk tensor copies (codes as four 128-byte and one
//     64-byte swizzled column boxes, scales as a 256-byte bulk copy) and
//     dequantize the codes once into an f16 tile [token][576] in shared
//     memory (E4M3 -> f16 is exact).  Token slots past L_b become zero codes
//     and zero scales, so neither a NaN code nor a NaN scale in the padding
//     reaches P.V (1Cat-vLLM PR #647, "Stop grouped-page4 null-block padding
//     from leaking E4M3 NaN", Fix);
//  2. S = q' K^T with m16n8k16 MMAs (warp w: rows 16(w%4).., tokens
//     32(w/4)..), scores scaled in fp32 by softmax_scale, the query row's
//     power-of-two factor and the token's scale, then masked (t >= vis);
//  3. online softmax in the exp2 domain; the two warps of a row tile trade
//     their row maxima through shared memory.  P' = p * scale_t * 2^-E (E
//     the exponent of the page's largest token scale, so P' fits f16 with
//     full precision) is stored as f16; the row sum keeps p alone;
//  4. O += P' V with m16n8k16 MMAs (warp w: rows 32(w%2).., channels
//     128(w/2)..); the factor exp2(m_old - m_new) * 2^(E_old - E) rescales O
//     first, so O always carries the current page's 2^-E.
// The query rows of a segment are staged once per piece as f16, each row
// scaled by a power of two into [-1, 1) (exact), the factor joining the score
// scale.
#include "pa_attn.cuh"

namespace pa {
namespace lat {

constexpr int DK = 576, DV = 512, BS = 64, LROWS = 64, THREADS = 256, NSLOT = 2;
constexpr int KB = DK / 64;                          // column blocks of 64 channels (128 B of f16)
constexpr int BLK = LROWS * 128;                      // bytes of one column block (64 rows)
constexpr int QS_OFF = 0;                            // q' [KB][64 rows][128 B], swizzled
constexpr int KS_OFF = QS_OFF + KB * BLK;            // f16 page [KB][64 tokens][128 B], swizzled
constexpr int RING_OFF = KS_OFF + KB * BLK;          // E4M3 pages as copied
constexpr int SLOT_BYTES = 4 * BS * 128 + BS * 64;   // four 128-B column boxes + one 64-B box
constexpr int PS_OFF = RING_OFF + NSLOT * SLOT_BYTES;  // P' [64 rows][64 tokens] f16, swizzled
constexpr int TSRAW_OFF = PS_OFF + LROWS * 128;       // [NSLOT][64] token scales as copied
constexpr int TSN_OFF = TSRAW_OFF + NSLOT * BS * 4;  // [64] scale_t * 2^-E (0 past L_b)
constexpr int RMAX_OFF = TSN_OFF + BS * 4;           // [2][64] row maxima of the two token halves
constexpr int LPART_OFF = RMAX_OFF;                  //   (at the end of a piece: row sums)
constexpr int ALPHA_OFF = RMAX_OFF + 2 * LROWS * 4;   // [64] O rescale factors
constexpr int MROW_OFF = ALPHA_OFF;                  //   (at the end of a piece: row maxima)
constexpr int ROWSC_OFF = ALPHA_OFF + LROWS * 4;      // [64] score factor of each query row
constexpr int BAR_OFF = ROWSC_OFF + LROWS * 4;        // [NSLOT] mbarriers
constexpr int FLAG_OFF = BAR_OFF + NSLOT * 8;        // [0] wait ok, [1] E of the page, [2 + s] slot s bad, [4] errors
constexpr int SMEM_USED = FLAG_OFF + 32;
constexpr int SMEM_BYTES = SMEM_USED + 1024;         // + alignment of the base to 1 KB
constexpr uint32_t PAGE_TX = SLOT_BYTES + BS * 4;    // bytes one page's copies deliver
static_assert(SMEM_BYTES <= 227 * 1024, "latent kernel exceeds the shared memory of one CTA");

// byte offset of the 16-byte chunk holding channels 8c..8c+7 (c < 72) of row
// r in a [KB][64][128 B] tile: chunk index XOR (r mod 8) inside each 128 B
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return (uint32_t)((c >> 3) * BLK + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ float load_qv(const LatentParams &P, size_t idx) {
    const uint16_t bits = reinterpret_cast<const uint16_t *>(P.q)[idx];
    if (P.q_dtype == PA_BF16) return __uint_as_float((uint32_t)bits << 16);
    return __half2float(__ushort_as_half(bits));
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((min(max(e, -126), 127) + 127) << 23); }

}  // namespace lat

__global__ void __launch_bounds__(lat::THREADS, 1)
    pa_latent_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                     LatentParams P) {
    using namespace lat;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t qs = sbase + QS_OFF, ks = sbase + KS_OFF, ps = sbase + PS_OFF;
    float *tsraw = reinterpret_cast<float *>(smem + TSRAW_OFF);
    float *tsn = reinterpret_cast<float *>(smem + TSN_OFF);
    float *rmax = reinterpret_cast<float *>(smem + RMAX_OFF);
    float *lpart = reinterpret_cast<float *>(smem + LPART_OFF);
    float *alpha = reinterpret_cast<float *>(smem + ALPHA_OFF);
    float *mrow = reinterpret_cast<float *>(smem + MROW_OFF);
    float *rowsc = reinterpret_cast<float *>(smem + ROWSC_OFF);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    int *flags = reinterpret_cast<int *>(smem + FLAG_OFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, c = lane & 3;
    const int X = P.Hkv * P.RBLK;

    grid_dependency_wait();
    const long long total = P.hdr[HDR_TOTAL_PAGES];
    if (total > (long long)P.B * P.mbps) {
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    const long long Ntot = total * X;
    const long long NW = gridDim.x;
    const long long kw = blockIdx.x;
    const long long x0 = kw * Ntot / NW, x1 = (kw + 1) * Ntot / NW;
    if (x0 >= x1) return;
    const int npg = (int)(x1 - x0);

    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
        tma_prefetch_desc(&tma);
        tma_prefetch_desc(&tmb);
    }
    __syncthreads();

    Cursor cc = cursor_at(x0, P.req, P.B, X, P.mbps);
    if (cc.b >= P.B) {  // uniform: every thread computed the same cursor
        if (tid == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    // ---- producer state (warp 0): issue cursor and a cache of 32 block ids
    Cursor ci = cc;
    int idc_b = -1, idc_w0 = 0, idc = 0;
    auto issue = [&](int j) {  // warp 0 only
        const int slot = j % NSLOT;
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
            flags[2 + slot] = ok ? 0 : 1;
            if (ok) {
                const int kvh = ci.q / P.RBLK;
                uint8_t *dst = smem + RING_OFF + slot * SLOT_BYTES;
                mbar_arrive_expect_tx(&full[slot], PAGE_TX);
#pragma unroll
                for (int sg = 0; sg < 4; ++sg) tma_load_4d(dst + sg * BS * 128, &tma, &full[slot], sg * 128, 0, kvh, blk);
                tma_load_4d(dst + 4 * BS * 128, &tmb, &full[slot], 512, 0, kvh, blk);
                const uint8_t *src = P.k_pool + (size_t)blk * P.block_stride + P.codes_bytes + (size_t)kvh * BS * 4;
                bulk_load(smem + TSRAW_OFF + slot * BS * 4, src, BS * 4, &full[slot]);
            } else {
                mbar_arrive(&full[slot]);  // no copy: the piece is NaN-filled
            }
        }
        if (ci.b < P.B) cursor_next(ci, P.req, P.B, X, P.mbps);
    };
    if (warp == 0) {
        for (int j = 0; j < min(NSLOT, npg); ++j) issue(j);
    }

    // ---- roles: QK warp (rows 16*mt.., tokens 32*th..), PV warp (rows 32*mr.., channels 128*dq..)
    const int mt = warp & 3, th = warp >> 2;
    const int mr = warp & 1, dq = warp >> 1;
    const int ra = 16 * mt + g, rb = ra + 8;  // the thread's two score rows within the segment

    float o[2][16][4];       // O rows 32mr + 16i + g (+8), channels 128dq + 8t + 2c (+1)
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    int vis_a = 0, vis_b = 0, L = 0, kvh = 0, rblk = 0;
    int piece_b = -1, piece_q = -1, piece_p0 = 0, last_p = 0;
    int E_run = 0;
    bool pbad = false;
    uint32_t err = 0;

    auto start_piece = [&]() {
        piece_b = cc.b;
        piece_q = cc.q;
        piece_p0 = cc.p;
        kvh = cc.q / P.RBLK;
        rblk = cc.q % P.RBLK;
        const int4 Rq = P.req[cc.b];
        L = P.context_lens[cc.b];
        pbad = false;
        if (Rq.w != 0) { pbad = true; err |= PA_DEV_ERR_CONTEXT_LEN; }
        if (L != Rq.x) { pbad = true; err |= PA_DEV_ERR_STALE_PLAN; }
        const int r0 = rblk * LROWS;
        auto vis_of = [&](int r) { return (r0 + r < P.R && P.causal) ? L - (P.n - 1 - (r0 + r) / P.G) : L; };
        vis_a = vis_of(ra);
        vis_b = vis_of(rb);
        // q rows: 4 threads per row, 18 chunks of 8 channels each
        const int qr = tid >> 2, part = tid & 3;
        const int r = r0 + qr;
        const bool rok = r < P.R;
        size_t qbase = 0;
        if (rok) {
            const int jq = r / P.G, h = kvh * P.G + r % P.G;
            qbase = (((size_t)cc.b * P.n + jq) * P.Hq + h) * DK;
        }
        float mx = 0.f;
        if (rok) {
#pragma unroll 1
            for (int k = 0; k < 18; ++k) {
                const int ch = part + 4 * k;
#pragma unroll
                for (int e = 0; e < 8; ++e) mx = fmaxf(mx, fabsf(load_qv(P, qbase + ch * 8 + e)));
            }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        float rho = 1.f;
        if (mx > 0.f && mx < 3.0e38f) {
            int e;
            frexpf(mx, &e);
            rho = ldexpf(1.0f, e);
        }
        const float inv = 1.0f / rho;
#pragma unroll 1
        for (int k = 0; k < 18; ++k) {
            const int ch = part + 4 * k;
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float u0 = 0.f, u1 = 0.f;
                if (rok) {
                    u0 = load_qv(P, qbase + ch * 8 + 2 * e) * inv;
                    u1 = load_qv(P, qbase + ch * 8 + 2 * e + 1) * inv;
                }
                w[e] = pack_f16x2(u0, u1);
            }
            *reinterpret_cast<uint4 *>(smem + QS_OFF + sw_off(qr, ch)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (part == 0) rowsc[qr] = rok ? P.softmax_scale * rho * LOG2E : 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int t = 0; t < 16; ++t) o[i][t][0] = o[i][t][1] = o[i][t][2] = o[i][t][3] = 0.f;
        m_a = m_b = -INFINITY;
        l_a = l_b = 0.f;
        E_run = 0;
    };

    auto finish_piece = [&]() {
        __syncthreads();  // every warp is past its last P.V (alpha is reused below)
        float la = l_a, lb = l_b;
        la += __shfl_xor_sync(0xffffffffu, la, 1);
        la += __shfl_xor_sync(0xffffffffu, la, 2);
        lb += __shfl_xor_sync(0xffffffffu, lb, 1);
        lb += __shfl_xor_sync(0xffffffffu, lb, 2);
        if (c == 0) {
            lpart[th * LROWS + ra] = la;
            lpart[th * LROWS + rb] = lb;
            if (th == 0) {
                mrow[ra] = m_a;
                mrow[rb] = m_b;
            }
        }
        __syncthreads();
        const int Pb = planned_pages(P.req, piece_b, P.mbps);
        const bool complete = (piece_p0 == 0 && last_p == Pb - 1);
        const long long slot_id = (long long)piece_b * X + piece_q + kw;
        const int r0 = rblk * LROWS;
        const float NaN = __int_as_float(0x7fc00000);
        const float escale = pow2f(E_run);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int row = 32 * mr + 16 * i + g + 8 * hh;
                const int r = r0 + row;
                if (r >= P.R) continue;
                const float l = lpart[row] + lpart[LROWS + row];
                const float m = mrow[row];
                const float f = l > 0.f ? escale / l : 0.f;
                const int jq = r / P.G, h = kvh * P.G + r % P.G;
                const size_t obase = (((size_t)piece_b * P.n + jq) * P.Hq + h) * DV;
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int d = 128 * dq + 8 * t + 2 * c;
                    float v0 = o[i][t][2 * hh] * f, v1 = o[i][t][2 * hh + 1] * f;
                    if (pbad) v0 = v1 = NaN;
                    if (complete) {
                        if (P.out_dtype == PA_F32) {
                            *reinterpret_cast<float2 *>(reinterpret_cast<float *>(P.out) + obase + d) = make_float2(v0, v1);
                        } else if (P.out_dtype == PA_F16) {
                            *reinterpret_cast<uint32_t *>(reinterpret_cast<__half *>(P.out) + obase + d) = pack_f16x2(v0, v1);
                        } else {
                            *reinterpret_cast<uint32_t *>(reinterpret_cast<__nv_bfloat16 *>(P.out) + obase + d) =
                                pack_bf16x2(v0, v1);
                        }
                    } else {
                        *reinterpret_cast<float2 *>(P.part_o + ((size_t)slot_id * LROWS + row) * DV + d) = make_float2(v0, v1);
                    }
                }
                if (dq == 0 && c == 0) {
                    float lse_v = l > 0.f ? (m + lg2(l)) * LN2 : -INFINITY;
                    if (pbad) lse_v = NaN;
                    if (complete) {
                        if (P.lse != nullptr) P.lse[((size_t)piece_b * P.n + jq) * P.Hq + h] = lse_v;
                    } else {
                        P.part_lse[(size_t)slot_id * LROWS + row] = lse_v;
                    }
                }
            }
        }
    };

    int j = 0;
    for (; j < npg; ++j) {
        if (cc.b >= P.B) {  // records shorter than the shares (uniform)
            err |= PA_DEV_ERR_STALE_PLAN;
            break;
        }
        if (cc.b != piece_b || cc.q != piece_q) {
            if (piece_b >= 0) finish_piece();
            start_piece();
        }
        const int slot = j % NSLOT;
        // ---- wait for the page (one thread waits; the outcome is shared)
        if (tid == 0) flags[0] = mbar_wait_bounded(&full[slot], (j / NSLOT) & 1, nullptr) ? 1 : 0;
        __syncthreads();
        if (!flags[0]) {
            err |= PA_DEV_ERR_TIMEOUT;
            pbad = true;
            break;
        }
        (void)mbar_try_wait(&full[slot], (j / NSLOT) & 1);  // acquire the copies' writes in every thread
        if (flags[2 + slot]) {
            err |= PA_DEV_ERR_BLOCK_ID;
            pbad = true;
        }
        const int nvalid = min(BS, L - cc.p * BS);  // real tokens of this page
        const uint8_t *pg8 = smem + RING_OFF + slot * SLOT_BYTES;
        // ---- token scales: zero past L_b, normalised by the page's largest power of two
        if (warp == 0) {
            const float s0 = lane < nvalid ? tsraw[slot * BS + lane] : 0.f;
            const float s1 = lane + 32 < nvalid ? tsraw[slot * BS + lane + 32] : 0.f;
            float mx = fmaxf(fabsf(s0), fabsf(s1));
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            int E = E_run;
            if (mx > 0.f && mx < 3.0e38f) {
                frexpf(mx, &E);
                E = min(max(E, -120), 120);
            }
            const float ne = pow2f(-E);
            tsn[lane] = s0 * ne;
            tsn[lane + 32] = s1 * ne;
            if (lane == 0) flags[1] = E;
        }
        // ---- dequantize the codes into the f16 tile (zero rows past L_b)
#pragma unroll 3
        for (int it = 0; it < 9; ++it) {
            const int item = it * THREADS + tid;  // 64 tokens x 36 chunks of 16 codes
            const int t = item / 36, c16 = item % 36;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t < nvalid) {
                const uint8_t *src;
                if (c16 < 32) src = pg8 + (c16 >> 3) * (BS * 128) + t * 128 + (((c16 & 7) ^ (t & 7)) << 4);
                else src = pg8 + 4 * BS * 128 + t * 64 + ((((c16 - 32) & 3) ^ ((t >> 1) & 3)) << 4);
                v = *reinterpret_cast<const uint4 *>(src);
            }
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                h[2 * e] = e4m3x2_f16x2(w[e]);
                h[2 * e + 1] = e4m3x2_f16x2(w[e] >> 16);
            }
            *reinterpret_cast<uint4 *>(smem + KS_OFF + sw_off(t, 2 * c16)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(smem + KS_OFF + sw_off(t, 2 * c16 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
        __syncthreads();  // f16 tile, scales and E ready; the ring slot is free
        const int E_page = flags[1];
        if (warp == 0) {
            fence_proxy_async_smem();
            if (j + NSLOT < npg) issue(j + NSLOT);
        }

        // ---- S = q' K^T: rows 16mt.., tokens 32th..
        float s[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
        {
            const int arow = 16 * mt + (lane & 15);
            const int brow0 = 32 * th + (lane & 7) + 8 * (lane >> 4);
#pragma unroll 4
            for (int kst = 0; kst < DK / 16; ++kst) {
                uint32_t a[4], b0[4], b1[4];
                ldsm_x4(a, qs + sw_off(arow, 2 * kst + (lane >> 4)));
                ldsm_x4(b0, ks + sw_off(brow0, 2 * kst + ((lane >> 3) & 1)));
                ldsm_x4(b1, ks + sw_off(brow0 + 16, 2 * kst + ((lane >> 3) & 1)));
                mma16816<false>(s[0], a, b0[0], b0[1]);
                mma16816<false>(s[1], a, b0[2], b0[3]);
                mma16816<false>(s[2], a, b1[0], b1[1]);
                mma16816<false>(s[3], a, b1[2], b1[3]);
            }
        }
        // ---- scale, mask, row maxima
        const float fe = pow2f(E_page);
        const float fa = rowsc[ra] * fe, fb = rowsc[rb] * fe;
        const int tpage = cc.p * BS;
        float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int tl = 32 * th + 8 * t + 2 * c;
            const float2 sn = *reinterpret_cast<const float2 *>(tsn + tl);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float sne = e ? sn.y : sn.x;
                float xa = s[t][e] * fa * sne, xb = s[t][2 + e] * fb * sne;
                xa = (tpage + tl + e < vis_a) ? xa : -INFINITY;
                xb = (tpage + tl + e < vis_b) ? xb : -INFINITY;
                s[t][e] = xa;
                s[t][2 + e] = xb;
                mxa = fmaxf(mxa, xa);
                mxb = fmaxf(mxb, xb);
            }
        }
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
        if (c == 0) {
            rmax[th * LROWS + ra] = mxa;
            rmax[th * LROWS + rb] = mxb;
        }
        named_barrier(1 + mt, 64);  // the two warps of row tile mt
        mxa = fmaxf(mxa, rmax[(1 - th) * LROWS + ra]);
        mxb = fmaxf(mxb, rmax[(1 - th) * LROWS + rb]);
        const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
        const float basea = (mna == -INFINITY) ? 0.f : mna;
        const float baseb = (mnb == -INFINITY) ? 0.f : mnb;
        const float ala = ex2(m_a - basea), alb = ex2(m_b - baseb);
        m_a = mna;
        m_b = mnb;
        float psa = 0.f, psb = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int tl = 32 * th + 8 * t + 2 * c;
            const float2 sn = *reinterpret_cast<const float2 *>(tsn + tl);
            const float pa0 = ex2(s[t][0] - basea), pa1 = ex2(s[t][1] - basea);
            const float pb0 = ex2(s[t][2] - baseb), pb1 = ex2(s[t][3] - baseb);
            psa += pa0 + pa1;
            psb += pb0 + pb1;
            const int chunk = 4 * th + t;  // tokens 8*chunk .. 8*chunk+7
            *reinterpret_cast<uint32_t *>(smem + PS_OFF + ra * 128 + ((chunk ^ (ra & 7)) << 4) + 4 * c) =
                pack_f16x2(pa0 * sn.x, pa1 * sn.y);
            *reinterpret_cast<uint32_t *>(smem + PS_OFF + rb * 128 + ((chunk ^ (rb & 7)) << 4) + 4 * c) =
                pack_f16x2(pb0 * sn.x, pb1 * sn.y);
        }
        l_a = l_a * ala + psa;
        l_b = l_b * alb + psb;
        if (th == 0 && c == 0) {
            const float fE = pow2f(E_run - E_page);
            alpha[ra] = ala * fE;
            alpha[rb] = alb * fE;
        }
        E_run = E_page;
        __syncthreads();  // P', alpha ready

        // ---- O = alpha O + P' V: rows 32mr.., channels 128dq..
        {
            float al[2][2];
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) al[i][hh] = alpha[32 * mr + 16 * i + g + 8 * hh];
            if (__any_sync(0xffffffffu, al[0][0] != 1.f || al[0][1] != 1.f || al[1][0] != 1.f || al[1][1] != 1.f)) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        o[i][t][0] *= al[i][0];
                        o[i][t][1] *= al[i][0];
                        o[i][t][2] *= al[i][1];
                        o[i][t][3] *= al[i][1];
                    }
            }
            const int prow = 32 * mr + (lane & 15);
            const int vtok = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
            for (int kst = 0; kst < BS / 16; ++kst) {
                uint32_t a0[4], a1[4];
                ldsm_x4(a0, ps + prow * 128 + (((2 * kst + (lane >> 4)) ^ (prow & 7)) << 4));
                ldsm_x4(a1, ps + (prow + 16) * 128 + (((2 * kst + (lane >> 4)) ^ ((prow + 16) & 7)) << 4));
                const int tok = 16 * kst + vtok;
#pragma unroll
                for (int pr = 0; pr < 8; ++pr) {
                    uint32_t b[4];
                    ldsm_x4_t(b, ks + sw_off(tok, 16 * dq + 2 * pr + (lane >> 4)));
                    mma16816<false>(o[0][2 * pr], a0, b[0], b[1]);
                    mma16816<false>(o[1][2 * pr], a1, b[0], b[1]);
                    mma16816<false>(o[0][2 * pr + 1], a0, b[2], b[3]);
                    mma16816<false>(o[1][2 * pr + 1], a1, b[2], b[3]);
                }
            }
        }
        last_p = cc.p;
        cursor_next(cc, P.req, P.B, X, P.mbps);
    }
    if (j < npg && tid == 0) {
        // a wait ran out: let every copy still in flight land before exiting
        for (int i = j; i < min(npg, j + NSLOT); ++i) mbar_wait_bounded(&full[i % NSLOT], (i / NSLOT) & 1, nullptr);
    }
    grid_dependents_launch();
    if (piece_b >= 0) finish_piece();
    // one word per CTA
    unsigned *s_err = reinterpret_cast<unsigned *>(flags + 4);
    if (tid == 0) *s_err = 0u;
    __syncthreads();
    if (err) atomicOr(s_err, err);
    __syncthreads();
    if (tid == 0) atomic_or_err(P.hdr, *s_err);
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
