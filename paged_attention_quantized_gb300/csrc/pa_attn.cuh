// Split-KV paged decode / verify attention for sm_103a.
//
// One CTA computes one work unit (request b, kv head, a run of logical pages)
// for up to 16 query rows of that kv head (the GQA group times next_n).
//
//  * warp NW (the producer) reads the unit's block ids 32 at a time, checks
//    each against [1, num_blocks) and copies the K and V tiles of page p --
//    [bs][row bytes] for this kv head, contiguous in the head-major pool -- into
//    a ring of shared-memory stages with 4-D bulk tensor copies (TMA), 128- or
//    64-byte swizzled so the consumers' 16-byte loads hit distinct banks;
//  * warps 0..NW-1 (consumers) take pages round-robin in logical order; for
//    every 16-token chunk they dequantize K codes in registers into mma B
//    fragments, compute S = q' K^T with m16n8k16 tensor-core MMAs (rows are the
//    16 query rows, fp32 accumulate), run the online softmax (exp2 domain,
//    warp-shuffle row maxima), and accumulate O += P V with V dequantized the
//    same way;
//  * at the end the consumer warps' (m, l, O) are merged in warp order, and
//    the unit writes either the final output (one split) or a normalised
//    partial and its log-sum-exp for the combine kernel.
//
// Pages are ordered by logical position only (1Cat-vLLM PR #494, "Stabilize
// QSA page4 order under KV relocation": physical addresses are payload), so
// results are bitwise identical under relocation.  Token slots at or past
// L_b on the last page are copied but never used: their scores are replaced
// by -inf with a select and their V codes are zeroed before the MMA, so a NaN
// code there cannot reach P.V (1Cat-vLLM PR #647, "Stop grouped-page4
// null-block padding from leaking E4M3 NaN", Root cause and Fix).  Columns of
// block_table past the request's pages are never read.
//
// The K scale: per-tensor scalars and max|k_scale| go into the fp32 score
// scale; a per-channel scale is folded into q as q * (k_scale / max|k_scale|)
// in fp32 and rounded once, so the folded query never exceeds |q|
// (onnxruntime PR #32520, "Normalize the PER_CHANNEL K scale folded into Q
// for paged XQA", Approach).  With f16 MMAs every query row is further scaled
// by a power of two into [-1, 1) (exact) and the factor joins the score scale,
// so bf16 queries of any magnitude fit the f16 operand.
#pragma once

#include "pa_common.cuh"

namespace pa {

constexpr int NW = 4;                      // consumer warps
#ifndef PA_MIN_BLOCKS_SMALL_D
#define PA_MIN_BLOCKS_SMALL_D 3
#endif
#ifndef PA_MIN_BLOCKS_LARGE_D
#define PA_MIN_BLOCKS_LARGE_D 2
#endif
// resident CTAs per SM the register allocation is sized for
template <int D>
constexpr int min_blocks() { return D <= 128 ? PA_MIN_BLOCKS_SMALL_D : PA_MIN_BLOCKS_LARGE_D; }
constexpr int ATTN_THREADS = (NW + 1) * 32;
constexpr int MAX_STAGES = 32;
constexpr int ROWS = 16;                   // query rows per CTA (mma M)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

template <int KVT>
struct KvTraits;
template <>
struct KvTraits<PA_F16> { static constexpr int BITS = 16; static constexpr bool BF = false; };
template <>
struct KvTraits<PA_BF16> { static constexpr int BITS = 16; static constexpr bool BF = true; };
template <>
struct KvTraits<PA_E4M3> { static constexpr int BITS = 8; static constexpr bool BF = false; };
template <>
struct KvTraits<PA_INT8> { static constexpr int BITS = 8; static constexpr bool BF = false; };
template <>
struct KvTraits<PA_INT4> { static constexpr int BITS = 4; static constexpr bool BF = false; };

template <int KVT, int D>
struct Geo {
    static constexpr int BITS = KvTraits<KVT>::BITS;
    static constexpr bool BF = KvTraits<KVT>::BF;    // bf16 MMA (else f16)
    static constexpr int RB = D * BITS / 8;          // bytes of one token row
    static constexpr int SW = RB >= 128 ? 128 : 64;  // segment = swizzle span
    static constexpr int NSEG = RB / SW;
    static constexpr int EPS = SW * 8 / BITS;        // elements per segment
    static constexpr int KSTEPS = D / 16;            // k-steps of S = q K^T
    static constexpr int KPS = KSTEPS / NSEG;        // k-steps per segment
    static constexpr int KWORDS = SW / 16;           // 32-bit K words per lane per segment
    static constexpr int VWORDS = SW / 32;           // 32-bit V words per lane per row per segment
    static constexpr int EPL = EPS / 8;              // V elements per lane per segment
    static constexpr int NT2 = D / 8;                // n-tiles of O
    static_assert(RB % SW == 0, "row must be whole segments");
    static_assert(NSEG * EPS == D, "segments must cover the row");
    static_assert(EPL * NSEG == NT2, "V lanes must cover the row");
    static_assert(KPS * NSEG == KSTEPS, "k-steps must split evenly");
};

// Byte offset of 16-byte chunk `chunk` of segment `seg` of token row `s` in a
// [NSEG][bs][SW] tile written by a swizzled tensor copy (the tile is 1024-byte
// aligned): 128B swizzle XORs the chunk index with s mod 8, 64B swizzle with
// (s / 2) mod 4.
template <int SW>
__device__ __forceinline__ uint32_t tile_off(int s, int seg, int chunk, int bs) {
    if constexpr (SW == 128) return (uint32_t)(seg * bs * 128 + s * 128 + ((chunk ^ (s & 7)) << 4));
    else return (uint32_t)(seg * bs * 64 + s * 64 + ((chunk ^ ((s >> 1) & 3)) << 4));
}

// Channel held by lane-quad index c in element e (0..3 -> mma k index 2c, 2c+1,
// 2c+8, 2c+9) of global k-step K.  K is contracted against q, so any
// bijection works as long as q uses the same one; this one lets every lane
// read 16-byte runs of a K row.
template <int KVT, int D>
__device__ __forceinline__ int phys_ch(int K, int c, int e) {
    using G = Geo<KVT, D>;
    const int seg = K / G::KPS, j = K % G::KPS;
    const int base = seg * G::EPS + c * (G::EPS / 4);
    if constexpr (G::BITS == 4) {
        const int x = base + 8 * (j >> 1);
        const int lo = (j & 1) ? 2 : 0;
        // e: 0 -> x+lo, 1 -> x+lo+4, 2 -> x+lo+1, 3 -> x+lo+5
        return x + lo + ((e & 1) ? 4 : 0) + (e >> 1);
    } else {
        return base + 4 * j + e;
    }
}

// B fragment of S = q K^T for k-step j of a segment from this lane's K words.
template <int KVT>
__device__ __forceinline__ void k_frag(const uint32_t *w, int j, uint32_t &b0, uint32_t &b1) {
    if constexpr (KVT == PA_F16 || KVT == PA_BF16) {
        b0 = w[2 * j];
        b1 = w[2 * j + 1];
    } else if constexpr (KVT == PA_E4M3) {
        b0 = e4m3x2_f16x2(w[j]);
        b1 = e4m3x2_f16x2(w[j] >> 16);
    } else if constexpr (KVT == PA_INT8) {
        const uint32_t u = w[j] ^ 0x80808080u;
        b0 = u8pair_f16x2(u, 0x4140);
        b1 = u8pair_f16x2(u, 0x4342);
    } else {  // INT4
        uint32_t u = w[j >> 1] ^ 0x88888888u;
        if (j & 1) u >>= 8;
        b0 = u4lo_f16x2(u);
        b1 = u4hi_f16x2(u);
    }
}

// B fragments of O += P V for the EPL elements of one segment.  ra, rb: rows
// 2c and 2c+1 (-> b0), rc, rd: rows 2c+8, 2c+9 (-> b1), VWORDS words each.
template <int KVT, int EPL, int VW>
__device__ __forceinline__ void v_frags(const uint32_t *ra, const uint32_t *rb, const uint32_t *rc,
                                        const uint32_t *rd, uint32_t (*bf)[2]) {
#pragma unroll
    for (int k = 0; k < VW; ++k) {
        if constexpr (KVT == PA_F16 || KVT == PA_BF16) {
            bf[2 * k][0] = __byte_perm(ra[k], rb[k], 0x5410);
            bf[2 * k + 1][0] = __byte_perm(ra[k], rb[k], 0x7632);
            bf[2 * k][1] = __byte_perm(rc[k], rd[k], 0x5410);
            bf[2 * k + 1][1] = __byte_perm(rc[k], rd[k], 0x7632);
        } else if constexpr (KVT == PA_E4M3) {
            const uint32_t t0 = __byte_perm(ra[k], rb[k], 0x5140), t1 = __byte_perm(ra[k], rb[k], 0x7362);
            const uint32_t u0 = __byte_perm(rc[k], rd[k], 0x5140), u1 = __byte_perm(rc[k], rd[k], 0x7362);
            bf[4 * k][0] = e4m3x2_f16x2(t0);
            bf[4 * k + 1][0] = e4m3x2_f16x2(t0 >> 16);
            bf[4 * k + 2][0] = e4m3x2_f16x2(t1);
            bf[4 * k + 3][0] = e4m3x2_f16x2(t1 >> 16);
            bf[4 * k][1] = e4m3x2_f16x2(u0);
            bf[4 * k + 1][1] = e4m3x2_f16x2(u0 >> 16);
            bf[4 * k + 2][1] = e4m3x2_f16x2(u1);
            bf[4 * k + 3][1] = e4m3x2_f16x2(u1 >> 16);
        } else if constexpr (KVT == PA_INT8) {
            const uint32_t xa = ra[k] ^ 0x80808080u, xb = rb[k] ^ 0x80808080u;
            const uint32_t xc = rc[k] ^ 0x80808080u, xd = rd[k] ^ 0x80808080u;
            const uint32_t t0 = __byte_perm(xa, xb, 0x5140), t1 = __byte_perm(xa, xb, 0x7362);
            const uint32_t u0 = __byte_perm(xc, xd, 0x5140), u1 = __byte_perm(xc, xd, 0x7362);
            bf[4 * k][0] = u8pair_f16x2(t0, 0x4140);
            bf[4 * k + 1][0] = u8pair_f16x2(t0, 0x4342);
            bf[4 * k + 2][0] = u8pair_f16x2(t1, 0x4140);
            bf[4 * k + 3][0] = u8pair_f16x2(t1, 0x4342);
            bf[4 * k][1] = u8pair_f16x2(u0, 0x4140);
            bf[4 * k + 1][1] = u8pair_f16x2(u0, 0x4342);
            bf[4 * k + 2][1] = u8pair_f16x2(u1, 0x4140);
            bf[4 * k + 3][1] = u8pair_f16x2(u1, 0x4342);
        } else {  // INT4: 8 channels per word
            const uint32_t xa = ra[k] ^ 0x88888888u, xb = rb[k] ^ 0x88888888u;
            const uint32_t xc = rc[k] ^ 0x88888888u, xd = rd[k] ^ 0x88888888u;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t sel = half ? 0x7632 : 0x5410;
                const uint32_t t = __byte_perm(xa, xb, sel), u = __byte_perm(xc, xd, sel);
                const int e = 8 * k + 4 * half;
                bf[e][0] = u4lo_f16x2(t);
                bf[e + 1][0] = u4hi_f16x2(t);
                bf[e + 2][0] = u4lo_f16x2(t >> 8);
                bf[e + 3][0] = u4hi_f16x2(t >> 8);
                bf[e][1] = u4lo_f16x2(u);
                bf[e + 1][1] = u4hi_f16x2(u);
                bf[e + 2][1] = u4lo_f16x2(u >> 8);
                bf[e + 3][1] = u4hi_f16x2(u >> 8);
            }
        }
    }
}

template <int N>
__device__ __forceinline__ void lds_words(uint32_t *w, const uint8_t *p) {
    if constexpr (N == 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (N == 2) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = v.x; w[1] = v.y;
    }
}

struct SmemMisc {
    float sc[ROWS];        // score scale per row (log2 domain)
    int vis[ROWS];         // visible tokens per row
    float m_w[NW][ROWS];   // per-warp running max (log2 domain)
    float l_w[NW][ROWS];   // per-warp running sum
    float rowmax[ROWS];    // max |q'| per row (prologue)
    int bad;               // unit must be NaN-filled
    int abort_flag;        // a bounded wait ran out
    uint32_t err;          // error bits to publish
};

template <int KVT, int D>
__device__ __forceinline__ float load_q(const AttnParams &P, int b, int j, int h, int d) {
    const size_t idx = (((size_t)b * P.n + j) * P.Hq + h) * D + d;
    const uint16_t bits = reinterpret_cast<const uint16_t *>(P.q)[idx];
    if (P.q_dtype == PA_BF16) return __uint_as_float((uint32_t)bits << 16);
    return __half2float(__ushort_as_half(bits));
}

template <int KVT, int D>
__global__ void __launch_bounds__(ATTN_THREADS, min_blocks<D>())
    pa_attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, AttnParams P) {
    using G = Geo<KVT, D>;
    constexpr bool BF = G::BF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int unit = blockIdx.x;
    const int rblk = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ST = P.stages;
    const int bs = P.bs;
    const int tile_bytes = bs * G::RB;

    // shared-memory carve-up
    uint8_t *ring = smem;
    uint32_t *qs = reinterpret_cast<uint32_t *>(ring + (size_t)ST * P.stage_bytes);  // [KSTEPS][32][4]
    // [ROWS][D] merge buffer: the ring is free once every page has been consumed
    // (all copies landed and were read); the host sizes the ring to hold it
    float *mbuf = reinterpret_cast<float *>(ring);
    SmemMisc *ms = reinterpret_cast<SmemMisc *>(qs + G::KSTEPS * 128);
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(ms) + ((sizeof(SmemMisc) + 15) & ~15));
    uint64_t *empty = full + MAX_STAGES;

    const uint32_t num_units = P.hdr[HDR_NUM_UNITS];
    if (unit >= (int)num_units || unit >= P.max_units) return;

    const int4 U = P.units[unit];
    // a unit record that does not fit this problem (workspace planned for
    // another problem) is rejected before anything it names is read
    const bool unit_ok = U.x >= 0 && U.x < P.B && (U.y >> 16) < P.Hkv && U.z >= 0 && U.z <= U.w &&
                         U.w <= P.mbps;
    const int b = unit_ok ? U.x : 0, kvh = unit_ok ? (U.y >> 16) : 0, split = U.y & 0xFFFF;
    const int p0 = unit_ok ? U.z : 0, p1 = unit_ok ? U.w : 0;
    const int4 Rq = P.req[b];
    const int L = P.context_lens[b];
    const int S_b = Rq.y;
    const int npages = p1 - p0;
    const int r0 = rblk * ROWS;

    if (threadIdx.x == 0) {
        uint32_t err = 0;
        int bad = 0;
        if (!unit_ok) { bad = 1; err |= PA_DEV_ERR_STALE_PLAN; }
        if (Rq.w != 0) { bad = 1; err |= PA_DEV_ERR_CONTEXT_LEN; }
        if (L != Rq.x || (long long)p1 * bs > (long long)L + bs - 1) { bad = 1; err |= PA_DEV_ERR_STALE_PLAN; }
        // the ring depth must be a positive multiple of the consumer warps
        // (see the host's stage choice); never run a ring that could alias
        if (ST < NW || ST > MAX_STAGES || ST % NW != 0) { bad = 1; err |= PA_DEV_ERR_TIMEOUT; }
        ms->bad = bad;
        ms->err = err;
        ms->abort_flag = 0;
        for (int s = 0; s < min(ST, MAX_STAGES); ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();

    const bool bad0 = ms->bad != 0;

    if (warp == NW) {
        // ------------------------------------------------------- producer
        int issued = 0;  // pages whose copy was started (in order)
        if (!bad0) {
            if (lane == 0) {
                tma_prefetch_desc(&tmk);
                tma_prefetch_desc(&tmv);
            }
            const int32_t *tab = P.block_table + (size_t)b * P.mbps + p0;
            bool stop = false;
            int id_next = (lane < npages) ? tab[lane] : 0;
            for (int base = 0; base < npages && !stop; base += 32) {
                const int n_here = min(32, npages - base);
                const int id = id_next;
                // block ids of the next batch, in flight while this one is issued
                id_next = (base + 32 + lane < npages) ? tab[base + 32 + lane] : 0;
                const bool ok = (lane >= n_here) || (id >= 1 && id < P.num_blocks);
                const unsigned okmask = __ballot_sync(0xffffffffu, ok);
                for (int k = 0; k < n_here; ++k) {
                    const int i = base + k;
                    const int slot = i % ST;
                    if (i >= ST && !mbar_wait_bounded(&empty[slot], ((i / ST) - 1) & 1, &ms->abort_flag)) {
                        if (lane == 0) { ms->abort_flag = 1; atomicOr(&ms->err, PA_DEV_ERR_TIMEOUT); }
                        stop = true;
                        break;
                    }
                    const int blk = __shfl_sync(0xffffffffu, id, k);
                    if (lane == 0) {
                        uint8_t *kt = ring + (size_t)slot * P.stage_bytes;
                        uint8_t *vt = kt + tile_bytes;
                        if ((okmask >> k) & 1u) {
                            mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * tile_bytes));
#pragma unroll
                            for (int sg = 0; sg < G::NSEG; ++sg) {
                                tma_load_4d(kt + sg * bs * G::SW, &tmk, &full[slot], sg * G::SW, 0, kvh, blk);
                                tma_load_4d(vt + sg * bs * G::SW, &tmv, &full[slot], sg * G::SW, 0, kvh, blk);
                            }
                        } else {
                            // invalid id: no copy; the unit is NaN-filled
                            atomicOr(&ms->err, PA_DEV_ERR_BLOCK_ID);
                            ms->bad = 1;
                            mbar_arrive(&full[slot]);
                        }
                    }
                    issued = i + 1;
                    __syncwarp();
                }
            }
        }
        // wait for the consumers, then make sure no copy is still landing
        asm volatile("bar.sync 2, %0;" ::"n"(ATTN_THREADS));
        if (lane == 0 && ms->abort_flag) {
            volatile int never = 0;
            for (int i = max(0, issued - ST); i < issued; ++i)
                mbar_wait_bounded(&full[i % ST], (i / ST) & 1, &never);
        }
        if (threadIdx.x == NW * 32) atomic_or_err(P.hdr, ms->err);
        return;
    }

    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, c = lane & 3;
    const int ctid = threadIdx.x;  // 0 .. NW*32-1

    // per-row constants
    if (ctid < ROWS) {
        const int r = r0 + ctid;
        int vis = L;
        if (r < P.R && P.causal) vis = L - (P.n - 1 - r / P.G);
        ms->vis[ctid] = vis;
    }
    const float kmax = (P.k_mode == PA_SCALE_CHANNEL) ? __uint_as_float(P.hdr[HDR_KMAX]) : 1.0f;
    const float kscal = (P.k_mode == PA_SCALE_TENSOR) ? P.k_scale[0] : kmax;
    // fold factor of channel d (per-channel K scale normalised by its max)
    auto fold = [&](int d) -> float {
        return (P.k_mode == PA_SCALE_CHANNEL) ? P.k_scale[(size_t)kvh * D + d] / kmax : 1.0f;
    };
    // row maxima of |q'| (f16 MMAs only)
    if constexpr (!BF) {
        const int row = ctid >> 3, sub = ctid & 7;  // 8 threads per row
        float mx = 0.f;
        const int r = r0 + row;
        if (r < P.R) {
            const int jq = r / P.G, h = kvh * P.G + (r % P.G);
            for (int d = sub; d < D; d += 8) mx = fmaxf(mx, fabsf(load_q<KVT, D>(P, b, jq, h, d) * fold(d)));
        }
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (sub == 0) ms->rowmax[row] = mx;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32));
    if (ctid < ROWS) {
        float rho = 1.0f;
        if constexpr (!BF) {
            const float mx = ms->rowmax[ctid];
            if (mx > 0.f && mx < 3.0e38f) {
                int e;
                frexpf(mx, &e);  // mx = f * 2^e, f in [0.5, 1)
                rho = ldexpf(1.0f, e);
            }
        }
        ms->rowmax[ctid] = rho;  // reuse: the power-of-two row factor
        ms->sc[ctid] = P.softmax_scale * kscal * rho * LOG2E;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32));
    // q' fragments, shared by all consumer warps: warp w builds k-steps w, w+NW, ...
    for (int K = warp; K < G::KSTEPS; K += NW) {
        uint32_t a[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {       // a0a1/a2a3 use e=0,1; a4a5/a6a7 use e=2,3
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {         // row g, row g+8
                const int row = g + 8 * rr, r = r0 + row;
                float v0 = 0.f, v1 = 0.f;
                if (r < P.R) {
                    const int jq = r / P.G, h = kvh * P.G + (r % P.G);
                    const float inv = 1.0f / ms->rowmax[row];
                    const int d0 = phys_ch<KVT, D>(K, c, 2 * half), d1 = phys_ch<KVT, D>(K, c, 2 * half + 1);
                    v0 = load_q<KVT, D>(P, b, jq, h, d0) * fold(d0) * inv;
                    v1 = load_q<KVT, D>(P, b, jq, h, d1) * fold(d1) * inv;
                }
                a[2 * half + rr] = pack2<BF>(v0, v1);
            }
        }
        reinterpret_cast<uint4 *>(qs)[K * 32 + lane] = make_uint4(a[0], a[1], a[2], a[3]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32));

    const float sc0 = ms->sc[g], sc1 = ms->sc[g + 8];
    const int vis0 = ms->vis[g], vis1 = ms->vis[g + 8];
    const int vis_min = min(vis0, vis1);

    float o[G::NT2][4];
#pragma unroll
    for (int t = 0; t < G::NT2; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool aborted = false;

    for (int i = warp; i < (bad0 ? 0 : npages); i += NW) {
        const int slot = i % ST;
        if (!mbar_wait_bounded(&full[slot], (i / ST) & 1, &ms->abort_flag)) {
            if (lane == 0) { ms->abort_flag = 1; atomicOr(&ms->err, PA_DEV_ERR_TIMEOUT); }
            aborted = true;
            break;
        }
        if (!*reinterpret_cast<volatile int *>(&ms->bad)) {
            const uint8_t *kt = ring + (size_t)slot * P.stage_bytes;
            const uint8_t *vt = kt + tile_bytes;
            const int page = p0 + i;
            const int t_page = page * bs;
            const int nvalid = min(bs, L - t_page);  // real tokens in this page
            for (int ch = 0; ch < bs; ch += 16) {
                // ---- S = q' K^T for tokens ch .. ch+15 (two n-tiles)
                float s[2][4];
#pragma unroll
                for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
                for (int sg = 0; sg < G::NSEG; ++sg) {
                    uint32_t kw[2][G::KWORDS];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int srow = ch + 8 * t + g;
                        if constexpr (G::SW == 128) {
                            lds_words<4>(kw[t], kt + tile_off<128>(srow, sg, 2 * c, bs));
                            lds_words<4>(kw[t] + 4, kt + tile_off<128>(srow, sg, 2 * c + 1, bs));
                        } else {
                            lds_words<4>(kw[t], kt + tile_off<64>(srow, sg, c, bs));
                        }
                    }
#pragma unroll
                    for (int j = 0; j < G::KPS; ++j) {
                        const uint4 av = reinterpret_cast<const uint4 *>(qs)[(sg * G::KPS + j) * 32 + lane];
                        const uint32_t a[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            uint32_t b0, b1;
                            k_frag<KVT>(kw[t], j, b0, b1);
                            mma16816<BF>(s[t], a, b0, b1);
                        }
                    }
                }
                // ---- scale, mask, online softmax
                const int tbase = t_page + ch + 2 * c;
                const bool need_mask = (t_page + ch + 16 > vis_min);
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = tbase + 8 * t + e;
                        float x0 = s[t][e] * sc0, x1 = s[t][2 + e] * sc1;
                        if (need_mask) {
                            x0 = (tok < vis0) ? x0 : -INFINITY;
                            x1 = (tok < vis1) ? x1 : -INFINITY;
                        }
                        s[t][e] = x0;
                        s[t][2 + e] = x1;
                        mx0 = fmaxf(mx0, x0);
                        mx1 = fmaxf(mx1, x1);
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
                const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
                const float al0 = ex2(m0 - base0), al1 = ex2(m1 - base1);  // m = -inf -> 0
                m0 = mn0;
                m1 = mn1;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        s[t][e] = ex2(s[t][e] - base0);
                        s[t][2 + e] = ex2(s[t][2 + e] - base1);
                        ps0 += s[t][e];
                        ps1 += s[t][2 + e];
                    }
                }
                l0 = l0 * al0 + ps0;
                l1 = l1 * al1 + ps1;
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int t = 0; t < G::NT2; ++t) {
                        o[t][0] *= al0;
                        o[t][1] *= al0;
                        o[t][2] *= al1;
                        o[t][3] *= al1;
                    }
                }
                // ---- O += P V
                uint32_t pa[4];
                pa[0] = pack2<BF>(s[0][0], s[0][1]);
                pa[1] = pack2<BF>(s[0][2], s[0][3]);
                pa[2] = pack2<BF>(s[1][0], s[1][1]);
                pa[3] = pack2<BF>(s[1][2], s[1][3]);
                const int rA = ch + 2 * c, rB = rA + 1, rC = rA + 8, rD = rA + 9;
                const bool zA = rA >= nvalid, zB = rB >= nvalid, zC = rC >= nvalid, zD = rD >= nvalid;
#pragma unroll
                for (int sg = 0; sg < G::NSEG; ++sg) {
                    uint32_t va[G::VWORDS], vb[G::VWORDS], vc[G::VWORDS], vd[G::VWORDS];
                    if constexpr (G::SW == 128) {
                        lds_words<4>(va, vt + tile_off<128>(rA, sg, g, bs));
                        lds_words<4>(vb, vt + tile_off<128>(rB, sg, g, bs));
                        lds_words<4>(vc, vt + tile_off<128>(rC, sg, g, bs));
                        lds_words<4>(vd, vt + tile_off<128>(rD, sg, g, bs));
                    } else {
                        const int hoff = 8 * (g & 1);
                        lds_words<2>(va, vt + tile_off<64>(rA, sg, g >> 1, bs) + hoff);
                        lds_words<2>(vb, vt + tile_off<64>(rB, sg, g >> 1, bs) + hoff);
                        lds_words<2>(vc, vt + tile_off<64>(rC, sg, g >> 1, bs) + hoff);
                        lds_words<2>(vd, vt + tile_off<64>(rD, sg, g >> 1, bs) + hoff);
                    }
#pragma unroll
                    for (int k = 0; k < G::VWORDS; ++k) {  // padding slots: codes -> 0
                        va[k] = zA ? 0u : va[k];
                        vb[k] = zB ? 0u : vb[k];
                        vc[k] = zC ? 0u : vc[k];
                        vd[k] = zD ? 0u : vd[k];
                    }
                    uint32_t bf[G::EPL][2];
                    v_frags<KVT, G::EPL, G::VWORDS>(va, vb, vc, vd, bf);
#pragma unroll
                    for (int e = 0; e < G::EPL; ++e) mma16816<BF>(o[sg * G::EPL + e], pa, bf[e][0], bf[e][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    (void)aborted;

    // ------------------------------------------------------ merge the warps
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (c == 0) {
        ms->m_w[warp][g] = m0;
        ms->m_w[warp][g + 8] = m1;
        ms->l_w[warp][g] = l0;
        ms->l_w[warp][g + 8] = l1;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32));
    float f0, f1;
    {
        float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            M0 = fmaxf(M0, ms->m_w[w][g]);
            M1 = fmaxf(M1, ms->m_w[w][g + 8]);
        }
        f0 = (M0 == -INFINITY) ? 0.f : ex2(m0 - M0);
        f1 = (M1 == -INFINITY) ? 0.f : ex2(m1 - M1);
    }
    for (int w = 0; w < NW; ++w) {
        if (warp == w) {
#pragma unroll
            for (int t = 0; t < G::NT2; ++t) {
                const int sg = t / G::EPL, e = t % G::EPL;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int d = sg * G::EPS + (2 * c + cc) * G::EPL + e;
                    float *p0r = mbuf + g * D + d;
                    float *p1r = mbuf + (g + 8) * D + d;
                    if (w == 0) {
                        *p0r = o[t][cc] * f0;
                        *p1r = o[t][2 + cc] * f1;
                    } else {
                        *p0r += o[t][cc] * f0;
                        *p1r += o[t][2 + cc] * f1;
                    }
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NW * 32));
    }

    // ---------------------------------------------------------- epilogue
    const bool bad = ms->bad || ms->abort_flag;
    const int rows_here = unit_ok ? min(ROWS, P.R - r0) : 0;
    const bool final_out = (S_b == 1);
    for (int idx = ctid; idx < rows_here * D; idx += NW * 32) {
        const int row = idx / D, d = idx % D;
        float M = -INFINITY, Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, ms->m_w[w][row]);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) Lsum += ms->l_w[w][row] * ex2(ms->m_w[w][row] - M);
        }
        float val = (Lsum > 0.f) ? mbuf[row * D + d] / Lsum : 0.f;
        float lse_v = (Lsum > 0.f) ? (M + lg2(Lsum)) * LN2 : -INFINITY;
        if (bad) { val = __int_as_float(0x7fc00000); lse_v = __int_as_float(0x7fc00000); }
        const int r = r0 + row;
        const int jq = r / P.G, h = kvh * P.G + (r % P.G);
        if (final_out) {
            float vsc = 1.0f;
            if (P.v_mode == PA_SCALE_TENSOR) vsc = P.v_scale[0];
            else if (P.v_mode == PA_SCALE_CHANNEL) vsc = P.v_scale[(size_t)kvh * D + d];
            const float y = val * vsc;
            const size_t oi = (((size_t)b * P.n + jq) * P.Hq + h) * D + d;
            if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = y;
            else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(y);
            else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(y);
            if (P.lse != nullptr && d == 0) P.lse[((size_t)b * P.n + jq) * P.Hq + h] = lse_v;
        } else {
            P.part_o[((size_t)unit * P.R + r) * D + d] = val;
            if (d == 0) P.part_lse[(size_t)unit * P.R + r] = lse_v;
        }
    }
    (void)split;
    asm volatile("bar.sync 2, %0;" ::"n"(ATTN_THREADS));
}

}  // namespace pa
