// Split-KV paged decode / verify attention for sm_103a.
//
// Persistent CTAs of 4 warps; each warp (or, for D = 256 with query rows on
// the MMA M axis, each pair of warps sharing one ring and splitting the
// channel segments between them) is an independent worker that streams its
// share of the logical page sequence for up to 16 query rows of a kv head.
// With more than 16 query rows per kv head the workers come in groups, one
// per block of 16 rows, that share one run of pages: each page of the
// group's share is read from HBM once and from L2 by the other row blocks.
//
//  * the worker's lane 0 reads block ids 32 at a time, checks each against
//    [1, num_blocks) and copies the K and V tiles of its next pages -- [bs][row
//    bytes] for one kv head, contiguous in the head-major pool -- into its ring
//    of shared-memory slots, one 5-D bulk tensor copy (TMA) per tile: rows of
//    more than 128 bytes are cut into 128-byte segments, the segment dimension
//    placed outside the rows, and each line 128- or 64-byte swizzled so the
//    16-byte loads of the lanes hit distinct banks (the copy instruction, not
//    the bytes, is what costs the issuing warp);
//  * for every 16-token chunk of a page the worker dequantizes K codes in
//    registers into mma fragments, computes S = q' K^T with m16n8k16 tensor-
//    core MMAs (query rows on M, or, with at most 8 rows per kv head, tokens
//    on M: S^T = K q'^T), runs the online softmax (exp2 domain; the row
//    maximum is lazy: it is reduced across lanes, and O and the row sum
//    rescaled, only when some score passes it by more than 2^8, so P stays
//    below 256) and accumulates O += P V with V dequantized the same way;
//  * its run of pages inside one segment (request, kv head, block of query
//    rows) is a piece: a whole segment writes the output, a cut one a
//    normalised partial and its log-sum-exp for the combine kernel.
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

constexpr int NWK = 4;                     // warps per CTA, each an independent stream
enum : int { WP_WHOLE = 0, WP_PART = 1, WP_MERGED = 2 };  // what a work page is (see pa_attn_kernel)
#ifndef PA_MERGE_BLOCKS
#define PA_MERGE_BLOCKS 2
#endif
constexpr int MERGE_BLOCKS = PA_MERGE_BLOCKS;  // blocks per merged work page
#ifndef PA_MIN_BLOCKS_SMALL_D
#define PA_MIN_BLOCKS_SMALL_D 2
#endif
#ifndef PA_MIN_BLOCKS_LARGE_D
#define PA_MIN_BLOCKS_LARGE_D 1
#endif
#ifndef PA_MIN_BLOCKS_TOKM
#define PA_MIN_BLOCKS_TOKM 4
#endif
#ifndef PA_MIN_BLOCKS_PAIR
#define PA_MIN_BLOCKS_PAIR 3
#endif
#ifndef PA_MIN_BLOCKS_TOKM_16BIT
#define PA_MIN_BLOCKS_TOKM_16BIT 3
#endif
// resident CTAs per SM the register and shared-memory budgets are sized for
// (tokens-as-M kernels need fewer registers; with 16-bit codes two ring pages
// per warp only fit 3 CTAs per SM at D = 128, so those are given the registers
// of 3)
__host__ __device__ constexpr int min_blocks(int bits, int D, bool tokm, bool pair) {
    return D <= 128 ? (tokm ? (bits == 16 && D == 128 ? PA_MIN_BLOCKS_TOKM_16BIT : PA_MIN_BLOCKS_TOKM)
                            : PA_MIN_BLOCKS_SMALL_D)
                    : (pair ? PA_MIN_BLOCKS_PAIR : PA_MIN_BLOCKS_LARGE_D);
}
// q' fragments live in registers for D <= 128, in the warp's shared memory above
template <int D>
__host__ __device__ constexpr bool q_in_regs() { return D <= 128; }
// Paired warps (D = 256, query rows on the MMA M axis, an even number of
// 128-byte channel segments): two warps share one worker's ring and each takes
// half of the channel segments -- half of the q.K contraction (the partial
// scores are summed through shared memory) and half of the output channels --
// so the O accumulator is 64 registers instead of 128.
__host__ __device__ constexpr bool pair_mode(int D, bool tokm, int nseg) { return !tokm && D == 256 && nseg % 2 == 0; }
constexpr int ATTN_THREADS = NWK * 32;
constexpr int MAX_SLOTS = 16;              // ring slots (pages) per warp
constexpr int ROWS = 16;                   // query rows per segment (mma M)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float LAZY_SLACK = 8.0f;         // lazy row maximum (exp2 domain): reduce and rescale only when a score exceeds m + 8

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
        uint32_t u = w[j >> 1];
        if (j & 1) u >>= 8;
        b0 = s4lo_f16x2(u);
        b1 = s4hi_f16x2(u);
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
            const uint32_t xa = ra[k], xb = rb[k], xc = rc[k], xd = rd[k];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t sel = half ? 0x7632 : 0x5410;
                const uint32_t t = __byte_perm(xa, xb, sel), u = __byte_perm(xc, xd, sel);
                const int e = 8 * k + 4 * half;
                bf[e][0] = s4lo_f16x2(t);
                bf[e + 1][0] = s4hi_f16x2(t);
                bf[e + 2][0] = s4lo_f16x2(t >> 8);
                bf[e + 3][0] = s4hi_f16x2(t >> 8);
                bf[e][1] = s4lo_f16x2(u);
                bf[e + 1][1] = s4hi_f16x2(u);
                bf[e + 2][1] = s4lo_f16x2(u >> 8);
                bf[e + 3][1] = s4hi_f16x2(u >> 8);
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

// Bytes of one worker's shared memory: its ring of pages, its q' fragments
// (when they do not live in registers), for paired warps the score exchange
// (2 buffers x 2 warps x 32 lanes x 8 floats) and per-slot flags, and the ring
// barriers, rounded to 1 KB.
constexpr int XCHG_BYTES = 2 * 2 * 32 * 8 * 4;
template <int D>
__host__ __device__ constexpr int warp_smem_bytes(int slots, int page_bytes, bool pair = false) {
    return (slots * page_bytes + (q_in_regs<D>() ? 0 : (D / 16) * 512) + (pair ? XCHG_BYTES + MAX_SLOTS * 4 + 16 : 0) +
            MAX_SLOTS * 8 + 1023) / 1024 * 1024;
}

// Position of logical page p of segment q (kv head * row blocks + row block)
// of request b in the global page sequence: PS_b * X + q * P_b + p, where
// PS_b = sum of P over earlier requests and X = segments per request.
struct Cursor {
    int b, q, p;  // request, segment within the request, page
    int Pb;       // pages of request b
    int L;        // its planned length (kept only by cursors that need it: WL)
};

// pages of request b as planned, clamped to the table width so that a
// workspace planned for another problem cannot send a read out of bounds
__device__ __forceinline__ int planned_pages(const int4 *req, int b, int mbps) {
    return min(max(req[b].y, 0), mbps);
}

template <bool WL = false>
__device__ __forceinline__ void cursor_next(Cursor &cu, const int4 *req, int B, int X, int mbps) {
    if (++cu.p < cu.Pb) return;
    cu.p = 0;
    if (++cu.q < X) return;
    cu.q = 0;
    do {
        ++cu.b;
        cu.Pb = cu.b < B ? planned_pages(req, cu.b, mbps) : 0;
        if constexpr (WL) cu.L = cu.b < B ? req[cu.b].x : 0;
    } while (cu.b < B && cu.Pb == 0);
}

// The cursor of global position x (< total pages): the request is the last
// one whose first position is <= x (it cannot be empty).  Returns b = B if
// the records do not describe such a request.
__device__ __forceinline__ Cursor cursor_at(long long x, const int4 *req, int B, int X, int mbps) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)req[mid].z * X <= x) lo = mid;
        else hi = mid - 1;
    }
    Cursor cu;
    cu.b = lo;
    cu.Pb = planned_pages(req, lo, mbps);
    cu.L = req[lo].x;
    const long long off = x - (long long)req[lo].z * X;
    if (cu.Pb < 1 || off < 0 || off >= (long long)cu.Pb * X) {
        cu.b = B;
        cu.q = cu.p = 0;
        return cu;
    }
    cu.q = (int)(off / cu.Pb);
    cu.p = (int)(off % cu.Pb);
    return cu;
}

// 8x8 transpose of 16-bit elements held in the mma fragment layout (lane t
// holds row t/4, columns 2(t%4) and 2(t%4)+1)
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(a));
    return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The 4 q values of row (b, j, h) that lane-quad index c uses in k-step K, in
// the element order e = 0..3 of phys_ch: with 8- or 16-bit codes they are 4
// consecutive channels (one 8-byte load when q is 8-byte aligned), with INT4
// two pairs of consecutive channels (two 4-byte loads when 4-byte aligned).
template <int KVT, int D>
__device__ __forceinline__ void load_q4(const AttnParams &P, int b, int j, int h, int K, int c, float *v) {
    using G = Geo<KVT, D>;
    const uint16_t *row = reinterpret_cast<const uint16_t *>(P.q) + (((size_t)b * P.n + j) * P.Hq + h) * D;
    auto f = [&](uint32_t bits) -> float {
        return (P.q_dtype == PA_BF16) ? __uint_as_float(bits << 16) : __half2float(__ushort_as_half((uint16_t)bits));
    };
    const int d0 = phys_ch<KVT, D>(K, c, 0);
    if constexpr (G::BITS == 4) {
        const int d1 = phys_ch<KVT, D>(K, c, 1);  // d0 + 4; e = 2, 3 are d0 + 1, d1 + 1
        if ((reinterpret_cast<uintptr_t>(P.q) & 3) == 0) {
            const uint32_t a = *reinterpret_cast<const uint32_t *>(row + d0);
            const uint32_t bb = *reinterpret_cast<const uint32_t *>(row + d1);
            v[0] = f(a & 0xFFFFu); v[2] = f(a >> 16); v[1] = f(bb & 0xFFFFu); v[3] = f(bb >> 16);
        } else {
            v[0] = f(row[d0]); v[2] = f(row[d0 + 1]); v[1] = f(row[d1]); v[3] = f(row[d1 + 1]);
        }
    } else {
        if ((reinterpret_cast<uintptr_t>(P.q) & 7) == 0) {
            const uint2 w = *reinterpret_cast<const uint2 *>(row + d0);
            v[0] = f(w.x & 0xFFFFu); v[1] = f(w.x >> 16); v[2] = f(w.y & 0xFFFFu); v[3] = f(w.y >> 16);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = f(row[d0 + e]);
        }
    }
}

// TOKM: at most 8 query rows per kv head.  Tokens then form the MMA M axis
// (S^T = K q'^T and O^T = V^T P^T with the rows as N = 8), which halves the
// tensor work and the O accumulator against padding 8 rows up to M = 16.
// WM, what a work page is (the plan counts work pages of P.bs tokens):
//  WP_WHOLE   one block;
//  WP_PART    one of P.wpb equal parts of a block (blocks too large for the ring);
//  WP_MERGED  MERGE_BLOCKS consecutive blocks of the request, for small blocks
//             whose row fits one swizzle line: each block's tile is its own copy,
//             landing below the previous one as further rows of the same tile,
//             and the per-page work (wait, copy issue, cursors) is paid once for
//             all of them.  Blocks past the request's length are not copied; their
//             rows are masked like any padding slot.
template <int KVT, int D, bool TOKM, int WM>
__global__ void __launch_bounds__(ATTN_THREADS, min_blocks(Geo<KVT, D>::BITS, D, TOKM, pair_mode(D, TOKM, Geo<KVT, D>::NSEG)))
    pa_attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, AttnParams P) {
    using G = Geo<KVT, D>;
    constexpr bool BF = G::BF;
    constexpr bool QREG = q_in_regs<D>();
    constexpr bool PAIR = pair_mode(D, TOKM, G::NSEG);
    constexpr int WPW = PAIR ? 2 : 1;               // warps per worker
    constexpr int NSEGW = G::NSEG / WPW;            // channel segments of this warp
    constexpr int KSW = G::KSTEPS / WPW;            // k-steps of S = q K^T of this warp
    constexpr int NO = TOKM ? D / 16 : G::NT2 / WPW;  // accumulator tiles of O (O^T with TOKM)
    constexpr int HEPL = G::EPL / 2;            // TOKM: O^T tiles per V segment
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int NS = P.slots;
    const int bs = P.bs;
    const int tile_bytes = bs * G::RB;
    const int page_bytes = 2 * tile_bytes;  // K tile then V tile
    // Workers come in groups of RBLK, one per row block of a kv head: the
    // cursors run over (request, kv head, page) and every worker of a group
    // takes its own row block of every page of the group's share, so the
    // group reads each page at about the same time (all but the first copy
    // of a page hit L2) instead of every row block streaming the KV again.
    const int GS = P.RBLK;
    // pages read by one worker only stream through L2 (evict first); a group
    // of row-block workers rereads each page from L2
    const uint64_t pol = GS > 1 ? l2_evict_normal_policy() : l2_evict_first_policy();

    // this worker's shared memory: ring of NS pages, q' fragments (each warp of
    // a pair its half), the pair's score exchange and slot flags, barriers
    const int wk = warp / WPW;                 // worker within the CTA
    const int hf = PAIR ? (warp & 1) : 0;      // half of the channel segments (paired warps)
    const int sg0 = hf * NSEGW;                // first channel segment of this warp
    uint8_t *ring = smem + (size_t)wk * P.warp_smem;
    uint8_t *qbase = ring + (size_t)NS * page_bytes;
    uint4 *qs = reinterpret_cast<uint4 *>(qbase) + (size_t)hf * KSW * 32;             // [KSW][32]
    float *xchg = reinterpret_cast<float *>(qbase + (QREG ? 0 : G::KSTEPS * 512));   // [2][2][8][32]
    volatile int *sflags = reinterpret_cast<volatile int *>(reinterpret_cast<uint8_t *>(xchg) + XCHG_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(xchg) +
                                                  (PAIR ? XCHG_BYTES + MAX_SLOTS * 4 + 16 : 0));  // [MAX_SLOTS]
    if (NS < 1 || NS > MAX_SLOTS) return;  // the host never launches this
    auto pair_sync = [&]() {
        if constexpr (PAIR) named_barrier(1 + wk, 64);
    };

    // the plan (and anything else earlier on the stream) must be complete
    grid_dependency_wait();
    // the warp's share of the global page sequence
    const long long total = P.hdr[HDR_TOTAL_PAGES];
    if (total > (long long)P.B * P.mbps) {  // not a plan of this problem
        if (threadIdx.x == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    const long long Ntot = total * P.Hkv;
    const long long NWt = (long long)gridDim.x * (NWK / WPW);
    const long long kw = (long long)blockIdx.x * (NWK / WPW) + wk;  // worker
    const long long NG = NWt / GS;                                   // worker groups
    const long long kg = kw / GS;                                    // this worker's group
    const int gi = (int)(kw - kg * GS);                              // and its row block
    if (kg >= NG) return;  // the host sizes the launch in whole groups
    const long long x0 = kg * Ntot / NG, x1 = (kg + 1) * Ntot / NG;
    if (x0 >= x1) return;
    const int npg = (int)(x1 - x0);

    if (lane == 0 && hf == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
        tma_prefetch_desc(&tmk);
        tma_prefetch_desc(&tmv);
    }
    __syncwarp();
    pair_sync();  // the barriers are initialised before the partner waits on them

    uint32_t err = 0;
    Cursor cc = cursor_at(x0, P.req, P.B, P.Hkv, P.mbps);  // compute cursor (q = kv head)
    if (cc.b >= P.B) {
        if (lane == 0) atomic_or_err(P.hdr, PA_DEV_ERR_STALE_PLAN);
        return;
    }
    Cursor ci = cc;                             // issue cursor (runs NS pages ahead)
    int idc_b = -1, idc_w0 = 0, idc = 0;        // block ids of ci.b, pages [idc_w0, idc_w0 + 32)
    int idc_nb = 0;                             // merged work pages: blocks of request ci.b
    unsigned slot_bad = 0;                      // slots whose page had an invalid id

    int islot = 0;  // ring slot of the next copy
#ifdef PA_FAULT_INJECT
    const unsigned fi_withhold = P.hdr[HDR_WITHHOLD];
    long long fi_pos = x0;  // position of the next page issued
#endif
    auto issue = [&]() {
        const int slot = islot;
        islot = (islot + 1 == NS) ? 0 : islot + 1;
#ifdef PA_FAULT_INJECT
        if (fi_withhold != 0 && fi_pos++ + 1 == (long long)fi_withhold && ci.b < P.B) {
            if constexpr (WM == WP_MERGED) cursor_next<true>(ci, P.req, P.B, P.Hkv, P.mbps);
            else cursor_next(ci, P.req, P.B, P.Hkv, P.mbps);
            return;  // no copy and no arrive: the waits on this slot run out
        }
#endif
        if (ci.b >= P.B) {  // inconsistent records: no copy, the slot still completes
            if constexpr (PAIR) {
                if (lane == 0) sflags[slot] = 1;
            }
            if (lane == 0) mbar_arrive(&full[slot]);
            slot_bad |= 1u << slot;
            return;
        }
        if constexpr (WM == WP_MERGED) {
            // work page ci.p: blocks [bi0, bi0 + nbp) of the request, all rows
            const int bi0 = ci.p * MERGE_BLOCKS;
            if (ci.b != idc_b || bi0 < idc_w0 || bi0 + MERGE_BLOCKS > idc_w0 + 32) {
                idc_b = ci.b;
                idc_w0 = bi0;
                idc_nb = min((ci.L - 1) / P.bsb + 1, P.tbl_stride);  // blocks of the request (L >= 1)
                const int pg = idc_w0 + lane;
                idc = (pg < idc_nb) ? P.block_table[(size_t)ci.b * P.tbl_stride + pg] : 0;
            }
            const int nbp = min(MERGE_BLOCKS, idc_nb - bi0);
            int blk[MERGE_BLOCKS];
            bool ok = nbp >= 1;
#pragma unroll
            for (int i = 0; i < MERGE_BLOCKS; ++i) {
                blk[i] = __shfl_sync(0xffffffffu, idc, bi0 - idc_w0 + i);
                if (i < nbp) ok = ok && blk[i] >= 1 && blk[i] < P.num_blocks;
            }
            const int kvh = ci.q;
            if constexpr (PAIR) {
                if (lane == 0) sflags[slot] = ok ? 0 : 1;
            }
            if (lane == 0) {
                uint8_t *kt = ring + (size_t)slot * page_bytes;
                uint8_t *vt = kt + tile_bytes;
                const int sub = P.bsb * G::RB;  // bytes of one block's tile
                if (ok) {
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * nbp * sub));
#pragma unroll
                    for (int i = 0; i < MERGE_BLOCKS; ++i) {
                        if (i < nbp) {
                            tma_load_5d_hint(kt + i * sub, &tmk, &full[slot], 0, 0, 0, kvh, blk[i], pol);
                            tma_load_5d_hint(vt + i * sub, &tmv, &full[slot], 0, 0, 0, kvh, blk[i], pol);
                        }
                    }
                } else {
                    mbar_arrive(&full[slot]);
                }
            }
            slot_bad = ok ? (slot_bad & ~(1u << slot)) : (slot_bad | (1u << slot));
            cursor_next<true>(ci, P.req, P.B, P.Hkv, P.mbps);
            return;
        }
        // work page ci.p: rows [y0, y0 + bs) of block bi of the request
        int bi = ci.p, y0 = 0, nblk = ci.Pb;
        if constexpr (WM == WP_PART) {
            bi = ci.p / P.wpb;
            y0 = (ci.p - bi * P.wpb) * bs;
            nblk = (ci.Pb + P.wpb - 1) / P.wpb;
        }
        if (ci.b != idc_b || bi < idc_w0 || bi >= idc_w0 + 32) {
            idc_b = ci.b;
            idc_w0 = bi;
            const int pg = idc_w0 + lane;
            idc = (pg < nblk) ? P.block_table[(size_t)ci.b * P.tbl_stride + pg] : 0;
        }
        const int blk = __shfl_sync(0xffffffffu, idc, bi - idc_w0);
        const bool ok = blk >= 1 && blk < P.num_blocks;
        const int kvh = ci.q;
        if constexpr (PAIR) {
            if (lane == 0) sflags[slot] = ok ? 0 : 1;  // published with the barrier's phase
        }
        if (lane == 0) {
            uint8_t *kt = ring + (size_t)slot * page_bytes;
            uint8_t *vt = kt + tile_bytes;
            if (ok) {
                mbar_arrive_expect_tx(&full[slot], (uint32_t)page_bytes);
                tma_load_5d_hint(kt, &tmk, &full[slot], 0, y0, 0, kvh, blk, pol);  // all segments of the K tile
                tma_load_5d_hint(vt, &tmv, &full[slot], 0, y0, 0, kvh, blk, pol);
            } else {
                mbar_arrive(&full[slot]);  // no copy: the piece is NaN-filled
            }
        }
        slot_bad = ok ? (slot_bad & ~(1u << slot)) : (slot_bad | (1u << slot));
        cursor_next(ci, P.req, P.B, P.Hkv, P.mbps);
    };

    const int npre = min(NS, npg);
    if (hf == 0)
        for (int j = 0; j < npre; ++j) issue();

    // ---- per-piece state (a piece = this warp's run of pages of one segment)
    // o: rows g / g+8 x channels (rows-as-M), or channels x rows 2c / 2c+1 (TOKM);
    // m0/l0 and m1/l1 are the running max / sum of the lane's two rows
    float o[NO][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    uint32_t qreg[QREG ? G::KSTEPS : 1][4];
    float sc0 = 0.f, sc1 = 0.f;
    int vis0 = 0, vis1 = 0, L = 0, kvh = 0, rblk = 0, piece_b = -1, piece_q = -1, piece_p0 = 0, last_p = 0;
    bool pbad = false;

    auto start_piece = [&]() {
        piece_b = cc.b;
        piece_q = cc.q;
        piece_p0 = cc.p;
        kvh = cc.q;
        rblk = gi;
        const int4 Rq = P.req[cc.b];
        L = P.context_lens[cc.b];
        pbad = false;
        if (Rq.w != 0) { pbad = true; err |= PA_DEV_ERR_CONTEXT_LEN; }
        if (L != Rq.x) { pbad = true; err |= PA_DEV_ERR_STALE_PLAN; }
        const int r0 = rblk * ROWS;
        const int rg0 = r0 + g, rg1 = r0 + g + 8;
        vis0 = (rg0 < P.R && P.causal) ? L - (P.n - 1 - rg0 / P.G) : L;
        vis1 = (rg1 < P.R && P.causal) ? L - (P.n - 1 - rg1 / P.G) : L;
        const float kmax = (P.k_mode == PA_SCALE_CHANNEL) ? __uint_as_float(P.hdr[HDR_KMAX]) : 1.0f;
        const float kscal = (P.k_mode == PA_SCALE_TENSOR) ? P.k_scale[0] : kmax;
        auto fold = [&](int d) -> float {
            return (P.k_mode == PA_SCALE_CHANNEL) ? P.k_scale[(size_t)kvh * D + d] / kmax : 1.0f;
        };
        // rows g and g+8 of this segment: query position jq, query head h
        const bool ok0 = rg0 < P.R, ok1 = rg1 < P.R;
        const int jq0 = ok0 ? rg0 / P.G : 0, h0 = kvh * P.G + (ok0 ? rg0 % P.G : 0);
        const int jq1 = ok1 ? rg1 / P.G : 0, h1 = kvh * P.G + (ok1 ? rg1 % P.G : 0);
        // power-of-two row factors so that f16 operands of any bf16 query fit
        float rho0 = 1.f, rho1 = 1.f;
        if constexpr (!BF) {
            float mx0 = 0.f, mx1 = 0.f;
#pragma unroll 4
            for (int K = 0; K < G::KSTEPS; ++K) {
                float v0[4] = {0.f, 0.f, 0.f, 0.f}, v1[4] = {0.f, 0.f, 0.f, 0.f};
                if (ok0) load_q4<KVT, D>(P, cc.b, jq0, h0, K, c, v0);
                if (ok1) load_q4<KVT, D>(P, cc.b, jq1, h1, K, c, v1);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float f = fold(phys_ch<KVT, D>(K, c, e));
                    mx0 = fmaxf(mx0, fabsf(v0[e] * f));
                    mx1 = fmaxf(mx1, fabsf(v1[e] * f));
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            int e;
            if (mx0 > 0.f && mx0 < 3.0e38f) { frexpf(mx0, &e); rho0 = ldexpf(1.0f, e); }
            if (mx1 > 0.f && mx1 < 3.0e38f) { frexpf(mx1, &e); rho1 = ldexpf(1.0f, e); }
        }
        sc0 = P.softmax_scale * kscal * rho0 * LOG2E;
        sc1 = P.softmax_scale * kscal * rho1 * LOG2E;
        if constexpr (TOKM) {
            // this lane's score rows are 2c and 2c+1; their q rows were folded
            // by the lanes with g = 2c and g = 2c+1
            const float sA = __shfl_sync(0xffffffffu, sc0, 8 * c), sB = __shfl_sync(0xffffffffu, sc0, 8 * c + 4);
            const int ra = r0 + 2 * c, rb = ra + 1;
            vis0 = (ra < P.R && P.causal) ? L - (P.n - 1 - ra / P.G) : L;
            vis1 = (rb < P.R && P.causal) ? L - (P.n - 1 - rb / P.G) : L;
            sc0 = sA;
            sc1 = sB;
        }
        const float inv0 = 1.0f / rho0, inv1 = 1.0f / rho1;
#pragma unroll
        for (int K = 0; K < KSW; ++K) {
            const int Kg = hf * KSW + K;  // k-step of the whole row (paired warps: this half)
            uint32_t a[4];
            float v0[4] = {0.f, 0.f, 0.f, 0.f}, v1[4] = {0.f, 0.f, 0.f, 0.f};
            if (ok0) load_q4<KVT, D>(P, cc.b, jq0, h0, Kg, c, v0);
            if (ok1) load_q4<KVT, D>(P, cc.b, jq1, h1, Kg, c, v1);
#pragma unroll
            for (int half = 0; half < 2; ++half) {  // a0a1/a2a3 use e=0,1; a4a5/a6a7 use e=2,3
                const float f0 = fold(phys_ch<KVT, D>(Kg, c, 2 * half)), f1 = fold(phys_ch<KVT, D>(Kg, c, 2 * half + 1));
                const float u0 = v0[2 * half] * f0 * inv0, u1 = v0[2 * half + 1] * f1 * inv0;
                const float w0 = v1[2 * half] * f0 * inv1, w1 = v1[2 * half + 1] * f1 * inv1;
                a[2 * half] = pack2<BF>(u0, u1);
                a[2 * half + 1] = pack2<BF>(w0, w1);
            }
            if constexpr (QREG) {
                qreg[K][0] = a[0]; qreg[K][1] = a[1]; qreg[K][2] = a[2]; qreg[K][3] = a[3];
            } else {
                qs[K * 32 + lane] = make_uint4(a[0], a[1], a[2], a[3]);
            }
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < NO; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    };

    auto finish_piece = [&]() {
        float la = l0, lb = l1;
        if constexpr (TOKM) {  // the lane's rows were summed over its tokens g, g+8
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                la += __shfl_xor_sync(0xffffffffu, la, off);
                lb += __shfl_xor_sync(0xffffffffu, lb, off);
            }
        } else {
            la += __shfl_xor_sync(0xffffffffu, la, 1);
            la += __shfl_xor_sync(0xffffffffu, la, 2);
            lb += __shfl_xor_sync(0xffffffffu, lb, 1);
            lb += __shfl_xor_sync(0xffffffffu, lb, 2);
        }
        const int Pb = planned_pages(P.req, piece_b, P.mbps);
        const bool complete = (piece_p0 == 0 && last_p == Pb - 1);
        const long long slot_id = ((long long)piece_b * P.Hkv + piece_q + kg) * GS + gi;  // partial slot of this piece
        const int r0 = rblk * ROWS;
        const float NaN = __int_as_float(0x7fc00000);
        // store value `val` of (row index within the segment, channel d)
        auto put = [&](int row, int d, float val) {
            const int r = r0 + row;
            if (pbad) val = NaN;
            if (complete) {
                float vsc = 1.0f;
                if (P.v_mode == PA_SCALE_TENSOR) vsc = P.v_scale[0];
                else if (P.v_mode == PA_SCALE_CHANNEL) vsc = P.v_scale[(size_t)kvh * D + d];
                const float y = val * vsc;
                const int jq = r / P.G, h = kvh * P.G + (r % P.G);
                const size_t oi = (((size_t)piece_b * P.n + jq) * P.Hq + h) * D + d;
                if (P.out_dtype == PA_F32) reinterpret_cast<float *>(P.out)[oi] = y;
                else if (P.out_dtype == PA_F16) reinterpret_cast<__half *>(P.out)[oi] = __float2half_rn(y);
                else reinterpret_cast<__nv_bfloat16 *>(P.out)[oi] = __float2bfloat16_rn(y);
            } else {
                P.part_o[((size_t)slot_id * ROWS + row) * D + d] = val;
            }
        };
        auto put_lse = [&](int row, float l, float m) {
            const int r = r0 + row;
            float lse_v = l > 0.f ? (m + lg2(l)) * LN2 : -INFINITY;
            if (pbad) lse_v = NaN;
            if (complete) {
                const int jq = r / P.G, h = kvh * P.G + (r % P.G);
                if (P.lse != nullptr) P.lse[((size_t)piece_b * P.n + jq) * P.Hq + h] = lse_v;
            } else {
                P.part_lse[(size_t)slot_id * ROWS + row] = lse_v;
            }
        };
        if constexpr (TOKM) {
            const int ra = 2 * c, rb = 2 * c + 1;
            const float ia = la > 0.f ? 1.0f / la : 0.f, ib = lb > 0.f ? 1.0f / lb : 0.f;
#pragma unroll
            for (int t = 0; t < NO; ++t) {
                const int sg = t / HEPL, mm = t % HEPL;
                const int dlo = sg * G::EPS + g * G::EPL + 2 * mm;
                if (r0 + ra < P.R) {
                    put(ra, dlo, o[t][0] * ia);
                    put(ra, dlo + 1, o[t][2] * ia);
                }
                if (r0 + rb < P.R) {
                    put(rb, dlo, o[t][1] * ib);
                    put(rb, dlo + 1, o[t][3] * ib);
                }
            }
            if (g == 0) {
                if (r0 + ra < P.R) put_lse(ra, la, m0);
                if (r0 + rb < P.R) put_lse(rb, lb, m1);
            }
        } else {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int row = g + 8 * rr;
                if (r0 + row >= P.R) continue;
                const float l = rr ? lb : la;
                const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
                for (int t = 0; t < NO; ++t) {
                    const int sg = sg0 + t / G::EPL, e = t % G::EPL;
#pragma unroll
                    for (int cc2 = 0; cc2 < 2; ++cc2)
                        put(row, sg * G::EPS + (2 * c + cc2) * G::EPL + e, o[t][2 * rr + cc2] * inv);
                }
                if (c == 0 && hf == 0) put_lse(row, l, rr ? m1 : m0);
            }
        }
    };

    int xb = 0;  // paired warps: exchange buffer parity
    int cslot = 0;       // ring slot of page j
    uint32_t cpar = 0;   // its barrier phase parity
    int j = 0;
    for (; j < npg; ++j) {
        if (cc.b >= P.B) {  // records shorter than the shares: stop, copies drained below
            err |= PA_DEV_ERR_STALE_PLAN;
            break;
        }
        if (cc.b != piece_b || cc.q != piece_q) {
            if (piece_b >= 0) finish_piece();
            start_piece();
        }
        const int slot = cslot;
        const uint32_t par = cpar;
        if (++cslot == NS) { cslot = 0; cpar ^= 1u; }
        bool ok_wait = mbar_wait_bounded(&full[slot], par, nullptr);
        if constexpr (PAIR) {
            // both warps of the pair leave together: each publishes its outcome
            const int okw = __all_sync(0xffffffffu, ok_wait) ? 1 : 0;
            if (lane == 0) sflags[MAX_SLOTS + hf] = okw;
            pair_sync();
            ok_wait = sflags[MAX_SLOTS] && sflags[MAX_SLOTS + 1];
            pair_sync();  // both have read the votes before the next page's
            if (ok_wait) (void)mbar_try_wait(&full[slot], par);
        }
        if (!ok_wait) {
            err |= PA_DEV_ERR_TIMEOUT;
            pbad = true;
            break;
        }
        const bool bad_slot = PAIR ? (sflags[slot] != 0) : (((slot_bad >> slot) & 1u) != 0);
        if (bad_slot) {
            err |= PA_DEV_ERR_BLOCK_ID;
            pbad = true;
        }
        if (!pbad) {
            const uint8_t *kt = ring + (size_t)slot * page_bytes;
            const uint8_t *vt = kt + tile_bytes;
            const int t_page = cc.p * bs;
            const int nvalid = min(bs, L - t_page);  // real tokens in this page
            const int vis_min = min(vis0, vis1);
            for (int ch = 0; ch < bs; ch += 16) {
              if constexpr (TOKM) {
                // ---- S^T = K q'^T for tokens ch .. ch+15 (M) x query rows (N = 8);
                // two partial accumulators halve the dependent MMA chain
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int sg = 0; sg < G::NSEG; ++sg) {
                    uint32_t kw2[2][G::KWORDS];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int srow = ch + 8 * t + g;
                        if constexpr (G::SW == 128) {
                            lds_words<4>(kw2[t], kt + tile_off<128>(srow, sg, 2 * c, bs));
                            lds_words<4>(kw2[t] + 4, kt + tile_off<128>(srow, sg, 2 * c + 1, bs));
                        } else {
                            lds_words<4>(kw2[t], kt + tile_off<64>(srow, sg, c, bs));
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < G::KPS; ++jj) {
                        const int K = sg * G::KPS + jj;
                        uint32_t q0, q1;
                        if constexpr (QREG) {
                            q0 = qreg[K][0];
                            q1 = qreg[K][2];
                        } else {
                            const uint4 av = qs[K * 32 + lane];
                            q0 = av.x;
                            q1 = av.z;
                        }
                        uint32_t a[4];
                        k_frag<KVT>(kw2[0], jj, a[0], a[2]);  // token row g
                        k_frag<KVT>(kw2[1], jj, a[1], a[3]);  // token row g+8
                        if (K & 1) mma16816<BF>(sb, a, q0, q1);
                        else mma16816<BF>(sa, a, q0, q1);
                    }
                }
                // ---- scale, mask, online softmax (rows 2c, 2c+1; tokens g, g+8)
                float x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) x[e] = (sa[e] + sb[e]) * ((e & 1) ? sc1 : sc0);
                if (t_page + ch + 16 > vis_min) {
                    const int tg = t_page + ch + g;
                    x[0] = (tg < vis0) ? x[0] : -INFINITY;
                    x[1] = (tg < vis1) ? x[1] : -INFINITY;
                    x[2] = (tg + 8 < vis0) ? x[2] : -INFINITY;
                    x[3] = (tg + 8 < vis1) ? x[3] : -INFINITY;
                }
                float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
                if (__any_sync(0xffffffffu, mx0 > m0 + LAZY_SLACK || mx1 > m1 + LAZY_SLACK)) {
#pragma unroll
                    for (int off = 4; off <= 16; off <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
                    }
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float al0 = ex2(m0 - ((mn0 == -INFINITY) ? 0.f : mn0));
                    const float al1 = ex2(m1 - ((mn1 == -INFINITY) ? 0.f : mn1));
                    m0 = mn0;
                    m1 = mn1;
                    l0 *= al0;
                    l1 *= al1;
#pragma unroll
                    for (int t = 0; t < NO; ++t) {
                        o[t][0] *= al0;
                        o[t][1] *= al1;
                        o[t][2] *= al0;
                        o[t][3] *= al1;
                    }
                }
                const float base0 = (m0 == -INFINITY) ? 0.f : m0;
                const float base1 = (m1 == -INFINITY) ? 0.f : m1;
                x[0] = ex2(x[0] - base0);
                x[2] = ex2(x[2] - base0);
                x[1] = ex2(x[1] - base1);
                x[3] = ex2(x[3] - base1);
                l0 += x[0] + x[2];
                l1 += x[1] + x[3];
                // ---- P^T fragments: transpose the [token][row] pairs
                const uint32_t pb0 = movmatrix_trans(pack2<BF>(x[0], x[1]));  // tokens 2c,2c+1 of row g
                const uint32_t pb1 = movmatrix_trans(pack2<BF>(x[2], x[3]));  // tokens 2c+8,2c+9
                // ---- O^T += V^T P^T
                const int rA = ch + 2 * c, rB = rA + 1, rC = rA + 8, rD = rA + 9;
                const bool tail = ch + 16 > nvalid;
                const bool zA = tail && rA >= nvalid, zB = tail && rB >= nvalid;
                const bool zC = tail && rC >= nvalid, zD = tail && rD >= nvalid;
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
                    if (tail) {
#pragma unroll
                        for (int k = 0; k < G::VWORDS; ++k) {
                            va[k] = zA ? 0u : va[k];
                            vb[k] = zB ? 0u : vb[k];
                            vc[k] = zC ? 0u : vc[k];
                            vd[k] = zD ? 0u : vd[k];
                        }
                    }
                    uint32_t bf[G::EPL][2];
                    v_frags<KVT, G::EPL, G::VWORDS>(va, vb, vc, vd, bf);
#pragma unroll
                    for (int mm = 0; mm < HEPL; ++mm) {
                        const uint32_t a[4] = {bf[2 * mm][0], bf[2 * mm + 1][0], bf[2 * mm][1], bf[2 * mm + 1][1]};
                        mma16816<BF>(o[sg * HEPL + mm], a, pb0, pb1);
                    }
                }
              } else {
                // ---- S = q' K^T for tokens ch .. ch+15 (two n-tiles); paired
                // warps each take their half of the channel segments
                float s[2][4];
#pragma unroll
                for (int t = 0; t < 2; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
                for (int sgl = 0; sgl < NSEGW; ++sgl) {
                    const int sg = sg0 + sgl;
                    uint32_t kw2[2][G::KWORDS];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const int srow = ch + 8 * t + g;
                        if constexpr (G::SW == 128) {
                            lds_words<4>(kw2[t], kt + tile_off<128>(srow, sg, 2 * c, bs));
                            lds_words<4>(kw2[t] + 4, kt + tile_off<128>(srow, sg, 2 * c + 1, bs));
                        } else {
                            lds_words<4>(kw2[t], kt + tile_off<64>(srow, sg, c, bs));
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < G::KPS; ++jj) {
                        uint32_t a[4];
                        if constexpr (QREG) {
                            a[0] = qreg[sg * G::KPS + jj][0]; a[1] = qreg[sg * G::KPS + jj][1];
                            a[2] = qreg[sg * G::KPS + jj][2]; a[3] = qreg[sg * G::KPS + jj][3];
                        } else {
                            const uint4 av = qs[(sgl * G::KPS + jj) * 32 + lane];
                            a[0] = av.x; a[1] = av.y; a[2] = av.z; a[3] = av.w;
                        }
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            uint32_t b0, b1;
                            k_frag<KVT>(kw2[t], jj, b0, b1);
                            mma16816<BF>(s[t], a, b0, b1);
                        }
                    }
                }
                if constexpr (PAIR) {
                    // the partner's partial scores; both warps add them in the same order
                    // [buffer][warp][value][lane]: consecutive lanes, consecutive banks
                    float *mine = xchg + ((xb & 1) * 2 + hf) * 256 + lane;
                    const float *theirs = xchg + ((xb & 1) * 2 + (hf ^ 1)) * 256 + lane;
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int e = 0; e < 4; ++e) mine[(4 * t + e) * 32] = s[t][e];
                    pair_sync();
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float o2 = theirs[(4 * t + e) * 32];
                            s[t][e] = hf == 0 ? s[t][e] + o2 : o2 + s[t][e];
                        }
                    ++xb;
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
                        float x0v = s[t][e] * sc0, x1v = s[t][2 + e] * sc1;
                        if (need_mask) {
                            x0v = (tok < vis0) ? x0v : -INFINITY;
                            x1v = (tok < vis1) ? x1v : -INFINITY;
                        }
                        s[t][e] = x0v;
                        s[t][2 + e] = x1v;
                        mx0 = fmaxf(mx0, x0v);
                        mx1 = fmaxf(mx1, x1v);
                    }
                }
                if (__any_sync(0xffffffffu, mx0 > m0 + LAZY_SLACK || mx1 > m1 + LAZY_SLACK)) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float al0 = ex2(m0 - ((mn0 == -INFINITY) ? 0.f : mn0));  // m = -inf -> 0
                    const float al1 = ex2(m1 - ((mn1 == -INFINITY) ? 0.f : mn1));
                    m0 = mn0;
                    m1 = mn1;
                    l0 *= al0;
                    l1 *= al1;
#pragma unroll
                    for (int t = 0; t < NO; ++t) {
                        o[t][0] *= al0;
                        o[t][1] *= al0;
                        o[t][2] *= al1;
                        o[t][3] *= al1;
                    }
                }
                const float base0 = (m0 == -INFINITY) ? 0.f : m0;
                const float base1 = (m1 == -INFINITY) ? 0.f : m1;
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
                l0 += ps0;
                l1 += ps1;
                // ---- O += P V
                uint32_t pa[4];
                pa[0] = pack2<BF>(s[0][0], s[0][1]);
                pa[1] = pack2<BF>(s[0][2], s[0][3]);
                pa[2] = pack2<BF>(s[1][0], s[1][1]);
                pa[3] = pack2<BF>(s[1][2], s[1][3]);
                const int rA = ch + 2 * c, rB = rA + 1, rC = rA + 8, rD = rA + 9;
                const bool tail = ch + 16 > nvalid;  // padding slots in this chunk: codes -> 0
                const bool zA = tail && rA >= nvalid, zB = tail && rB >= nvalid;
                const bool zC = tail && rC >= nvalid, zD = tail && rD >= nvalid;
#pragma unroll
                for (int sgl = 0; sgl < NSEGW; ++sgl) {
                    const int sg = sg0 + sgl;
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
                    if (tail) {
#pragma unroll
                        for (int k = 0; k < G::VWORDS; ++k) {
                            va[k] = zA ? 0u : va[k];
                            vb[k] = zB ? 0u : vb[k];
                            vc[k] = zC ? 0u : vc[k];
                            vd[k] = zD ? 0u : vd[k];
                        }
                    }
                    uint32_t bf[G::EPL][2];
                    v_frags<KVT, G::EPL, G::VWORDS>(va, vb, vc, vd, bf);
#pragma unroll
                    for (int e = 0; e < G::EPL; ++e) mma16816<BF>(o[sgl * G::EPL + e], pa, bf[e][0], bf[e][1]);
                }
              }
            }
        }
        last_p = cc.p;
        // every lane (of both warps of a pair) is done reading the slot before
        // a copy may overwrite it
        __syncwarp();
        pair_sync();
        fence_proxy_async_smem();
        if (j + NS < npg && hf == 0) issue();
        cursor_next(cc, P.req, P.B, P.Hkv, P.mbps);
    }
    if (j < npg && hf == 0) {
        // a wait ran out: let every copy still in flight land before exiting
        for (int i = j; i < min(npg, j + NS); ++i) mbar_wait_bounded(&full[i % NS], (i / NS) & 1, nullptr);
    }
    if (j < npg) {
        // every piece this worker still owned -- the one in progress and any
        // later one of its share -- is written as NaN (outputs, or partials the
        // combine turns into NaN rows), so no row keeps stale values
        pbad = true;
        for (; j < npg && cc.b < P.B; ++j) {
            if (cc.b != piece_b || cc.q != piece_q) {
                if (piece_b >= 0) finish_piece();
                piece_b = cc.b;
                piece_q = cc.q;
                piece_p0 = cc.p;
                kvh = cc.q;
                rblk = gi;
            }
            last_p = cc.p;
            cursor_next(cc, P.req, P.B, P.Hkv, P.mbps);
        }
    }
    // the combine may start launching while the last pieces are written
    grid_dependents_launch();
    if (piece_b >= 0) finish_piece();
    if (lane == 0) atomic_or_err(P.hdr, err);
}

}  // namespace pa
