// Host side of the C ABI declared in include/pa.h: argument validation,
// workspace layout, tensor-map encoding and kernel dispatch.  No allocation,
// no synchronisation (except pa_get_error), no global state beyond cached
// driver entry points and per-device SM counts.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pa_attn_launch.cuh"

namespace pa {
cudaError_t launch_plan(const PlanParams &P, const float *k_scale, int k_count, cudaStream_t s);
cudaError_t launch_combine(const CombineParams &P, cudaStream_t s);
cudaError_t launch_latent(const CUtensorMap &ta, const CUtensorMap &tb, const LatentParams &P, int ctas,
                          cudaStream_t s);
cudaError_t launch_e4m3_tc(const CUtensorMap &tk, const CUtensorMap &tv, const E4TcParams &P, int ctas,
                           cudaStream_t s);
}  // namespace pa

namespace {

constexpr int VERSION = 100;
#ifndef PA_MIN_RING_PAGES
#define PA_MIN_RING_PAGES 2  // pages per worker before the resident CTAs per SM are stepped down
#endif
#ifndef PA_MIN_RING_PAGES_PAIR
#define PA_MIN_RING_PAGES_PAIR 1  // paired warps: more resident workers beat a deeper ring
#endif
#ifndef PA_TOKM_MAX_ROWS
#define PA_TOKM_MAX_ROWS 8  // at most 8: the rows are the MMA N axis then
#endif
constexpr size_t SM_SMEM_BYTES = 228 * 1024;     // shared memory per SM
constexpr size_t CTA_RESERVED_BYTES = 1024;       // reserved by the runtime per resident CTA
constexpr size_t MAX_DYN_SMEM_BYTES = 227 * 1024; // opt-in limit per CTA
// the single-latent kernel's fixed shape (one CTA of 64 query rows per SM)
constexpr int LAT_DK = 576, LAT_DV = 512, LAT_BS = 64, LAT_ROWS = 64, LAT_RING = 2;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int dtype_bits(int dt) {
    switch (dt) {
        case PA_F16: case PA_BF16: return 16;
        case PA_E4M3: case PA_INT8: return 8;
        case PA_INT4: return 4;
        default: return 0;
    }
}

std::atomic<int> g_sms[64];

pa_status device_sms(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev >= 0 && dev < 64) {
        const int c = g_sms[dev].load(std::memory_order_relaxed);
        if (c > 0) { *sms = c; return PA_OK; }
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return PA_ERR_CUDA;
    if (dev >= 0 && dev < 64) g_sms[dev].store(v, std::memory_order_relaxed);
    *sms = v;
    return PA_OK;
}

// Everything derived from a problem on the host.
struct Derived {
    int G, R, row_blocks, sms, ctas, minb;
    bool tokm, latent;
    bool e4tc;     // the E4M3 tensor-core kernel (head dim 256, 16..64 rows per kv head)
    int rows_seg;  // query rows per segment
    int gs;        // workers per group (they share one run of pages, one row block each)
    long long nwarps, slots_partial;
    int D, RB, SW, slots, warp_smem;
    int wp;        // work page: tokens the kernel handles as one page (a block, an equal part of one, or merged blocks)
    int wpb, mpb;  // parts per block (split blocks), blocks per work page (merged blocks); at least one is 1
    int box_rows;  // rows of one tile copy: the work page, or one block of a merged page
    size_t k_block, v_block, smem;
    pa_layout L;
};

pa_status derive_grouped(const pa_problem *p, Derived *d);
int work_pages_per_seq(const pa_problem *p, const Derived &d);

pa_status derive(const pa_problem *p, Derived *d) {
    if (p == nullptr || d == nullptr) return PA_ERR_INVALID_ARG;
    if (p->batch < 0 || p->next_n < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1 ||
        p->num_q_heads % p->num_kv_heads != 0 || p->head_dim_k < 1 || p->head_dim_v < 1 ||
        p->block_size < 1 || p->num_blocks < 1 || p->max_blocks_per_seq < 1 || p->max_context_len < 0 ||
        p->num_sms < 0 || p->grid_ctas < 0 || p->grid_ctas > (1 << 20))
        return PA_ERR_INVALID_ARG;
    if ((p->q_dtype != PA_F16 && p->q_dtype != PA_BF16) || dtype_bits(p->kv_dtype) == 0 ||
        (p->out_dtype != PA_F32 && p->out_dtype != PA_F16 && p->out_dtype != PA_BF16))
        return PA_ERR_INVALID_ARG;
    if (p->k_scale_mode < PA_SCALE_NONE || p->k_scale_mode > PA_SCALE_TOKEN || p->v_scale_mode < PA_SCALE_NONE ||
        p->v_scale_mode > PA_SCALE_TOKEN)
        return PA_ERR_INVALID_ARG;
    if (!std::isfinite(p->softmax_scale)) return PA_ERR_INVALID_ARG;
    if (p->causal != 0 && p->causal != 1) return PA_ERR_INVALID_ARG;
    if (p->v_is_k_prefix != 0 && p->v_is_k_prefix != 1) return PA_ERR_INVALID_ARG;
    if (p->kv_dtype == PA_INT4 && ((p->head_dim_k & 1) || (p->head_dim_v & 1))) return PA_ERR_INVALID_ARG;

    if (p->v_is_k_prefix && p->head_dim_v > p->head_dim_k) return PA_ERR_INVALID_ARG;
    d->G = p->num_q_heads / p->num_kv_heads;
    {
        const long long R = (long long)d->G * p->next_n;
        if (R > (1 << 20)) return PA_ERR_UNSUPPORTED;
        d->R = (int)R;
    }
    if (p->num_sms > 0) d->sms = p->num_sms;
    else {
        const pa_status st = device_sms(&d->sms);
        if (st != PA_OK) return st;
    }
    d->latent = p->v_is_k_prefix != 0;
    d->e4tc = !d->latent && p->kv_dtype == PA_E4M3 && p->head_dim_k == 256 && p->head_dim_v == 256 &&
              (p->k_scale_mode == PA_SCALE_NONE || p->k_scale_mode == PA_SCALE_TENSOR) &&
              (p->v_scale_mode == PA_SCALE_NONE || p->v_scale_mode == PA_SCALE_TENSOR) && d->R % 16 == 0 &&
              d->R >= 16 && d->R <= 64 &&
              (p->block_size == 16 || p->block_size == 32 || p->block_size == 64 || p->block_size == 128) &&
              p->num_kv_heads <= 65535;
    if (d->e4tc) {
        // tokens on the MMA M axis in 128-token chunks (the plan's pages), all R
        // rows of a kv head in one segment, one CTA per SM
        d->D = 256;
        d->rows_seg = d->R;
        d->row_blocks = 1;
        d->tokm = false;
        d->minb = 1;
        d->RB = 256;
        d->SW = 128;
        d->k_block = (size_t)p->num_kv_heads * p->block_size * 256;
        d->v_block = d->k_block;
        d->slots = d->R <= 48 ? 3 : 2;  // K stages of a chunk (V: 3 at 16 rows, else 2)
        d->wp = 128;
        d->wpb = 1;
        d->mpb = 128 / p->block_size;
        d->box_rows = p->block_size;
        d->warp_smem = 0;
        d->smem = 0;
        d->gs = 1;
        d->ctas = p->grid_ctas > 0 ? p->grid_ctas : d->sms;
        d->nwarps = d->ctas;
    } else if (d->latent) {
        // single-latent MQA: one E4M3 plane, V = its first 512 of 576
        // channels, a per-token fp32 scale after the codes of each block
        if (p->kv_dtype != PA_E4M3 || p->k_scale_mode != PA_SCALE_TOKEN || p->head_dim_k != LAT_DK ||
            p->head_dim_v != LAT_DV || p->block_size != LAT_BS || p->num_kv_heads > 65535)
            return PA_ERR_UNSUPPORTED;
        d->D = LAT_DK;
        d->rows_seg = LAT_ROWS;
        d->row_blocks = (d->R + LAT_ROWS - 1) / LAT_ROWS;
        if (d->row_blocks > 65535) return PA_ERR_UNSUPPORTED;
        d->tokm = false;
        d->minb = 1;
        d->RB = LAT_DK;
        d->SW = 128;
        d->k_block = (size_t)p->num_kv_heads * LAT_BS * (LAT_DK + 4);
        d->v_block = d->k_block;
        d->slots = LAT_RING;
        d->wp = LAT_BS;
        d->wpb = 1;
        d->mpb = 1;
        d->box_rows = LAT_BS;
        d->warp_smem = 0;
        d->smem = 0;
        // the workers are CTAs, in groups of one per row block
        d->gs = d->row_blocks;
        const int want = p->grid_ctas > 0 ? p->grid_ctas : d->sms;
        d->ctas = std::max(d->gs, want / d->gs * d->gs);
        d->nwarps = d->ctas;
    } else {
        const pa_status st = derive_grouped(p, d);
        if (st != PA_OK) return st;
    }

    // Every request has at most the table width of pages (longer ones are
    // flagged, not planned), and the plan keeps page prefix sums in 32 bits:
    // problems that could need more are refused here rather than flagged by
    // the planner on the device.
    if ((long long)p->batch * work_pages_per_seq(p, *d) > 0x7fffffffll) return PA_ERR_UNSUPPORTED;
    const long long X = (long long)p->num_kv_heads * d->row_blocks;
    d->slots_partial = ((long long)p->batch * (X / d->gs) + d->nwarps / d->gs) * d->gs;
    if (d->slots_partial > (1ll << 31)) return PA_ERR_UNSUPPORTED;

    pa_layout &Lo = d->L;
    std::memset(&Lo, 0, sizeof(Lo));
    size_t off = 0;
    Lo.header_offset = off;
    off = align_up(off + 64, 256);
    Lo.requests_offset = off;
    off = align_up(off + (size_t)p->batch * 16, 256);
    Lo.partial_o_offset = off;
    off = align_up(off + (size_t)d->slots_partial * d->rows_seg * p->head_dim_v * 4, 256);
    Lo.partial_lse_offset = off;
    off = align_up(off + (size_t)d->slots_partial * d->rows_seg * 4, 256);
    Lo.total_bytes = off;
    Lo.partial_slots = d->slots_partial;
    Lo.rows_per_kv_head = d->R;
    Lo.row_blocks = d->row_blocks;
    Lo.num_sms = d->sms;
    Lo.grid_ctas = d->ctas;
    Lo.warps = (int32_t)d->nwarps;
    Lo.ring_pages_per_warp = d->slots;
    Lo.rows_per_segment = d->rows_seg;
    Lo.group_size = d->gs;
    Lo.work_page_tokens = d->wp;
    return PA_OK;
}

// The grouped kernel (K and V planes of their own, per-tensor / per-channel
// scales): launch shape and shared-memory budget.
pa_status derive_grouped(const pa_problem *p, Derived *d) {
    if (p->k_scale_mode == PA_SCALE_TOKEN || p->v_scale_mode == PA_SCALE_TOKEN) return PA_ERR_UNSUPPORTED;
    if (p->head_dim_k != p->head_dim_v) return PA_ERR_UNSUPPORTED;
    const int D = p->head_dim_k;
    if (D != 64 && D != 128 && D != 256) return PA_ERR_UNSUPPORTED;
    if (p->kv_dtype == PA_INT4 && D == 64) return PA_ERR_UNSUPPORTED;
    if (p->block_size % 16 != 0 || p->block_size > 128) return PA_ERR_UNSUPPORTED;
    if (p->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;

    d->D = D;
    d->rows_seg = 16;
    d->row_blocks = (d->R + 15) / 16;
    if (d->row_blocks > 65535) return PA_ERR_UNSUPPORTED;
    const int bs = p->block_size;
    const int bits = dtype_bits(p->kv_dtype);
    d->RB = D * bits / 8;
    d->SW = d->RB >= 128 ? 128 : 64;
    d->k_block = (size_t)p->num_kv_heads * bs * d->RB;
    d->v_block = d->k_block;
    // Ring pages per worker (a warp, or a pair of warps sharing one ring for
    // D = 256 with rows on the MMA M axis): as many as fit the shared memory of
    // the resident CTAs per SM the kernel's registers allow; with pages too
    // large for two per worker, fewer CTAs per SM, and one page per worker as
    // the last resort.  A block too large for that is handled as 2, 3, ...
    // equal work pages of at least 16 tokens (logical order is unchanged: the
    // parts of a block are consecutive positions), whichever split keeps the
    // most CTAs per SM with the minimum ring, the larger page on a tie.
    d->tokm = d->R <= PA_TOKM_MAX_ROWS;  // few query rows per kv head: tokens on the MMA M axis
    const bool pair = pa::pair_mode(D, d->tokm, d->RB / d->SW);
    const int workers = pa::NWK / (pair ? 2 : 1);  // per CTA
    const int min_pages = pair ? PA_MIN_RING_PAGES_PAIR : PA_MIN_RING_PAGES;
    auto wsm = [&](int s, int wp) {
        const int page_bytes = 2 * wp * d->RB;
        return D <= 128 ? pa::warp_smem_bytes<128>(s, page_bytes, pair) : pa::warp_smem_bytes<256>(s, page_bytes, pair);
    };
    auto fit = [&](int minb, int wp) {
        const size_t budget = std::min(MAX_DYN_SMEM_BYTES, SM_SMEM_BYTES / minb - CTA_RESERVED_BYTES) - 1024;
        int slots = 0;
        for (int s = 1; s <= pa::MAX_SLOTS; ++s)
            if ((size_t)workers * wsm(s, wp) <= budget) slots = s;
        return slots;
    };
    bool found = false;
    int best_ok = 0;
    for (int wp = bs; wp >= 16; wp -= 16) {
        if (bs % wp != 0) continue;  // work pages: equal parts of a block, multiples of 16 tokens
        // fewer resident CTAs until every worker holds two pages (one in flight
        // while it computes on the other); one page per worker as the last resort
        int minb = pa::min_blocks(bits, D, d->tokm, pair);
        int slots = fit(minb, wp);
        while (slots < min_pages && minb > 1) {
            minb -= 1;
            slots = fit(minb, wp);
        }
        if (slots < 1) continue;
        const int ok = slots >= min_pages ? 1 : 0;
        if (!found || ok > best_ok || (ok == best_ok && minb > d->minb)) {
            found = true;
            best_ok = ok;
            d->minb = minb;
            d->slots = slots;
            d->wp = wp;
        }
    }
    if (!found) return PA_ERR_UNSUPPORTED;
    d->wpb = bs / d->wp;
    d->mpb = 1;
    d->box_rows = d->wp;
    // 16-token blocks of short rows (2 KB pages): MERGE_BLOCKS consecutive blocks
    // per work page, when the ring still holds two of them at the same residency
    if (d->wpb == 1 && bs == 16 && pa::merge_rows(d->RB)) {
        const int wp2 = pa::MERGE_BLOCKS * bs;
        const int s2 = fit(d->minb, wp2);
        if (s2 >= min_pages) {
            d->mpb = pa::MERGE_BLOCKS;
            d->wp = wp2;
            d->slots = s2;
        }
    }
    d->warp_smem = wsm(d->slots, d->wp);
    d->smem = 1024 + (size_t)workers * d->warp_smem;
    d->ctas = p->grid_ctas > 0 ? p->grid_ctas : d->sms * d->minb;
    // workers come in groups of row_blocks (one per block of 16 query rows of
    // a kv head, walking the same pages): the launch holds whole groups
    d->gs = d->row_blocks;
    {
        int g = d->gs, w = workers;
        while (w != 0) { const int t = g % w; g = w; w = t; }  // gcd(gs, workers)
        const int m = d->gs / g;                               // CTAs per whole number of groups
        d->ctas = std::max(m, d->ctas / m * m);
    }
    d->nwarps = (long long)d->ctas * workers;
    return PA_OK;
}

// work pages per request at most: the table width in work pages
int work_pages_per_seq(const pa_problem *p, const Derived &d) {
    return d.mpb > 1 ? (p->max_blocks_per_seq + d.mpb - 1) / d.mpb : p->max_blocks_per_seq * d.wpb;
}

pa_status check_ws(const Derived &d, void *ws, size_t bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) != 0 || bytes < d.L.total_bytes)
        return PA_ERR_WORKSPACE;
    return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// [num_blocks][Hkv][bs][RB] bytes (block stride may exceed Hkv*bs*RB), box
// [SW bytes][bs][1][1], swizzled by SW.
pa_status make_tmap(CUtensorMap *tm, const void *base, const Derived &d, const pa_problem *p, size_t block_stride,
                    int box_bytes = 0) {
    auto enc = encode_fn();
    if (enc == nullptr) return PA_ERR_CUDA;
    const int bx = box_bytes > 0 ? box_bytes : d.SW;
    cuuint64_t dims[4] = {(cuuint64_t)d.RB, (cuuint64_t)p->block_size, (cuuint64_t)p->num_kv_heads,
                          (cuuint64_t)p->num_blocks};
    cuuint64_t strides[3] = {(cuuint64_t)d.RB, (cuuint64_t)p->block_size * d.RB, (cuuint64_t)block_stride};
    cuuint32_t box[4] = {(cuuint32_t)bx, (cuuint32_t)p->block_size, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     bx == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

// One tile of the grouped kernel -- all segments of [rows][RB] for one kv head of
// a whole block, a part of one, or one block of a merged work page -- as a single
// 5-D box {SW bytes, rows, NSEG segments, 1, 1}:
// the segment dimension (stride SW) is placed outside the rows, so the box
// lands as [segment][row][SW bytes], each SW-byte line swizzled by its row.
pa_status make_tmap_tile(CUtensorMap *tm, const void *base, const Derived &d, const pa_problem *p,
                         size_t block_stride) {
    auto enc = encode_fn();
    if (enc == nullptr) return PA_ERR_CUDA;
    const int nseg = d.RB / d.SW;
    cuuint64_t dims[5] = {(cuuint64_t)d.SW, (cuuint64_t)p->block_size, (cuuint64_t)nseg,
                          (cuuint64_t)p->num_kv_heads, (cuuint64_t)p->num_blocks};
    cuuint64_t strides[4] = {(cuuint64_t)d.RB, (cuuint64_t)d.SW, (cuuint64_t)p->block_size * d.RB,
                             (cuuint64_t)block_stride};
    cuuint32_t box[5] = {(cuuint32_t)d.SW, (cuuint32_t)d.box_rows, (cuuint32_t)nseg, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     d.SW == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

cudaError_t dispatch_attn(const pa_problem *p, const Derived &d, const CUtensorMap &tk, const CUtensorMap &tv,
                          const pa::AttnParams &P, cudaStream_t s) {
    const dim3 grid((unsigned)d.ctas);
    const bool tokm = d.tokm;
#define PA_CASE(KVT, DD)                                                                               \
    if (p->kv_dtype == KVT && d.D == DD)                                                               \
        return d.wpb > 1   ? pa::launch_attn_split<KVT, DD>(tk, tv, P, grid, d.smem, tokm, s)           \
               : d.mpb > 1 ? pa::launch_attn_merged<KVT, DD>(tk, tv, P, grid, d.smem, tokm, s)          \
                           : pa::launch_attn<KVT, DD>(tk, tv, P, grid, d.smem, tokm, s);
    PA_CASE(PA_F16, 64) PA_CASE(PA_F16, 128) PA_CASE(PA_F16, 256)
    PA_CASE(PA_BF16, 64) PA_CASE(PA_BF16, 128) PA_CASE(PA_BF16, 256)
    PA_CASE(PA_E4M3, 64) PA_CASE(PA_E4M3, 128) PA_CASE(PA_E4M3, 256)
    PA_CASE(PA_INT8, 64) PA_CASE(PA_INT8, 128) PA_CASE(PA_INT8, 256)
    PA_CASE(PA_INT4, 128) PA_CASE(PA_INT4, 256)
#undef PA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

extern "C" {

PA_API int pa_version(void) { return VERSION; }

PA_API const char *pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        default: return "PA_ERR_UNKNOWN";
    }
}

PA_API pa_status pa_workspace_layout(const pa_problem *p, pa_layout *layout) {
    if (layout == nullptr) return PA_ERR_INVALID_ARG;
    Derived d;
    const pa_status st = derive(p, &d);
    if (st != PA_OK) return st;
    *layout = d.L;
    return PA_OK;
}

PA_API pa_status pa_workspace_size(const pa_problem *p, size_t *bytes) {
    if (bytes == nullptr) return PA_ERR_INVALID_ARG;
    Derived d;
    const pa_status st = derive(p, &d);
    if (st != PA_OK) return st;
    *bytes = d.L.total_bytes;
    return PA_OK;
}

PA_API pa_status pa_plan(const pa_problem *p, const int32_t *context_lens, const float *k_scale, void *workspace,
                         size_t workspace_bytes, pa_stream_t stream) {
    Derived d;
    pa_status st = derive(p, &d);
    if (st != PA_OK) return st;
    if ((st = check_ws(d, workspace, workspace_bytes)) != PA_OK) return st;
    if (p->batch > 0 && context_lens == nullptr) return PA_ERR_INVALID_ARG;
    if (p->k_scale_mode == PA_SCALE_CHANNEL && k_scale == nullptr) return PA_ERR_INVALID_ARG;
    pa::PlanParams P;
    P.context_lens = context_lens;
    P.hdr = at<uint32_t>(workspace, d.L.header_offset);
    P.req = at<int4>(workspace, d.L.requests_offset);
    P.B = p->batch;
    P.bs = d.wp;                                        // work pages (a block, a part of one, or merged blocks)
    P.max_ctx = p->max_context_len;
    P.mbps = work_pages_per_seq(p, d);
    P.bsb = p->block_size;
    P.tbl = p->max_blocks_per_seq;
    const float *ks = (p->k_scale_mode == PA_SCALE_CHANNEL) ? k_scale : nullptr;
    cudaError_t e = pa::launch_plan(P, ks, p->num_kv_heads * p->head_dim_k, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_run(const pa_problem *p, const void *q, const void *k_pool, const void *v_pool,
                        const int32_t *block_table, const int32_t *context_lens, const float *k_scale,
                        const float *v_scale, void *workspace, size_t workspace_bytes, void *out, float *lse,
                        pa_stream_t stream) {
    Derived d;
    pa_status st = derive(p, &d);
    if (st != PA_OK) return st;
    if ((st = check_ws(d, workspace, workspace_bytes)) != PA_OK) return st;
    if (p->batch == 0) return PA_OK;
    if (q == nullptr || k_pool == nullptr || (v_pool == nullptr && !d.latent) || block_table == nullptr ||
        context_lens == nullptr || out == nullptr)
        return PA_ERR_INVALID_ARG;
    if (d.latent) {
        // q rows are read in 16-byte pieces, outputs as channel pairs
        const uintptr_t out_align = p->out_dtype == PA_F32 ? 7 : 3;
        if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(q) & 15) ||
            (reinterpret_cast<uintptr_t>(out) & out_align))
            return PA_ERR_INVALID_ARG;
        CUtensorMap ta, tb;
        if ((st = make_tmap(&ta, k_pool, d, p, d.k_block, 128)) != PA_OK) return st;
        if ((st = make_tmap(&tb, k_pool, d, p, d.k_block, 64)) != PA_OK) return st;
        pa::LatentParams P;
        P.q = static_cast<const uint8_t *>(q);
        P.k_pool = static_cast<const uint8_t *>(k_pool);
        P.block_table = block_table;
        P.context_lens = context_lens;
        P.hdr = at<uint32_t>(workspace, d.L.header_offset);
        P.req = at<const int4>(workspace, d.L.requests_offset);
        P.part_o = at<float>(workspace, d.L.partial_o_offset);
        P.part_lse = at<float>(workspace, d.L.partial_lse_offset);
        P.out = out;
        P.lse = lse;
        P.block_stride = (long long)d.k_block;
        P.codes_bytes = p->num_kv_heads * LAT_BS * LAT_DK;
        P.B = p->batch;
        P.n = p->next_n;
        P.Hq = p->num_q_heads;
        P.Hkv = p->num_kv_heads;
        P.G = d.G;
        P.R = d.R;
        P.RBLK = d.row_blocks;
        P.mbps = p->max_blocks_per_seq;
        P.num_blocks = p->num_blocks;
        P.q_dtype = p->q_dtype;
        P.out_dtype = p->out_dtype;
        P.causal = p->causal;
        P.softmax_scale = p->softmax_scale;
        cudaError_t e = pa::launch_latent(ta, tb, P, d.ctas, reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    if (d.e4tc) {
        // rows of q are read in 16-byte pieces; the pools are read by tensor copies
        if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(v_pool) & 15) ||
            (reinterpret_cast<uintptr_t>(q) & 15))
            return PA_ERR_INVALID_ARG;
        if ((p->k_scale_mode == PA_SCALE_TENSOR && k_scale == nullptr) ||
            (p->v_scale_mode == PA_SCALE_TENSOR && v_scale == nullptr))
            return PA_ERR_INVALID_ARG;
        CUtensorMap tk, tv;
        if ((st = make_tmap(&tk, k_pool, d, p, d.k_block, 128)) != PA_OK) return st;
        if ((st = make_tmap(&tv, v_pool, d, p, d.v_block, 128)) != PA_OK) return st;
        pa::E4TcParams P;
        P.q = static_cast<const uint8_t *>(q);
        P.k_pool = static_cast<const uint8_t *>(k_pool);
        P.v_pool = static_cast<const uint8_t *>(v_pool);
        P.block_table = block_table;
        P.context_lens = context_lens;
        P.k_scale = k_scale;
        P.v_scale = v_scale;
        P.hdr = at<uint32_t>(workspace, d.L.header_offset);
        P.req = at<const int4>(workspace, d.L.requests_offset);
        P.part_o = at<float>(workspace, d.L.partial_o_offset);
        P.part_lse = at<float>(workspace, d.L.partial_lse_offset);
        P.out = out;
        P.lse = lse;
        P.block_stride = (long long)d.k_block;
        P.B = p->batch;
        P.n = p->next_n;
        P.Hq = p->num_q_heads;
        P.Hkv = p->num_kv_heads;
        P.G = d.G;
        P.R = d.R;
        P.bs = p->block_size;
        P.tbl = p->max_blocks_per_seq;
        P.mbps = work_pages_per_seq(p, d);
        P.num_blocks = p->num_blocks;
        P.q_dtype = p->q_dtype;
        P.out_dtype = p->out_dtype;
        P.k_mode = p->k_scale_mode;
        P.v_mode = p->v_scale_mode;
        P.causal = p->causal;
        P.softmax_scale = p->softmax_scale;
        cudaError_t e = pa::launch_e4m3_tc(tk, tv, P, d.ctas, reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    if ((reinterpret_cast<uintptr_t>(k_pool) & 15) || (reinterpret_cast<uintptr_t>(v_pool) & 15) ||
        (reinterpret_cast<uintptr_t>(q) & 1))
        return PA_ERR_INVALID_ARG;
    if ((p->k_scale_mode == PA_SCALE_TENSOR || p->k_scale_mode == PA_SCALE_CHANNEL) && k_scale == nullptr)
        return PA_ERR_INVALID_ARG;
    if ((p->v_scale_mode == PA_SCALE_TENSOR || p->v_scale_mode == PA_SCALE_CHANNEL) && v_scale == nullptr)
        return PA_ERR_INVALID_ARG;
    CUtensorMap tk, tv;
    if ((st = make_tmap_tile(&tk, k_pool, d, p, d.k_block)) != PA_OK) return st;
    if ((st = make_tmap_tile(&tv, v_pool, d, p, d.v_block)) != PA_OK) return st;
    pa::AttnParams P;
    P.q = static_cast<const uint8_t *>(q);
    P.block_table = block_table;
    P.context_lens = context_lens;
    P.k_scale = k_scale;
    P.v_scale = v_scale;
    P.hdr = at<uint32_t>(workspace, d.L.header_offset);
    P.req = at<const int4>(workspace, d.L.requests_offset);
    P.part_o = at<float>(workspace, d.L.partial_o_offset);
    P.part_lse = at<float>(workspace, d.L.partial_lse_offset);
    P.out = out;
    P.lse = lse;
    P.B = p->batch;
    P.n = p->next_n;
    P.Hq = p->num_q_heads;
    P.Hkv = p->num_kv_heads;
    P.G = d.G;
    P.R = d.R;
    P.RBLK = d.row_blocks;
    P.bs = d.wp;                                    // work pages (a block, a part of one, or merged blocks)
    P.mbps = work_pages_per_seq(p, d);
    P.wpb = d.wpb;
    P.bsb = p->block_size;
    P.tbl_stride = p->max_blocks_per_seq;
    P.num_blocks = p->num_blocks;
    P.q_dtype = p->q_dtype;
    P.out_dtype = p->out_dtype;
    P.k_mode = p->k_scale_mode;
    P.v_mode = p->v_scale_mode;
    P.causal = p->causal;
    P.slots = d.slots;
    P.warp_smem = d.warp_smem;
    P.softmax_scale = p->softmax_scale;
    cudaError_t e = dispatch_attn(p, d, tk, tv, P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_combine(const pa_problem *p, const float *v_scale, void *workspace, size_t workspace_bytes,
                            void *out, float *lse, pa_stream_t stream) {
    Derived d;
    pa_status st = derive(p, &d);
    if (st != PA_OK) return st;
    if ((st = check_ws(d, workspace, workspace_bytes)) != PA_OK) return st;
    if (p->batch == 0) return PA_OK;
    if (out == nullptr) return PA_ERR_INVALID_ARG;
    const int v_mode = d.latent ? PA_SCALE_TOKEN : p->v_scale_mode;  // latent: V shares K's token scales
    if ((v_mode == PA_SCALE_TENSOR || v_mode == PA_SCALE_CHANNEL) && v_scale == nullptr)
        return PA_ERR_INVALID_ARG;
    pa::CombineParams P;
    P.req = at<const int4>(workspace, d.L.requests_offset);
    P.hdr = at<const uint32_t>(workspace, d.L.header_offset);
    P.part_o = at<const float>(workspace, d.L.partial_o_offset);
    P.part_lse = at<const float>(workspace, d.L.partial_lse_offset);
    P.v_scale = v_scale;
    P.out = out;
    P.lse = lse;
    P.B = p->batch;
    P.n = p->next_n;
    P.Hq = p->num_q_heads;
    P.Hkv = p->num_kv_heads;
    P.G = d.G;
    P.R = d.R;
    P.RBLK = d.row_blocks;
    P.Dv = p->head_dim_v;
    P.out_dtype = p->out_dtype;
    P.v_mode = v_mode;
    P.rows_seg = d.rows_seg;
    P.gs = d.gs;
    P.nwarps = d.nwarps;
    cudaError_t e = pa::launch_combine(P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_attention(const pa_problem *p, const void *q, const void *k_pool, const void *v_pool,
                              const int32_t *block_table, const int32_t *context_lens, const float *k_scale,
                              const float *v_scale, void *workspace, size_t workspace_bytes, void *out, float *lse,
                              pa_stream_t stream) {
    pa_status st = pa_plan(p, context_lens, k_scale, workspace, workspace_bytes, stream);
    if (st != PA_OK) return st;
    st = pa_run(p, q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale, workspace, workspace_bytes, out,
                lse, stream);
    if (st != PA_OK) return st;
    return pa_combine(p, v_scale, workspace, workspace_bytes, out, lse, stream);
}

PA_API pa_status pa_get_error(const void *workspace, uint32_t *bits, pa_stream_t stream) {
    if (workspace == nullptr || bits == nullptr) return PA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

}  // extern "C"
