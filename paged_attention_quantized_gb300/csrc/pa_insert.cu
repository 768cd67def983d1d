// pa_insert: quantize the next_n new K / V rows of every request and write
// them into their slots of the paged pool -- the write that precedes each
// decode or verify step of the attention.
//
// Sources (page title, section):
//  - CentML/vllm PR #167, "Q pad + KV insert", Design: the per-token
//    quantization and paged insert of the new K/V rows (this library takes
//    over only that part: no RoPE, no Q padding).
//  - onnxruntime PR #32520, "[CUDA] Normalize the PER_CHANNEL K scale folded
//    into Q for paged XQA", Description: symmetric INT8 / INT4 caches whose
//    scale spans max|K| / 127 or max|K| / 7.
//  - 1Cat-vLLM PR #647, "Stop grouped-page4 null-block padding from leaking
//    E4M3 NaN", Root cause: 0x7F / 0xFF are E4M3's NaN codes, so finite values
//    past 448 saturate instead.
//
// The kernel is HBM-bound.  The new rows of each plane are contiguous in
// their source buffer, so each CTA (3 per SM, 256 threads) takes chunks of
// up to 32 KB of them: one 1-D bulk copy per chunk into a two-stage shared-
// memory ring, issued while the previous chunk is quantized, and the next
// chunk's slots (length check, block id) resolved during the same wait.  Each
// warp splits into row groups of 8, 16 or 32 lanes (the smallest power of two
// that covers the row's 8-channel chunks, 32 for rows longer than 256
// channels) that write one store of 4-16 bytes per 8 channels.  Rows are
// ordered (token, plane, kv head), so the warps of a CTA write neighbouring
// slots of the same blocks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "pa.h"

namespace {

constexpr int THREADS = 256;
constexpr int MAX_D = 2048;  // channels per row at most (8 chunks of 8 per lane)

struct InsertParams {
    const uint8_t *src[2];       // new K rows, new V rows: [B][n][Hkv][D] of the source dtype
    uint8_t *pool[2];            // K plane, V plane
    const float *scale[2];       // per mode: NULL, 1 fp32, or [Hkv][D] fp32
    const int32_t *block_table;
    const int32_t *context_lens;
    uint32_t *err;               // device error word (NULL: not reported)
    long long block_stride[2];   // bytes per block of each plane
    int D[2], row_bytes[2], mode[2];
    int planes;
    int B, n, Hkv, bs, num_blocks, mbps, max_ctx;
    int rows;                    // B * n * planes * Hkv
    int lpr_log2;                // lanes per row = 1 << lpr_log2
    int any_token;               // some plane computes per-token scales
};

template <int SRC>
struct Src;
template <>
struct Src<PA_F32> {
    static constexpr int BYTES = 4;
    __device__ static void load8(const uint8_t *p, float *x) {
        const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};
template <>
struct Src<PA_F16> {
    static constexpr int BYTES = 2;
    __device__ static void load8(const uint8_t *p, float *x) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], 4);
            const float2 f = __half22float2(h);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
};
template <>
struct Src<PA_BF16> {
    static constexpr int BYTES = 2;
    __device__ static void load8(const uint8_t *p, float *x) {
        const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // a bf16 value is the upper half of its fp32
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

// NaN-propagating maximum (a NaN anywhere in a row makes its scale NaN).
__device__ __forceinline__ float nan_max(float a, float b) { return (a != a || a > b) ? a : b; }

// Round to nearest, ties to even, clamp to [-lim, lim]; NaN gives 0.
__device__ __forceinline__ int quant_int(float y, float lim) {
    if (y != y) return 0;
    return (int)fminf(fmaxf(rintf(y), -lim), lim);
}

// Two fp32 values to E4M3 (nearest, ties to even, saturating to +-448, NaN
// stays NaN): `lo` lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Encode 8 quotients and store them at `dst` (16, 8 or 4 bytes).
template <int KV>
__device__ __forceinline__ void store8(uint8_t *dst, const float *y) {
    if constexpr (KV == PA_F16) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(y[2 * i], y[2 * i + 1]);
            memcpy(&w[i], &h, 4);
        }
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (KV == PA_BF16) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
            memcpy(&w[i], &h, 4);
        }
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (KV == PA_E4M3) {
        const uint32_t a = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
        const uint32_t b = e4m3x2(y[4], y[5]) | (e4m3x2(y[6], y[7]) << 16);
        *reinterpret_cast<uint2 *>(dst) = make_uint2(a, b);
    } else if constexpr (KV == PA_INT8) {
        uint32_t w[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i >> 2] |= (uint32_t)(quant_int(y[i], 127.f) & 0xFF) << (8 * (i & 3));
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    } else {  // INT4: channel 2i in the low nibble of byte i
        uint32_t w = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) w |= (uint32_t)(quant_int(y[i], 7.f) & 0xF) << (4 * i);
        *reinterpret_cast<uint32_t *>(dst) = w;
    }
}

// Where one row goes: its source, destination slot, scales and validity.
struct Row {
    const uint8_t *src;
    uint8_t *dst;          // first code byte of the slot's row
    float *tok_scale;      // per-token scale slot of the row
    const float *scale;
    int D, mode, g;
    bool valid;
};

template <int SRC>
__device__ __forceinline__ Row locate(const InsertParams &P, int r, bool report) {
    Row w;
    const int per_tok = P.planes * P.Hkv;
    const int t = r / per_tok;
    const int rem = r - t * per_tok;
    const int plane = rem >= P.Hkv ? 1 : 0;
    const int g = rem - plane * P.Hkv;
    const int b = t / P.n;
    const int j = t - b * P.n;
    w.g = g;
    w.D = P.D[plane];
    w.mode = P.mode[plane];
    w.scale = P.scale[plane];
    w.src = P.src[plane] + ((long long)t * P.Hkv + g) * w.D * Src<SRC>::BYTES;
    w.dst = nullptr;
    w.tok_scale = nullptr;
    w.valid = false;
    const int L = __ldg(P.context_lens + b);
    // the contract: L >= n (the new tokens are counted), L <= max_context_len,
    // and the table holds every page of the request
    if (L < P.n || L > P.max_ctx || (L - 1) / P.bs + 1 > P.mbps) {
        if (report && j == 0 && rem == 0 && P.err) atomicOr(P.err, PA_DEV_ERR_CONTEXT_LEN);
        return w;
    }
    const int pos = L - P.n + j;
    const int page = pos / P.bs;
    const int slot = pos - page * P.bs;
    const int blk = __ldg(P.block_table + (long long)b * P.mbps + page);
    if (blk < 1 || blk >= P.num_blocks) {
        if (report && rem == 0 && P.err) atomicOr(P.err, PA_DEV_ERR_BLOCK_ID);
        return w;
    }
    uint8_t *block = P.pool[plane] + (long long)blk * P.block_stride[plane];
    w.dst = block + (long long)(g * P.bs + slot) * P.row_bytes[plane];
    w.tok_scale = reinterpret_cast<float *>(block + (long long)P.Hkv * P.bs * P.row_bytes[plane]) +
                  (g * P.bs + slot);
    w.valid = true;
    return w;
}

// Staged variant: the new rows of each plane are contiguous in their source
// buffer, so a CTA copies a chunk of up to STAGE_BYTES of them into shared
// memory with one 1-D bulk copy while it quantizes the previous chunk (two
// stages), and resolves the next chunk's slots (length, block id) during the
// same wait.  Every wait is bounded; on a timeout the CTA sets
// PA_DEV_ERR_TIMEOUT, stops, and waits (bounded) for its copies in flight.
constexpr int STAGES = 2;
constexpr int STAGE_BYTES = 32 * 1024;
constexpr int MAX_CHUNK_ROWS = 512;
constexpr unsigned long long WAIT_NS = 2000000000ull;

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool wait_full(uint64_t *bar, uint32_t parity, volatile int *abort) {
    const unsigned long long t0 = [] {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        return t;
    }();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(su32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (*abort) return false;
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > WAIT_NS) return false;
    }
}

struct Chunk {
    int plane, r0, nrows;
};

__device__ __forceinline__ Chunk chunk_of(int c, int nch0, const int (&cr)[2], int rows_p) {
    Chunk ch;
    ch.plane = c < nch0 ? 0 : 1;
    const int ci = c - (ch.plane ? nch0 : 0);
    ch.r0 = ci * cr[ch.plane];
    ch.nrows = min(cr[ch.plane], rows_p - ch.r0);
    return ch;
}

template <int SRC>
__device__ __forceinline__ void issue_chunk(const InsertParams &P, const Chunk &ch, uint8_t *dst, uint64_t *bar) {
    const uint32_t bytes = (uint32_t)ch.nrows * P.D[ch.plane] * Src<SRC>::BYTES;  // rows are multiples of 16 B
    const uint8_t *src = P.src[ch.plane] + (long long)ch.r0 * P.D[ch.plane] * Src<SRC>::BYTES;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(su32(bar))
                 : "memory");
}

// Slot of row i of a chunk: byte offset of its code row in its plane's pool,
// or -1 when the contract check fails (flags raised here).
__device__ __forceinline__ long long slot_of(const InsertParams &P, int plane, int rp) {
    const int t = rp / P.Hkv;
    const int g = rp - t * P.Hkv;
    const int b = t / P.n;
    const int j = t - b * P.n;
    const int L = __ldg(P.context_lens + b);
    if (L < P.n || L > P.max_ctx || (L - 1) / P.bs + 1 > P.mbps) {
        if (j == 0 && g == 0 && plane == 0 && P.err) atomicOr(P.err, PA_DEV_ERR_CONTEXT_LEN);
        return -1;
    }
    const int pos = L - P.n + j;
    const int page = pos / P.bs;
    const int slot = pos - page * P.bs;
    const int blk = __ldg(P.block_table + (long long)b * P.mbps + page);
    if (blk < 1 || blk >= P.num_blocks) {
        if (g == 0 && plane == 0 && P.err) atomicOr(P.err, PA_DEV_ERR_BLOCK_ID);
        return -1;
    }
    return (long long)blk * P.block_stride[plane] + (long long)(g * P.bs + slot) * P.row_bytes[plane];
}

template <int SRC, int KV, int NCK>
__global__ void __launch_bounds__(THREADS, 3)
pa_insert_staged_kernel(const InsertParams P, int cr0, int cr1, int nch0, int nch) {
    extern __shared__ __align__(128) uint8_t stage[];                 // STAGES * STAGE_BYTES
    __shared__ long long slots[STAGES][MAX_CHUNK_ROWS];
    __shared__ __align__(8) uint64_t full[STAGES];
    __shared__ int abort_flag;
    const int tid = threadIdx.x, lane = tid & 31;
    const int lpr = 1 << P.lpr_log2;
    const int sub = lane & (lpr - 1);
    const int rows_per_pass = THREADS >> P.lpr_log2;
    const int cr[2] = {cr0, cr1};  // indexed by plane
    const int rows_p = P.B * P.n * P.Hkv;
    constexpr int BITS = (KV == PA_F16 || KV == PA_BF16) ? 16 : (KV == PA_INT4 ? 4 : 8);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(&full[s])), "r"(1) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
    }
    __syncthreads();
    const int first = blockIdx.x, step = gridDim.x;
    if (first < nch) {
        const Chunk ch = chunk_of(first, nch0, cr, rows_p);
        if (tid == 0) issue_chunk<SRC>(P, ch, stage, &full[0]);
        for (int i = tid; i < ch.nrows; i += THREADS) slots[0][i] = slot_of(P, ch.plane, ch.r0 + i);
    }
    int k = 0;
    bool pending_next = false;
    for (int c = first; c < nch; c += step, ++k) {
        const int s = k & 1;
        const Chunk ch = chunk_of(c, nch0, cr, rows_p);
        const int nxt = c + step;
        pending_next = nxt < nch;
        if (pending_next) {  // stage s^1 and its slots were released by the barrier ending the previous iteration
            const Chunk cn = chunk_of(nxt, nch0, cr, rows_p);
            if (tid == 0) issue_chunk<SRC>(P, cn, stage + (s ^ 1) * STAGE_BYTES, &full[s ^ 1]);
            for (int i = tid; i < cn.nrows; i += THREADS) slots[s ^ 1][i] = slot_of(P, cn.plane, cn.r0 + i);
        }
        if (!wait_full(&full[s], (uint32_t)(k >> 1) & 1u, &abort_flag)) abort_flag = 1;
        __syncthreads();  // slots[s] written, abort decided
        if (abort_flag) break;
        const uint8_t *rows = stage + s * STAGE_BYTES;
        const int D = P.D[ch.plane];
        const int mode = P.mode[ch.plane];
        const float *scale = P.scale[ch.plane];
        uint8_t *pool = P.pool[ch.plane];
        const int passes = (ch.nrows + rows_per_pass - 1) / rows_per_pass;
        for (int pass = 0; pass < passes; ++pass) {
            const int i = pass * rows_per_pass + (tid >> P.lpr_log2);
            const bool in = i < ch.nrows;
            float x[NCK][8];
#pragma unroll
            for (int kk = 0; kk < NCK; ++kk) {
                const int cc = sub + kk * lpr;
                if (in && cc * 8 < D) {
                    const uint8_t *src = rows + ((long long)i * D + cc * 8) * Src<SRC>::BYTES;
                    if constexpr (SRC == PA_F32) {
                        const float4 a = *reinterpret_cast<const float4 *>(src);
                        const float4 b = *reinterpret_cast<const float4 *>(src + 16);
                        x[kk][0] = a.x; x[kk][1] = a.y; x[kk][2] = a.z; x[kk][3] = a.w;
                        x[kk][4] = b.x; x[kk][5] = b.y; x[kk][6] = b.z; x[kk][7] = b.w;
                    } else {
                        const uint4 u = *reinterpret_cast<const uint4 *>(src);
                        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if constexpr (SRC == PA_F16) {
                                __half2 h;
                                memcpy(&h, &w[q], 4);
                                const float2 f = __half22float2(h);
                                x[kk][2 * q] = f.x;
                                x[kk][2 * q + 1] = f.y;
                            } else {
                                x[kk][2 * q] = __uint_as_float(w[q] << 16);
                                x[kk][2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) x[kk][q] = 0.f;
                }
            }
            float s_tok = 1.f;
            if (P.any_token) {  // every lane of the warp takes part
                float m = 0.f;
#pragma unroll
                for (int kk = 0; kk < NCK; ++kk)
#pragma unroll
                    for (int q = 0; q < 8; ++q) m = nan_max(fabsf(x[kk][q]), m);
                for (int o = lpr >> 1; o > 0; o >>= 1) m = nan_max(__shfl_xor_sync(0xffffffffu, m, o), m);
                s_tok = __fdiv_rn(m, 448.f);
                if (s_tok == 0.f) s_tok = 1.f;
            }
            const long long off = in ? slots[s][i] : -1;
            if (off < 0) continue;
            const int rp = ch.r0 + i;
            const int g = rp - (rp / P.Hkv) * P.Hkv;
            uint8_t *dst = pool + off;
            float ts = 1.f;
            if (mode == PA_SCALE_TENSOR) ts = __ldg(scale);
            if (mode == PA_SCALE_TOKEN) ts = s_tok;
#pragma unroll
            for (int kk = 0; kk < NCK; ++kk) {
                const int cc = sub + kk * lpr;
                if (cc * 8 >= D) continue;
                float y[8];
                if (mode == PA_SCALE_NONE) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) y[q] = x[kk][q];
                } else if (mode == PA_SCALE_CHANNEL) {
                    const float4 *sp = reinterpret_cast<const float4 *>(scale + (long long)g * D + cc * 8);
                    const float4 a = __ldg(sp), b = __ldg(sp + 1);
                    const float s8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int q = 0; q < 8; ++q) y[q] = __fdiv_rn(x[kk][q], s8[q]);
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) y[q] = __fdiv_rn(x[kk][q], ts);
                }
                store8<KV>(dst + cc * BITS, y);
            }
            if (mode == PA_SCALE_TOKEN && sub == 0) {
                // the scale slot: after the block's codes, [Hkv][bs] fp32
                const long long blk_off = off - (off % P.block_stride[ch.plane]);
                const long long in_blk = off - blk_off;             // (g * bs + slot) * row_bytes
                const int gs = (int)(in_blk / P.row_bytes[ch.plane]);
                *reinterpret_cast<float *>(pool + blk_off + (long long)P.Hkv * P.bs * P.row_bytes[ch.plane] +
                                           (long long)gs * 4) = s_tok;
            }
        }
        __syncthreads();  // stage s and slots[s] free for the chunk after next
    }
    if (abort_flag && tid == 0) {
        if (P.err) atomicOr(P.err, PA_DEV_ERR_TIMEOUT);
        // copies still in flight on either stage: wait for them, bounded
        // (chunk k on stage k & 1, and chunk k + 1 on the other stage if it was issued)
        volatile int never = 0;
        for (int d = 0; d < 2; ++d) {
            const int kk = k + d;
            if (d == 1 && !pending_next) break;
            wait_full(&full[kk & 1], (uint32_t)(kk >> 1) & 1u, &never);
        }
    }
}

template <int SRC, int KV>
cudaError_t launch_kv(const InsertParams &P, int nck, int ctas, int cr0, int cr1, int nch0, int nch, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = STAGES * STAGE_BYTES;
    cfg.stream = s;
    if (nck == 1) {
        cudaFuncSetAttribute(pa_insert_staged_kernel<SRC, KV, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             STAGES * STAGE_BYTES);
        return cudaLaunchKernelEx(&cfg, pa_insert_staged_kernel<SRC, KV, 1>, P, cr0, cr1, nch0, nch);
    }
    if (nck == 4) {
        cudaFuncSetAttribute(pa_insert_staged_kernel<SRC, KV, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             STAGES * STAGE_BYTES);
        return cudaLaunchKernelEx(&cfg, pa_insert_staged_kernel<SRC, KV, 4>, P, cr0, cr1, nch0, nch);
    }
    cudaFuncSetAttribute(pa_insert_staged_kernel<SRC, KV, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         STAGES * STAGE_BYTES);
    return cudaLaunchKernelEx(&cfg, pa_insert_staged_kernel<SRC, KV, 8>, P, cr0, cr1, nch0, nch);
}

template <int SRC>
cudaError_t launch_src(const InsertParams &P, int kv, int nck, int ctas, int cr0, int cr1, int nch0, int nch,
                       cudaStream_t s) {
    switch (kv) {
        case PA_F16: return launch_kv<SRC, PA_F16>(P, nck, ctas, cr0, cr1, nch0, nch, s);
        case PA_BF16: return launch_kv<SRC, PA_BF16>(P, nck, ctas, cr0, cr1, nch0, nch, s);
        case PA_E4M3: return launch_kv<SRC, PA_E4M3>(P, nck, ctas, cr0, cr1, nch0, nch, s);
        case PA_INT8: return launch_kv<SRC, PA_INT8>(P, nck, ctas, cr0, cr1, nch0, nch, s);
        case PA_INT4: return launch_kv<SRC, PA_INT4>(P, nck, ctas, cr0, cr1, nch0, nch, s);
        default: return cudaErrorInvalidValue;
    }
}

int kv_bits(int dt) {
    switch (dt) {
        case PA_F16: case PA_BF16: return 16;
        case PA_E4M3: case PA_INT8: return 8;
        case PA_INT4: return 4;
        default: return 0;
    }
}

std::atomic<int> g_insert_sms[64];

pa_status sm_count(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev >= 0 && dev < 64) {
        const int c = g_insert_sms[dev].load(std::memory_order_relaxed);
        if (c > 0) { *sms = c; return PA_OK; }
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return PA_ERR_CUDA;
    if (dev >= 0 && dev < 64) g_insert_sms[dev].store(v, std::memory_order_relaxed);
    *sms = v;
    return PA_OK;
}

bool misaligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

}  // namespace

extern "C" PA_API pa_status pa_insert(const pa_problem *p, int32_t src_dtype, const void *k_new, const void *v_new,
                                      const int32_t *block_table, const int32_t *context_lens,
                                      const float *k_scale, const float *v_scale, void *k_pool, void *v_pool,
                                      uint32_t *dev_error, pa_stream_t stream) {
    if (p == nullptr) return PA_ERR_INVALID_ARG;
    if (p->batch < 0 || p->next_n < 1 || p->num_kv_heads < 1 || p->block_size < 1 || p->num_blocks < 1 ||
        p->max_blocks_per_seq < 1 || p->max_context_len < 0 || p->num_sms < 0)
        return PA_ERR_INVALID_ARG;
    if (src_dtype != PA_F32 && src_dtype != PA_F16 && src_dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    const int bits = kv_bits(p->kv_dtype);
    if (bits == 0) return PA_ERR_INVALID_ARG;
    if (p->v_is_k_prefix != 0 && p->v_is_k_prefix != 1) return PA_ERR_INVALID_ARG;
    const int planes = p->v_is_k_prefix ? 1 : 2;
    const int Ds[2] = {p->head_dim_k, p->head_dim_v};
    const int modes[2] = {p->k_scale_mode, p->v_scale_mode};
    const float *scales[2] = {k_scale, v_scale};
    if (p->v_is_k_prefix && (p->head_dim_v < 1 || p->head_dim_v > p->head_dim_k)) return PA_ERR_INVALID_ARG;
    for (int i = 0; i < planes; ++i) {
        if (Ds[i] < 8 || Ds[i] > MAX_D || Ds[i] % 8 != 0) return PA_ERR_UNSUPPORTED;
        if (modes[i] < PA_SCALE_NONE || modes[i] > PA_SCALE_TOKEN) return PA_ERR_INVALID_ARG;
        if (modes[i] == PA_SCALE_TOKEN && p->kv_dtype != PA_E4M3) return PA_ERR_UNSUPPORTED;
        if (modes[i] == PA_SCALE_TENSOR && (scales[i] == nullptr || misaligned(scales[i], 4)))
            return PA_ERR_INVALID_ARG;
        if (modes[i] == PA_SCALE_CHANNEL && (scales[i] == nullptr || misaligned(scales[i], 16)))
            return PA_ERR_INVALID_ARG;
    }
    const long long rows = (long long)p->batch * p->next_n * planes * p->num_kv_heads;
    if (rows > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
    if (dev_error != nullptr && misaligned(dev_error, 4)) return PA_ERR_INVALID_ARG;
    if (rows == 0) return PA_OK;

    InsertParams P = {};
    const void *srcs[2] = {k_new, v_new};
    void *pools[2] = {k_pool, v_pool};
    int dmax = 0;
    for (int i = 0; i < planes; ++i) {
        if (srcs[i] == nullptr || pools[i] == nullptr) return PA_ERR_INVALID_ARG;
        if (misaligned(srcs[i], 16) || misaligned(pools[i], 16)) return PA_ERR_INVALID_ARG;
        const int row_bytes = Ds[i] * bits / 8;
        const long long codes = (long long)p->num_kv_heads * p->block_size * row_bytes;
        const long long stride = codes + (modes[i] == PA_SCALE_TOKEN ? (long long)p->num_kv_heads * p->block_size * 4 : 0);
        if (stride % 16 != 0) return PA_ERR_UNSUPPORTED;
        P.src[i] = static_cast<const uint8_t *>(srcs[i]);
        P.pool[i] = static_cast<uint8_t *>(pools[i]);
        P.scale[i] = scales[i];
        P.block_stride[i] = stride;
        P.D[i] = Ds[i];
        P.row_bytes[i] = row_bytes;
        P.mode[i] = modes[i];
        if (modes[i] == PA_SCALE_TOKEN) P.any_token = 1;
        dmax = std::max(dmax, Ds[i]);
    }
    if (block_table == nullptr || context_lens == nullptr) return PA_ERR_INVALID_ARG;
    P.block_table = block_table;
    P.context_lens = context_lens;
    P.err = dev_error;
    P.planes = planes;
    P.B = p->batch;
    P.n = p->next_n;
    P.Hkv = p->num_kv_heads;
    P.bs = p->block_size;
    P.num_blocks = p->num_blocks;
    P.mbps = p->max_blocks_per_seq;
    P.max_ctx = p->max_context_len;
    P.rows = (int)rows;

    // lanes per row: the smallest power of two >= the row's 8-channel chunks
    // (at most 32); chunks per lane beyond that
    const int chunks = dmax / 8;
    int lg = 0;
    while ((1 << lg) < chunks && lg < 5) ++lg;
    P.lpr_log2 = lg;
    const int per_lane = (chunks + (1 << lg) - 1) >> lg;
    const int nck = per_lane <= 1 ? 1 : (per_lane <= 4 ? 4 : 8);

    int sms = p->num_sms;
    if (sms == 0) {
        const pa_status st = sm_count(&sms);
        if (st != PA_OK) return st;
    }
    const int esize = src_dtype == PA_F32 ? 4 : 2;
    int cr[2] = {1, 1}, nch_p[2] = {0, 0};
    const int rows_p = (int)(rows / planes);
    for (int i = 0; i < planes; ++i) {
        cr[i] = std::min(MAX_CHUNK_ROWS, STAGE_BYTES / (Ds[i] * esize));
        nch_p[i] = (rows_p + cr[i] - 1) / cr[i];
    }
    const int nch = nch_p[0] + nch_p[1];
    const int ctas = std::min(nch, sms * 3);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (src_dtype) {
        case PA_F32: e = launch_src<PA_F32>(P, p->kv_dtype, nck, ctas, cr[0], cr[1], nch_p[0], nch, s); break;
        case PA_F16: e = launch_src<PA_F16>(P, p->kv_dtype, nck, ctas, cr[0], cr[1], nch_p[0], nch, s); break;
        default: e = launch_src<PA_BF16>(P, p->kv_dtype, nck, ctas, cr[0], cr[1], nch_p[0], nch, s); break;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
