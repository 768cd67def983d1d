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
// The kernel is HBM-bound (16-byte vector loads of the new rows, one store of
// 4-16 bytes per 8 channels): a grid-stride loop over up to 8 CTAs of 256
// threads per SM, each warp split into row groups of 8, 16 or 32 lanes (the
// smallest power of two that covers the row's 8-channel chunks, 32 for rows
// longer than 256 channels).
// Rows are ordered (token, plane, kv head), so the warps of a CTA write
// neighbouring slots of the same blocks.
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

// NCK: 8-channel chunks per lane at most; UNR: row groups a warp loads
// before it encodes any (more bytes in flight for short rows).
template <int SRC, int KV, int NCK, int UNR>
__global__ void __launch_bounds__(THREADS, NCK == 1 ? 4 : 2) pa_insert_kernel(const InsertParams P) {
    const int lane = threadIdx.x & 31;
    const int lpr = 1 << P.lpr_log2;
    const int sub = lane & (lpr - 1);
    const int rpw = 32 >> P.lpr_log2;  // rows per warp and group
    const long long warp = ((long long)blockIdx.x * THREADS + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * THREADS) >> 5;
    constexpr int BITS = (KV == PA_F16 || KV == PA_BF16) ? 16 : (KV == PA_INT4 ? 4 : 8);
    for (long long base = warp * rpw * UNR; base < P.rows; base += nwarps * rpw * UNR) {
        float x[UNR][NCK][8];
        Row row[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const long long r = base + u * rpw + (lane >> P.lpr_log2);
            if (r < P.rows) {
                row[u] = locate<SRC>(P, (int)r, sub == 0);
            } else {
                row[u].valid = false;
                row[u].D = 0;
            }
#pragma unroll
            for (int k = 0; k < NCK; ++k) {
                const int c = sub + k * lpr;
                if (row[u].valid && c * 8 < row[u].D) {
                    Src<SRC>::load8(row[u].src + (long long)c * 8 * Src<SRC>::BYTES, x[u][k]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[u][k][i] = 0.f;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            float s_tok = 1.f;
            if (P.any_token) {  // uniform: every lane of the warp reduces
                float m = 0.f;
#pragma unroll
                for (int k = 0; k < NCK; ++k)
#pragma unroll
                    for (int i = 0; i < 8; ++i) m = nan_max(fabsf(x[u][k][i]), m);
                for (int o = lpr >> 1; o > 0; o >>= 1) m = nan_max(__shfl_xor_sync(0xffffffffu, m, o), m);
                s_tok = __fdiv_rn(m, 448.f);
                if (s_tok == 0.f) s_tok = 1.f;
            }
            const Row &w = row[u];
            if (!w.valid) continue;
            float ts = 1.f;
            if (w.mode == PA_SCALE_TENSOR) ts = __ldg(w.scale);
            if (w.mode == PA_SCALE_TOKEN) ts = s_tok;
#pragma unroll
            for (int k = 0; k < NCK; ++k) {
                const int c = sub + k * lpr;
                if (c * 8 >= w.D) continue;
                float y[8];
                if (w.mode == PA_SCALE_NONE) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = x[u][k][i];
                } else if (w.mode == PA_SCALE_CHANNEL) {
                    const float4 *sp = reinterpret_cast<const float4 *>(w.scale + (long long)w.g * w.D + c * 8);
                    const float4 a = __ldg(sp), b = __ldg(sp + 1);
                    const float s8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(x[u][k][i], s8[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(x[u][k][i], ts);
                }
                store8<KV>(w.dst + c * BITS, y);
            }
            if (w.mode == PA_SCALE_TOKEN && sub == 0) *w.tok_scale = s_tok;
        }
    }
}

template <int SRC, int KV>
cudaError_t launch_kv(const InsertParams &P, int nck, int ctas, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    if (nck == 1) return cudaLaunchKernelEx(&cfg, pa_insert_kernel<SRC, KV, 1, 2>, P);
    if (nck == 4) return cudaLaunchKernelEx(&cfg, pa_insert_kernel<SRC, KV, 4, 1>, P);
    return cudaLaunchKernelEx(&cfg, pa_insert_kernel<SRC, KV, 8, 1>, P);
}

template <int SRC>
cudaError_t launch_src(const InsertParams &P, int kv, int nck, int ctas, cudaStream_t s) {
    switch (kv) {
        case PA_F16: return launch_kv<SRC, PA_F16>(P, nck, ctas, s);
        case PA_BF16: return launch_kv<SRC, PA_BF16>(P, nck, ctas, s);
        case PA_E4M3: return launch_kv<SRC, PA_E4M3>(P, nck, ctas, s);
        case PA_INT8: return launch_kv<SRC, PA_INT8>(P, nck, ctas, s);
        case PA_INT4: return launch_kv<SRC, PA_INT4>(P, nck, ctas, s);
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
    const int unr = nck == 1 ? 2 : 1;

    int sms = p->num_sms;
    if (sms == 0) {
        const pa_status st = sm_count(&sms);
        if (st != PA_OK) return st;
    }
    const long long rows_per_cta = (long long)(THREADS / 32) * (32 >> lg) * unr;
    const long long want = (rows + rows_per_cta - 1) / rows_per_cta;
    const int ctas = (int)std::min<long long>(want, (long long)sms * (2048 / THREADS));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (src_dtype) {
        case PA_F32: e = launch_src<PA_F32>(P, p->kv_dtype, nck, ctas, s); break;
        case PA_F16: e = launch_src<PA_F16>(P, p->kv_dtype, nck, ctas, s); break;
        default: e = launch_src<PA_BF16>(P, p->kv_dtype, nck, ctas, s); break;
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
