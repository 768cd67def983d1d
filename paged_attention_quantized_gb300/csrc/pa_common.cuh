// Device helpers shared by the paged-attention kernels (sm_103a).
// Inline PTX for mbarriers, bulk tensor copies (TMA), warp-level MMA and the
// packed conversions used to dequantize KV codes in registers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// ------------------------------------------------------------ kernel params

struct AttnParams {
    const uint8_t *q;
    const int32_t *block_table;
    const int32_t *context_lens;
    const float *k_scale;
    const float *v_scale;
    uint32_t *hdr;       // workspace header words
    const int4 *req;     // per-request plan records {L, pages, pages before, flags}
    float *part_o;       // [slots][16][Dv] partial outputs of segment pieces
    float *part_lse;     // [slots][16]
    void *out;
    float *lse;
    int B, n, Hq, Hkv, G, R, RBLK, num_blocks;
    int bs;              // tokens of a work page: a block, an equal part of one, or merged blocks
    int mbps;            // work pages per request at most (table width x wpb, or / blocks merged)
    int wpb;             // work pages per block (parts of a block)
    int bsb;             // tokens of a block
    int tbl_stride;      // block_table row stride (blocks per request)
    int q_dtype, out_dtype, k_mode, v_mode, causal;
    int slots;           // ring pages per worker (a warp, or a pair of warps)
    int warp_smem;       // shared-memory bytes per warp
    float softmax_scale;
};

// The single-latent kernel: K and V share one E4M3 plane per kv head (V is
// the first 512 of 576 channels) with a per-token fp32 scale after the codes
// of every block.
struct LatentParams {
    const uint8_t *q;
    const uint8_t *k_pool;     // block b starts at k_pool + b * block_stride
    const int32_t *block_table;
    const int32_t *context_lens;
    uint32_t *hdr;
    const int4 *req;
    float *part_o;             // [slots][64][512]
    float *part_lse;           // [slots][64]
    void *out;
    float *lse;
    long long block_stride;    // bytes per pool block (codes + scales)
    int codes_bytes;           // Hkv * bs * 576: offset of the scales in a block
    int B, n, Hq, Hkv, G, R, RBLK, mbps, num_blocks;
    int q_dtype, out_dtype, causal;
    float softmax_scale;
};

// The E4M3 tensor-core kernel (head dim 256, 16..64 query rows per kv head):
// separate K and V planes, per-tensor (or no) scales, 128-token chunks.
struct E4TcParams {
    const uint8_t *q;
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    const int32_t *block_table;
    const int32_t *context_lens;
    const float *k_scale;  // per-tensor or NULL
    const float *v_scale;
    uint32_t *hdr;
    const int4 *req;       // plan over 128-token chunks
    float *part_o;         // [slots][R][256]
    float *part_lse;       // [slots][R]
    void *out;
    float *lse;
    long long block_stride;  // bytes per pool block (Hkv * bs * 256)
    int B, n, Hq, Hkv, G, R, bs, tbl, mbps, num_blocks;
    int q_dtype, out_dtype, k_mode, v_mode, causal;
    float softmax_scale;
};

struct PlanParams {
    const int32_t *context_lens;
    uint32_t *hdr;
    int4 *req;
    int B, bs, max_ctx, mbps;  // bs: tokens of a work page; mbps: work pages per request at most
    int bsb, tbl;              // tokens of a block, blocks per request at most (the table width)
};

struct CombineParams {
    const int4 *req;
    const uint32_t *hdr;
    const float *part_o;
    const float *part_lse;
    const float *v_scale;
    void *out;
    float *lse;
    int B, n, Hq, Hkv, G, R, RBLK, Dv, out_dtype, v_mode;
    int rows_seg;      // query rows per segment (16, or 64 for the latent kernel)
    int gs;            // workers per group (1, or the row blocks for the latent kernel)
    long long nwarps;  // workers of the attention launch (warps, or CTAs for the latent kernel)
};

// header word indices
constexpr int HDR_ERR = 0;
constexpr int HDR_TOTAL_PAGES = 1;  // sum over requests of their pages
constexpr int HDR_KMAX = 3;

// bounded waits: give up after this many nanoseconds of %globaltimer (2 s;
// a test build sets a shorter limit with -DPA_WAIT_LIMIT_NS=...)
#ifndef PA_WAIT_LIMIT_NS
#define PA_WAIT_LIMIT_NS 2000000000ull
#endif
constexpr unsigned long long WAIT_LIMIT_NS = PA_WAIT_LIMIT_NS;
// Test builds only (-DPA_FAULT_INJECT): header word 4 of the workspace names a
// page (its global position + 1, 0 = none) whose copy every producer that
// owns it withholds -- neither a copy nor an arrive -- so the waits on that
// ring slot run out, the way a copy lost on the device would look.
constexpr int HDR_WITHHOLD = 4;

// ------------------------------------------------------------------ basics

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity.  Gives up (returns
// false) when *abort (if given) becomes non-zero or after WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (globaltimer() - t0 > WAIT_LIMIT_NS) return false;
    }
}

// -------------------------------------------------------------------- TMA

// 4-D tiled bulk tensor copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *tm, uint64_t *bar, int x, int y, int z,
                                            int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// An L2 policy for data read once (the KV stream): its lines are the first
// to go, so the stream does not push out what is reused (code, queries,
// tables, plan records).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// the default L2 policy, as a value (for call sites that pick one at run time)
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_4d with an L2 cache policy
__device__ __forceinline__ void tma_load_4d_hint(void *dst, const CUtensorMap *tm, uint64_t *bar, int x, int y, int z,
                                                 int w, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// 5-D tiled bulk tensor copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *tm, uint64_t *bar, int c0, int c1, int c2,
                                            int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
        : "memory");
}

// tma_load_5d with an L2 cache policy
__device__ __forceinline__ void tma_load_5d_hint(void *dst, const CUtensorMap *tm, uint64_t *bar, int c0, int c1,
                                                 int c2, int c3, int c4, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar)),
        "l"(pol)
        : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// bulk_load with an L2 cache policy
__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// -------------------------------------------------------------------- MMA

// D = A * B + D, m16n8k16, fp32 accumulate.  A row-major (4 regs), B
// column-major (2 regs), C/D 4 floats.
template <bool BF16>
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// four 8x8 b16 matrices from shared memory (lane i supplies the row address
// of matrix i / 8); .trans delivers the transposed matrices
__device__ __forceinline__ void ldsm_x4(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// barrier `id` (1..15) over `count` threads (a multiple of 32)
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------- conversions

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) return pack_bf16x2(lo, hi);
    else return pack_f16x2(lo, hi);
}

// two E4M3 codes (low byte -> low half) to f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two_codes) {
    uint32_t r;
    const uint16_t v = static_cast<uint16_t>(two_codes & 0xFFFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
    __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b),
                        *reinterpret_cast<__half2 *>(&c));
    return *reinterpret_cast<uint32_t *>(&r);
}

// Integer codes to f16 through the exponent trick: the f16 with bits 0x64XX
// is exactly 1024 + XX, and 0x64XY (nibble form) 1024 + XY.
constexpr uint32_t F16X2_1152 = 0x64806480u;  // {1152, 1152}: 1024 + 128
constexpr uint32_t F16X2_1032 = 0x64086408u;  // {1032, 1032}: 1024 + 8
constexpr uint32_t F16X2_1_16 = 0x2C002C00u;  // {1/16, 1/16}
constexpr uint32_t F16X2_M72 = 0xD480D480u;   // {-72, -72}

// bytes b0, b1 of an (offset-binary) int8 word -> f16x2 {b0 - 128, b1 - 128}
__device__ __forceinline__ uint32_t u8pair_f16x2(uint32_t ux, uint32_t sel) {
    return hsub2_u(__byte_perm(ux, 0x64646464u, sel), F16X2_1152);
}

// low nibbles of bytes 0 and 2 (offset-binary) -> {n0 - 8, n2 - 8}
__device__ __forceinline__ uint32_t u4lo_f16x2(uint32_t ux) {
    return hsub2_u((ux & 0x000F000Fu) | 0x64006400u, F16X2_1032);
}

// high nibbles of bytes 0 and 2 (offset-binary) -> {n0 - 8, n2 - 8}
__device__ __forceinline__ uint32_t u4hi_f16x2(uint32_t ux) {
    return hfma2_u((ux & 0x00F000F0u) | 0x64006400u, F16X2_1_16, F16X2_M72);
}

// (a & b) ^ c in one instruction
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Two's-complement nibbles straight from the stored word (no offset-binary
// XOR first): ((w ^ 8) & 0xF) | 0x6400 equals (w & 0xF) ^ 0x6408, one LOP3.
// low nibbles of bytes 0 and 2 -> {n0, n2}
__device__ __forceinline__ uint32_t s4lo_f16x2(uint32_t w) {
    return hsub2_u(and_xor(w, 0x000F000Fu, 0x64086408u), F16X2_1032);
}

// high nibbles of bytes 0 and 2 -> {n0, n2}
__device__ __forceinline__ uint32_t s4hi_f16x2(uint32_t w) {
    return hfma2_u(and_xor(w, 0x00F000F0u, 0x64806480u), F16X2_1_16, F16X2_M72);
}

// ------------------------------------------------- programmatic dependent launch

// Block until the grid this launch depends on has finished and its writes are
// visible (a no-op when the launch had no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next launch on the stream start its prologue early.
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` with programmatic stream serialisation: it may begin while
// the previous kernel on the stream drains, and waits in grid_dependency_wait.
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// -------------------------------------------------------------- reductions

__device__ __forceinline__ void atomic_or_err(uint32_t *hdr, uint32_t bits) {
    if (bits) atomicOr(hdr + HDR_ERR, bits);
}

}  // namespace pa
