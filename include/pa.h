/*
 * pa.h -- paged decode / verify attention over a quantized paged KV cache.
 *
 * C ABI of the GB300 (sm_103a) library `libpa.so`.  Plain pointers and sizes
 * only.  Every call enqueues work on the caller's CUDA stream and returns
 * without synchronising (except pa_get_error), so a pa_plan -> pa_run ->
 * pa_combine sequence can be captured in a CUDA graph.
 *
 * The operation (for request b, query row j < next_n, query head h, kv head
 * g = h / (Hq / Hkv)):
 *
 *   vis   = causal ? L_b - (next_n - 1 - j) : L_b
 *   k^_t  = dec(K[block_table[b][t / bs], g, t % bs, :]) * k_scale
 *   v^_t  = dec(V[block_table[b][t / bs], g, t % bs, :]) * v_scale
 *   out   = softmax_t( softmax_scale * q[b, j, h, :] . k^_t ) . v^_t   for t < vis
 *   lse   = ln sum_t exp(softmax_scale * q . k^_t)                   (optional)
 *   vis <= 0 gives out = 0 and lse = -inf.
 *
 * Sources (page title, section):
 *  - FlashInfer docs, "flashinfer.fp4_paged_mqa_logits", Parameters: the
 *    problem statement -- q [batch, next_n, heads, dim], a paged pool indexed by
 *    block_table [batch, max_blocks_per_seq] int32, context_lens [batch] int32
 *    bounded by max_context_len, a device-side schedule that is only valid for
 *    the context_lens it was computed from, and a preallocated `out`.
 *  - onnxruntime PR #32520, "[CUDA] Normalize the PER_CHANNEL K scale folded into
 *    Q for paged XQA", Description / Approach: FP8 / INT8 / INT4 caches with a
 *    per-tensor or per-(kv head, channel) scale; a single-block max|k_scale|
 *    reduction, launched on the device so the step stays capturable, whose
 *    result normalises the scale folded into q.
 *  - 1Cat-vLLM PR #494, "[Bugfix][SM70] Stabilize QSA page4 order under KV
 *    relocation", Summary / Contract and limits: work is ordered by logical
 *    token position; results are bitwise identical when pages are relocated.
 *  - 1Cat-vLLM PR #647, "[Bugfix][SM70] Stop grouped-page4 null-block padding
 *    from leaking E4M3 NaN", Root cause / Fix: block 0 is the null block;
 *    padding and unused slots never reach P.V (0 * NaN = NaN).
 *
 * ------------------------------------------------------------------ layouts
 *  q            [batch][next_n][Hq][Dk]   fp16 or bf16, contiguous (16-byte
 *               aligned for the single-latent shape, 2-byte otherwise).
 *  k_pool       [num_blocks] blocks; each block is [Hkv][bs][row bytes] codes,
 *               followed -- only with PA_SCALE_TOKEN -- by [Hkv][bs] fp32
 *               per-token scales.  Row bytes = Dk * bits / 8 (fp16/bf16 16,
 *               E4M3/INT8 8, INT4 4).  INT4: two's-complement nibbles, channel
 *               2i in the low nibble of byte i.  INT8: two's complement.
 *               E4M3: the "fn" FP8 format (0x7F / 0xFF are NaN).
 *               Base address 16-byte aligned.
 *  v_pool       the same with Dv, or NULL when v_is_k_prefix (V is then the
 *               first Dv channels of the K plane and uses K's scales; this
 *               build supports it for the single-latent shape only: E4M3
 *               codes, PA_SCALE_TOKEN, Dk = 576, Dv = 512, bs = 64).
 *  block_table  [batch][max_blocks_per_seq] int32 physical block ids.  Columns
 *               p < ceil(L_b / bs) must hold ids in [1, num_blocks); block 0 is
 *               the null block.  Other columns are never read.
 *  context_lens [batch] int32, 0 <= L_b <= max_context_len.
 *  k_scale      PA_SCALE_NONE: NULL.  TENSOR: 1 fp32.  CHANNEL: [Hkv][Dk] fp32.
 *               TOKEN: NULL (the scales live in the pool blocks).
 *  v_scale      as k_scale with Dv (NULL when v_is_k_prefix).
 *  out          [batch][next_n][Hq][Dv] of out_dtype (f32 / f16 / bf16).
 *  lse          optional [batch][next_n][Hq] fp32 (natural log), or NULL.
 *  workspace    caller-owned device memory of pa_workspace_size() bytes,
 *               256-byte aligned.  It holds the plan, the split partials and a
 *               device error word; its layout is reported by
 *               pa_workspace_layout().
 *
 * ---------------------------------------------------------------- ownership
 *  The caller owns every buffer.  The library allocates no memory, keeps no
 *  per-call state outside the workspace, and reads device pointers only from
 *  kernels.  All calls for one workspace must be ordered on one stream.
 *  A plan is valid only for the context_lens it was made from: re-run pa_plan
 *  (into the same workspace) whenever they change, e.g. before every replay of
 *  a captured step.
 *
 * ------------------------------------------------------------------- errors
 *  Host-detectable problems return a status and launch nothing.  Among
 *  them: a batch whose table could name more than 2^31 - 1 pages in all
 *  (batch x max_blocks_per_seq work pages) is PA_ERR_UNSUPPORTED, since the
 *  plan keeps page counts in 32 bits.
 *  Contract violations only visible on the device (a block id outside
 *  [1, num_blocks) at a visible position, L_b outside [0, max_context_len] or
 *  needing more than max_blocks_per_seq columns, context_lens changed since
 *  pa_plan) set bits in the workspace's device error word and fill the
 *  affected request's output rows with NaN.  The kernels never trap and every
 *  wait they contain is bounded; a wait that runs out sets PA_DEV_ERR_TIMEOUT.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

/* A cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st *pa_stream_t;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* bad size, NULL or misaligned pointer, bad enum */
    PA_ERR_UNSUPPORTED = 2, /* valid problem this build has no kernel for */
    PA_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or too small */
    PA_ERR_CUDA = 4         /* a CUDA runtime call or launch failed */
} pa_status;

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_E4M3 = 3, PA_INT8 = 4, PA_INT4 = 5 } pa_dtype;

typedef enum {
    PA_SCALE_NONE = 0,    /* codes are the values */
    PA_SCALE_TENSOR = 1,  /* one fp32 scalar */
    PA_SCALE_CHANNEL = 2, /* one fp32 per (kv head, channel) */
    PA_SCALE_TOKEN = 3    /* one fp32 per (block, kv head, slot), inside the block */
} pa_scale_mode;

/* Bits of the device error word (pa_get_error). */
#define PA_DEV_ERR_BLOCK_ID 0x1u    /* visible position mapped to an id outside [1, num_blocks) */
#define PA_DEV_ERR_CONTEXT_LEN 0x2u /* L_b < 0, > max_context_len, or > max_blocks_per_seq pages */
#define PA_DEV_ERR_STALE_PLAN 0x4u  /* context_lens differ from the ones pa_plan saw */
#define PA_DEV_ERR_TIMEOUT 0x8u     /* a bounded wait inside a kernel ran out */
#define PA_DEV_ERR_PLAN_OVERFLOW 0x10u

typedef struct pa_problem {
    int32_t batch;              /* B >= 0 requests */
    int32_t next_n;             /* query rows per request, >= 1 */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv, divides Hq */
    int32_t head_dim_k;         /* Dk */
    int32_t head_dim_v;         /* Dv */
    int32_t block_size;         /* bs, tokens per block (grouped kernel: a multiple of 16, <= 128; latent: 64;
                                   the E4M3 tensor-core kernel: 16, 32, 64 or 128) */
    int32_t num_blocks;         /* blocks in the pool (block 0 = null block) */
    int32_t max_blocks_per_seq; /* block_table columns */
    int32_t max_context_len;    /* bound on every context_lens entry */
    int32_t q_dtype;            /* PA_F16 or PA_BF16 */
    int32_t kv_dtype;           /* PA_F16, PA_BF16, PA_E4M3, PA_INT8, PA_INT4 */
    int32_t out_dtype;          /* PA_F32, PA_F16, PA_BF16 */
    int32_t k_scale_mode;       /* pa_scale_mode */
    int32_t v_scale_mode;       /* pa_scale_mode (ignored when v_is_k_prefix) */
    int32_t causal;             /* 1: row j sees tokens [0, L_b - next_n + j] */
    int32_t v_is_k_prefix;      /* 1: V = first Dv channels of the K plane */
    int32_t num_sms;            /* SMs to size the launch for; 0 = current device's SM count */
    int32_t grid_ctas;          /* persistent CTAs of pa_run; 0 = num_sms x resident CTAs per SM */
    float softmax_scale;        /* e.g. 1/sqrt(Dk) */
} pa_problem;

/* Byte offsets inside the workspace (all 256-byte aligned) and the launch
 * shape.  Header words (uint32): [0] device error bits, [1] total pages
 * sum_b P_b of the plan, [3] max|k_scale| (fp32 bits).  Request records
 * (int32 x4 per request): {L_b seen by pa_plan, P_b = ceil(L_b / wp) (0 when
 * L_b breaks the contract), PS_b = sum of P over earlier requests, flags},
 * with wp = work_page_tokens: bs, or an equal part of a block when a block
 * is too large for the kernel's shared-memory ring (a "page" below is a work
 * page; the parts of a block are consecutive positions).
 *
 * pa_run orders every page of the batch by logical position -- request,
 * kv head, block of S query rows ("segment"), page -- and gives worker k of
 * the persistent launch (W workers) positions [k*N/W, (k+1)*N/W) of the N in
 * total.  A worker's run of pages inside one segment is a "piece"; a piece
 * that is a whole segment writes `out` directly, other pieces write a partial
 * (normalised output, log-sum-exp) to slot (segment index + k), which
 * pa_combine merges in ascending k.  Partials: fp32 [partial_slots][S][Dv]
 * outputs and fp32 [partial_slots][S] log-sum-exps, row i of a slot = query
 * row S * (row block) + i of the kv head, query row
 * r = j * (Hq / Hkv) + (h mod (Hq / Hkv)).
 *
 * Three kernels: the grouped kernel (separate K and V planes, per-tensor or
 * per-channel scales) has S = 16 and one worker per warp (or pair of warps);
 * the E4M3 tensor-core kernel (E4M3 K and V at Dk = Dv = 256, per-tensor or no
 * scales, 16, 32, 48 or 64 query rows per kv head, bs = 16, 32, 64 or 128) has
 * S = all rows of a kv head, pages of 128 tokens (work_page_tokens = 128,
 * whole blocks) and one worker per CTA (one CTA per SM); the single-latent
 * kernel (v_is_k_prefix: E4M3, PA_SCALE_TOKEN, Dk = 576, Dv = 512, bs = 64)
 * has S = 64 and one worker per CTA (one CTA per SM).  In all three, workers
 * come in groups of G = row_blocks (G = 1 on the E4M3 tensor-core kernel): positions run over
 * (request, kv head, page), the W / G groups share them as above, and worker
 * g*G + i takes row block i of every page of group g's share (the G workers
 * read the same pages at about the same time, so all but the first read hit
 * L2).  The piece of segment (b, kv head u, row block i) in group g has slot
 * (b*Hkv + u + g)*G + i; with one row block (G = 1) this is the rule above. */
typedef struct pa_layout {
    size_t total_bytes;
    size_t header_offset;
    size_t requests_offset;
    size_t partial_o_offset;
    size_t partial_lse_offset;
    int64_t partial_slots;       /* B * Hkv * row_blocks + warps (grouped: (B*Hkv + W/G)*G) */
    int32_t rows_per_kv_head;    /* (Hq / Hkv) * next_n */
    int32_t row_blocks;          /* ceil(rows_per_kv_head / rows_per_segment) */
    int32_t num_sms;             /* effective */
    int32_t grid_ctas;           /* effective persistent CTAs of pa_run */
    int32_t warps;               /* workers W: grid_ctas * 4 (grouped; * 2 with paired warps at D = 256
                                    and more than 8 query rows per kv head) or grid_ctas (latent, E4M3
                                    tensor-core); the launch is sized so that W is a multiple of group_size */
    int32_t ring_pages_per_warp; /* pages each worker keeps in flight (E4M3 tensor-core: K stages) */
    int32_t rows_per_segment;    /* S: 16 (grouped), 64 (latent) or all rows of a kv head (E4M3 tensor-core) */
    int32_t group_size;          /* G = row_blocks: workers sharing one run of pages */
    int32_t work_page_tokens;    /* tokens the attention handles as one page: block_size, or an equal
                                    part of a block (>= 16) when two whole blocks per worker do not fit */
} pa_layout;

/* Library version: major * 10000 + minor * 100 + patch. */
PA_API int pa_version(void);

/* Human-readable name of a status code (static string). */
PA_API const char *pa_status_string(pa_status s);

/* Workspace bytes needed by pa_plan / pa_run / pa_combine for problem *p.
 * Host only; with p->num_sms == 0 it queries the current device. */
PA_API pa_status pa_workspace_size(const pa_problem *p, size_t *bytes);

/* Workspace layout for *p (host only, as pa_workspace_size). */
PA_API pa_status pa_workspace_layout(const pa_problem *p, pa_layout *layout);

/* Plan the work for the current context_lens (device pointer): pages of
 * every request and their prefix sums (request records, header word 1).  With
 * PA_SCALE_CHANNEL K scales, also reduces max|k_scale| over every (kv head,
 * channel) on the device (k_scale: device [Hkv][Dk] fp32); otherwise k_scale
 * may be NULL.  Clears the device error word.  Launches 1-2 kernels. */
PA_API pa_status pa_plan(const pa_problem *p, const int32_t *context_lens, const float *k_scale,
                         void *workspace, size_t workspace_bytes, pa_stream_t stream);

/* The attention itself over the planned pages (see pa_layout for how they
 * are shared out).  Segments handled whole by one warp write `out` (and `lse`
 * if not NULL) directly; the others leave partials in the workspace for
 * pa_combine.  All pointers are device pointers. */
PA_API pa_status pa_run(const pa_problem *p, const void *q, const void *k_pool, const void *v_pool,
                        const int32_t *block_table, const int32_t *context_lens,
                        const float *k_scale, const float *v_scale, void *workspace,
                        size_t workspace_bytes, void *out, float *lse, pa_stream_t stream);

/* Merge the partials of every segment that several warps shared (log-sum-exp,
 * ascending warp order), apply the V scale and write `out` / `lse` for them;
 * write 0 / -inf for requests without pages (NaN for flagged ones).  Segments
 * one warp handled whole are left untouched.  Must follow pa_run with the same
 * problem (its launch shape decides the pieces). */
PA_API pa_status pa_combine(const pa_problem *p, const float *v_scale, void *workspace,
                            size_t workspace_bytes, void *out, float *lse, pa_stream_t stream);

/* pa_plan + pa_run + pa_combine in one call (same arguments). */
PA_API pa_status pa_attention(const pa_problem *p, const void *q, const void *k_pool,
                              const void *v_pool, const int32_t *block_table,
                              const int32_t *context_lens, const float *k_scale,
                              const float *v_scale, void *workspace, size_t workspace_bytes,
                              void *out, float *lse, pa_stream_t stream);

/* pa_attention without a workspace argument, for callers that cannot
 * allocate device memory: for example a plugin whose host application hands
 * it only its input and output buffers and owns every allocation itself.
 * The pages have no counterpart of this call; it exists for such callers.
 *
 * Its scratch is one static device array of 32 MiB that every GPU loading
 * this library reserves until the process exits; problems whose
 * pa_workspace_size exceeds 32 MiB are rejected with PA_ERR_WORKSPACE.  It
 * allocates nothing and calls no allocating routine.  The first call on a
 * device looks up the array's device address (once per device, with that
 * device current) and keeps it for the life of the process: make that first
 * call before any stream capture, and do not call this entry point again on
 * a device after cudaDeviceReset (the kept address would be stale).  All
 * calls share the one array, which keeps the last call's contents, so calls
 * that may overlap on the GPU (other streams, other host threads) race with
 * each other: order them on one stream.  Device error bits land in the shared
 * array and cannot be read back separately; a request that broke the contract
 * still gets NaN rows. */
PA_API pa_status pa_attention_noalloc(const pa_problem *p, const void *q, const void *k_pool,
                                      const void *v_pool, const int32_t *block_table,
                                      const int32_t *context_lens, const float *k_scale,
                                      const float *v_scale, void *out, float *lse,
                                      pa_stream_t stream);

/* Quantized paged KV insert: write the next_n new K / V rows of every
 * request into their pool slots, quantized to the pool's encoding -- the step
 * that precedes the attention of each decode / verify step.
 *
 * Sources (page title, section): CentML/vllm PR #167, "Q pad + KV insert",
 * Design (the per-token quantization and paged insert of the new rows; RoPE
 * and Q padding are not part of this call); onnxruntime PR #32520, "[CUDA]
 * Normalize the PER_CHANNEL K scale folded into Q for paged XQA", Description
 * (symmetric INT8 / INT4 codes with scales max|K| / 127 and max|K| / 7);
 * 1Cat-vLLM PR #647, "Stop grouped-page4 null-block padding from leaking E4M3
 * NaN", Root cause (0x7F / 0xFF are NaN, so finite values saturate at 448).
 *
 * Positions: context_lens already count the new tokens (as for pa_run), so
 * new token j of request b goes to logical position L_b - next_n + j, block
 * block_table[b][pos / bs], slot pos % bs.  Nothing else in the pool is
 * written: other slots of a partial block keep their bytes.
 *
 * Each row x (fp32 values of the source) is stored as codes of x / s, the
 * quotient rounded once in fp32 (IEEE division):
 *   PA_SCALE_NONE     s = 1
 *   PA_SCALE_TENSOR   s = *scale
 *   PA_SCALE_CHANNEL  s = scale[g][d]
 *   PA_SCALE_TOKEN    (E4M3 only) s = max_d |x_d| / 448 computed per row (1
 *                     when it is 0; NaN when the row holds a NaN) and stored
 *                     in the block's per-token scale slot.
 * Codes: f16 / bf16 round to nearest even (overflow gives inf); E4M3 rounds
 * to nearest, ties to even, saturating at +-448 (NaN stays NaN); INT8 / INT4
 * round half to even and clamp to [-127, 127] / [-7, 7] (NaN gives 0), INT4
 * packed two per byte, channel 2i in the low nibble.
 *
 * Arguments (device pointers unless stated):
 *  p            host; uses batch, next_n, num_kv_heads, head_dim_k/v (multiples
 *               of 8, at most 2048), block_size, num_blocks, max_blocks_per_seq,
 *               max_context_len, kv_dtype, k/v_scale_mode, v_is_k_prefix and
 *               num_sms (0 = the current device's); the other fields are not
 *               read.
 *  src_dtype    PA_F32, PA_F16 or PA_BF16: the dtype of k_new / v_new.
 *  k_new        [batch][next_n][Hkv][Dk] new K rows, 16-byte aligned.
 *  v_new        [batch][next_n][Hkv][Dv] new V rows, 16-byte aligned; not
 *               read when v_is_k_prefix (V is then part of the K rows).
 *  block_table, context_lens   as for pa_run.
 *  k_scale, v_scale  per mode: NULL (NONE, TOKEN), 1 fp32 (TENSOR) or
 *               [Hkv][D] fp32, 16-byte aligned (CHANNEL).
 *  k_pool, v_pool  the pool planes (layout as for pa_run), written in place;
 *               v_pool is not written when v_is_k_prefix.
 *  dev_error    optional device uint32 that the kernel ORs error bits into
 *               (read it with pa_get_error(dev_error, ...)); NULL to ignore.
 *
 * Errors: host-detectable problems return a status and launch nothing.  On
 * the device, a request with L_b < next_n, L_b > max_context_len or more
 * pages than table columns is left unwritten (PA_DEV_ERR_CONTEXT_LEN), and a
 * new token whose block id is outside [1, num_blocks) is left unwritten
 * (PA_DEV_ERR_BLOCK_ID).  Requests must not share a block at the positions
 * they write (concurrent writes to one slot race).  One kernel launch on
 * `stream`; no allocation, no synchronisation. */
PA_API pa_status pa_insert(const pa_problem *p, int32_t src_dtype, const void *k_new, const void *v_new,
                           const int32_t *block_table, const int32_t *context_lens, const float *k_scale,
                           const float *v_scale, void *k_pool, void *v_pool, uint32_t *dev_error,
                           pa_stream_t stream);

/* Sparse (selected-token) paged attention: query token j of request b (all
 * its heads) attends only to the logical positions sel[b][j][:] names.
 *
 * Sources (page title, section): 1Cat-vLLM PR #494, "[Bugfix][SM70]
 * Stabilize QSA page4 order under KV relocation", Summary / Contract and
 * limits (sparse attention over per-query selected token ids, work ordered
 * by logical position, bitwise stable under relocation) and Upstream and
 * duplicate-work check (unused selection entries are skipped).
 *
 *   T_bj = { t in sel[b][j][0..top_k) : 0 <= t < vis_bj }   (a set)
 *   out[b,j,h,:] = softmax_{t in T_bj}(softmax_scale * q . k^_t) . v^_t
 * with vis_bj as for pa_run (causal or not); entries < 0 or >= vis_bj are
 * skipped, a position listed twice counts once, and the order of the
 * entries does not matter (the result is bitwise the same).  An empty T_bj
 * gives out = 0, lse = -inf.
 *
 * Arguments as for pa_attention, plus:
 *  top_k      entries per selection row (>= 0).
 *  sel        device [batch][next_n][top_k] int32 logical positions.
 *  workspace  caller-owned device memory of pa_sparse_workspace_size()
 *             bytes, 256-byte aligned: word 0 is the device error word
 *             (read it with pa_get_error), then the per-token counts and the
 *             compacted token lists.
 * Supported: separate K and V planes (not v_is_k_prefix) with Dk = Dv in
 * {64, 128, 256}, Hq / Hkv <= min(16, 2048 / D), per-token scales for E4M3
 * only, max_context_len <= 1.8M (the planner's bitmap: one bit per position,
 * in shared memory); other problems return PA_ERR_UNSUPPORTED.
 * Device errors: a request whose length breaks the contract
 * (PA_DEV_ERR_CONTEXT_LEN) or a selected token whose block id is outside
 * [1, num_blocks) (PA_DEV_ERR_BLOCK_ID) gets NaN rows.  Three stream
 * operations (a 4-byte memset of the error word and two kernels); no
 * allocation, no synchronisation. */
PA_API pa_status pa_sparse_workspace_size(const pa_problem *p, int32_t top_k, size_t *bytes);

PA_API pa_status pa_sparse_attention(const pa_problem *p, int32_t top_k, const int32_t *sel, const void *q,
                                     const void *k_pool, const void *v_pool, const int32_t *block_table,
                                     const int32_t *context_lens, const float *k_scale, const float *v_scale,
                                     void *workspace, size_t workspace_bytes, void *out, float *lse,
                                     pa_stream_t stream);

/* FP4 (MXFP4) paged MQA logits: for every query row r = b * next_n + j and
 * token t of request b, a weighted sum over heads of the FP4 dot products.
 *
 * Source (page title, section): FlashInfer docs,
 * "flashinfer.fp4_paged_mqa_logits", Parameters -- q, sf_q, kv_fused, weights,
 * context_lens, block_table, max_context_len, sf_vec_size,
 * is_kv_sf_interleaved and a preallocated out of at least max_context_len
 * columns.
 *
 *   q^[h, d]  = e2m1(q[b][j][h] value d) * 2^(byte d / 32 of sf_q[b][j][h] - 127)
 *   k^[t, d]  = e2m1(value d of token t % bs in block block_table[b][t / bs])
 *               * 2^(scale byte d / 32 of that token - 127)
 *   logit[r][t] = sum_h weights[r][h] * f(q^[h, :] . k^[t, :])   for t < vis
 *   logit[r][t] = -inf                                  for vis <= t < max_context_len
 * with f the identity, or max(0, .) when rectify = 1 (the page does not print
 * how the heads combine: a plain weighted sum is this library's reading, the
 * rectified sum an option), and vis = L_b, or L_b - (next_n - 1 - j) when
 * causal = 1.  E2M1 is the OCP MX 4-bit float (values 0, 0.5, 1, 1.5, 2, 3,
 * 4, 6 and their negatives); UE8M0 is a power of two 2^(e - 127), 0xFF NaN.
 *
 * Layouts (device pointers):
 *  q         [batch][next_n][num_heads][64] uint8: 128 E2M1 values, value 2i
 *            in the low nibble of byte i; 16-byte aligned.
 *  sf_q      [batch][next_n][num_heads] int32: byte i (little-endian) scales
 *            values 32i .. 32i + 31.
 *  kv_fused  [num_blocks][block_size * 68] uint8: a block is block_size rows
 *            of 64 packed bytes (token order), then block_size 4-byte scale
 *            words, in token order or, with sf_interleaved = 1, word slot k
 *            holding token (k % 4) * (block_size / 4) + k / 4; 16-byte aligned.
 *  weights   [batch * next_n][num_heads] float32.
 *  context_lens [batch] int32 (<= max_context_len); block_table
 *            [batch][max_blocks_per_seq] int32 ids in [1, num_blocks) for the
 *            ceil(L_b / block_size) blocks each request uses (a narrower
 *            requirement than the page's round_up(L_b, 128) / block_size;
 *            columns past a request's blocks are never read).
 *  out       [batch * next_n][out_stride] of out_dtype (f32 / f16 / bf16);
 *            columns 0 .. max_context_len - 1 of every row are written.
 *  workspace caller-owned, pa_fp4_logits_workspace_size() bytes, 256-byte
 *            aligned: word 0 is the device error word (pa_get_error), then
 *            the plan over 128-token tiles and, for the plain weighted sum,
 *            the folded query rows sum_h weights[r][h] * q^[h] (fp32).
 * Supported: head_dim 128, sf_vec_size 32, block_size 16 / 32 / 64 / 128,
 * num_heads a multiple of 16, next_n * num_heads <= 192; other problems
 * return PA_ERR_UNSUPPORTED.  A request whose length breaks the contract
 * (PA_DEV_ERR_CONTEXT_LEN) or a block id outside [1, num_blocks)
 * (PA_DEV_ERR_BLOCK_ID) gets NaN logits; nothing outside the buffers is read
 * or written.  The plain weighted sum (rectify = 0, next_n <= 4) folds the
 * heads into one query vector per row first (the logit is linear in the
 * heads) and runs on the CUDA cores; rectified heads (and next_n > 4) keep
 * the per-head products on the tensor cores.  Three or four kernel launches
 * on `stream`; no allocation, no synchronisation. */
typedef struct pa_fp4_problem {
    int32_t batch;              /* B >= 0 requests */
    int32_t next_n;             /* query rows per request, >= 1 */
    int32_t num_heads;          /* H */
    int32_t head_dim;           /* 128 */
    int32_t sf_vec_size;        /* values per UE8M0 scale: 32 */
    int32_t block_size;         /* tokens per kv_fused block */
    int32_t num_blocks;         /* blocks in the pool (block 0 = null block) */
    int32_t max_blocks_per_seq; /* block_table columns */
    int32_t max_context_len;    /* columns of each output row written; bound on context_lens */
    int32_t out_dtype;          /* PA_F32, PA_F16, PA_BF16 */
    int32_t out_stride;         /* elements between output rows (>= max_context_len; 0 = max_context_len) */
    int32_t causal;             /* 1: row j sees tokens [0, L_b - next_n + j] */
    int32_t rectify;            /* 1: each head's dot product is clamped at 0 before weighting */
    int32_t sf_interleaved;     /* 1: interleaved scale words (see above) */
    int32_t num_sms;            /* SMs to size the launch for; 0 = current device's */
    int32_t grid_ctas;          /* persistent CTAs; 0 = one per SM */
} pa_fp4_problem;

PA_API pa_status pa_fp4_logits_workspace_size(const pa_fp4_problem *p, size_t *bytes);

PA_API pa_status pa_fp4_logits(const pa_fp4_problem *p, const uint8_t *q, const int32_t *sf_q,
                               const uint8_t *kv_fused, const float *weights, const int32_t *context_lens,
                               const int32_t *block_table, void *workspace, size_t workspace_bytes,
                               void *out, pa_stream_t stream);

/* Copy the device error word to *bits.  Synchronises `stream`. */
PA_API pa_status pa_get_error(const void *workspace, uint32_t *bits, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
