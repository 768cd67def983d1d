/*
 * Paged decode/verify attention over a quantized paged KV cache -- CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow definition that the
 * CUDA library is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.  It
 * shares no header, table or helper with the CUDA sources.
 *
 * What it computes (exact attention, evaluated in double precision):
 *
 *   For request b, query row j in [0, n) and query head h, with kv head
 *   g = h / (Hq / Hkv):
 *     vis      = L_b - (n - 1 - j)  if causal   (row j sits at logical position
 *                                               L_b - n + j and sees tokens up to it)
 *              = L_b                otherwise
 *     for t in [0, vis):
 *        blk   = block_table[b][t / bs],  slot = t % bs
 *        k^[d] = dec(Kcode[blk, g, slot, d]) * ks(g, d, blk, slot)
 *        v^[d] = dec(Vcode[blk, g, slot, d]) * vs(g, d, blk, slot)
 *        s_t   = softmax_scale * sum_d q[b, j, h, d] * k^[d]
 *     M = max_t s_t,  p_t = exp(s_t - M)
 *     out[d] = sum_t p_t v^[d] / sum_t p_t,    lse = M + ln(sum_t p_t)
 *     vis <= 0  ->  out = 0, lse = -inf.
 *
 * Sources (page title, section):
 *  - FlashInfer docs, "flashinfer.fp4_paged_mqa_logits", Parameters
 *    (block_table / context_lens / next_n): the logical-token walk through the
 *    block table; token t of request b lives in block block_table[b][t / bs],
 *    slot t % bs; entries past the request's pages are never used.
 *  - 1Cat-vLLM PR #647 "[Bugfix][SM70] Stop grouped-page4 null-block padding from
 *    leaking E4M3 NaN", Root cause: E4M3 bytes 0x7F / 0xFF are NaN; block 0 is a
 *    null block that must not contribute.  The oracle only ever touches slots
 *    t < vis, so padding and the null block are never read.
 *  - onnxruntime PR #32520 "[CUDA] Normalize the PER_CHANNEL K scale folded into Q
 *    for paged XQA", Description / Approach: INT8 / INT4 / FP8 codes with a
 *    per-tensor scalar or per-(kv head, channel) scale, k^ = code * scale.  The
 *    oracle applies scales to the codes directly; it does NOT fold them into q
 *    (folding is a GPU-side reorganisation of the same product).
 *  - 1Cat-vLLM PR #494 "[Bugfix][SM70] Stabilize QSA page4 order under KV
 *    relocation", Numerical follow-up: "CPU FP64 dot products" as the reference
 *    method.  The oracle's summation order is the logical token order, so its
 *    result is bitwise independent of the physical block ids.
 *
 * Readings where the pages are silent:
 *  - pool layout: head-major [num_blocks][Hkv][bs][row_bytes]; with per-token
 *    scales every block is [Hkv][bs][row_bytes] codes followed by [Hkv][bs] fp32
 *    scales (the FlashInfer page's "data region, then scale-factor region");
 *  - INT4: two's-complement nibbles, channel 2i in the low nibble of byte i;
 *  - INT8: two's complement, no zero point;
 *  - next_n causal alignment as written above;
 *  - with v_is_k_prefix, V is the first Dv channels of the K plane and shares
 *    K's scales.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Element encodings understood by the oracle (numbered independently of any
 * other component; the Python wrapper maps names to these). */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_INT8 = 3, ORC_INT4 = 4 };
/* Scale modes. */
enum { ORC_SCALE_NONE = 0, ORC_SCALE_TENSOR = 1, ORC_SCALE_CHANNEL = 2, ORC_SCALE_TOKEN = 3 };

/* Status codes. */
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_BLOCK = 2, ORC_NO_MEM = 3 };

typedef struct {
    int32_t B, n, Hq, Hkv, Dk, Dv, bs, num_blocks, max_blocks_per_seq;
    int32_t q_dtype, kv_dtype;
    int32_t k_scale_mode, v_scale_mode;
    int32_t v_is_k_prefix;
    int32_t causal;
    double softmax_scale;
} orc_problem;

/* ---------------------------------------------------------------- decoding */

/* FP8 E4M3 ("fn" variant used by KV caches): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits, subnormals when the exponent field is 0, no
 * infinities, and the two patterns S.1111.111 (0x7F, 0xFF) are NaN. */
double orc_e4m3_value(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

void orc_e4m3_table(double out[256]) {
    for (int c = 0; c < 256; ++c) out[c] = orc_e4m3_value((uint8_t)c);
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double orc_f16_value(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0x1F) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);
    else v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent with
 * bias 127, 7 mantissa bits). */
double orc_bf16_value(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int m = b & 0x7F;
    double v;
    if (e == 0xFF) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -126 - 7);
    else v = ldexp(1.0 + (double)m / 128.0, e - 127);
    return sign ? -v : v;
}

double orc_int4_value(uint8_t byte, int high) {
    int nib = high ? (byte >> 4) & 0xF : byte & 0xF;
    return (double)(nib >= 8 ? nib - 16 : nib);
}

int orc_bits(int dtype) {
    switch (dtype) {
        case ORC_F16: case ORC_BF16: return 16;
        case ORC_E4M3: case ORC_INT8: return 8;
        case ORC_INT4: return 4;
        default: return -1;
    }
}

static double g_e4m3[256];

/* Value of channel d of a row of codes stored at `row`. */
static double decode_elem(int dtype, const uint8_t *row, int d) {
    switch (dtype) {
        case ORC_F16: { uint16_t h; memcpy(&h, row + 2 * (size_t)d, 2); return orc_f16_value(h); }
        case ORC_BF16: { uint16_t h; memcpy(&h, row + 2 * (size_t)d, 2); return orc_bf16_value(h); }
        case ORC_E4M3: return g_e4m3[row[d]];
        case ORC_INT8: return (double)(int8_t)row[d];
        case ORC_INT4: return orc_int4_value(row[d / 2], d & 1);
        default: return NAN;
    }
}

/* Bytes of one pool block, and where (g, slot)'s codes and per-token scale sit
 * inside it. */
static size_t row_bytes_of(int dtype, int D) { return (size_t)D * (size_t)orc_bits(dtype) / 8; }

static size_t block_bytes_of(const orc_problem *p, int D, int token_scaled) {
    size_t codes = (size_t)p->Hkv * p->bs * row_bytes_of(p->kv_dtype, D);
    return codes + (token_scaled ? (size_t)p->Hkv * p->bs * 4 : 0);
}

typedef struct {
    const orc_problem *p;
    const uint8_t *q;
    const uint8_t *k_pool, *v_pool;
    const int32_t *block_table, *context_lens;
    const float *k_scale, *v_scale;
    const int32_t *rows; /* num_rows triples (b, j, h) */
    int64_t num_rows;
    double *out, *lse;
    int64_t next_row; /* work counter */
    pthread_mutex_t lock;
    int status;
} orc_job;

static double scale_of(int mode, const float *scale, const uint8_t *blk_base, size_t codes_bytes,
                       int g, int slot, int d, int D, int bs) {
    switch (mode) {
        case ORC_SCALE_NONE: return 1.0;
        case ORC_SCALE_TENSOR: return (double)scale[0];
        case ORC_SCALE_CHANNEL: return (double)scale[(size_t)g * D + d];
        case ORC_SCALE_TOKEN: {
            float s;
            memcpy(&s, blk_base + codes_bytes + ((size_t)g * bs + slot) * 4, 4);
            return (double)s;
        }
        default: return NAN;
    }
}

/* One output row: the definition written out (two passes over the logical
 * tokens: scores and their max, then weights and the weighted sum). */
static int one_row(const orc_job *J, int b, int j, int h, double *out, double *lse, double *s) {
    const orc_problem *p = J->p;
    const int G = p->Hq / p->Hkv;
    const int g = h / G;
    const int L = J->context_lens[b];
    const int vis = p->causal ? L - (p->n - 1 - j) : L;
    const int k_tok = p->k_scale_mode == ORC_SCALE_TOKEN;
    const int v_from_k = p->v_is_k_prefix != 0;
    const int v_mode = v_from_k ? p->k_scale_mode : p->v_scale_mode;
    const int v_tok = v_mode == ORC_SCALE_TOKEN;
    const int Dv_plane = v_from_k ? p->Dk : p->Dv;
    const size_t k_row = row_bytes_of(p->kv_dtype, p->Dk);
    const size_t v_row = row_bytes_of(p->kv_dtype, Dv_plane);
    const size_t k_blk = block_bytes_of(p, p->Dk, k_tok);
    const size_t v_blk = block_bytes_of(p, Dv_plane, v_tok);
    const size_t k_codes = (size_t)p->Hkv * p->bs * k_row;
    const size_t v_codes = (size_t)p->Hkv * p->bs * v_row;
    const uint8_t *vp = v_from_k ? J->k_pool : J->v_pool;
    const float *vsc = v_from_k ? J->k_scale : J->v_scale;

    /* decode the query row exactly */
    const size_t q_elem = 2;
    const uint8_t *qrow = J->q + (((size_t)b * p->n + j) * p->Hq + h) * p->Dk * q_elem;
    double qv[1024];
    if (p->Dk > 1024) return ORC_BAD_ARG;
    for (int d = 0; d < p->Dk; ++d) qv[d] = decode_elem(p->q_dtype, qrow, d);

    if (vis <= 0) {
        for (int d = 0; d < p->Dv; ++d) out[d] = 0.0;
        *lse = -INFINITY;
        return ORC_OK;
    }
    /* pass 1: scores */
    double M = -INFINITY;
    for (int t = 0; t < vis; ++t) {
        int blk = J->block_table[(size_t)b * p->max_blocks_per_seq + t / p->bs];
        int slot = t % p->bs;
        if (blk < 0 || blk >= p->num_blocks) return ORC_BAD_BLOCK;
        const uint8_t *base = J->k_pool + (size_t)blk * k_blk;
        const uint8_t *row = base + ((size_t)g * p->bs + slot) * k_row;
        double acc = 0.0;
        for (int d = 0; d < p->Dk; ++d) {
            double kh = decode_elem(p->kv_dtype, row, d) *
                        scale_of(p->k_scale_mode, J->k_scale, base, k_codes, g, slot, d, p->Dk, p->bs);
            acc += qv[d] * kh;
        }
        s[t] = p->softmax_scale * acc;
        if (s[t] > M) M = s[t];
    }
    /* pass 2: weights and weighted values */
    double denom = 0.0;
    for (int d = 0; d < p->Dv; ++d) out[d] = 0.0;
    for (int t = 0; t < vis; ++t) {
        int blk = J->block_table[(size_t)b * p->max_blocks_per_seq + t / p->bs];
        int slot = t % p->bs;
        const uint8_t *base = vp + (size_t)blk * v_blk;
        const uint8_t *row = base + ((size_t)g * p->bs + slot) * v_row;
        double pt = exp(s[t] - M);
        denom += pt;
        for (int d = 0; d < p->Dv; ++d) {
            double vh = decode_elem(p->kv_dtype, row, d) *
                        scale_of(v_mode, vsc, base, v_codes, g, slot, d, Dv_plane, p->bs);
            out[d] += pt * vh;
        }
    }
    for (int d = 0; d < p->Dv; ++d) out[d] /= denom;
    *lse = M + log(denom);
    return ORC_OK;
}

static void *worker(void *arg) {
    orc_job *J = (orc_job *)arg;
    int maxL = 0;
    for (int b = 0; b < J->p->B; ++b) maxL = J->context_lens[b] > maxL ? J->context_lens[b] : maxL;
    double *s = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    if (!s) {
        pthread_mutex_lock(&J->lock);
        J->status = ORC_NO_MEM;
        pthread_mutex_unlock(&J->lock);
        return NULL;
    }
    for (;;) {
        int64_t r;
        pthread_mutex_lock(&J->lock);
        r = J->next_row++;
        pthread_mutex_unlock(&J->lock);
        if (r >= J->num_rows) break;
        int b = J->rows[3 * r], j = J->rows[3 * r + 1], h = J->rows[3 * r + 2];
        int st = one_row(J, b, j, h, J->out + (size_t)r * J->p->Dv, J->lse + r, s);
        if (st != ORC_OK) {
            pthread_mutex_lock(&J->lock);
            J->status = st;
            pthread_mutex_unlock(&J->lock);
        }
    }
    free(s);
    return NULL;
}

static int check_problem(const orc_problem *p) {
    if (p->B < 0 || p->n < 1 || p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv) return ORC_BAD_ARG;
    if (p->Dk < 1 || p->Dv < 1 || p->bs < 1 || p->num_blocks < 1) return ORC_BAD_ARG;
    if (orc_bits(p->kv_dtype) < 0) return ORC_BAD_ARG;
    if (p->q_dtype != ORC_F16 && p->q_dtype != ORC_BF16) return ORC_BAD_ARG;
    if (p->kv_dtype == ORC_INT4 && ((p->Dk & 1) || (p->Dv & 1))) return ORC_BAD_ARG;
    if (p->v_is_k_prefix && p->Dv > p->Dk) return ORC_BAD_ARG;
    return ORC_OK;
}

/* Evaluate `num_rows` rows given as (b, j, h) triples.  out: [num_rows][Dv],
 * lse: [num_rows].  Returns ORC_OK, or ORC_BAD_BLOCK if a visible token maps
 * to a block id outside [0, num_blocks). */
int orc_attention(const orc_problem *p, const void *q, const void *k_pool, const void *v_pool,
                  const int32_t *block_table, const int32_t *context_lens, const float *k_scale,
                  const float *v_scale, const int32_t *rows, int64_t num_rows, double *out,
                  double *lse, int num_threads) {
    static int table_ready = 0;
    if (!table_ready) {
        orc_e4m3_table(g_e4m3);
        table_ready = 1;
    }
    int st = check_problem(p);
    if (st != ORC_OK) return st;
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.p = p;
    J.q = (const uint8_t *)q;
    J.k_pool = (const uint8_t *)k_pool;
    J.v_pool = (const uint8_t *)v_pool;
    J.block_table = block_table;
    J.context_lens = context_lens;
    J.k_scale = k_scale;
    J.v_scale = v_scale;
    J.rows = rows;
    J.num_rows = num_rows;
    J.out = out;
    J.lse = lse;
    pthread_mutex_init(&J.lock, NULL);
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 512) num_threads = 512;
    pthread_t th[512];
    int started = 0;
    for (int i = 1; i < num_threads; ++i)
        if (pthread_create(&th[started], NULL, worker, &J) == 0) ++started;
    worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    pthread_mutex_destroy(&J.lock);
    return J.status;
}

/* Near-tie analysis of one row, for rows whose softmax is almost one-hot:
 * there the token that wins can change with fp16 rounding of the folded
 * query (onnxruntime PR #32520 page, Validation status).
 *
 * Computes the row's scores s_t exactly, M = max s_t and the gap M - s_(2) to
 * the runner-up (+inf if only one token is visible), and, over the tokens with
 * s_t >= M - delta, the per-channel minimum and maximum of v^.  Any convex
 * combination of those tokens' values lies inside [vmin, vmax]. */
int orc_row_ties(const orc_problem *p, const void *q, const void *k_pool, const void *v_pool,
                 const int32_t *block_table, const int32_t *context_lens, const float *k_scale,
                 const float *v_scale, int b, int j, int h, double delta, double *vmin,
                 double *vmax, double *gap, int32_t *count) {
    static int table_ready = 0;
    if (!table_ready) {
        orc_e4m3_table(g_e4m3);
        table_ready = 1;
    }
    int st = check_problem(p);
    if (st != ORC_OK) return st;
    orc_job J;
    memset(&J, 0, sizeof(J));
    J.p = p;
    J.q = (const uint8_t *)q;
    J.k_pool = (const uint8_t *)k_pool;
    J.v_pool = (const uint8_t *)v_pool;
    J.block_table = block_table;
    J.context_lens = context_lens;
    J.k_scale = k_scale;
    J.v_scale = v_scale;
    const int L = context_lens[b];
    const int vis = p->causal ? L - (p->n - 1 - j) : L;
    *count = 0;
    *gap = INFINITY;
    for (int d = 0; d < p->Dv; ++d) { vmin[d] = INFINITY; vmax[d] = -INFINITY; }
    if (vis <= 0) return ORC_OK;
    double *s = (double *)malloc(sizeof(double) * (size_t)vis);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)p->Dv);
    if (!s || !tmp) { free(s); free(tmp); return ORC_NO_MEM; }
    /* scores via the row evaluator (pass 1 of the definition) */
    double lse;
    st = one_row(&J, b, j, h, tmp, &lse, s);
    if (st != ORC_OK) { free(s); free(tmp); return st; }
    double M = -INFINITY, M2 = -INFINITY;
    for (int t = 0; t < vis; ++t) {
        if (s[t] > M) { M2 = M; M = s[t]; }
        else if (s[t] > M2) M2 = s[t];
    }
    *gap = vis > 1 ? M - M2 : INFINITY;
    /* values of the tokens within delta of the max: run a one-hot weight
     * through the same value walk by evaluating each candidate token alone */
    const int G = p->Hq / p->Hkv;
    const int g = h / G;
    const int v_from_k = p->v_is_k_prefix != 0;
    const int v_mode = v_from_k ? p->k_scale_mode : p->v_scale_mode;
    const int v_tok = v_mode == ORC_SCALE_TOKEN;
    const int Dv_plane = v_from_k ? p->Dk : p->Dv;
    const size_t v_row = row_bytes_of(p->kv_dtype, Dv_plane);
    const size_t v_blk = block_bytes_of(p, Dv_plane, v_tok);
    const size_t v_codes = (size_t)p->Hkv * p->bs * v_row;
    const uint8_t *vp = v_from_k ? J.k_pool : J.v_pool;
    const float *vsc = v_from_k ? k_scale : v_scale;
    for (int t = 0; t < vis; ++t) {
        if (!(s[t] >= M - delta)) continue;
        ++*count;
        int blk = block_table[(size_t)b * p->max_blocks_per_seq + t / p->bs];
        int slot = t % p->bs;
        const uint8_t *base = vp + (size_t)blk * v_blk;
        const uint8_t *row = base + ((size_t)g * p->bs + slot) * v_row;
        for (int d = 0; d < p->Dv; ++d) {
            double vh = decode_elem(p->kv_dtype, row, d) *
                        scale_of(v_mode, vsc, base, v_codes, g, slot, d, Dv_plane, p->bs);
            if (vh < vmin[d]) vmin[d] = vh;
            if (vh > vmax[d]) vmax[d] = vh;
        }
    }
    free(s);
    free(tmp);
    return ORC_OK;
}
