/*
 * Plain CPU oracle for the paged KV cache decode path -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark use
 * this file. It shares no code, header or table with the CUDA library; it is
 * slow on purpose and written so that each step can be checked against the
 * definitions on the pages by eye.
 *
 * Sources (web pages, by title and section):
 *  [P1] "PagedAttention实现" (ainanfeng.cn teaching version), section
 *       "PagedAttention管理器": write_kv (logical position -> page index by
 *       division, offset by remainder, then a copy of the token's values) and
 *       cow_write (whole-block copy of a shared block).
 *  [P2] "CS349E lecture 7: 01_paged_attention.py", demo 2 (paper eq. 4):
 *       scores are formed block by block through the block table, ONE softmax
 *       is taken over the whole context, then V is accumulated block by block;
 *       the result equals attention over the concatenated (contiguous) K/V.
 *  [P3] "04 - Paged Attention 实现进度", section B.2: slot_mapping maps each new
 *       token to a physical slot (block id + offset), block_tables has shape
 *       [batch, max_blocks_per_seq], context_lens is each sequence's length,
 *       cu_seqlens_q (query_start_loc in vLLM's terms, section D.2) packs the
 *       variable-length query chunks of a prefill step.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - slot = physical_block * block_size + offset; slot -1 means "skip".
 *  - the query head h reads kv head h / (num_heads / num_kv_heads).
 *  - context length 0 gives an all-zero output row.
 *  - the cache layout is [num_blocks, block_size, num_kv_heads, head_dim].
 *
 * Arithmetic is float64. Cache and query elements are read in their storage
 * type (fp32, fp16, bf16 or fp64) and widened exactly to double.
 *
 * 8-bit cache (not on the pages; the design notes state the reading): the
 * cache may hold OCP FP8 E4M3 codes (OCP 8-bit Floating Point Specification,
 * "E4M3": sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * S.1111.111 = NaN, largest finite 448). A cache element stands for
 * decoded(code) * scale, with one float32 scale for all of K and one for all
 * of V. Writing divides the token's value by the scale in float32 and rounds
 * the quotient to the nearest code (ties to even mantissa), magnitudes from
 * 448 up (infinities included) saturating to 448.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_F64 = 3, OR_E4M3 = 4 };

enum {
    OR_OK = 0,
    OR_ERR_ARG = -1,
    OR_ERR_BLOCK_ID = -2,   /* a live logical block maps outside the pool */
    OR_ERR_CONTEXT = -3,    /* context longer than the table can describe */
    OR_ERR_NOMEM = -4
};

static int elem_bytes(int dtype)
{
    switch (dtype) {
    case OR_F32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_F64: return 8;
    case OR_E4M3: return 1;
    default: return 0;
    }
}

/* OCP FP8 E4M3 -> double, from the format's definition: exponent field 0 holds
 * the subnormals (m / 8) * 2^-6; otherwise (1 + m / 8) * 2^(e - 7); the
 * pattern with all exponent and mantissa bits set is NaN (no infinities). */
static double e4m3_bits_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* m * 2^-3 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);    /* (8 + m) * 2^-3 * 2^(e-7) */
    return sign ? -v : v;
}

double oracle_e4m3_to_double(uint8_t c) { return e4m3_bits_to_double(c); }

/* Nearest E4M3 code to x. The non-negative finite codes 0x00..0x7E are in
 * increasing order of magnitude, so |x| belongs to code c when it lies between
 * the midpoints of c with its two neighbours. Midpoints of codes are exact in
 * double and so is |x|, so every comparison is exact. On a midpoint the code
 * with the even mantissa (the even code) wins. |x| >= 448 (and infinity)
 * saturates to 448; NaN gives 0x7F; the sign bit is x's, also for results that
 * round to zero. */
uint8_t oracle_e4m3_from_float(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int c = 0;
    while (c < 0x7E) {
        double mid = 0.5 * (e4m3_bits_to_double((uint8_t)c) + e4m3_bits_to_double((uint8_t)(c + 1)));
        if (a < mid || (a == mid && (c & 1) == 0))
            break;
        ++c;
    }
    return (uint8_t)(sign | c);
}

/* IEEE-754 binary16 -> double, from the format's definition. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    double v;
    if (exp == 0)
        v = ldexp((double)man, -24);                 /* subnormal: man * 2^-14 / 2^10 */
    else if (exp == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man | 0x400), exp - 25);  /* (1024 + man) * 2^(exp-15-10) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of a binary32. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, int64_t i, int dtype)
{
    switch (dtype) {
    case OR_F32: return (double)((const float *)base)[i];
    case OR_F16: return half_bits_to_double(((const uint16_t *)base)[i]);
    case OR_BF16: return bf16_bits_to_double(((const uint16_t *)base)[i]);
    case OR_E4M3: return e4m3_bits_to_double(((const uint8_t *)base)[i]);
    default: return ((const double *)base)[i];
    }
}

/* ------------------------------------------------------------------------
 * Scatter of new tokens' K and V rows into cache slots  [P1 write_kv; P3 B.2]
 *
 * k, v:        [num_tokens, row_elems]   (row_elems = num_kv_heads * head_dim)
 * caches:      [num_blocks, block_size, row_elems]
 * Token t goes to block slot_mapping[t] / block_size, offset
 * slot_mapping[t] % block_size. Slot -1 is skipped. Any other slot outside
 * [0, num_blocks * block_size) is skipped and counted.
 * Returns the number of invalid slots, or OR_ERR_ARG.
 * ---------------------------------------------------------------------- */
int64_t oracle_kv_write(const void *k, const void *v, const int32_t *slot_mapping,
                        int64_t num_tokens, void *key_cache, void *value_cache,
                        int64_t num_blocks, int block_size, int64_t row_elems, int dtype)
{
    int es = elem_bytes(dtype);
    if (es == 0 || block_size <= 0 || row_elems <= 0 || num_tokens < 0 || num_blocks < 0)
        return OR_ERR_ARG;
    int64_t row_bytes = row_elems * es;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot == -1)
            continue;
        if (slot < 0 || slot >= num_blocks * (int64_t)block_size) {
            bad++;
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        int64_t dst = (block * block_size + offset) * row_bytes;
        memcpy((char *)key_cache + dst, (const char *)k + t * row_bytes, (size_t)row_bytes);
        memcpy((char *)value_cache + dst, (const char *)v + t * row_bytes, (size_t)row_bytes);
    }
    return bad;
}

/* ------------------------------------------------------------------------
 * Scatter into an 8-bit E4M3 cache  [P1 write_kv; P3 B.2 for the slots; the
 * encoding is this project's reading, see the file header]
 *
 * Same slots and layout as oracle_kv_write; each element x of k (v) is stored
 * as the E4M3 code nearest to the float32 quotient x / k_scale (x / v_scale).
 * k and v hold fp32, fp16 or bf16 values (all exact in float32).
 * Returns the number of invalid slots skipped, or OR_ERR_ARG.
 * ---------------------------------------------------------------------- */
int64_t oracle_kv_write_fp8(const void *k, const void *v, int src_dtype, const int32_t *slot_mapping,
                            int64_t num_tokens, uint8_t *key_cache, uint8_t *value_cache,
                            int64_t num_blocks, int block_size, int64_t row_elems, float k_scale,
                            float v_scale)
{
    if ((src_dtype != OR_F32 && src_dtype != OR_F16 && src_dtype != OR_BF16) || block_size <= 0 ||
        row_elems <= 0 || num_tokens < 0 || num_blocks < 0 || !(k_scale > 0.0f) || !(v_scale > 0.0f) ||
        isinf(k_scale) || isinf(v_scale))
        return OR_ERR_ARG;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot == -1)
            continue;
        if (slot < 0 || slot >= num_blocks * (int64_t)block_size) {
            bad++;
            continue;
        }
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        int64_t dst = (block * block_size + offset) * row_elems;
        for (int64_t i = 0; i < row_elems; ++i) {
            float xk = (float)load_elem(k, t * row_elems + i, src_dtype);
            float xv = (float)load_elem(v, t * row_elems + i, src_dtype);
            float qk = xk / k_scale;           /* float32 division, rounded to nearest */
            float qv = xv / v_scale;
            key_cache[dst + i] = oracle_e4m3_from_float(qk);
            value_cache[dst + i] = oracle_e4m3_from_float(qv);
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------
 * Whole-block copy for copy-on-write  [P1 cow_write: the block's full contents
 * are duplicated into a fresh block before the write]
 *
 * pairs: [num_pairs, 2] = (src, dst). block_elems = block_size * row_elems.
 * Pairs with an id outside [0, num_blocks) are skipped and counted.
 * Returns the number of invalid pairs, or OR_ERR_ARG.
 * ---------------------------------------------------------------------- */
int64_t oracle_copy_blocks(void *key_cache, void *value_cache, const int32_t *pairs,
                           int64_t num_pairs, int64_t num_blocks, int64_t block_elems, int dtype)
{
    int es = elem_bytes(dtype);
    if (es == 0 || block_elems <= 0 || num_pairs < 0)
        return OR_ERR_ARG;
    int64_t bb = block_elems * es;
    int64_t bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            bad++;
            continue;
        }
        memcpy((char *)key_cache + dst * bb, (const char *)key_cache + src * bb, (size_t)bb);
        memcpy((char *)value_cache + dst * bb, (const char *)value_cache + src * bb, (size_t)bb);
    }
    return bad;
}

/* ------------------------------------------------------------------------
 * Decode attention over a paged cache  [P2 demo 2, eq. 4; P3 B.2]
 *
 * For sequence b and query head h (kv head h / G, G = num_heads/num_kv_heads):
 *   1. gather K, V of positions 0..ctx-1 through block_tables[b] into
 *      contiguous arrays (position t lives in physical block
 *      block_tables[b][t / block_size] at offset t % block_size);
 *   2. s[t] = scale * sum_d q[b,h,d] * K[t,d];
 *   3. one softmax over all ctx scores: p[t] = exp(s[t] - max s) / sum;
 *   4. out[b,h,d] = sum_t p[t] * V[t,d]   (t in position order).
 * ---------------------------------------------------------------------- */
typedef struct {
    double *out;
    double *weights;          /* optional [ctx] of one (b, h) */
    int weights_b, weights_h;
    const void *q;
    int q_dtype;
    const void *key_cache, *value_cache;
    int cache_dtype;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size;
    int64_t num_blocks;
    double scale;
    double k_scale, v_scale;  /* cache element = stored value * scale (1 unless E4M3) */
    int64_t next_item;        /* work counter over (b, kv head) */
    int status;
} attn_job;

static int attend_one(attn_job *J, int b, int kvh, double *Kc, double *Vc, double *s)
{
    const int D = J->head_dim, Hk = J->num_kv_heads, bs = J->block_size;
    const int G = J->num_heads / Hk;
    const int ctx = J->context_lens[b];
    const int64_t row = (int64_t)Hk * D;

    /* step 1: gather through the block table */
    for (int t = 0; t < ctx; ++t) {
        int32_t phys = J->block_tables[(int64_t)b * J->max_blocks_per_seq + t / bs];
        if (phys < 0 || phys >= J->num_blocks)
            return OR_ERR_BLOCK_ID;
        int64_t base = ((int64_t)phys * bs + t % bs) * row + (int64_t)kvh * D;
        for (int d = 0; d < D; ++d) {
            Kc[(int64_t)t * D + d] = load_elem(J->key_cache, base + d, J->cache_dtype) * J->k_scale;
            Vc[(int64_t)t * D + d] = load_elem(J->value_cache, base + d, J->cache_dtype) * J->v_scale;
        }
    }
    for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;
        double *o = J->out + ((int64_t)b * J->num_heads + h) * D;
        if (ctx == 0) {
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            continue;
        }
        const int64_t qbase = ((int64_t)b * J->num_heads + h) * D;
        /* step 2: scores */
        for (int t = 0; t < ctx; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += load_elem(J->q, qbase + d, J->q_dtype) * Kc[(int64_t)t * D + d];
            s[t] = J->scale * acc;
        }
        /* step 3: one softmax over the whole context */
        double m = s[0];
        for (int t = 1; t < ctx; ++t)
            if (s[t] > m)
                m = s[t];
        double l = 0.0;
        for (int t = 0; t < ctx; ++t) {
            s[t] = exp(s[t] - m);
            l += s[t];
        }
        for (int t = 0; t < ctx; ++t)
            s[t] = s[t] / l;
        if (J->weights && b == J->weights_b && h == J->weights_h)
            memcpy(J->weights, s, sizeof(double) * (size_t)ctx);
        /* step 4: weighted sum of V */
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int t = 0; t < ctx; ++t)
                acc += s[t] * Vc[(int64_t)t * D + d];
            o[d] = acc;
        }
    }
    return OR_OK;
}

static void *attn_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    int max_ctx = 0;
    for (int b = 0; b < J->num_seqs; ++b)
        if (J->context_lens[b] > max_ctx)
            max_ctx = J->context_lens[b];
    size_t n = (size_t)(max_ctx > 0 ? max_ctx : 1);
    double *Kc = malloc(sizeof(double) * n * (size_t)J->head_dim);
    double *Vc = malloc(sizeof(double) * n * (size_t)J->head_dim);
    double *s = malloc(sizeof(double) * n);
    if (!Kc || !Vc || !s) {
        __atomic_store_n(&J->status, OR_ERR_NOMEM, __ATOMIC_RELAXED);
        free(Kc); free(Vc); free(s);
        return NULL;
    }
    const int64_t items = (int64_t)J->num_seqs * J->num_kv_heads;
    for (;;) {
        int64_t it = __atomic_fetch_add(&J->next_item, 1, __ATOMIC_RELAXED);
        if (it >= items)
            break;
        int rc = attend_one(J, (int)(it / J->num_kv_heads), (int)(it % J->num_kv_heads), Kc, Vc, s);
        if (rc != OR_OK)
            __atomic_store_n(&J->status, rc, __ATOMIC_RELAXED);
    }
    free(Kc); free(Vc); free(s);
    return NULL;
}

static int run_attention(attn_job *J, int num_threads)
{
    if (J->num_seqs < 0 || J->num_heads <= 0 || J->num_kv_heads <= 0 || J->head_dim <= 0 ||
        J->block_size <= 0 || J->num_heads % J->num_kv_heads != 0 ||
        elem_bytes(J->cache_dtype) == 0 || elem_bytes(J->q_dtype) == 0)
        return OR_ERR_ARG;
    for (int b = 0; b < J->num_seqs; ++b) {
        int ctx = J->context_lens[b];
        if (ctx < 0)
            return OR_ERR_ARG;
        if ((int64_t)ctx > (int64_t)J->max_blocks_per_seq * J->block_size)
            return OR_ERR_CONTEXT;
    }
    if (num_threads < 1)
        num_threads = 1;
    if (num_threads > 256)
        num_threads = 256;
    J->next_item = 0;
    J->status = OR_OK;
    pthread_t tid[256];
    int started = 0;
    for (int i = 1; i < num_threads; ++i) {
        if (pthread_create(&tid[started], NULL, attn_worker, J) == 0)
            started++;
    }
    attn_worker(J);
    for (int i = 0; i < started; ++i)
        pthread_join(tid[i], NULL);
    return J->status;
}

int oracle_paged_attention(double *out, const void *q, int q_dtype,
                           const void *key_cache, const void *value_cache, int cache_dtype,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           double scale, int num_threads)
{
    attn_job J;
    memset(&J, 0, sizeof J);
    J.out = out; J.q = q; J.q_dtype = q_dtype;
    J.key_cache = key_cache; J.value_cache = value_cache; J.cache_dtype = cache_dtype;
    J.block_tables = block_tables; J.max_blocks_per_seq = max_blocks_per_seq;
    J.context_lens = context_lens; J.num_seqs = num_seqs; J.num_heads = num_heads;
    J.num_kv_heads = num_kv_heads; J.head_dim = head_dim; J.block_size = block_size;
    J.num_blocks = num_blocks; J.scale = scale; J.weights = NULL;
    J.weights_b = -1; J.weights_h = -1;
    J.k_scale = 1.0; J.v_scale = 1.0;
    return run_attention(&J, num_threads);
}

/* Decode attention over an E4M3 cache: the same four steps, each cache element
 * read as decoded(code) * k_scale for K and decoded(code) * v_scale for V (the
 * product is exact in double). */
int oracle_paged_attention_fp8(double *out, const void *q, int q_dtype, const uint8_t *key_cache,
                               const uint8_t *value_cache, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                               int num_heads, int num_kv_heads, int head_dim, int block_size,
                               int64_t num_blocks, double scale, float k_scale, float v_scale,
                               int num_threads)
{
    attn_job J;
    memset(&J, 0, sizeof J);
    J.out = out; J.q = q; J.q_dtype = q_dtype;
    J.key_cache = key_cache; J.value_cache = value_cache; J.cache_dtype = OR_E4M3;
    J.block_tables = block_tables; J.max_blocks_per_seq = max_blocks_per_seq;
    J.context_lens = context_lens; J.num_seqs = num_seqs; J.num_heads = num_heads;
    J.num_kv_heads = num_kv_heads; J.head_dim = head_dim; J.block_size = block_size;
    J.num_blocks = num_blocks; J.scale = scale; J.weights = NULL;
    J.weights_b = -1; J.weights_h = -1;
    J.k_scale = (double)k_scale; J.v_scale = (double)v_scale;
    return run_attention(&J, num_threads);
}

/* The softmax weights p[0..ctx) of one (sequence b, query head h), together
 * with the full output (single thread). */
int oracle_attention_weights(double *weights, double *out, const void *q, int q_dtype,
                             const void *key_cache, const void *value_cache, int cache_dtype,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, int num_seqs, int num_heads,
                             int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                             double scale, int b, int h)
{
    attn_job J;
    memset(&J, 0, sizeof J);
    J.out = out; J.q = q; J.q_dtype = q_dtype;
    J.key_cache = key_cache; J.value_cache = value_cache; J.cache_dtype = cache_dtype;
    J.block_tables = block_tables; J.max_blocks_per_seq = max_blocks_per_seq;
    J.context_lens = context_lens; J.num_seqs = num_seqs; J.num_heads = num_heads;
    J.num_kv_heads = num_kv_heads; J.head_dim = head_dim; J.block_size = block_size;
    J.num_blocks = num_blocks; J.scale = scale;
    J.k_scale = 1.0; J.v_scale = 1.0;
    J.weights = weights; J.weights_b = b; J.weights_h = h;
    return run_attention(&J, 1);
}

/* ------------------------------------------------------------------------
 * Chunked-prefill attention over a paged cache  [P2 demo 1 and demo 2: a
 * paged step first writes the chunk's K/V, then every position of the chunk
 * attends; P3 B.2: cu_seqlens_q packs the chunks]
 *
 * Sequence b owns query rows query_start_loc[b] .. query_start_loc[b+1]-1
 * (q_len_b rows). Its context holds context_lens[b] tokens, the chunk being the
 * last q_len_b of them, so query row i sits at position
 * pos = context_lens[b] - q_len_b + i and sees positions 0..pos (causal). For
 * each query head h (kv head h / G): gather K, V of positions 0..pos through the
 * block table, s[t] = scale * q . K[t], p = softmax(s), out = sum_t p[t] V[t].
 * q, out: [total_q, num_heads, head_dim].
 * ---------------------------------------------------------------------- */
typedef struct {
    double *out;
    const void *q;
    int dtype;
    const void *key_cache, *value_cache;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    const int32_t *context_lens, *query_start_loc;
    int num_seqs, num_heads, num_kv_heads, head_dim, block_size;
    int64_t num_blocks;
    double scale;
    int64_t next_item;
    int status;
} prefill_job;

static void *prefill_worker(void *arg)
{
    prefill_job *J = (prefill_job *)arg;
    const int D = J->head_dim, Hk = J->num_kv_heads, bs = J->block_size, H = J->num_heads;
    const int G = H / Hk;
    const int64_t row = (int64_t)Hk * D;
    int max_ctx = 1;
    for (int b = 0; b < J->num_seqs; ++b)
        if (J->context_lens[b] > max_ctx)
            max_ctx = J->context_lens[b];
    double *Kc = malloc(sizeof(double) * (size_t)max_ctx * (size_t)D);
    double *Vc = malloc(sizeof(double) * (size_t)max_ctx * (size_t)D);
    double *s = malloc(sizeof(double) * (size_t)max_ctx);
    if (!Kc || !Vc || !s) {
        __atomic_store_n(&J->status, OR_ERR_NOMEM, __ATOMIC_RELAXED);
        free(Kc); free(Vc); free(s);
        return NULL;
    }
    const int64_t items = (int64_t)J->num_seqs * Hk;
    for (;;) {
        int64_t it = __atomic_fetch_add(&J->next_item, 1, __ATOMIC_RELAXED);
        if (it >= items)
            break;
        const int b = (int)(it / Hk), kvh = (int)(it % Hk);
        const int ctx = J->context_lens[b];
        const int q0 = J->query_start_loc[b], q_len = J->query_start_loc[b + 1] - q0;
        int bad = 0;
        /* gather the whole context once; each query uses a prefix of it */
        for (int t = 0; t < ctx && !bad; ++t) {
            int32_t phys = J->block_tables[(int64_t)b * J->max_blocks_per_seq + t / bs];
            if (phys < 0 || phys >= J->num_blocks) {
                bad = 1;
                break;
            }
            int64_t base = ((int64_t)phys * bs + t % bs) * row + (int64_t)kvh * D;
            for (int d = 0; d < D; ++d) {
                Kc[(int64_t)t * D + d] = load_elem(J->key_cache, base + d, J->dtype);
                Vc[(int64_t)t * D + d] = load_elem(J->value_cache, base + d, J->dtype);
            }
        }
        if (bad) {
            __atomic_store_n(&J->status, OR_ERR_BLOCK_ID, __ATOMIC_RELAXED);
            continue;
        }
        for (int i = 0; i < q_len; ++i) {
            const int n = ctx - q_len + i + 1;            /* positions 0..pos */
            for (int g = 0; g < G; ++g) {
                const int h = kvh * G + g;
                const int64_t qbase = ((int64_t)(q0 + i) * H + h) * D;
                double *o = J->out + qbase;
                for (int t = 0; t < n; ++t) {
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d)
                        acc += load_elem(J->q, qbase + d, J->dtype) * Kc[(int64_t)t * D + d];
                    s[t] = J->scale * acc;
                }
                double m = s[0];
                for (int t = 1; t < n; ++t)
                    if (s[t] > m)
                        m = s[t];
                double l = 0.0;
                for (int t = 0; t < n; ++t) {
                    s[t] = exp(s[t] - m);
                    l += s[t];
                }
                for (int t = 0; t < n; ++t)
                    s[t] = s[t] / l;
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int t = 0; t < n; ++t)
                        acc += s[t] * Vc[(int64_t)t * D + d];
                    o[d] = acc;
                }
            }
        }
    }
    free(Kc); free(Vc); free(s);
    return NULL;
}

int oracle_paged_prefill(double *out, const void *q, const void *key_cache, const void *value_cache,
                         int dtype, const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, const int32_t *query_start_loc, int num_seqs,
                         int num_heads, int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, double scale, int num_threads)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_heads % num_kv_heads != 0 || elem_bytes(dtype) == 0)
        return OR_ERR_ARG;
    for (int b = 0; b < num_seqs; ++b) {
        const int q_len = query_start_loc[b + 1] - query_start_loc[b];
        if (q_len < 0 || context_lens[b] < q_len)
            return OR_ERR_ARG;
        if ((int64_t)context_lens[b] > (int64_t)max_blocks_per_seq * block_size)
            return OR_ERR_CONTEXT;
    }
    prefill_job J;
    memset(&J, 0, sizeof J);
    J.out = out; J.q = q; J.dtype = dtype; J.key_cache = key_cache; J.value_cache = value_cache;
    J.block_tables = block_tables; J.max_blocks_per_seq = max_blocks_per_seq;
    J.context_lens = context_lens; J.query_start_loc = query_start_loc; J.num_seqs = num_seqs;
    J.num_heads = num_heads; J.num_kv_heads = num_kv_heads; J.head_dim = head_dim;
    J.block_size = block_size; J.num_blocks = num_blocks; J.scale = scale;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 256) num_threads = 256;
    pthread_t tid[256];
    int started = 0;
    for (int i = 1; i < num_threads; ++i)
        if (pthread_create(&tid[started], NULL, prefill_worker, &J) == 0)
            started++;
    prefill_worker(&J);
    for (int i = 0; i < started; ++i)
        pthread_join(tid[i], NULL);
    return J.status;
}
