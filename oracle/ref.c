/*
 * Oracle for attention over a paged (block-table) KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links
 * or calls this file; only the tests, the package's smoke check and the
 * bench's CPU-baseline leg do.  It shares no code, header, table or constant
 * with the CUDA path.
 *
 * Plain, slow, obviously correct: every floating-point step is done in
 * double precision on bf16-valued inputs (bf16 -> double is exact), with no
 * tiling, fusion or reordering beyond the definitions below.
 *
 * Sources (page title, section):
 *  - "手搓 vLLM 推理引擎" (LLM-101-CN nano-vllm walkthrough), Step 4
 *    "Triton Kernel：写入 KV Cache": a token whose slot is -1 is skipped,
 *    otherwise its num_kv_heads*head_dim K and V values are copied to
 *    cache row `slot`.
 *  - same page, Step 5 "prepare_prefill()" / "prepare_decode()": the new
 *    tokens of a sequence are positions [num_cached, len); their slots are
 *    block_table[pos / block_size] * block_size + pos % block_size (the
 *    decode form, block_table[-1]*bs + last_block_num_tokens - 1, is the same
 *    formula at pos = len - 1).
 *  - "mini-infer系统实战-03-向量化 KV Gather", sections 2.2-2.3: the physical
 *    block of logical position pos is block_table[pos // block_size] and the
 *    row inside it is pos % block_size; the gathered rows form dense K/V.
 *  - "推理系统" (CS 与 LLM 学习知识库), the KV-cache toy: new tokens sit at
 *    the end, new token i (of T) sees the first S - T + i + 1 keys (a lower
 *    triangular mask shifted by S - T), scores are q.k * scale, softmax over
 *    the visible keys, output is the probability-weighted sum of V.
 *  - "面试问答准备: nano-vLLM 推理引擎优化", Q1: the causal bound of a query
 *    at absolute position p is context_len = p + 1.
 *  - "vLLM / SGLang 面试源码深挖", section 4 (KV block fork): a child that
 *    appends into a shared, mutable block gets a new block holding a copy of
 *    the shared block's valid KV.
 *  - "面试问答准备: nano-vLLM 推理引擎优化", Q3 (INT8 KV): per (token, KV
 *    head) symmetric quantisation of the head_dim values: scale =
 *    max(max|x| / 127, 1e-8), code = x / scale rounded half away from zero
 *    (add +-0.5, truncate toward zero), scale kept as fp16; dequantised value
 *    = code * scale.  Computed in fp32 as the page's kernel does, so the codes
 *    (an integer decision) are taken in the same precision as on the GPU.
 *  - Grouped-query attention: query head h reads KV head h / (Hq / Hkv)
 *    (contiguous groups; the pages do not state the mapping, this is the
 *    plainest reading and reduces to multi-head attention when Hq == Hkv).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * fp32 -> IEEE binary16, round to nearest, ties to even, written from the
 * format's definition (1 sign, 5 exponent bits biased by 15, 10 fraction bits;
 * subnormals below 2^-14, infinities above 65504).
 */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    const uint32_t sign = (x >> 16) & 0x8000u;
    const int32_t exp = (int32_t)((x >> 23) & 0xffu);
    uint32_t man = x & 0x7fffffu;
    if (exp == 0xff)
        return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0u));
    const int32_t e = exp - 127 + 15; /* biased binary16 exponent */
    if (e >= 31)
        return (uint16_t)(sign | 0x7c00u);
    if (e <= 0) { /* binary16 subnormal (or zero) */
        if (e < -10)
            return (uint16_t)sign; /* below half the smallest subnormal */
        man |= 0x800000u;          /* explicit leading one */
        const uint32_t shift = (uint32_t)(14 - e);
        uint32_t h = man >> shift;
        const uint32_t rem = man & ((1u << shift) - 1u), half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (h & 1u)))
            ++h; /* may carry into the exponent field: still correct */
        return (uint16_t)(sign | h);
    }
    uint32_t h = sign | ((uint32_t)e << 10) | (man >> 13);
    const uint32_t rem = man & 0x1fffu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))
        ++h; /* carries into the exponent (or to infinity) as rounding requires */
    return (uint16_t)h;
}

float oracle_f16_to_f32(uint16_t h)
{
    const uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    const int32_t exp = (h >> 10) & 0x1f;
    const uint32_t man = h & 0x3ffu;
    float v;
    if (exp == 0)
        v = ldexpf((float)man, -24); /* subnormal: man * 2^-24 (exact in fp32) */
    else if (exp == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexpf((float)(man | 0x400u), exp - 25);
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    u |= sign;
    memcpy(&v, &u, sizeof v);
    return v;
}

/*
 * INT8 quantisation of `rows` head vectors of D bf16 values each (fp32
 * arithmetic, IEEE division): codes [rows][D] int8, scales [rows] fp16 bits.
 */
void oracle_quantize_rows(const uint16_t *x, int64_t rows, int d_len, int8_t *codes, uint16_t *scales)
{
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * d_len;
        float amax = 0.0f;
        for (int d = 0; d < d_len; ++d) {
            const float v = (float)bf16_to_double(xr[d]);
            const float a = fabsf(v);
            if (a > amax)
                amax = a;
        }
        float scale = amax / 127.0f;
        if (scale < 1e-8f)
            scale = 1e-8f;
        for (int d = 0; d < d_len; ++d) {
            const float q = (float)bf16_to_double(xr[d]) / scale;
            const float t = q >= 0.0f ? q + 0.5f : q - 0.5f;
            codes[r * d_len + d] = (int8_t)truncf(t);
        }
        scales[r] = oracle_f32_to_f16(scale);
    }
}

/*
 * INT8 scatter: quantise each new token's K and V head vectors into its slot.
 * Codes use the data layout [num_blocks][block_size][num_kv_heads][head_dim];
 * scales are stored head-major inside a block, [num_blocks][num_kv_heads]
 * [block_size] (the pages fix no layout for them; per-head token runs are
 * then contiguous).
 */
void oracle_store_kvcache_int8(int8_t *k_cache, int8_t *v_cache, uint16_t *k_scale, uint16_t *v_scale,
                               const uint16_t *k, const uint16_t *v, const int32_t *slots, int64_t num_tokens,
                               int num_kv_heads, int head_dim, int block_size)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int32_t s = slots[t];
        if (s == -1)
            continue;
        const int64_t blk = s / block_size, off = s % block_size;
        for (int g = 0; g < num_kv_heads; ++g) {
            const int64_t si = (blk * num_kv_heads + g) * block_size + off;
            oracle_quantize_rows(k + t * row + (int64_t)g * head_dim, 1, head_dim,
                                 k_cache + (int64_t)s * row + (int64_t)g * head_dim, k_scale + si);
            oracle_quantize_rows(v + t * row + (int64_t)g * head_dim, 1, head_dim,
                                 v_cache + (int64_t)s * row + (int64_t)g * head_dim, v_scale + si);
        }
    }
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Slot of every new token (prepare_prefill / prepare_decode).
 * Sequence b has seq_lens[b] tokens of which the last query_lens[b] are new;
 * its physical blocks are blk_ids[blk_off[b] .. blk_off[b+1]).
 * Writes sum(query_lens) slots in sequence order.  Returns the count, or -1
 * if a position falls outside the sequence's block list.
 */
int64_t oracle_slot_mapping(int num_seqs, const int32_t *seq_lens, const int32_t *query_lens,
                            const int32_t *blk_off, const int32_t *blk_ids, int block_size,
                            int32_t *slots)
{
    int64_t t = 0;
    for (int b = 0; b < num_seqs; ++b) {
        int first = seq_lens[b] - query_lens[b];
        for (int pos = first; pos < seq_lens[b]; ++pos) {
            int logical = pos / block_size;
            if (logical >= blk_off[b + 1] - blk_off[b])
                return -1;
            int phys = blk_ids[blk_off[b] + logical];
            slots[t++] = phys * block_size + pos % block_size;
        }
    }
    return t;
}

/*
 * KV scatter: cache row `slot` (row = num_kv_heads*head_dim bf16 values)
 * receives the token's K and V rows, bit for bit.  slot == -1 is skipped.
 */
void oracle_store_kvcache(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k, const uint16_t *v,
                          const int32_t *slots, int64_t num_tokens, int64_t row_elems)
{
    for (int64_t t = 0; t < num_tokens; ++t) {
        int32_t s = slots[t];
        if (s == -1)
            continue;
        memcpy(k_cache + (int64_t)s * row_elems, k + t * row_elems, (size_t)row_elems * 2);
        memcpy(v_cache + (int64_t)s * row_elems, v + t * row_elems, (size_t)row_elems * 2);
    }
}

/*
 * Block copy (copy-on-write fork): for each (src, dst, n) triple, cache rows
 * src*bs + i are copied to dst*bs + i for i < n, in K and in V, in order.
 */
void oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int32_t *triples, int64_t num_triples,
                        int block_size, int64_t row_elems)
{
    for (int64_t t = 0; t < num_triples; ++t) {
        const int64_t src = triples[3 * t], dst = triples[3 * t + 1], n = triples[3 * t + 2];
        for (int64_t i = 0; i < n; ++i) {
            memcpy(k_cache + (dst * block_size + i) * row_elems, k_cache + (src * block_size + i) * row_elems,
                   (size_t)row_elems * 2);
            memcpy(v_cache + (dst * block_size + i) * row_elems, v_cache + (src * block_size + i) * row_elems,
                   (size_t)row_elems * 2);
        }
    }
}

/*
 * Block copy of an INT8 cache: the same (src, dst, n) triples move the codes
 * of rows src*bs + i to dst*bs + i (i < n) and, for every KV head g, the
 * scales [src][g][i] to [dst][g][i] (scale layout [blocks][Hkv][bs]).
 */
void oracle_copy_blocks_int8(int8_t *k_cache, int8_t *v_cache, uint16_t *k_scale, uint16_t *v_scale,
                             const int32_t *triples, int64_t num_triples, int block_size, int num_kv_heads,
                             int head_dim)
{
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int64_t t = 0; t < num_triples; ++t) {
        const int64_t src = triples[3 * t], dst = triples[3 * t + 1], n = triples[3 * t + 2];
        for (int64_t i = 0; i < n; ++i) {
            memcpy(k_cache + (dst * block_size + i) * row, k_cache + (src * block_size + i) * row, (size_t)row);
            memcpy(v_cache + (dst * block_size + i) * row, v_cache + (src * block_size + i) * row, (size_t)row);
            for (int g = 0; g < num_kv_heads; ++g) {
                k_scale[(dst * num_kv_heads + g) * block_size + i] = k_scale[(src * num_kv_heads + g) * block_size + i];
                v_scale[(dst * num_kv_heads + g) * block_size + i] = v_scale[(src * num_kv_heads + g) * block_size + i];
            }
        }
    }
}

/*
 * Dense rebuild of one sequence's keys (or values) through its block list:
 * dense[j][g][d] = cache[blk[j / bs]][j % bs][g][d], for j < len.
 */
void oracle_gather_dense(const uint16_t *cache, int len, const int32_t *blocks, int num_kv_heads,
                         int head_dim, int block_size, double *dense)
{
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int j = 0; j < len; ++j) {
        int64_t phys = blocks[j / block_size];
        int64_t slot = phys * block_size + j % block_size;
        const uint16_t *src = cache + slot * row;
        for (int64_t e = 0; e < row; ++e)
            dense[(int64_t)j * row + e] = bf16_to_double(src[e]);
    }
}

/*
 * A finite fp32 value rounded to the nearest bf16 (the upper 16 bits of an fp32
 * pattern), ties to the even pattern: add half of the dropped 16-bit unit, less one
 * unless the kept part is odd, then drop the low 16 bits.
 */
static double round_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
    float r;
    memcpy(&r, &u, sizeof r);
    return (double)r;
}

/*
 * Same rebuild from an INT8 cache: dense value = code * fp16 scale of its (slot,
 * head) ("面试问答准备: nano-vLLM 推理引擎优化", Q3).  The page dequantises in two
 * ways: the decode kernel multiplies each code by its token scale in fp32 and feeds
 * the product straight into the online softmax (to_bf16 = 0: the exact product, as
 * code * scale needs at most 8 + 11 significant bits), and the prefill path
 * materialises the values as code * scale in fp32 cast to the model's dtype
 * (to_bf16 = 1: that product rounded to bf16).
 */
void oracle_gather_dense_int8(const int8_t *cache, const uint16_t *scales, int len, const int32_t *blocks,
                              int num_kv_heads, int head_dim, int block_size, int to_bf16, double *dense)
{
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int j = 0; j < len; ++j) {
        int64_t phys = blocks[j / block_size];
        int64_t slot = phys * block_size + j % block_size;
        for (int g = 0; g < num_kv_heads; ++g) {
            const double sc = (double)oracle_f16_to_f32(scales[(phys * num_kv_heads + g) * block_size + j % block_size]);
            for (int d = 0; d < head_dim; ++d) {
                const int8_t c = cache[slot * row + (int64_t)g * head_dim + d];
                dense[(int64_t)j * row + (int64_t)g * head_dim + d] =
                    to_bf16 ? round_to_bf16((float)c * (float)sc) : (double)c * sc;
            }
        }
    }
}

/*
 * Causal attention for every query row of every sequence.
 *   q:   [sum(query_lens), Hq, D] bf16 bits, rows in sequence order
 *   out: [sum(query_lens), Hq, D] double
 * Query row i of sequence b (0 <= i < query_lens[b]) is at absolute position
 * seq_lens[b] - query_lens[b] + i and sees keys 0..that position.
 * row_select (nullable): when given, only packed query rows t with
 * row_select[t] != 0 are computed (all heads); other output rows are left
 * untouched.  Returns the number of (query row, head, key) scores computed,
 * or -1 on malformed input.
 */
static int64_t attention_impl(const uint16_t *q, const void *k_cache, const void *v_cache, const uint16_t *k_scale,
                              const uint16_t *v_scale, int int8_mode, int num_seqs, const int32_t *seq_lens,
                              const int32_t *query_lens, const int32_t *blk_off, const int32_t *blk_ids,
                              int num_heads, int num_kv_heads, int head_dim, int block_size, double scale,
                              const uint8_t *row_select, double *out, int num_threads)
{
#ifdef _OPENMP
    /* thread count of this call only (0: the OpenMP default) */
    const int nthreads = num_threads > 0 ? num_threads : omp_get_max_threads();
#else
    (void)num_threads;
#endif
    if (num_heads % num_kv_heads != 0)
        return -1;
    const int group = num_heads / num_kv_heads;
    const int64_t kv_row = (int64_t)num_kv_heads * head_dim;
    int64_t pairs = 0;
    int64_t q_begin = 0;

    for (int b = 0; b < num_seqs; ++b) {
        const int lk = seq_lens[b], lq = query_lens[b];
        if (lq < 0 || lk < lq || (lq > 0 && lk < 1))
            return -1;
        if ((int64_t)(lk + block_size - 1) / block_size > blk_off[b + 1] - blk_off[b])
            return -1;
        int any = 0;
        for (int i = 0; i < lq; ++i)
            if (!row_select || row_select[q_begin + i])
                any = 1;
        if (!any) {
            q_begin += lq;
            continue;
        }
        /* step 1: dense K and V of this sequence through its block table */
        double *kd = (double *)malloc(sizeof(double) * (size_t)lk * (size_t)kv_row);
        double *vd = (double *)malloc(sizeof(double) * (size_t)lk * (size_t)kv_row);
        if (!kd || !vd) {
            free(kd);
            free(vd);
            return -1;
        }
        if (int8_mode) { /* 1: exact products, 2: products rounded to bf16 */
            oracle_gather_dense_int8((const int8_t *)k_cache, k_scale, lk, blk_ids + blk_off[b], num_kv_heads,
                                     head_dim, block_size, int8_mode == 2, kd);
            oracle_gather_dense_int8((const int8_t *)v_cache, v_scale, lk, blk_ids + blk_off[b], num_kv_heads,
                                     head_dim, block_size, int8_mode == 2, vd);
        } else {
            oracle_gather_dense((const uint16_t *)k_cache, lk, blk_ids + blk_off[b], num_kv_heads, head_dim,
                                block_size, kd);
            oracle_gather_dense((const uint16_t *)v_cache, lk, blk_ids + blk_off[b], num_kv_heads, head_dim,
                                block_size, vd);
        }

        /* step 2: causal softmax(q K^T * scale) V for each (row, head) */
        int64_t work = (int64_t)lq * num_heads;
        int64_t seq_pairs = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : seq_pairs) num_threads(nthreads)
        for (int64_t w = 0; w < work; ++w) {
            int i = (int)(w / num_heads), h = (int)(w % num_heads);
            int64_t t = q_begin + i;
            if (row_select && !row_select[t])
                continue;
            int g = h / group;
            int visible = lk - lq + i + 1; /* keys 0 .. position */
            const uint16_t *qrow = q + (t * num_heads + h) * head_dim;
            double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
            double *s = (double *)malloc(sizeof(double) * (size_t)visible);
            for (int d = 0; d < head_dim; ++d)
                qd[d] = bf16_to_double(qrow[d]);
            double m = -INFINITY;
            for (int j = 0; j < visible; ++j) {
                const double *kr = kd + (int64_t)j * kv_row + (int64_t)g * head_dim;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += qd[d] * kr[d];
                s[j] = dot * scale;
                if (s[j] > m)
                    m = s[j];
            }
            double l = 0.0;
            for (int j = 0; j < visible; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            double *o = out + (t * num_heads + h) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            for (int j = 0; j < visible; ++j) {
                const double *vr = vd + (int64_t)j * kv_row + (int64_t)g * head_dim;
                double p = s[j] / l;
                for (int d = 0; d < head_dim; ++d)
                    o[d] += p * vr[d];
            }
            seq_pairs += visible;
            free(qd);
            free(s);
        }
        pairs += seq_pairs;
        free(kd);
        free(vd);
        q_begin += lq;
    }
    return pairs;
}

int64_t oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                               int num_seqs, const int32_t *seq_lens, const int32_t *query_lens,
                               const int32_t *blk_off, const int32_t *blk_ids, int num_heads,
                               int num_kv_heads, int head_dim, int block_size, double scale,
                               const uint8_t *row_select, double *out, int num_threads)
{
    return attention_impl(q, k_cache, v_cache, NULL, NULL, 0, num_seqs, seq_lens, query_lens, blk_off, blk_ids,
                          num_heads, num_kv_heads, head_dim, block_size, scale, row_select, out, num_threads);
}

/* Causal attention over an INT8 cache: the same definition on the dequantised K/V
 * (values_bf16: the dequantised values rounded to bf16, as the page's prefill path). */
int64_t oracle_paged_attention_int8(const uint16_t *q, const int8_t *k_cache, const int8_t *v_cache,
                                    const uint16_t *k_scale, const uint16_t *v_scale, int values_bf16, int num_seqs,
                                    const int32_t *seq_lens, const int32_t *query_lens, const int32_t *blk_off,
                                    const int32_t *blk_ids, int num_heads, int num_kv_heads, int head_dim,
                                    int block_size, double scale, const uint8_t *row_select, double *out,
                                    int num_threads)
{
    return attention_impl(q, k_cache, v_cache, k_scale, v_scale, values_bf16 ? 2 : 1, num_seqs, seq_lens, query_lens, blk_off,
                          blk_ids, num_heads, num_kv_heads, head_dim, block_size, scale, row_select, out,
                          num_threads);
}
