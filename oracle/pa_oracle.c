/*
 * pa_oracle.c -- CPU oracle for paged decode attention and its cache ops.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can check the CUDA kernels against a plain,
 * slow, obviously correct restatement of what the method computes.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Sources (page titles and sections of the pages this restates):
 *  - "PagedAttention 完全拆解：操作系统分页思想如何拯救 LLM 推理的内存利用率",
 *    section "背景" (the softmax attention equation a_ij, o_i with the 1/sqrt(d)
 *    factor) and section "原理详解（二）：块式注意力的数学" (the block-wise form:
 *    paging only changes storage, the result is exactly standard attention).
 *  - same page, "原理详解（一）" Figure 6 (block table: logical block -> physical
 *    block, only the last block partially filled) and "原理详解（三）：kernel 实现"
 *    items 1 and 3 (fused reshape + block write; fused block copy).
 *  - same page, "内存共享" Figure 8 (copy-on-write copies one block src -> dst).
 *  - same page, "局限与未解决的问题" item 6, and "PagedAttention 与 vLLM 推理加速"
 *    section "一图总结" (chunked prefill and speculative verification: several
 *    new query tokens of one sequence attend to the paged cache causally).
 *  - iaim.asia/ai-infra/182, section "KV Cache 如何按块分配" (zero-based table:
 *    tokens 0..15 -> block_table[0], 16..31 -> block_table[1], ...; the in-block
 *    layout is the backend's choice and K, V may be two tensors).
 *
 * Layout conventions shared with the tests (the pages leave the in-block layout
 * to the backend, so one is fixed here):
 *   k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *   q, out           : [num_seqs][num_q_heads][head_dim]
 *   block_tables     : [num_seqs][bt_stride] int32
 *   context_lens     : [num_seqs] int32, includes the current token
 *   slot_mapping     : [num_tokens] int64, slot = block * block_size + offset,
 *                      slot < 0 means "skip this token"
 *   query head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 * Arithmetic is fp64.  fp16 and bf16 inputs are decoded to fp64 exactly by the
 * bit-level decoders below.  Nothing here is blocked, fused or reordered: the
 * attention routine gathers each sequence's keys and values through its block
 * table into contiguous arrays, then evaluates the textbook definition.
 *
 * Parity pins for every function are in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_E4M3 = 3 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                  /* zero / subnormal */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(frac | 0x400), expo - 25);  /* 1.frac * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE 754 binary32 word. */
double orc_bf16_to_f64(uint16_t b)
{
    uint32_t w = (uint32_t)b << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits;
 * exponent field 0 is subnormal (fraction x 2^-9), the all-ones code S.1111.111 is
 * NaN, there are no infinities, and the largest finite magnitude is 448. */
double orc_e4m3_to_f64(uint8_t c)
{
    int sign = c >> 7;
    int expo = (c >> 3) & 0xf;
    int frac = c & 0x7;
    double mag;
    if (expo == 15 && frac == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)frac, -9);
    else
        mag = ldexp((double)(8 + frac), expo - 10);      /* 1.frac * 2^(e-7) */
    return sign ? -mag : mag;
}

/* The e4m3 code nearest to x, ties to the even code (even fraction), saturating:
 * magnitudes of 448 and above (infinity included) give +-448, NaN gives 0x7f.
 * Found by comparing x with every finite code's value. */
uint8_t orc_f32_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7e;
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        const double d = fabs(a - orc_e4m3_to_f64((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return sign | (uint8_t)best;
}

static size_t orc_elem_size(int dtype)
{
    return dtype == ORC_F32 ? 4 : (dtype == ORC_E4M3 ? 1 : 2);
}

static double orc_load(const void* base, int dtype, int64_t idx)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char*)base + 4 * idx, 4);
        return (double)f;
    }
    if (dtype == ORC_E4M3)
        return orc_e4m3_to_f64(((const uint8_t*)base)[idx]);
    uint16_t bits;
    memcpy(&bits, (const char*)base + 2 * idx, 2);
    return dtype == ORC_F16 ? orc_f16_to_f64(bits) : orc_bf16_to_f64(bits);
}

/* Element index of k_cache[block][head][offset][0]. */
static int64_t orc_row(int64_t block, int head, int offset, int num_kv_heads,
                       int block_size, int head_dim)
{
    return ((block * num_kv_heads + head) * block_size + offset) * (int64_t)head_dim;
}

/*
 * One (sequence, query head): gather, then softmax attention in fp64.
 * Returns 0, or -1 when a block id read from the table lies outside the pool.
 */
static int orc_one_head(double* o, const void* q, int q_dtype, const void* k_cache,
                        const void* v_cache, int kv_dtype, const float* k_scale,
                        const float* v_scale, int64_t num_blocks,
                        const int32_t* table_row, int s, int h, int L, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, double scale)
{
    const int group = num_q_heads / num_kv_heads;
    const int hk = h / group;
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    if (L == 0)
        return 0;                       /* empty context: zero output (convention) */

    /* Step 1 -- gather: token t lives in physical block table_row[t / B] at slot t % B. */
    double* K = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
    double* V = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
    double* sc = (double*)malloc(sizeof(double) * (size_t)L);
    if (!K || !V || !sc) {
        free(K); free(V); free(sc);
        return -2;
    }
    for (int t = 0; t < L; ++t) {
        int64_t blk = table_row[t / block_size];
        int off = t % block_size;
        if (blk < 0 || blk >= num_blocks) {
            free(K); free(V); free(sc);
            return -1;
        }
        int64_t r = orc_row(blk, hk, off, num_kv_heads, block_size, head_dim);
        /* a quantised cache holds codes; the value is code * the kv head's scale */
        const double ks = k_scale ? (double)k_scale[hk] : 1.0;
        const double vs = v_scale ? (double)v_scale[hk] : 1.0;
        for (int d = 0; d < head_dim; ++d) {
            K[(size_t)t * head_dim + d] = orc_load(k_cache, kv_dtype, r + d) * ks;
            V[(size_t)t * head_dim + d] = orc_load(v_cache, kv_dtype, r + d) * vs;
        }
    }

    /* Step 2 -- scores s_t = scale * q . k_t. */
    const int64_t qoff = ((int64_t)s * num_q_heads + h) * head_dim;
    for (int t = 0; t < L; ++t) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += orc_load(q, q_dtype, qoff + d) * K[(size_t)t * head_dim + d];
        sc[t] = scale * dot;
    }

    /* Step 3 -- a_t = exp(s_t) / sum_u exp(s_u), evaluated as exp(s_t - m) / sum exp(s_u - m)
     * with m = max s (the same quotient, kept finite). */
    double m = sc[0];
    for (int t = 1; t < L; ++t)
        if (sc[t] > m)
            m = sc[t];
    double l = 0.0;
    for (int t = 0; t < L; ++t) {
        sc[t] = exp(sc[t] - m);
        l += sc[t];
    }

    /* Step 4 -- o = sum_t a_t v_t. */
    for (int t = 0; t < L; ++t) {
        double a = sc[t] / l;
        for (int d = 0; d < head_dim; ++d)
            o[d] += a * V[(size_t)t * head_dim + d];
    }
    free(K); free(V); free(sc);
    return 0;
}

/*
 * Paged decode attention: out[s][h][:] for every sequence s and query head h.
 * context_lens[s] tokens are attended (the current token included).  For an
 * E4M3 cache, k_scale / v_scale give each kv head's scale (NULL otherwise).
 * Returns 0; -1 for a block id outside [0, num_blocks); -3 for a context
 * longer than the table row (bt_stride * block_size) or negative; -2 on
 * allocation failure; -4 for bad sizes.
 */
int orc_paged_attention(double* out, const void* q, int q_dtype, const void* k_cache,
                        const void* v_cache, int kv_dtype, const float* k_scale,
                        const float* v_scale, int64_t num_blocks,
                        const int32_t* block_tables, int64_t bt_stride,
                        const int32_t* context_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, double scale,
                        int num_threads)
{
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_q_heads % num_kv_heads != 0)
        return -4;
    for (int s = 0; s < num_seqs; ++s)
        if (context_lens[s] < 0 || (int64_t)context_lens[s] > bt_stride * block_size)
            return -3;

    int status = 0;
    const int64_t work = (int64_t)num_seqs * num_q_heads;
#ifdef _OPENMP
    if (num_threads < 1)
        num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t i = 0; i < work; ++i) {
        int s = (int)(i / num_q_heads);
        int h = (int)(i % num_q_heads);
        int rc = orc_one_head(out + i * head_dim, q, q_dtype, k_cache, v_cache, kv_dtype,
                              k_scale, v_scale, num_blocks,
                              block_tables + (int64_t)s * bt_stride, s, h,
                              context_lens[s], num_q_heads, num_kv_heads, head_dim,
                              block_size, scale);
        if (rc != 0) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = rc;
        }
    }
    (void)num_threads;
    return status;
}

/*
 * Attention of a chunk of consecutive new query tokens per sequence: chunked
 * prefill and speculative verification, the later uses of the paged cache named
 * in "PagedAttention 完全拆解", section "局限与未解决的问题" item 6 (Chunked Prefill
 * on top of the paged KV cache) and in "PagedAttention 与 vLLM 推理加速", section
 * "一图总结" (a large model verifying a small model's guesses).
 *
 * Sequence s owns query rows query_start[s] .. query_start[s+1]-1 of q and out
 * ([rows][num_q_heads][head_dim]); with n = that count and L = context_lens[s],
 * the chunk's tokens are the last n of the L cached ones, so chunk token j sits at
 * position L - n + j and, causally, attends to cached tokens 0 .. L - n + j: the
 * decode attention of section "背景" over a context of L - n + j + 1 tokens.
 * Rows of a sequence whose chunk is longer than its context (n > L) are NaN.
 * Returns 0; -1 for a block id outside the pool; -3 for a context longer than
 * the table row or negative; -4 for bad sizes or a decreasing query_start.
 */
int orc_chunk_attention(double* out, const void* q, int q_dtype, const void* k_cache,
                        const void* v_cache, int kv_dtype, const float* k_scale,
                        const float* v_scale, int64_t num_blocks,
                        const int32_t* block_tables, int64_t bt_stride,
                        const int32_t* context_lens, const int32_t* query_start, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        double scale, int num_threads)
{
    if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_q_heads % num_kv_heads != 0 || query_start[0] != 0)
        return -4;
    for (int s = 0; s < num_seqs; ++s) {
        if (query_start[s + 1] < query_start[s])
            return -4;
        if (context_lens[s] < 0 || (int64_t)context_lens[s] > bt_stride * block_size)
            return -3;
    }

    int status = 0;
    const int64_t rows = query_start[num_seqs];
    const int64_t work = rows * num_q_heads;
#ifdef _OPENMP
    if (num_threads < 1)
        num_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
    for (int64_t i = 0; i < work; ++i) {
        const int64_t row = i / num_q_heads;            /* query token row of q / out */
        const int h = (int)(i % num_q_heads);
        int s = 0;                                      /* the sequence owning the row */
        while (query_start[s + 1] <= row)
            ++s;
        const int n = query_start[s + 1] - query_start[s];
        const int L = context_lens[s];
        double* o = out + i * head_dim;
        if (n > L) {
            for (int d = 0; d < head_dim; ++d)
                o[d] = NAN;
            continue;
        }
        const int j = (int)(row - query_start[s]);      /* index within the chunk */
        const int visible = L - n + j + 1;              /* tokens 0 .. L - n + j */
        int rc = orc_one_head(o, q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                              num_blocks, block_tables + (int64_t)s * bt_stride, (int)row, h,
                              visible, num_q_heads, num_kv_heads, head_dim, block_size, scale);
        if (rc != 0) {
#ifdef _OPENMP
#pragma omp critical
#endif
            status = rc;
        }
    }
    (void)num_threads;
    return status;
}

/*
 * reshape_and_cache: for every new token i with slot_mapping[i] >= 0 and every
 * kv head h, copy the bytes of k[i][h][:] to k_cache[slot / B][h][slot % B][:]
 * (likewise v).  A byte copy, so values, NaN payloads and signed zeros are kept.
 * Returns 0, or -1 if a slot lies beyond the pool (nothing is written then).
 */
int orc_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                          int head_dim, int block_size, int64_t num_blocks, int dtype)
{
    const size_t esz = orc_elem_size(dtype);
    const size_t row = esz * (size_t)head_dim;
    for (int64_t i = 0; i < num_tokens; ++i)
        if (slot_mapping[i] >= num_blocks * block_size)
            return -1;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int off = (int)(slot % block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t src = ((size_t)i * num_kv_heads + h) * row;
            size_t dst = (size_t)orc_row(blk, h, off, num_kv_heads, block_size, head_dim) * esz;
            memcpy((char*)k_cache + dst, (const char*)k + src, row);
            memcpy((char*)v_cache + dst, (const char*)v + src, row);
        }
    }
    return 0;
}

/*
 * reshape_and_cache into an E4M3 cache: for every new token i with a slot >= 0 and
 * every kv head h, k_cache[slot / B][h][slot % B][d] = e4m3(fp32(k[i][h][d]) / k_scale[h])
 * (fp32 division, rounded to the nearest code, ties to even, saturating), likewise v.
 * Returns 0, or -1 if a slot lies beyond the pool (nothing is written then).
 */
int orc_reshape_and_cache_e4m3(const void* k, const void* v, int src_dtype, uint8_t* k_cache,
                               uint8_t* v_cache, const float* k_scale, const float* v_scale,
                               const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int64_t num_blocks)
{
    for (int64_t i = 0; i < num_tokens; ++i)
        if (slot_mapping[i] >= num_blocks * block_size)
            return -1;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int offset = (int)(slot % block_size);
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim;
            int64_t dst = orc_row(block, h, offset, num_kv_heads, block_size, head_dim);
            for (int d = 0; d < head_dim; ++d) {
                float kx = (float)orc_load(k, src_dtype, src + d);
                float vx = (float)orc_load(v, src_dtype, src + d);
                k_cache[dst + d] = orc_f32_to_e4m3(kx / k_scale[h]);
                v_cache[dst + d] = orc_f32_to_e4m3(vx / v_scale[h]);
            }
        }
    }
    return 0;
}

/*
 * copy_blocks: for every layer and every pair (src, dst), the destination block
 * receives the bytes the source block held BEFORE any copy of this call.
 * caches[l] points to a pool of num_blocks blocks of block_bytes each (K and V
 * pools of every layer are passed in one list).  Returns 0, or -1 for a block
 * id outside the pool, or -2 on allocation failure.
 */
int orc_copy_blocks(void* const* caches, int num_caches, const int64_t* pairs,
                    int64_t num_pairs, int64_t block_bytes, int64_t num_blocks)
{
    for (int64_t p = 0; p < num_pairs; ++p)
        if (pairs[2 * p] < 0 || pairs[2 * p] >= num_blocks || pairs[2 * p + 1] < 0 ||
            pairs[2 * p + 1] >= num_blocks)
            return -1;
    if (num_pairs == 0)
        return 0;
    char* snap = (char*)malloc((size_t)(num_pairs * block_bytes));
    if (!snap)
        return -2;
    for (int c = 0; c < num_caches; ++c) {
        char* pool = (char*)caches[c];
        for (int64_t p = 0; p < num_pairs; ++p)      /* pre-copy state of every source */
            memcpy(snap + p * block_bytes, pool + pairs[2 * p] * block_bytes,
                   (size_t)block_bytes);
        for (int64_t p = 0; p < num_pairs; ++p)
            memcpy(pool + pairs[2 * p + 1] * block_bytes, snap + p * block_bytes,
                   (size_t)block_bytes);
    }
    free(snap);
    return 0;
}

/*
 * swap_blocks: moves whole blocks between two pools of one cache that live in
 * different memories -- the swapping of a preempted sequence group's KV blocks to
 * CPU memory and back ("PagedAttention 完全拆解", section "调度与抢占：内存不够时
 * 怎么办", 换出 (Swapping)).  For every cache c and pair (s, d):
 * dst[c][d] = src[c][s], block_bytes bytes; nothing else changes.  Returns 0, or -1
 * for a block id outside its pool.
 */
int orc_swap_blocks(void* const* dst, void* const* src, int num_caches, const int64_t* pairs,
                    int64_t num_pairs, int64_t block_bytes, int64_t src_blocks,
                    int64_t dst_blocks)
{
    for (int64_t p = 0; p < num_pairs; ++p)
        if (pairs[2 * p] < 0 || pairs[2 * p] >= src_blocks || pairs[2 * p + 1] < 0 ||
            pairs[2 * p + 1] >= dst_blocks)
            return -1;
    for (int c = 0; c < num_caches; ++c)
        for (int64_t p = 0; p < num_pairs; ++p)
            memcpy((char*)dst[c] + pairs[2 * p + 1] * block_bytes,
                   (const char*)src[c] + pairs[2 * p] * block_bytes, (size_t)block_bytes);
    return 0;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
