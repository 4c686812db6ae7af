/*
 * pa.h -- C ABI of the paged decode attention library (libpa.so), GB300 / sm_103a.
 *
 * Three operations over a paged KV cache, each a hand-written CUDA kernel:
 *
 *   pa_reshape_and_cache  write each new token's K/V rows into the cache slots
 *                         named by slot_mapping ("PagedAttention 完全拆解",
 *                         section 原理详解（三）：kernel 实现, item 1: fused reshape
 *                         and block write; Figure 6 decode steps).
 *   pa_decode             one query per sequence attends over its context through
 *                         its block table (same page, section 原理详解（二）：块式注意
 *                         力的数学, block-wise attention equation; section 原理详解
 *                         （三） item 2: fused block read and attention), with a
 *                         split-context second pass for long contexts
 *                         (iaim.asia/ai-infra/182, section vLLM 内核里的缓解写法:
 *                         segments merged by a reduce).
 *   pa_copy_blocks        copy whole blocks src -> dst for copy-on-write (first page,
 *                         section 原理详解（三） item 3: fused block copy; section
 *                         内存共享, Figure 8).
 *
 * Layout (the pages leave the in-block layout to the backend; iaim.asia page,
 * section KV Cache 如何按块分配).  All tensors are dense, row-major, in device
 * memory, and owned by the caller:
 *
 *   k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]   dtype T
 *   q, out            [num_seqs][num_q_heads][head_dim]   (out may be fp32)
 *   block_tables      [num_seqs][block_table_stride]      int32 physical block ids;
 *                     token t of sequence s lives in block block_tables[s][t / B]
 *                     at slot t % B
 *   context_lens      [num_seqs]                           int32, current token included
 *   new k, v          [num_tokens][num_kv_heads][head_dim] dtype T
 *   slot_mapping      [num_tokens]                         int64, slot = block * B + offset;
 *                                                          slot < 0 skips the token
 *   query head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 * Conventions:
 *   - Every call is asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  The library never synchronises,
 *     never allocates device memory and keeps no state except a per-device SM
 *     count and a per-device error word (see pa_get_device_error).
 *   - Host-side validation runs before any launch.  A failed check returns a
 *     negative pa_status and launches nothing.  A failed launch returns
 *     PA_ERR_CUDA.
 *   - Device-side checks (always on, one compare per block): a block id outside
 *     [0, num_blocks), a slot outside the pool, or a context length that is
 *     negative or exceeds max_context_len sets a bit in the device error word,
 *     skips the access and, for pa_decode, writes NaN to the affected outputs.
 *     Kernels never trap.
 *   - A context length of 0 yields an all-zero output row.
 *   - Per-device state (the SM count, the error word, encoded tensor maps and the
 *     no-alloc scratch address) is looked up once per device and process.  Do not
 *     call cudaDeviceReset on a device the library has been used on while the
 *     process still uses the library: the cached addresses would then point into
 *     the destroyed context.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID = -1,      /* a pointer, size, alignment or value is out of range */
    PA_ERR_UNSUPPORTED = -2,  /* head_dim / block_size / dtype combination not built */
    PA_ERR_WORKSPACE = -3,    /* split-context workspace missing or too small */
    PA_ERR_CUDA = -4          /* a CUDA runtime call or kernel launch failed */
} pa_status;

/* Bits of the device error word. */
#define PA_DEVERR_BLOCK_ID    0x1u  /* block table entry outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT_LEN 0x2u  /* context_len < 0 or > max_context_len */
#define PA_DEVERR_SLOT        0x4u  /* slot_mapping entry >= num_blocks * block_size */
#define PA_DEVERR_TIMEOUT     0x8u  /* a bounded pipeline wait gave up */
#define PA_DEVERR_RANGE       0x10u /* chunk attention over a bf16 cache: a row weighed a V
                                           element without an f16 value (|v| >= 65536,
                                           infinite or NaN) */

/*
 * Bytes of device workspace a pa_decode call with these sizes uses: when it splits
 * contexts into partitions of partition_size tokens (0 = the automatic choice, which
 * never needs more than this; < 0 = never split, returns 0), per (sequence, query
 * head, partition) one fp32 partial output row of head_dim values plus its running
 * max and sum; with the automatic choice, at least 8 bytes per sequence (rounded up
 * to 256) for the longest-first dispatch order of a one-pass call (see pa_decode).
 * Passing a workspace of this size to an automatic (partition_size 0) call is what
 * turns that order on: a call without a workspace that does not split runs the
 * sequences in index order, with the same results but a longer tail on mixed-length
 * batches.  Pure host arithmetic; no CUDA call.  Returns 0 for invalid sizes.
 */
size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t max_context_len, int32_t block_size,
                                 int32_t partition_size);

/*
 * Paged decode attention: for every sequence s and query head h,
 *   out[s][h][:] = sum_t a_t v_t,  a_t = exp(scale q.k_t) / sum_u exp(scale q.k_u),
 * over the context_lens[s] tokens reached through block_tables[s].
 *
 *   out               device, [S][Hq][D] of out_dtype (PA_F32 or kv_dtype)
 *   q                 device, [S][Hq][D] of kv_dtype
 *   k_cache, v_cache  device, 16-byte aligned, [num_blocks][Hkv][B][D] of kv_dtype
 *   block_tables      device, [S][block_table_stride] int32
 *   context_lens      device, [S] int32
 *   max_context_len   host upper bound on every context_lens[s]; sizes the grid
 *                     (no device-to-host read happens).  Must be <=
 *                     block_table_stride * block_size.
 *   head_dim          64 or 128; block_size 16 or 32; num_q_heads a multiple of
 *                     num_kv_heads.  kv_dtype PA_F32, PA_F16 or PA_BF16.
 *   scale             multiplies q.k (1/sqrt(head_dim) in the usual case)
 *   partition_size    0 = automatic; < 0 = one pass per (sequence, kv head);
 *                     > 0 = split each context into partitions of this many tokens
 *                     (a multiple of block_size) and merge them in a second kernel.
 *   workspace         device buffer of workspace_bytes; required only when the
 *                     call splits (see pa_decode_workspace_bytes).  An automatic
 *                     (partition_size 0) one-pass call on the CUDA-core kernel (fewer
 *                     than 4 query heads per kv head; over E4M3 caches, head_dim
 *                     64 only) whose grid holds more CTAs
 *                     than fit on the GPU at once uses its first 8 * S bytes, when
 *                     given, for a longest-first order of the sequences (one more
 *                     small launch; pa_decode_orders_sequences tells): a long
 *                     context started in the last wave would stretch the kernel's
 *                     tail.  Results are bitwise the same in either order.
 *   stream            cudaStream_t (as void*).
 * out must not overlap q or the caches, and the workspace none of out, q, the
 * caches, block_tables or context_lens (PA_ERR_INVALID, nothing launched).
 */
int pa_decode(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
              const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
              const int32_t* block_tables, int64_t block_table_stride,
              const int32_t* context_lens, int32_t max_context_len, int32_t num_seqs,
              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
              float scale, int32_t partition_size, void* workspace, size_t workspace_bytes,
              void* stream);

/*
 * Bytes of the static device scratch pa_decode_noalloc uses (32 MiB).  Every GPU
 * that loads the library's no-alloc module keeps this much device memory until
 * the process exits.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * pa_decode_noalloc -- the split-context pa_decode with its scratch in a fixed
 * static device array (PA_NOALLOC_SCRATCH_BYTES) instead of a caller workspace.
 * The pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory on the decode path, such as a plugin whose host runtime
 * owns all device memory and forbids cudaMalloc in its enqueue hook, or a C caller
 * with no allocator.  The caller still owns and passes every input and the output.
 *
 * Arguments, layout and results are those of pa_decode, minus the workspace.
 * partition_size: 0 = 512 tokens, > 0 = that many (a multiple of block_size),
 * < 0 is rejected (PA_ERR_INVALID): this entry point always splits.
 * Returns PA_ERR_WORKSPACE, launching nothing, when the split needs more than
 * PA_NOALLOC_SCRATCH_BYTES (pa_decode_workspace_bytes gives the need).
 * Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 * The first call on each device looks up the array's device address (with that
 * device current).
 * All calls share the one array, so calls that overlap on the GPU (say, on two
 * streams) race and corrupt each other's results; serialise them.  The array
 * keeps the last call's contents; nothing in it needs to start at zero, because
 * each call writes every partial it reads.
 */
int pa_decode_noalloc(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                      const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                      const int32_t* block_tables, int64_t block_table_stride,
                      const int32_t* context_lens, int32_t max_context_len, int32_t num_seqs,
                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, float scale, int32_t partition_size, void* stream);

/*
 * Cache write: for each token i < num_tokens with slot = slot_mapping[i] >= 0 and
 * each kv head h, k_cache[slot / B][h][slot % B][:] = k[i][h][:] and likewise for v.
 * A bit-exact copy.  k, v, k_cache, v_cache: device, 16-byte aligned;
 * slot_mapping: device int64.  Two tokens naming the same slot is a caller error
 * (which one lands is unspecified).  Slots >= num_blocks * B are skipped and flag
 * PA_DEVERR_SLOT.
 */
int pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int64_t num_tokens, int32_t num_kv_heads,
                         int32_t head_dim, int32_t block_size, int64_t num_blocks,
                         pa_dtype dtype, void* stream);

/*
 * Block copy for copy-on-write: for every layer l < num_layers and every pair p,
 * the whole block src = pairs[2p] of k_caches[l] and of v_caches[l] is copied to
 * block dst = pairs[2p+1] (block_bytes bytes each; every block of every pool).
 *   k_caches, v_caches  HOST arrays of num_layers DEVICE pointers (16-byte aligned)
 *   src_dst_pairs_host  HOST array of 2 * num_pairs int64 block ids
 *   block_bytes         bytes of one block (a multiple of 16)
 * Validation (host): ids in [0, num_blocks), destinations pairwise distinct, and
 * no destination is also a source -- so the result equals copying from the
 * pre-copy state.  The pairs travel as kernel parameters; one launch per chunk of
 * pairs and layers, nothing is allocated.
 */
int pa_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                   const int64_t* src_dst_pairs_host, int64_t num_pairs, int64_t block_bytes,
                   int64_t num_blocks, void* stream);

/*
 * pa_swap_blocks: batched block moves between two pools that live in different
 * memories -- swapping the KV blocks of a preempted sequence group out to a CPU
 * pool and back in ("PagedAttention 完全拆解", section 调度与抢占：内存不够时怎么办,
 * 换出 (Swapping); its Figure 19a shows per-block transfers leaving the link idle
 * when blocks are small, so every pair and cache moves in one launch here).
 *   src_caches, dst_caches  HOST arrays of num_caches pool base addresses (one per
 *                       layer and per K / V); each pool is device memory or pinned
 *                       host memory the device can address (cudaHostAlloc /
 *                       cudaHostRegister); a cache's src and dst pools must not overlap
 *   src_dst_pairs_host  HOST int64 [num_pairs][2]: (block id in src pool, block id in
 *                       dst pool)
 *   block_bytes         bytes of one block (a multiple of 16)
 *   src_num_blocks, dst_num_blocks   pool sizes in blocks
 * For every cache c and pair (s, d): dst_caches[c][d] = src_caches[c][s], byte for
 * byte.  Validation (host): ids in range, destination ids pairwise distinct, pools
 * 16-byte aligned, non-overlapping and device-addressable; otherwise a negative
 * pa_status with nothing launched.  Launches one kernel per 64 caches x 1024 pairs;
 * allocates nothing.  Whether a group is swapped out or in is the caller's choice of
 * src and dst (the pages swap whole sequence groups, all-or-nothing).
 */
int pa_swap_blocks(void* const* src_caches, void* const* dst_caches, int32_t num_caches,
                   const int64_t* src_dst_pairs_host, int64_t num_pairs, int64_t block_bytes,
                   int64_t src_num_blocks, int64_t dst_num_blocks, void* stream);

/*
 * FP8 KV cache (OCP E4M3: 4 exponent bits, bias 7, 3 fraction bits, largest finite
 * magnitude 448, no infinities).  A cache element is a one-byte code c; its value is
 * e4m3(c) * scale[h], with one fp32 scale per kv head for K (k_scale[Hkv]) and one
 * for V (v_scale[Hkv]), both DEVICE arrays owned by the caller.  Quantising halves
 * the bytes of the bandwidth-bound decode (the write-ups list FP8 KV caches among
 * the later vLLM optimisations: "PagedAttention 完全拆解", section 局限与未解决的问题,
 * item 6).  Layouts are those of pa.h's 16-bit caches with one byte per element.
 *
 * pa_reshape_and_cache_fp8: for each token i with slot = slot_mapping[i] >= 0 and each
 * kv head h, k_cache[slot / B][h][slot % B][d] = e4m3(fp32(k[i][h][d]) / k_scale[h]),
 * likewise v: IEEE fp32 division, round to the nearest code with ties to even,
 * magnitudes beyond 448 saturate to +-448, NaN stays NaN.  src_dtype: PA_F32, PA_F16
 * or PA_BF16 (the type of k and v).  head_dim must be a multiple of 16.  Errors and
 * slot checks as in pa_reshape_and_cache.
 */
int pa_reshape_and_cache_fp8(const void* k, const void* v, pa_dtype src_dtype, void* k_cache,
                             void* v_cache, const float* k_scale, const float* v_scale,
                             const int64_t* slot_mapping, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int64_t num_blocks, void* stream);

/*
 * pa_decode_fp8: pa_decode over E4M3 caches.  q (and a native-dtype out) have
 * q_dtype, PA_F16 or PA_BF16; out_dtype is PA_F32 or q_dtype.  Scores use the
 * dequantised keys (q . (c_k * k_scale[h])) and the output the dequantised values;
 * accumulation is fp32 as in pa_decode.  At head_dim 128 with up to 4 query heads per
 * kv head the products run on the tensor cores with the codes as operands: each query
 * row enters as four E4M3 terms after a power-of-two scaling (exact for elements down
 * to about 2^-21 of the row's largest magnitude for bf16 queries, 2^-18 for f16; the
 * smaller ones keep an absolute error below 2^-29 of it) and each probability as four
 * terms (2^-16 relative).  All other arguments, the split
 * rules and the workspace are those of pa_decode (pa_decode_workspace_bytes gives the
 * size).
 */
int pa_decode_fp8(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                  const void* k_cache, const void* v_cache, const float* k_scale,
                  const float* v_scale, int64_t num_blocks, const int32_t* block_tables,
                  int64_t block_table_stride, const int32_t* context_lens,
                  int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size, float scale,
                  int32_t partition_size, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Chunk attention: causal attention of several new query tokens per sequence over
 * the paged cache -- chunked prefill and speculative verification, the later uses
 * of the paged KV cache named in "PagedAttention 完全拆解", section 局限与未解决的问题
 * item 6, and in "PagedAttention 与 vLLM 推理加速", section 一图总结.
 *
 * Sequence s owns query rows query_start[s] .. query_start[s+1]-1 of q and out
 * (n_s rows; query_start[0] = 0, query_start[num_seqs] = num_query_tokens).  Its
 * chunk is the last n_s of its context_lens[s] = L_s cached tokens (write them with
 * pa_reshape_and_cache first), so chunk token j sits at position L_s - n_s + j and
 * attends to cached tokens 0 .. L_s - n_s + j:
 *   out[row][h] = sum_{t <= L_s - n_s + j} a_t v_t,
 *   a_t = exp(scale q[row][h] . k_t) / sum_{u <= L_s - n_s + j} exp(scale q[row][h] . k_u),
 * with k_t, v_t read through block_tables[s] as in pa_decode and query head h
 * reading kv head h / (num_q_heads / num_kv_heads).  n_s = 1 is pa_decode.
 *
 *   out        [num_query_tokens][num_q_heads][head_dim], out_dtype PA_F32 or kv_dtype
 *   q          [num_query_tokens][num_q_heads][head_dim], kv_dtype
 *   k_cache, v_cache, num_blocks, block_tables, block_table_stride, context_lens: as in
 *              pa_decode; kv_dtype PA_F16 or PA_BF16
 *   query_start  DEVICE int32 [num_seqs + 1], non-decreasing
 *   max_query_len    >= every n_s (sizes the grid); max_context_len >= every L_s
 *   partition_size   0 = automatic split of long contexts, < 0 never split, > 0 that
 *                    many tokens per partition (a multiple of 64)
 *   workspace        DEVICE scratch of pa_chunk_workspace_bytes(...) when a split
 *                    happens (16-byte aligned, caller-owned), else may be NULL; it
 *                    must not overlap out, q, the caches, block_tables,
 *                    context_lens or query_start (PA_ERR_INVALID)
 * Supported: head_dim 64 / 128, block_size 16 / 32, num_q_heads / num_kv_heads <= 128.
 * Accumulation is fp32 on the tensor cores.  A kv head with at most 32 (token, head)
 * rows (max_query_len * num_q_heads / num_kv_heads: e.g. verifying a few speculated
 * tokens) runs on the memory-bound decode kernel in a multi-row mode, where the
 * probabilities enter P.V as hi + lo halves of the 16-bit type (fp32-level accuracy).
 * Longer chunks run on the tcgen05 kernel (256 rows per CTA), where they enter as one
 * f16 term (11 significant bits): the output is then off by at most 2^-11 of the
 * largest |v| the row weighs, plus fp32 rounding.  That kernel multiplies P with V in
 * f16, so over a bf16 cache it converts each V tile to f16 in shared memory; a V
 * element of the context with |v| >= 65536, infinite or NaN, has no f16 value: the
 * rows that weigh it come out infinite or NaN and set PA_DEVERR_RANGE.
 * Errors: invalid arguments return a negative pa_status with nothing launched.  On
 * the device, n_s > L_s, L_s > max_context_len, n_s > max_query_len or rows beyond
 * query_start[num_seqs] set PA_DEVERR_CONTEXT_LEN (the offending sequence's rows
 * become NaN; rows that no sequence owns are left unwritten); a block id outside the
 * pool sets PA_DEVERR_BLOCK_ID; see above for PA_DEVERR_RANGE.
 */
size_t pa_chunk_workspace_bytes(int64_t num_query_tokens, int32_t num_q_heads, int32_t head_dim,
                                int32_t max_context_len, int32_t partition_size);
int pa_chunk_attention(void* out, pa_dtype out_dtype, const void* q, const void* k_cache,
                       const void* v_cache, pa_dtype kv_dtype, int64_t num_blocks,
                       const int32_t* block_tables, int64_t block_table_stride,
                       const int32_t* context_lens, const int32_t* query_start,
                       int64_t num_query_tokens, int32_t max_query_len, int32_t max_context_len,
                       int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, float scale, int32_t partition_size,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_chunk_attention_fp8: pa_chunk_attention over E4M3 caches (the FP8 cache of
 * pa_decode_fp8: value = code * per-kv-head scale, k_scale / v_scale DEVICE [Hkv]).
 * q (and a native-dtype out) have q_dtype, PA_F16 or PA_BF16; out_dtype is PA_F32 or
 * q_dtype.  Short chunks (at most 32 (token, head) rows per kv head) run on a decode
 * kernel's multi-row mode, which reads the one-byte tiles directly.  Longer chunks at
 * head_dim 128 run on the tcgen05 chunk kernel, whose converter warps turn each tile
 * into f16 operands (exact) in shared memory; a bf16 query row is scaled into f16
 * range by a power of two (exact).  At head_dim 64 every chunk length takes the
 * multi-row mode.  All other arguments, rules and errors are those of
 * pa_chunk_attention (returns PA_ERR_UNSUPPORTED when called with an E4M3 kv_dtype).
 */
int pa_chunk_attention_fp8(void* out, pa_dtype out_dtype, const void* q, pa_dtype q_dtype,
                           const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, int64_t num_blocks, const int32_t* block_tables,
                           int64_t block_table_stride, const int32_t* context_lens,
                           const int32_t* query_start, int64_t num_query_tokens,
                           int32_t max_query_len, int32_t max_context_len, int32_t num_seqs,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, float scale, int32_t partition_size,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * The partition length (tokens) a pa_decode / pa_decode_fp8 call, or a
 * pa_chunk_attention call, with these arguments splits contexts into; 0 when it
 * runs one pass per sequence (no merge launch).  partition_size as in those calls;
 * the automatic choice (0) depends on the current device's SM count and the
 * kernels' occupancy.  Returns a negative pa_status for invalid arguments, or
 * PA_ERR_CUDA when the automatic choice cannot query the device.
 */
int32_t pa_decode_partition_tokens(pa_dtype q_dtype, pa_dtype kv_dtype, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t max_context_len,
                                   int32_t partition_size);
/*
 * 1 when a pa_decode / pa_decode_fp8 call with these arguments and a workspace of
 * pa_decode_workspace_bytes(...) builds the longest-first dispatch order (one more
 * launch before the decode), else 0; a negative pa_status as for
 * pa_decode_partition_tokens.
 */
int32_t pa_decode_orders_sequences(pa_dtype q_dtype, pa_dtype kv_dtype, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t max_context_len,
                                   int32_t partition_size);
int32_t pa_chunk_partition_tokens(pa_dtype kv_dtype, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int32_t max_query_len, int32_t max_context_len,
                                  int32_t partition_size);

/*
 * Name of the attention kernel a pa_decode / pa_decode_fp8 call with these arguments
 * launches: "decode_kernel" (CUDA cores), "decode_mma_kernel" (mma.sync tensor cores)
 * or "decode_tc8_kernel" (tcgen05 over E4M3 codes); NULL for arguments those calls
 * reject.  The launchers route by the same rule.  A static string; no CUDA call.
 */
const char* pa_decode_kernel_name(pa_dtype kv_dtype, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim);
/*
 * The same for pa_chunk_attention (kv_dtype PA_F16 / PA_BF16) and
 * pa_chunk_attention_fp8 (kv_dtype PA_FP8_E4M3): "chunk_attn_kernel" (tcgen05, long
 * chunks; over E4M3 caches with an f16 conversion stage) or a decode kernel's chunk-row
 * mode; NULL for arguments those calls reject.
 */
const char* pa_chunk_kernel_name(pa_dtype kv_dtype, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_query_len);

/*
 * Test hook for the bounded pipeline waits; off unless armed, and not for production
 * use.  Arms a one-shot fault that the calling thread's next pa_decode / pa_decode_fp8
 * call consumes (whichever kernel it runs; only the CUDA-core decode kernel,
 * "decode_kernel" in pa_decode_kernel_name, acts on it).  In that call the CTA with
 * linear block index cta_index (blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y *
 * blockIdx.z), grid = (partitions, kv heads x head chunks, sequences)) issues no copy of
 * the cache at all, so nothing is ever in flight for it, and its waits give up after
 * wait_limit_us microseconds instead of 2 s: the device error word gets
 * PA_DEVERR_TIMEOUT and that CTA's output rows become NaN, while every other CTA
 * computes as usual.  No GPU fault, trap or hang is involved.  Returns PA_ERR_INVALID
 * for cta_index < 0 or wait_limit_us outside [1, 1000000].
 */
int pa_test_arm_wait_timeout(int32_t cta_index, uint32_t wait_limit_us);

/*
 * Measurement helper, outside the attention path: reads every byte of buf once with
 * 16-byte loads (8 CTAs of 128 threads per SM) and XORs a checksum into
 * *sink, so that a caller timing it on `stream` learns the read-only bandwidth a
 * kernel that reads a buffer and writes almost nothing can reach (a copy benchmark
 * also writes).  buf: device, 16-byte aligned, bytes a nonzero multiple of 16;
 * sink: device uint32, caller-owned.  Asynchronous; PA_ERR_INVALID on bad arguments.
 */
int pa_stream_read(const void* buf, size_t bytes, uint32_t* sink, void* stream);

/*
 * pa_stream_read_runs: measurement helper, the read ceiling of scattered runs.  buf
 * (DEVICE, 16-byte aligned) is divided into runs of run_bytes (1024, 2048, 4096, 8192
 * or 16384); the call reads run order[i] for every i < num_runs (order: DEVICE int32,
 * values in [0, bytes / run_bytes)), CTAs taking consecutive entries as a decode CTA
 * walks a block table.  sink: DEVICE uint32[2]; sink[0] receives a checksum, sink[1]
 * counts entries outside the range (skipped).  Asynchronous on stream.  Returns
 * PA_ERR_INVALID for a null or misaligned pointer, num_runs <= 0 or another run size.
 */
int pa_stream_read_runs(const void* buf, size_t bytes, uint32_t run_bytes, const int32_t* order,
                        int64_t num_runs, uint32_t* sink, void* stream);

/*
 * Reads and clears the calling device's error word (PA_DEVERR_* bits).
 * Synchronises with `stream` to do so.  flags: host pointer.
 */
int pa_get_device_error(uint32_t* flags, void* stream);

/* Human-readable name of a pa_status value.  Never NULL. */
const char* pa_status_string(int status);

/* Library version string, e.g. "paged_kv_cache_119_gb300 0.1 sm_103a". */
const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
