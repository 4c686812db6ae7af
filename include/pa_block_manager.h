/*
 * pa_block_manager.h -- C ABI of the host-side KV block manager (in libpa.so).
 *
 * The manager owns no device memory.  It decides, for every sequence, which
 * physical blocks of a pool of num_blocks blocks hold its tokens, and emits what
 * the CUDA kernels consume: the int64 slot of each new token (for
 * pa_reshape_and_cache), int32 block-table rows and context lengths (for
 * pa_decode), and (src, dst) copy pairs (for pa_copy_blocks).
 *
 * Semantics ("PagedAttention 完全拆解", sections 原理详解（一） (Figure 6), 内存共享 /
 * 引用计数 (Figure 8), Beam Search (Figure 9) and 三种原语：fork、append、free):
 *   - a sequence's tokens fill logical blocks left to right; a new physical block
 *     is taken from the free list only when the last block is full (Figure 6);
 *   - every physical block has a reference count (the number of sequences whose
 *     table names it);
 *   - fork: the child gets a copy of the parent's block table, and every block's
 *     count goes up by one;
 *   - append: before the new token is written into the sequence's last block,
 *     if that block is shared (count > 1) a new block is taken, the old block's
 *     contents are scheduled to be copied into it (a copy pair), the old count
 *     goes down by one and the sequence's table points at the new block
 *     (copy-on-write: the writer takes the copy, the others keep the original);
 *   - free: every block's count goes down by one; blocks reaching zero return to
 *     the free list.
 * The free list is first-in first-out: blocks are handed out in the order given
 * at creation (or 0, 1, 2, ...) and freed blocks are reused after all blocks
 * that were free before them.
 *
 * Errors: every call returns PA_OK or a negative pa_status (PA_ERR_INVALID for an
 * unknown or duplicate sequence id, a bad argument or an exhausted pool; on an
 * exhausted pool nothing is changed).  Not thread-safe: one manager per thread.
 */
#ifndef PA_BLOCK_MANAGER_H_
#define PA_BLOCK_MANAGER_H_

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

/* A manager for num_blocks blocks of block_size tokens.  alloc_order: NULL, or a
 * HOST array of num_blocks distinct ids in [0, num_blocks) giving the free list's
 * initial order.  Returns NULL on invalid arguments or allocation failure. */
pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* alloc_order);
void pa_bm_destroy(pa_block_manager* bm);

/* Registers sequence seq_id with num_tokens prompt tokens and allocates their
 * blocks.  slots_out (HOST, num_tokens entries, may be NULL) receives the slot of
 * each prompt token in order. */
int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, int32_t num_tokens,
                       int64_t* slots_out);

/* The child shares every block of the parent (fork). */
int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id);

/* Reserves the slot of one new token of every listed sequence, in list order
 * (one decode step of a batch).  slots_out (HOST, n entries) receives the slots;
 * pairs_out (HOST, room for 2 * n int64) receives the copy-on-write pairs as
 * (src, dst) and *num_pairs their count.  All-or-nothing: if the pool cannot serve
 * the whole step, nothing changes and PA_ERR_INVALID is returned. */
int pa_bm_append(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                 int64_t* pairs_out, int32_t* num_pairs);

/* Drops the sequence; blocks whose count reaches zero return to the free list. */
int pa_bm_free(pa_block_manager* bm, int64_t seq_id);

/* Block-table rows and context lengths for a batch: row i of table_out (HOST,
 * n x stride int32) gets sequence seq_ids[i]'s physical blocks, padded with -1;
 * context_lens_out[i] its token count.  PA_ERR_INVALID if a row needs more than
 * stride entries. */
int pa_bm_block_tables(const pa_block_manager* bm, const int64_t* seq_ids, int32_t n,
                       int32_t* table_out, int32_t stride, int32_t* context_lens_out);

int32_t pa_bm_num_free_blocks(const pa_block_manager* bm);
/* Reference count of a physical block (0 = free), or -1 for an invalid id. */
int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block);
/* Token count of a sequence, or -1 if unknown. */
int32_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq_id);

/*
 * Swapping ("PagedAttention 完全拆解", section 调度与抢占：内存不够时怎么办, 换出
 * (Swapping)): a preempted sequence group moves to CPU memory as a whole and comes
 * back as a whole; the pages' workers keep a CPU block allocator beside the GPU one.
 *
 * pa_bm_set_cpu_pool: gives the manager a CPU pool of num_cpu_blocks block ids
 * (0 .. num_cpu_blocks-1, handed out first-in first-out).  Once, before swapping.
 *
 * pa_bm_swap_out: every distinct GPU block of the listed sequences (in order of first
 * appearance) gets one CPU block; pairs_out (HOST, room for max_pairs pairs) receives
 * (gpu block, cpu block) pairs -- the pairs pa_swap_blocks takes to copy the GPU pools
 * into the CPU pools -- and *num_pairs their count.  Blocks the group shares stay
 * shared on the CPU (one copy, the group's references counted on it); the group's
 * references leave the GPU blocks, which return to the free list when no other
 * sequence names them.  The sequences are then swapped out: pa_bm_append, pa_bm_fork
 * and pa_bm_block_tables refuse them; pa_bm_free releases their CPU blocks.
 * pa_bm_swap_in: the reverse, with (cpu block, gpu block) pairs for pa_swap_blocks
 * from the CPU pools into the GPU pools; sharing is preserved again.
 * Both are all-or-nothing: PA_ERR_INVALID with nothing changed if no CPU pool was set,
 * a sequence is unknown, listed twice or already on the target side, the target pool
 * has too few free blocks, or the pairs do not fit in max_pairs.
 */
int pa_bm_set_cpu_pool(pa_block_manager* bm, int32_t num_cpu_blocks);
int pa_bm_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs_out,
                   int32_t max_pairs, int32_t* num_pairs);
int pa_bm_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs_out,
                  int32_t max_pairs, int32_t* num_pairs);
int32_t pa_bm_num_free_cpu_blocks(const pa_block_manager* bm);
/* Reference count of a CPU block (0 = free), or -1 for an invalid id. */
int32_t pa_bm_cpu_ref_count(const pa_block_manager* bm, int32_t block);
/* 1 if the sequence is swapped out, 0 if on the GPU, -1 if unknown. */
int32_t pa_bm_is_swapped(const pa_block_manager* bm, int64_t seq_id);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H_ */
