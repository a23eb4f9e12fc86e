/*
 * pagedkv_blocks.h -- host-side block manager of the paged KV cache and the
 * device block copy used by copy-on-write.  Part of libpagedkv.so.
 *
 * Sources (page title, section):
 *  - "Distributed LLM Inference Serving Platform", section 2 (Mental Model):
 *    physical blocks are allocated from one pool only when needed; prompt
 *    blocks are shared by parallel completions with a reference count and
 *    cloned only when a diverging token is appended (copy-on-write).
 *  - same page, section 7 (PagedBlockManager listing): a LIFO free list,
 *    allocation that fails with an out-of-memory error when the list is
 *    empty, a reference-counted free, share = reference count + 1.
 *  - same page, Lab 1 and its worked solution: forkSequence copies the
 *    parent's block table into each child and raises every block's
 *    reference count; on the first decode step each child that appends into
 *    a shared, partially filled tail block gets a fresh block holding a copy
 *    of the tail's tokens plus its own token, while the last sharer (count
 *    back to 1) writes in place.  Full prefix blocks stay shared.
 *
 * Reading where the page's listing and its worked solution disagree: the
 * listing clones before checking whether the tail block is full (a full
 * shared block would then hold 17 tokens) and its scheduler appends the
 * clone to the table instead of replacing the tail.  This manager follows
 * the worked solution: only a partially filled shared tail is cloned, the
 * clone replaces the tail entry, and a full tail (shared or not) is followed
 * by a fresh block.
 *
 * The manager is plain host C++ (no CUDA calls) and not thread-safe: one
 * caller at a time per manager.  Slots follow the library's encoding,
 * slot = physical_block * block_size + row.
 */
#ifndef PAGEDKV_BLOCKS_H
#define PAGEDKV_BLOCKS_H

#include <stddef.h>
#include <stdint.h>

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Status of an allocation that found the free list empty. */
#define PKV_ERR_OUT_OF_BLOCKS (-6)

typedef struct pkv_block_manager pkv_block_manager;

/* A pool of num_blocks blocks of block_size tokens, all free.  NULL on bad
 * arguments or allocation failure.  Blocks are handed out LIFO, starting
 * with block num_blocks - 1. */
pkv_block_manager *pkv_bm_create(int64_t num_blocks, int block_size);
void pkv_bm_destroy(pkv_block_manager *bm);

/* Registers an empty sequence.  PKV_ERR_INVALID_ARG if the id exists. */
int pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id);

/* Child gets a copy of the parent's block table and length; every block of
 * the table gains one reference.  PKV_ERR_INVALID_ARG if the parent is
 * unknown or the child exists. */
int pkv_bm_fork(pkv_block_manager *bm, int64_t parent, int64_t child);

/*
 * Reserves the slot of the sequence's next token (host pointers):
 *  *slot          where the token's K/V go (paged_kv_append's slot_mapping)
 *  *copy_src, *copy_dst, *copy_tokens
 *                 a copy-on-write the caller must run on the device before
 *                 writing the token (paged_kv_copy_blocks): rows
 *                 [0, copy_tokens) of block copy_src to block copy_dst, all
 *                 KV heads.  copy_src = -1 when there is nothing to copy.
 * Returns PKV_ERR_OUT_OF_BLOCKS (state unchanged) when a block is needed and
 * none is free.
 */
int pkv_bm_append_slot(pkv_block_manager *bm, int64_t seq_id, int64_t *slot, int32_t *copy_src,
                       int32_t *copy_dst, int32_t *copy_tokens);

/* Drops the sequence; blocks whose reference count reaches 0 return to the
 * free list (in table order). */
int pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);

int64_t pkv_bm_num_free_blocks(const pkv_block_manager *bm);

/* Token count of a sequence (host out-pointer). */
int pkv_bm_sequence_length(const pkv_block_manager *bm, int64_t seq_id, int64_t *length);

/* Copies up to `capacity` block ids of the sequence's table into out (host)
 * and stores the table's length in *num_blocks (host). */
int pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *out,
                       int64_t capacity, int64_t *num_blocks);

/* Reference count and filled rows of a physical block (host out-pointers). */
int pkv_bm_block_info(const pkv_block_manager *bm, int32_t block, int32_t *refcount,
                      int32_t *tokens);

/*
 * Prefix groups of a batch, for paged_decode_attention_prefix_shared
 * ("Distributed LLM Inference Serving Platform", section 2 and Lab 1:
 * completions forked from one prompt share its blocks; section 5.1
 * Ingestion: a cached common prefix referenced by several requests).
 *
 * seq_ids (host, n entries) lists the batch's sequences in row order (row b
 * of q and of the block tables the caller passes to the attention).  The
 * batch is cut into maximal runs of consecutive rows whose sequences hold
 * the same physical block as their first table entry; each run is a group,
 * and its prefix is the number of leading table entries that every member
 * holds in common with the run's first sequence, times block_size (rows of
 * a shared block are never written by one sharer alone: copy-on-write gives
 * the writer its own block first).  A sequence with an empty table, or whose
 * first block no neighbour holds, is a group of one with prefix 0.  Sharers
 * must sit in consecutive rows to be grouped (forked siblings usually do).
 *  group_offsets     (host) int32 [n + 1]: group i is rows
 *                    [group_offsets[i], group_offsets[i + 1])
 *  group_prefix_lens (host) int32 [n]: prefix tokens of group i
 *  *num_groups, *max_group_size, *max_prefix_len  (host, may be NULL)
 * These are the arrays and bounds the prefix-aware attention takes (copy the
 * two arrays to the device).  PKV_ERR_INVALID_ARG on an unknown id or a null
 * array; n == 0 gives no groups.
 */
int pkv_bm_prefix_groups(const pkv_block_manager *bm, const int64_t *seq_ids, int n,
                         int32_t *group_offsets, int32_t *group_prefix_lens, int *num_groups,
                         int *max_group_size, int *max_prefix_len);

/*
 * Device block copy for copy-on-write: for each i < num_copies and every KV
 * head, rows [0, tokens[i]) of block src[i] are copied bit for bit to block
 * dst[i] in both caches (tokens == NULL: whole blocks).  src, dst, tokens are
 * device int32 arrays.  A block id outside [0, num_blocks) or a row count
 * outside [0, block_size] sets PKV_ERRBIT_SLOT in *err_word (if given) and
 * that copy is skipped.  Asynchronous on cuda_stream; allocates nothing.
 * Copies with the same dst, or whose dst is another copy's src, race.
 */
int paged_kv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src, const int32_t *dst,
                         const int32_t *tokens, int num_copies, int n_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, int32_t *err_word,
                         void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_BLOCKS_H */
