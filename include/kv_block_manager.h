/*
 * kv_block_manager.h -- host-side allocator of the paged KV pool's blocks.
 *
 * The bookkeeping around the pool, as the pages describe it:
 *   - A free list of physical blocks; a sequence takes a new block only when its
 *     last one is full, and gives all of its blocks back when it finishes or is
 *     preempted (xuewyang.github.io/posts/kv, "PagedAttention: the KV cache in
 *     blocks" and "A toy vLLM"; brunomaga.github.io, PagedKVCache.append / free).
 *   - Reference counts on shared blocks and copy-on-write: a sequence about to
 *     write into a block that other sequences also hold gets a private copy first
 *     (learn.mohebi.ai lesson 12, "PagedAttention", sharing 4.4).
 *   - Automatic prefix caching: each full block is named by a hash chained over
 *     the previous block's hash and its own token ids; a new prompt reuses cached
 *     blocks from its start up to the first miss; blocks that no sequence holds
 *     stay cached and are evicted least recently used first; an optional salt is
 *     mixed into the first block's hash so that requests with different salts
 *     never share blocks (brunomaga.github.io, "Prefix caching"; kongchang.com,
 *     "Automatic Prefix Caching").
 *
 * Everything here is host memory and host code (no CUDA call), guarded by one
 * mutex per manager.  Block ids are indices into a kv_pool of the same size; the
 * manager never touches the pool's contents: copy-on-write reports the copies
 * the caller must make on the device (kv_copy_blocks) before it writes.
 * Sequence ids are caller-chosen 64-bit values.  No call aborts or throws; all
 * return a kv_status (KV_ERR_INVALID_ARG for unknown sequences and bad sizes,
 * KV_ERR_OUT_OF_BLOCKS when the pool cannot hold a request, state unchanged).
 */
#ifndef KV_BLOCK_MANAGER_H
#define KV_BLOCK_MANAGER_H

#include <stddef.h>
#include <stdint.h>

#include "kv_paged.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kv_block_manager kv_block_manager;

/* Free-list order.  FIFO hands out the oldest free block first and is the
 * order of the first page's toy engine (pop from the front, return to the
 * back); LIFO hands out the most recently freed block first, like the second
 * page's PagedKVCache (pop from the back). */
#define KV_BM_FIFO 0x0
#define KV_BM_LIFO 0x1
/* Keep full blocks of finished sequences cached for prefix reuse. */
#define KV_BM_PREFIX_CACHING 0x2

/* One block copy a caller must make (device side) before writing: copy-on-write. */
typedef struct kv_block_copy {
    int32_t src;
    int32_t dst;
} kv_block_copy;

/* A manager of num_blocks blocks of block_size tokens; flags: KV_BM_* bits. */
kv_status kv_bm_create(int num_blocks, int block_size, int flags, kv_block_manager** out);
kv_status kv_bm_destroy(kv_block_manager* bm);

/* Registers an empty sequence (no blocks); salt is mixed into its first block's
 * hash (0: none).  KV_ERR_INVALID_ARG if the id is taken. */
kv_status kv_bm_add_sequence(kv_block_manager* bm, int64_t seq, uint64_t salt);

/* child becomes a new sequence sharing all of parent's blocks and tokens
 * (parallel sampling, beam search): every shared block's count goes up by one. */
kv_status kv_bm_fork(kv_block_manager* bm, int64_t parent, int64_t child);

/*
 * Reserves slots for n_tokens new tokens at the end of the sequence, taking new
 * blocks on demand (from the free list, else by evicting the least recently used
 * cached block).  If the sequence's last block is partly filled and shared, it is
 * first replaced by a private copy: the copy to make is written to *copy and
 * *n_copies is set to 1 (else 0).  token_ids (may be NULL) are the tokens' ids;
 * with prefix caching, every block they complete is registered under its chained
 * hash.  All-or-nothing: KV_ERR_OUT_OF_BLOCKS leaves the manager unchanged.
 * After the call the tokens sit at positions old_length .. old_length + n - 1 of
 * the sequence's block table.
 */
kv_status kv_bm_append_slots(kv_block_manager* bm, int64_t seq, int n_tokens,
                             const int32_t* token_ids, kv_block_copy* copy, int* n_copies);

/*
 * For a sequence with no tokens yet: walks the full blocks of the prompt
 * (token_ids, n_tokens), chaining hashes from the sequence's salt, and adopts
 * each cached block whose hash and tokens match, stopping at the first miss.
 * *cached_tokens = number of leading tokens now in the cache (a multiple of
 * block_size); the caller prefills the rest.  Without KV_BM_PREFIX_CACHING it is
 * always 0.
 */
kv_status kv_bm_match_prefix(kv_block_manager* bm, int64_t seq, const int32_t* token_ids,
                             int n_tokens, int* cached_tokens);

/* Releases the sequence's blocks (finish or preemption): each count goes down by
 * one; a block no longer held goes back to the free list, or -- with prefix
 * caching, if it is registered -- to the cached-and-evictable list (the tail of the
 * sequence is evicted first).  The sequence id is forgotten. */
kv_status kv_bm_free_sequence(kv_block_manager* bm, int64_t seq);

/* Blocks that a new allocation can take (free + cached-and-evictable). */
kv_status kv_bm_num_free_blocks(const kv_block_manager* bm, int* n_free, int* n_cached_evictable);

/* Number of tokens and blocks of a sequence. */
kv_status kv_bm_sequence_info(const kv_block_manager* bm, int64_t seq, int* n_tokens,
                              int* n_blocks);

/* Reference count of a block (0 for free or cached-and-evictable blocks). */
kv_status kv_bm_block_refcount(const kv_block_manager* bm, int32_t block, int* refcount);

/*
 * Host arrays for the kernels: block_tables [batch, max_blocks] (entries past a
 * sequence's blocks are -1) and context_lens [batch] (the sequences' token
 * counts), for the listed sequences in order.  KV_ERR_INVALID_ARG if a
 * sequence is unknown or holds more than max_blocks blocks.
 */
kv_status kv_bm_build_tables(const kv_block_manager* bm, const int64_t* seqs, int batch,
                             int max_blocks, int32_t* block_tables, int32_t* context_lens);

/*
 * Device: copies whole blocks of the pool (K and V, every slot and kv head),
 * copies[i].src -> copies[i].dst for i < n, on the stream.  copies is a DEVICE
 * array of n kv_block_copy.  Ids outside the pool are skipped and flagged
 * (KV_DEVERR_BLOCK_ID).  Pairs must not overlap (no block both source and
 * destination).  n == 0 is a no-op.
 */
kv_status kv_copy_blocks(kv_pool* pool, const kv_block_copy* copies, int n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KV_BLOCK_MANAGER_H */
