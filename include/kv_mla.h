/*
 * kv_mla.h -- decode over a paged cache of multi-head latent attention (MLA).
 *
 * xuewyang.github.io/posts/kv, "How big is the cache?" and "MLA: how does decode
 * get full-size keys and values back?": a model with MLA caches one small vector
 * per token and layer instead of per-head keys and values -- 512 latent numbers
 * c_t plus a 64-number rotary key shared by all heads (576 in all, DeepSeek-V2),
 * against 2 x 128 heads x 128 = 32,768 for multi-head attention.  In decode the
 * up-projections are absorbed: the query of head h is folded through W_UK,h
 * (q_lat,h = [W_UK,h^T q_nope,h ; q_rope,h], 576 numbers), every head scores the
 * cached vectors directly, and the attention-weighted sum of latents is
 * projected up by W_UV,h once afterwards.  Every head thus attends over one
 * shared key = value vector per token, multi-query attention with a wide head:
 *   s_t = scale * q_lat,h . c_t[0 .. 575]
 *   out_h = sum_t softmax(s)_t c_t[0 .. 511],   lse_h = log sum_t exp(s_t)
 * learn.mohebi.ai lesson 12, "Smaller caches", gives the same 512 + 64 numbers.
 *
 * This header adds the latent pool and the absorbed decode over it.  The folding
 * of W_UK into the query and of W_UV into the output are dense per-token matrix
 * products done by the caller before and after this call.
 *
 * The pool is a kv_pool (include/kv_paged.h) with one cached vector per token:
 * device memory [num_blocks, block_size, 576] bf16 (latent then rotary key), no
 * V half (kv_pool_tensors returns v_pool = NULL).  Appends go through
 * paged_kv_append with v_new = NULL and k_new = the new tokens' vectors
 * [num_tokens, 576] bf16; block copies through kv_copy_blocks.  Errors are the
 * kv_status codes and device error bits of kv_paged.h; nothing here aborts.
 */
#ifndef KV_MLA_H
#define KV_MLA_H

#include <stddef.h>
#include <stdint.h>

#include "kv_paged.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * A latent pool of num_blocks blocks of block_size tokens on `device`.
 * latent_dim must be 512 and rope_dim 64 (the kernels are laid out for them,
 * else KV_ERR_UNSUPPORTED); block_size 16, 32 or 64.  Contents start zeroed.
 */
kv_status kv_mla_pool_create(int num_blocks, int block_size, int latent_dim, int rope_dim,
                             int device, kv_pool** out);

/* Split-KV plan (see paged_decode_plan): chunk size in tokens, a multiple of
 * block_size (0 = automatic, from the batch, heads and SM count: 768 .. 2048
 * tokens), and the most chunks a sequence can have.
 *
 * Three kernels serve this call.  Latent pools with blocks of 64 tokens run a
 * tcgen05 form, accumulators in tensor memory, one CTA per SM: the wide one for at
 * least 64 query heads (tiles of 128 heads on the MMA's M dimension, each CTA
 * producing one half of the 512 latent outputs), the narrow one below that (tiles
 * of 16 heads; each MMA covers the 16 heads of a tile and 64 tokens, or 128 latent
 * numbers for the output).  Their work units ((latent half,) head tile, sequence,
 * block) are cut into equal contiguous ranges, one per CTA; a sequence cut by a
 * range boundary is merged from its pieces by a second kernel.  For them the chunk
 * argument is the least number of tokens a range holds (0 = automatic: 256 .. 1024
 * tokens), and max_splits the most pieces a sequence can be cut into.  Pools with
 * other block sizes run the mma.sync form with tiles of 16 heads, a CTA per
 * (sequence, head tile, chunk) and the merge inside the kernel. */
kv_status paged_mla_decode_plan(const kv_pool* pool, int batch, int q_heads, int max_blocks,
                                int kv_split_tokens, int* split_tokens, int* max_splits);

/* Bytes of device workspace for these sizes: the partial outputs of cut sequences
 * (fp16 in the tcgen05 forms, fp32 in the mma.sync form), an fp32 (max, sum) pair
 * per head and piece, and one 32-bit counter per (sequence, head tile[, latent
 * half]); 0 when no sequence can be cut into pieces.  The workspace must be zero-filled before its first use;
 * every call leaves the counters ready for the next.  Calls sharing a workspace
 * must not overlap in time. */
kv_status paged_mla_workspace_size(const kv_pool* pool, int batch, int q_heads, int max_blocks,
                                   int kv_split_tokens, size_t* bytes);

/*
 * Absorbed MLA decode for every sequence of a ragged batch, reading the latent
 * cache in place through the block tables (one query per sequence).
 *   q: bf16 [batch, q_heads, 576] absorbed queries (latent part then rotary part).
 *   block_tables: int32 [batch, max_blocks]; context_lens: int32 [batch]; token t
 *     of sequence b is at block block_tables[b][t / block_size], slot
 *     t % block_size; slots at or past context_lens[b] are never used.
 *   scale: softmax scale (the model's, e.g. 1/sqrt(128 + 64)).
 *   out: bf16 [batch, q_heads, 512]; lse: fp32 [batch, q_heads] natural-log
 *     log-sum-exp of the scaled scores, or NULL.  context_lens[b] == 0 gives
 *     out = 0 and lse = -inf.
 *   Bad block ids are skipped and flagged (KV_DEVERR_BLOCK_ID); out-of-range
 *   context lengths are clamped and flagged (KV_DEVERR_CONTEXT).
 *   Asynchronous on `stream` (NULL = legacy default stream); no allocation.
 *   KV_ERR_INVALID_ARG for a pool that is not a latent pool.
 */
kv_status paged_mla_decode_attention(const kv_pool* pool, const void* q, int q_heads,
                                     const int32_t* block_tables, int max_blocks,
                                     const int32_t* context_lens, int batch, float scale,
                                     int kv_split_tokens, void* workspace, size_t workspace_bytes,
                                     void* out, float* lse, void* stream);

/*
 * One decode step over a latent pool in one call: append each sequence's new cached
 * vector at position context_lens[b] - 1 (as paged_kv_append with token i = sequence i
 * and no V half), then paged_mla_decode_attention.  No separate append kernel runs:
 * each CTA that loads the block holding a sequence's new vector writes the vector into it
 * before that load (several CTAs may write the same bytes).  Pool bytes, outputs and device
 * error bits are identical to the two separate calls: a position outside the table
 * (context_lens[b] < 1 or beyond max_blocks * block_size) is flagged
 * KV_DEVERR_POSITION and not written, a bad block id KV_DEVERR_BLOCK_ID.
 *   kv_new: bf16 [batch, 576], 16-byte aligned (512 latent + 64 rotary-key numbers).
 *   Every other argument as for paged_mla_decode_attention.  All arguments are checked
 *   before anything is launched; on an error nothing is appended.
 */
kv_status paged_mla_decode_step(kv_pool* pool, const void* kv_new, const void* q, int q_heads,
                                const int32_t* block_tables, int max_blocks,
                                const int32_t* context_lens, int batch, float scale,
                                int kv_split_tokens, void* workspace, size_t workspace_bytes,
                                void* out, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KV_MLA_H */
