/*
 * kv_paged.h -- C ABI of the paged KV-cache decode library (GB300, sm_103a).
 *
 * The decode step of a serving engine over a paged KV cache:
 *   - The cache is a single pool of equal-sized blocks, made once when the
 *     engine starts; a per-sequence block table turns the sequence's logical
 *     block numbers into physical block ids, which can sit anywhere in the
 *     pool (xuewyang.github.io/posts/kv, section "PagedAttention: the KV cache
 *     in blocks").
 *   - In a decode step the new token's key and value are stored first; its
 *     query then attends over all cached tokens of the sequence, itself
 *     included (same page, section "Prefill and decode"; brunomaga.github.io
 *     "inference-prefill-decode-roofline-cache", section "PagedAttention: memory
 *     management for the KV cache", PagedKVCache.append and
 *     paged_decode_attention).
 *   - The attention kernel walks the table and reads the cache block by block,
 *     combining per-block partial results with the online-softmax update
 *     (learn.mohebi.ai lesson 12 "LLM inference serving", section
 *     "PagedAttention (4.1-4.3)"); long contexts are spread over the SMs by
 *     split-KV decoding (same lesson, section 6 "Where it shows up").
 *
 * Conventions common to every call:
 *   - All array pointers are DEVICE pointers on the pool's device, owned by the
 *     caller, except the pool's own K/V/scale memory (owned by the pool).
 *     Tensor data (q, k_new, v_new, out, workspace) must be 16-byte aligned;
 *     int32 / float arrays 4-byte aligned.
 *   - The calling thread's current CUDA device must be the pool's device.
 *   - `stream` is a cudaStream_t (NULL: the legacy default stream).  append and
 *     decode only enqueue work: they never allocate, never synchronise and
 *     never read device memory on the host, so they may be captured in a CUDA
 *     graph.  Their results are ready when the stream reaches them.
 *   - Errors detectable on the host (shapes, pointers, alignment, sizes) are
 *     returned before anything is launched.  Values that live on the device
 *     (block ids, context lengths, sequence indices) are checked by the
 *     kernels: a bad entry is skipped or clamped, never dereferenced, and a
 *     bit is set in the pool's device error word (kv_pool_device_errors).
 *   - No call aborts the process and no C++ exception crosses this ABI.
 */
#ifndef KV_PAGED_H
#define KV_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KV_PAGED_ABI_VERSION 1

typedef enum kv_status {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,     /* a host-checkable argument is wrong; nothing was launched */
    KV_ERR_OUT_OF_MEMORY = 2,   /* the pool allocation failed */
    KV_ERR_OUT_OF_BLOCKS = 3,   /* reserved for a host block allocator (no free block left) */
    KV_ERR_UNSUPPORTED = 4,     /* valid but not implemented (head_dim, block_size, dtype combo) */
    KV_ERR_CUDA = 5,            /* a CUDA runtime/driver call or a launch failed */
    KV_ERR_DEVICE_CHECK = 6     /* kv_pool_device_errors found device-side error bits */
} kv_status;

typedef enum kv_dtype {
    KV_DTYPE_BF16 = 0,          /* cache stores bf16 values bit for bit */
    KV_DTYPE_FP8_E4M3 = 1       /* cache stores OCP e4m3fn codes, value = code * scale[kv_head] */
} kv_dtype;

/* Bits of the pool's device error word. */
#define KV_DEVERR_BLOCK_ID 0x1u  /* a block-table entry outside [0, num_blocks) was skipped */
#define KV_DEVERR_CONTEXT  0x2u  /* a context length < 0 or > max_blocks * block_size was clamped */
#define KV_DEVERR_SEQ      0x4u  /* an appended token named a sequence outside [0, batch) */
#define KV_DEVERR_POSITION 0x8u  /* an appended token's position was < 0 or past the table */
#define KV_DEVERR_TIMEOUT  0x10u /* a pipeline wait gave up after its time limit (about 2 s) */

typedef struct kv_pool kv_pool;  /* opaque; owned by the library */

/* ABI version of the loaded library (KV_PAGED_ABI_VERSION when built). */
int kv_abi_version(void);

/* Static, never-NULL description of a status code. */
const char* kv_status_string(kv_status status);

/*
 * kv_pool_create -- one allocation holding the K pool, the V pool, the
 * per-kv-head fp8 scales and the device error word.  A single allocation at
 * start-up keeps every address fixed for the life of the pool, which is what
 * CUDA-graph capture of the step relies on (xuewyang.github.io/posts/kv,
 * section "Why vLLM sizes the cache at startup").
 *   K and V: [num_blocks, block_size, kv_heads, head_dim] elements each (the
 *   vLLM per-layer layout of that page's "Reading the code" section, with K and
 *   V as the two halves).  Token slot `s` of block `b` holds every kv head of
 *   one token.  Initial contents: all bytes zero; fp8 scales 1.0.
 *   Supported: block_size 16 or 32; bf16 with head_dim 64 or 128; fp8 e4m3
 *   with head_dim 128; kv_heads >= 1; num_blocks >= 1 and the pool below 2^40
 *   bytes.  One pool serves one layer.
 *   device: CUDA ordinal; the pool's memory lives there.  The caller's current
 *   device is restored before returning.
 *   Errors: KV_ERR_INVALID_ARG (NULL out, sizes <= 0), KV_ERR_UNSUPPORTED,
 *   KV_ERR_OUT_OF_MEMORY, KV_ERR_CUDA (no such device, tensor-map encoding).
 *   On error *out is set to NULL.
 */
kv_status kv_pool_create(int num_blocks, int block_size, int kv_heads, int head_dim,
                         kv_dtype dtype, int device, kv_pool** out);

/* Frees the pool's memory (synchronises the device first).  NULL is a no-op. */
kv_status kv_pool_destroy(kv_pool* pool);

/*
 * Device addresses of the pool's arrays (any output pointer may be NULL):
 * K and V pools as above, k_scale / v_scale float32 [kv_heads] (meaningful for
 * the fp8 cache; 1.0 otherwise).  The pointers stay valid until destroy.
 */
kv_status kv_pool_tensors(const kv_pool* pool, void** k_pool, void** v_pool,
                          float** k_scale, float** v_scale);

/* Shape of the pool (any output pointer may be NULL). */
kv_status kv_pool_shape(const kv_pool* pool, int* num_blocks, int* block_size, int* kv_heads,
                        int* head_dim, kv_dtype* dtype, int* device);

/*
 * Copies per-kv-head scales from HOST arrays of kv_heads floats into the pool
 * (synchronous; a set-up call, not part of the step).  Scales must be finite
 * and > 0.  Either pointer may be NULL to leave that scale unchanged.
 */
kv_status kv_pool_set_scales(kv_pool* pool, const float* k_scale_host, const float* v_scale_host);

/*
 * Reads the pool's device error word (synchronises the device).  *bits gets
 * the KV_DEVERR_* bits raised by kernels since the last clear; clear != 0
 * resets it.  Returns KV_ERR_DEVICE_CHECK when any bit is set, else KV_OK.
 */
kv_status kv_pool_device_errors(kv_pool* pool, uint32_t* bits, int clear);

/*
 * paged_kv_append -- writes the key and value of num_tokens tokens into the
 * pool: the token at position p lands in table entry p / block_size at slot
 * p % block_size (xuewyang.github.io/posts/kv, sections "A toy vLLM" (write_kv)
 * and "Reading the code: a warehouse of lockers"; brunomaga.github.io,
 * PagedKVCache.append).
 *   k_new, v_new: bf16 [num_tokens, kv_heads, head_dim].
 *   token_seq: int32 [num_tokens] sequence of each token, or NULL for token i
 *     -> sequence i (then num_tokens <= batch).
 *   token_pos: int32 [num_tokens] position of each token, or NULL for
 *     context_lens[seq] - 1 (the decode step: context_lens counts the token
 *     being appended).
 *   block_tables: int32 [batch, max_blocks]; context_lens: int32 [batch]
 *     (read only when token_pos is NULL).
 *   Token at position p of sequence s goes to block
 *   block_tables[s][p / block_size], slot p % block_size, for every kv head.
 *   bf16 pools store the input bits unchanged; fp8 pools store
 *   e4m3fn(round-to-nearest-even, saturating at +-448)(x / scale[kv_head])
 *   with the quotient rounded to binary32 first.
 *   Block allocation (and copy-on-write of shared blocks) is the caller's job:
 *   the entry must already name a block the sequence owns.
 *   Two tokens written to the same slot in one call race (either may win).
 *   num_tokens == 0 is a no-op.
 */
kv_status paged_kv_append(kv_pool* pool, const void* k_new, const void* v_new, int num_tokens,
                          const int32_t* token_seq, const int32_t* token_pos,
                          const int32_t* block_tables, int max_blocks,
                          const int32_t* context_lens, int batch, void* stream);

/*
 * Resolves the split-KV plan paged_decode_attention will use for these
 * sizes: *split_tokens (a multiple of block_size) and *max_splits (the most
 * chunks any sequence can have, ceil(max_blocks * block_size / split_tokens)).
 * kv_split_tokens: 0 = automatic (from batch, heads, max_blocks and the SM
 * count; between 64 and 192 blocks, 128 at most where one CTA covers two kv
 * heads), else a positive multiple of block_size.
 * KV_ERR_UNSUPPORTED when max_splits would exceed 65535.  Either output may
 * be NULL.
 */
kv_status paged_decode_plan(const kv_pool* pool, int batch, int q_heads, int max_blocks,
                            int kv_split_tokens, int* split_tokens, int* max_splits);

/*
 * The CTA layout paged_decode_attention (q_len = 1), paged_attention_multi_query and
 * paged_decode_step use for these sizes: *cta_heads = the kv heads one CTA covers --
 * 1 (one CTA per kv head and query-row tile) or 2 / 4 (one CTA per group of kv heads,
 * chosen with the automatic chunk for the pool layouts it is built for: bf16, head_dim
 * 128, blocks of 16 -> 2; fp8, head_dim 128, blocks of 32 -> 4; rows of a kv head <= 8).
 * Diagnostic only: both layouts compute the same attention.  Same errors as
 * paged_decode_plan.
 */
kv_status paged_decode_cta_heads(const kv_pool* pool, int batch, int q_heads, int q_len,
                                 int max_blocks, int kv_split_tokens, int* cta_heads);

/*
 * Bytes of device workspace paged_decode_attention needs for these sizes
 * (fp32 partial outputs, maxima and sums of the split-KV chunks, and one
 * 32-bit chunk counter per (sequence, kv head, head tile)); 0 when every
 * sequence fits one chunk.
 */
kv_status paged_decode_workspace_size(const kv_pool* pool, int batch, int q_heads,
                                      int max_blocks, int kv_split_tokens, size_t* bytes);

/*
 * paged_decode_attention -- single-query attention for every sequence of a
 * ragged batch, reading the cache in place through the block tables.
 *   q: bf16 [batch, q_heads, 1, head_dim] (the new token's query).
 *   Query head h uses kv head h / (q_heads / kv_heads): contiguous groups of
 *   g = q_heads / kv_heads query heads share one kv head (GQA; g = 1 is MHA),
 *   and all g heads of a group are computed from one read of that head's K/V.
 *   block_tables: int32 [batch, max_blocks]; context_lens: int32 [batch],
 *   counting the token appended in this step; tokens 0 .. ctx-1 of sequence b
 *   are at block_tables[b][t / block_size], slot t % block_size.  Slots at or
 *   past ctx in the last block are never used.  Entries past a sequence's
 *   blocks are not read.  ctx == 0 gives out = 0 and lse = -inf.
 *   out[b, h, :] = sum_t softmax_t(scale * q[b,h,:] . K[t, h/g, :]) V[t, h/g, :]
 *     as bf16 [batch, q_heads, head_dim] (round to nearest even), fp32
 *     accumulation; for the fp8 cache K and V are the dequantised values
 *     code * scale[kv_head].
 *   lse_out: optional float32 [batch, q_heads], natural-log log-sum-exp of the
 *     scaled scores (NULL to skip).
 *   kv_split_tokens: split-KV chunk in tokens (0 = automatic; else a positive
 *     multiple of block_size).  Chunk j of a sequence covers tokens
 *     [j * split, (j+1) * split); the chunks of a sequence are merged by
 *     log-sum-exp by whichever of its chunk CTAs finishes last.  The result
 *     does not depend on the split up to rounding.
 *   workspace: device memory of at least paged_decode_workspace_size() bytes
 *     (may be NULL when that size is 0).  It must be zero-filled before its
 *     first use: it holds the counters that tell the last chunk of a sequence
 *     to merge the others, and every successful call leaves them at zero
 *     again.  After a call that raised KV_DEVERR_TIMEOUT, zero it before
 *     reuse.  One kernel launch per call: the merge happens inside it.
 *   q_heads must be a positive multiple of the pool's kv_heads.
 *   Concurrent calls that share a workspace on different streams race.
 */
kv_status paged_decode_attention(const kv_pool* pool, const void* q, int q_heads,
                                 const int32_t* block_tables, int max_blocks,
                                 const int32_t* context_lens, int batch, float scale,
                                 int kv_split_tokens, void* workspace, size_t workspace_bytes,
                                 void* out, float* lse_out, void* stream);

/*
 * paged_decode_attention_split_merge -- the same attention in two kernels: the
 * split-KV grid leaves the fp32 partial (normalised output, maximum, sum) of
 * every chunk of a cut sequence in the workspace, and a separate log-sum-exp
 * merge kernel combines them (learn.mohebi.ai lesson 12, section 6: split-KV
 * decoding).  Sequences of one chunk are finished by the grid.  The merge does
 * the fused form's arithmetic in the same order: outputs and lse are bit-
 * identical to paged_decode_attention with the same arguments.
 *   Arguments, workspace size and errors as for paged_decode_attention; the
 *   workspace's chunk counters are not used (it need not be zero-filled).
 *   Two kernel launches when some sequence can have more than one chunk, one
 *   otherwise.
 */
kv_status paged_decode_attention_split_merge(const kv_pool* pool, const void* q, int q_heads,
                                             const int32_t* block_tables, int max_blocks,
                                             const int32_t* context_lens, int batch, float scale,
                                             int kv_split_tokens, void* workspace,
                                             size_t workspace_bytes, void* out, float* lse_out,
                                             void* stream);

/*
 * paged_merge_attention_states -- combines attention results over disjoint key
 * sets into the result over their union: source r attended over its own keys
 * and gave o_r and lse_r, and
 *   LSE = log sum_r exp(lse_r),   out = sum_r exp(lse_r - LSE) o_r
 * (the log-sum-exp merge of split-KV decoding, learn.mohebi.ai lesson 12,
 * section 6, with the chunks' (max, sum) pairs folded into lse).  It is the one
 * exchange a sequence split across devices needs: each device runs
 * paged_decode_attention over its share of the sequence's blocks (with
 * lse_out), the (out, lse) pairs are gathered, and this call merges them.
 *   outs: bf16 [n_src, rows, head_dim], 16-byte aligned; lses: fp32 [n_src,
 *   rows], natural log, -inf for a source that saw no key (left out).
 *   out: bf16 [rows, head_dim] (round to nearest even), 16-byte aligned;
 *   lse_out: fp32 [rows] or NULL.  A row whose sources are all empty gets
 *   out = 0, lse = -inf.
 *   n_src >= 1; head_dim a multiple of 8 in [8, 1024]; rows == 0 is a no-op.
 *   fp32 arithmetic.  Runs on the calling thread's current CUDA device (all
 *   pointers must be device memory of that device), asynchronously on `stream`
 *   (NULL = legacy default stream); no allocation.  out must not overlap outs.
 */
kv_status paged_merge_attention_states(const void* outs, const float* lses, int n_src,
                                       long long rows, int head_dim, void* out, float* lse_out,
                                       void* stream);

/*
 * paged_attention_multi_query -- attention of q_len new tokens per sequence
 * over the paged cache: the verify pass of speculative decoding (the target
 * model scores the draft's guesses in one pass) and the chunks of a chunked
 * prefill.  The q_len new tokens must already be appended; query token i of
 * sequence b sits at position context_lens[b] - q_len + i and attends to keys
 * 0 .. that position -- the shifted causal mask of cached attention
 * (xuewyang.github.io/posts/kv, "A KV cache in PyTorch"; 4yush.com "The KV
 * cache and the systems around it", section "Why the keys and values never
 * change").
 *   q: bf16 [batch, q_heads, q_len, head_dim]; out: bf16 [batch, q_heads,
 *   q_len, head_dim]; lse_out: optional float32 [batch, q_heads, q_len].
 *   The g = q_heads / kv_heads heads of a group and the q_len query tokens
 *   (g * q_len rows, at most 4096) share each read of a K/V block.
 *   context_lens[b] < q_len (but > 0) is a device-side error
 *   (KV_DEVERR_CONTEXT); queries whose position would be negative attend to
 *   nothing.  Everything else (tables, split, workspace, errors) as in
 *   paged_decode_attention, which is this call with q_len == 1.
 */
kv_status paged_attention_multi_query(const kv_pool* pool, const void* q, int q_heads, int q_len,
                                      const int32_t* block_tables, int max_blocks,
                                      const int32_t* context_lens, int batch, float scale,
                                      int kv_split_tokens, void* workspace,
                                      size_t workspace_bytes, void* out, float* lse_out,
                                      void* stream);

/* Workspace bytes of paged_attention_multi_query for these sizes. */
kv_status paged_multi_query_workspace_size(const kv_pool* pool, int batch, int q_heads,
                                           int q_len, int max_blocks, int kv_split_tokens,
                                           size_t* bytes);

/*
 * paged_decode_step -- one decode step of every sequence of the batch: the
 * append of its q_len new tokens (xuewyang.github.io/posts/kv, "A toy vLLM",
 * write_kv: the new token is appended first) followed by their attention over
 * the cache (paged_attention_multi_query), both enqueued on `stream`.
 *   k_new, v_new: bf16 [batch * q_len, kv_heads, head_dim]; row i is token
 *     i % q_len of sequence i / q_len, written at position
 *     context_lens[b] - q_len + i % q_len (context_lens already counts the new
 *     tokens).  The pool must not be a latent pool (KV_ERR_INVALID_ARG).
 *   Everything else -- q, tables, lengths, split, workspace, outputs, device
 *   error bits -- as in paged_attention_multi_query; all arguments are checked
 *   before anything is launched, so an error leaves the pool untouched.
 *   The result equals paged_kv_append (with those positions) followed by
 *   paged_attention_multi_query: the same pool bytes, the same output bits.
 *   Where a kv head's query rows (q_heads / kv_heads * q_len) fit one 8-row
 *   tile it is one kernel launch: the CTA that reads a block holding one of
 *   the new tokens writes that token's rows of its kv heads into the pool
 *   first (bf16 copied, fp8 quantised exactly as paged_kv_append does), then
 *   loads the block; new tokens whose position lies outside the block table
 *   are not written and set KV_DEVERR_POSITION, as the append would.  With
 *   more rows it is paged_kv_append's kernel followed by the attention's.
 */
kv_status paged_decode_step(kv_pool* pool, const void* k_new, const void* v_new, const void* q,
                            int q_heads, int q_len, const int32_t* block_tables, int max_blocks,
                            const int32_t* context_lens, int batch, float scale,
                            int kv_split_tokens, void* workspace, size_t workspace_bytes,
                            void* out, float* lse_out, void* stream);

/*
 * Test hook of the failure path of the decode kernels; the pages have no
 * counterpart (their engines raise on the host; this library's kernels bound
 * every pipeline wait instead, see KV_DEVERR_TIMEOUT).  Process-wide, read by
 * every later paged_decode_attention / paged_attention_multi_query /
 * paged_decode_step / split-merge / no-alloc launch:
 *   stop_stage: the producer of each CTA issues no load for the stages of its
 *     chunk from this index on (-1, the default: off), so the consumers' wait
 *     for that stage can only run out: they set KV_DEVERR_TIMEOUT, leave their
 *     loop and write what they have (the outputs are then meaningless), while
 *     every load that was issued lands before the CTA exits;
 *   consumer_wait_ns: the consumers' limit for a stage wait (0: the default,
 *     two seconds); the producer's waits keep the default.
 * KV_ERR_INVALID_ARG for stop_stage < -1.  Not for production use: call
 * kv_debug_decode_stall(-1, 0) to restore normal operation.
 */
kv_status kv_debug_decode_stall(int stop_stage, unsigned long long consumer_wait_ns);

/*
 * Allocation-free decode attention.  The paper has no counterpart to this call;
 * it exists for users of this library who cannot allocate device memory at the
 * call site: plug-in hosts that give a kernel only its input and output
 * buffers, engines whose own allocator has already reserved the whole GPU, and
 * latency-critical paths where cudaMalloc's implicit device-wide
 * synchronisation would stall other streams.
 *
 * Same arguments and result as paged_decode_attention, without the workspace:
 * the split-KV partials go to a static device array of
 * KV_NO_ALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  The call itself allocates
 * nothing (no cudaMalloc, no library allocator).
 *   - Returns KV_ERR_UNSUPPORTED, before launching anything, when the partials
 *     for these sizes (paged_decode_workspace_size) exceed
 *     KV_NO_ALLOC_SCRATCH_BYTES; pick a larger kv_split_tokens or use
 *     paged_decode_attention with your own workspace.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture.  The address is kept for the life of the process, so a
 *     cudaDeviceReset after that first call is not supported: the array is
 *     created again at a new address that this call would not see.
 *   - Arguments are validated before the array is touched: a rejected call
 *     writes nothing to it and launches nothing.
 *   - All calls on a device share the one array, which keeps what the last
 *     call left.  The chunk counters that must start at zero are cleared by
 *     each call on its stream before its kernel; the partial results need no
 *     clearing.  Calls whose kernels overlap on the GPU (different streams
 *     without ordering) race on the array and may corrupt each other's
 *     results.
 */
#define KV_NO_ALLOC_SCRATCH_BYTES (8u << 20)

kv_status paged_decode_attention_noalloc(const kv_pool* pool, const void* q, int q_heads,
                                         const int32_t* block_tables, int max_blocks,
                                         const int32_t* context_lens, int batch, float scale,
                                         int kv_split_tokens, void* out, float* lse_out,
                                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KV_PAGED_H */
