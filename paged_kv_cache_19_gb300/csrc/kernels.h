// kernels.h -- parameter blocks and launchers shared by the host layer and the
// CUDA translation units.  Internal to the library (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

struct kv_block_copy;

namespace kvp {

// One CTA of the main decode kernel covers (sequence, kv head, head group,
// split).  All pointers are device pointers.
// Query rows: q and out are [batch, q_heads, q_len, head_dim], i.e. rows
// (b * kv_heads + kvh) * rows + r with rows = group * q_len per kv head and
// r = (head in the group) * q_len + (query token).  Query token i of a
// sequence sits at position ctx - q_len + i and sees keys 0 .. that position.
struct DecodeParams {
    const uint16_t* q;        // bf16 [batch, q_heads, q_len, head_dim]
    const int32_t* tables;    // [batch, max_blocks]
    const int32_t* ctx;       // [batch]
    const float* k_scale;     // [kv_heads] (fp8 cache)
    const float* v_scale;     // [kv_heads] (fp8 cache)
    uint16_t* out;            // bf16 [batch, q_heads, q_len, head_dim]
    float* lse;               // [batch, q_heads, q_len] or null
    float* part_o;            // [batch, q_heads, q_len, max_splits, head_dim]
    float* part_ml;           // [batch, q_heads, q_len, max_splits, 2]: (max, sum), log2 units
    uint32_t* err;            // device error word
    int* tickets;             // per-unit count of finished chunks; zero between calls
    int batch, q_heads, kv_heads, group, head_groups;
    int q_len, rows;          // query tokens per sequence; rows per kv head = group * q_len
    int max_blocks, num_blocks;
    int split_blocks, max_splits;   // chunk length in blocks; most chunks a sequence can have
    float scale_log2;         // softmax scale * log2(e)
    // paged_decode_step: the step's new tokens (bf16 [batch * q_len, kv_heads, head_dim],
    // token t of sequence b at row b * q_len + t, position ctx - q_len + t), which the CTA
    // reading a block writes into the pool halves before it loads that block; null for the
    // attention alone.
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint8_t* k_pool;
    uint8_t* v_pool;
    // 0: the last chunk CTA of a cut sequence merges the chunks (tickets).  1: chunk CTAs
    // only leave their partials, and paged_decode_merge (launch_decode_merge) merges them.
    int merge_kernel;
    // Failure-path test hook (kv_debug_decode_stall): the producer issues no load for a
    // chunk's stages from stop_stage on (-1: all), and the consumers give up a stage wait
    // after consumer_wait_ns instead of WAIT_LIMIT_NS (0: the default).
    int stop_stage;
    unsigned long long consumer_wait_ns;
};

struct AppendParams {
    const uint16_t* k_new;    // bf16 [num_tokens, kv_heads, head_dim]
    const uint16_t* v_new;
    const int32_t* token_seq; // or null
    const int32_t* token_pos; // or null
    const int32_t* tables;
    const int32_t* ctx;
    uint8_t* k_pool;
    uint8_t* v_pool;
    const float* k_scale;
    const float* v_scale;
    uint32_t* err;
    int num_tokens, batch, max_blocks, num_blocks, block_size, kv_heads, head_dim;
    int fp8;
    int q_len;                // without token_seq / token_pos: token i is token i % q_len of
                              // sequence i / q_len, at position ctx - q_len + i % q_len
};

// Absorbed multi-head latent attention over a latent pool [num_blocks,
// block_size, MLA_DK] (latent numbers then the rotary key).  One CTA per
// (sequence, tile of 16 query heads, split chunk).
constexpr int MLA_DV = 512;                 // latent numbers: the value
constexpr int MLA_DR = 64;                  // rotary-key numbers
constexpr int MLA_DK = MLA_DV + MLA_DR;     // numbers a query scores against
struct MlaParams {
    const uint16_t* q;        // bf16 [batch, q_heads, MLA_DK] (absorbed queries)
    const int32_t* tables;    // [batch, max_blocks]
    const int32_t* ctx;       // [batch]
    uint16_t* out;            // bf16 [batch, q_heads, MLA_DV]
    float* lse;               // [batch, q_heads] or null
    float* part_o;            // [batch, q_heads, max_splits, MLA_DV]; the tcgen05 forms store
                              // fp16 here: wide, per piece (sequence, head tile, half, split)
                              // [8 chunks][8 slots of 4][128 heads]; narrow, per piece (sequence,
                              // head tile, split) [16 heads][MLA_DV]
    float* part_ml;           // [batch, q_heads, max_splits, 2]: (max, sum), log2 units;
                              // tcgen05 forms: [piece][128 or 16 heads][2]
    uint32_t* err;
    int* tickets;             // [batch, head_tiles]: finished chunks, zero between calls;
                              // tcgen05 forms: piece counts, [batch, head_tiles, 2 halves]
                              // (wide) or [batch, head_tiles] (narrow)
    int batch, q_heads, head_tiles;
    int max_blocks, num_blocks;
    int split_blocks, max_splits;   // chunk length in blocks (tcgen05 form: least blocks per CTA
                                    // range); most chunks (pieces) a sequence can have
    float scale_log2;
    // paged_mla_decode_step: the step's new vectors (bf16 [batch, MLA_DK], sequence b's at
    // position ctx - 1), which the CTA reading the block that holds one writes into the
    // latent pool first; null for the attention alone.
    const uint16_t* kv_new;
    uint8_t* pool;
};

// Launch with programmatic stream serialisation: the kernel may begin launching
// while the preceding kernel in the stream finishes (it waits for that kernel
// with griddepcontrol.wait before touching memory).  Falls back to an ordinary
// launch where the attribute is refused.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e == cudaErrorNotSupported || e == cudaErrorInvalidValue) {
        cudaGetLastError();
        cfg.numAttrs = 0;
        e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    }
    return e;
}

// Row tile of one CTA: 8 or 16 query rows of a kv head (padding unused rows).
inline int head_tile_for_group(int rows) { return rows <= 8 ? 8 : 16; }

// Raises the variant's dynamic shared-memory limit (once, at pool creation).
cudaError_t prepare_decode_bf16(int head_dim, int block_size, int head_tile);
cudaError_t prepare_decode_fp8(int head_dim, int block_size, int head_tile);
cudaError_t launch_decode_bf16(int head_dim, int block_size, int head_tile, dim3 grid,
                               const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_fp8(int head_dim, int block_size, int head_tile, dim3 grid,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeParams& p, cudaStream_t s);
// The decode kernel with one CTA per group of `heads` kv heads (decode_heads.cuh), `ctas`
// CTAs per SM; the variants built are listed in decode_heads.cu.
bool decode_heads_supported(bool fp8, int head_dim, int block_size, int head_tile, int heads,
                            int ctas);
cudaError_t prepare_decode_heads(bool fp8, int head_dim, int block_size);
cudaError_t launch_decode_heads(bool fp8, int head_dim, int block_size, int head_tile, int heads,
                                int ctas, dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv,
                                const DecodeParams& p, cudaStream_t s);
// The separate log-sum-exp merge of the chunk partials that paged_decode_main leaves
// with merge_kernel = 1: one thread per 4 numbers of a query row, sequences of one
// chunk skipped (their chunk wrote the output).
cudaError_t launch_decode_merge(const DecodeParams& p, int head_dim, int block_size,
                                cudaStream_t s);
// Merge of attention results over disjoint key sets: outs bf16 [n_src, rows, head_dim],
// lses [n_src, rows] (natural log) -> out bf16 [rows, head_dim], lse_out [rows] or null.
cudaError_t launch_merge_attention_states(const uint16_t* outs, const float* lses, int n_src,
                                          long long rows, int head_dim, uint16_t* out,
                                          float* lse_out, cudaStream_t s);
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
// Tokens per pipeline stage of the latent decode (0: block size not supported);
// prod: the variant with a producer warp (small grids), else the three-CTA one.
int mla_stage_tokens(int block_size, bool prod);
cudaError_t prepare_mla_decode(int block_size);
cudaError_t launch_mla_decode(int block_size, bool prod, dim3 grid, const CUtensorMap& tm,
                              const MlaParams& p, cudaStream_t s);
// The tcgen05 form: tiles of 128 heads, blocks of 64 tokens, one CTA per SM taking an
// equal contiguous range of the (latent half, head tile, sequence, block) units; the
// pieces of sequences cut by a range boundary are merged by a second kernel, launched
// by launch_mla_decode_tc when max_splits > 1.
constexpr int MLA_TC_HEADS = 128;
// Positions the tcgen05 forms' partition adds before each sequence's blocks: the cost of
// starting a segment (the queries' load and the epilogue), in blocks (mla_partition.cuh);
// the values timed best on GB300.
constexpr int MLA_SEG_PAD_WIDE = 4;
constexpr int MLA_SEG_PAD_NARROW = 2;
constexpr int MLA_TC_BLOCK = 64;
cudaError_t prepare_mla_decode_tc();
cudaError_t launch_mla_decode_tc(dim3 grid, const CUtensorMap& tm, const MlaParams& p,
                                 cudaStream_t s);
// The narrow tcgen05 form: tiles of 16 heads (columns of the score MMAs, whose rows are
// tokens), blocks of 64 tokens streamed as 32-token stages, one CTA per SM taking an equal
// contiguous range of the (head tile, sequence, block) units; cut sequences are merged by
// a second kernel when max_splits > 1.  tm: the latent pool's map with a box of one
// 64-number piece of 32 slots; tq: the queries' map, dims (MLA_DK, q_heads, batch), a box
// of one 64-number piece of min(16, q_heads) heads.
// Partials: part_o [piece][16 heads][MLA_DV], part_ml [piece][16 heads] (max, sum),
// piece = (sequence, head tile, split); tickets [batch, head_tiles] piece counts.
constexpr int MLA_TCN_HEADS = 16;
constexpr int MLA_TCN_STAGE_TOKENS = 32;
cudaError_t prepare_mla_decode_tcn();
cudaError_t launch_mla_decode_tcn(dim3 grid, const CUtensorMap& tm, const CUtensorMap& tq,
                                  const MlaParams& p, cudaStream_t s);
cudaError_t launch_copy_blocks(const struct kv_block_copy* copies, int n, uint8_t* k_pool,
                               uint8_t* v_pool, size_t block_bytes, int num_blocks, uint32_t* err,
                               cudaStream_t s);

}  // namespace kvp
