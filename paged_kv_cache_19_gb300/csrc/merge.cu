// merge.cu -- the log-sum-exp merge of split-KV chunk partials as a kernel of
// its own (paged_decode_attention_split_merge).
//
// Chunk j of a cut sequence leaves, per query row, its normalised output o_j,
// its running maximum m_j and its sum l_j (log2 units).  The row's result is
//   M = max_j m_j,  w_j = l_j 2^(m_j - M),  out = sum_j w_j o_j / sum_j w_j,
//   lse = (M + log2 sum_j w_j) ln 2
// (learn.mohebi.ai lesson 12, section 6: split-KV decoding; the identity is the
// online softmax of brunomaga.github.io "inference-prefill-decode-roofline-cache"
// applied to whole chunks).  Chunks that saw no token (l_j = 0) are left out.
// The arithmetic is the one the fused in-kernel merge of paged_decode_main does,
// in the same order, so both forms give the same bits.
#include "decode_common.cuh"
#include "kernels.h"

namespace kvp {

namespace {

constexpr int MERGE_THREADS = 128;

__global__ void __launch_bounds__(MERGE_THREADS)
paged_decode_merge(const DecodeParams p, int head_dim, int block_size)
{
    grid_dependency_wait();                          // the chunk partials of the decode grid
    grid_dependents_launch();
    const int per_row = head_dim >> 2;               // threads per query row, 4 numbers each
    const long long g = static_cast<long long>(blockIdx.x) * MERGE_THREADS + threadIdx.x;
    const long long rows = static_cast<long long>(p.batch) * p.q_heads * p.q_len;
    const long long row = g / per_row;
    if (row >= rows) return;
    const int d0 = static_cast<int>(g - row * per_row) * 4;
    const int b = static_cast<int>(row / (static_cast<long long>(p.q_heads) * p.q_len));

    // the chunk count of this sequence, from its context length clamped as the decode did
    int ctx = __ldg(p.ctx + b);
    const int cap = p.max_blocks * block_size;
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    const int nblk = (ctx + block_size - 1) / block_size;
    const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    if (nsplit == 1) return;                         // its only chunk wrote the output

    const float* ml = p.part_ml + row * p.max_splits * 2;
    float M = -INFINITY;
    for (int j = 0; j < nsplit; ++j) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(ml + 2 * j));
        if (v.y > 0.f) M = fmaxf(M, v.x);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float W = 0.f;
    const float* ob = p.part_o + row * p.max_splits * head_dim + d0;
#pragma unroll 4
    for (int j = 0; j < nsplit; ++j) {
        // every slot j < nsplit lies in the workspace: load unconditionally, add if used
        const float2 mlj = __ldcg(reinterpret_cast<const float2*>(ml + 2 * j));
        const float4 v = __ldcg(reinterpret_cast<const float4*>(ob + static_cast<size_t>(j) * head_dim));
        if (mlj.y > 0.f) {
            const float wj = mlj.y * fast_exp2(mlj.x - M);
            W += wj;
            acc[0] += wj * v.x;
            acc[1] += wj * v.y;
            acc[2] += wj * v.z;
            acc[3] += wj * v.w;
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint2 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(p.out + row * head_dim + d0) = o;
    if (p.lse != nullptr && d0 == 0) p.lse[row] = lse_from(M, W);
}

}  // namespace

cudaError_t launch_decode_merge(const DecodeParams& p, int head_dim, int block_size,
                                cudaStream_t s)
{
    const long long threads =
        static_cast<long long>(p.batch) * p.q_heads * p.q_len * (head_dim / 4);
    const long long blocks = (threads + MERGE_THREADS - 1) / MERGE_THREADS;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_dependent(paged_decode_merge, dim3(static_cast<unsigned>(blocks)),
                            dim3(MERGE_THREADS), 0, s, p, head_dim, block_size);
}

}  // namespace kvp

// ----------------------------------------------------------------------------
// Merge of attention results over disjoint key sets (paged_merge_attention_states).
//
// Source r attended over its own keys and left o_r (normalised, bf16) and lse_r
// (natural log).  Over the union of the keys,
//   LSE = log sum_r exp(lse_r),   out = sum_r exp(lse_r - LSE) o_r
// -- the split-KV identity above with l_r exp(m_r) = exp(lse_r).  This is the one
// exchange a sequence split across devices needs (each device decodes its share of
// the blocks; the (o_r, lse_r) pairs are gathered and merged).  Sources with
// lse_r = -inf saw no key and are left out; if every source is empty the row gets
// out = 0, lse = -inf.
namespace kvp {

namespace {

__global__ void __launch_bounds__(MERGE_THREADS)
merge_attention_states(const uint16_t* __restrict__ outs, const float* __restrict__ lses,
                       int n_src, long long rows, int head_dim, uint16_t* __restrict__ out,
                       float* __restrict__ lse_out)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int per_row = head_dim >> 2;               // threads per row, 4 numbers each
    const long long g = static_cast<long long>(blockIdx.x) * MERGE_THREADS + threadIdx.x;
    const long long row = g / per_row;
    if (row >= rows) return;
    const int d0 = static_cast<int>(g - row * per_row) * 4;
    constexpr float LOG2E = 1.4426950408889634f;

    float M = -INFINITY;                             // log2 units
    for (int r = 0; r < n_src; ++r) {
        const float l = __ldg(lses + r * rows + row);
        if (l > -INFINITY) M = fmaxf(M, l * LOG2E);
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float W = 0.f;
    if (M > -INFINITY) {
        for (int r = 0; r < n_src; ++r) {
            const float l = __ldg(lses + r * rows + row);
            if (!(l > -INFINITY)) continue;
            const float w = fast_exp2(l * LOG2E - M);
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(
                outs + (static_cast<size_t>(r) * rows + row) * head_dim + d0));
            W += w;
            acc[0] += w * bf16_bits_to_float(static_cast<uint16_t>(v.x & 0xffffu));
            acc[1] += w * bf16_bits_to_float(static_cast<uint16_t>(v.x >> 16));
            acc[2] += w * bf16_bits_to_float(static_cast<uint16_t>(v.y & 0xffffu));
            acc[3] += w * bf16_bits_to_float(static_cast<uint16_t>(v.y >> 16));
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint2 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(out + row * head_dim + d0) = o;
    if (lse_out != nullptr && d0 == 0) lse_out[row] = lse_from(M, W);
}

}  // namespace

cudaError_t launch_merge_attention_states(const uint16_t* outs, const float* lses, int n_src,
                                          long long rows, int head_dim, uint16_t* out,
                                          float* lse_out, cudaStream_t s)
{
    const long long threads = rows * (head_dim / 4);
    const long long blocks = (threads + MERGE_THREADS - 1) / MERGE_THREADS;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_dependent(merge_attention_states, dim3(static_cast<unsigned>(blocks)),
                            dim3(MERGE_THREADS), 0, s, outs, lses, n_src, rows, head_dim, out,
                            lse_out);
}

}  // namespace kvp
