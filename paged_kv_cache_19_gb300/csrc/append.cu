// append.cu -- the paged KV append.
#include "append_row.cuh"
#include "device_common.cuh"
#include "kernels.h"
#include "kv_block_manager.h"

namespace kvp {

// ---------------------------------------------------------------------------
// Append: token i goes to sequence token_seq[i] (or i / q_len) at position
// token_pos[i] (or ctx - q_len + i % q_len): block table entry pos / block_size, slot
// pos % block_size, all kv heads (xuewyang.github.io/posts/kv, "A toy vLLM",
// write_kv; brunomaga.github.io, PagedKVCache.append).  One CTA per token;
// each thread moves 8 elements (16 bytes of bf16 input) per step.
// fp8: code = e4m3fn(x / scale[head]) with the quotient rounded to binary32
// and the conversion rounding to nearest even, saturating at +-448 (e4m3_codes8).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) paged_kv_append_kernel(const AppendParams p)
{
    grid_dependency_wait();                        // inputs of the preceding kernel are ready
    grid_dependents_launch();
    const int i = blockIdx.x;
    const int seq = p.token_seq != nullptr ? __ldg(p.token_seq + i) : i / p.q_len;
    if (seq < 0 || seq >= p.batch) {
        if (threadIdx.x == 0) atomicOr(p.err, KV_DEVERR_SEQ);
        return;
    }
    const int pos = p.token_pos != nullptr ? __ldg(p.token_pos + i) : __ldg(p.ctx + seq) - p.q_len + i % p.q_len;
    if (pos < 0 || pos / p.block_size >= p.max_blocks) {
        if (threadIdx.x == 0) atomicOr(p.err, KV_DEVERR_POSITION);
        return;
    }
    const int blk = __ldg(p.tables + static_cast<size_t>(seq) * p.max_blocks + pos / p.block_size);
    if (blk < 0 || blk >= p.num_blocks) {
        if (threadIdx.x == 0) atomicOr(p.err, KV_DEVERR_BLOCK_ID);
        return;
    }
    const int slot = pos % p.block_size;
    const int row = p.kv_heads * p.head_dim;                 // elements per token
    const size_t dst = (static_cast<size_t>(blk) * p.block_size + slot) * row;
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_new + static_cast<size_t>(i) * row);
    const int nvec = row / 8;
    if (p.v_pool == nullptr) {                      // latent pool: one cached vector per token
        uint4* kd = reinterpret_cast<uint4*>(p.k_pool + dst * 2);
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) kd[v] = __ldg(ks + v);
        return;
    }
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_new + static_cast<size_t>(i) * row);
    if (!p.fp8) {
        uint4* kd = reinterpret_cast<uint4*>(p.k_pool + dst * 2);
        uint4* vd = reinterpret_cast<uint4*>(p.v_pool + dst * 2);
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
            kd[v] = __ldg(ks + v);
            vd[v] = __ldg(vs + v);
        }
        return;
    }
    uint2* kd = reinterpret_cast<uint2*>(p.k_pool + dst);
    uint2* vd = reinterpret_cast<uint2*>(p.v_pool + dst);
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        const int h = (v * 8) / p.head_dim;
        kd[v] = e4m3_codes8(__ldg(ks + v), __ldg(p.k_scale + h));
        vd[v] = e4m3_codes8(__ldg(vs + v), __ldg(p.v_scale + h));
    }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s)
{
    return launch_dependent(paged_kv_append_kernel, dim3(static_cast<unsigned>(p.num_tokens)),
                            dim3(128), 0, s, p);
}

// ---------------------------------------------------------------------------
// Whole-block copies for copy-on-write: block src -> dst of the K and the V
// pool, 16 bytes per thread.  One CTA per (copy, pool half) slice.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) kv_copy_blocks_kernel(const kv_block_copy* copies, int n,
                                                             uint8_t* k_pool, uint8_t* v_pool,
                                                             size_t block_bytes, int num_blocks,
                                                             uint32_t* err)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int i = blockIdx.x >> 1;
    if (i >= n) return;
    uint8_t* pool = (blockIdx.x & 1) ? v_pool : k_pool;
    if (pool == nullptr) return;                    // latent pools have no V half
    const int src = copies[i].src;
    const int dst = copies[i].dst;
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && (blockIdx.x & 1) == 0) atomicOr(err, KV_DEVERR_BLOCK_ID);
        return;
    }
    const uint4* from = reinterpret_cast<const uint4*>(pool + static_cast<size_t>(src) * block_bytes);
    uint4* to = reinterpret_cast<uint4*>(pool + static_cast<size_t>(dst) * block_bytes);
    const size_t nvec = block_bytes / 16;
    for (size_t v = threadIdx.x; v < nvec; v += blockDim.x) to[v] = from[v];
}

cudaError_t launch_copy_blocks(const kv_block_copy* copies, int n, uint8_t* k_pool, uint8_t* v_pool,
                               size_t block_bytes, int num_blocks, uint32_t* err, cudaStream_t s)
{
    return launch_dependent(kv_copy_blocks_kernel, dim3(static_cast<unsigned>(2 * n)), dim3(256), 0,
                            s, copies, n, k_pool, v_pool, block_bytes, num_blocks, err);
}

}  // namespace kvp
