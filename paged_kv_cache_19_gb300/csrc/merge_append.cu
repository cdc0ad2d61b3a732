// merge_append.cu -- split-KV log-sum-exp merge and the paged KV append.
#include "device_common.cuh"
#include "kernels.h"

namespace kvp {

// ---------------------------------------------------------------------------
// Merge of the split-KV chunks of one (sequence, query head) per warp.
// Chunk j carries its normalised output o_j, its running max m_j and its sum
// l_j = sum exp2(s - m_j) (log2 units).  With M = max_j m_j over non-empty
// chunks and w_j = l_j 2^(m_j - M):
//   out = sum_j w_j o_j / sum_j w_j,   lse = (M + log2 sum_j w_j) ln 2.
// This is the standard identity behind split-KV decoding (learn.mohebi.ai
// lesson 12, section 6: long contexts spread the cache read over all SMs).
// Sequences that fit one chunk were finished by the main kernel.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) paged_decode_merge(const MergeParams p)
{
    constexpr int PER = D / 32;
    const int gw = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= p.batch * p.q_heads) return;
    const int b = gw / p.q_heads;
    int ctx = __ldg(p.ctx + b);
    const int cap = p.max_blocks * p.block_size;
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    const int nblk = (ctx + p.block_size - 1) / p.block_size;
    const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    if (nsplit <= 1) return;

    const size_t bh = static_cast<size_t>(gw);            // == b * q_heads + h
    const float* ml = p.part_ml + bh * p.max_splits * 2;
    float M = -INFINITY;
    for (int j = lane; j < nsplit; j += 32) {
        const float lj = ml[2 * j + 1];
        if (lj > 0.f) M = fmaxf(M, ml[2 * j]);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, o));

    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float W = 0.f;
    const float* ob = p.part_o + bh * p.max_splits * D + lane * PER;
    for (int j = 0; j < nsplit; ++j) {
        const float lj = ml[2 * j + 1];
        if (!(lj > 0.f)) continue;                        // empty chunk: m = -inf, l = 0
        const float wj = lj * fast_exp2(ml[2 * j] - M);
        W += wj;
        const float* oj = ob + static_cast<size_t>(j) * D;
        if constexpr (PER == 4) {
            const float4 v = *reinterpret_cast<const float4*>(oj);
            acc[0] += wj * v.x;
            acc[1] += wj * v.y;
            acc[2] += wj * v.z;
            acc[3] += wj * v.w;
        } else {
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] += wj * oj[e];
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + bh * D + lane * PER);
#pragma unroll
    for (int e = 0; e < PER; e += 2) dst[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
    if (p.lse != nullptr && lane == 0)
        p.lse[bh] = W > 0.f ? (M + __log2f(W)) * 0.69314718055994531f : -INFINITY;
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t s)
{
    const long warps = static_cast<long>(p.batch) * p.q_heads;
    const int threads = 128;
    const long blocks = (warps * 32 + threads - 1) / threads;
    if (p.head_dim == 128)
        paged_decode_merge<128><<<static_cast<unsigned>(blocks), threads, 0, s>>>(p);
    else
        paged_decode_merge<64><<<static_cast<unsigned>(blocks), threads, 0, s>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Append: token i goes to sequence token_seq[i] (or i) at position
// token_pos[i] (or ctx - 1): block table entry pos / block_size, slot
// pos % block_size, all kv heads (xuewyang.github.io/posts/kv, "A toy vLLM",
// write_kv; brunomaga.github.io, PagedKVCache.append).  One CTA per token;
// each thread moves 8 elements (16 bytes of bf16 input) per step.
// fp8: code = e4m3fn(x / scale[head]) with the quotient rounded to binary32
// and the conversion rounding to nearest even, saturating at +-448.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) paged_kv_append_kernel(const AppendParams p)
{
    const int i = blockIdx.x;
    const int seq = p.token_seq != nullptr ? __ldg(p.token_seq + i) : i;
    if (seq < 0 || seq >= p.batch) {
        if (threadIdx.x == 0) atomicOr(p.err, KV_DEVERR_SEQ);
        return;
    }
    const int pos = p.token_pos != nullptr ? __ldg(p.token_pos + i) : __ldg(p.ctx + seq) - 1;
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
    const uint4* vs = reinterpret_cast<const uint4*>(p.v_new + static_cast<size_t>(i) * row);
    const int nvec = row / 8;
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
        const float sk = __ldg(p.k_scale + h);
        const float sv = __ldg(p.v_scale + h);
        const uint4 kx = __ldg(ks + v);
        const uint4 vx = __ldg(vs + v);
        const uint32_t kw[4] = {kx.x, kx.y, kx.z, kx.w};
        const uint32_t vw[4] = {vx.x, vx.y, vx.z, vx.w};
        uint32_t kc[2] = {0u, 0u}, vc[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float k0 = __fdiv_rn(__uint_as_float(kw[e] << 16), sk);
            const float k1 = __fdiv_rn(__uint_as_float(kw[e] & 0xffff0000u), sk);
            const float v0 = __fdiv_rn(__uint_as_float(vw[e] << 16), sv);
            const float v1 = __fdiv_rn(__uint_as_float(vw[e] & 0xffff0000u), sv);
            const uint32_t k2 = __nv_cvt_float2_to_fp8x2(make_float2(k0, k1), __NV_SATFINITE, __NV_E4M3);
            const uint32_t v2 = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
            kc[e >> 1] |= (k2 & 0xffffu) << (16 * (e & 1));
            vc[e >> 1] |= (v2 & 0xffffu) << (16 * (e & 1));
        }
        kd[v] = make_uint2(kc[0], kc[1]);
        vd[v] = make_uint2(vc[0], vc[1]);
    }
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s)
{
    paged_kv_append_kernel<<<static_cast<unsigned>(p.num_tokens), 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvp
