// append_row.cuh -- writing tokens' K and V rows into the pool: the arithmetic shared by the
// append kernel and the decode kernels' in-kernel append of paged_decode_step.
//
// A token at position pos of a sequence lives in block table entry pos / block_size, slot
// pos % block_size, one row of head_dim numbers per kv head (xuewyang.github.io/posts/kv,
// "A toy vLLM", write_kv; brunomaga.github.io, PagedKVCache.append).  bf16 rows are copied;
// fp8: code = e4m3fn(x / scale[head]), the quotient rounded to binary32 and the conversion
// rounding to nearest even, saturating at +-448.
#pragma once

#include "device_common.cuh"
#include "kernels.h"

namespace kvp {

// Eight bf16 values (one 16-byte vector) -> eight e4m3 codes (8 bytes), low element first.
__device__ __forceinline__ uint2 e4m3_codes8(uint4 x, float scale)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t c[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float a = __fdiv_rn(__uint_as_float(w[e] << 16), scale);
        const float b = __fdiv_rn(__uint_as_float(w[e] & 0xffff0000u), scale);
        const uint32_t two = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
        c[e >> 1] |= (two & 0xffffu) << (16 * (e & 1));
    }
    return make_uint2(c[0], c[1]);
}

// paged_decode_step's new tokens (row b * q_len + t of k_new / v_new, position
// ctx - q_len + t) that fall in the logical blocks [j_lo, j_hi) of sequence b, for the NH kv
// heads h0 .. h0 + NH - 1, written by the 32 lanes of a warp: every (token, head) row pair
// is one 16-byte vector per lane, all loaded before any is stored so that the loads are in
// flight together.  Blocks whose table entry is not a valid id are skipped (the caller
// flags them); positions outside the table never fall in a block and are left to the
// caller to flag.
template <bool FP8, int D, int BS, int NH>
__device__ __forceinline__ void write_step_rows(const DecodeParams& p, int b, int ctx_raw, int j_lo,
                                                int j_hi, int h0, int lane)
{
    constexpr int NV = D / 8;                                     // 16-byte vectors per row
    static_assert(2 * NV <= 32, "a K row and a V row take at most one vector per lane");
    if (lane >= 2 * NV) return;
    const int32_t* trow = p.tables + static_cast<size_t>(b) * p.max_blocks;
    const int t0 = max(0, j_lo * BS - (ctx_raw - p.q_len));       // first token in the range
    const bool is_k = lane < NV;
    const int u = is_k ? lane : lane - NV;                        // vector of the row
    uint8_t* pool = is_k ? p.k_pool : p.v_pool;
    const uint16_t* src = is_k ? p.k_new : p.v_new;
    for (int t = t0; t < p.q_len; ++t) {
        const int pos = ctx_raw - p.q_len + t;
        const int j = pos / BS;
        if (pos < 0) continue;
        if (j >= j_hi) break;
        const int blk = __ldg(trow + j);
        if (blk < 0 || blk >= p.num_blocks) continue;
        const size_t srow = (static_cast<size_t>(b) * p.q_len + t) * p.kv_heads + h0;
        const size_t drow = (static_cast<size_t>(blk) * BS + pos % BS) * p.kv_heads + h0;
        uint4 x[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) x[h] = __ldg(reinterpret_cast<const uint4*>(src + (srow + h) * D) + u);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
            if constexpr (!FP8) {
                reinterpret_cast<uint4*>(pool + (drow + h) * D * 2)[u] = x[h];
            } else {
                const float sc = __ldg((is_k ? p.k_scale : p.v_scale) + h0 + h);
                reinterpret_cast<uint2*>(pool + (drow + h) * D)[u] = e4m3_codes8(x[h], sc);
            }
        }
    }
}

// Generic-proxy writes to global memory ordered before later TMA (async-proxy) reads.
__device__ __forceinline__ void fence_proxy_async_all()
{
    asm volatile("fence.proxy.async;" ::: "memory");
}

// paged_mla_decode_step: the logical block that holds sequence b's new vector (position
// ctx - 1), or -1 when the call appends nothing or the position is outside the table
// (flagged KV_DEVERR_POSITION elsewhere, as the append would).
__device__ __forceinline__ int mla_step_block(const MlaParams& p, int b, int bs)
{
    if (p.kv_new == nullptr) return -1;
    const int raw = __ldg(p.ctx + b);
    if (raw < 1 || raw > p.max_blocks * bs) return -1;
    return (raw - 1) / bs;
}

// paged_mla_decode_step: thread t of nth (nth >= 24) copies its share of sequence b's new
// vector (row b of kv_new, MLA_DK bf16 numbers = 72 vectors of 16 bytes) into slot `slot`
// of pool block blk: vectors t, t + nth, t + 2 nth, all loaded before any is stored.  The
// caller orders the writes before the TMA loads of the block (fence_proxy_async_all, then a
// barrier the loading thread waits on).
__device__ __forceinline__ void load_latent_share(const MlaParams& p, int b, int t, int nth, uint4 (&x)[3])
{
    constexpr int NV = MLA_DK / 8;
    const uint4* src = reinterpret_cast<const uint4*>(p.kv_new + static_cast<size_t>(b) * MLA_DK);
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (t + i * nth < NV) x[i] = __ldg(src + t + i * nth);
}

__device__ __forceinline__ void store_latent_share(const MlaParams& p, int blk, int bs, int slot, int t,
                                                   int nth, const uint4 (&x)[3])
{
    constexpr int NV = MLA_DK / 8;
    uint4* dst = reinterpret_cast<uint4*>(p.pool + (static_cast<size_t>(blk) * bs + slot) * MLA_DK * 2);
#pragma unroll
    for (int i = 0; i < 3; ++i)
        if (t + i * nth < NV) dst[t + i * nth] = x[i];
}

__device__ __forceinline__ void write_latent_share(const MlaParams& p, int b, int blk, int bs, int slot,
                                                   int t, int nth)
{
    uint4 x[3];
    load_latent_share(p, b, t, nth, x);
    store_latent_share(p, blk, bs, slot, t, nth, x);
}

}  // namespace kvp
