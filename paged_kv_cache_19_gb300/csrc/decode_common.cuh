// decode_common.cuh -- the per-block work and the epilogue pieces of paged
// decode attention.
//
// What is computed (per sequence b and query head h, kv = h / g):
//   s_t = scale * q[b,h,:] . K[t,kv,:],  out = sum_t softmax(s)_t V[t,kv,:]
// over tokens 0 .. ctx_b - 1, read in place through the block table
// (brunomaga.github.io "inference-prefill-decode-roofline-cache", section
// "PagedAttention: memory management for the KV cache", paged_decode_attention;
// learn.mohebi.ai lesson 12, "PagedAttention (4.1-4.3)": the kernel reads the
// cache one block at a time and combines blocks with the online-softmax update).
//
// One consumer warp handles one cache block of one kv head at a time:
//   * scores S^T[16 tokens x 8 heads] = K[16 x d] . Q^T[d x 8] on the tensor
//     cores (mma.m16n8k16, tokens on M so a GQA group of up to 8 heads fills N);
//   * online softmax in the log2 domain with warp shuffles; slots at or past
//     ctx are replaced by -inf and their V rows zeroed, never used as values;
//   * O^T[d x 8] += V^T[d x 16] . P^T[16 x 8], with P moved from the
//     accumulator layout to the B-operand layout by movmatrix.
// bf16 caches feed the MMA from ldmatrix; fp8 e4m3 codes are converted to f16
// in registers (exact) and the per-head scales are applied in fp32.
#pragma once

#include "device_common.cuh"
#include "kernels.h"

namespace kvp {

template <bool FP8, int D, int BS, int NT>
struct DecodeCfg {
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROWB = D * ELEM;           // bytes of one token's row of one kv head
    static constexpr int DCH = ROWB / 128;          // 128-byte swizzle rows per token
    static constexpr int TILE = BS * ROWB;          // bytes of one K (or V) block tile
    static constexpr int STAGE = 2 * TILE;          // K tile then V tile
    // About 64 KB of stages per CTA, 3 CTAs per SM: ~192 KB in flight per SM (16-row
    // tiles fit 3 CTAs in 128 registers with a few spilled bytes, which measured faster
    // on GB300 than 2 CTAs with 96 KB rings: 125 us against 129 us for the verify pass).
    static constexpr int RING = 64 * 1024;
    static constexpr int NSTAGE = (RING / STAGE) / 4 * 4 >= 4 ? (RING / STAGE) / 4 * 4 : 4;
    static constexpr int NCW = 4;                   // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int MT = BS / 16;              // 16-token tiles per block
    static constexpr int NTT = NT / 8;              // 8-head tiles
    static constexpr int KS = D / 16;               // 16-wide slices of head_dim
    static constexpr int RED_STRIDE = D + 4;        // padded row of the epilogue buffer (floats)
    static constexpr int RED_FLOATS = NCW * NT * RED_STRIDE + 2 * NCW * NT;
    static constexpr int RED_BYTES = RED_FLOATS * 4;
    static constexpr int E = NT * D / (NCW * 32);   // output elements per consumer thread
    static_assert(ROWB % 128 == 0, "rows must be whole 128-byte swizzle rows");
    static_assert(NSTAGE % NCW == 0, "each consumer warp must own whole stages");
    static_assert(!FP8 || D == 128, "fp8 path is laid out for head_dim 128");
    static_assert(E % 4 == 0 && D % E == 0, "epilogue split (float4 partial reads)");
};

// Byte address of 16-byte chunk `ch` of token `tok` in a TMA tile written with
// the 128-byte swizzle: row = tok * DCH + ch / 8, and chunk (ch % 8) of a row
// sits at position (ch % 8) ^ (row % 8).  Tiles start on 1024-byte boundaries.
template <int DCH>
__device__ __forceinline__ uint32_t swz(uint32_t tile, int tok, int ch)
{
    const int row = tok * DCH + (ch >> 3);
    return tile + row * 128 + ((((ch & 7) ^ (row & 7))) << 4);
}

// Online-softmax state of one consumer warp for the heads of one tile.
// o[ms][nt][hi*2 + j] holds (d(ms, row r + 8 hi), head nt*8 + 2c + j).
template <class C>
struct WarpState {
    float o[C::KS][C::NTT][4];
    float m[C::NTT][2];
    float l[C::NTT][2];
};

template <class C>
__device__ __forceinline__ void reset_state(WarpState<C>& s)
{
#pragma unroll
    for (int ms = 0; ms < C::KS; ++ms)
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s.o[ms][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt) {
        s.m[nt][0] = s.m[nt][1] = -INFINITY;
        s.l[nt][0] = s.l[nt][1] = 0.f;
    }
}

// Q^T as the MMA B operand, element (k, n) = q[head n][d(k)], for the nh real
// heads starting at qb (rows past nh are zero).  Returns the fp32 factor that
// turns raw MMA scores into log2-domain logits.
template <bool FP8, int D, int BS, int NT>
__device__ __forceinline__ float load_q_frags(uint32_t (&qf)[D / 16][NT / 8][2], const uint16_t* qb,
                                              int nh, int lane, float scale_log2,
                                              const float* k_scale, int kvh)
{
    using C = DecodeCfg<FP8, D, BS, NT>;
    const int r = lane >> 2;
    const int c = lane & 3;
    if constexpr (!FP8) {
        // d(k) is the natural order: B rows 2c, 2c+1 and 2c+8, 2c+9 of slice ks.
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt) {
            const int hl = nt * 8 + r;
            const bool valid = hl < nh;
            const uint16_t* qh = qb + static_cast<size_t>(valid ? hl : 0) * D;
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                qf[ks][nt][0] = valid ? *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 2 * c) : 0u;
                qf[ks][nt][1] = valid ? *reinterpret_cast<const uint32_t*>(qh + ks * 16 + 8 + 2 * c) : 0u;
            }
        }
        return scale_log2;
    } else {
        // The fp8 K operand is read 4 bytes at a time, so slice ks of thread
        // column c holds d = 32c + 4ks + {0,1} (B rows 2c, 2c+1) and
        // d = 32c + 4ks + {2,3} (B rows 2c+8, 2c+9).  q goes to f16 (exact for
        // bf16 values inside the f16 range) after a power-of-two pre-scale that
        // keeps max|q| below 2^15; the scale is undone in the returned factor.
        float qv[C::KS][C::NTT][4];
        float qmax = 0.f;
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt) {
            const int hl = nt * 8 + r;
            const bool valid = hl < nh;
            const uint16_t* qh = qb + static_cast<size_t>(valid ? hl : 0) * D;
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = valid ? bf16_bits_to_float(qh[32 * c + 4 * ks + e]) : 0.f;
                    qv[ks][nt][e] = x;
                    qmax = fmaxf(qmax, fabsf(x));
                }
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(FULL_MASK, qmax, o));
        const int ex = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xffu) - 126;   // qmax < 2^ex
        const int shift = max(0, ex - 15);
        const float down = __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
        const float up = __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                qf[ks][nt][0] = pack_f16x2(qv[ks][nt][0] * down, qv[ks][nt][1] * down);
                qf[ks][nt][1] = pack_f16x2(qv[ks][nt][2] * down, qv[ks][nt][3] * down);
            }
        return scale_log2 * up * __ldg(k_scale + kvh);
    }
}

// Causal offsets of the rows this thread's accumulator columns belong to: row
// r (query token i = r % q_len) sees one token fewer than the sequence's last
// query for every later query token: dt = q_len - 1 - i.  Zero for decode.
template <int NTT>
__device__ __forceinline__ void row_offsets(int (&dt)[NTT][2], int row0, int q_len, int lane)
{
    const int c = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NTT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) dt[nt][j] = q_len - 1 - (row0 + nt * 8 + 2 * c + j) % q_len;
}

// One cache block (BS tokens of one kv head, K tile at tk, V tile at tv in
// shared memory) folded into the warp's online-softmax state.  lim = ctx minus
// the block's first token position (may exceed BS): token k of the block is a
// key for a row with causal offset dt when k < lim - dt; tokens at or past
// lim are not in the cache at all and their values are never used.
template <bool FP8, int D, int BS, int NT>
__device__ __forceinline__ void process_block(uint32_t tk, uint32_t tv, int lim,
                                              const int (&dt)[NT / 8][2],
                                              const uint32_t (&qf)[D / 16][NT / 8][2], float sl2,
                                              WarpState<DecodeCfg<FP8, D, BS, NT>>& st, int lane)
{
    using C = DecodeCfg<FP8, D, BS, NT>;
    const int r = lane >> 2;
    const int c = lane & 3;
    const int nvalid = min(BS, lim);

    // ---- scores S^T[tokens x heads] = K . Q^T
    float s[C::MT][C::NTT][4];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[mt][nt][e] = 0.f;
        if constexpr (!FP8) {
            // A fragments {rows 0-7, 8-15} x {k 0-7, 8-15} from four 8x8 ldmatrix tiles
            const int tok = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                uint32_t a[4];
                ldsm_x4(swz<C::DCH>(tk, tok, 2 * ks + (lane >> 4)), a);
#pragma unroll
                for (int nt = 0; nt < C::NTT; ++nt)
                    mma_bf16_16816(s[mt][nt], a, qf[ks][nt][0], qf[ks][nt][1]);
            }
        } else {
            const int ta = mt * 16 + r;
            const uint4 x0 = lds128(swz<1>(tk, ta, 2 * c));
            const uint4 x1 = lds128(swz<1>(tk, ta, 2 * c + 1));
            const uint4 y0 = lds128(swz<1>(tk, ta + 8, 2 * c));
            const uint4 y1 = lds128(swz<1>(tk, ta + 8, 2 * c + 1));
            const uint32_t wa[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t wb[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                uint32_t a[4];
                a[0] = e4m3x2_to_f16x2(wa[ks]);          // token ta,   d = 32c+4ks+{0,1}
                a[1] = e4m3x2_to_f16x2(wb[ks]);          // token ta+8
                a[2] = e4m3x2_to_f16x2(wa[ks] >> 16);    // token ta,   d = 32c+4ks+{2,3}
                a[3] = e4m3x2_to_f16x2(wb[ks] >> 16);
#pragma unroll
                for (int nt = 0; nt < C::NTT; ++nt)
                    mma_f16_16816(s[mt][nt], a, qf[ks][nt][0], qf[ks][nt][1]);
            }
        }
    }

    // ---- online softmax over this block (log2 domain)
    bool rescale = false;
    float alpha[C::NTT][2];
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float mx = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    const int tok = mt * 16 + r + 8 * hi;
                    const float x = tok < lim - dt[nt][j] ? s[mt][nt][2 * hi + j] * sl2 : -INFINITY;
                    s[mt][nt][2 * hi + j] = x;
                    mx = fmaxf(mx, x);
                }
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 16));
            const float m_new = fmaxf(st.m[nt][j], mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float a_ = fast_exp2(st.m[nt][j] - m_use);
            st.m[nt][j] = m_new;
            float ls = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    const float pr = fast_exp2(s[mt][nt][2 * hi + j] - m_use);
                    s[mt][nt][2 * hi + j] = pr;
                    ls += pr;
                }
            st.l[nt][j] = st.l[nt][j] * a_ + ls;
            alpha[nt][j] = a_;
            rescale |= (a_ != 1.f);
        }
    }
    if (__any_sync(FULL_MASK, rescale)) {
#pragma unroll
        for (int ms = 0; ms < C::KS; ++ms)
#pragma unroll
            for (int nt = 0; nt < C::NTT; ++nt) {
                st.o[ms][nt][0] *= alpha[nt][0];
                st.o[ms][nt][1] *= alpha[nt][1];
                st.o[ms][nt][2] *= alpha[nt][0];
                st.o[ms][nt][3] *= alpha[nt][1];
            }
    }

    // ---- P^T as the B operand: transpose each 8x8 quadrant of the accumulator
    // layout (rows = tokens) into the B layout (rows = heads).
    uint32_t pb[C::MT][C::NTT][2];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt) {
            if constexpr (!FP8) {
                pb[mt][nt][0] = movmatrix_trans(pack_bf16x2(s[mt][nt][0], s[mt][nt][1]));
                pb[mt][nt][1] = movmatrix_trans(pack_bf16x2(s[mt][nt][2], s[mt][nt][3]));
            } else {
                pb[mt][nt][0] = movmatrix_trans(pack_f16x2(s[mt][nt][0], s[mt][nt][1]));
                pb[mt][nt][1] = movmatrix_trans(pack_f16x2(s[mt][nt][2], s[mt][nt][3]));
            }
        }

    // ---- O^T[d x heads] += V^T[d x tokens] . P^T[tokens x heads]
    const bool partial = nvalid < BS;
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
        const int t0 = mt * 16 + 2 * c;     // tokens of this thread: t0, t0+1, t0+8, t0+9
        if constexpr (!FP8) {
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (partial) {
                mlo = (t0 < nvalid ? 0x0000ffffu : 0u) | (t0 + 1 < nvalid ? 0xffff0000u : 0u);
                mhi = (t0 + 8 < nvalid ? 0x0000ffffu : 0u) | (t0 + 9 < nvalid ? 0xffff0000u : 0u);
            }
            const int quad = lane >> 3;     // 8x8 tile: (d half = quad & 1, token half = quad >> 1)
            const int tok = mt * 16 + (lane & 7) + (quad >> 1) * 8;
#pragma unroll
            for (int ms = 0; ms < C::KS; ++ms) {
                uint32_t a[4];
                ldsm_x4_trans(swz<C::DCH>(tv, tok, 2 * ms + (quad & 1)), a);
                a[0] &= mlo;
                a[1] &= mlo;
                a[2] &= mhi;
                a[3] &= mhi;
#pragma unroll
                for (int nt = 0; nt < C::NTT; ++nt)
                    mma_bf16_16816(st.o[ms][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
            }
        } else {
            // Thread (r, c) reads d = 16r .. 16r+15 of tokens t0, t0+1, t0+8, t0+9.
            // Slice ms = 2w holds d = 16r + 4w (row r) and 16r + 4w + 1 (row r+8);
            // slice 2w+1 holds d = 16r + 4w + 2 and + 3.
            uint4 v0 = lds128(swz<1>(tv, t0, r));
            uint4 v1 = lds128(swz<1>(tv, t0 + 1, r));
            uint4 v2 = lds128(swz<1>(tv, t0 + 8, r));
            uint4 v3 = lds128(swz<1>(tv, t0 + 9, r));
            if (partial) {
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                if (t0 >= nvalid) v0 = z;
                if (t0 + 1 >= nvalid) v1 = z;
                if (t0 + 8 >= nvalid) v2 = z;
                if (t0 + 9 >= nvalid) v3 = z;
            }
            const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
            const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
            const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w};
            const uint32_t w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t x01 = __byte_perm(w0[w], w1[w], 0x5140);   // d+0 | d+1
                const uint32_t y01 = __byte_perm(w0[w], w1[w], 0x7362);   // d+2 | d+3
                const uint32_t x23 = __byte_perm(w2[w], w3[w], 0x5140);
                const uint32_t y23 = __byte_perm(w2[w], w3[w], 0x7362);
                uint32_t a[4];
                a[0] = e4m3x2_to_f16x2(x01);
                a[1] = e4m3x2_to_f16x2(x01 >> 16);
                a[2] = e4m3x2_to_f16x2(x23);
                a[3] = e4m3x2_to_f16x2(x23 >> 16);
#pragma unroll
                for (int nt = 0; nt < C::NTT; ++nt)
                    mma_f16_16816(st.o[2 * w][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
                a[0] = e4m3x2_to_f16x2(y01);
                a[1] = e4m3x2_to_f16x2(y01 >> 16);
                a[2] = e4m3x2_to_f16x2(y23);
                a[3] = e4m3x2_to_f16x2(y23 >> 16);
#pragma unroll
                for (int nt = 0; nt < C::NTT; ++nt)
                    mma_f16_16816(st.o[2 * w + 1][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
            }
        }
    }
}

// The per-thread row sums of a warp summed over the 8 row groups sharing a column.
template <class C>
__device__ __forceinline__ void reduce_row_sums(WarpState<C>& st)
{
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = st.l[nt][j];
            l += __shfl_xor_sync(FULL_MASK, l, 4);
            l += __shfl_xor_sync(FULL_MASK, l, 8);
            l += __shfl_xor_sync(FULL_MASK, l, 16);
            st.l[nt][j] = l;
        }
}

// Writes a warp's (reduced) state into the epilogue buffer:
// red_o [NCW][NT][RED_STRIDE], red_m [NCW][NT], red_l [NCW][NT].
template <bool FP8, class C>
__device__ __forceinline__ void stash_state(float* red, const WarpState<C>& st, int warp, int lane)
{
    constexpr int NT = C::NTT * 8;
    const int r = lane >> 2;
    const int c = lane & 3;
    float* red_o = red;
    float* red_m = red_o + C::NCW * NT * C::RED_STRIDE;
    float* red_l = red_m + C::NCW * NT;
#pragma unroll
    for (int ms = 0; ms < C::KS; ++ms)
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int head = nt * 8 + 2 * c + j;
                    const int d = FP8 ? (16 * r + 2 * ms + hi) : (16 * ms + r + 8 * hi);
                    red_o[(warp * NT + head) * C::RED_STRIDE + d] = st.o[ms][nt][2 * hi + j];
                }
    if (r == 0) {
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int head = nt * 8 + 2 * c + j;
                red_m[warp * NT + head] = st.m[nt][j];
                red_l[warp * NT + head] = st.l[nt][j];
            }
    }
}

// Merges the NCW warp states of local head `head`, elements d0 .. d0+E-1:
// acc = normalised output (times out_scale), M = max (log2 units), L = sum.
template <class C>
__device__ __forceinline__ void combine_warps(const float* red, int head, int d0, float out_scale,
                                              float (&acc)[C::E], float& M, float& L)
{
    constexpr int NT = C::NTT * 8;
    const float* red_o = red;
    const float* red_m = red_o + C::NCW * NT * C::RED_STRIDE;
    const float* red_l = red_m + C::NCW * NT;
    M = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, red_m[w * NT + head]);
    float f[C::NCW];
    L = 0.f;
#pragma unroll
    for (int w = 0; w < C::NCW; ++w) {
        f[w] = M == -INFINITY ? 0.f : fast_exp2(red_m[w * NT + head] - M);
        L += f[w] * red_l[w * NT + head];
    }
    const float inv = (L > 0.f ? 1.f / L : 0.f) * out_scale;
#pragma unroll
    for (int e = 0; e < C::E; ++e) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) x += f[w] * red_o[(w * NT + head) * C::RED_STRIDE + d0 + e];
        acc[e] = x * inv;
    }
}

__device__ __forceinline__ float lse_from(float M, float L)
{
    return L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace kvp
