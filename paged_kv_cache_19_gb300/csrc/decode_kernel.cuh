// decode_kernel.cuh -- main kernel of paged decode attention.
//
// What it computes (per sequence b and query head h, kv = h / g):
//   s_t = scale * q[b,h,:] . K[t,kv,:],  out = sum_t softmax(s)_t V[t,kv,:]
// over the tokens 0 .. ctx_b - 1 of the sequence, read in place through its
// block table (brunomaga.github.io "inference-prefill-decode-roofline-cache",
// section "PagedAttention: memory management for the KV cache",
// paged_decode_attention; learn.mohebi.ai lesson 12, "PagedAttention
// (4.1-4.3)": the kernel reads K and V block by block and merges them with the
// online-softmax update).  A CTA owns one (sequence, kv head, query-head tile,
// split-KV chunk); chunks are merged by log-sum-exp in the merge kernel.
//
// GB300 design:
//   * One producer warp streams K and V blocks with 5-D TMA tensor loads
//     (cp.async.bulk.tensor, 128-byte swizzle) into a ring of NSTAGE shared-
//     memory stages, one cache block per stage, completion tracked by
//     mbarriers; the block-table row is fetched 32 entries at a time with one
//     coalesced load and broadcast by shuffles.
//   * Four consumer warps take the stages round-robin (stage i -> warp i % 4,
//     so each warp owns NSTAGE / 4 stages and waits on them in order).  Each
//     warp keeps its own online-softmax state over its blocks; the four states
//     are merged in shared memory at the end.
//   * The g query heads of a GQA group share one read of K/V: scores are a
//     tensor-core product S^T[16 tokens x 8 heads] = K[16 x d] . Q^T[d x 8]
//     (mma.m16n8k16, tokens on the M side so a group of up to 8 heads fills the
//     N side), and P.V is O^T[d x 8] += V^T[d x 16] . P^T[16 x 8], with the
//     probabilities moved from the accumulator layout to the B-operand layout by
//     movmatrix.  bf16 caches feed the MMA straight from ldmatrix; fp8 e4m3
//     caches are converted to f16 in registers (exact) and the per-head scales
//     are applied to the fp32 scores and outputs.
//   * Every wait is bounded (WAIT_LIMIT_NS); a late barrier sets
//     KV_DEVERR_TIMEOUT and the CTA drains its copies and returns.
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
    static constexpr int NSTAGE = STAGE >= 16384 ? 4 : (STAGE >= 8192 ? 8 : 16);
    static constexpr int NCW = 4;                   // consumer warps
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int MT = BS / 16;              // 16-token tiles per block
    static constexpr int NTT = NT / 8;              // 8-head tiles
    static constexpr int KS = D / 16;               // 16-wide slices of head_dim
    static constexpr int RED_STRIDE = D + 4;        // padded row of the epilogue buffer (floats)
    static constexpr int RED_BYTES = (NCW * NT * RED_STRIDE + 2 * NCW * NT) * 4;
    static constexpr int SMEM = 1024 + NSTAGE * STAGE + NSTAGE * (8 + 8 + 4);
    static constexpr int MINB = NT == 8 ? 3 : 2;
    static_assert(ROWB % 128 == 0, "rows must be whole 128-byte swizzle rows");
    static_assert(NSTAGE % NCW == 0, "each consumer warp must own whole stages");
    static_assert(RED_BYTES <= NSTAGE * STAGE, "epilogue buffer reuses the stages");
    static_assert(!FP8 || D == 128, "fp8 path is laid out for head_dim 128");
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

template <bool FP8, int D, int BS, int NT>
__global__ void __launch_bounds__(DecodeCfg<FP8, D, BS, NT>::THREADS, DecodeCfg<FP8, D, BS, NT>::MINB)
paged_decode_main(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeParams p)
{
    using C = DecodeCfg<FP8, D, BS, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NSTAGE * C::STAGE);
    uint64_t* empty = full + C::NSTAGE;
    int* stage_blk = reinterpret_cast<int*>(empty + C::NSTAGE);

    const int b = blockIdx.z;
    const int kvh = blockIdx.y / p.head_groups;
    const int hg = blockIdx.y - kvh * p.head_groups;
    const int split = blockIdx.x;

    int ctx = __ldg(p.ctx + b);
    const int cap = p.max_blocks * BS;
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) atomicOr(p.err, KV_DEVERR_CONTEXT);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int nblk = (ctx + BS - 1) / BS;
    const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    if (split >= nsplit) return;                     // this sequence has fewer chunks
    const int blk0 = split * p.split_blocks;
    const int nb = max(0, min(nblk - blk0, p.split_blocks));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // ------------------------------------------------------------ producer warp
    if (warp == C::NCW) {
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        const int32_t* trow = p.tables + static_cast<size_t>(b) * p.max_blocks + blk0;
        int issued = 0;
        bool ok = true;
        for (int base = 0; base < nb && ok; base += 32) {
            const int j = base + lane;
            int id = -1;
            if (j < nb) {
                id = __ldg(trow + j);
                if (id < 0 || id >= p.num_blocks) {
                    atomicOr(p.err, KV_DEVERR_BLOCK_ID);
                    id = -1;                          // skipped: never addressed
                }
            }
            const int cnt = min(32, nb - base);
            for (int k = 0; k < cnt; ++k) {
                const int blk = __shfl_sync(FULL_MASK, id, k);
                const int it = base + k;
                const int st = it % C::NSTAGE;
                const uint32_t ph = static_cast<uint32_t>(it / C::NSTAGE) & 1u;
                int good = 1;
                if (lane == 0) {
                    if (!mbar_wait_bounded(smem_u32(empty + st), ph ^ 1u)) {
                        atomicOr(p.err, KV_DEVERR_TIMEOUT);
                        good = 0;
                    } else {
                        stage_blk[st] = blk;
                        const uint32_t fb = smem_u32(full + st);
                        if (blk >= 0) {
                            const uint32_t dst = smem_u32(smem + st * C::STAGE);
                            mbar_arrive_expect_tx(fb, C::STAGE);
                            tma_load_5d(dst, &tmk, 0, 0, kvh, 0, blk, fb);
                            tma_load_5d(dst + C::TILE, &tmv, 0, 0, kvh, 0, blk, fb);
                        } else {
                            mbar_arrive(fb);
                        }
                    }
                }
                good = __shfl_sync(FULL_MASK, good, 0);
                if (!good) {
                    ok = false;
                    break;
                }
                issued = it + 1;
            }
        }
        // Drain: the CTA must not exit while a copy into its shared memory is
        // in flight.  Only the last NSTAGE loads can still be pending.
        if (lane == 0) {
            for (int it = max(0, issued - C::NSTAGE); it < issued; ++it) {
                if (!mbar_wait_bounded(smem_u32(full + (it % C::NSTAGE)),
                                       static_cast<uint32_t>(it / C::NSTAGE) & 1u)) {
                    atomicOr(p.err, KV_DEVERR_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumer warps
    const int r = lane >> 2;          // row group of the MMA fragments
    const int c = lane & 3;           // column pair of the MMA fragments
    const int g = p.group;
    const int hq0 = kvh * g + hg * NT;                 // query head of local head 0
    const int nh = min(NT, g - hg * NT);               // real heads in this tile

    // Q^T as the MMA B operand: element (k, n) = q[head n][d(k)].
    uint32_t qf[C::KS][C::NTT][2];
    float sl2 = p.scale_log2;
    const uint16_t* qb = p.q + (static_cast<size_t>(b) * p.q_heads + hq0) * D;
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
    } else {
        // fp8 cache: the K operand is read 4 bytes at a time, so slice ks of
        // thread column c holds d = 32c + 4ks + {0,1} (B rows 2c, 2c+1) and
        // d = 32c + 4ks + {2,3} (B rows 2c+8, 2c+9).  Q uses the same map.
        // q goes to f16 (exact for bf16 values inside the f16 range); a power-
        // of-two pre-scale keeps max|q| below 2^15 and is undone in sl2.
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
        sl2 *= up * __ldg(p.k_scale + kvh);
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int ks = 0; ks < C::KS; ++ks) {
                qf[ks][nt][0] = pack_f16x2(qv[ks][nt][0] * down, qv[ks][nt][1] * down);
                qf[ks][nt][1] = pack_f16x2(qv[ks][nt][2] * down, qv[ks][nt][3] * down);
            }
    }

    // O^T accumulators: o[ms][nt][hi*2 + j] holds (d(ms, r + 8 hi), head nt*8 + 2c + j).
    float o[C::KS][C::NTT][4];
    float m_run[C::NTT][2], l_run[C::NTT][2];
#pragma unroll
    for (int ms = 0; ms < C::KS; ++ms)
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[ms][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -INFINITY;
        l_run[nt][0] = l_run[nt][1] = 0.f;
    }

    for (int it = warp; it < nb; it += C::NCW) {
        const int st = it % C::NSTAGE;
        const uint32_t ph = static_cast<uint32_t>(it / C::NSTAGE) & 1u;
        const bool arrived = mbar_wait_bounded(smem_u32(full + st), ph);
        if (!__all_sync(FULL_MASK, arrived)) {
            if (lane == 0) atomicOr(p.err, KV_DEVERR_TIMEOUT);
            break;
        }
        const int blk = stage_blk[st];
        if (blk >= 0) {
            const int nvalid = min(BS, ctx - (blk0 + it) * BS);
            const uint32_t tk = smem_u32(smem + st * C::STAGE);
            const uint32_t tv = tk + C::TILE;

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

            // ---- online softmax over this block (log2 domain); slots at or past
            // ctx are replaced by -inf, never read as values.
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
                            const float x = tok < nvalid ? s[mt][nt][2 * hi + j] * sl2 : -INFINITY;
                            s[mt][nt][2 * hi + j] = x;
                            mx = fmaxf(mx, x);
                        }
                    mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 16));
                    const float m_new = fmaxf(m_run[nt][j], mx);
                    const float m_use = m_new == -INFINITY ? 0.f : m_new;
                    const float a_ = fast_exp2(m_run[nt][j] - m_use);
                    m_run[nt][j] = m_new;
                    float ls = 0.f;
#pragma unroll
                    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                        for (int hi = 0; hi < 2; ++hi) {
                            const float pr = fast_exp2(s[mt][nt][2 * hi + j] - m_use);
                            s[mt][nt][2 * hi + j] = pr;
                            ls += pr;
                        }
                    l_run[nt][j] = l_run[nt][j] * a_ + ls;
                    alpha[nt][j] = a_;
                    rescale |= (a_ != 1.f);
                }
            }
            if (__any_sync(FULL_MASK, rescale)) {
#pragma unroll
                for (int ms = 0; ms < C::KS; ++ms)
#pragma unroll
                    for (int nt = 0; nt < C::NTT; ++nt) {
                        o[ms][nt][0] *= alpha[nt][0];
                        o[ms][nt][1] *= alpha[nt][1];
                        o[ms][nt][2] *= alpha[nt][0];
                        o[ms][nt][3] *= alpha[nt][1];
                    }
            }

            // ---- P^T as the B operand: transpose each 8x8 quadrant of the
            // accumulator layout (rows = tokens) into the B layout (rows = heads).
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
                            mma_bf16_16816(o[ms][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
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
                            mma_f16_16816(o[2 * w][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
                        a[0] = e4m3x2_to_f16x2(y01);
                        a[1] = e4m3x2_to_f16x2(y01 >> 16);
                        a[2] = e4m3x2_to_f16x2(y23);
                        a[3] = e4m3x2_to_f16x2(y23 >> 16);
#pragma unroll
                        for (int nt = 0; nt < C::NTT; ++nt)
                            mma_f16_16816(o[2 * w + 1][nt], a, pb[mt][nt][0], pb[mt][nt][1]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + st));
    }

    // ------------------------------------------------------------ epilogue
    // Row sums were kept per thread; add the 8 row groups that share a column.
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = l_run[nt][j];
            l += __shfl_xor_sync(FULL_MASK, l, 4);
            l += __shfl_xor_sync(FULL_MASK, l, 8);
            l += __shfl_xor_sync(FULL_MASK, l, 16);
            l_run[nt][j] = l;
        }

    named_barrier_sync(1, C::NCW * 32);     // every consumer is done with the stages
    float* red_o = reinterpret_cast<float*>(smem);                  // [NCW][NT][RED_STRIDE]
    float* red_m = red_o + C::NCW * NT * C::RED_STRIDE;             // [NCW][NT]
    float* red_l = red_m + C::NCW * NT;                             // [NCW][NT]
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
                    red_o[(warp * NT + head) * C::RED_STRIDE + d] = o[ms][nt][2 * hi + j];
                }
    if (r == 0) {
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int head = nt * 8 + 2 * c + j;
                red_m[warp * NT + head] = m_run[nt][j];
                red_l[warp * NT + head] = l_run[nt][j];
            }
    }
    named_barrier_sync(1, C::NCW * 32);

    constexpr int E = NT * D / (C::NCW * 32);     // output elements per thread
    static_assert(E % 2 == 0 && D % E == 0, "epilogue split");
    const int t = threadIdx.x;
    const int head = (t * E) / D;
    const int d0 = (t * E) % D;
    if (head < nh) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, red_m[w * NT + head]);
        float f[C::NCW];
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) {
            f[w] = M == -INFINITY ? 0.f : fast_exp2(red_m[w * NT + head] - M);
            L += f[w] * red_l[w * NT + head];
        }
        float inv = L > 0.f ? 1.f / L : 0.f;
        if constexpr (FP8) inv *= __ldg(p.v_scale + kvh);
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < C::NCW; ++w) x += f[w] * red_o[(w * NT + head) * C::RED_STRIDE + d0 + e];
            acc[e] = x * inv;
        }
        const int gq = hq0 + head;
        const size_t bh = static_cast<size_t>(b) * p.q_heads + gq;
        if (nsplit == 1) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + bh * D + d0);
#pragma unroll
            for (int e = 0; e < E; e += 2) dst[e / 2] = pack_bf16x2(acc[e], acc[e + 1]);
            if (p.lse != nullptr && d0 == 0)
                p.lse[bh] = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
        } else {
            float* dst = p.part_o + (bh * p.max_splits + split) * D + d0;
#pragma unroll
            for (int e = 0; e < E; ++e) dst[e] = acc[e];
            if (d0 == 0) {
                p.part_ml[(bh * p.max_splits + split) * 2 + 0] = M;
                p.part_ml[(bh * p.max_splits + split) * 2 + 1] = L;
            }
        }
    }
}

template <bool FP8, int D, int BS, int NT>
cudaError_t prepare_variant()
{
    using C = DecodeCfg<FP8, D, BS, NT>;
    return cudaFuncSetAttribute(paged_decode_main<FP8, D, BS, NT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
}

template <bool FP8, int D, int BS, int NT>
cudaError_t launch_variant(dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv,
                           const DecodeParams& p, cudaStream_t s)
{
    using C = DecodeCfg<FP8, D, BS, NT>;
    paged_decode_main<FP8, D, BS, NT><<<grid, C::THREADS, C::SMEM, s>>>(tk, tv, p);
    return cudaGetLastError();
}

}  // namespace kvp
