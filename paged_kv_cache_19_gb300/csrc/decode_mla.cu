// decode_mla.cu -- absorbed multi-head latent attention over a paged latent
// cache: every query head of a sequence attends over one shared cached vector
// per token (512 latent numbers followed by the 64-number rotary key); the key
// is the whole vector and the value its latent part (xuewyang.github.io/posts/kv,
// "MLA: how does decode get full-size keys and values back?": W_UK is folded
// into the query and W_UV applied after the attention, so full keys and values
// are never built).
//
// One CTA per (sequence, tile of 16 query heads, split-KV chunk).  Four consumer
// warps all work on every stage of SUB tokens x 1152 bytes:
//   * scores S^T[tokens x 16 heads] = C[tokens x 576] . Q^T are split over the
//     576 numbers (warp w sums its 144 on the tensor cores, with the query
//     fragments held in registers); the four partial sums are exchanged through
//     shared memory across one barrier per stage and added in the same order by
//     every warp, so all warps hold the same scores and run the same online
//     softmax; then warp w accumulates O^T[latent 128w .. 128w+127 x 16 heads]
//     += C^T . P^T.  Splitting the 576-long sums keeps each warp's chain of
//     dependent MMAs short (9) and its accumulator at 64 registers.
//   * stages arrive by 5-D TMA loads (128-byte swizzle) into a ring guarded by
//     "full" mbarriers, in one of two ways:
//       PROD: a fifth warp issues the loads and waits for "empty" mbarriers that
//         the consumers arrive on -- 32-token stages, 2 stages, 2 CTAs per SM;
//         the load of a stage starts as soon as its slot is released.
//       otherwise: the exchange barrier already tells that the previous stage is
//         free, so thread 0 issues the load NSTAGE - 1 stages ahead right there
//         -- no producer warp and no "empty" barriers, 16-token stages, 3
//         stages, 3 CTAs per SM (12 consumer warps).
//     The host takes the producer form for grids of up to three CTAs per SM and
//     the three-CTA form beyond.
//   * the swizzled shared-memory offsets each lane reads are fixed per warp and
//     computed once, before the loop.
//   * split chunks leave fp32 partials and the last one to finish merges them by
//     log-sum-exp (ticket in the workspace), as in the GQA decode kernel.
//   * paged_mla_decode_step: the CTA whose chunk holds the block with the sequence's
//     new vector writes it there (72 threads, 16 bytes each) before the barrier that
//     precedes every load.
// Every wait is bounded; a stage that does not arrive sets KV_DEVERR_TIMEOUT and
// all consumer warps leave the loop together (the decision is shared across the
// exchange barrier), after the loads in flight have landed (bounded waits).
#include "append_row.cuh"
#include "decode_common.cuh"
#include "kernels.h"

namespace kvp {

template <int BS, int SUB, int NSTAGE, bool PROD>
struct MlaCfg {
    static constexpr int DK = MLA_DK;               // numbers per cached token (key)
    static constexpr int DV = MLA_DV;               // latent numbers (value)
    static constexpr int DCH = DK * 2 / 128;        // 128-byte rows per token: 9
    static constexpr int STAGE = SUB * DK * 2;      // bytes of one stage
    static constexpr int SPB = BS / SUB;            // stages per block
    static constexpr int NCW = 4;
    static constexpr int THREADS = (NCW + (PROD ? 1 : 0)) * 32;
    static_assert(NCW * 32 >= MLA_DK / 8, "the step's new vector: one 16-byte vector a thread");
    static constexpr int NT = 16;                   // heads per CTA
    static constexpr int NTT = NT / 8;
    static constexpr int MT = SUB / 16;             // 16-token slices per stage
    static constexpr int KSW = DK / 16 / NCW;       // 16-wide k slices per warp: 9
    static constexpr int MSW = DV / 16 / NCW;       // 16-wide latent slices per warp: 8
    static constexpr int MT_BYTES = 16 * DCH * 128; // bytes between 16-token slices
    static constexpr int XFLOATS = NCW * MT * NTT * 32 * 4;   // one exchange buffer
    static constexpr int XBYTES = 2 * XFLOATS * 4;
    static constexpr int RED_STRIDE = DV + 4;
    static constexpr int RED_BYTES = (NT * RED_STRIDE + 2 * NT) * 4;
    static constexpr int E = NT * DV / (NCW * 32);  // output numbers per thread: 64
    static constexpr int RING = NSTAGE * STAGE;
    static constexpr int SMEM = 1024 + RING + XBYTES + NSTAGE * (8 + 8 + 4) + 16;
    static constexpr int MINB = PROD ? 2 : 3;      // CTAs per SM (shared memory allows it)
    static_assert(MINB * (SMEM + 1024) <= 228 * 1024, "CTAs per SM fit the shared memory");
    static_assert(BS % SUB == 0 && SUB % 16 == 0, "stages are whole 16-token slices of a block");
    static_assert(NSTAGE >= 2, "one stage in use, at least one loading");
    static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert((16 * DCH) % 8 == 0, "16-token slices keep the swizzle phase");
    static_assert(RED_BYTES <= RING, "epilogue buffer reuses the stages");
    static_assert(DK % (16 * NCW) == 0 && DV % (16 * NCW) == 0, "k / latent split");
};

struct MlaState {
    float o[MLA_DV / 16 / 4][2][4];                 // [latent slice][head tile][mma C]
    float m[2][2];
    float l[2][2];
};

// Byte offset, inside a stage, of the 16-byte chunk `ch` (of 72) of token `tok`:
// the 128-byte swizzle of a TMA tile whose rows are (token, 128-byte piece).
template <int DCH>
__device__ __forceinline__ uint32_t swz_off(int tok, int ch)
{
    const int row = tok * DCH + (ch >> 3);
    return static_cast<uint32_t>(row * 128 + ((((ch & 7) ^ (row & 7))) << 4));
}

// Thread 0: issue (or skip) the load of chunk stage `it` into ring slot it % NSTAGE.
// Returns the block id it used (-1: bad id, flagged; the stage arrives empty).
template <class C, int SUB, int NSTAGE>
__device__ __forceinline__ void issue_stage(int it, const int32_t* trow, int num_blocks,
                                            uint8_t* smem, uint64_t* full, int* stage_blk,
                                            const CUtensorMap* tmc, uint32_t* err)
{
    const int j = it / C::SPB;
    const int sub = it - j * C::SPB;
    int blk = __ldg(trow + j);
    if (blk < 0 || blk >= num_blocks) {
        atomicOr(err, KV_DEVERR_BLOCK_ID);
        blk = -1;
    }
    const int st = it % NSTAGE;
    stage_blk[st] = blk;
    const uint32_t fb = smem_u32(full + st);
    if (blk >= 0) {
        mbar_arrive_expect_tx(fb, C::STAGE);
        tma_load_5d(smem_u32(smem + st * C::STAGE), tmc, 0, 0, 0, sub * SUB, blk, fb);
    } else {
        mbar_arrive(fb);
    }
}

template <int BS, int SUB, int NSTAGE, bool PROD>
__global__ void __launch_bounds__(MlaCfg<BS, SUB, NSTAGE, PROD>::THREADS,
                                  MlaCfg<BS, SUB, NSTAGE, PROD>::MINB)
paged_mla_decode_main(const __grid_constant__ CUtensorMap tmc, const MlaParams p)
{
    using C = MlaCfg<BS, SUB, NSTAGE, PROD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* xbuf = reinterpret_cast<float*>(smem + C::RING);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING + C::XBYTES);
    uint64_t* empty = full + NSTAGE;                // PROD only
    int* stage_blk = reinterpret_cast<int*>(empty + NSTAGE);
    int* flags = stage_blk + NSTAGE;                // [0]: abort, [1]: merge

    const int ht = blockIdx.x;
    const int b = blockIdx.y;
    const int split = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = lane >> 2;
    const int c = lane & 3;
    const int blk0 = split * p.split_blocks;
    const int nh = min(C::NT, p.q_heads - ht * C::NT);
    const size_t row0 = static_cast<size_t>(b) * p.q_heads + ht * C::NT;   // global (b, head)

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(smem_u32(full + i), 1);
            if (PROD) mbar_init(smem_u32(empty + i), C::NCW);
        }
        flags[0] = 0;
        fence_mbar_init();
    }
    grid_dependency_wait();                          // inputs of the preceding kernel are ready

    const int32_t* trow = p.tables + static_cast<size_t>(b) * p.max_blocks + blk0;
    int id_first = -1;
    if (PROD && warp == C::NCW && blk0 + lane < p.max_blocks) id_first = __ldg(trow + lane);

    // Q^T fragments of this warp's 144 numbers: k slice kk is slice 9w + kk.
    uint32_t qf[C::KSW][C::NTT][2];
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt) {
        if (warp >= C::NCW) break;
        const int hl = nt * 8 + r;
        const bool valid = hl < nh;
        const uint16_t* qh = p.q + (row0 + (valid ? hl : 0)) * C::DK;
#pragma unroll
        for (int kk = 0; kk < C::KSW; ++kk) {
            const int k0 = (warp * C::KSW + kk) * 16;
            qf[kk][nt][0] = valid ? *reinterpret_cast<const uint32_t*>(qh + k0 + 2 * c) : 0u;
            qf[kk][nt][1] = valid ? *reinterpret_cast<const uint32_t*>(qh + k0 + 8 + 2 * c) : 0u;
        }
    }
    int ctx = __ldg(p.ctx + b);
    const int cap = p.max_blocks * BS;
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && split == 0 && ht == 0) atomicOr(p.err, KV_DEVERR_CONTEXT);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int nblk = (ctx + BS - 1) / BS;
    const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    const int nb = max(0, min(nblk - blk0, p.split_blocks));
    const int nstages = nb * C::SPB;
    // paged_mla_decode_step: a position outside the table is flagged once per sequence (as
    // the append would) and not written; a CTA whose chunk holds the block with the new
    // vector writes it there first (its first 72 threads, one 16-byte vector each), before
    // the barrier that precedes every load.  Several head tiles write the same bytes.
    if (p.kv_new != nullptr) {
        const int raw = __ldg(p.ctx + b);
        if (threadIdx.x == 0 && split == 0 && ht == 0 && (raw < 1 || raw > cap))
            atomicOr(p.err, KV_DEVERR_POSITION);
        const int step_j = mla_step_block(p, b, BS) - blk0;
        if (step_j >= 0 && step_j < nb && threadIdx.x < MLA_DK / 8) {
            const int bid = __ldg(trow + step_j);
            if (bid >= 0 && bid < p.num_blocks) {   // a bad id is flagged by the load path
                write_latent_share(p, b, bid, BS, (raw - 1) % BS, threadIdx.x, MLA_DK / 8);
                fence_proxy_async_all();
            }
        }
    }
    __syncthreads();                                 // barriers initialised
    if (split >= nsplit) {
        grid_dependents_launch();
        return;
    }

    // ------------------------------------------------------------ producer warp (PROD)
    if (PROD && warp == C::NCW) {
        if (lane == 0) prefetch_tensormap(&tmc);
        int issued = 0;
        bool ok = true;
        for (int base = 0; base < nb && ok; base += 32) {
            const int j = base + lane;
            int id = -1;
            if (j < nb) {
                id = base == 0 ? id_first : __ldg(trow + j);
                if (id < 0 || id >= p.num_blocks) {
                    atomicOr(p.err, KV_DEVERR_BLOCK_ID);
                    id = -1;
                }
            }
            const int cnt = min(32, nb - base);
            for (int k = 0; k < cnt && ok; ++k) {
                const int blk = __shfl_sync(FULL_MASK, id, k);
#pragma unroll 1
                for (int sub = 0; sub < C::SPB; ++sub) {
                    const int it = (base + k) * C::SPB + sub;
                    const int st = it % NSTAGE;
                    const uint32_t ph = static_cast<uint32_t>(it / NSTAGE) & 1u;
                    int good = 1;
                    if (lane == 0) {
                        if (!mbar_wait_bounded(smem_u32(empty + st), ph ^ 1u)) {
                            atomicOr(p.err, KV_DEVERR_TIMEOUT);
                            good = 0;
                        } else {
                            stage_blk[st] = blk;
                            const uint32_t fb = smem_u32(full + st);
                            if (blk >= 0) {
                                mbar_arrive_expect_tx(fb, C::STAGE);
                                tma_load_5d(smem_u32(smem + st * C::STAGE), &tmc, 0, 0, 0,
                                            sub * SUB, blk, fb);
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
        }
        grid_dependents_launch();
        if (lane == 0) {                            // the CTA must not exit with copies in flight
            for (int it = max(0, issued - NSTAGE); it < issued; ++it) {
                if (!mbar_wait_bounded(smem_u32(full + (it % NSTAGE)),
                                       static_cast<uint32_t>(it / NSTAGE) & 1u)) {
                    atomicOr(p.err, KV_DEVERR_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumer warps
    int issued = 0;                                  // thread 0 (not PROD): loads issued
    if (!PROD && threadIdx.x == 0) {
        prefetch_tensormap(&tmc);
        for (; issued < min(NSTAGE, nstages); ++issued)
            issue_stage<C, SUB, NSTAGE>(issued, trow, p.num_blocks, smem, full, stage_blk, &tmc,
                                        p.err);
    }

    MlaState st;
#pragma unroll
    for (int ms = 0; ms < C::MSW; ++ms)
#pragma unroll
        for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.o[ms][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt) {
        st.m[nt][0] = st.m[nt][1] = -INFINITY;
        st.l[nt][0] = st.l[nt][1] = 0.f;
    }
    const float sl2 = p.scale_log2;
    // Per-lane offsets of the ldmatrix reads (slice 0; slice mt adds mt * MT_BYTES,
    // which keeps the swizzle phase since 16 * 9 rows is a multiple of 8).
    uint32_t off_s[C::KSW], off_v[C::MSW];
    {
        const int tok_s = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < C::KSW; ++kk)
            off_s[kk] = swz_off<C::DCH>(tok_s, 2 * (warp * C::KSW + kk) + (lane >> 4));
        const int quad = lane >> 3;
        const int tok_v = (lane & 7) + (quad >> 1) * 8;
#pragma unroll
        for (int ms = 0; ms < C::MSW; ++ms)
            off_v[ms] = swz_off<C::DCH>(tok_v, 2 * (warp * C::MSW + ms) + (quad & 1));
    }
    float* xw = xbuf + warp * (C::MT * C::NTT * 32 * 4) + lane * 4;
    int waited = 0;                                  // stages this CTA has seen arrive

    for (int it = 0; it < nstages; ++it) {
        const int s = it % NSTAGE;
        const uint32_t ph = static_cast<uint32_t>(it / NSTAGE) & 1u;
        const bool arrived = __all_sync(FULL_MASK, mbar_wait_bounded(smem_u32(full + s), ph));
        if (!arrived && lane == 0) {
            atomicOr(p.err, KV_DEVERR_TIMEOUT);
            flags[0] = 1;
        }
        if (arrived) waited = it + 1;
        const int blk = arrived ? stage_blk[s] : -1;
        const uint32_t tile = smem_u32(smem + s * C::STAGE);
        const int xo = (it & 1) * C::XFLOATS;

        // ---- partial scores over this warp's 144 numbers
        float sc[C::MT][C::NTT][4];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[mt][nt][e] = 0.f;
        if (blk >= 0) {
#pragma unroll
            for (int kk = 0; kk < C::KSW; ++kk)
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    uint32_t a[4];
                    ldsm_x4(tile + mt * C::MT_BYTES + off_s[kk], a);
#pragma unroll
                    for (int nt = 0; nt < C::NTT; ++nt)
                        mma_bf16_16816(sc[mt][nt], a, qf[kk][nt][0], qf[kk][nt][1]);
                }
        }
        // ---- exchange: every warp publishes its partial sums, then adds all four.
        // Past this barrier every warp is also done with stage it - 1.
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < C::NTT; ++nt)
                *reinterpret_cast<float4*>(xw + xo + (mt * C::NTT + nt) * 128) =
                    make_float4(sc[mt][nt][0], sc[mt][nt][1], sc[mt][nt][2], sc[mt][nt][3]);
        named_barrier_sync(1, C::NCW * 32);
        if (flags[0]) break;                        // a stage never arrived: all warps leave
        if (!PROD && threadIdx.x == 0 && it >= 1 && issued < nstages) {
            issue_stage<C, SUB, NSTAGE>(issued, trow, p.num_blocks, smem, full, stage_blk, &tmc,
                                        p.err);   // into the slot of stage it - 1
            ++issued;
        }
        if (blk < 0) {                              // skipped (bad id): nothing to fold in
            if (PROD) {
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(empty + s));
            }
            continue;
        }
        {
            const float* xr = xbuf + xo + lane * 4;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < C::NTT; ++nt) {
                    const int o = (mt * C::NTT + nt) * 128;
                    float4 acc = *reinterpret_cast<const float4*>(xr + o);
#pragma unroll
                    for (int w = 1; w < C::NCW; ++w) {
                        const float4 v = *reinterpret_cast<const float4*>(
                            xr + w * (C::MT * C::NTT * 128) + o);
                        acc.x += v.x;
                        acc.y += v.y;
                        acc.z += v.z;
                        acc.w += v.w;
                    }
                    sc[mt][nt][0] = acc.x;
                    sc[mt][nt][1] = acc.y;
                    sc[mt][nt][2] = acc.z;
                    sc[mt][nt][3] = acc.w;
                }
        }
        // ---- online softmax (log2 domain); tokens at or past lim are not cached.
        // The max is taken on the raw scores (the scale is positive) and the scale
        // is applied inside the exponent: p = 2^(s * sl2 - m).
        const int lim = ctx - (blk0 * BS + it * SUB);
        const int nvalid = min(SUB, lim);
        const bool partial = nvalid < SUB;
        if (partial) {
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi)
                    if (mt * 16 + r + 8 * hi >= nvalid) {
#pragma unroll
                        for (int nt = 0; nt < C::NTT; ++nt) {
                            sc[mt][nt][2 * hi] = -INFINITY;
                            sc[mt][nt][2 * hi + 1] = -INFINITY;
                        }
                    }
        }
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
                    for (int hi = 0; hi < 2; ++hi) mx = fmaxf(mx, sc[mt][nt][2 * hi + j]);
                mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 16));
                const float m_new = fmaxf(st.m[nt][j], mx * sl2);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float a_ = fast_exp2(st.m[nt][j] - m_use);
                st.m[nt][j] = m_new;
                float ls = 0.f;
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        const float pr = fast_exp2(fmaf(sc[mt][nt][2 * hi + j], sl2, -m_use));
                        sc[mt][nt][2 * hi + j] = pr;
                        ls += pr;
                    }
                st.l[nt][j] = st.l[nt][j] * a_ + ls;
                alpha[nt][j] = a_;
                rescale |= (a_ != 1.f);
            }
        }
        if (__any_sync(FULL_MASK, rescale)) {
#pragma unroll
            for (int ms = 0; ms < C::MSW; ++ms)
#pragma unroll
                for (int nt = 0; nt < C::NTT; ++nt) {
                    st.o[ms][nt][0] *= alpha[nt][0];
                    st.o[ms][nt][1] *= alpha[nt][1];
                    st.o[ms][nt][2] *= alpha[nt][0];
                    st.o[ms][nt][3] *= alpha[nt][1];
                }
        }

        // ---- O^T[latent slice x heads] += C^T[latent x tokens] . P^T[tokens x heads]
        // (in a partial stage the values of tokens past the cache are zeroed: they
        // may hold anything, and 0 * NaN would poison the sums)
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            uint32_t pb[C::NTT][2];
#pragma unroll
            for (int nt = 0; nt < C::NTT; ++nt) {
                pb[nt][0] = movmatrix_trans(pack_bf16x2(sc[mt][nt][0], sc[mt][nt][1]));
                pb[nt][1] = movmatrix_trans(pack_bf16x2(sc[mt][nt][2], sc[mt][nt][3]));
            }
            if (!partial) {
#pragma unroll
                for (int ms = 0; ms < C::MSW; ++ms) {
                    uint32_t a[4];
                    ldsm_x4_trans(tile + mt * C::MT_BYTES + off_v[ms], a);
#pragma unroll
                    for (int nt = 0; nt < C::NTT; ++nt)
                        mma_bf16_16816(st.o[ms][nt], a, pb[nt][0], pb[nt][1]);
                }
            } else {
                const int t0 = mt * 16 + 2 * c;
                const uint32_t mlo = (t0 < nvalid ? 0x0000ffffu : 0u) | (t0 + 1 < nvalid ? 0xffff0000u : 0u);
                const uint32_t mhi = (t0 + 8 < nvalid ? 0x0000ffffu : 0u) | (t0 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
                for (int ms = 0; ms < C::MSW; ++ms) {
                    uint32_t a[4];
                    ldsm_x4_trans(tile + mt * C::MT_BYTES + off_v[ms], a);
                    a[0] &= mlo;
                    a[1] &= mlo;
                    a[2] &= mhi;
                    a[3] &= mhi;
#pragma unroll
                    for (int nt = 0; nt < C::NTT; ++nt)
                        mma_bf16_16816(st.o[ms][nt], a, pb[nt][0], pb[nt][1]);
                }
            }
        }
        if (PROD) {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(empty + s));
        }
    }
    if (!PROD && threadIdx.x == 0) {
        // loads issued but never waited for (only after a timeout) must land first
        for (int it = waited; it < issued; ++it) {
            if (!mbar_wait_bounded(smem_u32(full + (it % NSTAGE)),
                                   static_cast<uint32_t>(it / NSTAGE) & 1u))
                break;
        }
    }

    // ------------------------------------------------------------ epilogue
    grid_dependents_launch();
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
    named_barrier_sync(1, C::NCW * 32);             // every consumer is done with the stages
    float* red = reinterpret_cast<float*>(smem);    // [NT][RED_STRIDE] normalised out, then m, l
    float* red_m = red + C::NT * C::RED_STRIDE;
    float* red_l = red_m + C::NT;
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int head = nt * 8 + 2 * c + j;
            const float inv = st.l[nt][j] > 0.f ? 1.f / st.l[nt][j] : 0.f;
#pragma unroll
            for (int ms = 0; ms < C::MSW; ++ms)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi) {
                    const int d = (warp * C::MSW + ms) * 16 + r + 8 * hi;
                    red[head * C::RED_STRIDE + d] = st.o[ms][nt][2 * hi + j] * inv;
                }
            if (warp == 0 && r == 0) {
                red_m[head] = st.m[nt][j];
                red_l[head] = st.l[nt][j];
            }
        }
    named_barrier_sync(1, C::NCW * 32);

    const int t = threadIdx.x;
    const int head = (t * C::E) / C::DV;
    const int d0 = (t * C::E) % C::DV;
    const size_t bh = row0 + head;
    const float M = red_m[head];
    const float L = red_l[head];
    const float* src = red + head * C::RED_STRIDE + d0;
    if (head < nh) {
        if (nsplit == 1) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + bh * C::DV + d0);
#pragma unroll
            for (int e = 0; e < C::E; e += 8)
                dst[e / 8] = make_uint4(pack_bf16x2(src[e], src[e + 1]), pack_bf16x2(src[e + 2], src[e + 3]),
                                        pack_bf16x2(src[e + 4], src[e + 5]),
                                        pack_bf16x2(src[e + 6], src[e + 7]));
            if (p.lse != nullptr && d0 == 0) p.lse[bh] = lse_from(M, L);
        } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + (bh * p.max_splits + split) * C::DV + d0);
#pragma unroll
            for (int e = 0; e < C::E; e += 4) dst[e / 4] = make_float4(src[e], src[e + 1], src[e + 2], src[e + 3]);
            if (d0 == 0) {
                p.part_ml[(bh * p.max_splits + split) * 2 + 0] = M;
                p.part_ml[(bh * p.max_splits + split) * 2 + 1] = L;
            }
            __threadfence();
        }
    }
    if (nsplit == 1) return;

    // ---- ticket: the last chunk of this (sequence, head tile) merges all chunks
    named_barrier_sync(1, C::NCW * 32);
    int* ticket = p.tickets + static_cast<size_t>(b) * p.head_tiles + ht;
    if (t == 0) {
        const int last = atomicAdd(ticket, 1) == nsplit - 1;
        if (last) __threadfence();
        flags[1] = last;
    }
    named_barrier_sync(1, C::NCW * 32);
    if (!flags[1]) return;
    if (head < nh) {
        const float* ml = p.part_ml + bh * p.max_splits * 2;
        float Mx = -INFINITY;
        for (int j = 0; j < nsplit; ++j)
            if (__ldcg(ml + 2 * j + 1) > 0.f) Mx = fmaxf(Mx, __ldcg(ml + 2 * j));
        float acc[C::E];
#pragma unroll
        for (int e = 0; e < C::E; ++e) acc[e] = 0.f;
        float W = 0.f;
        const float* ob = p.part_o + bh * p.max_splits * C::DV + d0;
        for (int j = 0; j < nsplit; ++j) {
            const float lj = __ldcg(ml + 2 * j + 1);
            if (!(lj > 0.f)) continue;
            const float wj = lj * fast_exp2(__ldcg(ml + 2 * j) - Mx);
            W += wj;
            const float* oj = ob + static_cast<size_t>(j) * C::DV;
#pragma unroll
            for (int e = 0; e < C::E; e += 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(oj + e));
                acc[e] += wj * v.x;
                acc[e + 1] += wj * v.y;
                acc[e + 2] += wj * v.z;
                acc[e + 3] += wj * v.w;
            }
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(p.out + bh * C::DV + d0);
#pragma unroll
        for (int e = 0; e < C::E; e += 8)
            dst[e / 8] = make_uint4(pack_bf16x2(acc[e] * inv, acc[e + 1] * inv),
                                    pack_bf16x2(acc[e + 2] * inv, acc[e + 3] * inv),
                                    pack_bf16x2(acc[e + 4] * inv, acc[e + 5] * inv),
                                    pack_bf16x2(acc[e + 6] * inv, acc[e + 7] * inv));
        if (p.lse != nullptr && d0 == 0) p.lse[bh] = lse_from(Mx, W);
    }
    if (t == 0) *ticket = 0;
}

namespace {

template <int BS, bool PROD>
struct MlaVariant {
    static constexpr int SUB = PROD ? (BS < 32 ? BS : 32) : 16;
    static constexpr int NSTAGE = PROD ? (SUB == 16 ? 4 : 2) : 3;
    using C = MlaCfg<BS, SUB, NSTAGE, PROD>;
    static cudaError_t prepare()
    {
        return cudaFuncSetAttribute(paged_mla_decode_main<BS, SUB, NSTAGE, PROD>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    }
    static cudaError_t launch(dim3 grid, const CUtensorMap& tm, const MlaParams& p, cudaStream_t s)
    {
        return launch_dependent(paged_mla_decode_main<BS, SUB, NSTAGE, PROD>, grid,
                                dim3(C::THREADS), C::SMEM, s, tm, p);
    }
};

template <int BS>
cudaError_t prepare_both()
{
    cudaError_t e = MlaVariant<BS, false>::prepare();
    return e != cudaSuccess ? e : MlaVariant<BS, true>::prepare();
}

}  // namespace

int mla_stage_tokens(int block_size, bool prod)
{
    switch (block_size) {
    case 16: return prod ? MlaVariant<16, true>::SUB : MlaVariant<16, false>::SUB;
    case 32: return prod ? MlaVariant<32, true>::SUB : MlaVariant<32, false>::SUB;
    case 64: return prod ? MlaVariant<64, true>::SUB : MlaVariant<64, false>::SUB;
    default: return 0;
    }
}

cudaError_t prepare_mla_decode(int block_size)
{
    switch (block_size) {
    case 16: return prepare_both<16>();
    case 32: return prepare_both<32>();
    case 64: return prepare_both<64>();
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mla_decode(int block_size, bool prod, dim3 grid, const CUtensorMap& tm,
                              const MlaParams& p, cudaStream_t s)
{
    switch (block_size) {
    case 16: return prod ? MlaVariant<16, true>::launch(grid, tm, p, s)
                         : MlaVariant<16, false>::launch(grid, tm, p, s);
    case 32: return prod ? MlaVariant<32, true>::launch(grid, tm, p, s)
                         : MlaVariant<32, false>::launch(grid, tm, p, s);
    case 64: return prod ? MlaVariant<64, true>::launch(grid, tm, p, s)
                         : MlaVariant<64, false>::launch(grid, tm, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvp
