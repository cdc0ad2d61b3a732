// decode_heads.cuh -- paged decode attention with one CTA per (sequence, group of HC
// kv heads, query-row tile, split-KV chunk).
//
// The same operation as paged_decode_main (decode_kernel.cuh), with the CTA laid out
// after the pool: a cache block holds every kv head of its tokens
// ([num_blocks, block_size, kv_heads, head_dim], xuewyang.github.io/posts/kv,
// "Reading the code: a warehouse of lockers"), so one stage of the ring holds one
// block of HC kv heads -- K tiles of the HC heads, then their V tiles -- and the
// CTA's start (context length, table entries, queries, first loads) and its
// epilogue are paid once for HC heads instead of once per head.
//
//   * One producer warp: per stage, lane 0 waits for the slot and arms its
//     barrier, then lanes 0 .. 2 HC - 1 issue one 5-D TMA box load each (one
//     block of one kv head, K or V, 128-byte swizzle) -- the HC heads of a block
//     are adjacent in HBM, so the loads of a stage read one contiguous span.
//   * HC consumer warps: warp h owns kv head h of the group and folds every stage
//     of the chunk into its online-softmax state (the per-block work of
//     decode_common.cuh), so it holds the whole chunk's state for its rows and no
//     warp states are merged; a stage is free once the HC warps have read it.
//   * Each warp writes its rows: bf16 output and LSE for a sequence of one chunk,
//     else an fp32 partial; the CTA then takes a ticket and the last chunk CTA of
//     the (sequence, head group, row tile) merges every chunk by log-sum-exp
//     (learn.mohebi.ai lesson 12, section 6: split-KV decoding), unless the
//     separate merge kernel is asked for.
//   * The step form (STEP, paged_decode_step) also appends: the producer writes the
//     step's new K/V rows of the group's kv heads into the chunk's blocks
//     (append_row.cuh) once the ring is full or before the first block holding
//     one is loaded, and orders the writes before its TMA loads.
//   * Every wait is bounded (WAIT_LIMIT_NS); a late barrier sets
//     KV_DEVERR_TIMEOUT and the CTA drains its copies and returns.
#pragma once

#include "append_row.cuh"
#include "decode_common.cuh"

namespace kvp {

template <bool FP8, int D, int BS, int NT, int HC, int CTAS>
struct HeadsCfg {
    using C = DecodeCfg<FP8, D, BS, NT>;
    static constexpr int HSTAGE = 2 * HC * C::TILE;          // K tiles of HC heads, then V tiles
    // About 192 KB of stages in flight per SM, shared by its CTAS CTAs.
    static constexpr int RING = (192 / CTAS) * 1024;
    static constexpr int NST = RING / HSTAGE >= 2 ? RING / HSTAGE : 2;
    static constexpr int NCW = HC;                           // consumer warps, one per kv head
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int SMEM = 1024 + NST * HSTAGE + NST * (8 + 8 + 4) + 16;
    static constexpr int E = NT * D / 32;                    // merge: numbers per consumer thread
    static_assert(E % 4 == 0 && D % E == 0, "merge split (float4 partial reads)");
    static_assert(2 * HC <= 32, "one producer lane per TMA load of a stage");
    static_assert((SMEM + 1024) * CTAS <= 228 * 1024, "CTAs per SM");
};

// Writes one warp's rows from its (reduced) online-softmax state: bf16 output and LSE
// when the chunk is the whole sequence, else the chunk's fp32 partial (normalised
// output, max, sum).  Thread (r, c) holds rows nt*8 + 2c + j at the numbers d(ms, hi).
template <bool FP8, class C>
__device__ __forceinline__ void write_warp_rows(const WarpState<C>& st, const DecodeParams& p,
                                                size_t row0, int nh, int split, bool whole,
                                                float out_scale, int lane)
{
    constexpr int D = C::KS * 16;
    const int r = lane >> 2;
    const int c = lane & 3;
#pragma unroll
    for (int nt = 0; nt < C::NTT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int hl = nt * 8 + 2 * c + j;
            if (hl >= nh) continue;
            const size_t bh = row0 + hl;
            const float L = st.l[nt][j];
            const float inv = (L > 0.f ? 1.f / L : 0.f) * out_scale;
            if (whole) {
                uint16_t* dst = p.out + bh * D;
#pragma unroll
                for (int ms = 0; ms < C::KS; ++ms)
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        const int d = FP8 ? (16 * r + 2 * ms + hi) : (16 * ms + r + 8 * hi);
                        dst[d] = static_cast<uint16_t>(pack_bf16x2(st.o[ms][nt][2 * hi + j] * inv, 0.f));
                    }
                if (p.lse != nullptr && r == 0) p.lse[bh] = lse_from(st.m[nt][j], L);
            } else {
                float* dst = p.part_o + (bh * p.max_splits + split) * D;
#pragma unroll
                for (int ms = 0; ms < C::KS; ++ms)
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        const int d = FP8 ? (16 * r + 2 * ms + hi) : (16 * ms + r + 8 * hi);
                        dst[d] = st.o[ms][nt][2 * hi + j] * inv;
                    }
                if (r == 0) {
                    p.part_ml[(bh * p.max_splits + split) * 2 + 0] = st.m[nt][j];
                    p.part_ml[(bh * p.max_splits + split) * 2 + 1] = L;
                }
            }
        }
}

// STEP: paged_decode_step's form (writes the step's new rows before loading their blocks).
template <bool FP8, int D, int BS, int NT, int HC, int CTAS, bool STEP>
__global__ void __launch_bounds__(HeadsCfg<FP8, D, BS, NT, HC, CTAS>::THREADS, CTAS)
paged_decode_heads(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const DecodeParams p)
{
    using H = HeadsCfg<FP8, D, BS, NT, HC, CTAS>;
    using C = DecodeCfg<FP8, D, BS, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + H::NST * H::HSTAGE);
    uint64_t* empty = full + H::NST;
    int* stage_blk = reinterpret_cast<int*>(empty + H::NST);
    int* merge_flag = stage_blk + H::NST;

    const int b = blockIdx.y;
    const int kg = blockIdx.x / p.head_groups;               // group of HC kv heads
    const int hg = blockIdx.x - kg * p.head_groups;          // query-row tile
    const int split = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int blk0 = split * p.split_blocks;
    const int nh = min(NT, p.rows - hg * NT);                // real rows in this tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < H::NST; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), HC);
        }
        fence_mbar_init();
    }
    grid_dependency_wait();                                  // inputs of the preceding kernel

    const int32_t* trow = p.tables + static_cast<size_t>(b) * p.max_blocks + blk0;
    int id_first = -1;
    if (warp == H::NCW && blk0 + lane < p.max_blocks) id_first = __ldg(trow + lane);
    // the consumer warp's kv head
    const int h = warp;
    const int kvh = kg * HC + h;
    const size_t row0 = (static_cast<size_t>(b) * p.kv_heads + kvh) * p.rows + hg * NT;
    uint32_t qf[C::KS][C::NTT][2];
    float sl2 = 0.f;
    int dt[C::NTT][2];
    if (warp < H::NCW) {
        sl2 = load_q_frags<FP8, D, BS, NT>(qf, p.q + row0 * D, nh, lane, p.scale_log2, p.k_scale, kvh);
        row_offsets<C::NTT>(dt, hg * NT, p.q_len, lane);
    }
    int ctx = __ldg(p.ctx + b);
    const int cap = p.max_blocks * BS;

    if (ctx < 0 || ctx > cap || (ctx > 0 && ctx < p.q_len)) {
        if (threadIdx.x == 0 && split == 0 && blockIdx.x == 0) atomicOr(p.err, KV_DEVERR_CONTEXT);
        ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    }
    const int nblk = (ctx + BS - 1) / BS;
    const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    const int nb = max(0, min(nblk - blk0, p.split_blocks));
    __syncthreads();                                         // barriers initialised
    if (split >= nsplit) {
        grid_dependents_launch();
        return;
    }

    // ------------------------------------------------------------ producer warp
    if (warp == H::NCW) {
        if (lane == 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
        }
        int issued = 0;
        bool ok = true;
        // paged_decode_step: the length as given (re-read here rather than kept live across
        // the roles: the consumers' registers are the kernel's peak)
        const int ctx_raw = STEP ? __ldg(p.ctx + b) : 0;
        if (STEP && lane == 0 && split == 0 && blockIdx.x == 0) {
            // paged_decode_step: a new token whose position is not in the table is not written
            for (int t = 0; t < p.q_len; ++t) {
                const int pos = ctx_raw - p.q_len + t;
                if (pos < 0 || pos / BS >= p.max_blocks) atomicOr(p.err, KV_DEVERR_POSITION);
            }
        }
        // paged_decode_step: the first block that holds one of the step's new tokens
        const int new_blk = STEP ? max(0, ctx_raw - p.q_len) / BS : p.max_blocks;
        bool wrote = blk0 + nb <= new_blk;                    // nothing of the step in this chunk
        // lane i < 2 HC loads the K (i < HC) or V tile of kv head kg * HC + i % HC
        const int my_h = lane % HC;
        const CUtensorMap* my_map = lane < HC ? &tmk : &tmv;
        const uint32_t my_off = static_cast<uint32_t>((lane < HC ? 0 : HC * C::TILE) + my_h * C::TILE);
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
            for (int k = 0; k < cnt; ++k) {
                const int blk = __shfl_sync(FULL_MASK, id, k);
                const int it = base + k;
                if (it == p.stop_stage) {                // test hook: the rest never lands
                    ok = false;
                    break;
                }
                if (STEP && !wrote && (blk0 + it >= new_blk || it == H::NST)) {
                    // the step's new rows go into their blocks once the ring is full (the
                    // producer would wait for a slot anyway), or before the first block that
                    // holds one is loaded, whichever comes first
                    write_step_rows<FP8, D, BS, HC>(p, b, ctx_raw, max(blk0, new_blk), blk0 + nb, kg * HC, lane);
                    fence_proxy_async_all();
                    __syncwarp();
                    wrote = true;
                }
                const int st = it % H::NST;
                const uint32_t ph = static_cast<uint32_t>(it / H::NST) & 1u;
                int good = 1;
                if (lane == 0) {
                    if (!mbar_wait_bounded(smem_u32(empty + st), ph ^ 1u)) {
                        atomicOr(p.err, KV_DEVERR_TIMEOUT);
                        good = 0;
                    } else {
                        stage_blk[st] = blk;
                        if (blk >= 0)
                            mbar_arrive_expect_tx(smem_u32(full + st), H::HSTAGE);
                        else
                            mbar_arrive(smem_u32(full + st));
                    }
                }
                good = __shfl_sync(FULL_MASK, good, 0);
                if (!good) {
                    ok = false;
                    break;
                }
                // the barrier is armed before any of the stage's bytes can land
                if (blk >= 0 && lane < 2 * HC)
                    tma_load_5d(smem_u32(smem + st * H::HSTAGE) + my_off, my_map, 0, 0,
                                kg * HC + my_h, 0, blk, smem_u32(full + st));
                issued = it + 1;
            }
        }
        grid_dependents_launch();
        if (lane == 0) {
            for (int it = max(0, issued - H::NST); it < issued; ++it) {
                if (!mbar_wait_bounded(smem_u32(full + (it % H::NST)),
                                       static_cast<uint32_t>(it / H::NST) & 1u)) {
                    atomicOr(p.err, KV_DEVERR_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumer warps
    WarpState<C> st;
    reset_state(st);
    const unsigned long long wait_ns = p.consumer_wait_ns ? p.consumer_wait_ns : WAIT_LIMIT_NS;
    for (int it = 0; it < nb; ++it) {
        const int s = it % H::NST;
        const uint32_t ph = static_cast<uint32_t>(it / H::NST) & 1u;
        const bool arrived = mbar_wait_bounded(smem_u32(full + s), ph, wait_ns);
        if (!__all_sync(FULL_MASK, arrived)) {
            if (lane == 0) atomicOr(p.err, KV_DEVERR_TIMEOUT);
            break;
        }
        const int blk = stage_blk[s];
        if (blk >= 0) {
            const uint32_t tk = smem_u32(smem + s * H::HSTAGE) + h * C::TILE;
            process_block<FP8, D, BS, NT>(tk, tk + HC * C::TILE, ctx - (blk0 + it) * BS, dt, qf, sl2,
                                          st, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
    }
    grid_dependents_launch();
    reduce_row_sums(st);

    const bool whole = nsplit == 1;
    write_warp_rows<FP8, C>(st, p, row0, nh, split, whole, FP8 ? __ldg(p.v_scale + kvh) : 1.f, lane);
    if (whole || p.merge_kernel) return;
    __threadfence();                                         // partials visible before the ticket

    // ---- ticket: the last chunk of this (sequence, head group, row tile) merges all chunks
    named_barrier_sync(1, H::NCW * 32);
    const int t = threadIdx.x;
    int* ticket = p.tickets + (static_cast<size_t>(b) * p.kv_heads + kg) * p.head_groups + hg;
    if (t == 0) {
        const int last = atomicAdd(ticket, 1) == nsplit - 1;
        if (last) __threadfence();
        *merge_flag = last;
    }
    named_barrier_sync(1, H::NCW * 32);
    if (!*merge_flag) return;
    // thread t merges numbers d0 .. d0 + E - 1 of local row lr of head mh
    constexpr int E = H::E;
    const int flat = t * E;                                  // over HC x NT rows of D numbers
    const int mh = flat / (NT * D);
    const int lr = (flat / D) % NT;
    const int d0 = flat % D;
    if (lr < nh) {
        const size_t bh = (static_cast<size_t>(b) * p.kv_heads + kg * HC + mh) * p.rows + hg * NT + lr;
        const float* ml = p.part_ml + bh * p.max_splits * 2;
        float M = -INFINITY;
        for (int j = 0; j < nsplit; ++j) {
            if (__ldcg(ml + 2 * j + 1) > 0.f) M = fmaxf(M, __ldcg(ml + 2 * j));
        }
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        float Wt = 0.f;
        const float* ob = p.part_o + bh * p.max_splits * D + d0;
        for (int j = 0; j < nsplit; ++j) {
            const float lj = __ldcg(ml + 2 * j + 1);
            if (!(lj > 0.f)) continue;
            const float wj = lj * fast_exp2(__ldcg(ml + 2 * j) - M);
            Wt += wj;
            const float* oj = ob + static_cast<size_t>(j) * D;
#pragma unroll
            for (int e = 0; e < E; e += 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(oj + e));
                acc[e] += wj * v.x;
                acc[e + 1] += wj * v.y;
                acc[e + 2] += wj * v.z;
                acc[e + 3] += wj * v.w;
            }
        }
        const float inv = Wt > 0.f ? 1.f / Wt : 0.f;
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + bh * D + d0);
#pragma unroll
        for (int e = 0; e < E; e += 2) dst[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
        if (p.lse != nullptr && d0 == 0) p.lse[bh] = lse_from(M, Wt);
    }
    if (t == 0) *ticket = 0;
}

template <bool FP8, int D, int BS, int NT, int HC, int CTAS>
cudaError_t prepare_heads_variant()
{
    cudaError_t e = cudaFuncSetAttribute(paged_decode_heads<FP8, D, BS, NT, HC, CTAS, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         HeadsCfg<FP8, D, BS, NT, HC, CTAS>::SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(paged_decode_heads<FP8, D, BS, NT, HC, CTAS, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                HeadsCfg<FP8, D, BS, NT, HC, CTAS>::SMEM);
}

template <bool FP8, int D, int BS, int NT, int HC, int CTAS>
cudaError_t launch_heads_variant(dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeParams& p, cudaStream_t s)
{
    if (p.k_new != nullptr)
        return launch_dependent(paged_decode_heads<FP8, D, BS, NT, HC, CTAS, true>, grid,
                                dim3(HeadsCfg<FP8, D, BS, NT, HC, CTAS>::THREADS),
                                HeadsCfg<FP8, D, BS, NT, HC, CTAS>::SMEM, s, tk, tv, p);
    return launch_dependent(paged_decode_heads<FP8, D, BS, NT, HC, CTAS, false>, grid,
                            dim3(HeadsCfg<FP8, D, BS, NT, HC, CTAS>::THREADS),
                            HeadsCfg<FP8, D, BS, NT, HC, CTAS>::SMEM, s, tk, tv, p);
}

}  // namespace kvp
