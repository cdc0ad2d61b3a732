// decode_kernel.cuh -- paged decode attention: one CTA per (sequence, kv
// head, query-head tile, split-KV chunk).
//
// Chunk j of a sequence covers its blocks [j S, (j+1) S).  The grid is
// chunk-major (blockIdx.z = chunk), so every sequence's first chunks start
// before any remainder chunk and the shortest work is scheduled last.  A
// sequence with one chunk is finished by its CTA; otherwise each chunk CTA
// leaves an fp32 partial (normalised output, max, sum) and counts itself on
// the unit's ticket, and the CTA that completes the count merges the chunks by
// log-sum-exp (learn.mohebi.ai lesson 12, section 6: split-KV decoding) and
// resets the ticket -- no second kernel.  With merge_kernel set the chunk CTAs
// only leave their partials and paged_decode_merge (merge.cu) combines them.
//
//   * One producer warp streams K and V blocks with 5-D TMA tensor loads
//     (cp.async.bulk.tensor, 128-byte swizzle) into a ring of NSTAGE shared-
//     memory stages, one cache block per stage, tracked by mbarriers; the
//     block-table row is fetched 32 entries at a time with one coalesced load.
//   * Four consumer warps take the stages round-robin (stage i -> warp i % 4,
//     so each warp owns NSTAGE / 4 stages and waits on them in order), each
//     with its own online-softmax state (decode_common.cuh); the four states
//     are merged in shared memory at the end.
//   * The step form (STEP, paged_decode_step with 8-row tiles) also appends: the
//     producer writes the step's new K/V rows of its kv head into the chunk's
//     blocks (append_row.cuh) once the ring is full or before the first block
//     holding one is loaded, and orders the writes before its TMA loads.
//   * Every wait is bounded (WAIT_LIMIT_NS); a late barrier sets
//     KV_DEVERR_TIMEOUT and the CTA drains its copies and returns.
#pragma once

#include "append_row.cuh"
#include "decode_common.cuh"

namespace kvp {

template <bool FP8, int D, int BS, int NT>
struct GridCfg : DecodeCfg<FP8, D, BS, NT> {
    using C = DecodeCfg<FP8, D, BS, NT>;
    static constexpr int SMEM = 1024 + C::NSTAGE * C::STAGE + C::NSTAGE * (8 + 8 + 4) + 16;
    static constexpr int MINB = 3;                  // CTAs per SM (row tiles of 8 and 16)
    static_assert(C::RED_BYTES <= C::NSTAGE * C::STAGE, "epilogue buffer reuses the stages");
};

// STEP: paged_decode_step's form, which writes the step's new rows of each block into the
// pool before loading it (a separate instantiation, so that the attention-only kernel keeps
// its registers).
template <bool FP8, int D, int BS, int NT, bool STEP>
__global__ void __launch_bounds__(DecodeCfg<FP8, D, BS, NT>::THREADS, GridCfg<FP8, D, BS, NT>::MINB)
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
    int* merge_flag = stage_blk + C::NSTAGE;

    const int b = blockIdx.y;
    const int kvh = blockIdx.x / p.head_groups;
    const int hg = blockIdx.x - kvh * p.head_groups;
    const int split = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int blk0 = split * p.split_blocks;
    const int nh = min(NT, p.rows - hg * NT);          // real rows in this tile
    // global query row of local row 0 (rows = heads of the group x query tokens)
    const size_t row0 = (static_cast<size_t>(b) * p.kv_heads + kvh) * p.rows + hg * NT;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NSTAGE; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), 1);
        }
        fence_mbar_init();
    }
    grid_dependency_wait();                          // inputs of the preceding kernel are ready

    // Independent loads in flight together: the context length, the chunk's
    // first 32 table entries (producer) and the query fragments (consumers).
    const int32_t* trow = p.tables + static_cast<size_t>(b) * p.max_blocks + blk0;
    int id_first = -1;
    if (warp == C::NCW && blk0 + lane < p.max_blocks) id_first = __ldg(trow + lane);
    uint32_t qf[C::KS][C::NTT][2];
    float sl2 = 0.f;
    int dt[C::NTT][2];
    if (warp < C::NCW) {
        sl2 = load_q_frags<FP8, D, BS, NT>(qf, p.q + row0 * D, nh, lane, p.scale_log2, p.k_scale,
                                           kvh);
        row_offsets<C::NTT>(dt, hg * NT, p.q_len, lane);
    }
    int ctx = __ldg(p.ctx + b);
    const int cap = p.max_blocks * BS;

    if (ctx < 0 || ctx > cap || (ctx > 0 && ctx < p.q_len)) {
        // out of range (clamped), or fewer cached tokens than new queries (kept:
        // the queries at negative positions attend to nothing)
        if (threadIdx.x == 0 && split == 0 && blockIdx.x == 0) atomicOr(p.err, KV_DEVERR_CONTEXT);
        ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    }
    const int nblk = (ctx + BS - 1) / BS;
    const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
    const int nb = max(0, min(nblk - blk0, p.split_blocks));
    __syncthreads();                                 // barriers initialised
    if (split >= nsplit) {                           // this sequence has fewer chunks
        grid_dependents_launch();
        return;
    }

    // ------------------------------------------------------------ producer warp
    if (warp == C::NCW) {
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
        for (int base = 0; base < nb && ok; base += 32) {
            const int j = base + lane;
            int id = -1;
            if (j < nb) {
                id = base == 0 ? id_first : __ldg(trow + j);
                if (id < 0 || id >= p.num_blocks) {
                    atomicOr(p.err, KV_DEVERR_BLOCK_ID);
                    id = -1;                          // skipped: never addressed
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
                if (STEP && !wrote && (blk0 + it >= new_blk || it == C::NSTAGE)) {
                    // the step's new rows go into their blocks once the ring is full (the
                    // producer would wait for a slot anyway), or before the first block that
                    // holds one is loaded, whichever comes first
                    write_step_rows<FP8, D, BS, 1>(p, b, ctx_raw, max(blk0, new_blk), blk0 + nb, kvh, lane);
                    fence_proxy_async_all();
                    __syncwarp();
                    wrote = true;
                }
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
        grid_dependents_launch();                    // every load of this CTA is issued
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
    WarpState<C> st;
    reset_state(st);
    const unsigned long long wait_ns = p.consumer_wait_ns ? p.consumer_wait_ns : WAIT_LIMIT_NS;
    for (int it = warp; it < nb; it += C::NCW) {
        const int s = it % C::NSTAGE;
        const uint32_t ph = static_cast<uint32_t>(it / C::NSTAGE) & 1u;
        const bool arrived = mbar_wait_bounded(smem_u32(full + s), ph, wait_ns);
        if (!__all_sync(FULL_MASK, arrived)) {
            if (lane == 0) atomicOr(p.err, KV_DEVERR_TIMEOUT);
            break;
        }
        const int blk = stage_blk[s];
        if (blk >= 0) {
            const uint32_t tk = smem_u32(smem + s * C::STAGE);
            process_block<FP8, D, BS, NT>(tk, tk + C::TILE, ctx - (blk0 + it) * BS, dt, qf, sl2,
                                          st, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(empty + s));
    }

    // ------------------------------------------------------------ epilogue
    grid_dependents_launch();
    reduce_row_sums(st);
    named_barrier_sync(1, C::NCW * 32);     // every consumer is done with the stages
    float* red = reinterpret_cast<float*>(smem);
    stash_state<FP8>(red, st, warp, lane);
    named_barrier_sync(1, C::NCW * 32);

    const int t = threadIdx.x;
    const int head = (t * C::E) / D;
    const int d0 = (t * C::E) % D;
    const size_t bh = row0 + head;                   // global query row
    if (head < nh) {
        float acc[C::E], M, L;
        combine_warps<C>(red, head, d0, FP8 ? __ldg(p.v_scale + kvh) : 1.f, acc, M, L);
        if (nsplit == 1) {
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + bh * D + d0);
#pragma unroll
            for (int e = 0; e < C::E; e += 2) dst[e / 2] = pack_bf16x2(acc[e], acc[e + 1]);
            if (p.lse != nullptr && d0 == 0) p.lse[bh] = lse_from(M, L);
        } else {
            float* dst = p.part_o + (bh * p.max_splits + split) * D + d0;
#pragma unroll
            for (int e = 0; e < C::E; ++e) dst[e] = acc[e];
            if (d0 == 0) {
                p.part_ml[(bh * p.max_splits + split) * 2 + 0] = M;
                p.part_ml[(bh * p.max_splits + split) * 2 + 1] = L;
            }
            __threadfence();                        // partial visible before the ticket
        }
    }
    if (nsplit == 1 || p.merge_kernel) return;      // done, or merged by paged_decode_merge

    // ---- ticket: the last chunk of this unit to finish merges all chunks
    named_barrier_sync(1, C::NCW * 32);
    int* ticket = p.tickets + (static_cast<size_t>(b) * p.kv_heads + kvh) * p.head_groups + hg;
    if (t == 0) {
        const int last = atomicAdd(ticket, 1) == nsplit - 1;
        if (last) __threadfence();
        *merge_flag = last;
    }
    named_barrier_sync(1, C::NCW * 32);
    if (!*merge_flag) return;
    if (head < nh) {
        const float* ml = p.part_ml + bh * p.max_splits * 2;
        float M = -INFINITY;
        for (int j = 0; j < nsplit; ++j) {
            if (__ldcg(ml + 2 * j + 1) > 0.f) M = fmaxf(M, __ldcg(ml + 2 * j));
        }
        float acc[C::E];
#pragma unroll
        for (int e = 0; e < C::E; ++e) acc[e] = 0.f;
        float W = 0.f;
        const float* ob = p.part_o + bh * p.max_splits * D + d0;
        for (int j = 0; j < nsplit; ++j) {
            const float lj = __ldcg(ml + 2 * j + 1);
            if (!(lj > 0.f)) continue;               // empty chunk: m = -inf, l = 0
            const float wj = lj * fast_exp2(__ldcg(ml + 2 * j) - M);
            W += wj;
            const float* oj = ob + static_cast<size_t>(j) * D;
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
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + bh * D + d0);
#pragma unroll
        for (int e = 0; e < C::E; e += 2) dst[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
        if (p.lse != nullptr && d0 == 0) p.lse[bh] = lse_from(M, W);
    }
    if (t == 0) *ticket = 0;                        // ready for the next call
}

// The step form is built for 8-row tiles only: with 16-row tiles the consumers' state
// leaves no registers for it (measured: 134 us for the 4-token verify step against 125 us
// for its attention), so paged_decode_step runs the append kernel first there.
template <int NT>
constexpr bool step_form_built() { return NT == 8; }

template <bool FP8, int D, int BS, int NT>
cudaError_t prepare_variant()
{
    cudaError_t e = cudaFuncSetAttribute(paged_decode_main<FP8, D, BS, NT, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         GridCfg<FP8, D, BS, NT>::SMEM);
    if constexpr (step_form_built<NT>()) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(paged_decode_main<FP8, D, BS, NT, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     GridCfg<FP8, D, BS, NT>::SMEM);
    }
    return e;
}

template <bool FP8, int D, int BS, int NT>
cudaError_t launch_variant(dim3 grid, const CUtensorMap& tk, const CUtensorMap& tv,
                           const DecodeParams& p, cudaStream_t s)
{
    if (p.k_new != nullptr) {
        if constexpr (step_form_built<NT>())
            return launch_dependent(paged_decode_main<FP8, D, BS, NT, true>, grid,
                                    dim3(DecodeCfg<FP8, D, BS, NT>::THREADS),
                                    GridCfg<FP8, D, BS, NT>::SMEM, s, tk, tv, p);
        return cudaErrorInvalidValue;
    }
    return launch_dependent(paged_decode_main<FP8, D, BS, NT, false>, grid,
                            dim3(DecodeCfg<FP8, D, BS, NT>::THREADS),
                            GridCfg<FP8, D, BS, NT>::SMEM, s, tk, tv, p);
}

}  // namespace kvp
