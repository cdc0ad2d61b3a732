// decode_mla_tc.cu -- absorbed multi-head latent attention on the 5th-generation
// tensor cores (tcgen05), for wide head tiles: all 128 query heads of a sequence
// on the MMA's M dimension (xuewyang.github.io/posts/kv, "MLA: how does decode
// get full-size keys and values back?": every head scores the shared cached
// vector -- 512 latent + 64 rotary-key numbers -- and averages its latent part).
//
// Persistent: one CTA per SM holds its tensor memory for the whole launch and
// works through items (sequence, tile of 128 heads, quarter of the latent output,
// split chunk) taken from a counter in the workspace, first chunks first; the
// last CTA to finish resets the counter.  320 threads:
//   * warp 8 takes the next item, skips empty ones (chunks past a sequence's
//     end), passes the item to the other roles through a 4-slot ring in shared
//     memory, and streams the item's 64-token blocks, one per stage, with nine
//     TMA loads (one per 128-byte piece of the 576 numbers, 128-byte swizzle),
//     so a stage is nine [64 tokens x 64 numbers] K-major tiles: 72 KB, 3 stages.
//     The loads of the next item start while the current one is computed.
//   * warp 9 (one thread) issues the MMAs.  Scores S[128 heads x 64 tokens] =
//     Q . C^T: A = the absorbed queries, kept in tensor memory for the item
//     (128 lanes x 288 columns), B = the stage (K-major), 36 MMAs of K = 16.
//     Then O[128 heads x 128 latent] += P . C[:, quarter]: A = the probabilities
//     in tensor memory, B = the same stage read MN-major (the latent numbers of a
//     token are contiguous), 4 MMAs.  Completion is signalled by tcgen05.commit on
//     mbarriers.  The scores of stage i+1 are computed while the softmax of stage
//     i runs, and the output update of stage i while the softmax of stage i+1 runs.
//   * warps 0-7: head h (tensor-memory lane h) belongs to two threads, one in
//     warp h / 32 (tokens 0-31 of a stage, output columns 0-63) and one in warp
//     h / 32 + 4 (tokens 32-63, columns 64-127) -- a warp can only reach its own
//     quarter of the lanes, and two warps per quarter halve the serial work of
//     each.  Each reads its 32 scores, the pair exchanges its maxima through
//     shared memory, and each writes its 32 probabilities (bf16) back to tensor
//     memory; at the end of an item each normalises and stores its 64 outputs,
//     then loads the next item's queries.  The output is rescaled only when the
//     running max grows by more than 2^8 (log2 units); until then the older
//     maximum stays the reference, which is exact because the final division
//     uses the sum taken against the same reference.
//   * the four quarter-items of a sequence chunk compute the same scores (the
//     tensor memory of an SM holds the fp32 output of 128 heads x 128 latent
//     numbers beside the queries and one score tile, not more) and read the same
//     stages, which the L2 serves after the first.
//   * tensor memory: queries [0, 288), scores [288, 352), probabilities
//     [352, 384), output [384, 512).
// Every wait is bounded; a late barrier sets KV_DEVERR_TIMEOUT and every role
// leaves its loop, waits (bounded) for its copies and MMAs in flight, and the CTA
// frees its tensor memory before it exits.
#include "decode_common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace kvp {

namespace {

constexpr int TC_TOK = 64;                      // tokens per stage (one block)
constexpr int TC_NSTAGE = 3;
constexpr int TC_PIECE = TC_TOK * 128;          // one 64-number piece of 64 tokens
constexpr int TC_NPIECE = MLA_DK / 64;          // 9
constexpr int TC_STAGE = TC_NPIECE * TC_PIECE;  // 73,728 bytes
constexpr int TC_DQ = 128;                      // latent numbers per CTA
constexpr int TC_M = 128;                       // heads per CTA
constexpr int TC_THREADS = 320;                 // warps 0-7 softmax, 8 loads, 9 MMA
constexpr uint32_t TM_Q = 0, TM_S = 288, TM_P = 352, TM_O = 384, TM_COLS = 512;
constexpr uint32_t IDESC_S = tc_idesc_bf16(TC_M, TC_TOK, 0, 0);
constexpr uint32_t IDESC_O = tc_idesc_bf16(TC_M, TC_DQ, 0, 1);
constexpr float RESCALE_LOG2 = 8.f;
constexpr int TC_CTL = 4096;
constexpr int TC_SMEM = 1024 + TC_NSTAGE * TC_STAGE + TC_CTL;
static_assert(TC_SMEM <= 227 * 1024, "one CTA per SM");
static_assert(TM_O + TC_DQ <= TM_COLS && TM_P + TC_TOK / 2 <= TM_O && TM_S + TC_TOK <= TM_P &&
                  TM_Q + MLA_DK / 2 <= TM_S,
              "tensor-memory columns");

constexpr int TC_NITEM = 4;                     // ring of work items in shared memory

// A work item as the producer hands it on: n = stages, at least 1 (-1: no more items).
struct TcItem {
    int b, ht, dq, split, n, ctx;
};

struct TcCtl {
    uint64_t kv_full[TC_NSTAGE];
    uint64_t kv_empty[TC_NSTAGE];
    uint64_t s_full, s_free, p_full, p_free, q_ready, mma_done;
    uint64_t item_full[TC_NITEM];
    uint64_t item_empty[TC_NITEM];
    uint32_t tmem_base;
    int stage_blk[TC_NSTAGE];
    int abort_flag;
    int merge_flag;
    TcItem items[TC_NITEM];
    float xmax[2][2][TC_M];                         // [stage parity][token half][head]
    float xl[2][TC_M];                              // [token half][head]
};
static_assert(sizeof(TcCtl) <= TC_CTL, "control block");

__device__ __forceinline__ bool all_ok(bool ok) { return __all_sync(FULL_MASK, ok); }

// Named barrier that also returns, to every participant, the OR of their `pred`.
__device__ __forceinline__ bool named_barrier_or(int id, int threads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// The scores of a stage: S = Q . C^T, 36 MMAs of K = 16.  The descriptor of slice
// ks is the stage's base descriptor plus a constant (16-byte units in the low
// word), so each issue is one add: a single thread issues every MMA of the CTA
// and its issue rate, not the tensor pipe, bounds small-N MMAs like these.
__device__ __forceinline__ void issue_score_mma(uint32_t tbase, uint32_t stage_addr)
{
    const uint64_t d0 = tc_smem_desc(stage_addr, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < MLA_DK / 16; ++ks)
        tc_mma_ts(tbase + TM_S + 0u, tbase + TM_Q + ks * 8,
                  d0 + static_cast<uint64_t>(((ks >> 2) * TC_PIECE + (ks & 3) * 32) >> 4), IDESC_S,
                  ks > 0);
}

// The output update of stage k: O += P . C[:, quarter] over its 64 tokens.
__device__ __forceinline__ void issue_output_mma(uint32_t tbase, uint32_t stage_addr, int dq, bool first)
{
    const uint64_t d0 = tc_smem_desc(stage_addr + 2 * dq * TC_PIECE, TC_PIECE, 1024);
#pragma unroll
    for (int kk = 0; kk < TC_TOK / 16; ++kk)
        tc_mma_ts(tbase + TM_O, tbase + TM_P + kk * 8, d0 + static_cast<uint64_t>((kk * 2048) >> 4),
                  IDESC_O, !(first && kk == 0));
}

}  // namespace

__global__ void __launch_bounds__(TC_THREADS, 1)
paged_mla_decode_tc(const __grid_constant__ CUtensorMap tmp, const MlaParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    TcCtl* ctl = reinterpret_cast<TcCtl*>(smem + TC_NSTAGE * TC_STAGE);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int* abort_flag = &ctl->abort_flag;

    if (tid == 0) {
        for (int i = 0; i < TC_NSTAGE; ++i) {
            mbar_init(smem_u32(&ctl->kv_full[i]), 1);
            mbar_init(smem_u32(&ctl->kv_empty[i]), 1);
        }
        for (int i = 0; i < TC_NITEM; ++i) {
            mbar_init(smem_u32(&ctl->item_full[i]), 1);
            mbar_init(smem_u32(&ctl->item_empty[i]), 9);   // the MMA thread + 8 softmax warps
        }
        mbar_init(smem_u32(&ctl->s_full), 1);
        mbar_init(smem_u32(&ctl->s_free), 8);
        mbar_init(smem_u32(&ctl->p_full), 8);
        mbar_init(smem_u32(&ctl->p_free), 1);
        mbar_init(smem_u32(&ctl->q_ready), 8);
        mbar_init(smem_u32(&ctl->mma_done), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) tc_alloc(smem_u32(&ctl->tmem_base), TM_COLS);
    grid_dependency_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ctl->tmem_base;

    if (warp == 8) {
        // ------------------------------------------------------------ items and loads
        if (lane == 0) {
            prefetch_tensormap(&tmp);
            const int per_chunk = p.batch * p.head_tiles * 4;
            const int total = per_chunk * p.max_splits;
            int k = 0;                              // items handed on
            int g = 0;                              // stages issued (all items)
            bool ok = true;
            for (;;) {
                const int item = atomicAdd(p.queue, 1);
                const bool last = item >= total || *abort_flag;
                TcItem it{};
                if (!last) {
                    it.split = item / per_chunk;
                    const int rem = item - it.split * per_chunk;
                    it.b = rem / (p.head_tiles * 4);
                    const int x = rem - it.b * (p.head_tiles * 4);
                    it.ht = x >> 2;
                    it.dq = x & 3;
                    int ctx = __ldg(p.ctx + it.b);
                    const int cap = p.max_blocks * TC_TOK;
                    if (ctx < 0 || ctx > cap) {
                        if (it.split == 0 && x == 0) atomicOr(p.err, KV_DEVERR_CONTEXT);
                        ctx = ctx < 0 ? 0 : cap;
                    }
                    it.ctx = ctx;
                    const int nblk = (ctx + TC_TOK - 1) / TC_TOK;
                    const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
                    if (it.split >= nsplit) continue;       // past the sequence's end: skip
                    it.n = max(0, min(nblk - it.split * p.split_blocks, p.split_blocks));
                    if (it.n == 0) {
                        // an empty sequence: its output quarter is 0 (and its LSE -inf),
                        // written here, so every item handed on has stages -- the softmax
                        // warps then never run more than one item ahead of the MMA thread
                        const int nh = min(TC_M, p.q_heads - it.ht * TC_M);
                        const size_t row0 = static_cast<size_t>(it.b) * p.q_heads + it.ht * TC_M;
                        for (int hh = 0; hh < nh; ++hh) {
                            uint4* dst = reinterpret_cast<uint4*>(p.out + (row0 + hh) * MLA_DV + it.dq * TC_DQ);
                            for (int v = 0; v < TC_DQ / 8; ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
                            if (p.lse != nullptr && it.dq == 0) p.lse[row0 + hh] = -INFINITY;
                        }
                        continue;
                    }
                } else {
                    it.n = -1;
                }
                const int slot = k % TC_NITEM;
                if (!mbar_wait_bounded(smem_u32(&ctl->item_empty[slot]),
                                       (static_cast<uint32_t>(k / TC_NITEM) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
                ctl->items[slot] = it;
                mbar_arrive(smem_u32(&ctl->item_full[slot]));
                ++k;
                if (last) break;
                const int32_t* trow = p.tables + static_cast<size_t>(it.b) * p.max_blocks +
                                      it.split * p.split_blocks;
                int next_blk = it.n > 0 ? __ldg(trow) : -1;   // block id read one stage ahead
                for (int s = 0; s < it.n; ++s, ++g) {
                    const int st = g % TC_NSTAGE;
                    int blk = next_blk;
                    if (s + 1 < it.n) next_blk = __ldg(trow + s + 1);
                    if (!mbar_wait_bounded(smem_u32(&ctl->kv_empty[st]),
                                           (static_cast<uint32_t>(g / TC_NSTAGE) & 1u) ^ 1u) ||
                        *abort_flag) {
                        ok = false;
                        break;
                    }
                    if (blk < 0 || blk >= p.num_blocks) {
                        atomicOr(p.err, KV_DEVERR_BLOCK_ID);
                        blk = -1;
                    }
                    ctl->stage_blk[st] = blk;
                    const uint32_t fb = smem_u32(&ctl->kv_full[st]);
                    if (blk >= 0) {
                        mbar_arrive_expect_tx(fb, TC_STAGE);
                        const uint32_t dst = smem_u32(smem + st * TC_STAGE);
                        for (int pc = 0; pc < TC_NPIECE; ++pc)
                            tma_load_5d(dst + pc * TC_PIECE, &tmp, 0, pc, 0, 0, blk, fb);
                    } else {
                        mbar_arrive(fb);
                    }
                }
                if (!ok) break;
            }
            if (!ok) {
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ctl->abort_flag = 1;
            }
            // copies still in flight must land before the CTA moves on
            for (int j = max(0, g - TC_NSTAGE); j < g; ++j)
                if (!mbar_wait_bounded(smem_u32(&ctl->kv_full[j % TC_NSTAGE]),
                                       static_cast<uint32_t>(j / TC_NSTAGE) & 1u))
                    break;
        }
        grid_dependents_launch();
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            bool ok = true;
            int g = 0;                              // stages processed (all items)
            for (int k = 0; ok; ++k) {
                const int slot = k % TC_NITEM;
                ok = mbar_wait_bounded(smem_u32(&ctl->item_full[slot]),
                                       static_cast<uint32_t>(k / TC_NITEM) & 1u);
                if (!ok) break;
                const int n = ctl->items[slot].n;
                const int dq = ctl->items[slot].dq;
                mbar_arrive(smem_u32(&ctl->item_empty[slot]));
                if (n < 0) break;
                ok = mbar_wait_bounded(smem_u32(&ctl->q_ready), static_cast<uint32_t>(k) & 1u);
                for (int s = 0; ok && s < n; ++s) {
                    const int gs = g + s;
                    const int st = gs % TC_NSTAGE;
                    ok = mbar_wait_bounded(smem_u32(&ctl->kv_full[st]),
                                           static_cast<uint32_t>(gs / TC_NSTAGE) & 1u);
                    if (ok && gs >= 1)
                        ok = mbar_wait_bounded(smem_u32(&ctl->s_free), static_cast<uint32_t>(gs - 1) & 1u);
                    if (!ok || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_score_mma(tbase, smem_u32(smem + st * TC_STAGE));
                    tc_commit(smem_u32(&ctl->s_full));
                    if (s >= 1) {
                        ok = mbar_wait_bounded(smem_u32(&ctl->p_full), static_cast<uint32_t>(gs - 1) & 1u);
                        if (!ok) break;
                        tc_fence_after();
                        issue_output_mma(tbase, smem_u32(smem + ((gs - 1) % TC_NSTAGE) * TC_STAGE), dq, s == 1);
                        tc_commit(smem_u32(&ctl->p_free));
                        tc_commit(smem_u32(&ctl->kv_empty[(gs - 1) % TC_NSTAGE]));
                    }
                }
                if (ok && n >= 1) {
                    // the item's last output update, before the next item's queries
                    const int gl = g + n - 1;
                    ok = mbar_wait_bounded(smem_u32(&ctl->p_full), static_cast<uint32_t>(gl) & 1u);
                    if (ok) {
                        tc_fence_after();
                        issue_output_mma(tbase, smem_u32(smem + (gl % TC_NSTAGE) * TC_STAGE), dq, n == 1);
                        tc_commit(smem_u32(&ctl->p_free));
                        tc_commit(smem_u32(&ctl->kv_empty[gl % TC_NSTAGE]));
                    }
                }
                g += n;
            }
            if (!ok) {
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ctl->abort_flag = 1;
            }
            // every MMA issued must be complete before the tensor memory is freed
            tc_commit(smem_u32(&ctl->mma_done));
            mbar_wait_bounded(smem_u32(&ctl->mma_done), 0);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        const int half = warp >> 2;                 // token half of a stage, output half
        const int h = (warp & 3) * 32 + lane;       // head of the tile = tensor-memory lane
        const int st_id = warp * 32 + lane;         // 0 .. 255 among the softmax threads
        const uint32_t lrow = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const float sl2 = p.scale_log2;
        bool failed = false;                        // this thread has seen a wait give up
        int g = 0;                                  // stages processed (all items)
        for (int k = 0; !failed; ++k) {
            const int slot = k % TC_NITEM;
            bool ok = all_ok(mbar_wait_bounded(smem_u32(&ctl->item_full[slot]),
                                               static_cast<uint32_t>(k / TC_NITEM) & 1u));
            const TcItem item = ctl->items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->item_empty[slot]));
            // leave together: on a failure, or when there are no more items
            if (named_barrier_or(2, 256, !ok || item.n < 0 || *abort_flag != 0)) {
                failed = !ok || *abort_flag != 0;
                break;
            }
            const int b = item.b, dq = item.dq, split = item.split, n = item.n, ctx = item.ctx;
            const int ht = item.ht;
            const int blk0 = split * p.split_blocks;
            const int nblk = (ctx + TC_TOK - 1) / TC_TOK;
            const int nsplit = nblk > 0 ? (nblk + p.split_blocks - 1) / p.split_blocks : 1;
            const int nh = min(TC_M, p.q_heads - ht * TC_M);
            const size_t row0 = static_cast<size_t>(b) * p.q_heads + ht * TC_M;
            {
                // queries -> tensor memory (the previous item's score MMAs are complete:
                // this thread waited for its last scores)
                const uint4* qg = reinterpret_cast<const uint4*>(p.q + (row0 + (h < nh ? h : 0)) * MLA_DK);
#pragma unroll 1
                for (int c9 = half * 5; c9 < (half ? TC_NPIECE : 5); ++c9) {
                    uint32_t r[32];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const uint4 x = h < nh ? __ldg(qg + c9 * 8 + v) : make_uint4(0u, 0u, 0u, 0u);
                        r[4 * v] = x.x;
                        r[4 * v + 1] = x.y;
                        r[4 * v + 2] = x.z;
                        r[4 * v + 3] = x.w;
                    }
                    tc_st32(lrow + TM_Q + c9 * 32, r);
                }
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->q_ready));
            }
            float m_ref = -INFINITY, l = 0.f;
            for (int s = 0; s < n; ++s) {
                const int gs = g + s;
                const int st = gs % TC_NSTAGE;
                ok = mbar_wait_bounded(smem_u32(&ctl->kv_full[st]), static_cast<uint32_t>(gs / TC_NSTAGE) & 1u);
                if (ok) ok = mbar_wait_bounded(smem_u32(&ctl->s_full), static_cast<uint32_t>(gs) & 1u);
                ok = all_ok(ok);
                if (!ok) failed = true;
                const int blk = ok ? ctl->stage_blk[st] : -1;
                const int nvalid_all = blk < 0 ? 0 : min(TC_TOK, ctx - (blk0 + s) * TC_TOK);
                const int nvalid = nvalid_all - half * 32;   // of this thread's 32 tokens
                float sv[32];
                if (ok) {
                    tc_fence_after();
                    uint32_t r[32];
                    tc_ld32(lrow + TM_S + half * 32, r);
                    tc_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(r[j]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free));
                }
                if (nvalid < 32) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j >= nvalid) sv[j] = -INFINITY;   // not cached (may be NaN)
                }
                float mx = sv[0];
#pragma unroll
                for (int j = 1; j < 32; ++j) mx = fmaxf(mx, sv[j]);
                ctl->xmax[gs & 1][half][h] = mx;
                // Every softmax thread reaches this barrier each stage and leaves the loop
                // here together, on any failure seen so far (its own or another role's).
                if (named_barrier_or(2, 256, failed || *abort_flag != 0)) {
                    failed = true;
                    break;
                }
                mx = fmaxf(mx, ctl->xmax[gs & 1][half ^ 1][h]);
                const float m_new = fmaxf(m_ref, mx * sl2);
                float f = 1.f;
                if (m_ref == -INFINITY) {
                    m_ref = m_new;                  // nothing accumulated yet
                } else if (m_new > m_ref + RESCALE_LOG2) {
                    f = fast_exp2(m_ref - m_new);
                    l *= f;
                    m_ref = m_new;
                }
                // Past the exchange barrier no warp leaves the loop on its own (its partner
                // would wait at the next barrier): a failed wait is noted and the loop
                // ends at the next barrier.
                if (__any_sync(FULL_MASK, f != 1.f)) {
                    // O holds the item's stages < s: wait for the last of their updates,
                    // then scale this thread's half of the output row
                    ok = all_ok(mbar_wait_bounded(smem_u32(&ctl->p_free), static_cast<uint32_t>(gs - 1) & 1u));
                    if (!ok) {
                        failed = true;
                        continue;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c2 = 0; c2 < 2; ++c2) {
                        uint32_t r[32];
                        const uint32_t col = TM_O + half * 64 + c2 * 32;
                        tc_ld32(lrow + col, r);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * f);
                        tc_st32(lrow + col, r);
                    }
                    tc_wait_st();
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                uint32_t pk[16];
                float ls = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float p0 = fast_exp2(fmaf(sv[2 * j], sl2, -m_use));
                    const float p1 = fast_exp2(fmaf(sv[2 * j + 1], sl2, -m_use));
                    ls += p0 + p1;
                    pk[j] = pack_bf16x2(p0, p1);
                }
                l += ls;
                if (nvalid_all < TC_TOK) {
                    // values of tokens past the cache (or of a skipped block) are zeroed so
                    // that 0 * NaN cannot reach the output sums
                    uint8_t* sp = smem + st * TC_STAGE + 2 * dq * TC_PIECE;
                    const int v0 = max(0, nvalid_all);
                    for (int i = st_id; i < (TC_TOK - v0) * 16; i += 256) {
                        const int row = v0 + (i >> 4);
                        const int pc = (i >> 3) & 1;
                        const int ch = i & 7;
                        *reinterpret_cast<uint4*>(sp + pc * TC_PIECE + row * 128 + (ch << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                if (gs >= 1) {
                    // the previous probabilities must have been consumed
                    ok = all_ok(mbar_wait_bounded(smem_u32(&ctl->p_free), static_cast<uint32_t>(gs - 1) & 1u));
                    if (!ok) {
                        failed = true;
                        continue;
                    }
                }
                tc_fence_after();
                tc_st16(lrow + TM_P + half * 16, pk);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full));
            }
            // all threads leave the stage loop together (the exchange barrier), so this
            // barrier sees every softmax thread; a failure ends the item loop for all
            if (named_barrier_or(1, 256, failed)) {
                failed = true;
                break;
            }
            ok = n < 1 || all_ok(mbar_wait_bounded(smem_u32(&ctl->p_free), static_cast<uint32_t>(g + n - 1) & 1u));
            tc_fence_after();
            ctl->xl[half][h] = l;
            if (named_barrier_or(1, 256, !ok)) {
                failed = true;
                break;
            }
            l = ctl->xl[0][h] + ctl->xl[1][h];

            // ---- epilogue: this thread's head, latent numbers 128 dq + 64 half .. + 63
            const size_t bh = row0 + h;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const bool write = h < nh;
            const bool whole = nsplit == 1;
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r[32];
                if (n >= 1) {
                    tc_ld32(lrow + TM_O + half * 64 + c2 * 32, r);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                if (!write) continue;
                const int d0 = dq * TC_DQ + half * 64 + c2 * 32;
                if (whole) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + bh * MLA_DV + d0);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(
                            pack_bf16x2(__uint_as_float(r[8 * v]) * inv, __uint_as_float(r[8 * v + 1]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv),
                            pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv));
                } else {
                    float4* dst = reinterpret_cast<float4*>(p.part_o + (bh * p.max_splits + split) * MLA_DV + d0);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                             __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
                }
            }
            tc_fence_before();
            if (write && half == 0) {
                if (whole) {
                    if (p.lse != nullptr && dq == 0) p.lse[bh] = lse_from(m_ref, l);
                } else {
                    // every quarter writes the same (max, sum); the merge of a quarter reads
                    // the pairs its own siblings wrote before counting themselves
                    p.part_ml[(bh * p.max_splits + split) * 2 + 0] = m_ref;
                    p.part_ml[(bh * p.max_splits + split) * 2 + 1] = l;
                }
            }
            if (!whole) {
                __threadfence();
                named_barrier_sync(1, 256);
                int* ticket = p.tickets + (static_cast<size_t>(b) * p.head_tiles + ht) * 4 + dq;
                if (st_id == 0) {
                    const int last = atomicAdd(ticket, 1) == nsplit - 1;
                    if (last) __threadfence();
                    ctl->merge_flag = last;
                }
                named_barrier_sync(1, 256);
                const bool merge = ctl->merge_flag != 0;
                if (merge && h < nh) {
                    const float* ml = p.part_ml + bh * p.max_splits * 2;
                    float M = -INFINITY;
                    for (int j = 0; j < nsplit; ++j)
                        if (__ldcg(ml + 2 * j + 1) > 0.f) M = fmaxf(M, __ldcg(ml + 2 * j));
                    float W = 0.f;
                    for (int j = 0; j < nsplit; ++j) {
                        const float lj = __ldcg(ml + 2 * j + 1);
                        if (lj > 0.f) W += lj * fast_exp2(__ldcg(ml + 2 * j) - M);
                    }
                    const float winv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll 1
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const int d0 = dq * TC_DQ + half * 64 + c8 * 8;
                        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        for (int j = 0; j < nsplit; ++j) {
                            const float lj = __ldcg(ml + 2 * j + 1);
                            if (!(lj > 0.f)) continue;
                            const float wj = lj * fast_exp2(__ldcg(ml + 2 * j) - M);
                            const float4* src = reinterpret_cast<const float4*>(
                                p.part_o + (bh * p.max_splits + j) * MLA_DV + d0);
                            const float4 a0 = __ldcg(src), a1 = __ldcg(src + 1);
                            acc[0] += wj * a0.x;
                            acc[1] += wj * a0.y;
                            acc[2] += wj * a0.z;
                            acc[3] += wj * a0.w;
                            acc[4] += wj * a1.x;
                            acc[5] += wj * a1.y;
                            acc[6] += wj * a1.z;
                            acc[7] += wj * a1.w;
                        }
                        *reinterpret_cast<uint4*>(p.out + bh * MLA_DV + d0) =
                            make_uint4(pack_bf16x2(acc[0] * winv, acc[1] * winv), pack_bf16x2(acc[2] * winv, acc[3] * winv),
                                       pack_bf16x2(acc[4] * winv, acc[5] * winv), pack_bf16x2(acc[6] * winv, acc[7] * winv));
                    }
                    if (p.lse != nullptr && dq == 0 && half == 0) p.lse[bh] = lse_from(M, W);
                }
                if (merge && st_id == 0) *ticket = 0;
                named_barrier_sync(1, 256);         // merge_flag is reused by the next item
            }
            g += n;
        }
        if (failed && lane == 0) {
            atomicOr(p.err, KV_DEVERR_TIMEOUT);
            ctl->abort_flag = 1;
        }
        grid_dependents_launch();
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tc_dealloc(tbase, TM_COLS);
    }
    if (tid == 0) {
        // the last CTA to finish resets the work counter for the next call
        __threadfence();
        if (atomicAdd(p.queue + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            p.queue[0] = 0;
            p.queue[1] = 0;
            __threadfence();
        }
    }
}

cudaError_t prepare_mla_decode_tc()
{
    return cudaFuncSetAttribute(paged_mla_decode_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TC_SMEM);
}

cudaError_t launch_mla_decode_tc(dim3 grid, const CUtensorMap& tm, const MlaParams& p,
                                 cudaStream_t s)
{
    return launch_dependent(paged_mla_decode_tc, grid, dim3(TC_THREADS), TC_SMEM, s, tm, p);
}

}  // namespace kvp
