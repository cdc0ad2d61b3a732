// decode_mla_tc.cu -- absorbed multi-head latent attention on the 5th-generation
// tensor cores (tcgen05), for wide head tiles: all 128 query heads of a sequence
// on the MMA's M dimension (xuewyang.github.io/posts/kv, "MLA: how does decode
// get full-size keys and values back?": every head scores the shared cached
// vector -- 512 latent + 64 rotary-key numbers -- and averages its latent part).
//
// A CTA computes one 256-wide half of the latent output of a tile of 128 heads, and
// the full scores: the fp32 output of 128 heads x 512 latent numbers alone would fill
// an SM's tensor memory.
//
// Persistent: one CTA per SM holds its tensor memory for the whole launch and takes
// one equal contiguous range of the units (latent half, head tile, sequence, block)
// (mla_partition.cuh); a sequence cut by a range boundary leaves fp32 partials,
// merged by paged_mla_merge_tc.  352 threads:
//   * warp 8 walks the range's segments (item = a run of blocks of one sequence,
//     head tile and half), passes each to the other roles through a 4-slot ring in
//     shared memory, and streams its 64-token blocks, one per stage, with nine
//     TMA loads (one per 128-byte piece of the 576 numbers, 128-byte swizzle):
//     a stage is nine K-major [64 tokens x 64 numbers] tiles, 72 KB, 2 stages.
//     The five pieces only the scores read (the other half's latent numbers and
//     the rotary key) and the four pieces of this CTA's output half have
//     barriers of their own: the first five are reloaded as soon as the scores
//     of their stage are done, the other four once its output update is.
//   * warp 9 (one thread) issues the score MMAs.  Scores S[128 heads x 64 tokens] =
//     Q . C^T in 36 MMAs of K = 16: the 20 over the score-only pieces take A =
//     the queries' matching 320 numbers held in tensor memory, the 16 over the
//     output pieces (whose loads land last) take A = the other 256 numbers held
//     in shared memory.  Warp 10 (one thread) issues the output update
//     O[128 heads x 256 latent] += P . C[:, half]: A = the probabilities in tensor
//     memory, B = the four output pieces read MN-major (the latent numbers of a
//     token are contiguous), 4 MMAs of N = 256.  Completion is signalled by
//     tcgen05.commit on mbarriers.  With two issuing threads the scores of stage
//     i+1 start as soon as the softmax has read those of stage i, and the update of
//     stage i as soon as its probabilities are written; one thread issuing both in a
//     fixed order made each wait for the other.
//   * warps 0-7: head h (tensor-memory lane h) belongs to two threads, one in
//     warp h / 32 (tokens 0-31 of a stage, output columns 0-127) and one in warp
//     h / 32 + 4 (tokens 32-63, columns 128-255) -- a warp can only reach its
//     own quarter of the lanes, and two warps per quarter halve the serial work
//     of each.  Each reads its 32 scores, the pair exchanges its maxima through
//     shared memory, and each writes its 32 probabilities (bf16) back to tensor
//     memory; at the end of an item each normalises and stores its 128 outputs,
//     then loads the next item's queries.  The output is rescaled only when the
//     running max grows by more than 2^8 (log2 units); until then the older
//     maximum stays the reference, which is exact because the final division
//     uses the sum taken against the same reference.
//   * tensor memory: queries [0, 160), scores [160, 224), probabilities
//     [224, 256), output [256, 512).  Shared memory: 2 stages (144 KB), the
//     queries' other 256 numbers (64 KB, K-major, 128-byte swizzle), control.
//   * paged_mla_decode_step: lanes 1-31 of the producer warp walk the same partition and
//     write the new vector of each sequence whose last block lies in the range into that
//     block; the producer lane waits on an mbarrier for those writes before it loads such
//     a block.
// Every wait is bounded; a late barrier sets KV_DEVERR_TIMEOUT and every role
// leaves its loop, waits (bounded) for its copies and MMAs in flight, and the CTA
// frees its tensor memory before it exits.
#include "append_row.cuh"
#include "decode_common.cuh"
#include "kernels.h"
#include "mla_partition.cuh"
#include "tcgen05.cuh"

namespace kvp {

namespace {

constexpr int TC_TOK = 64;                      // tokens per stage (one block)
constexpr int TC_NSTAGE = 2;
constexpr int TC_PIECE = TC_TOK * 128;          // one 64-number piece of 64 tokens
constexpr int TC_NPIECE = MLA_DK / 64;          // 9
constexpr int TC_NEARLY = 5;                    // pieces only the scores read
constexpr int TC_NLATE = TC_NPIECE - TC_NEARLY; // 4: this CTA's output half
constexpr int TC_STAGE = TC_NPIECE * TC_PIECE;  // 73,728 bytes
constexpr int TC_DQ = 256;                      // latent numbers per CTA
constexpr int TC_M = 128;                       // heads per CTA
constexpr int TC_QPIECE = TC_M * 128;           // one 64-number piece of 128 heads
constexpr int TC_QS = TC_NLATE * TC_QPIECE;     // queries kept in shared memory
constexpr int TC_THREADS = 352;                 // warps 0-7 softmax, 8 loads, 9 score MMAs, 10 output MMAs
constexpr uint32_t TM_Q = 0, TM_S = 160, TM_P = 224, TM_O = 256, TM_COLS = 512;
constexpr uint32_t IDESC_S = tc_idesc_bf16(TC_M, TC_TOK, 0, 0);
constexpr uint32_t IDESC_O = tc_idesc_bf16(TC_M, TC_DQ, 0, 1);
constexpr float RESCALE_LOG2 = 8.f;
constexpr int TC_CTL = 4096;
constexpr int TC_SMEM = 1024 + TC_NSTAGE * TC_STAGE + TC_QS + TC_CTL;
static_assert(TC_SMEM <= 227 * 1024, "one CTA per SM");
static_assert(TM_Q + TC_NEARLY * 32 <= TM_S && TM_S + TC_TOK <= TM_P && TM_P + TC_TOK / 2 <= TM_O &&
                  TM_O + TC_DQ <= TM_COLS,
              "tensor-memory columns");
static_assert(TC_NLATE * 64 == TC_DQ, "the output half is the four late pieces");

constexpr int TC_NITEM = 4;                     // ring of work items in shared memory

// Piece of the 576 numbers held by score-only slot j (0..4) / output slot j (0..3)
// of a stage, for the CTA computing latent half dq.
__device__ __forceinline__ int early_piece(int dq, int j) { return j < 4 ? 4 * (1 - dq) + j : 8; }
__device__ __forceinline__ int late_piece(int dq, int j) { return 4 * dq + j; }

// A work item as the producer hands it on: blocks blk0 .. blk0 + n - 1 of sequence b
// (n >= 1; -1: no more items), piece `split` of the `nsplit` the sequence's units
// were cut into by the partition.
struct TcItem {
    int b, ht, dq, split, nsplit, blk0, n, ctx;
};

struct TcCtl {
    uint64_t kv_full_e[TC_NSTAGE];                  // score-only pieces landed
    uint64_t kv_full_l[TC_NSTAGE];                  // output pieces landed
    uint64_t kv_empty_e[TC_NSTAGE];                 // scores of the stage done
    uint64_t kv_empty_l[TC_NSTAGE];                 // output update of the stage done
    uint64_t s_full, s_free, p_full, p_free, q_ready, mma_done[2];
    uint64_t item_full[TC_NITEM];
    uint64_t item_empty[TC_NITEM];
    uint32_t tmem_base;
    int stage_blk[TC_NSTAGE];
    int abort_flag;
    TcItem items[TC_NITEM];
    float xmax[2][2][TC_M];                         // [stage parity][token half][head]
    float xl[2][TC_M];                              // [token half][head]
    uint64_t step_done;                             // paged_mla_decode_step: new vectors written
};
static_assert(sizeof(TcCtl) <= TC_CTL, "control block");

// Scores over the five score-only pieces: 20 MMAs of K = 16 with A = the queries'
// matching numbers in tensor memory.  The descriptor of slice ks is the stage's
// base descriptor plus a constant (16-byte units in the low word), so each issue
// is one add: a single thread issues every MMA of the CTA, and its issue rate, not
// the tensor pipe, bounds small-N MMAs like these.
__device__ __forceinline__ void issue_score_early(uint32_t tbase, uint32_t stage_addr)
{
    const uint64_t d0 = tc_smem_desc(stage_addr, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < TC_NEARLY * 4; ++ks)
        tc_mma_ts(tbase + TM_S, tbase + TM_Q + ks * 8,
                  d0 + static_cast<uint64_t>(((ks >> 2) * TC_PIECE + (ks & 3) * 32) >> 4), IDESC_S,
                  ks > 0);
}

// Scores over the four output pieces: 16 MMAs with A = the other query numbers,
// K-major in shared memory.
__device__ __forceinline__ void issue_score_late(uint32_t tbase, uint32_t stage_addr, uint32_t q_addr)
{
    const uint64_t b0 = tc_smem_desc(stage_addr + TC_NEARLY * TC_PIECE, 16, 1024);
    const uint64_t a0 = tc_smem_desc(q_addr, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < TC_NLATE * 4; ++ks)
        tc_mma_ss(tbase + TM_S, a0 + static_cast<uint64_t>(((ks >> 2) * TC_QPIECE + (ks & 3) * 32) >> 4),
                  b0 + static_cast<uint64_t>(((ks >> 2) * TC_PIECE + (ks & 3) * 32) >> 4), IDESC_S, true);
}

// The output update of a stage: O += P . C[:, half] over its 64 tokens; the four
// output pieces are the N = 256 operand read MN-major (64-number atoms one piece
// apart, 8-token groups 1 KB apart).
__device__ __forceinline__ void issue_output_mma(uint32_t tbase, uint32_t stage_addr, bool first)
{
    const uint64_t d0 = tc_smem_desc(stage_addr + TC_NEARLY * TC_PIECE, TC_PIECE, 1024);
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
    uint8_t* qsm = smem + TC_NSTAGE * TC_STAGE;
    TcCtl* ctl = reinterpret_cast<TcCtl*>(qsm + TC_QS);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int* abort_flag = &ctl->abort_flag;

    if (tid == 0) {
        for (int i = 0; i < TC_NSTAGE; ++i) {
            mbar_init(smem_u32(&ctl->kv_full_e[i]), 1);
            mbar_init(smem_u32(&ctl->kv_full_l[i]), 1);
            mbar_init(smem_u32(&ctl->kv_empty_e[i]), 1);
            mbar_init(smem_u32(&ctl->kv_empty_l[i]), 1);
        }
        for (int i = 0; i < TC_NITEM; ++i) {
            mbar_init(smem_u32(&ctl->item_full[i]), 1);
            mbar_init(smem_u32(&ctl->item_empty[i]), 10);  // the two MMA threads + 8 softmax warps
        }
        mbar_init(smem_u32(&ctl->s_full), 1);
        mbar_init(smem_u32(&ctl->s_free), 8);
        mbar_init(smem_u32(&ctl->p_full), 8);
        mbar_init(smem_u32(&ctl->p_free), 1);
        mbar_init(smem_u32(&ctl->q_ready), 8);
        mbar_init(smem_u32(&ctl->mma_done[0]), 1);
        mbar_init(smem_u32(&ctl->mma_done[1]), 1);
        mbar_init(smem_u32(&ctl->step_done), 31);   // lanes 1-31 of the producer warp
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) tc_alloc(smem_u32(&ctl->tmem_base), TM_COLS);
    grid_dependency_wait();                     // inputs of the preceding kernel are ready
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ctl->tmem_base;

    if (warp == 8) {
        // ------------------------------------------------------------ partition, items, loads
        // Units: (half dq, head tile ht, sequence b, block) in that order (outer index
        // dq * head_tiles + ht), cut into equal contiguous ranges (mla_partition.cuh).
        MlaPartition<TC_TOK, MLA_SEG_PAD_WIDE> part;
        part.init(p, p.head_tiles * 2, lane);
        if (lane == 0) {
            prefetch_tensormap(&tmp);
            int k = 0;                              // items handed on
            int g = 0;                              // stages issued (all items)
            int ge = 0, gl = 0;                     // stages with score-only / output loads issued
            bool ok = true;
            bool step_written = false;              // paged_mla_decode_step: waited for lanes 1-31
            for (;;) {
                TcItem it{};
                it.n = -1;
                if (!*abort_flag) {
                    const MlaSegment sg = part.next();
                    it.n = sg.n;
                    if (sg.n >= 0) {
                        it.b = sg.b;
                        it.dq = sg.outer / p.head_tiles;
                        it.ht = sg.outer - it.dq * p.head_tiles;
                        it.split = sg.split;
                        it.nsplit = sg.nsplit;
                        it.blk0 = sg.blk0;
                        it.ctx = sg.ctx;
                    }
                }
                const bool last = it.n < 0;
                if (!last) {
                    // the item's queries (rows of its head tile, contiguous) into L2: the
                    // softmax warps load them when the previous item is done
                    const size_t qrow0 = static_cast<size_t>(it.b) * p.q_heads + it.ht * TC_M;
                    const int nhq = min(TC_M, p.q_heads - it.ht * TC_M);
                    prefetch_l2_bulk(p.q + qrow0 * MLA_DK, static_cast<uint32_t>(nhq) * MLA_DK * 2);
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
                const int32_t* trow = p.tables + static_cast<size_t>(it.b) * p.max_blocks + it.blk0;
                int next_blk = __ldg(trow);         // block id read one stage ahead
                // paged_mla_decode_step: the segment's stage whose block holds the new vector
                const int step_s = mla_step_block(p, it.b, TC_TOK) - it.blk0;
                for (int s = 0; s < it.n; ++s, ++g) {
                    const int st = g % TC_NSTAGE;
                    const uint32_t ph = (static_cast<uint32_t>(g / TC_NSTAGE) & 1u) ^ 1u;
                    int bid = next_blk;
                    if (s + 1 < it.n) next_blk = __ldg(trow + s + 1);
                    if (bid < 0 || bid >= p.num_blocks) {
                        atomicOr(p.err, KV_DEVERR_BLOCK_ID);
                        bid = -1;
                    }
                    if (s == step_s && bid >= 0 && !step_written) {   // holds a new vector
                        if (!mbar_wait_bounded(smem_u32(&ctl->step_done), 0u)) {
                            ok = false;
                            break;
                        }
                        step_written = true;
                    }
                    const uint32_t dst = smem_u32(smem + st * TC_STAGE);
                    // score-only pieces: free once the scores of the stage two back are done
                    if (!mbar_wait_bounded(smem_u32(&ctl->kv_empty_e[st]), ph) || *abort_flag) {
                        ok = false;
                        break;
                    }
                    const uint32_t fe = smem_u32(&ctl->kv_full_e[st]);
                    if (bid >= 0) {
                        mbar_arrive_expect_tx(fe, TC_NEARLY * TC_PIECE);
                        for (int j = 0; j < TC_NEARLY; ++j)
                            tma_load_5d(dst + j * TC_PIECE, &tmp, 0, early_piece(it.dq, j), 0, 0, bid, fe);
                        // the output pieces load later (when their slot frees): bring them
                        // into L2 now so that load is short
                        for (int j = 0; j < TC_NLATE; ++j)
                            tma_prefetch_l2_5d(&tmp, 0, late_piece(it.dq, j), 0, 0, bid);
                    } else {
                        mbar_arrive(fe);
                    }
                    ge = g + 1;
                    // output pieces: free once that stage's output update is done (its
                    // softmax, which reads stage_blk, is then over too)
                    if (!mbar_wait_spin(smem_u32(&ctl->kv_empty_l[st]), ph) || *abort_flag) {
                        ok = false;
                        break;
                    }
                    ctl->stage_blk[st] = bid;
                    const uint32_t fl = smem_u32(&ctl->kv_full_l[st]);
                    if (bid >= 0) {
                        mbar_arrive_expect_tx(fl, TC_NLATE * TC_PIECE);
                        for (int j = 0; j < TC_NLATE; ++j)
                            tma_load_5d(dst + (TC_NEARLY + j) * TC_PIECE, &tmp, 0, late_piece(it.dq, j), 0,
                                        0, bid, fl);
                    } else {
                        mbar_arrive(fl);
                    }
                    gl = g + 1;
                }
                if (!ok) break;
            }
            if (!ok) {
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ctl->abort_flag = 1;
            }
            // copies still in flight must land before the CTA moves on
            for (int j = max(0, ge - TC_NSTAGE); j < ge; ++j)
                if (!mbar_wait_bounded(smem_u32(&ctl->kv_full_e[j % TC_NSTAGE]),
                                       static_cast<uint32_t>(j / TC_NSTAGE) & 1u))
                    break;
            for (int j = max(0, gl - TC_NSTAGE); j < gl; ++j)
                if (!mbar_wait_bounded(smem_u32(&ctl->kv_full_l[j % TC_NSTAGE]),
                                       static_cast<uint32_t>(j / TC_NSTAGE) & 1u))
                    break;
        } else {
            // the next kernel may start launching (it waits for this grid's completion
            // before reading anything); lanes 1-31 write the step's new vectors, if any
            grid_dependents_launch();
            if (p.kv_new != nullptr) part.write_step_rows(smem_u32(&ctl->step_done), lane - 1, 31);
        }
        grid_dependents_launch();
    } else if (warp == 9 || warp == 10) {
        // ------------------------------------------------------------ MMA issue
        // Two issuing threads: warp 9 the scores of each stage, as soon as it has landed
        // and the softmax has read the scores before (one score buffer); warp 10 the output
        // update of each stage, as soon as its probabilities are written.  The update of a
        // stage reads the probabilities and this half's pieces, the scores the queries and
        // all nine pieces: the two touch different tensor memory, and an item's first
        // update waits for its queries, which the softmax threads load only after their
        // epilogue has read the output of the item before.
        if (lane == 0) {
            const bool scores = warp == 9;
            const uint32_t q_addr = smem_u32(qsm);
            bool ok = true;
            int g = 0;                              // stages processed (all items)
            for (int k = 0; ok; ++k) {
                const int slot = k % TC_NITEM;
                ok = mbar_wait_bounded(smem_u32(&ctl->item_full[slot]),
                                       static_cast<uint32_t>(k / TC_NITEM) & 1u);
                if (!ok) break;
                const int n = ctl->items[slot].n;
                mbar_arrive(smem_u32(&ctl->item_empty[slot]));
                if (n < 0) break;
                ok = mbar_wait_bounded(smem_u32(&ctl->q_ready), static_cast<uint32_t>(k) & 1u);
                for (int s = 0; ok && s < n; ++s) {
                    const int gs = g + s;
                    const int st = gs % TC_NSTAGE;
                    const uint32_t ph = static_cast<uint32_t>(gs / TC_NSTAGE) & 1u;
                    const uint32_t stage_addr = smem_u32(smem + st * TC_STAGE);
                    if (!scores) {
                        // polled without suspending: this update frees the slot of this half's
                        // pieces, whose reload the scores two stages on wait for
                        ok = mbar_wait_spin(smem_u32(&ctl->p_full), static_cast<uint32_t>(gs) & 1u);
                        if (!ok || *abort_flag) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_output_mma(tbase, stage_addr, s == 0);
                        tc_commit(smem_u32(&ctl->p_free));
                        tc_commit(smem_u32(&ctl->kv_empty_l[st]));
                        continue;
                    }
                    ok = mbar_wait_bounded(smem_u32(&ctl->kv_full_e[st]), ph);
                    // the score buffer is free once the softmax has read the stage before
                    if (ok && gs >= 1) ok = mbar_wait_bounded(smem_u32(&ctl->s_free), static_cast<uint32_t>(gs - 1) & 1u);
                    if (!ok || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_score_early(tbase, stage_addr);
                    // then the scores over this half's pieces (their loads, issued once the
                    // update of the stage two back had finished with the slot)
                    ok = mbar_wait_bounded(smem_u32(&ctl->kv_full_l[st]), ph);
                    if (!ok) break;
                    tc_fence_after();
                    issue_score_late(tbase, stage_addr, q_addr);
                    tc_commit(smem_u32(&ctl->s_full));
                    tc_commit(smem_u32(&ctl->kv_empty_e[st]));
                }
                g += n;
            }
            if (!ok) {
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ctl->abort_flag = 1;
            }
            // every MMA issued must be complete before the tensor memory is freed
            const uint32_t done = smem_u32(&ctl->mma_done[scores ? 0 : 1]);
            tc_commit(done);
            mbar_wait_bounded(done, 0);
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
            const int ht = item.ht, blk0 = item.blk0, nsplit = item.nsplit;
            const int nh = min(TC_M, p.q_heads - ht * TC_M);
            const size_t row0 = static_cast<size_t>(b) * p.q_heads + ht * TC_M;
            {
                // queries (the previous item's score MMAs are complete: this thread
                // waited for its last scores).  The 128 rows of the tile are contiguous;
                // they are copied piece by piece into the queries' shared memory with
                // coalesced 16-byte asynchronous copies (consecutive threads: the eight
                // 16-byte chunks of a row, then the next rows; K-major with the 128-byte
                // swizzle, chunk c of row r at (c ^ (r & 7))), in three rounds: the four
                // score-only latent pieces and then the rotary piece go on to tensor
                // memory (each thread moving its head's row), the four pieces of this
                // CTA's output half stay in shared memory for the MMAs.
                const uint32_t qs = smem_u32(qsm);
                const uint16_t* qtile = p.q + row0 * MLA_DK;
                auto copy_pieces = [&](int npc, int first_slot, bool late) {
                    for (int idx = st_id; idx < npc * TC_M * 8; idx += 256) {
                        const int j = idx >> 10, r = (idx >> 3) & (TC_M - 1), cc = idx & 7;
                        const int pc = late ? late_piece(dq, j) : early_piece(dq, first_slot + j);
                        const uint32_t dst = qs + j * TC_QPIECE + r * 128 + ((cc ^ (r & 7)) << 4);
                        if (r < nh)
                            cp_async16(dst, qtile + static_cast<size_t>(r) * MLA_DK + pc * 64 + cc * 8);
                        else
                            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
                    }
                    cp_async_wait_all();
                    named_barrier_sync(1, 256);
                };
                auto row_chunk = [&](int j, int cc) {
                    uint4 v;
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                                 : "r"(qs + j * TC_QPIECE + h * 128 + ((cc ^ (h & 7)) << 4)));
                    return v;
                };
                // round 1: score-only latent pieces -> tensor-memory slots 0-3 (2 per half)
                copy_pieces(4, 0, false);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const int j = half * 2 + jj;
                    uint32_t r[32];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint4 v = row_chunk(j, cc);
                        r[4 * cc] = v.x;
                        r[4 * cc + 1] = v.y;
                        r[4 * cc + 2] = v.z;
                        r[4 * cc + 3] = v.w;
                    }
                    tc_st32(lrow + TM_Q + j * 32, r);
                }
                tc_wait_st();
                named_barrier_sync(1, 256);
                // round 2: the rotary piece -> tensor-memory slot 4 (16 columns per half)
                copy_pieces(1, 4, false);
                {
                    uint32_t r[16];
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 v = row_chunk(0, half * 4 + cc);
                        r[4 * cc] = v.x;
                        r[4 * cc + 1] = v.y;
                        r[4 * cc + 2] = v.z;
                        r[4 * cc + 3] = v.w;
                    }
                    tc_st16(lrow + TM_Q + 4 * 32 + half * 16, r);
                }
                tc_wait_st();
                named_barrier_sync(1, 256);
                // round 3: this half's pieces, kept in shared memory for the MMAs
                copy_pieces(4, 0, true);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctl->q_ready));
            }
            float m_ref = -INFINITY, l = 0.f;
            for (int s = 0; s < n; ++s) {
                const int gs = g + s;
                const int st = gs % TC_NSTAGE;
                ok = mbar_wait_bounded(smem_u32(&ctl->kv_full_l[st]), static_cast<uint32_t>(gs / TC_NSTAGE) & 1u);
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
                    for (int c2 = 0; c2 < 4; ++c2) {
                        uint32_t r[32];
                        const uint32_t col = TM_O + half * 128 + c2 * 32;
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
                    // that 0 * NaN cannot reach the output sums (the scores of the stage,
                    // which read these rows too, are complete)
                    uint8_t* sp = smem + st * TC_STAGE + TC_NEARLY * TC_PIECE;
                    const int v0 = max(0, nvalid_all);
                    for (int i = st_id; i < (TC_TOK - v0) * 32; i += 256) {
                        const int row = v0 + (i >> 5);
                        const int pc = (i >> 3) & 3;
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

            // ---- epilogue: this thread's head, latent numbers 256 dq + 128 half .. + 127,
            // in four chunks of 32.  A whole sequence's output goes through shared memory
            // (the queries' shared-memory part, idle until the next item's queries are
            // loaded by these threads) so that the global writes are whole rows: 32 heads
            // x 32 numbers per warp, row r = head 32 (warp % 4) + r, 16-byte chunk j of a
            // row at (j ^ (r & 7)).  A piece of a cut sequence leaves its partial for
            // paged_mla_merge_tc, and every item records its sequence's piece count.
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const bool whole = nsplit == 1;
            // piece index of a cut sequence's partial: (sequence, head tile, half, split)
            const size_t piece = ((static_cast<size_t>(b) * p.head_tiles + ht) * 2 + dq) * p.max_splits + split;
            if (!whole && h < nh && half == 0)
                reinterpret_cast<float2*>(p.part_ml)[piece * TC_M + h] = make_float2(m_ref, l);
            const uint32_t tile = smem_u32(qsm) + warp * 4096;
            const int hq = (warp & 3) * 32;         // first head of this warp's rows
#pragma unroll 1
            for (int c2 = 0; c2 < 4; ++c2) {
                uint32_t r[32];
                if (n >= 1) {
                    tc_ld32(lrow + TM_O + half * 128 + c2 * 32, r);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = 0u;
                }
                if (!whole) {
                    // a piece of a cut sequence: its normalised partial, in fp16 (values of
                    // the cache averaged: well inside its range, 11 significant bits against
                    // the output's 8), in the piece layout [32-number chunk][4-number slot]
                    // [head], coalesced as written (thread = head); its (max, sum) beside it
                    uint2* dst = reinterpret_cast<uint2*>(p.part_o) + piece * (TC_M * TC_DQ / 4) +
                                 static_cast<size_t>((half * 4 + c2) * 8) * TC_M + h;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j * TC_M] = make_uint2(pack_f16x2(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv),
                                                   pack_f16x2(__uint_as_float(r[4 * j + 2]) * inv, __uint_as_float(r[4 * j + 3]) * inv));
                    continue;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(tile + lane * 128 + ((j ^ (lane & 7)) << 4)),
                                 "f"(__uint_as_float(r[4 * j]) * inv), "f"(__uint_as_float(r[4 * j + 1]) * inv),
                                 "f"(__uint_as_float(r[4 * j + 2]) * inv), "f"(__uint_as_float(r[4 * j + 3]) * inv)
                                 : "memory");
                __syncwarp();
                const int d0 = dq * TC_DQ + half * 128 + c2 * 32;
                {
                    // bf16 rows of 64 bytes: lane -> row it * 8 + lane / 4, numbers 8 (lane % 4) ..
#pragma unroll
                    for (int it = 0; it < 4; ++it) {
                        const int rr = it * 8 + (lane >> 2), qd = lane & 3;
                        float4 a, bq;
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w)
                                     : "r"(tile + rr * 128 + (((2 * qd) ^ (rr & 7)) << 4)));
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(bq.x), "=f"(bq.y), "=f"(bq.z), "=f"(bq.w)
                                     : "r"(tile + rr * 128 + (((2 * qd + 1) ^ (rr & 7)) << 4)));
                        if (hq + rr < nh)
                            *reinterpret_cast<uint4*>(p.out + (row0 + hq + rr) * MLA_DV + d0 + qd * 8) =
                                make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(bq.x, bq.y),
                                           pack_bf16x2(bq.z, bq.w));
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            const size_t bh = row0 + h;
            if (h < nh && half == 0 && whole && p.lse != nullptr && dq == 0) p.lse[bh] = lse_from(m_ref, l);
            if (st_id == 0 && p.tickets != nullptr)
                p.tickets[(static_cast<size_t>(b) * p.head_tiles + ht) * 2 + dq] = nsplit;
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
}

// Merge of the pieces of every cut sequence: CTA (chunk of 32 latent numbers, head
// tile and half, sequence), thread = head.  The pieces' (max, sum) pairs give the
// weights w_j = l_j 2^(m_j - M) of the standard log-sum-exp merge; the output row is
// sum_j w_j o_j / sum_j w_j, staged through shared memory for whole-row writes.
__global__ void __launch_bounds__(TC_M, 4)
paged_mla_merge_tc(const MlaParams p)
{
    __shared__ uint32_t tile[TC_M][17];             // bf16 pairs, padded rows
    // The next kernel may start launching now (its CTAs set up beside this grid's small
    // CTAs); it reads nothing before waiting for this grid to complete.
    grid_dependents_launch();
    grid_dependency_wait();
    const int cg = blockIdx.x;                      // 32-number chunk of the half
    const int ht = blockIdx.y >> 1, dq = blockIdx.y & 1;
    const int b = blockIdx.z;
    const int h = threadIdx.x;
    const int ctx = __ldg(p.ctx + b);
    // an empty sequence (or a negative length, read as empty) has no pieces
    const int nsplit = ctx > 0 ? __ldcg(p.tickets + (static_cast<size_t>(b) * p.head_tiles + ht) * 2 + dq) : 1;
    if (nsplit > 1) {
        const int nh = min(TC_M, p.q_heads - ht * TC_M);
        const size_t piece0 = ((static_cast<size_t>(b) * p.head_tiles + ht) * 2 + dq) * p.max_splits;
        const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + piece0 * TC_M + h;
        const uint2* po = reinterpret_cast<const uint2*>(p.part_o) + piece0 * (TC_M * TC_DQ / 4) +
                          static_cast<size_t>(cg * 8) * TC_M + h;
        float M = -INFINITY, W = 0.f;
        float acc[32];
#pragma unroll
        for (int v = 0; v < 32; ++v) acc[v] = 0.f;
        // two pieces per round: their (max, sum) pairs and numbers are loaded together; the
        // running max and the accumulators are rescaled when a later piece raises the max
        for (int j0 = 0; j0 < nsplit; j0 += 2) {
            float2 mj[2];
            float4 x[2][8];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const bool in = j0 + i < nsplit;
                const size_t j = static_cast<size_t>(in ? j0 + i : j0);
                mj[i] = in ? __ldcg(ml + j * TC_M) : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint2 u = __ldcg(po + j * (TC_M * TC_DQ / 4) + v * TC_M);
                    const float2 a = unpack_f16x2(u.x), c = unpack_f16x2(u.y);
                    x[i][v] = make_float4(a.x, a.y, c.x, c.y);
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (!(mj[i].y > 0.f)) continue;
                const float m2 = fmaxf(M, mj[i].x);
                const float fo = fast_exp2(M - m2);        // 0 while nothing is accumulated
                const float wj = mj[i].y * fast_exp2(mj[i].x - m2);
                W = W * fo + wj;
                M = m2;
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    acc[4 * v] = acc[4 * v] * fo + wj * x[i][v].x;
                    acc[4 * v + 1] = acc[4 * v + 1] * fo + wj * x[i][v].y;
                    acc[4 * v + 2] = acc[4 * v + 2] * fo + wj * x[i][v].z;
                    acc[4 * v + 3] = acc[4 * v + 3] * fo + wj * x[i][v].w;
                }
            }
        }
        const float winv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
        for (int v = 0; v < 16; ++v) tile[h][v] = pack_bf16x2(acc[2 * v] * winv, acc[2 * v + 1] * winv);
        if (p.lse != nullptr && dq == 0 && cg == 0 && h < nh)
            p.lse[static_cast<size_t>(b) * p.q_heads + ht * TC_M + h] = lse_from(M, W);
        __syncthreads();
        // rows of 64 bytes: thread -> row it * 32 + h / 4, 16 bytes (h % 4)
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int rr = it * 32 + (h >> 2), qd = h & 3;
            if (rr < nh)
                *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(b) * p.q_heads + ht * TC_M + rr) * MLA_DV +
                                          dq * TC_DQ + cg * 32 + qd * 8) =
                    make_uint4(tile[rr][4 * qd], tile[rr][4 * qd + 1], tile[rr][4 * qd + 2], tile[rr][4 * qd + 3]);
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
    cudaError_t e = launch_dependent(paged_mla_decode_tc, grid, dim3(TC_THREADS), TC_SMEM, s, tm, p);
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    return launch_dependent(paged_mla_merge_tc, dim3(TC_DQ / 32, p.head_tiles * 2, p.batch), dim3(TC_M), 0, s, p);
}

}  // namespace kvp
