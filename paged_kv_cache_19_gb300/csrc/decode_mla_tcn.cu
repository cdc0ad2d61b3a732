// decode_mla_tcn.cu -- absorbed multi-head latent attention on the 5th-generation
// tensor cores (tcgen05) for narrow head tiles: 16 query heads per tile, as when a
// layer's heads are split over several GPUs (xuewyang.github.io/posts/kv, "MLA:
// how does decode get full-size keys and values back?": every head scores the
// shared cached vector -- 512 latent + 64 rotary-key numbers -- and averages its
// latent part).
//
// With 16 heads the work per cached byte is small (about 30 flop/byte), so the
// kernel is meant to stream the cache at HBM speed; a tcgen05 MMA costs a fixed
// ~50 cycles whatever its shape up to N = 64 (measured on GB300), so the shapes
// are chosen for few instructions per token:
//   * scores S[16 heads x 64 tokens] = Q . C^T: an M = 128 MMA whose rows 0-15
//     (tensor-memory lanes 0-15) are the tile's heads, the other rows never read --
//     A = the queries (latent part in tensor memory, rotary part in shared memory),
//     B = the stage's nine K-major pieces -- 36
//     MMAs of K = 16 per block.  (An M = 64 form costs the same per MMA, but
//     alternating it with the M = 128 output MMAs left ~700 idle cycles at every
//     switch in a trace of this kernel on GB300.)
//   * output O^T[512 latent x 16 heads] += C^T . P^T: four M = 128 tiles of the
//     latent numbers, A = two pieces of the stage read MN-major (a token's latent
//     numbers are contiguous), B = the probabilities P^T[16 x 64] in shared
//     memory -- 16 MMAs of K = 16 per block.
// About 3,100 cycles of MMA issue per 72 KB block: below the ~3,400 cycles an SM's
// share of the HBM bandwidth needs for it.
//
// Persistent, one CTA per SM (224 KB of shared memory, all 512 tensor-memory columns);
// the units (head tile, sequence, block) are cut into one equal contiguous range
// per CTA (mla_partition.cuh), a sequence cut by a range boundary leaving fp32
// partials merged by paged_mla_merge_tcn.  192 threads:
//   * warp 4 walks the range's segments, hands each to the other roles through a
//     4-slot ring, prefetches its queries into L2 and streams its 64-token blocks
//     with nine TMA loads each (one per 128-byte piece, 128-byte swizzle) into 3
//     stages of 72 KB;
//   * warp 5 (one thread) issues the MMAs in a fixed order -- the scores of block g
//     (two score buffers in tensor memory), then the output update of block g - 1 --
//     so that the scores of a block run while the softmax of the one before does;
//   * warp 0, lanes 0-15 (head h = lane h): the online softmax
//     over each stage's 64 scores in registers, P^T row h written to shared memory
//     (two buffers); the whole warp loads the next segment's queries into tensor
//     memory (lanes 16-31 fetch the second half of each row and pass it down);
//   * warps 0-3: each stage, a barrier at which warp 0 publishes whether the output
//     is to be rescaled (the running max grew by more than 2^8 -- until then the
//     older max stays the reference, exact since the final division uses the sum
//     taken against the same reference) and whether the block has tokens past the
//     cache (their value rows are zeroed: 0 * NaN must not reach the sums); at the
//     end of a segment each warp normalises and writes its quarter of the latent
//     rows.
//   * tensor memory: the queries' latent numbers [0, 256), two score buffers [256,
//     384), output tiles at 384, 416, 448, 480 (16 columns each); the queries' 64
//     rotary numbers sit in shared memory.
//   * paged_mla_decode_step (the STEP instantiation, 224 threads): warp 6 walks the
//     same partition and writes the new vector of each sequence whose last block lies in
//     the range into that block; warp 4 waits on an mbarrier for those writes before it
//     loads such a block.
// Every wait is bounded; a late barrier sets KV_DEVERR_TIMEOUT and every role leaves
// its loop, waits (bounded) for its copies and MMAs in flight, and the CTA frees its
// tensor memory before it exits.
#include "append_row.cuh"
#include "decode_common.cuh"
#include "kernels.h"
#include "mla_partition.cuh"
#include "tcgen05.cuh"

namespace kvp {

namespace {

constexpr int TN_H = MLA_TCN_HEADS;             // heads per tile
constexpr int TN_TOK = 64;                      // tokens per stage (one block)
constexpr int TN_NSTAGE = 3;
constexpr int TN_PIECE = TN_TOK * 128;          // one 64-number piece of 64 tokens
constexpr int TN_NPIECE = MLA_DK / 64;          // 9
constexpr int TN_STAGE = TN_NPIECE * TN_PIECE;  // 73,728 bytes
constexpr int TN_PBUF = TN_H * 128;             // P^T: a 128-byte row of 64 bf16 per head
constexpr int TN_THREADS = 192;                 // warps 0-3 softmax / epilogue, 4 loads, 5 MMA
constexpr int TN_THREADS_STEP = 224;            // + warp 6: the step's new vectors
constexpr int TN_EPI = 128;                     // threads of warps 0-3
// tensor memory: the queries' 512 latent numbers [0, 256), two score buffers [256, 320)
// and [320, 384), output tiles at 384, 416, 448, 480 (16 columns each)
constexpr uint32_t TN_Q = 0, TN_S = 256, TN_O = 384, TN_COLS = 512;
// shared memory: the queries' 64 rotary numbers (16 rows of 128 bytes, K-major,
// 128-byte swizzle) lead, the A operand of the rotary score MMAs, whose rows 16-127 fall
// on the first stage (read, never used)
constexpr int TN_QR = 2048;
constexpr uint32_t IDESC_S = tc_idesc_bf16(128, TN_TOK, 0, 0);
constexpr uint32_t IDESC_O = tc_idesc_bf16(128, TN_H, 1, 0);
constexpr float RESCALE_LOG2 = 8.f;
constexpr int TN_CTL = 1024;
constexpr int TN_SMEM = 1024 + TN_QR + TN_NSTAGE * TN_STAGE + 2 * TN_PBUF + TN_CTL;
constexpr int TN_NITEM = 4;
static_assert(TN_SMEM <= 227 * 1024, "one CTA per SM");
static_assert(TN_Q + MLA_DV / 2 <= TN_S && TN_S + 2 * TN_TOK <= TN_O && TN_O + 3 * 32 + TN_H <= TN_COLS,
              "tensor-memory columns");
static_assert(TN_QR + TN_STAGE >= 128 * 128, "rows 16-127 of the rotary A operand stay in the stages");
static_assert(TN_H == 16, "heads are lanes 0-15: warp 0 holds their scores");

struct TnCtl {
    uint64_t kv_full[TN_NSTAGE];                    // the stage's nine pieces landed
    uint64_t kv_empty[TN_NSTAGE];                   // its output update is done
    uint64_t q_full, o_full, o_free, mma_done;
    uint64_t s_full[2], s_free[2];                  // the two score buffers
    uint64_t p_full[2], p_free[2];
    uint64_t item_full[TN_NITEM], item_empty[TN_NITEM];
    uint32_t tmem_base;
    int stage_blk[TN_NSTAGE];
    int abort_flag;
    int flags[2];                                   // per stage (two in turn): 1 rescale the
                                                    // output, 2 tokens past the cache; >> 2: valid tokens
    MlaSegment items[TN_NITEM];
    float fac[TN_H];                                // per-head factors of a rescale
    float lsum[TN_H], mref[TN_H];                   // per-head (sum, max) at a segment's end
    uint64_t step_done;                             // paged_mla_decode_step: new vectors written
};
static_assert(sizeof(TnCtl) <= TN_CTL, "control block");

// One score MMA of S[128 x 64] = Q . C^T (rows 0-15 are the heads), slice ks of the 36
// (16 numbers each): slices 0-31 are the latent numbers, A = the queries in tensor memory
// (8 columns per slice), slices 32-35 the rotary key, A = the rotary queries in shared
// memory; B = the matching piece of the stage, K-major, advanced 32 bytes per slice.
__device__ __forceinline__ void score_mma(uint32_t d, uint32_t tbase, uint64_t st0, uint64_t qr0, int ks)
{
    const uint64_t b = st0 + static_cast<uint64_t>(((ks >> 2) * TN_PIECE + (ks & 3) * 32) >> 4);
    if (ks < 32)
        tc_mma_ts(d, tbase + TN_Q + ks * 8, b, IDESC_S, ks > 0);
    else
        tc_mma_ss(d, qr0 + static_cast<uint64_t>(((ks & 3) * 32) >> 4), b, IDESC_S, true);
}

// One output MMA: O^T[128 i .. 128 i + 127, 16 heads] += C^T . P^T over tokens 16 kk ..
// 16 kk + 15 -- A = pieces 2i and 2i + 1 read MN-major (64-number atoms one piece
// apart, 8-token groups 1 KB apart), B = P^T, K-major.
__device__ __forceinline__ void output_mma(uint32_t tbase, uint32_t stage_addr, uint64_t p0, int i, int kk,
                                           bool first)
{
    const uint64_t a = tc_smem_desc(stage_addr + 2 * i * TN_PIECE, TN_PIECE, 1024) +
                       static_cast<uint64_t>((kk * 2048) >> 4);
    tc_mma_ss(tbase + TN_O + 32 * i, a, p0 + static_cast<uint64_t>((kk * 32) >> 4), IDESC_O,
              !(first && kk == 0));
}

__device__ __forceinline__ void issue_scores(uint32_t tbase, uint32_t sbuf, uint32_t stage_addr, uint32_t qr_addr)
{
    const uint64_t st0 = tc_smem_desc(stage_addr, 16, 1024), qr0 = tc_smem_desc(qr_addr, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < TN_NPIECE * 4; ++ks) score_mma(tbase + sbuf, tbase, st0, qr0, ks);
}

__device__ __forceinline__ void issue_output(uint32_t tbase, uint32_t stage_addr, uint32_t p_addr, bool first)
{
    const uint64_t p0 = tc_smem_desc(p_addr, 16, 1024);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int kk = 0; kk < TN_TOK / 16; ++kk) output_mma(tbase, stage_addr, p0, i, kk, first);
}

// The MMA thread: the output update of stage go (segment ko; first / last: its place in
// the segment) once its probabilities are written -- and, for a segment's first stage,
// once the previous segment's output has been read.  Frees the stage's slot and the
// probabilities' buffer; after a segment's last stage, hands the output to the epilogue.
__device__ __forceinline__ bool mma_output_stage(TnCtl* ctl, uint32_t tbase, uint8_t* stages, uint8_t* pbuf, int go,
                                                 int ko, bool first, bool last)
{
    bool ok = mbar_wait_bounded(smem_u32(&ctl->p_full[go & 1]), static_cast<uint32_t>(go >> 1) & 1u);
    if (ok && first && ko >= 1) ok = mbar_wait_bounded(smem_u32(&ctl->o_free), static_cast<uint32_t>(ko - 1) & 1u);
    if (!ok) return false;
    tc_fence_after();
    issue_output(tbase, smem_u32(stages + (go % TN_NSTAGE) * TN_STAGE), smem_u32(pbuf + (go & 1) * TN_PBUF), first);
    tc_commit(smem_u32(&ctl->kv_empty[go % TN_NSTAGE]));
    tc_commit(smem_u32(&ctl->p_free[go & 1]));
    if (last) tc_commit(smem_u32(&ctl->o_full));
    return true;
}

// Warp 0: the queries of heads ht * 16 + 0..15 of sequence b -- the 512 latent numbers
// into tensor-memory lanes 0-15, columns [0, 256) (128-byte chunk j of a row -> columns
// 32 j .. 32 j + 31), the 64 rotary numbers into the shared-memory rows at qr (row h,
// 16-byte chunk c at (c ^ (h & 7))).  Lane h fetches chunks 0-4 of head h, lane h + 16
// chunks 5-8 (5-7 passed down by shuffles; lanes 16-31 store into tensor-memory lanes
// 16-31, which no result is read from), in two rounds of at most three chunks per lane
// (one round would spill registers).  Rows past q_heads are zero.
__device__ __forceinline__ void load_queries(const MlaParams& p, int b, int ht, uint32_t lrow, uint32_t qr,
                                             int lane)
{
    const int h = lane & 15, hi = lane >> 4;
    const int head = ht * TN_H + h;
    const bool valid = head < p.q_heads;
    const uint4* row = reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.q_heads + (valid ? head : 0)) * MLA_DK);
    // round 0: lanes 0-15 chunks 0-2, lanes 16-31 chunks 5-7; round 1: chunks 3-4 and 8
#pragma unroll
    for (int round = 0; round < 2; ++round) {
        const int nlo = round == 0 ? 3 : 2;         // chunks of lanes 0-15 this round
        const int nhi = round == 0 ? 3 : 1;         // chunks of lanes 16-31
        const int c_lo = round == 0 ? 0 : 3, c_hi = round == 0 ? 5 : 8;
        uint32_t r[3][32];
#pragma unroll
        for (int j = 0; j < 3; ++j)
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                if (valid && j < (hi ? nhi : nlo)) x = __ldg(row + ((hi ? c_hi : c_lo) + j) * 8 + v);
                r[j][4 * v] = x.x;
                r[j][4 * v + 1] = x.y;
                r[j][4 * v + 2] = x.z;
                r[j][4 * v + 3] = x.w;
            }
#pragma unroll
        for (int j = 0; j < 3; ++j)
            if (j < nlo) tc_st32(lrow + TN_Q + 32 * (c_lo + j), r[j]);
        if (round == 0) {
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                uint32_t x[32];
#pragma unroll
                for (int v = 0; v < 32; ++v) x[v] = __shfl_down_sync(FULL_MASK, r[j][v], 16);
                tc_st32(lrow + TN_Q + 32 * (c_hi + j), x);
            }
        } else if (hi) {
            // the rotary chunk: lane h + 16 writes row h
#pragma unroll
            for (int c = 0; c < 8; ++c)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(qr + h * 128 + ((c ^ (h & 7)) << 4)),
                             "r"(r[0][4 * c]), "r"(r[0][4 * c + 1]), "r"(r[0][4 * c + 2]), "r"(r[0][4 * c + 3])
                             : "memory");
        }
    }
    fence_proxy_async_smem();
    tc_wait_st();
}

}  // namespace

// STEP: paged_mla_decode_step (p.kv_new set), whose new vectors a seventh warp writes.
template <bool STEP>
__global__ void __launch_bounds__(STEP ? TN_THREADS_STEP : TN_THREADS, 1)
paged_mla_decode_tcn(const __grid_constant__ CUtensorMap tmp, const MlaParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem + TN_QR;
    uint8_t* pbuf = stages + TN_NSTAGE * TN_STAGE;
    TnCtl* ctl = reinterpret_cast<TnCtl*>(pbuf + 2 * TN_PBUF);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int* abort_flag = &ctl->abort_flag;

    if (tid == 0) {
        for (int i = 0; i < TN_NSTAGE; ++i) {
            mbar_init(smem_u32(&ctl->kv_full[i]), 1);
            mbar_init(smem_u32(&ctl->kv_empty[i]), 1);
        }
        for (int i = 0; i < TN_NITEM; ++i) {
            mbar_init(smem_u32(&ctl->item_full[i]), 1);
            mbar_init(smem_u32(&ctl->item_empty[i]), 5);   // the MMA thread + warps 0-3
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&ctl->p_full[i]), 1);
            mbar_init(smem_u32(&ctl->p_free[i]), 1);
            mbar_init(smem_u32(&ctl->s_full[i]), 1);
            mbar_init(smem_u32(&ctl->s_free[i]), 1);
        }
        mbar_init(smem_u32(&ctl->q_full), 1);
        mbar_init(smem_u32(&ctl->o_full), 1);
        mbar_init(smem_u32(&ctl->o_free), 4);
        mbar_init(smem_u32(&ctl->mma_done), 1);
        mbar_init(smem_u32(&ctl->step_done), 32);   // the lanes of warp 6 (STEP)
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) tc_alloc(smem_u32(&ctl->tmem_base), TN_COLS);
    grid_dependency_wait();                     // inputs of the preceding kernel are ready
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ctl->tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------------ segments and loads
        MlaPartition<TN_TOK, MLA_SEG_PAD_NARROW> part;
        part.init(p, p.head_tiles, lane);
        if (lane == 0) {
            prefetch_tensormap(&tmp);
            int k = 0;                              // segments handed on
            int g = 0;                              // stages issued (all segments)
            bool ok = true;
            bool step_written = false;              // paged_mla_decode_step: waited for lanes 1-31
            for (;;) {
                const MlaSegment it = *abort_flag ? MlaSegment{0, 0, 0, -1, 0, 0, 0} : part.next();
                const bool last = it.n < 0;
                if (!last) {
                    const int nhq = min(TN_H, p.q_heads - it.outer * TN_H);
                    prefetch_l2_bulk(p.q + (static_cast<size_t>(it.b) * p.q_heads + it.outer * TN_H) * MLA_DK,
                                     static_cast<uint32_t>(nhq) * MLA_DK * 2);
                }
                const int slot = k % TN_NITEM;
                if (!mbar_wait_bounded(smem_u32(&ctl->item_empty[slot]),
                                       (static_cast<uint32_t>(k / TN_NITEM) & 1u) ^ 1u)) {
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
                const int step_s = STEP ? mla_step_block(p, it.b, TN_TOK) - it.blk0 : -1;
                for (int s = 0; s < it.n; ++s, ++g) {
                    const int st = g % TN_NSTAGE;
                    int bid = next_blk;
                    if (s + 1 < it.n) next_blk = __ldg(trow + s + 1);
                    if (bid < 0 || bid >= p.num_blocks) {
                        atomicOr(p.err, KV_DEVERR_BLOCK_ID);
                        bid = -1;
                    }
                    if (STEP && s == step_s && bid >= 0 && !step_written) {   // warp 6 wrote it?
                        if (!mbar_wait_bounded(smem_u32(&ctl->step_done), 0u)) {
                            ok = false;
                            break;
                        }
                        step_written = true;
                    }
                    if (!mbar_wait_bounded(smem_u32(&ctl->kv_empty[st]),
                                           (static_cast<uint32_t>(g / TN_NSTAGE) & 1u) ^ 1u) ||
                        *abort_flag) {
                        ok = false;
                        break;
                    }
                    ctl->stage_blk[st] = bid;
                    const uint32_t fb = smem_u32(&ctl->kv_full[st]);
                    if (bid >= 0) {
                        const uint32_t dst = smem_u32(stages + st * TN_STAGE);
                        mbar_arrive_expect_tx(fb, TN_STAGE);
                        for (int j = 0; j < TN_NPIECE; ++j)
                            tma_load_5d(dst + j * TN_PIECE, &tmp, 0, j, 0, 0, bid, fb);
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
            for (int j = max(0, g - TN_NSTAGE); j < g; ++j)
                if (!mbar_wait_bounded(smem_u32(&ctl->kv_full[j % TN_NSTAGE]),
                                       static_cast<uint32_t>(j / TN_NSTAGE) & 1u))
                    break;
        }
        grid_dependents_launch();
    } else if (STEP && warp == 6) {
        // ------------------------------------------------------------ the step's new vectors
        // The same partition, walked beside the producer: every block of the range that holds
        // a sequence's new vector gets it before the producer loads that block.
        MlaPartition<TN_TOK, MLA_SEG_PAD_NARROW> part;
        part.init(p, p.head_tiles, lane, false);
        part.write_step_rows(smem_u32(&ctl->step_done), lane, 32);
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            // A fixed order: the scores of stage g, then the output update of stage g - 1,
            // so that the scores of the next block run while the softmax of the last one
            // does, and each wait blocks (try_wait) rather than polls.  At a segment
            // boundary the last output update of the old segment comes first.
            const uint32_t qr = smem_u32(smem);
            bool ok = true;
            int g = 0;                              // stages scored (all segments)
            int pk = -1, pfirst = 0, plast = 0;     // the stage whose output update is due, its
                                                    // segment, first / last in the segment
            for (int k = 0; ok; ++k) {
                const int slot = k % TN_NITEM;
                ok = mbar_wait_bounded(smem_u32(&ctl->item_full[slot]), static_cast<uint32_t>(k / TN_NITEM) & 1u);
                if (!ok) break;
                const int n = ctl->items[slot].n;
                mbar_arrive(smem_u32(&ctl->item_empty[slot]));
                if (n < 0) break;
                for (int s = 0; ok && s < n; ++s, ++g) {
                    const int st = g % TN_NSTAGE;
                    if (s == 0 && pk >= 0) {
                        // the previous segment's last output update goes first: it does not
                        // wait for this segment's queries, and its epilogue can then run
                        // while they load
                        ok = mma_output_stage(ctl, tbase, stages, pbuf, g - 1, pk, pfirst, plast);
                        pk = -1;
                        if (!ok) break;
                    }
                    ok = mbar_wait_bounded(smem_u32(&ctl->kv_full[st]), static_cast<uint32_t>(g / TN_NSTAGE) & 1u);
                    if (ok && g >= 2)
                        ok = mbar_wait_bounded(smem_u32(&ctl->s_free[g & 1]), static_cast<uint32_t>((g - 2) >> 1) & 1u);
                    if (ok && s == 0) ok = mbar_wait_bounded(smem_u32(&ctl->q_full), static_cast<uint32_t>(k) & 1u);
                    if (!ok || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_scores(tbase, TN_S + TN_TOK * (g & 1), smem_u32(stages + st * TN_STAGE), qr);
                    tc_commit(smem_u32(&ctl->s_full[g & 1]));
                    if (pk >= 0) ok = mma_output_stage(ctl, tbase, stages, pbuf, g - 1, pk, pfirst, plast);
                    pk = k;
                    pfirst = s == 0;
                    plast = s == n - 1;
                }
            }
            if (ok && pk >= 0) ok = mma_output_stage(ctl, tbase, stages, pbuf, g - 1, pk, pfirst, plast);
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
        const uint32_t lrow = tbase + (static_cast<uint32_t>(warp * 32) << 16);
        const int h = lane & 15;                    // warp 0: the head of this lane
        const bool soft = warp == 0 && lane < TN_H;
        const float sl2 = p.scale_log2;
        bool failed = false;
        int g = 0;                                  // stages processed (all segments)
        MlaSegment item{};
        {
            const bool ok = all_ok(mbar_wait_bounded(smem_u32(&ctl->item_full[0]), 0));
            item = ctl->items[0];
            failed = !ok;
        }
        if (warp == 0 && !failed && item.n >= 0) {
            load_queries(p, item.b, item.outer, lrow, smem_u32(smem), lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->q_full));
        }
        // every warp of the four reaches this barrier once per segment, failed or not: it is
        // the one place they leave the loop together
        for (int k = 0;; ++k) {
            const int slot = k % TN_NITEM;
            if (k > 0 && !failed) {
                const bool ok = all_ok(mbar_wait_bounded(smem_u32(&ctl->item_full[slot]),
                                                         static_cast<uint32_t>(k / TN_NITEM) & 1u));
                item = ctl->items[slot];
                if (!ok) failed = true;
            }
            __syncwarp();
            if (lane == 0 && !failed) mbar_arrive(smem_u32(&ctl->item_empty[slot]));
            if (named_barrier_or(1, TN_EPI, failed || item.n < 0 || *abort_flag != 0)) {
                failed = failed || *abort_flag != 0;
                break;
            }
            const int b = item.b, ht = item.outer, split = item.split, n = item.n, ctx = item.ctx;
            const int blk0 = item.blk0, nsplit = item.nsplit;
            const int nh = min(TN_H, p.q_heads - ht * TN_H);
            const size_t row0 = static_cast<size_t>(b) * p.q_heads + ht * TN_H;
            float m_ref = -INFINITY, l = 0.f;
            for (int s = 0; s < n; ++s) {
                const int gs = g + s;
                const int st = gs % TN_NSTAGE;
                float sv[64];
                int nvalid = 0;
                bool ok = true;
                if (warp == 0) {
                    ok = mbar_wait_bounded(smem_u32(&ctl->kv_full[st]), static_cast<uint32_t>(gs / TN_NSTAGE) & 1u);
                    if (ok) ok = mbar_wait_bounded(smem_u32(&ctl->s_full[gs & 1]), static_cast<uint32_t>(gs >> 1) & 1u);
                    ok = all_ok(ok);
                    const int blk = ok ? ctl->stage_blk[st] : -1;
                    nvalid = blk < 0 ? 0 : min(TN_TOK, ctx - (blk0 + s) * TN_TOK);
                    if (ok) {
                        tc_fence_after();
                        uint32_t r[32];
                        tc_ld32(lrow + TN_S + TN_TOK * (gs & 1), r);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(r[j]);
                        tc_ld32(lrow + TN_S + TN_TOK * (gs & 1) + 32, r);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) sv[32 + j] = __uint_as_float(r[j]);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[gs & 1]));
                    }
                    if (nvalid < TN_TOK) {
#pragma unroll
                        for (int j = 0; j < 64; ++j)
                            if (j >= nvalid) sv[j] = -INFINITY;   // not cached (may be NaN)
                    }
                    float mx = sv[0];
#pragma unroll
                    for (int j = 1; j < 64; ++j) mx = fmaxf(mx, sv[j]);
                    const float m_new = fmaxf(m_ref, mx * sl2);
                    float f = 1.f;
                    if (m_ref == -INFINITY) {
                        m_ref = m_new;              // nothing accumulated yet
                    } else if (m_new > m_ref + RESCALE_LOG2) {
                        f = fast_exp2(m_ref - m_new);
                        l *= f;
                        m_ref = m_new;
                    }
                    const bool any = __any_sync(FULL_MASK, soft && f != 1.f);
                    if (lane < TN_H) ctl->fac[h] = f;
                    if (lane == 0)
                        ctl->flags[gs & 1] = (any ? 1 : 0) | (nvalid < TN_TOK ? 2 : 0) | (max(0, nvalid) << 2);
                }
                // warp 0 publishes the stage's flags; a failure anywhere ends the loop here
                if (named_barrier_or(1, TN_EPI, failed || !ok || *abort_flag != 0)) {
                    failed = true;
                    break;
                }
                const int flags = ctl->flags[gs & 1];
                if (flags & 1) {
                    // scale the output columns by their heads' factors once the updates of
                    // the earlier stages are done
                    const bool w = all_ok(mbar_wait_bounded(smem_u32(&ctl->p_free[(gs - 1) & 1]),
                                                            static_cast<uint32_t>((gs - 1) >> 1) & 1u));
                    if (!w) failed = true;
                    if (w) {
                        tc_fence_after();
                        float fh[TN_H];
#pragma unroll
                        for (int j = 0; j < TN_H; ++j) fh[j] = ctl->fac[j];
#pragma unroll 1
                        for (int i = 0; i < 4; ++i) {
                            uint32_t r[32];
                            tc_ld32(lrow + TN_O + 32 * i, r);
                            tc_wait_ld();
                            uint32_t x[16];
#pragma unroll
                            for (int j = 0; j < TN_H; ++j) x[j] = __float_as_uint(__uint_as_float(r[j]) * fh[j]);
                            tc_st16(lrow + TN_O + 32 * i, x);
                        }
                        tc_wait_st();
                        tc_fence_before();
                    }
                }
                if (flags & 2) {
                    // value rows of tokens past the cache (or of a skipped block) are zeroed
                    // (the stage's scores, which read them too, are complete)
                    const int v0 = max(0, flags >> 2);
                    uint8_t* sp = stages + st * TN_STAGE;
                    for (int i = tid; i < (TN_TOK - v0) * 64; i += TN_EPI) {
                        const int row = v0 + (i >> 6);
                        const int pc = (i >> 3) & 7;
                        const int ch = i & 7;
                        *reinterpret_cast<uint4*>(sp + pc * TN_PIECE + row * 128 + (ch << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                if (flags != 0 && named_barrier_or(1, TN_EPI, failed)) {
                    failed = true;
                    break;
                }
                if (warp == 0) {
                    // probabilities (bf16) of this thread's head: P^T row h, 128-byte swizzle
                    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                    uint32_t pk[32];
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float p0 = fast_exp2(fmaf(sv[2 * j], sl2, -m_use));
                        const float p1 = fast_exp2(fmaf(sv[2 * j + 1], sl2, -m_use));
                        ls[j & 3] += p0 + p1;
                        pk[j] = pack_bf16x2(p0, p1);
                    }
                    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    bool w = true;
                    if (gs >= 2)
                        w = mbar_wait_bounded(smem_u32(&ctl->p_free[gs & 1]), static_cast<uint32_t>((gs - 2) >> 1) & 1u);
                    w = all_ok(w);
                    if (!w) {
                        failed = true;
                    } else {
                        if (lane < TN_H) {
                            const uint32_t row = smem_u32(pbuf + (gs & 1) * TN_PBUF) + h * 128;
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c ^ (h & 7)) << 4)),
                                             "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                                             : "memory");
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&ctl->p_full[gs & 1]));
                    }
                }
            }
            if (warp == 0 && lane < TN_H) {
                ctl->lsum[h] = l;
                ctl->mref[h] = m_ref;
            }
            if (named_barrier_or(1, TN_EPI, failed)) {
                failed = true;
                break;
            }
            // ---- warp 0 loads the next segment's queries first (its scores may then start
            // while this segment's output is written); each warp then writes its quarter
            // of the output.  A failure is passed on at the next segment's barrier.
            if (warp == 0) {
                const int nslot = (k + 1) % TN_NITEM;
                const bool ok = all_ok(mbar_wait_bounded(smem_u32(&ctl->item_full[nslot]),
                                                         static_cast<uint32_t>((k + 1) / TN_NITEM) & 1u));
                if (!ok) {
                    failed = true;
                } else {
                    const MlaSegment nx = ctl->items[nslot];
                    if (nx.n >= 0) {
                        load_queries(p, nx.b, nx.outer, lrow, smem_u32(smem), lane);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&ctl->q_full));
                    }
                }
            }
            if (!failed && !all_ok(mbar_wait_bounded(smem_u32(&ctl->o_full), static_cast<uint32_t>(k) & 1u)))
                failed = true;
            if (failed) continue;                   // leaves at the next segment's barrier
            tc_fence_after();
            // ---- epilogue: latent rows 128 i + 32 warp + lane of the four tiles, 16 heads
            // each; a whole sequence's output in bf16, a piece of a cut one as its fp32
            // partial [piece][head][512] with (max, sum) per head
            const bool whole = nsplit == 1;
            const size_t piece = (static_cast<size_t>(b) * p.head_tiles + ht) * p.max_splits + split;
            float inv[TN_H];
#pragma unroll
            for (int j = 0; j < TN_H; ++j) {
                const float lj = ctl->lsum[j];
                inv[j] = lj > 0.f ? 1.f / lj : 0.f;
            }
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                uint32_t r[32];
                tc_ld32(lrow + TN_O + 32 * i, r);
                tc_wait_ld();
                const int d = 128 * i + 32 * warp + lane;
                if (whole) {
                    uint16_t* dst = p.out + row0 * MLA_DV + d;
#pragma unroll
                    for (int j = 0; j < TN_H; ++j)
                        if (j < nh) dst[static_cast<size_t>(j) * MLA_DV] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(r[j]) * inv[j], 0.f));
                } else {
                    // fp16: averages of cached values, well inside its range, 11 significant
                    // bits against the output's 8
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.part_o) + piece * (TN_H * MLA_DV) + d;
#pragma unroll
                    for (int j = 0; j < TN_H; ++j)
                        dst[j * MLA_DV] = static_cast<uint16_t>(pack_f16x2(__uint_as_float(r[j]) * inv[j], 0.f));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->o_free));
            if (warp == 0 && lane < TN_H) {
                const float mj = ctl->mref[h], lj = ctl->lsum[h];
                if (!whole)
                    reinterpret_cast<float2*>(p.part_ml)[piece * TN_H + h] = make_float2(mj, lj);
                else if (p.lse != nullptr && h < nh)
                    p.lse[row0 + h] = lse_from(mj, lj);
            }
            if (tid == 0 && p.tickets != nullptr) p.tickets[static_cast<size_t>(b) * p.head_tiles + ht] = nsplit;
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
    if (warp == 5) {
        tc_fence_after();
        tc_dealloc(tbase, TN_COLS);
    }
}

// Merge of the pieces of every cut sequence: CTA (sequence, head tile, quarter of the
// latent numbers), thread (head, 8 numbers).  The pieces' (max, sum) pairs give the
// weights w_j = l_j 2^(m_j - M) of the standard log-sum-exp merge; out = sum_j w_j o_j /
// sum_j w_j.  Four pieces per round, their loads issued together.
__global__ void __launch_bounds__(256)
paged_mla_merge_tcn(const MlaParams p)
{
    // The next kernel may start launching now (its CTAs set up beside this grid's small
    // CTAs); it reads nothing before waiting for this grid to complete.
    grid_dependents_launch();
    grid_dependency_wait();
    const int b = blockIdx.x, ht = blockIdx.y, qd = blockIdx.z;
    const int h = threadIdx.x >> 4, cg = threadIdx.x & 15;
    const int ctx = __ldg(p.ctx + b);
    const int nsplit = ctx > 0 ? __ldcg(p.tickets + static_cast<size_t>(b) * p.head_tiles + ht) : 1;
    const int nh = min(TN_H, p.q_heads - ht * TN_H);
    if (nsplit > 1 && h < nh) {
        const size_t piece0 = (static_cast<size_t>(b) * p.head_tiles + ht) * p.max_splits;
        const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + piece0 * TN_H + h;
        const uint4* po = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.part_o) +
                                                         (piece0 * TN_H + h) * MLA_DV + qd * 128 + cg * 8);
        float M = -INFINITY, W = 0.f;
        float acc[8];
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[v] = 0.f;
        for (int j0 = 0; j0 < nsplit; j0 += 4) {
            float2 mj[4];
            float4 x[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const bool in = j0 + i < nsplit;
                const size_t j = static_cast<size_t>(in ? j0 + i : j0);
                mj[i] = in ? __ldcg(ml + j * TN_H) : make_float2(-INFINITY, 0.f);
                const uint4 u = __ldcg(po + j * (TN_H * MLA_DV / 8));
                const float2 a = unpack_f16x2(u.x), bq = unpack_f16x2(u.y), c = unpack_f16x2(u.z),
                             e = unpack_f16x2(u.w);
                x[i][0] = make_float4(a.x, a.y, bq.x, bq.y);
                x[i][1] = make_float4(c.x, c.y, e.x, e.y);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (!(mj[i].y > 0.f)) continue;   // an empty piece: m = -inf, l = 0
                const float m2 = fmaxf(M, mj[i].x);
                const float fo = fast_exp2(M - m2);   // 0 while nothing is accumulated
                const float wj = mj[i].y * fast_exp2(mj[i].x - m2);
                W = W * fo + wj;
                M = m2;
                const float xs[8] = {x[i][0].x, x[i][0].y, x[i][0].z, x[i][0].w,
                                     x[i][1].x, x[i][1].y, x[i][1].z, x[i][1].w};
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[v] = acc[v] * fo + wj * xs[v];
            }
        }
        const float winv = W > 0.f ? 1.f / W : 0.f;
        *reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(b) * p.q_heads + ht * TN_H + h) * MLA_DV + qd * 128 + cg * 8) =
            make_uint4(pack_bf16x2(acc[0] * winv, acc[1] * winv), pack_bf16x2(acc[2] * winv, acc[3] * winv),
                       pack_bf16x2(acc[4] * winv, acc[5] * winv), pack_bf16x2(acc[6] * winv, acc[7] * winv));
        if (p.lse != nullptr && qd == 0 && cg == 0)
            p.lse[static_cast<size_t>(b) * p.q_heads + ht * TN_H + h] = lse_from(M, W);
    }
}

cudaError_t prepare_mla_decode_tcn()
{
    cudaError_t e = cudaFuncSetAttribute(paged_mla_decode_tcn<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, TN_SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(paged_mla_decode_tcn<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TN_SMEM);
}

cudaError_t launch_mla_decode_tcn(dim3 grid, const CUtensorMap& tm, const MlaParams& p,
                                  cudaStream_t s)
{
    cudaError_t e = p.kv_new != nullptr
                        ? launch_dependent(paged_mla_decode_tcn<true>, grid, dim3(TN_THREADS_STEP), TN_SMEM, s, tm, p)
                        : launch_dependent(paged_mla_decode_tcn<false>, grid, dim3(TN_THREADS), TN_SMEM, s, tm, p);
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    return launch_dependent(paged_mla_merge_tcn, dim3(p.batch, p.head_tiles, MLA_DV / 128), dim3(256), 0, s, p);
}

}  // namespace kvp
