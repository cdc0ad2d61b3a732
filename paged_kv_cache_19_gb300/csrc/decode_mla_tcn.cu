// decode_mla_tcn.cu -- absorbed multi-head latent attention on the 5th-generation
// tensor cores (tcgen05) for narrow head tiles: 16 query heads per tile, as when a
// layer's heads are split over several GPUs (xuewyang.github.io/posts/kv, "MLA:
// how does decode get full-size keys and values back?": every head scores the
// shared cached vector -- 512 latent + 64 rotary-key numbers -- and averages its
// latent part).
//
// With 16 heads the work per cached byte is small (about 30 flop/byte), so the
// kernel is meant to stream the cache at HBM speed.  A tcgen05 MMA costs ~46 cycles of
// issue whatever its shape up to N = 64 (measured on GB300), so the shapes are chosen
// for few MMAs per token, with the tokens on the M dimension:
//   * a stage is 32 tokens (half a 64-token pool block) as nine 4 KB pieces, piece
//     j = numbers 64 j .. 64 j + 63 of every token (K-major, 128-byte swizzle);
//   * scores S^T = C . Q^T with M = 128 rows that stack four K-groups of the same 32
//     tokens: rows 32 w .. 32 w + 31 are piece 4 G + w of the stage (consecutive
//     pieces are 4 KB apart, the stride of 8-row groups times four), and the N = 64
//     columns stack the 16 heads four times, column group w holding the queries'
//     piece 4 G + w.  The diagonal blocks (rows 32 w.., columns 16 w..) are the
//     products wanted; the others are computed and never read.  Two such MMAs (G =
//     0, 1) per 16-number slice cover the eight latent pieces: 8 MMAs; the rotary
//     piece takes 4 more (N = 16, rows 96-127 = piece 8 are the ones read);
//   * output O^T[512 latent x 16 heads] += C^T . P^T: four M = 128 tiles of the
//     latent numbers, A = two pieces read MN-major, B = P^T[16 x 32] -- 8 MMAs;
//   so 20 MMAs per 32 tokens.
//   The four K-group partial scores of a token sit in four lane quarters of tensor
//   memory: the softmax warps add them through shared memory.
//
// Persistent, one CTA per SM (about 214 KB of shared memory, 512 tensor-memory columns);
// the units (head tile, sequence, 64-token block) are cut into one equal contiguous
// range per CTA (mla_partition.cuh), a sequence cut by a range boundary leaving fp16
// partials merged by paged_mla_merge_tcn.  512 threads:
//   * warp 4 walks the range's segments, hands each to the other roles through a
//     4-slot ring (prefetching its queries into L2) and streams the 32-token stages,
//     nine TMA loads each, into a ring of 5 stages;
//   * warp 5 (one thread) loads each segment's queries by TMA into shared memory once
//     the scores of the segment before are done, and issues the score MMAs of each stage
//     as soon as it has landed (two score buffers in tensor memory); warp 10 (one thread)
//     issues the output update of each stage as soon as its probabilities are written;
//   * two softmax teams take alternate stages, team 0 = warps 0-3, team 1 = warps 12-15
//     (one warp per tensor-memory lane quarter each).  A team's warps read their quarter's
//     diagonal block of the scores and add the four partials in one shared-memory round,
//     so that warp v holds heads 4 v .. 4 v + 3 (lane = token); a vote decides whether
//     any score exceeds its head's reference by more than 2^8 (the maxima are reduced
//     only then: a lazy rescale, exact since the final division uses the sum taken against
//     the same reference); the warps write the bf16 probabilities P^T, zero the value rows
//     of tokens past the cache (0 * NaN must not reach the sums) and apply a rescale to
//     the team's output.  Each team keeps its own running (max, sum) per head and its own
//     output accumulator, so the teams never wait for each other;
//   * warps 6-9 (the epilogue) merge the two teams' outputs of a segment by log-sum-exp
//     and write them; the output accumulators alternate between two sets per segment,
//     so a segment is written while the next one accumulates;
//   * tensor memory: score buffers at columns 0 and 128 (64 columns + 16 for the rotary
//     part), output sets at 256 and 384, each team's four 16-column tiles 64 apart.
//   * paged_mla_decode_step (the STEP instantiation): warp 11 walks the same partition
//     and writes the new vector of each sequence whose last block lies in the range into
//     that block; warp 4 waits on an mbarrier for those writes before it loads such a
//     block.
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
constexpr int TN_BLK = MLA_TC_BLOCK;            // tokens per pool block (the partition's unit)
constexpr int TN_TOK = 32;                      // tokens per stage
constexpr int TN_NSTAGE = 5;
constexpr int TN_PIECE = TN_TOK * 128;          // one 64-number piece of 32 tokens
constexpr int TN_NPIECE = MLA_DK / 64;          // 9
constexpr int TN_STAGE = TN_NPIECE * TN_PIECE;  // 36,864 bytes
constexpr int TN_QPIECE = TN_H * 128;           // one 64-number piece of the 16 query rows
constexpr int TN_QBUF = TN_NPIECE * TN_QPIECE;  // 18,432 bytes
constexpr int TN_PBUF = TN_H * 128;             // P^T: 128-byte rows, stage parity b in bytes [64 b, 64 b + 64)
constexpr int TN_XBUF = 12 * 32 * 16;           // one team's score partials exchanged between its warps
constexpr int TN_CTL = 2048;
constexpr int TN_THREADS = 512;                 // 0-3, 12-15 softmax; 4 loads; 5, 10 MMA; 6-9 epilogue; 11 step
constexpr int TN_SOFT = 128;                    // threads of a softmax team, of the epilogue
constexpr int TN_NITEM = 4;
constexpr int TN_ITEM_READERS = 14;             // the two MMA threads and twelve warps
// shared memory: the query buffer, the stages, P^T, the exchange buffers, the control block
constexpr int TN_OFF_Q = 0;
constexpr int TN_OFF_ST = TN_OFF_Q + TN_QBUF;
constexpr int TN_OFF_P = TN_OFF_ST + TN_NSTAGE * TN_STAGE;
constexpr int TN_OFF_X = TN_OFF_P + TN_PBUF;
constexpr int TN_OFF_CTL = TN_OFF_X + 2 * TN_XBUF;
constexpr int TN_SMEM = 1024 + TN_OFF_CTL + TN_CTL;
static_assert(TN_SMEM <= 227 * 1024, "one CTA per SM");
static_assert(TN_OFF_ST % 1024 == 0 && TN_STAGE % 1024 == 0 && TN_OFF_P % 1024 == 0 && TN_QBUF % 1024 == 0,
              "128-byte-swizzled operands start on 1 KB boundaries");
// tensor memory: score buffers (64 + 16 columns) at 0 and 128; output set b (segment
// parity), team t at 256 + 128 b + 64 t, tile i 16 i further
constexpr uint32_t TN_S = 0, TN_S_STRIDE = 128, TN_ROPE = 64, TN_O = 256, TN_COLS = 512;
__host__ __device__ constexpr uint32_t tn_obase(int b, int t) { return TN_O + 128 * b + 64 * t; }
static_assert(TN_S + TN_S_STRIDE + TN_ROPE + TN_H <= TN_O && tn_obase(1, 1) + 48 + TN_H <= TN_COLS,
              "tensor-memory columns");
static_assert(TN_H == 16 && TN_TOK == 32, "four 16-head column groups; a lane per token");
constexpr uint32_t IDESC_S = tc_idesc_bf16(128, 4 * TN_H, 0, 0);
constexpr uint32_t IDESC_R = tc_idesc_bf16(128, TN_H, 0, 0);
constexpr uint32_t IDESC_O = tc_idesc_bf16(128, TN_H, 1, 0);
constexpr float RESCALE_LOG2 = 8.f;

struct TnCtl {
    uint64_t kv_full[TN_NSTAGE];                    // the stage's nine pieces landed
    uint64_t kv_empty[TN_NSTAGE];                   // its output update is done
    uint64_t q_full, q_free;                        // the queries landed / their scores done
    uint64_t s_full[2], s_free[2];                  // score buffers (stage parity = team)
    uint64_t p_full[2], p_free[2];                  // P^T halves (stage parity = team)
    uint64_t o_full[2], o_free[2];                  // output sets: segment done / written
    uint64_t ml_full[2];                            // a segment's (max, sum) per head written
    uint64_t item_full[TN_NITEM], item_empty[TN_NITEM];
    uint64_t mma_done[2], step_done;
    uint32_t tmem_base;
    int abort_flag;
    int stage_blk[TN_NSTAGE];
    uint32_t resc[2];                               // per team, byte w: its warp w rescales
    MlaSegment items[TN_NITEM];
    float fac[2][TN_H];                             // per team: per-head factors of a rescale
    float lsum[2][2][TN_H], mref[2][2][TN_H];       // per output set, per team: (sum, max)
};
static_assert(sizeof(TnCtl) <= TN_CTL, "control block");

// Stages of a segment: two per block, one for a sequence's last block when it holds at
// most 32 tokens.
__device__ __forceinline__ int seg_stages(const MlaSegment& it)
{
    const int extra = (it.blk0 + it.n) * TN_BLK - it.ctx;
    return 2 * it.n - (extra >= TN_TOK ? 1 : 0);
}

// Score MMAs of one stage into the score buffer at tensor-memory address d: 8 for the
// latent pieces (two groups of four pieces stacked on M, 16 numbers per MMA) and 4 for
// the rotary piece (rows 96-127 = piece 8 against the rotary queries, N = 16, at d + 64).
// st_k, q_k: K-major descriptors of the stage and of the query buffer; every operand is
// their start moved by a constant (descriptor addresses count 16-byte units), so the
// issuing thread spends no time building descriptors.
__device__ __forceinline__ void issue_scores(uint32_t d, uint64_t st_k, uint64_t q_k)
{
#pragma unroll
    for (int grp = 0; grp < 2; ++grp)
#pragma unroll
        for (int c = 0; c < 4; ++c)
            tc_mma_ss(d, st_k + ((grp * 4 * TN_PIECE + c * 32) >> 4), q_k + ((grp * 4 * TN_QPIECE + c * 32) >> 4),
                      IDESC_S, (grp | c) != 0);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        tc_mma_ss(d + TN_ROPE, st_k + ((5 * TN_PIECE + c * 32) >> 4), q_k + ((8 * TN_QPIECE + c * 32) >> 4), IDESC_R,
                  c != 0);
}

// Output MMAs of one stage: O^T[128 i .. 128 i + 127, 16 heads] += C^T . P^T over tokens
// 16 kk .. 16 kk + 15 -- A = pieces 2i and 2i + 1 read MN-major (st_mn: the stage's
// descriptor with 64-number atoms one piece apart, 8-token groups 1 KB apart), B = the
// stage's half of P^T, K-major (p_k).  first: the team's first stage of the segment.
__device__ __forceinline__ void issue_output(uint32_t obase, uint64_t st_mn, uint64_t p_k, bool first)
{
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int kk = 0; kk < TN_TOK / 16; ++kk)
            tc_mma_ss(obase + 16 * i, st_mn + ((2 * i * TN_PIECE + kk * 2048) >> 4), p_k + ((kk * 32) >> 4), IDESC_O,
                      !(first && kk == 0));
}

// Four floats to / from shared memory (shared-space addresses).
__device__ __forceinline__ void sts_f4(uint32_t addr, const float* v)
{
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3])
                 : "memory");
}

__device__ __forceinline__ void lds_add_f4(uint32_t addr, float* v)
{
    float a, b, c, d;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(a), "=f"(b), "=f"(c), "=f"(d) : "r"(addr) : "memory");
    v[0] += a;
    v[1] += b;
    v[2] += c;
    v[3] += d;
}

__device__ __forceinline__ float pick4(const float* v, int i)
{
    return i == 0 ? v[0] : i == 1 ? v[1] : i == 2 ? v[2] : v[3];
}

}  // namespace

// STEP: paged_mla_decode_step (p.kv_new set), whose new vectors warp 11 writes.
template <bool STEP>
__global__ void __launch_bounds__(TN_THREADS, 1)
paged_mla_decode_tcn(const __grid_constant__ CUtensorMap tmp, const __grid_constant__ CUtensorMap tmq,
                     const MlaParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* qbuf = smem + TN_OFF_Q;
    uint8_t* stages = smem + TN_OFF_ST;
    uint8_t* pbuf = smem + TN_OFF_P;
    uint8_t* xbufs = smem + TN_OFF_X;
    TnCtl* ctl = reinterpret_cast<TnCtl*>(smem + TN_OFF_CTL);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    volatile int* abort_flag = &ctl->abort_flag;
    // query rows per TMA box: 16, or all heads when there are fewer (the other rows of
    // the buffer are zeroed once here)
    const int q_rows = min(TN_H, p.q_heads);

    if (tid == 0) {
        for (int i = 0; i < TN_NSTAGE; ++i) {
            mbar_init(smem_u32(&ctl->kv_full[i]), 1);
            mbar_init(smem_u32(&ctl->kv_empty[i]), 1);
        }
        for (int i = 0; i < TN_NITEM; ++i) {
            mbar_init(smem_u32(&ctl->item_full[i]), 1);
            mbar_init(smem_u32(&ctl->item_empty[i]), TN_ITEM_READERS);
        }
        mbar_init(smem_u32(&ctl->q_full), 1);
        mbar_init(smem_u32(&ctl->q_free), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&ctl->s_full[i]), 1);
            mbar_init(smem_u32(&ctl->s_free[i]), 4);
            mbar_init(smem_u32(&ctl->p_full[i]), 4);
            mbar_init(smem_u32(&ctl->p_free[i]), 1);
            mbar_init(smem_u32(&ctl->o_full[i]), 1);
            mbar_init(smem_u32(&ctl->o_free[i]), 4);
            mbar_init(smem_u32(&ctl->ml_full[i]), 8);
            mbar_init(smem_u32(&ctl->mma_done[i]), 1);
        }
        mbar_init(smem_u32(&ctl->step_done), 32);   // the lanes of warp 11 (STEP)
        ctl->abort_flag = 0;
        fence_mbar_init();
    }
    if (q_rows < TN_H) {
        for (int i = tid; i < TN_QBUF / 16; i += blockDim.x)
            reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    if (warp == 5) tc_alloc(smem_u32(&ctl->tmem_base), TN_COLS);
    grid_dependency_wait();                     // inputs of the preceding kernel are ready
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = ctl->tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------------ segments and loads
        MlaPartition<TN_BLK, MLA_SEG_PAD_NARROW> part;
        part.init(p, p.head_tiles, lane);
        if (lane == 0) {
            prefetch_tensormap(&tmp);
            int k = 0;                              // segments handed on
            int g = 0;                              // stages issued (all segments)
            bool ok = true;
            bool step_written = false;              // paged_mla_decode_step: waited for warp 11
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
                const int ns = seg_stages(it);
                const int32_t* trow = p.tables + static_cast<size_t>(it.b) * p.max_blocks + it.blk0;
                int next_bid = __ldg(trow);         // block id read one block ahead
                int bid = -1;
                // paged_mla_decode_step: the segment's block that holds the new vector
                const int step_j = STEP ? mla_step_block(p, it.b, TN_BLK) - it.blk0 : -1;
                for (int s = 0; s < ns; ++s, ++g) {
                    const int st = g % TN_NSTAGE;
                    if ((s & 1) == 0) {
                        bid = next_bid;
                        if ((s >> 1) + 1 < it.n) next_bid = __ldg(trow + (s >> 1) + 1);
                        if (bid < 0 || bid >= p.num_blocks) {
                            atomicOr(p.err, KV_DEVERR_BLOCK_ID);
                            bid = -1;
                        }
                        if (STEP && (s >> 1) == step_j && bid >= 0 && !step_written) {   // warp 11 wrote it?
                            if (!mbar_wait_bounded(smem_u32(&ctl->step_done), 0u)) {
                                ok = false;
                                break;
                            }
                            step_written = true;
                        }
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
                            tma_load_5d(dst + j * TN_PIECE, &tmp, 0, j, 0, TN_TOK * (s & 1), bid, fb);
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
    } else if (warp == 11) {
        // ------------------------------------------------------------ the step's new vectors
        // The same partition, walked beside the producer: every block of the range that holds
        // a sequence's new vector gets it before the producer loads that block.
        if (STEP) {
            MlaPartition<TN_BLK, MLA_SEG_PAD_NARROW> part;
            part.init(p, p.head_tiles, lane, false);
            part.write_step_rows(smem_u32(&ctl->step_done), lane, 32);
        }
    } else if (warp == 5 || warp == 10) {
        // ------------------------------------------------------------ MMA issue
        // Two issuing threads, so that neither kind of MMA waits behind the other: warp 5
        // loads each segment's queries and issues the scores of each stage as soon as it has
        // landed (and its score buffer is free), warp 10 the output update of each stage as
        // soon as its probabilities are written.  They touch different tensor memory; the
        // update of stage g follows the scores of stage g through the softmax's barrier.
        if (lane == 0) {
            const bool scores = warp == 5;
            bool ok = true;
            if (scores) prefetch_tensormap(&tmq);
            // descriptors of the first stage (K-major; MN-major with atoms a piece apart), of
            // the query buffer and of P^T; the others are these moved by a constant
            const uint64_t st_k0 = tc_smem_desc(smem_u32(stages), 16, 1024);
            const uint64_t st_mn0 = tc_smem_desc(smem_u32(stages), TN_PIECE, 1024);
            const uint64_t q_k = tc_smem_desc(smem_u32(qbuf), 16, 1024);
            const uint64_t p_k0 = tc_smem_desc(smem_u32(pbuf), 16, 1024);
            const uint32_t qbytes = static_cast<uint32_t>(TN_NPIECE * q_rows * 128);
            int nq = 0;                             // segments whose queries were requested
            int g = 0;                              // stages (all segments)
            for (int k = 0; ok; ++k) {
                const int slot = k % TN_NITEM;
                ok = mbar_wait_bounded(smem_u32(&ctl->item_full[slot]), static_cast<uint32_t>(k / TN_NITEM) & 1u);
                if (!ok) break;
                const MlaSegment it = ctl->items[slot];
                mbar_arrive(smem_u32(&ctl->item_empty[slot]));
                if (it.n < 0) break;
                const int ns = seg_stages(it);
                if (scores) {
                    // the segment's queries, once the scores of the segment before are done
                    if (k >= 1) ok = mbar_wait_bounded(smem_u32(&ctl->q_free), static_cast<uint32_t>(k - 1) & 1u);
                    if (!ok) break;
                    const uint32_t fb = smem_u32(&ctl->q_full);
                    mbar_arrive_expect_tx(fb, qbytes);
                    for (int j = 0; j < TN_NPIECE; ++j)
                        tma_load_3d(smem_u32(qbuf) + j * TN_QPIECE, &tmq, 64 * j, it.outer * TN_H, it.b, fb);
                    nq = k + 1;
                }
                for (int s = 0; ok && s < ns; ++s, ++g) {
                    const int st = g % TN_NSTAGE;
                    const int t = g & 1;            // the team of this stage
                    if (!scores) {
                        // the output update of stage g, once its probabilities are written --
                        // and, for the segment's first stage, once the epilogue has read the
                        // output set the segment reuses
                        ok = mbar_wait_bounded(smem_u32(&ctl->p_full[t]), static_cast<uint32_t>(g >> 1) & 1u);
                        if (ok && s == 0 && k >= 2)
                            ok = mbar_wait_bounded(smem_u32(&ctl->o_free[k & 1]), static_cast<uint32_t>((k >> 1) - 1) & 1u);
                        if (!ok || *abort_flag) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_output(tbase + tn_obase(k & 1, t), st_mn0 + static_cast<uint64_t>((st * TN_STAGE) >> 4),
                                     p_k0 + static_cast<uint64_t>((64 * t) >> 4), s < 2);
                        tc_commit(smem_u32(&ctl->kv_empty[st]));
                        tc_commit(smem_u32(&ctl->p_free[t]));
                        if (s == ns - 1) tc_commit(smem_u32(&ctl->o_full[k & 1]));
                        continue;
                    }
                    ok = mbar_wait_bounded(smem_u32(&ctl->kv_full[st]), static_cast<uint32_t>(g / TN_NSTAGE) & 1u);
                    if (ok && g >= 2)
                        ok = mbar_wait_bounded(smem_u32(&ctl->s_free[t]), static_cast<uint32_t>((g - 2) >> 1) & 1u);
                    if (ok && s == 0) ok = mbar_wait_bounded(smem_u32(&ctl->q_full), static_cast<uint32_t>(k) & 1u);
                    if (!ok || *abort_flag) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_scores(tbase + TN_S + TN_S_STRIDE * t, st_k0 + static_cast<uint64_t>((st * TN_STAGE) >> 4), q_k);
                    tc_commit(smem_u32(&ctl->s_full[t]));
                    if (s == ns - 1) tc_commit(smem_u32(&ctl->q_free));
                }
            }
            if (!ok) {
                atomicOr(p.err, KV_DEVERR_TIMEOUT);
                ctl->abort_flag = 1;
            }
            // every MMA issued must be complete before the tensor memory is freed, and the
            // query copies before the CTA exits
            const uint32_t done = smem_u32(&ctl->mma_done[scores ? 0 : 1]);
            tc_commit(done);
            mbar_wait_bounded(done, 0);
            if (scores && nq > 0) mbar_wait_bounded(smem_u32(&ctl->q_full), static_cast<uint32_t>(nq - 1) & 1u);
        }
    } else if (warp < 4 || warp >= 12) {
        // ------------------------------------------------------------ softmax teams
        const int team = warp < 4 ? 0 : 1;
        const int v = warp & 3;                     // this warp's lane quarter; heads 4 v .. 4 v + 3
        const int bar_id = 1 + team;
        const uint32_t lrow = tbase + (static_cast<uint32_t>(v * 32) << 16);
        const uint32_t xb = smem_u32(xbufs + team * TN_XBUF) + lane * 16;
        const float sl2 = p.scale_log2;
        bool failed = false;
        int g = 0;                                  // stages of all segments so far
        for (int k = 0;; ++k) {
            const int slot = k % TN_NITEM;
            // warp 0 of the team alone polls the segment ring; the others wait at the
            // team's named barrier (every warp of the team reaches it once per segment and
            // once per stage, failed or not: it is the one place they leave the loop
            // together)
            bool bad = failed;
            if (v == 0 && !bad)
                bad = !all_ok(mbar_wait_bounded(smem_u32(&ctl->item_full[slot]), static_cast<uint32_t>(k / TN_NITEM) & 1u));
            if (named_barrier_or(bar_id, TN_SOFT, bad || *abort_flag != 0)) {
                failed = true;
                break;
            }
            const MlaSegment item = ctl->items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->item_empty[slot]));
            if (item.n < 0) break;
            const int ns = seg_stages(item);
            // the team's running (max, sum) of heads 4 v + i, this lane's token of each stage
            float m_ref[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                m_ref[i] = -INFINITY;
                l[i] = 0.f;
            }
            // this team's stages of the segment: s = s0, s0 + 2, ...
            const int s0 = (g + team) & 1;
            for (int s = s0; s < ns; s += 2) {
                const int gs = g + s;
                const int st = gs % TN_NSTAGE;
                // each warp checks the stage's barriers itself (the scores are issued well
                // ahead, so these are normally complete already); a failure is passed on at
                // the stage's last barrier
                bool ok = !failed;
                if (ok) ok = mbar_wait_spin(smem_u32(&ctl->kv_full[st]), static_cast<uint32_t>(gs / TN_NSTAGE) & 1u);
                if (ok) ok = mbar_wait_spin(smem_u32(&ctl->s_full[team]), static_cast<uint32_t>(gs >> 1) & 1u);
                ok = all_ok(ok);
                if (!ok) failed = true;
                const int blk = ok ? ctl->stage_blk[st] : -1;
                const int nvalid = blk < 0 ? 0 : max(0, min(TN_TOK, item.ctx - item.blk0 * TN_BLK - TN_TOK * s));
                // this warp's K-group partial of token `lane`, 16 heads
                float sc[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) sc[j] = 0.f;
                if (ok) {
                    tc_fence_after();
                    const uint32_t sb = lrow + TN_S + TN_S_STRIDE * team;
                    uint32_t r[16];
                    tc_ld16(sb + 16 * v, r);
                    if (v == 3) {
                        uint32_t r2[16];
                        tc_ld16(sb + TN_ROPE, r2);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) sc[j] = __uint_as_float(r[j]) + __uint_as_float(r2[j]);
                    } else {
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) sc[j] = __uint_as_float(r[j]);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctl->s_free[team]));
                    if (nvalid < TN_TOK) {
                        // value rows of tokens past the cache (or of a skipped block) are
                        // zeroed; the scores, which read them too, are complete
                        uint8_t* sp = stages + st * TN_STAGE;
                        for (int i = v * 32 + lane; i < (TN_TOK - nvalid) * 64; i += TN_SOFT) {
                            const int row = nvalid + (i >> 6);
                            const int pc = (i >> 3) & 7;
                            const int ch = i & 7;
                            *reinterpret_cast<uint4*>(sp + pc * TN_PIECE + row * 128 + (ch << 4)) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                }
                // the four partials added in one round through shared memory: warp w hands
                // the partials of heads 4 u .. 4 u + 3 to warp u (slot 3 u + the rank of w
                // among the other three), then each warp adds the three it received to its
                // own, in the order of the sending warps
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (u != v) sts_f4(xb + (3 * u + (v < u ? v : v - 1)) * 512, sc + 4 * u);
                named_barrier_sync(bar_id, TN_SOFT);
                float s4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    s4[i] = v == 0 ? sc[i] : v == 1 ? sc[4 + i] : v == 2 ? sc[8 + i] : sc[12 + i];
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    if (w != v) lds_add_f4(xb + (3 * v + (w < v ? w : w - 1)) * 512, s4);
                if (lane >= nvalid) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) s4[i] = -INFINITY;   // not cached (may be NaN)
                }
                // The stage's maxima are needed only where some score exceeds its head's
                // reference by more than 2^8 (or no reference is set yet): a vote decides,
                // the maxima are reduced only then.
                bool over = false;
#pragma unroll
                for (int i = 0; i < 4; ++i) over = over || s4[i] * sl2 > m_ref[i] + RESCALE_LOG2;
                bool resc = false;
                if (__any_sync(FULL_MASK, over)) {
                    float mx[4], fi[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx[i] = s4[i];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], __shfl_xor_sync(FULL_MASK, mx[i], o));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float m_new = fmaxf(m_ref[i], mx[i] * sl2);
                        fi[i] = 1.f;
                        if (m_ref[i] == -INFINITY) {
                            m_ref[i] = m_new;       // nothing accumulated yet
                        } else if (m_new > m_ref[i] + RESCALE_LOG2) {
                            fi[i] = fast_exp2(m_ref[i] - m_new);
                            l[i] *= fi[i];
                            m_ref[i] = m_new;
                            resc = true;
                        }
                    }
                    // the factors of this warp's heads (1 where nothing changed), read by the
                    // team's four warps when this warp's flag is set
                    if (resc && lane < 4) ctl->fac[team][4 * v + lane] = pick4(fi, lane);
                }
                if (lane == 0) reinterpret_cast<volatile uint8_t*>(&ctl->resc[team])[v] = resc ? 1 : 0;
                // a failure anywhere ends the loop here; past it, every warp of the team knows
                // which heads' output columns are to be rescaled
                if (named_barrier_or(bar_id, TN_SOFT, failed || *abort_flag != 0)) {
                    failed = true;
                    break;
                }
                const uint32_t rw = *reinterpret_cast<volatile uint32_t*>(&ctl->resc[team]);
                const int rs = static_cast<int>((rw & 1u) | ((rw >> 7) & 2u) | ((rw >> 14) & 4u) | ((rw >> 21) & 8u));
                // the team's previous stage (two back) must have been folded into the output
                // before the output is rescaled or its half of P^T rewritten
                const bool pw = gs < 2 || all_ok(mbar_wait_spin(smem_u32(&ctl->p_free[team]),
                                                                static_cast<uint32_t>((gs - 2) >> 1) & 1u));
                if (!pw) failed = true;
                if (rs != 0 && !failed) {
                    // scale the output columns of the rescaled heads by their factors (a
                    // team's first stage of a segment never rescales)
                    tc_fence_after();
                    float fh[TN_H];
#pragma unroll
                    for (int j = 0; j < TN_H; ++j) fh[j] = (rs >> (j >> 2)) & 1 ? ctl->fac[team][j] : 1.f;
                    const uint32_t ob = lrow + tn_obase(k & 1, team);
#pragma unroll 1
                    for (int i = 0; i < 4; ++i) {
                        uint32_t r[16];
                        tc_ld16(ob + 16 * i, r);
                        tc_wait_ld();
#pragma unroll
                        for (int j = 0; j < TN_H; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * fh[j]);
                        tc_st16(ob + 16 * i, r);
                    }
                    tc_wait_st();
                }
                if (!failed) {
                    // probabilities (bf16) of this lane's token: P^T rows 4 v + i, the team's
                    // 64-byte half of each 128-byte swizzled row
                    const int chunk = 4 * team + (lane >> 3);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float m_use = m_ref[i] == -INFINITY ? 0.f : m_ref[i];
                        const float pi = fast_exp2(fmaf(s4[i], sl2, -m_use));
                        l[i] += pi;
                        const int hd = 4 * v + i;
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(smem_u32(pbuf) + hd * 128 + ((chunk ^ (hd & 7)) << 4) +
                                                                     (lane & 7) * 2),
                                     "h"(static_cast<unsigned short>(pack_bf16x2(pi, 0.f)))
                                     : "memory");
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && !failed) mbar_arrive(smem_u32(&ctl->p_full[team]));
            }
            if (!failed) {
                // the team's (max, sum) per head for the segment (a team without a stage in
                // it leaves l = 0), for the epilogue; the set's last reader was the epilogue
                // of segment k - 2
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int i = 0; i < 4; ++i) l[i] += __shfl_xor_sync(FULL_MASK, l[i], o);
                const bool w = k < 2 || all_ok(mbar_wait_bounded(smem_u32(&ctl->o_free[k & 1]),
                                                                 static_cast<uint32_t>((k >> 1) - 1) & 1u));
                if (!w) {
                    failed = true;
                } else {
                    if (lane < 4) {
                        ctl->lsum[k & 1][team][4 * v + lane] = pick4(l, lane);
                        ctl->mref[k & 1][team][4 * v + lane] = pick4(m_ref, lane);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&ctl->ml_full[k & 1]));
                }
            }
            g += ns;
        }
        if (failed && lane == 0) {
            atomicOr(p.err, KV_DEVERR_TIMEOUT);
            ctl->abort_flag = 1;
        }
        grid_dependents_launch();
    } else {
        // ------------------------------------------------------------ epilogue (warps 6-9)
        // warp 6 + i reads lane quarter (6 + i) & 3: latent rows 128 t + 32 q + lane of the
        // four tiles, 16 heads each, of both teams' outputs; their log-sum-exp merge is a
        // whole sequence's output in bf16, or a piece of a cut one as its fp16 partial
        // [piece][head][512] with (max, sum) per head
        const int q4 = warp & 3;
        const uint32_t lrow = tbase + (static_cast<uint32_t>(q4 * 32) << 16);
        bool failed = false;
        for (int k = 0;; ++k) {
            const int slot = k % TN_NITEM;
            // warp 6 alone polls (sleeping between polls: these waits last a segment); warps
            // 7-9 wait at named barrier 3
            bool bad = false;
            if (warp == 6)
                bad = !all_ok(mbar_wait_sleep(smem_u32(&ctl->item_full[slot]), static_cast<uint32_t>(k / TN_NITEM) & 1u));
            if (named_barrier_or(3, TN_SOFT, bad)) {
                failed = true;
                break;
            }
            const MlaSegment item = ctl->items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->item_empty[slot]));
            if (item.n < 0) break;
            if (warp == 6) {
                bool ok = mbar_wait_sleep(smem_u32(&ctl->o_full[k & 1]), static_cast<uint32_t>(k >> 1) & 1u);
                if (ok) ok = mbar_wait_sleep(smem_u32(&ctl->ml_full[k & 1]), static_cast<uint32_t>(k >> 1) & 1u);
                bad = !all_ok(ok);
            }
            if (named_barrier_or(3, TN_SOFT, bad || *abort_flag != 0)) {
                failed = true;
                break;
            }
            tc_fence_after();
            const int b = item.b, ht = item.outer;
            const int nh = min(TN_H, p.q_heads - ht * TN_H);
            const bool whole = item.nsplit == 1;
            const size_t row0 = static_cast<size_t>(b) * p.q_heads + ht * TN_H;
            const size_t piece = (static_cast<size_t>(b) * p.head_tiles + ht) * p.max_splits + item.split;
            // per head: the teams' weights 2^(m_t - M) / L, M the larger max of a team with a
            // sum, L = sum_t l_t 2^(m_t - M); a team with no sum has weight 0 (its output set
            // may hold anything)
            float w0[TN_H], w1[TN_H];
            float mh = 0.f, lh = 0.f;
#pragma unroll
            for (int j = 0; j < TN_H; ++j) {
                const float l0 = ctl->lsum[k & 1][0][j], l1 = ctl->lsum[k & 1][1][j];
                const float m0 = ctl->mref[k & 1][0][j], m1 = ctl->mref[k & 1][1][j];
                const bool h0 = l0 > 0.f, h1 = l1 > 0.f;
                const float M = h0 && h1 ? fmaxf(m0, m1) : (h0 ? m0 : (h1 ? m1 : -INFINITY));
                const float e0 = h0 ? fast_exp2(m0 - M) : 0.f, e1 = h1 ? fast_exp2(m1 - M) : 0.f;
                const float L = l0 * e0 + l1 * e1;
                const float inv = L > 0.f ? 1.f / L : 0.f;
                w0[j] = e0 * inv;
                w1[j] = e1 * inv;
                if (lane == j) {
                    mh = M;
                    lh = L;
                }
            }
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                uint32_t r0[16], r1[16];
                tc_ld16(lrow + tn_obase(k & 1, 0) + 16 * i, r0);
                tc_ld16(lrow + tn_obase(k & 1, 1) + 16 * i, r1);
                tc_wait_ld();
                float o[TN_H];
#pragma unroll
                for (int j = 0; j < TN_H; ++j)
                    o[j] = (w0[j] > 0.f ? __uint_as_float(r0[j]) * w0[j] : 0.f) +
                           (w1[j] > 0.f ? __uint_as_float(r1[j]) * w1[j] : 0.f);
                const int d = 128 * i + 32 * q4 + lane;
                if (whole) {
                    uint16_t* dst = p.out + row0 * MLA_DV + d;
#pragma unroll
                    for (int j = 0; j < TN_H; ++j)
                        if (j < nh) dst[static_cast<size_t>(j) * MLA_DV] = static_cast<uint16_t>(pack_bf16x2(o[j], 0.f));
                } else {
                    // fp16: averages of cached values, well inside its range, 11 significant
                    // bits against the output's 8
                    uint16_t* dst = reinterpret_cast<uint16_t*>(p.part_o) + piece * (TN_H * MLA_DV) + d;
#pragma unroll
                    for (int j = 0; j < TN_H; ++j) dst[j * MLA_DV] = static_cast<uint16_t>(pack_f16x2(o[j], 0.f));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->o_free[k & 1]));
            if (warp == 6 && lane < TN_H) {
                if (!whole)
                    reinterpret_cast<float2*>(p.part_ml)[piece * TN_H + lane] = make_float2(mh, lh);
                else if (p.lse != nullptr && lane < nh)
                    p.lse[row0 + lane] = lse_from(mh, lh);
            }
            if (warp == 6 && lane == 0 && p.tickets != nullptr)
                p.tickets[static_cast<size_t>(b) * p.head_tiles + ht] = item.nsplit;
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

cudaError_t launch_mla_decode_tcn(dim3 grid, const CUtensorMap& tm, const CUtensorMap& tq,
                                  const MlaParams& p, cudaStream_t s)
{
    cudaError_t e = p.kv_new != nullptr
                        ? launch_dependent(paged_mla_decode_tcn<true>, grid, dim3(TN_THREADS), TN_SMEM, s,
                                           tm, tq, p)
                        : launch_dependent(paged_mla_decode_tcn<false>, grid, dim3(TN_THREADS), TN_SMEM, s, tm,
                                           tq, p);
    if (e != cudaSuccess || p.max_splits <= 1) return e;
    return launch_dependent(paged_mla_merge_tcn, dim3(p.batch, p.head_tiles, MLA_DV / 128), dim3(256), 0, s, p);
}

}  // namespace kvp
