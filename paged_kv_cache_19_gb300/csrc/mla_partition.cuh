// mla_partition.cuh -- the balanced static partition of the latent-attention
// work shared by the tcgen05 MLA kernels.
//
// Units are (outer, sequence b, position) in that order, T = S * nouter of them,
// `outer` being whatever the kernel splits the heads into (head tiles, times the
// latent halves for the wide form).  A sequence of ctx tokens has nb =
// ceil(ctx / tok) blocks and occupies PAD + nb positions (none when it is empty):
// a pad, then its blocks.  The pad is no work; it stands for what starting a
// segment costs a CTA (the queries' load, the epilogue), so that ranges holding
// many sequence starts get fewer blocks (measured best on GB300: 2 positions for
// the narrow form, 4 for the wide one).  S is the
// positions of the whole batch.  CTA c of the G that have work takes the
// contiguous range [c T / G, (c + 1) T / G), with G chosen so that a range holds
// at least split_blocks positions; every CTA derives the same partition from the
// context lengths, so no CTA waits for another.  A sequence
// cut by range boundaries leaves one piece per CTA that holds some of its
// blocks: piece `split` of `nsplit`, merged afterwards by log-sum-exp.  A range
// that holds only pad positions has no work.
//
// A CTA walks its range as segments (runs of blocks of one sequence and one
// outer index), the last segment first: a sequence cut between CTA c and c + 1
// is then worked on first by both, so the merge of its pieces does not wait for
// the end of either range.
#pragma once

#include "append_row.cuh"
#include "device_common.cuh"
#include "kernels.h"

namespace kvp {

// One segment: blocks blk0 .. blk0 + n - 1 of sequence b for outer index `outer`;
// n < 0 marks the end of the range.
struct MlaSegment {
    int outer, b, blk0, n, ctx, split, nsplit;
};

// Quotient and remainder of non-negative 64-bit values, by a 32-bit division when both
// fit in 32 bits (the usual case: a 64-bit division is a long software sequence).
__device__ __forceinline__ long long udiv_ll(long long a, long long b)
{
    if ((static_cast<unsigned long long>(a) | static_cast<unsigned long long>(b)) >> 32 == 0)
        return static_cast<long long>(static_cast<unsigned>(a) / static_cast<unsigned>(b));
    return a / b;
}

__device__ __forceinline__ long long umod_ll(long long a, long long b)
{
    if ((static_cast<unsigned long long>(a) | static_cast<unsigned long long>(b)) >> 32 == 0)
        return static_cast<long long>(static_cast<unsigned>(a) % static_cast<unsigned>(b));
    return a % b;
}

template <int TOK, int PAD>
struct MlaPartition {
    const MlaParams* p;
    long long S, T, gact, u0, u1, c;
    int cap;
    // the cursor (each lane walks its own copy after init)
    long long u, ls, ub_l, pre;
    int outer, b, blk, outer_l, b_last, ctx_l, nb_l;
    bool last_done;

    __device__ __forceinline__ int seq_ctx(int bb) const
    {
        const int x = __ldg(p->ctx + bb);
        return x < 0 ? 0 : (x > cap ? cap : x);
    }

    // the CTA whose range holds unit x
    __device__ __forceinline__ int cta_of(long long x) const { return static_cast<int>(udiv_ll((x + 1) * gact - 1, T)); }

    // Warp-wide (all 32 lanes): block count of the batch, the range of this CTA and the
    // sequences at its ends.  Out-of-range context lengths are flagged and clamped; an
    // empty sequence has no units, so its output (0) and LSE (-inf) are written here, by
    // CTA b mod gridDim.x (all of this only when `outputs`; a second warp walking the same
    // partition passes false).  Batches of up to 256 sequences keep their lengths and block
    // prefix sums in registers (sequence 32 i + lane in slot i), so that the range ends
    // are located without loading the lengths again.
    __device__ void init(const MlaParams& params, int nouter, int lane, bool outputs = true)
    {
        p = &params;
        cap = p->max_blocks * TOK;
        S = 0;
        int ctxv[8], nbv[8], incl[8], tot[8];
        for (int b0 = 0; b0 < p->batch; b0 += 256) {
            int raw[8];                             // eight lengths per lane in flight
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int bb = b0 + i * 32 + lane;
                raw[i] = bb < p->batch ? __ldg(p->ctx + bb) : 0;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int bb = b0 + i * 32 + lane;
                int x = raw[i];
                if (bb < p->batch && (x < 0 || x > cap)) {
                    if (blockIdx.x == 0 && outputs) atomicOr(p->err, KV_DEVERR_CONTEXT);
                    x = x < 0 ? 0 : cap;
                }
                const int nb = (x + TOK - 1) / TOK;
                ctxv[i] = x;
                nbv[i] = nb > 0 ? nb + PAD : 0;     // positions of the sequence
                incl[i] = nbv[i];
            }
            // inclusive prefix sums over the lanes, the eight slots' shuffle chains interleaved
#pragma unroll
            for (int o = 1; o < 32; o <<= 1)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int y = __shfl_up_sync(FULL_MASK, incl[i], o);
                    if (lane >= o) incl[i] += y;
                }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                tot[i] = __shfl_sync(FULL_MASK, incl[i], 31);
                S += tot[i];
            }
            if (outputs) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int bb = b0 + i * 32 + lane;
                    if (bb < p->batch && nbv[i] == 0 &&
                        bb % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x)) {
                        uint4* dst = reinterpret_cast<uint4*>(p->out + static_cast<size_t>(bb) * p->q_heads * MLA_DV);
                        for (int v = 0; v < p->q_heads * (MLA_DV / 8); ++v) dst[v] = make_uint4(0u, 0u, 0u, 0u);
                        if (p->lse != nullptr)
                            for (int hh = 0; hh < p->q_heads; ++hh) p->lse[static_cast<size_t>(bb) * p->q_heads + hh] = -INFINITY;
                    }
                }
            }
        }
        T = S * nouter;
        gact = udiv_ll(T, p->split_blocks);
        if (gact < 1) gact = 1;
        if (gact > gridDim.x) gact = gridDim.x;
        c = blockIdx.x;
        u0 = c < gact ? udiv_ll(c * T, gact) : T;
        u1 = c < gact ? udiv_ll((c + 1) * T, gact) : T;
        int b_first = 0;
        long long pre_first = 0, pre_last = 0;
        b_last = 0;
        ctx_l = 0;
        if (u0 < u1) {
            if (p->batch <= 256) {
                // both ends at once from the registers: the slots' offsets, then sixteen
                // independent ballots, then the first slot past each end
                const long long v0 = umod_ll(u0, S), v1 = umod_ll(u1 - 1, S);
                long long off[8];
                long long acc = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    off[i] = acc;
                    acc += tot[i];
                }
                unsigned p0[8], p1[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    p0[i] = __ballot_sync(FULL_MASK, off[i] + incl[i] > v0);
                    p1[i] = __ballot_sync(FULL_MASK, off[i] + incl[i] > v1);
                }
                int i0 = 7, i1 = 7;
#pragma unroll
                for (int i = 7; i >= 0; --i) {
                    if (p0[i] != 0u) i0 = i;
                    if (p1[i] != 0u) i1 = i;
                }
                // the slot's values of the first lane past each end, picked without indexing
                unsigned q0 = 0u, q1 = 0u;
                long long o0 = 0, o1 = 0;
                int e0 = 0, e1 = 0, c1 = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i == i0) {
                        q0 = p0[i];
                        o0 = off[i];
                        e0 = incl[i] - nbv[i];
                    }
                    if (i == i1) {
                        q1 = p1[i];
                        o1 = off[i];
                        e1 = incl[i] - nbv[i];
                        c1 = ctxv[i];
                    }
                }
                const int fl0 = __ffs(q0) - 1, fl1 = __ffs(q1) - 1;
                b_first = i0 * 32 + fl0;
                pre_first = o0 + __shfl_sync(FULL_MASK, e0, fl0);
                b_last = i1 * 32 + fl1;
                pre_last = o1 + __shfl_sync(FULL_MASK, e1, fl1);
                ctx_l = __shfl_sync(FULL_MASK, c1, fl1);
            } else {
                locate(u0, b_first, pre_first, lane);
                locate(u1 - 1, b_last, pre_last, lane);
                ctx_l = seq_ctx(b_last);
            }
        }
        // cursor: the last segment first, then the rest of the range from its start
        ls = u1;
        outer_l = nb_l = 0;
        ub_l = 0;
        if (u0 < u1) {
            outer_l = static_cast<int>(udiv_ll(u1 - 1, S));
            ub_l = static_cast<long long>(outer_l) * S + pre_last;
            ls = ub_l > u0 ? ub_l : u0;
            nb_l = (ctx_l + TOK - 1) / TOK;
        }
        last_done = !(u0 < u1);
        u = u0;
        outer = u0 < u1 ? static_cast<int>(udiv_ll(u0, S)) : 0;
        b = b_first;
        pre = pre_first;
        blk = u0 < u1 ? static_cast<int>(umod_ll(u0, S) - pre_first) : 0;
    }

    // Warp-wide: the sequence holding position x < T, and the number of positions before
    // it (prefix sums, 32 sequences at a time).
    __device__ void locate(long long x, int& b_at, long long& pre_at, int lane) const
    {
        const long long v = umod_ll(x, S);
        long long acc = 0;
        b_at = 0;
        pre_at = 0;
        for (int b0 = 0; b0 < p->batch; b0 += 32) {
            const int bb = b0 + lane;
            const int nbr = bb < p->batch ? (seq_ctx(bb) + TOK - 1) / TOK : 0;
            const int nb = nbr > 0 ? nbr + PAD : 0;       // positions
            int in = nb;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(FULL_MASK, in, o);
                if (lane >= o) in += y;
            }
            const unsigned past = __ballot_sync(FULL_MASK, acc + in > v);
            if (past != 0u) {
                const int fl = __ffs(past) - 1;
                b_at = b0 + fl;
                pre_at = acc + __shfl_sync(FULL_MASK, in, fl) - __shfl_sync(FULL_MASK, nb, fl);
                return;
            }
            acc += __shfl_sync(FULL_MASK, in, 31);
        }
    }

    // A segment of blocks blk0 .. blk0 + n - 1 of a sequence whose positions start at ub
    // (its pad): the pieces are the ranges holding its blocks.
    __device__ __forceinline__ MlaSegment make(int o, int bb, long long ub, int blk0, int n, int x, int nb) const
    {
        MlaSegment it;
        const long long first = ub + PAD;   // position of block 0
        const int cf = cta_of(first);
        it.outer = o;
        it.b = bb;
        it.blk0 = blk0;
        it.n = n;
        it.ctx = x;
        it.split = static_cast<int>(c) - cf;
        it.nsplit = cta_of(first + nb - 1) - cf + 1;
        return it;
    }

    // paged_mla_decode_step, thread t of the nth (>= 24) lanes that walk the partition after
    // init, each on its own cursor: every segment of the range that holds the block with a
    // sequence's new vector (position ctx - 1) gets the vector written into that block, the
    // lanes sharing each copy; then each lane orders its writes before later TMA loads and
    // arrives once on `done` (expected count nth).  The thread that loads the blocks waits on
    // `done` before it loads such a block.  Blocks with a bad id are skipped (the loading
    // thread flags them when it reaches them); a position outside the table is not written
    // and is flagged KV_DEVERR_POSITION by CTA 0, as the append would flag it.  Several CTAs,
    // or both halves of one, may write the same bytes.
    __device__ void write_step_rows(uint32_t done, int t, int nth)
    {
        if (blockIdx.x == 0)
            for (int bb = t; bb < p->batch; bb += nth) {
                const int x = __ldg(p->ctx + bb);
                if (x < 1 || x > cap) atomicOr(p->err, KV_DEVERR_POSITION);
            }
        for (;;) {
            const MlaSegment sg = next();
            if (sg.n < 0) break;
            const int raw = __ldg(p->ctx + sg.b);
            if (raw < 1 || raw > cap) continue;
            const int j = (raw - 1) / TOK;
            if (j < sg.blk0 || j >= sg.blk0 + sg.n) continue;
            // the block id and the new vector are loaded together
            const int bid = __ldg(p->tables + static_cast<size_t>(sg.b) * p->max_blocks + j);
            uint4 x[3];
            load_latent_share(*p, sg.b, t, nth, x);
            if (bid < 0 || bid >= p->num_blocks) continue;
            store_latent_share(*p, bid, TOK, (raw - 1) % TOK, t, nth, x);
        }
        fence_proxy_async_all();
        mbar_arrive(done);
    }

    // One thread: the next segment of the range (n < 0: none left).
    __device__ MlaSegment next()
    {
        MlaSegment it{};
        it.n = -1;
        if (!last_done) {
            last_done = true;
            // positions [ls, u1) of the last sequence; its blocks among them, if any
            const long long r0 = ls - ub_l - PAD > 0 ? ls - ub_l - PAD : 0;
            const long long r1 = u1 - ub_l - PAD;
            if (r1 > r0)
                return make(outer_l, b_last, ub_l, static_cast<int>(r0), static_cast<int>(r1 - r0), ctx_l, nb_l);
        }
        while (u < ls) {
            const int x = seq_ctx(b);
            const int nb = (x + TOK - 1) / TOK;
            const int wv = nb > 0 ? nb + PAD : 0;
            if (blk >= wv) {                        // next sequence (or next outer index)
                pre += wv;
                blk = 0;
                if (++b == p->batch) {
                    b = 0;
                    pre = 0;
                    ++outer;
                }
                continue;
            }
            const int n = static_cast<int>(wv - blk < ls - u ? wv - blk : ls - u);
            const int r0 = blk - PAD > 0 ? blk - PAD : 0;
            const int r1 = blk + n - PAD;
            const long long ub = static_cast<long long>(outer) * S + pre;
            u += n;
            blk += n;
            if (r1 > r0) return make(outer, b, ub, r0, r1 - r0, x, nb);
            // only pad positions of this sequence: no work, walk on
        }
        return it;
    }
};

}  // namespace kvp
