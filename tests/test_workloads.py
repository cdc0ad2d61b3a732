"""Host-side checks of the workload generator and the byte accounting."""
import os

import numpy as np
import pytest

import workloads
from workloads import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_bytes_per_token_matches_the_pages():
    rows = []
    for line in open(os.path.join(GOLDEN, "kv_bytes_per_token.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            rows.append([c.strip() for c in line.split("|")])
    assert len(rows) == 2
    for _, layers, kvh, d, e, want in rows:
        assert accounting.kv_bytes_per_token(int(layers), int(kvh), int(d), int(e)) == int(want)


def test_generator_is_deterministic_and_shaped():
    spec = workloads.custom(batch=6, q_heads=8, kv_heads=2, head_dim=64, block_size=16,
                            ctx_uniform=(1, 90), seed=3)
    a, b = workloads.make(spec), workloads.make(spec)
    assert np.array_equal(a.k, b.k) and np.array_equal(a.q, b.q)
    assert np.array_equal(a.block_tables, b.block_tables)
    assert a.k.shape == (a.total_tokens, 2, 64) and a.q.shape == (6, 8, 64)
    nb = (a.context_lens + 15) // 16
    for i in range(6):
        assert (a.block_tables[i, :nb[i]] >= 0).all() and (a.block_tables[i, nb[i]:] == -1).all()
    used = a.block_tables[a.block_tables >= 0]
    assert np.unique(used).size == used.size                    # no sharing without prefix groups
    assert a.num_blocks == int(np.ceil(1.1 * used.size))


def test_prefix_groups_share_only_full_blocks_without_the_append_slot():
    spec = workloads.custom(batch=8, q_heads=4, kv_heads=1, head_dim=16, block_size=16,
                            ctx=[20, 70, 64, 129, 65, 200, 16, 90], seed=4, prefix_group=4,
                            prefix_tokens=64)
    w = workloads.make(spec)
    for b in range(8):
        ctx = int(w.context_lens[b])
        for j in range(int((ctx + 15) // 16)):
            if w.shared_block[b, j]:
                assert j < 4 and j < (ctx - 1) // 16
    # shared ids are the same inside a group and distinct across groups
    g0 = {int(w.block_tables[b, 0]) for b in range(4) if w.shared_block[b, 0]}
    g1 = {int(w.block_tables[b, 0]) for b in range(4, 8) if w.shared_block[b, 0]}
    assert len(g0) == 1 and len(g1) == 1 and g0 != g1
    # values of the shared prefix agree inside the group
    assert np.array_equal(w.seq_k(1)[:64], w.seq_k(3)[:64])
    # each shared block is written once by the prefill list
    assert accounting.unique_kv_tokens(w) < w.total_tokens


def test_decode_bytes_counts_kv_and_partials():
    spec = workloads.custom(batch=2, q_heads=8, kv_heads=2, head_dim=64, block_size=16,
                            ctx=[100, 10], seed=5)
    w = workloads.make(spec)
    one = accounting.decode_bytes(w, split_tokens=10 ** 6)
    assert one["kv_logical"] == 110 * 2 * 2 * 64 * 2 and one["partials"] == 0
    many = accounting.decode_bytes(w, split_tokens=32)         # sequence 0 -> 4 chunks
    assert many["partials"] == 4 * 8 * (64 + 2) * 4 * 2


def _brute_force_pieces(nb, tiles, split_blocks, grid, halves=2, pad=None):
    """Assign every position (latent half / head tile, sequence, position) to its range by
    scanning the range starts, then count the distinct ranges holding each sequence's
    blocks (a sequence's first `pad` positions hold none; by default the form's pad)."""
    if pad is None:
        pad = accounting.MLA_SEG_PAD_WIDE if halves == 2 else accounting.MLA_SEG_PAD_NARROW
    units = [(outer, b, j >= pad) for outer in range(tiles * halves) for b, n in enumerate(nb)
             for j in range(n + pad if n else 0)]
    T = len(units)
    g = max(1, min(grid, T // split_blocks))
    starts = [c * T // g for c in range(g + 1)]
    owner = []
    c = 0
    for u in range(T):
        while starts[c + 1] <= u:
            c += 1
        owner.append(c)
    sizes = [starts[c + 1] - starts[c] for c in range(g)]
    seen = {}
    for ((outer, b, real), c) in zip(units, owner):
        if real:
            seen.setdefault((outer, b), set()).add(c)
    pieces = [len(seen[(outer, b)]) for outer in range(tiles * halves) for b, n in enumerate(nb) if n > 0]
    return pieces, sizes, g


@pytest.mark.parametrize("ctx,heads,split_blocks,grid", [
    ([1, 70, 300, 2, 4096, 65], 128, 1, 152),
    ([640, 64, 3000, 129, 2000], 128, 16, 7),
    ([100] * 40, 256, 4, 33),
    ([5000, 1], 96, 8, 152),
])
def test_mla_tc_pieces_match_a_brute_force_partition(ctx, heads, split_blocks, grid):
    w = workloads.make(workloads.mla(batch=len(ctx), q_heads=heads, block_size=64, ctx=ctx, seed=3))
    nb = [-(-c // 64) for c in ctx]
    want, sizes, g = _brute_force_pieces(nb, -(-heads // 128), split_blocks, grid)
    got = accounting.mla_tc_pieces(w, split_blocks, grid)
    assert list(got) == want
    # every range but a lone one holds at least split_blocks units, and no sequence is cut
    # into more pieces than the workspace bound ceil((max_blocks - 1) / split_blocks) + 1
    if g > 1:
        assert min(sizes) >= split_blocks
    assert max(want) <= (max(nb) - 1 + split_blocks - 1) // split_blocks + 1


@pytest.mark.parametrize("ctx,heads,split_blocks,grid", [
    ([1, 70, 300, 2, 4096, 65], 16, 1, 152),
    ([640, 64, 3000, 129, 2000], 40, 13, 7),
    ([100] * 40, 16, 4, 33),
    ([5000, 1], 48, 8, 152),
])
def test_mla_narrow_pieces_match_a_brute_force_partition(ctx, heads, split_blocks, grid):
    """The narrow tensor-core form: units (head tile of 16, sequence, block), no halves."""
    w = workloads.make(workloads.mla(batch=len(ctx), q_heads=heads, block_size=64, ctx=ctx, seed=3))
    nb = [-(-c // 64) for c in ctx]
    want, sizes, g = _brute_force_pieces(nb, -(-heads // 16), split_blocks, grid, halves=1)
    got = accounting.mla_tc_pieces(w, split_blocks, grid, head_tile=16, halves=1)
    assert list(got) == want
    if g > 1:
        assert min(sizes) >= split_blocks
    assert max(want) <= (max(nb) - 1 + split_blocks - 1) // split_blocks + 1


def _walk_partition(nb, nouter, split_blocks, grid, pad):
    """The tensor-core MLA kernels' partition walk restated on the host: per CTA, the
    segments (outer, sequence, first block, blocks, split, nsplit) it hands on, the last
    one first, from the same integer arithmetic as the device code."""
    wv = [n + pad if n else 0 for n in nb]
    S = sum(wv)
    T = S * nouter
    gact = min(grid, max(1, T // split_blocks))
    pre = [sum(wv[:i]) for i in range(len(nb))]

    def cta_of(x):
        return ((x + 1) * gact - 1) // T

    def locate(v):
        for b in range(len(nb)):
            if wv[b] and pre[b] <= v < pre[b] + wv[b]:
                return b, pre[b]
        raise AssertionError("position outside the batch")

    def make(c, o, bb, ub, blk0, n):
        first = ub + pad
        cf = cta_of(first)
        return (o, bb, blk0, n, c - cf, cta_of(first + nb[bb] - 1) - cf + 1)

    segs = {}
    for c in range(grid):
        u0 = c * T // gact if c < gact else T
        u1 = (c + 1) * T // gact if c < gact else T
        out = []
        if u0 < u1:
            b_first, pre_first = locate(u0 % S)
            b_last, pre_last = locate((u1 - 1) % S)
            outer_l = (u1 - 1) // S
            ub_l = outer_l * S + pre_last
            ls = max(ub_l, u0)
            r0, r1 = max(ls - ub_l - pad, 0), u1 - ub_l - pad
            if r1 > r0:
                out.append(make(c, outer_l, b_last, ub_l, r0, r1 - r0))
            u, outer, b, p_, blk = u0, u0 // S, b_first, pre_first, u0 % S - pre_first
            while u < ls:
                if blk >= wv[b]:
                    p_ += wv[b]
                    blk = 0
                    b += 1
                    if b == len(nb):
                        b, p_, outer = 0, 0, outer + 1
                    continue
                n = min(wv[b] - blk, ls - u)
                r0, r1 = max(blk - pad, 0), blk + n - pad
                ub = outer * S + p_
                u += n
                blk += n
                if r1 > r0:
                    out.append(make(c, outer, b, ub, r0, r1 - r0))
        segs[c] = out
    return segs


@pytest.mark.parametrize("pad", [0, accounting.MLA_SEG_PAD_NARROW, accounting.MLA_SEG_PAD_WIDE, 7])
def test_mla_partition_walk_covers_every_block_once(pad):
    rng = np.random.default_rng(17)
    for trial in range(300):
        batch = int(rng.integers(1, 40))
        nb = [int(x) if rng.random() > 0.15 else 0 for x in rng.integers(1, 70, size=batch)]
        if sum(nb) == 0:
            nb[0] = 1
        nouter = int(rng.choice([1, 2, 3, 4, 6]))
        split_blocks = int(rng.choice([1, 2, 4, 13]))
        grid = int(rng.choice([1, 7, 33, 152]))
        segs = _walk_partition(nb, nouter, split_blocks, grid, pad)
        covered = {}
        for c, lst in segs.items():
            keys = [(o, b) for (o, b, *_rest) in lst]
            assert len(keys) == len(set(keys)), "two segments of one sequence in one CTA"
            for (o, b, blk0, n, split, nsplit) in lst:
                assert n >= 1 and 0 <= blk0 and blk0 + n <= nb[b]
                assert 0 <= split < nsplit
                covered.setdefault((o, b), []).append((blk0, n, split, nsplit))
        want_pieces, _, _ = _brute_force_pieces(nb, nouter, split_blocks, grid, halves=1, pad=pad)
        keys = [(o, b) for o in range(nouter) for b in range(batch) if nb[b]]
        assert sorted(covered) == sorted(keys)
        for key, want in zip(keys, want_pieces):
            parts = sorted(covered[key])
            blocks = [j for (blk0, n, _, _) in parts for j in range(blk0, blk0 + n)]
            assert blocks == list(range(nb[key[1]])), (trial, key)
            assert {s for (_, _, s, _) in parts} == set(range(want))
            assert all(ns == want for (_, _, _, ns) in parts)
