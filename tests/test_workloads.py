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


def _brute_force_pieces(nb, tiles, split_blocks, grid, halves=2):
    """Assign every unit (latent half / head tile, sequence, block) to its range by
    scanning the range starts, then count the distinct ranges each sequence touches."""
    units = [(outer, b) for outer in range(tiles * halves) for b, n in enumerate(nb) for _ in range(n)]
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
    for (key, c) in zip(units, owner):
        seen.setdefault(key, set()).add(c)
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
