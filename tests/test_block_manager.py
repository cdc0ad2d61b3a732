"""Host block manager (kv_bm_* in include/kv_block_manager.h), checked on the CPU
against the pages' worked examples and against invariants of the bookkeeping.

Sources:
  * xuewyang.github.io "KV cache, vLLM, SGLang...", "A toy vLLM": the block tables of
    a continuous-batching engine over 10 blocks of 4 tokens (tests/golden).
  * learn.mohebi.ai lesson 12 "Inference serving", section 8 question 3: parallel
    sampling of 3 answers to a 100-token prompt with blocks of 16 -> 21 blocks
    unshared, 7 shared, 9 after each sample writes one token (copy-on-write).
  * learn.mohebi.ai lesson 12, the NumPy check of paging memory: 200 live lengths
    from default_rng(1).integers(100, 3000) -> 322055 tokens in 323568 paged slots.
  * brunomaga.github.io, "Prefix caching, prompt caching or context caching", the
    figure on lookup with blocks of 4: request 2 reuses two blocks of request 1 and
    prefills 4 tokens; request 3 reuses one block and prefills 8 although its last
    block holds the same tokens as request 1's.
  * kongchang.com "KV cache and PagedAttention", "Automatic Prefix Caching": unused
    cached blocks are evicted least recently used first; a per-request salt mixed into
    the first block's hash keeps tenants from sharing blocks.
"""
import os

import numpy as np
import pytest

import paged_kv_cache_19_gb300 as kp
from paged_kv_cache_19_gb300 import build as cuda_build

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    cuda_build.build()
    kp.load_library()


def blocks_needed(n, bs):
    return -(-n // bs)


# ---------------------------------------------------------------------------
# Toy continuous-batching engine (block bookkeeping only; the model is replaced by
# counting tokens, which is all the block tables depend on).
# ---------------------------------------------------------------------------
def run_toy_engine(requests, num_blocks=10, block=4, max_running=3):
    bm = kp.BlockManager(num_blocks, block)
    waiting = [dict(rid=r, toks=p, n_prompt=p, n_new=n, cached=0) for r, p, n in requests]
    running, trace, step, preemptions, produced = [], [], 0, 0, {}

    def done(s):
        return s["toks"] - s["n_prompt"] >= s["n_new"]

    def free_blocks():
        return bm.num_free_blocks()[0]

    while waiting or running:
        step += 1
        while (waiting and len(running) < max_running
               and blocks_needed(waiting[0]["toks"] + 1, block) <= free_blocks()):
            s = waiting.pop(0)
            running.append(s)
            bm.add_sequence(s["rid"])
            assert bm.append_slots(s["rid"], s["toks"]) is None     # prefill the prompt
            s["cached"] = s["toks"]
            s["toks"] += 1                                          # first generated token
        while running and sum(s["cached"] % block == 0 for s in running) > free_blocks():
            s = running.pop()                                       # preempt the newest
            bm.free_sequence(s["rid"])
            preemptions += 1
            s["n_new"] -= s["toks"] - s["n_prompt"]
            s["n_prompt"], s["cached"] = s["toks"], 0
            waiting.insert(0, s)
        for s in running:
            if not done(s):
                bm.append_slots(s["rid"], 1)                        # K/V of the last token
                s["cached"] += 1
                s["toks"] += 1
        tables = {s["rid"]: bm.block_table(s["rid"]) for s in running}
        trace.append((step, [s["rid"] for s in running], free_blocks(), tables))
        for s in [s for s in running if done(s)]:
            running.remove(s)
            bm.free_sequence(s["rid"])
            produced[s["rid"]] = s["toks"]
    return trace, bm, preemptions, produced


def load_toy_golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "p1_toy_engine_tables.txt")):
        if line.startswith("#") or not line.strip():
            continue
        step, batch, free, tables = [f.strip() for f in line.split("|")]
        tab = {}
        for item in tables.split(";"):
            rid, blocks = item.split(":")
            tab[int(rid)] = [int(b) for b in blocks.split(",")]
        rows.append((int(step), [int(b) for b in batch.split(",")], int(free), tab))
    return rows


def test_toy_engine_block_tables_match_the_page():
    trace, bm, preemptions, _ = run_toy_engine([(0, 5, 3), (1, 2, 8), (2, 7, 2), (3, 3, 6),
                                                (4, 4, 4)])
    assert trace == load_toy_golden()
    assert preemptions == 0 and bm.num_free_blocks() == (10, 0)


def test_toy_engine_with_a_small_pool_preempts_and_still_finishes():
    # the page's suggestion: shrink the pool to 4 blocks and watch preemption
    requests = [(0, 5, 3), (1, 2, 8), (2, 7, 2), (3, 3, 6), (4, 4, 4)]
    trace, bm, preemptions, produced = run_toy_engine(requests, num_blocks=4)
    assert preemptions > 0
    assert produced == {r: p + n for r, p, n in requests}   # every request got all its tokens
    assert bm.num_free_blocks() == (4, 0)
    for _, batch, free, tables in trace:
        held = [b for t in tables.values() for b in t]
        assert len(held) == len(set(held)) and len(held) + free == 4


# ---------------------------------------------------------------------------
# Copy-on-write: parallel sampling
# ---------------------------------------------------------------------------
def test_parallel_sampling_copy_on_write_21_7_9():
    bs, prompt = 16, 100
    unshared = kp.BlockManager(64, bs)
    for s in range(3):
        unshared.add_sequence(s)
        unshared.append_slots(s, prompt)
    assert 64 - unshared.num_free_blocks()[0] == 21

    bm = kp.BlockManager(64, bs)
    bm.add_sequence(0)
    assert bm.append_slots(0, prompt) is None
    bm.fork(0, 1)
    bm.fork(0, 2)
    assert 64 - bm.num_free_blocks()[0] == 7
    table = bm.block_table(0)
    assert len(table) == 7 and all(bm.refcount(b) == 3 for b in table)
    last = table[-1]
    copies = [bm.append_slots(s, 1) for s in range(3)]
    # the first two writers copy the shared, partly filled last block; the third writes in place
    assert copies[0] is not None and copies[0][0] == last
    assert copies[1] is not None and copies[1][0] == last
    assert copies[2] is None
    assert bm.refcount(last) == 1 and bm.block_table(2)[-1] == last
    assert 64 - bm.num_free_blocks()[0] == 9
    for s in range(3):
        assert bm.sequence_info(s) == (101, 7)
        assert bm.block_table(s)[:6] == table[:6]
    for b in table[:6]:
        assert bm.refcount(b) == 3
    for s in range(3):
        bm.free_sequence(s)
    assert bm.num_free_blocks() == (64, 0)


def test_copy_on_write_only_for_a_partly_filled_shared_block():
    bm = kp.BlockManager(16, 4)
    bm.add_sequence(0)
    bm.append_slots(0, 8)                     # two full blocks
    bm.fork(0, 1)
    assert bm.append_slots(1, 1) is None      # new block, nothing shared is written
    t0, t1 = bm.block_table(0), bm.block_table(1)
    assert t1[:2] == t0 and len(t1) == 3 and bm.refcount(t1[2]) == 1


# ---------------------------------------------------------------------------
# Paging memory: allocation on demand wastes less than one block per sequence
# ---------------------------------------------------------------------------
def test_paging_simulation_matches_the_page():
    rng = np.random.default_rng(1)
    live = rng.integers(100, 3000, size=200)
    block = 16
    assert int(live.sum()) == 322055 and 8192 * len(live) == 1638400
    bm = kp.BlockManager(21000, block)
    for i, n in enumerate(live):
        bm.add_sequence(i)
        bm.append_slots(i, int(n))
    held = 21000 - bm.num_free_blocks()[0]
    assert held * block == 323568
    assert f"{live.sum() / (8192 * len(live)):.1%}" == "19.7%"
    assert f"{live.sum() / (held * block):.1%}" == "99.5%"
    for i, n in enumerate(live):
        toks, nb = bm.sequence_info(i)
        assert toks == n and 0 <= nb * block - n < block


def test_one_token_at_a_time_equals_one_bulk_append():
    a, b = kp.BlockManager(64, 16), kp.BlockManager(64, 16)
    a.add_sequence(7)
    b.add_sequence(7)
    a.append_slots(7, 37)
    for _ in range(37):
        b.append_slots(7, 1)
    assert a.block_table(7) == b.block_table(7) and a.sequence_info(7) == (37, 3)


# ---------------------------------------------------------------------------
# Free-list order, exhaustion, tables
# ---------------------------------------------------------------------------
def test_fifo_and_lifo_free_lists():
    # FIFO takes the oldest free block; LIFO the most recently returned one
    for lifo, first, second in ((False, [0, 1, 2], [3, 4, 5]), (True, [5, 4, 3], [3, 4, 5])):
        bm = kp.BlockManager(6, 2, lifo=lifo)
        bm.add_sequence(0)
        bm.append_slots(0, 6)
        assert bm.block_table(0) == first
        bm.free_sequence(0)
        bm.add_sequence(1)
        bm.append_slots(1, 6)
        assert bm.block_table(1) == second


def test_out_of_blocks_is_all_or_nothing():
    bm = kp.BlockManager(4, 4)
    bm.add_sequence(0)
    bm.append_slots(0, 10)                    # 3 blocks
    before = (bm.block_table(0), bm.sequence_info(0), bm.num_free_blocks())
    with pytest.raises(kp.KVError) as e:
        bm.append_slots(0, 7)                 # needs 2 more, 1 free
    assert e.value.status == kp.KV_ERR_OUT_OF_BLOCKS
    assert (bm.block_table(0), bm.sequence_info(0), bm.num_free_blocks()) == before
    bm.append_slots(0, 6)                     # exactly fills the pool
    assert bm.num_free_blocks() == (0, 0) and bm.sequence_info(0) == (16, 4)
    with pytest.raises(kp.KVError):
        bm.append_slots(0, 1)


def test_copy_on_write_counts_against_the_free_blocks():
    bm = kp.BlockManager(2, 4)
    bm.add_sequence(0)
    bm.append_slots(0, 3)
    bm.fork(0, 1)
    assert bm.append_slots(0, 1) is not None  # takes the last free block
    with pytest.raises(kp.KVError):
        bm.append_slots(1, 2)                 # in place, but then needs a new block: none
    assert bm.sequence_info(1) == (3, 1)


def test_build_tables_pads_with_minus_one():
    bm = kp.BlockManager(8, 4)
    for s, n in ((10, 5), (11, 0), (12, 9)):
        bm.add_sequence(s)
        bm.append_slots(s, n)
    tables, lens = bm.build_tables([12, 11, 10], 4)
    assert lens.tolist() == [9, 0, 5]
    assert tables.tolist() == [bm.block_table(12) + [-1], [-1] * 4, bm.block_table(10) + [-1, -1]]
    with pytest.raises(kp.KVError):
        bm.build_tables([12], 2)              # holds 3 blocks
    with pytest.raises(kp.KVError):
        bm.build_tables([99], 4)


def test_bad_arguments_are_rejected():
    with pytest.raises(kp.KVError):
        kp.BlockManager(0, 4)
    bm = kp.BlockManager(4, 4)
    bm.add_sequence(1)
    with pytest.raises(kp.KVError):
        bm.add_sequence(1)
    with pytest.raises(kp.KVError):
        bm.append_slots(2, 1)
    with pytest.raises(kp.KVError):
        bm.fork(2, 3)
    with pytest.raises(kp.KVError):
        bm.fork(1, 1)
    with pytest.raises(kp.KVError):
        bm.free_sequence(2)
    with pytest.raises(kp.KVError):
        bm.refcount(4)


# ---------------------------------------------------------------------------
# Automatic prefix caching
# ---------------------------------------------------------------------------
def serve(bm, seq, prompt, salt=0, generated=0):
    """Admit a request: reuse cached blocks, prefill the rest, decode, finish.
    Returns the number of prompt tokens prefilled."""
    bm.add_sequence(seq, salt)
    hit = bm.match_prefix(seq, prompt)
    bm.append_slots(seq, len(prompt) - hit, prompt[hit:])
    for t in range(generated):
        bm.append_slots(seq, 1, [10_000 + t])
    table = bm.block_table(seq)
    bm.free_sequence(seq)
    return len(prompt) - hit, table


def test_prefix_caching_figure_example():
    A, B, C, D, E = ([i] * 4 for i in (1, 2, 3, 4, 5))
    bm = kp.BlockManager(16, 4, prefix_caching=True)
    p1, t1 = serve(bm, 1, A + B + C)
    assert p1 == 12
    p2, t2 = serve(bm, 2, A + B + D)
    assert p2 == 4 and t2[:2] == t1[:2] and t2[2] != t1[2]
    p3, t3 = serve(bm, 3, A + E + C)
    # same tokens as request 1's last block, but the chain differs after block 2
    assert p3 == 8 and t3[0] == t1[0] and t3[1] not in t1 and t3[2] != t1[2]


def test_a_changed_early_token_breaks_the_chain():
    bm = kp.BlockManager(32, 4, prefix_caching=True)
    prompt = list(range(100, 124))
    assert serve(bm, 1, prompt)[0] == 24
    assert serve(bm, 2, prompt)[0] == 0
    changed = list(prompt)
    changed[5] = 7
    assert serve(bm, 3, changed)[0] == 20       # only block 0 matches
    assert serve(bm, 4, prompt[:22])[0] == 2    # only full blocks are reused


def test_running_sequences_share_cached_blocks_with_counts():
    bm = kp.BlockManager(16, 4, prefix_caching=True)
    sys_prompt = list(range(50, 58))
    bm.add_sequence(1)
    bm.append_slots(1, 10, sys_prompt + [1, 2])
    bm.add_sequence(2)
    assert bm.match_prefix(2, sys_prompt + [3, 4]) == 8
    shared = bm.block_table(1)[:2]
    assert bm.block_table(2) == shared and all(bm.refcount(b) == 2 for b in shared)
    bm.append_slots(2, 2, [3, 4])
    bm.free_sequence(1)
    assert all(bm.refcount(b) == 1 for b in shared)
    bm.free_sequence(2)
    free, cached = bm.num_free_blocks()
    assert cached == 2 and free + cached == 16   # partial blocks are never cached


def test_salt_isolates_tenants():
    bm = kp.BlockManager(16, 4, prefix_caching=True)
    prompt = list(range(8))
    assert serve(bm, 1, prompt, salt=111)[0] == 8
    assert serve(bm, 2, prompt, salt=222)[0] == 8
    assert serve(bm, 3, prompt, salt=111)[0] == 0
    assert serve(bm, 4, prompt, salt=222)[0] == 0
    assert serve(bm, 5, prompt)[0] == 8


def test_lru_eviction_order():
    bm = kp.BlockManager(6, 2, prefix_caching=True)
    a, b = [1, 1, 2, 2, 3, 3], [7, 7, 8, 8, 9, 9]
    _, ta = serve(bm, 1, a)
    _, tb = serve(bm, 2, b)
    assert bm.num_free_blocks() == (0, 6)
    assert serve(bm, 3, a)[0] == 0              # touches a: b is now least recently used
    bm.add_sequence(4)
    bm.append_slots(4, 2, [5, 5])               # evicts b's last block first
    assert bm.block_table(4) == [tb[2]]
    bm.append_slots(4, 2, [6, 6])
    assert bm.block_table(4) == [tb[2], tb[1]]
    bm.free_sequence(4)
    bm.add_sequence(5)
    assert bm.match_prefix(5, b) == 2           # b's first block survived
    bm.free_sequence(5)
    bm.add_sequence(6)
    assert bm.match_prefix(6, a) == 6           # a survived whole


def test_without_prefix_caching_nothing_is_reused():
    bm = kp.BlockManager(16, 4)
    prompt = list(range(12))
    assert serve(bm, 1, prompt)[0] == 12
    assert serve(bm, 2, prompt)[0] == 12
    assert bm.num_free_blocks() == (16, 0)


def test_randomised_bookkeeping_invariants():
    rng = np.random.default_rng(5)
    nb, bs = 40, 4
    bm = kp.BlockManager(nb, bs, prefix_caching=True)
    live, model, next_id = {}, {}, 0
    for it in range(600):
        op = rng.integers(0, 4)
        if op == 0 or not live:
            prompt = [int(x) for x in rng.integers(0, 3, size=int(rng.integers(1, 14)))]
            bm.add_sequence(next_id)
            hit = bm.match_prefix(next_id, prompt)
            assert hit % bs == 0 and hit <= len(prompt)
            try:
                bm.append_slots(next_id, len(prompt) - hit, prompt[hit:])
            except kp.KVError:
                bm.free_sequence(next_id)
            else:
                live[next_id] = len(prompt)
            next_id += 1
        elif op == 1:
            s = int(rng.choice(list(live)))
            try:
                bm.append_slots(s, 1, [int(rng.integers(0, 3))])
                live[s] += 1
            except kp.KVError:
                pass
        elif op == 2:
            s = int(rng.choice(list(live)))
            try:
                bm.append_slots(s, 0)
                bm.fork(s, next_id)
                live[next_id] = live[s]
                next_id += 1
            except kp.KVError:
                pass
        else:
            s = int(rng.choice(list(live)))
            bm.free_sequence(s)
            del live[s]
        # invariants: counts equal the number of tables holding a block; every
        # block is held, free or cached-and-evictable; no sequence exceeds its tokens
        refs = np.zeros(nb, dtype=int)
        for s, n in live.items():
            table = bm.block_table(s)
            assert bm.sequence_info(s) == (n, blocks_needed(n, bs))
            for b in table:
                refs[b] += 1
        for b in range(nb):
            assert bm.refcount(b) == refs[b]
        free, cached = bm.num_free_blocks()
        assert int((refs > 0).sum()) + free + cached == nb


def test_match_prefix_equals_brute_force_longest_cached_prefix():
    # brunomaga.github.io, "Prefix caching": the lookup walks full blocks from the
    # start and stops at the first miss; a block matches only when the whole prefix
    # up to its end matches.  Brute force: the longest full-block prefix of the
    # prompt that equals the prefix of something served before (pool never full).
    rng = np.random.default_rng(9)
    bs = 4
    bm = kp.BlockManager(4096, bs, prefix_caching=True)
    served = []
    for seq in range(300):
        if served and rng.random() < 0.7:
            base = served[int(rng.integers(0, len(served)))]
            cut = int(rng.integers(0, len(base) + 1))
            prompt = base[:cut] + [int(x) for x in rng.integers(0, 3, size=int(rng.integers(0, 9)))]
        else:
            prompt = [int(x) for x in rng.integers(0, 3, size=int(rng.integers(1, 20)))]
        if not prompt:
            prompt = [0]
        best = 0
        for old in served:
            n = 0
            while (n + bs <= min(len(old), len(prompt))
                   and old[n:n + bs] == prompt[n:n + bs]):
                n += bs
            best = max(best, n)
        bm.add_sequence(seq)
        assert bm.match_prefix(seq, prompt) == best
        bm.append_slots(seq, len(prompt) - best, prompt[best:])
        gen = [int(x) for x in rng.integers(0, 3, size=int(rng.integers(0, 6)))]
        for t in gen:
            bm.append_slots(seq, 1, [t])
        bm.free_sequence(seq)
        served.append(prompt + gen)
