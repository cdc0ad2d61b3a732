"""GPU checks of the block manager driving the kernels: copy-on-write copies
(kv_copy_blocks) bit for bit, and decode attention over tables the manager
builds -- parallel sampling with forks and prefix reuse across requests --
against the float64 oracle on each sequence's own contiguous keys and values."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import MAX_ABS, REL_L2, bf16_tensor, compare, i32

pytestmark = pytest.mark.gpu

HQ, HKV, D = 8, 2, 128


def rows(rng, n):
    return workloads.f32_to_bf16_bits(rng.standard_normal((n, HKV, D)).astype(np.float32))


def write(pool, seq_tables, k_bits, v_bits, seq_index, positions):
    tables, ctx = seq_tables
    n = len(positions)
    kp.paged_kv_append(pool, bf16_tensor(k_bits), bf16_tensor(v_bits), i32(tables).cuda(),
                       i32(ctx).cuda(), token_seq=i32(np.full(n, seq_index)),
                       token_pos=i32(positions))


def check_decode(pool, tables, ctx, per_seq_k, per_seq_v, rng):
    """Decode one query per sequence through the tables and compare with the oracle
    on the sequences' own contiguous K/V."""
    batch = len(per_seq_k)
    q = workloads.f32_to_bf16_bits(rng.standard_normal((batch, HQ, D)).astype(np.float32))
    scale = 1.0 / math.sqrt(D)
    out = torch.empty(batch, HQ, D, dtype=torch.bfloat16, device="cuda")
    kp.paged_decode_attention(pool, bf16_tensor(q), i32(tables), i32(ctx), scale, out=out)
    k_all = np.concatenate(per_seq_k)
    v_all = np.concatenate(per_seq_v)
    lens = np.array([len(k) for k in per_seq_k], dtype=np.int32)
    assert (lens == ctx).all()
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    ref, _ = oracle.decode(q, k_all, v_all, starts, lens, q_heads=HQ, kv_heads=HKV, head_dim=D,
                           scale=scale)
    max_abs, rel, _ = compare(out, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)


def pool_rows(pool, table, n):
    """The K and V bits of a sequence's first n tokens, read from the pool on the host."""
    k, v, _, _ = pool.tensors()
    bs = k.shape[1]
    kh = k.view(torch.int16).cpu().numpy().view(np.uint16)
    vh = v.view(torch.int16).cpu().numpy().view(np.uint16)
    idx = [(table[p // bs], p % bs) for p in range(n)]
    return (np.stack([kh[b, s] for b, s in idx]), np.stack([vh[b, s] for b, s in idx]))


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_copy_blocks_bit_exact_and_bad_ids_flagged(dtype):
    rng = np.random.default_rng(31)
    nb, bs = 12, 16
    pool = kp.kv_pool_create(nb, bs, HKV, D, dtype)
    kr, vr = pool.raw_bytes()
    k0 = rng.integers(0, 256, size=tuple(kr.shape), dtype=np.uint8)
    v0 = rng.integers(0, 256, size=tuple(vr.shape), dtype=np.uint8)
    kr.copy_(torch.from_numpy(k0))
    vr.copy_(torch.from_numpy(v0))
    pairs = np.array([[3, 7], [0, 11], [5, 1], [nb, 2], [4, -1]], dtype=np.int32)
    kp.kv_copy_blocks(pool, i32(pairs))
    torch.cuda.synchronize()
    ke, ve = k0.copy(), v0.copy()
    for s, d in pairs[:3]:
        ke[d], ve[d] = k0[s], v0[s]
    assert np.array_equal(kr.cpu().numpy(), ke) and np.array_equal(vr.cpu().numpy(), ve)
    assert pool.device_errors() & kp.DEVERR_BLOCK_ID
    kp.kv_copy_blocks(pool, i32(np.zeros((0, 2))))     # no-op
    assert pool.device_errors() == 0
    pool.destroy()


def test_parallel_sampling_with_copy_on_write_decodes_each_sample():
    rng = np.random.default_rng(32)
    bs, nb, prompt, samples, steps = 16, 48, 100, 3, 20
    pool = kp.kv_pool_create(nb, bs, HKV, D, "bf16")
    for t in pool.raw_bytes():
        t.fill_(workloads.POISON_BYTE)
    bm = kp.BlockManager(nb, bs)
    bm.add_sequence(0)
    bm.append_slots(0, prompt)
    pk, pv = rows(rng, prompt), rows(rng, prompt)
    write(pool, bm.build_tables([0], 8), pk, pv, 0, np.arange(prompt))
    for s in range(1, samples):
        bm.fork(0, s)
    ks = [[pk] for _ in range(samples)]
    vs = [[pv] for _ in range(samples)]
    seqs = list(range(samples))
    n_copies = 0
    for step in range(steps):
        copies = [c for c in (bm.append_slots(s, 1) for s in seqs) if c is not None]
        n_copies += len(copies)
        if copies:
            kp.kv_copy_blocks(pool, i32(np.array(copies)))
        tables, ctx = bm.build_tables(seqs, 8)
        kn, vn = rows(rng, samples), rows(rng, samples)
        kp.paged_kv_append(pool, bf16_tensor(kn), bf16_tensor(vn), i32(tables), i32(ctx))
        for s in seqs:
            ks[s].append(kn[s:s + 1])
            vs[s].append(vn[s:s + 1])
        if step in (0, 11, steps - 1):
            check_decode(pool, tables, ctx, [np.concatenate(k) for k in ks],
                         [np.concatenate(v) for v in vs], rng)
    assert n_copies == samples - 1
    # every sample's tokens sit bit for bit where its table says
    for s in seqs:
        got_k, got_v = pool_rows(pool, bm.block_table(s), prompt + steps)
        assert np.array_equal(got_k, np.concatenate(ks[s]))
        assert np.array_equal(got_v, np.concatenate(vs[s]))
    assert pool.device_errors() == 0
    pool.destroy()


def test_prefix_reuse_across_requests_and_after_eviction():
    rng = np.random.default_rng(33)
    bs, nb = 16, 10
    pool = kp.kv_pool_create(nb, bs, HKV, D, "bf16")
    for t in pool.raw_bytes():
        t.fill_(workloads.POISON_BYTE)
    bm = kp.BlockManager(nb, bs, prefix_caching=True)

    # a prefix's K/V is a function of its tokens: same leading tokens, same rows
    ids1 = [int(x) for x in rng.integers(0, 1000, size=40)]
    k1, v1 = rows(rng, 40), rows(rng, 40)
    ids2 = ids1[:32] + [int(x) for x in rng.integers(1000, 2000, size=21)]
    k2 = np.concatenate([k1[:32], rows(rng, 21)])
    v2 = np.concatenate([v1[:32], rows(rng, 21)])

    def serve(seq, ids, k, v, expect_hit):
        bm.add_sequence(seq)
        hit = bm.match_prefix(seq, ids)
        assert hit == expect_hit
        bm.append_slots(seq, len(ids) - hit, ids[hit:])
        tables, ctx = bm.build_tables([seq], 8)
        write(pool, (tables, ctx), k[hit:], v[hit:], 0, np.arange(hit, len(ids)))
        check_decode(pool, tables, ctx, [k], [v], rng)
        table = bm.block_table(seq)
        bm.free_sequence(seq)
        return table

    t1 = serve(1, ids1, k1, v1, 0)
    t2 = serve(2, ids2, k2, v2, 32)                 # two full blocks of request 1
    assert t2[:2] == t1[:2]
    # a burst of unrelated requests evicts everything cached
    bm.add_sequence(3)
    bm.append_slots(3, nb * bs)
    bm.free_sequence(3)
    serve(4, ids2, k2, v2, 0)
    assert pool.device_errors() == 0
    pool.destroy()
