"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (torch SDPA, torch's float8 / bfloat16 conversions, scipy logsumexp),
a closed form, an invariant, or a value printed on the pages (tests/golden).
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(shape, seed, scale=1.0):
    r = np.random.default_rng(seed)
    return workloads.f32_to_bf16_bits((r.standard_normal(shape) * scale).astype(np.float32))


def _f64(bits):
    return workloads.bf16_bits_to_f32(bits).astype(np.float64)


# --------------------------------------------------------------------------- formats
def test_bf16_decoder_matches_torch_on_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bf16_value(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(ours[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_decoder_matches_torch_on_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_value(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.nanmax(ours) == 448.0 and np.nanmin(ours) == -448.0
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert ours[1] == 2.0 ** -9                      # smallest subnormal


def test_e4m3_encoder_roundtrips_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_from_float(vals), codes)


def test_e4m3_encoder_matches_torch_rne_on_all_bf16_within_range():
    bits = np.arange(65536, dtype=np.uint16)
    x = workloads.bf16_bits_to_f32(bits)
    keep = np.isfinite(x) & (np.abs(x) <= 448.0)
    x = x[keep]
    ours = oracle.e4m3_from_float(x)
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encoder_saturates_beyond_448():
    x = np.array([448.5, 463.9, 464.0, 465.0, 480.0, 1e4, 3e38, -449.0, -1e30], dtype=np.float32)
    codes = oracle.e4m3_from_float(x)
    assert np.array_equal(codes[x > 0], np.full((x > 0).sum(), 0x7E, dtype=np.uint8))
    assert np.array_equal(codes[x < 0], np.full((x < 0).sum(), 0xFE, dtype=np.uint8))


def test_e4m3_quantize_divides_in_binary32_then_rounds():
    # torch: binary32 division, then RNE to e4m3 (values stay inside +-448 here)
    r = np.random.default_rng(5)
    xb = workloads.f32_to_bf16_bits(r.standard_normal(4000).astype(np.float32) * 3)
    for scale in (np.float32(0.0123), np.float32(4.5 / 448), np.float32(1.0), np.float32(0.3)):
        ours = oracle.e4m3_quantize(xb, scale)
        xt = torch.from_numpy(workloads.bf16_bits_to_f32(xb))
        q = xt / torch.tensor(scale, dtype=torch.float32)
        inside = q.abs() <= 448
        ref = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ours[inside.numpy()], ref[inside.numpy()])
        assert np.all(oracle.e4m3_value(ours[~inside.numpy()]) == np.sign(q[~inside].numpy()) * 448)


# --------------------------------------------------------------------------- addressing
def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([c.strip() for c in line.split("|")])
    return rows


def test_block_addressing_matches_the_page_examples():
    rows = _read_golden("p1_block_addresses.txt")
    assert len(rows) == 6
    hkv, d, nblk = 1, 8, 10
    for kind, bs, table, n, expected in rows:
        bs, n = int(bs), int(n)
        table = np.array([int(t) for t in table.split(",")], dtype=np.int32)[None, :]
        kp = np.full((nblk, bs, hkv, d * 2), 0xFF, dtype=np.uint8)
        vp = kp.copy()
        if kind == "fill":
            pos = np.arange(n, dtype=np.int32)
        else:
            pos = np.array([n], dtype=np.int32)
        kn = np.arange(1, pos.size * hkv * d + 1, dtype=np.uint16).reshape(pos.size, hkv, d)
        bad = oracle.append(kp, vp, "bf16", bs, kn, kn, table, np.array([pos.max() + 1]),
                            token_seq=np.zeros(pos.size, np.int32), token_pos=pos)
        assert bad == 0
        written = (kp.reshape(nblk, bs, -1) != 0xFF).any(axis=2)      # [block, slot]
        if kind == "fill":
            want = {int(a): int(b) for a, b in (p.split(":") for p in expected.split(","))}
            got = {blk: int(written[blk].sum()) for blk in range(nblk) if written[blk].any()}
            assert got == want
            for blk, cnt in want.items():          # slots fill from 0 upwards
                assert written[blk, :cnt].all()
        else:
            blk, slot = (int(x) for x in expected.split(":"))
            assert written.sum() == 1 and written[blk, slot]


def test_invalid_addresses_are_skipped_and_counted():
    kp = np.full((4, 4, 1, 4), 0xFF, dtype=np.uint8)
    vp = kp.copy()
    kn = np.ones((3, 1, 2), dtype=np.uint16)
    table = np.array([[0, 9], [1, -1]], dtype=np.int32)      # 9 and -1 are outside a 4-block pool
    bad = oracle.append(kp, vp, "bf16", 4, kn, kn, table, np.array([6, 5], np.int32),
                        token_seq=np.array([0, 1, 5], np.int32), token_pos=None)
    assert bad == 3
    assert (kp == 0xFF).all()


# --------------------------------------------------------------------------- attention
def _sdpa_causal(Q, K, V):
    # torch SDPA in float64: Q [H, T, d], K/V [H, T, d]
    return F.scaled_dot_product_attention(torch.from_numpy(Q)[None], torch.from_numpy(K)[None],
                                          torch.from_numpy(V)[None], is_causal=True)[0].numpy()


@pytest.mark.parametrize("hq,hkv,d,T", [(4, 4, 16, 37), (8, 2, 32, 50), (6, 1, 8, 20)])
def test_decode_equals_full_causal_attention(hq, hkv, d, T):
    """Decoding with a cache gives row t of full causal attention (the first page's self-check)."""
    Q = _f64(_bf16((T, hq, d), 11))
    K = _f64(_bf16((T, hkv, d), 12))
    V = _f64(_bf16((T, hkv, d), 13))
    g = hq // hkv
    # reference: GQA as MHA on K/V repeated g times per group (query head h uses kv head h // g)
    Kr = np.repeat(K, g, axis=1).transpose(1, 0, 2).copy()
    Vr = np.repeat(V, g, axis=1).transpose(1, 0, 2).copy()
    full = _sdpa_causal(Q.transpose(1, 0, 2).copy(), Kr, Vr)            # [hq, T, d]
    for t in range(1, T + 1):
        out, lse = oracle.attend(Q[t - 1], K[:t], V[:t], 1.0 / math.sqrt(d))
        assert np.max(np.abs(out - full[:, t - 1])) < 1e-13


def test_toy_layer_prefill_then_decode_through_the_paged_cache():
    """The first page's check: prefill 6 tokens, decode 4, compare with full causal attention.

    Here the keys and values go through the oracle's paged append (block size 4,
    a permuted 10-block pool) and are read back through the table by the gather.
    """
    torch.manual_seed(0)
    d, H = 64, 4
    hd = d // H
    Wq, Wk, Wv = (torch.randn(d, d, dtype=torch.float64) / 8 for _ in range(3))
    x = torch.randn(10, d, dtype=torch.float64)
    to_bits = lambda t: workloads.f32_to_bf16_bits(t.float().numpy())
    qb = to_bits((x @ Wq.T).view(10, H, hd))
    kb = to_bits((x @ Wk.T).view(10, H, hd))
    vb = to_bits((x @ Wv.T).view(10, H, hd))
    Qf, Kf, Vf = _f64(qb), _f64(kb), _f64(vb)
    ref = _sdpa_causal(Qf.transpose(1, 0, 2).copy(), Kf.transpose(1, 0, 2).copy(),
                       Vf.transpose(1, 0, 2).copy())                  # [H, 10, hd]
    table = np.array([[6, 2, 9]], dtype=np.int32)
    kp = np.full((10, 4, H, hd * 2), 0xFF, dtype=np.uint8)
    vp = kp.copy()
    oracle.append(kp, vp, "bf16", 4, kb[:6], vb[:6], table, np.array([6], np.int32),
                  token_seq=np.zeros(6, np.int32), token_pos=np.arange(6, dtype=np.int32))
    worst = 0.0
    for t in range(6, 10):          # decode: append the new token first, then attend
        oracle.append(kp, vp, "bf16", 4, kb[t:t + 1], vb[t:t + 1], table,
                      np.array([t + 1], np.int32))
        K = oracle.gather(kp, "bf16", table[0], t + 1)
        V = oracle.gather(vp, "bf16", table[0], t + 1)
        out, _ = oracle.attend(Qf[t], K, V, 1.0 / math.sqrt(hd))
        worst = max(worst, np.max(np.abs(out - ref[:, t])))
    assert worst < 1e-13


def test_paged_gather_equals_contiguous_cache_bit_exact():
    w = workloads.make(workloads.custom(batch=3, q_heads=4, kv_heads=2, head_dim=16, block_size=8,
                                        ctx=[1, 8, 29], seed=21))
    kp, vp = oracle.pool_image(w, after_step=True)
    for b in range(w.batch):
        n = int(w.context_lens[b])
        K = oracle.gather(kp, "bf16", w.block_tables[b], n)
        V = oracle.gather(vp, "bf16", w.block_tables[b], n)
        assert np.array_equal(K, _f64(w.seq_k(b)))
        assert np.array_equal(V, _f64(w.seq_v(b)))


def test_block_permutation_invariance_bit_exact():
    w = workloads.make(workloads.custom(batch=2, q_heads=4, kv_heads=2, head_dim=16, block_size=4,
                                        ctx=[13, 22], seed=22, pool_blocks=16))
    kp, vp = oracle.pool_image(w, after_step=True)
    perm = np.random.default_rng(3).permutation(w.num_blocks)       # new id of old block i
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    t2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    q = _f64(w.q)
    for b in range(w.batch):
        n = int(w.context_lens[b])
        a = oracle.attend(q[b], oracle.gather(kp, "bf16", w.block_tables[b], n),
                          oracle.gather(vp, "bf16", w.block_tables[b], n), w.scale)
        c = oracle.attend(q[b], oracle.gather(kp2, "bf16", t2[b], n),
                          oracle.gather(vp2, "bf16", t2[b], n), w.scale)
        assert np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1])


def test_batch_independence_bit_exact():
    w = workloads.make(workloads.custom(batch=5, q_heads=8, kv_heads=2, head_dim=16, block_size=16,
                                        ctx=[3, 40, 17, 1, 64], seed=23))
    out, lse = oracle.decode_workload(w, threads=3)
    for b in range(w.batch):
        o1, l1 = oracle.decode_workload(w, seqs=[b])
        assert np.array_equal(out[b], o1[0]) and np.array_equal(lse[b], l1[0])


def test_single_token_context_returns_its_value():
    q = _f64(_bf16((8, 32), 31))
    k = _f64(_bf16((1, 2, 32), 32))
    v = _f64(_bf16((1, 2, 32), 33))
    out, lse = oracle.attend(q, k, v, 0.25)
    for h in range(8):
        assert np.array_equal(out[h], v[0, h // 4])
        assert lse[h] == pytest.approx(0.25 * float(q[h] @ k[0, h // 4]), abs=1e-14)


def test_identical_keys_give_the_mean_of_values():
    q = _f64(_bf16((4, 16), 34))
    k = np.repeat(_f64(_bf16((1, 1, 16), 35)), 50, axis=0)
    v = _f64(_bf16((50, 1, 16), 36))
    out, lse = oracle.attend(q, k, v, 0.25)
    for h in range(4):
        assert np.max(np.abs(out[h] - v[:, 0].mean(axis=0))) < 1e-14
        assert lse[h] == pytest.approx(0.25 * float(q[h] @ k[0, 0]) + math.log(50), abs=1e-12)


def test_gqa_equals_mha_on_repeated_kv_bit_exact():
    q = _f64(_bf16((12, 16), 37))
    k = _f64(_bf16((23, 3, 16), 38))
    v = _f64(_bf16((23, 3, 16), 39))
    a = oracle.attend(q, k, v, 0.3)
    b = oracle.attend(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), 0.3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_lse_and_weights_against_library_logsumexp():
    q = _f64(_bf16((2, 16), 40))
    k = _f64(_bf16((300, 1, 16), 41, scale=3.0))
    v = np.eye(300)[:, None, :16].repeat(1, axis=1).copy()       # not used for the weights
    s = 0.25 * (k[:, 0] @ q.T)                                    # [300, 2] scores (numpy matmul)
    _, lse = oracle.attend(q, k, _f64(_bf16((300, 1, 16), 42)), 0.25)
    assert np.allclose(lse, logsumexp(s, axis=0), rtol=0, atol=1e-12)
    # weights sum to one: with V = one-hot rows the outputs are the weights themselves
    V1 = np.zeros((16, 1, 16))
    V1[np.arange(16), 0, np.arange(16)] = 1.0
    out, _ = oracle.attend(q, k[:16], V1, 0.25)
    assert np.all(np.abs(out.sum(axis=1) - 1.0) < 1e-12)
    del v


def test_shift_invariance():
    q = _f64(_bf16((4, 16), 43))
    k = _f64(_bf16((40, 1, 16), 44))
    v = _f64(_bf16((40, 1, 16), 45))
    w = np.zeros(16)
    w[3] = 1000.0                            # a common component added to every key
    out0, lse0 = oracle.attend(q, k, v, 0.25)
    out1, lse1 = oracle.attend(q, k + w, v, 0.25)
    assert np.max(np.abs(out1 - out0)) < 1e-12
    assert np.allclose(lse1 - lse0, 0.25 * q @ w, rtol=0, atol=1e-9)


@pytest.mark.parametrize("split", [1, 3, 16, 64, 1000])
def test_split_merge_equals_unsplit(split):
    q = _f64(_bf16((8, 32), 46))
    k = _f64(_bf16((157, 2, 32), 47, scale=2.0))
    v = _f64(_bf16((157, 2, 32), 48))
    o1, l1 = oracle.attend(q, k, v, 0.2)
    n = -(-157 // split)
    o2, l2 = oracle.attend_split(q, k, v, 0.2, split, n + 3)      # 3 trailing empty chunks
    assert np.max(np.abs(o2 - o1)) < 1e-12 and np.max(np.abs(l2 - l1)) < 1e-12


@pytest.mark.parametrize("cuts", [(0, 157), (0, 64, 157), (0, 0, 40, 41, 100, 157), (0, 157, 157)])
def test_merge_of_shards_equals_attention_over_all_keys(cuts):
    """A context cut into consecutive shards (some empty), attended shard by shard and merged
    from the (out, lse) pairs alone, gives attention over the whole context."""
    q = _f64(_bf16((8, 32), 51))
    k = _f64(_bf16((157, 2, 32), 52, scale=2.0))
    v = _f64(_bf16((157, 2, 32), 53))
    o_all, l_all = oracle.attend(q, k, v, 0.2)
    outs, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b > a:
            o, l = oracle.attend(q, k[a:b], v[a:b], 0.2)
        else:                                   # a shard with no key
            o, l = np.full((8, 32), np.nan), np.full(8, -np.inf)
        outs.append(o)
        lses.append(l)
    o_m, l_m = oracle.merge_states(np.stack(outs), np.stack(lses))
    assert np.max(np.abs(o_m - o_all)) < 1e-12 and np.max(np.abs(l_m - l_all)) < 1e-12


def test_merge_states_special_cases():
    rng = np.random.default_rng(54)
    o = rng.standard_normal((3, 5, 8))
    # one source: unchanged
    m1, l1 = oracle.merge_states(o[:1], np.array([[0.5, -1.0, 2.0, 0.0, 3.0]]))
    assert np.array_equal(m1, o[0]) and np.allclose(l1, [0.5, -1.0, 2.0, 0.0, 3.0], atol=1e-15)
    # equal lse: the plain mean, and lse grows by log n
    m3, l3 = oracle.merge_states(o, np.zeros((3, 5)))
    assert np.allclose(m3, o.mean(0), atol=1e-15) and np.allclose(l3, np.log(3.0), atol=1e-15)
    # weights exp(lse_r) / sum: lse (0, log 3) gives weights 1/4 and 3/4
    m2, _ = oracle.merge_states(o[:2], np.stack([np.zeros(5), np.full(5, np.log(3.0))]))
    assert np.allclose(m2, 0.25 * o[0] + 0.75 * o[1], atol=1e-14)
    # a row whose sources are all empty: out 0, lse -inf
    me, le = oracle.merge_states(o[:2], np.full((2, 5), -np.inf))
    assert np.array_equal(me, np.zeros((5, 8))) and np.all(le == -np.inf)


def test_empty_context_attends_to_nothing():
    q = _f64(_bf16((4, 8), 49))
    out, lse = oracle.attend(q, np.zeros((0, 2, 8)), np.zeros((0, 2, 8)), 0.5)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_padded_masked_library_attention_matches_oracle_decode():
    """The second page's batched form: gather into a padded tensor, mask past each length, softmax."""
    w = workloads.make(workloads.custom(batch=4, q_heads=8, kv_heads=2, head_dim=16, block_size=4,
                                        ctx=[1, 5, 12, 30], seed=24))
    out, _ = oracle.decode_workload(w)
    L = int(w.context_lens.max())
    g = 4
    Kp = np.zeros((w.batch, 8, L, 16))
    Vp = np.zeros((w.batch, 8, L, 16))
    for b in range(w.batch):
        n = int(w.context_lens[b])
        Kp[b, :, :n] = np.repeat(_f64(w.seq_k(b)), g, axis=1).transpose(1, 0, 2)
        Vp[b, :, :n] = np.repeat(_f64(w.seq_v(b)), g, axis=1).transpose(1, 0, 2)
    mask = torch.arange(L)[None, :] < torch.from_numpy(w.context_lens.astype(np.int64))[:, None]
    ref = F.scaled_dot_product_attention(torch.from_numpy(_f64(w.q))[:, :, None],
                                         torch.from_numpy(Kp), torch.from_numpy(Vp),
                                         attn_mask=mask[:, None, None, :], scale=w.scale)[:, :, 0]
    assert np.max(np.abs(out - ref.numpy())) < 1e-13


def test_fp8_decode_uses_dequantised_codes():
    w = workloads.make(workloads.custom(batch=2, q_heads=2, kv_heads=2, head_dim=16, block_size=8,
                                        ctx=[9, 20], seed=25, cache_dtype="fp8_e4m3"))
    out, _ = oracle.decode_workload(w)
    for b in range(w.batch):
        n = int(w.context_lens[b])
        kq = np.stack([oracle.e4m3_value(oracle.e4m3_quantize(w.seq_k(b)[:, h], w.k_scale[h]))
                       * np.float64(w.k_scale[h]) for h in range(2)], axis=1)
        vq = np.stack([oracle.e4m3_value(oracle.e4m3_quantize(w.seq_v(b)[:, h], w.v_scale[h]))
                       * np.float64(w.v_scale[h]) for h in range(2)], axis=1)
        ref = F.scaled_dot_product_attention(torch.from_numpy(_f64(w.q[b]))[:, None],
                                             torch.from_numpy(kq.transpose(1, 0, 2).copy()),
                                             torch.from_numpy(vq.transpose(1, 0, 2).copy()),
                                             scale=w.scale)[:, 0]
        assert np.max(np.abs(out[b] - ref.numpy())) < 1e-13
        assert n == kq.shape[0]
    # the pool image holds exactly those codes
    kp, _ = oracle.pool_image(w, after_step=True)
    blk, slot = w.block_tables[1, 19 // 8], 19 % 8
    assert np.array_equal(kp[blk, slot, 0],
                          oracle.e4m3_quantize(w.seq_k(1)[19, 0], w.k_scale[0]))


# --------------------------------------------------------------------------- several new tokens
def test_multi_query_visibility_matches_the_printed_masks():
    """With q = 0 every visible key gets the same weight; one-hot values reveal which keys."""
    rows = _read_golden("p4_shifted_masks.txt")
    assert len(rows) == 2
    for start, T, masks in rows:
        start, T = int(start), int(T)
        want = np.array([[int(ch) for ch in m] for m in masks.split(";")], dtype=float)
        ctx = start + T
        d = 8
        v = np.zeros((ctx, 1, d), dtype=np.uint16)
        for t in range(ctx):                                # one-hot rows (bf16 1.0 = 0x3F80)
            v[t, 0, t] = 0x3F80
        k = _bf16((ctx, 1, d), 50)
        q = np.zeros((1, 1, T, d), dtype=np.uint16)
        out, _ = oracle.decode_multi(q, k, v, np.array([0]), np.array([ctx], np.int32), q_heads=1,
                                     q_len=T, kv_heads=1, head_dim=d, scale=0.5)
        seen = (out[0, 0, :, :ctx] > 0).astype(float)
        assert np.array_equal(seen, want)
        assert np.allclose(out[0, 0, :, :ctx].sum(axis=1), 1.0)


@pytest.mark.parametrize("hq,hkv,t", [(4, 4, 3), (8, 2, 5)])
def test_multi_query_equals_the_last_rows_of_full_causal_attention(hq, hkv, t):
    T, d = 29, 16
    Q = _f64(_bf16((T, hq, d), 51))
    Kb, Vb = _bf16((T, hkv, d), 52), _bf16((T, hkv, d), 53)
    K, V = _f64(Kb), _f64(Vb)
    g = hq // hkv
    full = _sdpa_causal(Q.transpose(1, 0, 2).copy(), np.repeat(K, g, axis=1).transpose(1, 0, 2).copy(),
                        np.repeat(V, g, axis=1).transpose(1, 0, 2).copy())           # [hq, T, d]
    qb = _bf16((T, hq, d), 51)[T - t:].transpose(1, 0, 2)[None].copy()              # [1, hq, t, d]
    out, _ = oracle.decode_multi(qb, Kb, Vb, np.array([0]), np.array([T], np.int32), q_heads=hq,
                                 q_len=t, kv_heads=hkv, head_dim=d, scale=1 / math.sqrt(d))
    assert np.max(np.abs(out[0] - full[:, T - t:])) < 1e-13


def test_multi_query_of_one_token_is_the_decode():
    w = workloads.make(workloads.custom(batch=3, q_heads=8, kv_heads=2, head_dim=16, block_size=8,
                                        ctx=[1, 9, 30], seed=54))
    a, la = oracle.decode_workload(w)
    b, lb = oracle.decode_multi_workload(w, w.q[:, :, None, :], 1)
    assert np.array_equal(a, b[:, :, 0]) and np.array_equal(la, lb[:, :, 0])


# --------------------------------------------------------------------------- MLA (absorbed)
# xuewyang.github.io/posts/kv, "MLA: how does decode get full-size keys and values back?":
# folding W_UK into the query and W_UV into the output gives the same result as rebuilding
# every head's keys and values from the cached latents (the page's float32 check prints a
# difference of 4.5e-07); DeepSeek-V2 caches 512 latent + 64 rotary-key numbers per token.
@pytest.mark.parametrize("heads,dh,dl,dr,ctx", [(4, 16, 32, 8, 23), (3, 8, 24, 0, 5),
                                                (2, 32, 64, 16, 1)])
def test_mla_absorbed_equals_expanded_attention(heads, dh, dl, dr, ctx):
    r = np.random.default_rng(heads * 100 + ctx)
    w_uk = r.standard_normal((heads, dh, dl)) / math.sqrt(dl)
    w_uv = r.standard_normal((heads, dh, dl)) / math.sqrt(dl)
    lat = r.standard_normal((ctx, dl))
    rope_k = r.standard_normal((ctx, dr))
    q_nope = r.standard_normal((heads, dh))
    q_rope = r.standard_normal((heads, dr))
    scale = 1.0 / math.sqrt(dh + dr)
    # (a) expand: per head, full keys [W_UK c ; k_rope] and values W_UV c, normal attention
    out_a, lse_a = np.zeros((heads, dh)), np.zeros(heads)
    for h in range(heads):
        k_h = np.concatenate([lat @ w_uk[h].T, rope_k], axis=1)[:, None, :]
        v_h = np.concatenate([lat @ w_uv[h].T, np.zeros((ctx, dr))], axis=1)[:, None, :]
        q_h = np.concatenate([q_nope[h], q_rope[h]])[None, :]
        o, l = oracle.attend(q_h, k_h, v_h, scale)
        out_a[h], lse_a[h] = o[0, :dh], l[0]
    # (b) absorb: q into latent space, attend over the cached vectors, project up once
    q_lat = np.concatenate([np.einsum("hkc,hk->hc", w_uk, q_nope), q_rope], axis=1)
    o_lat, lse_b = oracle.mla_attend(q_lat, np.concatenate([lat, rope_k], axis=1), dl, scale)
    out_b = np.einsum("hkc,hc->hk", w_uv, o_lat)
    assert np.max(np.abs(out_a - out_b)) < 1e-12
    assert np.max(np.abs(lse_a - lse_b)) < 1e-12


def test_mla_matches_torch_sdpa_with_a_narrower_value():
    r = np.random.default_rng(77)
    heads, dl, dr, ctx = 5, 48, 16, 37
    q = r.standard_normal((heads, dl + dr))
    cache = r.standard_normal((ctx, dl + dr))
    scale = 0.11
    out, lse = oracle.mla_attend(q, cache, dl, scale)
    qt = torch.from_numpy(q)[:, None, :]                       # [H, 1, dk]
    kt = torch.from_numpy(cache)[None].expand(heads, ctx, dl + dr)
    vt = torch.from_numpy(cache[:, :dl])[None].expand(heads, ctx, dl)
    ref = F.scaled_dot_product_attention(qt, kt, vt, scale=scale)[:, 0]
    assert np.max(np.abs(out - ref.numpy())) < 1e-12
    s = scale * (q @ cache.T)
    assert np.max(np.abs(lse - logsumexp(s, axis=1))) < 1e-12


def test_mla_decode_batch_is_single_kv_head_decode_with_key_equal_value():
    # bf16 batch form against the (pinned) GQA decode with one kv head whose key and
    # value are both the cached vector; the MLA output is its first dl numbers
    heads, dl, dr = 8, 64, 16
    ctx = np.array([1, 17, 40, 0], dtype=np.int32)
    starts = np.concatenate([[0], np.cumsum(ctx)[:-1]]).astype(np.int64)
    cache = _bf16((int(ctx.sum()), dl + dr), 5)
    q = _bf16((ctx.size, heads, dl + dr), 6)
    scale = 1.0 / math.sqrt(dl + dr)
    out, lse = oracle.mla_decode(q, cache, starts, ctx, latent_dim=dl, scale=scale)
    ref, ref_lse = oracle.decode(q, cache[:, None, :], cache[:, None, :], starts, ctx,
                                 q_heads=heads, kv_heads=1, head_dim=dl + dr, scale=scale)
    assert np.array_equal(out, ref[:, :, :dl])
    assert np.array_equal(lse, ref_lse)
    assert np.all(out[3] == 0) and np.all(np.isneginf(lse[3]))


def test_mla_cache_numbers_per_token():
    # 512 + 64 = 576 numbers per token and layer against 2 x 128 heads x 128 for MHA
    from workloads import accounting
    assert accounting.mla_numbers_per_token(512, 64) == 576
    assert 2 * 128 * 128 == 32768
    assert accounting.mla_bytes_per_token(512, 64, 2) == 1152
