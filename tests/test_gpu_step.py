"""GPU parity of paged_decode_step: the append of the step's new tokens and their attention
in one call (for K/V pools one kernel, whose CTAs write the new rows of the blocks they read
before loading them; for latent pools the append kernel, then the attention streaming the
blocks the append does not touch while it runs).

The pool after the step must equal the oracle's append image bit for bit, the outputs the
oracle within the attention tolerances, and both must be bit-identical to the separate
paged_kv_append + attention calls.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import LSE_ABS, MAX_ABS, REL_L2, Staged, compare, i32

pytestmark = pytest.mark.gpu

C = workloads.custom
STEP = {
    "tiny": workloads.CONFIGS["tiny"],
    "g4_one_chunk": C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                      ctx=[1, 16, 203], seed=301),
    "g8_split64": C(batch=3, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                    ctx=[37, 300, 1000], seed=302, split_tokens=64),
    "g2_d64_bs32_ctx_on_block_edges": C(batch=5, q_heads=4, kv_heads=2, head_dim=64, block_size=32,
                                        ctx=[1, 32, 33, 64, 700], seed=303, split_tokens=96),
    "fp8_g4": C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                ctx=[3, 150, 400], seed=304, cache_dtype="fp8_e4m3", split_tokens=32),
    "verify_t4": C(batch=4, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                   ctx=[4, 17, 130, 700], q_len=4, seed=305),
    "verify_t3_fp8": C(batch=3, q_heads=4, kv_heads=4, head_dim=128, block_size=32,
                       ctx=[3, 64, 200], q_len=3, seed=306, cache_dtype="fp8_e4m3"),
    "long_ragged_auto_split": C(batch=3, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                                ctx=[5000, 17, 2500], seed=307),
}


def _step_inputs(st):
    w = st.w
    if w.q_len > 1:
        return st.k_step, st.v_step, st.q_multi
    return st.k_new, st.v_new, st.q


def _lse_shape(q):
    return q.shape[:3] if q.dim() == 4 else q.shape[:2]


@pytest.mark.parametrize("name", sorted(STEP))
def test_step_matches_the_oracle_and_the_separate_calls(name):
    w = workloads.make(STEP[name])
    fused = Staged(w, step_append=False)
    k, v, q = _step_inputs(fused)
    out = torch.empty_like(q)
    lse = torch.empty(_lse_shape(q), dtype=torch.float32, device="cuda")
    kp.paged_decode_step(fused.pool, k, v, q, fused.tables, fused.ctx, w.scale,
                         kv_split_tokens=w.spec.split_tokens, out=out, lse=lse)
    torch.cuda.synchronize()

    # the pool: bit for bit the oracle's image after the append
    kimg, vimg = oracle.pool_image(w, after_step=True)
    kr, vr = fused.pool.raw_bytes()
    assert np.array_equal(kr.cpu().numpy(), kimg)
    assert np.array_equal(vr.cpu().numpy(), vimg)

    # the outputs: the oracle within tolerance
    if w.q_len > 1:
        ref, ref_lse = oracle.decode_multi_workload(w, w.q_multi, w.q_len)
    else:
        ref, ref_lse = oracle.decode_workload(w)
    max_abs, rel, got = compare(out, ref)
    assert np.isfinite(got).all()
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.nanmax(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    assert fused.pool.device_errors() == 0

    # the separate calls give the same bits
    sep = Staged(w, step_append=True)
    if w.q_len > 1:
        out2, lse2 = sep.multi()
    else:
        out2, lse2 = sep.decode()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    sep.destroy()
    fused.destroy()


def test_repeated_steps_on_one_stream_stay_exact():
    """Several steps back to back on one stream (each step's attention overlapping the
    append that precedes it), each checked against the oracle of its own step."""
    spec = C(batch=4, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
             ctx=[15, 16, 17, 300], seed=308, split_tokens=64)
    w = workloads.make(spec)
    st = Staged(w, step_append=False)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            out = torch.empty_like(st.q)
            kp.paged_decode_step(st.pool, st.k_new, st.v_new, st.q, st.tables, st.ctx, w.scale,
                                 kv_split_tokens=spec.split_tokens, out=out, stream=s)
            outs.append(out)
    s.synchronize()
    ref, _ = oracle.decode_workload(w)
    for out in outs:                                   # the same step repeated: same result
        max_abs, rel, _ = compare(out, ref)
        assert max_abs <= MAX_ABS and rel <= REL_L2
        assert torch.equal(out, outs[0])
    assert st.pool.device_errors() == 0
    st.destroy()


def test_step_writes_and_flags_what_the_separate_append_does():
    """Context lengths that put a new token outside its block table (an empty sequence, one
    longer than the table): the step writes the same pool bytes as paged_kv_append followed
    by the attention, sets the same device error bits and gives the same output bits."""
    w = workloads.make(C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                         ctx=[10, 40, 33], seed=310))
    bad_ctx = np.array([0, 40, w.max_blocks * 16 + 5], dtype=np.int32)
    results = []
    for fused in (True, False):
        st = Staged(w, step_append=False)
        ctx = i32(bad_ctx)
        out = torch.empty_like(st.q)
        lse = torch.empty(st.q.shape[:2], dtype=torch.float32, device="cuda")
        if fused:
            kp.paged_decode_step(st.pool, st.k_new, st.v_new, st.q, st.tables, ctx, w.scale,
                                 out=out, lse=lse)
        else:
            kp.paged_kv_append(st.pool, st.k_new, st.v_new, st.tables, ctx)
            kp.paged_decode_attention(st.pool, st.q, st.tables, ctx, w.scale, out=out, lse=lse)
        torch.cuda.synchronize()
        bits = st.pool.device_errors()
        kr, vr = st.pool.raw_bytes()
        results.append((bits, kr.clone(), vr.clone(), out.clone(), lse.clone()))
        st.destroy()
    (b1, k1, v1, o1, l1), (b2, k2, v2, o2, l2) = results
    assert b1 == b2, (hex(b1), hex(b2))
    assert b1 & kp.DEVERR_POSITION and b1 & kp.DEVERR_CONTEXT
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_step_rejects_bad_arguments_before_launching():
    w = workloads.make(C(batch=2, q_heads=4, kv_heads=2, head_dim=64, block_size=16,
                         ctx=[10, 40], seed=309))
    st = Staged(w, step_append=False)
    before = [t.clone() for t in st.pool.raw_bytes()]
    bad_q = torch.empty(2, 5, 64, dtype=torch.bfloat16, device="cuda")   # 5 heads over 2 kv heads
    with pytest.raises(kp.KVError):
        kp.paged_decode_step(st.pool, st.k_new, st.v_new, bad_q, st.tables, st.ctx, w.scale)
    torch.cuda.synchronize()
    after = st.pool.raw_bytes()
    assert all(torch.equal(a, b) for a, b in zip(before, after))      # nothing was appended
    st.destroy()
    lat = kp.kv_mla_pool_create(8, 64, 512, 64)
    with pytest.raises(kp.KVError):
        kp.paged_decode_step(lat, torch.zeros(1, 576, dtype=torch.bfloat16, device="cuda"),
                             torch.zeros(1, 576, dtype=torch.bfloat16, device="cuda"),
                             torch.zeros(1, 16, 576, dtype=torch.bfloat16, device="cuda"),
                             torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                             torch.ones(1, dtype=torch.int32, device="cuda"), 0.1)
    lat.destroy()


# ---- latent pools: paged_mla_decode_step, one case per form of the attention kernel
M = workloads.mla
MLA_STEP = {
    "mma_bs16_h16": M(batch=4, q_heads=16, block_size=16, ctx=[1, 16, 17, 300], seed=311,
                      split_tokens=64),
    "narrow_bs64_h16": M(batch=5, q_heads=16, block_size=64, ctx=[1, 64, 65, 700, 2000], seed=312,
                         split_tokens=64),
    "narrow_bs64_h40": M(batch=3, q_heads=40, block_size=64, ctx=[63, 129, 1500], seed=313),
    "wide_bs64_h128": M(batch=3, q_heads=128, block_size=64, ctx=[1, 70, 900], seed=314,
                        split_tokens=64),
    # a grid of more than three CTAs per SM: the mma.sync form without a producer warp, whose
    # loads (and the write of the new vector before them) are issued by a consumer thread
    "mma_bs16_h128_many_ctas": M(batch=24, q_heads=128, block_size=16, ctx_uniform=(1, 300),
                                 seed=316, split_tokens=64),
}


@pytest.mark.parametrize("name", sorted(MLA_STEP))
def test_mla_step_matches_the_oracle_and_the_separate_calls(name):
    w = workloads.make(MLA_STEP[name])
    s = w.spec
    fused = Staged(w, step_append=False)
    out = torch.empty(w.batch, s.q_heads, s.latent_dim, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.batch, s.q_heads, dtype=torch.float32, device="cuda")
    kp.paged_mla_decode_step(fused.pool, fused.k_new, fused.q, fused.tables, fused.ctx, w.scale,
                             kv_split_tokens=s.split_tokens, out=out, lse=lse,
                             latent_dim=s.latent_dim)
    torch.cuda.synchronize()
    # the pool holds every vector, the appended ones included, bit for bit
    k, _, _, _ = fused.pool.tensors()
    pool = k.view(torch.int16).cpu().numpy().view(np.uint16)[:, :, 0, :]
    for b in range(w.batch):
        n = int(w.context_lens[b])
        t = np.arange(n)
        assert np.array_equal(pool[w.block_tables[b, t // s.block_size], t % s.block_size],
                              w.seq_k(b)[:, 0, :]), b
    ref, ref_lse = oracle.mla_decode_workload(w)
    max_abs, rel, got = compare(out, ref)
    assert np.isfinite(got).all()
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.nanmax(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    assert fused.pool.device_errors() == 0
    # the separate calls give the same bits
    sep = Staged(w, step_append=True)
    out2, lse2 = sep.mla()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    sep.destroy()
    fused.destroy()


MLA_EDGE = {
    "mma_bs16_h16": (M(batch=4, q_heads=16, block_size=16, ctx=[10, 40, 33, 50], seed=318), 16),
    "narrow_bs64_h16": (M(batch=4, q_heads=16, block_size=64, ctx=[10, 140, 70, 200], seed=319),
                        64),
    "wide_bs64_h128": (M(batch=4, q_heads=128, block_size=64, ctx=[10, 140, 70, 200], seed=320),
                       64),
    "mma_bs16_h128_many_ctas": (M(batch=24, q_heads=128, block_size=16, ctx_uniform=(20, 300),
                                  seed=321), 16),
}


@pytest.mark.parametrize("name", sorted(MLA_EDGE))
def test_mla_step_writes_and_flags_what_the_separate_append_does(name):
    """A latent step whose new vectors fall outside the block table (an empty sequence, one
    longer than the table) or into a block with a bad id: the same pool bytes, device error
    bits and output bits as paged_kv_append followed by the attention."""
    spec, bs = MLA_EDGE[name]
    w = workloads.make(spec)
    bad_ctx = w.context_lens.astype(np.int32)
    bad_ctx[0] = 0
    bad_ctx[2] = w.max_blocks * bs + 5
    bad_tables = w.block_tables.copy()
    bad_tables[3, (bad_ctx[3] - 1) // bs] = -7        # the block that would hold the new vector
    results = []
    for fused in (True, False):
        st = Staged(w, step_append=False)
        ctx, tables = i32(bad_ctx), i32(bad_tables)
        out = torch.empty(w.batch, spec.q_heads, spec.latent_dim, dtype=torch.bfloat16,
                          device="cuda")
        lse = torch.empty(w.batch, spec.q_heads, dtype=torch.float32, device="cuda")
        if fused:
            kp.paged_mla_decode_step(st.pool, st.k_new, st.q, tables, ctx, w.scale, out=out,
                                     lse=lse, latent_dim=spec.latent_dim)
        else:
            kp.paged_kv_append(st.pool, st.k_new, None, tables, ctx)
            kp.paged_mla_decode_attention(st.pool, st.q, tables, ctx, w.scale, out=out, lse=lse,
                                          latent_dim=spec.latent_dim)
        torch.cuda.synchronize()
        bits = st.pool.device_errors()
        kr = st.pool.raw_bytes()[0]
        results.append((bits, kr.clone(), out.clone(), lse.clone()))
        st.destroy()
    (b1, k1, o1, l1), (b2, k2, o2, l2) = results
    assert b1 == b2, (hex(b1), hex(b2))
    assert b1 & kp.DEVERR_POSITION and b1 & kp.DEVERR_CONTEXT and b1 & kp.DEVERR_BLOCK_ID
    assert torch.equal(k1, k2)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_mla_step_rejects_bad_arguments_before_launching():
    w = workloads.make(M(batch=2, q_heads=16, block_size=64, ctx=[10, 100], seed=315))
    st = Staged(w, step_append=False)
    before = [t.clone() for t in st.pool.raw_bytes() if t is not None]
    buf = torch.empty(2 * 16 * 512 + 8, dtype=torch.bfloat16, device="cuda")
    bad_out = buf[1:1 + 2 * 16 * 512].view(2, 16, 512)               # 2 bytes off a 16-byte boundary
    with pytest.raises(kp.KVError):
        kp.paged_mla_decode_step(st.pool, st.k_new, st.q, st.tables, st.ctx, w.scale, out=bad_out)
    torch.cuda.synchronize()
    after = [t for t in st.pool.raw_bytes() if t is not None]
    assert all(torch.equal(a, b) for a, b in zip(before, after))      # nothing was appended
    st.destroy()
    gqa = kp.kv_pool_create(8, 16, 2, 64)
    with pytest.raises(kp.KVError):                                   # not a latent pool
        kp.paged_mla_decode_step(gqa, torch.zeros(1, 576, dtype=torch.bfloat16, device="cuda"),
                                 torch.zeros(1, 16, 576, dtype=torch.bfloat16, device="cuda"),
                                 torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                                 torch.ones(1, dtype=torch.int32, device="cuda"), 0.1)
    gqa.destroy()


def test_repeated_mla_steps_on_one_stream_stay_exact():
    """Several latent steps back to back on one stream, each kernel starting while the one
    before it finishes (the same step repeated: same bits each time)."""
    w = workloads.make(M(batch=4, q_heads=16, block_size=64, ctx=[15, 64, 65, 600], seed=317,
                         split_tokens=64))
    st = Staged(w, step_append=False)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(3):
            out = torch.empty(w.batch, w.spec.q_heads, w.spec.latent_dim, dtype=torch.bfloat16,
                              device="cuda")
            kp.paged_mla_decode_step(st.pool, st.k_new, st.q, st.tables, st.ctx, w.scale,
                                     kv_split_tokens=w.spec.split_tokens, out=out, stream=s,
                                     latent_dim=w.spec.latent_dim)
            outs.append(out)
    s.synchronize()
    ref, _ = oracle.mla_decode_workload(w)
    for out in outs:
        max_abs, rel, _ = compare(out, ref)
        assert max_abs <= MAX_ABS and rel <= REL_L2
        assert torch.equal(out, outs[0])
    assert st.pool.device_errors() == 0
    st.destroy()
