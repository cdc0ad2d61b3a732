"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Append, indexing and fp8 codes are compared bit for bit; attention outputs
within max |err| <= 2e-2 and relative L2 <= 5e-3 (bf16 storage, fp32
accumulation); for the fp8 cache also within 6e-2 of the oracle on the
unquantised values.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import (FP8_GATE_MIN_CTX, FP8_VS_UNQUANTISED_MAX_ABS, LSE_ABS, MAX_ABS, REL_L2,
                      Staged, bf16_tensor, compare, i32)

pytestmark = pytest.mark.gpu

C = workloads.custom
SMALL = {
    "tiny": workloads.CONFIGS["tiny"],
    "g4_d128_bs16": C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                      ctx=[1, 16, 203], seed=101),
    "g8_split64": C(batch=3, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                    ctx=[37, 300, 1000], seed=102, split_tokens=64),
    "g1_d64_bs32": C(batch=4, q_heads=4, kv_heads=4, head_dim=64, block_size=32,
                     ctx=[5, 33, 64, 95], seed=103),
    "g16_nt16": C(batch=2, q_heads=32, kv_heads=2, head_dim=128, block_size=16,
                  ctx=[100, 257], seed=104),
    "g32_two_head_groups": C(batch=2, q_heads=32, kv_heads=1, head_dim=64, block_size=16,
                             ctx=[70, 500], seed=105, split_tokens=128),
    "g12_padded_bs32": C(batch=3, q_heads=24, kv_heads=2, head_dim=128, block_size=32,
                         ctx=[31, 32, 333], seed=106),
    "g2_d64": C(batch=5, q_heads=4, kv_heads=2, head_dim=64, block_size=16,
                ctx=[2, 17, 48, 129, 700], seed=107, split_tokens=96),
    "prefix_shared": C(batch=8, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                       ctx=[20, 70, 64, 129, 65, 200, 16, 90], seed=108, prefix_group=4,
                       prefix_tokens=64),
    "fp8_g1_bs32": C(batch=5, q_heads=4, kv_heads=4, head_dim=128, block_size=32,
                     ctx=[1, 31, 32, 33, 200], seed=109, cache_dtype="fp8_e4m3"),
    "fp8_g4_split32": C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                        ctx=[3, 150, 400], seed=110, cache_dtype="fp8_e4m3", split_tokens=32),
    "fp8_g16": C(batch=2, q_heads=32, kv_heads=2, head_dim=128, block_size=32,
                 ctx=[64, 300], seed=111, cache_dtype="fp8_e4m3"),
    "long_ragged_auto_split": C(batch=3, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                                ctx=[5000, 17, 2500], seed=112),
    # eight kv heads: the layouts whose CTA covers a group of kv heads
    "hkv8_g4_split256": C(batch=3, q_heads=32, kv_heads=8, head_dim=128, block_size=16,
                          ctx=[1, 300, 1900], seed=113, split_tokens=256),
    "hkv8_g2_auto": C(batch=5, q_heads=16, kv_heads=8, head_dim=128, block_size=16,
                      ctx=[17, 64, 700, 2500, 33], seed=114),
    "hkv8_g16_nt16": C(batch=2, q_heads=128, kv_heads=8, head_dim=128, block_size=16,
                       ctx=[100, 1000], seed=116, split_tokens=512),
    "hkv8_prefix_shared": C(batch=8, q_heads=32, kv_heads=8, head_dim=128, block_size=16,
                            ctx=[20, 70, 64, 129, 65, 200, 16, 90], seed=117, prefix_group=4,
                            prefix_tokens=64, split_tokens=32),
    "fp8_hkv8_split256": C(batch=3, q_heads=8, kv_heads=8, head_dim=128, block_size=32,
                           ctx=[5, 700, 1500], seed=115, cache_dtype="fp8_e4m3", split_tokens=256),
    # the automatic chunk on kv-head counts the group layouts divide (6 -> pairs, 12 -> fours)
    # or do not (fp8 with 2 kv heads keeps one CTA per kv head)
    "hkv6_g3_pairs": C(batch=4, q_heads=18, kv_heads=6, head_dim=128, block_size=16,
                       ctx=[2, 160, 1300, 47], seed=118),
    "fp8_hkv12_fours": C(batch=3, q_heads=12, kv_heads=12, head_dim=128, block_size=32,
                         ctx=[33, 900, 2100], seed=119, cache_dtype="fp8_e4m3"),
    "fp8_hkv2_per_head": C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=32,
                           ctx=[64, 250, 3000], seed=120, cache_dtype="fp8_e4m3"),
}


@pytest.fixture(scope="module", params=sorted(SMALL))
def staged(request):
    w = workloads.make(SMALL[request.param])
    st = Staged(w)
    yield st
    st.destroy()


def test_append_pool_image_bit_exact(staged):
    w = staged.w
    kimg, vimg = oracle.pool_image(w, after_step=True)
    kr, vr = staged.pool.raw_bytes()
    assert np.array_equal(kr.cpu().numpy(), kimg)
    assert np.array_equal(vr.cpu().numpy(), vimg)
    assert staged.pool.device_errors() == 0


def test_decode_matches_oracle(staged):
    w = staged.w
    out, lse = staged.decode()
    ref, ref_lse = oracle.decode_workload(w)
    max_abs, rel, got = compare(out, ref)
    assert np.isfinite(got).all()
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    if w.spec.cache_dtype == "fp8_e4m3":
        # Against the unquantised values the error is dominated by e4m3 rounding itself
        # (up to 2^-4 |v| per value), which only averages out over many tokens: the 6e-2
        # gate applies to contexts of at least 64 tokens.
        raw, _ = oracle.decode_workload(w, cache_dtype="bf16")
        long_ctx = w.context_lens >= FP8_GATE_MIN_CTX
        assert np.max(np.abs(got - raw)[long_ctx]) <= FP8_VS_UNQUANTISED_MAX_ABS
    assert staged.pool.device_errors() == 0


def test_decode_is_invariant_to_the_split(staged):
    w = staged.w
    a, la = staged.decode(split_tokens=w.spec.block_size)          # one block per chunk
    b, lb = staged.decode(split_tokens=w.spec.block_size * w.max_blocks)   # one chunk
    c, lc = staged.decode(split_tokens=0)                          # automatic
    ref, _ = oracle.decode_workload(w)
    for out in (a, b, c):
        max_abs, rel, _ = compare(out, ref)
        assert max_abs <= MAX_ABS and rel <= REL_L2
    assert torch.allclose(la, lb, atol=LSE_ABS, rtol=0)
    assert torch.allclose(la, lc, atol=LSE_ABS, rtol=0)


def test_chunk_counters_return_to_zero(staged):
    """The in-kernel merge counts finished chunks per (sequence, kv head, head tile)
    in the workspace and resets the counts: repeated calls on one workspace give
    identical bits and leave the counters at zero."""
    w = staged.w
    s = w.spec
    split = s.block_size * 2                                       # many chunks per sequence
    need = kp.paged_decode_workspace_size(staged.pool, w.batch, s.q_heads, w.max_blocks, split)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.empty_like(staged.q)
        kp.paged_decode_attention(staged.pool, staged.q, staged.tables, staged.ctx, w.scale,
                                  kv_split_tokens=split, workspace=ws, out=out)
        outs.append(out.view(torch.int16).clone())
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    g = s.q_heads // s.kv_heads
    tiles = 1 if g <= 8 else -(-g // 16)
    counters = ws[need - w.batch * s.kv_heads * tiles * 4:]
    assert torch.count_nonzero(counters) == 0


def _split_merge(st, split):
    out = torch.empty_like(st.q)
    lse = torch.empty(st.q.shape[:2], dtype=torch.float32, device="cuda")
    kp.paged_decode_attention_split_merge(st.pool, st.q, st.tables, st.ctx, st.w.scale,
                                          kv_split_tokens=split, out=out, lse=lse)
    return out, lse


def test_separate_merge_kernel_gives_the_fused_bits(staged):
    """The two-kernel form (split-KV grid, then a separate log-sum-exp merge kernel) against
    the fused form, whose last chunk CTA merges: identical output and lse bits at one block
    per chunk, three blocks per chunk and the automatic chunk, and within tolerance of the
    oracle."""
    w = staged.w
    bs = w.spec.block_size
    ref, ref_lse = oracle.decode_workload(w)
    for split in (bs, 3 * bs, 0):
        a, la = staged.decode(split_tokens=split)
        b, lb = _split_merge(staged, split)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), split
        assert torch.equal(la.view(torch.int32), lb.view(torch.int32)), split
        max_abs, rel, _ = compare(b, ref)
        assert max_abs <= MAX_ABS and rel <= REL_L2, (split, max_abs, rel)
        assert np.max(np.abs(lb.cpu().numpy() - ref_lse)) <= LSE_ABS
    assert staged.pool.device_errors() == 0


def test_block_permutation_gives_identical_bits():
    w = workloads.make(SMALL["g4_d128_bs16"])
    st = Staged(w)
    out1, lse1 = st.decode(split_tokens=32)
    perm = np.random.default_rng(9).permutation(w.num_blocks)
    kr, vr = st.pool.raw_bytes()
    idx = torch.from_numpy(np.argsort(perm)).cuda()          # new block j holds old block argsort[j]
    kr.copy_(kr[idx].clone())
    vr.copy_(vr[idx].clone())
    t2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    st.tables = i32(t2)
    out2, lse2 = st.decode(split_tokens=32)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    st.destroy()


def test_block_permutation_gives_identical_bits_with_automatic_chunks():
    w = workloads.make(SMALL["long_ragged_auto_split"])
    st = Staged(w)
    out1, lse1 = st.decode(split_tokens=0)
    perm = np.random.default_rng(10).permutation(w.num_blocks)
    kr, vr = st.pool.raw_bytes()
    idx = torch.from_numpy(np.argsort(perm)).cuda()
    kr.copy_(kr[idx].clone())
    vr.copy_(vr[idx].clone())
    st.tables = i32(np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1))
    out2, lse2 = st.decode(split_tokens=0)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    st.destroy()


def test_many_tiny_and_empty_sequences():
    """Zero-length sequences between long ones; chunked and one-chunk sequences mixed."""
    ctx = [0, 1, 0, 3000, 0, 16, 17, 0, 1, 999, 0, 0]
    spec = C(batch=len(ctx), q_heads=8, kv_heads=2, head_dim=128, block_size=16, seed=124,
             ctx=[max(c, 1) for c in ctx])
    w = workloads.make(spec)
    st = Staged(w)
    st.ctx = i32(np.array(ctx, dtype=np.int32))
    out, lse = st.decode(split_tokens=0)
    live = [i for i, c in enumerate(ctx) if c > 0]
    dead = [i for i, c in enumerate(ctx) if c == 0]
    w2 = workloads.make(spec)
    ref, ref_lse = oracle.decode_workload(w2, seqs=[i for i in live if ctx[i] == max(ctx[i], 1)])
    max_abs, rel, _ = compare(out[live], ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2
    assert torch.count_nonzero(out[dead].float()) == 0 and torch.isneginf(lse[dead]).all()
    assert st.pool.device_errors() == 0
    few = np.zeros(len(ctx), dtype=np.int32)
    few[[1, 3]] = [1, 16]                    # two sequences of one block each
    st.ctx = i32(few)
    out3, _ = st.decode(split_tokens=0)
    assert torch.isfinite(out3.float()).all()
    v0 = w.seq_v(1)[0]                        # one token: the output is its value, exactly
    want = np.repeat(v0, 4, axis=0).view(np.int16)
    assert np.array_equal(out3[1].view(torch.int16).cpu().numpy(), want)
    assert torch.count_nonzero(out3[[0, 2, 4]].float()) == 0
    st.destroy()


def test_batch_independence_bit_exact():
    w = workloads.make(SMALL["g8_split64"])
    st = Staged(w)
    full, _ = st.decode(split_tokens=64)
    for b in range(w.batch):
        out = torch.empty_like(st.q[b:b + 1])
        kp.paged_decode_attention(st.pool, st.q[b:b + 1], st.tables[b:b + 1], st.ctx[b:b + 1],
                                  w.scale, kv_split_tokens=64, out=out)
        assert torch.equal(out.view(torch.int16), full[b:b + 1].view(torch.int16))
    st.destroy()


def test_empty_context_gives_zero_output_and_minus_inf_lse():
    spec = C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16, ctx=[5, 40, 9], seed=120)
    w = workloads.make(spec)
    st = Staged(w)
    st.ctx = i32(np.array([5, 0, 9], dtype=np.int32))
    out, lse = st.decode()
    ref, _ = oracle.decode_workload(w, seqs=[0, 2])
    assert torch.count_nonzero(out[1].float()) == 0
    assert torch.isneginf(lse[1]).all()
    max_abs, rel, _ = compare(out[[0, 2]], ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2
    st.destroy()


def test_bad_block_id_is_skipped_and_reported():
    spec = C(batch=2, q_heads=8, kv_heads=2, head_dim=128, block_size=16, ctx=[40, 40], seed=121)
    w = workloads.make(spec)
    st = Staged(w)
    assert st.pool.device_errors() == 0
    t = w.block_tables.copy()
    t[1, 1] = w.num_blocks + 7          # outside the pool
    st.tables = i32(t)
    out, _ = st.decode()
    torch.cuda.synchronize()
    assert st.pool.device_errors() & kp.DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    ref, _ = oracle.decode_workload(w, seqs=[0])
    max_abs, rel, _ = compare(out[:1], ref)           # the other sequence is untouched
    assert max_abs <= MAX_ABS and rel <= REL_L2
    st.ctx = i32(np.array([40, 10_000], dtype=np.int32))     # past max_blocks * block_size
    st.decode()
    assert st.pool.device_errors() & kp.DEVERR_CONTEXT
    st.destroy()


def test_append_rejects_bad_addresses_on_device():
    spec = C(batch=2, q_heads=2, kv_heads=2, head_dim=64, block_size=16, ctx=[3, 20], seed=122)
    w = workloads.make(spec)
    st = Staged(w)
    before = [x.clone() for x in st.pool.raw_bytes()]
    kn = bf16_tensor(w.k_new[:1])
    kp.paged_kv_append(st.pool, kn, kn, st.tables, st.ctx, token_seq=i32([5]), token_pos=i32([0]))
    assert st.pool.device_errors() & kp.DEVERR_SEQ
    kp.paged_kv_append(st.pool, kn, kn, st.tables, st.ctx, token_seq=i32([0]), token_pos=i32([-1]))
    assert st.pool.device_errors() & kp.DEVERR_POSITION
    bad = w.block_tables.copy()
    bad[0, 0] = -3
    kp.paged_kv_append(st.pool, kn, kn, i32(bad), st.ctx, token_seq=i32([0]), token_pos=i32([0]))
    assert st.pool.device_errors() & kp.DEVERR_BLOCK_ID
    after = st.pool.raw_bytes()
    assert all(torch.equal(a, b) for a, b in zip(before, after))
    st.destroy()


def test_host_validation_rejects_before_launch():
    spec = C(batch=2, q_heads=8, kv_heads=2, head_dim=128, block_size=16, ctx=[3, 20], seed=123)
    w = workloads.make(spec)
    st = Staged(w)
    bad_heads = torch.zeros(2, 7, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kp.KVError) as e:
        kp.paged_decode_attention(st.pool, bad_heads, st.tables, st.ctx, w.scale)
    assert e.value.status == kp.KV_ERR_INVALID_ARG
    with pytest.raises(kp.KVError):
        kp.paged_decode_attention(st.pool, st.q, st.tables, st.ctx, w.scale, kv_split_tokens=24)
    need = kp.paged_decode_workspace_size(st.pool, 2, 8, w.max_blocks, 16)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kp.KVError):
        kp.paged_decode_attention(st.pool, st.q, st.tables, st.ctx, w.scale, kv_split_tokens=16,
                                  workspace=small)
    storage = torch.empty(st.q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    misaligned = storage[1:1 + st.q.numel()].view(st.q.shape)
    with pytest.raises(kp.KVError):
        kp.paged_decode_attention(st.pool, misaligned, st.tables, st.ctx, w.scale)
    with pytest.raises(kp.KVError):
        kp.kv_pool_create(10, 24, 2, 128)                            # block size not supported
    assert st.pool.device_errors() == 0
    st.destroy()


def test_fp8_append_codes_match_the_oracle_encoder_on_every_bf16_value():
    bits = np.arange(65536, dtype=np.uint16)
    x = workloads.bf16_bits_to_f32(bits)
    bits = bits[~np.isnan(x)]                       # NaN inputs are outside the encoder's domain
    bits = np.concatenate([bits, bits[: (-bits.size) % 128]])
    tokens = bits.size // 128
    for scale in (1.0, 0.37, 3.5e-3):
        pool = kp.kv_pool_create(tokens // 16 + 1, 16, 1, 128, "fp8_e4m3")
        pool.set_scales([scale], [scale])
        table = i32(np.arange(tokens // 16 + 1, dtype=np.int32)[None, :])
        kn = bf16_tensor(bits.reshape(tokens, 1, 128))
        kp.paged_kv_append(pool, kn, kn, table, i32([tokens]), token_seq=i32(np.zeros(tokens)),
                           token_pos=i32(np.arange(tokens)))
        kr, _ = pool.raw_bytes()
        got = kr.cpu().numpy().reshape(-1)[: bits.size]
        want = oracle.e4m3_quantize(bits, np.float32(scale))
        assert np.array_equal(got, want)
        pool.destroy()


# ----------------------------------------------------------------- full-size configurations
FULL = ["tiny", "llama3_8b", "long_context", "ragged_prefix", "mha_fp8"]


def _equal_in_slabs(dev_bytes: torch.Tensor, image: np.ndarray, slab: int = 4096) -> bool:
    """Every byte of a device pool half against the oracle's image, a slab of blocks at a
    time (the full-size pools are a few GB)."""
    for a in range(0, image.shape[0], slab):
        if not np.array_equal(dev_bytes[a:a + slab].cpu().numpy(), image[a:a + slab]):
            return False
    return True


@pytest.mark.parametrize("name", FULL)
def test_full_size_config_parity(name):
    """At the benchmark's sizes and in its launch configuration (append + attention in one
    paged_decode_step call): the whole K and V pools bit for bit against the oracle's image
    (every prefilled and appended slot, and the poisoned ones), and every sequence's output
    and LSE against the oracle."""
    w = workloads.make(workloads.CONFIGS[name])
    st = Staged(w, step_append=False)
    s = w.spec
    out = torch.empty_like(st.q)
    lse = torch.empty(st.q.shape[:2], dtype=torch.float32, device="cuda")
    kp.paged_decode_step(st.pool, st.k_new, st.v_new, st.q, st.tables, st.ctx, w.scale,
                         kv_split_tokens=s.split_tokens, out=out, lse=lse)
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    threads = os.cpu_count() or 1
    kimg, vimg = oracle.pool_image(w, after_step=True, threads=threads)
    kr, vr = st.pool.raw_bytes()
    assert tuple(kr.shape) == kimg.shape and tuple(vr.shape) == vimg.shape
    assert _equal_in_slabs(kr, kimg) and _equal_in_slabs(vr, vimg)
    del kimg, vimg
    # every sequence against the oracle
    ref, ref_lse = oracle.decode_workload(w, threads=threads)
    max_abs, rel, got = compare(out, ref)
    assert np.isfinite(got).all() and torch.isfinite(lse).all()
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    if s.cache_dtype == "fp8_e4m3":
        raw, _ = oracle.decode_workload(w, threads=threads, cache_dtype="bf16")
        long_ctx = w.context_lens >= FP8_GATE_MIN_CTX
        assert np.max(np.abs(got - raw)[long_ctx]) <= FP8_VS_UNQUANTISED_MAX_ABS
    # the attention alone and the two-kernel form (separate log-sum-exp merge) give the
    # same bits at this size
    out1, lse1 = st.decode()
    assert torch.equal(out.view(torch.int16), out1.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse1.view(torch.int32))
    out2, lse2 = _split_merge(st, s.split_tokens)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse2.view(torch.int32))
    assert st.pool.device_errors() == 0
    st.destroy()
