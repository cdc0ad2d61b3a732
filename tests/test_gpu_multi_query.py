"""GPU parity of attention with several new tokens per sequence (speculative verify,
prefill chunks): paged_attention_multi_query against the float64 oracle."""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import (FP8_GATE_MIN_CTX, FP8_VS_UNQUANTISED_MAX_ABS, LSE_ABS, MAX_ABS, REL_L2,
                      Staged, compare, i32)

pytestmark = pytest.mark.gpu

C = workloads.custom
CASES = {
    "g4_t4_verify": C(batch=4, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                      ctx=[4, 17, 130, 700], q_len=4, seed=201),
    "g8_t2_rows16": C(batch=3, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                      ctx=[2, 33, 500], q_len=2, seed=202, split_tokens=64),
    "g4_t5_two_row_tiles": C(batch=3, q_heads=8, kv_heads=2, head_dim=64, block_size=32,
                             ctx=[5, 40, 300], q_len=5, seed=203),
    "g32_t2_four_tiles": C(batch=2, q_heads=32, kv_heads=1, head_dim=64, block_size=16,
                           ctx=[3, 260], q_len=2, seed=204),
    "prefill_chunk_t16": C(batch=2, q_heads=4, kv_heads=4, head_dim=128, block_size=16,
                           ctx=[16, 77], q_len=16, seed=205),
    "fp8_g1_t3": C(batch=3, q_heads=4, kv_heads=4, head_dim=128, block_size=32, ctx=[3, 64, 200],
                   q_len=3, seed=206, cache_dtype="fp8_e4m3"),
    # the automatic chunk: two kv heads and both 8-row tiles of each per CTA
    "hkv8_g4_t4_verify": C(batch=3, q_heads=32, kv_heads=8, head_dim=128, block_size=16,
                           ctx=[4, 300, 1100], q_len=4, seed=207),
    "hkv8_g2_t3_rows6": C(batch=3, q_heads=16, kv_heads=8, head_dim=128, block_size=16,
                          ctx=[3, 500, 2000], q_len=3, seed=209),
}


@pytest.fixture(scope="module", params=sorted(CASES))
def staged(request):
    w = workloads.make(CASES[request.param])
    st = Staged(w)
    yield st
    st.destroy()


def test_append_of_the_step_tokens_bit_exact(staged):
    kimg, vimg = oracle.pool_image(staged.w, after_step=True)
    kr, vr = staged.pool.raw_bytes()
    assert np.array_equal(kr.cpu().numpy(), kimg) and np.array_equal(vr.cpu().numpy(), vimg)


@pytest.mark.parametrize("split", ["spec", 16, 10 ** 6])
def test_multi_query_matches_oracle(staged, split):
    w = staged.w
    sp = w.spec.split_tokens if split == "spec" else (w.spec.block_size if split == 16 else
                                                      w.spec.block_size * w.max_blocks)
    out, lse = staged.multi(split_tokens=sp)
    ref, ref_lse = oracle.decode_multi_workload(w, w.q_multi, w.q_len)
    max_abs, rel, got = compare(out, ref)
    assert np.isfinite(got).all()
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    if w.spec.cache_dtype == "fp8_e4m3":
        raw, _ = oracle.decode_multi_workload(w, w.q_multi, w.q_len, cache_dtype="bf16")
        long_ctx = np.repeat((w.context_lens >= FP8_GATE_MIN_CTX)[:, None], w.spec.q_heads, 1)
        assert np.max(np.abs(got - raw)[long_ctx]) <= FP8_VS_UNQUANTISED_MAX_ABS
    assert staged.pool.device_errors() == 0


def test_each_query_equals_a_decode_over_its_prefix(staged):
    """Query i of a sequence is the decode of a context ending at its own position."""
    w = staged.w
    t = w.q_len
    one_chunk = w.spec.block_size * w.max_blocks
    out, lse = staged.multi(split_tokens=one_chunk)
    for i in range(t):
        ctx_i = i32(w.context_lens - (t - 1 - i))
        q_i = staged.q_multi[:, :, i].contiguous()
        o_i = torch.empty_like(q_i)
        l_i = torch.empty(q_i.shape[:2], dtype=torch.float32, device="cuda")
        kp.paged_decode_attention(staged.pool, q_i, staged.tables, ctx_i, w.scale,
                                  kv_split_tokens=one_chunk, out=o_i, lse=l_i)
        assert torch.equal(out[:, :, i].view(torch.int16), o_i.view(torch.int16))
        assert torch.equal(lse[:, :, i], l_i)


def test_one_query_token_is_the_decode():
    w = workloads.make(C(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                         ctx=[1, 40, 333], seed=207))
    st = Staged(w)
    a, la = st.decode(split_tokens=64)
    b = torch.empty_like(st.q[:, :, None])
    lb = torch.empty(st.q.shape[:2] + (1,), dtype=torch.float32, device="cuda")
    kp.paged_attention_multi_query(st.pool, st.q[:, :, None].contiguous(), st.tables, st.ctx,
                                   w.scale, kv_split_tokens=64, out=b, lse=lb)
    assert torch.equal(a.view(torch.int16), b[:, :, 0].view(torch.int16))
    assert torch.equal(la, lb[:, :, 0])
    st.destroy()


def test_context_shorter_than_the_queries_is_flagged():
    w = workloads.make(C(batch=2, q_heads=4, kv_heads=2, head_dim=128, block_size=16,
                         ctx=[8, 20], q_len=4, seed=208))
    st = Staged(w)
    st.ctx = i32(np.array([2, 20], dtype=np.int32))      # 2 tokens, 4 queries
    out, lse = st.multi()
    assert st.pool.device_errors() & kp.DEVERR_CONTEXT
    assert torch.isfinite(out.float()).all()
    # queries 0 and 1 of sequence 0 would sit at negative positions: nothing to attend to
    assert torch.count_nonzero(out[0, :, :2].float()) == 0
    assert torch.isneginf(lse[0, :, :2]).all()
    st.destroy()


def test_full_size_speculative_verify():
    """At the benchmark's sizes (the 4-token verify pass on the Llama-3-8B-shaped layer, the
    automatic chunk): the whole K and V pools bit for bit, and every query of every sequence
    against the oracle."""
    w = workloads.make(workloads.CONFIGS["llama3_8b_verify4"])
    st = Staged(w)
    out, lse = st.multi()
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    threads = os.cpu_count() or 1
    kimg, vimg = oracle.pool_image(w, after_step=True, threads=threads)
    kr, vr = st.pool.raw_bytes()
    for a in range(0, kimg.shape[0], 4096):
        assert np.array_equal(kr[a:a + 4096].cpu().numpy(), kimg[a:a + 4096])
        assert np.array_equal(vr[a:a + 4096].cpu().numpy(), vimg[a:a + 4096])
    del kimg, vimg
    ref, ref_lse = oracle.decode_multi_workload(w, w.q_multi, w.q_len, threads=threads)
    max_abs, rel, got = compare(out, ref)
    assert np.isfinite(got).all()
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    st.destroy()
