"""The allocation-free decode entry point against the regular one (GPU).

paged_decode_attention_noalloc serves callers that cannot allocate device
memory at the call site (plug-in hosts that only hand over input and output
buffers, engines whose allocator already owns the GPU, latency-critical paths
that cannot afford cudaMalloc's device-wide synchronisation).  Its split-KV
partials live in a static array inside the library instead of a caller
workspace.  Each call is checked against the float64 oracle and against the regular
entry point (with a caller workspace) on the same inputs.  This file runs
last so that a failure here comes after every other test; it also passes on
its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import LSE_ABS, MAX_ABS, REL_L2, Staged, compare, i32

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 8 << 20        # KV_NO_ALLOC_SCRATCH_BYTES in include/kv_paged.h


def _entry(lib):
    fn = lib.paged_decode_attention_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, I, P, I, P, I, ctypes.c_float, I, P, P, P]
    fn.restype = I
    return fn


def _call(fn, st, q_heads, tables, max_blocks, split, out, lse):
    return fn(st.pool.handle, st.q.data_ptr(), q_heads, tables.data_ptr(), max_blocks,
              st.ctx.data_ptr(), st.w.batch, st.w.scale, split, out.data_ptr(),
              None if lse is None else lse.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _check_two_calls(fn, st, split):
    """Two calls in a row (the second reuses the scratch the first left behind), each
    against the oracle and against paged_decode_attention with its own workspace."""
    w = st.w
    ref, ref_lse = oracle.decode_workload(w)
    ws_out, ws_lse = st.decode(split_tokens=split)
    ws = ws_out.float().cpu().double().numpy()
    for _ in range(2):
        out = torch.full_like(st.q, float("nan"))
        lse = torch.full(st.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        assert _call(fn, st, w.spec.q_heads, st.tables, w.max_blocks, split, out, lse) == kp.KV_OK
        torch.cuda.synchronize()
        max_abs, rel, _ = compare(out, ref)
        assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
        assert np.max(np.abs(lse.cpu().double().numpy() - ref_lse)) <= LSE_ABS
        max_abs, rel, _ = compare(out, ws)
        assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
        assert torch.allclose(lse, ws_lse, atol=LSE_ABS, rtol=0)


def test_noalloc_matches_the_oracle_and_the_workspace_entry_point_on_two_calls():
    fn = _entry(kp.load_library())
    spec = workloads.custom(batch=3, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                            ctx=[5000, 17, 2500], seed=131)
    w = workloads.make(spec)
    st = Staged(w)
    split = 256                                          # several chunks: the scratch is used
    need = kp.paged_decode_workspace_size(st.pool, w.batch, spec.q_heads, w.max_blocks, split)
    assert 0 < need <= SCRATCH_LIMIT
    _check_two_calls(fn, st, split)
    assert st.pool.device_errors() == 0
    st.destroy()


def test_noalloc_automatic_chunks_match_on_two_calls():
    """Automatic chunk size, several chunks per sequence: the in-kernel merge keeps its
    chunk counters in the scratch."""
    fn = _entry(kp.load_library())
    spec = workloads.custom(batch=5, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                            ctx=[900, 17, 2500, 1, 64], seed=133)
    w = workloads.make(spec)
    st = Staged(w)
    _, max_splits = kp.paged_decode_plan(st.pool, w.batch, spec.q_heads, w.max_blocks, 0)
    assert max_splits > 1
    _check_two_calls(fn, st, 0)
    assert st.pool.device_errors() == 0
    st.destroy()


def test_noalloc_rejected_call_leaves_the_scratch_alone():
    """A call rejected by validation (an unaligned output here) returns the error before
    anything touches the shared array, and the calls after it are still correct."""
    fn = _entry(kp.load_library())
    spec = workloads.custom(batch=3, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                            ctx=[700, 33, 1200], seed=134)
    w = workloads.make(spec)
    st = Staged(w)
    split = 128
    big = torch.zeros(st.q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    bad = big[1:1 + st.q.numel()].view(st.q.shape)       # 2-byte offset: not 16-byte aligned
    assert _call(fn, st, spec.q_heads, st.tables, w.max_blocks, split, bad, None) == \
        kp.KV_ERR_INVALID_ARG
    _check_two_calls(fn, st, split)
    assert st.pool.device_errors() == 0
    st.destroy()


def test_noalloc_refuses_sizes_beyond_its_scratch():
    fn = _entry(kp.load_library())
    spec = workloads.custom(batch=3, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                            ctx=[300, 17, 250], seed=132)
    w = workloads.make(spec)
    st = Staged(w)
    max_blocks = 2000                                    # 2000 one-block chunks per sequence
    tables = np.full((w.batch, max_blocks), -1, dtype=np.int32)
    tables[:, :w.max_blocks] = w.block_tables
    t = i32(tables)
    need = kp.paged_decode_workspace_size(st.pool, w.batch, spec.q_heads, max_blocks, 16)
    assert need > SCRATCH_LIMIT
    out = torch.zeros_like(st.q)
    assert _call(fn, st, spec.q_heads, t, max_blocks, 16, out, None) == kp.KV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.count_nonzero(out.float()) == 0         # nothing was launched
    st.destroy()
