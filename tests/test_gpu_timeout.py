"""The bounded-wait failure path of the decode kernels, on the GPU and without a fault.

Every pipeline wait in the kernels gives up after a time limit, sets KV_DEVERR_TIMEOUT
and lets the CTA finish instead of spinning forever.  kv_debug_decode_stall makes one such
wait run out on purpose: the producer of each CTA issues no load from a given stage of its
chunk on, so the consumers wait on a barrier that nothing completes, while every load that
was issued still lands before the CTA exits.  The call must report the timeout, leave the
pool untouched and the device usable: the next call, with normal operation restored, must
match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import LSE_ABS, MAX_ABS, REL_L2, Staged, compare

pytestmark = pytest.mark.gpu

C = workloads.custom


@pytest.mark.parametrize("split,cta_heads", [(256, 1), (0, 2)])
def test_a_stage_that_never_lands_times_out_and_the_next_call_is_exact(split, cta_heads):
    w = workloads.make(C(batch=2, q_heads=8, kv_heads=2, head_dim=128, block_size=16,
                         ctx=[900, 300], seed=141))
    st = Staged(w)
    s = w.spec
    # both layouts of the kernel: one CTA per kv head (a chunk given by the caller) and
    # one CTA per pair of kv heads (the automatic chunk on this pool layout)
    assert kp.paged_decode_cta_heads(st.pool, w.batch, s.q_heads, 1, w.max_blocks, split) == cta_heads
    before = [t.clone() for t in st.pool.raw_bytes()]
    need = kp.paged_decode_workspace_size(st.pool, w.batch, s.q_heads, w.max_blocks, split)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(st.q)
    lse = torch.empty(st.q.shape[:2], dtype=torch.float32, device="cuda")
    kp.kv_debug_decode_stall(3, 20_000_000)         # stop at stage 3, consumers give up after 20 ms
    try:
        kp.paged_decode_attention(st.pool, st.q, st.tables, st.ctx, w.scale, kv_split_tokens=split,
                                  workspace=ws, out=out, lse=lse)
        torch.cuda.synchronize()
    finally:
        kp.kv_debug_decode_stall(-1, 0)
    assert st.pool.device_errors() & kp.DEVERR_TIMEOUT
    after = st.pool.raw_bytes()
    assert all(torch.equal(a, b) for a, b in zip(before, after))
    # the context is still usable and the next call is exact
    ws.zero_()
    kp.paged_decode_attention(st.pool, st.q, st.tables, st.ctx, w.scale, kv_split_tokens=split,
                              workspace=ws, out=out, lse=lse)
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    ref, ref_lse = oracle.decode_workload(w)
    max_abs, rel, _ = compare(out, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    st.destroy()

