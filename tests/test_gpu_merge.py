"""GPU parity of paged_merge_attention_states, the merge of attention results over
disjoint key sets (the one exchange of a sequence split across devices).

Two checks: the kernel against the oracle's merge on the same bf16 inputs (only fp32
arithmetic and the final bf16 rounding differ), and a sequence split by blocks into
shards -- each shard decoded by paged_decode_attention on its own block table, as a
device of a split would -- merged on the GPU against the oracle's attention over the
whole context.  On one GPU the shards run one after the other: no kernel waits on
another.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import LSE_ABS, MAX_ABS, REL_L2, Staged, compare, i32

pytestmark = pytest.mark.gpu


def _bf16_round_bound(ref):
    # one bf16 rounding (2^-9 relative) of an fp32 result, with margin
    return 2.0 ** -8 * np.abs(ref) + 1e-6


@pytest.mark.parametrize("n_src,rows,d", [(1, 7, 64), (2, 300, 128), (5, 1000, 128), (3, 33, 8)])
def test_merge_kernel_matches_the_oracle_merge(n_src, rows, d):
    g = torch.Generator().manual_seed(1000 + n_src * 7 + d)
    outs = torch.randn(n_src, rows, d, generator=g).to(torch.bfloat16)
    lses = (torch.randn(n_src, rows, generator=g) * 4.0).float()
    if n_src > 1:
        lses[0, ::3] = -float("inf")                  # sources with no key
        lses[:, 5] = -float("inf")                    # a row with no key at all
    outs_d, lses_d = outs.cuda(), lses.cuda()
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    out = kp.paged_merge_attention_states(outs_d, lses_d, lse=lse)
    ref, ref_lse = oracle.merge_states(outs.double().numpy(), lses.double().numpy())
    got = out.double().cpu().numpy()
    assert np.all(np.abs(got - ref) <= _bf16_round_bound(ref))
    got_lse = lse.double().cpu().numpy()
    empty = ~np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), ~empty)
    assert np.max(np.abs(got_lse[~empty] - ref_lse[~empty])) <= 1e-4
    if n_src > 1:
        assert np.all(got[5] == 0.0) and got_lse[5] == -np.inf


def _shard_tables(w, n_shards):
    """Per shard: a block table holding each sequence's r-th range of blocks, and the
    number of tokens in that range (0 for an empty shard)."""
    bs = w.spec.block_size
    tabs, ctxs = [], []
    for r in range(n_shards):
        t = np.zeros_like(w.block_tables)
        c = np.zeros(w.batch, dtype=np.int32)
        for b in range(w.batch):
            n = int(w.context_lens[b])
            nb = -(-n // bs)
            per = -(-nb // n_shards)
            j0, j1 = min(r * per, nb), min((r + 1) * per, nb)
            t[b, :j1 - j0] = w.block_tables[b, j0:j1]
            c[b] = max(0, min(n, j1 * bs) - j0 * bs)
        tabs.append(t)
        ctxs.append(c)
    return tabs, ctxs


@pytest.mark.parametrize("n_shards", [2, 3, 8])
def test_sequence_split_by_blocks_merges_to_the_whole_attention(n_shards):
    spec = workloads.custom(batch=4, q_heads=16, kv_heads=2, head_dim=128, block_size=16,
                            ctx=[3000, 700, 33, 16], seed=131)
    w = workloads.make(spec)
    st = Staged(w)
    s = w.spec
    tabs, ctxs = _shard_tables(w, n_shards)
    outs = torch.empty((n_shards, w.batch, s.q_heads, s.head_dim), dtype=torch.bfloat16,
                       device="cuda")
    lses = torch.empty((n_shards, w.batch, s.q_heads), dtype=torch.float32, device="cuda")
    for r in range(n_shards):
        kp.paged_decode_attention(st.pool, st.q, i32(tabs[r]), i32(ctxs[r]), w.scale,
                                  out=outs[r], lse=lses[r])
    lse = torch.empty((w.batch, s.q_heads), dtype=torch.float32, device="cuda")
    out = kp.paged_merge_attention_states(outs, lses, lse=lse)
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    assert any((c == 0).any() for c in ctxs)          # some shard of a short sequence is empty
    # against the oracle's attention over each whole context
    ref, ref_lse = oracle.decode_workload(w)
    max_abs, rel, got = compare(out, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= LSE_ABS
    # against the oracle's merge of the same shard results
    m_ref, _ = oracle.merge_states(outs.double().cpu().numpy().reshape(n_shards, -1, s.head_dim),
                                   lses.double().cpu().numpy().reshape(n_shards, -1))
    m_ref = m_ref.reshape(got.shape)
    assert np.all(np.abs(got - m_ref) <= _bf16_round_bound(m_ref))
    st.destroy()


def test_merge_rejects_bad_arguments_before_launching():
    outs = torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda")
    lses = torch.zeros(2, 4, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        kp.paged_merge_attention_states(outs, lses[:, :3].contiguous())
    with pytest.raises(kp.KVError):
        kp.paged_merge_attention_states(torch.zeros(2, 4, 12, dtype=torch.bfloat16,
                                                    device="cuda"), lses)
