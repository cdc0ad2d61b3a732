"""GPU parity of the absorbed multi-head latent attention decode over a paged
latent cache (paged_mla_decode_attention) against the float64 oracle.

Each head scores the shared cached vector (512 latent + 64 rotary-key numbers)
and averages its latent part (xuewyang.github.io/posts/kv, "MLA: how does decode
get full-size keys and values back?").  Outputs within max |err| <= 2e-2 and
relative L2 <= 5e-3, LSE within 2e-3; the latent pool's bytes bit for bit.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_19_gb300 as kp
import workloads
from gpu_util import LSE_ABS, MAX_ABS, REL_L2, Staged, compare, i32

pytestmark = pytest.mark.gpu

M = workloads.mla
SMALL = {
    "bs16_h16": M(batch=4, q_heads=16, block_size=16, ctx=[1, 15, 16, 300], seed=201),
    "bs32_h32_split128": M(batch=3, q_heads=32, block_size=32, ctx=[33, 500, 2000], seed=202,
                           split_tokens=128),
    "bs64_h20_padded": M(batch=3, q_heads=20, block_size=64, ctx=[64, 65, 700], seed=203),
    "bs64_h128": M(batch=2, q_heads=128, block_size=64, ctx=[100, 1500], seed=204),
    "bs64_auto_split_long": M(batch=2, q_heads=16, block_size=64, ctx=[9000, 40], seed=205),
    "bs64_split64_ragged": M(batch=5, q_heads=16, block_size=64, ctx=[1, 63, 64, 129, 1000],
                             seed=206, split_tokens=64),
    # grids of more than two CTAs per SM run the two-CTAs-per-SM variant
    "bs16_h128_many_ctas": M(batch=24, q_heads=128, block_size=16, ctx_uniform=(1, 300),
                             seed=209, split_tokens=64),
    "bs32_h64_many_ctas": M(batch=24, q_heads=64, block_size=32, ctx_uniform=(1, 400),
                            seed=210, split_tokens=64),
    # blocks of 64 and at least 64 heads run the wide tcgen05 form (128-head tiles, latent halves)
    "tc_h128_split128": M(batch=4, q_heads=128, block_size=64, ctx=[1, 64, 65, 700], seed=211,
                          split_tokens=128),
    "tc_h96_padded_tile": M(batch=3, q_heads=96, block_size=64, ctx=[63, 200, 1000], seed=212),
    "tc_h256_two_tiles": M(batch=2, q_heads=256, block_size=64, ctx=[130, 900], seed=213,
                           split_tokens=256),
    "tc_h64_long": M(batch=2, q_heads=64, block_size=64, ctx=[5000, 3], seed=214),
    # blocks of 64 and fewer heads run the narrow tcgen05 form (16-head tiles); these cut
    # many sequences into pieces and give CTAs several segments
    "tcn_h16_many_segments": M(batch=10, q_heads=16, block_size=64, ctx_uniform=(1, 1500), seed=215,
                               split_tokens=64),
    "tcn_h48_three_tiles": M(batch=3, q_heads=48, block_size=64, ctx=[65, 640, 3000], seed=216,
                             split_tokens=128),
    "tcn_h8_partial_tile": M(batch=4, q_heads=8, block_size=64, ctx=[1, 2, 4000, 127], seed=217),
}


@pytest.fixture(scope="module", params=sorted(SMALL))
def staged(request):
    st = Staged(workloads.make(SMALL[request.param]))
    yield st
    st.destroy()


def check(out, lse, w, seqs=None, threads=1):
    ref, ref_lse = oracle.mla_decode_workload(w, seqs=seqs, threads=threads)
    got = out if seqs is None else out[torch.as_tensor(seqs, device=out.device).long()]
    max_abs, rel, _ = compare(got, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)
    if lse is not None:
        gl = (lse if seqs is None else lse[torch.as_tensor(seqs, device=lse.device).long()])
        assert np.max(np.abs(gl.cpu().double().numpy() - ref_lse)) <= LSE_ABS


def test_latent_pool_holds_every_vector_bit_for_bit(staged):
    w = staged.w
    k, v, _, _ = staged.pool.tensors()
    assert v is None
    pool = k.view(torch.int16).cpu().numpy().view(np.uint16)[:, :, 0, :]
    bs = w.spec.block_size
    for b in range(w.batch):
        n = int(w.context_lens[b])
        t = np.arange(n)
        got = pool[w.block_tables[b, t // bs], t % bs]
        assert np.array_equal(got, w.seq_k(b)[:, 0, :]), b


def test_mla_decode_matches_oracle(staged):
    out, lse = staged.mla()
    torch.cuda.synchronize()
    check(out, lse, staged.w)
    assert staged.pool.device_errors() == 0


@pytest.mark.parametrize("split", [0, 64, 256])
def test_split_sizes_agree(staged, split):
    bs = staged.w.spec.block_size
    if split % bs:
        pytest.skip("chunk must be a multiple of the block size")
    out, lse = staged.mla(split_tokens=split)
    check(out, lse, staged.w)


def test_repeated_calls_are_identical(staged):
    a, la = staged.mla(split_tokens=staged.w.spec.block_size)
    b, lb = staged.mla(split_tokens=staged.w.spec.block_size)
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("bs,heads", [(16, 16), (64, 128), (64, 16)])
def test_empty_sequence_and_out_of_range_length(bs, heads):
    w = workloads.make(M(batch=2, q_heads=heads, block_size=bs, ctx=[40, 20], seed=207))
    st = Staged(w)
    ctx = torch.tensor([0, 20], dtype=torch.int32, device="cuda")
    out = torch.empty(2, heads, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(2, heads, dtype=torch.float32, device="cuda")
    kp.paged_mla_decode_attention(st.pool, st.q, st.tables, ctx, w.scale, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ref, ref_lse = oracle.mla_decode_workload(w, seqs=[1])
    assert compare(out[1:], ref)[0] <= MAX_ABS
    assert st.pool.device_errors() == 0
    bad = torch.tensor([40, 10 ** 6], dtype=torch.int32, device="cuda")
    kp.paged_mla_decode_attention(st.pool, st.q, st.tables, bad, w.scale, out=out, lse=lse)
    assert st.pool.device_errors() & kp.DEVERR_CONTEXT
    st.destroy()


@pytest.mark.parametrize("bs,heads", [(16, 16), (64, 128), (64, 16)])
def test_bad_block_ids_are_skipped_and_flagged(bs, heads):
    w = workloads.make(M(batch=2, q_heads=heads, block_size=bs, ctx=[150, 150], seed=208))
    st = Staged(w)
    tables = st.tables.clone()
    tables[0, 1] = w.num_blocks + 5
    out = torch.empty(2, heads, 512, dtype=torch.bfloat16, device="cuda")
    kp.paged_mla_decode_attention(st.pool, st.q, tables, st.ctx, w.scale, out=out)
    assert st.pool.device_errors() & kp.DEVERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    ref, _ = oracle.mla_decode_workload(w, seqs=[1])
    assert compare(out[1:], ref)[0] <= MAX_ABS
    st.destroy()


def test_api_rejects_mismatched_pools():
    gqa = kp.kv_pool_create(8, 16, 1, 128)
    q = torch.zeros(1, 16, 576, dtype=torch.bfloat16, device="cuda")
    t = torch.zeros(1, 1, dtype=torch.int32, device="cuda")
    c = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kp.KVError):
        kp.paged_mla_decode_attention(gqa, q, t, c, 0.1)
    lat = kp.kv_mla_pool_create(8, 16)
    with pytest.raises(kp.KVError):
        kp.paged_decode_attention(lat, torch.zeros(1, 8, 576, dtype=torch.bfloat16, device="cuda"),
                                  t, c, 0.1)
    with pytest.raises(kp.KVError):
        kp.paged_kv_append(lat, q[:, 0], q[:, 0], t, c)          # a latent pool takes no V
    with pytest.raises(kp.KVError):
        kp.kv_mla_pool_create(8, 16, latent_dim=256)
    gqa.destroy()
    lat.destroy()


@pytest.mark.parametrize("config", ["deepseek_mla", "deepseek_mla_tp8"])
def test_full_size_parity(config):
    """At the benchmark's sizes and in its launch configuration (append + attention in one
    paged_mla_decode_step call): the whole latent pool bit for bit against the oracle's
    image, and every sequence's output and LSE against the oracle."""
    w = workloads.make(workloads.CONFIGS[config])
    st = Staged(w, step_append=False)
    s = w.spec
    out = torch.empty(w.batch, s.q_heads, s.latent_dim, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.batch, s.q_heads, dtype=torch.float32, device="cuda")
    kp.paged_mla_decode_step(st.pool, st.k_new, st.q, st.tables, st.ctx, w.scale,
                             kv_split_tokens=s.split_tokens, out=out, lse=lse,
                             latent_dim=s.latent_dim)
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    threads = os.cpu_count() or 1
    kimg, _ = oracle.pool_image(w, after_step=True, threads=threads)
    kr, vr = st.pool.raw_bytes()
    assert vr is None and tuple(kr.shape) == kimg.shape
    for a in range(0, kimg.shape[0], 4096):
        assert np.array_equal(kr[a:a + 4096].cpu().numpy(), kimg[a:a + 4096]), a
    del kimg
    check(out, lse, w, threads=threads)
    out1, lse1 = st.mla()                        # the attention alone: the same bits
    assert torch.equal(out.view(torch.int16), out1.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse1.view(torch.int32))
    assert st.pool.device_errors() == 0
    st.destroy()


@pytest.mark.parametrize("heads", [16, 128])
def test_tcgen05_batches_over_256_sequences(heads):
    """Batches above 256 sequences take the tensor-core forms' prefix search over the
    segment-padded positions (a different path from smaller batches); short ragged
    sequences and small ranges give many segments per CTA."""
    w = workloads.make(M(batch=300, q_heads=heads, block_size=64, ctx_uniform=(1, 400),
                         seed=218, split_tokens=64))
    st = Staged(w)
    out, lse = st.mla()
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    check(out, lse, w, threads=os.cpu_count() or 1)
    out2, lse2 = st.mla(split_tokens=0)
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    check(out2, lse2, w, threads=os.cpu_count() or 1)
    st.destroy()


@pytest.mark.parametrize("heads", [16, 128])
def test_frequent_output_rescales(heads):
    """A softmax scale of 1 spreads the scores so widely (standard deviation ~24) that a
    head's running maximum keeps growing by more than 2^8 from one stage to the next:
    the tensor-core forms' lazy output rescale then runs in many stages, each time for
    some heads only, each head with its own factor."""
    w = workloads.make(workloads.custom("mla_scale_1", batch=4, q_heads=heads, kv_heads=1,
                                        head_dim=576, block_size=64, seed=219,
                                        ctx=[70, 700, 2000, 3000], latent_dim=512,
                                        qk_head_dim=1, split_tokens=1024))
    assert w.scale == 1.0
    st = Staged(w)
    out, lse = st.mla()
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0
    check(out, lse, w)
    st.destroy()


def test_copy_blocks_on_a_latent_pool():
    pool = kp.kv_mla_pool_create(6, 16)
    k, _ = pool.raw_bytes()
    rng = np.random.default_rng(3)
    k0 = rng.integers(0, 256, size=tuple(k.shape), dtype=np.uint8)
    k.copy_(torch.from_numpy(k0))
    kp.kv_copy_blocks(pool, i32(np.array([[2, 4]])))
    torch.cuda.synchronize()
    exp = k0.copy()
    exp[4] = k0[2]
    assert np.array_equal(k.cpu().numpy(), exp) and pool.device_errors() == 0
    pool.destroy()
