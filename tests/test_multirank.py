"""The multi-process path of bench.py on the CPU: world_size 2 over gloo.

The decode step shards by sequence with no exchange (each rank runs its own batch as an
independent replica), so what several ranks share is host logic only: the rendezvous, the
barrier around the timed region, the max of the ranks' times and the sum of their bytes, the
per-rank seeds of the synthetic batches, and the reference arm that rank 0 alone runs.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    import torch.distributed as dist
    r, w, local = bench.dist_setup(None)
    try:
        assert (r, w, local) == (rank, world, rank)
        assert dist.get_backend() == "gloo"
        bench.barrier(w)
        res = {
            "max": bench.max_over_ranks(1.5 + rank, w),
            "sum": bench.sum_over_ranks(10.0 * (rank + 1), w),
            "seed": bench.rank_spec("llama3_8b", rank).seed,
            "ctx_head": [int(x) for x in workloads.make(bench.rank_spec("tiny", rank)).context_lens],
        }
        bench.barrier(w)
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
        json.dump(res, fh)


def _shard_main(rank, world, port, out_dir):
    """One long sequence split by blocks across the ranks: each rank attends over its own
    blocks, the (out, lse) pairs are gathered -- the one exchange of a sequence split --
    and merged."""
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = workloads.custom(batch=1, q_heads=8, kv_heads=2, head_dim=64, block_size=16,
                                ctx=[1000], seed=121)
        w = workloads.make(spec)
        n = int(w.context_lens[0])                              # the sequence's K/V, contiguous
        k = workloads.bf16_bits_to_f32(w.k[:n]).astype(np.float64)
        v = workloads.bf16_bits_to_f32(w.v[:n]).astype(np.float64)
        q = workloads.bf16_bits_to_f32(w.q[0]).astype(np.float64).reshape(8, 64)
        nblk = -(-k.shape[0] // 16)
        per = -(-nblk // world)
        a, b = min(rank * per * 16, k.shape[0]), min((rank + 1) * per * 16, k.shape[0])
        o, l = oracle.attend(q, k[a:b], v[a:b], w.scale)
        o_all = [torch.zeros(8, 64, dtype=torch.float64) for _ in range(world)]
        l_all = [torch.zeros(8, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(o_all, torch.from_numpy(o))
        dist.all_gather(l_all, torch.from_numpy(l))
        merged, lse = oracle.merge_states(np.stack([t.numpy() for t in o_all]),
                                          np.stack([t.numpy() for t in l_all]))
        ref, ref_lse = oracle.attend(q, k, v, w.scale)
        res = {"err": float(np.max(np.abs(merged - ref))),
               "lse_err": float(np.max(np.abs(lse - ref_lse))), "shard": [a, b]}
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"shard{rank}.json"), "w") as fh:
        json.dump(res, fh)


def test_sequence_split_across_two_gloo_ranks_merges_to_the_whole_attention(tmp_path):
    port = _free_port()
    mp.start_processes(_shard_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    r = [json.load(open(tmp_path / f"shard{i}.json")) for i in range(2)]
    assert r[0]["shard"] == [0, 512] and r[1]["shard"] == [512, 1000]
    for x in r:
        assert x["err"] < 1e-12 and x["lse_err"] < 1e-12


def test_two_gloo_ranks_reduce_time_and_bytes_and_seed_their_own_batches(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    r0 = json.load(open(tmp_path / "rank0.json"))
    r1 = json.load(open(tmp_path / "rank1.json"))
    # the timed region is the slowest rank's; the throughput counts every rank's bytes
    assert r0["max"] == r1["max"] == 2.5
    assert r0["sum"] == r1["sum"] == 30.0
    # each rank its own seeded batch (independent replicas, weak scaling)
    assert r0["seed"] != r1["seed"]
    tiny = __import__("workloads").CONFIGS["tiny"]
    assert r0["ctx_head"] == list(tiny.ctx_fixed)       # rank 0 keeps the workload as given


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--config", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=540, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
