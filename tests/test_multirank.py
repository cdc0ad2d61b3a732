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
