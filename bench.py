#!/usr/bin/env python
"""Benchmark of the paged-KV decode step (append + paged decode attention).

One step = paged_kv_append of every sequence's new K/V, then
paged_decode_attention over the whole ragged batch, on the Llama-3-8B-shaped
layer by default (batch 64, GQA 32/8, head_dim 128, block_size 16, contexts
uniform in [512, 4096], bf16 N(0,1), blocks randomly permuted in a pool of
total blocks + 10%).  Prints one JSON line.

  python bench.py [--gpus N --steps K --warmup W] [--config NAME] [--impl reference]

value: whole-step algorithmic bytes / step time (GB/s), inputs resident in HBM.
e2e:   the same, measured with host (pinned) inputs and output copied inside the
       timed region.
--impl reference: the float64 CPU oracle on the host cores, each step a
       bounded sample of the same workload.
With torchrun (N > 1) every rank runs its own batch on its own GPU (weak
scaling, no collective on the data path); the barrier and the max-over-ranks
timing use torch.distributed.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time
from dataclasses import replace

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402
from workloads import accounting  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "paged decode step (append + decode attention): achieved algorithmic HBM GB/s"
PROFILES = os.path.join(ROOT, "profiles")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="llama3_8b", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--split-tokens", type=int, default=None,
                    help="override the split-KV chunk (0 = automatic)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="measure only --config (no other workloads in the same run)")
    ap.add_argument("--extra-cpu-seconds", type=float, default=3.0,
                    help="target CPU time of the oracle baseline of each other workload")
    return ap.parse_args()


# --------------------------------------------------------------------------- helpers
KERNEL_SOURCES = {
    "gqa": ["decode_kernel.cuh", "decode_common.cuh", "decode_bf16.cu", "decode_fp8.cu",
            "device_common.cuh", "append_row.cuh"],
    "gqa_heads": ["decode_heads.cuh", "decode_heads.cu", "decode_common.cuh", "device_common.cuh",
                  "append_row.cuh"],
    "mla": ["decode_mla.cu", "decode_common.cuh", "device_common.cuh", "append_row.cuh"],
    "mla_tc": ["decode_mla_tc.cu", "mla_partition.cuh", "tcgen05.cuh", "decode_common.cuh",
               "device_common.cuh", "append_row.cuh"],
    "mla_tcn": ["decode_mla_tcn.cu", "mla_partition.cuh", "tcgen05.cuh", "decode_common.cuh",
                "device_common.cuh", "append_row.cuh"],
}


def kernel_kind(spec, cta_heads: int = 1) -> str:
    """Which decode kernel a workload runs: the GQA kernel with one CTA per kv head or per
    group of cta_heads kv heads (the library's plan, paged_decode_cta_heads), or a form of
    the latent decode (tcgen05 for blocks of 64: the wide form for at least 64 query heads,
    the narrow one below; mma.sync for other block sizes)."""
    if not spec.mla:
        return "gqa" if cta_heads == 1 else "gqa_heads"
    if spec.block_size != 64:
        return "mla"
    return "mla_tc" if spec.q_heads >= 64 else "mla_tcn"


KERNEL_NAMES = {"gqa": "paged_decode_main", "gqa_heads": "paged_decode_heads (a CTA per group of kv heads)",
                "mla": "paged_mla_decode_main (mma.sync)",
                "mla_tc": "paged_mla_decode_tc (tcgen05)",
                "mla_tcn": "paged_mla_decode_tcn (tcgen05, 16-head tiles)"}


def kernel_source_sha(kind: str = "gqa") -> str:
    """Hash of the device sources the timed decode kernel is compiled from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_19_gb300", "csrc")
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(config: str, kind: str):
    """DRAM bytes per decode launch recorded by an ncu capture of the current kernels.

    A profile summary under profiles/ states `kernel_source_sha:` and
    `dram_bytes_per_launch:` for a workload; it counts only while the sources
    are unchanged."""
    sha = kernel_source_sha(kind)
    for path in glob.glob(os.path.join(PROFILES, "*.md")) + glob.glob(os.path.join(PROFILES, "*.txt")):
        text = open(path).read()
        m_sha = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", text)
        m_cfg = re.search(r"bench_config:\s*(\w+)", text)
        m_b = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
        if m_sha and m_b and m_cfg and m_sha.group(1) == sha and m_cfg.group(1) == config:
            return int(m_b.group(1)), os.path.relpath(path, ROOT)
    return None, None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor throughput (TFLOP/s, burst) and where it comes from."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, with host timestamps."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return None
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside:             # region shorter than the sampling period: nearest samples
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest to the timed region"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(p[0]) for _, p in inside]
        reasons = set()
        for _, p in inside:
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"], p[3:]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": num(inside[0][1][1]),
                "power_w_max": max(num(p[2]) for _, p in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


def dist_setup(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_spec(config: str, rank: int):
    spec = workloads.CONFIGS[config]
    return spec if rank == 0 else replace(spec, seed=spec.seed + 100_000 * rank)


def tc_grid(w, split_tokens, sms=152):
    """CTAs of the tensor-core MLA launch (the library's rule: one per SM, no more than
    ranges of split_blocks units the batch could hold)."""
    s = w.spec
    outer = -(-s.q_heads // 128) * 2 if kernel_kind(s) == "mla_tc" else -(-s.q_heads // 16)
    units = outer * w.batch * w.max_blocks
    return min(sms, max(1, units // max(1, split_tokens // s.block_size)))


def decode_bytes(w, split_tokens, sms=152):
    if w.spec.mla:
        kind = kernel_kind(w.spec)
        grid = tc_grid(w, split_tokens, sms) if kind in ("mla_tc", "mla_tcn") else 0
        return accounting.mla_decode_bytes(w, split_tokens, tc_grid=grid,
                                           form="wide" if kind == "mla_tc" else "narrow")
    return accounting.decode_bytes(w, split_tokens)


def workload_config(w, split_tokens, max_splits, world):
    s = w.spec
    kv = decode_bytes(w, split_tokens)
    return {
        "workload": s.name, "batch": s.batch, "q_heads": s.q_heads, "kv_heads": s.kv_heads,
        "head_dim": s.head_dim, "block_size": s.block_size, "cache_dtype": s.cache_dtype,
        "q_len": s.q_len,
        "context_tokens": w.total_tokens, "ctx_min": int(w.context_lens.min()),
        "ctx_max": int(w.context_lens.max()), "num_blocks": w.num_blocks,
        "split_tokens": split_tokens, "max_splits": max_splits,
        "kv_bytes_logical": kv["kv_logical"], "kv_bytes_unique": kv["kv_unique"],
        "l2": (f"no flush: the KV pool read per step ({kv['kv_logical'] / 1e6:.0f} MB) is larger "
               f"than the 129 MB L2" if kv["kv_logical"] > L2_BYTES else
               "working set smaller than L2: numbers include L2 hits"),
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        "seed": s.seed,
        **({"attention": "MLA absorbed (one cached vector per token: latent + rotary key)",
            "latent_dim": s.latent_dim, "rope_dim": s.head_dim - s.latent_dim,
            "softmax_scale": f"1/sqrt({s.qk_head_dim})"} if s.mla else {}),
    }


# --------------------------------------------------------------------------- CPU oracle legs
def oracle_step_sample(w, seqs, threads):
    """One oracle step on a sample of sequences: append their new tokens, then decode them."""
    import oracle
    s = w.spec
    # append: the sampled sequences' target blocks, remapped into a small pool image
    # (a latent pool has one cached vector per token: the V image is scratch)
    pos = w.context_lens[seqs] - 1
    blocks = w.block_tables[seqs, pos // s.block_size]
    uniq, inv = np.unique(blocks, return_inverse=True)
    table = np.zeros((len(seqs), w.max_blocks), dtype=np.int32)
    table[np.arange(len(seqs)), pos // s.block_size] = inv.astype(np.int32)
    shape = (uniq.size, s.block_size, s.kv_heads, s.head_dim * w.elem_bytes)
    kp_img = np.full(shape, 0xFF, dtype=np.uint8)
    vp_img = np.full(shape, 0xFF, dtype=np.uint8)
    oracle.append(kp_img, vp_img, s.cache_dtype, s.block_size, w.k_new[seqs], w.v_new[seqs], table,
                  w.context_lens[seqs], k_scale=w.k_scale, v_scale=w.v_scale)
    if s.mla:
        return oracle.mla_decode_workload(w, seqs=seqs)
    return oracle.decode_workload(w, seqs=seqs, threads=threads)


def sample_bytes(w, seqs):
    s = w.spec
    if s.mla:
        ntok = int(w.context_lens[seqs].astype(np.int64).sum())
        qo = len(seqs) * s.q_heads * (s.head_dim + s.latent_dim) * 2
        return ntok * s.head_dim * 2 + qo + len(seqs) * s.head_dim * 4, ntok
    row = 2 * s.kv_heads * s.head_dim * w.elem_bytes
    kv = int(w.context_lens[seqs].astype(np.int64).sum()) * row
    qo = 2 * len(seqs) * s.q_heads * s.head_dim * 2
    app = len(seqs) * s.kv_heads * s.head_dim * (4 + 2 * w.elem_bytes)
    return kv + qo + app, int(w.context_lens[seqs].astype(np.int64).sum())


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(w, target_s: float, gpu_out=None):
    """The oracle as it stands on the host cores, on a bounded sample of the workload."""
    threads = os.cpu_count() or 1
    order = np.random.default_rng(0).permutation(w.batch)
    n = min(w.batch, threads)
    t0 = time.perf_counter()
    out, _ = oracle_step_sample(w, order[:n], threads)
    dt = time.perf_counter() - t0
    seqs = order[:n]
    if dt < target_s / 4 and n < w.batch:        # grow the sample towards the target time
        n2 = int(min(w.batch, max(n + 1, n * target_s / max(dt, 1e-3) / 2)))
        seqs = order[:n2]
        t0 = time.perf_counter()
        out, _ = oracle_step_sample(w, seqs, threads)
        dt = time.perf_counter() - t0
    times = [dt]
    if dt < target_s / 3:                         # the whole batch is quick: repeat it
        for _ in range(int(min(200, (target_s / 3) / max(dt, 1e-3)))):
            t0 = time.perf_counter()
            oracle_step_sample(w, seqs, threads)
            times.append(time.perf_counter() - t0)
    best, mean = min(times), sum(times) / len(times)
    nbytes, ntok = sample_bytes(w, seqs)
    used = 1 if w.spec.mla else threads           # the MLA oracle runs on one thread
    res = {"value": round(nbytes / best / 1e9, 4), "unit": "GB/s", "cores": used,
           "kind": "oracle",
           "sample": (f"append + decode of {len(seqs)} of {w.batch} sequences ({ntok} cached "
                      f"tokens, all {w.spec.q_heads} query heads), float64 C oracle, "
                      f"{used} thread{'s' if used > 1 else ''}, best of {len(times)} "
                      f"pass{'es' if len(times) > 1 else ''} ({best * 1e3:.1f} ms; mean "
                      f"{mean * 1e3:.1f} ms; {sum(times):.1f} s in all)"),
           "mean_value": round(nbytes / mean / 1e9, 4),
           "kv_tokens_per_s": round(ntok / best, 1),
           "nproc": os.cpu_count(), "cpu_model": cpu_model()}
    if used > 1:                                  # the same oracle on one thread
        few = seqs[:max(1, min(len(seqs), 8))]
        t0 = time.perf_counter()
        oracle_step_sample(w, few, 1)
        t1 = time.perf_counter() - t0
        res["single_thread"] = {"value": round(sample_bytes(w, few)[0] / t1 / 1e9, 4),
                                "unit": "GB/s", "sequences": int(len(few)),
                                "seconds": round(t1, 3)}
    if gpu_out is not None:
        got = gpu_out[seqs].float().cpu().double().numpy()
        err = got - out
        res["sample_max_abs_err_vs_gpu"] = float(np.max(np.abs(err)))
        res["sample_rel_l2_err_vs_gpu"] = float(np.linalg.norm(err) / np.linalg.norm(out))
    return res


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = workloads.make(workloads.CONFIGS[args.config])
    threads = os.cpu_count() or 1
    order = np.random.default_rng(0).permutation(w.batch)
    # size each step so that warm-up + timed steps fit about two minutes
    t0 = time.perf_counter()
    oracle_step_sample(w, order[:1], threads)
    per_seq = max(time.perf_counter() - t0, 1e-4)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(w.batch, threads * budget / per_seq)))
    steps_seqs = [np.take(order, np.arange(i * n, i * n + n), mode="wrap")
                  for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        oracle_step_sample(w, steps_seqs[i], threads)
    total_bytes = 0
    total_tok = 0
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        oracle_step_sample(w, steps_seqs[i], threads)
        b, tok = sample_bytes(w, steps_seqs[i])
        total_bytes += b
        total_tok += tok
    dt = time.perf_counter() - t0
    value = total_bytes / dt / 1e9
    if w.spec.mla:
        threads = 1                                # the MLA oracle runs on one thread
    sample = (f"each step: append + decode of {n} of {w.batch} sequences, float64 C oracle, "
              f"{threads} thread{'s' if threads > 1 else ''}")
    line = {
        "impl": "reference", "metric": METRIC,
        "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "kv_tokens_per_s": round(total_tok / dt, 1),
        "config": {"workload": w.spec.name, "batch": w.spec.batch, "sample_sequences_per_step": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def mla_roofline(w, dec_bytes, dec_ms, hbm_peak):
    """Extra roofline figures of the MLA decode: its arithmetic is dense enough (every head
    of a sequence scores each cached vector) that the tensor-core time is reported too."""
    flops = accounting.mla_decode_flops(w)
    tpeak, tkind = measured_tensor_peak()
    t_hbm = dec_bytes["total"] / (hbm_peak * 1e9)
    t_mma = flops / (tpeak * 1e12)
    return {"flops_per_launch": flops,
            "intensity_flop_per_byte": round(flops / dec_bytes["total"], 1),
            "ridge_flop_per_byte": round(tpeak * 1e12 / (hbm_peak * 1e9), 1),
            "tensor_achieved_tflops": round(flops / (dec_ms / 1e3) / 1e12, 1),
            "tensor_peak_tflops": tpeak, "tensor_peak_kind": f"{tkind} cuBLAS bf16 (burst)",
            "tensor_frac": round(flops / (dec_ms / 1e3) / 1e12 / tpeak, 4),
            "bound_by_arithmetic": "tensor" if t_mma > t_hbm else "hbm",
            "l2_vector_reads_per_launch": dec_bytes["l2_reads"]}


# --------------------------------------------------------------------------- GPU arm
def stage(w, device):
    import torch
    import paged_kv_cache_19_gb300 as kp
    s = w.spec

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    if s.mla:
        pool = kp.kv_mla_pool_create(w.num_blocks, s.block_size, s.latent_dim,
                                     s.head_dim - s.latent_dim, device=device.index)
    else:
        pool = kp.kv_pool_create(w.num_blocks, s.block_size, s.kv_heads, s.head_dim,
                                 s.cache_dtype, device=device.index)
    for t in pool.raw_bytes():
        if t is not None:
            t.fill_(workloads.POISON_BYTE)
    if s.cache_dtype == "fp8_e4m3":
        pool.set_scales(w.k_scale, w.v_scale)
    tables, ctx = i32(w.block_tables), i32(w.context_lens)
    chunk = 1 << 16
    for a in range(0, w.prefill_seq.size, chunk):
        rows = w.prefill_row[a:a + chunk]
        kp.paged_kv_append(pool, bf16(w.k[rows]), None if s.mla else bf16(w.v[rows]), tables, ctx,
                           token_seq=i32(w.prefill_seq[a:a + chunk]),
                           token_pos=i32(w.prefill_pos[a:a + chunk]))
    step = {"q": bf16(w.q if w.q_len == 1 else w.q_multi), "k": bf16(w.k[w.step_rows]),
            "v": None if s.mla else bf16(w.v[w.step_rows]),
            "seq": None if w.q_len == 1 else i32(w.step_seq),
            "pos": None if w.q_len == 1 else i32(w.step_pos)}
    return pool, tables, ctx, step


NOMINAL_HBM_GBS = 8000.0          # GB300 HBM3e, nominal (about 8 TB/s)
# The workloads measured in the same run after the headline one (one GPU only): the other
# bench configurations (the tiny one is launch-bound: reported, not a roofline claim), the
# multi-token verify pass and both latent-attention layers.
EXTRA_CONFIGS = ["tiny", "long_context", "ragged_prefix", "mha_fp8", "llama3_8b_verify4",
                 "deepseek_mla", "deepseek_mla_tp8"]


class Staged:
    """One workload resident on the GPU and the library calls the bench times."""

    def __init__(self, w, device, split_override):
        import torch
        import paged_kv_cache_19_gb300 as kp
        self.kp = kp
        self.w = w
        s = self.s = w.spec
        self.device = device
        self.split_req = s.split_tokens if split_override is None else split_override
        self.pool, self.tables, self.ctx, self.stp = stage(w, device)
        self.q = self.stp["q"]
        if s.mla:
            self.split_tokens, self.max_splits = kp.paged_mla_decode_plan(
                self.pool, s.batch, s.q_heads, w.max_blocks, self.split_req)
            ws_bytes = kp.paged_mla_workspace_size(self.pool, s.batch, s.q_heads, w.max_blocks,
                                                   self.split_req)
            self.out = torch.empty(s.batch, s.q_heads, s.latent_dim, dtype=torch.bfloat16,
                                   device=device)
        else:
            self.split_tokens, self.max_splits = kp.paged_decode_plan(
                self.pool, s.batch, s.q_heads, w.max_blocks, self.split_req)
            ws_bytes = kp.paged_multi_query_workspace_size(self.pool, s.batch, s.q_heads, s.q_len,
                                                           w.max_blocks, self.split_req)
            self.out = torch.empty_like(self.q)
        self.workspace = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=device)
        self.lse = torch.empty(self.q.shape[:-1], dtype=torch.float32, device=device)
        self.stream = torch.cuda.current_stream()
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.dec_bytes = decode_bytes(w, self.split_tokens, sms)
        self.app_bytes = accounting.mla_append_bytes(w) if s.mla else accounting.append_bytes(w)
        self.step_bytes = self.dec_bytes["total"] + self.app_bytes
        # append + decode; the tensor-core MLA forms add their merge kernel when sequences
        # can be cut into pieces (the other kernels merge inside the decode kernel)
        self.cta_heads = 1 if s.mla else kp.paged_decode_cta_heads(
            self.pool, s.batch, s.q_heads, s.q_len, w.max_blocks, self.split_req)
        self.kind = kernel_kind(s, self.cta_heads)
        self.two_kernels = self.kind in ("mla_tc", "mla_tcn") and self.max_splits > 1
        # paged_decode_step on a K/V pool whose kv heads have at most 8 query rows is one
        # kernel (its CTAs write the new rows before loading their blocks), else the append
        # kernel then the attention; on a latent pool the attention kernel writes the new
        # vectors itself (plus the merge kernel of the tensor-core forms when sequences can
        # be cut)
        rows = s.q_heads // s.kv_heads * s.q_len
        if s.mla:
            self.launches_per_step = 2 if self.two_kernels else 1
        else:
            self.launches_per_step = 1 if rows <= 8 else 2

    def attend(self, out=None):
        kp, s, w = self.kp, self.s, self.w
        out = self.out if out is None else out
        if s.mla:
            kp.paged_mla_decode_attention(self.pool, self.q, self.tables, self.ctx, w.scale,
                                          kv_split_tokens=self.split_req, workspace=self.workspace,
                                          out=out, lse=self.lse, stream=self.stream,
                                          latent_dim=s.latent_dim)
        elif s.q_len == 1:
            kp.paged_decode_attention(self.pool, self.q, self.tables, self.ctx, w.scale,
                                      kv_split_tokens=self.split_req, workspace=self.workspace,
                                      out=out, lse=self.lse, stream=self.stream)
        else:
            kp.paged_attention_multi_query(self.pool, self.q, self.tables, self.ctx, w.scale,
                                           kv_split_tokens=self.split_req,
                                           workspace=self.workspace, out=out, lse=self.lse,
                                           stream=self.stream)

    def run_step(self, kk, vv, qq, tt, cc, out=None):
        """One decode step through the public API: append + attention in one call --
        paged_decode_step for K/V caches, paged_mla_decode_step for latent pools.  The step's tokens are the last q_len of
        every sequence, in sequence order, which is the layout both calls take."""
        kp, s, w = self.kp, self.s, self.w
        out = self.out if out is None else out
        if s.mla:
            kp.paged_mla_decode_step(self.pool, kk, qq, tt, cc, w.scale,
                                     kv_split_tokens=self.split_req, workspace=self.workspace,
                                     out=out, lse=self.lse, stream=self.stream,
                                     latent_dim=s.latent_dim)
        else:
            kp.paged_decode_step(self.pool, kk, vv, qq, tt, cc, w.scale,
                                 kv_split_tokens=self.split_req, workspace=self.workspace,
                                 out=out, lse=self.lse, stream=self.stream)

    def step(self):
        self.run_step(self.stp["k"], self.stp["v"], self.q, self.tables, self.ctx)

    def _loop_ms(self, fn, n):
        import torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(self.stream)
        for _ in range(n):
            fn()
        e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def decode_ms(self, n):
        """The decode kernel alone: n launches back to back; mean ms per call."""
        return self._loop_ms(self.attend, n) / n

    def append_ms(self, n):
        """The append kernel alone: n launches back to back (rewriting the same slots)."""
        kp, stp = self.kp, self.stp

        def app():
            kp.paged_kv_append(self.pool, stp["k"], stp["v"], self.tables, self.ctx,
                               token_seq=stp["seq"], token_pos=stp["pos"], stream=self.stream)

        return self._loop_ms(app, n) / n

    def per_call_us(self, n):
        """The decode kernel per call, L2 flushed before each (a read of twice the L2 size
        between the calls, outside the event pair: it evicts every earlier line and, unlike
        a write, leaves no dirty lines for the timed kernel to write back)."""
        import torch
        flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=self.device)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(n)]
        for e0, e1 in pairs:
            flush.sum()
            e0.record(self.stream)
            self.attend()
            e1.record(self.stream)
        torch.cuda.synchronize()
        del flush
        return sorted(e0.elapsed_time(e1) * 1e3 for e0, e1 in pairs)

    def e2e(self, steps, warmup, world, all_bytes):
        """The step end to end: every step copies its inputs from pinned host memory and
        reads its output back.  Two device input buffers and two outputs let step i + 1's
        host-to-device copy and step i's device-to-host copy run on a copy stream while
        step i + 1 / step i computes; every step still moves its own bytes both ways."""
        import torch
        stp = self.stp
        inputs = [("q", self.q), ("k", stp["k"]), ("tables", self.tables), ("ctx", self.ctx)]
        if stp["v"] is not None:
            inputs.append(("v", stp["v"]))
        if stp["seq"] is not None:
            inputs += [("seq", stp["seq"]), ("pos", stp["pos"])]
        # the step's inputs packed into one pinned host buffer (16-byte aligned pieces) and
        # copied with one host-to-device copy per step into a device buffer whose views the
        # call takes
        offs, total = {}, 0
        for name, t in inputs:
            offs[name] = total
            total += -(-t.numel() * t.element_size() // 16) * 16
        h_buf = torch.empty(total, dtype=torch.uint8, pin_memory=True)
        d_bufs = [torch.empty(total, dtype=torch.uint8, device=self.device) for _ in range(2)]

        def view(buf, name, t):
            n = t.numel() * t.element_size()
            return buf[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)

        for name, t in inputs:
            view(h_buf, name, t).copy_(t.cpu())
        views = [{name: view(b, name, t) for name, t in inputs} for b in d_bufs]
        outs = [self.out, torch.empty_like(self.out)]
        h_outs = [torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
                  for _ in range(2)]
        comp = self.stream
        copy = torch.cuda.Stream(device=self.device)
        ev = lambda: torch.cuda.Event()                                  # noqa: E731
        in_ready, done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        for e in done + out_read:
            e.record(comp)

        def h2d(i):
            j = i % 2
            copy.wait_event(done[j])               # step i - 2 has finished reading d_bufs[j]
            with torch.cuda.stream(copy):
                d_bufs[j].copy_(h_buf, non_blocking=True)
            in_ready[j].record(copy)

        def run(n):
            h2d(0)
            for i in range(n):
                j = i % 2
                if i + 1 < n:
                    h2d(i + 1)                     # overlaps step i
                comp.wait_event(in_ready[j])
                comp.wait_event(out_read[j])       # step i - 2's output has been read
                d = views[j]
                self.run_step(d["k"], d.get("v"), d["q"], d["tables"], d["ctx"], out=outs[j])
                done[j].record(comp)
                copy.wait_event(done[j])
                with torch.cuda.stream(copy):
                    h_outs[j].copy_(outs[j], non_blocking=True)
                out_read[j].record(copy)

        run(max(3, warmup))
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(copy)
        run(steps)
        e1.record(copy)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
        bo = h_outs[0].numel() * h_outs[0].element_size()
        return {"value": round(all_bytes / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": total, "d2h_bytes_per_step": bo,
                "ms_per_step": round(e2e_ms / steps, 5),
                "overlap": "double-buffered inputs and outputs; copies on a second stream "
                           "overlap the neighbouring steps' compute"}

    def destroy(self):
        self.pool.destroy()


def roofline_obj(st, dec_ms, peak, peak_kind, config_name):
    """The roofline figures of a workload's decode kernel: algorithmic bytes per launch over
    the back-to-back launch time, against the measured copy bandwidth and the nominal HBM
    bandwidth, with the DRAM traffic of an ncu capture of the same sources."""
    s = st.s
    achieved = st.dec_bytes["total"] / (dec_ms / 1e3) / 1e9
    kind = st.kind
    traffic, traffic_src = profiled_traffic(config_name, kind)
    return {"kernel": KERNEL_NAMES[kind]
                      + ((" + paged_mla_merge_tc" + ("n" if kind == "mla_tcn" else "")
                          + " (the decode call's two launches; ") if st.two_kernels else
                         " (one launch per decode call, in-kernel split-KV merge; ")
                      + "K calls timed back to back)",
            "bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": traffic, "traffic_source": traffic_src,
            "algorithmic_bytes_per_launch": st.dec_bytes["total"],
            "algorithmic_bytes_unique_per_launch": st.dec_bytes["total_unique"],
            **(mla_roofline(st.w, st.dec_bytes, dec_ms, peak) if s.mla else {})}


def measure_extra(name, args, device, peak, peak_kind):
    """One more workload in the same run: the step and the decode kernel back to back, the
    decode per call with L2 flushed, and the oracle on a short sample of host work."""
    import torch
    w = workloads.make(workloads.CONFIGS[name])
    st = Staged(w, device, None)
    steps = 200
    for _ in range(max(3, args.warmup)):
        st.step()
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0, f"device-side error during warm-up ({name})"
    step_ms = st._loop_ms(st.step, steps) / steps
    dec_ms = st.decode_ms(steps)
    per_call = st.per_call_us(20)
    assert st.pool.device_errors() == 0, f"device-side error during the timed calls ({name})"
    res = {
        "workload": name, "steps": steps,
        "config": workload_config(w, st.split_tokens, st.max_splits, 1),
        "step_ms": round(step_ms, 5),
        "step_gbs": round(st.step_bytes / (step_ms / 1e3) / 1e9, 2),
        "kv_tokens_per_s": round(w.total_tokens / (step_ms / 1e3), 1),
        "decode_us_back_to_back": round(dec_ms * 1e3, 2),
        "decode_per_call": {"calls": len(per_call), "median_us": round(statistics.median(per_call), 2),
                            "min_us": round(per_call[0], 2),
                            "l2": "flushed before each call (a read of twice the L2 size)",
                            "median_gbs": round(st.dec_bytes["total"]
                                                / (statistics.median(per_call) * 1e-6) / 1e9, 2)},
        "roofline": roofline_obj(st, dec_ms, peak, peak_kind, name),
    }
    out = st.out
    st.destroy()
    if not args.no_cpu_baseline and w.spec.q_len == 1:
        res["cpu_baseline"] = cpu_baseline(w, args.extra_cpu_seconds, gpu_out=out)
    del out
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local):
    import torch
    import paged_kv_cache_19_gb300 as kp
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    kp.load_library()
    w = workloads.make(rank_spec(args.config, rank))
    s = w.spec
    st = Staged(w, device, args.split_tokens)
    stream = st.stream

    for _ in range(max(3, args.warmup)):
        st.step()
    torch.cuda.synchronize()
    assert st.pool.device_errors() == 0, "device-side error during warm-up"

    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(device).uuid)
        gpu_uuid = gpu_uuid if gpu_uuid.startswith("GPU-") else "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = str(local)
    sampler = None if args.no_clocks else ClockSampler(gpu_uuid)
    if sampler is not None:
        time.sleep(0.3)

    # ---- timed region: K steps (append + decode) back to back, events on the
    # launching stream at both ends only (an event between the two kernels would
    # stop the decode from launching while the append finishes)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    host0 = time.time()
    t_start.record(stream)
    for _ in range(args.steps):
        st.step()
    t_end.record(stream)
    torch.cuda.synchronize()
    host1 = time.time()
    barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    total_ms_max = max_over_ranks(total_ms, world)

    # ---- the decode kernel alone (roofline of the kernel), per call with L2 flushed, and
    # the append kernel alone
    dec_avg_ms = st.decode_ms(args.steps)
    n_calls = min(50, max(5, args.steps))
    per_call_us = st.per_call_us(n_calls)
    app_avg_ms = st.append_ms(args.steps)
    assert st.pool.device_errors() == 0, "device-side error during the timed region"
    if sampler is not None:
        time.sleep(0.2)
        sampler.stop()
        clocks = sampler.summary(host0, host1)
    else:
        clocks = None

    all_bytes = sum_over_ranks(st.step_bytes * args.steps, world)
    value = all_bytes / (total_ms_max / 1e3) / 1e9
    kv_tok = sum_over_ranks(w.total_tokens * args.steps, world) / (total_ms_max / 1e3)
    peak, peak_kind = measured_peaks()

    # ---- end to end: host (pinned) inputs copied in and the output copied out every step
    e2e = None if args.no_e2e else st.e2e(args.steps, args.warmup, world, all_bytes)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and s.q_len == 1:
        cpu = cpu_baseline(w, args.cpu_seconds, gpu_out=st.out)
    line_cfg = workload_config(w, st.split_tokens, st.max_splits, world)
    app_bytes = st.app_bytes
    launches = st.launches_per_step * args.steps
    roof = roofline_obj(st, dec_avg_ms, peak, peak_kind, args.config)
    st.destroy()
    del st
    torch.cuda.empty_cache()

    # ---- the other workloads, in the same run (one GPU only)
    extra = None
    if world == 1 and not args.no_extra:
        extra = {}
        for name in EXTRA_CONFIGS:
            if name == args.config:
                continue
            extra[name] = measure_extra(name, args, device, peak, peak_kind)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms_max / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if s.cache_dtype == "bf16" else "fp8_e4m3 cache, bf16 q/out",
            "data": "synthetic (seeded N(0,1) bf16, no trained weights)",
            "config": line_cfg,
            "pct_of_peak": round(100 * value / peak, 2),
            "pct_of_nominal_peak": round(100 * value / NOMINAL_HBM_GBS, 2),
            "kv_tokens_per_s": round(kv_tok, 1),
            "decode_ms_per_call": round(dec_avg_ms, 5),
            "decode_per_call": {"calls": n_calls, "median_us": round(statistics.median(per_call_us), 2),
                                "min_us": round(per_call_us[0], 2),
                                "l2": "flushed before each call (a read of twice the L2 size)",
                                "median_gbs": round(roof["algorithmic_bytes_per_launch"]
                                                    / (statistics.median(per_call_us) * 1e-6) / 1e9, 2)},
            "append": {"kernel": "paged_kv_append_kernel (K launches back to back after the timed "
                                 "steps)",
                       "ms_per_call": round(app_avg_ms, 5), "bytes_per_call": app_bytes,
                       "achieved_gbs": round(app_bytes / (app_avg_ms / 1e3) / 1e9, 2),
                       "frac": round(app_bytes / (app_avg_ms / 1e3) / 1e9 / peak, 4),
                       "bound": "launch latency (a few hundred KB per call)"},
            "roofline": roof,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": launches,
            "clocks": clocks,
            "other_workloads": extra,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
