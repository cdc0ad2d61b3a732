"""Seeded synthetic decode-step workloads for the paged KV cache.

This module only draws inputs: shapes, context lengths, block tables, and
N(0,1) values rounded to bf16.  It contains none of the attention arithmetic,
so the CUDA path and the float64 oracle can both consume its output without
sharing any of the method's code.

Shapes follow the workloads named for the method (Llama-3-8B-like GQA 32/8 at
head_dim 128, long contexts with split-KV, prefix-shared ragged batches, an
MHA fp8 cache).  The pool layout is [num_blocks, block_size, kv_heads,
head_dim] for K and for V, as in the vLLM layout described on
"The KV cache and PagedAttention" (xuewyang.github.io/posts/kv, section
"Reading the code: a warehouse of lockers").

Reproducibility: every stream is a numpy PCG64 generator keyed by
(seed, role, index), so any one sequence can be regenerated on its own.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

# Byte that poisons unused pool memory: 0xFFFF is a bf16 NaN and 0xFF an e4m3fn
# NaN (S.1111.111), so any slot the kernels should skip reads as NaN if touched.
POISON_BYTE = 0xFF
DTYPES = ("bf16", "fp8_e4m3")


@dataclass(frozen=True)
class Spec:
    """Shape and sampling recipe of one decode step."""
    name: str
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    block_size: int
    cache_dtype: str = "bf16"
    seed: int = 0
    ctx_fixed: tuple = ()           # explicit context lengths (overrides sampling)
    ctx_uniform: tuple = ()         # (lo, hi) inclusive integers
    ctx_lognormal: tuple = ()       # (median, sigma, lo, hi)
    prefix_group: int = 0           # sequences per shared-prefix group (0: no sharing)
    prefix_tokens: int = 0          # tokens of the shared prefix
    pool_blocks: int = 0            # fixed pool size; 0 -> ceil(1.1 * blocks in use)
    split_tokens: int = 0           # split-KV chunk (0 = library's automatic choice)
    q_len: int = 1                  # new tokens per sequence in the step (1: decode)
    latent_dim: int = 0             # MLA: one cached vector per token, its first latent_dim
                                    # numbers are the value (kv_heads 1, head_dim = latent + rope)
    qk_head_dim: int = 0            # softmax scale 1/sqrt(qk_head_dim) (0: head_dim)
    note: str = ""

    @property
    def mla(self) -> bool:
        return self.latent_dim > 0


# The five workloads.  Seeds are 1000 + index.
CONFIGS = {
    "tiny": Spec("tiny", batch=4, q_heads=4, kv_heads=4, head_dim=64, block_size=16,
                 seed=1001, ctx_fixed=(17, 64, 100, 129), pool_blocks=64,
                 note="tiny paged decode, one layer"),
    "llama3_8b": Spec("llama3_8b", batch=64, q_heads=32, kv_heads=8, head_dim=128,
                      block_size=16, seed=1002, ctx_uniform=(512, 4096),
                      note="Llama-3-8B-shaped decode layer, GQA 32/8"),
    "long_context": Spec("long_context", batch=8, q_heads=64, kv_heads=8, head_dim=128,
                         block_size=16, seed=1003, ctx_uniform=(32768, 131072),
                         split_tokens=4096,
                         note="long-context split-KV decode, GQA 64/8, 4096-token chunks"),
    "ragged_prefix": Spec("ragged_prefix", batch=256, q_heads=32, kv_heads=8, head_dim=128,
                          block_size=16, seed=1004, ctx_lognormal=(1024, 0.8, 16, 8192),
                          prefix_group=8, prefix_tokens=512,
                          note="ragged lognormal batch, groups of 8 share a 512-token prefix"),
    "llama3_8b_verify4": Spec("llama3_8b_verify4", batch=64, q_heads=32, kv_heads=8,
                              head_dim=128, block_size=16, seed=1012, ctx_uniform=(512, 4096),
                              q_len=4,
                              note="speculative verify pass: 4 new tokens per sequence on the "
                                   "Llama-3-8B-shaped layer"),
    "mha_fp8": Spec("mha_fp8", batch=128, q_heads=32, kv_heads=32, head_dim=128,
                    block_size=32, cache_dtype="fp8_e4m3", seed=1005, ctx_fixed=(2048,) * 128,
                    note="MHA 7B-shaped decode with an fp8 e4m3 cache"),
    # Multi-head latent attention, absorbed decode: 512 latent + 64 rotary-key numbers
    # per token (DeepSeek-V2/V3), softmax scale 1/sqrt(128 + 64), blocks of 64 tokens.
    "deepseek_mla": Spec("deepseek_mla", batch=64, q_heads=128, kv_heads=1, head_dim=576,
                         block_size=64, seed=1013, ctx_uniform=(512, 4096), latent_dim=512,
                         qk_head_dim=192,
                         note="DeepSeek-V3-shaped MLA decode layer, all 128 heads on one GPU"),
    "deepseek_mla_tp8": Spec("deepseek_mla_tp8", batch=64, q_heads=16, kv_heads=1, head_dim=576,
                             block_size=64, seed=1014, ctx_uniform=(512, 4096), latent_dim=512,
                             qk_head_dim=192,
                             note="the same layer with its heads split over 8 GPUs (16 per GPU)"),
}


def custom(name="custom", *, batch, q_heads, kv_heads, head_dim, block_size,
           cache_dtype="bf16", seed=7, ctx=None, ctx_uniform=(), prefix_group=0,
           prefix_tokens=0, pool_blocks=0, split_tokens=0, q_len=1, latent_dim=0,
           qk_head_dim=0) -> Spec:
    """A small workload for tests: explicit lengths or a uniform range."""
    return Spec(name, batch=batch, q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
                block_size=block_size, cache_dtype=cache_dtype, seed=seed,
                ctx_fixed=tuple(int(c) for c in ctx) if ctx is not None else (),
                ctx_uniform=tuple(ctx_uniform), prefix_group=prefix_group,
                prefix_tokens=prefix_tokens, pool_blocks=pool_blocks,
                split_tokens=split_tokens, q_len=q_len, latent_dim=latent_dim,
                qk_head_dim=qk_head_dim)


def mla(name="mla", *, batch, q_heads, block_size, seed=7, ctx=None, ctx_uniform=(),
        split_tokens=0, pool_blocks=0) -> Spec:
    """A small MLA workload (512 latent + 64 rotary-key numbers per token)."""
    return custom(name, batch=batch, q_heads=q_heads, kv_heads=1, head_dim=576,
                  block_size=block_size, seed=seed, ctx=ctx, ctx_uniform=ctx_uniform,
                  split_tokens=split_tokens, pool_blocks=pool_blocks, latent_dim=512,
                  qk_head_dim=192)


def _rng(*key) -> np.random.Generator:
    return np.random.default_rng([int(k) for k in key])


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(shape, *key) -> np.ndarray:
    return f32_to_bf16_bits(_rng(*key).standard_normal(shape, dtype=np.float32))


def context_lengths(spec: Spec) -> np.ndarray:
    """Context lengths, counting the token appended in this step."""
    if spec.ctx_fixed:
        ctx = np.array(spec.ctx_fixed, dtype=np.int64)
        assert ctx.size == spec.batch, "ctx_fixed must list one length per sequence"
    elif spec.ctx_uniform:
        lo, hi = spec.ctx_uniform
        ctx = _rng(spec.seed, 0).integers(lo, hi, size=spec.batch, endpoint=True)
    elif spec.ctx_lognormal:
        median, sigma, lo, hi = spec.ctx_lognormal
        z = _rng(spec.seed, 0).standard_normal(spec.batch)
        ctx = np.clip(np.rint(np.exp(math.log(median) + sigma * z)), lo, hi).astype(np.int64)
    else:
        raise ValueError("spec gives no context lengths")
    return ctx.astype(np.int32)


@dataclass
class Workload:
    spec: Spec
    context_lens: np.ndarray        # int32 [B]
    block_tables: np.ndarray        # int32 [B, max_blocks]; entries past a sequence's blocks are -1
    num_blocks: int
    q: np.ndarray                   # uint16 bf16 bits [B, Hq, d]
    k: np.ndarray                   # uint16 bf16 bits [T_total, Hkv, d], sequences back to back
    v: np.ndarray                   # same
    seq_start: np.ndarray           # int64 [B]: row of position 0 of each sequence in k / v
    shared_block: np.ndarray        # bool [B, max_blocks]: entry is a block shared with another sequence
    k_scale: np.ndarray | None      # float32 [Hkv] (fp8 cache only)
    v_scale: np.ndarray | None
    prefill_seq: np.ndarray = field(default=None)   # int32 [N]: tokens written before the step
    prefill_pos: np.ndarray = field(default=None)   # int32 [N]
    prefill_row: np.ndarray = field(default=None)   # int64 [N]: row in k / v
    q_multi: np.ndarray | None = None               # uint16 bf16 [B, Hq, q_len, d] when q_len > 1

    @property
    def q_len(self) -> int:
        return self.spec.q_len

    @property
    def step_seq(self) -> np.ndarray:
        """Sequence of each token appended in the step (q_len per sequence)."""
        return np.repeat(np.arange(self.batch, dtype=np.int32), self.q_len)

    @property
    def step_pos(self) -> np.ndarray:
        ctx = self.context_lens.astype(np.int32)
        t = self.q_len
        return (np.repeat(ctx - t, t) + np.tile(np.arange(t, dtype=np.int32), self.batch)).astype(np.int32)

    @property
    def step_rows(self) -> np.ndarray:
        return np.repeat(self.seq_start, self.q_len) + self.step_pos.astype(np.int64)

    @property
    def batch(self):
        return self.spec.batch

    @property
    def max_blocks(self):
        return self.block_tables.shape[1]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.qk_head_dim or self.spec.head_dim)

    @property
    def new_rows(self) -> np.ndarray:
        return self.seq_start + self.context_lens.astype(np.int64) - 1

    @property
    def k_new(self) -> np.ndarray:
        return self.k[self.new_rows]

    @property
    def v_new(self) -> np.ndarray:
        return self.v[self.new_rows]

    def seq_k(self, b: int) -> np.ndarray:
        s = int(self.seq_start[b])
        return self.k[s:s + int(self.context_lens[b])]

    def seq_v(self, b: int) -> np.ndarray:
        s = int(self.seq_start[b])
        return self.v[s:s + int(self.context_lens[b])]

    @property
    def total_tokens(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    @property
    def elem_bytes(self) -> int:
        return 1 if self.spec.cache_dtype == "fp8_e4m3" else 2

    def unique_blocks(self) -> int:
        used = self.block_tables[self.block_tables >= 0]
        return int(np.unique(used).size)


def _assign_blocks(spec: Spec, ctx: np.ndarray):
    """Block tables: a seeded permutation of the pool handed out in (sequence, block) order.

    With prefix groups, logical block j of a group member is the group's shared
    block when j < prefix_blocks and the block is full and does not hold the
    slot appended this step (j < (ctx - 1) // block_size); any other block is
    private, which is what copy-on-write would have produced before a write.
    """
    bs = spec.block_size
    nb = (ctx.astype(np.int64) + bs - 1) // bs
    max_blocks = int(nb.max())
    # count the blocks in use
    owner = []                       # (kind, key) per table entry in allocation order
    shared_of = {}
    entries = []
    for b in range(spec.batch):
        row = []
        for j in range(int(nb[b])):
            is_shared = False
            if (spec.prefix_group and j < spec.prefix_tokens // bs
                    and j < (int(ctx[b]) - spec.q_len) // bs):
                is_shared = True
            if is_shared:
                key = (b // spec.prefix_group, j)
                if key not in shared_of:
                    shared_of[key] = len(owner)
                    owner.append(key)
                row.append((shared_of[key], True))
            else:
                row.append((len(owner), False))
                owner.append(("private", b, j))
        entries.append(row)
    in_use = len(owner)
    num_blocks = spec.pool_blocks or int(math.ceil(1.1 * in_use))
    if num_blocks < in_use:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {in_use} blocks")
    perm = _rng(spec.seed, 1).permutation(num_blocks).astype(np.int32)
    tables = np.full((spec.batch, max_blocks), -1, dtype=np.int32)
    shared = np.zeros((spec.batch, max_blocks), dtype=bool)
    for b, row in enumerate(entries):
        for j, (slot, is_shared) in enumerate(row):
            tables[b, j] = perm[slot]
            shared[b, j] = is_shared
    return tables, shared, num_blocks


def make(spec: Spec, threads: int | None = None) -> Workload:
    """Draw the whole workload (all K/V values, tables, queries)."""
    ctx = context_lengths(spec)
    if (ctx < spec.q_len).any():
        raise ValueError("every context must hold at least the tokens appended in the step")
    tables, shared, num_blocks = _assign_blocks(spec, ctx)
    B, Hq, Hkv, d = spec.batch, spec.q_heads, spec.kv_heads, spec.head_dim
    seq_start = np.zeros(B, dtype=np.int64)
    seq_start[1:] = np.cumsum(ctx.astype(np.int64))[:-1]
    total = int(ctx.astype(np.int64).sum())
    if spec.mla and (Hkv != 1 or spec.cache_dtype != "bf16" or spec.q_len != 1
                     or spec.prefix_group or not 0 < spec.latent_dim < d):
        raise ValueError("an MLA workload has one bf16 cached vector per token and one query")
    k = np.empty((total, Hkv, d), dtype=np.uint16)
    v = k if spec.mla else np.empty((total, Hkv, d), dtype=np.uint16)   # MLA: value = the vector

    # per (sequence, tensor, head) largest |bf16| bit pattern, for the fp8 scales
    amax_bits = np.zeros((B, 2, Hkv), dtype=np.uint16)

    def fill(job):
        b, which = job
        dst = k if which == 0 else v
        s, n = int(seq_start[b]), int(ctx[b])
        dst[s:s + n] = _normal_bf16((n, Hkv, d), spec.seed, 2, b, which)
        if spec.prefix_group:
            p = min(n, spec.prefix_tokens)
            g = b // spec.prefix_group
            dst[s:s + p] = _normal_bf16((spec.prefix_tokens, Hkv, d), spec.seed, 3, g, which)[:p]
        if spec.cache_dtype == "fp8_e4m3":
            # for non-NaN bf16, (bits & 0x7FFF) orders like the magnitude
            amax_bits[b, which] = (dst[s:s + n] & np.uint16(0x7FFF)).max(axis=(0, 2))

    nthreads = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(fill, [(b, which) for b in range(B) for which in ((0,) if spec.mla else (0, 1))]))

    q = _normal_bf16((B, Hq, d), spec.seed, 4)
    q_multi = _normal_bf16((B, Hq, spec.q_len, d), spec.seed, 5) if spec.q_len > 1 else None

    k_scale = v_scale = None
    if spec.cache_dtype == "fp8_e4m3":
        # Per-kv-head scale: the largest magnitude of that head's data maps to 448,
        # the largest finite e4m3 value.  This is input calibration, not the method.
        amax = bf16_bits_to_f32(amax_bits.max(axis=0))          # [2, Hkv]
        k_scale = (amax[0] / np.float32(448.0)).astype(np.float32)
        v_scale = (amax[1] / np.float32(448.0)).astype(np.float32)
    elif spec.cache_dtype != "bf16":
        raise ValueError(f"unknown cache dtype {spec.cache_dtype}")

    # tokens written before this step: positions 0 .. ctx-q_len-1; a shared block is written once
    seqs, poss, rows = [], [], []
    written = set()
    bs = spec.block_size
    for b in range(B):
        n = int(ctx[b]) - spec.q_len
        if n <= 0:
            continue
        p = np.arange(n, dtype=np.int64)
        keep = np.ones(n, dtype=bool)
        for j in range(int(((n + bs - 1) // bs))):
            if shared[b, j]:
                blk = int(tables[b, j])
                if blk in written:
                    keep[j * bs:(j + 1) * bs] = False
                else:
                    written.add(blk)
        p = p[keep]
        seqs.append(np.full(p.size, b, dtype=np.int32))
        poss.append(p.astype(np.int32))
        rows.append(seq_start[b] + p)
    cat = (lambda xs, dt: np.concatenate(xs).astype(dt) if xs else np.zeros(0, dtype=dt))
    return Workload(spec=spec, context_lens=ctx, block_tables=tables, num_blocks=num_blocks,
                    q=q, k=k, v=v, seq_start=seq_start, shared_block=shared,
                    k_scale=k_scale, v_scale=v_scale,
                    prefill_seq=cat(seqs, np.int32), prefill_pos=cat(poss, np.int32),
                    prefill_row=cat(rows, np.int64), q_multi=q_multi)
