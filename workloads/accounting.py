"""Algorithmic byte and FLOP counts of the decode step (for throughput and roofline).

The counts are the minimum traffic the step needs, from the definitions:
every cached K and V element of the tokens 0 .. ctx-1 of each sequence read
once, q read, the output written, the block-table entries and context lengths
read, and the split-KV partials written and read back.  Bytes per token of
cache follow k = 2 * layers * kv_heads * head_dim * bytes_per_value
(learn.mohebi.ai lesson 12, section 3 "KV-cache memory"; xuewyang.github.io/
posts/kv, "How big is the cache?"), with one layer per pool here.
FLOPs follow the decode-step proposition of the same lesson (proof, step 3):
2 C d_h for the scores and 2 C d_h for the weighted values, per query head.
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_value: int) -> int:
    return 2 * layers * kv_heads * head_dim * bytes_per_value


def mla_numbers_per_token(latent_dim: int, rope_dim: int) -> int:
    """Numbers an MLA cache keeps per token and layer: the latent plus the rotary key."""
    return latent_dim + rope_dim


def mla_bytes_per_token(latent_dim: int, rope_dim: int, bytes_per_value: int) -> int:
    return mla_numbers_per_token(latent_dim, rope_dim) * bytes_per_value


def _nb(w):
    bs = w.spec.block_size
    return (w.context_lens.astype(np.int64) + bs - 1) // bs


def unique_kv_tokens(w) -> int:
    """Cached tokens counting each physically shared block once."""
    s = w.spec
    total = int(w.context_lens.astype(np.int64).sum())
    if not w.shared_block.any():
        return total
    shared_entries = int(w.shared_block.sum())
    shared_ids = np.unique(w.block_tables[w.shared_block])
    return total - shared_entries * s.block_size + int(shared_ids.size) * s.block_size


def decode_bytes(w, split_tokens: int) -> dict:
    """Algorithmic bytes of one paged_decode_attention call with chunks of split_tokens."""
    s = w.spec
    e = w.elem_bytes
    ctx = w.context_lens.astype(np.int64)
    nb = _nb(w)
    row = 2 * s.kv_heads * s.head_dim * e                      # K and V of one token
    kv_logical = int(ctx.sum()) * row
    kv_unique = unique_kv_tokens(w) * row
    # Each K/V element counts once, whatever the kernel does: a kernel that tiles a GQA
    # group's query rows and reads a block once per tile shows the extra reads as DRAM
    # traffic above these bytes, not as work of the method.
    rows = s.q_heads * s.q_len                                  # query rows per sequence
    qo = 2 * w.batch * rows * s.head_dim * 2                    # q read + out written (bf16)
    meta = 4 * int(nb.sum()) + 4 * w.batch + 4 * w.batch * rows  # tables, ctx, lse
    sb = max(1, split_tokens // s.block_size)
    nsplit = np.maximum(1, (nb + sb - 1) // sb)
    multi = nsplit > 1
    partial = int((nsplit[multi] * rows).sum()) * (s.head_dim + 2) * 4 * 2
    scales = 2 * 4 * s.kv_heads if s.cache_dtype == "fp8_e4m3" else 0
    other = qo + meta + partial + scales
    return {"kv_logical": kv_logical, "kv_unique": kv_unique, "other": other,
            "total": kv_logical + other, "total_unique": kv_unique + other,
            "partials": partial}


def append_bytes(w) -> int:
    """Algorithmic bytes of one paged_kv_append of the step's new tokens."""
    s = w.spec
    n = w.batch * s.q_len * s.kv_heads * s.head_dim
    return 2 * n * 2 + 2 * n * w.elem_bytes + 8 * w.batch * s.q_len


def decode_flops(w) -> int:
    s = w.spec
    return int(4 * w.context_lens.astype(np.int64).sum() * s.head_dim * s.q_heads * s.q_len)


# Positions the tensor-core MLA partition puts before each sequence's blocks (the cost of
# starting a segment, in blocks): the wide form's and the narrow form's.
MLA_SEG_PAD_WIDE = 4
MLA_SEG_PAD_NARROW = 2


def mla_tc_pieces(w, split_blocks: int, grid: int, head_tile: int = 128, halves: int = 2,
                  pad: int | None = None) -> np.ndarray:
    """Pieces each (outer, sequence) is cut into by a tensor-core MLA decode's partition:
    its positions (outer, sequence, position) -- outer = (latent half, head tile) for the
    wide form (tiles of 128 heads, two halves), the head tile for the narrow one (tiles of
    16, halves=1); a sequence with nb blocks has pad + nb positions, the pad first (none
    when empty) -- T in all, are cut into G = min(grid, T // split_blocks) (at least 1)
    equal contiguous ranges, range c = [c T / G, (c + 1) T / G); a sequence is cut at every
    range boundary among its blocks.  Same integer arithmetic as the kernels."""
    if pad is None:
        pad = MLA_SEG_PAD_WIDE if halves == 2 else MLA_SEG_PAD_NARROW
    nb = _nb(w)
    tiles = -(-w.spec.q_heads // head_tile)
    wv = np.where(nb > 0, nb + pad, 0).astype(np.int64)
    S = int(wv.sum())
    T = S * tiles * halves
    if T == 0:
        return np.zeros(0, dtype=np.int64)
    g = max(1, min(grid, T // max(1, split_blocks)))
    pre = np.concatenate([[0], np.cumsum(wv)[:-1]]).astype(np.int64)
    out = []
    for outer in range(tiles * halves):
        ub = outer * S + pre + pad                # position of each sequence's block 0
        for u, n in zip(ub, nb):
            if n == 0:
                continue
            first = ((u + 1) * g - 1) // T
            last = ((u + n) * g - 1) // T
            out.append(last - first + 1)
    return np.array(out, dtype=np.int64)


def mla_decode_bytes(w, split_tokens: int, head_tile: int = 16, tc_grid: int = 0,
                     form: str = "wide") -> dict:
    """Algorithmic bytes of one paged_mla_decode_attention call: every cached vector once
    (kv), the absorbed queries, the latent outputs, tables, lengths, LSE and the split
    partials.  l2_reads: vector bytes read by all head tiles (each tile reads the
    sequence's vectors; the copies after the first come from L2).

    tc_grid > 0: a tensor-core form with that many CTAs and pieces from mla_tc_pieces --
    form "wide": tiles of 128 heads, two latent halves each reading every vector, each
    piece of a cut sequence writing (and the merge reading) 128 heads x 256 fp16 numbers
    and an fp32 (max, sum) pair per head; form "narrow": tiles of 16 heads, 16 x 512 fp16
    numbers and 16 pairs per piece."""
    s = w.spec
    ctx = w.context_lens.astype(np.int64)
    nb = _nb(w)
    kv = int(ctx.sum()) * s.head_dim * 2
    rows = w.batch * s.q_heads
    qo = rows * (s.head_dim + s.latent_dim) * 2
    meta = 4 * int(nb.sum()) + 4 * w.batch + 4 * rows
    if tc_grid > 0 and form == "wide":
        tiles = -(-s.q_heads // 128) * 2
        pieces = mla_tc_pieces(w, max(1, split_tokens // s.block_size), tc_grid)
        partial = int(pieces[pieces > 1].sum()) * 128 * ((s.latent_dim // 2) * 2 + 8) * 2
    elif tc_grid > 0:
        tiles = -(-s.q_heads // 16)
        pieces = mla_tc_pieces(w, max(1, split_tokens // s.block_size), tc_grid, 16, 1)
        partial = int(pieces[pieces > 1].sum()) * 16 * (s.latent_dim * 2 + 8) * 2
    else:
        tiles = -(-s.q_heads // head_tile)
        sb = max(1, split_tokens // s.block_size)
        nsplit = np.maximum(1, (nb + sb - 1) // sb)
        multi = nsplit > 1
        partial = int(nsplit[multi].sum()) * s.q_heads * (s.latent_dim + 2) * 4 * 2
    other = qo + meta + partial
    return {"kv_logical": kv, "kv_unique": kv, "other": other, "total": kv + other,
            "total_unique": kv + other, "partials": partial, "l2_reads": kv * tiles}


def mla_append_bytes(w) -> int:
    n = w.batch * w.spec.head_dim
    return 2 * n * 2 + 8 * w.batch


def mla_decode_flops(w) -> int:
    """2 flops per multiply-add: scores over head_dim numbers, values over latent_dim."""
    s = w.spec
    return int(2 * w.context_lens.astype(np.int64).sum() * (s.head_dim + s.latent_dim) * s.q_heads)
