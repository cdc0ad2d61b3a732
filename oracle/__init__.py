"""float64 CPU oracle for the paged-KV decode step (test infrastructure).

Only the tests, the smoke check and the bench's CPU-baseline / reference arm
may import this package.  The product path never does, and the two share no
code: this file marshals numpy arrays into ``kv_oracle.c`` and holds one numpy
function of its own, ``merge_states`` (the merge of attention results over
disjoint key sets).

The C source states each step with its source page and section.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kv_oracle.c")
LIB = os.path.join(HERE, "libkvoracle.so")

BF16 = 0
FP8_E4M3 = 1
_DTYPE = {"bf16": BF16, "fp8_e4m3": FP8_E4M3}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE semantics: no fast-math, no contraction)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-D_DEFAULT_SOURCE", "-fPIC", "-shared",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.kvo_bf16_value.argtypes = [ctypes.c_uint16]
            lib.kvo_bf16_value.restype = ctypes.c_double
            lib.kvo_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.kvo_e4m3_value.restype = ctypes.c_double
            lib.kvo_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.kvo_e4m3_from_float.restype = ctypes.c_uint8
            lib.kvo_e4m3_quantize.argtypes = [ctypes.c_uint16, ctypes.c_float]
            lib.kvo_e4m3_quantize.restype = ctypes.c_uint8
            lib.kvo_append.argtypes = [P, P, I, I, I, I, I, P, P, I, P, P, P, I, P, I, P, P]
            lib.kvo_append.restype = I
            lib.kvo_gather.argtypes = [P, I, I, I, I, I, P, I, P, P]
            lib.kvo_gather.restype = I
            lib.kvo_attend.argtypes = [P, I, I, I, P, P, I, ctypes.c_double, P, P]
            lib.kvo_attend.restype = None
            lib.kvo_attend_split.argtypes = [P, I, I, I, P, P, I, ctypes.c_double, I, I, P, P]
            lib.kvo_attend_split.restype = None
            lib.kvo_decode.argtypes = [P, I, I, I, I, P, P, P, P, I, P, P, ctypes.c_double,
                                       P, I, P, P, I]
            lib.kvo_decode.restype = I
            lib.kvo_decode_multi.argtypes = [P, I, I, I, I, I, P, P, P, P, I, P, P, ctypes.c_double,
                                             P, I, P, P]
            lib.kvo_decode_multi.restype = I
            lib.kvo_mla_attend.argtypes = [P, I, I, I, P, I, ctypes.c_double, P, P]
            lib.kvo_mla_attend.restype = None
            lib.kvo_mla_decode.argtypes = [P, I, I, I, I, P, P, P, ctypes.c_double, P, I, P, P]
            lib.kvo_mla_decode.restype = I
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- formats
def bf16_value(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.kvo_bf16_value(int(x)) for x in b.ravel()]).reshape(b.shape)


def e4m3_value(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.kvo_e4m3_value(int(x)) for x in c.ravel()]).reshape(c.shape)


def e4m3_from_float(x) -> np.ndarray:
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.kvo_e4m3_from_float(float(v)) for v in a.ravel()],
                    dtype=np.uint8).reshape(a.shape)


def e4m3_quantize(bits, scale: float) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    s = float(np.float32(scale))
    return np.array([lib.kvo_e4m3_quantize(int(x), s) for x in b.ravel()],
                    dtype=np.uint8).reshape(b.shape)


# ---------------------------------------------------------------- append / gather
def append(k_pool: np.ndarray, v_pool: np.ndarray, cache_dtype: str, block_size: int,
           k_new, v_new, block_tables, context_lens, token_seq=None, token_pos=None,
           k_scale=None, v_scale=None) -> int:
    """Write new tokens into the pool images in place; returns the count of skipped tokens.

    k_pool / v_pool: uint8 arrays of the raw pool bytes, [num_blocks, bs, Hkv, d * elem].
    """
    lib = _load()
    num_blocks, bs, hkv = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    assert bs == block_size
    eb = 1 if cache_dtype == "fp8_e4m3" else 2
    d = k_pool.shape[3] // eb
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous and k_pool.dtype == np.uint8
    kn = _c(k_new, np.uint16).reshape(-1, hkv, d)
    vn = _c(v_new, np.uint16).reshape(-1, hkv, d)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    ts = _c(token_seq, np.int32)
    tp = _c(token_pos, np.int32)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    return lib.kvo_append(_ptr(k_pool), _ptr(v_pool), _DTYPE[cache_dtype], num_blocks, bs, hkv, d,
                          _ptr(kn), _ptr(vn), kn.shape[0], _ptr(ts), _ptr(tp), _ptr(bt),
                          bt.shape[1], _ptr(cl), cl.shape[0], _ptr(ks), _ptr(vs))


def gather(pool: np.ndarray, cache_dtype: str, table_row, ctx: int, scale=None) -> np.ndarray:
    """Contiguous float64 [ctx, Hkv, d] copy of one sequence read through its table."""
    lib = _load()
    num_blocks, bs, hkv = pool.shape[0], pool.shape[1], pool.shape[2]
    eb = 1 if cache_dtype == "fp8_e4m3" else 2
    d = pool.shape[3] // eb
    out = np.zeros((ctx, hkv, d), dtype=np.float64)
    tr = _c(table_row, np.int32)
    sc = _c(scale, np.float32)
    rc = lib.kvo_gather(_ptr(np.ascontiguousarray(pool)), _DTYPE[cache_dtype], num_blocks, bs, hkv,
                        d, _ptr(tr), ctx, _ptr(sc), _ptr(out))
    if rc != 0:
        raise ValueError("block table entry outside the pool")
    return out


# ---------------------------------------------------------------- attention
def attend(q, k, v, scale: float):
    """q [Hq, d], k/v [ctx, Hkv, d] float64 -> (out [Hq, d], lse [Hq])."""
    lib = _load()
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    hq, d = q.shape
    ctx, hkv = k.shape[0], k.shape[1]
    out = np.zeros((hq, d), dtype=np.float64)
    lse = np.zeros(hq, dtype=np.float64)
    lib.kvo_attend(_ptr(q), hq, hkv, d, _ptr(k), _ptr(v), ctx, float(scale), _ptr(out), _ptr(lse))
    return out, lse


def attend_split(q, k, v, scale: float, split_tokens: int, num_chunks: int | None = None):
    lib = _load()
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    hq, d = q.shape
    ctx, hkv = k.shape[0], k.shape[1]
    if num_chunks is None:
        num_chunks = max(1, -(-ctx // split_tokens))
    out = np.zeros((hq, d), dtype=np.float64)
    lse = np.zeros(hq, dtype=np.float64)
    lib.kvo_attend_split(_ptr(q), hq, hkv, d, _ptr(k), _ptr(v), ctx, float(scale), split_tokens,
                         num_chunks, _ptr(out), _ptr(lse))
    return out, lse


def merge_states(outs, lses):
    """Attention over the union of disjoint key sets from the attention over each set.

    outs [n, rows, d] (normalised outputs), lses [n, rows] (natural-log log-sum-exp of the
    scaled scores; -inf for a set with no key) -> (out [rows, d], lse [rows]).  Written out
    from the split-KV merge (learn.mohebi.ai lesson 12, section 6: split-KV decoding), with
    each set's (max, sum) pair folded into lse = max + log(sum):
        LSE = log sum_r exp(lse_r),   out = sum_r exp(lse_r - LSE) out_r.
    Sets with no key are left out; a row with none gets out = 0, lse = -inf."""
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    n, rows, d = outs.shape
    out = np.zeros((rows, d), dtype=np.float64)
    lse = np.full(rows, -np.inf)
    for i in range(rows):
        used = [r for r in range(n) if lses[r, i] > -np.inf]
        if not used:
            continue
        m = max(lses[r, i] for r in used)
        w = {r: np.exp(lses[r, i] - m) for r in used}
        total = sum(w.values())
        for r in used:
            out[i] += w[r] * outs[r, i]
        out[i] /= total
        lse[i] = m + np.log(total)
    return out, lse


def decode(q, k, v, seq_start, context_lens, *, q_heads: int, kv_heads: int, head_dim: int,
           scale: float, cache_dtype: str = "bf16", k_scale=None, v_scale=None,
           seqs=None, threads: int = 1):
    """Decode attention for a batch kept contiguously per sequence.

    q: uint16 bf16 [B, Hq, d]; k, v: uint16 bf16 [T_total, Hkv, d]; sequence b at rows
    seq_start[b] .. seq_start[b] + ctx[b] - 1.  With cache_dtype "fp8_e4m3" the oracle
    quantises the values with its own e4m3 encoder and attends over code * scale.
    Returns (out float64 [n, Hq, d], lse float64 [n, Hq]) for the listed sequences.
    """
    lib = _load()
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    ss = _c(seq_start, np.int64)
    cl = _c(context_lens, np.int32)
    batch = cl.shape[0]
    sl = None if seqs is None else _c(seqs, np.int32)
    n = batch if sl is None else sl.shape[0]
    out = np.zeros((n, q_heads, head_dim), dtype=np.float64)
    lse = np.zeros((n, q_heads), dtype=np.float64)
    rc = lib.kvo_decode(_ptr(q), batch, q_heads, kv_heads, head_dim, _ptr(k), _ptr(v), _ptr(ss),
                        _ptr(cl), _DTYPE[cache_dtype], _ptr(_c(k_scale, np.float32)),
                        _ptr(_c(v_scale, np.float32)), float(scale), _ptr(sl), n, _ptr(out),
                        _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("q_heads must be a multiple of kv_heads")
    return out, lse


def decode_workload(w, seqs=None, threads: int = 1, cache_dtype: str | None = None):
    """Oracle decode of a ``workloads.Workload`` (optionally a subset of sequences)."""
    s = w.spec
    return decode(w.q, w.k, w.v, w.seq_start, w.context_lens, q_heads=s.q_heads,
                  kv_heads=s.kv_heads, head_dim=s.head_dim, scale=w.scale,
                  cache_dtype=cache_dtype or s.cache_dtype, k_scale=w.k_scale,
                  v_scale=w.v_scale, seqs=seqs, threads=threads)


def pool_image(w, after_step: bool, threads: int = 1) -> tuple[np.ndarray, np.ndarray]:
    """Expected raw bytes of the K and V pools of a workload.

    Poisoned with 0xFF, then every prefilled token written; with after_step the
    token appended in this step as well.  Shape [num_blocks, bs, Hkv, d * elem].
    threads > 1 writes disjoint sets of tokens in concurrent calls of the C routine:
    every token has its own slot, so the image is the same whatever the order.
    """
    s = w.spec
    eb = w.elem_bytes
    shape = (w.num_blocks, s.block_size, s.kv_heads, s.head_dim * eb)
    kp = np.full(shape, 0xFF, dtype=np.uint8)
    vp = np.full(shape, 0xFF, dtype=np.uint8)

    def write(rows, seq, pos):
        n = rows.size
        parts = max(1, min(threads, n // 4096))
        cuts = [(i * n // parts, (i + 1) * n // parts) for i in range(parts)]

        def one(c):
            a, b = c
            return append(kp, vp, s.cache_dtype, s.block_size, w.k[rows[a:b]], w.v[rows[a:b]],
                          w.block_tables, w.context_lens, token_seq=seq[a:b], token_pos=pos[a:b],
                          k_scale=w.k_scale, v_scale=w.v_scale)

        if parts == 1:
            bad = one(cuts[0])
        else:
            from concurrent.futures import ThreadPoolExecutor
            with ThreadPoolExecutor(parts) as ex:
                bad = sum(ex.map(one, cuts))
        assert bad == 0

    if w.prefill_seq.size:
        write(w.prefill_row, w.prefill_seq, w.prefill_pos)
    if after_step:
        write(np.asarray(w.step_rows), np.asarray(w.step_seq), np.asarray(w.step_pos))
    return kp, vp


def decode_multi(q, k, v, seq_start, context_lens, *, q_heads: int, q_len: int, kv_heads: int,
                 head_dim: int, scale: float, cache_dtype: str = "bf16", k_scale=None,
                 v_scale=None, seqs=None):
    """Attention of q_len new tokens per sequence (causal among themselves).

    q: uint16 bf16 [B, Hq, q_len, d]; the last q_len cached tokens of each sequence are the
    new ones.  Returns (out float64 [n, Hq, q_len, d], lse float64 [n, Hq, q_len]).
    """
    lib = _load()
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    ss = _c(seq_start, np.int64)
    cl = _c(context_lens, np.int32)
    batch = cl.shape[0]
    sl = None if seqs is None else _c(seqs, np.int32)
    n = batch if sl is None else sl.shape[0]
    out = np.zeros((n, q_heads, q_len, head_dim), dtype=np.float64)
    lse = np.zeros((n, q_heads, q_len), dtype=np.float64)
    rc = lib.kvo_decode_multi(_ptr(q), batch, q_heads, q_len, kv_heads, head_dim, _ptr(k), _ptr(v),
                              _ptr(ss), _ptr(cl), _DTYPE[cache_dtype],
                              _ptr(_c(k_scale, np.float32)), _ptr(_c(v_scale, np.float32)),
                              float(scale), _ptr(sl), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("bad multi-query arguments")
    return out, lse


def decode_multi_workload(w, q_multi, q_len: int, seqs=None, cache_dtype: str | None = None,
                          threads: int = 1):
    """Oracle attention of q_len new tokens per sequence of a workload (q_multi [B, Hq, q_len, d]).

    threads > 1 runs disjoint sets of sequences in concurrent calls of the C routine
    (ctypes releases the interpreter lock); each sequence's arithmetic is unchanged."""
    s = w.spec
    seq_list = list(range(w.batch)) if seqs is None else [int(b) for b in seqs]

    def run(part):
        return decode_multi(q_multi, w.k, w.v, w.seq_start, w.context_lens, q_heads=s.q_heads,
                            q_len=q_len, kv_heads=s.kv_heads, head_dim=s.head_dim, scale=w.scale,
                            cache_dtype=cache_dtype or s.cache_dtype, k_scale=w.k_scale,
                            v_scale=w.v_scale, seqs=part)

    if threads <= 1 or len(seq_list) <= 1:
        return run(seq_list)
    from concurrent.futures import ThreadPoolExecutor
    parts = [seq_list[i::threads] for i in range(min(threads, len(seq_list)))]
    with ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(run, parts))
    out = np.zeros((len(seq_list), s.q_heads, q_len, s.head_dim), dtype=np.float64)
    lse = np.zeros((len(seq_list), s.q_heads, q_len), dtype=np.float64)
    for i, (o, l) in enumerate(res):
        out[i::len(parts)] = o
        lse[i::len(parts)] = l
    return out, lse


def mla_attend(q, cache, latent_dim: int, scale: float):
    """Absorbed multi-head latent attention for one sequence, float64.

    q [Hq, dl + dr] (queries already folded through W_UK, rotary part last), cache
    [ctx, dl + dr] (latent then rotary key).  Returns (out [Hq, dl], lse [Hq])."""
    lib = _load()
    q = _c(q, np.float64)
    cache = _c(cache, np.float64)
    hq, dk = q.shape
    ctx = cache.shape[0]
    assert cache.shape[1] == dk and 0 < latent_dim <= dk
    out = np.zeros((hq, latent_dim), dtype=np.float64)
    lse = np.zeros(hq, dtype=np.float64)
    lib.kvo_mla_attend(_ptr(q), hq, latent_dim, dk - latent_dim, _ptr(cache), ctx, float(scale),
                       _ptr(out), _ptr(lse))
    return out, lse


def mla_decode(q, cache, seq_start, context_lens, *, latent_dim: int, scale: float, seqs=None):
    """Absorbed MLA decode of a batch: q uint16 bf16 [B, Hq, dl + dr], cache uint16 bf16
    [T_total, dl + dr] contiguous per sequence.  Returns (out [n, Hq, dl], lse [n, Hq])."""
    lib = _load()
    q = _c(q, np.uint16)
    cache = _c(cache, np.uint16)
    ss = _c(seq_start, np.int64)
    cl = _c(context_lens, np.int32)
    batch, hq, dk = q.shape
    sl = None if seqs is None else _c(seqs, np.int32)
    n = batch if sl is None else sl.shape[0]
    out = np.zeros((n, hq, latent_dim), dtype=np.float64)
    lse = np.zeros((n, hq), dtype=np.float64)
    rc = lib.kvo_mla_decode(_ptr(q), batch, hq, latent_dim, dk - latent_dim, _ptr(cache), _ptr(ss),
                            _ptr(cl), float(scale), _ptr(sl), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("bad MLA arguments")
    return out, lse


def mla_decode_workload(w, seqs=None, threads: int = 1):
    """Oracle absorbed-MLA decode of a workload whose cache holds one vector per token.

    threads > 1 runs disjoint sets of sequences in concurrent calls of the C routine
    (ctypes releases the interpreter lock); each sequence's arithmetic is unchanged."""
    s = w.spec
    seq_list = list(range(w.batch)) if seqs is None else [int(b) for b in seqs]

    def run(part):
        return mla_decode(w.q, w.k[:, 0, :], w.seq_start, w.context_lens, latent_dim=s.latent_dim,
                          scale=w.scale, seqs=part)

    if threads <= 1 or len(seq_list) <= 1:
        return run(seq_list)
    from concurrent.futures import ThreadPoolExecutor
    parts = [seq_list[i::threads] for i in range(min(threads, len(seq_list)))]
    with ThreadPoolExecutor(len(parts)) as ex:
        res = list(ex.map(run, parts))
    out = np.zeros((len(seq_list), s.q_heads, s.latent_dim), dtype=np.float64)
    lse = np.zeros((len(seq_list), s.q_heads), dtype=np.float64)
    for i, (o, l) in enumerate(res):
        out[i::len(parts)] = o
        lse[i::len(parts)] = l
    return out, lse
