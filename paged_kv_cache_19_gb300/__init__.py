"""Paged KV cache for the decode step on GB300: Python binding of libkvpaged.so.

The functions mirror the C ABI in include/kv_paged.h, include/kv_mla.h and
include/kv_block_manager.h one to one and only
marshal arguments (torch tensors -> device pointers, the current stream).
Every step of the computation runs in the library's CUDA kernels; there is no
CPU path, and importing a function without the built library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "KVError", "Pool", "kv_pool_create", "kv_pool_destroy", "paged_kv_append", "paged_decode_plan",
    "paged_decode_cta_heads", "kv_debug_decode_stall",
    "paged_decode_workspace_size", "paged_decode_attention", "paged_decode_attention_split_merge",
    "paged_merge_attention_states",
    "paged_attention_multi_query",
    "paged_decode_step",
    "paged_multi_query_workspace_size", "library_path", "load_library", "BlockManager",
    "kv_copy_blocks", "BM_FIFO", "BM_LIFO", "BM_PREFIX_CACHING", "kv_mla_pool_create",
    "paged_mla_decode_plan", "paged_mla_workspace_size", "paged_mla_decode_attention",
    "paged_mla_decode_step",
    "DEVERR_BLOCK_ID", "DEVERR_CONTEXT", "DEVERR_SEQ", "DEVERR_POSITION", "DEVERR_TIMEOUT",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkvpaged.so")

KV_OK = 0
KV_ERR_INVALID_ARG = 1
KV_ERR_OUT_OF_MEMORY = 2
KV_ERR_OUT_OF_BLOCKS = 3
KV_ERR_UNSUPPORTED = 4
KV_ERR_CUDA = 5
KV_ERR_DEVICE_CHECK = 6
DEVERR_BLOCK_ID = 0x1
DEVERR_CONTEXT = 0x2
DEVERR_SEQ = 0x4
DEVERR_POSITION = 0x8
DEVERR_TIMEOUT = 0x10
_DTYPES = {"bf16": 0, "fp8_e4m3": 1}
BM_FIFO = 0x0
BM_LIFO = 0x1
BM_PREFIX_CACHING = 0x2

_lock = threading.Lock()
_lib = None


class _BlockCopy(ctypes.Structure):
    _fields_ = [("src", ctypes.c_int32), ("dst", ctypes.c_int32)]


class KVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib.kv_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {msg} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libkvpaged.so (built by __graft_entry__.build()); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, S, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int64
        sig = {
            "kv_abi_version": ([], I),
            "kv_status_string": ([I], ctypes.c_char_p),
            "kv_pool_create": ([I, I, I, I, I, I, ctypes.POINTER(P)], I),
            "kv_pool_destroy": ([P], I),
            "kv_pool_tensors": ([P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P),
                                 ctypes.POINTER(P)], I),
            "kv_pool_shape": ([P] + [ctypes.POINTER(I)] * 6, I),
            "kv_pool_set_scales": ([P, P, P], I),
            "kv_pool_device_errors": ([P, ctypes.POINTER(ctypes.c_uint32), I], I),
            "paged_kv_append": ([P, P, P, I, P, P, P, I, P, I, P], I),
            "paged_decode_plan": ([P, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "paged_decode_cta_heads": ([P, I, I, I, I, I, ctypes.POINTER(I)], I),
            "kv_debug_decode_stall": ([I, ctypes.c_ulonglong], I),
            "paged_decode_workspace_size": ([P, I, I, I, I, ctypes.POINTER(S)], I),
            "paged_decode_attention": ([P, P, I, P, I, P, I, ctypes.c_float, I, P, S, P, P, P], I),
            "paged_merge_attention_states": ([P, P, I, L, I, P, P, P], I),
            "paged_decode_attention_split_merge": ([P, P, I, P, I, P, I, ctypes.c_float, I, P, S, P,
                                                    P, P], I),
            "paged_attention_multi_query": ([P, P, I, I, P, I, P, I, ctypes.c_float, I, P, S, P, P,
                                             P], I),
            "paged_multi_query_workspace_size": ([P, I, I, I, I, I, ctypes.POINTER(S)], I),
            "paged_decode_step": ([P, P, P, P, I, I, P, I, P, I, ctypes.c_float, I, P, S, P, P, P],
                                  I),
            "kv_bm_create": ([I, I, I, ctypes.POINTER(P)], I),
            "kv_bm_destroy": ([P], I),
            "kv_bm_add_sequence": ([P, L, ctypes.c_uint64], I),
            "kv_bm_fork": ([P, L, L], I),
            "kv_bm_append_slots": ([P, L, I, P, ctypes.POINTER(_BlockCopy), ctypes.POINTER(I)], I),
            "kv_bm_match_prefix": ([P, L, P, I, ctypes.POINTER(I)], I),
            "kv_bm_free_sequence": ([P, L], I),
            "kv_bm_num_free_blocks": ([P, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "kv_bm_sequence_info": ([P, L, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "kv_bm_block_refcount": ([P, ctypes.c_int32, ctypes.POINTER(I)], I),
            "kv_bm_build_tables": ([P, P, I, I, P, P], I),
            "kv_copy_blocks": ([P, P, I, P], I),
            "kv_mla_pool_create": ([I, I, I, I, I, ctypes.POINTER(P)], I),
            "paged_mla_decode_plan": ([P, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)], I),
            "paged_mla_workspace_size": ([P, I, I, I, I, ctypes.POINTER(S)], I),
            "paged_mla_decode_attention": ([P, P, I, P, I, P, I, ctypes.c_float, I, P, S, P, P,
                                            P], I),
            "paged_mla_decode_step": ([P, P, P, I, P, I, P, I, ctypes.c_float, I, P, S, P, P, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int, what: str):
    if status != KV_OK:
        raise KVError(status, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t, dtype, name):
    if t is None:
        return None
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}, got "
                         f"{t.dtype} on {t.device} (contiguous={t.is_contiguous()})")
    return t


class _CudaBytes:
    """Exposes a device byte range to torch through __cuda_array_interface__."""

    def __init__(self, ptr: int, shape):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3, "strides": None}


class Pool:
    """One layer's paged K/V pool (owned by the library)."""

    def __init__(self, handle: int, num_blocks, block_size, kv_heads, head_dim, dtype, device,
                 latent: bool = False):
        self._h = ctypes.c_void_p(handle)
        self.num_blocks, self.block_size = num_blocks, block_size
        self.kv_heads, self.head_dim = kv_heads, head_dim
        self.dtype, self.device = dtype, device
        self.elem_bytes = 1 if dtype == "fp8_e4m3" else 2
        self.latent = latent            # MLA latent pool: one cached vector per token, no V

    @property
    def handle(self):
        if not self._h:
            raise RuntimeError("pool was destroyed")
        return self._h

    def tensors(self):
        """Torch views (no copy) of the pool: K, V as raw bytes [num_blocks, bs, Hkv, d*elem]
        viewed as bf16 or float8_e4m3fn (V is None for a latent pool), and the float32
        scales [Hkv]."""
        lib = load_library()
        k, v, ks, vs = (ctypes.c_void_p() for _ in range(4))
        _check(lib.kv_pool_tensors(self.handle, ctypes.byref(k), ctypes.byref(v), ctypes.byref(ks),
                                   ctypes.byref(vs)), "kv_pool_tensors")
        dev = torch.device("cuda", self.device)
        shape = (self.num_blocks, self.block_size, self.kv_heads, self.head_dim * self.elem_bytes)
        kt = torch.as_tensor(_CudaBytes(k.value, shape), device=dev)
        vt = torch.as_tensor(_CudaBytes(v.value, shape), device=dev) if v.value else None
        st = torch.as_tensor(_CudaBytes(ks.value, (self.kv_heads * 4,)), device=dev).view(torch.float32)
        sv = torch.as_tensor(_CudaBytes(vs.value, (self.kv_heads * 4,)), device=dev).view(torch.float32)
        cache = torch.float8_e4m3fn if self.dtype == "fp8_e4m3" else torch.bfloat16
        return kt.view(cache), None if vt is None else vt.view(cache), st, sv

    def raw_bytes(self):
        """K and V pools as uint8 views [num_blocks, bs, Hkv, d*elem] (V None if latent)."""
        k, v, _, _ = self.tensors()
        return k.view(torch.uint8), None if v is None else v.view(torch.uint8)

    def set_scales(self, k_scale=None, v_scale=None):
        lib = load_library()
        arr = lambda s: None if s is None else (ctypes.c_float * self.kv_heads)(*[float(x) for x in s])
        _check(lib.kv_pool_set_scales(self.handle, arr(k_scale), arr(v_scale)), "kv_pool_set_scales")

    def device_errors(self, clear: bool = True) -> int:
        lib = load_library()
        bits = ctypes.c_uint32(0)
        st = lib.kv_pool_device_errors(self.handle, ctypes.byref(bits), int(clear))
        if st not in (KV_OK, KV_ERR_DEVICE_CHECK):
            _check(st, "kv_pool_device_errors")
        return bits.value

    def destroy(self):
        if self._h:
            _check(load_library().kv_pool_destroy(self._h), "kv_pool_destroy")
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            if self._h and _lib is not None:
                _lib.kv_pool_destroy(self._h)
                self._h = ctypes.c_void_p(None)
        except Exception:
            pass


def kv_pool_create(num_blocks: int, block_size: int, kv_heads: int, head_dim: int,
                   dtype: str = "bf16", device: int | None = None) -> Pool:
    lib = load_library()
    if device is None:
        device = torch.cuda.current_device()
    h = ctypes.c_void_p()
    _check(lib.kv_pool_create(int(num_blocks), int(block_size), int(kv_heads), int(head_dim),
                              _DTYPES[dtype], int(device), ctypes.byref(h)), "kv_pool_create")
    return Pool(h.value, num_blocks, block_size, kv_heads, head_dim, dtype, device)


def kv_pool_destroy(pool: Pool):
    pool.destroy()


def paged_kv_append(pool: Pool, k_new, v_new, block_tables, context_lens=None, token_seq=None,
                    token_pos=None, stream=None):
    """Write the key/value rows [T, Hkv, d] (bf16) of T tokens into the pool."""
    lib = load_library()
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")          # None for a latent pool
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    _need(token_seq, torch.int32, "token_seq")
    _need(token_pos, torch.int32, "token_pos")
    batch, max_blocks = block_tables.shape
    n = k_new.shape[0]
    _check(lib.paged_kv_append(pool.handle, _ptr(k_new), _ptr(v_new), int(n), _ptr(token_seq),
                               _ptr(token_pos), _ptr(block_tables), int(max_blocks),
                               _ptr(context_lens), int(batch), _stream(stream)), "paged_kv_append")


def paged_decode_plan(pool: Pool, batch: int, q_heads: int, max_blocks: int,
                      kv_split_tokens: int = 0):
    lib = load_library()
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(lib.paged_decode_plan(pool.handle, int(batch), int(q_heads), int(max_blocks),
                                 int(kv_split_tokens), ctypes.byref(a), ctypes.byref(b)),
           "paged_decode_plan")
    return a.value, b.value


def kv_debug_decode_stall(stop_stage: int = -1, consumer_wait_ns: int = 0) -> None:
    """Failure-path test hook (see include/kv_paged.h); (-1, 0) restores normal operation."""
    lib = load_library()
    _check(lib.kv_debug_decode_stall(int(stop_stage), int(consumer_wait_ns)),
           "kv_debug_decode_stall")


def paged_decode_cta_heads(pool: Pool, batch: int, q_heads: int, q_len: int, max_blocks: int,
                           kv_split_tokens: int = 0) -> int:
    """kv heads one CTA of the decode covers for these sizes (1, 2 or 4)."""
    lib = load_library()
    n = ctypes.c_int()
    _check(lib.paged_decode_cta_heads(pool.handle, int(batch), int(q_heads), int(q_len),
                                      int(max_blocks), int(kv_split_tokens), ctypes.byref(n)),
           "paged_decode_cta_heads")
    return n.value


def paged_decode_workspace_size(pool: Pool, batch: int, q_heads: int, max_blocks: int,
                                kv_split_tokens: int = 0) -> int:
    lib = load_library()
    n = ctypes.c_size_t()
    _check(lib.paged_decode_workspace_size(pool.handle, int(batch), int(q_heads), int(max_blocks),
                                           int(kv_split_tokens), ctypes.byref(n)),
           "paged_decode_workspace_size")
    return n.value


def paged_decode_attention(pool: Pool, q, block_tables, context_lens, scale: float,
                           kv_split_tokens: int = 0, workspace=None, out=None, lse=None,
                           stream=None):
    """Decode attention; q bf16 [B, Hq, 1, d] or [B, Hq, d].  Returns out (shape of q)."""
    lib = load_library()
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    batch, q_heads = q.shape[0], q.shape[1]
    d = q.shape[-1]
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        need = paged_decode_workspace_size(pool, batch, q_heads, max_blocks, kv_split_tokens)
        # zero-filled: it holds the per-sequence chunk counters of the in-kernel merge
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device) if need else None
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(lib.paged_decode_attention(pool.handle, _ptr(q), int(q_heads), _ptr(block_tables),
                                      int(max_blocks), _ptr(context_lens), int(batch),
                                      float(scale), int(kv_split_tokens), _ptr(workspace),
                                      int(ws_bytes), _ptr(out), _ptr(lse), _stream(stream)),
           "paged_decode_attention")
    return out


def paged_decode_attention_split_merge(pool: Pool, q, block_tables, context_lens,
                                       scale: float, kv_split_tokens: int = 0,
                                       workspace=None, out=None, lse=None, stream=None):
    """paged_decode_attention as two kernels: the split-KV grid, then a separate
    log-sum-exp merge kernel (same bits).  Returns out (shape of q)."""
    lib = load_library()
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    batch, q_heads = q.shape[0], q.shape[1]
    d = q.shape[-1]
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        need = paged_decode_workspace_size(pool, batch, q_heads, max_blocks, kv_split_tokens)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device) if need else None
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(lib.paged_decode_attention_split_merge(
        pool.handle, _ptr(q), int(q_heads), _ptr(block_tables), int(max_blocks),
        _ptr(context_lens), int(batch), float(scale), int(kv_split_tokens), _ptr(workspace),
        int(ws_bytes), _ptr(out), _ptr(lse), _stream(stream)), "paged_decode_attention_split_merge")
    return out


def paged_merge_attention_states(outs, lses, out=None, lse=None, stream=None):
    """Attention over the union of disjoint key sets from the results over each set.

    outs: bf16 [n_src, *rows, d]; lses: fp32 [n_src, *rows] (natural log, -inf for a set
    with no key).  Returns out bf16 [*rows, d]; writes lse fp32 [*rows] when given."""
    lib = load_library()
    _need(outs, torch.bfloat16, "outs")
    _need(lses, torch.float32, "lses")
    n_src, d = outs.shape[0], outs.shape[-1]
    if tuple(lses.shape) != tuple(outs.shape[:-1]):
        raise ValueError("lses must have the shape of outs without its last dimension")
    rows = lses[0].numel() if n_src else 0
    if out is None:
        out = torch.empty(outs.shape[1:], dtype=torch.bfloat16, device=outs.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if out.numel() != rows * d or (lse is not None and lse.numel() != rows):
        raise ValueError("out / lse sizes do not match outs")
    _check(lib.paged_merge_attention_states(_ptr(outs), _ptr(lses), int(n_src), int(rows), int(d),
                                            _ptr(out), _ptr(lse), _stream(stream)),
           "paged_merge_attention_states")
    return out


def paged_multi_query_workspace_size(pool: Pool, batch: int, q_heads: int, q_len: int,
                                     max_blocks: int, kv_split_tokens: int = 0) -> int:
    lib = load_library()
    n = ctypes.c_size_t()
    _check(lib.paged_multi_query_workspace_size(pool.handle, int(batch), int(q_heads), int(q_len),
                                                int(max_blocks), int(kv_split_tokens),
                                                ctypes.byref(n)),
           "paged_multi_query_workspace_size")
    return n.value


def paged_attention_multi_query(pool: Pool, q, block_tables, context_lens, scale: float,
                                kv_split_tokens: int = 0, workspace=None, out=None, lse=None,
                                stream=None):
    """Attention of q_len new tokens per sequence; q bf16 [B, Hq, q_len, d].  Returns out."""
    lib = load_library()
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    if q.dim() != 4:
        raise ValueError("q must be [batch, q_heads, q_len, head_dim]")
    batch, q_heads, q_len, d = q.shape
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        need = paged_multi_query_workspace_size(pool, batch, q_heads, q_len, max_blocks,
                                                kv_split_tokens)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device) if need else None
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(lib.paged_attention_multi_query(pool.handle, _ptr(q), int(q_heads), int(q_len),
                                           _ptr(block_tables), int(max_blocks), _ptr(context_lens),
                                           int(batch), float(scale), int(kv_split_tokens),
                                           _ptr(workspace), int(ws_bytes), _ptr(out), _ptr(lse),
                                           _stream(stream)),
           "paged_attention_multi_query")
    return out


def paged_decode_step(pool: Pool, k_new, v_new, q, block_tables, context_lens,
                      scale: float, kv_split_tokens: int = 0, workspace=None,
                      out=None, lse=None, stream=None):
    """One decode step: append k_new / v_new (bf16 [B * q_len, Hkv, d]; row i is token i %
    q_len of sequence i / q_len, at position ctx - q_len + i % q_len), then the attention of
    q (bf16 [B, Hq, q_len, d], or [B, Hq, d] for one token per sequence) over the cache.
    Returns out (shaped like q)."""
    lib = load_library()
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    if q.dim() == 3:
        batch, q_heads, d = q.shape
        q_len = 1
    elif q.dim() == 4:
        batch, q_heads, q_len, d = q.shape
    else:
        raise ValueError("q must be [batch, q_heads, head_dim] or [batch, q_heads, q_len, head_dim]")
    if k_new.shape[0] != batch * q_len or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must hold batch * q_len tokens")
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        need = paged_multi_query_workspace_size(pool, batch, q_heads, q_len, max_blocks,
                                                kv_split_tokens)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device) if need else None
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(lib.paged_decode_step(pool.handle, _ptr(k_new), _ptr(v_new), _ptr(q), int(q_heads),
                                 int(q_len), _ptr(block_tables), int(max_blocks), _ptr(context_lens),
                                 int(batch), float(scale), int(kv_split_tokens), _ptr(workspace),
                                 int(ws_bytes), _ptr(out), _ptr(lse), _stream(stream)),
           "paged_decode_step")
    return out


def kv_copy_blocks(pool: Pool, copies, stream=None):
    """Copy whole pool blocks (K and V) on the device: copies is an int32 CUDA tensor [n, 2]
    of (src, dst) pairs, as BlockManager.append_slots reports them for copy-on-write."""
    lib = load_library()
    _need(copies, torch.int32, "copies")
    if copies.dim() != 2 or copies.shape[1] != 2:
        raise ValueError("copies must have shape [n, 2]")
    _check(lib.kv_copy_blocks(pool.handle, _ptr(copies), int(copies.shape[0]), _stream(stream)),
           "kv_copy_blocks")


class BlockManager:
    """Host allocator of a pool's blocks (free list, copy-on-write, prefix caching).

    A thin wrapper of the kv_bm_* calls; all bookkeeping runs in the library."""

    def __init__(self, num_blocks: int, block_size: int, lifo: bool = False,
                 prefix_caching: bool = False):
        self._lib = load_library()
        flags = (BM_LIFO if lifo else BM_FIFO) | (BM_PREFIX_CACHING if prefix_caching else 0)
        h = ctypes.c_void_p()
        _check(self._lib.kv_bm_create(int(num_blocks), int(block_size), flags, ctypes.byref(h)),
               "kv_bm_create")
        self._h = h.value
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    @staticmethod
    def _ids(token_ids):
        if token_ids is None:
            return None, None
        arr = (ctypes.c_int32 * len(token_ids))(*[int(t) for t in token_ids])
        return arr, ctypes.cast(arr, ctypes.c_void_p)

    def add_sequence(self, seq: int, salt: int = 0):
        _check(self._lib.kv_bm_add_sequence(self._h, int(seq), int(salt) & (2**64 - 1)),
               "kv_bm_add_sequence")

    def fork(self, parent: int, child: int):
        _check(self._lib.kv_bm_fork(self._h, int(parent), int(child)), "kv_bm_fork")

    def append_slots(self, seq: int, n_tokens: int, token_ids=None):
        """Returns the copy-on-write copy to make first, as (src, dst), or None."""
        if token_ids is not None and len(token_ids) != n_tokens:
            raise ValueError("token_ids must hold n_tokens ids")
        keep, ids = self._ids(token_ids)
        cp, n = _BlockCopy(), ctypes.c_int()
        _check(self._lib.kv_bm_append_slots(self._h, int(seq), int(n_tokens), ids,
                                            ctypes.byref(cp), ctypes.byref(n)),
               "kv_bm_append_slots")
        return (cp.src, cp.dst) if n.value else None

    def match_prefix(self, seq: int, token_ids) -> int:
        keep, ids = self._ids(token_ids)
        c = ctypes.c_int()
        _check(self._lib.kv_bm_match_prefix(self._h, int(seq), ids, len(token_ids),
                                            ctypes.byref(c)), "kv_bm_match_prefix")
        return c.value

    def free_sequence(self, seq: int):
        _check(self._lib.kv_bm_free_sequence(self._h, int(seq)), "kv_bm_free_sequence")

    def num_free_blocks(self):
        """(free, cached-and-evictable)."""
        a, b = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.kv_bm_num_free_blocks(self._h, ctypes.byref(a), ctypes.byref(b)),
               "kv_bm_num_free_blocks")
        return a.value, b.value

    def sequence_info(self, seq: int):
        """(tokens, blocks) of a sequence."""
        a, b = ctypes.c_int(), ctypes.c_int()
        _check(self._lib.kv_bm_sequence_info(self._h, int(seq), ctypes.byref(a), ctypes.byref(b)),
               "kv_bm_sequence_info")
        return a.value, b.value

    def refcount(self, block: int) -> int:
        r = ctypes.c_int()
        _check(self._lib.kv_bm_block_refcount(self._h, int(block), ctypes.byref(r)),
               "kv_bm_block_refcount")
        return r.value

    def build_tables(self, seqs, max_blocks: int):
        """Host int32 tensors (block_tables [batch, max_blocks], context_lens [batch])."""
        batch = len(seqs)
        ids = (ctypes.c_int64 * max(batch, 1))(*[int(s) for s in seqs])
        tables = torch.empty(batch, int(max_blocks), dtype=torch.int32)
        lens = torch.empty(batch, dtype=torch.int32)
        _check(self._lib.kv_bm_build_tables(self._h, ctypes.cast(ids, ctypes.c_void_p), batch,
                                            int(max_blocks), tables.data_ptr(), lens.data_ptr()),
               "kv_bm_build_tables")
        return tables, lens

    def block_table(self, seq: int):
        """The sequence's block ids, in order."""
        n = self.sequence_info(seq)[1]
        return self.build_tables([seq], max(n, 1))[0][0, :n].tolist()

    def close(self):
        if getattr(self, "_h", None):
            self._lib.kv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------------------- MLA
def kv_mla_pool_create(num_blocks: int, block_size: int, latent_dim: int = 512,
                       rope_dim: int = 64, device: int | None = None) -> Pool:
    """Latent pool [num_blocks, block_size, latent_dim + rope_dim] bf16 (no V half)."""
    lib = load_library()
    if device is None:
        device = torch.cuda.current_device()
    h = ctypes.c_void_p()
    _check(lib.kv_mla_pool_create(int(num_blocks), int(block_size), int(latent_dim),
                                  int(rope_dim), int(device), ctypes.byref(h)),
           "kv_mla_pool_create")
    return Pool(h.value, num_blocks, block_size, 1, latent_dim + rope_dim, "bf16", device,
                latent=True)


def paged_mla_decode_plan(pool: Pool, batch: int, q_heads: int, max_blocks: int,
                          kv_split_tokens: int = 0):
    lib = load_library()
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(lib.paged_mla_decode_plan(pool.handle, int(batch), int(q_heads), int(max_blocks),
                                     int(kv_split_tokens), ctypes.byref(a), ctypes.byref(b)),
           "paged_mla_decode_plan")
    return a.value, b.value


def paged_mla_workspace_size(pool: Pool, batch: int, q_heads: int, max_blocks: int,
                             kv_split_tokens: int = 0) -> int:
    lib = load_library()
    n = ctypes.c_size_t()
    _check(lib.paged_mla_workspace_size(pool.handle, int(batch), int(q_heads), int(max_blocks),
                                        int(kv_split_tokens), ctypes.byref(n)),
           "paged_mla_workspace_size")
    return n.value


def paged_mla_decode_attention(pool: Pool, q, block_tables, context_lens, scale: float,
                               kv_split_tokens: int = 0, workspace=None, out=None, lse=None,
                               stream=None, latent_dim: int = 512):
    """Absorbed MLA decode: q bf16 [B, Hq, latent + rope] -> out bf16 [B, Hq, latent]."""
    lib = load_library()
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    batch, q_heads = q.shape[0], q.shape[1]
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty(batch, q_heads, latent_dim, dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        need = paged_mla_workspace_size(pool, batch, q_heads, max_blocks, kv_split_tokens)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device) if need else None
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(lib.paged_mla_decode_attention(pool.handle, _ptr(q), int(q_heads), _ptr(block_tables),
                                          int(max_blocks), _ptr(context_lens), int(batch),
                                          float(scale), int(kv_split_tokens), _ptr(workspace),
                                          int(ws_bytes), _ptr(out), _ptr(lse), _stream(stream)),
           "paged_mla_decode_attention")
    return out


def paged_mla_decode_step(pool: Pool, kv_new, q, block_tables, context_lens, scale: float,
                          kv_split_tokens: int = 0, workspace=None, out=None, lse=None,
                          stream=None, latent_dim: int = 512):
    """One step over a latent pool: append kv_new bf16 [B, latent + rope] at position
    context_lens[b] - 1 of each sequence, then the absorbed MLA decode (one call: the
    attention kernel writes the new vectors before it loads their blocks).  Returns out
    bf16 [B, Hq, latent]."""
    lib = load_library()
    _need(kv_new, torch.bfloat16, "kv_new")
    _need(q, torch.bfloat16, "q")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    batch, q_heads = q.shape[0], q.shape[1]
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty(batch, q_heads, latent_dim, dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    if workspace is None:
        need = paged_mla_workspace_size(pool, batch, q_heads, max_blocks, kv_split_tokens)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=q.device) if need else None
    _need(workspace, torch.uint8, "workspace")
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check(lib.paged_mla_decode_step(pool.handle, _ptr(kv_new), _ptr(q), int(q_heads),
                                     _ptr(block_tables), int(max_blocks), _ptr(context_lens),
                                     int(batch), float(scale), int(kv_split_tokens),
                                     _ptr(workspace), int(ws_bytes), _ptr(out), _ptr(lse),
                                     _stream(stream)),
           "paged_mla_decode_step")
    return out
