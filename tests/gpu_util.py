"""Helpers shared by the GPU tests: stage a workload into a pool through the
C-ABI binding and compare results with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import paged_kv_cache_19_gb300 as kp
import workloads

# Tolerances for attention outputs (bf16 storage, fp32 accumulation).
MAX_ABS = 2e-2
REL_L2 = 5e-3
FP8_VS_UNQUANTISED_MAX_ABS = 6e-2
FP8_GATE_MIN_CTX = 64        # the unquantised-data gate needs the rounding errors to average out
LSE_ABS = 2e-3


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


class Staged:
    """A workload resident on the GPU: pool (poisoned, prefilled), tables, q."""

    def __init__(self, w: workloads.Workload, step_append: bool = True, chunk: int = 1 << 16):
        s = w.spec
        self.w = w
        if s.mla:
            self.pool = kp.kv_mla_pool_create(w.num_blocks, s.block_size, s.latent_dim,
                                              s.head_dim - s.latent_dim)
        else:
            self.pool = kp.kv_pool_create(w.num_blocks, s.block_size, s.kv_heads, s.head_dim,
                                          s.cache_dtype)
        for t in self.pool.raw_bytes():
            if t is not None:
                t.fill_(workloads.POISON_BYTE)
        if s.cache_dtype == "fp8_e4m3":
            self.pool.set_scales(w.k_scale, w.v_scale)
        self.tables = i32(w.block_tables)
        self.ctx = i32(w.context_lens)
        self.q = bf16_tensor(w.q)
        n = w.prefill_seq.size
        for a in range(0, n, chunk):
            rows = w.prefill_row[a:a + chunk]
            kp.paged_kv_append(self.pool, bf16_tensor(w.k[rows]),
                               None if s.mla else bf16_tensor(w.v[rows]),
                               self.tables, self.ctx, token_seq=i32(w.prefill_seq[a:a + chunk]),
                               token_pos=i32(w.prefill_pos[a:a + chunk]))
        self.k_new = bf16_tensor(w.k_new)
        self.v_new = None if s.mla else bf16_tensor(w.v_new)
        if w.q_len > 1:
            self.q_multi = bf16_tensor(w.q_multi)
            self.k_step = bf16_tensor(w.k[w.step_rows])
            self.v_step = bf16_tensor(w.v[w.step_rows])
            self.step_seq = i32(w.step_seq)
            self.step_pos = i32(w.step_pos)
        if step_append:
            self.append_step()

    def append_step(self, stream=None):
        if self.w.q_len > 1:
            kp.paged_kv_append(self.pool, self.k_step, self.v_step, self.tables, self.ctx,
                               token_seq=self.step_seq, token_pos=self.step_pos, stream=stream)
        else:
            kp.paged_kv_append(self.pool, self.k_new, self.v_new, self.tables, self.ctx,
                               stream=stream)

    def multi(self, split_tokens=None, lse=True, stream=None):
        s = self.w.spec
        split = s.split_tokens if split_tokens is None else split_tokens
        out = torch.empty_like(self.q_multi)
        l = (torch.empty(self.q_multi.shape[:3], dtype=torch.float32, device="cuda")
             if lse else None)
        kp.paged_attention_multi_query(self.pool, self.q_multi, self.tables, self.ctx, self.w.scale,
                                       kv_split_tokens=split, out=out, lse=l, stream=stream)
        return out, l

    def decode(self, split_tokens=None, lse=True, stream=None):
        s = self.w.spec
        split = s.split_tokens if split_tokens is None else split_tokens
        out = torch.empty_like(self.q)
        l = torch.empty(self.q.shape[:2], dtype=torch.float32, device="cuda") if lse else None
        kp.paged_decode_attention(self.pool, self.q, self.tables, self.ctx, self.w.scale,
                                  kv_split_tokens=split, out=out, lse=l, stream=stream)
        return out, l

    def mla(self, split_tokens=None, lse=True, stream=None):
        s = self.w.spec
        split = s.split_tokens if split_tokens is None else split_tokens
        out = torch.empty(self.q.shape[0], self.q.shape[1], s.latent_dim, dtype=torch.bfloat16,
                          device="cuda")
        l = torch.empty(self.q.shape[:2], dtype=torch.float32, device="cuda") if lse else None
        kp.paged_mla_decode_attention(self.pool, self.q, self.tables, self.ctx, self.w.scale,
                                      kv_split_tokens=split, out=out, lse=l, stream=stream,
                                      latent_dim=s.latent_dim)
        return out, l

    def destroy(self):
        self.pool.destroy()


def compare(out: torch.Tensor, ref: np.ndarray):
    """max |err| and relative L2 error of a bf16 GPU result against float64."""
    got = out.float().cpu().double().numpy().reshape(ref.shape)
    err = got - ref
    max_abs = float(np.max(np.abs(err))) if err.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(err) / den) if den > 0 else float(np.linalg.norm(err))
    return max_abs, rel, got
