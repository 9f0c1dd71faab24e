"""Helpers shared by the GPU parity tests: run the oracle and the CUDA path on
the same seeded workload and compare."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

ATOL = 1e-2   # max |gpu - oracle|
RTOL = 2e-2   # max |gpu - oracle| / max |oracle|


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def oracle_step(w: W.Workload, theta: float | None = None):
    """RoPE + append + attention on the host.  Returns (qkv, k_cache,
    v_cache, out fp64, append error bits, attention error bits)."""
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    qkv, kc, vc = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
    table = oracle.rope_table(w.theta if theta is None else theta, w.max_pos, D)
    e1 = oracle.rope_cache_append(qkv, w.positions, w.slot_mapping, kc, vc, table, H, Hkv, D, BS)
    q = np.ascontiguousarray(qkv[:, :H * D])
    cu = None if w.is_decode else w.cu_seqlens_q
    out, e2 = oracle.paged_attention(q, kc, vc, w.block_tables, w.context_lens, H, Hkv, D, BS,
                                     cu_seqlens_q=cu)
    return qkv, kc, vc, out, e1, e2


@functools.lru_cache(maxsize=8)
def oracle_for(idx: int):
    return oracle_step(W.build(idx))


@functools.lru_cache(maxsize=4)
def device_table(max_pos: int, theta: float, dev: str):
    return Q.qattn_rope_table_build(max_pos, 128, theta).to(dev)


class GpuRun:
    """The CUDA path on one workload: append, then decode or varlen."""

    def __init__(self, w: W.Workload, dev="cuda:0", theta=None, max_context_len=None):
        self.w = w
        self.dev = torch.device(dev)
        self.g = W.to_device(w, self.dev)
        self.dims = Q.make_dims(w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
        self.table = device_table(w.max_pos, w.theta if theta is None else theta, str(self.dev))
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.max_ctx = max_context_len or max(1, w.max_context_len)
        n = w.num_seqs
        size = (Q.qattn_paged_decode_workspace_size(n, self.max_ctx, self.dims) if w.is_decode
                else Q.qattn_varlen_prefill_workspace_size(n, self.max_ctx, self.dims))
        self.ws = torch.empty(max(size, 256), dtype=torch.uint8, device=self.dev)
        self.out = torch.empty((w.num_tokens, w.num_heads, w.head_dim), dtype=torch.bfloat16,
                               device=self.dev)

    def append(self):
        g = self.g
        Q.qattn_rope_cache_append(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                  g.slot_mapping, g.k_cache, g.v_cache, self.table, self.dims,
                                  self.err)
        return self

    def attend(self, varlen: bool | None = None):
        g = self.g
        if varlen is None:
            varlen = not self.w.is_decode
        if varlen:
            Q.qattn_varlen_prefill(self.out, g.q_view(), g.cu_seqlens_q, self.w.max_q_len,
                                   g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                   self.max_ctx, self.dims, self.ws, self.err)
        else:
            Q.qattn_paged_decode(self.out, g.q_view(), g.k_cache, g.v_cache, g.block_tables,
                                 g.context_lens, self.max_ctx, self.dims, self.ws, self.err)
        return self

    def sync(self):
        torch.cuda.synchronize(self.dev)
        return self

    @property
    def err_bits(self) -> int:
        return int(self.err.item())


def compare(got: torch.Tensor, ref: np.ndarray, rows=None):
    """Max abs / max-rel errors of a bf16 GPU output against the fp64 oracle."""
    g = got.float().cpu().double().numpy()
    if rows is not None:
        g, ref = g[rows], ref[rows]
    assert np.isfinite(g).all(), "non-finite GPU output"
    d = np.abs(g - ref)
    mx = float(d.max()) if d.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 1.0
    return mx, mx / max(scale, 1e-30)


def assert_close(got, ref, rows=None):
    mx, rel = compare(got, ref, rows)
    assert mx <= ATOL and rel <= RTOL, f"max abs {mx:.3e} (<= {ATOL}), max rel {rel:.3e} (<= {RTOL})"
    return mx, rel
