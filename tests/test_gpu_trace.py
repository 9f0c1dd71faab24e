"""The tracing build's diagnostics on the GPU: the per-CTA phase stamps of a
decode call, and the copy probe (the decode's K/V tile copies alone) -- both
finish with no device error and stay within their documented argument
ranges."""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_gqa_07_gb300 import build as B
from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import device_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tlib():
    B.build()
    Q.load_library()
    T = ctypes.CDLL(B.build(trace=True))
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    T.qattn_trace_copy_stream.argtypes = [P, P, I32, Q.qattn_dims, I32, P, I32, I32, P, P]
    T.qattn_trace_copy_stream.restype = ctypes.c_int
    T.qattn_trace_dims.argtypes = [P, P, P]
    T.qattn_trace_read.argtypes = [P, P]
    return T


def _tiles(w):
    bs, bpt = w.block_size, 128 // w.block_size
    bt = w.block_tables.tolist()
    out = []
    for b, L in enumerate(w.context_lens.tolist()):
        nblk = (L + bs - 1) // bs
        for g in range(w.num_kv_heads):
            for i in range((L + 127) // 128):
                out.append([g] + [bt[b][i * bpt + j] if i * bpt + j < nblk else -1
                                  for j in range(8)])
    return out


@pytest.mark.parametrize("fp8,bs,stages", [(0, 16, 2), (0, 64, 3), (1, 16, 4), (1, 32, 6)])
def test_copy_probe_runs_clean(tlib, fp8, bs, stages):
    w = W.custom(28, 4, ctx=[1, 129, 700, 3000, 4096, 17], q_lens=[1] * 6, seed=850 + bs,
                 block_size=bs)
    if fp8:
        w = W.with_fp8_cache(w)
    dev = torch.device("cuda", 0)
    g = W.to_device(w, dev)
    dims = Q.make_dims(w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
    tiles = torch.tensor(_tiles(w), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream()
    args = (g.k_cache.data_ptr(), g.v_cache.data_ptr(), int(g.k_cache.shape[0]), dims, fp8,
            tiles.data_ptr(), int(tiles.shape[0]))
    for _ in range(3):
        assert tlib.qattn_trace_copy_stream(*args, stages, err.data_ptr(), s.cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # stage counts outside the ring the shared memory holds are refused
    for bad in (1, 4 if not fp8 else 8):
        assert tlib.qattn_trace_copy_stream(*args, bad, err.data_ptr(), s.cuda_stream) == 1


def test_copy_probe_flags_bad_block(tlib):
    w = W.custom(16, 8, ctx=[300, 40], q_lens=[1, 1], seed=851)
    dev = torch.device("cuda", 0)
    g = W.to_device(w, dev)
    dims = Q.make_dims(w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
    t = _tiles(w)
    t[1][1] = int(g.k_cache.shape[0])  # one past the last block: skipped and flagged
    tiles = torch.tensor(t, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    assert tlib.qattn_trace_copy_stream(g.k_cache.data_ptr(), g.v_cache.data_ptr(),
                                        int(g.k_cache.shape[0]), dims, 0, tiles.data_ptr(),
                                        len(t), 2, err.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) & Q.DEVERR_BLOCK


def test_phase_stamps_of_a_decode_call(tlib):
    """The tracing build's decode call gives the right output and stamps
    every phase in order on the CTAs that ran."""
    w = W.custom(28, 4, ctx=[4096, 1000, 33], q_lens=[1] * 3, seed=852)
    dev = torch.device("cuda", 0)
    g = W.to_device(w, dev)
    dims = Q.make_dims(w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    tlib.qattn_paged_decode.argtypes = [P, P, I64, P, P, I32, P, I32, P, I32, I32, Q.qattn_dims,
                                        P, ctypes.c_size_t, P, P]
    tlib.qattn_paged_decode_workspace_size.argtypes = [I32, I32, Q.qattn_dims]
    tlib.qattn_paged_decode_workspace_size.restype = ctypes.c_size_t
    ws = torch.empty(tlib.qattn_paged_decode_workspace_size(3, w.max_context_len, dims),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((3, 28, 128), dtype=torch.bfloat16, device=dev)
    ref = torch.empty_like(out)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # the new tokens' K/V into the cache first (their slots hold NaN codes)
    Q.qattn_rope_cache_append(g.q_view(), g.k_view(), g.v_view(), g.positions, g.slot_mapping,
                              g.k_cache, g.v_cache, device_table(w.max_pos, w.theta, "cuda:0"),
                              dims, err)
    q = g.q_view()
    assert tlib.qattn_trace_clear() == 0
    assert tlib.qattn_paged_decode(out.data_ptr(), q.data_ptr(), q.stride(0), g.k_cache.data_ptr(),
                                   g.v_cache.data_ptr(), int(g.k_cache.shape[0]),
                                   g.block_tables.data_ptr(), int(g.block_tables.shape[1]),
                                   g.context_lens.data_ptr(), 3, w.max_context_len, dims,
                                   ws.data_ptr(), ws.numel(), err.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    Q.qattn_paged_decode(ref, q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                         w.max_context_len, dims, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.isfinite(ref.float()).all()
    assert torch.equal(out, ref)  # the stamps change no result
    n = (ctypes.c_int32 * 3)()
    tlib.qattn_trace_dims(ctypes.byref(n, 0), ctypes.byref(n, 4), ctypes.byref(n, 8))
    dec = np.zeros(n[0] * n[1], dtype=np.uint64)
    mer = np.zeros(n[2] * 4, dtype=np.uint64)
    assert tlib.qattn_trace_read(dec.ctypes.data, mer.ctypes.data) == 0
    d = dec.reshape(n[0], n[1]).astype(np.int64)
    ran = d[d[:, 5] > 0]
    assert len(ran) > 0
    assert (np.diff(ran[:, [0, 1, 2, 4, 5]], axis=1) >= 0).all()
