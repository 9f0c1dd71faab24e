"""The decode kernel's failure path, made to run on purpose without faulting
anything.  Through the testing hook qattn_debug_decode_faults the first CTA
of the decode kernel skips one K copy, so the barrier of that tile never
completes and the waits on it run out after a 1 ms limit.  The call must
come back, set QATTN_DEVERR_TIMEOUT in the error word (every role gave up,
drained its copies and MMAs, and freed tensor memory), and leave the
context usable: the next call, defaults restored, matches the oracle."""
import time

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import GpuRun, assert_close, oracle_step, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_07_gb300 import build
    build.build()
    Q.load_library()
    yield
    Q.qattn_debug_decode_faults(0, -1)


@pytest.mark.parametrize("skip", [0, 1, 5])
def test_decode_wait_runs_out_then_next_call_is_clean(skip):
    w = W.build(1)
    _, _, _, ref, e1, e2 = oracle_step(w)
    r = GpuRun(w).append().sync()
    assert r.err_bits == 0
    try:
        Q.qattn_debug_decode_faults(1_000_000, skip)
        t0 = time.perf_counter()
        r.attend().sync()
        dt = time.perf_counter() - t0
    finally:
        Q.qattn_debug_decode_faults(0, -1)
    assert r.err_bits & Q.DEVERR_TIMEOUT, f"error bits {r.err_bits}"
    assert dt < 5.0
    r.err.zero_()
    r.attend().sync()
    assert e1 == e2 == 0 and r.err_bits == 0
    assert_close(r.out, ref)


def test_fp8_decode_wait_runs_out_then_next_call_is_clean():
    w = W.with_fp8_cache(W.build(1))
    ks, vs = W.FP8_K_SCALE, W.FP8_V_SCALE
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    qkv, kc, vc = u16(w.qkv), w.k_cache.numpy().copy(), w.v_cache.numpy().copy()
    table = oracle.rope_table(w.theta, w.max_pos, D)
    assert oracle.rope_cache_append_fp8(qkv, w.positions, w.slot_mapping, kc, vc, table, H, Hkv,
                                        D, BS, ks, vs) == 0
    ref, e = oracle.paged_attention_fp8(np.ascontiguousarray(qkv[:, :H * D]), kc, vc, ks, vs,
                                        w.block_tables, w.context_lens, H, Hkv, D, BS)
    assert e == 0
    dev = torch.device("cuda:0")
    g = W.to_device(w, dev)
    dims = Q.make_dims(H, Hkv, D, BS)
    tab = Q.qattn_rope_table_build(w.max_pos, D, w.theta).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    Q.qattn_rope_cache_append_fp8(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                  g.slot_mapping, g.k_cache, g.v_cache, tab, ks, vs, dims,
                                  err_word=err)
    out = torch.empty((w.num_seqs, H, D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(Q.qattn_paged_decode_workspace_size(w.num_seqs, w.max_context_len, dims),
                     dtype=torch.uint8, device=dev)

    def call():
        Q.qattn_paged_decode_fp8(out, g.q_view(), g.k_cache, g.v_cache, g.block_tables,
                                 g.context_lens, w.max_context_len, ks, vs, dims, ws, err)
        torch.cuda.synchronize()
    try:
        Q.qattn_debug_decode_faults(1_000_000, 2)
        call()
    finally:
        Q.qattn_debug_decode_faults(0, -1)
    assert int(err.item()) & Q.DEVERR_TIMEOUT
    err.zero_()
    call()
    assert int(err.item()) == 0
    got = out.float().cpu().double().numpy()
    d = (np.abs(got - ref) - 2.0 ** -8 * np.abs(ref)).max()
    assert d <= 1e-2 and np.abs(got - ref).max() / np.abs(ref).max() <= 2e-2
