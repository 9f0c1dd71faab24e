"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle
on the same seeded inputs.

Bar: the cache append and all slot/block indexing bit-exact (the whole
k_cache and v_cache, sentinel-filled unused slots included, and the rotated
queries); attention outputs within max-abs 1e-2 and max-abs / max|ref| 2e-2
of the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import GpuRun, assert_close, compare, oracle_for, oracle_step, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_07_gb300 import build
    build.build()
    Q.load_library()


# ------------------------------------------------------------ append ----

@pytest.mark.parametrize("idx", range(5))
def test_append_bit_exact(idx):
    w = W.build(idx)
    qkv, kc, vc, _, e1, _ = oracle_for(idx)
    r = GpuRun(w).append().sync()
    assert r.err_bits == 0 and e1 == 0
    assert np.array_equal(u16(r.g.k_cache), kc), "k_cache differs"
    assert np.array_equal(u16(r.g.v_cache), vc), "v_cache differs"
    assert np.array_equal(u16(r.g.qkv), qkv), "rotated q (or k/v rows) differ"


def test_append_theta_pitfall_detected():
    """rope_theta 1e4 (the pages' pitfall) produces a different cache."""
    w = W.build(0)
    a = GpuRun(w).append().sync()
    b = GpuRun(w, theta=1e4).append().sync()
    assert not np.array_equal(u16(a.g.k_cache), u16(b.g.k_cache))
    _, kc4, _, _, _, _ = oracle_step(w, theta=1e4)
    assert np.array_equal(u16(b.g.k_cache), kc4)


def test_append_error_bits_and_padding():
    w = W.build(0)
    bad = W.to_device(w, "cpu")
    n_slots = w.num_blocks * w.block_size
    bad.slot_mapping = w.slot_mapping.clone()
    bad.positions = w.positions.clone()
    bad.slot_mapping[0] = n_slots + 3        # out of range: skipped, bit 1
    bad.slot_mapping[1] = -1                 # padding: q rotated, nothing written
    bad.positions[2] = w.max_pos             # out of range: token skipped, bit 16
    qkv, kc, vc, _, e1, _ = oracle_step(bad)
    assert e1 == Q.DEVERR_SLOT | Q.DEVERR_POSITION
    r = GpuRun(bad).append().sync()
    assert r.err_bits == Q.DEVERR_SLOT | Q.DEVERR_POSITION
    assert np.array_equal(u16(r.g.k_cache), kc)
    assert np.array_equal(u16(r.g.v_cache), vc)
    assert np.array_equal(u16(r.g.qkv), qkv)


def test_append_large_token_count():
    """A prefill-sized append (4 x 512 + 60 tokens) and a 16k-token one."""
    w = W.custom(28, 4, ctx=[4096] * 4, q_lens=[4096] * 4, seed=21)
    qkv, kc, vc, _, _, _ = oracle_step_append_only(w)
    r = GpuRun(w).append().sync()
    assert r.err_bits == 0
    assert np.array_equal(u16(r.g.k_cache), kc) and np.array_equal(u16(r.g.v_cache), vc)
    assert np.array_equal(u16(r.g.qkv), qkv)


def oracle_step_append_only(w):
    qkv, kc, vc = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
    table = oracle.rope_table(w.theta, w.max_pos, 128)
    e = oracle.rope_cache_append(qkv, w.positions, w.slot_mapping, kc, vc, table,
                                 w.num_heads, w.num_kv_heads, 128, 16)
    return qkv, kc, vc, None, e, 0


# ------------------------------------------------------------ decode ----

@pytest.mark.parametrize("idx", [0, 1, 3, 4])
def test_decode_parity(idx):
    w = W.build(idx)
    _, _, _, ref, _, e2 = oracle_for(idx)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


def test_decode_deterministic():
    w = W.build(1)
    r = GpuRun(w).append().attend().sync()
    first = r.out.clone()
    for _ in range(3):
        r.attend().sync()
        assert torch.equal(r.out, first)


def test_decode_block_permutation_bit_identical():
    w = W.build(1)
    a = GpuRun(w).append().attend().sync()
    b = GpuRun(W.permute_blocks(w, seed=5)).append().attend().sync()
    assert torch.equal(a.out, b.out)


@pytest.mark.parametrize("group", [1, 2, 3, 4, 5, 6, 7, 8])
def test_decode_ragged_contexts_every_group(group):
    """Contexts around the block (16) and chunk (32) edges, for every GQA
    group size the library supports."""
    ctx = [1, 2, 15, 16, 17, 31, 32, 33, 47, 63, 64, 65, 100, 257, 511, 512, 513, 1000]
    Hkv = 2
    w = W.custom(group * Hkv, Hkv, ctx=ctx, q_lens=[1] * len(ctx), seed=30 + group)
    _, _, vc, ref, _, e2 = oracle_step(w)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)
    # a one-token context returns V exactly
    v0 = torch.from_numpy(vc[int(w.block_tables[0, 0]), :, 0, :].astype(np.int16)).view(torch.bfloat16)
    assert torch.equal(r.out[0].cpu(), v0.repeat_interleave(group, dim=0))


def test_decode_many_sequences():
    """More sequences than threads in a CTA (the chunk-list scan runs in
    several tiles), short and long mixed."""
    gen = torch.Generator().manual_seed(40)
    ctx = torch.randint(1, 300, (700,), generator=gen).tolist()
    w = W.custom(16, 8, ctx=ctx, q_lens=[1] * 700, seed=41)
    _, _, _, ref, _, _ = oracle_step(w)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0
    assert_close(r.out, ref)


def test_varlen_api_on_decode_rows_matches_decode():
    w = W.build(1)
    a = GpuRun(w).append().attend(varlen=False).sync()
    b = GpuRun(w).append().attend(varlen=True).sync()
    assert torch.equal(a.out, b.out)


def test_decode_error_bits():
    w = W.build(0)
    r = GpuRun(w).append().sync()
    r.g.context_lens[1] = 0                   # invalid context: zero row, bit 4
    r.g.block_tables[2, 3] = w.num_blocks + 9  # bad block id: bit 2
    r.attend().sync()
    bits = r.err_bits
    assert bits & Q.DEVERR_CONTEXT and bits & Q.DEVERR_BLOCK and not bits & Q.DEVERR_TIMEOUT
    assert torch.count_nonzero(r.out[1]) == 0
    _, _, _, ref, _, _ = oracle_for(0)
    assert_close(r.out, ref, rows=[0, 3])     # untouched sequences still right


def test_decode_context_above_hint_is_flagged():
    w = W.build(0)
    r = GpuRun(w, max_context_len=200).append().attend().sync()   # one context is 255
    assert r.err_bits & Q.DEVERR_CONTEXT
    assert torch.count_nonzero(r.out[3]) == 0
    _, _, _, ref, _, _ = oracle_for(0)
    assert_close(r.out, ref, rows=[0, 1, 2])


def test_zero_sized_calls_are_noops():
    w = W.build(0)
    r = GpuRun(w)
    empty_i = torch.empty(0, dtype=torch.int32, device=r.dev)
    empty_q = torch.empty((0, w.num_heads * 128), dtype=torch.bfloat16, device=r.dev)
    Q.qattn_rope_cache_append(empty_q, empty_q[:, :1024], empty_q[:, :1024], empty_i, empty_i,
                              r.g.k_cache, r.g.v_cache, r.table, r.dims, r.err)
    Q.qattn_paged_decode(r.out[:0], empty_q, r.g.k_cache, r.g.v_cache,
                         r.g.block_tables[:0], r.g.context_lens[:0], 16, r.dims, r.ws, r.err)
    r.sync()
    assert r.err_bits == 0


def test_workspace_too_small_is_rejected():
    w = W.build(0)
    r = GpuRun(w).append()
    small = r.ws[:128]
    with pytest.raises(Q.QattnError) as ei:
        Q.qattn_paged_decode(r.out, r.g.q_view(), r.g.k_cache, r.g.v_cache, r.g.block_tables,
                             r.g.context_lens, r.max_ctx, r.dims, small, r.err)
    assert ei.value.status == Q.QATTN_ERR_WORKSPACE


# ------------------------------------------------------ workspace ----

def test_decode_workspace_needs_no_initialisation():
    """The split-KV parts and their counts live in the workspace.  A
    workspace of random bytes, and one reused across shapes, give the clean
    result."""
    ref = GpuRun(W.build(1)).append().attend().sync().out.clone()
    w1, w3 = W.build(1), W.build(3)
    r1, r3 = GpuRun(w1).append(), GpuRun(w3).append()
    size = max(r1.ws.numel(), r3.ws.numel())
    gen = torch.Generator(device=r1.dev).manual_seed(77)
    ws = torch.randint(0, 256, (size,), dtype=torch.uint8, device=r1.dev, generator=gen)
    r1.ws, r3.ws = ws, ws
    r1.attend().sync()
    assert r1.err_bits == 0 and torch.equal(r1.out, ref)
    r3.attend().sync()                        # other segments, other part counts
    _, _, _, ref3, _, _ = oracle_for(3)
    assert r3.err_bits == 0
    assert_close(r3.out, ref3)
    r1.attend().sync()
    assert r1.err_bits == 0 and torch.equal(r1.out, ref)


@pytest.mark.parametrize("idx", [1, 3])
def test_decode_graph_replay(idx):
    """The step (append, decode, merge; chained by programmatic dependent
    launch) captured in a CUDA graph replays to the same result."""
    w = W.build(idx)
    r = GpuRun(w)
    qkv0 = r.g.qkv.clone()
    r.append().attend().sync()
    first = r.out.clone()
    s = torch.cuda.Stream(device=r.dev)
    s.wait_stream(torch.cuda.current_stream(r.dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            r.g.qkv.copy_(qkv0)
            r.append().attend()
    for _ in range(3):
        r.out.zero_()
        graph.replay()
        r.sync()
        assert r.err_bits == 0
        assert torch.equal(r.out, first)
