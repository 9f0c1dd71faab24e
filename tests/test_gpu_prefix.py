"""GPU parity of the shared-prefix decode (qattn_paged_decode_shared_prefix:
the prefix once per kv head for the whole batch on tensor cores, beside the
decode kernel on each sequence's own tokens, parts merged) against the CPU
oracle's plain paged attention on the same inputs."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import GpuRun, assert_close, oracle_for, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_07_gb300 import build
    build.build()
    Q.load_library()


def run_prefix(r: GpuRun, prefix_len: int, ws=None):
    g = r.g
    if ws is None:
        n = Q.qattn_paged_decode_shared_prefix_workspace_size(r.w.num_seqs, r.max_ctx, r.dims)
        ws = torch.empty(n, dtype=torch.uint8, device=r.dev)
    Q.qattn_paged_decode_shared_prefix(r.out, g.q_view(), g.k_cache, g.v_cache, g.block_tables,
                                       g.context_lens, r.max_ctx, prefix_len, r.dims, ws, r.err)
    return r.sync()


def test_prefix_workload_parity():
    """128 sequences on a 2048-token shared prefix (Qwen3-0.6B heads)."""
    w = W.build(4)
    _, _, _, ref, _, e2 = oracle_for(4)
    r = run_prefix(GpuRun(w).append().sync(), w.shared_prefix_tokens)
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


@pytest.mark.parametrize("group,kv,prefix", [(1, 4, 16), (2, 8, 272), (3, 2, 128),
                                            (7, 4, 400), (8, 2, 1024)])
def test_prefix_every_group(group, kv, prefix):
    """Prefixes of 1 block, a ragged tile count, whole tiles; suffixes from
    1 token to several tiles."""
    suffix = [1, 2, 15, 16, 17, 100, 128, 129, 300, 700, 31, 64]
    ctx = [prefix + s for s in suffix]
    w = W.custom(group * kv, kv, ctx=ctx, q_lens=[1] * len(ctx), seed=400 + group,
                 shared_prefix_tokens=prefix)
    _, _, _, ref, _, e2 = oracle_step(w)
    r = run_prefix(GpuRun(w).append().sync(), prefix)
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


def test_prefix_many_row_tiles():
    """150 sequences of G = 2: three 64-sequence row tiles, the last partial."""
    gen = torch.Generator().manual_seed(410)
    ctx = (256 + torch.randint(1, 200, (150,), generator=gen)).tolist()
    w = W.custom(16, 8, ctx=ctx, q_lens=[1] * 150, seed=411, shared_prefix_tokens=256)
    _, _, _, ref, _, _ = oracle_step(w)
    r = run_prefix(GpuRun(w).append().sync(), 256)
    assert r.err_bits == 0
    assert_close(r.out, ref)


def test_prefix_deterministic_and_zero_prefix_equals_decode():
    w = W.custom(28, 4, ctx=[900, 1000, 513, 2000], q_lens=[1] * 4, seed=420,
                 shared_prefix_tokens=512)
    r = run_prefix(GpuRun(w).append().sync(), 512)
    first = r.out.clone()
    run_prefix(r, 512)
    assert torch.equal(r.out, first)
    plain = GpuRun(w).append().attend().sync().out.clone()
    run_prefix(r, 0)                      # no prefix: the plain decode path
    assert torch.equal(r.out, plain)


def test_prefix_errors():
    w = W.custom(16, 8, ctx=[300, 400, 500, 350], q_lens=[1] * 4, seed=430,
                 shared_prefix_tokens=256)
    r = GpuRun(w).append().sync()
    r.g.context_lens[1] = 256             # no token beyond the prefix: zero row, bit 4
    run_prefix(r, 256)
    assert r.err_bits & Q.DEVERR_CONTEXT and not r.err_bits & Q.DEVERR_PREFIX
    assert torch.count_nonzero(r.out[1]) == 0
    _, _, _, ref, _, _ = oracle_for_custom(w)
    assert_close(r.out, ref, rows=[0, 2, 3])
    r2 = GpuRun(w).append().sync()
    r2.g.block_tables[2, 3] = r2.g.block_tables[2, 20]   # breaks the shared prefix
    run_prefix(r2, 256)
    assert r2.err_bits & Q.DEVERR_PREFIX


def oracle_for_custom(w):
    return oracle_step(w)


def test_prefix_long_prefix_several_splits():
    """A 2304-token prefix (18 tiles: two splits of the prefix pass, the
    second ragged) under short and long suffixes."""
    ctx = [2304 + s for s in (1, 64, 129, 700, 1500, 33, 256, 2)]
    w = W.custom(28, 4, ctx=ctx, q_lens=[1] * len(ctx), seed=450, shared_prefix_tokens=2304)
    _, _, _, ref, _, e2 = oracle_step(w)
    r = run_prefix(GpuRun(w).append().sync(), 2304)
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


def test_prefix_graph_replay():
    """The append and the shared-prefix call (its prefix pass on the
    library's side stream, forked from and joined back into the captured
    stream) captured in a CUDA graph replay to the eager result."""
    w = W.build(4)
    r = GpuRun(w)
    qkv0 = r.g.qkv.clone()
    n = Q.qattn_paged_decode_shared_prefix_workspace_size(w.num_seqs, r.max_ctx, r.dims)
    ws = torch.empty(n, dtype=torch.uint8, device=r.dev)
    run_prefix(r.append().sync(), w.shared_prefix_tokens, ws)
    first = r.out.clone()
    g = r.g
    s = torch.cuda.Stream(device=r.dev)
    s.wait_stream(torch.cuda.current_stream(r.dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.qkv.copy_(qkv0)
            r.append()
            Q.qattn_paged_decode_shared_prefix(r.out, g.q_view(), g.k_cache, g.v_cache,
                                               g.block_tables, g.context_lens, r.max_ctx,
                                               w.shared_prefix_tokens, r.dims, ws, r.err)
    for _ in range(2):
        r.out.zero_()
        graph.replay()
        r.sync()
        assert r.err_bits == 0
        assert torch.equal(r.out, first)


def test_prefix_host_validation():
    w = W.custom(16, 8, ctx=[300, 400], q_lens=[1, 1], seed=440, shared_prefix_tokens=256)
    r = GpuRun(w).append().sync()
    for bad in (-16, 8, 400 + 16):
        with pytest.raises(Q.QattnError) as ei:
            run_prefix(r, bad)
        assert ei.value.status == Q.QATTN_ERR_INVALID_ARG
