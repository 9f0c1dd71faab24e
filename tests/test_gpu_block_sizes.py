"""GPU parity with 32- and 64-token cache blocks (the paged cache's block
size is a deployment knob: vLLM's block_size, PagedAttention section 4.2)
against the CPU oracle, which takes the block size as an argument: the
append bit-exact, decode, varlen prefill and the shared-prefix decode within
the bf16 tolerance."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import GpuRun, assert_close, oracle_step, u16

pytestmark = pytest.mark.gpu

# Context lengths around the block and tile edges of both sizes.
EDGE_CTX = [1, 2, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 1000, 1500]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_07_gb300 import build
    build.build()
    Q.load_library()


@pytest.mark.parametrize("bs", [32, 64])
def test_append_bit_exact(bs):
    w = W.custom(28, 4, ctx=EDGE_CTX, q_lens=[1] * len(EDGE_CTX), seed=700 + bs,
                 block_size=bs)
    assert w.block_size == bs and w.k_cache.shape[2] == bs
    qkv, kc, vc, _, e1, _ = oracle_step(w)
    r = GpuRun(w).append().sync()
    assert r.err_bits == 0 and e1 == 0
    assert np.array_equal(u16(r.g.qkv), qkv)
    assert np.array_equal(u16(r.g.k_cache), kc)
    assert np.array_equal(u16(r.g.v_cache), vc)


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("group,kv", [(1, 8), (2, 4), (7, 4), (8, 2)])
def test_decode(bs, group, kv):
    w = W.custom(group * kv, kv, ctx=EDGE_CTX, q_lens=[1] * len(EDGE_CTX),
                 seed=710 + bs + group, block_size=bs)
    _, _, _, ref, _, e2 = oracle_step(w)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


@pytest.mark.parametrize("bs", [32, 64])
def test_decode_long_split(bs):
    """Contexts of several thousand tokens: split-KV parts and the merge."""
    ctx = [4096, 3000, 5000, 129]
    w = W.custom(28, 4, ctx=ctx, q_lens=[1] * 4, seed=730 + bs, block_size=bs)
    _, _, _, ref, _, _ = oracle_step(w)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0
    assert_close(r.out, ref)


@pytest.mark.parametrize("bs", [32, 64])
def test_varlen_prefill_mixed(bs):
    """Chunked prefill over cached context plus decode rows in one call."""
    ctx = [300, 700, 64, 1, 129, 900]
    q_lens = [200, 33, 64, 1, 1, 1]
    w = W.custom(28, 4, ctx=ctx, q_lens=q_lens, seed=740 + bs, block_size=bs)
    _, _, _, ref, _, e2 = oracle_step(w)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


@pytest.mark.parametrize("bs,prefix", [(32, 32), (32, 416), (64, 192), (64, 1024)])
def test_shared_prefix(bs, prefix):
    suffix = [1, 2, 31, 32, 33, 64, 65, 128, 129, 300]
    ctx = [prefix + s for s in suffix]
    w = W.custom(16, 2, ctx=ctx, q_lens=[1] * len(ctx), seed=750 + bs + prefix,
                 shared_prefix_tokens=prefix, block_size=bs)
    _, _, _, ref, _, e2 = oracle_step(w)
    r = GpuRun(w).append().sync()
    n = Q.qattn_paged_decode_shared_prefix_workspace_size(w.num_seqs, r.max_ctx, r.dims)
    ws = torch.empty(n, dtype=torch.uint8, device=r.dev)
    g = r.g
    Q.qattn_paged_decode_shared_prefix(r.out, g.q_view(), g.k_cache, g.v_cache, g.block_tables,
                                       g.context_lens, r.max_ctx, prefix, r.dims, ws, r.err)
    r.sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


def test_prefix_not_block_multiple_rejected():
    w = W.custom(16, 2, ctx=[200, 300], q_lens=[1, 1], seed=760, block_size=64,
                 shared_prefix_tokens=128)
    r = GpuRun(w).append().sync()
    n = Q.qattn_paged_decode_shared_prefix_workspace_size(w.num_seqs, r.max_ctx, r.dims)
    ws = torch.empty(n, dtype=torch.uint8, device=r.dev)
    g = r.g
    with pytest.raises(Q.QattnError):
        Q.qattn_paged_decode_shared_prefix(r.out, g.q_view(), g.k_cache, g.v_cache,
                                           g.block_tables, g.context_lens, r.max_ctx, 96,
                                           r.dims, ws, r.err)
