"""GPU parity of the causal varlen / chunked-prefill path (tcgen05 kernel plus
the decode rows of a mixed batch) against the CPU oracle."""
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


def test_mixed_varlen_batch_parity():
    """4 chunks of 512 new tokens on 0-1536 cached tokens + 60 decode rows."""
    w = W.build(2)
    _, _, _, ref, _, e2 = oracle_for(2)
    r = GpuRun(w).append().attend().sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref, rows=slice(0, 2048))     # prefill rows
    assert_close(r.out, ref, rows=slice(2048, None))  # decode rows
    assert_close(r.out, ref)


@pytest.mark.parametrize("q_len,cached", [(2, 0), (5, 3), (17, 0), (128, 0), (129, 1),
                                          (300, 50), (256, 700), (513, 1000)])
def test_prefill_ragged_shapes(q_len, cached):
    w = W.custom(28, 4, ctx=[cached + q_len, 40, cached + q_len // 2 + 2],
                 q_lens=[q_len, 1, q_len // 2 + 2], seed=100 + q_len + cached)
    _, _, _, ref, _, e2 = oracle_step(w)
    r = GpuRun(w).append().attend(varlen=True).sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)


@pytest.mark.parametrize("group,kv", [(1, 4), (2, 8), (7, 4), (8, 2)])
def test_prefill_every_group(group, kv):
    w = W.custom(group * kv, kv, ctx=[200, 77, 333], q_lens=[200, 30, 133], seed=200 + group)
    _, _, _, ref, _, _ = oracle_step(w)
    r = GpuRun(w).append().attend(varlen=True).sync()
    assert r.err_bits == 0
    assert_close(r.out, ref)


def test_prefill_first_row_returns_v0():
    """With no cached tokens, query 0 sees key 0 only: its output is v_0."""
    w = W.custom(4, 2, ctx=[160], q_lens=[160], seed=300)
    r = GpuRun(w).append().attend(varlen=True).sync()
    H, Hkv, D = 4, 2, 128
    v0 = w.qkv[0, (H + Hkv) * D:].view(Hkv, D)          # raw v of token 0
    assert torch.equal(r.out[0].cpu(), v0.repeat_interleave(2, dim=0))


def test_prefill_block_permutation_bit_identical():
    w = W.custom(28, 4, ctx=[900, 300], q_lens=[400, 300], seed=301)
    a = GpuRun(w).append().attend(varlen=True).sync()
    b = GpuRun(W.permute_blocks(w, seed=9)).append().attend(varlen=True).sync()
    assert torch.equal(a.out, b.out)


def test_prefill_deterministic():
    w = W.build(2)
    r = GpuRun(w).append().attend().sync()
    first = r.out.clone()
    r.attend().sync()
    assert torch.equal(r.out, first)


def test_prefill_chunk_equals_decode_steps():
    """A 9-token chunk gives (within tolerance) the same rows as 9 decode
    steps over growing contexts -- the chunked-prefill equivalence."""
    w = W.custom(16, 8, ctx=[100], q_lens=[9], seed=302)
    r = GpuRun(w).append().attend(varlen=True).sync()
    g = r.g
    outs = []
    for i in range(9):
        L = 100 - 9 + 1 + i
        out = torch.empty((1, 16, 128), dtype=torch.bfloat16, device=r.dev)
        Q.qattn_paged_decode(out, g.q_view()[i:i + 1], g.k_cache, g.v_cache, g.block_tables,
                             torch.tensor([L], dtype=torch.int32, device=r.dev), 100, r.dims,
                             r.ws, r.err)
        outs.append(out)
    torch.cuda.synchronize()
    dec = torch.cat(outs).float()
    assert (dec - r.out.float()).abs().max().item() <= 1e-2


def test_prefill_context_error_rows():
    w = W.custom(4, 2, ctx=[50, 60], q_lens=[20, 30], seed=303)
    r = GpuRun(w).append().sync()
    r.g.context_lens[0] = 10           # fewer keys than queries: zero rows, bit 4
    r.attend(varlen=True).sync()
    assert r.err_bits & Q.DEVERR_CONTEXT
    assert torch.count_nonzero(r.out[:20]) == 0
    _, _, _, ref, _, _ = oracle_step(w)
    assert_close(r.out, ref, rows=slice(20, 50))


def test_prefill_split_into_sequence_batches():
    """A generous max_q_len hint (40000 tokens: 313 row tiles per sequence)
    makes the library plan one sequence per launch; the result is the same
    as the one-launch plan, bit for bit."""
    w = W.custom(28, 4, ctx=[700, 40, 333, 520], q_lens=[300, 1, 200, 129], seed=304)
    r = GpuRun(w).append().attend(varlen=True).sync()
    first = r.out.clone()
    g = r.g
    r.out.zero_()
    Q.qattn_varlen_prefill(r.out, g.q_view(), g.cu_seqlens_q, 40000, g.k_cache, g.v_cache,
                           g.block_tables, g.context_lens, r.max_ctx, r.dims, r.ws, r.err)
    r.sync()
    assert r.err_bits == 0
    assert torch.equal(r.out, first)
    _, _, _, ref, _, _ = oracle_step(w)
    assert_close(r.out, ref)


def test_prefill_many_tiles_ranked_order():
    """More (sequence, row tile) pairs than CTAs and KV lengths from 1 to 12
    tiles: every item is computed once whatever the ranked order."""
    ctx = [1500, 90, 700, 1300, 260, 1100, 30, 900]
    ql = [600, 90, 650, 130, 260, 1000, 2, 400]
    w = W.custom(8, 2, ctx=ctx, q_lens=ql, seed=305)
    _, _, _, ref, _, e2 = oracle_step(w)
    r = GpuRun(w).append().attend(varlen=True).sync()
    assert r.err_bits == 0 and e2 == 0
    assert_close(r.out, ref)

