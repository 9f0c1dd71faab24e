"""GPU parity of the FP8 (e4m3fn) KV cache (kv_cache_dtype "fp8" with a cache
scale per tensor, "Qwen2大模型架构解析与vLLM优化实践" sections 4.1, 4.2, 6.3)
against the CPU oracle: the append bit-exact (q bits and every cache code),
decode within the bf16 tolerance.  Cached tokens are e4m3 codes (unused
slots hold the NaN code 0x7F), new tokens go through each side's append."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import ATOL, RTOL, device_table, u16

pytestmark = pytest.mark.gpu

KS, VS = W.FP8_K_SCALE, W.FP8_V_SCALE
BF16_HALF_ULP = 2.0 ** -8   # relative rounding of a bf16 output


def assert_close(got, ref):
    """The bf16 bar (max abs 1e-2, max rel 2e-2) with the output's own bf16
    rounding allowed on top, element by element: keys and values are
    code * scale, which bf16 cannot hold, so even a one-key context's
    output (= its V row) carries up to half an ulp, 0.0156 at |o| in [4, 8)."""
    g = got.float().cpu().double().numpy()
    assert np.isfinite(g).all(), "non-finite GPU output"
    d = np.abs(g - ref)
    excess = float((d - BF16_HALF_ULP * np.abs(ref)).max())
    rel = float(d.max()) / max(float(np.abs(ref).max()), 1e-30)
    assert excess <= ATOL and rel <= RTOL, f"abs excess {excess:.3e}, rel {rel:.3e}"
EDGE_CTX = [1, 2, 15, 16, 17, 100, 127, 128, 129, 255, 256, 257, 700, 1500]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_07_gb300 import build
    build.build()
    Q.load_library()


def oracle_fp8(w, ks=KS, vs=VS, extras=None):
    """Append into the host copies of the e4m3 caches, then attention."""
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    qkv = u16(w.qkv)
    kc = w.k_cache.numpy().copy()
    vc = w.v_cache.numpy().copy()
    table = oracle.rope_table(w.theta, w.max_pos, D)
    ex = extras or {}
    e1 = oracle.rope_cache_append_fp8(qkv, w.positions, w.slot_mapping, kc, vc, table, H, Hkv,
                                      D, BS, ks, vs, bias=ex.get("bias"),
                                      q_norm_w=ex.get("q_norm"), k_norm_w=ex.get("k_norm"))
    q = np.ascontiguousarray(qkv[:, :H * D])
    cu = None if w.is_decode else w.cu_seqlens_q
    out, e2 = oracle.paged_attention_fp8(q, kc, vc, ks, vs, w.block_tables, w.context_lens,
                                         H, Hkv, D, BS, cu_seqlens_q=cu)
    return qkv, kc, vc, out, e1, e2


class Fp8Run:
    def __init__(self, w, ks=KS, vs=VS, dev="cuda:0"):
        self.w, self.ks, self.vs = w, ks, vs
        self.dev = torch.device(dev)
        self.g = W.to_device(w, self.dev)
        self.dims = Q.make_dims(w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
        self.table = device_table(w.max_pos, w.theta, str(self.dev))
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.max_ctx = max(1, w.max_context_len)
        n = Q.qattn_paged_decode_workspace_size(w.num_seqs, self.max_ctx, self.dims)
        self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.dev)
        self.out = torch.empty((w.num_tokens, w.num_heads, w.head_dim), dtype=torch.bfloat16,
                               device=self.dev)

    def append(self, extras=None):
        g, ex = self.g, {k: v.to(self.dev) for k, v in (extras or {}).items()}
        Q.qattn_rope_cache_append_fp8(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                      g.slot_mapping, g.k_cache, g.v_cache, self.table, self.ks,
                                      self.vs, self.dims, qkv_bias=ex.get("bias"),
                                      q_norm_weight=ex.get("q_norm"),
                                      k_norm_weight=ex.get("k_norm"), err_word=self.err)
        return self

    def decode(self):
        g = self.g
        Q.qattn_paged_decode_fp8(self.out, g.q_view(), g.k_cache, g.v_cache, g.block_tables,
                                 g.context_lens, self.max_ctx, self.ks, self.vs, self.dims,
                                 self.ws, self.err)
        return self

    def varlen(self, num_prefill_seqs=None):
        g, w = self.g, self.w
        npf = sum(1 for n in w.q_lens if n >= 2) if num_prefill_seqs is None else num_prefill_seqs
        n = Q.qattn_varlen_prefill_fp8_workspace_size(w.num_seqs, npf, self.max_ctx, self.dims)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=self.dev)
        Q.qattn_varlen_prefill_fp8(self.out, g.q_view(), g.cu_seqlens_q, w.max_q_len, g.k_cache,
                                   g.v_cache, g.block_tables, g.context_lens, self.max_ctx, npf,
                                   self.ks, self.vs, self.dims, ws, self.err)
        return self

    def sync(self):
        torch.cuda.synchronize(self.dev)
        return self


@pytest.mark.parametrize("bs", [16, 64])
def test_append_fp8_bit_exact(bs):
    w = W.with_fp8_cache(W.custom(28, 4, ctx=EDGE_CTX, q_lens=[1] * len(EDGE_CTX), seed=800 + bs,
                                  block_size=bs))
    qkv, kc, vc, _, e1, _ = oracle_fp8(w)
    r = Fp8Run(w).append().sync()
    assert int(r.err.item()) == 0 and e1 == 0
    assert np.array_equal(u16(r.g.qkv), qkv)
    assert np.array_equal(r.g.k_cache.cpu().numpy(), kc)
    assert np.array_equal(r.g.v_cache.cpu().numpy(), vc)


def test_append_fp8_with_bias_and_norm_bit_exact():
    w = W.with_fp8_cache(W.custom(16, 8, ctx=[5, 40, 300], q_lens=[5, 3, 64], seed=810))
    gen = torch.Generator().manual_seed(811)
    H, Hkv, D = 16, 8, 128
    extras = {"bias": (torch.randn((H + 2 * Hkv) * D, generator=gen) * 0.5).to(torch.bfloat16),
              "q_norm": (1 + 0.1 * torch.randn(D, generator=gen)).to(torch.bfloat16),
              "k_norm": (1 + 0.1 * torch.randn(D, generator=gen)).to(torch.bfloat16)}
    host = {k: u16(v) for k, v in extras.items()}
    qkv, kc, vc, _, e1, _ = oracle_fp8(w, extras=host)
    r = Fp8Run(w).append(extras).sync()
    assert int(r.err.item()) == 0 and (e1 & ~oracle.ERR_NORM_INEXACT) == 0
    assert np.array_equal(u16(r.g.qkv), qkv)
    assert np.array_equal(r.g.k_cache.cpu().numpy(), kc)
    assert np.array_equal(r.g.v_cache.cpu().numpy(), vc)


def test_append_fp8_saturates_and_scales():
    """Large values saturate to +-448 codes; other scales change the codes
    exactly as the oracle does."""
    w = W.custom(4, 2, ctx=[3, 20], q_lens=[3, 1], seed=812)
    w.qkv.mul_(40)                           # |x| / scale far past 448
    w = W.with_fp8_cache(w)
    saturated = []
    for ks, vs in [(KS, VS), (0.5, 3.0)]:
        qkv, kc, vc, _, e1, _ = oracle_fp8(w, ks, vs)
        r = Fp8Run(w, ks, vs).append().sync()
        assert np.array_equal(r.g.k_cache.cpu().numpy(), kc)
        assert np.array_equal(r.g.v_cache.cpu().numpy(), vc)
        saturated.append(bool(((kc & 0x7F) == 0x7E).any()))
    assert saturated == [True, False]


@pytest.mark.parametrize("bs", [16, 32, 64])
@pytest.mark.parametrize("group,kv", [(1, 8), (2, 8), (7, 4), (8, 2)])
def test_decode_fp8(bs, group, kv):
    w = W.with_fp8_cache(W.custom(group * kv, kv, ctx=EDGE_CTX, q_lens=[1] * len(EDGE_CTX),
                                  seed=820 + bs + group, block_size=bs))
    _, _, _, ref, _, e2 = oracle_fp8(w)
    r = Fp8Run(w).append().decode().sync()
    assert int(r.err.item()) == 0 and e2 == 0
    assert_close(r.out, ref)


def test_decode_fp8_long_split_and_scales():
    """Split-KV parts and the merge; k_scale moves the logits, v_scale the
    output."""
    ctx = [5000, 4096, 129, 2000]
    base = W.custom(28, 4, ctx=ctx, q_lens=[1] * 4, seed=830)
    for ks, vs in [(KS, VS), (0.004, 0.05)]:
        w = W.with_fp8_cache(base, ks, vs)
        _, _, _, ref, _, _ = oracle_fp8(w, ks, vs)
        r = Fp8Run(w, ks, vs).append().decode().sync()
        assert int(r.err.item()) == 0
        assert_close(r.out, ref)


@pytest.mark.parametrize("group,kv", [(7, 4), (8, 2), (1, 8)])
def test_decode_fp8_query_magnitude_per_head(group, kv):
    """Query heads whose magnitudes differ by up to 2^16, and all-zero heads:
    the decode takes the dot products on the e4m3 codes, with q split into
    two e4m3 parts under a power-of-two scale of its own per head."""
    ctx = [1, 17, 100, 700, 1500, 129, 3000]
    w = W.with_fp8_cache(W.custom(group * kv, kv, ctx=ctx, q_lens=[1] * len(ctx),
                                  seed=840 + group))
    H, D = w.num_heads, w.head_dim
    exps = [-12, -3, 0, 2, 4, None]
    with torch.no_grad():
        for h in range(H):
            e = exps[h % len(exps)]
            cols = w.qkv[:, h * D:(h + 1) * D]
            if e is None:
                cols.zero_()
            else:
                cols.mul_(2.0 ** e)  # exact in bf16: a power of two
    _, _, _, ref, _, e2 = oracle_fp8(w)
    r = Fp8Run(w).append().decode().sync()
    assert int(r.err.item()) == 0 and e2 == 0
    assert_close(r.out, ref)


def test_decode_fp8_workload_b64_and_deterministic():
    w = W.with_fp8_cache(W.build(1))
    _, _, _, ref, _, _ = oracle_fp8(w)
    r = Fp8Run(w).append().decode().sync()
    assert int(r.err.item()) == 0
    assert_close(r.out, ref)
    first = r.out.clone()
    r.decode().sync()
    assert torch.equal(r.out, first)


def test_decode_fp8_bad_scale_rejected():
    w = W.with_fp8_cache(W.custom(8, 2, ctx=[10], q_lens=[1], seed=840))
    r = Fp8Run(w)
    for ks in (0.0, -1.0, float("nan"), float("inf")):
        r.ks = ks
        with pytest.raises(Q.QattnError):
            r.decode()


def test_varlen_fp8_mixed_workload():
    """4 prefill chunks of 512 on 0-1536 cached tokens + 60 decode rows."""
    w = W.with_fp8_cache(W.build(2))
    _, _, _, ref, _, e2 = oracle_fp8(w)
    r = Fp8Run(w).append().varlen().sync()
    assert int(r.err.item()) == 0 and e2 == 0
    assert_close(r.out, ref)


@pytest.mark.parametrize("bs", [16, 64])
def test_varlen_fp8_ragged(bs):
    ctx = [300, 700, 64, 1, 129, 900, 2, 40]
    q_lens = [200, 33, 64, 1, 1, 130, 2, 1]
    w = W.with_fp8_cache(W.custom(28, 4, ctx=ctx, q_lens=q_lens, seed=850 + bs, block_size=bs))
    _, _, _, ref, _, e2 = oracle_fp8(w)
    r = Fp8Run(w).append().varlen().sync()
    assert int(r.err.item()) == 0 and e2 == 0
    assert_close(r.out, ref)


def test_varlen_fp8_capacity_exceeded_sets_error():
    w = W.with_fp8_cache(W.custom(8, 2, ctx=[100, 200, 50], q_lens=[10, 20, 5], seed=860))
    _, _, _, ref, _, _ = oracle_fp8(w)
    r = Fp8Run(w).append().varlen(num_prefill_seqs=2).sync()
    assert int(r.err.item()) & Q.DEVERR_CONTEXT
    # the first two prefill sequences are still right
    rows = slice(0, 30)
    g = r.out.float().cpu().double().numpy()[rows]
    d = np.abs(g - ref[rows]) - BF16_HALF_ULP * np.abs(ref[rows])
    assert float(d.max()) <= ATOL


def run_prefix_fp8(r, prefix):
    g, w = r.g, r.w
    n = Q.qattn_paged_decode_shared_prefix_fp8_workspace_size(w.num_seqs, r.max_ctx, prefix,
                                                              r.dims)
    ws = torch.empty(n, dtype=torch.uint8, device=r.dev)
    Q.qattn_paged_decode_shared_prefix_fp8(r.out, g.q_view(), g.k_cache, g.v_cache,
                                           g.block_tables, g.context_lens, r.max_ctx, prefix,
                                           r.ks, r.vs, r.dims, ws, r.err)
    return r.sync()


def test_shared_prefix_fp8_workload():
    """128 sequences on a 2048-token shared prefix (Qwen3-0.6B heads)."""
    w = W.with_fp8_cache(W.build(4))
    _, _, _, ref, _, e2 = oracle_fp8(w)
    r = run_prefix_fp8(Fp8Run(w).append().sync(), w.shared_prefix_tokens)
    assert int(r.err.item()) == 0 and e2 == 0
    assert_close(r.out, ref)


@pytest.mark.parametrize("group,kv,prefix,bs", [(1, 4, 16, 16), (7, 4, 400, 16),
                                               (8, 2, 1024, 32), (2, 8, 192, 64)])
def test_shared_prefix_fp8(group, kv, prefix, bs):
    suffix = [1, 2, 15, 16, 17, 100, 128, 129, 300, 64]
    ctx = [prefix + s_ for s_ in suffix]
    w = W.with_fp8_cache(W.custom(group * kv, kv, ctx=ctx, q_lens=[1] * len(ctx),
                                  seed=870 + group + bs, shared_prefix_tokens=prefix,
                                  block_size=bs))
    _, _, _, ref, _, e2 = oracle_fp8(w)
    r = run_prefix_fp8(Fp8Run(w).append().sync(), prefix)
    assert int(r.err.item()) == 0 and e2 == 0
    assert_close(r.out, ref)


def test_shared_prefix_fp8_table_mismatch_flagged():
    w = W.with_fp8_cache(W.custom(16, 8, ctx=[300, 400], q_lens=[1, 1], seed=880,
                                  shared_prefix_tokens=256))
    w.block_tables[1, 3] = w.block_tables[1, 20]    # second table leaves the prefix
    r = run_prefix_fp8(Fp8Run(w).append().sync(), 256)
    assert int(r.err.item()) & Q.DEVERR_PREFIX


def test_decode_fp8_error_bits():
    """A bad context or block id flags its bit and leaves the other rows
    right (the same device-side checks as the bf16 path)."""
    w = W.with_fp8_cache(W.build(0))
    _, _, _, ref, _, _ = oracle_fp8(w)
    r = Fp8Run(w).append().sync()
    r.g.context_lens[1] = 0                     # invalid context: zero row
    r.g.block_tables[2, 3] = w.num_blocks + 9   # bad block id
    r.decode().sync()
    bits = int(r.err.item())
    assert bits & Q.DEVERR_CONTEXT and bits & Q.DEVERR_BLOCK and not bits & Q.DEVERR_TIMEOUT
    assert torch.count_nonzero(r.out[1]) == 0
    g = r.out.float().cpu().double().numpy()
    for row in (0, 3):
        d = np.abs(g[row] - ref[row]) - BF16_HALF_ULP * np.abs(ref[row])
        assert float(d.max()) <= ATOL


def test_fp8_step_graph_replay():
    """Append + FP8 decode + merge captured in a CUDA graph replays to the
    eager result."""
    w = W.with_fp8_cache(W.build(1))
    r = Fp8Run(w)
    qkv0 = r.g.qkv.clone()
    k0, v0 = r.g.k_cache.clone(), r.g.v_cache.clone()
    r.append().decode().sync()
    first = r.out.clone()
    s = torch.cuda.Stream(device=r.dev)
    s.wait_stream(torch.cuda.current_stream(r.dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            r.g.qkv.copy_(qkv0)
            r.g.k_cache.copy_(k0)
            r.g.v_cache.copy_(v0)
            r.append().decode()
    for _ in range(3):
        r.out.zero_()
        graph.replay()
        r.sync()
        assert int(r.err.item()) == 0
        assert torch.equal(r.out, first)
