"""GPU parity of the extended append (qattn_rope_cache_append_ex: qkv
projection bias and Qwen3 per-head q/k RMSNorm before RoPE) against the
oracle: bit-exact over the whole cache and the rotated queries.  The oracle's
RMSNorm sums the squares in fp64 in index order (the plain definition); the
kernel forms the exact sum in integers and rounds it to fp64 once, so the two
agree wherever the fp64 sum is exact.  N(0, 1) heads occasionally hold a
value below 2^-18 of their largest, where the fp64 sum rounds (the oracle
reports it, ERR_NORM_INEXACT); the sums then differ by a few fp64 ulps,
which reach the bf16 output only if fp32(ss / 128 + eps) sits on a rounding
boundary -- the tests still require bit equality there."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import GpuRun, assert_close, u16

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))   # the value the library sees as a C float


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_07_gb300 import build
    build.build()
    Q.load_library()


def extras(w, seed, bias=True, norm=True):
    g = torch.Generator().manual_seed(seed)
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
    b = (0.5 * torch.randn((H + 2 * Hkv) * D, generator=g)).to(torch.bfloat16) if bias else None
    qn = (1.0 + 0.2 * torch.randn(D, generator=g)).to(torch.bfloat16) if norm else None
    kn = (1.0 + 0.2 * torch.randn(D, generator=g)).to(torch.bfloat16) if norm else None
    return b, qn, kn


def oracle_append_ex(w, b, qn, kn):
    qkv, kc, vc = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
    table = oracle.rope_table(w.theta, w.max_pos, w.head_dim)
    conv = [None if t is None else u16(t) for t in (b, qn, kn)]
    e = oracle.rope_cache_append_ex(qkv, w.positions, w.slot_mapping, kc, vc, table,
                                    w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                    bias=conv[0], q_norm_w=conv[1], k_norm_w=conv[2], eps=EPS)
    return qkv, kc, vc, e


def gpu_append_ex(r: GpuRun, b, qn, kn):
    g = r.g
    dev = [None if t is None else t.to(r.dev) for t in (b, qn, kn)]
    Q.qattn_rope_cache_append_ex(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                 g.slot_mapping, g.k_cache, g.v_cache, r.table, r.dims,
                                 qkv_bias=dev[0], q_norm_weight=dev[1], k_norm_weight=dev[2],
                                 norm_eps=EPS, err_word=r.err)
    return r.sync()


@pytest.mark.parametrize("idx,bias,norm", [(0, False, True), (0, True, True), (1, True, False),
                                          (2, True, True), (4, False, True)])
def test_append_ex_bit_exact(idx, bias, norm):
    w = W.build(idx)
    b, qn, kn = extras(w, 500 + idx, bias, norm)
    qkv, kc, vc, e = oracle_append_ex(w, b, qn, kn)
    r = gpu_append_ex(GpuRun(w), b, qn, kn)
    assert (e & ~oracle.ERR_NORM_INEXACT) == 0 and r.err_bits == 0
    assert np.array_equal(u16(r.g.k_cache), kc), "k_cache differs"
    assert np.array_equal(u16(r.g.v_cache), vc), "v_cache differs"
    assert np.array_equal(u16(r.g.qkv), qkv), "rotated q differs"


def test_append_ex_norm_wide_range_bit_exact():
    """Heads whose values span about 2^15 (a different power-of-two scale
    per element), exact zeros, and heads made only of bf16 subnormals: the
    kernel's integer sum of squares must meet the oracle's fp64 sum bit for
    bit wherever that sum is exact."""
    w = W.custom(16, 8, ctx=[40, 75, 130], q_lens=[5, 1, 3], seed=530)
    g = torch.Generator().manual_seed(531)
    T, width = w.qkv.shape
    z = torch.randn(T, width, generator=g)
    base = torch.sign(z) * (0.25 + z.abs())
    expo = torch.randint(-8, 4, (T, width), generator=g).float()
    x = base * torch.exp2(expo)
    x[torch.rand(T, width, generator=g) < 0.05] = 0.0
    # token 0: every head subnormal (|x| < 2^-126); token 1: q head 3 all zero
    x[0] = torch.randn(width, generator=g) * 2.0 ** -130
    x[1, 3 * 128:4 * 128] = 0.0
    w.qkv = x.to(torch.bfloat16)
    b, qn, kn = extras(w, 532, bias=False, norm=True)
    qkv, kc, vc, e = oracle_append_ex(w, b, qn, kn)
    assert e == 0, "the oracle's fp64 sum of squares was not exact on this input"
    r = gpu_append_ex(GpuRun(w), b, qn, kn)
    assert r.err_bits == 0
    assert np.array_equal(u16(r.g.k_cache), kc), "k_cache differs"
    assert np.array_equal(u16(r.g.v_cache), vc), "v_cache differs"
    assert np.array_equal(u16(r.g.qkv), qkv), "rotated q differs"


def test_append_ex_all_null_equals_append():
    w = W.build(1)
    a = GpuRun(w).append().sync()
    b = gpu_append_ex(GpuRun(w), None, None, None)
    # bit patterns: unused slots hold a NaN sentinel
    assert np.array_equal(u16(a.g.k_cache), u16(b.g.k_cache))
    assert np.array_equal(u16(a.g.v_cache), u16(b.g.v_cache))
    assert np.array_equal(u16(a.g.qkv), u16(b.g.qkv))


def test_append_ex_then_decode_matches_oracle():
    """Qwen3-shaped step with q/k norms, then decode, against the oracle."""
    w = W.build(0)
    b, qn, kn = extras(w, 510, bias=False, norm=True)
    qkv, kc, vc, _ = oracle_append_ex(w, b, qn, kn)
    H, D = w.num_heads, w.head_dim
    ref, e2 = oracle.paged_attention(np.ascontiguousarray(qkv[:, :H * D]), kc, vc,
                                     w.block_tables, w.context_lens, H, w.num_kv_heads, D,
                                     w.block_size)
    r = gpu_append_ex(GpuRun(w), b, qn, kn).attend().sync()
    assert e2 == 0 and r.err_bits == 0
    assert_close(r.out, ref)


def test_append_ex_rejects_bad_args():
    w = W.build(0)
    r = GpuRun(w)
    g = r.g
    qn = torch.ones(128, dtype=torch.bfloat16, device=r.dev)
    with pytest.raises(Q.QattnError) as ei:
        Q.qattn_rope_cache_append_ex(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                     g.slot_mapping, g.k_cache, g.v_cache, r.table, r.dims,
                                     q_norm_weight=qn, norm_eps=-1.0, err_word=r.err)
    assert ei.value.status == Q.QATTN_ERR_INVALID_ARG
    with pytest.raises(Q.QattnError):
        Q.qattn_rope_cache_append_ex(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                     g.slot_mapping, g.k_cache, g.v_cache, r.table, r.dims,
                                     q_norm_weight=qn[1:], err_word=r.err)   # misaligned


def test_append_with_dynamic_ntk_table():
    """A dynamic-NTK table (factor 2, original 4096) covering 8192 positions:
    the append is bit-exact against the oracle with the oracle's table."""
    w = W.custom(16, 8, ctx=[8000, 5000, 4200, 300], q_lens=[3, 1, 2, 1], seed=520)
    table_h = Q.qattn_rope_table_build_scaled(8192, 128, w.theta, Q.QATTN_ROPE_SCALING_DYNAMIC,
                                              2.0, 4096)
    to = oracle.rope_table_scaled(w.theta, 8192, 128, oracle.SCALING_DYNAMIC, 2.0, 4096)
    assert np.array_equal(table_h.numpy().view(np.uint32), to.view(np.uint32))
    qkv, kc, vc = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
    e = oracle.rope_cache_append(qkv, w.positions, w.slot_mapping, kc, vc, to, 16, 8, 128, 16)
    r = GpuRun(w)
    g = r.g
    Q.qattn_rope_cache_append(g.q_view(), g.k_view(), g.v_view(), g.positions, g.slot_mapping,
                              g.k_cache, g.v_cache, table_h.to(r.dev), r.dims, r.err)
    r.sync()
    assert e == 0 and r.err_bits == 0
    assert np.array_equal(u16(r.g.k_cache), kc) and np.array_equal(u16(r.g.v_cache), vc)
    assert np.array_equal(u16(r.g.qkv), qkv)
