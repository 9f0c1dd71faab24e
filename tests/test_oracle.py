"""Pins for the CPU oracle (no GPU).

The oracle is only trusted once it agrees with something other than itself:
the configuration values the pages print (tests/golden), closed forms of the
rotation and of the softmax, invariants (rotation preserves the norm, the
relative-position identity, block relabelling, GQA == MHA on repeated heads,
split == unsplit), special cases (one key returns V, equal keys average V)
and a multiprecision brute force on tiny inputs.  Each pin is chosen so that
a plausible mistake -- a dropped scale, a wrong sign or pairing in the
rotation, a wrong head grouping, a transposed or mis-indexed gather, a
wrong causal offset -- fails at least one of them.
"""
import cmath
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_07_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def bf16_of(x) -> np.ndarray:
    """Round fp64 values to bf16 payloads (via torch, an independent path)."""
    return u16(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def f64(u: np.ndarray) -> np.ndarray:
    return oracle.bf16_to_f64(u)


# ------------------------------------------------------------ golden ----

def test_golden_qwen2_7b_config_and_derived_shape():
    g = json.load(open(os.path.join(GOLDEN, "qwen2_7b_config.json")))
    head_dim = g["hidden_size"] // g["num_attention_heads"]
    assert head_dim == g["stated"]["head_dim"] == W.HEAD_DIM
    assert g["num_attention_heads"] // g["num_key_value_heads"] == g["stated"]["gqa_group"]
    assert W.QWEN2_7B == dict(num_heads=g["num_attention_heads"],
                              num_kv_heads=g["num_key_value_heads"])
    assert W.ROPE_THETA == g["rope_theta"] == g["stated"]["rope_theta_default"]
    assert W.MAX_POS == g["max_position_embeddings"]
    assert (head_dim ** -0.5) ** -2 == pytest.approx(g["stated"]["scaling_squared_inverse"])


def test_golden_qwen3_config():
    g = json.load(open(os.path.join(GOLDEN, "qwen3_0_6b_config.json")))
    assert W.QWEN3_0_6B == dict(num_heads=g["num_attention_heads"],
                                num_kv_heads=g["num_key_value_heads"])
    assert g["head_dim"] == W.HEAD_DIM


def test_fourteen_token_prefill_gives_fourteen_rows():
    """nano-vllm page section 5: 14 tokens at positions 0..13 -> 14 rows."""
    g = json.load(open(os.path.join(GOLDEN, "qwen3_0_6b_config.json")))["integration_check"]
    n = g["prefill_tokens"]
    w = W.custom(16, 8, ctx=[n], q_lens=[n], seed=3)
    qkv = u16(w.qkv)
    kc, vc = u16(w.k_cache), u16(w.v_cache)
    cs = oracle.rope_table(w.theta, 64, 128)
    assert oracle.rope_cache_append(qkv, w.positions, w.slot_mapping, kc, vc, cs,
                                    16, 8, 128, 16) == 0
    q = np.ascontiguousarray(qkv[:, :16 * 128])
    out, err = oracle.paged_attention(q, kc, vc, w.block_tables, w.context_lens,
                                      16, 8, 128, 16, cu_seqlens_q=w.cu_seqlens_q)
    assert err == 0 and out.shape == (g["rows_out"], 16, 128)
    # causal row 0 sees only key 0: it returns v_0 exactly
    v0 = f64(vc[int(w.block_tables[0, 0]), :, 0, :])  # [Hkv, D]
    assert np.array_equal(out[0], np.repeat(v0, 2, axis=0))


# ------------------------------------------------------------- table ----

def test_table_position_zero_is_identity():
    t = oracle.rope_table(1e6, 4, 128)
    assert np.all(t[0, :64] == 1.0) and np.all(t[0, 64:] == 0.0)


def test_table_first_frequency_is_one():
    """i = 0: theta^0 = 1, so column 0 is cos(pos) and column D/2 sin(pos)."""
    P = 32768
    t = oracle.rope_table(1e6, P, 128)
    pos = np.arange(P, dtype=np.float64)
    assert np.array_equal(t[:, 0], np.cos(pos).astype(np.float32))
    assert np.array_equal(t[:, 64], np.sin(pos).astype(np.float32))


def test_table_quarter_frequency_closed_form():
    """i = D/4: theta^(-1/2) = 1e-3 for theta = 1e6 (and 1e-2 for 1e4)."""
    for theta, f in ((1e6, 1e-3), (1e4, 1e-2)):
        t = oracle.rope_table(theta, 4096, 128)
        pos = np.arange(4096, dtype=np.float64)
        np.testing.assert_allclose(t[:, 32], np.cos(pos * f), rtol=0, atol=2e-7)
        np.testing.assert_allclose(t[:, 96], np.sin(pos * f), rtol=0, atol=2e-7)


def test_theta_pitfall_changes_table():
    """The pages' pitfall: rope_theta 1e4 instead of 1e6 gives other angles."""
    a = oracle.rope_table(1e6, 256, 128)
    b = oracle.rope_table(1e4, 256, 128)
    assert np.array_equal(a[:, 0], b[:, 0])           # frequency 1 in both
    assert np.count_nonzero(a[1:, 1:64] != b[1:, 1:64]) > 0.99 * 255 * 63


# -------------------------------------------------------------- RoPE ----

def test_rope_d2_is_complex_multiplication():
    """D = 2: rotate-half is x1 + i x2 times e^(i pos)."""
    rng = np.random.default_rng(0)
    for _ in range(50):
        x = rng.standard_normal(2)
        pos = float(rng.integers(0, 32768))
        y = oracle.rope_head_f64(x, pos, 1e6)
        z = complex(x[0], x[1]) * cmath.exp(1j * pos)
        assert abs(y[0] - z.real) < 1e-12 and abs(y[1] - z.imag) < 1e-12


def test_rope_pairs_i_with_i_plus_half():
    """One-hot inputs: e_i only mixes with e_{i+D/2}, with the signs of a
    counter-clockwise rotation."""
    D, pos = 8, 5.0
    for i in range(D // 2):
        c = math.cos(pos * 1e6 ** (-2 * i / D))
        s = math.sin(pos * 1e6 ** (-2 * i / D))
        e = np.zeros(D); e[i] = 1.0
        y = oracle.rope_head_f64(e, pos, 1e6)
        want = np.zeros(D); want[i] = c; want[i + D // 2] = s
        np.testing.assert_allclose(y, want, atol=1e-15)
        e = np.zeros(D); e[i + D // 2] = 1.0
        y = oracle.rope_head_f64(e, pos, 1e6)
        want = np.zeros(D); want[i] = -s; want[i + D // 2] = c
        np.testing.assert_allclose(y, want, atol=1e-15)


def test_rope_preserves_norm():
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.standard_normal(128)
        y = oracle.rope_head_f64(x, float(rng.integers(0, 32768)), 1e6)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12


def test_rope_relative_position_identity():
    """rot(q, m) . rot(k, n) depends only on m - n."""
    rng = np.random.default_rng(2)
    for _ in range(40):
        q, k = rng.standard_normal(128), rng.standard_normal(128)
        m, n, s = (float(v) for v in rng.integers(0, 16384, 3))
        a = oracle.rope_head_f64(q, m, 1e6) @ oracle.rope_head_f64(k, n, 1e6)
        b = oracle.rope_head_f64(q, m + s, 1e6) @ oracle.rope_head_f64(k, n + s, 1e6)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


def test_rope_exact_position_zero_keeps_bits():
    g = torch.Generator().manual_seed(4)
    x = u16(torch.randn(128, generator=g).to(torch.bfloat16))
    row = oracle.rope_table(1e6, 1, 128)[0]
    assert np.array_equal(oracle.rope_head_exact(x, row), x)


def test_rope_exact_within_fp32_bound_of_f64():
    """The fp32 recipe lands within half a bf16 ulp of the exact rotation of
    the same bf16 input plus the fp32 error of its two products and the
    table's rounding (bounded by 4 * 2^-24 * (|x1 c| + |x2 s|))."""
    g = torch.Generator().manual_seed(5)
    t = oracle.rope_table(1e6, 32768, 128)
    for pos in [1, 2, 3, 100, 4095, 17000, 32767]:
        xb = u16(torch.randn(128, generator=g).to(torch.bfloat16))
        y = f64(oracle.rope_head_exact(xb, t[pos]))
        x = f64(xb)
        ref = oracle.rope_head_f64(x, float(pos), 1e6)
        mag = np.abs(np.concatenate([x[:64], x[64:]])) + np.abs(np.concatenate([x[64:], x[:64]]))
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) * 2 ** 16
        bound = 0.5 * ulp + 4 * 2.0 ** -24 * mag
        assert np.all(np.abs(y - ref) <= bound), pos


# ------------------------------------------------------------ append ----

def test_append_hand_example():
    """2 blocks of 16, one KV head, D = 8; tokens at position 0 (rotation is
    the identity there) go to slots 17, 0, 31; a padding token (slot -1)
    writes nothing.  Every other cache entry keeps the sentinel."""
    H, Hkv, D, BS = 2, 1, 8, 16
    g = torch.Generator().manual_seed(6)
    qkv = u16(torch.randn(4, (H + 2 * Hkv) * D, generator=g).to(torch.bfloat16))
    q_before = qkv[:, :H * D].copy()
    kc = np.full((2, Hkv, BS, D), W.SENTINEL_BF16, dtype=np.uint16)
    vc = kc.copy()
    table = oracle.rope_table(1e6, 8, D)
    err = oracle.rope_cache_append(qkv, np.zeros(4, np.int32),
                                   np.array([17, 0, 31, -1], np.int32),
                                   kc, vc, table, H, Hkv, D, BS)
    assert err == 0
    want_k = np.full_like(kc, W.SENTINEL_BF16)
    want_v = want_k.copy()
    for t, (blk, off) in enumerate([(1, 1), (0, 0), (1, 15)]):
        want_k[blk, 0, off] = qkv[t, H * D:(H + 1) * D]
        want_v[blk, 0, off] = qkv[t, (H + 1) * D:]
    assert np.array_equal(kc, want_k) and np.array_equal(vc, want_v)
    assert np.array_equal(qkv[:, :H * D], q_before)


def test_append_rotates_k_and_q_at_position():
    H, Hkv, D, BS = 2, 2, 128, 16
    g = torch.Generator().manual_seed(7)
    qkv = u16(torch.randn(3, (H + 2 * Hkv) * D, generator=g).to(torch.bfloat16))
    orig = qkv.copy()
    kc = np.full((3, Hkv, BS, D), W.SENTINEL_BF16, dtype=np.uint16)
    vc = kc.copy()
    table = oracle.rope_table(1e6, 100, D)
    pos = np.array([5, 99, 40], np.int32)
    slots = np.array([33, 2, 47], np.int32)
    assert oracle.rope_cache_append(qkv, pos, slots, kc, vc, table, H, Hkv, D, BS) == 0
    for t in range(3):
        for h in range(H):
            want = oracle.rope_head_exact(orig[t, h * D:(h + 1) * D], table[pos[t]])
            assert np.array_equal(qkv[t, h * D:(h + 1) * D], want)
        blk, off = divmod(int(slots[t]), BS)
        for gh in range(Hkv):
            kin = orig[t, (H + gh) * D:(H + gh + 1) * D]
            assert np.array_equal(kc[blk, gh, off], oracle.rope_head_exact(kin, table[pos[t]]))
            assert np.array_equal(vc[blk, gh, off], orig[t, (H + Hkv + gh) * D:(H + Hkv + gh + 1) * D])
    assert np.array_equal(qkv[:, H * D:], orig[:, H * D:])   # k, v rows untouched


def test_append_error_bits():
    H, Hkv, D, BS = 1, 1, 8, 16
    qkv = np.zeros((3, 3 * D), np.uint16)
    kc = np.full((1, 1, BS, D), W.SENTINEL_BF16, np.uint16)
    vc = kc.copy()
    table = oracle.rope_table(1e6, 10, D)
    err = oracle.rope_cache_append(qkv, np.array([0, 10, 1], np.int32),
                                   np.array([16, 0, 3], np.int32), kc, vc, table,
                                   H, Hkv, D, BS)
    assert err == oracle.ERR_SLOT | oracle.ERR_POSITION
    assert np.all(kc[0, 0, 0] == W.SENTINEL_BF16)    # bad-position token skipped
    assert np.all(kc[0, 0, 3] == 0)                   # good token written


def test_theta_pitfall_changes_cache():
    w = W.build(0)
    outs = []
    for theta in (1e6, 1e4):
        qkv, kc, vc = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
        table = oracle.rope_table(theta, 256, 128)
        oracle.rope_cache_append(qkv, w.positions, w.slot_mapping, kc, vc, table,
                                 16, 8, 128, 16)
        outs.append(kc)
    assert not np.array_equal(outs[0], outs[1])


# ------------------------------------------------------- rope_scaling ----

def test_scaled_table_reduces_to_plain():
    plain = oracle.rope_table(1e6, 300, 128)
    assert np.array_equal(oracle.rope_table_scaled(1e6, 300, 128, oracle.SCALING_NONE), plain)
    assert np.array_equal(oracle.rope_table_scaled(1e6, 300, 128, oracle.SCALING_LINEAR, 1.0),
                          plain)
    # dynamic NTK leaves a table within the original length untouched
    assert np.array_equal(
        oracle.rope_table_scaled(1e6, 300, 128, oracle.SCALING_DYNAMIC, 2.0, 4096), plain)


def test_linear_scaling_is_position_interpolation():
    plain = oracle.rope_table(1e6, 400, 128)
    for f in (2, 4):
        t = oracle.rope_table_scaled(1e6, 400 * f, 128, oracle.SCALING_LINEAR, float(f))
        assert np.array_equal(t[::f], plain)         # row f*k == plain row k, bit for bit


def test_dynamic_ntk_base_closed_form():
    """factor 2, original 4096, a table of 8192 rows: base' = theta * 3^(D/(D-2)).
    Frequency 0 stays 1; the lowest frequency theta^(-(D-2)/D) is divided by
    exactly (2 * 8192/4096 - 1) = 3."""
    D, theta = 128, 1e6
    t = oracle.rope_table_scaled(theta, 8192, D, oracle.SCALING_DYNAMIC, 2.0, 4096)
    plain = oracle.rope_table(theta, 8192, D)
    assert np.array_equal(t[:, 0], plain[:, 0])       # cos(pos) at frequency 1
    lowest = theta ** (-(D - 2) / D)
    ang = np.arctan2(t[1:50, D - 1].astype(np.float64), t[1:50, D // 2 - 1].astype(np.float64))
    assert np.allclose(ang / np.arange(1, 50), lowest / 3.0, rtol=1e-5)
    # and a longer table gets a larger base (lower frequency)
    t2 = oracle.rope_table_scaled(theta, 16384, D, oracle.SCALING_DYNAMIC, 2.0, 4096)
    assert t2[1, D - 1] < t[1, D - 1]


def test_scaled_table_rejects_bad_args():
    for args in [(1e6, 10, 128, 3, 2.0, 4096), (1e6, 10, 128, 1, 0.5, 0),
                 (1e6, 10, 128, 2, 2.0, 0), (1e6, 10, 2, 1, 2.0, 0)]:
        with pytest.raises(ValueError):
            oracle.rope_table_scaled(*args)


# --------------------------------- qkv bias, Qwen3 per-head RMSNorm ----

def test_bias_add_rounds_once_to_nearest_even():
    one = bf16_of([1.0])[0]
    assert one == 0x3F80
    # 1 + 2^-8 is half an ulp above 1.0: ties to even -> 1.0
    assert oracle.add_bias_head(np.array([one]), bf16_of([2.0 ** -8]))[0] == 0x3F80
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: even -> 1 + 2^-6
    assert oracle.add_bias_head(np.array([one]), bf16_of([3 * 2.0 ** -8]))[0] == 0x3F82
    g = torch.Generator().manual_seed(11)
    x = u16(torch.randn(300, generator=g).to(torch.bfloat16))
    assert np.array_equal(oracle.add_bias_head(x, np.zeros_like(x)), x)      # zero bias
    neg = x ^ np.uint16(0x8000)                                              # b = -x
    assert np.all(f64(oracle.add_bias_head(x, neg)) == 0.0)
    # against fp64 addition then bf16 rounding (exact sums for these values)
    b = u16(torch.randn(300, generator=g).to(torch.bfloat16))
    assert np.array_equal(oracle.add_bias_head(x, b), bf16_of(f64(x) + f64(b)))


def test_rmsnorm_closed_forms():
    D = 128
    w1 = bf16_of(np.ones(D))
    two = bf16_of(np.full(D, 2.0))
    # constant 2.0: mean(x^2) = 4, r = 1/2 exactly, y = 1.0 exactly
    assert np.all(f64(oracle.rmsnorm_head(two, w1, 0.0)) == 1.0)
    # ... and y_i = w_i exactly for any weights
    g = torch.Generator().manual_seed(12)
    w = u16(torch.randn(D, generator=g).to(torch.bfloat16))
    assert np.array_equal(oracle.rmsnorm_head(two, w, 0.0), w)
    # sign is kept per element
    alt = bf16_of(np.where(np.arange(D) % 2 == 0, 2.0, -2.0))
    assert np.array_equal(f64(oracle.rmsnorm_head(alt, w1, 0.0)),
                          np.where(np.arange(D) % 2 == 0, 1.0, -1.0))
    # the zero vector stays zero with eps > 0 (no 0/0)
    z = np.zeros(D, np.uint16)
    assert np.all(f64(oracle.rmsnorm_head(z, w1, 1e-6)) == 0.0)


def test_rmsnorm_scale_invariance_and_unit_rms():
    D = 128
    g = torch.Generator().manual_seed(13)
    x = torch.randn(D, generator=g).to(torch.bfloat16)
    w1 = bf16_of(np.ones(D))
    y = oracle.rmsnorm_head(u16(x), w1, 0.0)
    for k in (-6, -1, 3, 9):          # power-of-two scaling is exact in bf16 and fp32
        assert np.array_equal(oracle.rmsnorm_head(u16(x * (2.0 ** k)), w1, 0.0), y)
    yv = f64(y)
    assert abs(np.sqrt(np.mean(yv * yv)) - 1.0) < 4e-3       # unit RMS up to bf16 rounding
    # the defining formula in fp64, within one bf16 rounding of the output
    xv = f64(u16(x))
    wv = f64(u16(torch.randn(D, generator=g).to(torch.bfloat16)))
    ref = xv / np.sqrt(np.mean(xv * xv) + 1e-6) * wv
    got = f64(oracle.rmsnorm_head(u16(x), bf16_of(wv), 1e-6))
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_rmsnorm_against_40_digit_arithmetic():
    """The defining formula y = x / sqrt(mean(x^2) + eps) * w evaluated with
    40-digit arithmetic on small integer-valued heads (and the same heads
    scaled by 2^-10, where eps = fp32(1e-6) is about 5% of mean(x^2)): the
    oracle's fp32 steps stay within 2^-21 relative of the exact value, so its
    bf16 result is the exact value's bf16 rounding up to that margin."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(21)
    D = 128
    eps32 = float(np.float32(1e-6))
    mismatched = 0
    for scale_exp in (0, -10):
        for _ in range(6):
            xi = rng.integers(-8, 9, D).astype(np.float64) * 2.0 ** scale_exp
            wi = rng.integers(-6, 7, D).astype(np.float64) / 4.0
            x, w = bf16_of(xi), bf16_of(wi)
            assert np.array_equal(f64(x), xi) and np.array_equal(f64(w), wi)
            y, exact = oracle.rmsnorm_head(x, w, 1e-6, with_exactness=True)
            assert exact
            ms = mp.fsum(mp.mpf(float(v)) ** 2 for v in xi) / D
            r = 1 / mp.sqrt(ms + mp.mpf(eps32))
            got = f64(y)
            for i in range(D):
                ref = mp.mpf(float(xi[i])) * r * mp.mpf(float(wi[i]))
                err = abs(mp.mpf(float(got[i])) - ref)
                assert err <= (2.0 ** -8 + 2.0 ** -21) * abs(ref) + mp.mpf(10) ** -30
                if got[i] != f64(bf16_of([float(ref)]))[0]:
                    mismatched += 1
    # only values within 2^-21 of a bf16 rounding boundary may round the other way
    assert mismatched <= 4


def test_rmsnorm_reports_an_inexact_sum_of_squares():
    """The reading needs the exact sum of squares; the oracle says when fp64
    could not hold it (magnitudes spanning ~2^60) and holds it otherwise."""
    D = 128
    w1 = bf16_of(np.ones(D))
    g = torch.Generator().manual_seed(22)
    x = u16(torch.randn(D, generator=g).to(torch.bfloat16))
    assert oracle.rmsnorm_head(x, w1, 1e-6, with_exactness=True)[1]
    wide = np.concatenate([np.full(D // 2, 1.0), np.full(D // 2, 1.0 + 2.0 ** -7) * 2.0 ** -60])
    _, exact = oracle.rmsnorm_head(bf16_of(wide), w1, 1e-6, with_exactness=True)
    assert not exact


def test_append_ex_without_extras_equals_append():
    w = W.build(0)
    a_qkv, a_kc, a_vc = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
    b_qkv, b_kc, b_vc = a_qkv.copy(), a_kc.copy(), a_vc.copy()
    table = oracle.rope_table(1e6, w.max_pos, 128)
    e1 = oracle.rope_cache_append(a_qkv, w.positions, w.slot_mapping, a_kc, a_vc, table,
                                  16, 8, 128, 16)
    e2 = oracle.rope_cache_append_ex(b_qkv, w.positions, w.slot_mapping, b_kc, b_vc, table,
                                     16, 8, 128, 16)
    assert e1 == e2 == 0
    assert np.array_equal(a_qkv, b_qkv) and np.array_equal(a_kc, b_kc)
    assert np.array_equal(a_vc, b_vc)


def test_append_ex_bias_goes_to_the_right_head():
    """A bias that is nonzero only on kv head 1 of k changes only that head
    in the cache, by bias-then-rope of the raw k."""
    H, Hkv, D, BS = 4, 2, 128, 16
    g = torch.Generator().manual_seed(14)
    qkv0 = u16(torch.randn(3, (H + 2 * Hkv) * D, generator=g).to(torch.bfloat16))
    pos = np.array([0, 7, 30], np.int32)
    slots = np.array([3, 20, 41], np.int32)
    table = oracle.rope_table(1e6, 64, D)
    bias = np.zeros((H + 2 * Hkv) * D, np.uint16)
    bias[(H + 1) * D:(H + 2) * D] = bf16_of(np.linspace(-1, 1, D))
    runs = []
    for bb in (None, bias):
        qkv = qkv0.copy()
        kc = np.full((3, Hkv, BS, D), W.SENTINEL_BF16, np.uint16)
        vc = kc.copy()
        assert oracle.rope_cache_append_ex(qkv, pos, slots, kc, vc, table, H, Hkv, D, BS,
                                           bias=bb) == 0
        runs.append((qkv, kc, vc))
    (q0, k0, v0), (q1, k1, v1) = runs
    assert np.array_equal(q0, q1) and np.array_equal(v0, v1)
    assert np.array_equal(k0[:, 0], k1[:, 0])
    for t in range(3):
        blk, off = divmod(int(slots[t]), BS)
        kin = qkv0[t, (H + 1) * D:(H + 2) * D]
        want = oracle.rope_head_exact(oracle.add_bias_head(kin, bias[(H + 1) * D:(H + 2) * D]),
                                      table[pos[t]])
        assert np.array_equal(k1[blk, 1, off], want)


def test_append_ex_norm_then_rope_has_unit_rms():
    """With unit weights, a normalised head rotated by RoPE keeps RMS 1 (RoPE
    preserves the norm), for q in place and k in the cache."""
    H, Hkv, D, BS = 2, 1, 128, 16
    g = torch.Generator().manual_seed(15)
    qkv = u16((3.0 * torch.randn(2, (H + 2 * Hkv) * D, generator=g)).to(torch.bfloat16))
    kc = np.full((1, Hkv, BS, D), W.SENTINEL_BF16, np.uint16)
    vc = kc.copy()
    table = oracle.rope_table(1e6, 100, D)
    w1 = bf16_of(np.ones(D))
    assert oracle.rope_cache_append_ex(qkv, np.array([17, 90], np.int32),
                                       np.array([4, 9], np.int32), kc, vc, table, H, Hkv, D,
                                       BS, q_norm_w=w1, k_norm_w=w1, eps=1e-6) == 0
    for t in range(2):
        for h in range(H):
            y = f64(qkv[t, h * D:(h + 1) * D])
            assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 8e-3
    for off in (4, 9):
        y = f64(kc[0, 0, off])
        assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 8e-3


# --------------------------------------------------------- attention ----

def _run_workload(w, theta=1e6, partition=0):
    qkv, kc, vc = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
    table = oracle.rope_table(theta, w.max_pos, D)
    assert oracle.rope_cache_append(qkv, w.positions, w.slot_mapping, kc, vc, table,
                                    H, Hkv, D, w.block_size) == 0
    q = np.ascontiguousarray(qkv[:, :H * D])
    cu = None if w.is_decode else w.cu_seqlens_q
    out, err = oracle.paged_attention(q, kc, vc, w.block_tables, w.context_lens, H,
                                      Hkv, D, w.block_size, cu_seqlens_q=cu,
                                      partition_tokens=partition)
    assert err == 0
    return out, kc, vc, q


def test_block_permutation_invariance():
    w = W.build(0)
    a, kca, _, _ = _run_workload(w)
    wp = W.permute_blocks(w, seed=11)
    b, kcb, _, _ = _run_workload(wp)
    assert np.array_equal(a, b)
    # logical cache identical: block x of one is block pi(x) of the other
    for bidx in range(w.num_seqs):
        for j in range(int(w.context_lens[bidx])):
            x = int(w.block_tables[bidx, j // 16])
            y = int(wp.block_tables[bidx, j // 16])
            assert np.array_equal(kca[x, :, j % 16], kcb[y, :, j % 16])


def _relayout(w, bs):
    """The same logical cache contents and new tokens in blocks of ``bs``
    tokens, placed in reverse order (a plain host copy, no oracle code)."""
    B, Hkv, D = w.num_seqs, w.num_kv_heads, w.head_dim
    need = [(int(L) + bs - 1) // bs for L in w.context_lens]
    pool = sum(need) + 1
    order = list(range(pool))[::-1]
    bt = np.zeros((B, max(need)), dtype=np.int32)
    used = 0
    for b, n in enumerate(need):
        bt[b, :n] = order[used:used + n]
        used += n
    kc = np.full((pool, Hkv, bs, D), 0x7FC1, dtype=np.uint16)
    vc = kc.copy()
    k0, v0 = u16(w.k_cache), u16(w.v_cache)
    slots = w.slot_mapping.numpy().astype(np.int32).copy()
    t = 0
    for b in range(B):
        L = int(w.context_lens[b])
        for j in range(L):
            x = int(w.block_tables[b, j // w.block_size])
            kc[bt[b, j // bs], :, j % bs] = k0[x, :, j % w.block_size]
            vc[bt[b, j // bs], :, j % bs] = v0[x, :, j % w.block_size]
        for i in range(w.q_lens[b]):
            p = L - w.q_lens[b] + i
            slots[t] = bt[b, p // bs] * bs + p % bs
            t += 1
    return kc, vc, bt, slots


@pytest.mark.parametrize("bs", [32, 64])
def test_block_size_invariance(bs):
    """16-, 32- and 64-token blocks holding the same tokens give the same
    append rows and bit-identical attention (prefill and decode rows)."""
    w = W.custom(8, 2, ctx=[5, 40, 100, 200], q_lens=[3, 1, 40, 1], seed=14)
    ref, kc16, vc16, _ = _run_workload(w)
    kc, vc, bt, slots = _relayout(w, bs)
    qkv = u16(w.qkv)
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
    table = oracle.rope_table(1e6, w.max_pos, D)
    assert oracle.rope_cache_append(qkv, w.positions, slots, kc, vc, table, H, Hkv, D, bs) == 0
    q = np.ascontiguousarray(qkv[:, :H * D])
    out, err = oracle.paged_attention(q, kc, vc, bt, w.context_lens, H, Hkv, D, bs,
                                      cu_seqlens_q=w.cu_seqlens_q)
    assert err == 0
    assert np.array_equal(out, ref)
    for b in range(w.num_seqs):
        for j in range(int(w.context_lens[b])):
            x = int(w.block_tables[b, j // 16])
            assert np.array_equal(kc[bt[b, j // bs], :, j % bs], kc16[x, :, j % 16])
            assert np.array_equal(vc[bt[b, j // bs], :, j % bs], vc16[x, :, j % 16])


def test_one_token_context_returns_v_exactly():
    w = W.custom(4, 2, ctx=[1, 1, 1], q_lens=[1, 1, 1], seed=12)
    out, kc, vc, _ = _run_workload(w)
    for b in range(3):
        v = f64(vc[int(w.block_tables[b, 0]), :, 0, :])
        assert np.array_equal(out[b], np.repeat(v, 2, axis=0))


def test_equal_keys_average_values():
    H, Hkv, D, BS, L = 2, 1, 128, 16, 37
    g = torch.Generator().manual_seed(13)
    k_row = u16(torch.randn(D, generator=g).to(torch.bfloat16))
    kc = np.tile(k_row, (3, Hkv, BS, 1)).astype(np.uint16)
    vc = u16(torch.randn(3, Hkv, BS, D, generator=g).to(torch.bfloat16))
    q = u16(torch.randn(1, H * D, generator=g).to(torch.bfloat16))
    bt = np.array([[2, 0, 1]], np.int32)
    out, err = oracle.paged_attention(q, kc, vc, bt, np.array([L], np.int32), H, Hkv, D, BS)
    vals = np.stack([f64(vc[bt[0, j // BS], 0, j % BS]) for j in range(L)])
    np.testing.assert_allclose(out[0, 0], vals.mean(axis=0), rtol=0, atol=1e-13)
    np.testing.assert_allclose(out[0, 1], vals.mean(axis=0), rtol=0, atol=1e-13)


def _gather_contiguous(w, kc, vc, b):
    L = int(w.context_lens[b])
    idx = [(int(w.block_tables[b, j // 16]), j % 16) for j in range(L)]
    k = np.stack([kc[x, :, o] for x, o in idx])   # [L, Hkv, D]
    v = np.stack([vc[x, :, o] for x, o in idx])
    return np.ascontiguousarray(k), np.ascontiguousarray(v)


def test_paged_equals_contiguous():
    w = W.build(0)
    out, kc, vc, q = _run_workload(w)
    for b in range(w.num_seqs):
        k, v = _gather_contiguous(w, kc, vc, b)
        ref = oracle.contiguous_attention(q[b:b + 1].reshape(1, 16, 128), k, v, 16, 8, 128)
        assert np.array_equal(out[b], ref[0])


def _numpy_attention(q, k, v, scale, causal_offset=None):
    """Dense fp64 attention for one head: q [n, D], k/v [L, D]."""
    s = (q @ k.T) * scale
    if causal_offset is not None:
        n, L = s.shape
        mask = np.arange(L)[None, :] > (causal_offset + np.arange(n))[:, None]
        s = np.where(mask, -np.inf, s)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def test_mha_case_matches_dense_numpy():
    w = W.custom(4, 4, ctx=[50, 7], q_lens=[1, 1], seed=14)
    out, kc, vc, q = _run_workload(w)
    for b in range(2):
        k, v = _gather_contiguous(w, kc, vc, b)
        for h in range(4):
            ref = _numpy_attention(f64(q[b, h * 128:(h + 1) * 128])[None],
                                   f64(k[:, h]), f64(v[:, h]), 128 ** -0.5)
            np.testing.assert_allclose(out[b, h], ref[0], rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_on_repeated_heads():
    """Query head h uses KV head h // G: GQA equals MHA over K/V heads
    repeated G times consecutively."""
    H, Hkv, D, BS, G = 8, 2, 128, 16, 4
    g = torch.Generator().manual_seed(15)
    kc = u16(torch.randn(6, Hkv, BS, D, generator=g).to(torch.bfloat16))
    vc = u16(torch.randn(6, Hkv, BS, D, generator=g).to(torch.bfloat16))
    q = u16(torch.randn(2, H * D, generator=g).to(torch.bfloat16))
    bt = np.array([[5, 1, 3], [0, 2, 4]], np.int32)
    cl = np.array([40, 33], np.int32)
    gqa, e1 = oracle.paged_attention(q, kc, vc, bt, cl, H, Hkv, D, BS)
    mha, e2 = oracle.paged_attention(q, np.ascontiguousarray(np.repeat(kc, G, axis=1)),
                                     np.ascontiguousarray(np.repeat(vc, G, axis=1)),
                                     bt, cl, H, H, D, BS)
    assert e1 == e2 == 0 and np.array_equal(gqa, mha)


def test_brute_force_multiprecision():
    """Tiny integer-valued inputs, D in {4, 8}, L <= 5, blocks of 2 tokens:
    the softmax is evaluated with 40-digit arithmetic."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    rng = np.random.default_rng(16)
    for D in (4, 8):
        for L in range(1, 6):
            H, Hkv, BS = 2, 1, 2
            nb = (L + BS - 1) // BS
            q = rng.integers(-3, 4, (1, H * D)).astype(np.float64)
            k = rng.integers(-3, 4, (nb, Hkv, BS, D)).astype(np.float64)
            v = rng.integers(-3, 4, (nb, Hkv, BS, D)).astype(np.float64)
            perm = rng.permutation(nb).astype(np.int32)
            kc = np.empty_like(k); vc = np.empty_like(v)
            kc[perm] = k; vc[perm] = v      # logical block i lives at perm[i]
            out, err = oracle.paged_attention(bf16_of(q), bf16_of(kc), bf16_of(vc),
                                              perm[None, :], np.array([L], np.int32),
                                              H, Hkv, D, BS)
            assert err == 0
            scale = mp.mpf(D) ** mp.mpf(-0.5)
            for h in range(H):
                z = [scale * sum(mp.mpf(q[0, h * D + d]) * mp.mpf(k[j // BS, 0, j % BS, d])
                                 for d in range(D)) for j in range(L)]
                e = [mp.e ** zi for zi in z]
                tot = sum(e)
                for d in range(D):
                    ref = sum(e[j] * mp.mpf(v[j // BS, 0, j % BS, d]) for j in range(L)) / tot
                    assert abs(out[0, h, d] - float(ref)) <= 1e-13 * (1 + abs(float(ref)))


@pytest.mark.parametrize("partition", [1, 3, 16, 100, 512])
def test_split_kv_merge_equals_unsplit(partition):
    w = W.build(0)
    a, *_ = _run_workload(w)
    b, *_ = _run_workload(w, partition=partition)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-13)


def test_chunked_prefill_equals_successive_decodes():
    """A chunk of n queries at the end of a context of L equals n decode
    steps with contexts L - n + 1 .. L."""
    n, L = 9, 40
    w = W.custom(4, 2, ctx=[L], q_lens=[n], seed=17)
    out, kc, vc, q = _run_workload(w)
    for i in range(n):
        d, err = oracle.paged_attention(q[i:i + 1], kc, vc, w.block_tables,
                                        np.array([L - n + 1 + i], np.int32), 4, 2, 128, 16)
        assert err == 0 and np.array_equal(d[0], out[i])


def test_full_causal_prefill_matches_dense_numpy():
    L = 23
    w = W.custom(2, 1, ctx=[L], q_lens=[L], seed=18)
    out, kc, vc, q = _run_workload(w)
    k, v = _gather_contiguous(w, kc, vc, 0)
    for h in range(2):
        ref = _numpy_attention(f64(q[:, h * 128:(h + 1) * 128]), f64(k[:, 0]), f64(v[:, 0]),
                               128 ** -0.5, causal_offset=0)
        np.testing.assert_allclose(out[:, h], ref, rtol=1e-12, atol=1e-13)
    assert np.array_equal(out[0, 0], f64(v[0, 0]))


def test_attention_error_rows():
    H, Hkv, D, BS = 2, 1, 8, 16
    kc = np.zeros((2, Hkv, BS, D), np.uint16)
    vc = np.full((2, Hkv, BS, D), 0x3F80, np.uint16)   # 1.0
    q = np.zeros((3, H * D), np.uint16)
    bt = np.array([[0, 1], [7, 1], [1, 0]], np.int32)
    cl = np.array([0, 5, 20], np.int32)
    out, err = oracle.paged_attention(q, kc, vc, bt, cl, H, Hkv, D, BS)
    assert err == oracle.ERR_CONTEXT | oracle.ERR_BLOCK
    assert np.all(out[0] == 0) and np.all(out[1] == 0)
    assert np.allclose(out[2], 1.0)


def test_workload_recipes():
    """The five workloads have the shapes their descriptions give."""
    w = W.build(0)
    assert w.context_lens.tolist() == [17, 64, 100, 255] and w.num_blocks == 64
    assert sorted(w.block_tables[w.block_tables >= 0].tolist()) != []
    w = W.build(1)
    assert w.num_seqs == 64 and int(w.context_lens.min()) >= 128 and int(w.context_lens.max()) <= 4096
    w = W.build(2)
    assert w.num_tokens == 2108 and w.q_lens[:4] == [512] * 4 and w.q_lens[4:] == [1] * 60
    assert w.num_seqs == 64
    w = W.build(4)
    bt = w.block_tables
    assert w.num_seqs == 128 and bool((bt[:, :128] == bt[0, :128]).all())
    assert int(w.context_lens.min()) >= 2048 + 64 and int(w.context_lens.max()) <= 2048 + 512


# ------------------------------------------------------ FP8 (e4m3fn) ----
#
# The FP8 KV cache: kv_cache_dtype "fp8" with fp8_e4m3fn and a cache scale
# per tensor ("Qwen2大模型架构解析与vLLM优化实践" sections 4.1, 4.2, 6.3).

def test_e4m3_closed_forms():
    v = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert v[0x38] == 1.0                      # exponent field 7 = bias
    assert v[0x7E] == 448.0                    # largest finite: 1.75 * 2^8
    assert v[0x08] == 2.0 ** -6                # smallest normal
    assert v[0x01] == 2.0 ** -9                # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9            # largest subnormal
    assert v[0x3C] == 1.5 and v[0x40] == 2.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.sum(np.isnan(v)) == 2
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])
    fin = v[:0x7F]
    assert np.all(np.diff(fin) > 0)            # codes 0..126 increase


def test_e4m3_decode_matches_torch_float8():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    v = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert np.array_equal(np.isnan(t), np.isnan(v))
    assert np.array_equal(t[~np.isnan(t)], v[~np.isnan(v)])


def _nearest_e4m3(x):
    """Brute force: the finite code nearest to x, ties to the even code,
    magnitudes past 448 saturated."""
    vals = np.array([float(np.ldexp(1.0 + (c & 7) / 8.0, ((c >> 3) & 15) - 7)) if c >> 3
                     else float(np.ldexp(c & 7, -9)) for c in range(0x7F)])
    out = []
    for xv in np.asarray(x, dtype=np.float64):
        a = min(abs(xv), 448.0)
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        c = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        out.append(c | (0x80 if np.signbit(xv) else 0))
    return np.array(out, dtype=np.uint8)


def test_e4m3_encode_brute_force_nearest_even():
    v = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (v[:-1] + v[1:]) / 2                # every tie
    rng = np.random.default_rng(21)
    x = np.concatenate([mids, -mids, v, -v, rng.standard_normal(3000) * 50,
                        rng.standard_normal(500) * 2.0 ** -7, [447.9, 448.0, 460.0, 464.0,
                                                               1e6, -1e6, 2.0 ** -10,
                                                               3 * 2.0 ** -11]])
    x = x.astype(np.float32)
    assert np.array_equal(oracle.f32_to_e4m3(x), _nearest_e4m3(x.astype(np.float64)))
    # the midpoint between 1 and 1.125 goes to 1 (even), between 1.125 and
    # 1.25 to 1.25 (even)
    assert oracle.f32_to_e4m3(np.float32(1.0625)) == 0x38
    assert oracle.f32_to_e4m3(np.float32(1.1875)) == 0x3A
    assert oracle.f32_to_e4m3(np.float32(np.inf)) == 0x7E
    assert oracle.f32_to_e4m3(np.float32(-np.inf)) == 0xFE
    assert oracle.f32_to_e4m3(np.float32(np.nan)) == 0x7F


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(22)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 6, 200000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.f32_to_e4m3(x), t)


def _fp8_caches(w):
    shape = tuple(w.k_cache.shape)
    return np.zeros(shape, dtype=np.uint8), np.zeros(shape, dtype=np.uint8)


def test_append_fp8_is_bf16_append_then_quantize():
    w = W.custom(8, 2, ctx=[5, 40, 100], q_lens=[5, 1, 7], seed=23)
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    table = oracle.rope_table(1e6, w.max_pos, D)
    q16, kc16, vc16 = u16(w.qkv), u16(w.k_cache), u16(w.v_cache)
    assert oracle.rope_cache_append(q16, w.positions, w.slot_mapping, kc16, vc16, table,
                                    H, Hkv, D, BS) == 0
    q8 = u16(w.qkv)
    kc8, vc8 = _fp8_caches(w)
    ks, vs = 0.037, 0.011
    assert oracle.rope_cache_append_fp8(q8, w.positions, w.slot_mapping, kc8, vc8, table,
                                        H, Hkv, D, BS, ks, vs) == 0
    assert np.array_equal(q8, q16)             # q as before
    slots = w.slot_mapping.numpy()
    blk, off = slots // BS, slots % BS
    k16 = f64(kc16[blk, :, off]).astype(np.float32)
    v16 = f64(vc16[blk, :, off]).astype(np.float32)
    assert np.array_equal(kc8[blk, :, off], oracle.f32_to_e4m3(k16 / np.float32(ks)))
    assert np.array_equal(vc8[blk, :, off], oracle.f32_to_e4m3(v16 / np.float32(vs)))
    # untouched slots stay as they were
    mask = np.ones(kc8.shape[:1] + kc8.shape[2:3], dtype=bool)
    mask[blk, off] = False
    assert not kc8.transpose(0, 2, 1, 3)[mask].any()


def test_append_fp8_hand_example():
    """Position 0 (no rotation): k = 1.0 under k_scale 0.5 is 2.0 = 0x40;
    v = 3.0 under v_scale 2 is 1.5 = 0x3C; v = 1000 saturates to 0x7E."""
    H, Hkv, D, BS = 1, 1, 128, 16
    qkv = np.zeros((1, (H + 2 * Hkv) * D), dtype=np.uint16)
    qkv[0, D:2 * D] = oracle.bf16_round(np.full(D, 1.0))
    qkv[0, 2 * D:] = oracle.bf16_round(np.full(D, 3.0))
    qkv[0, 2 * D + 5] = oracle.bf16_round(np.array([1000.0]))[0]
    kc = np.zeros((2, Hkv, BS, D), dtype=np.uint8)
    vc = kc.copy()
    table = oracle.rope_table(1e6, 8, D)
    assert oracle.rope_cache_append_fp8(qkv, [0], [19], kc, vc, table, H, Hkv, D, BS,
                                        0.5, 2.0) == 0
    assert np.all(kc[1, 0, 3] == 0x40)
    assert vc[1, 0, 3, 5] == 0x7E
    assert np.all(np.delete(vc[1, 0, 3], 5) == 0x3C)
    assert not kc[0].any() and not vc[0].any()


def test_attention_fp8_equals_bf16_on_representable_values():
    """Codes whose values times a power-of-two scale are bf16 numbers: the
    FP8 attention equals the bf16 attention over those numbers exactly."""
    w = W.custom(8, 2, ctx=[3, 70, 200], q_lens=[1, 1, 1], seed=24)
    rng = np.random.default_rng(24)
    codes_k = rng.integers(0, 256, size=w.k_cache.shape, dtype=np.uint8)
    codes_v = rng.integers(0, 256, size=w.v_cache.shape, dtype=np.uint8)
    for c in (codes_k, codes_v):
        c[(c & 0x7F) == 0x7F] = 0x3A            # no NaN codes
    ks, vs = 2.0 ** -3, 2.0 ** 2
    kb = oracle.bf16_round(oracle.e4m3_to_f64(codes_k) * ks)
    vb = oracle.bf16_round(oracle.e4m3_to_f64(codes_v) * vs)
    assert np.array_equal(f64(kb), oracle.e4m3_to_f64(codes_k) * ks)
    q = u16(w.q_view())
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    ref, e1 = oracle.paged_attention(q, kb, vb, w.block_tables, w.context_lens, H, Hkv, D, BS)
    out, e2 = oracle.paged_attention_fp8(q, codes_k, codes_v, ks, vs, w.block_tables,
                                         w.context_lens, H, Hkv, D, BS)
    assert e1 == 0 and e2 == 0
    assert np.array_equal(out, ref)


def test_attention_fp8_scale_identities():
    """v_scale multiplies the output; k_scale multiplies the logits."""
    w = W.custom(4, 2, ctx=[50, 300], q_lens=[4, 1], seed=25)
    rng = np.random.default_rng(25)
    ck = rng.integers(0, 0x7F, size=w.k_cache.shape, dtype=np.uint8) | \
        (rng.integers(0, 2, size=w.k_cache.shape, dtype=np.uint8) << 7)
    cv = rng.integers(0, 0x7F, size=w.v_cache.shape, dtype=np.uint8) | \
        (rng.integers(0, 2, size=w.v_cache.shape, dtype=np.uint8) << 7)
    q = u16(w.q_view())
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    args = (w.block_tables, w.context_lens, H, Hkv, D, BS)
    base, _ = oracle.paged_attention_fp8(q, ck, cv, 0.01, 1.0, *args,
                                         cu_seqlens_q=w.cu_seqlens_q)
    sv, _ = oracle.paged_attention_fp8(q, ck, cv, 0.01, 0.3, *args, cu_seqlens_q=w.cu_seqlens_q)
    assert np.allclose(sv, 0.3 * base, rtol=1e-12, atol=0)
    sk, _ = oracle.paged_attention_fp8(q, ck, cv, 1.0, 1.0, *args, cu_seqlens_q=w.cu_seqlens_q,
                                       scale=0.01 * D ** -0.5)
    assert np.allclose(sk, base, rtol=1e-12, atol=1e-15)
