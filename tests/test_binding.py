"""The Python binding's argument checks, on the CPU.

Every entry point hands the library the pointers and sizes that the C ABI
(include/qattn.h) expects for well-formed workloads, and a tensor whose
shape, dtype, layout or device disagrees with the call's dims is refused
before the library is called (QattnArgError: status QATTN_ERR_INVALID_ARG,
also a ValueError).  The library is replaced by a recorder and the device
check by a plain data_ptr(), so no GPU is needed.
"""
import pytest
import torch

from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W


class Recorder:
    """Stands in for the loaded library: records each entry-point call."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return 0
        return call

    def last(self, name):
        hits = [a for n, a in self.calls if n == name]
        assert hits, f"{name} was not called"
        return hits[-1]


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(Q, "_lib", r)
    monkeypatch.setattr(Q._Args, "device_ptr", lambda self, t, name: t.data_ptr())
    monkeypatch.setattr(Q, "_stream", lambda s: None)
    return r


class Call:
    """The arguments of one workload's calls (CPU tensors)."""

    def __init__(self, w, fp8=False):
        self.w = W.with_fp8_cache(w) if fp8 else w
        w = self.w
        self.dims = Q.make_dims(w.num_heads, w.num_kv_heads, w.head_dim, w.block_size)
        self.table = torch.zeros((w.max_pos, w.head_dim), dtype=torch.float32)
        self.out = torch.empty((w.num_tokens, w.num_heads, w.head_dim), dtype=torch.bfloat16)
        self.ws = torch.empty(4096, dtype=torch.uint8)
        self.err = torch.zeros(1, dtype=torch.int32)

    def append(self, **kw):
        w = self.w
        a = dict(q=w.q_view(), k=w.k_view(), v=w.v_view(), positions=w.positions,
                 slot_mapping=w.slot_mapping, k_cache=w.k_cache, v_cache=w.v_cache,
                 cos_sin=self.table, dims=self.dims, err_word=self.err)
        a.update(kw)
        Q.qattn_rope_cache_append(**a)

    def decode(self, **kw):
        w = self.w
        a = dict(out=self.out, q=w.q_view(), k_cache=w.k_cache, v_cache=w.v_cache,
                 block_tables=w.block_tables, context_lens=w.context_lens,
                 max_context_len=w.max_context_len, dims=self.dims, workspace=self.ws,
                 err_word=self.err)
        a.update(kw)
        Q.qattn_paged_decode(**a)

    def varlen(self, **kw):
        w = self.w
        a = dict(out=self.out, q=w.q_view(), cu_seqlens_q=w.cu_seqlens_q,
                 max_q_len=w.max_q_len, k_cache=w.k_cache, v_cache=w.v_cache,
                 block_tables=w.block_tables, context_lens=w.context_lens,
                 max_context_len=w.max_context_len, dims=self.dims, workspace=self.ws,
                 err_word=self.err)
        a.update(kw)
        Q.qattn_varlen_prefill(**a)


def small_workloads():
    return [
        W.custom(16, 8, ctx=[17, 64, 100, 255], q_lens=[1] * 4, seed=1),
        W.custom(28, 4, ctx=[300, 700, 64, 1, 129], q_lens=[200, 33, 64, 1, 1], seed=2),
        W.custom(16, 2, ctx=[64 + s for s in (1, 31, 300)], q_lens=[1] * 3, seed=3,
                 shared_prefix_tokens=64, block_size=32),
        W.custom(28, 4, ctx=[200, 129], q_lens=[1, 1], seed=4, block_size=64),
    ]


@pytest.mark.parametrize("idx", range(4))
def test_well_formed_calls_pass_sizes_through(rec, idx):
    w = small_workloads()[idx]
    c = Call(w)
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
    c.append()
    a = rec.last("qattn_rope_cache_append")
    assert a[1] == (H + 2 * Hkv) * D  # q row stride of the fused QKV rows
    assert a[8] == w.num_tokens and a[11] == w.k_cache.shape[0] and a[13] == w.max_pos
    bias = torch.zeros((H + 2 * Hkv) * D, dtype=torch.bfloat16)
    nw = torch.ones(D, dtype=torch.bfloat16)
    Q.qattn_rope_cache_append_ex(w.q_view(), w.k_view(), w.v_view(), w.positions,
                                 w.slot_mapping, w.k_cache, w.v_cache, c.table, c.dims,
                                 qkv_bias=bias, q_norm_weight=nw, k_norm_weight=nw,
                                 err_word=c.err)
    assert rec.last("qattn_rope_cache_append_ex")[14] == bias.data_ptr()
    if w.is_decode:
        c.decode()
        a = rec.last("qattn_paged_decode")
        assert a[5] == w.k_cache.shape[0] and a[7] == w.block_tables.shape[1]
        assert a[9] == w.num_seqs and a[10] == w.max_context_len
        assert a[13] == c.ws.numel()
        Q.qattn_paged_decode_noalloc(c.out, w.q_view(), w.k_cache, w.v_cache, w.block_tables,
                                     w.context_lens, w.max_context_len, c.dims, c.err)
        assert rec.last("qattn_paged_decode_noalloc")[9] == w.num_seqs
    if w.shared_prefix_tokens:
        Q.qattn_paged_decode_shared_prefix(c.out, w.q_view(), w.k_cache, w.v_cache,
                                           w.block_tables, w.context_lens, w.max_context_len,
                                           w.shared_prefix_tokens, c.dims, c.ws, c.err)
        assert rec.last("qattn_paged_decode_shared_prefix")[11] == w.shared_prefix_tokens
    c.varlen()
    a = rec.last("qattn_varlen_prefill")
    assert a[4] == w.num_seqs and a[5] == w.num_tokens and a[6] == w.max_q_len


@pytest.mark.parametrize("idx", range(4))
def test_fp8_calls_pass_sizes_through(rec, idx):
    c = Call(small_workloads()[idx], fp8=True)
    w = c.w
    assert w.k_cache.dtype == torch.uint8
    Q.qattn_rope_cache_append_fp8(w.q_view(), w.k_view(), w.v_view(), w.positions,
                                  w.slot_mapping, w.k_cache, w.v_cache, c.table, 0.5, 0.25,
                                  c.dims, err_word=c.err)
    a = rec.last("qattn_rope_cache_append_fp8")
    assert a[11] == w.k_cache.shape[0] and a[18:20] == (0.5, 0.25)
    if w.is_decode:
        Q.qattn_paged_decode_fp8(c.out, w.q_view(), w.k_cache.view(torch.float8_e4m3fn),
                                 w.v_cache, w.block_tables, w.context_lens, w.max_context_len,
                                 0.5, 0.25, c.dims, c.ws, c.err)
        assert rec.last("qattn_paged_decode_fp8")[11:13] == (0.5, 0.25)
    if w.shared_prefix_tokens:
        Q.qattn_paged_decode_shared_prefix_fp8(c.out, w.q_view(), w.k_cache, w.v_cache,
                                               w.block_tables, w.context_lens,
                                               w.max_context_len, w.shared_prefix_tokens, 0.5,
                                               0.25, c.dims, c.ws, c.err)
    npf = sum(1 for n in w.q_lens if n >= 2)
    Q.qattn_varlen_prefill_fp8(c.out, w.q_view(), w.cu_seqlens_q, w.max_q_len, w.k_cache,
                               w.v_cache, w.block_tables, w.context_lens, w.max_context_len, npf,
                               0.5, 0.25, c.dims, c.ws, c.err)
    assert rec.last("qattn_varlen_prefill_fp8")[14] == npf


def test_zero_sized_calls_pass(rec):
    c = Call(small_workloads()[0])
    w = c.w
    empty_i = torch.empty(0, dtype=torch.int32)
    empty_q = torch.empty((0, w.num_heads * 128), dtype=torch.bfloat16)
    kv = w.num_kv_heads * 128
    c.append(q=empty_q, k=empty_q[:, :kv], v=empty_q[:, :kv], positions=empty_i,
             slot_mapping=empty_i)
    c.decode(out=c.out[:0], q=empty_q, block_tables=w.block_tables[:0],
             context_lens=w.context_lens[:0])
    assert rec.last("qattn_paged_decode")[9] == 0


def _refused(fn, match):
    with pytest.raises(Q.QattnArgError, match=match) as ei:
        fn()
    assert ei.value.status == Q.QATTN_ERR_INVALID_ARG
    assert isinstance(ei.value, Q.QattnError) and isinstance(ei.value, ValueError)


def test_mismatched_caches_are_refused(rec):
    c = Call(small_workloads()[1])
    w = c.w
    _refused(lambda: c.decode(k_cache=w.k_cache[:, :1]), "k_cache is")          # kv heads
    bs32 = torch.zeros((4, w.num_kv_heads, 32, 128), dtype=torch.bfloat16)
    _refused(lambda: c.append(v_cache=bs32), "v_cache is")                      # block size
    _refused(lambda: c.varlen(v_cache=w.v_cache[:-1]), "same number of blocks")
    _refused(lambda: c.decode(k_cache=w.k_cache.transpose(1, 2).contiguous()
                              .transpose(1, 2)), "k_cache must be contiguous")
    _refused(lambda: c.decode(k_cache=w.k_cache.float()), "k_cache must be")  # dtype
    fp8 = Call(small_workloads()[1], fp8=True)
    _refused(lambda: Q.qattn_paged_decode_fp8(
        fp8.out, fp8.w.q_view(), w.k_cache, w.v_cache, fp8.w.block_tables, fp8.w.context_lens,
        fp8.w.max_context_len, 0.5, 0.5, fp8.dims, fp8.ws, fp8.err), "k_cache must be")
    assert rec.calls == []


def test_mismatched_tables_and_rows_are_refused(rec):
    c = Call(small_workloads()[0])
    w = c.w
    _refused(lambda: c.decode(block_tables=w.block_tables[:-1]), "block_tables is")
    wide = torch.zeros((w.num_seqs, 2 * w.block_tables.shape[1]), dtype=torch.int32)
    _refused(lambda: c.decode(block_tables=wide[:, ::2]), "block_tables must be contiguous")
    _refused(lambda: c.decode(context_lens=w.context_lens.long()), "context_lens must be")
    _refused(lambda: c.decode(q=w.q_view()[:, :64]), "q is")
    _refused(lambda: c.decode(q=w.q_view()[:-1]), "q is")
    _refused(lambda: c.decode(out=c.out[:-1]), "out has")
    _refused(lambda: c.decode(err_word=c.err[:0]), "err_word has")
    _refused(lambda: c.decode(workspace=c.ws[::2]), "workspace must be contiguous")
    _refused(lambda: c.varlen(context_lens=w.context_lens[:-1]), "context_lens has")
    _refused(lambda: c.varlen(cu_seqlens_q=w.cu_seqlens_q[:0]), "cu_seqlens_q has")
    _refused(lambda: c.append(slot_mapping=w.slot_mapping[:-1]), "slot_mapping has")
    _refused(lambda: c.append(positions=w.positions.view(2, -1)), "positions must be 1-D")
    _refused(lambda: c.append(k=w.k_view()[:, :-128]), "k is")
    _refused(lambda: c.append(cos_sin=c.table[:, :64]), "cos_sin is")
    _refused(lambda: c.append(cos_sin=c.table.double()), "cos_sin must be")
    assert rec.calls == []


def test_short_extras_are_refused(rec):
    c = Call(small_workloads()[0])
    w = c.w
    nw = torch.ones(128, dtype=torch.bfloat16)
    for kw, name in ((dict(q_norm_weight=nw[1:]), "q_norm_weight"),
                     (dict(k_norm_weight=nw[:64]), "k_norm_weight"),
                     (dict(qkv_bias=nw), "qkv_bias")):
        _refused(lambda: Q.qattn_rope_cache_append_ex(
            w.q_view(), w.k_view(), w.v_view(), w.positions, w.slot_mapping, w.k_cache,
            w.v_cache, c.table, c.dims, err_word=c.err, **kw), f"{name} has")
    assert rec.calls == []


def test_host_tensors_are_refused_before_the_library_is_called(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(Q, "_lib", r)
    c = Call(small_workloads()[0])
    _refused(c.decode, "must be a CUDA tensor")
    _refused(c.append, "must be a CUDA tensor")
    assert r.calls == []
