"""The decode entry point for callers that cannot allocate device memory.

Some callers may not call cudaMalloc at all -- code inside another
framework's CUDA-graph capture, a serving loop with a memory pool fixed at
start-up -- so they cannot hand qattn_paged_decode a workspace.
qattn_paged_decode_noalloc keeps its split-KV scratch in a fixed array inside
the library instead.  This test calls it through the C ABI three times in a row
(each call starts from whatever the previous one left in the shared array)
and checks each result against the CPU oracle and against qattn_paged_decode
with a workspace of its own, within the tolerance the parity tests use, and
that the device's free memory does not move across the later calls.  It lives in its own file,
named to be collected last, and passes alone or after the other tests.
"""
import ctypes

import pytest
import torch

from paged_kv_gqa_07_gb300 import build as B
from paged_kv_gqa_07_gb300 import qattn as Q
from paged_kv_gqa_07_gb300 import workloads as W

from _util import ATOL, RTOL, GpuRun, assert_close, oracle_for

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    B.build()
    lib = Q.load_library()
    fn = lib.qattn_paged_decode_noalloc
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [P, P, I64, P, P, I32, P, I32, P, I32, I32, Q.qattn_dims, P, P]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, r, out):
    g = r.g
    q = g.q_view()
    return fn(out.data_ptr(), q.data_ptr(), q.stride(0), g.k_cache.data_ptr(),
              g.v_cache.data_ptr(), int(g.k_cache.shape[0]), g.block_tables.data_ptr(),
              int(g.block_tables.shape[1]), g.context_lens.data_ptr(), int(g.context_lens.shape[0]),
              r.max_ctx, r.dims, r.err.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("idx", [1, 3])
def test_noalloc_decode_matches_workspace_decode_twice(idx):
    fn = _noalloc_fn()
    w = W.build(idx)
    r = GpuRun(w).append().sync()
    ref = r.attend().sync().out.clone()
    assert r.err_bits == 0
    outs = [torch.full_like(ref, float("nan")) for _ in range(3)]
    free = []
    for out in outs:   # nothing in this loop allocates on the torch side
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        assert _call(fn, r, out) == Q.QATTN_OK
        torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
    assert r.err_bits == 0
    _, _, _, oracle_out, e1, e2 = oracle_for(idx)
    assert e1 == e2 == 0
    for out in outs:
        assert_close(out, oracle_out)
        d = (out.float() - ref.float()).abs().max().item()
        scale = ref.float().abs().max().item()
        assert d <= ATOL and d / scale <= RTOL
    # after the first call (which may load the library's device code), the
    # calls take no device memory
    assert free[1] == free[2] == free[3]


def test_noalloc_refuses_shapes_beyond_its_scratch():
    fn = _noalloc_fn()
    w = W.build(0)
    r = GpuRun(w).append().sync()
    dims = r.dims
    big_ctx = 1 << 20   # a 1M-token hint: the split workspace would exceed 32 MiB
    assert Q.qattn_paged_decode_workspace_size(w.num_seqs, big_ctx, dims) > (32 << 20)
    g = r.g
    q = g.q_view()
    out = torch.empty_like(r.out)
    rc = fn(out.data_ptr(), q.data_ptr(), q.stride(0), g.k_cache.data_ptr(), g.v_cache.data_ptr(),
            int(g.k_cache.shape[0]), g.block_tables.data_ptr(), int(g.block_tables.shape[1]),
            g.context_lens.data_ptr(), w.num_seqs, big_ctx, dims, None,
            torch.cuda.current_stream().cuda_stream)
    assert rc == Q.QATTN_ERR_WORKSPACE
