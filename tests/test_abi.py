"""C-ABI library checks that need no GPU: it builds, loads, exports every
symbol include/qattn.h declares, validates arguments on the host before any
CUDA call, and its host-side RoPE table equals the oracle's bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_gqa_07_gb300 import build as B
from paged_kv_gqa_07_gb300 import qattn as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return Q.load_library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "qattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qattn_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_three_entry_points():
    syms = declared_symbols()
    for name in ("qattn_rope_cache_append", "qattn_paged_decode", "qattn_varlen_prefill"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert sorted(Q.EXPORTED) == declared_symbols()


def test_tracing_build_exports_its_readers_and_the_regular_one_does_not(lib):
    """The tracing build (-DQATTN_TRACE) exports the functions of
    include/qattn_trace.h (stamp readers and the copy probe) on top of the
    regular entry points; the library the entry points ship in has none of
    them."""
    path = B.build(trace=True)
    tl = ctypes.CDLL(path)
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "qattn_trace.h")).read(),
                 flags=re.S)
    names = sorted(set(re.findall(r"\b(qattn_[a-z_0-9]+)\s*\(", src)))
    assert names == ["qattn_trace_clear", "qattn_trace_copy_stream", "qattn_trace_dims",
                     "qattn_trace_read"]
    for name in names + declared_symbols():
        assert hasattr(tl, name), name
    for name in names:
        assert not hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert Q.qattn_status_string(0) == "ok"
    assert "workspace" in Q.qattn_status_string(4)
    assert Q.qattn_version() >= 100


def test_host_rope_table_equals_oracle(lib):
    """The library's host table and the oracle's own table are computed by
    separate code from the same definition: they must agree bit for bit."""
    for theta in (1e6, 1e4):
        t = Q.qattn_rope_table_build(4096, 128, theta).numpy()
        o = oracle.rope_table(theta, 4096, 128)
        assert np.array_equal(t.view(np.uint32), o.view(np.uint32))


def test_host_rope_table_full_length(lib):
    t = Q.qattn_rope_table_build(32768, 128, 1e6).numpy()
    o = oracle.rope_table(1e6, 32768, 128)
    assert np.array_equal(t.view(np.uint32), o.view(np.uint32))


@pytest.mark.parametrize("scaling,factor,orig,max_pos", [(0, 1.0, 0, 64), (1, 2.0, 0, 300),
                                                        (1, 4.0, 0, 130), (2, 2.0, 100, 300),
                                                        (2, 2.0, 4096, 300)])
def test_host_scaled_table_equals_oracle(lib, scaling, factor, orig, max_pos):
    t = Q.qattn_rope_table_build_scaled(max_pos, 128, 1e6, scaling, factor, orig).numpy()
    o = oracle.rope_table_scaled(1e6, max_pos, 128, scaling, factor, orig)
    assert np.array_equal(t.view(np.uint32), o.view(np.uint32))


def test_table_build_rejects_bad_args(lib):
    buf = (ctypes.c_float * 16)()
    assert lib.qattn_rope_table_build(None, 4, 4, 1e6) == Q.QATTN_ERR_INVALID_ARG
    assert lib.qattn_rope_table_build(buf, 4, 3, 1e6) == Q.QATTN_ERR_INVALID_ARG
    assert lib.qattn_rope_table_build(buf, 0, 4, 1e6) == Q.QATTN_ERR_INVALID_ARG
    assert lib.qattn_rope_table_build(buf, 4, 4, -1.0) == Q.QATTN_ERR_INVALID_ARG
    f = lib.qattn_rope_table_build_scaled
    assert f(buf, 4, 4, 1e6, 3, 2.0, 10) == Q.QATTN_ERR_INVALID_ARG     # unknown scaling
    assert f(buf, 4, 4, 1e6, 1, 0.5, 0) == Q.QATTN_ERR_INVALID_ARG      # factor < 1
    assert f(buf, 4, 4, 1e6, 2, 2.0, 0) == Q.QATTN_ERR_INVALID_ARG      # dynamic, no original
    assert f(buf, 4, 2, 1e6, 1, 2.0, 0) == Q.QATTN_ERR_INVALID_ARG      # head_dim 2


def test_workspace_size_grows_with_context(lib):
    d = Q.make_dims(28, 4)
    a = Q.qattn_paged_decode_workspace_size(64, 4096, d)
    b = Q.qattn_paged_decode_workspace_size(64, 32768, d)
    assert 0 < a < b
    assert Q.qattn_paged_decode_workspace_size(64, 4096, Q.make_dims(28, 5)) == 0


def test_debug_fault_hook_checks_its_range(lib):
    """The decode testing hook refuses limits below 1 us or above 2 s and
    skip indices below -1, and (0, -1) restores the defaults; host only."""
    f = lib.qattn_debug_decode_faults
    assert f(5, -1) == Q.QATTN_ERR_INVALID_ARG
    assert f(3_000_000_000, -1) == Q.QATTN_ERR_INVALID_ARG
    assert f(0, -2) == Q.QATTN_ERR_INVALID_ARG
    assert f(1_000_000, 3) == Q.QATTN_OK
    assert f(0, -1) == Q.QATTN_OK


def test_host_validation_before_any_cuda_call(lib):
    """Every rejected call returns before touching CUDA (this machine may
    have no GPU): unsupported shapes, null pointers, bad strides."""
    fake = ctypes.c_void_p(256)
    d = Q.make_dims(28, 4)
    st = lib.qattn_rope_cache_append(fake, 28 * 128 + 1024, fake, 0, fake, 0, fake, fake, 4,
                                     fake, fake, 10, fake, 100, Q.make_dims(28, 4, 64), None, None)
    assert st == Q.QATTN_ERR_UNSUPPORTED                      # head_dim 64
    st = lib.qattn_rope_cache_append(fake, 4608, fake, 4608, fake, 4608, fake, fake, 4,
                                     fake, fake, 10, fake, 100, Q.make_dims(28, 4, 128, 48), None,
                                     None)
    assert st == Q.QATTN_ERR_UNSUPPORTED                      # block_size 48
    st = lib.qattn_rope_cache_append(fake, 4608, fake, 4608, fake, 4608, fake, fake, 4,
                                     fake, fake, 10, fake, 100, Q.make_dims(28, 4, 128, 8), None,
                                     None)
    assert st == Q.QATTN_ERR_UNSUPPORTED                      # block_size 8
    st = lib.qattn_rope_cache_append(fake, 4608, fake, 4608, fake, 4608, fake, fake, 4,
                                     fake, fake, 10, fake, 100, Q.make_dims(27, 4), None, None)
    assert st == Q.QATTN_ERR_UNSUPPORTED                      # 27 % 4
    st = lib.qattn_rope_cache_append(fake, 4608, fake, 4608, fake, 4608, None, fake, 4,
                                     fake, fake, 10, fake, 100, d, None, None)
    assert st == Q.QATTN_ERR_INVALID_ARG                      # null positions
    st = lib.qattn_rope_cache_append(fake, 4607, fake, 4608, fake, 4608, fake, fake, 4,
                                     fake, fake, 10, fake, 100, d, None, None)
    assert st == Q.QATTN_ERR_INVALID_ARG                      # stride % 8
    st = lib.qattn_rope_cache_append(None, 0, None, 0, None, 0, None, None, 0,
                                     None, None, 0, None, 0, d, None, None)
    assert st == Q.QATTN_OK                                   # zero tokens: no-op
    st = lib.qattn_paged_decode(fake, fake, 4608, fake, fake, 10, fake, 4, fake, 0, 100, d,
                                fake, 0, None, None)
    assert st == Q.QATTN_OK                                   # zero sequences: no-op
    st = lib.qattn_paged_decode(None, fake, 4608, fake, fake, 10, fake, 4, fake, 3, 100, d,
                                fake, 1 << 20, None, None)
    assert st == Q.QATTN_ERR_INVALID_ARG                      # null out
    st = lib.qattn_paged_decode(fake, ctypes.c_void_p(258), 4608, fake, fake, 10, fake, 4, fake,
                                3, 100, d, fake, 1 << 20, None, None)
    assert st == Q.QATTN_ERR_INVALID_ARG                      # misaligned q
    st = lib.qattn_varlen_prefill(fake, fake, 4608, None, 3, 10, 4, fake, fake, 10, fake, 4, fake,
                                  100, d, fake, 1 << 20, None, None)
    assert st == Q.QATTN_ERR_INVALID_ARG                      # null cu_seqlens_q
    st = lib.qattn_varlen_prefill(fake, fake, 4608, fake, 3, 50000, 49153, fake, fake, 10, fake,
                                  4, fake, 60000, d, fake, 1 << 30, None, None)
    assert st == Q.QATTN_ERR_UNSUPPORTED                      # a 49153-token chunk
    st = lib.qattn_paged_decode(fake, fake, 4608, fake, fake, 10, fake, 4, fake, 3, 100,
                                Q.make_dims(72, 8), fake, 1 << 20, None, None)
    assert st == Q.QATTN_ERR_UNSUPPORTED                      # group 9 > 8


def test_fp8_host_validation_before_any_cuda_call(lib):
    """The FP8 entry points reject bad scales and shapes on the host."""
    fake = ctypes.c_void_p(256)
    d = Q.make_dims(28, 4)
    good = (fake, 4608, fake, 4608, fake, 4608, fake, fake, 4, fake, fake, 10, fake, 100,
            None, None, None, 1e-6)
    for ks, vs in [(0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf")),
                   (1e-40, 1.0)]:
        assert lib.qattn_rope_cache_append_fp8(*good, ks, vs, d, None, None) == \
            Q.QATTN_ERR_INVALID_ARG
        assert lib.qattn_paged_decode_fp8(fake, fake, 4608, fake, fake, 10, fake, 4, fake, 3,
                                          100, ks, vs, d, fake, 1 << 20, None, None) == \
            Q.QATTN_ERR_INVALID_ARG
    assert lib.qattn_rope_cache_append_fp8(*good, 0.5, 0.5, Q.make_dims(28, 4, 128, 48), None,
                                           None) == Q.QATTN_ERR_UNSUPPORTED
    assert lib.qattn_paged_decode_fp8(fake, fake, 4608, fake, fake, 10, fake, 4, fake, 0, 100,
                                      0.5, 0.5, d, fake, 0, None, None) == Q.QATTN_OK
    assert lib.qattn_paged_decode_fp8(None, fake, 4608, fake, fake, 10, fake, 4, fake, 3, 100,
                                      0.5, 0.5, d, fake, 1 << 20, None, None) == \
        Q.QATTN_ERR_INVALID_ARG
    vf = lib.qattn_varlen_prefill_fp8
    assert vf(fake, fake, 4608, fake, 3, 10, 4, fake, fake, 10, fake, 4, fake, 100, 4, 0.5, 0.5,
              d, fake, 1 << 30, None, None) == Q.QATTN_ERR_INVALID_ARG   # 4 prefill of 3
    assert vf(fake, fake, 4608, fake, 3, 10, 4, fake, fake, 10, fake, 4, fake, 100, 2, 0.0, 0.5,
              d, fake, 1 << 30, None, None) == Q.QATTN_ERR_INVALID_ARG   # bad k_scale
    assert vf(fake, fake, 4608, fake, 3, 10, 4, fake, fake, 10, fake, 4, fake, 100, 2, 0.5, 0.5,
              d, fake, 16, None, None) == Q.QATTN_ERR_WORKSPACE          # workspace too small
    assert Q.qattn_varlen_prefill_fp8_workspace_size(3, 2, 100, d) > \
        Q.qattn_varlen_prefill_fp8_workspace_size(3, 1, 100, d) > 0
    assert Q.qattn_varlen_prefill_fp8_workspace_size(3, 4, 100, d) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        Q.load_library(str(tmp_path / "missing.so"))


C_CLIENT = r"""
#include <stdio.h>
#include <stdlib.h>
#include "qattn.h"

int main(void) {
  qattn_dims d = {28, 4, 128, 16, 0.0f};
  float* table = (float*)malloc(sizeof(float) * 8 * 128);
  int32_t ctx = 17;
  int rc;
  printf("version %d\n", qattn_version());
  printf("status %s\n", qattn_status_string(QATTN_ERR_WORKSPACE));
  rc = qattn_rope_table_build(table, 8, 128, 1e6);
  printf("table %d %.9g %.9g\n", rc, table[0], table[64]);
  printf("workspace %d\n", qattn_paged_decode_workspace_size(64, 4096, d) > 0);
  /* host validation, before any CUDA call: null caches */
  rc = qattn_paged_decode(NULL, NULL, 3584, NULL, NULL, 10, NULL, 4, &ctx, 1, 17, d, NULL, 0,
                          NULL, NULL);
  printf("decode %d\n", rc);
  d.block_size = 48;
  rc = qattn_paged_decode(NULL, NULL, 3584, NULL, NULL, 10, NULL, 4, &ctx, 1, 17, d, NULL, 0,
                          NULL, NULL);
  printf("unsupported %d\n", rc);
  free(table);
  return 0;
}
"""


def test_header_is_plain_c_and_the_library_links_from_c(lib, tmp_path):
    """include/qattn.h compiles as strict C99, and a C program linked against
    libqattn.so runs its host-side entry points (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(B.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lqattn", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    assert out[0] == f"version {int(lib.qattn_version())}"
    assert out[1] == "status " + lib.qattn_status_string(Q.QATTN_ERR_WORKSPACE).decode()
    assert out[2] == "table 0 1 0"           # position 0: cos 1, sin 0
    assert out[3] == "workspace 1"
    assert out[4] == f"decode {Q.QATTN_ERR_INVALID_ARG}"
    assert out[5] == f"unsupported {Q.QATTN_ERR_UNSUPPORTED}"
