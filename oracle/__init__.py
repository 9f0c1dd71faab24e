"""CPU oracle for the paged-KV GQA attention step (TEST INFRASTRUCTURE).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never links or calls it, and it shares
no code with the CUDA library: ``oracle.c`` is a plain fp64 restatement of
the maths, compiled with ``gcc -O2 -ffp-contract=off`` into ``liboracle.so``.

What each function follows (pages named by title and section):

* :func:`rope_table`   -- get_rope(head_dim, rotary_dim=head_dim, max_position,
  base=rope_theta) in "Qwen2大模型架构解析与vLLM优化实践" section 2.2, with
  rope_theta = 1e6 from "Qwen2 模型结构代码详解" section 2.
* :func:`rope_table_scaled` -- the table with rope_scaling (linear, or
  dynamic NTK: a raised base when the table covers more than the original
  positions), "Qwen2大模型架构解析与vLLM优化实践" section 7.1.
* :func:`rope_cache_append` -- rotate-half RoPE on q and k, then the write of
  k and v into fixed-size cache blocks through a slot mapping (PagedAttention
  block cache, vLLM-deploys-Qwen notes section 2.1; nano-vllm block_table and
  prepare_prefill, Qwen3 skeleton page section 5).
* :func:`rope_cache_append_ex`, :func:`add_bias_head`, :func:`rmsnorm_head`
  -- the same append with the qkv projection bias (bias=True,
  "Qwen2大模型架构解析与vLLM优化实践") and the Qwen3 per-head q_norm /
  k_norm RMSNorms (nano-vllm Qwen3 skeleton page, module tree) applied
  before RoPE.
* :func:`paged_attention` -- grouped-query attention with scaling
  head_dim ** -0.5 ("Qwen2 模型结构代码详解" section 2; Attention(...) in
  "Qwen2大模型架构解析与vLLM优化实践" section 4.1), gathering keys through the
  block table, for decode and for causal varlen / chunked prefill
  (FlashAttention-2 varlen, Qwen engineering notes section 2.1), optionally
  in the split-KV partition + log-sum-exp merge form.
* :func:`contiguous_attention` -- the same attention on unpaged K/V.
* :func:`f32_to_e4m3`, :func:`e4m3_to_f64`, :func:`rope_cache_append_fp8`,
  :func:`paged_attention_fp8` -- the FP8 KV cache (kv_cache_dtype "fp8",
  fp8_e4m3fn, a cache scale per tensor: "Qwen2大模型架构解析与vLLM优化实践"
  sections 4.1, 4.2 and 6.3): the OCP E4M3 format written out from its
  definition, codes = e4m3(x / scale) of the bf16 values a bf16 cache would
  hold, attention over code * scale.

Every function here is pinned by ``tests/test_oracle.py`` against closed
forms, invariants, a brute-force multiprecision softmax and the configuration
values the pages print (``tests/golden``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_SLOT = 1
ERR_BLOCK = 2
ERR_CONTEXT = 4
ERR_POSITION = 16
ERR_NORM_INEXACT = 64  # oracle only: an RMSNorm sum of squares was rounded in fp64

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F64 = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (idempotent); returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.oracle_rope_table.argtypes = [_F64, _I32, _I32, _P]
            L.oracle_rope_table.restype = ctypes.c_int
            L.oracle_rope_table_scaled.argtypes = [_F64, _I32, _I32, _I32, _F64, _I32, _P]
            L.oracle_rope_table_scaled.restype = ctypes.c_int
            L.oracle_rope_head_exact.argtypes = [_P, _I32, _P, _P]
            L.oracle_rope_head_exact.restype = None
            L.oracle_rope_head_f64.argtypes = [_P, _I32, _F64, _F64, _P]
            L.oracle_rope_head_f64.restype = None
            L.oracle_rope_cache_append.argtypes = [
                _P, _I64, _P, _I64, _P, _I64, _P, _P, _I32, _P, _P, _I32, _P,
                _I32, _I32, _I32, _I32, _I32]
            L.oracle_rope_cache_append.restype = _I32
            L.oracle_add_bias_head.argtypes = [_P, _P, _I32, _P]
            L.oracle_add_bias_head.restype = None
            L.oracle_rmsnorm_head.argtypes = [_P, _P, _I32, _F64, _P]
            L.oracle_rmsnorm_head.restype = _I32
            L.oracle_rope_cache_append_ex.argtypes = (
                L.oracle_rope_cache_append.argtypes + [_P, _P, _P, _F64])
            L.oracle_rope_cache_append_ex.restype = _I32
            L.oracle_paged_attention.argtypes = [
                _P, _P, _I64, _P, _I32, _P, _P, _I32, _P, _I32, _P, _I32, _I32,
                _I32, _I32, _F64, _I32, _I32]
            L.oracle_paged_attention.restype = _I32
            L.oracle_contiguous_attention.argtypes = [
                _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _F64]
            L.oracle_contiguous_attention.restype = _I32
            L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            L.oracle_f32_to_bf16.restype = ctypes.c_uint16
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = _F64
            L.oracle_f32_to_e4m3_array.argtypes = [_P, _I64, _P]
            L.oracle_f32_to_e4m3_array.restype = None
            L.oracle_e4m3_to_f64_array.argtypes = [_P, _I64, _P]
            L.oracle_e4m3_to_f64_array.restype = None
            L.oracle_rope_cache_append_fp8.argtypes = (
                L.oracle_rope_cache_append_ex.argtypes + [ctypes.c_float, ctypes.c_float])
            L.oracle_rope_cache_append_fp8.restype = _I32
            L.oracle_paged_attention_fp8.argtypes = [
                _P, _P, _I64, _P, _I32, _P, _P, _F64, _F64, _I32, _P, _I32, _P, _I32,
                _I32, _I32, _I32, _F64, _I32, _I32]
            L.oracle_paged_attention_fp8.restype = _I32
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """bf16 payload as a C-contiguous uint16 numpy array (torch or numpy in)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16
    return a


def _i32(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().cpu().contiguous().to(torch.int32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.int32)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def rope_table(theta: float, max_pos: int, head_dim: int) -> np.ndarray:
    """[max_pos, head_dim] fp32: cos in columns < D/2, sin in the rest."""
    out = np.empty((max_pos, head_dim), dtype=np.float32)
    rc = lib().oracle_rope_table(float(theta), int(max_pos), int(head_dim), _ptr(out))
    if rc != 0:
        raise ValueError("bad rope table arguments")
    return out


SCALING_NONE, SCALING_LINEAR, SCALING_DYNAMIC = 0, 1, 2


def rope_table_scaled(theta: float, max_pos: int, head_dim: int, scaling: int,
                      factor: float = 1.0, original_max: int = 0) -> np.ndarray:
    """rope_table with rope_scaling: 0 none, 1 linear, 2 dynamic NTK."""
    out = np.empty((max_pos, head_dim), dtype=np.float32)
    rc = lib().oracle_rope_table_scaled(float(theta), int(max_pos), int(head_dim),
                                        int(scaling), float(factor), int(original_max),
                                        _ptr(out))
    if rc != 0:
        raise ValueError("bad rope table arguments")
    return out


def rope_head_exact(x_u16: np.ndarray, cos_sin_row: np.ndarray) -> np.ndarray:
    """Rotate one bf16 head vector with the fp32 recipe; returns uint16."""
    x = np.ascontiguousarray(x_u16, dtype=np.uint16)
    row = np.ascontiguousarray(cos_sin_row, dtype=np.float32)
    y = np.empty_like(x)
    lib().oracle_rope_head_exact(_ptr(x), x.size, _ptr(row), _ptr(y))
    return y


def rope_head_f64(x: np.ndarray, pos: float, theta: float) -> np.ndarray:
    """Rotate one fp64 head vector at an exact fp64 angle."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().oracle_rope_head_f64(_ptr(x), x.size, float(pos), float(theta), _ptr(y))
    return y


def f32_to_bf16(f: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(f)))


def rope_cache_append(qkv, positions, slot_mapping, k_cache, v_cache, cos_sin,
                      num_heads, num_kv_heads, head_dim, block_size):
    """RoPE + cache append on host arrays, in place.

    qkv: uint16 [T, (H + 2 Hkv) D] fused rows (q heads first, then k, then
    v); its q heads are rotated in place.  k_cache / v_cache: uint16
    [num_blocks, Hkv, BS, D], written at the slots.  Returns the error bits.
    """
    assert qkv.dtype == np.uint16 and qkv.flags["C_CONTIGUOUS"]
    assert k_cache.dtype == np.uint16 and k_cache.flags["C_CONTIGUOUS"]
    assert v_cache.dtype == np.uint16 and v_cache.flags["C_CONTIGUOUS"]
    H, Hkv, D = num_heads, num_kv_heads, head_dim
    W = qkv.shape[1]
    assert W == (H + 2 * Hkv) * D
    pos = _i32(positions)
    slots = _i32(slot_mapping)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    base = qkv.ctypes.data
    return int(lib().oracle_rope_cache_append(
        base, W, base + H * D * 2, W, base + (H + Hkv) * D * 2, W,
        _ptr(pos), _ptr(slots), int(pos.shape[0]), _ptr(k_cache), _ptr(v_cache),
        int(k_cache.shape[0]), _ptr(cs), cs.shape[0], H, Hkv, D, block_size))


def add_bias_head(x, b):
    """bf16(float(x) + float(b)) element-wise on uint16 bf16 bit arrays."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    y = np.empty_like(x)
    lib().oracle_add_bias_head(_ptr(x), _ptr(b), int(x.size), _ptr(y))
    return y


def rmsnorm_head(x, w, eps, with_exactness=False):
    """RMSNorm of one head vector (uint16 bf16 bits) with weight w, eps.
    With ``with_exactness``, returns (y, exact) where exact says the fp64 sum
    of squares was exact (the reading's premise)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    y = np.empty_like(x)
    inexact = lib().oracle_rmsnorm_head(_ptr(x), _ptr(w), int(x.size), float(eps), _ptr(y))
    return (y, inexact == 0) if with_exactness else y


def rope_cache_append_ex(qkv, positions, slot_mapping, k_cache, v_cache, cos_sin,
                         num_heads, num_kv_heads, head_dim, block_size, bias=None,
                         q_norm_w=None, k_norm_w=None, eps=1e-6):
    """rope_cache_append with the qkv projection bias ([(H + 2 Hkv) D] bf16
    bits) added first and the per-head RMSNorms (weights [D]) of q and k
    before RoPE; None skips a step.  In place; returns the error bits."""
    assert qkv.dtype == np.uint16 and qkv.flags["C_CONTIGUOUS"]
    H, Hkv, D = num_heads, num_kv_heads, head_dim
    W = qkv.shape[1]
    assert W == (H + 2 * Hkv) * D
    pos = _i32(positions)
    slots = _i32(slot_mapping)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    keep = [None if a is None else np.ascontiguousarray(a, dtype=np.uint16)
            for a in (bias, q_norm_w, k_norm_w)]
    ptrs = [None if a is None else _ptr(a) for a in keep]
    base = qkv.ctypes.data
    return int(lib().oracle_rope_cache_append_ex(
        base, W, base + H * D * 2, W, base + (H + Hkv) * D * 2, W,
        _ptr(pos), _ptr(slots), int(pos.shape[0]), _ptr(k_cache), _ptr(v_cache),
        int(k_cache.shape[0]), _ptr(cs), cs.shape[0], H, Hkv, D, block_size,
        ptrs[0], ptrs[1], ptrs[2], float(eps)))


def paged_attention(q, k_cache, v_cache, block_tables, context_lens,
                    num_heads, num_kv_heads, head_dim, block_size, scale=None,
                    cu_seqlens_q=None, partition_tokens=0, nthreads=None):
    """fp64 paged attention.  q: uint16 [rows, row_stride] (heads packed at
    the front of each row).  Returns (out[rows, H, D] float64, error bits)."""
    qn = _u16(q)
    if qn.ndim == 3:
        qn = qn.reshape(qn.shape[0], -1)
    kc = _u16(k_cache)
    vc = _u16(v_cache)
    bt = _i32(block_tables)
    cl = _i32(context_lens)
    cu = None if cu_seqlens_q is None else _i32(cu_seqlens_q)
    num_seqs = int(cl.shape[0])
    rows = num_seqs if cu is None else int(cu[-1])
    out = np.zeros((rows, num_heads, head_dim), dtype=np.float64)
    if scale is None:
        scale = float(head_dim) ** -0.5
    err = lib().oracle_paged_attention(
        _ptr(out), _ptr(qn), qn.shape[1], _ptr(cu), num_seqs, _ptr(kc), _ptr(vc),
        int(kc.shape[0]), _ptr(bt), int(bt.shape[1]), _ptr(cl), num_heads,
        num_kv_heads, head_dim, block_size, float(scale), int(partition_tokens),
        int(nthreads or default_threads()))
    if err < 0:
        raise ValueError("bad attention arguments")
    return out, int(err)


def contiguous_attention(q, k, v, num_heads, num_kv_heads, head_dim, scale=None):
    """q: uint16 [q_len, H, D]; k, v: uint16 [L, Hkv, D]; bottom-right causal."""
    qn, kn, vn = _u16(q), _u16(k), _u16(v)
    q_len, L = qn.shape[0], kn.shape[0]
    out = np.zeros((q_len, num_heads, head_dim), dtype=np.float64)
    if scale is None:
        scale = float(head_dim) ** -0.5
    rc = lib().oracle_contiguous_attention(
        _ptr(out), _ptr(qn), _ptr(kn), _ptr(vn), L, q_len, num_heads,
        num_kv_heads, head_dim, float(scale))
    if rc != 0:
        raise ValueError("bad contiguous attention arguments")
    return out


def f32_to_e4m3(x) -> np.ndarray:
    """fp32 values -> e4m3fn codes (uint8), nearest-even, saturating."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint8)
    lib().oracle_f32_to_e4m3_array(_ptr(f), int(f.size), _ptr(out))
    return out


def e4m3_to_f64(c) -> np.ndarray:
    """e4m3fn codes (uint8) -> their values (NaN for the NaN codes)."""
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_to_f64_array(_ptr(c), int(c.size), _ptr(out))
    return out


def rope_cache_append_fp8(qkv, positions, slot_mapping, k_cache, v_cache, cos_sin,
                          num_heads, num_kv_heads, head_dim, block_size, k_scale, v_scale,
                          bias=None, q_norm_w=None, k_norm_w=None, eps=1e-6):
    """rope_cache_append_ex into uint8 e4m3 caches: k and v are stored as
    e4m3(x / k_scale) and e4m3(x / v_scale) of the bf16 rows a bf16 cache
    would receive.  In place; returns the error bits."""
    assert qkv.dtype == np.uint16 and qkv.flags["C_CONTIGUOUS"]
    assert k_cache.dtype == np.uint8 and k_cache.flags["C_CONTIGUOUS"]
    assert v_cache.dtype == np.uint8 and v_cache.flags["C_CONTIGUOUS"]
    H, Hkv, D = num_heads, num_kv_heads, head_dim
    W = qkv.shape[1]
    assert W == (H + 2 * Hkv) * D
    pos = _i32(positions)
    slots = _i32(slot_mapping)
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    keep = [None if a is None else np.ascontiguousarray(a, dtype=np.uint16)
            for a in (bias, q_norm_w, k_norm_w)]
    ptrs = [None if a is None else _ptr(a) for a in keep]
    base = qkv.ctypes.data
    return int(lib().oracle_rope_cache_append_fp8(
        base, W, base + H * D * 2, W, base + (H + Hkv) * D * 2, W,
        _ptr(pos), _ptr(slots), int(pos.shape[0]), _ptr(k_cache), _ptr(v_cache),
        int(k_cache.shape[0]), _ptr(cs), cs.shape[0], H, Hkv, D, block_size,
        ptrs[0], ptrs[1], ptrs[2], float(eps), float(k_scale), float(v_scale)))


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                        num_heads, num_kv_heads, head_dim, block_size, scale=None,
                        cu_seqlens_q=None, partition_tokens=0, nthreads=None):
    """paged_attention over uint8 e4m3 caches read as code * scale."""
    qn = _u16(q)
    if qn.ndim == 3:
        qn = qn.reshape(qn.shape[0], -1)
    kc = np.ascontiguousarray(_as_numpy(k_cache), dtype=np.uint8)
    vc = np.ascontiguousarray(_as_numpy(v_cache), dtype=np.uint8)
    bt = _i32(block_tables)
    cl = _i32(context_lens)
    cu = None if cu_seqlens_q is None else _i32(cu_seqlens_q)
    num_seqs = int(cl.shape[0])
    rows = num_seqs if cu is None else int(cu[-1])
    out = np.zeros((rows, num_heads, head_dim), dtype=np.float64)
    if scale is None:
        scale = float(head_dim) ** -0.5
    err = lib().oracle_paged_attention_fp8(
        _ptr(out), _ptr(qn), qn.shape[1], _ptr(cu), num_seqs, _ptr(kc), _ptr(vc),
        float(k_scale), float(v_scale), int(kc.shape[0]), _ptr(bt), int(bt.shape[1]),
        _ptr(cl), num_heads, num_kv_heads, head_dim, block_size, float(scale),
        int(partition_tokens), int(nthreads or default_threads()))
    if err < 0:
        raise ValueError("bad attention arguments")
    return out, int(err)


def _as_numpy(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().cpu().contiguous().view(torch.uint8).numpy()
    except ImportError:
        pass
    return np.asarray(a)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 payload (uint16), via fp32 then round-to-nearest-even."""
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def bf16_to_f64(u: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(u, dtype=np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
