"""Thin Python binding of the qattn C ABI (argument marshalling only).

Each function has the name of the C entry point it calls and forwards
``tensor.data_ptr()``, row strides and the current CUDA stream; all work runs
in the library's CUDA kernels.  A non-zero return code raises
:class:`QattnError`.  There is no fallback: if the library is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

QATTN_OK = 0
QATTN_ERR_INVALID_ARG = 1
QATTN_ERR_UNSUPPORTED = 2
QATTN_ERR_CUDA = 3
QATTN_ERR_WORKSPACE = 4

DEVERR_SLOT = 1
DEVERR_BLOCK = 2
DEVERR_CONTEXT = 4
DEVERR_TIMEOUT = 8
DEVERR_POSITION = 16
DEVERR_PREFIX = 32

EXPORTED = [
    "qattn_status_string",
    "qattn_version",
    "qattn_rope_table_build",
    "qattn_rope_table_build_scaled",
    "qattn_rope_cache_append",
    "qattn_rope_cache_append_ex",
    "qattn_rope_cache_append_fp8",
    "qattn_paged_decode_kernel",
    "qattn_paged_decode_workspace_size",
    "qattn_paged_decode",
    "qattn_paged_decode_fp8",
    "qattn_paged_decode_noalloc",
    "qattn_paged_decode_shared_prefix_workspace_size",
    "qattn_paged_decode_shared_prefix",
    "qattn_paged_decode_shared_prefix_fp8_workspace_size",
    "qattn_paged_decode_shared_prefix_fp8",
    "qattn_varlen_prefill_workspace_size",
    "qattn_varlen_prefill",
    "qattn_varlen_prefill_fp8_workspace_size",
    "qattn_varlen_prefill_fp8",
]


class QattnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status} ({qattn_status_string(status)})")


class qattn_dims(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("scale", ctypes.c_float)]


def make_dims(num_heads, num_kv_heads, head_dim=128, block_size=16, scale=0.0) -> qattn_dims:
    return qattn_dims(int(num_heads), int(num_kv_heads), int(head_dim), int(block_size),
                      float(scale))


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


def load_library(path: str | None = None):
    """Load libqattn.so (must already be built) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"qattn CUDA library not found at {p}; build it with "
                "paged_kv_gqa_07_gb300.build.build() (there is no non-CUDA path)")
        L = ctypes.CDLL(p)
        L.qattn_status_string.argtypes = [ctypes.c_int]
        L.qattn_status_string.restype = ctypes.c_char_p
        L.qattn_version.argtypes = []
        L.qattn_version.restype = ctypes.c_int
        L.qattn_rope_table_build.argtypes = [_P, _I32, _I32, ctypes.c_double]
        L.qattn_rope_table_build.restype = ctypes.c_int
        L.qattn_rope_table_build_scaled.argtypes = [_P, _I32, _I32, ctypes.c_double, _I32,
                                                    ctypes.c_double, _I32]
        L.qattn_rope_table_build_scaled.restype = ctypes.c_int
        L.qattn_rope_cache_append.argtypes = [
            _P, _I64, _P, _I64, _P, _I64, _P, _P, _I32, _P, _P, _I32, _P, _I32, qattn_dims, _P, _P]
        L.qattn_rope_cache_append.restype = ctypes.c_int
        L.qattn_rope_cache_append_ex.argtypes = [
            _P, _I64, _P, _I64, _P, _I64, _P, _P, _I32, _P, _P, _I32, _P, _I32, _P, _P, _P,
            ctypes.c_float, qattn_dims, _P, _P]
        L.qattn_rope_cache_append_ex.restype = ctypes.c_int
        L.qattn_rope_cache_append_fp8.argtypes = [
            _P, _I64, _P, _I64, _P, _I64, _P, _P, _I32, _P, _P, _I32, _P, _I32, _P, _P, _P,
            ctypes.c_float, ctypes.c_float, ctypes.c_float, qattn_dims, _P, _P]
        L.qattn_rope_cache_append_fp8.restype = ctypes.c_int
        L.qattn_paged_decode_kernel.argtypes = [qattn_dims]
        L.qattn_paged_decode_kernel.restype = ctypes.c_int
        L.qattn_paged_decode_workspace_size.argtypes = [_I32, _I32, qattn_dims]
        L.qattn_paged_decode_workspace_size.restype = _SZ
        L.qattn_paged_decode.argtypes = [
            _P, _P, _I64, _P, _P, _I32, _P, _I32, _P, _I32, _I32, qattn_dims, _P, _SZ, _P, _P]
        L.qattn_paged_decode.restype = ctypes.c_int
        L.qattn_paged_decode_fp8.argtypes = [
            _P, _P, _I64, _P, _P, _I32, _P, _I32, _P, _I32, _I32, ctypes.c_float, ctypes.c_float,
            qattn_dims, _P, _SZ, _P, _P]
        L.qattn_paged_decode_fp8.restype = ctypes.c_int
        L.qattn_paged_decode_shared_prefix_workspace_size.argtypes = [_I32, _I32, qattn_dims]
        L.qattn_paged_decode_shared_prefix_workspace_size.restype = _SZ
        L.qattn_paged_decode_shared_prefix.argtypes = [
            _P, _P, _I64, _P, _P, _I32, _P, _I32, _P, _I32, _I32, _I32, qattn_dims, _P, _SZ, _P,
            _P]
        L.qattn_paged_decode_shared_prefix.restype = ctypes.c_int
        L.qattn_paged_decode_shared_prefix_fp8_workspace_size.argtypes = [_I32, _I32, _I32,
                                                                          qattn_dims]
        L.qattn_paged_decode_shared_prefix_fp8_workspace_size.restype = _SZ
        L.qattn_paged_decode_shared_prefix_fp8.argtypes = [
            _P, _P, _I64, _P, _P, _I32, _P, _I32, _P, _I32, _I32, _I32, ctypes.c_float,
            ctypes.c_float, qattn_dims, _P, _SZ, _P, _P]
        L.qattn_paged_decode_shared_prefix_fp8.restype = ctypes.c_int
        L.qattn_varlen_prefill_workspace_size.argtypes = [_I32, _I32, qattn_dims]
        L.qattn_varlen_prefill_workspace_size.restype = _SZ
        L.qattn_varlen_prefill.argtypes = [
            _P, _P, _I64, _P, _I32, _I32, _I32, _P, _P, _I32, _P, _I32, _P, _I32, qattn_dims,
            _P, _SZ, _P, _P]
        L.qattn_varlen_prefill.restype = ctypes.c_int
        L.qattn_varlen_prefill_fp8_workspace_size.argtypes = [_I32, _I32, _I32, qattn_dims]
        L.qattn_varlen_prefill_fp8_workspace_size.restype = _SZ
        L.qattn_varlen_prefill_fp8.argtypes = [
            _P, _P, _I64, _P, _I32, _I32, _I32, _P, _P, _I32, _P, _I32, _P, _I32, _I32,
            ctypes.c_float, ctypes.c_float, qattn_dims, _P, _SZ, _P, _P]
        L.qattn_varlen_prefill_fp8.restype = ctypes.c_int
        if path is None:
            _lib = L
        return L


def lib():
    return _lib if _lib is not None else load_library()


# ---------------------------------------------------------------- helpers --

def _dev_ptr(t: torch.Tensor | None, name: str, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _rows(t: torch.Tensor, name: str):
    """(pointer, row stride in elements) of a 2-D bf16 view with unit inner stride."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D view with unit inner stride")
    return _dev_ptr(t, name, torch.bfloat16), t.stride(0)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(fn: str, rc: int):
    if rc != QATTN_OK:
        raise QattnError(fn, rc)


# ------------------------------------------------------------ entry points --

def qattn_status_string(status: int) -> str:
    return lib().qattn_status_string(int(status)).decode()


def qattn_version() -> int:
    return int(lib().qattn_version())


def qattn_rope_table_build(max_pos: int, head_dim: int, theta: float) -> torch.Tensor:
    """Host-built [max_pos, head_dim] fp32 cos/sin table (CPU tensor)."""
    out = torch.empty((max_pos, head_dim), dtype=torch.float32)
    _check("qattn_rope_table_build",
           lib().qattn_rope_table_build(out.data_ptr(), int(max_pos), int(head_dim), float(theta)))
    return out


QATTN_ROPE_SCALING_NONE, QATTN_ROPE_SCALING_LINEAR, QATTN_ROPE_SCALING_DYNAMIC = 0, 1, 2


def qattn_rope_table_build_scaled(max_pos: int, head_dim: int, theta: float, scaling: int,
                                  factor: float = 1.0, original_max_position: int = 0
                                  ) -> torch.Tensor:
    """Host-built table with rope_scaling (none, linear, dynamic NTK)."""
    out = torch.empty((max_pos, head_dim), dtype=torch.float32)
    _check("qattn_rope_table_build_scaled",
           lib().qattn_rope_table_build_scaled(out.data_ptr(), int(max_pos), int(head_dim),
                                               float(theta), int(scaling), float(factor),
                                               int(original_max_position)))
    return out


def qattn_rope_cache_append(q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin, dims,
                            err_word=None, stream=None):
    qp, qs = _rows(q, "q")
    kp, ks = _rows(k, "k")
    vp, vs = _rows(v, "v")
    rc = lib().qattn_rope_cache_append(
        qp, qs, kp, ks, vp, vs, _dev_ptr(positions, "positions", torch.int32),
        _dev_ptr(slot_mapping, "slot_mapping", torch.int32), int(positions.shape[0]),
        _dev_ptr(k_cache, "k_cache", torch.bfloat16), _dev_ptr(v_cache, "v_cache", torch.bfloat16),
        int(k_cache.shape[0]), _dev_ptr(cos_sin, "cos_sin", torch.float32), int(cos_sin.shape[0]),
        dims, _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_rope_cache_append", rc)


def qattn_rope_cache_append_ex(q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin, dims,
                               qkv_bias=None, q_norm_weight=None, k_norm_weight=None,
                               norm_eps=1e-6, err_word=None, stream=None):
    """qattn_rope_cache_append with the qkv projection bias and the Qwen3
    per-head q/k RMSNorms applied before the rotation (None skips a step)."""
    qp, qs = _rows(q, "q")
    kp, ks = _rows(k, "k")
    vp, vs = _rows(v, "v")
    rc = lib().qattn_rope_cache_append_ex(
        qp, qs, kp, ks, vp, vs, _dev_ptr(positions, "positions", torch.int32),
        _dev_ptr(slot_mapping, "slot_mapping", torch.int32), int(positions.shape[0]),
        _dev_ptr(k_cache, "k_cache", torch.bfloat16), _dev_ptr(v_cache, "v_cache", torch.bfloat16),
        int(k_cache.shape[0]), _dev_ptr(cos_sin, "cos_sin", torch.float32), int(cos_sin.shape[0]),
        _dev_ptr(qkv_bias, "qkv_bias", torch.bfloat16),
        _dev_ptr(q_norm_weight, "q_norm_weight", torch.bfloat16),
        _dev_ptr(k_norm_weight, "k_norm_weight", torch.bfloat16), float(norm_eps), dims,
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_rope_cache_append_ex", rc)


def _fp8_ptr(t: torch.Tensor, name: str):
    """Device pointer of an e4m3 cache (uint8 or float8_e4m3fn storage)."""
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError(f"{name} must be uint8 or float8_e4m3fn, got {t.dtype}")
    return _dev_ptr(t, name)


def qattn_rope_cache_append_fp8(q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin,
                                k_scale, v_scale, dims, qkv_bias=None, q_norm_weight=None,
                                k_norm_weight=None, norm_eps=1e-6, err_word=None, stream=None):
    """qattn_rope_cache_append_ex into e4m3 caches: keys and values stored
    as e4m3(x / k_scale), e4m3(x / v_scale)."""
    qp, qs = _rows(q, "q")
    kp, ks = _rows(k, "k")
    vp, vs = _rows(v, "v")
    rc = lib().qattn_rope_cache_append_fp8(
        qp, qs, kp, ks, vp, vs, _dev_ptr(positions, "positions", torch.int32),
        _dev_ptr(slot_mapping, "slot_mapping", torch.int32), int(positions.shape[0]),
        _fp8_ptr(k_cache, "k_cache"), _fp8_ptr(v_cache, "v_cache"),
        int(k_cache.shape[0]), _dev_ptr(cos_sin, "cos_sin", torch.float32), int(cos_sin.shape[0]),
        _dev_ptr(qkv_bias, "qkv_bias", torch.bfloat16),
        _dev_ptr(q_norm_weight, "q_norm_weight", torch.bfloat16),
        _dev_ptr(k_norm_weight, "k_norm_weight", torch.bfloat16), float(norm_eps),
        float(k_scale), float(v_scale), dims,
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_rope_cache_append_fp8", rc)


QATTN_DECODE_CUDA_CORE = 0
QATTN_DECODE_TENSOR_CORE = 1


def qattn_paged_decode_kernel(dims) -> int:
    """QATTN_DECODE_CUDA_CORE or QATTN_DECODE_TENSOR_CORE: the decode kernel used for dims."""
    return int(lib().qattn_paged_decode_kernel(dims))


def qattn_paged_decode_workspace_size(num_seqs: int, max_context_len: int, dims) -> int:
    return int(lib().qattn_paged_decode_workspace_size(int(num_seqs), int(max_context_len), dims))


def qattn_paged_decode(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                       dims, workspace, err_word=None, stream=None):
    qp, qs = _rows(q, "q")
    rc = lib().qattn_paged_decode(
        _dev_ptr(out, "out", torch.bfloat16), qp, qs,
        _dev_ptr(k_cache, "k_cache", torch.bfloat16), _dev_ptr(v_cache, "v_cache", torch.bfloat16),
        int(k_cache.shape[0]), _dev_ptr(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev_ptr(context_lens, "context_lens", torch.int32),
        int(context_lens.shape[0]), int(max_context_len), dims,
        _dev_ptr(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_paged_decode", rc)


def qattn_paged_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, k_scale, v_scale, dims, workspace, err_word=None,
                           stream=None):
    """qattn_paged_decode over e4m3 caches read as code * scale."""
    qp, qs = _rows(q, "q")
    rc = lib().qattn_paged_decode_fp8(
        _dev_ptr(out, "out", torch.bfloat16), qp, qs,
        _fp8_ptr(k_cache, "k_cache"), _fp8_ptr(v_cache, "v_cache"),
        int(k_cache.shape[0]), _dev_ptr(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev_ptr(context_lens, "context_lens", torch.int32),
        int(context_lens.shape[0]), int(max_context_len), float(k_scale), float(v_scale), dims,
        _dev_ptr(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_paged_decode_fp8", rc)


def qattn_paged_decode_shared_prefix_workspace_size(num_seqs: int, max_context_len: int,
                                                    dims) -> int:
    return int(lib().qattn_paged_decode_shared_prefix_workspace_size(
        int(num_seqs), int(max_context_len), dims))


def qattn_paged_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens,
                                     max_context_len, shared_prefix_len, dims, workspace,
                                     err_word=None, stream=None):
    qp, qs = _rows(q, "q")
    rc = lib().qattn_paged_decode_shared_prefix(
        _dev_ptr(out, "out", torch.bfloat16), qp, qs,
        _dev_ptr(k_cache, "k_cache", torch.bfloat16), _dev_ptr(v_cache, "v_cache", torch.bfloat16),
        int(k_cache.shape[0]), _dev_ptr(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev_ptr(context_lens, "context_lens", torch.int32),
        int(context_lens.shape[0]), int(max_context_len), int(shared_prefix_len), dims,
        _dev_ptr(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_paged_decode_shared_prefix", rc)


def qattn_varlen_prefill_workspace_size(num_seqs: int, max_context_len: int, dims) -> int:
    return int(lib().qattn_varlen_prefill_workspace_size(int(num_seqs), int(max_context_len), dims))


def qattn_varlen_prefill(out, q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables,
                         context_lens, max_context_len, dims, workspace, err_word=None,
                         stream=None):
    qp, qs = _rows(q, "q")
    rc = lib().qattn_varlen_prefill(
        _dev_ptr(out, "out", torch.bfloat16), qp, qs,
        _dev_ptr(cu_seqlens_q, "cu_seqlens_q", torch.int32), int(cu_seqlens_q.shape[0]) - 1,
        int(q.shape[0]), int(max_q_len),
        _dev_ptr(k_cache, "k_cache", torch.bfloat16), _dev_ptr(v_cache, "v_cache", torch.bfloat16),
        int(k_cache.shape[0]), _dev_ptr(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev_ptr(context_lens, "context_lens", torch.int32),
        int(max_context_len), dims, _dev_ptr(workspace, "workspace"),
        int(workspace.numel() * workspace.element_size()),
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_varlen_prefill", rc)



def qattn_varlen_prefill_fp8_workspace_size(num_seqs: int, num_prefill_seqs: int,
                                            max_context_len: int, dims) -> int:
    return int(lib().qattn_varlen_prefill_fp8_workspace_size(
        int(num_seqs), int(num_prefill_seqs), int(max_context_len), dims))


def qattn_varlen_prefill_fp8(out, q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables,
                             context_lens, max_context_len, num_prefill_seqs, k_scale, v_scale,
                             dims, workspace, err_word=None, stream=None):
    """qattn_varlen_prefill over e4m3 caches read as code * scale."""
    qp, qs = _rows(q, "q")
    rc = lib().qattn_varlen_prefill_fp8(
        _dev_ptr(out, "out", torch.bfloat16), qp, qs,
        _dev_ptr(cu_seqlens_q, "cu_seqlens_q", torch.int32), int(cu_seqlens_q.shape[0]) - 1,
        int(q.shape[0]), int(max_q_len), _fp8_ptr(k_cache, "k_cache"),
        _fp8_ptr(v_cache, "v_cache"), int(k_cache.shape[0]),
        _dev_ptr(block_tables, "block_tables", torch.int32), int(block_tables.shape[1]),
        _dev_ptr(context_lens, "context_lens", torch.int32), int(max_context_len),
        int(num_prefill_seqs), float(k_scale), float(v_scale), dims,
        _dev_ptr(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_varlen_prefill_fp8", rc)


def qattn_paged_decode_shared_prefix_fp8_workspace_size(num_seqs: int, max_context_len: int,
                                                        shared_prefix_len: int, dims) -> int:
    return int(lib().qattn_paged_decode_shared_prefix_fp8_workspace_size(
        int(num_seqs), int(max_context_len), int(shared_prefix_len), dims))


def qattn_paged_decode_shared_prefix_fp8(out, q, k_cache, v_cache, block_tables, context_lens,
                                         max_context_len, shared_prefix_len, k_scale, v_scale,
                                         dims, workspace, err_word=None, stream=None):
    """qattn_paged_decode_shared_prefix over e4m3 caches read as code * scale."""
    qp, qs = _rows(q, "q")
    rc = lib().qattn_paged_decode_shared_prefix_fp8(
        _dev_ptr(out, "out", torch.bfloat16), qp, qs,
        _fp8_ptr(k_cache, "k_cache"), _fp8_ptr(v_cache, "v_cache"),
        int(k_cache.shape[0]), _dev_ptr(block_tables, "block_tables", torch.int32),
        int(block_tables.shape[1]), _dev_ptr(context_lens, "context_lens", torch.int32),
        int(context_lens.shape[0]), int(max_context_len), int(shared_prefix_len),
        float(k_scale), float(v_scale), dims, _dev_ptr(workspace, "workspace"),
        int(workspace.numel() * workspace.element_size()),
        _dev_ptr(err_word, "err_word", torch.int32), _stream(stream))
    _check("qattn_paged_decode_shared_prefix_fp8", rc)
