"""Thin Python binding of the qattn C ABI (argument marshalling only).

Each function has the name of the C entry point it calls and forwards
``tensor.data_ptr()``, row strides and the current CUDA stream; all work runs
in the library's CUDA kernels.  Since the C ABI sees only pointers, each
tensor's device, dtype, shape and layout are first checked against the call's
dims (:class:`QattnArgError`, status QATTN_ERR_INVALID_ARG, if they disagree).
A non-zero return code raises :class:`QattnError`.  There is no fallback: if
the library is missing the first call raises.
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
    "qattn_debug_decode_faults",
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


class QattnArgError(QattnError, ValueError):
    """A tensor the binding refuses before calling the library (status
    QATTN_ERR_INVALID_ARG): its device, dtype, shape or layout disagrees with
    what the C ABI assumes of the pointer it would pass."""

    def __init__(self, fn: str, detail: str):
        self.status = QATTN_ERR_INVALID_ARG
        RuntimeError.__init__(self, f"{fn}: {detail}")


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
        L.qattn_debug_decode_faults.argtypes = [_I64, _I32]
        L.qattn_debug_decode_faults.restype = ctypes.c_int
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
        L.qattn_paged_decode_noalloc.argtypes = [
            _P, _P, _I64, _P, _P, _I32, _P, _I32, _P, _I32, _I32, qattn_dims, _P, _P]
        L.qattn_paged_decode_noalloc.restype = ctypes.c_int
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
#
# The C ABI sees plain pointers.  The layouts it assumes of them (include/
# qattn.h) are checked here, where the tensors' metadata is still at hand, so
# that a tensor of the wrong shape, dtype, layout or device is refused instead
# of being read or written out of bounds on the device.

_BF16 = (torch.bfloat16,)
_I32T = (torch.int32,)
_F32 = (torch.float32,)
_E4M3 = (torch.uint8, torch.float8_e4m3fn)


class _Args:
    """The tensors of one call: checked, then reduced to device pointers."""

    def __init__(self, fn: str, dims=None):
        self.fn = fn
        self.dims = dims
        self.dev = None  # the current device, looked up at the first tensor

    def bad(self, detail: str):
        raise QattnArgError(self.fn, detail)

    def ptr(self, t, name, dtypes=None, numel=0, contiguous=True):
        """Device pointer of `t` (None stays None): of one of `dtypes`,
        contiguous unless told otherwise, >= numel elements, on the current
        device."""
        if t is None:
            return None
        if dtypes is not None and t.dtype not in dtypes:
            self.bad(f"{name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
        if contiguous and not t.is_contiguous():
            self.bad(f"{name} must be contiguous")
        if numel and t.numel() < numel:
            self.bad(f"{name} has {t.numel()} elements, needs at least {numel}")
        return self.device_ptr(t, name)

    def device_ptr(self, t, name):
        if not t.is_cuda:
            self.bad(f"{name} must be a CUDA tensor, got {t.device}")
        if self.dev is None:
            self.dev = torch.cuda.current_device()
        if t.device.index != self.dev:
            self.bad(f"{name} is on {t.device}, not on the current device cuda:{self.dev}")
        return t.data_ptr()

    def rows(self, t, name, rows, cols):
        """(pointer, row stride in elements) of a bf16 row view: 2-D with unit
        inner stride, at least `rows` rows of at least `cols` elements."""
        if t.dim() != 2 or t.stride(1) != 1:
            self.bad(f"{name} must be a 2-D view with unit inner stride")
        if t.shape[0] < rows or t.shape[1] < cols:
            self.bad(f"{name} is {tuple(t.shape)}, needs at least {rows} rows of {cols}")
        return self.ptr(t, name, _BF16, contiguous=False), t.stride(0)

    def vec(self, t, name, n=0):
        """A contiguous 1-D int32 vector of at least n entries."""
        if t.dim() != 1:
            self.bad(f"{name} must be 1-D, got shape {tuple(t.shape)}")
        return self.ptr(t, name, _I32T, numel=n)

    def cache(self, k, v, fp8=False):
        """K and V caches: contiguous [num_blocks, Hkv, block_size, head_dim]
        (bf16, or e4m3 codes); returns their pointers and num_blocks."""
        d = self.dims
        want = (d.num_kv_heads, d.block_size, d.head_dim)
        for t, name in ((k, "k_cache"), (v, "v_cache")):
            if t.dim() != 4 or tuple(t.shape[1:]) != want:
                self.bad(f"{name} is {tuple(t.shape)}, must be [num_blocks, {want[0]}, "
                         f"{want[1]}, {want[2]}]")
        if k.shape[0] != v.shape[0]:
            self.bad("k_cache and v_cache must hold the same number of blocks")
        dt = _E4M3 if fp8 else _BF16
        return self.ptr(k, "k_cache", dt), self.ptr(v, "v_cache", dt), int(k.shape[0])

    def table(self, bt, num_seqs):
        """Block tables: contiguous int32 [>= num_seqs, max_blocks_per_seq]."""
        if bt.dim() != 2 or bt.shape[0] < num_seqs:
            self.bad(f"block_tables is {tuple(bt.shape)}, needs [>= {num_seqs}, "
                     "max_blocks_per_seq]")
        return self.ptr(bt, "block_tables", _I32T), int(bt.shape[1])

    def out(self, t, rows):
        """Output rows: contiguous bf16 [rows, num_heads, head_dim]."""
        d = self.dims
        return self.ptr(t, "out", _BF16, numel=rows * d.num_heads * d.head_dim)

    def workspace(self, t):
        """(pointer, bytes) of a contiguous workspace of any dtype."""
        return self.ptr(t, "workspace"), int(t.numel() * t.element_size())

    def err(self, t):
        return self.ptr(t, "err_word", _I32T, numel=1)

    def cos_sin(self, t):
        """The cos/sin table: contiguous fp32 [max_pos, head_dim]; returns
        its pointer and max_pos."""
        if t.dim() != 2 or t.shape[1] != self.dims.head_dim:
            self.bad(f"cos_sin is {tuple(t.shape)}, must be [max_pos, {self.dims.head_dim}]")
        return self.ptr(t, "cos_sin", _F32), int(t.shape[0])


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


def _append_args(a: _Args, q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin, fp8,
                 qkv_bias=None, q_norm_weight=None, k_norm_weight=None):
    """The argument list shared by the three append entry points, up to the
    optional extras: q/k/v rows, positions, slots, caches and the table."""
    d = a.dims
    pos = a.vec(positions, "positions")
    T = int(positions.shape[0])
    qp, qs = a.rows(q, "q", T, d.num_heads * d.head_dim)
    kp, ks = a.rows(k, "k", T, d.num_kv_heads * d.head_dim)
    vp, vs = a.rows(v, "v", T, d.num_kv_heads * d.head_dim)
    slots = a.vec(slot_mapping, "slot_mapping", T)
    kc, vc, nb = a.cache(k_cache, v_cache, fp8)
    cs, max_pos = a.cos_sin(cos_sin)
    args = [qp, qs, kp, ks, vp, vs, pos, slots, T, kc, vc, nb, cs, max_pos]
    extras = [a.ptr(qkv_bias, "qkv_bias", _BF16,
                    numel=(d.num_heads + 2 * d.num_kv_heads) * d.head_dim),
              a.ptr(q_norm_weight, "q_norm_weight", _BF16, numel=d.head_dim),
              a.ptr(k_norm_weight, "k_norm_weight", _BF16, numel=d.head_dim)]
    return args, extras


def qattn_rope_cache_append(q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin, dims,
                            err_word=None, stream=None):
    fn = "qattn_rope_cache_append"
    a = _Args(fn, dims)
    args, _ = _append_args(a, q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin, False)
    _check(fn, lib().qattn_rope_cache_append(*args, dims, a.err(err_word), _stream(stream)))


def qattn_rope_cache_append_ex(q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin, dims,
                               qkv_bias=None, q_norm_weight=None, k_norm_weight=None,
                               norm_eps=1e-6, err_word=None, stream=None):
    """qattn_rope_cache_append with the qkv projection bias and the Qwen3
    per-head q/k RMSNorms applied before the rotation (None skips a step)."""
    fn = "qattn_rope_cache_append_ex"
    a = _Args(fn, dims)
    args, extras = _append_args(a, q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin,
                                False, qkv_bias, q_norm_weight, k_norm_weight)
    _check(fn, lib().qattn_rope_cache_append_ex(*args, *extras, float(norm_eps), dims,
                                                a.err(err_word), _stream(stream)))


def qattn_rope_cache_append_fp8(q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin,
                                k_scale, v_scale, dims, qkv_bias=None, q_norm_weight=None,
                                k_norm_weight=None, norm_eps=1e-6, err_word=None, stream=None):
    """qattn_rope_cache_append_ex into e4m3 caches (uint8 or float8_e4m3fn
    storage): keys and values stored as e4m3(x / k_scale), e4m3(x / v_scale)."""
    fn = "qattn_rope_cache_append_fp8"
    a = _Args(fn, dims)
    args, extras = _append_args(a, q, k, v, positions, slot_mapping, k_cache, v_cache, cos_sin,
                                True, qkv_bias, q_norm_weight, k_norm_weight)
    _check(fn, lib().qattn_rope_cache_append_fp8(*args, *extras, float(norm_eps), float(k_scale),
                                                 float(v_scale), dims, a.err(err_word),
                                                 _stream(stream)))


def qattn_debug_decode_faults(wait_limit_ns: int, skip_k_copy: int) -> None:
    """Testing hook: the wait limit of later decode launches (0: default)
    and the K copy the decode kernel's first CTA skips (-1: none)."""
    _check("qattn_debug_decode_faults",
           lib().qattn_debug_decode_faults(int(wait_limit_ns), int(skip_k_copy)))


def qattn_paged_decode_workspace_size(num_seqs: int, max_context_len: int, dims) -> int:
    return int(lib().qattn_paged_decode_workspace_size(int(num_seqs), int(max_context_len), dims))


def _decode_args(a: _Args, out, q, k_cache, v_cache, block_tables, context_lens, fp8):
    """out, q rows, caches, tables and lengths of a decode call (one query
    row per sequence)."""
    d = a.dims
    lens = a.vec(context_lens, "context_lens")
    B = int(context_lens.shape[0])
    qp, qs = a.rows(q, "q", B, d.num_heads * d.head_dim)
    kc, vc, nb = a.cache(k_cache, v_cache, fp8)
    bt, mbps = a.table(block_tables, B)
    return [a.out(out, B), qp, qs, kc, vc, nb, bt, mbps, lens, B]


def qattn_paged_decode(out, q, k_cache, v_cache, block_tables, context_lens, max_context_len,
                       dims, workspace, err_word=None, stream=None):
    fn = "qattn_paged_decode"
    a = _Args(fn, dims)
    args = _decode_args(a, out, q, k_cache, v_cache, block_tables, context_lens, False)
    _check(fn, lib().qattn_paged_decode(*args, int(max_context_len), dims, *a.workspace(workspace),
                                        a.err(err_word), _stream(stream)))


def qattn_paged_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens,
                           max_context_len, k_scale, v_scale, dims, workspace, err_word=None,
                           stream=None):
    """qattn_paged_decode over e4m3 caches read as code * scale."""
    fn = "qattn_paged_decode_fp8"
    a = _Args(fn, dims)
    args = _decode_args(a, out, q, k_cache, v_cache, block_tables, context_lens, True)
    _check(fn, lib().qattn_paged_decode_fp8(*args, int(max_context_len), float(k_scale),
                                            float(v_scale), dims, *a.workspace(workspace),
                                            a.err(err_word), _stream(stream)))


def qattn_paged_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                               max_context_len, dims, err_word=None, stream=None):
    """qattn_paged_decode with its split-KV scratch in the library's own
    device array (no workspace); calls must not overlap on the GPU."""
    fn = "qattn_paged_decode_noalloc"
    a = _Args(fn, dims)
    args = _decode_args(a, out, q, k_cache, v_cache, block_tables, context_lens, False)
    _check(fn, lib().qattn_paged_decode_noalloc(*args, int(max_context_len), dims,
                                                a.err(err_word), _stream(stream)))


def qattn_paged_decode_shared_prefix_workspace_size(num_seqs: int, max_context_len: int,
                                                    dims) -> int:
    return int(lib().qattn_paged_decode_shared_prefix_workspace_size(
        int(num_seqs), int(max_context_len), dims))


def qattn_paged_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens,
                                     max_context_len, shared_prefix_len, dims, workspace,
                                     err_word=None, stream=None):
    fn = "qattn_paged_decode_shared_prefix"
    a = _Args(fn, dims)
    args = _decode_args(a, out, q, k_cache, v_cache, block_tables, context_lens, False)
    _check(fn, lib().qattn_paged_decode_shared_prefix(
        *args, int(max_context_len), int(shared_prefix_len), dims, *a.workspace(workspace),
        a.err(err_word), _stream(stream)))


def qattn_paged_decode_shared_prefix_fp8_workspace_size(num_seqs: int, max_context_len: int,
                                                        shared_prefix_len: int, dims) -> int:
    return int(lib().qattn_paged_decode_shared_prefix_fp8_workspace_size(
        int(num_seqs), int(max_context_len), int(shared_prefix_len), dims))


def qattn_paged_decode_shared_prefix_fp8(out, q, k_cache, v_cache, block_tables, context_lens,
                                         max_context_len, shared_prefix_len, k_scale, v_scale,
                                         dims, workspace, err_word=None, stream=None):
    """qattn_paged_decode_shared_prefix over e4m3 caches read as code * scale."""
    fn = "qattn_paged_decode_shared_prefix_fp8"
    a = _Args(fn, dims)
    args = _decode_args(a, out, q, k_cache, v_cache, block_tables, context_lens, True)
    _check(fn, lib().qattn_paged_decode_shared_prefix_fp8(
        *args, int(max_context_len), int(shared_prefix_len), float(k_scale), float(v_scale),
        dims, *a.workspace(workspace), a.err(err_word), _stream(stream)))


def qattn_varlen_prefill_workspace_size(num_seqs: int, max_context_len: int, dims) -> int:
    return int(lib().qattn_varlen_prefill_workspace_size(int(num_seqs), int(max_context_len), dims))


def _varlen_args(a: _Args, out, q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables,
                 context_lens, fp8):
    """out, q rows, sequence offsets, caches, tables and lengths of a varlen
    call: q holds total_q = q.shape[0] rows, cu_seqlens_q num_seqs + 1."""
    d = a.dims
    cu = a.vec(cu_seqlens_q, "cu_seqlens_q", 1)
    S = int(cu_seqlens_q.shape[0]) - 1
    total_q = int(q.shape[0]) if q.dim() == 2 else 0
    qp, qs = a.rows(q, "q", total_q, d.num_heads * d.head_dim)
    kc, vc, nb = a.cache(k_cache, v_cache, fp8)
    bt, mbps = a.table(block_tables, S)
    lens = a.vec(context_lens, "context_lens", S)
    return [a.out(out, total_q), qp, qs, cu, S, total_q, int(max_q_len), kc, vc, nb, bt, mbps,
            lens]


def qattn_varlen_prefill(out, q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables,
                         context_lens, max_context_len, dims, workspace, err_word=None,
                         stream=None):
    fn = "qattn_varlen_prefill"
    a = _Args(fn, dims)
    args = _varlen_args(a, out, q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables,
                        context_lens, False)
    _check(fn, lib().qattn_varlen_prefill(*args, int(max_context_len), dims,
                                          *a.workspace(workspace), a.err(err_word),
                                          _stream(stream)))


def qattn_varlen_prefill_fp8_workspace_size(num_seqs: int, num_prefill_seqs: int,
                                            max_context_len: int, dims) -> int:
    return int(lib().qattn_varlen_prefill_fp8_workspace_size(
        int(num_seqs), int(num_prefill_seqs), int(max_context_len), dims))


def qattn_varlen_prefill_fp8(out, q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables,
                             context_lens, max_context_len, num_prefill_seqs, k_scale, v_scale,
                             dims, workspace, err_word=None, stream=None):
    """qattn_varlen_prefill over e4m3 caches read as code * scale."""
    fn = "qattn_varlen_prefill_fp8"
    a = _Args(fn, dims)
    args = _varlen_args(a, out, q, cu_seqlens_q, max_q_len, k_cache, v_cache, block_tables,
                        context_lens, True)
    _check(fn, lib().qattn_varlen_prefill_fp8(*args, int(max_context_len), int(num_prefill_seqs),
                                              float(k_scale), float(v_scale), dims,
                                              *a.workspace(workspace), a.err(err_word),
                                              _stream(stream)))
