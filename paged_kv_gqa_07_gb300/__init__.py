"""qattn: the attention step of a Qwen2 decoder layer over a block-paged KV
cache (rotate-half RoPE + cache append, paged GQA decode, causal varlen
prefill) as hand-written sm_103a CUDA kernels behind a C ABI.

``qattn`` is the ctypes binding of that ABI (the library loads on first
use), ``build`` compiles the library in-tree, ``workloads`` builds seeded
synthetic inputs.
"""
from . import build, qattn, workloads  # noqa: F401

__all__ = ["build", "workloads", "qattn"]
