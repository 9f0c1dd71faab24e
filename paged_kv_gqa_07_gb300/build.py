"""Build the qattn shared library in-tree with nvcc for sm_103a.

``python -m paged_kv_gqa_07_gb300.build`` (or :func:`build`) compiles every
translation unit under ``csrc/`` in parallel and links
``paged_kv_gqa_07_gb300/_build/libqattn.so`` (CUDA runtime linked
statically, the driver API reached through cudaGetDriverEntryPointByVersion,
so nothing but the driver is needed at run time).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libqattn.so")
# The tracing build (-DQATTN_TRACE): the same sources with per-CTA phase
# stamps in the decode and merge kernels (include/qattn_trace.h); used only
# by bench.py --phases, never by the entry points' own library.
TRACE_DIR = os.path.join(BUILD_DIR, "trace")
TRACE_LIB_PATH = os.path.join(TRACE_DIR, "libqattn_trace.so")
SOURCES = ["api.cu", "rope_append.cu", "decode_merge.cu", "paged_decode_tc.cu", "fp8_gather.cu",
           "varlen_prefill.cu", "decode_noalloc.cu", "copy_probe.cu"]
HEADERS = ["common.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the qattn CUDA library cannot be built")


def _deps():
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "qattn.h"))
    deps.append(os.path.join(ROOT, "include", "qattn_trace.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          trace: bool = False) -> str:
    """Compile and link libqattn.so (with trace=True: the tracing build,
    _build/trace/libqattn_trace.so) if any source changed; return its path."""
    lib_path = TRACE_LIB_PATH if trace else LIB_PATH
    out_dir = TRACE_DIR if trace else BUILD_DIR
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = nvcc_path()
    os.makedirs(out_dir, exist_ok=True)
    common = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-I", os.path.join(ROOT, "include")]
    if trace:
        common.append("-DQATTN_TRACE")
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_info or p.returncode != 0):
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    subprocess.run(link, check=True)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                ptxas_info="--ptxas" in sys.argv, trace="--trace" in sys.argv))
