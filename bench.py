"""Benchmark of one attention step over a paged KV cache on GB300.

A step is the whole path for one batch: RoPE + cache append of the new tokens
(qattn_rope_cache_append), then paged GQA attention (qattn_paged_decode for a
decode workload, qattn_varlen_prefill for a mixed one).  Inputs are resident
in HBM when timing starts; L2 is flushed (a 512 MB buffer is written)
before every timed step, and each step is timed with CUDA events on the
launching stream.  The headline workload is the Qwen2-7B-shaped decode step
(28 query / 4 KV heads, head_dim 128, batch 64, contexts U[128, 4096], block
size 16, random block placement).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
step shards by sequence with no exchange), the time is the max over ranks and
the value counts all ranks' bytes ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_gqa_07_gb300 import workloads as W  # noqa: E402

METRIC = "paged GQA decode: KV HBM GB/s (% of GB300 peak), seqs/s; prefill tokens/s"
DEFAULT_WORKLOAD = "qwen2_7b_decode_b64"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.WORKLOAD_NAMES)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--append-sweep", action="store_true",
                   help="supplementary: time RoPE + append alone at 16k and 64k new tokens "
                        "(Qwen2-7B heads), one JSON line per size")
    p.add_argument("--block-size", type=int, choices=[16, 32, 64], default=16,
                   help="cache block size of the decode / mixed workloads")
    p.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                   help="cache dtype: bf16, or e4m3 codes with a per-tensor scale")
    p.add_argument("--extras", choices=["none", "bias", "qknorm", "both"], default="none",
                   help="add the qkv projection bias and/or the Qwen3 q/k RMSNorms to the "
                        "RoPE + append step (synthetic weights)")
    return p.parse_args()


# ----------------------------------------------------------- distributed --

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local_rank)
            dist.init_process_group(backend)
            self.pg = dist

    @classmethod
    def single(cls):
        d = cls.__new__(cls)
        d.world, d.rank, d.local_rank, d.pg = int(os.environ.get("WORLD_SIZE", "1")), 0, 0, None
        return d

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if self.pg is None:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_index: int, enabled=True):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu = ids[local_index] if local_index < len(ids) else str(local_index)
        self.enabled = enabled
        self.proc = None
        self.lines = []

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ peaks etc --

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_gqa_07_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, sha: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on
    this workload, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha") != sha:
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ----------------------------------------------------------------- ours --

def run_ours(args, dist: Dist):
    import numpy as np  # noqa: F401
    from paged_kv_gqa_07_gb300 import build as B
    from paged_kv_gqa_07_gb300 import qattn as Q

    B.build()
    Q.load_library()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    w = W.build(args.workload, seed=W.SEED_BASE + W.WORKLOAD_NAMES.index(args.workload) + 1000 * dist.rank,
                block_size=args.block_size)
    fp8 = args.kv == "fp8"
    if fp8:
        w = W.with_fp8_cache(w)
    ks, vs = W.FP8_K_SCALE, W.FP8_V_SCALE
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    dims = Q.make_dims(H, Hkv, D, BS)
    g = W.to_device(w, dev)
    qkv0 = g.qkv.clone()
    table = Q.qattn_rope_table_build(w.max_pos, D, w.theta).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    decode = w.is_decode
    max_ctx = w.max_context_len
    # a decode batch on a shared cached prefix takes the shared-prefix entry point
    prefix = w.shared_prefix_tokens if decode else 0
    n_prefill = sum(1 for n in w.q_lens if n >= 2)
    if prefix and fp8:
        ws_size = Q.qattn_paged_decode_shared_prefix_fp8_workspace_size(w.num_seqs, max_ctx,
                                                                         prefix, dims)
    elif not decode and fp8:
        ws_size = Q.qattn_varlen_prefill_fp8_workspace_size(w.num_seqs, n_prefill, max_ctx, dims)
    elif prefix:
        ws_size = Q.qattn_paged_decode_shared_prefix_workspace_size(w.num_seqs, max_ctx, dims)
    elif decode:
        ws_size = Q.qattn_paged_decode_workspace_size(w.num_seqs, max_ctx, dims)
    else:
        ws_size = Q.qattn_varlen_prefill_workspace_size(w.num_seqs, max_ctx, dims)
    ws = torch.empty(max(ws_size, 256), dtype=torch.uint8, device=dev)
    out = torch.empty((w.num_tokens, H, D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    gx = torch.Generator().manual_seed(W.SEED_BASE + 77)
    bias = qn = kn = None
    if args.extras in ("bias", "both"):
        bias = (0.5 * torch.randn((H + 2 * Hkv) * D, generator=gx)).to(torch.bfloat16).to(dev)
    if args.extras in ("qknorm", "both"):
        qn = (1.0 + 0.2 * torch.randn(D, generator=gx)).to(torch.bfloat16).to(dev)
        kn = (1.0 + 0.2 * torch.randn(D, generator=gx)).to(torch.bfloat16).to(dev)

    def append():
        if fp8:
            Q.qattn_rope_cache_append_fp8(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                          g.slot_mapping, g.k_cache, g.v_cache, table, ks, vs,
                                          dims, qkv_bias=bias, q_norm_weight=qn,
                                          k_norm_weight=kn, err_word=err)
        elif args.extras == "none":
            Q.qattn_rope_cache_append(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                      g.slot_mapping, g.k_cache, g.v_cache, table, dims, err)
        else:
            Q.qattn_rope_cache_append_ex(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                         g.slot_mapping, g.k_cache, g.v_cache, table, dims,
                                         qkv_bias=bias, q_norm_weight=qn, k_norm_weight=kn,
                                         err_word=err)

    def attend():
        if prefix and fp8:
            Q.qattn_paged_decode_shared_prefix_fp8(out, g.q_view(), g.k_cache, g.v_cache,
                                                   g.block_tables, g.context_lens, max_ctx,
                                                   prefix, ks, vs, dims, ws, err)
        elif not decode and fp8:
            Q.qattn_varlen_prefill_fp8(out, g.q_view(), g.cu_seqlens_q, w.max_q_len, g.k_cache,
                                       g.v_cache, g.block_tables, g.context_lens, max_ctx,
                                       n_prefill, ks, vs, dims, ws, err)
        elif prefix:
            Q.qattn_paged_decode_shared_prefix(out, g.q_view(), g.k_cache, g.v_cache,
                                               g.block_tables, g.context_lens, max_ctx, prefix,
                                               dims, ws, err)
        elif fp8:
            Q.qattn_paged_decode_fp8(out, g.q_view(), g.k_cache, g.v_cache, g.block_tables,
                                     g.context_lens, max_ctx, ks, vs, dims, ws, err)
        elif decode:
            Q.qattn_paged_decode(out, g.q_view(), g.k_cache, g.v_cache, g.block_tables,
                                 g.context_lens, max_ctx, dims, ws, err)
        else:
            Q.qattn_varlen_prefill(out, g.q_view(), g.cu_seqlens_q, w.max_q_len, g.k_cache,
                                   g.v_cache, g.block_tables, g.context_lens, max_ctx, dims, ws,
                                   err)

    for _ in range(args.warmup):
        g.qkv.copy_(qkv0)
        append()
        attend()
    torch.cuda.synchronize(dev)

    # (A) the step: events only at step boundaries, so the attention kernel
    # may overlap the append kernel's tail (programmatic dependent launch).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    with ClockSampler(dev.index, enabled=not args.no_clocks) as clocks:
        dist.barrier()
        torch.cuda.synchronize(dev)
        for s in range(args.steps):
            flush.fill_(s & 0xff)        # evict the cache and KV from L2
            g.qkv.copy_(qkv0)            # every step starts from the same rows
            ev[s][0].record(stream)
            append()
            attend()
            ev[s][1].record(stream)
        torch.cuda.synchronize(dev)
        dist.barrier()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    step_ms = [ev[s][0].elapsed_time(ev[s][1]) for s in range(args.steps)]

    # (B) the attention call alone (its kernels, on the launching stream), L2
    # flushed before each: the roofline's kernel duration.  (C) the append.
    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for i in range(n):
            flush.fill_(i & 0xff)
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in evs]
    attn_ms = timed(attend, args.steps)
    app_ms = timed(append, args.steps)
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"
    local_total_ms = sum(step_ms)
    total_ms = dist.max(local_total_ms)
    ms_per_step = total_ms / args.steps

    kv_bytes = w.kv_bytes_read()
    qo_bytes = 2 * w.num_tokens * H * D * 2
    all_kv = dist.sum(kv_bytes)
    value = all_kv * args.steps / (total_ms * 1e-3) / 1e9
    seqs_per_s = dist.sum(w.num_seqs) * args.steps / (total_ms * 1e-3)
    tokens_per_s = dist.sum(w.num_tokens) * args.steps / (total_ms * 1e-3)

    hbm_peak, tf_peak, peak_kind = measured_peaks()
    attn_avg_s = statistics.mean(attn_ms) * 1e-3
    result = {}
    if prefix:
        # HBM-bound on the distinct blocks: each is read from DRAM once
        alg = w.unique_kv_bytes() + qo_bytes
        achieved = alg / attn_avg_s / 1e9
        result["roofline"] = {"bound": "hbm",
                              "kernel": "varlen_prefill_kernel (prefix pass) + paged_decode",
                              "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                              "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                              "traffic": None, "algorithmic_bytes_per_launch": alg,
                              "logical_kv_bytes_per_launch": kv_bytes}
    elif decode:
        alg = kv_bytes + qo_bytes
        achieved = alg / attn_avg_s / 1e9
        if fp8 or Q.qattn_paged_decode_kernel(dims) == Q.QATTN_DECODE_TENSOR_CORE:
            kname, src = "paged_decode_tc_kernel", "paged_decode_tc.cu"
        else:
            kname, src = "paged_decode_kernel", "paged_decode.cu"
        sha = kernel_source_sha([src, "common.cuh", "internal.h"])
        traffic = profiled_traffic(kname + ("_fp8" if fp8 else ""), args.workload, sha)
        result["roofline"] = {"bound": "hbm", "kernel": kname,
                              "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                              "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                              "traffic": traffic, "algorithmic_bytes_per_launch": alg}
    else:
        flops = 4 * D * w.causal_pairs()
        achieved = flops / attn_avg_s / 1e12
        result["roofline"] = {"bound": "tensor", "kernel": "varlen prefill + decode rows",
                              "achieved": round(achieved, 2), "peak": tf_peak, "unit": "TFLOP/s",
                              "frac": round(achieved / tf_peak, 4), "peak_kind": peak_kind,
                              "traffic": None, "algorithmic_flops_per_launch": flops}

    # ---- end to end through the C ABI with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, dims, g, table, ws, err, dev, decode, max_ctx, dist, prefix,
                      (ks, vs) if fp8 else None)

    clk = clocks.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if not fp8 else "bf16 q/out, e4m3 cache, f16 tensor-core products",
        "data": "synthetic (seeded N(0,1) q/k/v and cache, random block placement)",
        "config": {"workload": args.workload, "num_heads": H, "num_kv_heads": Hkv,
                   "head_dim": D, "block_size": BS, "batch": w.num_seqs,
                   "new_tokens": w.num_tokens, "kv_bytes_per_step": kv_bytes,
                   "max_context_len": max_ctx, "l2": "flushed before every timed step (512 MB write)",
                   "append_extras": args.extras, "kv_cache_dtype": args.kv,
                   "parallelism": f"replicas x{dist.world}"},
        "seqs_per_s": round(seqs_per_s, 1),
        "tokens_per_s": round(tokens_per_s, 1),
        "append_ms": round(statistics.mean(app_ms), 5),
        "attention_ms": round(statistics.mean(attn_ms), 5),
        # per step: RoPE + append, the decode kernel and its merge kernel
        # (and, with prefill rows, the prefill kernel)
        # (+1 for the FP8 gather of the prefill / prefix blocks)
        "gpu_launches": ((4 if prefix else 3 if decode else 4) +
                         (1 if fp8 and (prefix or not decode) else 0)) * args.steps,
        **result,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if clk is not None:
        line["clocks"] = clk
    if dist.rank == 0 and not args.no_cpu_baseline and dist.world == 1:
        line["cpu_baseline"] = cpu_baseline(w, kv_bytes)
    return line


def run_e2e(args, w, dims, g, table, ws, err, dev, decode, max_ctx, dist, prefix=0,
            fp8_scales=None):
    """Same step through the public API, inputs copied from pinned host memory
    each step and the attention output read back."""
    from paged_kv_gqa_07_gb300 import qattn as Q

    H, D = w.num_heads, w.head_dim
    # The step's host inputs packed into one pinned buffer (256-byte aligned
    # segments): one host->device copy per step, the device tensors are views.
    names = ("qkv", "positions", "slot_mapping", "block_tables", "context_lens", "cu_seqlens_q")
    src = {k: getattr(w, k).contiguous() for k in names}
    offs, total = {}, 0
    for k, t in src.items():
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    dev_in = {}
    for k, t in src.items():
        n = t.numel() * t.element_size()
        host_buf[offs[k]:offs[k] + n].copy_(t.view(-1).view(torch.uint8))
        dev_in[k] = dev_buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    out = torch.empty((w.num_tokens, H, D), dtype=torch.bfloat16, device=dev)
    host_out = torch.empty_like(out, device="cpu").pin_memory()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    Hkv = w.num_kv_heads

    def step():
        dev_buf.copy_(host_buf, non_blocking=True)
        qkv = dev_in["qkv"]
        if fp8_scales is not None:
            Q.qattn_rope_cache_append_fp8(qkv[:, :H * D], qkv[:, H * D:(H + Hkv) * D],
                                          qkv[:, (H + Hkv) * D:], dev_in["positions"],
                                          dev_in["slot_mapping"], g.k_cache, g.v_cache, table,
                                          *fp8_scales, dims, err_word=err)
            if prefix:
                Q.qattn_paged_decode_shared_prefix_fp8(
                    out, qkv[:, :H * D], g.k_cache, g.v_cache, dev_in["block_tables"],
                    dev_in["context_lens"], max_ctx, prefix, *fp8_scales, dims, ws, err)
            elif decode:
                Q.qattn_paged_decode_fp8(out, qkv[:, :H * D], g.k_cache, g.v_cache,
                                         dev_in["block_tables"], dev_in["context_lens"], max_ctx,
                                         *fp8_scales, dims, ws, err)
            else:
                n_prefill = sum(1 for n in w.q_lens if n >= 2)
                Q.qattn_varlen_prefill_fp8(out, qkv[:, :H * D], dev_in["cu_seqlens_q"],
                                           w.max_q_len, g.k_cache, g.v_cache,
                                           dev_in["block_tables"], dev_in["context_lens"],
                                           max_ctx, n_prefill, *fp8_scales, dims, ws, err)
            host_out.copy_(out, non_blocking=True)
            return
        Q.qattn_rope_cache_append(qkv[:, :H * D], qkv[:, H * D:(H + Hkv) * D],
                                  qkv[:, (H + Hkv) * D:], dev_in["positions"],
                                  dev_in["slot_mapping"], g.k_cache, g.v_cache, table, dims, err)
        if prefix:
            Q.qattn_paged_decode_shared_prefix(out, qkv[:, :H * D], g.k_cache, g.v_cache,
                                               dev_in["block_tables"], dev_in["context_lens"],
                                               max_ctx, prefix, dims, ws, err)
        elif decode:
            Q.qattn_paged_decode(out, qkv[:, :H * D], g.k_cache, g.v_cache, dev_in["block_tables"],
                                 dev_in["context_lens"], max_ctx, dims, ws, err)
        else:
            Q.qattn_varlen_prefill(out, qkv[:, :H * D], dev_in["cu_seqlens_q"], w.max_q_len,
                                   g.k_cache, g.v_cache, dev_in["block_tables"],
                                   dev_in["context_lens"], max_ctx, dims, ws, err)
        host_out.copy_(out, non_blocking=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    dist.barrier()
    for s in range(args.steps):
        flush.fill_(s & 0xff)
        evs[s][0].record(stream)
        step()
        evs[s][1].record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    total_ms = dist.max(sum(a.elapsed_time(b) for a, b in evs))
    h2d = total
    d2h = host_out.numel() * host_out.element_size()
    value = dist.sum(w.kv_bytes_read()) * args.steps / (total_ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(total_ms / args.steps, 5)}


# --------------------------------------------------------------- oracle --

def oracle_sample(w: W.Workload, n_seqs: int):
    """The first n_seqs sequences of the workload as a smaller workload."""
    q_lens = w.q_lens[:n_seqs]
    T = sum(q_lens)
    sub = dict(w.__dict__)
    sub.update(qkv=w.qkv[:T].contiguous(), positions=w.positions[:T].contiguous(),
               slot_mapping=w.slot_mapping[:T].contiguous(),
               block_tables=w.block_tables[:n_seqs].contiguous(),
               context_lens=w.context_lens[:n_seqs].contiguous(),
               cu_seqlens_q=w.cu_seqlens_q[:n_seqs + 1].contiguous(), q_lens=q_lens)
    return W.Workload(**sub)


def oracle_time(w: W.Workload, n_seqs: int, reps: int = 1):
    """Seconds per oracle step (append + attention) on a sample, and its KV bytes."""
    import numpy as np

    import oracle

    s = oracle_sample(w, n_seqs)
    H, Hkv, D, BS = s.num_heads, s.num_kv_heads, s.head_dim, s.block_size
    table = oracle.rope_table(s.theta, s.max_pos, D)

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    fp8 = s.k_cache.dtype == torch.uint8
    if fp8:
        kc0, vc0 = s.k_cache.numpy().copy(), s.v_cache.numpy().copy()
    else:
        kc0, vc0 = u16(s.k_cache), u16(s.v_cache)
    cu = None if s.is_decode else s.cu_seqlens_q
    ks, vs = W.FP8_K_SCALE, W.FP8_V_SCALE
    times = []
    for _ in range(reps):
        qkv = u16(s.qkv)
        kc, vc = kc0.copy(), vc0.copy()
        t0 = time.perf_counter()
        if fp8:
            oracle.rope_cache_append_fp8(qkv, s.positions, s.slot_mapping, kc, vc, table, H,
                                         Hkv, D, BS, ks, vs)
            q = np.ascontiguousarray(qkv[:, :H * D])
            oracle.paged_attention_fp8(q, kc, vc, ks, vs, s.block_tables, s.context_lens, H,
                                       Hkv, D, BS, cu_seqlens_q=cu)
        else:
            oracle.rope_cache_append(qkv, s.positions, s.slot_mapping, kc, vc, table, H, Hkv,
                                     D, BS)
            q = np.ascontiguousarray(qkv[:, :H * D])
            oracle.paged_attention(q, kc, vc, s.block_tables, s.context_lens, H, Hkv, D, BS,
                                   cu_seqlens_q=cu)
        times.append(time.perf_counter() - t0)
    return statistics.median(times), s.kv_bytes_read(), s


def sample_size(w: W.Workload) -> int:
    """Sequences per oracle step: the whole batch unless that is more than
    about 2e9 fp64 multiply-adds (a few seconds on the host)."""
    per_seq = [2 * w.num_heads * w.head_dim * int(L) * q for L, q in
               zip(w.context_lens.tolist(), w.q_lens)]
    n, tot = 0, 0
    for c in per_seq:
        if n > 0 and tot + c > 2e9:
            break
        n, tot = n + 1, tot + c
    return max(1, n)


def cpu_model() -> str:
    """The host CPU's model, for the record: /proc/cpuinfo's model name, or on
    Arm (which prints none) its implementer and part numbers."""
    try:
        with open("/proc/cpuinfo") as f:
            lines = f.read().splitlines()
    except OSError:
        return platform.machine()
    fields = {}
    for line in lines:
        k, _, v = line.partition(":")
        fields.setdefault(k.strip(), v.strip())
    if fields.get("model name"):
        return fields["model name"]
    if fields.get("CPU implementer") and fields.get("CPU part"):
        return (f"{platform.machine()} (CPU implementer {fields['CPU implementer']}, "
                f"part {fields['CPU part']})")
    return platform.machine()


def cpu_baseline(w: W.Workload, kv_bytes_full: int, budget_s: float = 10.0):
    """The oracle, as it stands, timed on this host: repeated over a sample
    of the workload for about budget_s seconds."""
    import oracle
    n = sample_size(w)
    total, reps, kvb = 0.0, 0, 0
    while total < budget_s or reps == 0:
        sec, kvb, _ = oracle_time(w, n)
        total += sec
        reps += 1
    return {"value": round(kvb * reps / total / 1e9, 4), "unit": "GB/s",
            "cores": oracle.default_threads(), "cpu_model": cpu_model(), "kind": "oracle",
            "sample": f"first {n} of {w.num_seqs} sequences ({kvb} of {kv_bytes_full} KV bytes) "
                      f"x {reps} repetitions, append + attention in fp64, {total:.1f} s"}


def run_append_sweep(args):
    """K1 alone at sizes where bandwidth is meaningful (the decode step's
    64-token append is launch-bound): T new tokens in sequences of 16384,
    28/4 heads, L2 flushed before every timed launch."""
    from paged_kv_gqa_07_gb300 import build as B
    from paged_kv_gqa_07_gb300 import qattn as Q
    B.build()
    Q.load_library()
    dev = torch.device("cuda", 0)
    hbm_peak, _, peak_kind = measured_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for T in (16384, 65536):
        n = T // 16384  # sequences of 16384 new tokens (positions stay below max_pos)
        w = W.custom(28, 4, ctx=[16384] * n, q_lens=[16384] * n, seed=T)
        g = W.to_device(w, dev)
        dims = Q.make_dims(28, 4)
        table = Q.qattn_rope_table_build(w.max_pos, 128, w.theta).to(dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        qkv0 = g.qkv.clone()

        def append():
            Q.qattn_rope_cache_append(g.q_view(), g.k_view(), g.v_view(), g.positions,
                                      g.slot_mapping, g.k_cache, g.v_cache, table, dims, err)
        for _ in range(args.warmup):
            append()
        ms = []
        for i in range(args.steps):
            g.qkv.copy_(qkv0)
            flush.fill_(i & 0xff)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            append()
            e1.record()
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
        assert int(err.item()) == 0
        t = statistics.median(ms) * 1e-3
        alg = T * 18944  # read q/k/v + a table row, write q and the cache rows
        print(json.dumps({"metric": "rope + cache append GB/s (supplementary)", "tokens": T,
                          "value": round(alg / t / 1e9, 1), "unit": "GB/s",
                          "us": round(t * 1e6, 2), "algorithmic_bytes": alg,
                          "frac": round(alg / t / 1e9 / hbm_peak, 4), "peak_kind": peak_kind,
                          "l2": "flushed before every timed launch"}), flush=True)


def run_reference(args, dist: Dist):
    import oracle
    w = W.build(args.workload, block_size=args.block_size)
    if args.kv == "fp8":
        w = W.with_fp8_cache(w)
    n = sample_size(w)
    for _ in range(args.warmup):
        oracle_time(w, n)
    t0 = time.perf_counter()
    per = []
    for _ in range(args.steps):
        sec, kvb, s = oracle_time(w, n)
        per.append(sec)
    total = time.perf_counter() - t0
    value = kvb * args.steps / sum(per) / 1e9
    sample = (f"first {n} of {w.num_seqs} sequences per step ({kvb} KV bytes), "
              "append + attention in fp64")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(per) / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "batch_sampled": n, "block_size": w.block_size,
                   "kv_cache_dtype": args.kv},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                         "cores": oracle.default_threads(), "cpu_model": cpu_model(),
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(total, 2),
    }


def main():
    args = parse()
    if args.append_sweep:
        run_append_sweep(args)
        return
    if args.impl == "reference":
        # The reference arm is the CPU oracle: rank 0 alone runs it.
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps(run_reference(args, Dist.single())), flush=True)
        return
    dist = Dist()
    try:
        line = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
