"""Benchmark of one attention step over a paged KV cache on GB300.

A step is the whole path for one batch: RoPE + cache append of the new tokens
(qattn_rope_cache_append), then paged GQA attention (qattn_paged_decode for a
decode workload, qattn_varlen_prefill for a mixed one).  Inputs are resident
in HBM when timing starts.  The workload's cache and QKV rows are repeated as
a stack of layers at different addresses and consecutive steps use
consecutive layers, as a model's forward pass does, so every step's KV comes
from HBM (the layers between two uses of one span more than L2) without a
flush kernel.  Each step is timed with CUDA events on the launching stream.
The headline workload is the Qwen2-7B-shaped decode step (28 query / 4 KV
heads, head_dim 128, batch 64, contexts U[128, 4096], block size 16, random
block placement); a single-GPU run also times the other configurations
(tiny decode, mixed prefill + decode, long-context decode, shared-prefix
decode, FP8 cache) with the same harness under "workloads".

The "e2e" figure is the same step through the public API with the step's
inputs copied from pinned host memory and its output read back every step,
the copies on an upload and a download stream, double-buffered so that they
overlap the neighbouring steps' compute, timed over the whole loop.

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
    p.add_argument("--no-workloads", action="store_true",
                   help="time only --workload (by default a single-GPU run of the headline "
                        "workload also times the other four configurations and the FP8 cache)")
    p.add_argument("--phases", action="store_true",
                   help="diagnostic: the tracing build's per-CTA phase stamps of the decode "
                        "call (b64 and 8 x 32K), one JSON line per workload")
    p.add_argument("--copy-ceiling", action="store_true",
                   help="diagnostic: the tracing build's copy probe -- the decode's K/V tile "
                        "copies alone -- beside the decode call, b64 and 8 x 32K, bf16 and "
                        "FP8, one JSON line each")
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

# Launches per call of each entry point, as the library issues them: the
# append is one kernel; a decode call is the decode kernel and its merge
# kernel; a shared-prefix call adds the prefix pass; a varlen call with
# decode rows is the prefill kernel plus the decode pair; an FP8 varlen or
# shared-prefix call adds the gather of the blocks the prefill kernel reads.
LAUNCHES = {"append": 1, "decode": 2, "prefix": 3, "varlen": 3, "varlen_fp8": 4,
            "prefix_fp8": 4}

# Bytes of cache the rotated layers must span so that a call never finds its
# KV in L2 (129 MB) from the previous calls.
LAYER_SPAN_BYTES = 512 << 20


class Harness:
    """One workload resident on the device, with `layers` independent copies
    of its KV cache and QKV rows at different addresses -- the same layer
    shape repeated, as in a model's stack.  Timed calls cycle through the
    layers, so every call reads KV that the previous calls left out of L2
    (each layer's cache, or the span of layers between two uses of one, is
    larger than L2), with no flush kernel between calls."""

    def __init__(self, args, name, dev, kv="bf16", rank=0, sub_seqs=None, extras="none"):
        from paged_kv_gqa_07_gb300 import qattn as Q
        self.Q = Q
        idx = W.WORKLOAD_NAMES.index(name)
        w = W.build(name, seed=W.SEED_BASE + idx + 1000 * rank, block_size=args.block_size)
        if sub_seqs is not None:
            w = first_sequences(w, sub_seqs)
        self.fp8 = kv == "fp8"
        if self.fp8:
            w = W.with_fp8_cache(w)
        self.w, self.dev, self.extras = w, dev, extras
        self.ks, self.vs = W.FP8_K_SCALE, W.FP8_V_SCALE
        H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
        self.dims = Q.make_dims(H, Hkv, D, BS)
        g = W.to_device(w, dev)
        self.g = g
        self.table = Q.qattn_rope_table_build(w.max_pos, D, w.theta).to(dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.decode = w.is_decode
        self.max_ctx = w.max_context_len
        self.prefix = w.shared_prefix_tokens if self.decode else 0
        self.n_prefill = sum(1 for n in w.q_lens if n >= 2)
        B = w.num_seqs
        if self.prefix and self.fp8:
            ws = Q.qattn_paged_decode_shared_prefix_fp8_workspace_size(B, self.max_ctx,
                                                                      self.prefix, self.dims)
        elif not self.decode and self.fp8:
            ws = Q.qattn_varlen_prefill_fp8_workspace_size(B, self.n_prefill, self.max_ctx,
                                                           self.dims)
        elif self.prefix:
            ws = Q.qattn_paged_decode_shared_prefix_workspace_size(B, self.max_ctx, self.dims)
        elif self.decode:
            ws = Q.qattn_paged_decode_workspace_size(B, self.max_ctx, self.dims)
        else:
            ws = Q.qattn_varlen_prefill_workspace_size(B, self.max_ctx, self.dims)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.out = torch.empty((w.num_tokens, H, D), dtype=torch.bfloat16, device=dev)
        cache_bytes = 2 * g.k_cache.numel() * g.k_cache.element_size()
        self.nlayers = max(2, min(256, -(-LAYER_SPAN_BYTES // max(cache_bytes, 1))))
        self.layers = [(g.qkv, g.k_cache, g.v_cache)]
        for _ in range(self.nlayers - 1):
            self.layers.append((g.qkv.clone(), g.k_cache.clone(), g.v_cache.clone()))
        gx = torch.Generator().manual_seed(W.SEED_BASE + 77)
        self.bias = self.qn = self.kn = None
        if extras in ("bias", "both"):
            self.bias = (0.5 * torch.randn((H + 2 * Hkv) * D, generator=gx)).to(torch.bfloat16).to(dev)
        if extras in ("qknorm", "both"):
            self.qn = (1.0 + 0.2 * torch.randn(D, generator=gx)).to(torch.bfloat16).to(dev)
            self.kn = (1.0 + 0.2 * torch.randn(D, generator=gx)).to(torch.bfloat16).to(dev)

    @property
    def kind(self) -> str:
        if self.prefix:
            return "prefix_fp8" if self.fp8 else "prefix"
        if self.decode:
            return "decode"
        return "varlen_fp8" if self.fp8 and self.n_prefill else "varlen"

    def views(self, qkv):
        w = self.w
        H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
        return qkv[:, :H * D], qkv[:, H * D:(H + Hkv) * D], qkv[:, (H + Hkv) * D:]

    def append(self, l, qkv=None, positions=None, slots=None):
        Q, g = self.Q, self.g
        lq, kc, vc = self.layers[l % self.nlayers]
        q, k, v = self.views(lq if qkv is None else qkv)
        pos = g.positions if positions is None else positions
        sl = g.slot_mapping if slots is None else slots
        if self.fp8:
            Q.qattn_rope_cache_append_fp8(q, k, v, pos, sl, kc, vc, self.table, self.ks, self.vs,
                                          self.dims, qkv_bias=self.bias, q_norm_weight=self.qn,
                                          k_norm_weight=self.kn, err_word=self.err)
        elif self.extras == "none":
            Q.qattn_rope_cache_append(q, k, v, pos, sl, kc, vc, self.table, self.dims, self.err)
        else:
            Q.qattn_rope_cache_append_ex(q, k, v, pos, sl, kc, vc, self.table, self.dims,
                                         qkv_bias=self.bias, q_norm_weight=self.qn,
                                         k_norm_weight=self.kn, err_word=self.err)

    def attend(self, l, qkv=None, block_tables=None, context_lens=None, cu=None, out=None):
        Q, g, w = self.Q, self.g, self.w
        lq, kc, vc = self.layers[l % self.nlayers]
        q = self.views(lq if qkv is None else qkv)[0]
        bt = g.block_tables if block_tables is None else block_tables
        cl = g.context_lens if context_lens is None else context_lens
        cu = g.cu_seqlens_q if cu is None else cu
        out = self.out if out is None else out
        mc, ws, err, d = self.max_ctx, self.ws, self.err, self.dims
        if self.prefix and self.fp8:
            Q.qattn_paged_decode_shared_prefix_fp8(out, q, kc, vc, bt, cl, mc, self.prefix,
                                                   self.ks, self.vs, d, ws, err)
        elif not self.decode and self.fp8:
            Q.qattn_varlen_prefill_fp8(out, q, cu, w.max_q_len, kc, vc, bt, cl, mc,
                                       self.n_prefill, self.ks, self.vs, d, ws, err)
        elif self.prefix:
            Q.qattn_paged_decode_shared_prefix(out, q, kc, vc, bt, cl, mc, self.prefix, d, ws,
                                               err)
        elif self.fp8:
            Q.qattn_paged_decode_fp8(out, q, kc, vc, bt, cl, mc, self.ks, self.vs, d, ws, err)
        elif self.decode:
            Q.qattn_paged_decode(out, q, kc, vc, bt, cl, mc, d, ws, err)
        else:
            Q.qattn_varlen_prefill(out, q, cu, w.max_q_len, kc, vc, bt, cl, mc, d, ws, err)

    def step(self, l):
        self.append(l)
        self.attend(l)

    def timed(self, fn, steps, warmup, stream):
        """Per-call device times (ms) of `steps` calls fn(layer), layers in
        rotation, after `warmup` untimed calls.  A GPU sleep queued first
        lets the host enqueue ahead, so the events time the device."""
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize(self.dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(20_000_000)
        for s in range(steps):
            evs[s][0].record(stream)
            fn(warmup + s)
            evs[s][1].record(stream)
        torch.cuda.synchronize(self.dev)
        assert int(self.err.item()) == 0, f"device error bits {int(self.err.item())}"
        return [a.elapsed_time(b) for a, b in evs]

    def qo_bytes(self) -> int:
        w = self.w
        return 2 * w.num_tokens * w.num_heads * w.head_dim * 2

    def free(self):
        self.layers = None
        self.g = None


def decode_summary(h: Harness, attn_ms, step_ms, hbm_peak, peak_kind):
    """KV bandwidth of a decode call and its fraction of the HBM peak."""
    w = h.w
    a = statistics.median(attn_ms) * 1e-3
    s = statistics.median(step_ms) * 1e-3
    kv = w.kv_bytes_read()
    alg = kv + h.qo_bytes()
    d = {"attention_us": round(a * 1e6, 2), "step_us": round(s * 1e6, 2),
         "kv_bytes": kv, "algorithmic_bytes": alg,
         "kv_GBps": round(alg / a / 1e9, 1), "frac": round(alg / a / 1e9 / hbm_peak, 4),
         "peak_kind": peak_kind, "seqs_per_s": round(w.num_seqs / s, 1)}
    if h.prefix:
        uniq = w.unique_kv_bytes() + h.qo_bytes()
        d.update(logical_kv_GBps=d.pop("kv_GBps"), distinct_bytes=uniq,
                 distinct_GBps=round(uniq / a / 1e9, 1),
                 frac=round(uniq / a / 1e9 / hbm_peak, 4),
                 frac_basis="distinct blocks (each read from DRAM once)")
    return d


def run_ours(args, dist: Dist):
    from paged_kv_gqa_07_gb300 import build as B
    from paged_kv_gqa_07_gb300 import qattn as Q

    B.build()
    Q.load_library()
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    # The calls run on a stream of their own, as in a serving engine, not on
    # the legacy default stream.
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    hbm_peak, tf_peak, peak_kind = measured_peaks()
    h = Harness(args, args.workload, dev, kv=args.kv, rank=dist.rank, extras=args.extras)
    w = h.w
    H, Hkv, D, BS = w.num_heads, w.num_kv_heads, w.head_dim, w.block_size

    # (A) the step (append + attention), layers in rotation: events only at
    # step boundaries, so the attention kernels may overlap the append
    # kernel's tail (programmatic dependent launch).
    with ClockSampler(dev.index, enabled=not args.no_clocks) as clocks:
        dist.barrier()
        torch.cuda.synchronize(dev)
        step_ms = h.timed(h.step, args.steps, args.warmup, stream)
        torch.cuda.synchronize(dev)
        dist.barrier()
    # (B) the attention call alone: the roofline's kernel duration.  (C) the append.
    attn_ms = h.timed(h.attend, args.steps, args.warmup, stream)
    app_ms = h.timed(h.append, args.steps, args.warmup, stream)
    local_total_ms = sum(step_ms)
    total_ms = dist.max(local_total_ms)
    ms_per_step = total_ms / args.steps

    kv_bytes = w.kv_bytes_read()
    qo_bytes = h.qo_bytes()
    value = dist.sum(kv_bytes) * args.steps / (total_ms * 1e-3) / 1e9
    seqs_per_s = dist.sum(w.num_seqs) * args.steps / (total_ms * 1e-3)
    tokens_per_s = dist.sum(w.num_tokens) * args.steps / (total_ms * 1e-3)

    attn_avg_s = statistics.mean(attn_ms) * 1e-3
    result = {}
    if h.prefix:
        alg = w.unique_kv_bytes() + qo_bytes
        achieved = alg / attn_avg_s / 1e9
        result["roofline"] = {"bound": "hbm",
                              "kernel": "varlen_prefill_kernel (prefix pass) + paged_decode",
                              "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                              "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                              "traffic": None, "algorithmic_bytes_per_launch": alg,
                              "logical_kv_bytes_per_launch": kv_bytes}
    elif h.decode:
        alg = kv_bytes + qo_bytes
        achieved = alg / attn_avg_s / 1e9
        kname = "paged_decode_tc_kernel"
        sha = kernel_source_sha(["paged_decode_tc.cu", "decode_merge.cu", "common.cuh",
                                 "internal.h"])
        traffic = profiled_traffic(kname + ("_fp8" if h.fp8 else ""), args.workload, sha)
        result["roofline"] = {"bound": "hbm", "kernel": kname + " + decode_merge_kernel",
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
        e2e = run_e2e(args, h, dist, stream)
    nlayers, kind, fp8 = h.nlayers, h.kind, h.fp8
    h.free()
    del h
    torch.cuda.empty_cache()

    # ---- the other workloads, same harness (rank 0 of a single-GPU run) ----
    others = None
    if not args.no_workloads and dist.world == 1 and args.workload == DEFAULT_WORKLOAD \
            and args.kv == "bf16" and args.extras == "none" and args.block_size == 16:
        others = run_other_workloads(args, dev, stream, hbm_peak, tf_peak, peak_kind)

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
        "dtype": "bf16" if not fp8 else "bf16 q/out, e4m3 cache; decode q.k on e4m3 codes, P V in f16",
        "data": "synthetic (seeded N(0,1) q/k/v and cache, random block placement)",
        "config": {"workload": args.workload, "num_heads": H, "num_kv_heads": Hkv,
                   "head_dim": D, "block_size": BS, "batch": w.num_seqs,
                   "new_tokens": w.num_tokens, "kv_bytes_per_step": kv_bytes,
                   "max_context_len": w.max_context_len,
                   "l2": (f"inputs larger than L2: {nlayers} layers of the workload's cache "
                          "and QKV rows in rotation, consecutive steps read different layers"),
                   "append_extras": args.extras, "kv_cache_dtype": args.kv,
                   "parallelism": f"replicas x{dist.world}"},
        "seqs_per_s": round(seqs_per_s, 1),
        "tokens_per_s": round(tokens_per_s, 1),
        "append_ms": round(statistics.mean(app_ms), 5),
        "attention_ms": round(statistics.mean(attn_ms), 5),
        "gpu_launches": (LAUNCHES["append"] + LAUNCHES[kind]) * args.steps,
        **result,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if others is not None:
        line["workloads"] = others
    if clk is not None:
        line["clocks"] = clk
    if dist.rank == 0 and not args.no_cpu_baseline and dist.world == 1:
        line["cpu_baseline"] = cpu_baseline(w, kv_bytes)
    return line


def run_other_workloads(args, dev, stream, hbm_peak, tf_peak, peak_kind):
    """Every other configuration of the benchmark through the same harness:
    the tiny Qwen3 decode (launch-bound), the mixed prefill + decode batch
    (and its prefill part alone), the long-context decode, the shared-prefix
    decode, and the FP8-cache b64 decode."""
    res = {}

    def measure(name, **kw):
        h = Harness(args, name, dev, **kw)
        attn = h.timed(h.attend, args.steps, args.warmup, stream)
        if kw.get("sub_seqs") is None:
            step = h.timed(h.step, args.steps, args.warmup, stream)
        else:
            step = attn
        return h, attn, step

    h, attn, step = measure("tiny_qwen3_decode")
    d = decode_summary(h, attn, step, hbm_peak, peak_kind)
    d["bound"] = "launch (4 sequences, 1.8 MB of KV): the fraction is not a roofline claim"
    res["tiny_qwen3_decode"] = d
    h.free()

    h, attn, step = measure("qwen2_7b_long_decode")
    res["qwen2_7b_long_decode"] = decode_summary(h, attn, step, hbm_peak, peak_kind)
    h.free()

    h, attn, step = measure("qwen3_prefix_decode")
    res["qwen3_prefix_decode"] = decode_summary(h, attn, step, hbm_peak, peak_kind)
    h.free()

    h, attn, step = measure("qwen2_7b_decode_b64", kv="fp8")
    d = decode_summary(h, attn, step, hbm_peak, peak_kind)
    d["kv_cache_dtype"] = "fp8 (e4m3 codes, 1 byte per value)"
    res["qwen2_7b_decode_b64_fp8"] = d
    h.free()

    # the mixed batch: one varlen call (4 prefill chunks + 60 decode rows)
    h, attn, step = measure("qwen2_7b_mixed_varlen")
    w = h.w
    a, s = statistics.median(attn) * 1e-3, statistics.median(step) * 1e-3
    flops = 4 * w.head_dim * w.causal_pairs()
    mixed = {"attention_us": round(a * 1e6, 2), "step_us": round(s * 1e6, 2),
             "new_tokens": w.num_tokens, "tokens_per_s": round(w.num_tokens / s, 1),
             "causal_flops": flops, "call_TFLOPs": round(flops / a / 1e12, 2)}
    h.free()
    # its prefill part alone (the 4 chunks, no decode rows): the prefill kernel
    h, attn, _ = measure("qwen2_7b_mixed_varlen", sub_seqs=4)
    w = h.w
    k3 = statistics.median(attn) * 1e-3
    pf = 4 * w.head_dim * w.causal_pairs()
    mixed.update(prefill_only_us=round(k3 * 1e6, 2), prefill_tokens=w.num_tokens,
                 prefill_tokens_per_s=round(w.num_tokens / k3, 1),
                 prefill_TFLOPs=round(pf / k3 / 1e12, 2),
                 prefill_frac=round(pf / k3 / 1e12 / tf_peak, 4), peak_kind=peak_kind,
                 prefill_bound="tensor (bf16 dense peak)")
    res["qwen2_7b_mixed_varlen"] = mixed
    h.free()
    torch.cuda.empty_cache()
    return res


def run_e2e(args, h: Harness, dist, stream):
    """The same step through the public API, its inputs copied from pinned
    host memory every step and the attention output read back every step.
    As a serving loop would, the copies run on an upload and a download
    stream, double-buffered: step i+1's inputs go up and step i-1's output
    comes down while step i computes.  The timed region spans the whole loop, from before the
    first step's host->device copy to the end of the last step's
    device->host read."""
    w, dev = h.w, h.dev
    # The step's host inputs packed into one pinned buffer (256-byte aligned
    # segments): one host->device copy per step, the device tensors are views.
    names = ("qkv", "positions", "slot_mapping", "block_tables", "context_lens", "cu_seqlens_q")
    src = {k: getattr(w, k).contiguous() for k in names}
    offs, total = {}, 0
    for k, t in src.items():
        offs[k] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for k, t in src.items():
        n = t.numel() * t.element_size()
        host_buf[offs[k]:offs[k] + n].copy_(t.view(-1).view(torch.uint8))
    dev_bufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_in = []
    for buf in dev_bufs:
        views = {}
        for k, t in src.items():
            n = t.numel() * t.element_size()
            views[k] = buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        dev_in.append(views)
    outs = [torch.empty_like(h.out) for _ in range(2)]
    host_outs = [torch.empty_like(h.out, device="cpu").pin_memory() for _ in range(2)]
    # one stream for the uploads and one for the downloads: on a single copy
    # stream, step i+1's upload would queue behind step i's download, which
    # waits for step i's compute
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d = [ev(), ev()]
    comp = [ev(), ev()]
    d2h = [ev(), ev()]
    used = [False, False]

    def run(n_steps, first_layer):
        for i in range(n_steps):
            b = i & 1
            with torch.cuda.stream(up):
                if used[b]:
                    up.wait_event(comp[b])          # step i-2 is done with buffer b
                dev_bufs[b].copy_(host_buf, non_blocking=True)
                h2d[b].record(up)
            stream.wait_event(h2d[b])
            if used[b]:
                stream.wait_event(d2h[b])           # step i-2's output has been read
            d = dev_in[b]
            l = first_layer + i
            h.append(l, qkv=d["qkv"], positions=d["positions"], slots=d["slot_mapping"])
            h.attend(l, qkv=d["qkv"], block_tables=d["block_tables"],
                     context_lens=d["context_lens"], cu=d["cu_seqlens_q"], out=outs[b])
            comp[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(comp[b])
                host_outs[b].copy_(outs[b], non_blocking=True)
                d2h[b].record(down)
            used[b] = True
        for b in range(2):
            if used[b]:
                stream.wait_event(d2h[b])

    run(args.warmup, 0)
    torch.cuda.synchronize(dev)
    dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(20_000_000)
    t0.record(stream)
    up.wait_event(t0)  # the first copy is inside the timed region
    run(args.steps, args.warmup)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    assert int(h.err.item()) == 0, f"device error bits {int(h.err.item())}"
    total_ms = dist.max(t0.elapsed_time(t1))
    d2h_bytes = host_outs[0].numel() * host_outs[0].element_size()
    value = dist.sum(w.kv_bytes_read()) * args.steps / (total_ms * 1e-3) / 1e9

    # The same loop with every copy in line on the compute stream (upload,
    # step, download, one after the other): what the copies cost unhidden.
    def serial(i):
        dev_bufs[0].copy_(host_buf, non_blocking=True)
        d = dev_in[0]
        h.append(i, qkv=d["qkv"], positions=d["positions"], slots=d["slot_mapping"])
        h.attend(i, qkv=d["qkv"], block_tables=d["block_tables"],
                 context_lens=d["context_lens"], cu=d["cu_seqlens_q"], out=outs[0])
        host_outs[0].copy_(outs[0], non_blocking=True)

    serial_ms = dist.max(sum(h.timed(serial, args.steps, args.warmup, stream)))
    serial_value = dist.sum(w.kv_bytes_read()) * args.steps / (serial_ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": total,
            "d2h_bytes_per_step": d2h_bytes, "ms_per_step": round(total_ms / args.steps, 5),
            "serial": {"value": round(serial_value, 2),
                       "ms_per_step": round(serial_ms / args.steps, 5)},
            "copies": "pinned host <-> device every step on an upload and a download stream, "
                      "double-buffered, overlapped with the neighbouring steps' compute"}


# --------------------------------------------------------------- oracle --

def first_sequences(w: W.Workload, n_seqs: int):
    """The first n_seqs sequences of the workload as a smaller workload
    (input slicing only)."""
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

    s = first_sequences(w, n_seqs)
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


def run_phases(args):
    """Where the decode call's time goes, from the tracing build
    (include/qattn_trace.h): per-CTA %globaltimer stamps of the decode kernel
    and the merge kernel, layers in rotation as in the timed runs.  Times are
    us from the first decode CTA's entry; medians over the calls."""
    import ctypes

    import numpy as np

    from paged_kv_gqa_07_gb300 import build as B
    from paged_kv_gqa_07_gb300 import qattn as Q
    B.build()
    L = Q.load_library(B.build(trace=True))
    Q._lib = L
    L.qattn_trace_dims.argtypes = [ctypes.c_void_p] * 3
    L.qattn_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    dims = (ctypes.c_int32 * 3)()
    L.qattn_trace_dims(ctypes.byref(dims, 0), ctypes.byref(dims, 4), ctypes.byref(dims, 8))
    n_dec, n_slot, n_merge = int(dims[0]), int(dims[1]), int(dims[2])
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)  # as in the timed runs
    torch.cuda.set_stream(stream)
    for name in ("qwen2_7b_decode_b64", "qwen2_7b_long_decode", "qwen3_prefix_decode"):
        h = Harness(args, name, dev, kv=args.kv)
        event_ms = h.timed(h.attend, args.steps, args.warmup, stream)
        rows = []
        for r in range(max(5, args.steps)):
            assert L.qattn_trace_clear() == 0
            h.attend(r)
            torch.cuda.synchronize(dev)
            dec = np.zeros(n_dec * n_slot, dtype=np.uint64)
            mer = np.zeros(n_merge * 4, dtype=np.uint64)
            assert L.qattn_trace_read(dec.ctypes.data, mer.ctypes.data) == 0
            d = dec.reshape(n_dec, n_slot).astype(np.int64)
            d = d[d[:, 0] > 0]
            m = mer.reshape(n_merge, 4).astype(np.int64)
            m = m[m[:, 1] > 0]
            t0 = d[:, 0].min()
            us = lambda x: (x - t0) / 1e3
            rows.append({
                "plan_done": float(np.median(us(d[:, 1]))),
                "first_scores": float(np.median(us(d[:, 2]))),
                "copies_issued": float(np.median(us(d[:, 3]))),
                "softmax_done_median": float(np.median(us(d[:, 4]))),
                "softmax_done_max": float(us(d[:, 4]).max()),
                "cta_done_max": float(us(d[:, 5]).max()),
                "merge_released": float(us(m[:, 1]).min()),
                "merge_done": float(us(m[:, 2]).max()),
            })
        med = {k: round(statistics.median(r[k] for r in rows), 2) for k in rows[0]}
        phases = {
            "startup_us": med["first_scores"],
            "stream_us": round(med["softmax_done_median"] - med["first_scores"], 2),
            "tail_us": round(med["cta_done_max"] - med["softmax_done_median"], 2),
            "grid_end_to_merge_us": round(med["merge_released"] - med["cta_done_max"], 2),
            "merge_us": round(med["merge_done"] - med["merge_released"], 2),
            "kernels_us": med["merge_done"],
        }
        print(json.dumps({"phases": name, "kv_cache_dtype": args.kv, "ctas": int(d.shape[0]), "calls": len(rows),
                          "event_us_median": round(statistics.median(event_ms) * 1e3, 2),
                          "stamps_us_median": med, **phases,
                          "note": "tracing build; us from the first decode CTA's entry; "
                                  "event_us also holds the launch latency before it"}),
              flush=True)
        h.free()
        torch.cuda.empty_cache()


def decode_tile_list(w, prefix=0):
    """The decode kernel's work list: per (sequence, kv head) unit its
    128-token tiles, each as [kv head, block id of each cache block of the
    tile, -1 where there is none]; and the cache blocks it names.  With a
    shared prefix of `prefix` tokens (a multiple of the block size), the
    tokens after it, as the suffix decode of the shared-prefix call reads
    them."""
    bs = w.block_size
    bpt = 128 // bs
    pb = prefix // bs
    bt = w.block_tables.tolist()
    tiles, nblocks = [], 0
    for b, L in enumerate(w.context_lens.tolist()):
        L -= prefix
        nblk = (L + bs - 1) // bs
        for g in range(w.num_kv_heads):
            for i in range((L + 127) // 128):
                ids = [-1] * 8
                for j in range(bpt):
                    if i * bpt + j < nblk:
                        ids[j] = bt[b][pb + i * bpt + j]
                        nblocks += 1
                tiles.append([g] + ids)
    return tiles, nblocks


def run_copy_ceiling(args):
    """The copy pattern's own time: the tracing build's copy probe issues,
    per SM, the decode's K and V tile boxes (same tensor maps, same tiles,
    the decode's ring depth) with nothing consuming them, layers in
    rotation as in the timed runs; the decode call of the same harness is
    timed beside it with the regular library."""
    import ctypes

    from paged_kv_gqa_07_gb300 import build as B
    from paged_kv_gqa_07_gb300 import qattn as Q
    B.build()
    Q.load_library()
    T = ctypes.CDLL(B.build(trace=True))
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    T.qattn_trace_copy_stream.argtypes = [P, P, I32, Q.qattn_dims, I32, P, I32, I32, P, P]
    T.qattn_trace_copy_stream.restype = ctypes.c_int
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)  # as in the timed runs
    torch.cuda.set_stream(stream)
    hbm_peak, _, peak_kind = measured_peaks()
    for name in ("qwen2_7b_decode_b64", "qwen2_7b_long_decode", "qwen3_prefix_decode"):
        for kv in ("bf16", "fp8"):
            if name == "qwen3_prefix_decode" and kv == "fp8":
                continue
            h = Harness(args, name, dev, kv=kv)
            w = h.w
            # the shared-prefix call: the copies of its suffix decode (the
            # prefix pass beside it reads the prefix once)
            tiles, nblocks = decode_tile_list(w, w.shared_prefix_tokens)
            d_tiles = torch.tensor(tiles, dtype=torch.int32, device=dev)
            stages = 4 if kv == "fp8" else 3  # the decode kernel's K / V ring depth
            copy_bytes = 2 * nblocks * w.block_size * 128 * (1 if kv == "fp8" else 2)

            def copy(l):
                _, kc, vc = h.layers[l % h.nlayers]
                rc = T.qattn_trace_copy_stream(kc.data_ptr(), vc.data_ptr(), int(kc.shape[0]),
                                               h.dims, 1 if kv == "fp8" else 0,
                                               d_tiles.data_ptr(), len(tiles), stages,
                                               h.err.data_ptr(), stream.cuda_stream)
                assert rc == 0, rc

            copy_ms = h.timed(copy, args.steps, args.warmup, stream)
            attn_ms = h.timed(h.attend, args.steps, args.warmup, stream)
            c = statistics.median(copy_ms) * 1e-3
            a = statistics.median(attn_ms) * 1e-3
            print(json.dumps({"copy_ceiling": name, "kv_cache_dtype": kv,
                              "block_size": w.block_size, "stages": stages,
                              "copy_bytes": copy_bytes, "copy_us": round(c * 1e6, 2),
                              "copy_GBps": round(copy_bytes / c / 1e9, 1),
                              "copy_frac": round(copy_bytes / c / 1e9 / hbm_peak, 4),
                              "peak_kind": peak_kind, "decode_us": round(a * 1e6, 2),
                              "copy_over_decode": round(c / a, 3),
                              **({"note": "copies of the suffix decode only; decode_us is the "
                                          "whole shared-prefix call"}
                                 if w.shared_prefix_tokens else {})}), flush=True)
            h.free()
            del d_tiles
            torch.cuda.empty_cache()


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
    if args.phases:
        run_phases(args)
        return
    if args.copy_ceiling:
        run_copy_ceiling(args)
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
