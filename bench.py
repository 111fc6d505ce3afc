#!/usr/bin/env python3
"""Benchmark of one layer step of the paged-KV hot path on GB300.

A step is one pass of the whole path over one synthetic ragged batch:
paged_kv_write of the step's new K/V rows, then ragged paged attention
(decode kernel, prefill kernel, split combine: whatever the planner
launches).  Inputs are resident in HBM when the timed region starts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 1..5] [--no-breakdown]

Prints ONE JSON line on rank 0.  The headline workload is the largest one
that fits one GPU and the only full-size step with both kernel classes: the
mixed step of a 2048-token prefill chunk at position 16384, two fresh
1024-token prompts and 64 decodes.  The other four workloads are measured
too and reported under "workloads", each with its own kernel roofline, CPU
oracle baseline and end-to-end number.  `--impl reference` times the CPU
oracle (the only reference there is) on the host cores.  `--gpus N` without
torchrun's environment re-launches itself under torch.distributed.run with
N ranks (one independent replica per GPU).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import Batch, CONFIG_NAMES, config_spec, fill_normal_bf16, make_batch, subset_spec  # noqa: E402

METRIC = "ragged paged-attn step µs + KV-read HBM GB/s vs 8 TB/s; query tokens/s"
UNIT = "query tokens/s"
HEADLINE = 4
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0
SM_COUNT = 152
SM_MAX_MHZ = 2070.0
FP32_LANES_PER_SM = 128


# ---------------------------------------------------------------------------- environment

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest of every rank's x (the job's time is its slowest rank's).
    dist: torch.distributed (or None for one process); NCCL reduces a CUDA
    tensor on `device`, gloo a CPU one."""
    if dist is None:
        return float(x)
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own copy of the step's
    tokens (weak scaling, replicas), timed by the slowest rank."""
    return tokens_per_step * world / (ms_per_step / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "sm_max_mhz": float(pk.get("sm_max_mhz", SM_MAX_MHZ)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": SM_MAX_MHZ, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        if not self.samples:
            return None
        inside = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed region"
        if not inside:
            inside = [s for _, s in self.samples]
            window = "whole GPU phase (timed region shorter than the sampling interval)"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max((num(s[3]) or 0.0) for s in inside)}


# ---------------------------------------------------------------------------- accounting

def accounting(spec, meta, classes):
    """Algorithmic bytes and FLOPs of one step, whole and per kernel class.

    KV bytes count every pool slot a request must read (positions < L) once,
    however many requests share its block; FLOPs are 4*d*Hq per unmasked
    (query, key) pair.  The kernel class of each request is the library's
    own planner decision (pkv.plan_request_kernels)."""
    hq, hkv, d, bs = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    slot_bytes = hkv * d * 2 * 2                       # K and V of one slot
    n = meta.num_tokens
    per_class = {}
    rows_used = {}                                     # class -> {block: rows}
    for r, cls in enumerate(classes):
        t = meta.query_start_loc[r + 1] - meta.query_start_loc[r]
        L = meta.seq_lens[r]
        c = per_class.setdefault(cls, {"kv_bytes": 0, "q_out_bytes": 0, "flops": 0.0, "tokens": 0, "write_bytes": 0})
        c["q_out_bytes"] += 2 * t * hq * d * 2
        c["tokens"] += t
        c["write_bytes"] += t * hkv * d * 2 * 2 * 2 + t * 8  # its new K/V rows read + written, slots
        if L == 0 or t == 0:
            continue
        c["flops"] += 4.0 * d * hq * (t * (L - t) + t * (t + 1) / 2)
        table = spec.reqs[r].table
        used = rows_used.setdefault(cls, {})
        for blk_i in range(-(-L // bs)):
            rows = min(bs, L - blk_i * bs)
            blk = table[blk_i]
            if used.get(blk, 0) < rows:
                used[blk] = rows
    all_used = {}
    for cls, used in rows_used.items():
        per_class[cls]["kv_bytes"] = sum(used.values()) * slot_bytes
        for blk, rows in used.items():
            if all_used.get(blk, 0) < rows:
                all_used[blk] = rows
    unique_kv = sum(all_used.values()) * slot_bytes
    logical_kv = sum(meta.seq_lens) * slot_bytes
    write_bytes = n * hkv * d * 2 * 2 * 2 + n * 8     # new K/V read + written, slots
    q_out = 2 * n * hq * d * 2
    flops = sum(c["flops"] for c in per_class.values())
    return {"unique_kv_bytes": unique_kv, "logical_kv_bytes": logical_kv, "write_bytes": write_bytes,
            "q_out_bytes": q_out, "step_bytes": unique_kv + q_out + write_bytes, "flops": flops,
            "per_class": per_class, "tokens": n}


KERNEL_CLASS = {"attn_mma_decode": ("decode", "padding"), "attn_mma_prefill": ("prefill_mma",),
                "attn_tc_prefill": ("prefill_tensor",),
                # one launch for a mixed batch: decode CTAs ahead of the tcgen05 prefill CTAs
                "attn_tc_mixed": ("prefill_tensor", "decode", "padding")}
KERNEL_BOUND = {"paged_kv_write": "hbm", "attn_mma_decode": "hbm", "attn_mma_prefill": "tensor",
                "attn_tc_prefill": "tensor", "attn_tc_mixed": "tensor", "attn_split_combine": "hbm"}


DECODE_CLASSES = ("decode", "padding")


def kernel_work(name, acc, combined=True):
    """(algorithmic bytes, FLOPs) of one step attributable to kernel `name`.
    combined: the step is one pkv_paged_kv_write_attention call, whose decode
    kernels write the decode-class rows and whose scatter writes the rest."""
    if name == "paged_kv_write":
        if not combined:
            return acc["write_bytes"], 0.0
        return sum(c["write_bytes"] for cls, c in acc["per_class"].items() if cls not in DECODE_CLASSES), 0.0
    b = f = 0.0
    for cls in KERNEL_CLASS.get(name, ()):
        c = acc["per_class"].get(cls)
        if c:
            b += c["kv_bytes"] + c["q_out_bytes"] + (c["write_bytes"] if combined and cls in DECODE_CLASSES else 0)
            f += c["flops"]
    return b, f


def alu_peak_tflops(peaks):
    return SM_COUNT * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12


def source_hash(name):
    """Hash of a kernel's source file and the shared device headers, to tell
    whether stored ncu counters are current."""
    fname = {"paged_kv_write": "kv_write.cu", "attn_split_combine": "attn_combine.cu", "attn_tc_prefill": "attn_tc.cu",
             "attn_tc_mixed": "attn_tc.cu", "attn_mma_decode": "attn_mma.cu", "attn_mma_prefill": "attn_mma.cu"}.get(name)
    csrc = os.path.join(ROOT, "paged_kv_cache_84_gb300", "csrc")
    if not fname or not os.path.exists(os.path.join(csrc, fname)):
        return None
    h = hashlib.sha256()
    for f in (fname, "common.cuh", "sm100.cuh", "mma_tiles.cuh", "decode_warp.cuh"):
        path = os.path.join(csrc, f)
        if os.path.exists(path):
            with open(path, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:12]


def stored_traffic(name, workload):
    """DRAM bytes per launch from a committed ncu summary (profiles/ncu_traffic.txt:
    `kernel workload bytes_per_launch source_hash`), or None when absent or stale."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    h = source_hash(name)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == name and parts[1] == workload:
            return float(parts[2]) if parts[3] == h else None
    return None


def roofline(name, avg_s, launches_per_step, acc, peaks, workload):
    b, f = kernel_work(name, acc)
    b /= launches_per_step
    f /= launches_per_step
    bound = KERNEL_BOUND.get(name, "hbm")
    # A kernel whose class is tensor-bound at scale may be closer to the HBM
    # roofline on a small, latency-bound workload: report the binding one,
    # the roofline this launch comes closest to.
    hbm_frac = b / avg_s / 1e9 / peaks["hbm_gbs"]
    tensor_frac = f / avg_s / 1e12 / peaks["bf16_tflops"]
    if bound == "tensor" and hbm_frac > tensor_frac:
        bound = "hbm"
    if bound == "hbm":
        achieved, peak, unit = b / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
        note = f"of {peaks['source']} HBM copy bandwidth"
    elif bound == "tensor":
        achieved, peak, unit = f / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        note = f"of {peaks['source']} bf16 dense (burst)"
    else:
        achieved, peak, unit = f / avg_s / 1e12, alu_peak_tflops(peaks), "TFLOP/s"
        note = "of fp32 FMA peak derived as 152 SMs x 128 lanes x 2 flop x max SM clock"
    res = {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
           "frac": achieved / peak, "traffic": stored_traffic(name, workload), "peak_note": note,
           "hbm_frac": hbm_frac, "tensor_frac": tensor_frac,
           "algorithmic_bytes_per_launch": b, "algorithmic_flops_per_launch": f,
           "avg_launch_us": avg_s * 1e6}
    if bound == "tensor" and peaks.get("bf16_tflops_sustained"):
        # beside the burst peak: the measured rate of a seconds-long GEMM loop under the power cap
        res["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    return res


# ---------------------------------------------------------------------------- GPU arm

def upload_graph(g, stream):
    """Upload an instantiated CUDA graph to the device (driver cuGraphUpload)
    before it is timed.  Otherwise the graph's first launch uploads it, a
    one-time cost of ~2 us per node that would land in the timed region.
    Returns whether the upload ran."""
    try:
        h = g.raw_cuda_graph_exec()
        h = h if isinstance(h, int) else int(h)
        lib = ctypes.CDLL("libcuda.so.1")
        lib.cuGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.cuGraphUpload.restype = ctypes.c_int
        ok = lib.cuGraphUpload(ctypes.c_void_p(h), ctypes.c_void_p(stream.cuda_stream)) == 0
        torch.cuda.synchronize()
        return ok
    except Exception:
        return False


class Step:
    """One copy of a workload resident on the device."""

    def __init__(self, pkv, batch, device):
        m, s = batch.meta, batch.spec
        self.pkv, self.spec, self.meta = pkv, s, m
        self.kc = batch.k_cache.to(device)
        self.vc = batch.v_cache.to(device)
        self.q, self.k, self.v = batch.q.to(device), batch.k.to(device), batch.v.to(device)
        self.qsl = torch.tensor(m.query_start_loc, dtype=torch.int32, device=device)
        self.sl = torch.tensor(m.seq_lens, dtype=torch.int32, device=device)
        self.bt = m.block_table.to(device)
        self.slots = m.slot_mapping.to(device)
        self.out = torch.empty_like(self.q)
        self.ws = pkv.make_workspace(pkv.attention_workspace_bytes(
            max(1, m.num_reqs), max(1, m.num_tokens), s.num_q_heads, s.head_dim, max(1, m.max_seq_len)), device)
        self.qsl_h = torch.tensor(m.query_start_loc, dtype=torch.int32)
        self.sl_h = torch.tensor(m.seq_lens, dtype=torch.int32)

    def nbytes(self):
        ts = (self.kc, self.vc, self.q, self.k, self.v, self.out, self.bt, self.slots)
        return sum(t.numel() * t.element_size() for t in ts)

    def run(self, q=None, k=None, v=None, qsl=None, sl=None, bt=None, slots=None, out=None):
        """The step: the write and the attention as one pkv_paged_kv_write_attention call."""
        self.pkv.paged_kv_write_attention(
            k if k is not None else self.k, v if v is not None else self.v, self.kc, self.vc,
            slots if slots is not None else self.slots, out if out is not None else self.out,
            q if q is not None else self.q, qsl if qsl is not None else self.qsl,
            sl if sl is not None else self.sl, bt if bt is not None else self.bt,
            self.qsl_h, self.sl_h, self.meta.max_query_len, self.meta.max_seq_len, self.spec.scale, self.ws)

    def run_two_calls(self):
        """The same step as pkv_paged_kv_write followed by pkv_ragged_paged_attention."""
        pkv = self.pkv
        pkv.paged_kv_write(self.k, self.v, self.kc, self.vc, self.slots)
        pkv.ragged_paged_attention(self.out, self.q, self.kc, self.vc, self.qsl, self.sl, self.bt,
                                   self.qsl_h, self.sl_h, self.meta.max_query_len, self.meta.max_seq_len,
                                   self.spec.scale, self.ws)


def build_copies(pkv, cfg, device, max_copies=512, subset=0):
    spec = config_spec(cfg)
    if subset:
        spec = subset_spec(spec, subset)
    gen_dev = "cpu" if cfg in (1, 2) else device
    batch = make_batch(spec, device=gen_dev)
    first = Step(pkv, batch, device)
    copies = [first]
    per = first.nbytes()
    n = 1 if per > 2 * L2_BYTES else min(max_copies, math.ceil(2 * L2_BYTES / per) + 1)
    for _ in range(n - 1):
        copies.append(Step(pkv, batch, device))
    del batch
    return spec, copies


def time_workload(pkv, cfg, steps, warmup, device, peaks, dist=None, use_graph=True, subset=0):
    spec, copies = build_copies(pkv, cfg, device, subset=subset)
    meta = copies[0].meta
    classes = pkv.plan_request_kernels(meta.query_start_loc, meta.seq_lens, spec.num_q_heads,
                                       spec.num_kv_heads, spec.head_dim)
    acc = accounting(spec, meta, classes)
    stream = torch.cuda.current_stream()
    for i in range(max(3, warmup)):
        copies[i % len(copies)].run()
    torch.cuda.synchronize()
    before = pkv.launch_count()
    copies[0].run()
    torch.cuda.synchronize()
    launches_per_step = pkv.launch_count() - before

    # The timed region replays ONE CUDA graph that holds exactly `steps`
    # steps, each on the next rotated copy: the steps run back to back on the
    # device, as one layer's attention does inside a model's graph.  Graphs of
    # one step each are also timed, as a diagnostic of the per-replay cost.
    run_graph, per_graphs, uploaded = None, [], False
    if use_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for c in copies:
                c.run()
        torch.cuda.synchronize()
        warm_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(warm_graph, stream=side):
            for i in range(max(3, warmup)):
                copies[i % len(copies)].run()
        run_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(run_graph, stream=side):
            for i in range(steps):
                copies[i % len(copies)].run()
        for c in copies[:8]:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                c.run()
            per_graphs.append(g)
        torch.cuda.synchronize()
        uploaded = all([upload_graph(g, stream) for g in [warm_graph, run_graph] + per_graphs])
        warm_graph.replay()                               # the W untimed warm-up steps
        torch.cuda.synchronize()
    else:
        for i in range(max(3, warmup)):
            copies[i % len(copies)].run()
        torch.cuda.synchronize()

    # ---- timed region: exactly `steps` steps
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    if run_graph is not None:
        run_graph.replay()
    else:
        for i in range(steps):
            copies[i % len(copies)].run()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist is not None:
        dist.barrier()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), dist, device)
    ms_per_step = elapsed_ms / steps

    # The same steps as two calls (pkv_paged_kv_write, then the attention),
    # one graph of `steps` steps: the separate-call path, for comparison.
    two_calls_ms = None
    if use_graph:
        side2 = torch.cuda.Stream()
        side2.wait_stream(stream)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=side2):
            for i in range(steps):
                copies[i % len(copies)].run_two_calls()
        torch.cuda.synchronize()
        upload_graph(g2, stream)
        ev0.record(stream)
        g2.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        two_calls_ms = ev0.elapsed_time(ev1) / steps
        del g2

    # Workloads whose inputs fit in L2 (rotated across copies for the timed
    # value): the same steps on one copy, its inputs warm in L2, as a
    # diagnostic beside the L2-cold value.
    warm_ms = None
    if use_graph and len(copies) > 1:
        side4 = torch.cuda.Stream()
        side4.wait_stream(stream)
        g4 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g4, stream=side4):
            for _ in range(steps):
                copies[0].run()
        torch.cuda.synchronize()
        upload_graph(g4, stream)
        g4.replay()
        torch.cuda.synchronize()
        ev0.record(stream)
        g4.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        warm_ms = ev0.elapsed_time(ev1) / steps
        del g4

    # Latency-bound workloads (inputs that fit in L2): the floor of one
    # library launch, a graph of `steps` back-to-back 16-byte device copies
    # (pkv_copy_async, each a programmatic dependent of the one before, as
    # the step's launches are), reported beside the step.
    floor_ms = None
    if use_graph and len(copies) > 1:
        a = torch.zeros(4, dtype=torch.int32, device=device)
        b_ = torch.ones(4, dtype=torch.int32, device=device)
        side5 = torch.cuda.Stream()
        side5.wait_stream(stream)
        with torch.cuda.stream(side5):
            pkv.copy_async(a, b_, stream=side5)
        torch.cuda.synchronize()
        g5 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g5, stream=side5):
            for i in range(steps):
                pkv.copy_async(a if i % 2 else b_, b_ if i % 2 else a, stream=side5)
        torch.cuda.synchronize()
        upload_graph(g5, stream)
        g5.replay()
        torch.cuda.synchronize()
        ev0.record(stream)
        g5.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        floor_ms = ev0.elapsed_time(ev1) / steps
        del g5

    per_replay_ms = None
    if per_graphs:
        n = max(len(per_graphs), min(steps, 200))
        ev0.record(stream)
        for i in range(n):
            per_graphs[i % len(per_graphs)].replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        per_replay_ms = ev0.elapsed_time(ev1) / n

    # ---- per-kernel durations: CUDA events around every library launch,
    # recorded as event nodes of a second graph of the same `steps` steps
    # (the step as timed above: overlapped classes, rotated copies), read
    # after that graph has run once.  Event nodes sit between the kernels,
    # so each event pair spans its kernel alone; the per-launch eager
    # events used when capture is unavailable add the launch overhead.
    recs, kernel_timing = None, None
    if use_graph:
        try:
            pkv.profile_start(steps * launches_per_step + 16)
            side3 = torch.cuda.Stream()
            side3.wait_stream(stream)
            gp = torch.cuda.CUDAGraph()
            try:
                with torch.cuda.graph(gp, stream=side3):
                    for i in range(steps):
                        copies[i % len(copies)].run()
            finally:
                n_rec = pkv.profile_stop(read=False)
            torch.cuda.synchronize()
            upload_graph(gp, stream)
            gp.replay()
            torch.cuda.synchronize()
            recs = pkv.profile_records(n_rec)
            kernel_timing = "event nodes around every launch in a CUDA graph of %d steps" % steps
            del gp
        except Exception as e:                          # noqa: BLE001 - fall back to eager events
            torch.cuda.synchronize()
            kernel_timing = "eager per-launch events (graph capture of the events failed: %s)" % (
                str(e).splitlines()[0][:120] if str(e) else type(e).__name__)
            recs = None
    if recs is None:
        prof_steps = max(3, min(steps, 50))
        pkv.profile_start(prof_steps * launches_per_step + 16)
        for i in range(prof_steps):
            copies[i % len(copies)].run()
        recs = pkv.profile_stop()
        kernel_timing = kernel_timing or "eager per-launch events over %d steps" % prof_steps
        prof_steps_seen = prof_steps
    else:
        prof_steps_seen = steps
    kern = {}
    for name, ms in recs:
        k = kern.setdefault(name, {"launches": 0, "total_ms": 0.0})
        k["launches"] += 1
        k["total_ms"] += ms
    total = sum(k["total_ms"] for k in kern.values()) or 1.0
    kernels = {}
    for name, k in kern.items():
        kernels[name] = {"launches_per_step": k["launches"] / prof_steps_seen,
                         "avg_launch_us": 1e3 * k["total_ms"] / k["launches"],
                         "share": k["total_ms"] / total}
    # The kernel that bounds the step is the one with the most algorithmic
    # work against its own roofline (bytes at HBM peak, flops at tensor
    # peak).  Event spans cannot pick it when the classes overlap: a decode
    # kernel on the side stream stays resident, filling the SMs the prefill
    # leaves, for about as long as the whole step.
    def ideal_s(name):
        b, f = kernel_work(name, acc)
        return max(b / (peaks["hbm_gbs"] * 1e9), f / (peaks["bf16_tflops"] * 1e12))

    dominant = max(kern, key=lambda n: (ideal_s(n), kern[n]["total_ms"])) if kern else None
    roof = None
    if dominant:
        avg_s = kern[dominant]["total_ms"] / kern[dominant]["launches"] / 1e3
        bounded = False
        # a kernel cannot take longer than the whole step it is part of:
        # where the event bracket says so (launch overhead on a latency-bound
        # kernel), the step time bounds the kernel time instead
        if avg_s * kernels[dominant]["launches_per_step"] > ms_per_step / 1e3:
            avg_s = ms_per_step / 1e3 / kernels[dominant]["launches_per_step"]
            bounded = True
        roof = roofline(dominant, avg_s, kernels[dominant]["launches_per_step"], acc, peaks, f"cfg{cfg}")
        roof["timing"] = kernel_timing + ("; bounded by the step time" if bounded else "")
        roof["dominant_rule"] = "the launch with the most algorithmic work against its roofline"

    step_s = ms_per_step / 1e3
    res = {
        "workload": spec.name, "config_index": cfg,
        "ms_per_step": ms_per_step, "step_us": ms_per_step * 1e3,
        "query_tokens_per_s": acc["tokens"] / step_s,
        "kv_read_gbs": acc["unique_kv_bytes"] / step_s / 1e9,
        "kv_read_frac_of_8tbs": acc["unique_kv_bytes"] / step_s / 1e9 / NOMINAL_HBM_GBS,
        "step_hbm_frac": acc["step_bytes"] / step_s / 1e9 / peaks["hbm_gbs"],
        "step_tensor_frac": acc["flops"] / step_s / 1e12 / peaks["bf16_tflops"],
        "algorithmic": {k: acc[k] for k in ("unique_kv_bytes", "logical_kv_bytes", "q_out_bytes",
                                            "write_bytes", "step_bytes", "flops", "tokens")},
        "launches_per_step": launches_per_step, "copies": len(copies),
        "inputs_bytes_per_copy": copies[0].nbytes(),
        "l2": ("rotating %d copies of the inputs (%.0f MB > 2x L2)" % (len(copies), len(copies) * copies[0].nbytes() / 1e6)
               if len(copies) > 1 else "inputs larger than 2x L2"),
        "launch": (("one CUDA graph of %d steps (pkv_paged_kv_write_attention each) over the rotated copies" % steps) +
                   (", uploaded to the device before the timed region" if uploaded else "")
                   if run_graph is not None else "eager"),
        "ms_per_step_one_graph_per_step": per_replay_ms,
        "ms_per_step_two_calls": two_calls_ms,
        "step_us_warm_l2": warm_ms * 1e3 if warm_ms is not None else None,
        "launch_floor_us": floor_ms * 1e3 if floor_ms is not None else None,
        "kernels": kernels, "roofline": roof, "timed_wall": (t_wall0, t_wall1),
    }
    return spec, copies, res


def e2e_workload(pkv, copies, steps, device, dist=None, world=1):
    """Same step through the C ABI from pinned host memory: every step copies
    that step's inputs (q, k, v and the batch metadata, packed in one pinned
    buffer as a batch builder lays them out) to the device, runs the write and
    the attention, and copies the output back to pinned host memory, all inside
    the timed region.  Timed as one CUDA graph holding exactly `steps` such
    steps over the rotated device copies (like the kernel-only timing), with
    the input and output copies on streams of their own, overlapping other
    steps' attention (the reported value), with
    each step's copies in line (serial_ms_per_step), and as eager calls from
    Python (a diagnostic of the per-call host cost)."""
    c0 = copies[0]
    names = ("q", "k", "v", "qsl", "sl", "bt", "slots")
    offs, total = {}, 0
    for name in names:
        t = getattr(c0, name)
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()

    def views(buf):
        out = {}
        for name in names:
            t = getattr(c0, name)
            n = t.numel() * t.element_size()
            out[name] = buf[offs[name]:offs[name] + n].view(t.dtype).view(t.shape)
        return out

    hv = views(host)
    for name in names:
        hv[name].copy_(getattr(c0, name).cpu())
    # at least four input and output buffers, so that a step's copies can
    # overlap other steps even when one device copy of the workload fills
    # L2: step i's input copy waits only for the output copy of step i - 4
    devbufs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(max(4, len(copies)))]
    dev = [views(b) for b in devbufs]
    outbufs = [torch.empty_like(c0.out) for _ in devbufs]
    outs_h = torch.empty_like(c0.out, device="cpu").pin_memory()
    stream = torch.cuda.current_stream()
    h2d = sum(hv[name].numel() * hv[name].element_size() for name in names)
    d2h = outs_h.numel() * outs_h.element_size()

    def one(i):
        # the library's copy kernel moves the packed inputs in and the output
        # out (pinned host memory addressed by the kernel)
        c, b, d = copies[i % len(copies)], devbufs[i % len(devbufs)], dev[i % len(dev)]
        pkv.copy_async(b, host)
        c.run(q=d["q"], k=d["k"], v=d["v"], qsl=d["qsl"], sl=d["sl"], bt=d["bt"], slots=d["slots"])
        pkv.copy_async(outs_h, c.out)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, n):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(ev0.elapsed_time(ev1) / n, dist, device)

    eager_ms = timed(lambda: [one(i) for i in range(steps)], steps)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined(n):
        # Each step's input copy on one stream, its output copy on another,
        # the steps themselves on the current stream.  Step i waits for its
        # inputs; its output copy waits for step i.  Step i reads input buffer
        # i % L and writes output buffer i % L (L >= 2 of each), which step
        # i - L used: its input copy waits for step i - L's output copy alone,
        # so the input copies run ahead of the steps and step i's output
        # buffer is free once its inputs are in.
        cur = torch.cuda.current_stream()
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        L = len(devbufs)
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_c = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]

        def copy_in(i):
            with torch.cuda.stream(s_in):
                if i >= L:
                    s_in.wait_event(ev_out[i - L])
                pkv.copy_async(devbufs[i % L], host)
                ev_in[i].record(s_in)

        nxt = 0
        for i in range(n):
            while nxt < n and nxt - L < i:                  # issue every input copy whose wait is recorded
                copy_in(nxt)
                nxt += 1
            c, d, o = copies[i % len(copies)], dev[i % L], outbufs[i % L]
            cur.wait_event(ev_in[i])
            c.run(q=d["q"], k=d["k"], v=d["v"], qsl=d["qsl"], sl=d["sl"], bt=d["bt"], slots=d["slots"], out=o)
            ev_c[i].record(cur)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[i])
                pkv.copy_async(outs_h, o)
                ev_out[i].record(s_out)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    graph_ms, pipe_ms, why = None, None, None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(steps):
                one(i)
        torch.cuda.synchronize()
        upload_graph(g, stream)
        graph_ms = timed(g.replay, steps)
        side.wait_stream(stream)
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=side):
            pipelined(steps)
        torch.cuda.synchronize()
        upload_graph(gp, stream)
        pipe_ms = timed(gp.replay, steps)
    except Exception as e:                                  # capture of host copies unsupported
        why = str(e).splitlines()[0][:160] if str(e) else type(e).__name__
        torch.cuda.synchronize()
    ms = pipe_ms if pipe_ms is not None else graph_ms if graph_ms is not None else eager_ms
    if pipe_ms is not None:
        path = ("one CUDA graph of %d steps with the copies on two more streams: each step's packed pinned "
                "inputs move in by pkv_copy_async ahead of the step (up to the rotated buffers), the step runs "
                "pkv_paged_kv_write_attention once its inputs are in, and its output moves out to pinned "
                "memory by pkv_copy_async once it is done" % steps)
    elif graph_ms is not None:
        path = ("one CUDA graph of %d steps; each: pkv_copy_async of the packed pinned inputs to the device, "
                "pkv_paged_kv_write_attention, pkv_copy_async of the output to pinned memory" % steps)
    else:
        path = ("eager Python calls per step: pkv_copy_async of the packed pinned inputs to the device, "
                "pkv_paged_kv_write_attention, pkv_copy_async of the output to pinned memory")
    res = {"value": job_value(c0.meta.num_tokens, world, ms), "unit": UNIT, "ms_per_step": ms,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "path": path,
           "serial_ms_per_step": graph_ms, "eager_ms_per_step": eager_ms}
    if why is not None:
        res["graph_unavailable"] = why
    return res


def fp8_workload(pkv, cfg, device, peaks, steps=20, subset=0):
    """Workload `cfg` on a quantized pool: the whole bf16 pool is quantized
    once by the library's quantizing write, then each timed step is the
    quantizing write of the step's rows + attention over E4M3 codes and per
    (slot, head) scales as one pkv_paged_kv_write_attention_fp8 call, one
    CUDA graph of `steps` steps.  The workspace
    includes pkv_fp8_prefill_scratch_bytes, so prefill chunks run on tcgen05
    over bf16 copies of their blocks.  subset: the first N requests only."""
    spec = config_spec(cfg)
    if subset:
        spec = subset_spec(spec, subset)
    b = make_batch(spec, device=device)
    m = b.meta
    nbt, bs, hkv, d = b.k_cache.shape
    kc = torch.empty((nbt, bs, hkv, d), dtype=torch.uint8, device=device)
    vc = torch.empty_like(kc)
    ks = torch.empty((nbt, bs, hkv), dtype=torch.float32, device=device)
    vs = torch.empty_like(ks)
    all_slots = torch.arange(nbt * bs, dtype=torch.int64, device=device)
    for s0 in range(0, nbt * bs, 1 << 20):                 # quantize the pool in slices
        sl = all_slots[s0:s0 + (1 << 20)]
        pkv.paged_kv_write_fp8(b.k_cache.view(-1, hkv, d)[sl], b.v_cache.view(-1, hkv, d)[sl], kc, vc, ks, vs, sl)
    del b.k_cache, b.v_cache
    torch.cuda.empty_cache()
    q, k, v = b.q.to(device), b.k.to(device), b.v.to(device)
    slots = m.slot_mapping.to(device)
    qsl = torch.tensor(m.query_start_loc, dtype=torch.int32, device=device)
    sln = torch.tensor(m.seq_lens, dtype=torch.int32, device=device)
    bt = m.block_table.to(device)
    out = torch.empty_like(q)
    extra = pkv.fp8_prefill_scratch_bytes(m.query_start_loc, m.seq_lens, spec.num_q_heads, spec.num_kv_heads, d)
    ws = pkv.make_workspace(pkv.attention_workspace_bytes(m.num_reqs, m.num_tokens, spec.num_q_heads, d,
                                                          m.max_seq_len) + extra, device)

    def step():
        pkv.paged_kv_write_attention_fp8(k, v, kc, vc, ks, vs, slots, out, q, qsl, sln, bt, m.query_start_loc,
                                         m.seq_lens, m.max_query_len, m.max_seq_len, spec.scale, ws)

    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(steps):
            step()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    step_s = e0.elapsed_time(e1) / steps / 1e3
    # per-kernel durations: event nodes around every launch of a second graph
    # of the same steps (as in time_workload)
    kernels = None
    try:
        before = pkv.launch_count()
        step()
        torch.cuda.synchronize()
        per_step = pkv.launch_count() - before
        pkv.profile_start(steps * per_step + 16)
        gp = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(gp, stream=side):
                for _ in range(steps):
                    step()
        finally:
            n_rec = pkv.profile_stop(read=False)
        torch.cuda.synchronize()
        gp.replay()
        torch.cuda.synchronize()
        kern = {}
        for name, ms in pkv.profile_records(n_rec):
            k = kern.setdefault(name, [0, 0.0])
            k[0] += 1
            k[1] += ms
        kernels = {name: {"launches_per_step": c / steps, "avg_launch_us": 1e3 * t / c} for name, (c, t) in kern.items()}
        del gp
    except Exception:                                   # noqa: BLE001 - a diagnostic only
        torch.cuda.synchronize()
    # algorithmic bytes: every unique slot read once (codes of K and V + their scales), q, out, the write
    used = set()
    for r in range(m.num_reqs):
        L = m.seq_lens[r]
        used.update(m.block_table[r, :(L + bs - 1) // bs].tolist())
    kv_bytes = sum(min(bs, max(0, m.seq_lens[r] - j * bs)) for r in range(m.num_reqs)
                   for j in range((m.seq_lens[r] + bs - 1) // bs)) * hkv * (2 * d + 8)
    other = 2 * q.numel() * 2 + m.num_tokens * hkv * (2 * d * 2 + 2 * d + 8)
    flops = sum(4.0 * d * spec.num_q_heads * (t * (L - t) + t * (t + 1) / 2)
                for t, L in ((m.query_start_loc[r + 1] - m.query_start_loc[r], m.seq_lens[r]) for r in range(m.num_reqs))
                if L > 0 and t > 0)
    res = {"workload": spec.name, "step_us": step_s * 1e6, "query_tokens_per_s": m.num_tokens / step_s,
           "kv_bytes": kv_bytes, "kv_read_gbs": kv_bytes / step_s / 1e9,
           "step_hbm_frac": (kv_bytes + other) / step_s / 1e9 / peaks["hbm_gbs"],
           "step_tensor_frac": flops / step_s / 1e12 / peaks["bf16_tflops"],
           "prefill_scratch_bytes": extra,
           "pool": "E4M3 codes + fp32 scale per (slot, head)", "kernels": kernels}
    del kc, vc, ks, vs, q, k, v, out, ws, g
    torch.cuda.empty_cache()
    return res


def block_copy_workload(pkv, device, peaks, reps=20):
    """Copy-on-write and swap-out/in of whole blocks over 8 pools (4 layers' K and V, 16 x 8 heads x
    128 dims per block = 32 KB), 1 GB of pools: the block copies of the block manager, timed with CUDA
    events over `reps` calls each.  Copy-on-write moves 1024 blocks per pool per call; swap-out
    gathers 256 blocks per pool into pinned host memory, swap-in scatters them back."""
    nbt, bs, hkv, d = 4096, 16, 8, 128
    gen = torch.Generator(device=device).manual_seed(77)
    pools = [torch.empty((nbt, bs, hkv, d), dtype=torch.bfloat16, device=device) for _ in range(8)]
    for t in pools:
        fill_normal_bf16(t, gen)
    bb = bs * hkv * d * 2
    perm = torch.randperm(nbt, generator=torch.Generator().manual_seed(78)).to(torch.int32)
    srcs = [perm[i * 2048:i * 2048 + 1024].to(device) for i in range(2)]
    dsts = [perm[i * 2048 + 1024:(i + 1) * 2048].to(device) for i in range(2)]
    ids = perm[:256].to(device)
    host = torch.empty((len(pools), 256, bb), dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream()

    def timed(fn):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps / 1e3

    cow_s = timed(lambda i: pkv.copy_blocks(pools, srcs[i % 2], dsts[i % 2]))
    out_s = timed(lambda i: pkv.gather_blocks(pools, ids, host))
    in_s = timed(lambda i: pkv.scatter_blocks(pools, ids, host))
    cow_bytes = 2 * len(pools) * 1024 * bb                     # read + write
    swap_bytes = len(pools) * 256 * bb
    res = {
        "pools": len(pools), "block_bytes": bb, "pool_bytes_total": len(pools) * nbt * bb,
        "copy_on_write": {"blocks_per_pool": 1024, "us": cow_s * 1e6, "gbs": cow_bytes / cow_s / 1e9,
                          "frac_of_hbm": cow_bytes / cow_s / 1e9 / peaks["hbm_gbs"],
                          "bytes": "HBM read + write of the copied blocks"},
        "swap_out_to_pinned_host": {"blocks_per_pool": 256, "us": out_s * 1e6, "gbs": swap_bytes / out_s / 1e9},
        "swap_in_from_pinned_host": {"blocks_per_pool": 256, "us": in_s * 1e6, "gbs": swap_bytes / in_s / 1e9},
    }
    del pools, host
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------- CPU oracle

class OracleStep:
    """The workload's step on the CPU oracle: the write of the step's rows,
    then attention.  Its inputs are drawn exactly as the GPU arm draws them
    (on the device when there is one, for the multi-GB pools, then copied to
    host memory).  A step's attention can be timed whole or on a sample of
    its query tokens (all heads of every sampled token); a sample's time is
    scaled to the whole step by the keys the step's rows attend to, which
    the oracle's work follows (one pass over each visible key per row)."""

    def __init__(self, cfg, threads):
        import oracle
        self.oracle = oracle
        self.spec = spec = config_spec(cfg)
        dev = "cuda" if (cfg not in (1, 2) and torch.cuda.is_available()) else "cpu"
        b = make_batch(spec, device=dev)
        if dev != "cpu":
            b = Batch(spec, b.meta, b.q.cpu(), b.k.cpu(), b.v.cpu(), b.k_cache.cpu(), b.v_cache.cpu())
            torch.cuda.empty_cache()
        self.b, self.m, self.threads = b, b.meta, threads
        m = self.m
        self.keys = []                                   # keys each query row attends to
        for r in range(m.num_reqs):
            t, L = m.query_start_loc[r + 1] - m.query_start_loc[r], m.seq_lens[r]
            self.keys.extend(0 if L == 0 else L - t + i + 1 for i in range(t))
        self.total_keys = sum(self.keys)
        self.tokens = m.num_tokens

    def write(self):
        b = self.b
        self.oracle.paged_kv_write(b.k_cache, b.v_cache, b.k, b.v, self.m.slot_mapping)

    def attend_full(self):
        b, m = self.b, self.m
        self.oracle.ragged_paged_attention(b.q, b.k_cache, b.v_cache, m.query_start_loc, m.seq_lens,
                                           m.block_table, self.spec.scale, self.threads)

    def attend_sample(self, stride, offset):
        """Attention of every stride-th query token (all heads); returns the
        factor that scales its time to the whole step's attention."""
        b, m, hq = self.b, self.m, self.spec.num_q_heads
        toks = list(range(offset % stride, self.tokens, stride))
        keys = sum(self.keys[t] for t in toks)
        if not toks or keys == 0:
            toks, keys = [int(max(range(self.tokens), key=lambda t: self.keys[t]))], 0
            keys = self.keys[toks[0]]
        tt = [t for t in toks for _ in range(hq)]
        hh = [h for _ in toks for h in range(hq)]
        self.oracle.attention_rows(tt, hh, b.q, b.k_cache, b.v_cache, m.query_start_loc, m.seq_lens,
                                   m.block_table, self.spec.scale, self.threads)
        return self.total_keys / keys

    def timed_step(self, stride, offset=0):
        """Seconds of one step (write + attention), the attention measured on
        a sample when stride > 1 and scaled to the whole step."""
        t0 = time.perf_counter()
        self.write()
        t1 = time.perf_counter()
        if stride <= 1:
            self.attend_full()
            scale = 1.0
        else:
            scale = self.attend_sample(stride, offset)
        t2 = time.perf_counter()
        return (t1 - t0) + (t2 - t1) * scale

    def stride_for(self, seconds):
        """Token stride whose sampled step takes about `seconds` (1: whole steps)."""
        probe = max(1, self.tokens // 64)
        t0 = time.perf_counter()
        scale = self.attend_sample(probe, 0) if probe > 1 else 1.0
        if probe == 1:
            self.attend_full()
        full = (time.perf_counter() - t0) * scale
        return max(1, math.ceil(full / max(seconds, 1e-3)))

    def describe(self, n, stride, per_step_s):
        what = ("whole steps" if stride <= 1 else
                f"steps whose attention ran on every {stride}-th query token (all heads), its time scaled "
                f"by the keys those rows attend to ({self.total_keys} keys over all rows)")
        return (f"{n} {what} of the {self.spec.name} workload (write + attention) on {self.threads} threads; "
                f"{per_step_s * 1e3:.1f} ms per full step")


def cpu_baseline(cfg, budget_s=6.0):
    """The oracle on the host cores, a bounded sample of the workload's step:
    whole steps where a step fits in a third of the budget, otherwise steps
    whose attention covers every stride-th query token."""
    threads = os.cpu_count() or 1
    st = OracleStep(cfg, threads)
    stride = st.stride_for(budget_s / 3)
    times = []
    t0 = time.perf_counter()
    while not times or time.perf_counter() - t0 < budget_s:
        times.append(st.timed_step(stride, offset=len(times)))
    dt = statistics.median(times)
    # one step on a single thread: whole if that takes under the budget,
    # else on a sample `threads` times sparser (about the same wall time)
    s1 = stride * threads if stride > 1 else (1 if dt * threads < budget_s else threads)
    st.threads = 1
    one_s = st.timed_step(s1)
    st.threads = threads
    return {"value": st.tokens / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": st.describe(len(times), stride, dt),
            "ms_per_step": dt * 1e3, "one_thread_ms_per_step": one_s * 1e3,
            "one_thread_sample_stride": s1, "wall_s": time.perf_counter() - t0}


def run_reference(args):
    """The reference arm: the oracle as it stands on the host cores, K timed
    steps after W warm-up steps of the same workload; each step's attention
    runs on a token sample sized so that the whole run ends within about two
    minutes (whole steps where they are that cheap), scaled to the whole
    step.  Under torchrun rank 0 alone runs and prints."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    st = OracleStep(args.workload, threads)
    warm = max(3, args.warmup)
    per_step = min(5.0, max(0.02, 120.0 / (args.steps + warm)))
    stride = st.stride_for(per_step)
    for i in range(warm):
        st.timed_step(stride, offset=i)
    times = [st.timed_step(stride, offset=warm + i) for i in range(args.steps)]
    dt = sum(times) / len(times)
    value = st.tokens / dt
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": warm, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) values, shapes of the pages' workloads)",
            "config": {"workload": CONFIG_NAMES[args.workload], "query_tokens": st.tokens,
                       "requests": st.m.num_reqs, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": st.describe(args.steps, stride, dt)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import paged_kv_cache_84_gb300 as pkv
    from paged_kv_cache_84_gb300 import build as pkv_build
    if local == 0:
        pkv_build.build()                                # one build per node, in-tree
    if dist is not None:
        dist.barrier()
    pkv.load()
    peaks = load_peaks()
    warmup = max(3, args.warmup)

    clocks = ClockSampler(local).start()
    spec, copies, head = time_workload(pkv, args.workload, args.steps, warmup, device, peaks, dist,
                                       subset=args.subset)
    t0, t1 = head.pop("timed_wall")
    e2e = e2e_workload(pkv, copies, max(3, min(args.steps, 200)), device, dist, world)
    del copies
    torch.cuda.empty_cache()

    breakdown = {}
    block_copies = None
    fp8 = None
    if not args.no_breakdown:
        block_copies = block_copy_workload(pkv, device, peaks)
        fp8 = {str(c): fp8_workload(pkv, c, device, peaks) for c in (3, 4, 5)}
        for cfg in (1, 2, 3, 4, 5):
            if cfg == args.workload:
                r = dict(head)
                r["e2e"] = e2e
            else:
                _, cps, r = time_workload(pkv, cfg, max(10, min(args.steps, 50)), warmup, device, peaks, None)
                r.pop("timed_wall")
                r["e2e"] = e2e_workload(pkv, cps, max(10, min(args.steps, 50)), device)
                del cps
                torch.cuda.empty_cache()
            breakdown[str(cfg)] = r
    clocks.stop()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)
        for cfg, r in breakdown.items():
            r["cpu_baseline"] = cpu if int(cfg) == args.workload else cpu_baseline(int(cfg), budget_s=4.0)
    tokens = head["algorithmic"]["tokens"]
    line = {
        "metric": METRIC, "value": job_value(tokens, world, head["ms_per_step"]), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 values, shapes of the pages' workloads)",
        "config": {"workload": head["workload"], "query_tokens": tokens, "requests": len(spec.reqs),
                   "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
                   "block_size": spec.block_size, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": head["l2"], "launch": head["launch"]},
        "step_us": head["step_us"],
        "step_us_two_calls": (head["ms_per_step_two_calls"] * 1e3 if head["ms_per_step_two_calls"] is not None
                              else None),
        "step_us_one_graph_per_step": (head["ms_per_step_one_graph_per_step"] * 1e3
                                       if head["ms_per_step_one_graph_per_step"] is not None else None),
        "step_us_warm_l2": head["step_us_warm_l2"],
        "launch_floor_us": head["launch_floor_us"],
        "kv_read_gbs": head["kv_read_gbs"],
        "kv_read_frac_of_8tbs": head["kv_read_frac_of_8tbs"],
        "step_tensor_frac": head["step_tensor_frac"], "step_hbm_frac": head["step_hbm_frac"],
        "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": head["launches_per_step"] * args.steps,
        "clocks": clocks.summary(t0, t1), "peaks": peaks, "kernels": head["kernels"],
        "workloads": breakdown, "block_copies": block_copies, "fp8_pool": fp8,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def relaunch_with_ranks(n):
    """Run this same command as n ranks under torch.distributed.run on
    127.0.0.1 (one process per GPU); returns its exit status."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=HEADLINE, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-breakdown", action="store_true", help="time only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--subset", type=int, default=0,
                    help="keep only the first N requests of the workload (smaller profiling runs)")
    ap.add_argument("--fp8", action="store_true",
                    help="time only the workload on a quantized pool (a diagnostic line, for profiling runs)")
    args = ap.parse_args()
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        return relaunch_with_ranks(args.gpus)
    if world is not None and int(world) != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU", file=sys.stderr)
        return 2
    if args.impl == "reference":
        return run_reference(args)
    if args.fp8:
        return run_fp8(args)
    return run_ours(args)


def run_fp8(args):
    """One workload (or its first --subset requests) on a quantized pool,
    --steps steps in a CUDA graph; prints the fp8 line (not the headline)."""
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    import paged_kv_cache_84_gb300 as pkv
    from paged_kv_cache_84_gb300 import build as pkv_build
    pkv_build.build()
    pkv.load()
    res = fp8_workload(pkv, args.workload, device, load_peaks(), steps=max(1, args.steps), subset=args.subset)
    print(json.dumps({"fp8_pool": res, "steps": args.steps}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
