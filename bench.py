#!/usr/bin/env python
"""Benchmark of one striped paged attention step on GB300.

A step is the whole hot path over one batch: ``cp_kv_write`` of the step's
new K/V into the P-way striped pool, ``cp_paged_attn_partial`` (every
partner's partial with its log-sum-exp), ``own_token_attn`` for non-decode
workloads, and ``lse_merge`` of the partials.  Metric: algorithmic KV bytes the
step reads (every visible key and value once) per second, plus decode
tokens/s; inputs (the KV pool, 1.14 GB for the default workload) are larger
than L2, so no flush is needed between steps.

Default workload: GQA decode, batch 64, 32 query / 8 KV heads, head_dim 128,
page 16, P = 4, context lengths uniform in [512, 8192], bf16, fp32 LSE.

Each timed measurement is ``--windows`` windows of exactly K steps (after W
warm-up steps, a barrier and a synchronize around each window); the line
reports the median window and the spread.  Besides the headline workload the
line carries ``configs``: all five workloads of the specification, each timed
on both paths (``unfused``: partial + lse_merge; ``fused``: the partials merged
by the partial launch), with its partial launch's roofline (HBM, and for MLA
the tensor pipe against the sustained bf16 peak), the end-to-end step through
host buffers on its faster path, and the SM clocks sampled meanwhile.

``--impl reference`` times the float64 CPU oracle on the host cores instead
(the pages publish no implementation or figures to run); under torchrun only
rank 0 runs it.  ``--gpus N`` under torchrun runs N independent replicas (the
path has no cross-GPU step on one box): whole-job value = sum of the ranks'
bytes over the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV-read HBM GB/s (% of peak) and decode tokens/s, striped paged attn + merge"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
# sources whose digest keys the recorded ncu traffic of each partial kernel
KERNEL_SOURCES = {
    # one-token rows (decode steps): the plan, the dispatch, the decode kernels, the merges
    "gqa_partial": ["partial_gqa.cu", "partial_gqa_mma.cu", "partial_gqa_mmat.cu", "gqa_core.cuh",
                    "split_combine.cuh", "common.cuh", "mma_sync.cuh"],
    # non-decode steps add the multi-token kernel
    "gqa_mixed_partial": ["partial_gqa.cu", "partial_gqa_mma.cu", "partial_gqa_mmat.cu", "partial_gqa_ext_ws.cu",
                          "gqa_core.cuh", "split_combine.cuh", "common.cuh", "mma_sync.cuh", "tc05.cuh"],
    "mla_partial": ["partial_gqa.cu", "partial_mla_pair.cu", "tc05.cuh", "split_combine.cuh", "common.cuh"],
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="gqa_decode",
                    choices=["tiny_fp32", "gqa_decode", "long_gqa_decode", "mla_decode", "mixed_step",
                             "gqa_decode_fp8", "mixed_step_fp8"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi")
    ap.add_argument("--path", choices=["fused", "unfused"], default="unfused",
                    help="unfused: partial + lse_merge (the faster on every workload measured); fused: partials "
                         "merged inside the partial launch")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--windows", type=int, default=5,
                    help="timed windows of K steps each (median and spread reported)")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the headline workload only (skip the per-config object)")
    return ap.parse_args()


# the five workloads of the specification, in its order; the headline is the second
CONFIG_NAMES = ["tiny_fp32", "gqa_decode", "long_gqa_decode", "mla_decode", "mixed_step"]


# ---------------------------------------------------------------- workloads

def make_workload(name):
    from context_paged_attention_gb300 import workloads as W

    if name == "gqa_decode_fp8":
        return W.gqa_decode_fp8()
    if name == "mixed_step_fp8":
        return W.fp8_pool(W.mixed_step(), 0.0123, 0.0137)
    return W.WORKLOADS[{"tiny_fp32": 1, "gqa_decode": 2, "long_gqa_decode": 3, "mla_decode": 4,
                        "mixed_step": 5}[name]]()


def describe(w):
    lens = w.ctx_len[: w.num_real_rows] + w.new_len[: w.num_real_rows]
    return {
        "workload": f"{w.name}: {w.num_real_rows} rows, {w.num_q_heads}q/{w.num_kv_heads}kv heads, "
                    f"D {w.head_dim}/{w.head_dim_v}, page {w.page_size}, P {w.P}, {w.dtype}",
        "rows": int(w.num_real_rows),
        "tokens": int(w.num_tokens),
        "q_heads": w.num_q_heads,
        "kv_heads": w.num_kv_heads,
        "head_dim": w.head_dim,
        "head_dim_v": w.head_dim_v,
        "page_size": w.page_size,
        "P": w.P,
        "kv_len_mean": float(lens.mean()),
        "kv_bytes_per_step": int(w.kv_bytes_read()),
        "l2": "inputs larger than L2 (KV pool read each step exceeds 129 MB); no flush",
        "seed": w.meta.get("seed"),
    }


def algorithmic_bytes(w, fused=True):
    """Bytes the partial launch must move at minimum: every visible key once,
    the queries, and its outputs -- the P partials (unfused), or the merged
    output and LSE plus the own-token partial it folds in (fused)."""
    esz = 2 if w.dtype == "bf16" else 4
    T, Hq, D, Dv, P = w.num_tokens, w.num_q_heads, w.head_dim, w.head_dim_v, w.P
    kv = w.kv_bytes_read()
    q = T * Hq * D * esz
    if fused:
        out = T * Hq * (Dv * esz + 4) + (0 if w.decode else T * Hq * (Dv + 1) * 4)
    else:
        out = P * T * Hq * (Dv + 1) * 4
    return {"partial": kv + q + out, "kv": kv}


def launches_per_step(w, fused=True):
    """Kernels of one step: kv_write, the partial (a second kernel for the
    multi-token rows of a non-decode step), own_token (non-decode), and
    lse_merge (unfused) or, for fused MLA steps over 64-slot logical pages,
    the merge of the tokens cut between clusters."""
    n = 1 + 1
    if not w.decode:
        n += 2
    if not fused:
        n += 1
    elif w.mla and w.page_size == 64:
        n += 1
    return n


def algorithmic_flops(w):
    """Tensor-core FLOPs of the pool partial: 2 (D + Dv) per query head, per
    new token of a row and per key it sees in the pool."""
    kv = w.kv_len[: w.num_real_rows].astype("int64")
    n = w.new_len[: w.num_real_rows].astype("int64")
    return int(2 * (w.head_dim + w.head_dim_v) * w.num_q_heads * int((kv * n).sum()))


# ---------------------------------------------------------------- environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(kernel="gqa_partial"):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "context_paged_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel sources still match."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    digest = source_digest(kernel)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = dict(x.split("=", 1) for x in line.split())
            if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("source") == digest:
                return int(kv["dram_bytes_per_launch"])
    return None


_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40}


class _Nvml:
    """Read-only NVML queries through ctypes: SM clock, its maximum, power and
    the active clock-event reasons of one GPU (found by its UUID)."""

    def __init__(self, uuid: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        if self.lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + u)
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def read(self):
        ct = self.ct
        sm, mx, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(sm))       # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reasons_fn(self.h, ct.byref(rs))
        return float(sm.value), float(mx.value), mw.value / 1000.0, int(rs.value)


class ClockSampler:
    """SM clocks and clock-event reasons sampled in the background.

    NVML (read-only) polled every 5 ms, so that even a timed region of a few
    tens of milliseconds holds several samples; ``nvidia-smi -lms 100`` if
    NVML cannot be opened.  Samples are (wall time, sm MHz, max MHz, reasons set).
    """

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    SMI_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int, uuid: str | None = None, period_s: float = 0.005):
        self.samples = []
        self.proc = None
        self.device_index = device_index
        self.uuid = uuid
        self.period = period_s
        self.source = None
        self._stop = threading.Event()

    def start(self):
        nv = None
        if self.uuid:
            try:
                nv = _Nvml(self.uuid)
                nv.read()
            except Exception:
                nv = None
        if nv is not None:
            self.source = "nvml 5 ms"
            threading.Thread(target=self._poll, args=(nv,), daemon=True).start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.source = "nvidia-smi 100 ms"
        threading.Thread(target=self._read, daemon=True).start()

    def _poll(self, nv):
        while not self._stop.is_set():
            try:
                sm, mx, _, bits = nv.read()
            except Exception:
                return
            reasons = {n for n, b in _REASON_BITS.items() if bits & b}
            self.samples.append((time.time(), sm, mx, reasons))
            self._stop.wait(self.period)

    def _read(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                reasons = {self.SMI_NAMES[i] for i in range(4) if parts[4 + i].lower() == "active"}
                self.samples.append((time.time(), num(parts[0]), num(parts[1]), reasons))

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside if inside else [min(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))]
        sm = [s[1] for s in used if s[1] is not None]
        smax = [s[2] for s in used if s[2] is not None]
        reasons = sorted(set().union(*[s[3] for s in used]))
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(used), "window_samples": len(inside), "source": self.source}


# ---------------------------------------------------------------- replicas (N ranks, one GPU each)

def max_over_ranks(dist, values, device):
    """Max of each timing over the ranks (the slowest replica sets the job's time)."""
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world, bytes_per_rank, ms_per_step):
    """Whole-job GB/s: every replica's bytes over the slowest replica's step time."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- CPU oracle timing

def _oracle_row_task(task):
    """One row of the decode step by the float64 oracle (runs in a spawned worker)."""
    import numpy as np

    import oracle

    q_raw, k_raw, v_raw, scale, dv, mla = task
    t0 = time.perf_counter()
    q = oracle.raw_to_f64(q_raw)
    K = oracle.raw_to_f64(k_raw)
    V = K[:, :, :dv] if mla else oracle.raw_to_f64(v_raw)
    for i in range(q.shape[0]):
        oracle.attention(q[i], K[: K.shape[0] - q.shape[0] + i + 1], V[: K.shape[0] - q.shape[0] + i + 1], scale)
    del np
    return time.perf_counter() - t0


def oracle_tasks(w, max_keys=None):
    """Per-row oracle tasks (the step's real rows), optionally a prefix of rows bounded by total keys."""
    tasks, keys, nbytes = [], 0, 0
    esz = 2 if w.dtype == "bf16" else 4
    per_key = w.num_kv_heads * (w.head_dim + (0 if w.mla else w.head_dim_v)) * esz
    for b in range(w.num_real_rows):
        c, n = int(w.ctx_len[b]), int(w.new_len[b])
        s0 = int(w.seq_indptr[b])
        t0 = int(w.qo_indptr[b])
        m = c + n
        tasks.append((w.q[t0: t0 + n], w.k_seq[s0: s0 + m], None if w.mla else w.v_seq[s0: s0 + m], w.scale,
                      w.head_dim_v, w.mla))
        kv = int(w.kv_len[b]) if w.decode else c + n
        keys += kv
        nbytes += kv * per_key
        if max_keys is not None and keys >= max_keys:
            break
    return tasks, nbytes


class OraclePool:
    """Spawned single-threaded workers, one per host core (BLAS threads pinned to 1)."""

    def __init__(self):
        import multiprocessing as mp

        self.cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        for k in saved:
            os.environ[k] = "1"
        self.pool = mp.get_context("spawn").Pool(self.cores)
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v

    def run(self, tasks):
        t0 = time.perf_counter()
        self.pool.map(_oracle_row_task, tasks, chunksize=1)
        return time.perf_counter() - t0

    def run_for(self, tasks, min_s=5.0, max_passes=20):
        """Repeat the sample until at least min_s of wall time (at most max_passes): (seconds, passes)."""
        secs, passes = 0.0, 0
        while passes < max_passes and (passes == 0 or secs < min_s):
            secs += self.run(tasks)
            passes += 1
        return secs, passes

    def close(self):
        self.pool.terminate()


def sample_keys(w):
    """Bound the oracle sample to roughly 10-30 s of single-core float64 work."""
    per_key_cost = w.num_q_heads * (w.head_dim + w.head_dim_v) * 8  # bytes of float64 traffic per key per step
    budget_bytes = 6e10  # ~ 20 s of single-core float64 streaming at ~3 GB/s
    return max(1, int(budget_bytes / per_key_cost))


# ---------------------------------------------------------------- our arm

def load_tflops():
    """Sustained dense bf16 TFLOP/s (for a kernel inside a long step)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


def make_step(att, w, fused, stream):
    """One step of the hot path; ev0/ev1 bracket the partial launch."""

    def step(ev0=None, ev1=None):
        att.write_new()
        if fused:
            if not w.decode:
                att.own()
            if ev0 is not None:
                ev0.record(stream)
            att.fused()
            if ev1 is not None:
                ev1.record(stream)
            return
        if ev0 is not None:
            ev0.record(stream)
        att.partial()
        if ev1 is not None:
            ev1.record(stream)
        if not w.decode:
            att.own()
        att.merge()

    return step


def time_windows(step, K, windows, warmup, stream, dist):
    """W warm-up steps, then `windows` timed windows of exactly K steps, each
    bracketed by a barrier and a synchronize.  Returns per-window ms per step
    and mean partial-launch ms, and the wall-clock span of the windows."""
    import torch

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    win, part = [], []
    t0 = time.time()
    for _ in range(windows):
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(K):
            step(e0[i], e1[i])
        end.record(stream)
        torch.cuda.synchronize()
        win.append(start.elapsed_time(end) / K)
        part.append(sum(e0[i].elapsed_time(e1[i]) for i in range(K)) / K)
    t1 = time.time()
    return win, part, (t0, t1)


def spread(xs):
    return {"median": round(statistics.median(xs), 5), "min": round(min(xs), 5), "max": round(max(xs), 5),
            "windows": len(xs)}


def measure_config(name, args, world, local_rank, dist, sampler, stream, paths=("unfused", "fused"), att_w=None):
    """All of one workload's numbers: both paths timed in repeated windows,
    the partial launch's roofline, the end-to-end step with host buffers and
    the clocks seen meanwhile."""
    import torch
    from context_paged_attention_gb300.step import StripedAttention

    if att_w is None:
        w = make_workload(name)
        att = StripedAttention(w, device=f"cuda:{local_rank}")
    else:
        att, w = att_w
    torch.cuda.synchronize()
    if att.status() != 0:
        raise RuntimeError(f"{name}: device status {att.status()} after filling the pool")
    peak, peak_src = load_peaks()
    tflops, tf_src = load_tflops()
    out = {"workload": describe(w)["workload"], "kv_bytes_per_step": int(w.kv_bytes_read())}
    spans = []
    best = None
    for path in paths:
        fused = path == "fused"
        win, part, span = time_windows(make_step(att, w, fused, stream), args.steps, args.windows, args.warmup,
                                       stream, dist)
        spans.append(span)
        if att.status() != 0:
            raise RuntimeError(f"{name} ({path}): device status {att.status()} during the timed steps")
        if dist is not None:
            win = max_over_ranks(dist, win, f"cuda:{local_rank}")
            part = max_over_ranks(dist, part, f"cuda:{local_rank}")
        ms = statistics.median(win)
        pms = statistics.median(part)
        alg = algorithmic_bytes(w, fused)
        achieved = alg["partial"] / (pms * 1e-3) / 1e9
        roof = {"kernel": ("cp_paged_attn_fused" if fused else "cp_paged_attn_partial"), "bound": "hbm",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "algorithmic_bytes": alg["partial"], "ms_per_launch": round(pms, 5),
                "launch_windows": spread(part), "peak_note": f"of {peak_src}",
                "traffic": recorded_traffic(traffic_kernel(w), name + (":fused" if fused else ""))}
        if w.mla:
            fl = algorithmic_flops(w)
            roof["tensor"] = {"achieved": round(fl / (pms * 1e-3) / 1e12, 1), "peak": tflops, "unit": "TFLOP/s",
                              "frac": round(fl / (pms * 1e-3) / 1e12 / tflops, 4), "flops": fl,
                              "peak_note": f"bf16_tflops_sustained, of {tf_src}"}
        entry = {"ms_per_step": round(ms, 5), "step_windows": spread(win),
                 "value": round(job_throughput(world, alg["kv"], ms), 2), "unit": "GB/s",
                 "frac_of_peak": round(alg["kv"] / (ms * 1e-3) / 1e9 / peak, 4),
                 "decode_tokens_per_s": round(world * int(w.qo_indptr[w.num_real_rows]) / (ms * 1e-3), 1),
                 "roofline": roof, "gpu_launches_per_step": launches_per_step(w, fused)}
        out[path] = entry
        if best is None or ms < out[best]["ms_per_step"]:
            best = path
    out["best_path"] = best
    if not args.no_e2e:
        e = time_e2e(att, w, args, stream, best == "fused")
        if dist is not None:
            e["ms_per_step"] = max_over_ranks(dist, [e["ms_per_step"]], f"cuda:{local_rank}")[0]
        out["e2e"] = {"value": round(world * w.kv_bytes_read() / (e["ms_per_step"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                      "ms_per_step": round(e["ms_per_step"], 5), "path": best}
    if sampler is not None:
        out["clocks"] = sampler.summary(spans[0][0], spans[-1][1])
    return out, att, w


def traffic_kernel(w):
    return "mla_partial" if w.mla else ("gqa_partial" if w.decode else "gqa_mixed_partial")


def run_ours(args, rank, world, local_rank):
    import torch

    import __graft_entry__
    from context_paged_attention_gb300.step import StripedAttention

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    __graft_entry__.build()

    # the oracle workers are spawned before the first GPU call
    opool = OraclePool() if (rank == 0 and not args.no_cpu_baseline) else None
    stream = torch.cuda.current_stream()

    sampler = None
    if not args.no_clocks and rank == 0:
        try:
            uuid = str(torch.cuda.get_device_properties(local_rank).uuid)
        except Exception:
            uuid = None
        sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0, uuid)
        sampler.start()
        time.sleep(0.3)

    # ---- the headline workload, on the requested path
    w = make_workload(args.config)
    att = StripedAttention(w, device=f"cuda:{local_rank}")
    fused = args.path == "fused"
    head, att, w = measure_config(args.config, args, world, local_rank, dist, sampler, stream, paths=(args.path,),
                                  att_w=(att, w))
    h = head[args.path]
    ms = h["ms_per_step"]

    # the same step captured once as a CUDA graph and replayed K times
    graph = None
    if not args.no_graph:
        att.capture(fused)
        for _ in range(args.warmup):
            att.replay()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        g0.record(stream)
        for _ in range(args.steps):
            att.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        gms = g0.elapsed_time(g1) / args.steps
        graph = {"ms_per_step": round(gms, 5), "value": round(world * w.kv_bytes_read() / (gms * 1e-3) / 1e9, 2),
                 "unit": "GB/s", "note": "informational: the same step replayed from one captured CUDA graph"}
    cpu_tasks = oracle_tasks(w, sample_keys(w)) if opool is not None else None
    del att
    torch.cuda.empty_cache()

    # ---- every workload of the specification, both paths
    configs = None
    if not args.no_configs:
        configs = {}
        for name in CONFIG_NAMES:
            entry, a2, _ = measure_config(name, args, world, local_rank, dist, sampler, stream)
            configs[name] = entry
            del a2
            torch.cuda.empty_cache()

    if rank != 0:
        return
    peak, peak_src = load_peaks()
    roof = dict(h["roofline"])
    roof["kernel"] += (" (MLA, tcgen05)" if w.mla else
                       " (GQA, mma.sync decode rows + tcgen05 multi-token rows)" if w.dtype == "bf16" else
                       " (GQA, CUDA cores)")
    roof["traffic"] = recorded_traffic(traffic_kernel(w), args.config + (":fused" if fused else ""))
    line = {
        "metric": METRIC,
        "value": h["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) values, uniform lengths, random page permutation)",
        "config": describe(w) | {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                                 "timing": f"{args.windows} windows of {args.steps} steps after {args.warmup} "
                                           f"warm-up steps; ms_per_step is the median window"},
        "frac_of_peak": h["frac_of_peak"],
        "peak_source": f"{peak_src} hbm_gbs {peak}",
        "decode_tokens_per_s": h["decode_tokens_per_s"],
        "step_windows": h["step_windows"],
        "roofline": roof,
        "gpu_launches": args.steps * launches_per_step(w, fused),
        "launch_note": "per timed window of K steps: " +
                       ("kv_write, the fused partial+merge" if fused else "kv_write, partial, lse_merge") +
                       (" (+ own_token and the multi-token-row partial kernel for non-decode steps)" if not w.decode
                        else "") + "; plus one cudaMemsetAsync of the split-KV tickets when a stripe splits "
                                   "or the call is fused",
        "path": args.path,
    }
    if graph is not None:
        line["graph"] = graph
    if "e2e" in head:
        line["e2e"] = {k: v for k, v in head["e2e"].items() if k != "path"}
    if "clocks" in head:
        line["clocks"] = head["clocks"]
    if configs is not None:
        line["configs"] = configs
    if opool is not None:
        tasks, nbytes = cpu_tasks
        secs, passes = opool.run_for(tasks)
        opool.close()
        line["cpu_baseline"] = {"value": round(passes * nbytes / secs / 1e9, 4), "unit": "GB/s",
                                "cores": opool.cores, "kind": "oracle",
                                "sample": f"float64 oracle over {len(tasks)} of {w.num_real_rows} rows of the same "
                                          f"step ({nbytes / 1e9:.3f} GB of KV), {passes} pass(es), one spawned "
                                          f"single-threaded worker per core, {secs:.2f} s"}
    if sampler is not None:
        sampler.stop()
    print(json.dumps(line), flush=True)


def time_e2e(att, w, args, stream, fused=True):
    """Same step through the public API, its inputs copied each step from one
    pinned host buffer (the step's packed inputs) and its output and LSE read
    back into another."""
    import torch

    host_in = torch.empty(att.packed_inputs.shape, dtype=torch.uint8, pin_memory=True)
    host_in.copy_(att.packed_inputs)
    host_out = torch.empty(att.packed_outputs.shape, dtype=torch.uint8, pin_memory=True)
    h2d = att.packed_inputs.numel()
    d2h = att.packed_outputs.numel()

    def e2e_step():
        att.packed_inputs.copy_(host_in, non_blocking=True)
        if fused:
            att.run_step_fused()
        else:
            att.run_step()
        host_out.copy_(att.packed_outputs, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        e2e_step()
    end.record(stream)
    torch.cuda.synchronize()
    return {"ms_per_step": start.elapsed_time(end) / args.steps, "h2d": h2d, "d2h": d2h}


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return
    opool = OraclePool()
    w = make_workload(args.config)
    tasks, nbytes = oracle_tasks(w, sample_keys(w) // 4)
    for _ in range(args.warmup):
        opool.run(tasks[: max(1, len(tasks) // 8)])
    # time K bounded steps, scaled down so the whole run stays within a few minutes
    per = opool.run(tasks)
    budget = 120.0
    k = max(1, min(args.steps, int(budget / max(per, 1e-3))))
    secs = per
    for _ in range(k - 1):
        secs += opool.run(tasks)
    opool.close()
    ms = secs / k * 1e3
    value = nbytes / (secs / k) / 1e9
    sample = (f"float64 oracle over {len(tasks)} of {w.num_real_rows} rows ({nbytes / 1e9:.3f} GB of KV) per step, "
              f"{k} timed steps, one spawned single-threaded worker per core")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": k,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) values, uniform lengths, random page permutation)",
        "config": describe(w),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": opool.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
