#!/usr/bin/env python
"""Benchmark of the GB300 ragged paged attention library.

One step = one pass of the hot path over one mixed prefill+decode batch shaped like
Llama-3-8B serving (32 q / 8 kv heads, head_dim 128, page_size 16, 128 decode
sequences with kv_len U[512, 4096] and 4 prefill chunks of 512 queries with kv_len
U[512, 2048]): the batch's new K/V rows are written into their pages
and attention runs over the whole batch, in one call (rpa_forward_update: the cache write
of rpa_update_kv_cache shares a launch with rpa_forward's plan).

Printed as one JSON line:
  value      query tokens/s over the whole job, inputs resident in HBM (CUDA events)
  e2e        the same through the public API from pinned host buffers, with the
             host->device copy of every step's inputs and the device->host read of
             its output inside the timed region (double-buffered on two copy
             streams, so the copies of neighbouring steps run under the compute)
  roofline   the dominant kernel's algorithmic bytes (or flops) per launch over its
             CUDA-event duration, against the measured HBM / bf16 peak
  cpu_baseline  the float64 oracle on a bounded sample of the same batch, host cores
  variants   the Gemma-2-style fp8 batch, the DeepSeek MLA batch and the DSA sparse
             MLA batches, measured in the same run (parity cases of the test-suite)

``--impl reference`` times the oracle instead (the reference arm).  Under torchrun
(N > 1) every rank runs an independent replica of the step on its own GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "ragged paged attn tokens/s, HBM GB/s & TFLOP/s as % of GB300 roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer pass (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="llama_mixed",
                    choices=["llama_mixed", "gemma2_fp8_sw_cap", "mla_deepseek_v3", "dsa_sparse_prefill_token",
                             "dsa_sparse_prefill_page", "dsa_sparse_decode_token", "dsa_sparse_decode_page",
                             "dsa_sparse_ragged_token", "dsa_sparse_ragged_page"],
                    help="the headline step is llama_mixed; the others time one variant alone (profiling runs)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# environment: ranks, peaks, clocks
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except Exception:
        return dict(FALLBACK), "fallback"


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (the driver's libnvidia-ml, read-only
    queries) every ~0.5 ms by a thread, so a timed region of a few milliseconds is covered."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, local_rank):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        ident = vis.split(",")[local_rank].strip() if vis else str(local_rank)
        self.h = ctypes.c_void_p()
        if ident.startswith("GPU-") or ident.startswith("MIG-"):
            rc = self.lib.nvmlDeviceGetHandleByUUID(ident.encode(), ctypes.byref(self.h))
        else:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(int(ident), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError(f"nvml handle: {rc}")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None
        self.sm, self.bits, self.stop_flag = [], 0, False

    def _poll(self):
        ct = self.ct
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag:
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) == 0:
                self.sm.append(float(mhz.value))
            if self.reasons_fn(self.h, ct.byref(rs)) == 0:
                self.bits |= rs.value
            time.sleep(0.0005)

    def start(self):
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        return self

    def stop(self):
        self.stop_flag = True
        self.thread.join(timeout=2)
        return {"sm_mhz": statistics.median(self.sm) if self.sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if self.bits & b), "samples": len(self.sm),
                "source": "nvml, ~0.5 ms polling during the timed region"}


def clock_sampler(local_rank):
    try:
        return NvmlSampler(local_rank)
    except Exception:
        return ClockSampler(local_rank)


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.index = vis.split(",")[local_rank] if vis else str(local_rank)
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self.index], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names[1:], parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# algorithmic bytes and flops (what the method must move / compute)
# ---------------------------------------------------------------------------
def _visible(kv_len, q_len, sw):
    """Per query of a sequence: number of visible keys; and unique keys read."""
    qpos = kv_len - q_len + np.arange(q_len, dtype=np.int64)
    lo = np.maximum(0, qpos - sw + 1) if sw else np.zeros_like(qpos)
    vis = qpos + 1 - lo
    uniq = kv_len - (int(lo[0]) if q_len else kv_len)
    return vis, uniq


def rpa_accounting(b):
    Hq, D = b.q.shape[1], b.q.shape[2]
    C = b.kv_pages.shape[2]
    esz = b.kv_pages.element_size()
    G = Hq // (C // 2)
    acc = {"decode": [0, 0, 0], "prefill": [0, 0, 0]}  # tokens, bytes, flops
    for ql, kl in zip(b.q_lens, b.kv_lens_list):
        if ql == 0:
            continue
        vis, uniq = _visible(kl, ql, b.sliding_window)
        part = "decode" if ql * G <= 16 else "prefill"
        acc[part][0] += ql
        acc[part][1] += uniq * C * D * esz + ql * Hq * D * 2 * 2
        acc[part][2] += int(vis.sum()) * 4 * Hq * D
    return acc


def mla_accounting(m):
    H = m.ql_nope.shape[1]
    tok = byt = fl = 0
    dec = [0, 0, 0]
    for ql, kl in zip(m.q_lens, m.kv_lens_list):
        vis, uniq = _visible(kl, ql, m.sliding_window)
        b_ = uniq * 576 * 2 + ql * H * (576 * 2 + 512 * 2) + ql * 576 * 2 * 2
        f_ = int(vis.sum()) * 2 * H * (576 + 512)
        tok, byt, fl = tok + ql, byt + b_, fl + f_
        if ql == 1:
            dec = [dec[0] + 1, dec[1] + b_, dec[2] + f_]
    return tok, byt, fl, dec


def sparse_accounting(s):
    B, S, H, _ = s.q.shape
    RB = s.read_block
    idx = s.indices.numpy().astype(np.int64)
    pos = s.positions.numpy().astype(np.int64)
    units = idx[..., None] * RB + np.arange(RB)  # [B,S,K,RB]
    valid = (idx[..., None] >= 0) & (units <= pos[..., None, None]) & (units < s.seq_len)
    pairs = int(valid.sum())
    rows = 0
    for b in range(B):
        rows += np.unique(units[b][valid[b]]).size
    byt = rows * 576 * 2 + B * S * H * (576 * 2 + 512 * 4)
    fl = pairs * 2 * H * (576 + 512)
    return B * S, byt, fl


def sparse_ragged_accounting(s):
    """Tokens, bytes (the distinct selected rows, Q, the written rows, fp32 O) and flops of one
    packed-ragged call."""
    T, H, _ = s.ql.shape
    RB, ps = s.read_block, s.page_size
    cu_q = s.cu_q_lens.numpy()
    rid = np.clip(np.searchsorted(cu_q[1:], np.arange(T), side="right"), 0, len(s.seq_lens) - 1)
    bound = s.seq_lens.numpy().astype(np.int64)[rid]
    base = s.cu_kv_lens.numpy().astype(np.int64)[rid] // ps
    idx = s.topk.numpy().astype(np.int64)
    pos = s.positions.numpy().astype(np.int64)
    units = idx[..., None] * RB + np.arange(RB)  # [T, K, RB] request-local keys
    valid = (idx[..., None] >= 0) & (units <= pos[:, None, None]) & (units < bound[:, None, None])
    pages = s.page_indices.numpy().astype(np.int64)
    slot = pages[np.minimum(base[:, None, None] + units // ps, len(pages) - 1)] * ps + units % ps
    rows = np.unique(slot[valid]).size
    byt = rows * 576 * 2 + T * H * (576 * 2 + 512 * 4) + T * 640 * 2
    fl = int(valid.sum()) * 2 * H * (576 + 512)
    return T, byt, fl


def roof_time(byt, fl, peaks, sustained=False):
    tf = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return max(byt / (peaks["hbm_gbs"] * 1e9), fl / (tf * 1e12))


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------
def time_steps(fn, steps, warmup, world, timer=False, launches=False):
    """ms per step over `steps` timed steps (CUDA events on the current stream). timer=True
    also brackets every library launch with events (per-kernel times; the library then
    serialises launches it would otherwise overlap); launches=True also returns how many
    library kernels the timed steps launched."""
    from ragged_paged_attention_gb300 import api
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kt = api.KernelTimer() if timer else None
    if kt:
        kt.__enter__()
    n0 = api.launch_count()
    e0.record(st)
    for _ in range(steps):
        fn()
    e1.record(st)
    n1 = api.launch_count()
    torch.cuda.synchronize()
    if kt:
        kt.__exit__(None, None, None)
    barrier(world)
    ms = e0.elapsed_time(e1) / steps
    if launches:
        return ms, (kt.result if kt else {}), n1 - n0
    return ms, (kt.result if kt else {})


def source_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """dram bytes per launch from a committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    m_src = re.search(r"source_file:\s*(\S+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_src and m_b):
        return None
    src = os.path.join(ROOT, m_src.group(1))
    if not os.path.exists(src) or source_sha(src) != m_sha.group(1):
        return None
    return float(m_b.group(1))


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def llama_batch():
    from ragged_paged_attention_gb300 import workloads
    return workloads.llama_mixed()


def cpu_sample(run, total, seconds, n_cal=4, seed=0):
    """Times ``run(ids)`` -- the oracle on a subset of the ``total`` units (query tokens) of a
    workload: a calibration call on ``n_cal`` units, then one call on as many uniformly drawn
    units as fit in about ``seconds``.  Returns (units, seconds taken)."""
    rng = np.random.default_rng(seed)
    n_cal = min(n_cal, total)
    t0 = time.perf_counter()
    run(np.sort(rng.choice(total, n_cal, replace=False)))
    cal = time.perf_counter() - t0
    n = int(max(n_cal, min(total, n_cal * seconds / max(cal, 1e-3))))
    ids = np.sort(rng.choice(total, n, replace=False))
    t0 = time.perf_counter()
    run(ids)
    return n, time.perf_counter() - t0


def cpu_record(n, total, dt, what):
    return {"value": n / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} of {total} query tokens drawn uniformly from {what}, all heads, float64 C oracle "
                      f"with OpenMP, {dt:.1f} s"}


def cpu_baseline_rpa(b, seconds, seed=0, what="the Llama-3-8B mixed batch"):
    """The float64 oracle on a random sample of the batch's query tokens."""
    import oracle
    oracle.build()
    T = b.num_tokens
    n, dt = cpu_sample(lambda ids: oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens,
                                              len(b.q_lens), tokens=ids, **b.options()), T, seconds, 8, seed)
    return cpu_record(n, T, dt, what)


def cpu_baseline_mla(m, seconds, seed=0):
    """The oracle's update_kv_cache and attention on a random sample of the MLA batch's tokens."""
    import oracle
    oracle.build()
    T = m.num_tokens
    n, dt = cpu_sample(lambda ids: oracle.mla_forward(m.ql_nope, m.q_pe, m.new_kv_c, m.new_k_pe, m.cache_kv_c,
                                                      m.cache_k_pe, m.kv_lens, m.page_indices, m.cu_q_lens,
                                                      m.distribution, tokens=ids, **m.options()),
                       T, seconds, 4, seed)
    return cpu_record(n, T, dt, "the DeepSeek-V3 MLA batch (cache update included)")


def cpu_baseline_sparse(s, seconds, what, seed=0):
    """The oracle on a random sample of the sparse batch's queries."""
    import oracle
    oracle.build()
    B, S = s.q.shape[:2]
    n, dt = cpu_sample(lambda ids: oracle.sparse_mla(s.q, s.cache, s.indices, s.positions, s.page_table,
                                                     queries=ids, **s.options()), B * S, seconds, 2, seed)
    return cpu_record(n, B * S, dt, what)


def cpu_baseline_sparse_ragged(s, seconds, what, seed=0):
    """The oracle's self-write and attention on a random sample of the packed batch's tokens."""
    import oracle
    oracle.build()
    T = s.ql.shape[0]
    cache = oracle.sparse_ragged_write(s.kvc, s.kpe, s.cache, s.loc, page_size=s.page_size)
    n, dt = cpu_sample(lambda ids: oracle.sparse_mla_ragged(s.ql, s.qpe, cache, s.topk, s.positions, s.seq_lens,
                                                            s.cu_q_lens, s.cu_kv_lens, s.page_indices, queries=ids,
                                                            **s.options()), T, seconds, 2, seed)
    return cpu_record(n, T, dt, what)


def run_reference(args, world, rank):
    """Reference arm: the oracle on the host cores, timed per step on a bounded sample."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    b = llama_batch()
    rng = np.random.default_rng(1)
    T = b.num_tokens
    per_step = max(4, int(64 * 8 / max(args.steps + args.warmup, 1)))
    times, toks_done = [], 0
    for i in range(args.warmup + args.steps):
        toks = np.sort(rng.choice(T, per_step, replace=False))
        t0 = time.perf_counter()
        oracle.rpa(b.q, b.kv_pages, b.kv_lens, b.page_indices, b.cu_q_lens, len(b.q_lens), tokens=toks, **b.options())
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            toks_done += per_step
    value = toks_done / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "llama3_8b_mixed_batch", "sample_tokens_per_step": per_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{per_step} random query tokens of {T} per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    from ragged_paged_attention_gb300 import api
    from ragged_paged_attention_gb300 import build as rpa_build
    rpa_build.build()
    api.load_library()
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda", torch.cuda.current_device())
    cpu_ok = rank == 0 and world == 1 and not args.no_cpu_baseline
    if args.workload != "llama_mixed":
        res = run_variants(dev, peaks, args, world, only=args.workload,
                           cpu_secs=args.cpu_seconds / 3 if cpu_ok else 0.0)
        if rank == 0:
            v = res[args.workload]
            print(json.dumps({"metric": METRIC, "value": v["tokens_per_s"] * world, "unit": "tokens/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": v["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                              "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                              "config": {"workload": args.workload}, "detail": v}), flush=True)
        return

    b = llama_batch()
    acc = rpa_accounting(b)
    g = b.to(dev)
    opts = b.options()
    prm = api.make_rpa_params(g.q, g.kv_pages, g.page_indices, **opts)
    ws = torch.zeros(api.rpa_workspace_size(prm), dtype=torch.uint8, device=dev)
    out = torch.empty_like(g.q)

    def step():
        # the batch's new K/V rows into the cache, then attention: one call (rpa_forward_update)
        api.rpa_forward_update(g.q, g.new_k, g.new_v, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens,
                               g.num_seqs, out=out, workspace=ws, **opts)

    clocks = clock_sampler(local).start()
    ms, _, n_launch = time_steps(step, args.steps, args.warmup, world, launches=True)
    clk = clocks.stop()
    # per-kernel durations: a second pass with every launch bracketed by CUDA events (the
    # library runs its kernels one after another while they are timed)
    _, ktimes = time_steps(step, args.steps, 1, world, timer=True)
    assert api.check_device_status(ws) == 0
    ms = max_over_ranks(ms, world)
    T = b.num_tokens
    value = T * world / (ms * 1e-3)

    # dominant kernel of the step and its roofline
    step_total = sum(v[1] for v in ktimes.values())
    dom = max(ktimes.items(), key=lambda kv: kv[1][1])[0] if ktimes else None
    kernels = {k: {"launches": v[0], "avg_us": 1e3 * v[1] / max(v[0], 1),
                   "share": v[1] / step_total if step_total else None} for k, v in ktimes.items()}
    dec_bytes = acc["decode"][1]
    pre_flops = acc["prefill"][2]
    if dom == "rpa_prefill_attn":
        avg_s = ktimes[dom][1] / ktimes[dom][0] * 1e-3
        ach = pre_flops / avg_s / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / peaks["bf16_tflops"], "traffic": profiled_traffic(dom, "llama_mixed")}
    else:
        dom = "rpa_decode_attn"
        avg_s = ktimes[dom][1] / ktimes[dom][0] * 1e-3
        ach = dec_bytes / avg_s / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": profiled_traffic(dom, "llama_mixed")}
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["algorithmic_bytes_per_launch" if roof["bound"] == "hbm" else "algorithmic_flops_per_launch"] = (
        dec_bytes if roof["bound"] == "hbm" else pre_flops)
    step_bytes = acc["decode"][1] + acc["prefill"][1]
    step_flops = acc["decode"][2] + acc["prefill"][2]
    t_roof = roof_time(step_bytes, step_flops, peaks)
    # the step's other attention kernel against its own bound, from the same per-kernel pass
    other_roofs = {}
    if dom != "rpa_prefill_attn" and ktimes.get("rpa_prefill_attn") and pre_flops > 0:
        s_pre = ktimes["rpa_prefill_attn"][1] / ktimes["rpa_prefill_attn"][0] * 1e-3
        a_pre = pre_flops / s_pre / 1e12
        other_roofs["rpa_prefill_attn"] = {"bound": "tensor", "achieved": a_pre, "peak": peaks["bf16_tflops"],
                                           "unit": "TFLOP/s", "frac": a_pre / peaks["bf16_tflops"],
                                           "algorithmic_flops_per_launch": pre_flops}

    # end to end: pinned host inputs -> device, update + attention, output -> host, every
    # step. Served the way a serving loop would: inputs and outputs double-buffered on the
    # device, the host-to-device copies on one copy stream and the device-to-host copy on
    # another, so step i+1's inputs and step i-1's output move while step i computes.
    host = {k: v.pin_memory() for k, v in
            dict(q=b.q, new_k=b.new_k, new_v=b.new_v, kv_lens=b.kv_lens, page_indices=b.page_indices,
                 cu_q_lens=b.cu_q_lens, num_seqs=b.num_seqs).items()}
    dq = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    outs_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {n: [torch.cuda.Event() for _ in range(2)] for n in ("in_free", "in_ready", "out_ready", "out_free")}

    def e2e_step(i):
        k = i % 2
        s_in.wait_event(ev["in_free"][k])  # step i-2 is done with these device inputs
        with torch.cuda.stream(s_in):
            for name, v in host.items():
                dq[k][name].copy_(v, non_blocking=True)
        ev["in_ready"][k].record(s_in)
        comp.wait_event(ev["in_ready"][k])
        comp.wait_event(ev["out_free"][k])  # step i-2's output has reached the host
        d = dq[k]
        api.rpa_forward_update(d["q"], d["new_k"], d["new_v"], g.kv_pages, d["kv_lens"], d["page_indices"],
                               d["cu_q_lens"], d["num_seqs"], out=outs[k], workspace=ws, **opts)
        ev["in_free"][k].record(comp)
        ev["out_ready"][k].record(comp)
        s_out.wait_event(ev["out_ready"][k])
        with torch.cuda.stream(s_out):
            outs_h[k].copy_(outs[k], non_blocking=True)
        ev["out_free"][k].record(s_out)

    def time_e2e(steps, warmup):
        for i in range(warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        for i in range(warmup, warmup + steps):
            e2e_step(i)
        comp.wait_event(ev["out_free"][(warmup + steps - 1) % 2])  # the last output is on the host
        e1.record(comp)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / steps

    ms_e2e = None
    if not args.no_e2e:
        ms_e2e = max_over_ranks(time_e2e(args.steps, args.warmup), world)
        # the host copy of the last output is the device result of the same inputs (one more
        # resident step in the same launch mode: the decode shares depend on the SM split)
        step()
        torch.cuda.synchronize()
        assert torch.equal(outs_h[(args.warmup + args.steps - 1) % 2][:b.num_tokens].to(dev), out[:b.num_tokens])

    # same-run variants (decode/prefill sub-launches are in `kernels`)
    variants = {}
    if not args.no_variants:
        variants = run_variants(dev, peaks, args, world, cpu_secs=args.cpu_seconds / 3 if cpu_ok else 0.0)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_rpa(b, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "llama3_8b_mixed_batch", "num_q_heads": 32, "num_kv_heads": 8, "head_dim": 128,
                       "page_size": 16, "decode_seqs": 128, "prefill_chunks": "4 x 512", "query_tokens": T,
                       "kv_cache_bytes": g.kv_pages.numel() * g.kv_pages.element_size(),
                       "step": "rpa_forward_update (cache write of the new K/V rows + attention)",
                       "l2": "inputs larger than L2 (KV cache >1 GB read each step)", "parallelism": "replicas"},
            "step_roofline": {"bytes": step_bytes, "flops": step_flops, "roofline_us": t_roof * 1e6,
                              "frac": t_roof / (ms * 1e-3), "hbm_gbs": step_bytes / (ms * 1e-3) / 1e9,
                              "tflops": step_flops / (ms * 1e-3) / 1e12},
            "roofline": roof,
            "kernel_rooflines": other_roofs,
            "kernels": kernels,
            "gpu_launches": int(n_launch),
            "kernel_timing": "kernels/roofline: separate pass of the same steps with each launch bracketed by "
                             "CUDA events (kernels serialised); value/ms_per_step: unbracketed steps",
            "clocks": clk,
            "e2e": None if ms_e2e is None else {
                "value": T * world / (ms_e2e * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "copies": "pinned host buffers; inputs and outputs double-buffered on the device, "
                          "host-to-device and device-to-host copies on their own streams beside the compute"},
            "cpu_baseline": cpu,
            "variants": variants,
        }
        print(json.dumps(line), flush=True)


def run_variants(dev, peaks, args, world, only=None, cpu_secs=0.0):
    """The other workloads, each measured on its own; with cpu_secs > 0 each also carries the
    oracle timed on a bounded sample of it (about cpu_secs of host time)."""
    from ragged_paged_attention_gb300 import api, workloads
    res = {}
    steps, warm = (max(3, args.steps // 2), 3) if only is None else (args.steps, args.warmup)

    def want(name):
        return only is None or only == name

    def report(name, tok, byt, fl, ms, kt, extra=None):
        t_roof = roof_time(byt, fl, peaks)
        r = {"tokens_per_s": tok / (ms * 1e-3), "ms_per_step": ms, "hbm_gbs": byt / (ms * 1e-3) / 1e9,
             "tflops": fl / (ms * 1e-3) / 1e12, "roofline_frac": t_roof / (ms * 1e-3),
             "bound": "hbm" if byt / (peaks["hbm_gbs"] * 1e9) >= fl / (peaks["bf16_tflops"] * 1e12) else "tensor",
             "kernels_us": {k: 1e3 * v[1] / max(v[0], 1) for k, v in kt.items()}}
        if extra:
            r.update(extra)
        res[name] = r

    # Gemma-2-style fp8 KV, sliding window, soft cap
    if want("gemma2_fp8_sw_cap"):
        _variant_gemma(dev, peaks, api, workloads, steps, warm, world, report, cpu_secs)
    if want("mla_deepseek_v3"):
        _variant_mla(dev, peaks, api, workloads, steps, warm, world, report, cpu_secs)
    for phase in ("prefill", "decode"):
        for mode in ("token", "page"):
            if want(f"dsa_sparse_{phase}_{mode}"):
                _variant_sparse(dev, api, workloads, phase, mode, steps, warm, world, report, cpu_secs)
    for mode in ("token", "page"):
        if want(f"dsa_sparse_ragged_{mode}"):
            _variant_sparse_ragged(dev, api, workloads, mode, steps, warm, world, report, cpu_secs)
    return res


def _variant_gemma(dev, peaks, api, workloads, steps, warm, world, report, cpu_secs=0.0):
    b = workloads.gemma_options()
    acc = rpa_accounting(b)
    g = b.to(dev)
    opts = b.options()
    ws = torch.zeros(api.rpa_workspace_size(api.make_rpa_params(g.q, g.kv_pages, g.page_indices, **opts)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(g.q)
    def fwd():
        api.rpa_forward(g.q, g.kv_pages, g.kv_lens, g.page_indices, g.cu_q_lens, g.num_seqs, out=out, workspace=ws,
                        **opts)

    ms, _ = time_steps(fwd, steps, warm, world)
    _, kt = time_steps(fwd, steps, 1, world, timer=True)  # per-kernel pass (serialised)
    dec_us = 1e3 * kt["rpa_decode_attn"][1] / kt["rpa_decode_attn"][0]
    extra = {"decode_hbm_frac": acc["decode"][1] / (dec_us * 1e-6) / 1e9 / peaks["hbm_gbs"]}
    if kt.get("rpa_prefill_attn"):
        pre_us = 1e3 * kt["rpa_prefill_attn"][1] / kt["rpa_prefill_attn"][0]
        extra["prefill_tensor_frac"] = acc["prefill"][2] / (pre_us * 1e-6) / 1e12 / peaks["bf16_tflops"]
    if cpu_secs > 0:
        extra["cpu_baseline"] = cpu_baseline_rpa(b, cpu_secs, what="the Gemma-2-style fp8 batch")
    report("gemma2_fp8_sw_cap", b.num_tokens, acc["decode"][1] + acc["prefill"][1],
           acc["decode"][2] + acc["prefill"][2], ms, kt, extra)
    del b, g, out, ws
    torch.cuda.empty_cache()


def _mla_call(api, g, out, ws, opts):
    return lambda: api.mla_rpa_forward(g.ql_nope, g.q_pe, g.new_kv_c, g.new_k_pe, g.cache_kv_c, g.cache_k_pe,
                                       g.kv_lens, g.page_indices, g.cu_q_lens, g.distribution, out=out, workspace=ws,
                                       **opts)


def _variant_mla(dev, peaks, api, workloads, steps, warm, world, report, cpu_secs=0.0):
    m = workloads.mla_deepseek()
    tok, byt, fl, dec = mla_accounting(m)
    g = m.to(dev)
    opts = m.options()
    prm = api.make_mla_params(g.ql_nope, g.q_pe, g.cache_kv_c, g.cache_k_pe, g.kv_lens, g.page_indices, **opts)
    ws = torch.zeros(api.mla_workspace_size(prm), dtype=torch.uint8, device=dev)
    out = torch.empty_like(g.ql_nope)
    ms, kt = time_steps(_mla_call(api, g, out, ws, opts), steps, warm, world, timer=True)
    att_us = 1e3 * kt["mla_attn"][1] / kt["mla_attn"][0]
    extra = {"attn_tensor_frac": fl / (att_us * 1e-6) / 1e12 / peaks["bf16_tflops"]}
    # the decode-only and prefill-only sub-launches: the batch's own sequence lengths, each
    # class on its own (decode sits near the ridge, prefill is tensor-bound)
    nd = sum(1 for x in m.q_lens if x == 1)
    for name, ql, kl in (("decode_sub", m.q_lens[:nd], m.kv_lens_list[:nd]),
                         ("prefill_sub", m.q_lens[nd:], m.kv_lens_list[nd:])):
        sub = workloads.make_mla(ql, kl, seed=2003 + len(ql), num_decode=nd if name == "decode_sub" else 0,
                                 pages_per_seq=m.page_indices.numel() // len(m.q_lens))
        s_tok, s_byt, s_fl, _ = mla_accounting(sub)
        gs = sub.to(dev)
        prm_s = api.make_mla_params(gs.ql_nope, gs.q_pe, gs.cache_kv_c, gs.cache_k_pe, gs.kv_lens, gs.page_indices,
                                    **opts)
        ws_s = torch.zeros(api.mla_workspace_size(prm_s), dtype=torch.uint8, device=dev)
        out_s = torch.empty_like(gs.ql_nope)
        _, kt_s = time_steps(_mla_call(api, gs, out_s, ws_s, opts), steps, warm, world, timer=True)
        us = 1e3 * kt_s["mla_attn"][1] / kt_s["mla_attn"][0]
        t_roof = roof_time(s_byt, s_fl, peaks)
        extra[name] = {"tokens": s_tok, "attn_us": us, "bytes": s_byt, "flops": s_fl,
                       "hbm_gbs": s_byt / (us * 1e-6) / 1e9, "tflops": s_fl / (us * 1e-6) / 1e12,
                       "bound": "hbm" if s_byt / (peaks["hbm_gbs"] * 1e9) >= s_fl / (peaks["bf16_tflops"] * 1e12)
                       else "tensor", "roofline_frac": t_roof / (us * 1e-6),
                       "tensor_frac": s_fl / (us * 1e-6) / 1e12 / peaks["bf16_tflops"]}
        del sub, gs, ws_s, out_s
    if cpu_secs > 0:
        extra["cpu_baseline"] = cpu_baseline_mla(m, cpu_secs)
    report("mla_deepseek_v3", tok, byt, fl, ms, kt, extra)
    del m, g, out, ws
    torch.cuda.empty_cache()


def _variant_sparse_ragged(dev, api, workloads, mode, steps, warm, world, report, cpu_secs=0.0):
    s = workloads.dsa_sparse_ragged(mode=mode)
    tok, byt, fl = sparse_ragged_accounting(s)
    g = s.to(dev)
    prm = api.make_sparse_ragged_params(g.ql, g.qpe, g.cache, g.topk, g.seq_lens, g.page_indices, **s.options())
    ws = torch.zeros(api.sparse_mla_ragged_workspace_size(prm), dtype=torch.uint8, device=dev)
    out = torch.empty(s.ql.shape[:2] + (512,), dtype=torch.float32, device=dev)

    def call():
        api.sparse_mla_write_and_attend_ragged(g.ql, g.qpe, g.kvc, g.kpe, g.cache, g.topk, g.positions, g.loc,
                                               g.seq_lens, g.cu_q_lens, g.cu_kv_lens, g.page_indices, out=out,
                                               workspace=ws, **s.options())

    ms, kt = time_steps(call, max(3, steps // 2), warm, world, timer=True)
    extra = None
    if cpu_secs > 0:
        extra = {"cpu_baseline": cpu_baseline_sparse_ragged(
            s, cpu_secs, f"the packed-ragged DSA batch ({mode}-level selection, self-write included)")}
    report(f"dsa_sparse_ragged_{mode}", tok, byt, fl, ms, kt, extra)
    del s, g, out, ws
    torch.cuda.empty_cache()


def _variant_sparse(dev, api, workloads, phase, mode, steps, warm, world, report, cpu_secs=0.0):
    s = workloads.dsa_sparse(mode=mode, phase=phase)
    tok, byt, fl = sparse_accounting(s)
    g = s.to(dev)
    prm = api.make_sparse_params(g.q, g.cache, g.indices, g.page_table, read_block=s.read_block,
                                 page_size=s.page_size, seq_len=s.seq_len, sm_scale=s.sm_scale)
    ws = torch.zeros(api.sparse_mla_workspace_size(prm), dtype=torch.uint8, device=dev)
    out = torch.empty(s.q.shape[:3] + (512,), dtype=torch.float32, device=dev)
    ms, kt = time_steps(lambda: api.sparse_mla_forward(g.q, g.cache, g.indices, g.positions, g.page_table,
                                                       out=out, workspace=ws, **s.options()),
                        steps if phase == "decode" else max(3, steps // 4), warm, world, timer=True)
    extra = None
    if cpu_secs > 0:
        extra = {"cpu_baseline": cpu_baseline_sparse(s, cpu_secs, f"the DSA {phase} batch ({mode}-level selection)")}
    report(f"dsa_sparse_{phase}_{mode}", tok, byt, fl, ms, kt, extra)
    del s, g, out, ws
    torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
