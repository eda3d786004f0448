"""Benchmark of the fused SDPA forward on one or more GB300s.

One step is one pass of the whole hot path over one batch of synthetic input:
  1. a causal GQA prefill through a paged cache -- workload
     prefill_causal_bf16_gqa_s2048: bf16, B=1, Hq=32, Hkv=8 (GQA 4:1),
     Sq=Sk=2048, d=128, block size 64 with a randomly permuted block table;
  2. one split-KV decode step -- workload decode_bf16_b64_paged16: bf16,
     B=64, Hq=32, Hkv=8, d=128, kv lengths uniform in [512, 8192], block
     size 16, shared permuted pool, 8 splits + log-sum-exp combine.
Inputs are seeded synthetic N(0,1) tensors already resident in HBM when the
timed region starts.  L2 is flushed before every step (a 256 MiB write).

Reported (one JSON line on rank 0):
  value        prefill attention TFLOP/s (unmasked FLOPs, 4*d per visible
               (query, key) pair per query head) from CUDA events around the
               prefill launches, summed over all ranks;
  decode       decode KV GB/s (K+V bytes read + Q + O) from CUDA events around
               the decode call (split kernel + combine kernel);
  roofline     for the kernel with the larger share of device time: achieved
               vs the measured peak (HBM copy GB/s, or dense bf16 TFLOP/s);
  e2e          the same metric with host buffers: per step the host->device
               copy of the step's inputs from pinned memory, the calls, and
               the device->host copy of the outputs, all timed;
  configs      every configuration on its own (C1 fp16 S=128 d=64, C2, C3,
               C4a causal S=8192, C4b chunked B=4 Sq=512 Sk=8192, C5 dense
               non-causal BSHD B=4 H=16 S=16384 in each rounding mode RTNE,
               RTNA, RTZ): device time per call, throughput and fractions of
               the measured peaks, clocks sampled over them;
  cpu_baseline the fp64 CPU oracle on a bounded row sample of the same
               workloads (rank 0, single-GPU runs only).
`--impl reference` times the oracle instead (the reference arm).
`--sweep` times every named workload on its own instead (one JSON line each:
one call per timed iteration, L2 flushed before each, median of CUDA-event
times, clocks sampled meanwhile, plus a "protocol" object with the pages' own
protocol: 10 measurements of 50 back-to-back calls, trimmed mean, median,
noise flag; fractions of the measured peak and of NVIDIA's nominal peak);
these lines are not the benchmark line.
Multi-GPU: every rank runs its own copy of the workload (independent
problems, no collective on the data path); value is the sum over ranks of the
work divided by the slowest rank's time (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import attn_inputs  # noqa: E402

METRIC = "prefill attn TFLOP/s & decode KV GB/s on 1 GB300; % of tensor/HBM roofline"
PREFILL_WL = "prefill_causal_bf16_gqa_s2048"
DECODE_WL = "decode_bf16_b64_paged16"
DECODE_SPLITS = 8
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's nominal dense figures for one GB300 (the second denominator)
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}
CSRC = os.path.join(ROOT, "attention_forward_sdpa_gb300", "csrc")
# DRAM bytes (read + write) per launch from one ncu capture of the bench
# workload, valid only while the kernel's code has the recorded hash (sha256
# prefix of the source with comments and white space removed, so that an
# edit of comments alone keeps it; the ncu summaries under profiles/ record
# each capture).
MEASURED_TRAFFIC = {
    "prefill": ("prefill_tcgen05.cu", "8f6cfb695f3291b9", 25.273088e6 + 1536.0),
    "decode": ("decode_tcgen05.cu", "58e05c9cf0c323d8", 1.130844e9 + 8.962560e6),
}


# ----------------------------------------------------------------------------
# algorithmic work
# ----------------------------------------------------------------------------

def visible_pairs(q_lens, kv_lens, causal: bool, window=(-1, -1)) -> int:
    """(query row, key) pairs left visible by the mask, per query head;
    bottom-right causal alignment: row i of a sequence sees j <= i + Sk - Sq,
    a sliding window (left, right) keeps diag - left <= j <= diag + right."""
    tot = 0
    for sq, sk in zip(q_lens, kv_lens):
        diag = np.arange(sq, dtype=np.int64) + (sk - sq)
        hi = np.full(sq, sk, dtype=np.int64)                 # exclusive upper bound
        if causal:
            hi = np.minimum(hi, diag + 1)
        if window[1] >= 0:
            hi = np.minimum(hi, diag + window[1] + 1)
        lo = np.zeros(sq, dtype=np.int64)
        if window[0] >= 0:
            lo = np.maximum(lo, diag - window[0])
        tot += int(np.clip(hi - lo, 0, None).sum())
    return tot


def prefill_flops(prob, window=(-1, -1)) -> float:
    return 4.0 * prob.head_size * prob.num_q_heads * visible_pairs(prob.q_lens, prob.kv_lens,
                                                                   prob.causal, window)


# Feature-flagged sweep workloads: (base workload, flags).  The per-head
# arrays are built on the device from these recipes.
FEATURE_WORKLOADS = {
    "prefill_causal_bf16_s8192_window1024": ("prefill_causal_bf16_s8192", {"window": (1024, -1)}),
    "prefill_causal_bf16_s8192_softcap": ("prefill_causal_bf16_s8192", {"softcap": 30.0}),
    "prefill_causal_bf16_s8192_alibi_sinks": ("prefill_causal_bf16_s8192",
                                              {"alibi": True, "sinks": True}),
    "decode_bf16_b64_paged16_window1024": ("decode_bf16_b64_paged16", {"window": (1024, -1)}),
    "decode_bf16_b64_paged16_softcap_alibi_sinks": ("decode_bf16_b64_paged16",
                                                    {"softcap": 30.0, "alibi": True,
                                                     "sinks": True}),
    # fp8 E4M3 caches (per-tensor factors): the same draws, stored as codes
    "decode_bf16_b64_paged16_fp8kv": ("decode_bf16_b64_paged16", {"kv_fp8": True}),
    "prefill_chunked_bf16_b4_fp8kv": ("prefill_chunked_bf16_b4", {"kv_fp8": True}),
    "prefill_causal_bf16_gqa_s2048_fp8kv": ("prefill_causal_bf16_gqa_s2048", {"kv_fp8": True}),
}


def feature_args(recipe: dict, num_q_heads: int, dev, prob=None) -> dict:
    out = {}
    if recipe.get("kv_fp8"):
        out["kv_scales"] = (prob.k_scale, prob.v_scale)
    if "window" in recipe:
        out["window"] = recipe["window"]
    if "softcap" in recipe:
        out["softcap"] = recipe["softcap"]
    if recipe.get("alibi"):
        out["alibi_slopes"] = torch.tensor([2.0 ** (-8.0 * (h + 1) / num_q_heads)
                                            for h in range(num_q_heads)],
                                           dtype=torch.float32, device=dev)
    if recipe.get("sinks"):
        out["sinks"] = torch.zeros(num_q_heads, dtype=torch.float32, device=dev)
    return out


def decode_bytes(prob, window=(-1, -1)) -> float:
    """K + V bytes of the visible keys (a left window keeps the last
    left + 1 keys of each sequence; fp8 caches hold one byte per element)
    plus Q and O."""
    el = 2
    kv_el = 1 if getattr(prob, "kv_fp8", False) else 2
    keys = [min(k, window[0] + 1) if window[0] >= 0 else k for k in prob.kv_lens]
    kv = 2.0 * sum(keys) * prob.num_kv_heads * prob.head_size * kv_el
    qo = 2.0 * prob.num_seqs * prob.num_q_heads * prob.head_size * el
    return kv + qo


def code_hash(text: str) -> str:
    """sha256 of C/CUDA source with comments and white space removed."""
    import hashlib
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    text = re.sub(r"\s+", "", text)
    return hashlib.sha256(text.encode()).hexdigest()


def measured_traffic(kind):
    fname, digest, nbytes = MEASURED_TRAFFIC[kind]
    try:
        with open(os.path.join(CSRC, fname)) as f:
            cur = code_hash(f.read())
    except OSError:
        return None
    return nbytes if cur.startswith(digest) else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    @staticmethod
    def _parse(line):
        parts = [x.strip() for x in line.split(",")]
        try:
            return (float(parts[0]), float(parts[1]), parts[3:])
        except Exception:
            return None

    def parsed(self, t0: float, t1: float):
        """The samples taken between wall times t0 and t1, parsed."""
        inside = [self._parse(l) for t, l in self.samples if t0 <= t <= t1]
        return [x for x in inside if x]

    def summary(self, t0: float, t1: float):
        inside = self.parsed(t0, t1)
        window = "timed"
        if not inside:
            inside = [x for x in (self._parse(l) for _, l in self.samples) if x]
            window = "whole run"
        return clock_summary(inside, window)


def clock_summary(inside, window):
    """Median SM clock, the highest maximum seen and every throttle reason
    active in any of the parsed samples."""
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = set()
    for _, _, flags in inside:
        for n, v in zip(names, flags[1:5]):
            if v.lower().startswith("active"):
                reasons.add(n)
    return {"sm_mhz": statistics.median(x[0] for x in inside),
            "sm_max_mhz": max(x[1] for x in inside), "reasons": sorted(reasons),
            "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------
# the library arm
# ----------------------------------------------------------------------------

def bench_config(world: int) -> dict:
    """The workload description both arms report."""
    return {"workload": f"{PREFILL_WL} + {DECODE_WL}",
            "prefill": "causal bf16 B=1 Hq=32 Hkv=8 Sq=Sk=2048 d=128 paged bs=64 permuted",
            "decode": "bf16 B=64 Hq=32 Hkv=8 d=128 Sk~U[512,8192] paged bs=16 splits=8",
            "l2": "flushed before every step (256 MiB write)",
            "parallelism": f"replica x{world}" if world > 1 else "single GPU"}


def make_problems(seed: int):
    return attn_inputs.workload(PREFILL_WL, seed=seed), attn_inputs.workload(DECODE_WL, seed=seed)


def device_args(prob, dev):
    return {k: getattr(prob, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_table",
                                                  "query_start_loc", "seq_lens")}


def run_ours(args, rank, world, dev):
    import attention_forward_sdpa_gb300 as attn

    attn.load_library()
    pp, dp = make_problems(seed=rank)
    pt, dt = device_args(pp, dev), device_args(dp, dev)
    p_out = torch.empty_like(pt["q"])
    d_out = torch.empty_like(dt["q"])
    ws_n = attn.attn_decode_workspace_size(dp.num_seqs, dp.num_q_heads, dp.head_size, DECODE_SPLITS)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def do_prefill(t, out):
        attn.attn_fwd_prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                              t["query_start_loc"], t["seq_lens"], max_seqlen_q=pp.max_seqlen_q,
                              max_seqlen_k=pp.max_seqlen_k, scale=pp.scale, causal=True,
                              stream=stream)

    def do_decode(t, out):
        attn.attn_fwd_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                             t["seq_lens"], max_seqlen_k=dp.max_seqlen_k, scale=dp.scale,
                             num_splits=DECODE_SPLITS, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        do_prefill(pt, p_out)
        do_decode(dt, d_out)
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    ev_all = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    host_gate(stream, K)
    ev_all[0].record(stream)
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        do_prefill(pt, p_out)
        ev[k][1].record(stream)
        do_decode(dt, d_out)
        ev[k][2].record(stream)
    ev_all[1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    sampler.stop()

    p_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    d_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    step_ms = ev_all[0].elapsed_time(ev_all[1]) / K
    p_ms_tot, d_ms_tot = sum(p_ms), sum(d_ms)
    # slowest rank decides
    p_ms_tot, d_ms_tot, step_ms = max_over_ranks(world, dev, [p_ms_tot, d_ms_tot, step_ms])

    flops = prefill_flops(pp)
    dbytes = decode_bytes(dp)
    # whole-job work: every rank's own problem (decode lengths differ by seed)
    flops_all, dbytes_all = sum_over_ranks(world, dev, [flops, dbytes])
    tflops = flops_all * K / (p_ms_tot * 1e-3) / 1e12
    gbs = dbytes_all * K / (d_ms_tot * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    p_avg_s = p_ms_tot / K * 1e-3
    d_avg_s = d_ms_tot / K * 1e-3
    roof_p = {"kernel": "prefill_kernel<128,bf16>", "bound": "tensor",
              "achieved": flops / p_avg_s / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
              "frac": flops / p_avg_s / 1e12 / peaks["bf16_tflops"],
              "traffic": measured_traffic("prefill"),
              "peak_source": f"{peak_src} bf16 burst", "avg_launch_us": p_avg_s * 1e6,
              "algorithmic_per_launch": flops}
    roof_d = {"kernel": "decode_tc_kernel<bf16,4> + decode_combine_kernel", "bound": "hbm",
              "achieved": dbytes / d_avg_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
              "frac": dbytes / d_avg_s / 1e9 / peaks["hbm_gbs"],
              "traffic": measured_traffic("decode"),
              "peak_source": f"{peak_src} HBM copy", "avg_launch_us": d_avg_s * 1e6,
              "algorithmic_per_launch": dbytes}
    dominant, other = (roof_d, roof_p) if d_ms_tot >= p_ms_tot else (roof_p, roof_d)
    clocks = sampler.summary(t_wall0, t_wall1)
    step_samples = sampler.parsed(t_wall0, t_wall1)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, pp, dp, dev, stream, attn, ws, world)

    graph = None
    if not args.no_graph:
        try:
            graph = measure_graph(pp, dp, pt, dt, p_out, d_out, ws, flush, attn, dev)
        except Exception as exc:  # reported, never fatal: the eager numbers stand
            graph = {"error": f"{type(exc).__name__}: {exc}"[:200]}

    configs = None
    if not args.no_configs:
        configs = measure_configs(args, dev, attn, flush, peaks, peak_src)
        # The step's timed region lasts a few ms, shorter than the sampling
        # period, so the clocks reported for the run pool its samples with
        # those of the configuration set's timed calls (same process, same
        # kernels, right after it).
        cfg_samples = configs.pop("_clock_samples", [])
        if cfg_samples:
            clocks = clock_summary(step_samples + cfg_samples,
                                   f"timed: the step ({len(step_samples)} samples) and the "
                                   f"configuration set ({len(cfg_samples)} samples)")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(pp, dp, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world),
        "decode": {"value": gbs, "unit": "GB/s", "frac_of_hbm": gbs / world / peaks["hbm_gbs"],
                   "bytes_per_step": dbytes, "ms_per_call": d_avg_s * 1e3},
        "prefill": {"value": tflops, "unit": "TFLOP/s",
                    "frac_of_bf16": tflops / world / peaks["bf16_tflops"],
                    "flops_per_step": flops, "ms_per_call": p_avg_s * 1e3},
        "roofline": dominant, "roofline_other": other,
        "gpu_launches": K * 3,
        "clocks": clocks,
        "e2e": e2e,
        "graph": graph,
        "configs": configs,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# Every configuration of the workload set, timed in the default run next to
# the step: (label, workload, rounding mode).  The dense 16384 workload is
# timed in each output rounding mode.
CONFIG_SET = (
    ("C1", "prefill_causal_fp16_s128_d64", 0),
    ("C2", PREFILL_WL, 0),
    ("C3", DECODE_WL, 0),
    ("C4a", "prefill_causal_bf16_s8192", 0),
    ("C4b", "prefill_chunked_bf16_b4", 0),
    ("C5_rtne", "dense_bf16_bshd_s16384", 0),
    ("C5_rtna", "dense_bf16_bshd_s16384", 1),
    ("C5_rtz", "dense_bf16_bshd_s16384", 2),
)


# configurations also timed through the split (persistent, key-range-balanced) prefill
SPLIT_TIMED = ("C2", "C4a", "C4b", "C5_rtne")


def measure_configs(args, dev, attn, flush, peaks, peak_src):
    """Each configuration on its own: W warm-up calls, then K calls (the
    run's --steps, at most 20 for the dense 16384 workload), each after the
    256 MiB L2 flush, CUDA events around each call on the launching stream;
    mean and median device time, throughput and fractions of the measured
    peaks (burst, and sustained for the long runs), clocks sampled over the
    whole set.  The small fp16 case is launch-bound: its CUDA-graph replay
    time is reported too.  The causal, chunked and dense prefill workloads
    are also timed through attn_fwd_prefill_split (object "split")."""
    stream = torch.cuda.current_stream(dev)
    res = {}
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    launches = 0
    spans = []          # wall-time spans of the timed calls (clock samples are kept from these)
    probs = {}
    split_ws = torch.empty(attn.attn_prefill_split_workspace_size(128), dtype=torch.uint8,
                           device=dev)
    for label, name, rnd in CONFIG_SET:
        prob = probs.get(name)
        if prob is None:
            probs.clear()
            torch.cuda.empty_cache()
            prob = probs[name] = attn_inputs.workload(name)
        t = device_args(prob, dev)
        out = torch.empty_like(t["q"])
        is_decode = prob.max_seqlen_q == 1
        if is_decode:
            ws = torch.empty(attn.attn_decode_workspace_size(prob.num_seqs, prob.num_q_heads,
                                                             prob.head_size, DECODE_SPLITS),
                             dtype=torch.uint8, device=dev)

            def call(s=stream):
                attn.attn_fwd_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                     t["seq_lens"], max_seqlen_k=prob.max_seqlen_k,
                                     scale=prob.scale, num_splits=DECODE_SPLITS, workspace=ws,
                                     stream=s)
            per_call = 2
        else:
            def call(s=stream, split=False):
                attn.attn_fwd_prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                      t["query_start_loc"], t["seq_lens"],
                                      max_seqlen_q=prob.max_seqlen_q,
                                      max_seqlen_k=prob.max_seqlen_k, scale=prob.scale,
                                      causal=prob.causal, rounding=rnd, stream=s,
                                      split_workspace=split_ws if split else None)
            per_call = 1
        work_est = decode_bytes(prob) if is_decode else prefill_flops(prob)
        long_run = not is_decode and work_est > 1e11     # the 8192, chunked and dense workloads
        n = min(args.steps, 20) if work_est > 1e12 else args.steps
        for _ in range(args.warmup):
            flush.zero_()
            call()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        ta = time.time()
        host_gate(stream, n)
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        spans.append((ta, time.time()))
        launches += n * per_call
        us = [a.elapsed_time(b) * 1e3 for a, b in evs]
        mean_us, med_us = sum(us) / len(us), statistics.median(us)
        entry = {"workload": name, "rounding": ("RTNE", "RTNA", "RTZ")[rnd], "calls": n,
                 "mean_us": mean_us, "median_us": med_us}
        if is_decode:
            work = decode_bytes(prob)
            entry.update({"unit": "GB/s", "value": work / mean_us / 1e3,
                          "bytes_per_call": work,
                          "frac_of_hbm": work / mean_us / 1e3 / peaks["hbm_gbs"]})
        else:
            work = prefill_flops(prob)
            v = work / mean_us / 1e6
            entry.update({"unit": "TFLOP/s", "value": v, "flops_per_call": work,
                          "frac_of_bf16": v / peaks["bf16_tflops"]})
            if long_run:
                entry["frac_of_bf16_sustained"] = v / peaks["bf16_tflops_sustained"]
            if label in SPLIT_TIMED:
                # the same configuration through attn_fwd_prefill_split
                for _ in range(args.warmup):
                    flush.zero_()
                    call(split=True)
                torch.cuda.synchronize(dev)
                sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(n)]
                ta = time.time()
                host_gate(stream, n)
                for a, b in sev:
                    flush.zero_()
                    a.record(stream)
                    call(split=True)
                    b.record(stream)
                torch.cuda.synchronize(dev)
                spans.append((ta, time.time()))
                launches += n
                sus = [a.elapsed_time(b) * 1e3 for a, b in sev]
                smean = sum(sus) / len(sus)
                entry["split"] = {"entry_point": "attn_fwd_prefill_split", "mean_us": smean,
                                  "median_us": statistics.median(sus),
                                  "value": work / smean / 1e6,
                                  "frac_of_bf16": work / smean / 1e6 / peaks["bf16_tflops"]}
        if label == "C1":
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.graph(g, stream=cap):
                call(cap)
            torch.cuda.synchronize(dev)
            gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for a, b in gev:
                flush.zero_()
                a.record(stream)
                g.replay()
                b.record(stream)
            torch.cuda.synchronize(dev)
            launches += n
            entry["graph_median_us"] = statistics.median(a.elapsed_time(b) * 1e3 for a, b in gev)
            entry["note"] = "launch-bound (no roofline claim)"
            del g
        res[label] = entry
        del t, out
    t1 = time.time()
    sampler.stop()
    probs.clear()
    torch.cuda.empty_cache()
    res["peaks"] = {"bf16_tflops": peaks["bf16_tflops"],
                    "bf16_tflops_sustained": peaks["bf16_tflops_sustained"],
                    "hbm_gbs": peaks["hbm_gbs"], "source": peak_src}
    timed = [x for ta, tb in spans for x in sampler.parsed(ta, tb)]
    res["clocks"] = (clock_summary(timed, "timed calls") if timed else sampler.summary(t0, t1))
    res["_clock_samples"] = timed
    res["gpu_launches"] = launches
    res["l2"] = "flushed before every call (256 MiB write)"
    res["gpu"] = "this rank's GPU (rank 0 prints)"
    return res


def host_gate(stream, calls, host_ms_per_call=0.4):
    """Holds the stream in a device-side spin (torch.cuda._sleep) long enough
    for the host to enqueue `calls` timed calls behind it, so that no CUDA
    event span includes time the GPU spent waiting for the Python host to
    issue the next launch.  The spin runs before the first timed event."""
    cycles = int((calls * host_ms_per_call + 5.0) * 1e-3 * 2.1e9)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(cycles)


def measure_graph(pp, dp, pt, dt, p_out, d_out, ws, flush, attn, dev, n=50):
    """CUDA-graph replay of one call (kernel-only launch path): each call is
    captured once on a side stream and replayed with the 256 MiB L2 flush
    outside the graph; medians of n replays, CUDA events on the replay stream.
    Also the small causal fp16 S=128 d=64 case, whose time is launch cost."""
    c1 = attn_inputs.workload("prefill_causal_fp16_s128_d64")
    c1t = device_args(c1, dev)
    c1_out = torch.empty_like(c1t["q"])
    cap = torch.cuda.Stream(dev)

    def prefill(s):
        attn.attn_fwd_prefill(p_out, pt["q"], pt["k_cache"], pt["v_cache"], pt["block_table"],
                              pt["query_start_loc"], pt["seq_lens"], max_seqlen_q=pp.max_seqlen_q,
                              max_seqlen_k=pp.max_seqlen_k, scale=pp.scale, causal=True, stream=s)

    def decode(s):
        attn.attn_fwd_decode(d_out, dt["q"], dt["k_cache"], dt["v_cache"], dt["block_table"],
                             dt["seq_lens"], max_seqlen_k=dp.max_seqlen_k, scale=dp.scale,
                             num_splits=DECODE_SPLITS, workspace=ws, stream=s)

    def small(s):
        attn.attn_fwd_prefill(c1_out, c1t["q"], c1t["k_cache"], c1t["v_cache"], c1t["block_table"],
                              c1t["query_start_loc"], c1t["seq_lens"], max_seqlen_q=c1.max_seqlen_q,
                              max_seqlen_k=c1.max_seqlen_k, scale=c1.scale, causal=True, stream=s)

    cap.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(cap):
        for fn in (prefill, decode, small):   # first calls (one-time setup) outside any capture
            fn(cap)
    torch.cuda.synchronize(dev)
    graphs = {}
    for name, fn in (("prefill", prefill), ("decode", decode), ("small_prefill", small)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn(cap)
        graphs[name] = g
    torch.cuda.synchronize(dev)
    cur = torch.cuda.current_stream(dev)
    res = {}
    for name, g in graphs.items():
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for a, b in evs:
            flush.zero_()
            a.record(cur)
            g.replay()
            b.record(cur)
        torch.cuda.synchronize(dev)
        res[name] = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
    flops, dbytes = prefill_flops(pp), decode_bytes(dp)
    return {"prefill_us": res["prefill"], "prefill_tflops": flops / res["prefill"] / 1e6,
            "decode_us": res["decode"], "decode_gbs": dbytes / res["decode"] / 1e3,
            "small_prefill_us": res["small_prefill"],
            "small_prefill_workload": "prefill_causal_fp16_s128_d64",
            "note": "median of %d graph replays, L2 flushed before each (outside the graph)" % n}


def measure_e2e(args, pp, dp, dev, stream, attn, ws, world):
    """Host buffers through the public API: copy inputs in, run, copy outputs out."""
    host_p = {k: getattr(pp, k).pin_memory() for k in ("q", "k_cache", "v_cache", "block_table",
                                                       "query_start_loc", "seq_lens")}
    host_d = {k: getattr(dp, k).pin_memory() for k in ("q", "k_cache", "v_cache", "block_table",
                                                       "query_start_loc", "seq_lens")}
    dev_p = {k: torch.empty_like(v, device=dev) for k, v in host_p.items()}
    dev_d = {k: torch.empty_like(v, device=dev) for k, v in host_d.items()}
    p_out = torch.empty_like(dev_p["q"])
    d_out = torch.empty_like(dev_d["q"])
    p_host_out = torch.empty_like(host_p["q"]).pin_memory()
    d_host_out = torch.empty_like(host_d["q"]).pin_memory()
    h2d_p = sum(v.numel() * v.element_size() for v in host_p.values())
    h2d_d = sum(v.numel() * v.element_size() for v in host_d.values())
    d2h_p = p_host_out.numel() * 2
    d2h_d = d_host_out.numel() * 2

    def step(ev):
        ev[0].record(stream)
        for k in dev_p:
            dev_p[k].copy_(host_p[k], non_blocking=True)
        attn.attn_fwd_prefill(p_out, dev_p["q"], dev_p["k_cache"], dev_p["v_cache"],
                              dev_p["block_table"], dev_p["query_start_loc"], dev_p["seq_lens"],
                              max_seqlen_q=pp.max_seqlen_q, max_seqlen_k=pp.max_seqlen_k,
                              scale=pp.scale, causal=True, stream=stream)
        p_host_out.copy_(p_out, non_blocking=True)
        ev[1].record(stream)
        for k in dev_d:
            dev_d[k].copy_(host_d[k], non_blocking=True)
        attn.attn_fwd_decode(d_out, dev_d["q"], dev_d["k_cache"], dev_d["v_cache"],
                             dev_d["block_table"], dev_d["seq_lens"], max_seqlen_k=dp.max_seqlen_k,
                             scale=dp.scale, num_splits=DECODE_SPLITS, workspace=ws, stream=stream)
        d_host_out.copy_(d_out, non_blocking=True)
        ev[2].record(stream)

    n = max(3, min(args.steps, args.e2e_steps))
    for _ in range(2):
        step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    barrier(world)
    for e in evs:
        step(e)
    torch.cuda.synchronize(dev)
    p_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    d_ms = sum(e[1].elapsed_time(e[2]) for e in evs)
    p_ms, d_ms = max_over_ranks(world, dev, [p_ms, d_ms])
    flops = prefill_flops(pp)
    flops_all, dbytes_all = sum_over_ranks(world, dev, [flops, decode_bytes(dp)])
    return {"value": flops_all * n / (p_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d_p + h2d_d, "d2h_bytes_per_step": d2h_p + d2h_d,
            "steps": n,
            "decode": {"value": dbytes_all * n / (d_ms * 1e-3) / 1e9, "unit": "GB/s"},
            "note": "prefill part: H2D of its inputs + kernel + D2H of O; decode part likewise"}


# ----------------------------------------------------------------------------
# the oracle (CPU baseline and reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(prob, n_rows, seed):
    rng = np.random.default_rng(seed)
    total = prob.total_q * prob.num_q_heads
    return np.sort(rng.choice(total, size=min(n_rows, total), replace=False)).astype(np.int64)


def oracle_cost(prob, rows):
    """Unmasked FLOPs of the sampled rows (same count as the GPU metric)."""
    H = prob.num_q_heads
    qsl = prob.query_start_loc.numpy()
    tok = rows // H
    b = np.searchsorted(qsl, tok, side="right") - 1
    i = tok - qsl[b]
    sq = qsl[b + 1] - qsl[b]
    sk = np.asarray(prob.kv_lens)[b]
    vis = np.minimum(sk, i + (sk - sq) + 1) if prob.causal else sk
    return 4.0 * prob.head_size * float(np.clip(vis, 0, None).sum())


def oracle_bytes(prob, rows):
    """K/V bytes the sampled decode rows read, scaled like the GPU metric
    (one K/V read per kv head shared by its group)."""
    H, G = prob.num_q_heads, prob.num_q_heads // prob.num_kv_heads
    tok = rows // H
    sk = np.asarray(prob.kv_lens)[tok]
    per_row = sk * prob.head_size * 2 * 2 / G + 2 * prob.head_size * 2
    return float(per_row.sum())


def time_oracle(prob, rows, threads):
    from oracle import oracle
    t0 = time.perf_counter()
    oracle.sdpa(prob.q, prob.k_cache, prob.v_cache, prob.block_table, prob.query_start_loc,
                prob.seq_lens, num_q_heads=prob.num_q_heads, num_kv_heads=prob.num_kv_heads,
                head_size=prob.head_size, block_size=prob.block_size, scale=prob.scale,
                causal=prob.causal,
                dtype=oracle.BF16 if prob.dtype == torch.bfloat16 else oracle.F16, rows=rows,
                n_threads=threads, want_lse=False)
    return time.perf_counter() - t0


# (workload, rows: "full" or a sample size, threads: "all" or 1)
CPU_SWEEP_PLAN = (
    ("prefill_causal_fp16_s128_d64", "full", "all"),
    ("prefill_causal_fp16_s128_d64", "full", 1),
    ("prefill_causal_bf16_gqa_s2048", "full", "all"),
    ("prefill_causal_bf16_gqa_s2048", 4096, 1),
    ("decode_bf16_b64_paged16", "full", "all"),
    ("prefill_chunked_bf16_b4", "full", "all"),
    ("prefill_causal_bf16_s8192", 16384, "all"),
    ("dense_bf16_bshd_s16384", 2048, "all"),
)


def run_cpu_sweep(args):
    """The fp64 oracle timed on the host cores for every measured workload:
    in full where that takes up to a couple of minutes (C1, C2, C3, C4b),
    else on a random row sample whose time is extrapolated to the workload
    by its FLOPs (labelled so); C1 and C2 also single-threaded.  One JSON
    line per entry.  A baseline, not a target."""
    import platform
    cores = os.cpu_count() or 1
    cpu = platform.processor() or platform.machine()
    for name, rows, th in CPU_SWEEP_PLAN:
        prob = attn_inputs.workload(name)
        threads = cores if th == "all" else int(th)
        total = prob.total_q * prob.num_q_heads
        full = rows == "full"
        r = np.arange(total, dtype=np.int64) if full else oracle_sample(prob, int(rows), 11)
        secs = time_oracle(prob, r, threads)
        if prob.max_seqlen_q == 1:
            work, unit = oracle_bytes(prob, r), "GB/s"
            value, whole = work / secs / 1e9, decode_bytes(prob)
        else:
            work, unit = oracle_cost(prob, r), "TFLOP/s"
            value, whole = work / secs / 1e12, prefill_flops(prob)
        print(json.dumps({"workload": name, "kind": "oracle", "threads": threads, "cpu": cpu,
                          "rows": int(len(r)), "rows_total": int(total), "seconds": secs,
                          "value": value, "unit": unit, "extrapolated": not full,
                          "workload_seconds": secs if full else secs * whole / max(work, 1.0)}),
              flush=True)


def cpu_baseline(pp, dp, seconds):
    threads = os.cpu_count() or 1
    # calibrate on a small sample, then size the sample for ~seconds/2 each
    r0 = oracle_sample(pp, 256, 7)
    t0 = time_oracle(pp, r0, threads)
    n_p = int(max(256, min(pp.total_q * pp.num_q_heads, 256 * (seconds / 2) / max(t0, 1e-3))))
    rp = oracle_sample(pp, n_p, 8)
    tp = time_oracle(pp, rp, threads)
    rd0 = oracle_sample(dp, 64, 9)
    td0 = time_oracle(dp, rd0, threads)
    n_d = int(max(64, min(dp.total_q * dp.num_q_heads, 64 * (seconds / 2) / max(td0, 1e-3))))
    rd = oracle_sample(dp, n_d, 10)
    td = time_oracle(dp, rd, threads)
    return {"value": oracle_cost(pp, rp) / tp / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": f"prefill: {len(rp)} random (token, head) rows of {PREFILL_WL} in {tp:.1f}s; "
                      f"decode: {len(rd)} rows of {DECODE_WL} in {td:.1f}s",
            "decode": {"value": oracle_bytes(dp, rd) / td / 1e9, "unit": "GB/s"}}


def run_reference(args, rank, world):
    """Reference arm: the fp64 oracle on the host cores, each step a bounded
    row sample of the same two workloads."""
    if rank != 0:
        return
    pp, dp = make_problems(seed=0)
    threads = os.cpu_count() or 1
    rows_p = oracle_sample(pp, args.ref_rows, 11)
    rows_d = oracle_sample(dp, max(16, args.ref_rows // 4), 12)
    for _ in range(args.warmup):
        time_oracle(pp, rows_p, threads)
        time_oracle(dp, rows_d, threads)
    tp = td = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tp += time_oracle(pp, rows_p, threads)
        td += time_oracle(dp, rows_d, threads)
    wall = time.perf_counter() - t0
    K = args.steps
    value = oracle_cost(pp, rows_p) * K / tp / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": wall / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": bench_config(1),
        "decode": {"value": oracle_bytes(dp, rows_d) * K / td / 1e9, "unit": "GB/s"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{len(rows_p)} random prefill rows + {len(rows_d)} decode "
                                   f"rows per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def pages_protocol(call, stream, dev, measurements=10, launches=50, trim=0.2):
    """The timing protocol of "gfx942 unified attention -- parity + benchmark
    harness" (the shapes-check flags table under "Running": 10 warm-up
    launches, 50 launches per measurement, 10 measurements reduced by a
    trimmed mean with 0.2 cut from each end; "Troubleshooting" flags cells
    whose spread passes ~10% as noisy): `measurements` CUDA-event measurements
    of `launches` back-to-back calls each (no L2 flush inside a measurement,
    so small problems run warm), the per-call time of each; trimmed mean,
    median, and 'noisy' when (max - min) exceeds 10% of the median."""
    for _ in range(10):
        call()
    times = []
    for _ in range(measurements):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        host_gate(stream, launches)
        a.record(stream)
        for _ in range(launches):
            call()
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b) * 1e3 / launches)
    srt = sorted(times)
    k = int(len(srt) * trim)
    kept = srt[k:len(srt) - k] if len(srt) > 2 * k else srt
    med = statistics.median(srt)
    spread = (srt[-1] - srt[0]) / med if med > 0 else 0.0
    return {"trimmed_mean_us": sum(kept) / len(kept), "median_us": med, "spread": spread,
            "noisy": spread > 0.10, "measurements": measurements,
            "launches_per_measurement": launches, "l2": "warm (no flush inside a measurement)"}


def run_sweep(args, dev):
    """One line per named workload (see --sweep)."""
    import attention_forward_sdpa_gb300 as attn

    attn.load_library()
    peaks, peak_src = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    names = (args.sweep.split(",") if args.sweep != "all"
             else list(attn_inputs.WORKLOADS) + list(FEATURE_WORKLOADS))
    for name in names:
        base, recipe = FEATURE_WORKLOADS.get(name, (name, {}))
        prob = (attn_inputs.workload(base, kv_dtype=torch.float8_e4m3fn) if recipe.get("kv_fp8")
                else attn_inputs.workload(base))
        feat = feature_args(recipe, prob.num_q_heads, dev, prob)
        if recipe.get("kv_fp8") and prob.max_seqlen_q > 1:
            feat["fp8_workspace"] = torch.empty(
                attn.attn_fp8_prefill_workspace_size(prob.num_seqs, prob.max_seqlen_k,
                                                     prob.num_kv_heads, prob.head_size,
                                                     prob.block_size),
                dtype=torch.uint8, device=dev)
        window = recipe.get("window", (-1, -1))
        t = device_args(prob, dev)
        out = torch.empty_like(t["q"])
        is_decode = prob.max_seqlen_q == 1
        if is_decode:
            ws = torch.empty(attn.attn_decode_workspace_size(prob.num_seqs, prob.num_q_heads,
                                                             prob.head_size, DECODE_SPLITS),
                             dtype=torch.uint8, device=dev)

            def call():
                attn.attn_fwd_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                     t["seq_lens"], max_seqlen_k=prob.max_seqlen_k,
                                     scale=prob.scale, num_splits=DECODE_SPLITS, workspace=ws,
                                     stream=stream, **feat)
        else:
            if args.split and not feat:
                feat = {"split_workspace": torch.empty(
                    attn.attn_prefill_split_workspace_size(prob.head_size), dtype=torch.uint8,
                    device=dev)}

            def call():
                attn.attn_fwd_prefill(out, t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                      t["query_start_loc"], t["seq_lens"],
                                      max_seqlen_q=prob.max_seqlen_q,
                                      max_seqlen_k=prob.max_seqlen_k, scale=prob.scale,
                                      causal=prob.causal, stream=stream, **feat)
        for _ in range(args.warmup):
            flush.zero_()
            call()
        torch.cuda.synchronize(dev)
        n = 5 if prob.total_q * prob.num_q_heads > (1 << 22) else 20
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        sampler = ClockSampler(dev.index if dev.index is not None else 0)
        sampler.start()
        time.sleep(0.3)
        t0 = time.time()
        host_gate(stream, n)
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            call()
            b.record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        time.sleep(0.1)
        sampler.stop()
        us = statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3
        proto = pages_protocol(call, stream, dev)
        if is_decode:
            work = decode_bytes(prob, window)
            value, unit, peak = work / us / 1e3, "GB/s", peaks["hbm_gbs"]
            nominal, sustained = NOMINAL_PEAKS["hbm_gbs"], None
            proto["value_trimmed"] = work / proto["trimmed_mean_us"] / 1e3
        else:
            work = prefill_flops(prob, window)
            value, unit, peak = work / us / 1e6, "TFLOP/s", peaks["bf16_tflops"]
            nominal = NOMINAL_PEAKS["bf16_tflops"]
            sustained = peaks.get("bf16_tflops_sustained")
            proto["value_trimmed"] = work / proto["trimmed_mean_us"] / 1e6
        line = {"workload": name, "entry_point": ("attn_fwd_prefill_split"
                                                  if "split_workspace" in feat else None),
                "us": us, "value": value, "unit": unit,
                "frac": value / peak, "peak": peak, "peak_source": peak_src,
                "frac_nominal": value / nominal, "peak_nominal": nominal,
                "calls": n, "clocks": sampler.summary(t0, t1), "protocol": proto}
        if sustained:
            line["frac_sustained"] = value / sustained
            line["peak_sustained"] = sustained
        print(json.dumps(line), flush=True)
        del t, out
        torch.cuda.empty_cache()


# ----------------------------------------------------------------------------
# distributed plumbing
# ----------------------------------------------------------------------------

def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce_over_ranks(world, dev, vals, op):
    if world == 1:
        return list(vals)
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return t.tolist()


def max_over_ranks(world, dev, vals):
    """Element-wise maximum over the ranks (the slowest rank's times)."""
    import torch.distributed as dist
    return _reduce_over_ranks(world, dev, vals, dist.ReduceOp.MAX if world > 1 else None)


def sum_over_ranks(world, dev, vals):
    """Element-wise sum over the ranks (the whole job's work)."""
    import torch.distributed as dist
    return _reduce_over_ranks(world, dev, vals, dist.ReduceOp.SUM if world > 1 else None)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timings")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration timings (C1-C5) of the default line")
    ap.add_argument("--cpu-seconds", type=float, default=16.0)
    ap.add_argument("--ref-rows", type=int, default=128)
    ap.add_argument("--cpu-sweep", action="store_true",
                    help="time the fp64 oracle on the host cores for every measured workload")
    ap.add_argument("--sweep", nargs="?", const="all", default=None,
                    help="time each named workload (comma-separated names, default all)")
    ap.add_argument("--split", action="store_true",
                    help="with --sweep: run flag-free prefill workloads through "
                         "attn_fwd_prefill_split")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.cpu_sweep:
        if rank == 0:
            run_cpu_sweep(args)
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.sweep:
        if rank == 0:
            run_sweep(args, dev)
        return
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=dev)
    try:
        run_ours(args, rank, world, dev)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
