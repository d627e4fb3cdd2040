#!/usr/bin/env python
"""Benchmark of one DSpark decoding cycle's hot path on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
Markov-head drafting (gamma sequential positions), the confidence scheduler,
and rejection-sampling verification of every drafted position.  Workload
(default): R = 256 requests, gamma = 5, V = 151936, r = 256, T = 1, U and P
float32, W1/W2 bf16, verify-all-gamma.

Prints ONE JSON line (rank 0).  `value` is draft+verify positions per second
(R * gamma per step, all ranks) with inputs resident in HBM; `e2e` is the same
metric through the C ABI with host buffers (pinned host -> device copies of
U, P, anchors and confidences, and device -> host reads of the outputs,
inside the timed region).  The timed region holds the cycles alone; a second
pass over the same steps brackets every launch with CUDA events for the
kernel table and the roofline figure (`ms_per_step_profiled`).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dspark|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from speculative_decoding_drafting_gb300 import synth  # noqa: E402

WORKLOAD = "headline"
L2_FLUSH_BYTES = 512 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


class ClockSampler:
    """nvidia-smi sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples go to DSPARK_CLOCKS_DIR (default: the temp directory)
        import tempfile
        d = os.environ.get("DSPARK_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


CSRC = os.path.join(ROOT, "speculative_decoding_drafting_gb300", "csrc")
# kernel (as the library's profiling names it) -> (ncu summary under profiles/, its source file)
KERNEL_PROFILES = {
    "draft_sweep_tc": ("draft_sweep_tc_headline.md", "draft_tc.cu"),
    "verify_pass1": ("verify_pass1_headline.md", "verify.cu"),
    "verify_residual_tc": ("residual_tc_headline.md", "verify_tc.cu"),
}


def source_digest(cu_file: str) -> str:
    """sha256 over a kernel's .cu file and every header of the library: a
    capture's counters stay valid only while this digest is unchanged."""
    import hashlib
    h = hashlib.sha256()
    files = [os.path.join(CSRC, cu_file)] + sorted(
        os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    files.append(os.path.join(ROOT, "include", "dspark.h"))
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel: str):
    """DRAM bytes (read + write) of one launch of `kernel` from its committed
    ncu summary, or None if there is none or the kernel changed since."""
    ent = KERNEL_PROFILES.get(kernel)
    if not ent:
        return None
    path = os.path.join(ROOT, "profiles", ent[0])
    try:
        text = open(path).read()
    except OSError:
        return None
    import re
    m = re.search(r"source sha256: ([0-9a-f]{64})", text)
    if not m or m.group(1) != source_digest(ent[1]):
        return None
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    tot = 0.0
    for key in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
        m = re.search(re.escape(key) + r" = ([0-9.]+) (byte|Kbyte|Mbyte|Gbyte)", text)
        if not m:
            return None
        tot += float(m.group(1)) * scale[m.group(2)]
    return int(tot)


def rank_request_ids(R: int, rank: int) -> np.ndarray:
    """Request ids of one rank: every rank drafts and verifies its own block of
    R requests (weak scaling, no data-path exchange)."""
    return (np.arange(R) + rank * R).astype(np.uint32)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks: the job takes as long as its
    slowest rank.  CPU tensors with gloo, device tensors with NCCL."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(positions_per_rank_step: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job positions per second: every rank's positions over the slowest
    rank's time."""
    return positions_per_rank_step * world * steps / (max_ms / 1000.0)


def algorithmic_bytes(w, n_rej: float, verify_rows: float):
    """Bytes the cycle must move: U, W2 and the W1 rows once; the target rows
    verification must read (each request's rows up to its first rejection,
    or through the bonus row: accept_len + 1 rows); the residual pass's
    re-read of U_j and P_j of every rejecting request and W2 once.  Greedy
    verification (T = 0) has no residual: a mismatch emits the target row's
    argmax, which the row's own read gives."""
    su = 4 if w.u_dtype == synth.F32 else 2
    sp = 4 if w.p_dtype == synth.F32 else 2
    sw = 4 if w.w_dtype == synth.F32 else 2
    if not w.T > 0:
        n_rej = 0
    draft = w.R * w.gamma * w.V * su + w.r * w.V * sw + w.R * w.gamma * w.r * sw
    verify1 = verify_rows * w.V * sp
    resid = n_rej * w.V * (su + sp) + (w.r * w.V * sw if n_rej > 0 else 0)
    return dict(draft=draft, verify_rows=verify1, residual=resid, total=draft + verify1 + resid,
                sweep_per_launch=(w.R * w.V * su + w.r * w.V * sw / w.gamma + w.R * w.r * sw),
                residual_per_launch=resid)


GUMBEL_FLAG = 1e-4     # a draft (Gumbel-max or greedy) margin below this is a flagged decision
UNIFORM_FLAG = 1e-6    # so is a uniform this close to its acceptance or tree threshold


def count_flags(od: dict, ov: dict, g_tokens: np.ndarray, g_out: np.ndarray, g_acc: np.ndarray, acc: dict):
    """Flag accounting of one cycle: the oracle's draft od and verification ov
    against the GPU's tokens, output tokens and accept lengths on the same
    seed and request ids.  A decision is flagged where the oracle's own
    margin lies inside a band the kernels' rounding could cross; only there
    may the two disagree.  Adds to acc: positions compared, flagged decisions,
    flagged and unflagged disagreements."""
    R, gamma = od["tokens"].shape
    for i in range(R):
        diff = np.nonzero(g_tokens[i] != od["tokens"][i])[0]
        kc = int(diff[0]) + 1 if diff.size else gamma          # compared up to the first disagreement
        acc["positions"] += kc
        acc["flagged"] += int((od["margin"][i, :kc] < GUMBEL_FLAG).sum())
        if diff.size:
            k = int(diff[0])
            acc["flagged_disagreements" if od["margin"][i, k] < GUMBEL_FLAG else "unflagged_disagreements"] += 1
            continue
        vflag = bool(ov["min_gap"][i] < UNIFORM_FLAG)
        acc["flagged"] += int(vflag)
        if (g_out[i] != ov["out_tokens"][i]).any() or g_acc[i] != ov["accept_len"][i]:
            acc["flagged_disagreements" if vflag else "unflagged_disagreements"] += 1


def cpu_oracle_sample(w, x, target_s: float = 10.0, gpu_cycle=None):
    """Time the CPU oracle (draft + schedule + verify) on the workload itself:
    whole cycles over all R requests, repeated with fresh seeds until about
    target_s of CPU work; returns positions/s.  With gpu_cycle (seed ->
    numpy tokens, out_tokens, accept_len of the GPU cycle with request ids
    0..R-1, run outside the oracle's timing) the same cycles also give the
    flag accounting of the GPU path against the oracle."""
    import oracle
    cores = oracle.default_threads()
    idx = np.arange(w.R).astype(np.uint32)
    t_tot, cycles = 0.0, 0
    acc = dict(positions=0, flagged=0, flagged_disagreements=0, unflagged_disagreements=0)
    while t_tot < target_s and cycles < 8:
        seed = 7 + cycles
        t0 = time.perf_counter()
        d = oracle.draft_markov(x["U"], x["anchor"], x["W1"], x["W2"], w.T, seed, req_ids=idx)
        oracle.schedule_loop(x["c"], x["sps"])
        v = oracle.verify(x["P"], x["U"], x["W2"], d["tokens"], d["qx"], d["lse"], d["code"], w.T, seed,
                          req_ids=idx)
        t_tot += time.perf_counter() - t0
        cycles += 1
        if gpu_cycle is not None:
            count_flags(d, v, *gpu_cycle(seed), acc)
    cpu = dict(value=cycles * w.R * w.gamma / t_tot, unit="positions/s", cores=cores, kind="oracle",
               sample=f"{cycles} full cycle(s) of the workload (all {w.R} requests x {w.gamma} positions, "
                      f"V={w.V}): draft+schedule+verify, {t_tot:.2f} s on {cores} threads")
    flags = None
    if gpu_cycle is not None:
        n = max(1, acc["positions"])
        flags = dict(acc, flagged_rate=acc["flagged"] / n,
                     disagreement_rate=(acc["flagged_disagreements"] + acc["unflagged_disagreements"]) / n,
                     bands={"gumbel_margin": GUMBEL_FLAG, "uniform_gap": UNIFORM_FLAG},
                     sample=f"the CPU baseline's {cycles} cycle(s), GPU cycles on the same seeds and request ids")
    return cpu, flags


MULTI_GPU_REFUSAL = ("the GPU arm runs on one GPU: the draft sweep and the residual pass share W2 tiles among the "
                     "CTAs of a thread-block cluster by TMA multicast, which is defined for this GPU's own memory "
                     "only; requests shard as independent replicas, not measured on several GPUs")


def refuse_multi_gpu(rank: int, world: int) -> int:
    """Under torchrun with more than one rank the GPU arm does no work: rank 0
    prints one line saying why, every rank exits 0."""
    if rank == 0:
        print(json.dumps({"metric": "draft+verify positions/s", "unit": "positions/s", "n_gpus": world,
                          "value": None, "unavailable": MULTI_GPU_REFUSAL}), flush=True)
    return 0


def run_reference(args):
    """The oracle as the reference arm: K bounded samples of the workload."""
    rank, world, _ = _dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    cores = oracle.default_threads()
    n = min(cores, w.R)
    idx = np.arange(n)
    x = synth.gen_all(w, rows=idx)
    times = []
    for step in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        d = oracle.draft_markov(x["U"], x["anchor"], x["W1"], x["W2"], w.T, 100 + step, req_ids=idx.astype(np.uint32))
        oracle.schedule_loop(x["c"], x["sps"])
        oracle.verify(x["P"], x["U"], x["W2"], d["tokens"], d["qx"], d["lse"], d["code"], w.T, 100 + step,
                      req_ids=idx.astype(np.uint32))
        if step >= args.warmup:
            times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = n * w.gamma * len(times) / tot
    line = {
        "impl": "reference", "metric": "draft+verify positions/s", "value": value, "unit": "positions/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "R": w.R, "gamma": w.gamma, "V": w.V, "r": w.r, "T": w.T,
                   "sample_requests_per_step": n},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {w.R} requests per step, all {w.gamma} positions, V={w.V}"},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def measure_config(name: str, scheduled: bool, steps: int, devc, flush):
    """One more workload's whole cycle (Markov draft, scheduler, verification)
    at its own sizes, timed as the headline is (L2 flushed between cycles,
    CUDA events on the launch stream): positions per second, the cycle's
    algorithmic bytes and their fraction of the measured HBM peak.  With
    `scheduled` the verify lengths come from the scheduler's output (for the
    long block at rho = 0.9 it chooses l = 0 everywhere: one token per
    request, drawn from the first target row); otherwise every position is
    verified.  Inputs are drawn on the device (synth.gen_device)."""
    import torch
    from speculative_decoding_drafting_gb300 import binding
    w = synth.WORKLOADS[name]
    x = synth.gen_device(w, devc, seed=1)
    stream = torch.cuda.current_stream()
    wss = [None, None, None]

    def cycle(seed):
        d = binding.draft_markov(x["U"], x["anchor"], x["W1"], x["W2"], w.T, seed, ws=wss[0])
        s = binding.schedule(x["c"], x["sps"], ws=wss[1])
        v = binding.verify(x["P"], x["U"], x["W2"], d, w.T, seed, verify_len=s["verify_len"] if scheduled else None,
                           ws=wss[2])
        wss[:] = [d["ws"], s["ws"], v["ws"]]
        return d, s, v

    for i in range(3):
        cycle(10 + i)
    ms, rej, rows, vl = [], [], [], []
    for i in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        d, s, v = cycle(100 + i)
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
        lens = s["verify_len"] if scheduled else torch.full((w.R,), w.gamma, dtype=torch.int32, device=devc)
        acc = v["accept_len"]
        rej.append(int((acc < lens).sum().item()))
        rows.append(int((acc + 1).sum().item()))
        vl.append(float(lens.float().mean().item()))
    per = float(np.median(ms))
    ab = algorithmic_bytes(w, float(np.mean(rej)), float(np.mean(rows)))
    hbm_peak, _, peak_src = _peaks()
    gbs = ab["total"] / (per / 1000.0) / 1e9
    st = {synth.F32: "f32", synth.BF16: "bf16"}
    del x
    torch.cuda.empty_cache()
    return {"workload": (f"{w.name}: R={w.R} gamma={w.gamma} V={w.V} r={w.r} T={w.T} U {st[w.u_dtype]} "
                         f"P {st[w.p_dtype]} W {st[w.w_dtype]}"),
            "verify": ("scheduler (rho = %.1f)" % w.rho) if scheduled else "all gamma positions",
            "metric": "draft+verify positions/s", "value": round(w.R * w.gamma / (per / 1000.0), 1),
            "ms_per_cycle": round(per, 4), "mean_verify_len": round(float(np.mean(vl)), 3),
            "rejecting_requests": float(np.mean(rej)), "target_rows_read": float(np.mean(rows)),
            "algorithmic_bytes": int(ab["total"]), "achieved_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / hbm_peak, 4), "peak_source": f"{peak_src} hbm_gbs",
            "inputs": "drawn on the device (same distributions as the numpy generator)"}


def measure_rnn_draft(steps: int, warmup: int, devc, flush):
    """The RNN-head variant of the draft at its own workload (rnn: R = 256,
    gamma = 8, V = 151936, r = 256, d = 2048): draft positions per second,
    L2 flushed between calls, and the per-kernel table of a profiled pass."""
    import torch
    from speculative_decoding_drafting_gb300 import binding
    w = synth.WORKLOADS["rnn"]

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(devc)

    U, anchor = to_dev(synth.gen_U(w)), to_dev(synth.gen_anchor(w))
    W1, W2, Wgco, H = to_dev(synth.gen_W1(w)), to_dev(synth.gen_W2(w)), to_dev(synth.gen_Wgco(w)), to_dev(synth.gen_H(w))
    d = binding.draft_rnn(U, anchor, W1, W2, Wgco, H, w.T, 1)
    for i in range(warmup):
        binding.draft_rnn(U, anchor, W1, W2, Wgco, H, w.T, 2 + i, ws=d["ws"], out=d)
    stream = torch.cuda.current_stream()
    ms = []
    for prof in (False, True):
        binding.profile_enable(prof)
        for i in range(steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            binding.draft_rnn(U, anchor, W1, W2, Wgco, H, w.T, 100 + i, ws=d["ws"], out=d)
            b.record(stream)
            torch.cuda.synchronize()
            if not prof:
                ms.append(a.elapsed_time(b))
        binding.profile_enable(False)
    table = {}
    for name, t in binding.profile_collect():
        e = table.setdefault(name, [0, 0.0])
        e[0] += 1
        e[1] += t
    per = float(np.mean(ms))
    return {"workload": f"{w.name}: R={w.R} gamma={w.gamma} V={w.V} r={w.r} d={w.d} T={w.T} U f32, W/H/Wgco bf16",
            "metric": "draft positions/s", "value": round(w.R * w.gamma / (per / 1000.0), 1),
            "ms_per_draft": round(per, 4),
            "kernels_us_per_launch": {k: round(1000 * v / n, 2) for k, (n, v) in table.items()}}


def measure_confidence_and_threshold(w, U, anchor, W1, W2, c, steps: int, devc, flush, d_conf: int = 2048):
    """The fused confidence head and the threshold filter on the headline
    workload.  The head: the Markov draft with and without a d = 2048 head
    (alternating calls, L2 flushed before each), its extra time per draft and
    per prep launch.  The threshold filter: one call on c [R, gamma]."""
    import torch
    from speculative_decoding_drafting_gb300 import binding

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(devc)

    H, wc = to_dev(synth.gen_conf_H(w, d_conf)), to_dev(synth.gen_conf_w(w, d_conf))
    base = binding.draft_markov(U, anchor, W1, W2, w.T, 1)
    withc = binding.draft_markov(U, anchor, W1, W2, w.T, 1, conf_w=wc, conf_H=H)
    stream = torch.cuda.current_stream()
    ms = {False: [], True: []}
    for i in range(3 + steps):
        for on in (False, True):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if on:
                binding.draft_markov(U, anchor, W1, W2, w.T, 50 + i, ws=withc["ws"], out=withc, conf_w=wc, conf_H=H)
            else:
                binding.draft_markov(U, anchor, W1, W2, w.T, 50 + i, ws=base["ws"], out=base)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                ms[on].append(a.elapsed_time(b))
    prep = {}
    for on in (False, True):
        binding.profile_enable(True)
        for i in range(steps):
            flush.zero_()
            if on:
                binding.draft_markov(U, anchor, W1, W2, w.T, 90 + i, ws=withc["ws"], out=withc, conf_w=wc, conf_H=H)
            else:
                binding.draft_markov(U, anchor, W1, W2, w.T, 90 + i, ws=base["ws"], out=base)
        torch.cuda.synchronize()
        binding.profile_enable(False)
        t = [ms_ for name, ms_ in binding.profile_collect() if name == "draft_prep"]
        prep[on] = 1000.0 * float(np.mean(t))
    # threshold filter: one call per event pair (launch-bound: R * gamma floats)
    out = torch.empty((w.R,), dtype=torch.int32, device=devc)
    for i in range(5):
        binding.schedule_threshold(c, 0.5, 0, out=out)
    th = []
    for i in range(max(10, steps)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.schedule_threshold(c, 0.5, 0, out=out)
        b.record(stream)
        torch.cuda.synchronize()
        th.append(a.elapsed_time(b))
    m0, m1 = float(np.median(ms[False])), float(np.median(ms[True]))
    return {
        "confidence_head": {"workload": f"{w.name} draft with a d={d_conf} head (h bf16 [R, gamma, d], w f32 [d + r])",
                            "ms_per_draft_without": round(m0, 4), "ms_per_draft_with": round(m1, 4),
                            "extra_us_per_draft": round(1000 * (m1 - m0), 2),
                            "prep_us_without": round(prep[False], 2), "prep_us_with": round(prep[True], 2),
                            "h_bytes_per_draft": int(w.R * w.gamma * d_conf * 2)},
        "threshold_filter": {"workload": f"c [{w.R}, {w.gamma}] float32, theta 0.5, prefix-survival mode",
                             "us_per_call": round(1000 * float(np.median(th)), 2)},
    }


def measure_sts(steps: int, devc):
    """Sequential Temperature Scaling fit on a calibration set of 65536 draft
    blocks (gamma = 8, 256 log-spaced temperatures in [0.1, 10], 15 bins):
    fits per second and the per-kernel table.  Each fit evaluates
    N gamma G calibrated prefix-survival values."""
    import torch
    from speculative_decoding_drafting_gb300 import binding
    N, gamma, G, M = 65536, 8, 256, 15
    c, al = synth.gen_sts_set(N, gamma, tau=2.0, seed=1)
    cd = torch.from_numpy(c).to(devc)
    ad = torch.from_numpy(al).to(devc)
    grid = torch.from_numpy(synth.sts_grid(G, 0.1, 10.0)).to(devc)
    out = binding.sts_fit(cd, ad, grid, M)
    for _ in range(3):
        binding.sts_fit(cd, ad, grid, M, ws=out["ws"], out=out)
    stream = torch.cuda.current_stream()
    ms = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.sts_fit(cd, ad, grid, M, ws=out["ws"], out=out)
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    binding.profile_enable(True)
    for _ in range(steps):
        binding.sts_fit(cd, ad, grid, M, ws=out["ws"], out=out)
    torch.cuda.synchronize()
    binding.profile_enable(False)
    table = {}
    for name, t in binding.profile_collect():
        e = table.setdefault(name, [0, 0.0])
        e[0] += 1
        e[1] += t
    per = float(np.median(ms))
    return {"workload": f"calibration set N={N} gamma={gamma}, G={G} temperatures, M={M} bins",
            "ms_per_fit": round(per, 4), "evaluations_per_s": round(N * gamma * G / (per / 1000.0), 1),
            "t": [round(float(v), 4) for v in out["t"].cpu().numpy()],
            "kernels_us_per_launch": {k: round(1000 * v / n, 2) for k, (n, v) in table.items()}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dspark", choices=["dspark", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the RNN-head draft, confidence-head, threshold-filter and STS measurements")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    rank, world, local = _dist_env()
    if world > 1:
        return refuse_multi_gpu(rank, world)

    import torch

    from speculative_decoding_drafting_gb300 import binding

    torch.cuda.set_device(local)
    devc = torch.device("cuda", local)
    binding.load()
    w = synth.WORKLOADS[args.workload]
    if w.head != "markov":
        raise SystemExit("bench times the Markov-head cycle")
    x = synth.gen_all(w)
    req_ids = rank_request_ids(w.R, rank)                       # distinct requests on every rank

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(devc)

    U, P, W1, W2 = to_dev(x["U"]), to_dev(x["P"]), to_dev(x["W1"]), to_dev(x["W2"])
    anchor, c, sps, rid = to_dev(x["anchor"]), to_dev(x["c"]), to_dev(x["sps"]), to_dev(req_ids)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=devc)
    stream = torch.cuda.current_stream()

    def step(seed, ws=None):
        d = binding.draft_markov(U, anchor, W1, W2, w.T, seed, req_ids=rid, ws=ws and ws[0])
        s = binding.schedule(c, sps, ws=ws and ws[1])
        v = binding.verify(P, U, W2, d, w.T, seed, verify_len=None, req_ids=rid, ws=ws and ws[2])
        return d, s, v

    d, s, v = step(1)
    wss = (d["ws"], s["ws"], v["ws"])
    for i in range(args.warmup):
        step(10 + i, wss)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)

    def timed(k_steps, seed0, profiled):
        """k_steps cycles, each between a pair of events on the launch stream,
        L2 flushed before each; with `profiled` the library also brackets
        every launch with its own events (kernel table, roofline)."""
        binding.profile_enable(profiled)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k_steps)]
        outs = []
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(k_steps):
            flush.zero_()                                   # evict L2 between steps
            ev[i][0].record(stream)
            d, s, v = step(seed0 + i, wss)
            ev[i][1].record(stream)
            outs.append((v["accept_len"].clone(),))
        torch.cuda.synchronize()
        t_w = time.perf_counter() - t0
        binding.profile_enable(False)
        return [a.elapsed_time(b) for a, b in ev], outs, t_w, (binding.profile_collect() if profiled else [])

    # the timed region: nothing but the cycles (and the flush between them)
    step_ms, outs, t_wall, _ = timed(args.steps, 1000, False)
    # the same steps again with an event pair around every launch: the per-kernel
    # durations of the kernel table and the roofline (events between launches
    # also keep consecutive kernels from overlapping, so this pass is slower)
    prof_ms, _, _, launches = timed(args.steps, 1000, True)
    clk = clocks.stop()
    tot_ms = max_over_ranks(sum(step_ms), world, devc)
    value = job_throughput(w.R * w.gamma, world, args.steps, tot_ms)

    # kernel table from the per-launch events
    table = {}
    for name, ms in launches:
        e = table.setdefault(name, [0, 0.0])
        e[0] += 1
        e[1] += ms
    n_rej = float(np.mean([int((o[0] < w.gamma).sum().item()) for o in outs]))
    sweeps = [ms for name, ms in launches if name.startswith("draft_sweep")]
    sweep_by_k = [round(float(np.mean(sweeps[k::w.gamma])), 4) for k in range(w.gamma)] if sweeps else None
    rows_read = float(np.mean([int((o[0] + 1).sum().item()) for o in outs]))
    ab = algorithmic_bytes(w, n_rej, rows_read)
    hbm_peak, bf16_peak, peak_src = _peaks()
    dom = max(table.items(), key=lambda kv: kv[1][1])
    dom_name, (dom_n, dom_ms) = dom[0], dom[1]
    per_launch = {"draft_sweep_tc": ab["sweep_per_launch"], "draft_sweep_generic": ab["sweep_per_launch"],
                  "verify_residual_tc": ab["residual_per_launch"],
                  "verify_residual_generic": ab["residual_per_launch"]}
    dom_bytes = per_launch.get(dom_name)
    roofline = None
    if dom_bytes:
        achieved = dom_bytes / (dom_ms / dom_n / 1000.0) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(achieved / hbm_peak, 4), "traffic": measured_traffic(dom_name),
                    "kernel": dom_name, "peak_source": f"{peak_src} hbm_gbs",
                    "algorithmic_bytes_per_launch": int(dom_bytes)}
    cycle_gbs = ab["total"] / (tot_ms / args.steps / 1000.0) / 1e9 if world == 1 else None

    # end to end through the C ABI with host buffers
    e2e = None
    if args.e2e_steps > 0:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        hU, hP, hA, hC = pin(x["U"]), pin(x["P"]), pin(x["anchor"]), pin(x["c"])
        if x["U"].dtype == np.uint16:
            hU = hU.view(torch.bfloat16)
        if x["P"].dtype == np.uint16:
            hP = hP.view(torch.bfloat16)
        n_e2e = args.e2e_steps
        h_out = torch.empty((w.R, w.gamma + 1), dtype=torch.int32).pin_memory()
        h_n = [torch.empty((w.R,), dtype=torch.int32).pin_memory() for _ in range(n_e2e)]
        # the target logits stay in pinned host memory and verification reads
        # them in place (zero copy): only the rows its decisions need cross the
        # host link; U (all of it is drafted from), the anchors and c are
        # copied.  The device holds two sets of the copied inputs: the copy of
        # step i + 1 runs on its own stream while step i computes.  The timed
        # region opens before the first copy and closes after the last result
        # is read back.
        try:
            Pv = binding.host_view(hP, devc)
        except Exception:                                   # not mapped: copy P as well
            Pv = None
        stage = P if Pv is not None else None             # device rows of P, filled by verification's pass 1
        bufs = [dict(U=U, P=Pv if Pv is not None else P, anchor=anchor, c=c),
                dict(U=torch.empty_like(U), P=Pv if Pv is not None else torch.empty_like(P),
                     anchor=torch.empty_like(anchor), c=torch.empty_like(c))]
        cstream = torch.cuda.Stream(device=devc)
        ev_copied = [torch.cuda.Event() for _ in range(2)]
        ev_free = [torch.cuda.Event() for _ in range(2)]

        def copy_in(bi):
            b = bufs[bi]
            with torch.cuda.stream(cstream):
                b["U"].copy_(hU, non_blocking=True)
                if Pv is None:
                    b["P"].copy_(hP, non_blocking=True)
                b["anchor"].copy_(hA, non_blocking=True)
                b["c"].copy_(hC, non_blocking=True)
                ev_copied[bi].record(cstream)

        def step_on(b, seed):
            d = binding.draft_markov(b["U"], b["anchor"], W1, W2, w.T, seed, req_ids=rid, ws=wss[0])
            s_ = binding.schedule(b["c"], sps, ws=wss[1])
            v = binding.verify(b["P"], b["U"], W2, d, w.T, seed, verify_len=None, req_ids=rid, ws=wss[2],
                               p_stage=stage)
            return d, s_, v

        def pipeline(n, seed0, keep):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            cstream.wait_event(t0)
            copy_in(0)
            for i in range(n):
                bi = i % 2
                stream.wait_event(ev_copied[bi])
                d, s_, v = step_on(bufs[bi], seed0 + i)
                h_out.copy_(v["out_tokens"], non_blocking=True)
                keep[i].copy_(v["n_out"], non_blocking=True)
                ev_free[bi].record(stream)
                if i + 1 < n:
                    nb = (i + 1) % 2
                    if i >= 1:
                        cstream.wait_event(ev_free[nb])     # step i - 1 is done with that buffer
                    copy_in(nb)
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)

        pipeline(2, 4000, h_n)                              # warm-up
        flush.zero_()
        torch.cuda.synchronize()
        e2e_ms = [pipeline(n_e2e, 5000, h_n) / n_e2e] * n_e2e
        copied = int(hU.numel() * hU.element_size() + hA.numel() * 4 + hC.numel() * 4)
        if Pv is None:
            p_bytes = float(hP.numel() * hP.element_size())
        else:
            # target bytes fetched: with a staging buffer verification reads one
            # row per wave, so exactly rows 0 .. accept_len of each request
            # (n_out rows); the later passes read the device copy pass 1 made
            sp_ = hP.element_size()
            per = [int(hn.numpy().astype(np.int64).sum()) * w.V * sp_ for hn in h_n]
            p_bytes = float(np.mean(per))
        h2d = int(copied + p_bytes)
        d2h = int(h_out.numel() * 4 + h_n[0].numel() * 4)
        e2e_tot = max_over_ranks(sum(e2e_ms), world, devc)
        e2e_value = job_throughput(w.R * w.gamma, world, len(e2e_ms), e2e_tot)
        e2e = {"value": round(e2e_value, 1), "unit": "positions/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_tot / len(e2e_ms), 3),
               "steps": len(e2e_ms),
               "inputs": ("U, anchors, c copied from pinned host memory on a second stream, double-buffered (the copy "
                          "of step i + 1 overlaps step i); P read in place from pinned host memory, only the rows "
                          "verification needs (one row per wave), each once: pass 1 copies them to a device staging "
                          "buffer for the later passes (h2d_bytes_per_step counts the bytes fetched)" if Pv is not None else
                          "U, P, anchors, c copied from pinned host memory on a second stream, double-buffered"),
               "p_zero_copy": Pv is not None}

    variants = None
    if rank == 0 and world == 1 and not args.no_variants:
        variants = {"dspark5": measure_config("dspark5", False, max(5, args.steps // 2), devc, flush),
                    "greedy": measure_config("greedy", False, max(5, args.steps // 2), devc, flush),
                    "longblock_verify_all": measure_config("longblock", False, max(5, args.steps // 2), devc, flush),
                    "longblock_scheduled": measure_config("longblock", True, max(5, args.steps // 2), devc, flush),
                    "rnn_draft": measure_rnn_draft(max(3, args.steps // 2), 3, devc, flush)}
        variants.update(measure_confidence_and_threshold(w, U, anchor, W1, W2, c, max(5, args.steps // 2), devc,
                                                         flush))
        variants["sts_fit"] = measure_sts(max(5, args.steps // 2), devc)

    cpu = flags = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def gpu_cycle(seed):
            d_, s_, v_ = step(seed, wss)
            torch.cuda.synchronize()
            return (d_["tokens"].cpu().numpy(), v_["out_tokens"].cpu().numpy(), v_["accept_len"].cpu().numpy())

        cpu, flags = cpu_oracle_sample(w, x, gpu_cycle=gpu_cycle)

    if rank == 0:
        kernels = {k: {"launches": n, "ms_total": round(ms, 3), "share": round(ms / max(1e-9, sum(
            t[1] for t in table.values())), 4)} for k, (n, ms) in sorted(table.items(), key=lambda kv: -kv[1][1])}
        line = {
            "metric": "draft+verify positions/s", "value": round(value, 1), "unit": "positions/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{w.name}: R={w.R} gamma={w.gamma} V={w.V} r={w.r} T={w.T} U/P f32 W bf16, "
                                   "verify-all-gamma, scheduler computed each step",
                       "R": w.R, "gamma": w.gamma, "V": w.V, "r": w.r, "T": w.T,
                       "l2": "flushed between steps (512 MB write); inputs 1.7 GB > L2",
                       "parallelism": f"replicas x{world} (requests sharded, no collective)"},
            "roofline": roofline,
            "cycle": {"algorithmic_bytes": int(ab["total"]), "achieved_gbs": round(cycle_gbs, 1) if cycle_gbs else None,
                      "hbm_frac": round(cycle_gbs / hbm_peak, 4) if cycle_gbs else None,
                      "rejecting_requests_per_step": n_rej, "target_rows_read_per_step": rows_read},
            "kernels": kernels,
            "draft_sweep_ms_by_position": sweep_by_k,
            "ms_per_step_profiled": round(sum(prof_ms) / len(prof_ms), 4),
            "gpu_launches": len(launches),
            "clocks": clk,
            "wall_s_timed": round(t_wall, 3),
            "e2e": e2e,
            "cpu_baseline": cpu,
            "flags": flags,
            "variants": variants,
        }
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
