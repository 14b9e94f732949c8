#!/usr/bin/env python3
"""Benchmark of the verification step: verified draft positions per second and
achieved HBM bandwidth on GB300, one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c1] [--impl reference]

``--workload ng1`` / ``ng2`` time the n-gram drafter instead (one
spec_ngram_propose call over a batch of contexts per step); ``--workload eg1``
times the EAGLE-2 tree budget (one budget build for a batch of trees per step).

A step is one call of the verification on one batch of the workload
(default c1: chain, B=64, K=5, V=128256, bf16 logits, T=0.7), inputs resident
in HBM.  Consecutive steps rotate through input copies whose total exceeds
twice the L2, so no step finds its logits in L2.  Under torchrun each rank
verifies its own batch (weak scaling, no collective on the data path); the
time is the max over ranks.

``--impl reference`` times the fp64 CPU oracle on the host cores instead (the
reference arm): each step verifies one sequence of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
UNIT = "positions/s"
LAUNCHES_PER_CALL = 2  # the streaming row kernel and the per-sequence decision kernel


NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal
EX2_PER_SM_CLOCK = 16      # MUFU base-2 exponentials per SM per clock, nominal
STAT_CALLS = 200           # calls behind every per-call percentile (independent of --steps)


def _quantile(sorted_vals, q):
    i = min(len(sorted_vals) - 1, max(0, int(round(q * (len(sorted_vals) - 1)))))
    return sorted_vals[i]


def _cpu_model():
    """The host CPU's name from /proc/cpuinfo (x86: 'model name'; Arm:
    implementer and part numbers), else the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        names = {"0xd4f": "Neoverse V2", "0xd40": "Neoverse V1", "0xd49": "Neoverse N2", "0xd0c": "Neoverse N1"}
        part = fields["CPU part"]
        return (f"{platform.machine()} {names.get(part, 'part ' + part)} "
                f"(implementer {fields.get('CPU implementer', '?')}, part {part})")
    return platform.machine()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _source_hash():
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "sampling_row_online_gb300", "csrc", "*"))):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profile_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    m_h = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != _source_hash():
        return None
    return int(m_b.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 50):
        self.proc = None
        self.err = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:  # pragma: no cover
            self.err = str(e)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": self.err}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:  # pragma: no cover
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


def parse_clock_samples(text: str):
    sm, smax, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            smax.append(float(parts[1]))
        except ValueError:
            continue
        for nm, v in zip(names, parts[4:8]):
            if v.lower().startswith("active"):
                reasons.add(nm)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm)}


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, backend_device=None) -> float:
    """Max of a float over all ranks (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64,
                     device=backend_device if backend_device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
def make_inputs(w, device):
    from sampling_row_online_gb300.workloads import make_chain, make_tree, make_tree_sample
    if w.kind == "tree":
        return make_tree(w, device=device)
    if w.kind == "tree_sample":
        return make_tree_sample(w, device=device)
    return make_chain(w, device=device)


def time_oracle(w, n_sequences: int, host_inputs=None, nthreads=None):
    """Verifies n_sequences sequences of workload w with the oracle (cycling through
    the batch, all host cores); returns (seconds, threads, description)."""
    import numpy as np
    import torch
    import oracle
    nthreads = nthreads or max(1, os.cpu_count() or 1)
    if host_inputs is None:
        host_inputs = make_inputs(w, "cpu")
    done = 0
    t0 = time.perf_counter()
    while done < n_sequences:
        nb = min(w.B, n_sequences - done)
        if w.kind == "tree":
            zt, parent, tok = host_inputs
            oracle.verify_tree_greedy(zt[:nb], parent, tok[:nb], nthreads=nthreads)
        elif w.kind == "tree_sample":
            zt, zd, parent, tok = host_inputs
            oracle.verify_tree_sample(zt[:nb], zd[:nb], parent, tok[:nb], w.T, w.verify_seed,
                                      b_ids=np.arange(nb), nthreads=nthreads)
        else:
            zt, zd, x = host_inputs
            oracle.verify_chain(zt[:nb], None if zd is None else zd[:nb], x[:nb], w.T,
                                w.verify_seed, b_ids=np.arange(nb), nthreads=nthreads)
        done += nb
    return time.perf_counter() - t0, nthreads


def chain_config(w, ws):
    """The config of a verification workload's line, the same for both arms."""
    from sampling_row_online_gb300.workloads import describe, input_copies_for_cold_l2
    per_copy = w.algorithmic_bytes
    ncopies = input_copies_for_cold_l2(per_copy)
    return {"workload": f"{w.name}: {describe(w)}", "logits": w.dtype,
            "per_rank_batch": w.B, "parallelism": f"replicas x{ws} (sequences sharded, no collective)",
            "l2": f"rotating {ncopies} input copies ({ncopies * per_copy / 1e6:.0f} MB > 2x L2)"}


def run_reference(args, w):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    from sampling_row_online_gb300.workloads import describe
    host = make_inputs(w, "cpu")
    per_seq_positions = w.positions // w.B
    if args.warmup > 0:
        time_oracle(w, min(args.warmup, w.B), host)
    secs, threads = time_oracle(w, args.steps, host)
    value = args.steps * per_seq_positions / secs
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": chain_config(w, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} sequences of {w.name} (cycling through its "
                                   f"batch of {w.B}), fp64 oracle, {threads} OpenMP threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_gpu(args, w):
    import numpy as np
    import torch
    import torch.distributed as dist
    from sampling_row_online_gb300 import binding
    from sampling_row_online_gb300.workloads import describe, input_copies_for_cold_l2
    ws, rank, local = _dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    lib = binding.library()
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)

    # inputs (rank-specific seed: each rank verifies its own batch)
    wr = w.scaled(data_seed=w.data_seed + 7919 * rank)
    first = make_inputs(wr, dev)
    per_copy = w.algorithmic_bytes
    ncopies = input_copies_for_cold_l2(per_copy)
    copies = [first] + [tuple(t.clone() if t.dim() >= 2 and t.numel() * t.element_size() > 1 << 20
                              else t for t in first) for _ in range(ncopies - 1)]
    B, V = w.B, w.V
    dt = 0 if w.dtype == "f32" else 1
    if w.kind in ("tree", "tree_sample"):
        D = binding.spec_tree_max_depth(first[-2].cpu())
        out_a = torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    else:
        D = 0
        out_a = torch.empty((B, w.K + 1), dtype=torch.int32, device=dev)
    out_b = torch.empty((B,), dtype=torch.int32, device=dev)

    def make_call(c):
        if w.kind == "tree_sample":
            zt, zd, parent, tok = c
            a = (ctypes.c_void_p(zt.data_ptr()), ctypes.c_void_p(zd.data_ptr()),
                 ctypes.c_void_p(parent.data_ptr()), ctypes.c_void_p(tok.data_ptr()), B, w.K, V, dt,
                 ctypes.c_float(w.T), ctypes.c_uint64(w.verify_seed), D,
                 ctypes.c_void_p(out_a.data_ptr()), ctypes.c_void_p(out_b.data_ptr()), sp)
            return lambda: lib.spec_verify_tree(*a)
        if w.kind == "tree":
            zt, parent, tok = c
            a = (ctypes.c_void_p(zt.data_ptr()), ctypes.c_void_p(parent.data_ptr()),
                 ctypes.c_void_p(tok.data_ptr()), B, w.K, V, dt, D,
                 ctypes.c_void_p(out_a.data_ptr()), ctypes.c_void_p(out_b.data_ptr()), sp)
            return lambda: lib.spec_verify_tree_greedy(*a)
        zt, zd, x = c
        a = (ctypes.c_void_p(zt.data_ptr()),
             ctypes.c_void_p(zd.data_ptr()) if zd is not None else None,
             ctypes.c_void_p(x.data_ptr()), B, w.K, V, dt, ctypes.c_float(w.T),
             ctypes.c_uint64(w.verify_seed), ctypes.c_void_p(out_a.data_ptr()),
             ctypes.c_void_p(out_b.data_ptr()), sp)
        return lambda: lib.spec_verify(*a)

    calls = [make_call(c) for c in copies]
    for k in range(max(3, args.warmup)):
        st = calls[k % ncopies]()
        if st != 0:
            raise SystemExit(f"spec call failed: {st} {lib.spec_last_error_message().decode()}")
    torch.cuda.synchronize()
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error during warm-up")

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    wall0 = time.perf_counter()
    t_start.record(stream)
    for k in range(args.steps):
        calls[k % ncopies]()
    t_end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if ws > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    status = lib.spec_get_status(sp)
    if status != 0:
        raise SystemExit(f"device status error in the timed region: {status}")
    region_ms = t_start.elapsed_time(t_end)
    region_ms = max_over_ranks(region_ms, dev)
    # calls run back to back on the stream (each call's first kernel is a
    # programmatic dependent of the previous call's last): the average call
    # time is the region over the steps
    call_ms = region_ms / args.steps
    # the dominant kernel alone: an event before each call and one the library
    # records between its two launches (spec_arm_rows_event); a fixed sample
    # of STAT_CALLS calls, whatever --steps is
    n_rows = STAT_CALLS
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rows)]
    for a, b in ev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for k in range(n_rows):
        ev[k][0].record(stream)
        lib.spec_arm_rows_event(ctypes.c_void_p(ev[k][1].cuda_event))
        calls[k % ncopies]()
    torch.cuda.synchronize()
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error in the kernel-timing loop")
    avg_launch_ms = max_over_ranks(statistics.fmean(a.elapsed_time(b) for a, b in ev), dev)
    launch_us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
    # the same kernel with warm L2: calls on one input copy, so the end of the
    # previous call's stream is still resident
    n_warm = min(n_rows, 50)
    evw = ev[:n_warm]
    calls[0]()
    for k in range(n_warm):
        evw[k][0].record(stream)
        lib.spec_arm_rows_event(ctypes.c_void_p(evw[k][1].cuda_event))
        calls[0]()
    torch.cuda.synchronize()
    warm_ms = max_over_ranks(statistics.fmean(a.elapsed_time(b) for a, b in evw), dev)
    # the same calls chained back to back (as in the timed region), each with
    # device stamps (spec_arm_timer: no stream operation between launches):
    # the dominant kernel's time as it runs there, the call's device time, and
    # the start-to-start period of consecutive calls
    stamps = torch.empty((STAT_CALLS, 3), dtype=torch.int64, device=dev)
    stamps[:, 0] = -1
    stamps[:, 1:] = 0
    torch.cuda.synchronize()
    for k in range(STAT_CALLS):
        lib.spec_arm_timer(ctypes.c_void_p(stamps[k].data_ptr()))
        calls[k % ncopies]()
    torch.cuda.synchronize()
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error in the chained-stamps loop")
    st_np = stamps.cpu().numpy().view(np.uint64).astype(np.float64)
    chained_row_us = sorted(((st_np[:, 1] - st_np[:, 0]) / 1e3).tolist())
    chained_call_us = sorted(((st_np[:, 2] - st_np[:, 0]) / 1e3).tolist())
    chained_period_us = sorted(((st_np[1:, 0] - st_np[:-1, 0]) / 1e3).tolist())
    positions = w.positions * args.steps * ws
    value = positions / (region_ms / 1e3)

    # end to end through the host-buffer entry point (copies in the timed region)
    e2e = None
    if w.kind == "chain" and not args.no_e2e:
        zt, zd, x = first
        hzt, hzd, hx = (zt.cpu().pin_memory(), None if zd is None else zd.cpu().pin_memory(),
                        x.cpu().pin_memory())
        hout = torch.empty((B, w.K + 1), dtype=torch.int32, pin_memory=True)
        hn = torch.empty((B,), dtype=torch.int32, pin_memory=True)
        e_args = (ctypes.c_void_p(hzt.data_ptr()),
                  ctypes.c_void_p(hzd.data_ptr()) if hzd is not None else None,
                  ctypes.c_void_p(hx.data_ptr()), B, w.K, V, dt, ctypes.c_float(w.T),
                  ctypes.c_uint64(w.verify_seed), ctypes.c_void_p(hout.data_ptr()),
                  ctypes.c_void_p(hn.data_ptr()), sp)
        e_steps = max(5, min(args.steps, 30))
        for _ in range(3):
            lib.spec_verify_host(*e_args)
        if ws > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e_steps):
            st = lib.spec_verify_host(*e_args)
            if st != 0:
                raise SystemExit(f"spec_verify_host failed: {st}")
        e_sec = max_over_ranks(time.perf_counter() - t0, dev)
        h2d = hzt.numel() * hzt.element_size() + (0 if hzd is None else hzd.numel() * hzd.element_size()) \
            + hx.numel() * 4
        d2h = hout.numel() * 4 + hn.numel() * 4
        e2e = {"value": w.positions * e_steps * ws / e_sec, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = _peaks()
    kernel = "row_kernel"
    achieved = w.algorithmic_bytes / (avg_launch_ms / 1e3) / 1e9
    call_achieved = w.algorithmic_bytes / (call_ms / 1e3) / 1e9
    med_launch_ms = _quantile(launch_us, 0.5) / 1e3
    achieved_med = w.algorithmic_bytes / (med_launch_ms / 1e3) / 1e9
    q3 = lambda v: [_quantile(v, q) for q in (0.1, 0.5, 0.9)]
    row_med = _quantile(chained_row_us, 0.5)
    period_med = _quantile(chained_period_us, 0.5)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "frac_median": achieved_med / peak,
                "peak_source": f"{peak_kind} hbm_gbs",
                "traffic": _profile_traffic(kernel, w.name), "kernel": kernel,
                "timed": (f"{kernel} alone: CUDA events on the call's stream before the call and "
                          f"between its two launches (spec_arm_rows_event), mean of {n_rows} calls "
                          f"(frac_median: their median)"),
                "algorithmic_bytes_per_launch": w.algorithmic_bytes,
                "avg_launch_us": avg_launch_ms * 1e3,
                "launch_us_p10_median_p90": [_quantile(launch_us, q) for q in (0.1, 0.5, 0.9)],
                "warm_avg_launch_us": warm_ms * 1e3,
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "whole_call": {"achieved": call_achieved, "frac": call_achieved / peak,
                               "avg_call_us": call_ms * 1e3,
                               "timed": "region over the steps, calls chained back to back",
                               "period_us_p10_median_p90": q3(chained_period_us),
                               "frac_median_period": w.algorithmic_bytes / (period_med / 1e6) / 1e9 / peak},
                "chained": {"calls": STAT_CALLS,
                            "timed": ("device global-timer stamps of calls chained back to back "
                                      "(spec_arm_timer): first streaming-CTA start, last streaming-CTA "
                                      "end, last output"),
                            "row_kernel_us_p10_median_p90": q3(chained_row_us),
                            "row_kernel_frac_median": w.algorithmic_bytes / (row_med / 1e6) / 1e9 / peak,
                            "call_device_us_p10_median_p90": q3(chained_call_us),
                            "period_us_p10_median_p90": q3(chained_period_us)}}
    if w.T > 0:  # one MUFU ex2 per streamed logit
        exps = w.algorithmic_bytes / (4 if w.dtype == "f32" else 2)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = (clk or {}).get("sm_mhz") or (clk or {}).get("sm_max_mhz") or 2070.0
        exp_peak = sms * EX2_PER_SM_CLOCK * mhz * 1e6
        roofline["exp"] = {"per_s": exps / (avg_launch_ms / 1e3), "peak_per_s": exp_peak,
                           "frac": exps / (avg_launch_ms / 1e3) / exp_peak,
                           "peak_basis": f"{sms} SMs x {EX2_PER_SM_CLOCK} ex2 per clock x {mhz:.0f} MHz"}
    # CPU baseline: the oracle as it stands on the host cores, bounded sample
    cpu = None
    if not args.no_cpu_baseline:
        nseq = w.B
        secs, threads = time_oracle(w, nseq)
        reps = 1
        while secs * reps < 3.0 and reps < 8:
            more, _ = time_oracle(w, nseq)
            secs += more
            reps += 1
        per_seq = w.positions // w.B
        n1 = min(w.B, 16)
        secs1, _ = time_oracle(w, n1, nthreads=1)
        cpu = {"value": nseq * reps * per_seq / secs, "unit": UNIT, "cores": threads,
               "kind": "oracle",
               "sample": f"{reps} pass(es) over the {nseq} sequences of {w.name}, fp64 oracle",
               "one_core": {"value": n1 * per_seq / secs1, "unit": UNIT,
                            "sample": f"the first {n1} sequences of {w.name}, one thread"},
               "cpu_model": _cpu_model(), "nproc": os.cpu_count()}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": region_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": chain_config(w, ws),
        "roofline": roofline,
        "achieved_hbm_gbs": achieved,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * LAUNCHES_PER_CALL,
        "clocks": clk,
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# n-gram drafting workloads (ng1, ng2): one spec_ngram_propose call per step
# ----------------------------------------------------------------------------
NGRAM_METRIC = "n-gram drafts/sec (sequences drafted from their context), 1 GPU"
NGRAM_UNIT = "sequences/s"
NGRAM_BATCH = 10          # calls per chained-latency sample
NGRAM_FLOOR_US = 2.0      # 3 dependent round trips x ~0.6 us, plus one cluster barrier


def _ngram_bytes(lengths_host, K):
    """Algorithmic bytes of one call: every context token once, the lengths,
    the drafts and counts."""
    B = len(lengths_host)
    return 4 * int(lengths_host.sum()) + 4 * B + 4 * B * (K + 1)


def time_ngram_oracle(w, tokens_h, lengths_h, min_seconds):
    import oracle
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.ngram_propose(tokens_h, lengths_h, w.n_min, w.n_max, w.K, min_hits=w.min_hits)
        reps += 1
        secs = time.perf_counter() - t0
        if secs >= min_seconds:
            return secs, reps


def ngram_describe(w):
    return (f"n-gram drafting B={w.B} contexts of up to L={w.L} tokens (lengths uniform in [L/2, L]), "
            f"n in [{w.n_min}, {w.n_max}], min_hits={w.min_hits}, K={w.K}")


def ngram_config(w, ws, lengths_h):
    """The config of an n-gram workload's line, the same for both arms."""
    from sampling_row_online_gb300.workloads import input_copies_for_cold_l2
    alg = _ngram_bytes(lengths_h, w.K)
    ncopies = input_copies_for_cold_l2(alg)
    return {"workload": f"{w.name}: {ngram_describe(w)}", "per_rank_batch": w.B,
            "context_tokens_per_step": int(lengths_h.sum()),
            "parallelism": f"replicas x{ws} (sequences sharded, no collective)",
            "l2": f"rotating {ncopies} context copies ({ncopies * alg / 1e6:.0f} MB > 2x L2)"}


def run_reference_ngram(args, w):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    from sampling_row_online_gb300.workloads import make_contexts
    tokens, lengths = make_contexts(w, "cpu")
    th, lh = tokens.numpy(), lengths.numpy()
    for _ in range(max(0, args.warmup)):
        time_ngram_oracle(w, th, lh, 0.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_ngram_oracle(w, th, lh, 0.0)
    secs = time.perf_counter() - t0
    value = args.steps * w.B / secs
    line = {
        "metric": NGRAM_METRIC, "value": value, "unit": NGRAM_UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic", "impl": "reference",
        "config": ngram_config(w, ws, lh),
        "cpu_baseline": {"value": value, "unit": NGRAM_UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} passes over the {w.B} contexts of {w.name}, oracle, 1 thread"},
        "e2e": {"value": value, "unit": NGRAM_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu_ngram(args, w):
    import torch
    import torch.distributed as dist
    from sampling_row_online_gb300 import binding
    from sampling_row_online_gb300.workloads import input_copies_for_cold_l2, make_contexts
    ws, rank, local = _dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    lib = binding.library()
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    # generated on the host (the reference arm's contexts, bit for bit), then copied
    tokens, lengths = make_contexts(w, "cpu", seed=w.data_seed + 7919 * rank)
    tokens, lengths = tokens.to(dev), lengths.to(dev)
    lengths_h = lengths.cpu().numpy()
    alg = _ngram_bytes(lengths_h, w.K)
    ncopies = input_copies_for_cold_l2(alg)
    copies = [tokens] + [tokens.clone() for _ in range(ncopies - 1)]
    draft = torch.empty((w.B, w.K), dtype=torch.int32, device=dev)
    count = torch.empty((w.B,), dtype=torch.int32, device=dev)

    def make_call(t):
        a = (ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(lengths.data_ptr()), w.B, w.L, w.n_min, w.n_max,
             w.min_hits, w.K, ctypes.c_void_p(draft.data_ptr()), ctypes.c_void_p(count.data_ptr()), sp)
        return lambda: lib.spec_ngram_propose(*a)

    calls = [make_call(t) for t in copies]
    for k in range(max(3, args.warmup)):
        st = calls[k % ncopies]()
        if st != 0:
            raise SystemExit(f"spec_ngram_propose failed: {st} {lib.spec_last_error_message().decode()}")
    torch.cuda.synchronize()
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error during warm-up")
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    wall0 = time.perf_counter()
    t_start.record(stream)
    for k in range(args.steps):
        calls[k % ncopies]()
    t_end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if ws > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error in the timed region")
    region_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
    call_ms = region_ms / args.steps
    # the kernel alone: events around single calls (STAT_CALLS of them)
    n_one = STAT_CALLS
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_one)]
    for k in range(n_one):
        ev[k][0].record(stream)
        calls[k % ncopies]()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    avg_launch_ms = max_over_ranks(statistics.fmean(a.elapsed_time(b) for a, b in ev), dev)
    one_us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
    # chained latency: STAT_CALLS batches of NGRAM_BATCH calls back to back,
    # events around each batch (the call time inside a decode loop)
    evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_one)]
    for k in range(n_one):
        evb[k][0].record(stream)
        for j in range(NGRAM_BATCH):
            calls[(k + j) % ncopies]()
        evb[k][1].record(stream)
    torch.cuda.synchronize()
    chained_us = sorted(a.elapsed_time(b) * 1e3 / NGRAM_BATCH for a, b in evb)
    value = w.B * args.steps * ws / (region_ms / 1e3)

    # end to end through the binding: contexts copied in from pinned host
    # memory, drafts and counts copied out, every step
    e2e = None
    if not args.no_e2e:
        th = tokens.cpu().pin_memory()
        lh = lengths.cpu().pin_memory()
        dh = torch.empty((w.B, w.K), dtype=torch.int32, pin_memory=True)
        ch = torch.empty((w.B,), dtype=torch.int32, pin_memory=True)
        td = torch.empty_like(tokens)
        ld = torch.empty_like(lengths)
        e_steps = max(5, min(args.steps, 50))

        def e2e_step():
            td.copy_(th, non_blocking=True)
            ld.copy_(lh, non_blocking=True)
            binding.spec_ngram_propose(td, ld, w.n_min, w.n_max, w.K, min_hits=w.min_hits, out_draft=draft,
                                       out_count=count)
            dh.copy_(draft, non_blocking=True)
            ch.copy_(count, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            e2e_step()
        if ws > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(e_steps):
            e2e_step()
        e_sec = max_over_ranks(time.perf_counter() - t0, dev)
        e2e = {"value": w.B * e_steps * ws / e_sec, "unit": NGRAM_UNIT,
               "h2d_bytes_per_step": th.numel() * 4 + lh.numel() * 4,
               "d2h_bytes_per_step": dh.numel() * 4 + ch.numel() * 4}
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = _peaks()
    kernel = "ngram_kernel"
    achieved = alg / (avg_launch_ms / 1e3) / 1e9
    call_achieved = alg / (call_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} hbm_gbs", "traffic": _profile_traffic(kernel, w.name),
                "kernel": kernel,
                "timed": f"single calls bracketed by CUDA events on the call's stream, mean of {n_one}",
                "algorithmic_bytes_per_launch": alg, "avg_launch_us": avg_launch_ms * 1e3,
                "whole_call": {"achieved": call_achieved, "frac": call_achieved / peak,
                               "avg_call_us": call_ms * 1e3,
                               "timed": "region over the steps, calls chained back to back"}}
    cpu = None
    if not args.no_cpu_baseline:
        th_np, lh_np = tokens.cpu().numpy(), lengths_h
        secs, reps = time_ngram_oracle(w, th_np, lh_np, 3.0)
        cpu = {"value": w.B * reps / secs, "unit": NGRAM_UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{reps} passes over the {w.B} contexts of {w.name}, oracle, 1 thread"}
    q3 = lambda v: [_quantile(v, q) for q in (0.1, 0.5, 0.9)]
    latency = {"unit": "us per call",
               "chained_p10_median_p90": q3(chained_us),
               "standalone_p10_median_p90": q3(one_us),
               "floor_us": NGRAM_FLOOR_US,
               "floor_basis": ("3 dependent global round trips of the kernel (lengths; context and "
                               "suffix; the draft's tokens) x ~0.6 us idle L2/HBM round trip on GB300, "
                               "plus one cluster barrier (the G <= 8 CTAs of a sequence combine on chip)"),
               "timed": (f"chained: {n_one} batches of {NGRAM_BATCH} calls back to back between CUDA "
                         f"events; standalone: {n_one} calls each between CUDA events (includes "
                         f"the ~4 us fixed cost of a launch between two events)")}
    line = {
        "metric": NGRAM_METRIC, "latency": latency, "value": value, "unit": NGRAM_UNIT, "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": call_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": ngram_config(w, ws, lengths_h),
        "context_tokens_per_s": int(lengths_h.sum()) * args.steps * ws / (region_ms / 1e3),
        "roofline": roofline, "achieved_hbm_gbs": achieved, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps, "clocks": clk, "wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


# ----------------------------------------------------------------------------
# EAGLE-2 tree budget (eg1): one budget build (all expansion steps and the
# rerank) for a batch of trees per step
# ----------------------------------------------------------------------------
EAGLE_METRIC = "EAGLE-2 draft trees built/sec (expansion steps + rerank, draft rows resident), 1 GPU"
EAGLE_UNIT = "trees/s"


def eagle_describe(w):
    return (f"EAGLE-2 budget B={w.B} trees, V={w.V} {w.dtype} draft rows, T={w.T}, k={w.k} candidates per node, "
            f"{w.k} nodes grown per step, depth {w.depth}, rerank keeps {w.m}")


def _eagle_bytes(w):
    rows = sum(w.frontier_size(d) for d in range(w.depth))
    return w.B * rows * w.V * (4 if w.dtype == "f32" else 2)


def _eagle_oracle_build(w, rows, B):
    """The oracle's budget build over per-step rows [B, F, V] (CPU tensors)."""
    import numpy as np
    import oracle
    tok = np.zeros((B, w.M), np.int32)
    val = np.zeros((B, w.M), np.float64)
    par = np.zeros((B, w.M), np.int32)
    val[:, 0], par[:, 0] = 1.0, -1
    frontier = np.zeros((B, 1), np.int32)
    for d in range(w.depth):
        F = w.frontier_size(d)
        tt, tp = oracle.topk_prob(rows[d][:B].reshape(B * F, w.V), w.k, w.T)
        kn = w.k if d < w.depth - 1 else 0
        frontier, _ = oracle.eagle2_expand(frontier, tt.reshape(B, F, w.k), tp.reshape(B, F, w.k), tok, val, par,
                                           w.offset(d), kn)
    return oracle.eagle2_rerank(val, par, tok, w.m)


def eagle_config(w, ws):
    """The config of an EAGLE-2 workload's line, the same for both arms."""
    alg = _eagle_bytes(w)
    return {"workload": f"{w.name}: {eagle_describe(w)}", "per_rank_batch": w.B,
            "parallelism": f"replicas x{ws} (trees sharded, no collective)",
            "l2": f"draft rows of one build {alg / 1e6:.0f} MB (> 2x L2), read once per build"}


def run_reference_eagle2(args, w):
    ws, rank, _ = _dist_env()
    if rank != 0:
        return 0
    from sampling_row_online_gb300.workloads import eagle2_step_rows
    nb = 2  # trees per step: a bounded sample of the batch
    rows = [eagle2_step_rows(w, d, "cpu")[:nb].contiguous() for d in range(w.depth)]
    for _ in range(max(0, args.warmup)):
        _eagle_oracle_build(w, rows, nb)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _eagle_oracle_build(w, rows, nb)
    secs = time.perf_counter() - t0
    value = args.steps * nb / secs
    line = {
        "metric": EAGLE_METRIC, "value": value, "unit": EAGLE_UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": eagle_config(w, ws),
        "cpu_baseline": {"value": value, "unit": EAGLE_UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} builds of {nb} trees of {w.name}, oracle, 1 thread"},
        "e2e": {"value": value, "unit": EAGLE_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu_eagle2(args, w):
    import torch
    import torch.distributed as dist
    from sampling_row_online_gb300 import binding
    from sampling_row_online_gb300.workloads import eagle2_step_rows
    ws, rank, local = _dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    lib = binding.library()
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    vp = ctypes.c_void_p
    B, M = w.B, w.M
    rows = [eagle2_step_rows(w, d, dev) for d in range(w.depth)]   # > 2x L2 in total
    tok = torch.zeros((B, M), dtype=torch.int32, device=dev)
    val = torch.zeros((B, M), dtype=torch.float32, device=dev)
    par = torch.zeros((B, M), dtype=torch.int32, device=dev)
    val[:, 0], par[:, 0] = 1.0, -1
    fronts = [torch.zeros((B, 1), dtype=torch.int32, device=dev)] + \
             [torch.empty((B, w.k), dtype=torch.int32, device=dev) for _ in range(w.depth)]
    out = [torch.empty((B, w.m + 1), dtype=torch.int32, device=dev) for _ in range(3)]
    dt = 0 if w.dtype == "f32" else 1
    calls = []
    for d in range(w.depth):
        F = w.frontier_size(d)
        kn = w.k if d < w.depth - 1 else 0
        a = (vp(rows[d].data_ptr()), vp(fronts[d].data_ptr()), B, F, w.V, dt, ctypes.c_float(w.T), w.k,
             vp(tok.data_ptr()), vp(val.data_ptr()), vp(par.data_ptr()), M, w.offset(d), kn,
             vp(fronts[d + 1].data_ptr()), sp)
        calls.append(lambda a=a: lib.spec_eagle2_expand(*a))
    ra = (vp(val.data_ptr()), vp(par.data_ptr()), vp(tok.data_ptr()), B, M, w.m, vp(out[0].data_ptr()),
          vp(out[1].data_ptr()), vp(out[2].data_ptr()), sp)
    calls.append(lambda: lib.spec_eagle2_rerank(*ra))

    def step():
        for c in calls:
            st = c()
            if st != 0:
                raise SystemExit(f"EAGLE-2 call failed: {st} {lib.spec_last_error_message().decode()}")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error during warm-up")
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    wall0 = time.perf_counter()
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if ws > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error in the timed region")
    region_ms = max_over_ranks(t_start.elapsed_time(t_end), dev)
    step_ms = region_ms / args.steps
    value = B * args.steps * ws / (region_ms / 1e3)
    # the dominant kernel alone: spec_topk over the rows of one full step, the
    # calls rotating over the four full steps' rows (4 x 65.7 MB > 2x L2), so
    # each call's rows were last read 197 MB of reads earlier
    ttk = torch.empty((B * w.k, w.k), dtype=torch.int32, device=dev)
    tpk = torch.empty((B * w.k, w.k), dtype=torch.float32, device=dev)
    tas = [(vp(r.data_ptr()), B * w.k, w.V, dt, ctypes.c_float(w.T), w.k, vp(ttk.data_ptr()), vp(tpk.data_ptr()), sp)
           for r in rows[1:]]
    n_one = STAT_CALLS
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_one)]
    for k in range(len(tas)):   # one untimed pass over the copies
        lib.spec_topk(*tas[k])
    for k in range(n_one):
        ev[k][0].record(stream)
        lib.spec_topk(*tas[k % len(tas)])
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    one_ms = [a.elapsed_time(b) for a, b in ev]
    avg_launch_ms = max_over_ranks(statistics.fmean(one_ms), dev)
    med_launch_ms = max_over_ranks(statistics.median(one_ms), dev)
    # the same calls chained back to back, each with device stamps
    # (spec_arm_timer: no stream operation between the launches): the
    # kernel's time as it runs in the chain, and the start-to-start period
    import numpy as np
    tst = torch.empty((STAT_CALLS, 3), dtype=torch.int64, device=dev)
    tst[:, 0] = -1
    tst[:, 1:] = 0
    torch.cuda.synchronize()
    for k in range(STAT_CALLS):
        lib.spec_arm_timer(ctypes.c_void_p(tst[k].data_ptr()))
        lib.spec_topk(*tas[k % len(tas)])
    torch.cuda.synchronize()
    if lib.spec_get_status(sp) != 0:
        raise SystemExit("device status error in the chained top-k loop")
    ts = tst.cpu().numpy().view(np.uint64).astype(np.float64)
    ch_kernel_us = sorted(((ts[:, 1] - ts[:, 0]) / 1e3).tolist())
    ch_period_us = sorted(((ts[1:, 0] - ts[:-1, 0]) / 1e3).tolist())
    topk_bytes = B * w.k * w.V * (4 if w.dtype == "f32" else 2)

    e2e = None
    if not args.no_e2e:
        hrows = [r.cpu().pin_memory() for r in rows]
        drows = [torch.empty_like(r) for r in rows]
        hout = [torch.empty((B, w.m + 1), dtype=torch.int32, pin_memory=True) for _ in range(3)]
        e_calls = []
        for d in range(w.depth):
            F = w.frontier_size(d)
            kn = w.k if d < w.depth - 1 else 0
            a = (vp(drows[d].data_ptr()), vp(fronts[d].data_ptr()), B, F, w.V, dt, ctypes.c_float(w.T), w.k,
                 vp(tok.data_ptr()), vp(val.data_ptr()), vp(par.data_ptr()), M, w.offset(d), kn,
                 vp(fronts[d + 1].data_ptr()), sp)
            e_calls.append((d, a))

        def e2e_step():
            for d, a in e_calls:
                drows[d].copy_(hrows[d], non_blocking=True)
                lib.spec_eagle2_expand(*a)
            lib.spec_eagle2_rerank(*ra)
            for h, o in zip(hout, out):
                h.copy_(o, non_blocking=True)
            stream.synchronize()

        for _ in range(2):
            e2e_step()
        e_steps = max(3, min(args.steps, 20))
        t0 = time.perf_counter()
        for _ in range(e_steps):
            e2e_step()
        e_sec = max_over_ranks(time.perf_counter() - t0, dev)
        e2e = {"value": B * e_steps * ws / e_sec, "unit": EAGLE_UNIT,
               "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in hrows),
               "d2h_bytes_per_step": sum(h.numel() * 4 for h in hout)}
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0
    peak, peak_kind = _peaks()
    kernel = "topk_kernel"
    achieved = topk_bytes / (avg_launch_ms / 1e3) / 1e9

    def pct(v, q):
        return v[min(len(v) - 1, int(q * (len(v) - 1) + 0.5))]

    ch_med = pct(ch_kernel_us, 0.5)
    chained = {"kernel_us_p10_median_p90": [pct(ch_kernel_us, 0.1), ch_med, pct(ch_kernel_us, 0.9)],
               "achieved": topk_bytes / (ch_med / 1e6) / 1e9, "frac": topk_bytes / (ch_med / 1e6) / 1e9 / peak,
               "period_us_p10_median_p90": [pct(ch_period_us, 0.1), pct(ch_period_us, 0.5), pct(ch_period_us, 0.9)],
               "timed": (f"{STAT_CALLS} spec_topk calls chained back to back over the same rotating rows, "
                         "device global-timer stamps (spec_arm_timer): first CTA start to last CTA end, "
                         "and start-to-start period")}
    alg = _eagle_bytes(w)
    step_achieved = alg / (step_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} hbm_gbs", "traffic": _profile_traffic(kernel, w.name), "kernel": kernel,
                "timed": (f"spec_topk over one full step's rows ({B * w.k} rows of {w.V}), single calls bracketed "
                          f"by CUDA events, rotating over the {len(tas)} full steps' rows (> 2x L2), "
                          f"mean of {n_one}"),
                "algorithmic_bytes_per_launch": topk_bytes, "avg_launch_us": avg_launch_ms * 1e3,
                "median_launch_us": med_launch_ms * 1e3,
                "frac_median": topk_bytes / (med_launch_ms / 1e3) / 1e9 / peak,
                "chained": chained,
                "whole_step": {"achieved": step_achieved, "frac": step_achieved / peak, "avg_step_us": step_ms * 1e3,
                               "algorithmic_bytes": alg,
                               "timed": "region over the steps (all expansion calls and the rerank), back to back"}}
    cpu = None
    if not args.no_cpu_baseline:
        nb = 2
        hr = [r[:nb].cpu() for r in rows]
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 3.0:
            _eagle_oracle_build(w, hr, nb)
            reps += 1
        secs = time.perf_counter() - t0
        cpu = {"value": nb * reps / secs, "unit": EAGLE_UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{reps} builds of {nb} trees of {w.name} on the same rows, oracle, 1 thread"}
    line = {
        "metric": EAGLE_METRIC, "value": value, "unit": EAGLE_UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": eagle_config(w, ws),
        "roofline": roofline, "achieved_hbm_gbs": achieved, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps * (2 * w.depth + 1), "clocks": clk, "wall_s": wall,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="c1", choices=["c0", "c1", "c2", "c3", "c4", "c3s", "ng1", "ng2", "eg1"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args(argv)
    from sampling_row_online_gb300.workloads import EAGLE2_WORKLOADS, NGRAM_WORKLOADS, WORKLOADS
    if args.workload in EAGLE2_WORKLOADS:
        w = EAGLE2_WORKLOADS[args.workload]
        return run_reference_eagle2(args, w) if args.impl == "reference" else run_gpu_eagle2(args, w)
    if args.workload in NGRAM_WORKLOADS:
        w = NGRAM_WORKLOADS[args.workload]
        return run_reference_ngram(args, w) if args.impl == "reference" else run_gpu_ngram(args, w)
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    sys.exit(main())
