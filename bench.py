#!/usr/bin/env python
"""Benchmark of the lightning-indexer logits call on GB300.

One step = one indexer_logits call (the whole hot path: schedule, TMA loads,
tcgen05 MMA, ReLU.w head reduction, masked store and -inf clean) over one
synthetic workload resident in HBM. Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--split replicas|rows] [--zero-inputs]

Default workload: MXFP8 S_q=8192, S_kv=65536 (the largest single-GPU
configuration; DeepGEMM's MX logits numbers are quoted on this shape).

Timing: W untimed warm-up calls; then K calls, each preceded by an untimed
256 MiB write that flushes L2, each bracketed by CUDA events on the launch
stream; barrier + synchronize around the timed region; max over ranks.
`value` is in-window TFLOP/s = 2*H*D*(sum of window lengths) / time, for all
ranks together. `protocol` repeats the measurement the way DeepGEMM's MX
reproducer times its kernel: each sample is 5 back-to-back calls into 5
distinct output buffers between one pair of events (L2 flushed before the
sample), 40 samples with the buffer order rotated, median/p10/p90 per call;
`protocol_zero_inputs` does the same on all-zero Q/K/W with unit MX scales,
the inputs DeepGEMM times. `e2e` measures the same call end to end from
pinned host memory: inputs copied in and logits copied out inside the timed
region, on three streams (copy in / compute / copy out) with two device
buffer sets, so step i+1's inputs and step i-1's logits move while step i
computes. `--impl reference` times the float64 CPU oracle on bounded row
samples of the same workload.

Multi-GPU (torchrun, one process per GPU): `--split replicas` (default) runs
the whole workload on every rank (weak scaling); `--split rows` splits the
query rows of ONE problem across the ranks, balanced by in-window work, each
rank with the keys whole and its own output rows (strong scaling, no
collective on the data path).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("indexer logits µs/call and in-window TFLOP/s; "
          "% of GB300 dense tensor peak")
DEFAULT_WORKLOAD = "mxfp8_8192x65536"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DTYPES = {0: "bf16", 1: "e4m3", 2: "mxfp8(e4m3+e8m0)", 3: "mxfp4(e2m1+e8m0)"}
# dense tensor peak of a format relative to BF16 (nominal GB300 ratios)
FMT_PEAK_RATIO = {0: 1.0, 1: 2.0, 2: 2.0, 3: 6.0}
L2_FLUSH_BYTES = 256 << 20
# Files that define the logits kernel: a DRAM-traffic figure taken with ncu
# (profiles/) is reported as roofline.traffic only while these still hash to
# the digest it was taken on.
KERNEL_FILES = ("indexer_kernel.cuh", "ptx.cuh", "plan_kernel.cuh", "page_div.h")
# DRAM bytes (read + write) of one logits-kernel launch from an ncu capture,
# keyed by workload, with the kernel-source digest it was taken on.
PROFILED_TRAFFIC = {
    "bf16_batched_causal_4096": ("b9ac376f7fef89a9", 137480960 + 79439872),
    "fp8_per_token_2048x32768": ("b9ac376f7fef89a9", 21690112 + 207621120),
    "mxfp8_2048x32768": ("b9ac376f7fef89a9", 22220544 + 207505664),
    "mxfp4_2048x32768": ("b9ac376f7fef89a9", 11735040 + 207220736),
    "paged_fp8_decode_64x2_32768": ("b9ac376f7fef89a9", 208141568 + 7877120),
    "mxfp8_8192x65536": ("b9ac376f7fef89a9", 80191232 + 2086541312),
    "mxfp4_8192x65536": ("b9ac376f7fef89a9", 42626304 + 2086549248),
    "mxfp4_irregular_8192x65536": ("b9ac376f7fef89a9", 44206336 + 2086041600),
    "thd_bf16_3seq_8192x32768": ("b9ac376f7fef89a9", 144901888 + 1012543232),
}


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or the machine type."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def kernel_source_digest() -> str:
    """Digest of the sources that define the logits kernel."""
    import hashlib
    d = os.path.join(ROOT, "infra_dsa_indexer_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_FILES:
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--split", choices=["replicas", "rows"], default="replicas",
                    help="multi-GPU: whole problem per rank, or one problem's rows split")
    ap.add_argument("--zero-inputs", action="store_true",
                    help="time all-zero Q/K/W (unit MX scales) in the main measurement too")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--protocol-samples", type=int, default=40)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: CPU seconds all its steps together aim for")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-protocol", action="store_true")
    ap.add_argument("--topk", type=int, default=0,
                    help="also time indexer_topk (k columns per row) on the call's logits")
    ap.add_argument("--fused-topk", type=int, default=0,
                    help="also time indexer_logits_topk (k columns per row, no logits written) "
                         "against indexer_logits + indexer_topk")
    ap.add_argument("--out-bf16", action="store_true",
                    help="write the logits as BF16 (IDX_FLAG_OUT_BF16) instead of FP32")
    return ap.parse_args(argv)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; weak scaling, no collective on
# the data path: every rank runs the whole workload on its own GPU)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend or "nccl")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 - 0.05 <= ts <= t1 + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded row sample)
# ---------------------------------------------------------------------------

def oracle_sample_rate(case, seconds, rng_seed=0):
    """Time the float64 oracle on a row sample of about `seconds`; return
    (in-window TFLOP/s, threads, sample description)."""
    import oracle
    nth = oracle.num_threads()
    rng = np.random.default_rng(rng_seed)
    total_rows = case.B * case.S
    lo = np.clip(case.ks.reshape(-1).astype(np.int64), 0, case.N)
    hi = np.clip(case.ke.reshape(-1).astype(np.int64), 0, case.N)
    pairs = np.maximum(hi - lo, 0)

    def run(rows):
        t0 = time.perf_counter()
        oracle.logits(case.fmt, case.q, case.k, case.w, case.ks, case.ke, case.sm_scale,
                      q_sf=case.q_sf, k_sf=case.k_sf, k_tok=case.k_tok, w_fmt=case.w_fmt,
                      rows=rows, want_den=False, nthreads=nth)
        return time.perf_counter() - t0

    # calibrate on a probe large enough that thread start-up does not dominate
    probe = rng.choice(total_rows, size=min(total_rows, 8 * nth), replace=False)
    dt = run(probe)
    rate = max(pairs[probe].sum(), 1) / max(dt, 1e-6)       # pairs per second
    n = int(min(total_rows, max(nth, seconds * rate / max(pairs.mean(), 1))))
    rows = np.sort(rng.choice(total_rows, size=n, replace=False))
    dt = run(rows)
    flops = 2.0 * case.H * case.D * pairs[rows].sum()
    desc = (f"{n} of {total_rows} rows drawn uniformly (seed {rng_seed}), "
            f"{pairs[rows].sum()} in-window pairs, {dt:.1f} s")
    return flops / dt / 1e12, nth, desc


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, _dist):
    """The float64 CPU oracle on row samples (rank 0 only)."""
    from infra_dsa_indexer_gb300 import synth
    case = synth.make_workload(args.workload)
    import oracle
    oracle.build()
    budget = args.ref_seconds / max(1, args.steps + args.warmup)   # seconds per step
    nth = oracle.num_threads()
    lo = np.clip(case.ks.reshape(-1).astype(np.int64), 0, case.N)
    hi = np.clip(case.ke.reshape(-1).astype(np.int64), 0, case.N)
    pairs = np.maximum(hi - lo, 0)
    rng = np.random.default_rng(0)
    total_rows = case.B * case.S

    def step(nrows):
        rows = np.sort(rng.choice(total_rows, size=nrows, replace=False))
        t0 = time.perf_counter()
        oracle.logits(case.fmt, case.q, case.k, case.w, case.ks, case.ke, case.sm_scale,
                      q_sf=case.q_sf, k_sf=case.k_sf, k_tok=case.k_tok, w_fmt=case.w_fmt,
                      rows=rows, want_den=False, nthreads=nth)
        return time.perf_counter() - t0, pairs[rows].sum()

    dt, pr = step(min(total_rows, nth))
    rate = max(pr, 1) / max(dt, 1e-6)
    nrows = int(max(1, min(total_rows, budget * rate / max(pairs.mean(), 1))))
    for _ in range(args.warmup):
        step(nrows)
    tot_t, tot_p = 0.0, 0
    for _ in range(args.steps):
        dt, pr = step(nrows)
        tot_t += dt
        tot_p += pr
    value = 2.0 * case.H * case.D * tot_p / tot_t / 1e12
    sample = (f"{nrows} uniformly drawn rows per step of {total_rows}; ms_per_step is scaled "
              f"to the whole workload by in-window pairs ({tot_p / args.steps:.0f} sampled "
              f"of {int(pairs.sum())} per step)")
    sample_ms = 1e3 * tot_t / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sample_ms * max(int(pairs.sum()), 1) / max(tot_p / args.steps, 1.0),
        "sample_ms_per_step": sample_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(case, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
                         "sample": sample, "cpu_model": host_cpu_model()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(case, args):
    from infra_dsa_indexer_gb300 import synth
    split = getattr(args, "split", "replicas")
    return {"workload": args.workload, "B": case.B, "S_q": case.S, "S_kv": case.N,
            "H": case.H, "D": case.D, "format": synth.FMT_NAMES[case.fmt],
            "w_format": "bf16" if case.w_fmt == synth.W_BF16 else "f32",
            "in_window_pairs": case.in_window_pairs(), "clean": bool(case.clean),
            "group_rows": bool(case.group_rows),
            "out_format": "bf16" if getattr(args, "out_bf16", False) else "f32",
            "inputs": "all-zero (unit MX scales)" if getattr(args, "zero_inputs", False)
                      else "seeded N(0,1), quantised",
            "l2": "flushed before every timed call (256 MiB write)",
            "parallelism": (f"query-row split x{args.gpus}" if split == "rows"
                            else f"replicas x{args.gpus}")}


def zero_inputs_(t):
    """All-zero Q/K/W with unit MX scales (E8M0 0x7f) and unit per-key FP8
    scales, in place: the inputs DeepGEMM's reproducer times."""
    for key in ("q", "k", "w"):
        t[key].zero_()
    for key in ("q_sf", "k_sf"):
        if t.get(key) is not None:
            t[key].fill_(0x7F)
    if t.get("k_scales") is not None:
        t["k_scales"].fill_(1.0)


def _pct(sorted_vals, q):
    return sorted_vals[int(q * (len(sorted_vals) - 1))]


def run_ours(args, dist):
    import torch
    from infra_dsa_indexer_gb300 import binding, split, synth
    from infra_dsa_indexer_gb300 import build as lib_build

    dev = dist.local_rank
    torch.cuda.set_device(dev)
    if dist.rank == 0:
        lib_build.build()
    dist.barrier()
    binding.load()
    case = synth.make_workload(args.workload)
    flops_total = case.in_window_flops()
    t = binding.case_to_device(case, device=f"cuda:{dev}", out_bf16=args.out_bf16)
    if args.zero_inputs:
        zero_inputs_(t)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=f"cuda:{dev}")
    launches_per_call = binding.indexer_launches_per_call(t["shape"])

    # What this rank computes in one step: the whole problem (replicas), or
    # its query rows of the one problem (rows; one B=1 call per batch slice).
    if args.split == "rows" and dist.world > 1:
        if case.page_size:
            raise SystemExit("--split rows covers contiguous keys only")
        mine = split.row_split(case.ks, case.ke, case.N, dist.world)[dist.rank]
        views = []
        for b, s0, s1 in mine:
            v = split.slice_tensors(t, b, s0, s1)
            v["shape"] = binding.make_shape(1, s1 - s0, case.N, case.H, case.D, case.fmt,
                                            case.w_fmt, out_row_stride=t["shape"].out_row_stride,
                                            flags=t["shape"].flags)
            views.append(v)
        lo = np.clip(case.ks.astype(np.int64), 0, case.N)
        hi = np.clip(case.ke.astype(np.int64), 0, case.N)
        pairs = np.maximum(hi - lo, 0)
        my_pairs = sum(int(pairs[b, s0:s1].sum()) for b, s0, s1 in mine)
        flops_rank = 2.0 * case.H * case.D * my_pairs
        flops_all = flops_total                       # one problem, split
        scaling = "strong"
    else:
        views = [t]
        flops_rank = flops_total
        flops_all = dist.world * flops_total          # one problem per rank
        scaling = "weak"
    calls_per_step = len(views)

    def step(out=None, st=stream):
        for v in views:
            if out is not None:
                v = dict(v, out=out)
            binding.run_case(case, v, stream=st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = binding.indexer_get_last_error(stream)
    if st != binding.IDX_OK:
        raise RuntimeError(f"device error after warm-up: {binding.indexer_status_string(st)}")

    uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    clocks = ClockSampler(uuid) if dist.rank == 0 else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    time.sleep(0.3 if clocks else 0)
    dist.barrier()
    torch.cuda.synchronize()
    w0 = time.time()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    w1 = time.time()
    clk = clocks.stop(w0, w1) if clocks else None
    st = binding.indexer_get_last_error(stream)
    if st != binding.IDX_OK:
        raise RuntimeError(f"device error in timed region: {binding.indexer_status_string(st)}")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]      # ms, one step each
    ms_local = sum(per) / len(per)
    ms = dist.max(ms_local, device=f"cuda:{dev}")
    value = flops_all / (ms * 1e-3) / 1e12

    # --- DeepGEMM-style protocol: 5 calls into 5 distinct outputs per sample
    def protocol():
        if args.no_protocol or len(views) != 1:
            return None
        outs = [t["out"]] + [torch.empty_like(t["out"]) for _ in range(4)]
        for o in outs:
            step(out=o)
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.protocol_samples)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.protocol_samples)]
        torch.cuda.synchronize()
        for smp in range(args.protocol_samples):
            flush.fill_(float(smp))
            e0[smp].record(stream)
            for c in range(len(outs)):
                step(out=outs[(smp + c) % len(outs)])
            e1[smp].record(stream)
        torch.cuda.synchronize()
        us = sorted(1e3 * a.elapsed_time(b) / len(outs) for a, b in zip(e0, e1))
        med = statistics.median(us)
        del outs
        return {"calls_per_sample": 5, "samples": args.protocol_samples,
                "distinct_outputs": 5, "us_per_call_median": med,
                "us_per_call_p10": _pct(us, 0.1), "us_per_call_p90": _pct(us, 0.9),
                "tflops_median": flops_rank / (med * 1e-6) / 1e12}

    prot = protocol()

    # --- top-k over the logits of the call (its own launches and events)
    topk = None
    if args.topk and len(views) == 1:
        idx = torch.empty(case.B, case.S, args.topk, dtype=torch.int32, device=f"cuda:{dev}")
        for _ in range(3):
            binding.indexer_topk(t["out"], args.topk, idx=idx, n=case.N, stream=stream)
        torch.cuda.synchronize()
        k_st = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        k_en = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(float(i))
            k_st[i].record(stream)
            binding.indexer_topk(t["out"], args.topk, idx=idx, n=case.N, stream=stream)
            k_en[i].record(stream)
        torch.cuda.synchronize()
        k_ms = statistics.mean(s.elapsed_time(e) for s, e in zip(k_st, k_en))
        k_bytes = t["out"].numel() * t["out"].element_size() + idx.numel() * 4
        topk = {"k": args.topk, "us_per_call": 1e3 * k_ms, "kernel": "dsa::topk_rows_kernel",
                "bound": "hbm", "algorithmic_bytes_per_launch": k_bytes,
                "achieved_gbs": k_bytes / (k_ms * 1e-3) / 1e9, "gpu_launches": args.steps}

    # --- the fused call (logits never written) against logits + top-k
    fused = None
    if args.fused_topk and len(views) == 1 and not case.page_size and not args.out_bf16:
        kf = args.fused_topk
        shape_f = binding.make_shape(case.B, case.S, case.N, case.H, case.D, case.fmt,
                                     case.w_fmt,
                                     flags=binding.IDX_FLAG_GROUP_ROWS if case.group_rows else 0)
        ws = torch.empty(binding.indexer_logits_topk_workspace_bytes(shape_f), dtype=torch.uint8,
                         device=f"cuda:{dev}")
        idx_f = torch.empty(case.B * case.S, kf, dtype=torch.int32, device=f"cuda:{dev}")
        idx_s = torch.empty(case.B * case.S, kf, dtype=torch.int32, device=f"cuda:{dev}")

        def fused_call():
            binding.topk_case(case, t, kf, idx=idx_f, workspace=ws, stream=stream)

        def separate_call():
            step()
            binding.indexer_topk(t["out"], kf, idx=idx_s.view(case.B, case.S, kf), n=case.N,
                                 stream=stream)

        res = {}
        for name, fn in (("fused", fused_call), ("logits_then_topk", separate_call)):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            for i in range(args.steps):
                flush.fill_(float(i))
                ev[i][0].record(stream)
                fn()
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            res[name] = statistics.median(1e3 * a.elapsed_time(b) for a, b in ev)
        st_ = binding.indexer_get_last_error(stream)
        if st_ != binding.IDX_OK:
            raise RuntimeError(f"device error in fused top-k: {binding.indexer_status_string(st_)}")
        fused = {"k": kf, "us_per_call_fused": res["fused"],
                 "us_per_call_logits_then_topk": res["logits_then_topk"],
                 "speedup": res["logits_then_topk"] / res["fused"],
                 "workspace_bytes": int(ws.numel()),
                 "launches_fused": 5 + (1 if case.group_rows else 0)}
        del ws

    # --- end to end through the same call: pinned host inputs in, logits out
    def e2e(out_bf16):
        """Three streams (copy in, compute, copy out) over two device buffer
        sets: step i's call overlaps step i+1's input copy and step i-1's
        logits copy. Timed from the first input copy to the last logits copy."""
        keys = [key for key in ("q", "k", "w", "ks", "ke", "q_sf", "k_sf", "k_scales",
                                "block_table") if t.get(key) is not None]
        host = {key: t[key].cpu().pin_memory() for key in keys}
        sets = []
        for i in range(2):
            d = dict(t)
            for key in keys:
                d[key] = t[key] if i == 0 else torch.empty_like(t[key])
            d["out"] = torch.empty(t["out"].shape, device=t["out"].device,
                                   dtype=torch.bfloat16 if out_bf16 else torch.float32)
            d["shape"] = binding.make_shape(
                case.B, case.S, case.N, case.H, case.D, case.fmt, case.w_fmt,
                out_row_stride=t["shape"].out_row_stride,
                flags=(t["shape"].flags & ~binding.IDX_FLAG_OUT_BF16) |
                      (binding.IDX_FLAG_OUT_BF16 if out_bf16 else 0))
            sets.append(d)
        out_host = [torch.empty(sets[0]["out"].shape, dtype=sets[0]["out"].dtype).pin_memory()
                    for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_host[0].numel() * out_host[0].element_size()
        s_in, s_run, s_out = (torch.cuda.Stream() for _ in range(3))
        n = max(3, min(args.e2e_steps, args.steps))
        ev = lambda: torch.cuda.Event()

        def pipeline(steps, e0=None, e1=None):
            in_done = [ev() for _ in range(steps)]
            run_done = [ev() for _ in range(steps)]
            out_done = [ev() for _ in range(steps)]
            if e0 is not None:
                e0.record(s_in)
            for i in range(steps):
                d = sets[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(run_done[i - 2])      # set's inputs no longer read
                    for key in keys:
                        d[key].copy_(host[key], non_blocking=True)
                    in_done[i].record(s_in)
                with torch.cuda.stream(s_run):
                    s_run.wait_event(in_done[i])
                    if i >= 2:
                        s_run.wait_event(out_done[i - 2])     # set's logits copied out
                    binding.run_case(case, d, stream=s_run)
                    run_done[i].record(s_run)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(run_done[i])
                    out_host[i % 2].copy_(d["out"], non_blocking=True)
                    out_done[i].record(s_out)
            if e1 is not None:
                e1.record(s_out)
            torch.cuda.synchronize()

        # Untimed warm-up steps over both buffer sets and both pinned output
        # buffers: the first copies into fresh pinned memory are slower.
        pipeline(max(2, min(args.warmup, 4)))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        dist.barrier()
        torch.cuda.synchronize()
        pipeline(n, e0, e1)
        st_ = binding.indexer_get_last_error(s_run)
        if st_ != binding.IDX_OK:
            raise RuntimeError(f"device error in e2e: {binding.indexer_status_string(st_)}")
        e2e_ms = dist.max(e0.elapsed_time(e1) / n, device=f"cuda:{dev}")
        res = {"value": dist.world * flops_total / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "steps": n, "logits": "bf16" if out_bf16 else "f32",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "host_link_gbs": (h2d + d2h) / (e2e_ms * 1e-3) / 1e9,
               "warmup_steps": max(2, min(args.warmup, 4)),
               "pipeline": "3 streams (copy in / compute / copy out), 2 buffer sets"}
        del sets, out_host, host
        torch.cuda.empty_cache()
        return res

    e2e_main = e2e_bf16 = None
    if not args.no_e2e and len(views) == 1:
        e2e_main = e2e(args.out_bf16)
        if not args.out_bf16:
            e2e_bf16 = e2e(True)

    # --- the protocol again on all-zero inputs (unit MX scales)
    prot_zero = None
    if not args.zero_inputs and prot is not None:
        zero_inputs_(t)
        torch.cuda.synchronize()
        prot_zero = protocol()

    if dist.rank != 0:
        return
    peaks, peak_src = load_peaks()
    if topk is not None:
        topk["peak_gbs"] = peaks["hbm_gbs"]
        topk["frac"] = topk["achieved_gbs"] / peaks["hbm_gbs"]
    peak = peaks["bf16_tflops"] * FMT_PEAK_RATIO[case.fmt]
    achieved = flops_rank / (ms_local * 1e-3) / 1e12
    srt = sorted(per)
    prof = None if (args.out_bf16 or len(views) != 1) else PROFILED_TRAFFIC.get(args.workload)
    traffic = prof[1] if prof and prof[0] == kernel_source_digest() else None
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": (f"{peak_src} bf16 burst x{FMT_PEAK_RATIO[case.fmt]:g} "
                            "(nominal format ratio)" if case.fmt else f"{peak_src} bf16 burst"),
            "kernel": "dsa::indexer_logits_kernel",
            "kernel_source_digest": kernel_source_digest(),
            "algorithmic_flops_per_launch": flops_rank / calls_per_step,
            "hbm_write_gbs": case.B * case.S * case.N * (2 if args.out_bf16 else 4)
                             / (ms_local * 1e-3) / 1e9 * (flops_rank / flops_total),
            "hbm_peak_gbs": peaks["hbm_gbs"]}
    # The three floors of one call: tensor (in-window FLOPs at the format's
    # peak), epilogue FP32 arithmetic (two FP32 lane-ops per in-window
    # (pair, head) -- the ReLU and the weighted add -- at 128 FP32 lanes per
    # SM per cycle at the maximum SM clock: the GB300's FP32 throughput), and
    # HBM (inputs read once plus the logits written once, at the measured copy
    # rate). The largest is the bound a perfect kernel would meet.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_hz = 1e6 * float((clk or {}).get("sm_max_mhz") or 2070.0)
    in_bytes = sum(a.nbytes for a in (case.q, case.k, case.w, case.ks, case.ke, case.q_sf,
                                      case.k_sf, case.k_tok) if a is not None)
    out_bytes = case.B * case.S * case.N * (2 if args.out_bf16 else 4)
    floors = {"tensor_us": 1e6 * flops_rank / (peak * 1e12),
              "epilogue_fp32_us": 1e6 * (flops_rank / (2.0 * case.D)) * 2.0 / (sms * 128 * sm_hz),
              "hbm_us": 1e6 * (in_bytes + out_bytes) / (peaks["hbm_gbs"] * 1e9)}
    bound_name = max(floors, key=floors.get)
    roof["floors"] = floors
    roof["largest_floor"] = bound_name[:-3]
    roof["frac_of_largest_floor"] = floors[bound_name] / (1e3 * ms_local / calls_per_step)
    if case.page_size:
        # Decode reads each batch's keys once and is bound by HBM: report
        # the algorithmic bytes (keys up to each batch's longest window with
        # their scales, Q, W, windows, logits) against the measured copy rate.
        hi = np.clip(case.ke.astype(np.int64), 0, case.N).max(axis=1)
        key_bytes = case.k.shape[-1] * case.k.itemsize + (4 if case.k_tok is not None else 0) + \
            (case.k_sf.shape[-1] if case.k_sf is not None else 0)
        nbytes = (int(hi.sum()) * key_bytes + case.q.nbytes + case.w.nbytes + case.ks.nbytes +
                  case.ke.nbytes + (case.q_sf.nbytes if case.q_sf is not None else 0) +
                  case.B * case.S * case.N * (2 if args.out_bf16 else 4))
        gbs = nbytes / (ms_local * 1e-3) / 1e9
        roof.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes_per_launch": nbytes,
                     "peak_source": f"{peak_src} HBM copy",
                     "tensor_tflops": achieved})
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc = oracle_sample_rate(case, args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "cpu_model": host_cpu_model()}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "us_per_call": 1e3 * ms / calls_per_step,
        "us_per_call_median": 1e3 * statistics.median(per) / calls_per_step,
        "us_per_call_p10": 1e3 * _pct(srt, 0.1) / calls_per_step,
        "us_per_call_p90": 1e3 * _pct(srt, 0.9) / calls_per_step,
        "higher_is_better": True, "scaling": scaling, "vs_baseline": None,
        "dtype": DTYPES[case.fmt], "data": "synthetic (seeded N(0,1) inputs, quantised)"
        if not args.zero_inputs else "synthetic (all-zero inputs, unit MX scales)",
        "config": workload_config(case, args),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e_main, "e2e_bf16_logits": e2e_bf16,
        "protocol": prot, "protocol_zero_inputs": prot_zero, "topk": topk,
        "fused_topk": fused,
        "gpu_launches": args.steps * launches_per_call * calls_per_step,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        # the CPU oracle runs on rank 0 only; other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            run_reference(args, Dist.__new__(Dist))
        return
    dist = Dist()
    try:
        run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
