#!/usr/bin/env python
"""Benchmark of the lightning-indexer logits call on GB300.

One step = one indexer_logits call (the whole hot path: schedule, TMA loads,
tcgen05 MMA, ReLU.w head reduction, masked store and -inf clean) over one
synthetic workload resident in HBM. Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Timing: W untimed warm-up calls; then K calls, each preceded by an untimed
256 MiB write that flushes L2, each bracketed by CUDA events on the launch
stream; barrier + synchronize around the timed region; max over ranks.
`value` is in-window TFLOP/s = 2*H*D*(sum of window lengths) / time, for all
ranks together. `e2e` repeats the measurement through the same public call
with the inputs copied from pinned host memory and the logits copied back
inside the timed region. `--impl reference` times the float64 CPU oracle on
bounded row samples of the same workload.
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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DTYPES = {0: "bf16", 1: "e4m3", 2: "mxfp8(e4m3+e8m0)", 3: "mxfp4(e2m1+e8m0)"}
# dense tensor peak of a format relative to BF16 (nominal GB300 ratios)
FMT_PEAK_RATIO = {0: 1.0, 1: 2.0, 2: 2.0, 3: 6.0}
L2_FLUSH_BYTES = 256 << 20
# DRAM bytes (read + write) of one kernel launch from an ncu capture, keyed by
# workload, with the digest of the kernel sources it was taken on (see
# profiles/). Reported as roofline.traffic only while the sources still match.
PROFILED_TRAFFIC = {
    "bf16_batched_causal_4096": ("a0ab85169a9d316f", 137.495040e6 + 79.709440e6),
    "fp8_per_token_2048x32768": ("a0ab85169a9d316f", 21.721088e6 + 207.723008e6),
    "mxfp8_2048x32768": ("a0ab85169a9d316f", 22.222592e6 + 207.570432e6),
    "mxfp4_2048x32768": ("a0ab85169a9d316f", 11.900160e6 + 207.955968e6),
    "paged_fp8_decode_64x2_32768": ("a0ab85169a9d316f", 208.284160e6 + 11.974400e6),
    "mxfp8_8192x65536": ("a0ab85169a9d316f", 80375552 + 2087707904),
    "mxfp4_8192x65536": ("a0ab85169a9d316f", 42581504 + 2087260416),
    "mxfp4_irregular_8192x65536": ("a0ab85169a9d316f", 43101952 + 2086262272),
    "thd_bf16_3seq_8192x32768": ("a0ab85169a9d316f", 145004800 + 1013174528),
}


def kernel_source_digest() -> str:
    """Digest of the sources that define and launch the logits kernel (the
    top-k kernel's file is left out: it does not change the logits launch)."""
    import hashlib
    d = os.path.join(ROOT, "infra_dsa_indexer_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f.startswith("topk"):
            continue
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bf16_batched_causal_4096")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: CPU seconds all its steps together aim for")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--topk", type=int, default=0,
                    help="also time indexer_topk (k columns per row) on the call's logits")
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
    sample = f"{nrows} uniformly drawn rows per step of {total_rows}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(case, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nth, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(case, args):
    from infra_dsa_indexer_gb300 import synth
    return {"workload": args.workload, "B": case.B, "S_q": case.S, "S_kv": case.N,
            "H": case.H, "D": case.D, "format": synth.FMT_NAMES[case.fmt],
            "w_format": "bf16" if case.w_fmt == synth.W_BF16 else "f32",
            "in_window_pairs": case.in_window_pairs(), "clean": bool(case.clean),
            "group_rows": bool(case.group_rows),
            "out_format": "bf16" if getattr(args, "out_bf16", False) else "f32",
            "l2": "flushed before every timed call (256 MiB write)",
            "parallelism": f"replicas x{args.gpus}"}


def run_ours(args, dist):
    import torch
    from infra_dsa_indexer_gb300 import binding, synth
    from infra_dsa_indexer_gb300 import build as lib_build

    dev = dist.local_rank
    torch.cuda.set_device(dev)
    if dist.rank == 0:
        lib_build.build()
    dist.barrier()
    binding.load()
    case = synth.make_workload(args.workload)
    flops = case.in_window_flops()
    t = binding.case_to_device(case, device=f"cuda:{dev}", out_bf16=args.out_bf16)
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=f"cuda:{dev}")
    launches_per_call = binding.indexer_launches_per_call(t["shape"])

    for _ in range(args.warmup):
        binding.run_case(case, t, stream=stream)
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
        binding.run_case(case, t, stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    w1 = time.time()
    clk = clocks.stop(w0, w1) if clocks else None
    st = binding.indexer_get_last_error(stream)
    if st != binding.IDX_OK:
        raise RuntimeError(f"device error in timed region: {binding.indexer_status_string(st)}")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]      # ms, one launch each
    ms_local = sum(per) / len(per)
    ms = dist.max(ms_local, device=f"cuda:{dev}")
    value = dist.world * flops / (ms * 1e-3) / 1e12

    # --- top-k over the logits of the call (its own launches and events)
    topk = None
    if args.topk:
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

    # --- end to end through the same call: pinned host inputs in, logits out
    e2e = None
    if not args.no_e2e:
        host = {}
        for key in ("q", "k", "w", "ks", "ke", "q_sf", "k_sf", "k_scales", "block_table"):
            if t.get(key) is not None:
                host[key] = t[key].cpu().pin_memory()
        out_host = torch.empty(t["out"].shape, dtype=t["out"].dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_host.numel() * out_host.element_size()
        n_e2e = max(3, min(args.e2e_steps, args.steps))
        dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            for key, v in host.items():
                t[key].copy_(v, non_blocking=True)
            binding.run_case(case, t, stream=stream)
            out_host.copy_(t["out"], non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = dist.max(e0.elapsed_time(e1) / n_e2e, device=f"cuda:{dev}")
        e2e = {"value": dist.world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "steps": n_e2e,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    if dist.rank != 0:
        return
    peaks, peak_src = load_peaks()
    if topk is not None:
        topk["peak_gbs"] = peaks["hbm_gbs"]
        topk["frac"] = topk["achieved_gbs"] / peaks["hbm_gbs"]
    peak = peaks["bf16_tflops"] * FMT_PEAK_RATIO[case.fmt]
    achieved = flops / (ms_local * 1e-3) / 1e12
    srt = sorted(per)
    prof = None if args.out_bf16 else PROFILED_TRAFFIC.get(args.workload)
    traffic = prof[1] if prof and prof[0] == kernel_source_digest() else None
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": (f"{peak_src} bf16 burst x{FMT_PEAK_RATIO[case.fmt]:g} "
                            "(nominal format ratio)" if case.fmt else f"{peak_src} bf16 burst"),
            "kernel": "dsa::indexer_logits_kernel",
            "algorithmic_flops_per_launch": flops,
            "hbm_write_gbs": case.B * case.S * case.N * (2 if args.out_bf16 else 4)
                             / (ms_local * 1e-3) / 1e9,
            "hbm_peak_gbs": peaks["hbm_gbs"]}
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
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "us_per_call": 1e3 * ms, "us_per_call_median": 1e3 * statistics.median(per),
        "us_per_call_p10": 1e3 * srt[int(0.1 * (len(srt) - 1))],
        "us_per_call_p90": 1e3 * srt[int(0.9 * (len(srt) - 1))],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPES[case.fmt], "data": "synthetic (seeded N(0,1) inputs, quantised)",
        "config": workload_config(case, args),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "topk": topk,
        "gpu_launches": args.steps * launches_per_call,
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
