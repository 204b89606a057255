"""Benchmark: fused top-k / top-p filtering of B=256 x V=128256 bf16 logits.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--op filter|sample|sort|fused|v2] [--workload 1|2|3|4]

One step = one topkp_apply call over the whole batch (joint top-k + top-p,
workload 3: logits 2*N(0,1) in bf16, k ~ U{1..1024} with 10% of rows
disabled, p ~ U[0.5,1] with 5% of rows at 1.0), inputs resident in HBM.
Each timed step is bracketed by CUDA events on the launching stream, after a
512 MiB memset that flushes L2 (the flush itself is outside the events).
Under torchrun every rank filters its own batch (weak scaling, no collective:
rows are independent); the reported time is the maximum over ranks.

Prints one JSON line.  `roofline` compares the algorithmic bytes of the
kernel (read logits + write out = 4 bytes per element) per launch with the
measured HBM copy bandwidth; `cpu_baseline` times the CPU oracle (test
infrastructure, single-threaded numpy) on a bounded sample of the same rows;
`e2e` runs the same call from pinned host buffers with the copies inside the
timed region (the batch pipelined in row chunks over three streams; the
serial figure beside it).  `--workload` times the filter on another of the five seeded
configurations instead (1: 4 x 1024 fp32 joint, 2: 64 x 32000 fp16 top-p
only, 4: 1024 x 151936 fp32 top-k only; the default is 3), with the same
line; the committed ncu traffic applies to configuration 3 only.  `--impl reference` times that oracle alone as the reference
arm (on rank 0; other ranks exit without work).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

WORKLOAD = 3
METRIC = "rows/s and achieved HBM GB/s (% of peak), B=256 V=128256 bf16 joint top-k+top-p"
FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(value: float, ws: int, device) -> float:
    """The largest value over all ranks: a job's time is its slowest rank's."""
    if ws <= 1:
        return value
    import torch
    t = torch.tensor([value], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _job_rows_per_s(ws: int, rows: int, steps: int, total_s: float) -> float:
    """Whole-job throughput of weak-scaling replicas: every rank filters
    `rows` rows per step, and the job takes the slowest rank's time."""
    return ws * rows * steps / total_s


def _peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_hash():
    """Hash of the sources that define the filter kernel's device code (its
    own file and the device helpers it includes); declarations of the other
    kernels do not change it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "top_logit_filter_gb300", "csrc")
    for name in ("apply.cu", "common.cuh", "cluster.cuh"):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_per_launch():
    """DRAM bytes per launch of the filter kernel from the committed ncu
    summary, or None when the kernel sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "apply_kernel_B256_V128256_bf16.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_hash") != _kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def _opt(a, b):
    return None if a is None else a[b]


def _mode_of(w) -> str:
    if w["k"] is not None and w["p"] is not None:
        return "joint top-k + top-p"
    return "top-k only" if w["k"] is not None else "top-p only"


def _cpu_baseline(w, budget_s: float, gpu_out=None):
    """The oracle as it stands, one row at a time, for about budget_s seconds.
    When the GPU's output of the same batch is given, the rows the oracle
    produced are also compared with it (the tests' parity rule)."""
    import oracle as O
    t0 = time.perf_counter()
    rows = 0
    infos = []
    while rows < w["B"] and (rows < 4 or time.perf_counter() - t0 < budget_s):
        kk = _opt(w["k"], rows)
        infos.append(O.apply_row(w["x"][rows], w["dtype"], _opt(w["p"], rows), None if kk is None else int(kk))[1])
        rows += 1
    dt = time.perf_counter() - t0
    line = {"value": rows / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"first {rows} rows of the B={w['B']} x V={w['V']} {w['dtype']} workload, {dt:.1f} s, single-threaded numpy",
            "host": {"cpu": _cpu_model(), "cpu_count": os.cpu_count()}}
    if gpu_out is not None:
        from parity import compare_row
        flips = mismatches = 0
        for b, info in enumerate(infos):
            try:
                flips += compare_row(gpu_out[b], w["x"][b], info, w["dtype"], where=f"bench row {b}")
            except AssertionError:
                mismatches += 1
        line["parity"] = {"rows_checked": rows, "rows_outside_the_bar": mismatches, "top_p_flips_in_band": flips}
    return line


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from top_logit_filter_gb300 import workloads
    import oracle as O
    w = workloads.make(WORKLOAD)
    for i in range(args.warmup):
        b = i % w["B"]
        O.apply_row(w["x"][b], w["dtype"], w["p"][b], int(w["k"][b]))
    t0 = time.perf_counter()
    for i in range(args.steps):
        b = i % w["B"]
        O.apply_row(w["x"][b], w["dtype"], w["p"][b], int(w["k"][b]))
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64+f32 (numpy)",
        "data": "synthetic",
        "config": {"workload": w["name"], "B": w["B"], "V": w["V"], "mode": "joint top-k + top-p",
                   "step": "one row of the workload per step (CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} rows (cycling over the 256-row batch), single-threaded numpy"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


E2E_CHUNKS = 4


def _e2e_filter(tk, w, dev, stream, x, p, k, out, args, ws):
    """The filter end to end through the public API: each step copies the
    batch's logits, p and k from pinned host memory, filters them and copies
    the output back, all inside the timed region, and the next step starts
    only when the output is on the host.  Two ways: serial (copy in, filter,
    copy out on the caller's stream) and pipelined (the batch in E2E_CHUNKS
    row chunks: copies in, filtering and copies out on three streams, so
    that the two copy directions overlap).  `value` is the pipelined rate."""
    import torch
    from rawutil import raw_to_torch

    B, dt = w["B"], w["dtype"]
    hx = raw_to_torch(w["x"], dt).pin_memory()
    hp = raw_to_torch(w["p"], dt).pin_memory() if p is not None else None
    hk = torch.from_numpy(w["k"]).pin_memory() if k is not None else None
    hout = torch.empty_like(hx).pin_memory()
    steps = max(3, min(50, args.steps))
    dx = torch.empty_like(x)
    dp = torch.empty_like(p) if p is not None else None
    dk = torch.empty_like(k) if k is not None else None
    dout = torch.empty_like(x)

    def serial_step():
        dx.copy_(hx, non_blocking=True)
        if dp is not None:
            dp.copy_(hp, non_blocking=True)
        if dk is not None:
            dk.copy_(hk, non_blocking=True)
        hout.copy_(tk.apply(dx, p=dp, k=dk, out=dout), non_blocking=True)

    chunks = [(B * i // E2E_CHUNKS, B * (i + 1) // E2E_CHUNKS) for i in range(min(E2E_CHUNKS, B))]
    s_in, s_run, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in chunks]
    ev_run = [torch.cuda.Event() for _ in chunks]
    ev_out = [torch.cuda.Event() for _ in chunks]

    def piped_step():
        s_in.wait_stream(stream)
        with torch.cuda.stream(s_in):
            # p and k whole (a few hundred bytes), then the logits chunk by chunk
            if dp is not None:
                dp.copy_(hp, non_blocking=True)
            if dk is not None:
                dk.copy_(hk, non_blocking=True)
        for c, (r0, r1) in enumerate(chunks):
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_run[c])  # the last step's filter of this chunk has read its inputs
                dx[r0:r1].copy_(hx[r0:r1], non_blocking=True)
                ev_in[c].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev_in[c])
                s_run.wait_event(ev_out[c])  # the last step's copy out of this chunk is done
                tk.apply(dx[r0:r1], p=dp[r0:r1] if dp is not None else None, k=dk[r0:r1] if dk is not None else None,
                         out=dout[r0:r1])
                ev_run[c].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[c])
                hout[r0:r1].copy_(dout[r0:r1], non_blocking=True)
                ev_out[c].record(s_out)
        stream.wait_stream(s_out)  # the step ends with its output on the host

    def timed(step):
        for _ in range(2):
            step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return _max_over_ranks(e0.elapsed_time(e1) / 1e3, ws, dev)

    def same_bits(a, b):
        it = torch.int16 if a.element_size() == 2 else torch.int32
        return torch.equal(a.view(it), b.view(it))

    serial_s = timed(serial_step)
    serial_ok = same_bits(hout, out.cpu())
    hout.zero_()
    piped_s = timed(piped_step)
    piped_ok = same_bits(hout, out.cpu())
    h2d = sum(t.numel() * t.element_size() for t in (hx, hp, hk) if t is not None)
    d2h = hout.numel() * hout.element_size()
    return {"value": _job_rows_per_s(ws, B, steps, piped_s), "unit": "rows/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "pipeline": f"{len(chunks)} row chunks; copies in, filter and copies out on three streams",
            "serial": {"value": _job_rows_per_s(ws, B, steps, serial_s), "unit": "rows/s"},
            "output_matches_device_run": bool(serial_ok and piped_ok)}


def run_ours(args):
    import numpy as np
    import torch

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import top_logit_filter_gb300 as tk
    from rawutil import raw_to_torch
    from top_logit_filter_gb300 import workloads

    w = workloads.make(args.workload)
    B, V, dt = w["B"], w["V"], w["dtype"]
    x = raw_to_torch(w["x"], dt, dev)
    p = raw_to_torch(w["p"], dt, dev) if w["p"] is not None else None
    k = torch.from_numpy(w["k"]).to(dev) if w["k"] is not None else None
    out = torch.empty_like(x)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        flush.zero_()
        tk.apply(x, p=p, k=k, out=out)
    launches_per_step = tk.last_launch_count()
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clocks:
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            tk.apply(x, p=p, k=k, out=out)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        if ws > 1:
            torch.distributed.barrier()
        t_wall = time.perf_counter() - t_wall
    tk.device_status(dev)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_s = sum(step_ms) / 1e3
    q = sorted(step_ms)
    step_pct = {"p10_us": 1e3 * q[len(q) // 10], "p50_us": 1e3 * q[len(q) // 2], "p90_us": 1e3 * q[(9 * len(q)) // 10]}
    total_s = _max_over_ranks(total_s, ws, dev)
    ms_per_step = 1e3 * total_s / args.steps
    value = _job_rows_per_s(ws, B, args.steps, total_s)

    # roofline of the filter kernel: one launch per step
    esize = 4 if dt == "f32" else 2
    alg_bytes = B * V * esize * 2
    kernel_s = total_s / args.steps / max(1, launches_per_step)
    achieved = alg_bytes / kernel_s / 1e9
    peak, peak_kind = _peak_hbm()
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": _traffic_per_launch() if args.workload == WORKLOAD else None, "peak_source": f"{peak_kind} (copy bandwidth, burst)",
                "algorithmic_bytes_per_launch": alg_bytes}

    e2e = _e2e_filter(tk, w, dev, stream, x, p, k, out, args, ws)

    if rank == 0:
        line = {
            "metric": METRIC if args.workload == WORKLOAD else
                      f"rows/s and achieved HBM GB/s (% of peak), B={B} V={V} {dt} {_mode_of(w)}",
            "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dt, "data": "synthetic",
            "config": {"workload": w["name"], "B": B, "V": V, "mode": _mode_of(w),
                       "l2": "flushed before every timed step (512 MiB memset, outside the events)",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "1 GPU",
                       "wall_s_timed_region": t_wall, "step_time": step_pct},
            "achieved_GBps": achieved,
            "roofline": roofline,
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks.summary(),
            "e2e": e2e,
        }
        if not args.no_cpu_baseline:
            from rawutil import torch_to_raw
            line["cpu_baseline"] = _cpu_baseline(w, args.cpu_budget, torch_to_raw(out, dt))
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_sample(args):
    """The post-filter stage on the filter's output of the same batch: one
    topkp_sample call per step (min-p, QSample with Exp(1) variates, the
    output row), after the same L2 flush.  One JSON line."""
    import numpy as np
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import top_logit_filter_gb300 as tk
    from rawutil import raw_to_torch
    from top_logit_filter_gb300 import workloads

    w = workloads.make(WORKLOAD)
    B, V, dt = w["B"], w["V"], w["dtype"]
    x = raw_to_torch(w["x"], dt, dev)
    f = tk.apply(x, p=raw_to_torch(w["p"], dt, dev), k=torch.from_numpy(w["k"]).to(dev))
    rng = np.random.default_rng(SAMPLE_SEED)
    q = torch.from_numpy(rng.exponential(1.0, size=(B, V)).astype(np.float32)).to(dev)
    mp = torch.from_numpy(rng.uniform(0.001, 0.2, size=B).astype(np.float32)).to(dev)
    out = torch.empty_like(f)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush.zero_()
        tok, _ = tk.sample(f, min_p=mp, q=q, out=out)
    torch.cuda.synchronize(dev)
    kept = int((out.view(torch.int16) != -128).sum().item())   # bf16 -inf is 0xFF80

    def timed(call, prep=None):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            if prep is not None:
                prep()
            flush.zero_()
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        return sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3

    with ClockSampler(0) as clocks:
        total_s = timed(lambda: tk.sample(f, min_p=mp, q=q, out=out))
    # the same stage writing only what min-p removes (in place on a copy of
    # the filter's output, restored before the flush of every step), and the
    # token alone
    f2 = f.clone()
    in_place_s = timed(lambda: tk.sample(f2, min_p=mp, q=q, out=f2), prep=lambda: f2.copy_(f))
    token_s = timed(lambda: tk.sample(f, min_p=mp, q=q, want_out=False))
    tk.device_status(dev)
    alg_bytes = B * V * 2 * 2 + 4 * kept
    kernel_s = total_s / args.steps
    peak, peak_kind = _peak_hbm()
    achieved = alg_bytes / kernel_s / 1e9
    line = {
        "metric": "rows/s and achieved HBM GB/s, post-filter stage (min-p + exponential-race sample), "
                  "B=256 V=128256 bf16",
        "value": B * args.steps / total_s, "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * kernel_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "sample_after_apply_joint_B256_V128256_bf16", "B": B, "V": V,
                   "input": "the filter's output of the joint top-k + top-p batch; min_p ~ U[0.001, 0.2]; "
                            "q ~ Exp(1) fp32",
                   "kept_after_min_p": kept,
                   "ms_per_step_in_place": 1e3 * in_place_s / args.steps,
                   "ms_per_step_token_only": 1e3 * token_s / args.steps,
                   "l2": "flushed before every timed step (512 MiB memset, outside the events)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": f"{peak_kind} (copy bandwidth, burst)",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


SAMPLE_SEED = 4242


def _timed_steps(args, dev, stream, flush, call, prep=None):
    """Seconds over args.steps calls of `call`, each after the L2 flush,
    bracketed by CUDA events on the launching stream."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        if prep is not None:
            prep()
        flush.zero_()
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    return sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3


def run_fused(args):
    """The filter and the sample in one pass (topkp_apply_sample) on the
    B=256 x V=128256 bf16 joint batch, min_p ~ U[0.001, 0.2] and q ~ Exp(1):
    one call per step, token only (the decode case) and with the output
    row.  One JSON line (the token-only time is the headline)."""
    import numpy as np
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import top_logit_filter_gb300 as tk
    from rawutil import raw_to_torch
    from top_logit_filter_gb300 import workloads

    w = workloads.make(WORKLOAD)
    B, V, dt = w["B"], w["V"], w["dtype"]
    x = raw_to_torch(w["x"], dt, dev)
    p = raw_to_torch(w["p"], dt, dev)
    k = torch.from_numpy(w["k"]).to(dev)
    rng = np.random.default_rng(SAMPLE_SEED)
    q = torch.from_numpy(rng.exponential(1.0, size=(B, V)).astype(np.float32)).to(dev)
    mp = torch.from_numpy(rng.uniform(0.001, 0.2, size=B).astype(np.float32)).to(dev)
    out = torch.empty_like(x)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush.zero_()
        tk.apply_sample(x, p=p, k=k, min_p=mp, q=q, want_out=False)
        tk.apply_sample(x, p=p, k=k, min_p=mp, q=q, out=out)
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clocks:
        tok_s = _timed_steps(args, dev, stream, flush, lambda: tk.apply_sample(x, p=p, k=k, min_p=mp, q=q, want_out=False))
    out_s = _timed_steps(args, dev, stream, flush, lambda: tk.apply_sample(x, p=p, k=k, min_p=mp, q=q, out=out))
    two_s = _timed_steps(args, dev, stream, flush, lambda: tk.sample(tk.apply(x, p=p, k=k), min_p=mp, q=q,
                                                                     want_out=False))
    tk.device_status(dev)
    peak, peak_kind = _peak_hbm()
    alg_tok = B * V * 2        # the logits read; q is read only at the few survivors
    line = {
        "metric": "rows/s, fused top-k/top-p filter + min-p + sample (token only), B=256 V=128256 bf16",
        "value": B * args.steps / tok_s, "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * tok_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "apply_sample_joint_B256_V128256_bf16", "B": B, "V": V,
                   "min_p": "U[0.001, 0.2]", "q": "Exp(1) fp32",
                   "ms_per_step_with_out": 1e3 * out_s / args.steps,
                   "ms_per_step_two_calls_token_only": 1e3 * two_s / args.steps,
                   "l2": "flushed before every timed step (512 MiB memset, outside the events)"},
        "roofline": {"bound": "hbm", "achieved": alg_tok / (tok_s / args.steps) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": alg_tok / (tok_s / args.steps) / 1e9 / peak, "traffic": None,
                     "peak_source": f"{peak_kind} (copy bandwidth, burst)", "algorithmic_bytes_per_launch": alg_tok},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def run_v2(args):
    """The TopKTopPSampleV2 semantics (topkp_sample_v2) on a B=256 x
    V=152064 bf16 decode batch (2*N(0,1) logits; k ~ U{1..1024}, 10% of the
    rows 0 so top-k is skipped; p ~ U[0.5, 1]; min_p ~ U[0, 0.2]; q ~ Exp(1);
    ks_max = 1024): one call per step, the token and the filtered row."""
    import numpy as np
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import top_logit_filter_gb300 as tk
    from rawutil import raw_to_torch, to_raw

    rng = np.random.default_rng(SAMPLE_SEED + 1)
    B, V = 256, 152064
    x = raw_to_torch(to_raw((rng.standard_normal(B * V) * 2).astype(np.float32), "bf16").reshape(B, V), "bf16", dev)
    kk = rng.integers(1, 1025, size=B).astype(np.int32)
    kk[rng.random(B) < 0.1] = 0
    k = torch.from_numpy(kk).to(dev)
    p = torch.from_numpy(rng.uniform(0.5, 1.0, size=B).astype(np.float32)).to(dev)
    mp = torch.from_numpy(rng.uniform(0.0, 0.2, size=B).astype(np.float32)).to(dev)
    q = torch.from_numpy(rng.exponential(1.0, size=(B, V)).astype(np.float32)).to(dev)
    ws = torch.empty(int(tk._lib.load().topkp_sample_v2_workspace_size(B, V, 2)), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    call = lambda: tk.sample_v2(x, k=k, p=p, min_p=mp, q=q, ks_max=1024, workspace=ws)
    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clocks:
        total_s = _timed_steps(args, dev, stream, flush, call)
    tk.device_status(dev)
    peak, peak_kind = _peak_hbm()
    alg = B * V * 2 * 2
    kernel_s = total_s / args.steps
    line = {
        "metric": "rows/s, TopKTopPSampleV2 semantics (token + filtered row), B=256 V=152064 bf16",
        "value": B * args.steps / total_s, "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * kernel_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "sample_v2_B256_V152064_bf16", "B": B, "V": V, "ks_max": 1024,
                   "rows_topk_skipped": int((kk == 0).sum()),
                   "l2": "flushed before every timed step (512 MiB memset, outside the events)"},
        "roofline": {"bound": "hbm", "achieved": alg / kernel_s / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": alg / kernel_s / 1e9 / peak, "traffic": None,
                     "peak_source": f"{peak_kind} (copy bandwidth, burst)", "algorithmic_bytes_per_launch": alg},
        "gpu_launches": 3 * args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def run_sort(args):
    """The stable sort (topkp_sort) of the pre-sorted workload's logits
    (B=512 x V=152064 bf16): one call per step after the same L2 flush, the
    workspace allocated once outside the timed region.  One JSON line."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import top_logit_filter_gb300 as tk
    from rawutil import raw_to_torch
    from top_logit_filter_gb300 import workloads

    w = workloads.make(5)
    B, V, dt = w["B"], w["V"], w["dtype"]
    x = raw_to_torch(w["x"], dt, dev)
    ws = torch.empty(tk.sort_workspace_size(B, V, x.dtype), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush.zero_()
        tk.sort(x, workspace=ws)
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(0) as clocks:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            tk.sort(x, workspace=ws)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    total_s = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / 1e3
    # bytes a sort must move at least: read the logits, write values and indices
    alg_bytes = B * V * (2 + 2 + 4)
    kernel_s = total_s / args.steps
    peak, peak_kind = _peak_hbm()
    achieved = alg_bytes / kernel_s / 1e9
    line = {
        "metric": "rows/s and achieved HBM GB/s, stable sort of B=512 V=152064 bf16 rows",
        "value": B * args.steps / total_s, "unit": "rows/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * kernel_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "sort_B512_V152064_bf16", "B": B, "V": V,
                   "l2": "flushed before every timed step (512 MiB memset, outside the events)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": f"{peak_kind} (copy bandwidth, burst)",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--op", choices=("filter", "sample", "sort", "fused", "v2"), default="filter",
                    help="filter: the headline topkp_apply step; sample: the post-filter stage alone; "
                         "sort: the stable sort alone; fused: filter + min-p + sample in one call; "
                         "v2: the TopKTopPSampleV2 semantics")
    ap.add_argument("--workload", type=int, choices=(1, 2, 3, 4), default=WORKLOAD,
                    help="filter op only: which seeded configuration (3 is the headline batch)")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle timing (profiling runs)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of CPU oracle work for cpu_baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "sample":
        run_sample(args)
    elif args.op == "sort":
        run_sort(args)
    elif args.op == "fused":
        run_fused(args)
    elif args.op == "v2":
        run_v2(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
