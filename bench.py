"""Benchmark of the attention forward (one JSON line on stdout).

A step is one pass of the whole forward hot path over one batch of synthetic
input: one non-causal and one causal fa_fwd call on the N = 4096 comparison
workload of the pages (B=2, H=16, N=4096, D=64, bf16, scale 1/8).  ``value``
is the pages' FLOP count (4*B*H*N^2*D non-causal, half causal) of all steps of
all ranks divided by the summed device time of the calls, in TFLOP/s; each
call is bracketed by CUDA events on the stream it is launched on, and L2 is
flushed (a 256 MiB write) between calls, outside the events.

Other keys: ``configs`` (every workload of the task -- the five shapes, each
mask it is run with -- timed per call the same way: mean and median ms,
TFLOP/s and the fraction of the measured bf16 tensor peak), ``e2e`` (same
metric through the C ABI with pinned host buffers,
host->device and device->host copies of every step inside the timed region,
pipelined so one step's calls overlap its neighbours' copies), ``backward``
(fa_bwd on the same workload, per call), ``decode`` (split-KV decoding of a
few queries against long key sequences, per call, as K/V bandwidth against
the measured HBM copy rate), ``roofline``
(the non-causal kernel against the measured bf16 tensor peak), ``clocks``
(nvidia-smi samples taken during the timed region), ``cpu_baseline`` (the fp64
CPU oracle on a bounded sample, timed on this host's cores).

``--impl reference`` times the CPU oracle as the reference arm on the same
metric.  Under torchrun every rank runs its own replica of the workload (weak
scaling, no data-path collective); ranks only meet at the timing barriers.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and ms/call on 1 GB300 (causal & non-causal), % of tensor peak"
DEFAULT_WORKLOAD = "b2h16_n4096"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


# Split-KV decode shapes timed beside the headline (B, H, query rows, keys, D):
# a few queries against long key sequences, bf16, automatic schedule.
DECODE_SHAPES = ((1, 32, 4, 32768, 128), (8, 32, 1, 8192, 128))


def decode_timings(steps: int, dev, stream, flush, hbm_gbs: float) -> dict:
    """Mean time of `steps` fa_fwd_qkv calls per decode shape (CUDA events on
    the launching stream, L2 flushed before each call) and the K/V bandwidth
    it implies, against the measured HBM copy rate.  The same calls are also
    timed back to back without the flush (``us_mean_no_flush``): their K/V
    (0.5-1 GB, 4-8x the 129 MB L2) is larger than L2 either way, which the
    timing rules accept in place of a flush.  The difference is the cost of
    starting each call with the kernel's code and scheduling data cold, and of
    writing back the dirty lines the flush leaves in L2 (up to its 129 MB)
    while the call streams its K/V."""
    import torch
    from exact_attention_10_gb300 import fa
    out = {"dtype": "bf16", "schedule": "auto", "l2": "flushed between calls", "steps": steps, "shapes": []}
    for B, H, Nq, Nkv, D in DECODE_SHAPES:
        g = torch.Generator(device=dev).manual_seed(Nq * 131 + Nkv)
        q = torch.randn(B, H, Nq, D, device=dev, generator=g).to(torch.bfloat16)
        k = torch.randn(B, H, Nkv, D, device=dev, generator=g).to(torch.bfloat16)
        v = torch.randn(B, H, Nkv, D, device=dev, generator=g).to(torch.bfloat16)
        o, lse = torch.empty_like(q), torch.empty(B, H, Nq, dtype=torch.float32, device=dev)
        for _ in range(3):
            fa.forward(q, k, v, scale=D ** -0.5, out=o, lse=lse)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            fa.forward(q, k, v, scale=D ** -0.5, out=o, lse=lse)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        rc = fa.sync_status(stream.cuda_stream)
        if rc != 0:
            raise fa.FAError(rc, "decode")
        ms = statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends))
        for i in range(steps):
            starts[i].record(stream)
            fa.forward(q, k, v, scale=D ** -0.5, out=o, lse=lse)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        rc = fa.sync_status(stream.cuda_stream)
        if rc != 0:
            raise fa.FAError(rc, "decode")
        ms_nf = statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends))
        kv = 2 * B * H * Nkv * D * 2
        out["shapes"].append({"B": B, "H": H, "Nq": Nq, "Nkv": Nkv, "D": D, "us_mean": ms * 1e3,
                              "kv_bytes": kv, "kv_gbs": kv / (ms * 1e-3) / 1e9,
                              "frac_of_measured_hbm": kv / (ms * 1e-3) / 1e9 / hbm_gbs,
                              "us_mean_no_flush": ms_nf * 1e3,
                              "frac_of_measured_hbm_no_flush": kv / (ms_nf * 1e-3) / 1e9 / hbm_gbs})
        del q, k, v, o, lse
    return out


# The task's workloads, in order, each with the masks it is run with; the
# long-context one is causal at N = 32768 and non-causal at N = 16384.
CONFIG_WORKLOADS = ("tiny_n256", "b4h16_n1024", "b2h16_n4096", "ragged_n3000_d128_fp16", "long_n32768_d128",
                    "long_n16384_d128")
# ... of which these also time fa_bwd (the headline workload's backward is in
# the line's own "backward" object)
BWD_CONFIG_WORKLOADS = ("b4h16_n1024", "ragged_n3000_d128_fp16", "long_n16384_d128")


def config_timings(steps: int, dev, stream, flush, peak: float) -> dict:
    """Per-call timings of every task workload and mask (fa_fwd, automatic
    schedule; CUDA events on the launching stream, L2 flushed before each
    call, after 3 untimed calls), with the pages' FLOP count (4*B*H*N^2*D,
    half causal) and the exact causal count beside it."""
    import torch
    from exact_attention_10_gb300 import fa
    from exact_attention_10_gb300.accounting import flops, flops_causal_exact, fused_bytes
    from exact_attention_10_gb300.inputs import WORKLOADS, make_custom, make_qkv
    out = {"schedule": "auto", "l2": "flushed between calls", "steps": steps, "inputs": "make_qkv(seed=0)",
           "peak_tflops": peak, "workloads": {}}
    for name in CONFIG_WORKLOADS:
        w = WORKLOADS[name]
        q, k, v = (x.to(dev) for x in make_qkv(w, seed=0))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        entry = {"shape": w.describe()}
        for causal in w.masks:
            for _ in range(3):
                fa.forward(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse)
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            for i in range(steps):
                flush.zero_()
                starts[i].record(stream)
                fa.forward(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse)
                ends[i].record(stream)
            torch.cuda.synchronize(dev)
            rc = fa.sync_status(stream.cuda_stream)
            if rc != 0:
                raise fa.FAError(rc, name)
            ts = [a.elapsed_time(b) for a, b in zip(starts, ends)]
            avg = statistics.mean(ts)
            fl = flops(w.B, w.H, w.N, w.D, causal)
            tf = fl / (avg * 1e-3) / 1e12
            rec = {"ms_mean": avg, "ms_median": statistics.median(ts), "tflops": tf,
                   "frac_of_measured_peak": tf / peak, "flops_per_call": fl}
            if causal:
                rec["tflops_exact_causal_count"] = flops_causal_exact(w.B, w.H, w.N, w.D) / (avg * 1e-3) / 1e12
            # DRAM bytes per launch from a committed ncu capture of this kernel
            # on this workload (current kernel source only), beside the
            # algorithmic bytes (Q, K, V read, O written, fp32 LSE)
            kname = f"fa_fwd_sm103<{w.D},{w.dtype},{'causal' if causal else 'noncausal'}>"
            rec["algorithmic_bytes"] = fused_bytes(w.B, w.H, w.N, w.D)
            rec["traffic"] = _traffic_record(kname, workload_name=name)
            if name in BWD_CONFIG_WORKLOADS:   # fa_bwd from this forward's O and LSE, timed the same way
                do = make_custom(w.B, w.H, w.N, w.D, w.dtype, seed=1)[0].to(dev)
                grads = tuple(torch.empty_like(x) for x in (q, k, v))
                for _ in range(3):
                    fa.backward(q, k, v, o, do, lse, causal=causal, scale=w.scale, dq=grads[0], dk=grads[1],
                                dv=grads[2])
                for i in range(steps):
                    flush.zero_()
                    starts[i].record(stream)
                    fa.backward(q, k, v, o, do, lse, causal=causal, scale=w.scale, dq=grads[0], dk=grads[1],
                                dv=grads[2])
                    ends[i].record(stream)
                torch.cuda.synchronize(dev)
                rc = fa.sync_status(stream.cuda_stream)
                if rc != 0:
                    raise fa.FAError(rc, name + " backward")
                bavg = statistics.mean(a.elapsed_time(b) for a, b in zip(starts, ends))
                btf = 2.5 * fl / (bavg * 1e-3) / 1e12
                rec["backward"] = {"ms_mean": bavg, "tflops": btf, "frac_of_measured_peak": btf / peak,
                                   "flops_convention": "2.5 x forward",
                                   "dq_path": "one pass (fp32 accumulator)" if w.D == 64 else "second pass"}
                del do, grads
            entry["causal" if causal else "noncausal"] = rec
        out["workloads"][name] = entry
        del q, k, v, o, lse
        torch.cuda.empty_cache()
    return out


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest of every rank's value (this rank's value when single)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, steps: int, flops_per_step: float, slowest_ms: float) -> float:
    """Whole-job throughput: every rank runs `steps` steps of the same
    replica, and the job takes as long as its slowest rank."""
    return world * steps * flops_per_step / (slowest_ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= (self.t1 or r[0]) + 1]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use)}


def _traffic_record(kernel_name: str, workload_name: str | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (matched by content hash) and, when
    ``workload_name`` is given, on that workload; otherwise None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for rel in ("exact_attention_10_gb300/csrc/fa_fwd_kernel.cuh", "exact_attention_10_gb300/csrc/sm103_ptx.cuh",
                "exact_attention_10_gb300/csrc/fa_schedule.h"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    entry = rec.get(kernel_name)
    if not entry or entry.get("source_sha256") != h.hexdigest():
        return None
    if workload_name is not None and entry.get("workload_name") != workload_name:
        return None
    return entry.get("dram_bytes_per_launch")


def cpu_oracle_sample(w, budget_s: float, rows_per_head: int | None = None):
    """Time the fp64 oracle on sampled rows of the workload, both masks.

    Rows are spread evenly over [0, N) so a causal sample has the average row
    cost.  Returns (TFLOP/s in the pages' convention, description, threads)."""
    import numpy as np
    import oracle
    from exact_attention_10_gb300.accounting import flops
    from exact_attention_10_gb300.inputs import make_qkv
    q, k, v = make_qkv(w, seed=0)
    BH = w.B * w.H
    per_row = {c: flops(1, 1, w.N, w.D, c) / w.N for c in (False, True)}
    rows = rows_per_head or w.N
    done_flops, spent, heads = 0.0, 0.0, 0
    while spent < budget_s and heads < BH:
        bh = np.full(rows, heads, dtype=np.int64)
        ri = np.linspace(0, w.N - 1, rows).round().astype(np.int64)
        for causal in (False, True):
            t = time.perf_counter()
            oracle.rows(q, k, v, causal, w.scale, bh, ri)
            spent += time.perf_counter() - t
            done_flops += per_row[causal] * rows
        heads += 1
    what = "all rows" if rows == w.N else f"{rows} rows spread over [0, N)"
    desc = (f"{heads} of {BH} heads x {what}, non-causal and causal, of {w.describe()}; "
            f"{spent:.1f} s of CPU time")
    return done_flops / spent / 1e12, desc, oracle.num_threads(), spent


def run_reference(args, w):
    """Reference arm: the fp64 CPU oracle, timed as it stands."""
    rank, world, _ = _dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    from exact_attention_10_gb300.accounting import flops
    from exact_attention_10_gb300.inputs import make_qkv
    q, k, v = make_qkv(w, seed=0)
    # size each step so warmup + steps take about a minute on this host
    probe_rows = 32
    ri = np.linspace(0, w.N - 1, probe_rows).round().astype(np.int64)
    t = time.perf_counter()
    for causal in (False, True):
        oracle.rows(q, k, v, causal, w.scale, np.zeros(probe_rows, dtype=np.int64), ri)
    per_row_s = (time.perf_counter() - t) / probe_rows
    target = 60.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(w.N, target / max(per_row_s, 1e-9))))
    BH = w.B * w.H
    per_row = {c: flops(1, 1, w.N, w.D, c) / w.N for c in (False, True)}

    def step(i):
        bh = np.full(rows, i % BH, dtype=np.int64)
        ri = np.linspace(0, w.N - 1, rows).round().astype(np.int64)
        for causal in (False, True):
            oracle.rows(q, k, v, causal, w.scale, bh, ri)

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t
    fl = args.steps * rows * (per_row[False] + per_row[True])
    value = fl / dt / 1e12
    sample = (f"each step: {rows} query rows of one head (rows spread over [0, N)), non-causal and causal, "
              f"of {w.describe()}")
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.describe() + ", causal + non-causal per step", "B": w.B, "H": w.H,
                       "N": w.N, "D": w.D, "parallelism": "rank 0 only (CPU)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of CPU oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--bwd-steps", type=int, default=50, help="timed backward calls per mask (0: skip)")
    ap.add_argument("--decode-steps", type=int, default=30, help="timed split-KV decode calls per shape (0: skip)")
    ap.add_argument("--config-steps", type=int, default=20, help="timed calls per task workload and mask (0: skip)")
    args = ap.parse_args(argv)

    from exact_attention_10_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    import torch
    from exact_attention_10_gb300 import fa
    from exact_attention_10_gb300.accounting import flops
    from exact_attention_10_gb300.inputs import make_qkv

    rank, world, local = _dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load()

    q_h, k_h, v_h = make_qkv(w, seed=0)
    q, k, v = (x.to(dev) for x in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    modes = (False, True)
    F = {c: flops(w.B, w.H, w.N, w.D, c) for c in modes}
    code = fa.FA_BF16 if w.dtype == "bf16" else fa.FA_FP16

    def call(causal):
        rc = fa.fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H, w.N,
                        w.D, int(causal), w.scale, code, sp)
        if rc != 0:
            raise fa.FAError(rc, "fa_fwd")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        for c in modes:
            flush.zero_()
            call(c)
    rc = fa.sync_status(sp)
    if rc != 0:
        raise fa.FAError(rc, "warm-up")

    starts = {c: [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] for c in modes}
    ends = {c: [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)] for c in modes}
    barrier()
    clocks.mark_start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        for c in modes:
            flush.zero_()
            starts[c][i].record(stream)
            call(c)
            ends[c][i].record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    clocks.mark_end()
    rc = fa.sync_status(sp)
    if rc != 0:
        raise fa.FAError(rc, "timed region")
    ms = {c: [s.elapsed_time(e) for s, e in zip(starts[c], ends[c])] for c in modes}
    total_ms = max_over_ranks(sum(sum(v) for v in ms.values()), dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, args.steps, F[False] + F[True], total_ms)
    clk = clocks.finish()

    # End to end through the C ABI: every step copies its inputs in from pinned
    # host memory, makes both calls, and copies both O and LSE back out.  The
    # steps are pipelined over two sets of device buffers and three streams
    # (copies in, calls, copies out), so step i's calls overlap step i+1's
    # input copies and step i-1's output copies; every copy of every timed step
    # is inside the timed region.
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    qp, kp, vp = (x.pin_memory() for x in (q_h, k_h, v_h))
    outs_h = {c: (torch.empty(q_h.shape, dtype=q_h.dtype).pin_memory(),
                  torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()) for c in modes}
    h2d = sum(x.numel() * x.element_size() for x in (qp, kp, vp))
    d2h = sum(op_.numel() * op_.element_size() + lp_.numel() * lp_.element_size() for op_, lp_ in outs_h.values())
    sets = [{"in": (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)),
             "out": {c: (torch.empty_like(o), torch.empty_like(lse)) for c in modes}} for _ in range(2)]
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = [{name: torch.cuda.Event() for name in ("in", "run", "out")} for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        b = i % 2
        bq, bk, bv = sets[b]["in"]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev[b]["run"])      # the calls of step i-2 have read this set's inputs
            bq.copy_(qp, non_blocking=True)
            bk.copy_(kp, non_blocking=True)
            bv.copy_(vp, non_blocking=True)
            ev[b]["in"].record(s_in)
        s_run.wait_event(ev[b]["in"])
        if used[b]:
            s_run.wait_event(ev[b]["out"])         # step i-2's outputs have been copied out
        for c in modes:
            bo, bl = sets[b]["out"][c]
            rc = fa.fwd_raw(bq.data_ptr(), bk.data_ptr(), bv.data_ptr(), bo.data_ptr(), bl.data_ptr(), w.B, w.H,
                            w.N, w.D, int(c), w.scale, code, s_run.cuda_stream)
            if rc != 0:
                raise fa.FAError(rc, "fa_fwd")
        ev[b]["run"].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev[b]["run"])
            for c in modes:
                bo, bl = sets[b]["out"][c]
                outs_h[c][0].copy_(bo, non_blocking=True)
                outs_h[c][1].copy_(bl, non_blocking=True)
            ev[b]["out"].record(s_out)
        used[b] = True

    for i in range(4):
        e2e_step(i)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)   # after the last step's output copies
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_value = job_tflops(world, e2e_steps, F[False] + F[True], e2e_ms)
    rc = fa.sync_status(s_run.cuda_stream)
    if rc != 0:
        raise fa.FAError(rc, "e2e")
    # the last step's results, as read back, match the device-timed calls' outputs
    for c in modes:
        call(c)
        torch.cuda.synchronize(dev)
        if not (torch.equal(outs_h[c][0], o.cpu()) and torch.equal(outs_h[c][1], lse.cpu())):
            raise RuntimeError("end-to-end results differ from the device-timed calls")

    # backward (fa_bwd) on the same workload, from this forward's O and LSE and
    # a seeded upstream gradient; timed per call like the forward, outside the
    # step above.  FLOPs in the usual convention: 2.5 x the forward's (five
    # tile products per (query tile, key tile) pair: S, dP, dV, dK, dQ).
    bwd_info = None
    if args.bwd_steps > 0:
        from exact_attention_10_gb300.inputs import make_custom
        do = make_custom(w.B, w.H, w.N, w.D, w.dtype, seed=1)[0].to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bwd_info = {"flops_convention": "2.5 x forward (five tile products per tile pair)",
                    "kernels_per_call": 3,
                    "dq_path": ("one pass: dQ products added into an fp32 accumulator by TMA reductions"
                                if w.D == 64 else "second pass over the key tiles")}
        for c in modes:
            call(c)
            for _ in range(3):
                fa.backward(q, k, v, o, do, lse, causal=c, scale=w.scale, dq=dq, dk=dk, dv=dv)
            bs = [torch.cuda.Event(enable_timing=True) for _ in range(args.bwd_steps)]
            be = [torch.cuda.Event(enable_timing=True) for _ in range(args.bwd_steps)]
            barrier()
            for i in range(args.bwd_steps):
                flush.zero_()
                bs[i].record(stream)
                fa.backward(q, k, v, o, do, lse, causal=c, scale=w.scale, dq=dq, dk=dk, dv=dv)
                be[i].record(stream)
            barrier()
            rc = fa.sync_status(sp)
            if rc != 0:
                raise fa.FAError(rc, "backward")
            bms = statistics.mean(s_.elapsed_time(e_) for s_, e_ in zip(bs, be))
            btf = 2.5 * F[c] / (bms * 1e-3) / 1e12
            bwd_info["causal" if c else "noncausal"] = {"ms_mean": bms, "tflops": btf,
                                                       "frac_of_measured_peak": btf / _peaks()[0],
                                                       "flops_per_call": 2.5 * F[c]}

    peak, peak_sus, _, peak_src = _peaks()
    mode_info = {}
    for c in modes:
        avg = statistics.mean(ms[c])
        tf = F[c] / (avg * 1e-3) / 1e12
        mode_info["causal" if c else "noncausal"] = {
            "ms_mean": avg, "ms_median": statistics.median(ms[c]), "tflops": tf,
            "frac_of_measured_peak": tf / peak, "flops_per_call": F[c]}
    nc = mode_info["noncausal"]
    kernel_name = f"fa_fwd_sm103<{w.D},{'bf16' if w.dtype == 'bf16' else 'fp16'},noncausal>"
    roofline = {"bound": "tensor", "achieved": nc["tflops"], "peak": peak, "unit": "TFLOP/s",
                "frac": nc["tflops"] / peak, "traffic": _traffic_record(kernel_name),
                "kernel": kernel_name, "peak_source": f"bf16_tflops (burst, {peak_src})",
                "frac_of_sustained": nc["tflops"] / peak_sus}

    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.describe() + ", one non-causal + one causal call per step", "B": w.B,
                       "H": w.H, "N": w.N, "D": w.D, "l2": "flushed between timed calls (256 MiB write)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "modes": mode_info, "roofline": roofline,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                    "pipelined": "step i's calls overlap step i+1's input copies and step i-1's output copies "
                                 "(two device buffer sets, three streams)"},
            "clocks": clk, "gpu_launches": args.steps * len(modes), "wall_s_timed_region": wall}
    if bwd_info is not None:
        line["backward"] = bwd_info
    if args.config_steps > 0:
        # every task workload, outside the headline's timed region
        line["configs"] = config_timings(args.config_steps, dev, stream, flush, peak)
    if args.decode_steps > 0:
        # outside the timed region; a failure here is reported in the object
        # and leaves the line's own measurements as they are
        try:
            line["decode"] = decode_timings(args.decode_steps, dev, stream, flush, _peaks()[2])
        except Exception as e:
            line["decode"] = {"error": f"{type(e).__name__}: {e}"}
    if rank == 0 and not args.no_cpu_baseline:
        v_cpu, desc, cores, spent = cpu_oracle_sample(w, args.cpu_budget)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
