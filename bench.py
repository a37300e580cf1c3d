"""Benchmark of hybrid prefill+decode attention on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one hybrid batch: the fused persistent kernel
computes the chunked-prefill attention and every decode attention of the batch (one attention
layer of one serving iteration). The default run times the Yi-6B attention shape (32 query / 4 KV
heads, head_dim 128, one 2048-token chunk after a 28672-token prefix, 16 decodes with contexts
uniform in [16384, 32768], paged block 16) as the headline, the prefill-bound configuration;
the same JSON line carries, as keyed extras, the Llama-2-7B and Llama-3-8B configurations
(HBM-bound) and the two 200-iteration hybrid-batching trace mixes. Synthetic N(0,1) bf16 inputs.

Timing: CUDA events on the launching stream around each step. Between steps (outside the
events) a 1 GiB buffer is written and a 512 MiB one read, so every step starts with a cold L2
whose lines are clean: with the write alone, the ~126 MB of dirty lines it leaves would be
written back during the timed step (measured: 9-19 us of extra time per step). The headline
value is the fused variant's mean us/iter; the serial (two launches back to back) and
two-stream variants run on the same buffers for the speedup figures. `e2e` repeats the fused
step through the public C ABI from pinned host buffers (plan + upload + run + copies in the
timed region) and splits it into its parts.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]
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

METRIC = "hybrid prefill+decode attention µs/iter, % of roofline, speedup vs serial"
UNIT = "us/iter"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]),
                "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


L2_NOTE = ("flushed between steps: 1 GiB written, then 512 MiB read, so every step starts with a "
           "cold L2 that holds no dirty lines of the flush itself")


class L2Flush:
    """Between timed steps (outside the events): write a 1 GiB buffer (evicts everything the
    last step left in the 126 MB L2), then read a 512 MiB one, so the dirty lines of that write
    are written back here rather than inside the next timed step. The L2 the step sees is cold
    for all of its inputs, as under a profiler's cache flush."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(1 << 30, dtype=torch.uint8, device=device)
        self.r = torch.zeros(512 << 20, dtype=torch.uint8, device=device)

    def __call__(self):
        self.w.fill_(1)
        self.r.max()


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of a list of floats over all ranks (the list itself for one process).
    Every rank times the same work on its own GPU, so the job takes as long as its slowest rank."""
    if not dist:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _workload_name(cfg, batch) -> str:
    from hybrid_prefill_decode_gb300 import workloads as W
    name = W.CONFIG_NAMES.get(cfg) or W.PROFILE_CASES[cfg][0]
    return name + ", head_dim 128, paged block 16, bf16"


def _config_dict(args, batch, world):
    """The workload description both arms print (identical keys and values)."""
    d = {"workload": _workload_name(args.case or args.config, batch),
         "config_index": args.case or args.config,
         "l2": L2_NOTE,
         "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}
    if getattr(args, "append", False):
        d["kv_append"] = "new K/V rows written into the pools inside each step"
    return d


def _make_batch(args, device):
    from hybrid_prefill_decode_gb300 import workloads as W
    if args.case:
        return W.profile_case(args.case, device=device)
    return W.config(args.config, device=device)


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed region runs.

    Reads NVML through ctypes every ~1 ms (read-only queries), so even a timed region of a few
    milliseconds gets samples; if NVML cannot be loaded the summary says so."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device_index: int):
        self.dev = torch_device_index
        self.samples = []      # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.error = None
        self._stop = False
        self._thread = None

    def _handle(self):
        import ctypes
        import torch
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        props = torch.cuda.get_device_properties(self.dev)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        h = ctypes.c_void_p()
        if nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
            raise RuntimeError(f"no NVML device for bus id {bus}")
        return nvml, h

    def _loop(self, nvml, h):
        import ctypes
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop:
            if nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(0.001)

    def __enter__(self):
        import ctypes
        import threading
        try:
            nvml, h = self._handle()
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._thread = threading.Thread(target=self._loop, args=(nvml, h), daemon=True)
            self._thread.start()
            time.sleep(0.01)
        except Exception as e:  # no NVML: nothing sampled, say so
            self.error = str(e)
        return self

    def __exit__(self, *a):
        self._stop = True
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": [f"no samples ({self.error or 'region too short'})"],
                    "samples": 0}
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "nvml"}


def cpu_baseline(batch, target_s: float = 12.0):
    """The fp64 oracle as it stands, on this host's cores, on a bounded sample of the workload's
    query rows (every decode row and every k-th prefill row, all heads), scaled to one iteration
    by the number of visible (query, key) pairs."""
    import numpy as np
    import oracle
    Hq = batch.num_q_heads
    cu = batch.host_cu_seqlens
    pre_rows = []                         # (token index, visible keys)
    for s, (q, L) in enumerate(zip(batch.q_lens, batch.prefill_kv_lens)):
        for i in range(q):
            pre_rows.append((cu[s] + i, L - q + i + 1))
    dec_rows = [(d, L) for d, L in enumerate(batch.decode_kv_lens)]
    total_pairs = Hq * (sum(v for _, v in pre_rows) + sum(v for _, v in dec_rows))
    # calibrate on the decode rows, then pick the prefill stride to fill the time budget
    t0 = time.perf_counter()
    kinds = [1] * (len(dec_rows) * Hq)
    idx = [d for d, _ in dec_rows for _ in range(Hq)]
    heads = list(range(Hq)) * len(dec_rows)
    if kinds:
        oracle.rows(batch, kinds, idx, heads)
    t_dec = time.perf_counter() - t0
    dec_pairs = Hq * sum(v for _, v in dec_rows)
    rate = dec_pairs / max(t_dec, 1e-6)   # pairs per second
    stride = 1
    if pre_rows:
        want = max(1.0, target_s - t_dec) * rate
        pre_pairs_all = Hq * sum(v for _, v in pre_rows)
        stride = max(1, int(math.ceil(pre_pairs_all / want)))
    sample = pre_rows[::stride]
    t1 = time.perf_counter()
    if sample:
        oracle.rows(batch, [0] * (len(sample) * Hq), [r for r, _ in sample for _ in range(Hq)],
                    list(range(Hq)) * len(sample))
    t_pre = time.perf_counter() - t1
    samp_pairs = dec_pairs + Hq * sum(v for _, v in sample)
    elapsed = t_dec + t_pre
    us_per_iter = elapsed * 1e6 * total_pairs / max(samp_pairs, 1)
    return {"value": us_per_iter, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"all {len(dec_rows)} decode rows and every {stride}-th of "
                       f"{len(pre_rows)} prefill rows, all {Hq} heads "
                       f"({samp_pairs / total_pairs:.1%} of the iteration's visible pairs, "
                       f"{elapsed:.1f} s), scaled by visible (query, key) pairs"),
            "seconds": elapsed}


def run_reference(args, rank, world):
    """--impl reference: the fp64 CPU oracle timed on this host (rank 0 only)."""
    if rank != 0:
        return
    from hybrid_prefill_decode_gb300 import workloads as W
    batch = _make_batch(args, "cpu")
    vals = []
    for k in range(args.warmup + args.steps):
        r = cpu_baseline(batch, target_s=args.ref_step_s)
        if k >= args.warmup:
            vals.append(r)
    value = statistics.mean(v["value"] for v in vals)
    out = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": value / 1e3, "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": _config_dict(args, batch, world),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": vals[0]["cores"],
                            "kind": "oracle", "sample": vals[0]["sample"]},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


HEADLINE_CONFIG = 4           # Yi-6B shape, 2048-token chunk at 28K: the prefill-bound batch
EXTRA_CONFIGS = (2, 3)        # the HBM-bound batches
EXTRA_TRACES = ("a", "b")     # the long-context hybrid-batching mixes


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=None,
                    help="one configuration only (default: configuration 4 as the headline, with "
                         "configurations 2, 3 and the trace mixes a, b as extras in the same line)")
    ap.add_argument("--case", default=None, help="a small profiling case instead of --config")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-step-s", type=float, default=4.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="the headline configuration alone (no configurations 2, 3 or traces)")
    ap.add_argument("--only", default=None, help="profile mode: run only this variant, no extras")
    ap.add_argument("--trace", default=None, choices=["a", "b"],
                    help="the 200-iteration hybrid-batching trace (mix a or b) instead of --config")
    ap.add_argument("--trace-iters", type=int, default=200)
    ap.add_argument("--mix", action="store_true",
                    help="diagnostic: one instrumented fused launch of --config; prints the per-SM "
                         "prefill/decode mix from the kernel's own per-item records")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="decode attention over an FP8 (e4m3) cache: the decodes of --config, "
                         "with the bf16 cache of the same decodes timed beside it")
    ap.add_argument("--append", action="store_true",
                    help="every step also writes the iteration's new K/V rows into the pools "
                         "(pod_attn_run_append); the metric then includes that step")
    args = ap.parse_args()
    with_extras = (args.config is None and not args.case and not args.no_extras and
                   not args.only and not args.append)
    if args.config is None:
        args.config = HEADLINE_CONFIG

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    assert args.warmup >= 3 or args.only, "at least 3 warm-up steps"
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))

    from hybrid_prefill_decode_gb300 import binding as B
    from hybrid_prefill_decode_gb300 import build as build_mod
    from hybrid_prefill_decode_gb300 import roofline as R
    from hybrid_prefill_decode_gb300 import workloads as W
    build_mod.build()
    B.load()

    dev = torch.device(f"cuda:{local}")
    if args.trace:
        out = run_trace(args, args.trace, dev, B, R, W, world, dist)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return
    if args.kv_fp8:
        run_fp8(args, dev, B, R, W, rank, world, dist)
        return
    if args.mix:
        run_mix(args, dev, B, W, rank)
        return

    out = measure_config(args, args.config, args.case, dev, B, R, W, world, dist, local,
                         full=True)
    if out is None:                      # profile mode printed its own line
        return
    if with_extras:
        extras = {}
        for c in EXTRA_CONFIGS:
            extras[f"config{c}"] = _summary(
                measure_config(args, c, None, dev, B, R, W, world, dist, local, full=False))
        for mix in EXTRA_TRACES:
            extras[f"trace_{mix}"] = _trace_summary(
                run_trace(args, mix, dev, B, R, W, world, dist))
        out["extras"] = extras
        out["gpu_launches"] += sum(e.get("gpu_launches", 0) for e in extras.values())
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


def _summary(d):
    """The keyed extra of one configuration: its us/iter, fraction of the hybrid roofline and
    speedups over the serial and two-stream variants."""
    keys = ("value", "median_us", "serial_us", "streams_us", "speedup_vs_serial",
            "speedup_vs_streams", "tbs", "prefill_tflops", "gpu_launches")
    r = {k: d[k] for k in keys if k in d}
    r["workload"] = d["config"]["workload"]
    r["frac_of_t_star"] = d["hybrid_roofline"]["frac_of_t_star"]
    r["t_star_us"] = d["hybrid_roofline"]["t_star_us"]
    r["bound"] = d["roofline"]["bound"]
    r["clocks"] = d.get("clocks")
    return r


def _trace_summary(d):
    keys = ("value", "fused", "serial", "streams", "frac_of_t_star", "speedup_vs_serial",
            "speedup_vs_streams", "mean_t_star_us", "steps", "gpu_launches")
    r = {k: d[k] for k in keys if k in d}
    r["workload"] = d["config"]["workload"]
    return r


def measure_config(args, cfg, case, dev, B, R, W, world, dist, local, full):
    """One hybrid batch (configuration `cfg`, or the profiling case `case`): the fused, serial and
    two-stream variants timed on identical device buffers, cold L2 before every step. With
    `full`, also the step end to end through the C ABI (plan, upload, host copies, launch) with
    a breakdown of its parts, and the CPU oracle baseline. Returns the JSON dict (every rank),
    or None in profile mode."""
    import torch
    batch = W.profile_case(case, device=dev) if case else W.config(cfg, device=dev)
    work = R.batch_work(batch.num_q_heads, batch.num_kv_heads, batch.q_lens,
                        batch.prefill_kv_lens, batch.decode_kv_lens)
    hbm, tf_burst, tf_sust, peak_src = _peaks()
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(device=dev)
    o_p = torch.empty_like(batch.q_prefill)
    o_d = torch.empty_like(batch.q_decode)
    flush = L2Flush(dev)

    variants = [args.only] if args.only else ["fused", "serial", "streams"]
    plans = {}
    for v in variants:
        plan = B.Plan.for_batch(batch, variant=v)
        ws = plan.alloc_workspace(dev)
        plan.upload(ws, stream)
        plans[v] = (plan, ws)

    if args.append:
        # the new rows come separately; the pools start without them (NaN) and every step
        # writes them again (the same bytes: the step's work does not change)
        k_new, v_new, batch.k_pool, batch.v_pool = W.split_off_new_rows(batch)

    def step(v):
        plan, ws = plans[v]
        if args.append:
            plan.run_append(batch.q_prefill, batch.q_decode, k_new, v_new, batch.k_pool,
                            batch.v_pool, batch.block_tables, batch.cu_seqlens_q, batch.kv_lens,
                            o_p, o_d, ws, stream=stream, stream2=side)
        else:
            B.run_batch(plan, batch, ws, o_p, o_d, stream=stream, stream2=side)

    if args.only:                    # profiling mode: warm-up + K plain steps, nothing else
        for _ in range(args.warmup + args.steps):
            step(args.only)
        torch.cuda.synchronize()
        st = plans[args.only][0].device_status(plans[args.only][1])
        print(json.dumps({"profile_run": args.only, "status": st}))
        return None

    def timed(v, k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for a, b in evs:
            flush()                              # cold L2 for every step (outside the events)
            a.record(stream)
            step(v)
            b.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return [a.elapsed_time(b) * 1e3 for a, b in evs]

    for v in variants:
        for _ in range(args.warmup):
            step(v)
    torch.cuda.synchronize()
    for v in variants:
        assert plans[v][0].device_status(plans[v][1]) == B.OK, v

    results = {}
    clocks = None
    for v in variants:
        if v == "fused":
            with ClockSampler(local) as cs:
                results[v] = timed(v, args.steps)
            clocks = cs.summary()
        else:
            results[v] = timed(v, args.steps)
    for v in variants:
        assert plans[v][0].device_status(plans[v][1]) == B.OK, v

    def agg(us_list):
        return max_over_ranks([statistics.mean(us_list)], dist, dev)[0]

    us = {v: agg(results[v]) for v in variants}
    med = {v: statistics.median(results[v]) for v in variants}

    e2e = None
    if full and not args.no_e2e:
        e2e = _e2e(args, batch, plans["fused"][1], o_p, o_d, B, flush, stream, dist, dev, agg)

    t_fused = us["fused"] * 1e-6
    tstar = work.t_star(hbm, tf_burst)
    bound = work.bound(hbm, tf_burst)
    if bound == "hbm":
        achieved = work.bytes / t_fused / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": None,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src}
    else:
        achieved = work.prefill_flops / t_fused / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_burst, "unit": "TFLOP/s",
                "frac": achieved / tf_burst, "traffic": None,
                "peak_source": f"{peak_src} bf16 burst"}
    traffic = None if case else _traffic_from_profiles(cfg)
    if traffic is not None:
        roof["traffic"] = traffic
    cfg_args = argparse.Namespace(case=case, config=cfg, append=args.append)
    out = {
        "metric": METRIC, "value": us["fused"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us["fused"] / 1e3,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": _config_dict(cfg_args, batch, world),
        "median_us": med["fused"],
        "hybrid_roofline": {"t_star_us": tstar * 1e6, "frac_of_t_star": tstar / t_fused,
                            "bytes": work.bytes, "prefill_flops": work.prefill_flops,
                            "hbm_gbs": hbm, "bf16_tflops": tf_burst,
                            "frac_vs_8tbs_spec": (work.bytes / 8000e9) / t_fused},
        "tbs": work.bytes / t_fused / 1e12,
        "prefill_tflops": work.prefill_flops / t_fused / 1e12,
        "roofline": roof,
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if "serial" in us:
        out["serial_us"] = us["serial"]
        out["speedup_vs_serial"] = us["serial"] / us["fused"]
    if "streams" in us:
        out["streams_us"] = us["streams"]
        out["speedup_vs_streams"] = us["streams"] / us["fused"]
    if e2e:
        out["e2e"] = e2e
    if full and not args.no_cpu and world == 1:
        cpu_batch = batch.to("cpu")
        out["cpu_baseline"] = {k: v for k, v in cpu_baseline(cpu_batch).items() if k != "seconds"}
    return out


def _e2e(args, batch, ws, o_p, o_d, B, flush, stream, dist, dev, agg):
    """The fused step end to end through the C ABI, as a serving loop runs it: enqueue the copies
    of this step's q, block tables and lengths from pinned host buffers, plan the batch on the
    host while they run, upload the plan's work lists, launch, copy the outputs back, wait. Host
    time around the whole step; CUDA events split its device-side parts (the span between the
    input copies and the upload is the device waiting for the host's planning), host timers the
    planning and the other host calls."""
    import torch
    host = {k: getattr(batch, k).cpu().pin_memory() for k in
            ("q_prefill", "q_decode", "block_tables", "cu_seqlens_q", "kv_lens")}
    dq_p, dq_d = torch.empty_like(batch.q_prefill), torch.empty_like(batch.q_decode)
    dbt, dcu, dkv = (torch.empty_like(batch.block_tables), torch.empty_like(batch.cu_seqlens_q),
                     torch.empty_like(batch.kv_lens))
    ho_p = torch.empty(o_p.shape, dtype=o_p.dtype, pin_memory=True)
    ho_d = torch.empty(o_d.shape, dtype=o_d.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = ho_p.numel() * ho_p.element_size() + ho_d.numel() * ho_d.element_size()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]

    def e2e_step(parts):
        t0 = time.perf_counter()
        ev[0].record(stream)
        for dst, key in ((dq_p, "q_prefill"), (dq_d, "q_decode"), (dbt, "block_tables"),
                         (dcu, "cu_seqlens_q"), (dkv, "kv_lens")):
            dst.copy_(host[key], non_blocking=True)
        ev[1].record(stream)
        t1 = time.perf_counter()
        plan = B.Plan.for_batch(batch, variant="fused")   # host planning, beside the copies
        t2 = time.perf_counter()
        ev[2].record(stream)
        plan.upload(ws, stream)
        ev[3].record(stream)
        plan.run(dq_p, dq_d, batch.k_pool, batch.v_pool, dbt, dcu, dkv, o_p, o_d, ws,
                 stream=stream)
        ev[4].record(stream)
        ho_p.copy_(o_p, non_blocking=True)
        ho_d.copy_(o_d, non_blocking=True)
        ev[5].record(stream)
        t3 = time.perf_counter()
        stream.synchronize()
        t4 = time.perf_counter()
        if parts is not None:
            parts["plan_host"].append((t2 - t1) * 1e6)
            parts["enqueue_host"].append(((t1 - t0) + (t3 - t2)) * 1e6)
            parts["wait_host"].append((t4 - t3) * 1e6)
            parts["h2d_device"].append(ev[0].elapsed_time(ev[1]) * 1e3)
            parts["idle_for_plan_device"].append(ev[1].elapsed_time(ev[2]) * 1e3)
            parts["upload_device"].append(ev[2].elapsed_time(ev[3]) * 1e3)
            parts["kernel_device"].append(ev[3].elapsed_time(ev[4]) * 1e3)
            parts["d2h_device"].append(ev[4].elapsed_time(ev[5]) * 1e3)
        return (t4 - t0) * 1e6

    for _ in range(args.warmup):
        e2e_step(None)
    ts = []
    parts = {k: [] for k in ("plan_host", "enqueue_host", "wait_host", "h2d_device",
                             "idle_for_plan_device", "upload_device", "kernel_device",
                             "d2h_device")}
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for _ in range(args.steps):
        flush()
        torch.cuda.synchronize()
        ts.append(e2e_step(parts))
    return {"value": agg(ts), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "breakdown_us": {k: round(statistics.mean(v), 2) for k, v in parts.items()},
            "breakdown_note": ("plan_host: pod_attn_plan through the binding (runs while the "
                               "input copies do); enqueue_host: the step's other host calls; "
                               "wait_host: the final stream synchronisation; *_device: "
                               "CUDA-event spans on the stream in order: input copies, idle "
                               "until the plan is ready, upload, kernel, output copies")}


def run_trace(args, mix, dev, B, R, W, world, dist):
    """Configuration 5: every iteration of a seeded hybrid-batching trace is one step. The plan
    and upload of each iteration happen before its timed events (they are host work of the
    serving loop); the events time pod_attn_run. Reports mean/p50/p99 us/iter per variant and
    the sum of measured times over the sum of per-iteration hybrid rooflines."""
    import torch
    hbm, tf_burst, _, _ = _peaks()
    tr = W.trace(mix, iters=args.trace_iters, decode_targets=W.trace_decode_targets(
        torch.cuda.get_device_properties(dev).multi_processor_count))
    pool = W.TracePool(tr, device=dev)
    batches = [pool.batch(i) for i in range(len(tr.steps))]
    variants = ["fused", "serial", "streams"]
    plans = {v: [B.Plan.for_batch(b, variant=v) for b in batches] for v in variants}
    wsb = max(pl.workspace_bytes for v in variants for pl in plans[v])
    ws = {v: torch.empty(max(256, wsb), dtype=torch.uint8, device=dev) for v in variants}
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(device=dev)
    flush = L2Flush(dev)
    outs = [(torch.empty_like(b.q_prefill), torch.empty_like(b.q_decode)) for b in batches]
    tstar = [R.batch_work(b.num_q_heads, b.num_kv_heads, b.q_lens, b.prefill_kv_lens,
                          b.decode_kv_lens).t_star(hbm, tf_burst) * 1e6 for b in batches]
    times = {}
    for v in variants:
        for i in range(min(args.warmup, len(batches))):            # warm-up iterations
            plans[v][i].upload(ws[v], stream)
            B.run_batch(plans[v][i], batches[i], ws[v], *outs[i], stream=stream, stream2=side)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in batches]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for i, b in enumerate(batches):
            plans[v][i].upload(ws[v], stream)
            flush()
            evs[i][0].record(stream)
            B.run_batch(plans[v][i], b, ws[v], *outs[i], stream=stream, stream2=side)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        # per iteration, the slowest rank's time
        times[v] = max_over_ranks([a.elapsed_time(e) * 1e3 for a, e in evs], dist, dev)
        assert plans[v][-1].device_status(ws[v]) == B.OK, v

    def stats(xs):
        xs = sorted(xs)
        return {"mean": statistics.mean(xs), "p50": xs[len(xs) // 2],
                "p99": xs[min(len(xs) - 1, int(round(0.99 * (len(xs) - 1))))]}

    f = stats(times["fused"])
    return {"metric": METRIC, "value": f["mean"], "unit": UNIT, "n_gpus": world,
            "steps": len(batches), "warmup": args.warmup, "ms_per_step": f["mean"] / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"hybrid-batching trace mix {mix}: Llama-3-8B attention "
                                   f"(32/8, head_dim 128, paged block 16), 2048-token budget, "
                                   f"decodes first, {len(batches)} iterations",
                       "decode_targets": list(tr.decode_targets),
                       "l2": L2_NOTE},
            "fused": f, "serial": stats(times["serial"]), "streams": stats(times["streams"]),
            "sum_measured_over_sum_tstar": sum(times["fused"]) / sum(tstar),
            "frac_of_t_star": sum(tstar) / sum(times["fused"]),
            "speedup_vs_serial": sum(times["serial"]) / sum(times["fused"]),
            "speedup_vs_streams": sum(times["streams"]) / sum(times["fused"]),
            "mean_t_star_us": statistics.mean(tstar),
            "gpu_launches": len(batches),
            "pool_gb": pool.k_pool.numel() * 4 / 1e9}


def run_mix(args, dev, B, W, rank):
    """--mix: the per-SM mix of one fused launch, from the per-item records the kernel writes
    when the plan is instrumented (SM id, kind, start and end on the global timer). Cold L2 as
    in the timed runs; a diagnostic line, not a benchmark value."""
    import torch
    if rank != 0:
        return
    batch = _make_batch(args, dev)
    plan = B.Plan.for_batch(batch, instrument=True)
    ws = plan.alloc_workspace(dev)
    plan.upload(ws)
    flush = L2Flush(dev)
    for _ in range(max(3, args.warmup)):
        B.run_batch(plan, batch, ws)
    flush()
    B.run_batch(plan, batch, ws)
    torch.cuda.synchronize()
    assert plan.device_status(ws) == B.OK
    recs = plan.records(ws)
    t0 = min(r["t_start"] for r in recs)
    t1 = max(r["t_end"] for r in recs)
    span = (t1 - t0) / 1e3
    kinds = {}
    busy = {}
    end = {0: 0.0, 1: 0.0}
    dur = {0: [], 1: []}
    for r in recs:
        kinds.setdefault(r["smid"], set()).add(r["kind"])
        busy[r["cta"]] = busy.get(r["cta"], 0.0) + (r["t_end"] - r["t_start"]) / 1e3
        end[r["kind"]] = max(end[r["kind"]], (r["t_end"] - t0) / 1e3)
        dur[r["kind"]].append((r["t_end"] - r["t_start"]) / 1e3)
    n_sm = len(kinds)
    out = {"diagnostic": "per-SM prefill/decode mix of one fused launch (kernel records)",
           "config": _config_dict(args, batch, 1),
           "span_us": round(span, 1), "sms": n_sm,
           "sms_with_both_kinds": sum(1 for v in kinds.values() if v == {0, 1}),
           "sms_prefill_only": sum(1 for v in kinds.values() if v == {0}),
           "sms_decode_only": sum(1 for v in kinds.values() if v == {1}),
           "items": {"prefill": len(dur[0]), "decode": len(dur[1])},
           "mean_item_us": {k: (round(statistics.mean(v), 1) if v else None)
                            for k, v in (("prefill", dur[0]), ("decode", dur[1]))},
           "last_item_end_us": {"prefill": round(end[0], 1), "decode": round(end[1], 1)},
           "items_in_flight_per_cta": round(sum(busy.values()) / (span * max(1, len(busy))), 2)}
    print(json.dumps(out), flush=True)


def cpu_baseline_fp8(fb, target_s: float = 12.0):
    """The fp64 oracle of the FP8-cache decode on this host's cores, on the first decodes of the
    batch (as many as fill about `target_s`), scaled to the whole batch by cached rows read."""
    import oracle
    from hybrid_prefill_decode_gb300 import workloads as W
    lens = list(fb.decode_kv_lens)
    n, elapsed = 1, 0.0
    while True:
        sub = W.Fp8DecodeBatch(fb.num_q_heads, fb.num_kv_heads, fb.head_dim, fb.block_size,
                               lens[:n], fb.scale, fb.q_decode[:n], fb.k8, fb.v8, fb.k_scale,
                               fb.v_scale, fb.block_tables[:n], fb.kv_lens[:n], fb.seed)
        t0 = time.perf_counter()
        oracle.decode_fp8(sub)
        elapsed = time.perf_counter() - t0
        if n == len(lens) or elapsed * (2 * n) / n > target_s:
            break
        n = min(len(lens), 2 * n)
    us = elapsed * 1e6 * sum(lens) / sum(lens[:n])
    return {"value": us, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": (f"the first {n} of {len(lens)} decodes, all {fb.num_q_heads} heads "
                       f"({sum(lens[:n]) / sum(lens):.1%} of the cached rows read, "
                       f"{elapsed:.1f} s), scaled by cached rows")}


def run_fp8(args, dev, B, R, W, rank, world, dist):
    """--kv-fp8: one step = decode attention of every decode of --config over an e4m3 cache with
    per-(kv-head, channel) K scales and per-(row, kv-head) V scales (pod_attn_run_decode_fp8).
    The bf16-cache decode of the same decodes (pod_attn_run, decode-only plan) is timed beside it
    on the same lengths; the roofline counts the FP8 cache's bytes."""
    import torch
    hbm, _, _, peak_src = _peaks()
    Hq, Hkv, _, _, dkv = W.config_lengths(args.config)
    fb = W.make_fp8_decode_batch(Hq, Hkv, dkv, seed=args.config, device=dev)
    bb = W.make_batch(Hq, Hkv, [], [], dkv, seed=args.config, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    p8 = B.Plan(Hq, Hkv, [], list(dkv), len(dkv), fb.num_blocks, fb.max_blocks_per_seq, fb.scale,
                kv_fp8=True)
    ws8 = p8.alloc_workspace(dev)
    p8.upload(ws8, stream)
    o8 = torch.empty_like(fb.q_decode)
    p16 = B.Plan.for_batch(bb)
    ws16 = p16.alloc_workspace(dev)
    p16.upload(ws16, stream)
    o16 = torch.empty_like(bb.q_decode)
    op16 = torch.empty_like(bb.q_prefill)

    def step8():
        p8.run_decode_fp8(fb.q_decode, fb.k8, fb.v8, fb.k_scale, fb.v_scale, fb.block_tables,
                          fb.kv_lens, o8, ws8, stream=stream)

    def step16():
        B.run_batch(p16, bb, ws16, op16, o16, stream=stream)

    def timed(fn, k):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(k)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        for a, b in evs:
            flush()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return [a.elapsed_time(b) * 1e3 for a, b in evs]

    def agg(xs):
        return max_over_ranks([statistics.mean(xs)], dist, dev)[0]

    for fn in (step8, step16):
        for _ in range(args.warmup):
            fn()
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as cs:
        t8 = timed(step8, args.steps)
    clocks = cs.summary()
    t16 = timed(step16, args.steps)
    assert p8.device_status(ws8) == B.OK and p16.device_status(ws16) == B.OK
    us8, us16 = agg(t8), agg(t16)

    e2e = None
    if not args.no_e2e:
        host = {k: getattr(fb, k).cpu().pin_memory() for k in ("q_decode", "block_tables",
                                                               "kv_lens")}
        dq, dbt, dkv_t = (torch.empty_like(fb.q_decode), torch.empty_like(fb.block_tables),
                          torch.empty_like(fb.kv_lens))
        ho = torch.empty(o8.shape, dtype=o8.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in host.values())

        def e2e_step():
            for dst, key in ((dq, "q_decode"), (dbt, "block_tables"), (dkv_t, "kv_lens")):
                dst.copy_(host[key], non_blocking=True)
            plan = B.Plan(Hq, Hkv, [], list(dkv), len(dkv), fb.num_blocks,
                          fb.max_blocks_per_seq, fb.scale, kv_fp8=True)
            plan.upload(ws8, stream)
            plan.run_decode_fp8(dq, fb.k8, fb.v8, fb.k_scale, fb.v_scale, dbt, dkv_t, o8, ws8,
                                stream=stream)
            ho.copy_(o8, non_blocking=True)
            stream.synchronize()
            return plan

        for _ in range(args.warmup):
            e2e_step()
        ts = []
        for _ in range(args.steps):
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e2e_step()
            ts.append((time.perf_counter() - t0) * 1e6)
        e2e = {"value": agg(ts), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(ho.numel() * ho.element_size())}
    if rank != 0:
        return
    nbytes = R.fp8_decode_bytes(Hq, Hkv, dkv)
    bytes16 = R.batch_work(Hq, Hkv, [], [], dkv).bytes
    achieved = nbytes / (us8 * 1e-6) / 1e9
    out = {"metric": "FP8-cache decode attention µs/iter", "value": us8, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": us8 / 1e3, "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "e4m3 cache, f16 MMA, fp32 accumulate",
           "data": "synthetic",
           "config": {"workload": (f"the {len(dkv)} decodes of {W.CONFIG_NAMES[args.config]}, "
                                   f"head_dim 128, paged block 16, e4m3 K/V with per-(kv-head, "
                                   f"channel) K and per-(row, kv-head) V fp32 scales"),
                      "config_index": args.config,
                      "l2": L2_NOTE,
                      "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
           "median_us": statistics.median(t8),
           "bf16_cache_us": us16, "speedup_vs_bf16_cache": us16 / us8,
           "bf16_cache_tbs": bytes16 / (us16 * 1e-6) / 1e12,
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                        "frac": achieved / hbm, "traffic": None,
                        "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                        "algorithmic_bytes": nbytes},
           "gpu_launches": args.steps, "clocks": clocks}
    if e2e:
        out["e2e"] = e2e
    if not args.no_cpu and world == 1:
        out["cpu_baseline"] = cpu_baseline_fp8(fb.to("cpu"))
    print(json.dumps(out), flush=True)


def _traffic_from_profiles(cfg):
    """DRAM bytes (read + write) per launch of the fused kernel, from the committed ncu summary
    `profiles/traffic_config<cfg>.md` (its line `dram_bytes_per_launch: N`), if present."""
    path = os.path.join(ROOT, "profiles", f"traffic_config{cfg}.md")
    try:
        for line in open(path):
            if line.strip().startswith("dram_bytes_per_launch:"):
                return int(line.split(":", 1)[1].strip())
    except (OSError, ValueError):
        pass
    return None


if __name__ == "__main__":
    main()
