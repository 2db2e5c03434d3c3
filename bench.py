#!/usr/bin/env python3
"""Benchmark of libbeamnorm on GB300: µs per call and achieved HBM GB/s.

One step = one fused finalize_reduce_norm call (per-shard MoE finalize with
local BF16 rounding, rank-ordered FP32 sum, post-RMSNorm, residual add,
pre-RMSNorm) over one batch of synthetic input resident in HBM.  The default
workload is R=8 shards, H=8192, top-k=10, T=1024 tokens (1.53 GB per call,
far larger than L2, so no flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload C4:1024] [--no-sweep] [--no-e2e] [--no-cpu]

Rank 0 prints ONE JSON line on stdout; progress goes to stderr.  Under
torchrun each rank runs its own replica of the workload (weak scaling); the
time is the maximum over ranks.  ``--impl reference`` times the CPU oracle
(plain single-threaded C) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from tp_reduce_residual_gb300 import inputs  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (% of GB300 peak) vs tokens T, per H/R/top-k"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0       # GB300 HBM3e nominal, the peak the workload's target names
L2_ROTATION = 8                # rotate over input sets covering at least this many L2s
L2_BYTES_FALLBACK = 129 * 1024 * 1024


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; also exercised with gloo on CPU in tests)

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value: float, device="cpu") -> float:
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def row_range(T: int, world: int, rank: int):
    """Contiguous token rows of one rank when a batch is sharded by token."""
    base, extra = divmod(T, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


# ---------------------------------------------------------------------------------------
# measured peaks, clocks, profile evidence

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C++ source with comments and blank space removed (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments do not count): the recorded
    ncu traffic stays valid across comment edits and lapses on any code change."""
    h = hashlib.sha256()
    for name in ("bn_device.cuh", "bn_kernels.cu", "bn_internal.h"):
        with open(os.path.join(ROOT, "tp_reduce_residual_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload_key: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload_key)
        if e and e.get("kernel_hash") == kernel_source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception as e:  # no nvidia-smi: report no clocks
            log(f"clock sampling unavailable: {e}")
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# workloads

def parse_workload(spec: str):
    """'C4:1024' -> (Workload, T)."""
    name, _, t = spec.partition(":")
    wl = inputs.WORKLOADS[int(name.lstrip("Cc"))]
    T = int(t) if t else wl.tokens[-1]
    return wl, T


def workload_bytes(wl, T, split=False, with_shared=True):
    return inputs.algorithmic_bytes(wl.op, wl.R, T, wl.H, wl.k, split=split, with_shared=with_shared)


def headline_sets(B, l2):
    """Input sets the headline loop rotates over: one when a call's inputs are
    at least twice L2 (the default workload), else enough to pass 8x L2, at
    most 64."""
    if B >= 2 * l2:
        return 1
    return int(min(64, max(1, math.ceil(8 * l2 / B))))


def l2_label(B, l2):
    """How the headline loop keeps its inputs out of L2, for the config."""
    n = headline_sets(B, l2)
    if n == 1:
        return f"inputs {B / 1e9:.2f} GB per step > L2 {l2 / 1e6:.0f} MB; no flush"
    warm = "" if n * B >= 8 * l2 else ", below 8x L2: partly L2-warm"
    return (f"inputs rotate over {n} sets ({n * B / 1e9:.2f} GB{warm}) against L2 "
            f"{l2 / 1e6:.0f} MB; no flush")


def line_config(wl, T, B, world, with_ws, l2):
    """The workload description both arms print (the same keys and values)."""
    return {"workload": wl.describe(T), "op": wl.op, "R": wl.R, "H": wl.H, "k": wl.k, "T": T,
            "bytes_per_step": B, "parallelism": f"replicas x{world}", "workspace": with_ws,
            "l2": l2_label(B, l2)}


def call_fused(bn, d, res, out, stream=None, workspace=None):
    if d["op"] == "reduce_norm":
        bn.reduce_norm(d["partials"], res, d["gamma_post"], d["gamma_pre"], d["eps"], out=out,
                       stream=stream)
    else:
        bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=out, stream=stream,
                                workspace=workspace)


def call_split(bn, d, res, out, s):
    bn.finalize_reduce_only(d["expert_out"], d["perm"], d["w"], d["shared"], sum_out=s)
    bn.norm_only(s, res, d["gamma_post"], d["gamma_pre"], d["eps"], out=out)


def clone_set(d):
    """A copy of an input set at new addresses (same values)."""
    c = {}
    for key, v in d.items():
        c[key] = v.clone() if isinstance(v, torch.Tensor) else v
    return c


# ---------------------------------------------------------------------------------------
# the timed headline (our arm)

def time_headline(bn, wl, T, steps, warmup, dev_index, use_workspace=False, l2=L2_BYTES_FALLBACK):
    """Back-to-back calls on a created stream: programmatic dependent launch
    (the next call's launch and setup overlapping the previous kernel) takes
    effect on created streams and in graphs, not on the legacy default stream.
    use_workspace: the finalize calls take a workspace (rows over many CTAs
    where the shape is served).  A workload smaller than twice L2 rotates
    over several input sets (headline_sets)."""
    d = inputs.make_inputs(wl, T, device="cuda")
    n_sets = headline_sets(workload_bytes(wl, T), l2)
    sets = [d] + [clone_set(d) for _ in range(n_sets - 1)]
    ress = [s["residual"].clone() for s in sets]
    outs = [torch.empty_like(ress[0]) for _ in sets]
    it = [0]

    def call(workspace):
        i = it[0] % n_sets
        it[0] += 1
        call_fused(bn, sets[i], ress[i], outs[i], workspace=workspace)

    ws = None
    if use_workspace and wl.op == "finalize_reduce_norm":
        ws = bn.finalize_workspace(wl.R, T, wl.k, wl.H, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call(ws)
    torch.cuda.synchronize()
    if bn.check_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    sampler = ClockSampler(dev_index)
    sampler.start()
    time.sleep(0.3)  # let the sampler attach before the load starts
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            call(ws)
        end.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = start.elapsed_time(end)
    # keep the GPU loaded (untimed) until the clock record spans at least one second
    t_extra = time.time() + max(0.0, 1.0 - elapsed_ms / 1000.0)
    while time.time() < t_extra:
        with torch.cuda.stream(stream):
            for _ in range(20):
                call(ws)
        torch.cuda.synchronize()
    clocks = sampler.stop()
    if bn.check_device_error() != 0:
        raise RuntimeError("device error in the timed region")
    del d, sets, ress, outs, ws
    torch.cuda.empty_cache()
    return elapsed_ms, clocks


def time_e2e(bn, wl, T, steps, copy_streams=4):
    """The same call through the public API with host buffers: every step copies
    the inputs from pinned host memory and reads both outputs back.  Two
    device input sets alternate, so that one step's uploads (split by leading
    dimension over `copy_streams` side streams, several copy engines) overlap
    the previous step's call and downloads, as a serving loop would pipeline
    them; a set is overwritten only after the downloads of the step that last
    used it.  Every step still moves all of its bytes inside the timed region."""
    dd = inputs.make_inputs(wl, T, device="cuda")
    host = {k: (v.cpu().pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in dd.items()}
    devs = [{k: (torch.empty_like(v) if isinstance(v, torch.Tensor) else v) for k, v in dd.items()}
            for _ in range(2)]
    del dd
    outs = [torch.empty_like(devs[0]["residual"]) for _ in range(2)]
    out_h = [torch.empty(outs[0].shape, dtype=outs[0].dtype, pin_memory=True) for _ in range(2)]
    res_h = [torch.empty(outs[0].shape, dtype=outs[0].dtype, pin_memory=True) for _ in range(2)]
    names = [k for k, v in host.items() if isinstance(v, torch.Tensor)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = 2 * outs[0].numel() * outs[0].element_size()

    main = torch.cuda.current_stream()
    side = [torch.cuda.Stream() for _ in range(max(1, copy_streams))]
    down = torch.cuda.Stream()
    pieces = []  # per set: (host piece, device piece), largest first
    for dev in devs:
        ps = []
        for k in names:
            nparts = min(len(side), host[k].shape[0]) if host[k].dim() > 0 else 1
            for hp, dp in zip(host[k].chunk(nparts), dev[k].chunk(nparts)):
                ps.append((hp, dp))
        ps.sort(key=lambda x: -x[0].numel() * x[0].element_size())
        pieces.append(ps)
    freed = [torch.cuda.Event() for _ in range(2)]  # set b's downloads are done
    for ev in freed:
        ev.record(down)

    def step(i):
        b = i & 1
        load = [0] * len(side)
        for s_ in side:
            s_.wait_event(freed[b])
        for hp, dp in pieces[b]:   # largest first onto the least loaded stream
            j = load.index(min(load))
            with torch.cuda.stream(side[j]):
                dp.copy_(hp, non_blocking=True)
            load[j] += hp.numel() * hp.element_size()
        for s_ in side:
            main.wait_stream(s_)
        call_fused(bn, devs[b], devs[b]["residual"], outs[b])
        down.wait_stream(main)
        with torch.cuda.stream(down):
            out_h[b].copy_(outs[b], non_blocking=True)
            res_h[b].copy_(devs[b]["residual"], non_blocking=True)
            freed[b].record(down)

    step(0)
    step(1)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(main)
    for s_ in side + [down]:
        s_.wait_stream(main)
    for i in range(steps):
        step(i)
    for s_ in side + [down]:
        main.wait_stream(s_)
    end.record(main)
    torch.cuda.synchronize()
    barrier()
    ms = start.elapsed_time(end)
    del host, devs, outs
    torch.cuda.empty_cache()
    return ms, h2d, d2h


# ---------------------------------------------------------------------------------------
# per-config sweep (µs/call vs T), CUDA-graph timing as on the pages

def graph_time_us(fn_list, reps=10):
    """Capture fn_list (one call each) in a CUDA graph; median per-call µs over reps."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for fn in fn_list[:2]:
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for fn in fn_list:
            fn()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1000.0 / len(fn_list))
    del g
    return statistics.median(times)


def sweep(bn, peak, l2_bytes, max_sets=64):
    rows = []
    for wl in inputs.WORKLOADS:
        for T in wl.tokens:
            B = workload_bytes(wl, T)
            base = inputs.make_inputs(wl, T, device="cuda")
            n_sets = int(min(max_sets, max(1, math.ceil(L2_ROTATION * l2_bytes / B))))
            sets = [base] + [clone_set(base) for _ in range(n_sets - 1)]
            outs = [torch.empty_like(base["residual"]) for _ in range(n_sets)]
            hot = graph_time_us([lambda: call_fused(bn, base, base["residual"], outs[0])] * 20)
            ncalls = max(20, n_sets)
            cold_fns = [(lambda i=i: call_fused(bn, sets[i % n_sets], sets[i % n_sets]["residual"],
                                               outs[i % n_sets])) for i in range(ncalls)]
            cold = graph_time_us(cold_fns)
            row = {"workload": wl.describe(T), "cfg": f"C{wl.index}", "T": T, "bytes": B,
                   "us_cold": round(cold, 3), "us_hot": round(hot, 3),
                   "gbs_cold": round(B / cold / 1e3, 1), "frac_cold": round(B / cold / 1e3 / peak, 4),
                   "frac_cold_nominal": round(B / cold / 1e3 / NOMINAL_HBM_GBS, 4),
                   "input_sets": n_sets,
                   "l2_cold": bool(n_sets * B >= L2_ROTATION * l2_bytes)}
            if wl.op == "finalize_reduce_norm" and bn.finalize_workspace_bytes(wl.R, T, wl.k, wl.H):
                # the same calls with a workspace: each token row over many CTAs
                ws = bn.finalize_workspace(wl.R, T, wl.k, wl.H, device="cuda")
                ws_fns = [(lambda i=i: call_fused(bn, sets[i % n_sets], sets[i % n_sets]["residual"],
                                                  outs[i % n_sets], workspace=ws))
                          for i in range(ncalls)]
                wu = graph_time_us(ws_fns)
                row.update(us_ws_cold=round(wu, 3), frac_ws_cold=round(B / wu / 1e3 / peak, 4))
                del ws
            if wl.index == 4:
                Bs = workload_bytes(wl, T, split=True)
                sums = [torch.empty(T, wl.H, device="cuda") for _ in range(n_sets)]
                split_fns = [(lambda i=i: call_split(bn, sets[i % n_sets], sets[i % n_sets]["residual"],
                                                     outs[i % n_sets], sums[i % n_sets]))
                             for i in range(ncalls)]
                su = graph_time_us(split_fns)
                row.update(us_split_cold=round(su, 3), split_bytes=Bs,
                           fusion_gain=round(su / cold, 3))
                del sums
            if bn.check_device_error() != 0:
                raise RuntimeError(f"device error in sweep {wl.describe(T)}")
            log(f"sweep {row}")
            rows.append(row)
            del base, sets, outs
            torch.cuda.empty_cache()
    return rows


# ---------------------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)

def host_cpu() -> dict:
    """The host the oracle runs on: logical CPUs and the CPU's name."""
    name = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip() in ("model name", "Model", "Hardware") and val.strip():
                    name = val.strip()
                    break
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "cpu": name, "arch": platform.machine()}


def oracle_sample_time(wl, T, target_s, seed_rows=0):
    """Time the oracle on enough sampled token rows of the workload to take
    about target_s seconds; return (GB/s, rows, seconds)."""
    import numpy as np

    import oracle

    d = inputs.make_inputs(wl, T, device="cuda")

    def run(rows):
        c = inputs.to_numpy(inputs.select_rows(d, rows))
        t0 = time.perf_counter()
        if wl.op == "reduce_norm":
            oracle.reduce_norm(c["partials"], c["residual"], c["gamma_post"], c["gamma_pre"], c["eps"])
        else:
            oracle.finalize_reduce_norm(c["expert_out"], c["perm"], c["w"], c["shared"], c["residual"],
                                        c["gamma_post"], c["gamma_pre"], c["eps"])
        return time.perf_counter() - t0

    rng = np.random.default_rng(seed_rows)
    probe = sorted(rng.choice(T, size=min(T, 4), replace=False).tolist())
    t_probe = run(probe) / len(probe)
    n = int(max(1, min(T, target_s / max(t_probe, 1e-6))))
    rows = sorted(rng.choice(T, size=n, replace=False).tolist())
    secs = run(rows)
    B = workload_bytes(wl, n)
    del d
    torch.cuda.empty_cache()
    return B / secs / 1e9, n, secs


# ---------------------------------------------------------------------------------------

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="C4:1024")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--workspace", action="store_true",
                    help="finalize calls of the timed loop take a workspace (T <= 8)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--copy-streams", type=int, default=4,
                    help="side streams for the per-step host-to-device copies of the e2e leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: approximate total CPU seconds of the run")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        log("warning: fewer than 3 warm-up steps")

    rank, world, local = dist_env()
    wl, T = parse_workload(args.workload)
    B = workload_bytes(wl, T)
    peak, peak_kind = measured_peak()

    if args.impl == "reference":
        return main_reference(args, rank, world, wl, T, B)

    torch.cuda.set_device(local)
    dist_init("nccl")
    import __graft_entry__
    __graft_entry__.build()
    from tp_reduce_residual_gb300 import beamnorm as bn

    dev_index = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev_index)
    l2 = getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK
    log(f"rank {rank}/{world} on {props.name}: {wl.describe(T)}, {B / 1e9:.3f} GB per call")

    elapsed_ms, clocks = time_headline(bn, wl, T, args.steps, args.warmup, dev_index,
                                       use_workspace=args.workspace, l2=l2)
    with_ws = bool(args.workspace and wl.op == "finalize_reduce_norm"
                   and bn.finalize_workspace_bytes(wl.R, T, wl.k, wl.H))
    elapsed_ms = max_over_ranks(elapsed_ms, device="cuda")
    ms_per_step = elapsed_ms / args.steps
    achieved = B / (ms_per_step * 1e-3) / 1e9
    value = world * B * args.steps / (elapsed_ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        ms, h2d, d2h = time_e2e(bn, wl, T, args.e2e_steps, args.copy_streams)
        ms = max_over_ranks(ms, device="cuda")
        e2e = {"value": round(world * B * args.e2e_steps / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(ms / args.e2e_steps, 4), "copy_streams": args.copy_streams,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    rows = None
    if not args.no_sweep and rank == 0:
        rows = sweep(bn, peak, l2)

    cpu = None
    if not args.no_cpu and rank == 0:
        gbs, n, secs = oracle_sample_time(wl, T, args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} of {T} token rows of {wl.describe(T)}, {secs:.1f} s single-threaded",
               "host": host_cpu()}

    if rank == 0:
        key = f"C{wl.index}:{T}"
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "us_per_call": round(ms_per_step * 1000.0, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "io_dtype": "bf16", "data": "synthetic",
            "config": line_config(wl, T, B, world, with_ws, l2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_kind": peak_kind,
                         "peak_nominal": NOMINAL_HBM_GBS,
                         "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                         "traffic": None if with_ws else recorded_traffic(key)},
            "clocks": clocks,
            "gpu_launches": args.steps,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "sweep": rows,
        }
        print(json.dumps(line), flush=True)
    return 0


def main_reference(args, rank, world, wl, T, B):
    """The reference arm: the CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return 0
    import numpy as np

    import oracle

    torch.manual_seed(0)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    # bounded per-step sample: a few token rows, sized so the whole run takes ~1 minute
    d = inputs.make_inputs(wl, min(T, 64) if dev == "cpu" else T, device=dev)
    Tg = d["T"]
    rng = np.random.default_rng(0)

    def sample(n):
        rows = sorted(rng.choice(Tg, size=n, replace=False).tolist())
        return inputs.to_numpy(inputs.select_rows(d, rows))

    def run(c):
        if wl.op == "reduce_norm":
            oracle.reduce_norm(c["partials"], c["residual"], c["gamma_post"], c["gamma_pre"], c["eps"])
        else:
            oracle.finalize_reduce_norm(c["expert_out"], c["perm"], c["w"], c["shared"], c["residual"],
                                        c["gamma_post"], c["gamma_pre"], c["eps"])

    probe = sample(2)
    t0 = time.perf_counter()
    run(probe)
    per_row = (time.perf_counter() - t0) / 2
    total_steps = args.steps + args.warmup
    n = int(max(1, min(Tg, args.ref_seconds / total_steps / max(per_row, 1e-6))))
    c = sample(n)
    for _ in range(args.warmup):
        run(c)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(c)
    secs = time.perf_counter() - t0
    Bn = workload_bytes(wl, n)
    value = Bn * args.steps / secs / 1e9
    l2 = L2_BYTES_FALLBACK
    if torch.cuda.is_available():
        l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0) or L2_BYTES_FALLBACK
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1000.0, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic",
        "config": line_config(wl, T, B, world, False, l2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} token rows of {wl.describe(T)} per step "
                                   f"({Bn} algorithmic bytes)", "host": host_cpu()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
