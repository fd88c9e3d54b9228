#!/usr/bin/env python
"""Benchmark of the fused SwiGLU MLP forward + backward on GB300.

Metric: fwd+bwd TFLOPS with the pages' FLOP convention 18 M D H (M = B S) and
its fraction of the measured dense-bf16 tensor peak.  Workload: B=8, S=8192,
D=4096, H=11008, bf16 storage with fp32 accumulation, seeded synthetic data
(X ~ N(0,1), Wg/Wu ~ N(0,1/D), Wd ~ N(0,1/H), dY ~ N(0,1e-2)).

One step = swiglu_mlp_fwd + swiglu_mlp_bwd (all six kernels) on device-resident
inputs; every input is larger than the 129 MB L2, so no flush is needed.
Prints ONE JSON line (rank 0).  Under torchrun each rank runs an independent
replica (the path has no exchange step on one GPU): value = all ranks' FLOPs /
the slowest rank's time.

--impl reference times the CPU fp64 oracle on a bounded token sample of the
same workload (the reference arm); only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    "B8_S8192_D4096_H11008": dict(B=8, S=8192, D=4096, H=11008),
    "B8_S4096_D2048_H5632": dict(B=8, S=4096, D=2048, H=5632),
    "B8_S2048_D1024_H2816": dict(B=8, S=2048, D=1024, H=2816),
    # the main workload's layer at 1/8 and 1/4 of its tokens: small enough for
    # multi-metric ncu captures, from which its per-launch traffic is scaled
    "B1_S8192_D4096_H11008": dict(B=1, S=8192, D=4096, H=11008),
    "B2_S8192_D4096_H11008": dict(B=2, S=8192, D=4096, H=11008),
}
MAIN = "B8_S8192_D4096_H11008"
# the pages' own number for this workload: 1049.66 ms on an RTX 5060 Ti
# (SM120), i.e. 18 M D H / t = 50.67 TFLOPS ("Training results" table)
PAGES_TFLOPS = {MAIN: 18.0 * 65536 * 4096 * 11008 / 1.04966 / 1e12}
NOGRAD_S = [1, 2, 4, 8, 16, 32, 48, 64, 128, 256]
CPU_SAMPLE_TOKENS = 256
REF_STEP_TOKENS = 8


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _strip_comments(src: str) -> str:
    """C/CUDA source without its comments and blank lines (string literals in
    these sources hold no comment markers)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())


def _csrc_hash() -> str:
    """Hash of the kernel sources' code (comments excluded), which keys the
    committed ncu traffic figures to the kernels they were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "backward_tcgen05_tma_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(kernel: str, workload: str):
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(workload, {}).get(kernel)
    if not e or e.get("csrc_hash") != _csrc_hash():
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_over_ranks(sec: float, flops_per_rank: float, world: int, device="cpu"):
    """Replicas: every rank times its own steps; the job's step time is the
    slowest rank's (all_reduce MAX) and the job's throughput counts every
    rank's work.  Returns (max seconds per step, job TFLOPS)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([sec], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        sec = float(t.item())
    return sec, flops_per_rank * world / sec / 1e12


def _config(workload, w, dtype, world):
    return {"workload": workload, "B": w["B"], "S": w["S"], "D": w["D"], "H": w["H"],
            "M": w["B"] * w["S"], "dtype": dtype, "parallelism": "replicas%d" % world,
            "l2": "inputs larger than L2 (no flush)"}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import torch

    import oracle
    from backward_tcgen05_tma_gb300 import metrics, synthetic
    w = WORKLOADS[args.workload]
    D, H = w["D"], w["H"]
    m = REF_STEP_TOKENS
    t = synthetic.make_inputs(m, D, H, "bf16", seed=0, device="cpu", kind="device")
    cores = oracle.num_threads()

    def step():
        f = oracle.forward(t["X"], t["Wg"], t["Wu"], t["Wd"])
        oracle.backward(t["dY"], t["X"], t["Wg"], t["Wu"], t["Wd"], f)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = metrics.fwd_bwd_flops(m, D, H) / dt / 1e12
    sample = ("fwd+bwd of %d token rows per step through the fp64 oracle, full D=%d, H=%d "
              "weights of the workload" % (m, D, H))
    line = {"impl": "reference", "metric": "SwiGLU MLP fwd+bwd TFLOPS (18*M*D*H)",
            "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(args.workload, w, "bf16", world),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def _alloc(M, D, H, dt, device, minimal_ws=False):
    import torch
    from backward_tcgen05_tma_gb300 import api
    size = api.lib().swiglu_mlp_workspace_min_bytes if minimal_ws else \
        api.lib().swiglu_mlp_workspace_bytes
    e = {"Y": torch.empty(M, D, dtype=dt, device=device),
         "saved": torch.empty(M, 3 * H, dtype=dt, device=device),
         "dX": torch.empty(M, D, dtype=dt, device=device),
         "dWgu": torch.empty(2 * H, D, dtype=dt, device=device),
         "dWd": torch.empty(D, H, dtype=dt, device=device)}
    e["ws"] = torch.zeros(max(size(M, D, H, api.dtype_code(dt), op)
                              for op in (api.SWIGLU_OP_FWD, api.SWIGLU_OP_BWD)),
                          dtype=torch.uint8, device=device)
    return e


def _step(api, t, o):
    api.swiglu_mlp_fwd(t["X"], t["Wgu"], t["Wd"], out=o, ws=o["ws"])
    n = api.swiglu_mlp_last_launch_count()
    api.swiglu_mlp_bwd(t["dY"], t["X"], t["Wgu"], t["Wd"], o["saved"], out=o, ws=o["ws"])
    return n + api.swiglu_mlp_last_launch_count()


def _kernel_flops(name, M, D, H):
    return {"gate_up_swiglu": 2.0 * M * 2 * H * D, "down_proj": 2.0 * M * D * H,
            "dgu_inplace": 2.0 * M * H * D, "dwd": 2.0 * D * H * M,
            "dwgu": 2.0 * 2 * H * D * M, "dx": 2.0 * M * D * 2 * H}[name]


def _time_training(api, w, dtype_name, steps, warmup, seed, device, profile=False,
                   minimal_ws=False):
    """Times `steps` fwd+bwd steps (CUDA events on the launching stream);
    returns (mean seconds per step, kernel launches, per-kernel profile,
    buffers, median seconds per step).

    With profile=True a second pass of the same number of steps runs with the
    library's per-kernel events; they sit between the kernels and so launch
    them in plain stream order (no programmatic overlap), which is why the
    step time comes from the first, unprofiled pass."""
    import torch
    from backward_tcgen05_tma_gb300 import synthetic
    dt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype_name]
    M, D, H = w["B"] * w["S"], w["D"], w["H"]
    t = synthetic.make_inputs(M, D, H, dtype_name, seed=seed, device=device, kind="device")
    o = _alloc(M, D, H, dt, device, minimal_ws)
    for _ in range(warmup):
        _step(api, t, o)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    # one event after each step (a marker on the same stream: no extra sync)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    launches = 0
    ev[0].record(st)
    for i in range(steps):
        launches += _step(api, t, o)
        ev[i + 1].record(st)
    torch.cuda.synchronize()
    sec = ev[0].elapsed_time(ev[-1]) / 1e3 / steps
    med = statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(steps)) / 1e3
    prof = None
    if profile:
        api.swiglu_mlp_profile_read()
        api.swiglu_mlp_profile_enable(True)
        for _ in range(steps):
            _step(api, t, o)
        torch.cuda.synchronize()
        api.swiglu_mlp_profile_enable(False)
        prof = api.swiglu_mlp_profile_read()
    return sec, launches, prof, (t, o), med


def _e2e(api, t, o, steps):
    """The same step fed from and returned to the host, as a training loop
    would run it: every step copies its X and dY from pinned host memory and
    reads its result -- the parameter gradients dWgu, dWd, what the optimiser
    consumes -- back into pinned host memory, all inside the timed region.
    Y and dX stay on the device, as they do in a model, where they feed the
    neighbouring layers.  The copies run on a second stream into double-buffered device
    slots, so step i+1's inputs arrive and step i-1's results leave while step
    i computes (the saved buffer is reused: each step's backward consumes it
    before the next forward writes it)."""
    import torch
    dev = t["X"].device
    hx = torch.empty_like(t["X"], device="cpu").pin_memory()
    hdy = torch.empty_like(t["dY"], device="cpu").pin_memory()
    hx.copy_(t["X"])
    hdy.copy_(t["dY"])
    keys = ("dWgu", "dWd")
    slots = []
    for i in range(2):
        si = {"X": t["X"] if i == 0 else torch.empty_like(t["X"]),
              "dY": t["dY"] if i == 0 else torch.empty_like(t["dY"]),
              "Wgu": t["Wgu"], "Wd": t["Wd"]}
        # own gradient buffers per slot (they are copied out while the next
        # step runs); Y, dX, saved and ws are shared: no step allocates
        oi = dict(o) if i == 0 else {**{k: torch.empty_like(o[k]) for k in keys},
                                     "Y": o["Y"], "dX": o["dX"], "saved": o["saved"],
                                     "ws": o["ws"]}
        host = {k: torch.empty_like(o[k], device="cpu").pin_memory() for k in keys}
        slots.append((si, oi, host))
    h2d = hx.numel() * hx.element_size() + hdy.numel() * hdy.element_size()
    d2h = sum(v.numel() * v.element_size() for v in slots[0][2].values())
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()

    def run(n):
        in_ready = [ev(), ev()]
        done = [None, None]   # compute of the slot's last step finished
        freed = [None, None]  # results of the slot's last step copied out
        with torch.cuda.stream(copy):
            t0 = slots[0][0]
            t0["X"].copy_(hx, non_blocking=True)
            t0["dY"].copy_(hdy, non_blocking=True)
            in_ready[0].record(copy)
        for i in range(n):
            si, oi, host = slots[i % 2]
            comp.wait_event(in_ready[i % 2])
            if freed[i % 2] is not None:
                comp.wait_event(freed[i % 2])  # its outputs were read out
            _step(api, si, oi)
            done[i % 2] = ev()
            done[i % 2].record(comp)
            with torch.cuda.stream(copy):
                if i + 1 < n:  # next step's inputs, into the other slot
                    sn = slots[(i + 1) % 2][0]
                    if done[(i + 1) % 2] is not None:
                        copy.wait_event(done[(i + 1) % 2])
                    sn["X"].copy_(hx, non_blocking=True)
                    sn["dY"].copy_(hdy, non_blocking=True)
                    in_ready[(i + 1) % 2] = ev()
                    in_ready[(i + 1) % 2].record(copy)
                copy.wait_event(done[i % 2])
                for k in keys:
                    host[k].copy_(oi[k], non_blocking=True)
                freed[i % 2] = ev()
                freed[i % 2].record(copy)
        comp.wait_stream(copy)

    def copy_gbps(dst, src):
        # one copy alone on the copy stream: this machine's host path, idle
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(copy)
        with torch.cuda.stream(copy):
            dst.copy_(src, non_blocking=True)
        c1.record(copy)
        c1.synchronize()
        return round(src.numel() * src.element_size() / (c0.elapsed_time(c1) / 1e3) / 1e9, 1)

    run(1)
    torch.cuda.synchronize()
    idle = {"h2d": copy_gbps(slots[1][0]["X"], hx),
            "d2h": copy_gbps(slots[1][2]["dWgu"], slots[1][1]["dWgu"])}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    run(steps)
    e1.record(comp)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / steps, h2d, d2h, idle


def _nograd_sweep(api, device, peaks, sizes=NOGRAD_S):
    import torch
    from backward_tcgen05_tma_gb300 import metrics, synthetic
    D, H = 4096, 11008
    # L2 flush by READING 512 MiB (> 129 MB L2): a write-based flush would leave
    # dirty lines whose write-back lands inside the timed call
    flush = torch.ones(128 * 2 ** 20, dtype=torch.float32, device=device)
    wts = synthetic.make_inputs(1, D, H, "bf16", seed=1, device=device, kind="device")
    res = []
    for S in sizes:
        X = synthetic.device_normal((S, D), 1.0, "bf16", 1, 0, device)
        Y = torch.empty(S, D, dtype=torch.bfloat16, device=device)
        A = torch.empty(S, H, dtype=torch.bfloat16, device=device)
        ws = api.workspace(S, D, H, torch.bfloat16, api.SWIGLU_OP_FWD_NOGRAD, device)
        o = {"Y": Y, "A": A}
        # warm-up long enough for the clocks to settle after the training runs
        for _ in range(30):
            flush.sum()
            api.swiglu_mlp_fwd_nograd(X, wts["Wgu"], wts["Wd"], out=o, ws=ws)
        times = []
        st = torch.cuda.current_stream()
        api.swiglu_mlp_profile_read()
        for it in range(40):
            flush.sum()
            if it == 20:  # second half: per-kernel events too
                api.swiglu_mlp_profile_enable(True)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            api.swiglu_mlp_fwd_nograd(X, wts["Wgu"], wts["Wd"], out=o, ws=ws)
            e1.record(st)
            e1.synchronize()
            if it < 20:
                times.append(e0.elapsed_time(e1) / 1e3)
        api.swiglu_mlp_profile_enable(False)
        kern = {k: round(v[1] / v[0] * 1e3, 2) for k, v in api.swiglu_mlp_profile_read().items()}
        tmed = statistics.median(times)
        byts = metrics.nograd_algorithmic_bytes(S, D, H)
        loop = _decode_loop(api, X, wts, o, ws)
        packed = {}
        if S <= NOGRAD_PACKED_MAX_S:
            # the same call on the packed weight copy (same bytes, contiguous blocks)
            pk = api.swiglu_mlp_pack_weights(wts["Wgu"], wts["Wd"])
            call = lambda: api.swiglu_mlp_fwd_nograd_packed(X, pk, H, out=o, ws=ws)
            for _ in range(10):
                flush.sum()
                call()
            tp = []
            for it in range(20):
                flush.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                call()
                e1.record(st)
                e1.synchronize()
                tp.append(e0.elapsed_time(e1) / 1e3)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(DECODE_REPS):
                call()
            torch.cuda.synchronize()
            lp = (time.perf_counter() - t0) / DECODE_REPS
            tpm = statistics.median(tp)
            packed = {"us_packed": round(tpm * 1e6, 2),
                      "hbm_frac_packed": round(byts / tpm / 1e9 / peaks["hbm_gbs"], 4),
                      "loop_us_packed": round(lp * 1e6, 2),
                      "loop_hbm_frac_packed": round(byts / lp / 1e9 / peaks["hbm_gbs"], 4)}
            del pk
        res.append({"S": S, "us": round(tmed * 1e6, 2), "GBps": round(byts / tmed / 1e9, 1),
                    "hbm_frac": round(byts / tmed / 1e9 / peaks["hbm_gbs"], 4),
                    "TFLOPS": round(metrics.fwd_flops(S, D, H) / tmed / 1e12, 2),
                    "kernel_us": kern, **loop,
                    # the same bytes per call in the back-to-back loop (host wall clock)
                    "loop_hbm_frac": round(byts / (loop["loop_us_direct"] * 1e-6) / 1e9
                                           / peaks["hbm_gbs"], 4), **packed})
    return {"workload": "B1_D4096_H11008_bf16_nograd", "l2": "flushed (512 MiB read) before "
            "each timed call", "median_of": 20,
            "decode_loop": "%d back-to-back calls, host wall clock per call (launch cost "
                           "included, no flush: the 270 MB of weights exceed L2): direct C-ABI "
                           "calls vs replays of the captured graph" % DECODE_REPS,
            "packed": "*_packed: the same call on the weight copy written by "
                      "swiglu_mlp_pack_weights (S <= %d)" % NOGRAD_PACKED_MAX_S,
            "sweep": res}


DECODE_REPS = 200
NOGRAD_PACKED_MAX_S = 64  # the packed-weights form serves the few-token path


def _decode_loop(api, X, wts, o, ws):
    """Per-call wall time of a decode loop: direct calls vs CUDA-graph replays."""
    import torch
    g = api.FwdNogradGraph(wts["Wgu"], wts["Wd"], X.shape[0], X=X, out=o, ws=ws)
    out = {}
    for name, call in (("direct", lambda: api.swiglu_mlp_fwd_nograd(X, wts["Wgu"], wts["Wd"],
                                                                     out=o, ws=ws)),
                       ("graph", g.launch)):
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(DECODE_REPS):
            call()
        torch.cuda.synchronize()
        out["loop_us_" + name] = round((time.perf_counter() - t0) / DECODE_REPS * 1e6, 2)
    g.close()
    return out


# The pages' training intermediate memory (MB as printed), fwd+bwd, bf16, B=8,
# D=4096, H=11008: fused implementation and Liger, by sequence length.
PAGES_TRAIN_MEMORY = {256: (178.0, 107.0), 8192: (5664.0, 6356.0)}


def _memory_report(api, w, device):
    """Training intermediates (the [G|U|A] buffer + workspace) at the pages'
    memory-table shapes, with the recommended and the minimal workspace, and
    the main workload's step time with the minimal workspace."""
    import torch
    L = api.lib()
    D, H = w["D"], w["H"]
    rows = {}
    for S, (flash, liger) in PAGES_TRAIN_MEMORY.items():
        M = 8 * S
        saved = L.swiglu_mlp_saved_bytes(M, H, 0)
        full = max(L.swiglu_mlp_workspace_bytes(M, D, H, 0, op) for op in (0, 2))
        least = max(L.swiglu_mlp_workspace_min_bytes(M, D, H, 0, op) for op in (0, 2))
        mib = 1.0 / 2 ** 20
        rows["B8_S%d_D%d_H%d" % (S, D, H)] = {
            "saved_MiB": round(saved * mib, 1), "ws_MiB": round(full * mib, 1),
            "ws_min_MiB": round(least * mib, 3), "total_MiB": round((saved + full) * mib, 1),
            "total_min_ws_MiB": round((saved + least) * mib, 1),
            "pages_MB": {"fused": flash, "liger": liger}}
    sec, _, _, keep, _ = _time_training(api, w, "bf16", 10, 3, 0, device, minimal_ws=True)
    del keep
    torch.cuda.empty_cache()
    return {"intermediates": rows, "unit_note": "MiB = 2^20 bytes; the pages print MB",
            "main_workload_min_ws_ms_per_step": round(sec * 1e3, 3)}


def _cpu_baseline(t_dev, w):
    """The oracle, as it stands, on a bounded sample: fwd+bwd of the first
    CPU_SAMPLE_TOKENS token rows of the workload with its full weights."""
    import oracle
    from backward_tcgen05_tma_gb300 import metrics
    m = CPU_SAMPLE_TOKENS
    D, H = w["D"], w["H"]
    c = {k: t_dev[k][:m].cpu() if k in ("X", "dY") else t_dev[k].cpu()
         for k in ("X", "dY", "Wg", "Wu", "Wd")}
    t0 = time.perf_counter()
    f = oracle.forward(c["X"], c["Wg"], c["Wu"], c["Wd"])
    b = oracle.backward(c["dY"], c["X"], c["Wg"], c["Wu"], c["Wd"], f)
    dt = time.perf_counter() - t0
    return {"value": metrics.fwd_bwd_flops(m, D, H) / dt / 1e12, "unit": "TFLOPS",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "fwd+bwd of %d token rows (full D=%d, H=%d weights) of the workload, "
                      "fp64 loops, %.1f s" % (m, D, H, dt),
            "parity": _sample_parity(t_dev, f, b)}


def _sample_parity(t_dev, f, b):
    """The same sample through the library (C ABI, the training kernels):
    relative Frobenius error of each output against the oracle's."""
    import numpy as np
    import oracle
    from backward_tcgen05_tma_gb300 import api
    Y, saved = api.swiglu_mlp_fwd(t_dev["X"], t_dev["Wgu"], t_dev["Wd"])
    dX, dWgu, dWd = api.swiglu_mlp_bwd(t_dev["dY"], t_dev["X"], t_dev["Wgu"], t_dev["Wd"], saved)
    H = t_dev["Wd"].shape[1]
    got = {"Y": Y, "dX": dX, "dWg": dWgu[:H], "dWu": dWgu[H:], "dWd": dWd}
    ref = {"Y": f["Y"], "dX": b["dX"], "dWg": b["dWg"], "dWu": b["dWu"], "dWd": b["dWd"]}
    out = {k: float("%.3e" % oracle.rel_frob(got[k].double().cpu().numpy(), np.asarray(ref[k])))
           for k in got}
    out["metric"] = "relative Frobenius error vs the oracle (tolerance 1e-2)"
    return out


def run_nograd_only(args):
    """Only the no-grad sweep at the listed sizes (one JSON line)."""
    import torch
    from backward_tcgen05_tma_gb300 import api, build
    torch.cuda.set_device(0)
    build.build()
    api.lib()
    sizes = [int(x) for x in args.nograd.split(",")]
    out = _nograd_sweep(api, "cuda:0", _peaks(), sizes)
    print(json.dumps({"metric": "SwiGLU MLP no-grad forward, HBM GB/s", "nograd": out}), flush=True)
    return 0


def run_ours(args):
    import torch
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    device = "cuda:%d" % local
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(device))
    from backward_tcgen05_tma_gb300 import api, build, metrics
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    api.lib()
    if args.cta_pairs is not None:
        api.swiglu_mlp_set_cta_pairs(args.cta_pairs)
    peaks = _peaks()
    w = WORKLOADS[args.workload]
    M, D, H = w["B"] * w["S"], w["D"], w["H"]

    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sec, launches, prof, (t, o), med = _time_training(api, w, "bf16", args.steps, args.warmup,
                                                 seed=rank, device=device, profile=True)
    clocks = sampler.stop()
    flops = metrics.fwd_bwd_flops(M, D, H)
    sec, value = aggregate_over_ranks(sec, flops, world, device)
    if world > 1:
        torch.distributed.barrier()

    # dominant kernel from live event timings of the timed region
    dom = max(prof.items(), key=lambda kv: kv[1][1])
    name, (n_l, ms) = dom
    per_launch_s = ms / 1e3 / n_l
    achieved = _kernel_flops(name, M, D, H) / per_launch_s / 1e12
    traffic = _traffic(name, args.workload)
    kernels = {k: {"launches": v[0], "ms_per_launch": round(v[1] / v[0], 4),
                   "share": round(v[1] / sum(x[1] for x in prof.values()), 4),
                   "TFLOPS": round(_kernel_flops(k, M, D, H) / (v[1] / 1e3 / v[0]) / 1e12, 1)}
               for k, v in prof.items()}

    e2e_sec, h2d, d2h, idle_copy = _e2e(api, t, o, max(2, args.steps // 2))
    del t, o
    torch.cuda.empty_cache()

    line = {"metric": "SwiGLU MLP fwd+bwd TFLOPS (18*M*D*H)", "value": value, "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "ms_per_step_median": med * 1e3,
            "vs_baseline": value / world / PAGES_TFLOPS[args.workload]
            if args.workload in PAGES_TFLOPS else None,
            "dtype": "bf16", "data": "synthetic (seeded, device generator)",
            "config": _config(args.workload, w, "bf16", world),
            "pct_of_bf16_peak": {"burst": value / world / peaks["bf16_tflops"],
                                 "sustained": value / world / peaks["bf16_tflops_sustained"],
                                 "source": peaks["source"]},
            "roofline": {"bound": "tensor", "kernel": name, "achieved": achieved,
                         "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops_sustained"],
                         "peak_kind": "bf16 sustained (%s)" % peaks["source"],
                         "traffic": traffic,
                         "timing": "CUDA events around each launch on its stream, over a "
                                   "second pass of the same steps (events serialise the "
                                   "kernels; value comes from the unprofiled pass)"},
            "kernels": kernels,
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": {"value": flops / e2e_sec / 1e12, "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_sec * 1e3,
                    "copies": "X, dY in and the parameter gradients dWgu, dWd out (Y, dX stay "
                              "on the device), pinned host <-> device on a second stream, "
                              "double-buffered device slots, overlapping the neighbouring "
                              "steps' compute",
                    # one copy each way (X in, dWgu out), alone, just before the loop
                    "host_copy_GBps_idle": idle_copy}}

    if world == 1 and not args.quick:
        extra = {}
        # each timed over about 100 ms after a pause and a warm-up, so that the
        # short steps are not measured while the clocks recover from the
        # power-capped main workload
        # each timed over about 1 s after a pause and a warm-up, so that the
        # short steps are not measured while the clocks recover from the
        # power-capped main workload, with the SM clock sampled meanwhile
        # (TFLOPS per GHz compares dtypes whose clocks differ under the cap)
        for wl, dts, n in (("B8_S2048_D1024_H2816", ["bf16"], 1500),
                           ("B8_S4096_D2048_H5632", ["bf16", "f16"], 220)):
            for dn in dts:
                time.sleep(1.0)
                cs = ClockSampler(local)
                cs.start()
                s2, _, prof2, keep, med2 = _time_training(api, WORKLOADS[wl], dn, n, 10, 0, device,
                                                    profile=True)
                ck = cs.stop()
                del keep
                w2 = WORKLOADS[wl]
                M2, D2, H2 = w2["B"] * w2["S"], w2["D"], w2["H"]
                f2 = metrics.fwd_bwd_flops(M2, D2, H2)
                tf = f2 / s2 / 1e12
                extra["%s_%s" % (wl, dn)] = {
                    "ms_per_step": round(s2 * 1e3, 3), "ms_per_step_median": round(med2 * 1e3, 3),
                    "TFLOPS": round(tf, 1),
                    "kernel_ms": {k: round(v[1] / v[0], 4) for k, v in prof2.items()},
                    "clocks": ck,
                    "TFLOPS_per_GHz": round(tf / (ck["sm_mhz"] / 1e3), 1)
                    if ck.get("sm_mhz") else None}
                torch.cuda.empty_cache()
        line["other_workloads"] = extra
        line["memory"] = _memory_report(api, w, device)
        time.sleep(1.0)
        line["nograd"] = _nograd_sweep(api, device, peaks)
    if world == 1 or rank == 0:
        if world == 1 and not args.no_cpu:
            from backward_tcgen05_tma_gb300 import synthetic
            tc = synthetic.make_inputs(CPU_SAMPLE_TOKENS, D, H, "bf16", seed=0, device=device,
                                       kind="device")
            line["cpu_baseline"] = _cpu_baseline(tc, w)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=MAIN)
    ap.add_argument("--quick", action="store_true", help="main workload only")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cta-pairs", type=int, choices=[0, 1, 2], default=None,
                    help="tensor-core GEMMs on SM pairs: 1 by size (library default), 2 always, 0 never")
    ap.add_argument("--nograd", default=None,
                    help="comma-separated S values: run only the no-grad sweep (B=1, D=4096, H=11008)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.nograd:
        return run_nograd_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
