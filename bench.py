#!/usr/bin/env python
"""Packed variable-length context-parallel attention forward: throughput on GB300.

Metric: packed varlen attention fwd TFLOP/s over valid tokens (THD-aware FLOPs
4*D*H*sum pairs(L), counted from real sequence lengths) and the fraction of
the measured dense BF16 tensor peak.

A step is one pass of the hot path over one synthetic micro-batch already
resident in HBM: the whole packed forward (every virtual rank's ring steps
with the exact LSE merge fused in, one launch) plus the per-token loss
normalisation, which does not depend on the attention and runs beside it on
a second stream.  The context-parallel plan is built once per micro-batch
layout on the host, outside the timed region, as the pages' Dynamic-CP
scheduler also plans asynchronously off the critical path; its host time is
reported as plan_ms.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 oracle on host cores

Under torchrun (N>1) every rank runs an independent replica of the workload
on its own GPU (no data-path collective); a barrier and a max over ranks
bracket the timed region.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Host-only legs pin BLAS to one thread per worker before numpy loads.
if "--cpu-baseline-child" in sys.argv or ("--impl" in sys.argv and "reference" in sys.argv):
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np  # noqa: E402

METRIC = "packed varlen attention fwd TFLOP/s (valid tokens) and % of GB300 BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "dynamic_cp_microbatch"
FALLBACK_BF16_TFLOPS = 1900.0
# a kernel's DRAM traffic depends on its source and on the work list the planner hands it
TC_SOURCES = ("context_attention_cpattn_gb300/csrc/attn_tc.cu", "context_attention_cpattn_gb300/csrc/common.cuh",
              "context_attention_cpattn_gb300/csrc/plan.cpp")
TRAFFIC_FILE = "profiles/traffic.json"
BWD_SOURCES = ("context_attention_cpattn_gb300/csrc/attn_bwd_tc.cu", "context_attention_cpattn_gb300/csrc/common.cuh",
               "context_attention_cpattn_gb300/csrc/plan.cpp")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the CPU oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the long-sequence workloads after the headline one")
    ap.add_argument("--aux", action="store_true",
                    help="time the HBM-bound kernels (merge, shard gather, loss norm) instead of the forward")
    ap.add_argument("--mesh", default="",
                    help="UxR: run the workload on the 2D-Attention mesh of U Ulysses x R ring virtual ranks")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward (cpattn_bwd) on the workload instead of the forward")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--rows", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ------------------------------------------------------------------ replicas

class Replicas:
    """Rank bookkeeping for N independent replicas: a barrier and a max over
    ranks around the timed region, nothing in the data path."""

    def __init__(self, backend: str | None = None):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local = int(os.environ.get("LOCAL_RANK", str(self.rank)))
        self.backend = backend
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend or "nccl")
            self.dist = dist

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        dev = f"cuda:{self.local}" if self.backend in (None, "nccl") else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


# ------------------------------------------------------------------ clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

# NVML clock-event reason bits (read-only queries; nothing is ever set)
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}


def clock_csv_path(tag: str) -> str:
    """Where the raw clock samples go: the directory in CPATTN_CLOCKS_DIR, else /tmp."""
    return os.path.join(os.environ.get("CPATTN_CLOCKS_DIR", "/tmp"), f"cpattn_clocks_{tag}.csv")


def nvml_index(local_rank: int) -> int:
    """NVML index of the GPU this process uses: CUDA_VISIBLE_DEVICES maps the
    CUDA ordinal to the physical one when it lists plain indices."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    if ids and all(x.isdigit() for x in ids) and local_rank < len(ids):
        return int(ids[local_rank])
    return local_rank


class _Nvml:
    """The few read-only NVML queries the sampler needs, through ctypes."""

    def __init__(self, index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)

    def sample(self):
        c = self.c
        mhz, mw, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz))          # NVML_CLOCK_SM
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw))
        self.reasons_fn(self.h, c.byref(rs))
        return float(mhz.value), mw.value / 1e3, int(rs.value)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock, power and throttle reasons sampled every 2 ms from a host
    thread (NVML, read-only), or by nvidia-smi every 200 ms where NVML cannot
    be loaded.  ``mark()`` brackets a region; ``summary(region)`` gives the
    median SM clock under load and the reasons seen in it."""

    def __init__(self, local_rank: int, path: str, period_s: float = 0.002):
        import threading
        self.samples = []   # (host time, sm MHz, max MHz, power W, reasons set)
        self.marks = {}
        self.proc = None
        self.nvml = None
        self.path = path
        try:
            self.nvml = _Nvml(nvml_index(local_rank))
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.stop_ev = threading.Event()

            def loop():
                while not self.stop_ev.is_set():
                    mhz, w, rs = self.nvml.sample()
                    self.samples.append((time.perf_counter(), mhz, self.nvml.max_mhz, w,
                                         {n for bit, n in _NVML_REASONS.items() if rs & bit}))
                    self.stop_ev.wait(period_s)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
        else:
            try:
                self.f = open(path, "w")
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                     "-i", str(nvml_index(local_rank))], stdout=self.f, stderr=subprocess.DEVNULL)
            except (OSError, FileNotFoundError):
                self.proc = None

    def mark(self, name: str):
        self.marks[name] = time.perf_counter()

    def stop(self):
        if self.nvml is not None:
            time.sleep(0.02)
            self.stop_ev.set()
            self.thread.join(timeout=2)
            self.nvml.close()
        elif self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, start: str | None = None, end: str | None = None) -> dict | None:
        if self.nvml is None:
            if self.proc is None:
                return None
            return summarise_clocks(open(self.path).read())
        t0 = self.marks.get(start, -1e30) if start else -1e30
        t1 = self.marks.get(end, 1e30) if end else 1e30
        sel = [x for x in self.samples if t0 <= x[0] <= t1]
        if not sel:
            return None
        sm = [x[1] for x in sel]
        top = max(sm)
        loaded = [v for v in sm if v >= 0.5 * top] or sm
        reasons = sorted(set().union(*(x[4] for x in sel)))
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(x[2] for x in sel), "samples": len(sel),
                "power_w_max": max(x[3] for x in sel), "reasons": reasons, "source": "nvml, 2 ms period"}


def summarise_clocks(text: str) -> dict | None:
    sm, mx, reasons = [], [], set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for line in text.strip().splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    top = max(sm)
    loaded = [s for s in sm if s >= 0.5 * top] or sm
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "samples": len(sm),
            "reasons": sorted(reasons), "source": "nvidia-smi 200 ms"}


# ------------------------------------------------------------------ peaks, traffic

def measured_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "of measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "of fallback"


def tc_source_hash(sources=TC_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str = "attn_fwd_tc_kernel", sources=TC_SOURCES):
    """DRAM bytes per launch of a kernel from profiles/traffic.json, if they
    were taken on the current kernel source and this workload."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_FILE)) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("workload") != workload or rec.get("source_sha256") != tc_source_hash(sources):
        return None
    return float(rec["dram_bytes_per_launch"])


# ------------------------------------------------------------------ CPU oracle legs

def row_flops(cu, rows, H, D, causal) -> int:
    cu = np.asarray(cu, dtype=np.int64)
    seq = np.searchsorted(cu, rows, side="right") - 1
    vis = (rows - cu[seq] + 1) if causal else (cu[seq + 1] - cu[seq])
    return int(4 * D * H * int(vis.sum()))


def oracle_rows(w, rows, q, k, v, threads):
    from oracle import attention as A
    t0 = time.perf_counter()
    A.attention_at_rows(q, k, v, w.cu_seqlens, rows, w.causal, w.scale, threads=threads)
    return time.perf_counter() - t0


def cpu_baseline_child(args):
    """Runs in a subprocess with single-threaded BLAS: the oracle on sampled
    query rows (all heads) of the workload, on every host core."""
    import inputs
    w = inputs.workload(args.workload)
    q, k, v = inputs.make_qkv(w)
    cores = host_cores()
    n = max(8, args.rows or 64)
    rows = inputs.sample_rows(w.T, n, seed=w.seed + 1)
    dt = oracle_rows(w, rows, q, k, v, cores)
    # grow the sample (at least doubling) until it takes about the target time
    attempt = 0
    while not args.rows and dt < 0.5 * args.cpu_seconds and n < w.T and attempt < 8:
        n = int(min(w.T, n * max(2.0, args.cpu_seconds / max(dt, 1e-3))))
        rows = inputs.sample_rows(w.T, n, seed=w.seed + 2 + attempt)
        dt = oracle_rows(w, rows, q, k, v, cores)
        attempt += 1
    fl = row_flops(w.cu_seqlens, rows, w.H, w.D, w.causal)
    print(json.dumps({"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                      "sample": f"{len(rows)} seeded query rows x {w.H} heads of {w.name} "
                                f"({fl:.3e} FLOPs, {dt:.2f} s, fp64 numpy, {cores} threads)"}))


def run_cpu_baseline(args) -> dict | None:
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", "--workload", args.workload,
           "--cpu-seconds", str(args.cpu_seconds)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as ex:  # noqa: BLE001
        return {"value": None, "unit": UNIT, "cores": host_cores(), "kind": "oracle", "sample": f"failed: {ex}"}


def config_of(w, flops):
    cfg = {"workload": w.name, "T": w.T, "n_seqs": w.n_seqs, "H": w.H, "Hkv": w.Hkv, "D": w.D, "causal": w.causal,
           "mode": w.mode, "cp": w.cp, "flops_per_step": flops, "seed": w.seed}
    if w.grid:
        cfg["grid"] = list(w.grid)
    in_bytes = w.T * (w.H + 2 * w.Hkv) * w.D * (2 if w.dtype == "bf16" else 4)
    cfg["l2"] = f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB read per step)"
    return cfg


def run_reference(args):
    """The oracle as it stands, on the host cores, as the reference arm."""
    import inputs
    from oracle import flops as OF
    w = inputs.workload(args.workload)
    q, k, v = inputs.make_qkv(w)
    cores = host_cores()
    rows_per_step = args.rows or w.T  # every row: K and V are converted to fp64 once per step either way
    times, fl_total = [], 0
    for i in range(args.warmup + args.steps):
        rows = inputs.sample_rows(w.T, rows_per_step, seed=w.seed + 100 + i)
        dt = oracle_rows(w, rows, q, k, v, cores)
        if i >= args.warmup:
            times.append(dt)
            fl_total += row_flops(w.cu_seqlens, rows, w.H, w.D, w.causal)
    total = sum(times)
    value = fl_total / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, OF.fwd_flops(w.cu_seqlens, w.H, w.D, w.causal)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step {rows_per_step} seeded query rows x {w.H} heads of {w.name}, "
                                       f"fp64 numpy on {cores} threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def run_ours(args, rep: Replicas):
    import torch

    import context_attention_cpattn_gb300 as cp
    import inputs

    torch.cuda.set_device(rep.local)
    dev = torch.device("cuda", rep.local)
    w = inputs.workload(args.workload)
    q_h, k_h, v_h = inputs.make_qkv(w, pin=True)
    loss_h, valid_h = inputs.make_loss_inputs(w)
    loss_h, valid_h = loss_h.pin_memory(), valid_h.pin_memory()
    qd, kd, vd = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    loss_d, valid_d = loss_h.to(dev), valid_h.to(dev)

    t0 = time.perf_counter()
    if args.mesh:
        u, r = (int(x) for x in args.mesh.lower().split("x"))
        plan = cp.cpattn_plan_2d(w.cu_seqlens, u, r)
    elif w.mode == "paired":
        plan = cp.cpattn_plan_paired(w.cu_seqlens, w.cp, w.grid[0])
    else:
        plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    ws_bytes = cp.cpattn_workspace_size(plan, w.H, w.Hkv, w.D, qd.dtype, w.causal)
    plan_ms = 1e3 * (time.perf_counter() - t0)
    # FLOPs over the pairs the mask allows (teacher forcing for paired plans)
    flops = (4 * w.D * w.H * plan.allowed_pairs(True) if w.mode == "paired"
             else cp.cpattn_fwd_flops(w.cu_seqlens, w.H, w.D, w.causal))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.H, w.T), dtype=torch.float32, device=dev)
    out_loss = torch.empty(1, dtype=torch.float64, device=dev)
    out_cnt = torch.empty(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    # attention + loss; grid2d adds 3 shard gathers; the mesh adds 3 all-to-all gathers,
    # the reverse all-to-all of O and the LSE regroup
    launches_per_step = 2 + (5 if args.mesh or w.mode == "paired" else 3 if w.mode == "grid2d" else 0)

    # The loss normalisation does not depend on the attention, so it runs on a
    # second stream beside it: forked from the step's start and joined before
    # the step ends, both inside the timed region.
    side = torch.cuda.Stream(dev)
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    def step(ev0=None, ev1=None):
        if ev0 is not None:
            ev0.record(stream)
        fork.record(stream)
        side.wait_event(fork)
        cp.cpattn_token_loss_norm(loss_d, valid_d, out_loss, out_cnt, stream=side)
        cp.cpattn_fwd(plan, qd, kd, vd, o, lse, ws, scale=w.scale, causal=w.causal, stream=stream)
        if ev1 is not None:
            ev1.record(stream)
        join.record(side)
        stream.wait_event(join)

    sampler = ClockSampler(rep.local, clock_csv_path(f"rank{rep.rank}"))
    sampler.mark("warmup")
    for _ in range(args.warmup):
        step()
    cp.cpattn_sync_status(ws, stream)

    fwd_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rep.barrier()
    torch.cuda.synchronize(dev)
    sampler.mark("timed")
    start.record(stream)
    for i in range(args.steps):
        step(*fwd_ev[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark("timed_end")
    rep.barrier()
    clocks = sampler.summary("timed", "timed_end")
    clocks_run = sampler.summary("warmup", "timed_end")
    cp.cpattn_sync_status(ws, stream)
    elapsed = start.elapsed_time(end) / 1e3
    fwd_ms = [a.elapsed_time(b) for a, b in fwd_ev]
    elapsed_max = rep.max(elapsed)
    value = rep.world * args.steps * flops / elapsed_max / 1e12

    # end to end through the public API: every step copies its inputs from pinned host memory
    # and reads its outputs back inside the timed region, pipelined as a training input
    # pipeline would be: step i's upload (copy stream) overlaps step i-1's compute, whose
    # read-back (a third stream) overlaps step i's; two buffer sets alternate.
    e2e = None
    if not args.no_e2e:
        # uploads on three copy streams (Q; K; V and the loss inputs) so that several copy engines work
        s_ins = [torch.cuda.Stream(dev) for _ in range(3)]
        s_out = torch.cuda.Stream(dev)
        sets = []
        for _ in range(2):
            sets.append({
                "q": torch.empty_like(qd), "k": torch.empty_like(kd), "v": torch.empty_like(vd),
                "loss": torch.empty_like(loss_d), "valid": torch.empty_like(valid_d),
                "o": torch.empty_like(o), "lse": torch.empty_like(lse),
                "l": torch.empty(1, dtype=torch.float64, device=dev), "c": torch.empty(1, dtype=torch.int64, device=dev),
                "res": torch.empty(2, dtype=torch.float64, device=dev),
                "o_h": torch.empty(o.shape, dtype=o.dtype, pin_memory=True),
                "lse_h": torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True),
                "res_h": torch.empty(2, dtype=torch.float64, pin_memory=True)})
        h2d_done = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        d2h_done = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            b = i % 2
            B = sets[b]
            groups = ((("q", q_h),), (("k", k_h),), (("v", v_h), ("loss", loss_h), ("valid", valid_h)))
            for si, group in enumerate(groups):
                with torch.cuda.stream(s_ins[si]):
                    if i >= 2:
                        s_ins[si].wait_event(comp_done[b])  # step i-2's compute has read this set's inputs
                    for name, src in group:
                        B[name].copy_(src, non_blocking=True)
                    h2d_done[b][si].record(s_ins[si])
            for ev in h2d_done[b]:
                stream.wait_event(ev)
            if i >= 2:
                stream.wait_event(d2h_done[b])  # step i-2's read-back has left this set's outputs
            cp.cpattn_fwd(plan, B["q"], B["k"], B["v"], B["o"], B["lse"], ws, scale=w.scale, causal=w.causal,
                          stream=stream)
            cp.cpattn_token_loss_norm(B["loss"], B["valid"], B["l"], B["c"], stream=stream)
            B["res"][0:1].copy_(B["l"])
            B["res"][1:2].copy_(B["c"].to(torch.float64))
            comp_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                B["o_h"].copy_(B["o"], non_blocking=True)
                B["lse_h"].copy_(B["lse"], non_blocking=True)
                B["res_h"].copy_(B["res"], non_blocking=True)
                d2h_done[b].record(s_out)

        for i in range(args.warmup):
            e2e_step(i)
        rep.barrier()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for si in s_ins:
            si.wait_event(e0)
        for i in range(args.warmup, args.warmup + args.steps):
            e2e_step(i)
        e1.record(s_out)  # after the last read-back, which follows the last compute
        torch.cuda.synchronize(dev)
        rep.barrier()
        e2e_s = rep.max(e0.elapsed_time(e1) / 1e3)
        B = sets[0]
        h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h, loss_h, valid_h))
        d2h = (B["o_h"].numel() * B["o_h"].element_size() + B["lse_h"].numel() * B["lse_h"].element_size() +
               B["res_h"].numel() * 8)
        e2e = {"value": rep.world * args.steps * flops / e2e_s / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "pipelined": True,
               "ms_per_step": 1e3 * e2e_s / args.steps,
               "host_link_GB_s": (h2d + d2h) * args.steps / e2e_s / 1e9}
        cp.cpattn_sync_status(ws, stream)
        # the read-back of the last step holds the same result as the device-timed steps
        if not torch.equal(sets[(args.warmup + args.steps - 1) % 2]["o_h"].to(dev), o):
            raise RuntimeError("end-to-end output differs from the device-resident run")

    per_config = backward = None
    if rep.world == 1 and not args.no_per_config and not args.mesh and args.workload == DEFAULT_WORKLOAD:
        backward = time_backward(cp, w, qd, kd, vd, dev, stream, sampler, max(args.steps, 3), max(args.warmup, 3),
                                 tag="bwd_" + w.name)
        del qd, kd, vd, o, lse, ws
        if e2e is not None:
            del sets
        torch.cuda.empty_cache()
        per_config = {name: time_config(cp, name, n, dev, stream, sampler) for name, n in PER_CONFIG}
    sampler.stop()

    if rep.rank != 0:
        return
    peak, peak_src = measured_peak()
    fwd_mean_s = statistics.fmean(fwd_ms) / 1e3
    achieved = flops / fwd_mean_s / 1e12
    traffic = recorded_traffic(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": rep.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * elapsed_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_of(w, flops), **({"mode": "ulysses2d", "mesh": args.mesh + " (ulysses x ring)",
                                                 "cp": plan.cp} if args.mesh else {})),
        "pct_of_bf16_peak": 100.0 * value / (peak * rep.world),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                     "peak_source": peak_src, "traffic": traffic,
                     "kernel": "attn_fwd_tc_kernel (cpattn_fwd, CUDA events per call)"},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "clocks_warmup_and_timed": clocks_run,
        "plan_ms": plan_ms,
        "fwd_ms_mean": 1e3 * fwd_mean_s,
        "fwd_ms_min": min(fwd_ms),
        "tc_source_sha256": tc_source_hash(),
        "mma_area_useful": useful_mma_fraction(plan, w.causal, w.dtype),
    }
    add_sustained(line["roofline"], achieved, clocks)
    if per_config is not None:
        line["per_config"] = per_config
    if backward is not None:
        line["backward"] = backward
    if not args.no_cpu_baseline and rep.world == 1 and w.mode != "paired":
        # (the CPU legs evaluate the causal / bidirectional oracle; paired plans use another mask)
        line["cpu_baseline"] = run_cpu_baseline(args)
    print(json.dumps(line), flush=True)


# The other full-size workloads, timed in the same process after the headline
# one: (name, timed steps).  Three warm-up calls each; inputs larger than L2.
PER_CONFIG = (("long_video_200k_gqa", 5), ("video_latent_grid2d", 20), ("single_seq_1m_gqa", 2))


def measured_sustained() -> float | None:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        return None


def add_sustained(roofline: dict, achieved: float, clocks) -> None:
    """When the power cap held the clocks down during the timed region, the
    fraction of the measured sustained bf16 peak (a long loop under the same
    cap) goes beside the fraction of the burst peak."""
    sustained = measured_sustained()
    if sustained and clocks and "sw_power_cap" in clocks.get("reasons", []):
        roofline["frac_of_sustained"] = achieved / sustained
        roofline["peak_sustained"] = sustained


def time_config(cp, name, steps, dev, stream, sampler, warmup=3):
    """cpattn_fwd on one workload: TFLOP/s of valid-token FLOPs over `steps`
    calls timed by CUDA events on the launching stream."""
    import torch

    import inputs
    w = inputs.workload(name)
    q_h, k_h, v_h = inputs.make_qkv(w)
    qd, kd, vd = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    del q_h, k_h, v_h
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    flops = cp.cpattn_fwd_flops(w.cu_seqlens, w.H, w.D, w.causal)
    ws = torch.empty(cp.cpattn_workspace_size(plan, w.H, w.Hkv, w.D, qd.dtype, w.causal), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.H, w.T), dtype=torch.float32, device=dev)

    def call():
        cp.cpattn_fwd(plan, qd, kd, vd, o, lse, ws, scale=w.scale, causal=w.causal, stream=stream)

    for _ in range(warmup):
        call()
    cp.cpattn_sync_status(ws, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    sampler.mark(name)
    for a, b in ev:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark(name + "_end")
    cp.cpattn_sync_status(ws, stream)
    ms = [a.elapsed_time(b) for a, b in ev]
    mean_s = statistics.fmean(ms) / 1e3
    value = flops / mean_s / 1e12
    peak, src = measured_peak()
    out = {"value": value, "unit": UNIT, "frac": value / peak, "peak": peak, "peak_source": src,
           "ms_per_step": 1e3 * mean_s, "ms_min": min(ms), "steps": steps, "warmup": warmup,
           "flops_per_step": flops, "T": w.T, "H": w.H, "Hkv": w.Hkv, "mode": w.mode, "cp": w.cp,
           "causal": w.causal, "clocks": sampler.summary(name, name + "_end"),
           "mma_area_useful": useful_mma_fraction(plan, w.causal, w.dtype),
           "l2": "inputs larger than L2"}
    sustained = measured_sustained()
    if sustained and mean_s > 1.0:
        out["frac_of_sustained"] = value / sustained
        out["peak_sustained"] = sustained
    del qd, kd, vd, o, lse, ws
    torch.cuda.empty_cache()
    return out


# Kernel tile shapes (rows per tile, keys or queries per kernel tile) of the
# bf16 and fp32 forward and backward kernels.
TILE_SHAPES = {(False, "bf16"): (128, 64), (False, "fp32"): (64, 32),
               (True, "bf16"): (128, 64), (True, "fp32"): (32, 64)}


def useful_mma_fraction(plan, causal: bool, dtype: str = "bf16", backward: bool = False):
    """Share of a kernel's executed tile area (per query head) that falls on
    pairs the mask allows: allowed pairs over the tile area summed over the
    work list the call uploads (one head group's copy for head-sharded plans).
    The rest is the padding of partial tiles and pieces and the masked-out
    triangles of diagonal tiles."""
    tiles, _ = plan.worklist(backward, dtype, causal)
    tm, tn = TILE_SHAPES[(backward, dtype)]
    executed = int(tiles[:, 6].astype(np.int64).sum()) * tm * tn
    groups = plan.info()["split_h"] if plan.mode in (3, 4) else 1   # ulysses2d, paired
    return groups * plan.allowed_pairs(causal) / executed if executed else None


def time_backward(cp, w, qd, kd, vd, dev, stream, sampler, steps, warmup, tag="bwd"):
    """cpattn_bwd (delta/LSE prep, the tensor-core kernel, dQ conversion) on
    one workload, timed per call with CUDA events on its stream.  FLOPs = 2.5 x
    the forward's (five products of the forward's shape where the forward has
    two), over valid (causal) pairs only.  Returns the result as a dict."""
    import torch

    import inputs
    dod = inputs.make_dout(w).to(dev)
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    fwd_flops = cp.cpattn_fwd_flops(w.cu_seqlens, w.H, w.D, w.causal)
    flops = fwd_flops * 5 // 2
    ws = torch.empty(max(cp.cpattn_workspace_size(plan, w.H, w.Hkv, w.D, qd.dtype, w.causal),
                         cp.cpattn_bwd_workspace_size(plan, w.H, w.Hkv, w.D, qd.dtype, w.causal)),
                     dtype=torch.uint8, device=dev)
    o = torch.empty_like(qd)
    lse = torch.empty((w.H, w.T), dtype=torch.float32, device=dev)
    cp.cpattn_fwd(plan, qd, kd, vd, o, lse, ws, scale=w.scale, causal=w.causal, stream=stream)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)

    def step():
        cp.cpattn_bwd(plan, qd, kd, vd, o, lse, dod, dq, dk, dv, ws, scale=w.scale, causal=w.causal, stream=stream)

    for _ in range(warmup):
        step()
    cp.cpattn_sync_status(ws, stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    sampler.mark(tag)
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark(tag + "_end")
    cp.cpattn_sync_status(ws, stream)
    ms = [a.elapsed_time(b) for a, b in ev]
    mean_s = statistics.fmean(ms) / 1e3
    peak, peak_src = measured_peak()
    achieved = flops / mean_s / 1e12
    launches = 3 + (4 if w.mode == "grid2d" else 0)
    clocks = sampler.summary(tag, tag + "_end")
    out = {
        "metric": "packed varlen attention bwd TFLOP/s (valid tokens, 2.5x forward FLOPs)", "value": achieved,
        "unit": UNIT, "steps": steps, "warmup": warmup, "ms_per_step": 1e3 * mean_s,
        "ms_min": min(ms), "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(w, flops),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                     "peak_source": peak_src,
                     "traffic": recorded_traffic(w.name, "attn_bwd_tc_kernel", BWD_SOURCES),
                     "kernel": "cpattn_bwd call (pre + attn_bwd_tc_kernel + post), CUDA events per call"},
        "gpu_launches": launches * steps, "clocks": clocks,
        "mma_area_useful": useful_mma_fraction(plan, w.causal, w.dtype, backward=True)}
    add_sustained(out["roofline"], achieved, clocks)
    return out


def run_bwd(args):
    """Backward on the workload (see time_backward), printed as one JSON line."""
    import torch

    import context_attention_cpattn_gb300 as cp
    import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = inputs.workload(args.workload)
    q_h, k_h, v_h = inputs.make_qkv(w)
    qd, kd, vd = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    sampler = ClockSampler(0, clock_csv_path("bwd"))
    line = time_backward(cp, w, qd, kd, vd, dev, torch.cuda.current_stream(dev), sampler, args.steps, args.warmup)
    sampler.stop()
    print(json.dumps(line), flush=True)


def measured_hbm() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "of fallback"


def run_aux(args):
    """GB/s of the HBM-bound kernels on shapes of the workloads: the exact LSE
    merge of cp=4 partials over the 32K micro-batch, the grid2d shard gather of
    the 16x45x80 latent's Q, and the loss normalisation (micro-batch size and
    a 64M-token vector).  Algorithmic bytes: everything read once + written once.
    Also: the host link, the ring written out as block steps and merges (the
    micro-batch and the 200K-token sequence) against the fused forward, and
    the Dynamic-CP solver's host time."""
    import torch

    import context_attention_cpattn_gb300 as cp
    import inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, src = measured_hbm()
    out = []

    def timeit(fn, reps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps / 1e3

    def record(kernel, what, nbytes, sec):
        gbs = nbytes / sec / 1e9
        out.append({"kernel": kernel, "shape": what, "bytes": nbytes, "us": sec * 1e6, "GB_s": gbs,
                    "frac": gbs / peak})

    # merge: 4 partials x [32768, 32, 128] fp32 -> bf16 O and fp32 LSE
    T, H, D, n = 32768, 32, 128, 4
    g = torch.Generator(device=dev).manual_seed(1)
    o_parts = [torch.randn(T, H, D, device=dev, generator=g) for _ in range(n)]
    l_parts = [torch.randn(H, T, device=dev, generator=g) for _ in range(n)]
    o = torch.empty(T, H, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(H, T, device=dev)
    sec = timeit(lambda: cp.cpattn_merge(o_parts, l_parts, o, lse))
    record("merge_kernel", "4 x [32768,32,128] fp32 -> bf16", n * (T * H * D * 4 + H * T * 4) + T * H * D * 2 + H * T * 4, sec)
    del o_parts, l_parts, o, lse
    # shard gather of the latent's Q rows (split_cp_2d)
    w = inputs.workload("video_latent_grid2d")
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    idx = torch.from_numpy(plan.index_map()).to(dev)
    x = torch.randn(w.T, w.H, w.D, device=dev, generator=g).to(torch.bfloat16)
    y = torch.empty_like(x)
    sec = timeit(lambda: cp.cpattn_gather_rows(x, y, idx))
    record("permute_rows_kernel (gather)", "[57600,24,128] bf16", 2 * x.numel() * 2 + idx.numel() * 8, sec)
    sec = timeit(lambda: cp.cpattn_scatter_rows(y, x, idx))
    record("permute_rows_kernel (scatter)", "[57600,24,128] bf16", 2 * x.numel() * 2 + idx.numel() * 8, sec)
    del x, y
    # loss normalisation
    res = torch.empty(1, dtype=torch.float64, device=dev)
    cnt = torch.empty(1, dtype=torch.int64, device=dev)
    for Tl in (32768, 1 << 26):
        loss = torch.rand(Tl, device=dev, generator=g)
        valid = (torch.rand(Tl, device=dev, generator=g) > 0.1).to(torch.uint8)
        sec = timeit(lambda: cp.cpattn_token_loss_norm(loss, valid, res, cnt))
        record("loss_norm_kernel", f"T={Tl}", Tl * 5, sec)
    # host link: pinned host memory to and from HBM, 805 MB (the micro-batch's Q, K and V),
    # by copy engines (cudaMemcpyAsync on 1 or 3 streams) and by the copy kernel reading or
    # writing host memory directly
    nb = 805306368
    hbuf = torch.empty(nb, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(nb, dtype=torch.uint8, device=dev)
    link = []

    def rec(what, sec):
        link.append({"what": what, "bytes": nb, "ms": sec * 1e3, "GB_s": nb / sec / 1e9})

    rec("H2D cudaMemcpyAsync, 1 stream", timeit(lambda: dbuf.copy_(hbuf, non_blocking=True), reps=5))
    streams = [torch.cuda.Stream(dev) for _ in range(3)]
    thirds = [(i * nb // 3) // 16 * 16 for i in range(4)]

    def three(h2d):
        cur = torch.cuda.current_stream(dev)
        evs = []
        for si, st in enumerate(streams):
            st.wait_stream(cur)
            with torch.cuda.stream(st):
                a, b = thirds[si], thirds[si + 1]
                if h2d:
                    dbuf[a:b].copy_(hbuf[a:b], non_blocking=True)
                else:
                    hbuf[a:b].copy_(dbuf[a:b], non_blocking=True)
            evs.append(st)
        for st in evs:
            cur.wait_stream(st)

    rec("H2D cudaMemcpyAsync, 3 streams", timeit(lambda: three(True), reps=5))
    rec("D2H cudaMemcpyAsync, 1 stream", timeit(lambda: hbuf.copy_(dbuf, non_blocking=True), reps=5))
    rec("D2H cudaMemcpyAsync, 3 streams", timeit(lambda: three(False), reps=5))
    for blocks in (38, 152, 608):
        rec(f"H2D copy kernel, {blocks} blocks", timeit(lambda: cp.cpattn_copy(dbuf, hbuf, n_blocks=blocks), reps=5))
        rec(f"D2H copy kernel, {blocks} blocks", timeit(lambda: cp.cpattn_copy(hbuf, dbuf, n_blocks=blocks), reps=5))
    # both directions at once, as the pipelined end-to-end step moves them: H2D of the
    # 805 MB above beside D2H of 805 MB from a second pair of buffers (bytes = both)
    hbuf2 = torch.empty(nb, dtype=torch.uint8, pin_memory=True)
    dbuf2 = torch.empty(nb, dtype=torch.uint8, device=dev)

    def both():
        cur = torch.cuda.current_stream(dev)
        for st in streams[:2]:
            st.wait_stream(cur)
        with torch.cuda.stream(streams[0]):
            dbuf.copy_(hbuf, non_blocking=True)
        with torch.cuda.stream(streams[1]):
            hbuf2.copy_(dbuf2, non_blocking=True)
        for st in streams[:2]:
            cur.wait_stream(st)

    sec = timeit(both, reps=5)
    link.append({"what": "H2D and D2H at once, cudaMemcpyAsync on two streams", "bytes": 2 * nb, "ms": sec * 1e3,
                 "GB_s": 2 * nb / sec / 1e9})
    del hbuf, dbuf, hbuf2, dbuf2
    ring = [materialised_ring(cp, inputs, dev, timeit),
            materialised_ring(cp, inputs, dev, timeit, "long_video_200k_gqa", reps=2)]
    # Dynamic-CP solver (host C++): the micro-batch count sweep over a global
    # batch of 2048 long-tailed samples, dp 8, pp 4, V 2, m = 4..16
    rng = np.random.default_rng(3)
    L = np.clip(np.exp(rng.normal(np.log(512), 1.2, 2048)), 64, 16384).astype(np.int64)
    reps, t0 = 5, time.perf_counter()
    for _ in range(reps):
        r = cp.cpattn_dcp_sweep(L, 8, 4, 2, 4, 8, 16384, 4 * 128 * 32, 0)
    host = [{"solver": "cpattn_dcp_sweep", "shape": "2048 samples, dp 8, pp 4, V 2, m 4..16 (13 schedules)",
             "ms": (time.perf_counter() - t0) / reps * 1e3, "knee_m": r["knee_m"], "best_m": r["best_m"]}]
    print(json.dumps({"aux": out, "host_link": link, "ring": ring, "host": host, "hbm_peak_GB_s": peak,
                      "peak_source": src}), flush=True)


def materialised_ring(cp, inputs, dev, timeit, name="dynamic_cp_microbatch", reps=5):
    """A workload's ring written out step by step: for each of the cp virtual
    ranks, cp block attention steps (cpattn_block_fwd, fp32 partial O and LSE
    per step) and one exact merge of the partials into the rank's rows; beside
    it the fused forward (cpattn_fwd) on the same inputs.  The ring's steps
    together cover every valid (query, key) pair once, so their FLOPs are the
    forward's.  The ranks run one after another and share the partial
    buffers; the block steps are also timed on their own."""
    import torch

    w = inputs.workload(name)
    q_h, k_h, v_h = inputs.make_qkv(w)
    qd, kd, vd = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    del q_h, k_h, v_h
    plan = cp.cpattn_plan(w.cu_seqlens, w.cp, w.mode, w.grid)
    ws = torch.empty(cp.cpattn_workspace_size(plan, w.H, w.Hkv, w.D, qd.dtype, w.causal), dtype=torch.uint8,
                     device=dev)
    ro = plan.rank_offsets()
    idx = torch.from_numpy(plan.index_map()).to(dev)
    rows = [int(ro[r + 1] - ro[r]) for r in range(w.cp)]
    n_max = max(rows)
    po_buf = [torch.empty(n_max * w.H * w.D, dtype=torch.float32, device=dev) for _ in range(w.cp)]
    pl_buf = [torch.empty(w.H * n_max, dtype=torch.float32, device=dev) for _ in range(w.cp)]
    po = [[b[:n * w.H * w.D].view(n, w.H, w.D) for b in po_buf] for n in rows]
    pl = [[b[:w.H * n].view(w.H, n) for b in pl_buf] for n in rows]
    o = torch.empty_like(qd)
    lse = torch.empty((w.H, w.T), dtype=torch.float32, device=dev)
    flops = cp.cpattn_fwd_flops(w.cu_seqlens, w.H, w.D, w.causal)
    peak, _ = measured_peak()

    def steps(r):
        for t in range(w.cp):
            cp.cpattn_block_fwd(plan, qd, kd, vd, po[r][t], pl[r][t], ws, r, t, scale=w.scale, causal=w.causal)

    def merge(r):
        cp.cpattn_merge(po[r], pl[r], o, lse, out_rows=idx[int(ro[r]):int(ro[r + 1])])

    def ring():
        for r in range(w.cp):
            steps(r)
            merge(r)

    def all_steps():
        for r in range(w.cp):
            steps(r)

    def fused():
        cp.cpattn_fwd(plan, qd, kd, vd, o, lse, ws, scale=w.scale, causal=w.causal)

    res = {}
    for key, fn in (("ring (steps + merges)", ring), ("block steps", all_steps), ("fused forward", fused)):
        sec = timeit(fn, reps=reps)
        tf = flops / sec / 1e12
        res[key] = {"ms": sec * 1e3, "TFLOP/s": tf, "frac": tf / peak}
    cp.cpattn_sync_status(ws)
    return {"workload": w.name, "shape": f"cp={w.cp} ranks x {w.cp} steps, T={w.T}, H={w.H}, Hkv={w.Hkv}, D={w.D}",
            "flops": flops, "launches": w.cp * (w.cp + 1), **res}


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_baseline_child:
        cpu_baseline_child(args)
        return
    if args.aux:
        run_aux(args)
        return
    if args.bwd:
        run_bwd(args)
        return
    if args.impl == "reference":
        # host-only: rank 0 runs it, other ranks exit without work (no process group)
        if int(os.environ.get("RANK", "0")) != 0:
            return
        if os.environ.get("OPENBLAS_NUM_THREADS") != "1":
            # the oracle's thread pool supplies the parallelism: restart with
            # single-threaded BLAS, as the cpu_baseline child does
            env = dict(os.environ)
            for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
                env[var] = "1"
            sys.stdout.flush()
            os.execve(sys.executable, [sys.executable, os.path.abspath(__file__)] + sys.argv[1:], env)
        run_reference(args)
        return
    rep = Replicas()
    try:
        run_ours(args, rep)
    finally:
        rep.close()


if __name__ == "__main__":
    main()
