#!/usr/bin/env python
"""Benchmark of the fused selective scan (and the decode step) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one forward selective scan over the Mamba-2.8B-shaped layer
(batch 4, 5,120 channels, N = 16, L = 2,048, bf16 I/O, fp32 state), inputs
resident in HBM.  Under torchrun every rank scans its own copy of the layer
(channels are independent: no data-path collective, weak scaling); rank 0
prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on the
host cores on a bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan Gelem/s (batch·D·L) and HBM GB/s, % of min(HBM,MUFU) roofline"
UNIT = "Gelem/s"
WORKLOAD = "mamba2.8b_layer_L2048"
DECODE = "decode_b256_64tok"
HBM_FALLBACK_GBS = 6400.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-conv", action="store_true", help="skip the convolution kernels")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward scan")
    ap.add_argument("--no-ssd", action="store_true", help="skip the Mamba-2 (SSD) layer scan")
    ap.add_argument("--bwd-batch", type=int, default=0,
                    help="sequences of the layer the backward runs on (default: all of them)")
    ap.add_argument("--no-other", action="store_true", help="skip the other scan workloads")
    ap.add_argument("--settle-s", type=float, default=0.5,
                    help="seconds of untimed load before the timed region (clock settling)")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "MEASURED_PEAKS.json (copy, measured)"
    return HBM_FALLBACK_GBS, "fallback"


# ------------------------------------------------------------------ ranks
# Every rank scans its own copy of the workload: channels (and sequences) are
# independent recurrences, so there is no data-path exchange between ranks.
# Ranks meet only at the barriers around the timed region and in the max of
# their timings.

def rank_barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value of x over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(elems_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job Gelem/s: the elements every rank processed over the slowest rank's time."""
    return elems_per_rank * world / (ms_max / 1e3) / 1e9


# ------------------------------------------------------------------ ncu record
TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "scan_ws_kernel": ["scan_fwd.cu", "ssm_device.cuh", "ssm_internal.h"],
    "step_stream_kernel": ["state_update.cu", "ssm_device.cuh", "ssm_internal.h"],
    "conv1d_stream_kernel": ["conv1d.cu", "ssm_device.cuh", "ssm_internal.h"],
    "conv1d_step8_kernel": ["conv1d.cu", "ssm_device.cuh", "ssm_internal.h"],
    "bwd_rev_kernel": ["scan_bwd.cu", "ssm_device.cuh", "ssm_internal.h"],
    "ssd_kernel": ["ssd.cu", "ssm_device.cuh", "ssm_internal.h"],
}


def source_hash(kernel: str) -> str:
    """sha256 over the CUDA sources a kernel is built from."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "mamba_selective_scan_02_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu record, or None when the
    record is missing or was taken on different kernel sources."""
    try:
        with open(TRAFFIC) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons during the timed region (read-only).

    Uses NVML through pynvml when it is importable, else a ``nvidia-smi
    --query-gpu ... -lms`` child process; both only read the GPU's state."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown",
                  "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, torch_index: int, period_s: float = 0.05):
        self.samples, self.period, self.ok, self.mode = [], period_s, False, None
        self.max_mhz = None
        self._stop = threading.Event()
        import torch
        uuid = str(torch.cuda.get_device_properties(torch_index).uuid)
        self.uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        try:
            import pynvml
            pynvml.nvmlInit()
            self.h = pynvml.nvmlDeviceGetHandleByUUID(self.uuid)
            self.nv = pynvml
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.ok, self.mode = True, "nvml"
        except Exception as e:
            self.err = repr(e)
            import shutil
            if shutil.which("nvidia-smi"):
                self.ok, self.mode = True, "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                mhz = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                reasons = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                self.samples.append((mhz, reasons))
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run_nvml, daemon=True)
            self.t.start()
        elif self.mode == "nvidia-smi":
            import subprocess
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, "--query-gpu=" + ",".join(self.SMI_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(int(self.period * 1000))],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self.mode == "nvml":
            self.t.join()
        elif self.mode == "nvidia-smi":
            self.proc.terminate()
            out, _ = self.proc.communicate()
            bits = {2: 0x8, 3: 0x40, 4: 0x20, 5: 0x4}
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) != len(self.SMI_FIELDS):
                    continue
                try:
                    mhz, self.max_mhz = float(f[0]), float(f[1])
                except ValueError:
                    continue
                mask = 0
                for i, bit in bits.items():
                    if f[i].lower() == "active":
                        mask |= bit
                self.samples.append((mhz, mask))

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": getattr(self, "err", "no samples")}
        mask = 0
        for _, r in self.samples:
            mask |= r
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(v for k, v in self.REASONS.items() if mask & k),
                "samples": len(self.samples), "source": self.mode}


# ------------------------------------------------------------------ CPU oracle
def oracle_rate(w, seconds: float, cores: int, seed_offset: int = 0):
    """Gelem/s of the fp64 oracle on a bounded sample of ``w``: the unchanged
    sequential oracle, its independent (b, d) channels split over host threads.
    The sample is the first ``dim`` channels of one sequence (all L tokens),
    repeated until about ``seconds`` of CPU work has been timed."""
    from mamba_selective_scan_02_b300.inputs import make_inputs
    from oracle import oracle as orc

    probe = make_inputs(w, batch=1, dim=max(1, cores), seed=w.seed + 1000 + seed_offset)
    t0 = time.perf_counter()
    orc.scan(probe["u"], probe["delta"], probe["A"], probe["B"], probe["C"], Dskip=probe["Dskip"],
             z=probe["z"], bias=probe["bias"], threads=cores)
    per_round = max(time.perf_counter() - t0, 1e-3)        # one channel per core
    rounds = max(1, int(seconds / per_round))
    dim = min(w.dim, cores * rounds)
    inp = make_inputs(w, batch=1, dim=dim, seed=w.seed + 2000 + seed_offset)
    reps, dt = 0, 0.0
    while reps == 0 or dt < 0.8 * seconds:
        t0 = time.perf_counter()
        orc.scan(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], Dskip=inp["Dskip"], z=inp["z"],
                 bias=inp["bias"], threads=cores)
        dt += time.perf_counter() - t0
        reps += 1
    elems = reps * dim * w.seqlen
    return elems / dt / 1e9, dt, (f"{reps} x ({dim} channels x {w.seqlen} tokens, N={w.dstate}) "
                                  f"of {w.name}")


def run_reference(args):
    from mamba_selective_scan_02_b300.inputs import WORKLOADS
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[WORKLOAD]
    cores = os.cpu_count() or 1
    per_step = max(0.5, 90.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup):
        oracle_rate(w, per_step, cores, seed_offset=i)
    rates, secs = [], 0.0
    sample = ""
    for i in range(args.steps):
        r, dt, sample = oracle_rate(w, per_step, cores, seed_offset=100 + i)
        rates.append(r)
        secs += dt
    value = statistics.median(rates)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                   "seqlen": w.seqlen, "io_dtype": w.io_dtype},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample + " per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------ GPU path
def run_ours(args):
    import torch
    import torch.distributed as dist

    from mamba_selective_scan_02_b300 import api, capi
    from mamba_selective_scan_02_b300.inputs import WORKLOADS, make_inputs
    from mamba_selective_scan_02_b300.roofline import (algorithmic_bytes_scan,
                                                        algorithmic_bytes_step, exps_scan)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        rank_barrier(world)

    def allmax(x):
        return max_over_ranks(x, world, dev)

    w = WORKLOADS[WORKLOAD]
    inp = make_inputs(w, device=dev)
    y = torch.empty_like(inp["u"])
    hL = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=dev)
    ws = torch.empty(api.workspace_bytes(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"]),
                     dtype=torch.uint8, device=dev)
    p = api.scan_params(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], inp["Dskip"], inp["z"],
                        inp["bias"], None, y=y, hL=hL, workspace=ws)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        """Evict L2: write a buffer twice its size, then read another one, so the
        dirty lines are written back before (not during) the timed launch."""
        flush_w.zero_()
        flush_r.sum()
    plan = capi.ssm_scan_plan(p)
    # B/C widening + scan (chained, one chunk, or look-back alike)
    launches_per_step = 2

    # MUFU ex2 peak, measured on this GPU (the roofline's exponential side)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.empty(sms * 8 * 256, dtype=torch.float32, device=dev)
    iters = 2048
    ex2_count = sms * 8 * 256 * iters * 16
    best = math.inf
    for i in range(8):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        capi.check(capi.ssm_bench_mufu_ex2(sink.data_ptr(), sms * 8, iters, sh), "mufu bench")
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            best = min(best, e0.elapsed_time(e1))
    mufu_peak = ex2_count / (best / 1e3) / 1e9  # G ex2/s

    elems = w.batch * w.dim * w.seqlen
    alg_bytes = algorithmic_bytes_scan(w.batch, w.dim, w.dstate, w.seqlen, 2)
    exps = exps_scan(w.batch, w.dim, w.dstate, w.seqlen)
    hbm_peak, hbm_src = measured_peaks()

    for _ in range(max(3, args.warmup)):
        capi.check(capi.ssm_scan_fwd(p, sh), "ssm_scan_fwd")
    torch.cuda.synchronize(dev)
    capi.check(api.workspace_status(ws), "scan status")

    clocks = ClockSampler(local)
    with clocks:
        # keep warming until clocks settle (>= 0.5 s of load), then time exactly K steps
        t_end = time.perf_counter() + args.settle_s
        while time.perf_counter() < t_end:
            for _ in range(50):
                capi.ssm_scan_fwd(p, sh)
            torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        ev[0].record(stream)
        for i in range(args.steps):
            capi.ssm_scan_fwd(p, sh)
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    capi.check(api.workspace_status(ws), "scan status")
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    total_ms_max = allmax(total_ms)
    ms_step = total_ms_max / args.steps
    value = weak_scaling_value(elems * args.steps, world, total_ms_max)
    kern_ms = statistics.mean(per_step)
    achieved_ex2 = exps / (kern_ms / 1e3) / 1e9
    achieved_gbs = alg_bytes / (kern_ms / 1e3) / 1e9

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate,
                   "seqlen": w.seqlen, "io_dtype": w.io_dtype, "state_dtype": "f32",
                   "parallelism": f"replicas x{world} (independent channels)",
                   "scan_plan": plan,
                   "l2": f"inputs larger than L2 ({alg_bytes / 1e6:.1f} MB per step)"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {
            "bound": "alu", "unit": "Gex2/s", "achieved": achieved_ex2, "peak": mufu_peak,
            "frac": achieved_ex2 / mufu_peak, "traffic": recorded_traffic("scan_ws_kernel"),
            "peak_source": "MUFU ex2.approx throughput measured in this run (ssm_bench_mufu_ex2)",
            "kernel_ms": kern_ms,
            "hbm": {"achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved_gbs / hbm_peak, "peak_source": hbm_src,
                    "algorithmic_bytes": alg_bytes},
            "roofline_gelem_s": min(mufu_peak / w.dstate, hbm_peak / (alg_bytes / elems)),
        },
        "clocks": clocks.summary(),
    }

    # ---- the other scan workloads (parity cases), timed the same way, kernel only
    if not args.no_other:
        others = {}
        for name in ("small_layer_L2048", "long_seq_L131072"):
            wo = WORKLOADS[name]
            oi = make_inputs(wo, device=dev)
            oy = torch.empty_like(oi["u"])
            oh = torch.empty((wo.batch, wo.dim, wo.dstate), dtype=torch.float32, device=dev)
            ows = torch.empty(api.workspace_bytes(oi["u"], oi["delta"], oi["A"], oi["B"], oi["C"]),
                              dtype=torch.uint8, device=dev)
            op = api.scan_params(oi["u"], oi["delta"], oi["A"], oi["B"], oi["C"], oi["Dskip"], oi["z"],
                                 oi["bias"], None, y=oy, hL=oh, workspace=ows)
            reps = 3 if wo.seqlen > 100000 else 50
            for _ in range(3):
                capi.ssm_scan_fwd(op, sh)
            tms = []
            for _ in range(reps):
                flush_l2()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                capi.ssm_scan_fwd(op, sh)
                e1.record(stream)
                tms.append((e0, e1))
            torch.cuda.synchronize(dev)
            capi.check(api.workspace_status(ows), name)
            oms = statistics.median(a_.elapsed_time(b_) for a_, b_ in tms)
            oel = wo.batch * wo.dim * wo.seqlen
            oex = exps_scan(wo.batch, wo.dim, wo.dstate, wo.seqlen)
            obytes = algorithmic_bytes_scan(wo.batch, wo.dim, wo.dstate, wo.seqlen, 2)
            others[name] = {"ms": oms, "Gelem_s": oel / (oms / 1e3) / 1e9,
                            "mufu_frac": oex / (oms / 1e3) / 1e9 / mufu_peak,
                            "hbm_frac": obytes / (oms / 1e3) / 1e9 / hbm_peak,
                            "l2": "L2 flushed before every timed launch (256 MB written, 256 MB read)"}
            out["gpu_launches"] += reps + 3
            del oi, oy, oh, ows
        out["other_workloads"] = others

    # ---- end to end through the C ABI from pinned host buffers.  Steps
    # alternate between two buffer sets on two streams, so one step's
    # device-to-host read overlaps the next step's host-to-device copy (the two
    # directions use different copy engines); every step still moves its whole
    # input and output across PCIe inside the timed region.
    if not args.no_e2e:
        names = ("u", "delta", "z", "B", "C")
        small = ("A", "Dskip", "bias")
        host = {k: inp[k].cpu().pin_memory() for k in names + small}
        streams = [stream, torch.cuda.Stream(dev)]
        sets = []
        for si_ in range(2):
            dbuf = {k: torch.empty_like(inp[k]) for k in names + small}
            ye, he = torch.empty_like(y), torch.empty_like(hL)
            wse = torch.empty_like(ws)
            hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
            hh = torch.empty(hL.shape, dtype=hL.dtype).pin_memory()
            pe = api.scan_params(dbuf["u"], dbuf["delta"], dbuf["A"], dbuf["B"], dbuf["C"], dbuf["Dskip"],
                                 dbuf["z"], dbuf["bias"], None, y=ye, hL=he, workspace=wse)
            sets.append((dbuf, ye, he, hy, hh, pe))
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = y.numel() * y.element_size() + hL.numel() * hL.element_size()

        def e2e_step(i):
            dbuf, ye, he, hy, hh, pe = sets[i % 2]
            st_ = streams[i % 2]
            with torch.cuda.stream(st_):
                for k, t in host.items():
                    dbuf[k].copy_(t, non_blocking=True)
                capi.ssm_scan_fwd(pe, st_.cuda_stream)
                hy.copy_(ye, non_blocking=True)
                hh.copy_(he, non_blocking=True)

        for i in range(max(3, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        ksteps = max(4, min(args.steps, 50))
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(streams[0])
        streams[1].wait_event(e0)
        for i in range(ksteps):
            e2e_step(i)
        done1 = torch.cuda.Event()
        done1.record(streams[1])
        streams[0].wait_event(done1)
        e1.record(streams[0])
        torch.cuda.synchronize(dev)
        barrier()
        ms = allmax(e0.elapsed_time(e1))
        out["e2e"] = {"value": elems * ksteps * world / (ms / 1e3) / 1e9, "unit": UNIT,
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": ksteps,
                      "ms_per_step": ms / ksteps,
                      "pipelining": "two buffer sets on two streams (copy directions overlap)"}
        out["gpu_launches"] += launches_per_step * ksteps
        del host, sets

    # ---- decode: 64 consecutive tokens, L2 flushed before each (cold state as in a deep stack)
    if not args.no_decode:
        wd = WORKLOADS[DECODE]
        dinp = make_inputs(wd, device=dev)
        state = dinp["h0"].clone()
        ydec = torch.empty((wd.batch, wd.dim), dtype=dinp["u"].dtype, device=dev)
        tok = [api.step_params(state, dinp["u"][t], dinp["delta"][t], dinp["A"], dinp["B"][t], dinp["C"][t],
                               dinp["Dskip"], dinp["z"][t], dinp["bias"], y=ydec) for t in range(wd.seqlen)]
        for t in range(4):
            capi.check(capi.ssm_state_update(tok[t], sh), "ssm_state_update")
        state.copy_(dinp["h0"])
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(wd.seqlen)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(wd.seqlen)]
        for t in range(wd.seqlen):
            flush_l2()
            starts[t].record(stream)
            capi.ssm_state_update(tok[t], sh)
            ends[t].record(stream)
        torch.cuda.synchronize(dev)
        tms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        dbytes = algorithmic_bytes_step(wd.batch, wd.dim, wd.dstate, 2)
        flushed_ms = statistics.mean(tms)
        flushed_gbs = dbytes / (flushed_ms / 1e3) / 1e9
        # The workload as it is stated: the 64 tokens back to back, one launch
        # after the other with nothing in between (each token's state
        # write-back is paid wherever it lands), the mean over three passes
        # from the same starting state.
        b2b = []
        for rep in range(3):
            state.copy_(dinp["h0"])
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for t in range(wd.seqlen):
                capi.ssm_state_update(tok[t], sh)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            b2b.append(e0.elapsed_time(e1) / wd.seqlen)
        mean_ms = statistics.median(b2b)
        gbs = dbytes / (mean_ms / 1e3) / 1e9
        out["decode"] = {"workload": wd.name, "tokens": wd.seqlen, "ms_per_token": mean_ms,
                         "value": wd.batch * wd.dim / (mean_ms / 1e3) / 1e9, "unit": UNIT,
                         "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                                      "frac": gbs / hbm_peak,
                                      "traffic": recorded_traffic("step_stream_kernel"),
                                      "algorithmic_bytes": dbytes},
                         "timing": "64 tokens back to back from one event pair (median of 3 passes; "
                                   "L2 flushed once before each pass); state 83.9 MB",
                         "flushed": {"ms_per_token": flushed_ms, "achieved": flushed_gbs,
                                     "frac": flushed_gbs / hbm_peak,
                                     "l2": "L2 flushed before every token (256 MB written, then another "
                                           "256 MB read so the written lines are back in HBM)"}}
        out["gpu_launches"] += 4 * wd.seqlen + 4

    # ---- the backward scan on the same layer: dy drawn like y, L2 flushed
    # before every launch (its inputs and outputs exceed L2 anyway)
    if not args.no_bwd:
        from mamba_selective_scan_02_b300.roofline import algorithmic_bytes_bwd
        bb = args.bwd_batch or w.batch          # sequences of the layer the backward runs on
        bi = {k: (inp[k][:bb] if k in ("u", "delta", "z", "B", "C") else inp[k]) for k in inp}
        g = torch.Generator(device=dev).manual_seed(41)
        dy = torch.randn(bi["u"].shape, generator=g, device=dev).to(bi["u"].dtype)
        bshape = (bb, w.dstate, w.seqlen)
        bout = dict(du=torch.empty_like(bi["u"]), ddelta=torch.empty_like(bi["u"]), dz=torch.empty_like(bi["u"]),
                    dB=torch.empty(bshape, dtype=torch.float32, device=dev),
                    dC=torch.empty(bshape, dtype=torch.float32, device=dev),
                    dA=torch.empty((w.dim, w.dstate), dtype=torch.float32, device=dev),
                    dD=torch.empty(w.dim, dtype=torch.float32, device=dev),
                    ddelta_bias=torch.empty(w.dim, dtype=torch.float32, device=dev))
        bws = torch.empty(api.bwd_workspace_bytes(bb, w.dim, w.dstate, w.seqlen, dtype=bi["u"].dtype),
                          dtype=torch.uint8, device=dev)
        # With room for it, the checkpoint pass runs on the forward scan kernel
        # (B, C widening + checkpoint launch) ahead of the reverse pass.
        fwd_ckpt = bws.numel() > api.bwd_workspace_bytes(bb, w.dim, w.dstate, w.seqlen, dtype=torch.float32)
        kpc = 3 if fwd_ckpt else 2
        bp = api.bwd_params(bi["u"], bi["delta"], bi["A"], bi["B"], bi["C"], dy, bi["Dskip"], bi["z"],
                            bi["bias"], None, None, workspace=bws, **bout)
        for _ in range(3):
            capi.check(capi.ssm_scan_bwd(bp, sh), "ssm_scan_bwd")
        tms = []
        for _ in range(20):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            capi.ssm_scan_bwd(bp, sh)
            e1.record(stream)
            tms.append((e0, e1))
        torch.cuda.synchronize(dev)
        capi.check(api.workspace_status(bws), "ssm_scan_bwd")
        bms = statistics.median(a_.elapsed_time(b_) for a_, b_ in tms)
        bbytes = algorithmic_bytes_bwd(bb, w.dim, w.dstate, w.seqlen, bi["u"].element_size())
        bgbs = bbytes / (bms / 1e3) / 1e9
        bex = exps * bb / w.batch / (bms / 1e3) / 1e9
        out["backward"] = {
            "workload": w.name, "ms": bms, "value": elems * bb / w.batch / (bms / 1e3) / 1e9, "unit": UNIT,
            "roofline": {"bound": "hbm", "achieved": bgbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": bgbs / hbm_peak, "algorithmic_bytes": bbytes,
                         "traffic": recorded_traffic("bwd_rev_kernel"),
                         "mufu": {"achieved": bex, "peak": mufu_peak, "unit": "Gex2/s", "frac": bex / mufu_peak,
                                  "note": "one exp per (b, d, n, t), the forward's count"}},
            "kernels_per_call": kpc, "batch": bb,
            "checkpoints": "forward scan kernel, checkpoint mode" if fwd_ckpt else "backward checkpoint kernel",
            "l2": "L2 flushed before every launch (256 MB written, 256 MB read)"}
        out["gpu_launches"] += 23 * kpc
        del dy, bout, bws, bi

    # ---- the Mamba-2 layer scan (SSD): the Mamba-2 2.7B layer (80 heads of 64,
    # N = 128) at the same batch and length, L2 flushed before every launch
    if not args.no_ssd:
        from mamba_selective_scan_02_b300.inputs import make_ssd_inputs
        from mamba_selective_scan_02_b300.roofline import algorithmic_bytes_ssd, flops_ssd
        sb, sL, sH, sP, sN = w.batch, w.seqlen, 80, 64, 128
        si = make_ssd_inputs(sb, sL, sH, sP, sN, seed=51, device=dev)
        sy = torch.empty_like(si["x"])
        shL = torch.empty((sb, sH, sP, sN), dtype=torch.float32, device=dev)
        sws = torch.empty(api.ssd_workspace_bytes(sb, sL, sH, sP, sN), dtype=torch.uint8, device=dev)
        sp = api.ssd_params(si["x"], si["dt"], si["A"], si["B"], si["C"], si["D"], si["dt_bias"], None,
                            y=sy, hL=shL, workspace=sws)
        for _ in range(3):
            capi.check(capi.ssm_ssd_fwd(sp, sh), "ssm_ssd_fwd")
        tms = []
        for _ in range(30):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            capi.ssm_ssd_fwd(sp, sh)
            e1.record(stream)
            tms.append((e0, e1))
        torch.cuda.synchronize(dev)
        sms_ = statistics.median(a_.elapsed_time(b_) for a_, b_ in tms)
        sbytes = algorithmic_bytes_ssd(sb, sL, sH, sP, sN)
        sflops = flops_ssd(sb, sL, sH, sP, sN, chunk=128)   # the kernel's chunk length
        sgbs = sbytes / (sms_ / 1e3) / 1e9
        stf = sflops / (sms_ / 1e3) / 1e12
        bf16_peak = None
        try:
            with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                bf16_peak = float(json.load(f)["bf16_tflops"])
        except (OSError, ValueError, KeyError):
            bf16_peak = 1800.0  # the profiling recipe's fallback burst figure
        t_hbm, t_tc = sbytes / (hbm_peak * 1e9), (sflops / (bf16_peak * 1e12) if bf16_peak else 0.0)
        bound = "hbm" if t_hbm >= t_tc else "tensor"
        out["ssd"] = {
            "workload": f"mamba2_2.7b_layer_b{sb}_L{sL}_H{sH}_P{sP}_N{sN}", "ms": sms_,
            "value": sb * sL * sH * sP / (sms_ / 1e3) / 1e9, "unit": UNIT,
            "roofline": ({"bound": "hbm", "achieved": sgbs, "peak": hbm_peak, "unit": "GB/s",
                          "frac": sgbs / hbm_peak, "traffic": recorded_traffic("ssd_kernel")} if bound == "hbm" else
                         {"bound": "tensor", "achieved": stf, "peak": bf16_peak, "unit": "TFLOP/s",
                          "frac": stf / bf16_peak}),
            "algorithmic_bytes": sbytes, "flops": sflops, "tflops": stf,
            "tensor_path": "tcgen05.mma kind::f16 (bf16 operands, fp32 accumulators in TMEM), TMA-fed 128-token chunks",
            "chains": "each (sequence, head) chain in segments handing the state on through the workspace",
            "l2": "L2 flushed before every launch (256 MB written, 256 MB read)"}
        out["gpu_launches"] += 33
        del si, sy, shL, sws

    # ---- the short convolution in front of the scan: the layer shape (sequence
    # form) and the decode batch (one token), L2 flushed before every launch
    if not args.no_conv:
        from mamba_selective_scan_02_b300.inputs import make_conv_inputs
        from mamba_selective_scan_02_b300.roofline import algorithmic_bytes_conv, algorithmic_bytes_conv_step
        cw = 4
        ci = make_conv_inputs(w.batch, w.dim, w.seqlen, cw, w.io_dtype, seed=31, device=dev)
        cu = torch.empty_like(ci["x"])
        cso = torch.empty_like(ci["state"])
        cp = api.conv_params(ci["x"], ci["weight"], ci["bias"], ci["state"], u=cu, state_out=cso)
        for _ in range(3):
            capi.check(capi.ssm_conv1d_fwd(cp, sh), "ssm_conv1d_fwd")
        tms = []
        for _ in range(50):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            capi.ssm_conv1d_fwd(cp, sh)
            e1.record(stream)
            tms.append((e0, e1))
        torch.cuda.synchronize(dev)
        cms = statistics.median(a_.elapsed_time(b_) for a_, b_ in tms)
        cbytes = algorithmic_bytes_conv(w.batch, w.dim, w.seqlen, cw, ci["x"].element_size())
        cgbs = cbytes / (cms / 1e3) / 1e9
        conv = {"workload": f"conv1d_W{cw}_b{w.batch}_D{w.dim}_L{w.seqlen}", "ms": cms,
                "value": w.batch * w.dim * w.seqlen / (cms / 1e3) / 1e9, "unit": UNIT,
                "roofline": {"bound": "hbm", "achieved": cgbs, "peak": hbm_peak, "unit": "GB/s",
                             "frac": cgbs / hbm_peak, "traffic": recorded_traffic("conv1d_stream_kernel"),
                             "algorithmic_bytes": cbytes},
                "l2": "L2 flushed before every launch (256 MB written, 256 MB read)"}
        del ci, cu, cso
        wd = WORKLOADS[DECODE]
        si = make_conv_inputs(wd.batch, wd.dim, 8, cw, wd.io_dtype, seed=32, device=dev, decode=True)
        sstate = si["state"].clone()
        su = torch.empty((wd.batch, wd.dim), dtype=si["x"].dtype, device=dev)
        sp = []
        for t in range(8):
            q = capi.ConvStepParams()
            q.batch, q.dim, q.width = wd.batch, wd.dim, cw
            q.io_dtype = capi.SSM_BF16 if si["x"].dtype == torch.bfloat16 else capi.SSM_F32
            q.state, q.x, q.weight, q.bias = (sstate.data_ptr(), si["x"][t].data_ptr(),
                                              si["weight"].data_ptr(), si["bias"].data_ptr())
            q.silu, q.u = 1, su.data_ptr()
            sp.append(q)
        for t in range(3):
            capi.check(capi.ssm_conv1d_step(sp[t], sh), "ssm_conv1d_step")
        tms = []
        for t in range(8):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            capi.ssm_conv1d_step(sp[t], sh)
            e1.record(stream)
            tms.append((e0, e1))
        torch.cuda.synchronize(dev)
        sms = statistics.median(a_.elapsed_time(b_) for a_, b_ in tms)
        sbytes = algorithmic_bytes_conv_step(wd.batch, wd.dim, cw, si["x"].element_size())
        sgbs = sbytes / (sms / 1e3) / 1e9
        conv["decode_step"] = {"workload": f"conv1d_step_W{cw}_b{wd.batch}_D{wd.dim}", "ms": sms,
                               "roofline": {"bound": "hbm", "achieved": sgbs, "peak": hbm_peak,
                                            "unit": "GB/s", "frac": sgbs / hbm_peak,
                                            "traffic": recorded_traffic("conv1d_step8_kernel"),
                                            "algorithmic_bytes": sbytes}}
        out["conv1d"] = conv
        out["gpu_launches"] += 53 + 11
        del si, sstate, su

    # ---- CPU baseline: the fp64 oracle on a bounded sample (rank 0 only)
    if rank == 0 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        r, dt, sample = oracle_rate(w, 15.0, cores)
        r1, dt1, sample1 = oracle_rate(w, 6.0, 1, seed_offset=7)
        out["cpu_baseline"] = {"value": r, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": sample, "seconds": dt,
                               "single_thread": {"value": r1, "unit": UNIT, "cores": 1, "sample": sample1,
                                                 "seconds": dt1}}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
