#!/usr/bin/env python
"""Throughput of the chunked TTT-Linear scan on B300, one JSON line.

A step is one ttt_linear_fwd over the whole long-context workload
(B1 H32 T131072 d64, chunk b = 16, bf16 Q/K/V, fp32 state): every stage of the
hot path (chunk loads, error at the chunk start, intra-chunk scores, read-out,
state update, write-back of Z and W_out). With 32 heads the library runs the
segment-parallel form: an affine-map kernel, a combine kernel and the read-out
kernel. Metric: token·heads per second, and the dominant kernel's fraction of
the HBM roofline (its algorithmic bytes over its own event-timed duration; for
the read-out kernel: Q, K, V read and Z written, plus the states), with every
kernel's share and the whole step's fraction beside it.

Arms
  default            our CUDA library through its C ABI (device-resident inputs),
                     plus an end-to-end figure through host buffers and the
                     oracle timed on the host cores as a CPU baseline.
  --impl reference   the fp64 CPU oracle on the host cores (a bounded sample of
                     the same workload per step): the baseline arm.

Multi-GPU: the (batch row, head) units are independent, so N GPUs run N
replicas of the workload (weak scaling, no collective); value = all ranks'
token·heads over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "TTT-Linear scan tokens·heads/sec and % of binding roofline (1×B300)"
UNIT = "token·heads/s"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6400.0
REFERENCE_BUDGET_S = 120.0  # wall time of the reference arm's warm-up and timed steps together
NOMINAL_HBM_GBS = 7700.0  # B300 HBM3e, vendor figure: context beside the measured copy bandwidth
# kernel -> (source files whose digest a committed ncu summary must match, summary file)
KERNEL_PROFILES = {
    "linear_mma_kernel": (("test_sequence_layers_06_b300/csrc/linear_mma.cu",), "profiles/linear_mma_long_b16.md"),
    "linear_seg_affine_kernel": (("test_sequence_layers_06_b300/csrc/linear_seg.cu",),
                                 "profiles/linear_seg_affine_long_b16.md"),
    "linear_seg_affine_wy_kernel": (("test_sequence_layers_06_b300/csrc/linear_seg_wy.cu",),
                                    "profiles/linear_seg_affine_wy_long_b16.md"),
    "linear_seg_combine_kernel": (("test_sequence_layers_06_b300/csrc/linear_seg.cu",),
                                  "profiles/linear_seg_combine_long_b16.md"),
}
BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="linear_long")
    ap.add_argument("--b", type=int, default=16)
    ap.add_argument("--T", type=int, default=0, help="override the workload's sequence length (profiling cases)")
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--mode", choices=["fwd", "bwd", "momentum", "ln", "decode"], default="fwd",
                    help="bwd: time the TTT-Linear backward (ttt_linear_bwd) on the workload instead; "
                         "momentum / ln: the inner-model variant's tensor-core kernel (bf16, d = 64, b = 16); "
                         "decode: ttt_linear_decode on the workload's heads, --T tokens per launch (default 1)")
    return ap.parse_args()


# --------------------------------------------------------------------------- helpers
def algorithmic_bytes(w: synth.Workload) -> int:
    """Bytes one pass must move: Q, K, V read and Z written once, W0 read once, W_out written once."""
    es = 2 if w.dtype == "bf16" else 4
    return w.token_heads * 4 * w.d * es + w.H * w.d * w.d * 4 + w.units * w.d * w.d * 4


def kernel_bytes(w: synth.Workload, plan) -> tuple:
    """Algorithmic bytes of each kernel of one step: (affine maps, combine, read-out).
    Affine maps: K, V of every segment that has a map read once, the maps written.
    Combine: the maps read, the start states written (and W0). Read-out: Q, K, V
    read and Z written once, W0 and the start states read, W_out written."""
    es = 2 if w.dtype == "bf16" else 4
    state = w.d * w.d * 4
    bounds = w.units * (plan["seg_count"] - 1)
    if bounds == 0:
        return 0, 0, algorithmic_bytes(w)
    affine = bounds * plan["seg_len"] * 2 * w.d * es + bounds * 2 * state
    combine = bounds * 3 * state + w.units * state
    return affine, combine, algorithmic_bytes(w) + bounds * state


def algorithmic_flops(w: synth.Workload, b: int) -> int:
    """Per chunk of b tokens: E, Q W and K^T E (2 b d^2 each) plus Q K^T and S E (2 b^2 d each)."""
    return w.token_heads * (6 * w.d * w.d + 4 * b * w.d)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, 1800.0, "fallback"


def source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_PROFILES[kernel][0]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """dram bytes per launch from the committed ncu summary of `kernel`, if it was taken on today's
    kernel source and on this workload."""
    path = os.path.join(ROOT, KERNEL_PROFILES[kernel][1])
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "kernel_source_sha",
                                                        "workload")):
                k, v = line.strip().split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != source_digest(kernel) or vals.get("workload") != workload:
        return None
    try:
        return int(float(vals["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def roofline_summary(names, kernel_ms, kbytes, ms_per_step: float, step_bytes: int, hbm_gbs: float,
                     peak_kind: str, traffic_of) -> dict:
    """The JSON line's roofline block: for each kernel with algorithmic bytes, those bytes over its
    mean event-timed duration against the HBM peak; the dominant (longest) kernel at the top level;
    the whole step's fraction; and each fraction also against the nominal HBM bandwidth."""
    kernels = {}
    for name, ms, nbytes in zip(names, kernel_ms, kbytes):
        if nbytes == 0:
            continue
        gbs = nbytes / (ms * 1e-3) / 1e9
        kernels[name] = {"ms": round(ms, 4), "share": round(ms / ms_per_step, 4), "algorithmic_bytes": nbytes,
                         "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm_gbs, 4),
                         "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4), "traffic": traffic_of(name)}
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["achieved_gbs"], "peak": hbm_gbs,
            "unit": "GB/s", "frac": kernels[dom]["frac"], "traffic": kernels[dom]["traffic"],
            "peak_kind": f"{peak_kind} (copy bandwidth, MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.4 TB/s",
            "frac_of_nominal": kernels[dom]["frac_of_nominal"], "nominal_gbs": NOMINAL_HBM_GBS,
            "algorithmic_bytes_per_launch": kernels[dom]["algorithmic_bytes"], "kernel_ms": kernels[dom]["ms"],
            "kernels": kernels,
            "step": {"algorithmic_bytes": step_bytes, "ms": round(ms_per_step, 4),
                     "frac": round(step_gbs / hbm_gbs, 4), "frac_of_nominal": round(step_gbs / NOMINAL_HBM_GBS, 4)}}


class _Nvml:
    """The few NVML calls the clock record needs, through ctypes on the driver's
    libnvidia-ml (no Python NVML package required)."""

    CLOCK_SM = 1

    def __init__(self, uuid: str | None, index: int):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        ok = False
        if uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for the device")
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def clock(self) -> int:
        c = ctypes.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ctypes.byref(c)) != 0:
            raise RuntimeError("nvmlDeviceGetClockInfo failed")
        return int(c.value)

    def max_clock(self) -> int:
        c = ctypes.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, ctypes.byref(c)) != 0:
            raise RuntimeError("nvmlDeviceGetMaxClockInfo failed")
        return int(c.value)

    def reasons(self) -> int:
        r = ctypes.c_ulonglong()
        if self._reasons(self.h, ctypes.byref(r)) != 0:
            raise RuntimeError("clock event reasons query failed")
        return int(r.value)


def _device_uuid(index: int):
    """'GPU-…' UUID of CUDA device `index` (NVML's numbering may differ from CUDA's)."""
    try:
        import torch
        u = getattr(torch.cuda.get_device_properties(index), "uuid", None)
        if u is None:
            return None
        u = str(u)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


class ClockSampler:
    """Samples the SM clock and the clock event (throttle) reasons while the timed region runs:
    NVML every ~2 ms (through ctypes), else nvidia-smi every 20 ms. Fewer than 3 samples are
    reported as unknown, never as clean."""

    NAMES = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
             0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
             0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}
    MIN_SAMPLES = 3

    def __init__(self, index: int, period_s: float = 0.002):
        self.ok = False
        self.samples = []
        self.reasons = 0
        self.period = period_s
        self.index = index
        self.mode = None
        self.error = None
        self.max_mhz = None
        try:
            self.nv = _Nvml(_device_uuid(index), index)
            self.max_mhz = self.nv.max_clock()
            self.ok, self.mode = True, "nvml"
        except Exception as e:  # no NVML: sample nvidia-smi instead
            self.error = repr(e)
            import shutil
            if shutil.which("nvidia-smi"):
                self.ok, self.mode = True, "nvidia-smi"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.clock())
                self.reasons |= self.nv.reasons()
            except Exception as e:
                self.error = repr(e)
            time.sleep(self.period)

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active")

    def _smi_reader(self):
        for line in self._p.stdout:
            if self._stop.is_set():
                continue  # drain without recording
            try:
                sm, mx, reasons = [x.strip() for x in line.split(",")]
                self.samples.append(float(sm))
                self.max_mhz = float(mx)
                self.reasons |= int(reasons, 16)
                self._first.set()
            except ValueError:
                continue

    def __enter__(self):
        self._stop = threading.Event()
        if self.mode == "nvml":
            self.samples.append(self.nv.clock())  # one sample before the timed work is enqueued
            self.reasons |= self.nv.reasons()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        elif self.mode == "nvidia-smi":
            import subprocess
            self._first = threading.Event()
            uuid = _device_uuid(self.index)
            self._p = subprocess.Popen(["nvidia-smi", "-i", uuid or str(self.index),
                                        f"--query-gpu={self.SMI_FIELDS}",
                                        "--format=csv,noheader,nounits", "-lms", "20"],
                                       stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._smi_reader, daemon=True)
            self._t.start()
            self._first.wait(5.0)  # the timed region starts once sampling runs
            self.samples.clear()
            self.reasons = 0
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self.mode == "nvml":
            self._t.join()
            try:  # one sample after the timed work has finished
                self.samples.append(self.nv.clock())
                self.reasons |= self.nv.reasons()
            except Exception as e:
                self.error = repr(e)
        elif self.mode == "nvidia-smi":
            self._p.terminate()
            self._t.join(2.0)

    def report(self):
        reasons = sorted(n for bit, n in self.NAMES.items() if self.reasons & bit and n != "gpu_idle")
        med = statistics.median(self.samples) if self.samples else None
        r = {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples),
             "source": self.mode}
        if len(self.samples) < self.MIN_SAMPLES:
            r["state"] = "unknown (too few samples in the timed region)"
        if self.error:
            r["error"] = self.error
        return r

    def rejected(self):
        """True: throttled or stuck clocks (measure again); None: unknown (too few samples)."""
        r = self.report()
        if set(r["reasons"]) & BAD_REASONS:
            return True
        if r["samples"] < self.MIN_SAMPLES:
            return None
        if r["sm_mhz"] and r["sm_max_mhz"] and not r["reasons"] and r["sm_mhz"] < 0.7 * r["sm_max_mhz"]:
            return True
        return False


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank runs its own replica of the workload
    (independent units, no collective on the data path), so the job takes as long
    as its slowest rank. The process group's backend decides the device (NCCL: the
    rank's GPU; gloo: the host)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: int, ms_per_step: float) -> float:
    """Whole-job token·heads/s: all ranks' units over the slowest rank's step time."""
    return world * units_per_rank / (ms_per_step * 1e-3)


# --------------------------------------------------------------------------- CPU oracle
def oracle_rate(w: synth.Workload, b: int, target_s: float):
    """The oracle (as it stands) on a bounded sample: every head of batch row 0, the first Ts tokens.
    Returns (token·heads/s, threads, sample description, seconds)."""
    import oracle
    threads = oracle.max_threads()

    def prepare(Ts):
        inp = synth.make_inputs(w.with_(B=1, T=Ts))
        if w.variant == "mlp":
            return lambda: oracle.mlp_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W1_64, inp.W2_64, b)
        return lambda: oracle.linear_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, b)

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    probe = max(b, 1024)
    dt = timed(prepare(probe))
    Ts = int(min(w.T, max(probe, probe * target_s / max(dt, 1e-6))))
    Ts = max(b, Ts // b * b)
    fn = prepare(Ts)
    reps, total = 0, 0.0
    while True:  # one pass over the sample, repeated until about target_s of work
        total += timed(fn)
        reps += 1
        if total >= 0.8 * target_s or reps >= 20:
            break
    sample = (f"{w.name}: batch row 0, all {w.H} heads, first {Ts} of {w.T} tokens, {reps} pass(es) "
              f"(fp64 primal oracle)")
    return reps * w.H * Ts / total, threads, sample, total


# --------------------------------------------------------------------------- our arm
def bench_ours(args, world, rank, local):
    import torch
    import test_sequence_layers_06_b300 as ttt
    sys.path.insert(0, os.path.join(ROOT, "tests"))

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = synth.WORKLOADS[args.workload].with_(b=args.b)
    if args.T:
        w = w.with_(T=args.T)
    inp = synth.make_inputs(w, want_exact=False)

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    Q, K, V = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
    eta, W0 = torch.from_numpy(inp.eta).to(dev), torch.from_numpy(inp.W0).to(dev)
    Z = torch.empty_like(Q)
    Wo = torch.empty((w.B, w.H, w.d, w.d), dtype=torch.float32, device=dev)
    ws = torch.zeros(ttt.ttt_workspace_bytes(w.B, w.H, w.T, w.d, args.b), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    plan = ttt.ttt_linear_plan(w.B, w.H, w.T, w.d, args.b, ttt.TTT_BF16 if w.dtype == "bf16" else ttt.TTT_F32)
    launches_per_step = plan["kernels"]  # plus a 16-byte status memset per call

    # Per-step phase events, recorded by the library on its stream around each kernel:
    # [start, after affine maps, after combine, after read-out].
    phase = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for evs in phase:  # create the CUDA events (torch makes them on first record)
        for e in evs:
            e.record(stream)
    phase_handles = [(ctypes.c_void_p * 4)(*[e.cuda_event for e in evs]) for evs in phase]
    phase_opts = [ttt.ttt_options(0, 0, 0, 0, ctypes.cast(h, ctypes.c_void_p)) for h in phase_handles]

    def step(i=None):
        ttt.ttt_linear_fwd(Q, K, V, eta, W0, args.b, Z=Z, W_out=Wo, workspace=ws, stream=stream,
                           options=None if i is None else phase_opts[i])

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if ttt.ttt_last_device_status(ws, stream) != 0:
        raise RuntimeError("device status not OK after warm-up")

    def timed():
        barrier()
        torch.cuda.synchronize()
        sampler = ClockSampler(local)
        with sampler:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for i in range(args.steps):
                step(i)
            t1.record(stream)
            torch.cuda.synchronize()
        barrier()
        total_ms = t0.elapsed_time(t1)
        per = [[evs[k].elapsed_time(evs[k + 1]) for k in range(3)] for evs in phase]
        return total_ms, per, sampler

    total_ms, per, sampler = timed()
    if sampler.rejected():  # throttled or stuck clocks: measure once more
        total_ms, per, sampler = timed()
    if ttt.ttt_last_device_status(ws, stream) != 0:
        raise RuntimeError("device status not OK after the timed region")

    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, w.token_heads, ms_per_step)

    # roofline: every kernel's algorithmic bytes over its own mean event-timed duration
    hbm_gbs, _, peak_kind = measured_peaks()
    kernel_ms = [float(np.mean([p[k] for p in per])) for k in range(3)]
    names = ("linear_seg_affine_wy_kernel" if plan["affine"] == 2 else "linear_seg_affine_kernel",
             "linear_seg_combine_kernel", "linear_mma_kernel")
    profile_key = f"{w.name} B{w.B} H{w.H} T{w.T} b{args.b}"
    roofline = roofline_summary(names, kernel_ms, kernel_bytes(w, plan), ms_per_step, algorithmic_bytes(w),
                                hbm_gbs, peak_kind, lambda name: profiled_traffic(name, profile_key))
    roofline["flops_per_step"] = algorithmic_flops(w, args.b)

    # end to end: pinned host buffers in, Z and W_out back out, through the public call
    e2e = None
    if args.e2e_steps > 0:
        hq = torch.from_numpy(inp.q.view(np.int16)).pin_memory() if inp.q.dtype == np.uint16 else \
            torch.from_numpy(inp.q).pin_memory()
        hk = torch.from_numpy(inp.k.view(np.int16)).pin_memory() if inp.k.dtype == np.uint16 else \
            torch.from_numpy(inp.k).pin_memory()
        hv = torch.from_numpy(inp.v.view(np.int16)).pin_memory() if inp.v.dtype == np.uint16 else \
            torch.from_numpy(inp.v).pin_memory()
        hz = torch.empty(hq.shape, dtype=hq.dtype).pin_memory()
        hw = torch.empty(tuple(Wo.shape), dtype=torch.float32).pin_memory()
        as_raw = (lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t)
        Qi, Ki, Vi, Zi = as_raw(Q), as_raw(K), as_raw(V), as_raw(Z)

        def e2e_step():
            Qi.copy_(hq, non_blocking=True)
            Ki.copy_(hk, non_blocking=True)
            Vi.copy_(hv, non_blocking=True)
            step()
            hz.copy_(Zi, non_blocking=True)
            hw.copy_(Wo, non_blocking=True)

        # Serial form: every step copies in, computes and copies out on one stream.
        e2e_step()
        torch.cuda.synchronize()
        barrier()
        a, bq = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        bq.record(stream)
        torch.cuda.synchronize()
        serial_ms = max_over_ranks(a.elapsed_time(bq) / args.e2e_steps, world, dev)

        # Streamed form (the e2e number): two sets of device buffers; step i's inputs go in on a
        # copy stream while step i - 1 computes and its results go out on a third stream, so
        # the host-to-device and device-to-host copies of neighbouring steps overlap. Every
        # step still copies its own inputs in and its own Z and W_out back.
        sets = [(Qi, Ki, Vi, Zi, Wo), tuple(torch.empty_like(t) for t in (Qi, Ki, Vi, Zi, Wo))]
        ws2 = [ws, torch.zeros_like(ws)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for e in ev_done + ev_out:
            e.record(stream)

        def streamed(n):
            for i in range(n):
                k = i % 2
                q_, k_, v_, z_, w_ = sets[k]
                s_in.wait_event(ev_done[k])        # step i - 2 has read this set's inputs
                with torch.cuda.stream(s_in):
                    q_.copy_(hq, non_blocking=True)
                    k_.copy_(hk, non_blocking=True)
                    v_.copy_(hv, non_blocking=True)
                    ev_in[k].record(s_in)
                stream.wait_event(ev_in[k])
                stream.wait_event(ev_out[k])       # step i - 2's results have left this set
                ttt.ttt_linear_fwd(q_.view(Q.dtype), k_.view(Q.dtype), v_.view(Q.dtype), eta, W0, args.b,
                                   Z=z_.view(Z.dtype), W_out=w_, workspace=ws2[k], stream=stream)
                ev_done[k].record(stream)
                s_out.wait_event(ev_done[k])
                with torch.cuda.stream(s_out):
                    hz.copy_(z_, non_blocking=True)
                    hw.copy_(w_, non_blocking=True)
                    ev_out[k].record(s_out)

        streamed(2)
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        streamed(args.e2e_steps)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, world, dev)
        for k in range(2):
            if ttt.ttt_last_device_status(ws2[k], stream) != 0:
                raise RuntimeError("device status not OK after the streamed end-to-end steps")
        h2d = hq.numel() * hq.element_size() * 3
        d2h = hz.numel() * hz.element_size() + hw.numel() * 4
        e2e = {"value": job_throughput(world, w.token_heads, e2e_ms), "unit": UNIT, "ms_per_step": round(e2e_ms, 3),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "form": "streamed: two device buffer sets, neighbouring steps' copies overlap (host clock)",
               "serial": {"value": job_throughput(world, w.token_heads, serial_ms), "ms_per_step": round(serial_ms, 3),
                          "form": "copy in, compute, copy out on one stream (CUDA events)"}}

    extras = {}
    if rank == 0 and not args.no_extras:
        try:
            extras = bench_extras(ttt, dev, stream)
        except Exception as exc:  # secondary workloads; the headline line is printed regardless
            extras = {"error": f"{type(exc).__name__}: {exc}"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, threads, sample, secs = oracle_rate(w, args.b, target_s=10.0)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
               "seconds": round(secs, 2)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "b": args.b,
                       "inputs": f"Q/K/V {w.dtype} {w.note}", "state": "fp32",
                       "path": {1: "fp32 SIMT", 2: "tensor-core one pass", 3: "segment-parallel"}[plan["path"]],
                       "seg_len": plan["seg_len"], "seg_count": plan["seg_count"],
                       "l2": "inputs larger than L2 (%.2f GB vs 126 MB)" % (3 * w.token_heads * w.d * 2 / 1e9),
                       "parallelism": f"replicas x{world} (independent units, no collective)"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": sampler.report(),
            "extras": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def bench_extras(ttt, dev, stream):
    """Secondary workloads, a few steps each (device-resident inputs)."""
    import torch
    hbm_gbs, tflops, _ = measured_peaks()
    out = {}

    def t_ms(fn, n, ahead=True):
        """Device time per call. With `ahead`, a bounded sleep kernel (torch's, a fixed cycle count)
        holds the stream while the n calls are enqueued, so the host cost of the binding does not
        show in the device time of short calls."""
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if ahead:
            with torch.cuda.stream(stream):
                torch.cuda._sleep(int(4e6) * (n + 1))  # about 2 ms per call at 2 GHz
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    def dev_inputs(w):
        inp = synth.make_inputs(w, want_exact=False)
        cv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev))
        return inp, cv(inp.q), cv(inp.k), cv(inp.v), torch.from_numpy(inp.eta).to(dev)

    for name, b in (("linear_125m", 16), ("linear_small", 16), ("linear_long", 64), ("linear_long", 256),
                    ("linear_long", 2048)):
        w = synth.WORKLOADS[name].with_(b=b)
        inp, Q, K, V, eta = dev_inputs(w)
        W0 = torch.from_numpy(inp.W0).to(dev)
        Z = torch.empty_like(Q)
        Wo = torch.empty((w.B, w.H, w.d, w.d), dtype=torch.float32, device=dev)
        ws = torch.zeros(ttt.ttt_workspace_bytes(w.B, w.H, w.T, w.d, b), dtype=torch.uint8, device=dev)
        ms = t_ms(lambda: ttt.ttt_linear_fwd(Q, K, V, eta, W0, b, Z=Z, W_out=Wo, workspace=ws, stream=stream),
                  10 if w.T < 100000 else 5)
        gbs = algorithmic_bytes(w) / (ms * 1e-3) / 1e9
        out[f"{name}_b{b}"] = {"ms": round(ms, 4), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                               "hbm_frac": round(gbs / hbm_gbs, 4)}
        del Q, K, V, Z
    # TTT-MLP
    w = synth.WORKLOADS["mlp_125m"]
    inp, Q, K, V, eta = dev_inputs(w)
    W1, W2 = torch.from_numpy(inp.W1).to(dev), torch.from_numpy(inp.W2).to(dev)
    ms = t_ms(lambda: ttt.ttt_mlp_fwd(Q, K, V, eta, W1, W2, 16, stream=stream), 2)
    m = w.hidden
    flops = w.token_heads * (16 * w.d * m + 4 * 16 * (w.d + m))
    out["mlp_125m_b16"] = {"ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                           "tensor_frac": round(flops / (ms * 1e-3) / (tflops * 1e12), 5)}
    # inner-model variants (fp32 SIMT kernel, one CTA per unit) on the small workload's shape
    try:
        w = synth.WORKLOADS["linear_small"]
        inp, Q, K, V, eta = dev_inputs(w)
        W0 = torch.from_numpy(inp.W0).to(dev)
        vec = torch.zeros((w.H, w.d), device=dev)
        gam = torch.ones((w.H, w.d), device=dev)
        et = torch.full((w.B, w.H, w.T), 0.1, device=dev)
        calls = {"bias": lambda: ttt.ttt_linear_bias_fwd(Q, K, V, eta, W0, vec, 16, stream=stream),
                 "token_eta": lambda: ttt.ttt_linear_token_eta_fwd(Q, K, V, et, W0, 16, stream=stream),
                 "ln_residual": lambda: ttt.ttt_linear_ln_fwd(Q, K, V, eta, W0, gam, vec, 16, stream=stream),
                 "momentum": lambda: ttt.ttt_linear_momentum_fwd(Q, K, V, eta, eta, W0, 16, stream=stream)}
        for name, fn in calls.items():
            ms = t_ms(fn, 3)
            out[f"variant_{name}_small_b16"] = {
                "ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                "hbm_frac": round(algorithmic_bytes(w) / (ms * 1e-3) / 1e9 / hbm_gbs, 5),
                "note": "B2 H4 T2048 d64 bf16 in, fp32 SIMT kernel, one CTA per (batch row, head)"}
        del Q, K, V
        # The bias (d = 63, padded to 64) and the per-token rate (d = 64) on the tensor-core
        # kernels, long-context shape: prep pass + ttt_linear_fwd's plan + copy-out.
        for name in ("bias", "token_eta"):
            d = 63 if name == "bias" else 64
            w = synth.WORKLOADS["linear_long"].with_(d=d)
            inp, Q, K, V, eta = dev_inputs(w)
            W0 = torch.from_numpy(inp.W0).to(dev)
            code = ttt.TTT_INNER_BIAS if name == "bias" else ttt.TTT_INNER_TOKEN_ETA
            vws = torch.empty(ttt.ttt_linear_variant_workspace_bytes(code, ttt.TTT_BF16, w.B, w.H, w.T, d, 16),
                              dtype=torch.uint8, device=dev)
            if name == "bias":
                vec = torch.zeros((w.H, d), dtype=torch.float32, device=dev)
                fn = lambda: ttt.ttt_linear_bias_fwd(Q, K, V, eta, W0, vec, 16, stream=stream, fast=True, workspace=vws)
            else:
                et = torch.full((w.B, w.H, w.T), 0.1, dtype=torch.float32, device=dev)
                fn = lambda: ttt.ttt_linear_token_eta_fwd(Q, K, V, et, W0, 16, stream=stream, fast=True,
                                                          workspace=vws)
            ms = t_ms(fn, 5)
            if ttt.ttt_last_device_status(vws, stream) != 0:
                raise RuntimeError(f"variant {name}: device status not OK")
            out[f"variant_{name}_fast_long_b16"] = {
                "ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                "hbm_frac": round(algorithmic_bytes(w) / (ms * 1e-3) / 1e9 / hbm_gbs, 4),
                "note": f"B1 H32 T131072 d{d} bf16: changed inputs (padded to 64 features) through the "
                        "tensor-core segment-parallel path; bytes counted at d"}
            del Q, K, V, vws
        # Momentum and LN + residual on their tensor-core kernels (bf16, d = 64, b = 16, one CTA per unit).
        for wname, tag in (("linear_small", "small"), ("linear_125m", "125m")):
            w = synth.WORKLOADS[wname]
            inp, Q, K, V, eta = dev_inputs(w)
            W0 = torch.from_numpy(inp.W0).to(dev)
            mbeta = torch.full((w.H,), 0.9, dtype=torch.float32, device=dev)
            malpha = torch.full((w.H,), 0.05, dtype=torch.float32, device=dev)  # a stable momentum step
            gam, lnb = torch.ones((w.H, w.d), device=dev), torch.zeros((w.H, w.d), device=dev)
            mws = torch.zeros(256, dtype=torch.uint8, device=dev)
            fns = {"momentum": (lambda: ttt.ttt_linear_momentum_fwd(Q, K, V, malpha, mbeta, W0, 16, stream=stream,
                                                                    fast=True, workspace=mws,
                                                                    options={"force_path": ttt.PATH_TENSOR}),
                                "alpha 0.05, beta 0.9: tensor-core momentum kernel"),
                   "ln_residual": (lambda: ttt.ttt_linear_ln_fwd(Q, K, V, malpha, W0, gam, lnb, 16, stream=stream,
                                                                 fast=True, workspace=mws,
                                                                 options={"force_path": ttt.PATH_TENSOR}),
                                   "eta 0.05: tensor-core LN + residual kernel")}
            for vname, (fn, what) in fns.items():
                ms = t_ms(fn, 5)
                if ttt.ttt_last_device_status(mws, stream) != 0:
                    raise RuntimeError(f"{vname}: device status not OK")
                out[f"variant_{vname}_fast_{tag}_b16"] = {
                    "ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                    "hbm_frac": round(algorithmic_bytes(w) / (ms * 1e-3) / 1e9 / hbm_gbs, 4),
                    "note": f"B{w.B} H{w.H} T{w.T} d64 bf16, {what}, one CTA per (batch row, head)"}
            del Q, K, V
    except Exception as exc:  # reported in the line, never silently dropped
        out["variants"] = {"error": f"{type(exc).__name__}: {exc}"}
    # backward of TTT-Linear on the tensor cores (bf16, b = 16), 125M-shaped: B8 H12 T8192
    try:
        w = synth.WORKLOADS["linear_125m"]
        inp, Q, K, V, eta = dev_inputs(w)
        W0 = torch.from_numpy(inp.W0).to(dev)
        dZ = torch.randn_like(Q, dtype=torch.float32).to(torch.bfloat16)
        dW = torch.randn(w.B, w.H, w.d, w.d, device=dev)
        ws = torch.empty(ttt.ttt_linear_bwd_workspace_bytes(w.B, w.H, w.T, w.d, 16), dtype=torch.uint8, device=dev)
        ms = t_ms(lambda: ttt.ttt_linear_bwd(Q, K, V, eta, W0, 16, dZ, dW, workspace=ws, stream=stream), 5)
        # algorithmic bytes: Q, K, V, dZ read and dQ, dK, dV written once (bf16), states aside
        bwd_bytes = w.token_heads * 7 * w.d * 2
        out["linear_bwd_125m_bf16_b16"] = {"ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                                           "hbm_frac": round(bwd_bytes / (ms * 1e-3) / 1e9 / hbm_gbs, 4),
                                           "note": "B8 H12 T8192 d64 bf16; tensor-core backward, one CTA per "
                                                   "(batch row, head), W kept every 64 tokens"}
        del Q, K, V, dZ
    except Exception as exc:  # reported in the line, never silently dropped
        out["linear_bwd_125m_bf16_b16"] = {"error": f"{type(exc).__name__}: {exc}"}
    # backward of TTT-Linear, fp32 operands (the SIMT kernel: one CTA per unit)
    try:
        w = synth.WORKLOADS["linear_small"].with_(dtype="f32")
        inp = synth.make_inputs(w, want_exact=False)
        Q, K, V = (torch.from_numpy(a).to(dev) for a in (inp.q, inp.k, inp.v))
        eta, W0 = torch.from_numpy(inp.eta).to(dev), torch.from_numpy(inp.W0).to(dev)
        dZ = torch.randn_like(Q)
        dW = torch.randn(w.B, w.H, w.d, w.d, device=dev)
        ws = torch.empty(ttt.ttt_linear_bwd_workspace_bytes(w.B, w.H, w.T, w.d, 16), dtype=torch.uint8, device=dev)
        ms = t_ms(lambda: ttt.ttt_linear_bwd(Q, K, V, eta, W0, 16, dZ, dW, workspace=ws, stream=stream), 3)
        # algorithmic bytes: Q, K, V, dZ read and dQ, dK, dV written once (fp32), states aside
        bwd_bytes = w.token_heads * 7 * w.d * 4
        out["linear_bwd_small_f32_b16"] = {"ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                                           "hbm_frac": round(bwd_bytes / (ms * 1e-3) / 1e9 / hbm_gbs, 5),
                                           "note": "B2 H4 T2048 d64 fp32; dQ, dK, dV, d eta, dW0 for given dZ, "
                                                   "dW_out; one CTA per (batch row, head)"}
        del Q, K, V, dZ
    except Exception as exc:  # reported in the line, never silently dropped
        out["linear_bwd_small_f32_b16"] = {"error": f"{type(exc).__name__}: {exc}"}
    # backward of TTT-Linear with few units: the segment-parallel form (B2 H4 T8192, B1 H32 T131072)
    for tag, w in (("linear_bwd_seg_small_bf16_b16", synth.WORKLOADS["linear_small"].with_(T=8192)),
                   ("linear_bwd_seg_long_bf16_b16", synth.WORKLOADS["linear_long"])):
        try:
            inp, Q, K, V, eta = dev_inputs(w)
            W0 = torch.from_numpy(inp.W0).to(dev)
            dZ = torch.randn_like(Q, dtype=torch.float32).to(torch.bfloat16)
            dW = torch.randn(w.B, w.H, w.d, w.d, device=dev)
            ws = torch.empty(ttt.ttt_linear_bwd_workspace_bytes(w.B, w.H, w.T, w.d, 16), dtype=torch.uint8,
                             device=dev)
            ms = t_ms(lambda: ttt.ttt_linear_bwd(Q, K, V, eta, W0, 16, dZ, dW, workspace=ws, stream=stream), 3)
            if ttt.ttt_last_device_status(ws, stream) != 0:
                raise RuntimeError("device status not OK")
            bwd_bytes = w.token_heads * 7 * w.d * 2
            out[tag] = {"ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                        "hbm_frac": round(bwd_bytes / (ms * 1e-3) / 1e9 / hbm_gbs, 4),
                        "note": f"B{w.B} H{w.H} T{w.T} d64 bf16: segments of whole 64-token blocks, one "
                                "tensor-core backward CTA each"}
            del Q, K, V, dZ, ws
        except Exception as exc:  # reported in the line, never silently dropped
            out[tag] = {"error": f"{type(exc).__name__}: {exc}"}
    # backward of TTT-MLP (fp32 parity kernel), B2 H4 T512 d64 hidden 256
    try:
        w = synth.WORKLOADS["mlp_125m"].with_(B=2, H=4, T=512, dtype="f32")
        inp = synth.make_inputs(w, want_exact=False)
        Q, K, V = (torch.from_numpy(a).to(dev) for a in (inp.q, inp.k, inp.v))
        eta, W1, W2 = (torch.from_numpy(a).to(dev) for a in (inp.eta, inp.W1, inp.W2))
        dZ = torch.randn_like(Q)
        dW1 = torch.randn(w.B, w.H, w.d, 4 * w.d, device=dev)
        dW2 = torch.randn(w.B, w.H, 4 * w.d, w.d, device=dev)
        ws = torch.empty(ttt.ttt_mlp_bwd_workspace_bytes(w.B, w.H, w.T, w.d, 16), dtype=torch.uint8, device=dev)
        ms = t_ms(lambda: ttt.ttt_mlp_bwd(Q, K, V, eta, W1, W2, 16, dZ, dW1, dW2, workspace=ws, stream=stream), 2)
        out["mlp_bwd_small_f32_b16"] = {"ms": round(ms, 3), "token_heads_per_s": w.token_heads / (ms * 1e-3),
                                        "note": "B2 H4 T512 d64 hidden 256 fp32; dQ, dK, dV, d eta, dW1, dW2; "
                                                "fp32 parity kernel, one CTA per (batch row, head)"}
        del Q, K, V, dZ
    except Exception as exc:  # reported in the line, never silently dropped
        out["mlp_bwd_small_f32_b16"] = {"error": f"{type(exc).__name__}: {exc}"}
    # decode: one token for B1 H32 from a state
    try:
        q = torch.randn(1, 32, 64, device=dev).to(torch.bfloat16)
        Wa = torch.zeros(1, 32, 64, 64, device=dev)
        Wr = torch.zeros(1, 32, 64, 64, device=dev)
        e32 = torch.full((32,), 0.1, device=dev)
        ms = t_ms(lambda: ttt.ttt_linear_decode_step(q, q, q, e32, Wa, Wr, 5, 16, stream=stream), 200,
                  ahead=False)
        # The same 100 tokens replayed from a CUDA graph: the GPU-side cost per token
        # without the Python call overhead of the loop above.
        z = torch.empty_like(q)
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                ttt.ttt_linear_decode_step(q, q, q, e32, Wa, Wr, 5, 16, z=z, stream=side)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for i in range(100):
                ttt.ttt_linear_decode_step(q, q, q, e32, Wa, Wr, 5 + i, 16, z=z, stream=side)
        gms = t_ms(graph.replay, 10) / 100
        per_launch = {}
        for n in (16, 128):  # n tokens per launch (ttt_linear_decode), state kept in registers between them
            qn = torch.randn(1, 32, n, 64, device=dev).to(torch.bfloat16)
            zn = torch.empty_like(qn)
            per_launch[str(n)] = round(t_ms(lambda: ttt.ttt_linear_decode(qn, qn, qn, e32, Wa, Wr, 5, 16, z=zn,
                                                                          stream=stream), 20) * 1e3 / n, 3)
        out["decode_long_1tok"] = {"us_per_step": round(ms * 1e3, 2),
                                   "us_per_step_cuda_graph": round(gms * 1e3, 2),
                                   "us_per_token_n_per_launch": per_launch,
                                   "note": "B1 H32 d64 bf16: one token per call through the Python binding, "
                                           "100 one-token calls replayed from a CUDA graph, and n tokens per "
                                           "ttt_linear_decode launch (us per token); floor ~0.25 us (state bytes)"}
    except Exception as exc:  # reported in the line, never silently dropped
        out["decode_long_1tok"] = {"error": f"{type(exc).__name__}: {exc}"}
    return out


# --------------------------------------------------------------------------- reference arm
def bench_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    w = synth.WORKLOADS[args.workload].with_(b=args.b)
    # bounded sample per step: batch row 0, all heads, the first Ts tokens, sized so that the
    # whole run stays within a few minutes
    steps = args.steps
    warm = max(3, args.warmup)
    budget_s = REFERENCE_BUDGET_S
    threads = oracle.max_threads()
    probe = synth.make_inputs(w.with_(B=1, T=256))
    t0 = time.perf_counter()
    oracle.linear_primal(probe.q64, probe.k64, probe.v64, probe.eta64, probe.W0_64, args.b)
    per_tok = (time.perf_counter() - t0) / 256
    Ts = int(max(args.b, min(w.T, budget_s / (steps + warm) / max(per_tok, 1e-9))))
    Ts = max(args.b, Ts // args.b * args.b)
    inp = synth.make_inputs(w.with_(B=1, T=Ts))
    run = lambda: oracle.linear_primal(inp.q64, inp.k64, inp.v64, inp.eta64, inp.W0_64, args.b)
    for _ in range(warm):
        run()
    t0 = time.perf_counter()
    for _ in range(steps):
        run()
    dt = (time.perf_counter() - t0) / steps
    value = w.H * Ts / dt
    sample = f"{w.name}: batch row 0, all {w.H} heads, first {Ts} of {w.T} tokens per step (fp64 primal oracle)"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "b": args.b,
                       "inputs": f"Q/K/V {w.dtype} (exact fp64 values) {w.note}"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_mlp(args, world, rank, local):
    """A TTT-MLP workload through ttt_mlp_fwd (secondary; used for profiling the
    tensor-core TTT-MLP kernel). Reports against the bf16 tensor roofline."""
    import torch
    import test_sequence_layers_06_b300 as ttt
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload].with_(b=args.b)
    if args.T:
        w = w.with_(T=args.T)
    inp = synth.make_inputs(w, want_exact=False)
    cv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev))
    Q, K, V = cv(inp.q), cv(inp.k), cv(inp.v)
    eta = torch.from_numpy(inp.eta).to(dev)
    W1, W2 = torch.from_numpy(inp.W1).to(dev), torch.from_numpy(inp.W2).to(dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: ttt.ttt_mlp_fwd(Q, K, V, eta, W1, W2, args.b, stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / args.steps
    _, tflops, kind = measured_peaks()
    flops = w.token_heads * (16 * w.d * w.hidden + 4 * args.b * (w.d + w.hidden))
    achieved = flops / (ms * 1e-3) / 1e12
    if rank == 0:
        print(json.dumps({"metric": "TTT-MLP scan tokens·heads/sec", "value": w.token_heads / (ms * 1e-3),
                          "unit": UNIT, "n_gpus": world, "steps": args.steps, "ms_per_step": round(ms, 4),
                          "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                          "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "hidden": w.hidden,
                                     "b": args.b},
                          "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": tflops,
                                       "unit": "TFLOP/s", "frac": round(achieved / tflops, 5),
                                       "peak_kind": f"{kind} bf16 burst"}}), flush=True)


def bench_decode(args, world, rank, local):
    """Decode after a prefill: N = --T tokens (default 1) per ttt_linear_decode launch for every (batch
    row, head) of the workload, from a state (secondary; used for profiling the decode kernel)."""
    import torch
    import test_sequence_layers_06_b300 as ttt
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    n = args.T or 1
    g = torch.Generator(device=dev).manual_seed(5)
    q = torch.randn(w.B, w.H, n, w.d, device=dev, generator=g).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn(w.B, w.H, n, w.d, device=dev, generator=g), dim=-1).to(torch.bfloat16)
    v = torch.randn(w.B, w.H, n, w.d, device=dev, generator=g).to(torch.bfloat16)
    eta = torch.full((w.H,), 0.1, device=dev)
    Wa = 0.02 * torch.randn(w.B, w.H, w.d, w.d, device=dev, generator=g)
    Wr = Wa.clone()
    z = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    step = lambda: ttt.ttt_linear_decode(q, k, v, eta, Wa, Wr, 5, args.b, z=z, stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(4e6) * (args.steps + 1))  # hold the stream while the launches are enqueued
    a.record(stream)
    for _ in range(args.steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / args.steps
    if rank == 0:
        print(json.dumps({"metric": "TTT-Linear decode tokens·heads/sec", "value": w.units * n / (ms * 1e-3),
                          "unit": UNIT, "n_gpus": world, "steps": args.steps, "us_per_launch": round(ms * 1e3, 3),
                          "us_per_token": round(ms * 1e3 / n, 3), "higher_is_better": True, "dtype": "bf16",
                          "data": "synthetic", "config": {"workload": w.name, "B": w.B, "H": w.H, "d": w.d,
                                                          "b": args.b, "tokens_per_launch": n}}), flush=True)


def bench_variant(args, world, rank, local):
    """The momentum or LN + residual variant through its *_ex call on the workload's shape (secondary;
    used for profiling those tensor-core kernels). Reports against the HBM roofline of the plain
    read-out's bytes."""
    import torch
    import test_sequence_layers_06_b300 as ttt
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload].with_(b=16)
    if args.T:
        w = w.with_(T=args.T)
    inp = synth.make_inputs(w, want_exact=False)
    cv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev))
    Q, K, V = cv(inp.q), cv(inp.k), cv(inp.v)
    W0 = torch.from_numpy(inp.W0).to(dev)
    rate = torch.full((w.H,), 0.05, dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    opts = {"force_path": ttt.PATH_TENSOR}
    if args.mode == "momentum":
        mbeta = torch.full((w.H,), 0.9, dtype=torch.float32, device=dev)
        step = lambda: ttt.ttt_linear_momentum_fwd(Q, K, V, rate, mbeta, W0, 16, stream=stream, fast=True,
                                                   workspace=ws, options=opts)
    else:
        gam, lnb = torch.ones((w.H, w.d), device=dev), torch.zeros((w.H, w.d), device=dev)
        step = lambda: ttt.ttt_linear_ln_fwd(Q, K, V, rate, W0, gam, lnb, 16, stream=stream, fast=True,
                                             workspace=ws, options=opts)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    if ttt.ttt_last_device_status(ws, stream) != 0:
        raise RuntimeError("device status not OK")
    ms = a.elapsed_time(e) / args.steps
    hbm_gbs, _, kind = measured_peaks()
    gbs = algorithmic_bytes(w) / (ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({"metric": f"TTT-Linear {args.mode} variant tokens·heads/sec", "value": w.token_heads / (ms * 1e-3),
                          "unit": UNIT, "n_gpus": world, "steps": args.steps, "ms_per_step": round(ms, 4),
                          "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                          "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "b": 16,
                                     "variant": args.mode},
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                                       "frac": round(gbs / hbm_gbs, 4), "peak_kind": kind}}), flush=True)


def bench_bwd(args, world, rank, local):
    """The TTT-Linear backward through ttt_linear_bwd on a workload (secondary; used for the
    backward's profiles). Reports against the HBM roofline of its algorithmic bytes: Q, K, V, dZ
    read and dQ, dK, dV written once."""
    import torch
    import test_sequence_layers_06_b300 as ttt
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload].with_(b=args.b)
    if args.T:
        w = w.with_(T=args.T)
    inp = synth.make_inputs(w, want_exact=False)
    cv = (lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev))
    Q, K, V = cv(inp.q), cv(inp.k), cv(inp.v)
    eta, W0 = torch.from_numpy(inp.eta).to(dev), torch.from_numpy(inp.W0).to(dev)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    dZ = torch.randn(Q.shape, device=dev, generator=g).to(torch.bfloat16)
    dW = torch.randn((w.B, w.H, w.d, w.d), device=dev, generator=g)
    ws = torch.empty(ttt.ttt_linear_bwd_workspace_bytes(w.B, w.H, w.T, w.d, args.b), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = lambda: ttt.ttt_linear_bwd(Q, K, V, eta, W0, args.b, dZ, dW, workspace=ws, stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    if ttt.ttt_last_device_status(ws, stream) != 0:
        raise RuntimeError("device status not OK after the timed region")
    ms = a.elapsed_time(e) / args.steps
    hbm_gbs, _, kind = measured_peaks()
    nbytes = w.token_heads * 7 * w.d * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({"metric": "TTT-Linear backward tokens·heads/sec", "value": w.token_heads / (ms * 1e-3),
                          "unit": UNIT, "n_gpus": world, "steps": args.steps, "ms_per_step": round(ms, 4),
                          "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
                          "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "b": args.b},
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                                       "frac": round(gbs / hbm_gbs, 4), "algorithmic_bytes": nbytes,
                                       "peak_kind": kind}}), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.impl == "reference":
        bench_reference(args, world, rank)
    elif args.mode == "bwd":
        bench_bwd(args, world, rank, local)
    elif args.mode in ("momentum", "ln"):
        bench_variant(args, world, rank, local)
    elif args.mode == "decode":
        bench_decode(args, world, rank, local)
    elif synth.WORKLOADS[args.workload].variant == "mlp":
        bench_mlp(args, world, rank, local)
    else:
        bench_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
