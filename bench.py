"""Benchmark of the exact attention forward on GB300.

Default workload: the sequence-length sweep point N = 8192, d = 128 (bf16,
B = 16384 / N = 2, H = 2048 / d = 16, non-causal; the causal run of the same
shapes is reported beside it).  A step is one launch of the fused attention
kernel over that batch, through attn_fwd_ws (its workspace gives full attention
the stream-K tail; the arrival counters are zeroed by one memset per launch).  Metric: attention forward TFLOP/s with
FLOPs = 4 B H N^2 d (halved when causal), and its fraction of the measured
dense BF16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the float64 CPU oracle, host cores

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(weak scaling: the path has no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "attention fwd TFLOP/s and % of GB300 dense BF16/FP8 tensor peak vs seq len"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL_SOURCES = [os.path.join(ROOT, "exact_attention_forward_05_gb300", "csrc", f)
                  for f in ("attn_kernel.cuh", "sm103.cuh", "attn_fwd.cu", "host_common.h", "host_common.cu")]
PROFILE_JSON = os.path.join(ROOT, "profiles", "attn_fwd_bf16_b2_h16_n8192_d128.json")

WORKLOADS = {}
for _n in (512, 1024, 2048, 4096, 8192, 16384):
    for _d in (64, 128, 256):
        for _c in (False, True):
            WORKLOADS[f"sweep_n{_n}_d{_d}{'_causal' if _c else ''}"] = dict(
                B=16384 // _n, H=2048 // _d, N=_n, d=_d, causal=_c, dtype="bf16")
WORKLOADS["b4_h16_n2048_d128"] = dict(B=4, H=16, N=2048, d=128, causal=False, dtype="bf16")
WORKLOADS["b4_h16_n2048_d128_causal"] = dict(B=4, H=16, N=2048, d=128, causal=True, dtype="bf16")
WORKLOADS["long_b1_h16_n32768_d128_causal"] = dict(B=1, H=16, N=32768, d=128, causal=True, dtype="bf16")
DEFAULT_WORKLOAD = "sweep_n8192_d128"


def flops(w) -> float:
    f = 4.0 * w["B"] * w["H"] * w["N"] ** 2 * w["d"]
    return f / 2 if w["causal"] else f


def describe(w) -> str:
    return (f"{w['dtype']} attention fwd, B={w['B']}, H={w['H']}, N={w['N']}, d={w['d']}, "
            f"{'causal' if w['causal'] else 'non-causal'}")


# NVIDIA's dense (no 2:4 sparsity) per-GPU tensor figures for GB300, for
# context beside the measured denominators.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_FP8_TFLOPS = 4500.0


def peaks(sustained: bool = False):
    """The bf16 denominator: the measured cuBLAS bf16 GEMM rate (burst,
    or the seconds-long sustained loop), i.e. what cuBLAS achieves on this
    GB300 -- below the datasheet figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        if sustained and "bf16_tflops_sustained" in p:
            return float(p["bf16_tflops_sustained"]), \
                "measured cuBLAS bf16 GEMM, sustained (MEASURED_PEAKS.json bf16_tflops_sustained; cuBLAS-achievable, not the datasheet peak)"
        return float(p["bf16_tflops"]), \
            "measured cuBLAS bf16 GEMM, burst (MEASURED_PEAKS.json bf16_tflops; cuBLAS-achievable, not the datasheet peak)"
    return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, one earlier GB300 measurement)"


def hbm_peak() -> float:
    """Measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"])
    return 6800.0


def roofline(achieved, fp8=False, sustained=False, **extra):
    """Roofline object: `peak` is the measured denominator (FP8: twice the
    measured bf16 rate, the nominal FP8/BF16 ratio of the tensor cores);
    `frac_nominal` is the same rate against NVIDIA's dense datasheet figure."""
    peak, src = peaks(sustained)
    if fp8:
        peak, src = 2.0 * peak, "2 x " + src + " (nominal FP8 / BF16 dense ratio)"
    nominal = NOMINAL_FP8_TFLOPS if fp8 else NOMINAL_BF16_TFLOPS
    return dict({"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": UNIT,
                 "frac": round(achieved / peak, 4), "peak_source": src, "peak_nominal": nominal,
                 "frac_nominal": round(achieved / nominal, 4),
                 "peak_nominal_source": "NVIDIA GB300 dense tensor figure (no sparsity)"}, **extra)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------------ clocks

REASON_BITS = {  # NVML clocks-event reason bits
    "sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
    "hw_power_brake_slowdown": 0x80}


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, power,
    clocks-event reasons).  Nothing here changes a GPU setting."""

    def __init__(self, device_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        ident = (uuid if uuid.startswith("GPU-") else f"GPU-{uuid}").encode()
        if self.lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(ident), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_sm = self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn):
        v = self.ct.c_uint()
        return float(v.value) if fn(self.h, 1, self.ct.byref(v)) == 0 else None  # 1 = SM clock

    def sample(self):
        """(sm_mhz, sm_max_mhz, power_w, reasons bitmask)"""
        p, r = self.ct.c_uint(), self.ct.c_ulonglong()
        pw = p.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, self.ct.byref(p)) == 0 else None
        rs = r.value if self.reasons_fn(self.h, self.ct.byref(r)) == 0 else 0
        return self._clock(self.lib.nvmlDeviceGetClockInfo), self.max_sm, pw, rs


class ClockSampler:
    """Clock samples with host timestamps, taken every 2 ms through NVML
    (every 100 ms through nvidia-smi when NVML cannot be loaded)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples = []  # (time, sm_mhz, sm_max_mhz, power_w, {reason names})
        self.proc = None
        self.source = None
        self._stop = threading.Event()
        try:
            nv = _Nvml(device_index)
            nv.sample()
            self.source = "nvml 2 ms"
            self.thread = threading.Thread(target=self._poll, args=(nv, period_s), daemon=True)
            self.thread.start()
            return
        except Exception:
            pass
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.source = "nvidia-smi 100 ms"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self, nv, period_s):
        while not self._stop.is_set():
            try:
                sm, mx, pw, bits = nv.sample()
            except Exception:
                return
            if sm is not None:
                self.samples.append((time.time(), sm, mx, pw,
                                     {n for n, b in REASON_BITS.items() if bits & b}))
            time.sleep(period_s)

    def _read(self):
        for line in self.proc.stdout:
            self.add_smi_line(time.time(), line)

    def add_smi_line(self, ts, line):
        f = [x.strip() for x in line.split(",")]
        if len(f) < 7:
            return
        try:
            sm, mx = float(f[0]), float(f[1])
        except ValueError:
            return
        try:
            pw = float(f[2])
        except ValueError:
            pw = None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = {n for n, val in zip(names, f[3:7]) if val.lower().startswith("active")}
        self.samples.append((ts, sm, mx, pw, reasons))

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sm, mx, pw, reasons = [], [], [], set()
        for ts, s_mhz, m_mhz, p_w, rs in list(self.samples):
            if not (t0 <= ts <= t1):
                continue
            sm.append(s_mhz)
            if m_mhz is not None:
                mx.append(m_mhz)
            if p_w is not None:
                pw.append(p_w)
            reasons |= rs
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "sm_min_mhz": min(sm), "power_w_max": max(pw) if pw else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": self.source}


# --------------------------------------------------------------- GPU arm

def time_kernel(fn, steps: int, warmup: int, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for _ in range(steps):
        fn()
    ev[1].record(stream)
    torch.cuda.synchronize()
    return ev[0].elapsed_time(ev[1])  # ms


def time_for(fn, seconds: float, stream, sampler=None, min_steps: int = 3):
    """Back-to-back launches for at least `seconds` of device time, in
    batches timed with CUDA events on `stream`; returns (ms per launch,
    launches, clocks of the window)."""
    ms = time_kernel(fn, 3, 0, stream) / 3  # estimate
    n = max(min_steps, int(seconds * 1e3 / max(ms, 1e-3)))
    t0 = time.time()
    total = time_kernel(fn, n, 0, stream)
    t1 = time.time()
    clocks = sampler.summary(t0, t1) if sampler else None
    return total / n, n, clocks


def barrier(world):
    """All ranks meet (process group barrier), then this rank's GPU work drains."""
    if world > 1:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x: float, world: int) -> float:
    """The largest value of x over all ranks (the elapsed time of the slowest
    rank); the reduction runs on the process group's own device (CUDA for
    NCCL, host memory for gloo)."""
    if world == 1:
        return x
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def kernel_source_sha256() -> str:
    """Hash of the sources the bf16 attention kernel is built from."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def traffic_from_profile():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source."""
    if not os.path.exists(PROFILE_JSON):
        return None
    with open(PROFILE_JSON) as f:
        prof = json.load(f)
    sha = kernel_source_sha256()
    if prof.get("kernel_source_sha256") != sha:
        return None
    return prof.get("dram_bytes_per_launch_full_workload")


def cpu_baseline(w, q, k, v, budget_s: float = 12.0):
    """The oracle as it stands, on every host core, on a bounded sample of the
    workload: whole heads (all their query rows) when one head fits the time
    budget, else seeded query rows of one head; throughput in TFLOP/s."""
    import oracle
    import synth
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    qf, kf, vf = (t.reshape(1, B * H, N, d) for t in (q, k, v))
    scale = d ** -0.5
    probe = synth.sample_rows(N, 64, seed=1, salt=99)
    t0 = time.time()
    oracle.attention(qf[:, :1], kf[:, :1], vf[:, :1], causal=w["causal"], scale=scale, rows=probe)
    t_head = max(time.time() - t0, 1e-4) * N / len(probe)
    if t_head <= budget_s:
        nh = int(min(B * H, max(1, budget_s // t_head)))
        rows = None
        keys = nh * (N * (N + 1) // 2 if w["causal"] else N * N)
        what = f"{nh} of {B * H} heads, all {N} query rows each"
    else:
        nh = 1
        rows = synth.sample_rows(N, int(max(16, N * budget_s / t_head)), seed=2, salt=98)
        keys = int((rows + 1).sum()) if w["causal"] else len(rows) * N
        what = f"{len(rows)} seeded query rows of head 0"
    t0 = time.time()
    _, _, used = oracle.attention(qf[:, :nh], kf[:, :nh], vf[:, :nh], causal=w["causal"],
                                  scale=scale, rows=rows, return_threads=True)
    dt = time.time() - t0
    fl = 4.0 * float(keys) * d
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{what} (float64 C oracle, {dt:.1f} s)", "seconds": dt}


def run_gpu(args):
    rank, world, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_forward_05_gb300 as attn
    import synth

    w = WORKLOADS[args.workload]
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    q, k, v = synth.attention_inputs(B, H, N, d, w["dtype"], seed=rank)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = d ** -0.5
    launches = [0]
    # With a workspace, full attention takes the stream-K tail (attn_fwd_ws:
    # the units that do not fill a last round are cut into equal key ranges);
    # causal launches ignore it.
    fws = torch.empty(attn.workspace_bytes(d, dev), dtype=torch.uint8, device=dev) if d <= 128 else None
    def step(causal=w["causal"]):
        attn.attn_fwd(qd, kd, vd, causal=causal, scale=scale, out=o, lse=lse, stream=stream, workspace=fws)
        launches[0] += 1

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(1.0 if sampler else 0.0)
    barrier(world)
    # warm-up, then exactly `steps` timed launches between barriers
    for _ in range(args.warmup):
        step()
    barrier(world)
    launches[0] = 0
    t_wall0 = time.time()
    ms = time_kernel(step, args.steps, 0, stream)
    t_wall1 = time.time()
    barrier(world)
    n_launch = launches[0]
    ms_max = max_over_ranks(ms, world)
    status = attn.device_status()
    if status != attn.ATTN_OK:
        raise RuntimeError(f"device status {attn.status_string(status)}")
    per_step = ms_max / args.steps
    value = flops(w) * world / (per_step * 1e-3) / 1e12

    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None

    # The same launch back to back for at least 1.5 s: its clocks (power cap
    # included) and its rate against the sustained cuBLAS denominator.
    ms_sus, n_sus, clocks_sus = time_for(step, 1.5, stream, sampler)
    ms_sus = max_over_ranks(ms_sus, world)
    sus_value = flops(w) / (ms_sus * 1e-3) / 1e12

    # the other mask setting of the same shapes, for context
    other = dict(w, causal=not w["causal"])
    ms_o, _, clocks_o = time_for(lambda: step(other["causal"]), 0.3, stream, sampler)
    ms_o = max_over_ranks(ms_o, world)
    other_value = flops(other) * world / (ms_o * 1e-3) / 1e12
    step()  # leave o / lse for the configured mask
    torch.cuda.synchronize()
    status = attn.device_status()
    if status != attn.ATTN_OK:
        raise RuntimeError(f"device status {attn.status_string(status)}")

    # end to end: host buffers (pinned) through the C ABI, copies in the timed region
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    op = torch.empty_like(qp).pin_memory()
    lp = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    hws = torch.empty(attn.host_workspace_bytes(B, H, N, d, qd.dtype), dtype=torch.uint8, device=dev)
    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        attn.attn_fwd_host(qp, kp, vp, causal=w["causal"], scale=scale, workspace=hws, out=op,
                           lse=lp, device=dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        attn.attn_fwd_host(qp, kp, vp, causal=w["causal"], scale=scale, workspace=hws, out=op,
                           lse=lp, device=dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world) / e2e_steps
    e2e_value = flops(w) * world / e2e_s / 1e12

    fp8 = fp8_leg(w, dev, stream, rank, args, sampler) if w["d"] == 128 else None
    host = host_cost(dev, stream) if rank == 0 else None
    if sampler:
        sampler.stop()

    achieved = flops(w) / (ms / args.steps * 1e-3) / 1e12
    line = None
    if rank == 0:
        cpu = cpu_baseline(w, q, k, v)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w["dtype"], "data": "synthetic (seeded iid N(0,1), splitmix64 + Box-Muller)",
            "config": {"workload": describe(w), "B": B, "H": H, "N": N, "d": d,
                       "causal": w["causal"], "scale": scale,
                       "flops_per_step_per_gpu": flops(w),
                       "schedule": ("persistent round-robin rounds plus a stream-K tail (attn_fwd_ws workspace; "
                                    "its arrival counters are zeroed by one cudaMemsetAsync before each launch)")
                                   if not w["causal"] else "persistent, longest-first causal units",
                       "l2": "inputs larger than L2 (Q, K, V, O = 4 x %.0f MiB)" % (B * H * N * d * 2 / 2 ** 20),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roofline(achieved, traffic=traffic_from_profile(), kernel="attn_fwd_kernel<128, bf16>"),
            "cpu_baseline": {k2: (round(v2, 6) if isinstance(v2, float) else v2)
                             for k2, v2 in cpu.items() if k2 != "seconds"},
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                    "h2d_bytes_per_step": 3 * q.numel() * q.element_size(),
                    "d2h_bytes_per_step": o.numel() * o.element_size() + lse.numel() * 4,
                    "path": "attn_fwd_host (pinned host buffers)"},
            "gpu_launches": n_launch,
            "clocks": clocks,
            "sustained": {"value": round(sus_value, 2), "unit": UNIT, "launches": n_sus,
                          "seconds": round(ms_sus * n_sus / 1e3, 2),
                          "roofline": roofline(sus_value, sustained=True), "clocks": clocks_sus},
            "other_mask": {"causal": other["causal"], "value": round(other_value, 2), "unit": UNIT,
                           "clocks": clocks_o},
            "fp8": fp8,
            "host": host,
            "device": torch.cuda.get_device_name(dev),
        }
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return line


def host_cost(dev, stream, calls: int = 500):
    """Host time per attn_fwd call in the library (C ABI called directly
    through ctypes, arguments marshalled once; the GPU is left to drain the
    launches after the loop) on the smallest sweep point, bf16 B=32, H=16,
    N=512, d=128, beside that launch's device time."""
    import ctypes
    import exact_attention_forward_05_gb300 as attn
    B, H, N, d = 32, 16, 512, 128
    q = torch.randn(B, H, N, d, device=dev, dtype=torch.bfloat16)
    k, v, o = torch.randn_like(q), torch.randn_like(q), torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev, dtype=torch.float32)
    lib = attn.lib()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, 0,
            ctypes.c_float(d ** -0.5), attn.ATTN_BF16, ctypes.c_void_p(stream.cuda_stream))
    for _ in range(10):
        lib.attn_fwd(*args)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        lib.attn_fwd(*args)
    host_us = (time.perf_counter() - t0) / calls * 1e6
    torch.cuda.synchronize()
    dev_us = time_kernel(lambda: lib.attn_fwd(*args), 200, 0, stream) / 200 * 1e3
    return {"workload": "bf16 attention fwd, B=32, H=16, N=512, d=128, non-causal",
            "host_us_per_call": round(host_us, 2), "device_us_per_launch": round(dev_us, 2),
            "note": "host time of the C entry point per call (argument checks, cached tensor maps, launch)"}


def fp8_leg(w, dev, stream, rank, args, sampler=None):
    """The FP8 path on the same shapes with 0.1 % outliers in Q, K, V: the FP8
    attention kernel alone (against the FP8 dense peak = 2 x the measured bf16
    peak, the nominal FP8/BF16 ratio of the tensor cores), the pre-pass
    (Hadamard rotation + block quantisation, HBM-bound), the pre-pass with the
    rotary embedding of Q and K fused in front, and pre-pass + kernel together;
    plus the RMS error against exact attention on sampled rows next to the
    naive per-tensor FP8 baseline.  The kernel is timed over the same number
    of back-to-back launches as the main line (a burst, like the bf16 figure)
    and again for 1.5 s (sustained); every timing carries its clock record."""
    import exact_attention_forward_05_gb300 as attn
    import synth
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=rank)
    signs = synth.hadamard_signs(H, d, seed=rank).to(dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    nblk = (N + 127) // 128
    bufs = [torch.empty((B, H, N, d), dtype=torch.uint8, device=dev) for _ in range(3)] + \
           [torch.empty((B, H, nblk), dtype=torch.float32, device=dev) for _ in range(3)]
    o8 = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    l8 = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    scale = d ** -0.5
    prep = lambda: attn.fp8_prepare(qd, kd, vd, signs=signs, out=bufs, stream=stream)
    rope = tuple(t.to(dev) for t in synth.rotary_tables(N, d))
    prep_rope = lambda: attn.fp8_prepare(qd, kd, vd, signs=signs, out=bufs, stream=stream, rope=rope)
    ws = torch.empty(max(attn.workspace_bytes(d, dev), 1), dtype=torch.uint8, device=dev)
    fwd = lambda: attn.attn_fwd_fp8(*bufs, causal=w["causal"], scale=scale, out=o8, lse=l8, stream=stream,
                                    workspace=ws)
    def both():
        prep()
        fwd()
    prep()
    for _ in range(3):
        fwd()
    torch.cuda.synchronize()
    n = max(args.steps, 20)
    t0 = time.time()
    t_fwd = time_kernel(fwd, n, 0, stream) / n
    clocks_fwd = sampler.summary(t0, time.time()) if sampler else None
    t_sus, n_sus, clocks_sus = time_for(fwd, 1.5, stream, sampler)
    t_prep, _, clocks_prep = time_for(prep, 0.3, stream, sampler)
    t_prep_rope, _, _ = time_for(prep_rope, 0.3, stream, sampler)
    t_both, _, _ = time_for(both, 0.3, stream, sampler)
    if attn.device_status() != attn.ATTN_OK:
        raise RuntimeError("device status after the FP8 leg")
    fl = flops(w)
    val = fl / (t_fwd * 1e-3) / 1e12
    sus = fl / (t_sus * 1e-3) / 1e12
    prep_bytes = 3 * q.numel() * 2 + 3 * q.numel() + 3 * B * H * nblk * 4
    out = {"workload": f"fp8 e4m3 attention fwd, B={B}, H={H}, N={N}, d={d}, "
                       f"{'causal' if w['causal'] else 'non-causal'}, per-block scales + Hadamard, "
                       "inputs N(0,1) + N(0,100) * Bernoulli(0.001), bf16 output",
           "value": round(val, 2), "unit": UNIT, "launches": n,
           "schedule": ("round-robin rounds plus a stream-K tail (attn_fwd_fp8_ws workspace; its arrival "
                        "counters are zeroed by one cudaMemsetAsync before each launch)") if not w["causal"]
                       else "persistent, longest-first causal units",
           "roofline": roofline(val, fp8=True, kernel="attn_fwd_kernel<128, e4m3>"),
           "clocks": clocks_fwd,
           "sustained": {"value": round(sus, 2), "launches": n_sus, "roofline": roofline(sus, fp8=True, sustained=True),
                         "clocks": clocks_sus},
           "prepare_us": round(t_prep * 1e3, 2),
           "prepare_rotary_us": round(t_prep_rope * 1e3, 2),
           "prepare_gbs": round(prep_bytes / (t_prep * 1e-3) / 1e9, 1),
           "prepare_roofline": {"bound": "hbm", "achieved": round(prep_bytes / (t_prep * 1e-3) / 1e9, 1),
                                "peak": hbm_peak(), "unit": "GB/s",
                                "frac": round(prep_bytes / (t_prep * 1e-3) / 1e9 / hbm_peak(), 4),
                                "algorithmic_bytes": prep_bytes, "clocks": clocks_prep},
           "pipeline_value": round(fl / (t_both * 1e-3) / 1e12, 2)}
    if rank == 0:
        # Accuracy beside the rate, outside the timed region: RMS of the FP8 output against the
        # bf16 kernel's on the same inputs, every element (parity against the float64 oracle is
        # the tests' job).
        ob = attn.attn_fwd(qd, kd, vd, causal=w["causal"], scale=scale)[0].float()
        on, _ = attn.attn_fwd_fp8_pipeline(qd, kd, vd, signs=None, causal=w["causal"], scale=scale,
                                           per_tensor=True)
        out["rms_vs_bf16_kernel"] = float((o8.float() - ob).square().mean().sqrt())
        out["rms_vs_bf16_kernel_naive_per_tensor"] = float((on.float() - ob).square().mean().sqrt())
        del ob, on
    return out


# --------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    import synth
    w = WORKLOADS[args.workload]
    N, d = w["N"], w["d"]
    # The oracle needs only the rows it computes plus the keys and values of head 0.
    q, k, v = synth.attention_inputs(1, 1, N, d, w["dtype"], seed=0)
    probe = synth.sample_rows(N, 16, seed=3, salt=97)
    t0 = time.time()
    _, _, used = oracle.attention(q, k, v, causal=w["causal"], scale=d ** -0.5, rows=probe,
                                  return_threads=True)
    per_row = max(time.time() - t0, 1e-4) / len(probe)
    budget = 90.0  # seconds for the whole run
    rows_per_step = int(max(1, min(N, budget / (args.steps + args.warmup) / per_row)))
    total_fl, total_t = 0.0, 0.0
    for i in range(args.warmup + args.steps):
        rows = synth.sample_rows(N, rows_per_step, seed=4 + i, salt=96)
        t0 = time.time()
        oracle.attention(q, k, v, causal=w["causal"], scale=d ** -0.5, rows=rows)
        dt = time.time() - t0
        if i >= args.warmup:
            keys = (rows + 1).sum() if w["causal"] else len(rows) * N
            total_fl += 4.0 * float(keys) * d
            total_t += dt
    value = total_fl / total_t / 1e12
    sample = (f"{rows_per_step} query rows of one head per step (all their keys), float64, "
              f"{args.steps} timed steps")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded iid N(0,1))",
            "config": {"workload": describe(w), "B": w["B"], "H": w["H"], "N": N, "d": d,
                       "causal": w["causal"], "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ablation(args):
    """Overlap ablation (in the spirit of the FlashAttention-3 page's ablation
    table): the bench workload, causal and not, and the FP8 kernel, timed with
    two Q tiles per CTA whose softmax and products overlap (ping-pong, the
    default) and with one Q tile per CTA at a time (no overlap).  Each line is
    at least 0.5 s of back-to-back launches and carries its clock record."""
    import exact_attention_forward_05_gb300 as attn
    import synth
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(0)
    time.sleep(0.5)
    B, H, N, d = 2, 16, 8192, 128
    q, k, v = (t.to(dev) for t in synth.attention_inputs(B, H, N, d, "bf16", seed=0))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    qo, ko, vo = (t.to(dev) for t in synth.outlier_inputs(B, H, N, d, "bf16", seed=0))
    bufs = attn.fp8_prepare(qo, ko, vo, signs=synth.hadamard_signs(H, d, seed=0).to(dev))
    o8 = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)

    def emit(name, w, f, fp8):
        for _ in range(max(args.warmup, 3)):
            f()
        ms, n, clocks = time_for(f, 0.5, stream, sampler)
        tf = flops(w) / (ms * 1e-3) / 1e12
        rl = roofline(tf, fp8=fp8)
        print(json.dumps({"schedule": name, "workload": describe(w), "value": round(tf, 1), "unit": UNIT,
                          "frac": rl["frac"], "frac_nominal": rl["frac_nominal"], "ms": round(ms, 4),
                          "launches": n, "clocks": clocks}), flush=True)

    try:
        for mode, name in ((attn.SCHEDULE_PINGPONG, "ping-pong (two Q tiles, overlap)"),
                           (attn.SCHEDULE_ONE_TILE, "one Q tile per CTA (no overlap)")):
            attn.set_schedule(mode)
            for causal in (False, True):
                emit(name, dict(B=B, H=H, N=N, d=d, causal=causal, dtype="bf16"),
                     lambda: attn.attn_fwd(q, k, v, causal=causal, scale=d ** -0.5, out=o, lse=lse,
                                           stream=stream), False)
            emit(name, dict(B=B, H=H, N=N, d=d, causal=False, dtype="fp8 e4m3"),
                 lambda: attn.attn_fwd_fp8(*bufs, causal=False, scale=d ** -0.5, out=o8,
                                           return_lse=False, stream=stream), True)
    finally:
        attn.set_schedule(attn.SCHEDULE_PINGPONG)
        sampler.stop()
    if attn.device_status() != attn.ATTN_OK:
        raise RuntimeError("device status after the ablation")


def run_sweep(args):
    """One device-timed line per point of the sequence-length sweep (bf16,
    B = 16384/N, H = 2048/d, causal and non-causal), the FP8 kernel at
    d = 128 (H = 16, inputs with 0.1 % outliers), and the long-context causal
    case (B = 1, H = 16, N = 32768, d = 128).  Each point: CUDA events on the
    launching stream around at least 0.5 s of back-to-back launches, with the
    clock record of that window."""
    import exact_attention_forward_05_gb300 as attn
    import synth
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(0)
    time.sleep(0.5)

    def emit(w, f, fp8=False):
        for _ in range(max(args.warmup, 3)):
            f()
        ms, n, clocks = time_for(f, 0.5, stream, sampler)
        tf = flops(w) / (ms * 1e-3) / 1e12
        rl = roofline(tf, fp8=fp8)
        print(json.dumps({"workload": describe(w), "value": round(tf, 1), "unit": UNIT,
                          "frac": rl["frac"], "frac_nominal": rl["frac_nominal"], "ms": round(ms, 4),
                          "launches": n, "clocks": clocks}), flush=True)

    try:
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            for d in (64, 128, 256):
                B, H = 16384 // N, 2048 // d
                q, k, v = (t.to(dev) for t in synth.attention_inputs(B, H, N, d, "bf16", seed=0))
                o = torch.empty_like(q)
                lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
                for causal in (False, True):
                    emit(dict(B=B, H=H, N=N, d=d, causal=causal, dtype="bf16"),
                         lambda: attn.attn_fwd(q, k, v, causal=causal, scale=d ** -0.5, out=o, lse=lse,
                                               stream=stream))
                del q, k, v, o, lse
            # FP8: d = 128 with H = 16 (the FP8 workload), d = 64 and 256 with the
            # bf16 sweep's H = 2048 / d.
            for d in (64, 128, 256):
                B, H = 16384 // N, (16 if d == 128 else 2048 // d)
                q, k, v = (t.to(dev) for t in synth.outlier_inputs(B, H, N, d, "bf16", seed=0))
                bufs = attn.fp8_prepare(q, k, v, signs=synth.hadamard_signs(H, d, seed=0).to(dev))
                o8 = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
                for causal in (False, True):
                    emit(dict(B=B, H=H, N=N, d=d, causal=causal, dtype="fp8 e4m3"),
                         lambda: attn.attn_fwd_fp8(*bufs, causal=causal, scale=d ** -0.5, out=o8,
                                                   return_lse=False, stream=stream), fp8=True)
                del q, k, v, bufs, o8
        # Long-context configuration: B = 1, H = 16, N = 32768, d = 128, causal.
        B, H, N, d = 1, 16, 32768, 128
        q, k, v = (t.to(dev) for t in synth.attention_inputs(B, H, N, d, "bf16", seed=0))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        emit(dict(B=B, H=H, N=N, d=d, causal=True, dtype="bf16"),
             lambda: attn.attn_fwd(q, k, v, causal=True, scale=d ** -0.5, out=o, lse=lse, stream=stream))
        del q, k, v, o, lse
    finally:
        sampler.stop()
    if attn.device_status() != attn.ATTN_OK:
        raise RuntimeError("device status after the sweep")


def run_backward(args):
    """Backward pass (attn_bwd: the row dot products D, the main kernel, the
    final dQ pass) on the bench workload's shapes, causal and not, each line
    at least 0.5 s of back-to-back calls with its clock record.  FLOPs:
    2.5 x the forward's 4 B H N^2 d (five products per block pair against the
    forward's two), halved when causal."""
    import exact_attention_forward_05_gb300 as attn
    import synth
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(0)
    time.sleep(0.5)
    w0 = WORKLOADS[args.workload]
    B, H, N, d = w0["B"], w0["H"], w0["N"], w0["d"]
    q, k, v = (t.to(dev) for t in synth.attention_inputs(B, H, N, d, "bf16", seed=0))
    g = synth.attention_inputs(B, H, N, d, "bf16", seed=1000)[0].to(dev)
    ws = torch.empty(attn.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)
    grads = tuple(torch.empty_like(q) for _ in range(3))
    try:
        for causal in (False, True):
            o, lse = attn.attn_fwd(q, k, v, causal=causal)
            f = lambda: attn.attn_bwd(q, k, v, o, g, lse, causal=causal, workspace=ws, out=grads, stream=stream)
            for _ in range(max(args.warmup, 3)):
                f()
            ms, n, clocks = time_for(f, 0.5, stream, sampler)
            w = dict(B=B, H=H, N=N, d=d, causal=causal, dtype="bf16")
            fl = 2.5 * flops(w)
            tf = fl / (ms * 1e-3) / 1e12
            rl = roofline(tf)
            print(json.dumps({"workload": "backward of " + describe(w), "value": round(tf, 1), "unit": UNIT,
                              "flops_convention": "2.5 x 4 B H N^2 d (halved when causal)",
                              "frac": rl["frac"], "frac_nominal": rl["frac_nominal"], "ms": round(ms, 4),
                              "launches": n, "clocks": clocks}), flush=True)
    finally:
        sampler.stop()
    if attn.device_status() != attn.ATTN_OK:
        raise RuntimeError("device status after the backward")


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--ablation", action="store_true",
                    help="overlap ablation: the bench workload under both work schedules, one line each")
    ap.add_argument("--sweep", action="store_true",
                    help="print one device-timed line per sweep configuration instead")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass on the workload's shapes (causal and not), one line each")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.backward:
        run_backward(args)
        return
    if args.ablation:
        run_ablation(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
