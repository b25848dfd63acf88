#!/usr/bin/env python
"""Attention-forward benchmark: TFLOP/s (bf16) and fraction of dense-BF16 peak.

One step is one exact attention forward (QK^T, online softmax, PV, O and
LSE) over the whole workload, i.e. one launch of the library's kernel.  The
default workload is B=2, H=32, N=4096, d=128, causal.  FLOPs per step are
4*B*H*Nq*Nk*d, halved for causal.

With --fp8 a step is one forward pass of the 8-bit path (fa_fwd_fp8) on the
workload quantized to e4m3 (V transposed); its roofline peak is the bf16 peak
times the nominal fp8 : bf16 ratio of 2.

With --bwd a step is instead one backward pass (dQ, dK, dV and delta from
Q, K, V, O, LSE and dO: three kernel launches); FLOPs per step are counted
as 2.5 times the forward's (the five products of the plain gradient), so the
products the kernels recompute are not credited.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--bwd]
    python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

With N > 1 (torchrun), every rank runs its own copy of the workload: the
units are independent (batch, head, query block) problems, so there is no
collective on the data path ("scaling": "weak"); the barrier and the
max-over-ranks timing are the only cross-rank steps.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s bf16 (N=4096,d=128,causal) and % of dense-BF16 peak"
METRIC_BWD = "attention bwd TFLOP/s bf16 (dQ, dK, dV; 2.5x the forward FLOPs) and % of dense-BF16 peak"
METRIC_FP8 = "attention fwd TFLOP/s fp8 e4m3 and % of dense-FP8 peak"
FP8_OVER_BF16 = 2.0   # nominal dense fp8 : bf16 tensor rate (4.5 : 2.25 PFLOP/s)
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["exact_attention_42_gb300/csrc/fa_fwd.cu", "exact_attention_42_gb300/csrc/ptx.cuh",
                      "exact_attention_42_gb300/csrc/fa_sched.cu"],
    "decode_kernel": ["exact_attention_42_gb300/csrc/fa_decode.cu", "exact_attention_42_gb300/csrc/ptx.cuh"],
    "fa_bwd": ["exact_attention_42_gb300/csrc/fa_bwd.cu", "exact_attention_42_gb300/csrc/ptx.cuh",
               "exact_attention_42_gb300/csrc/fa_sched.cu"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
ROTATE_MIN = 3        # input copies cycled through, so each step reads from HBM
ROTATE_MAX = 4096
L2_BYTES = 129 * 2 ** 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget-s", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--bwd", action="store_true", help="time the backward pass instead of the forward")
    ap.add_argument("--fp8", action="store_true", help="time the 8-bit (e4m3) forward")
    ap.add_argument("--graph", action="store_true",
                    help="capture the timed steps into one CUDA graph and time its replay (launch-bound workloads)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- helpers

def kernel_hash(kernel: str = "fa_fwd_kernel") -> str:
    """Digest of the sources one kernel is built from (ties ncu figures to them)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, k if not pre else pre + "." + k)
                elif isinstance(x, (int, float)):
                    flat[pre.split(".")[-1]] = float(x)
            walk(d)
            if "bf16_tflops" in flat:
                return {"hbm_gbs": flat.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]),
                        "bf16_tflops": flat["bf16_tflops"],
                        "bf16_tflops_sustained": flat.get("bf16_tflops_sustained", flat["bf16_tflops"]),
                        "source": "measured"}
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


def load_traffic(workload: str, kernel: str = "fa_fwd_kernel"):
    """ncu DRAM bytes per launch, if captured for this exact kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel_sha") != kernel_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (read-only
    queries) every millisecond on a background thread, so that even a timed
    region of a few milliseconds has samples.  mark_start / mark_stop bracket
    the timed region; stop() summarises the samples taken inside it."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str):
        import ctypes
        import threading
        self.ct = ctypes
        self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        if self.nvml.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML device with uuid %s" % uuid)
        self.get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.sm_max = float(mx.value)
        self.samples = []
        self.window = [None, None]
        self.stop_evt = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _read(self):
        ct = self.ct
        clk, mw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(clk))
        self.nvml.nvmlDeviceGetPowerUsage(self.handle, ct.byref(mw))
        self.get_reasons(self.handle, ct.byref(rs))
        return time.perf_counter(), float(clk.value), mw.value / 1000.0, int(rs.value)

    def _run(self):
        while not self.stop_evt.is_set():
            self.samples.append(self._read())
            time.sleep(0.001)

    def start(self):
        self.thread.start()

    def mark_start(self):
        self.samples.append(self._read())
        self.window[0] = time.perf_counter()

    def mark_stop(self):
        self.window[1] = time.perf_counter()
        self.samples.append(self._read())

    def stop(self):
        self.stop_evt.set()
        self.thread.join(timeout=5)
        try:
            self.nvml.nvmlShutdown()
        except Exception:
            pass
        t0, t1 = self.window
        inside = [x for x in self.samples if t0 is not None and t1 is not None and t0 <= x[0] <= t1]
        use = inside or self.samples
        if not use:
            return None
        reasons = sorted({name for x in use for bit, name in self.REASONS.items() if x[3] & bit})
        return {"sm_mhz": statistics.median(x[1] for x in use), "sm_max_mhz": self.sm_max, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside),
                "power_w_median": statistics.median(x[2] for x in use),
                "source": "NVML, 1 ms polling during the timed region"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms (used when NVML
    cannot be loaded)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.proc = None
        self.path = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="fa_clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "200"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        try:
            sm = [float(r[1]) for r in rows]
            smax = max(float(r[2]) for r in rows)
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows), "power_w_median": statistics.median(
                    [float(r[3]) for r in rows if r[3].replace(".", "", 1).isdigit()] or [0.0]),
                "source": "nvidia-smi -lms 200 over warm-up and timed region"}

    def mark_start(self):
        pass

    def mark_stop(self):
        pass


def host_cpu():
    """Logical CPUs of the host and its model name (for the CPU baseline)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    import platform
    return {"nproc": os.cpu_count(), "model": model or platform.processor() or platform.machine()}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Maximum of `value` over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def is_decode(prob) -> bool:
    """Whether fa_fwd runs this problem on the split-KV (decode) path."""
    return (not prob.varlen) and prob.Nk > 0 and (prob.Hq // prob.Hkv) * prob.Nq <= 16


def step_bytes(prob, bwd: bool = False, fp8: bool = False) -> int:
    """Bytes of one input set and its outputs (what one timed step touches)."""
    rows = prob.q.size // prob.d
    qkv = (prob.q.size + prob.k.size + prob.v.size) * (1 if fp8 else 2)
    out = 2 * prob.q.size + 4 * rows                      # O bf16, LSE fp32
    if bwd:
        # O, LSE and dO in; dQ, dK, dV and delta out.
        return qkv + out + 2 * prob.q.size + 2 * (prob.q.size + prob.k.size + prob.v.size) + 4 * rows
    return qkv + out


def rotation(prob, bwd: bool = False, fp8: bool = False) -> int:
    """Input copies the timed steps cycle through: enough that together they
    hold more than twice the L2, so that each step's inputs come from HBM
    (at least ROTATE_MIN, at most ROTATE_MAX)."""
    per = max(1, step_bytes(prob, bwd, fp8))
    return int(min(ROTATE_MAX, max(ROTATE_MIN, 2 * L2_BYTES // per + 1)))


def workload_config(prob, name, world: int = 1, bwd: bool = False, fp8: bool = False):
    cfg = {"workload": name, "B": prob.B, "Hq": prob.Hq, "Hkv": prob.Hkv, "Nq": prob.Nq, "Nk": prob.Nk,
           "d": prob.d, "causal": prob.causal, "flop_per_step": prob.flops()}
    if prob.varlen:
        cfg["seqlens"] = prob.seqlens()
        cfg["total_tokens"] = int(prob.cu_seqlens[-1])
    cfg["parallelism"] = "replicas" if world > 1 else "single"
    rot = rotation(prob, bwd, fp8)
    cfg["l2"] = "inputs rotated over %d copies (%.0f MB > %d MB L2)" % (
        rot, rot * step_bytes(prob, bwd, fp8) / 1e6, L2_BYTES // 2 ** 20)
    return cfg


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(prob, budget_s: float, start_head: int = 0, backward: bool = False):
    """Times the fp64 oracle, as it stands, on whole heads of the workload
    until `budget_s` is spent (at least one head).  Returns (TFLOP/s, threads,
    description).  With `backward`, the oracle's gradients of each head (dense
    workloads), counted at 2.5 times the forward FLOPs."""
    import numpy as np
    from fa_inputs import bf16_bits_to_f64, make_dout
    from oracle import attention_bwd, attention_fwd, oracle_threads
    dout = make_dout(prob, 1000) if backward else None

    flops = 0.0
    heads = 0
    t0 = time.perf_counter()
    hq = start_head
    while True:
        if prob.varlen:
            s = hq % prob.B
            h = (hq // prob.B) % prob.Hq
            t_0, t_1 = int(prob.cu_seqlens[s]), int(prob.cu_seqlens[s + 1])
            L = t_1 - t_0
            kvh = h // (prob.Hq // prob.Hkv)
            q = bf16_bits_to_f64(prob.q[h:h + 1, t_0:t_1])[None]
            k = bf16_bits_to_f64(prob.k[kvh:kvh + 1, t_0:t_1])[None]
            v = bf16_bits_to_f64(prob.v[kvh:kvh + 1, t_0:t_1])[None]
            f = 4.0 * L * L * prob.d * (0.5 if prob.causal else 1.0)
        else:
            b = (hq // prob.Hq) % prob.B
            h = hq % prob.Hq
            kvh = h // (prob.Hq // prob.Hkv)
            q = bf16_bits_to_f64(prob.q[b:b + 1, h:h + 1])
            k = bf16_bits_to_f64(prob.k[b:b + 1, kvh:kvh + 1])
            v = bf16_bits_to_f64(prob.v[b:b + 1, kvh:kvh + 1])
            f = 4.0 * prob.Nq * prob.Nk * prob.d * (0.5 if prob.causal else 1.0)
        if backward:
            attention_bwd(q, k, v, bf16_bits_to_f64(dout[b:b + 1, h:h + 1]), prob.scale, prob.causal)
            f *= 2.5
        else:
            attention_fwd(q, k, v, prob.scale, prob.causal)
        flops += f
        heads += 1
        hq += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    desc = "%d whole head(s) of %s (every query row of each), fp64%s, %.1f s" % (
        heads, prob.name, ", backward" if backward else "", dt)
    return flops / dt / 1e12, oracle_threads(), desc, dt


def run_reference(args):
    """The oracle on the host cores, on the same workload and metric."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    from fa_inputs import make_workload, HEADLINE
    name = args.workload or HEADLINE
    prob = make_workload(name)
    if (args.bwd or args.fp8) and prob.varlen:
        raise SystemExit("--bwd / --fp8: dense workloads only")
    per_step = max(1.0, args.cpu_budget_s / max(1, args.steps))
    for w in range(args.warmup):
        oracle_sample(prob, 0.0, start_head=w, backward=args.bwd)
    vals, secs, descs = [], [], []
    t0 = time.perf_counter()
    threads = None
    for i in range(args.steps):
        v, threads, desc, dt = oracle_sample(prob, per_step, start_head=i * 7, backward=args.bwd)
        vals.append(v)
        secs.append(dt)
        descs.append(desc)
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {"metric": METRIC_BWD if args.bwd else (METRIC_FP8 if args.fp8 else METRIC), "value": value,
            "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": workload_config(prob, name, args.gpus, args.bwd, args.fp8),
            "cpu_baseline": dict({"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                                  "sample": "per step: " + descs[-1]}, **host_cpu()),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU run

def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    import exact_attention_42_gb300 as fa
    if rank == 0:
        fa.build()
    barrier(world, dev)
    fa.lib()

    from fa_inputs import make_workload, make_dout, HEADLINE
    name = args.workload or HEADLINE
    prob = make_workload(name)
    if (args.bwd or args.fp8) and prob.varlen:
        raise SystemExit("--bwd / --fp8: dense workloads only")
    flops = prob.flops() * (2.5 if args.bwd else 1.0)

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    if args.fp8:
        from fa_inputs import make_fp8
        f8 = make_fp8(prob)
        u8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
        q0, k0, v0 = u8(f8.q8), u8(f8.k8), u8(f8.vt8)
        descales = (f32(f8.q_scale), f32(f8.k_scale), f32(f8.v_scale))
    else:
        q0, k0, v0 = dev_bf16(prob.q), dev_bf16(prob.k), dev_bf16(prob.v)
    do0 = dev_bf16(make_dout(prob, 1000)) if args.bwd else None
    cu = None if prob.cu_seqlens is None else torch.from_numpy(prob.cu_seqlens).to(dev)
    sets = []
    rotate = rotation(prob, args.bwd, args.fp8)
    for r in range(rotate):
        q, k, v = (q0, k0, v0) if r == 0 else (q0.clone(), k0.clone(), v0.clone())
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
        if args.bwd:
            # The forward pass's O and LSE are inputs of the backward step.
            fa.fwd(q, k, v, causal=prob.causal, scale=prob.scale, out=o, lse=lse)
            do = do0 if r == 0 else do0.clone()
            grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                     torch.empty(q.shape[:-1], dtype=torch.float32, device=dev))
            sets.append((q, k, v, o, lse, do) + grads)
        else:
            sets.append((q, k, v, o, lse))
    stream = torch.cuda.current_stream(dev)
    launches_per_step = 3 if args.bwd else 1

    def step(i, s=None):
        s = stream if s is None else s
        if args.bwd:
            q, k, v, o, lse, do, dq, dk, dv, dl = sets[i % rotate]
            fa.bwd(q, k, v, o, lse, do, causal=prob.causal, scale=prob.scale, stream=s,
                   dq=dq, dk=dk, dv=dv, delta=dl)
            return
        q, k, v, o, lse = sets[i % rotate]
        if args.fp8:
            fa.fwd_fp8(q, k, v, *descales, causal=prob.causal, scale=prob.scale, out=o, lse=lse, stream=s)
            return
        fa.fwd(q, k, v, causal=prob.causal, scale=prob.scale, cu_seqlens=cu, out=o, lse=lse, stream=s)

    # --graph: the timed steps are captured into one CUDA graph once (after
    # the warm-up) and the timed region is its replay, so that host launch
    # overhead drops out for launch-bound workloads.  The kernels and their
    # inputs are the same.
    graph = None
    if args.graph:
        for i in range(max(args.warmup, 1)):
            step(i)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(args.steps):
                step(i, torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)

    fa.fa_device_status()
    sampler = None
    if not args.no_clocks:
        gid = None
        try:
            gid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
        except Exception:
            gid = None
        try:
            sampler = NvmlClockSampler(gid)
        except (OSError, AttributeError, TypeError):
            sampler = ClockSampler(gid)
        sampler.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark_start()
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_stop()
    barrier(world, dev)
    clocks = sampler.stop() if sampler else None
    ms_total = ev0.elapsed_time(ev1)
    ms_step = reduce_max(ms_total / args.steps, world, dev)
    status_bits = fa.fa_device_status()
    value = world * flops / (ms_step * 1e-3) / 1e12

    # Warm-L2 figure, for context beside the cold one above: the same input
    # set every step (whatever of it fits stays in L2).  Not the bench value.
    warm_steps = max(3, min(args.steps, 50))
    for _ in range(3):
        step(0)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(warm_steps):
        step(0)
    w1.record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = w0.elapsed_time(w1) / warm_steps
    status_bits |= fa.fa_device_status()

    # End to end through the public API: pinned host inputs copied in, the
    # kernels, the results copied back, every step.
    if args.bwd:
        q, k, v, o, lse, do, dq, dk, dv, dl = sets[0]
        ins = (q, k, v, o, lse, do)
        outs = (dq, dk, dv, dl)
    else:
        q, k, v, o, lse = sets[0]
        ins = (q, k, v)
        outs = (o, lse)
    hins = tuple(t.cpu().pin_memory() for t in ins)
    houts = tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs)
    cu_host = None if cu is None else cu.cpu()
    h2d = sum(t.numel() * t.element_size() for t in hins) + (0 if cu_host is None else cu_host.numel() * 4)
    d2h = sum(t.numel() * t.element_size() for t in houts)
    host_api = not (args.bwd or args.fp8)

    def e2e_step():
        if host_api:
            # fwd_host: the forward for host tensors (copies in, kernels and
            # copies out pipelined over pieces of the batch), waits for O, LSE.
            fa.fwd_host(*hins, causal=prob.causal, scale=prob.scale, cu_seqlens=cu_host, device=dev,
                        out=houts[0], lse=houts[1])
            return
        for dst, src in zip(ins, hins):
            dst.copy_(src, non_blocking=True)
        if args.bwd:
            fa.bwd(q, k, v, o, lse, do, causal=prob.causal, scale=prob.scale, stream=stream,
                   dq=dq, dk=dk, dv=dv, delta=dl)
        elif args.fp8:
            fa.fwd_fp8(q, k, v, *descales, causal=prob.causal, scale=prob.scale, out=o, lse=lse, stream=stream)
        else:
            fa.fwd(q, k, v, causal=prob.causal, scale=prob.scale, cu_seqlens=cu, out=o, lse=lse, stream=stream)
        for dst, src in zip(houts, outs):
            dst.copy_(src, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1) / args.e2e_steps, world, dev)
    e2e_value = world * flops / (e2e_ms * 1e-3) / 1e12

    peaks = load_peaks()
    tag = "of measured" if peaks["source"] == "measured" else "of fallback"
    launch_s = ms_total / args.steps * 1e-3
    if args.bwd:
        # The whole backward step (delta, dQ and dK/dV kernels) against the
        # dense bf16 peak, credited with the plain gradient's FLOPs only.
        achieved = flops / launch_s / 1e12
        sustained = ms_total >= 1000.0
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": load_traffic(name + ":bwd", "fa_bwd"),
                    "peak_kind": "bf16 dense %s %s" % ("sustained" if sustained else "burst", tag),
                    "frac_of_burst": achieved / peaks["bf16_tflops"],
                    "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                    "kernel": "fa_bwd", "algorithmic_flop_per_launch": flops,
                    "executed_flop_per_launch": prob.flops() * 3.5,
                    "note": "one step = bwd_delta_kernel + bwd_dq_kernel + bwd_dkdv_kernel"}
    elif args.fp8:
        achieved = flops / launch_s / 1e12
        sustained = ms_total >= 1000.0
        peak = FP8_OVER_BF16 * (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"])
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": load_traffic(name + ":fp8"),
                    "peak_kind": "fp8 dense %s = bf16 %s x %.0f (nominal fp8:bf16 ratio)"
                                 % ("sustained" if sustained else "burst", tag, FP8_OVER_BF16),
                    "kernel": "fa_fwd_kernel", "algorithmic_flop_per_launch": flops,
                    "algorithmic_bytes_per_launch": prob.q.size + prob.k.size + prob.v.size + 2 * prob.q.size
                                                    + 4 * (prob.q.size // prob.d)}
    elif is_decode(prob):
        # Split-KV path: bound by reading K and V from HBM.
        achieved = prob.io_bytes() / launch_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "traffic": load_traffic(name, "decode_kernel"),
                    "peak_kind": "HBM copy bandwidth " + tag, "kernel": "decode_kernel",
                    "algorithmic_bytes_per_launch": prob.io_bytes(), "algorithmic_flop_per_launch": flops}
    else:
        achieved = flops / launch_s / 1e12
        # A timed region of a second or more runs under the power cap, like the
        # seconds-long GEMM loop behind the sustained peak; shorter runs compare
        # against the burst peak.
        sustained = ms_total >= 1000.0
        peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": load_traffic(name),
                    "peak_kind": "bf16 dense %s %s" % ("sustained" if sustained else "burst", tag),
                    "frac_of_burst": achieved / peaks["bf16_tflops"],
                    "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                    "kernel": "fa_fwd_kernel", "algorithmic_flop_per_launch": flops,
                    "algorithmic_bytes_per_launch": prob.io_bytes()}
    line = {"metric": METRIC_BWD if args.bwd else (METRIC_FP8 if args.fp8 else METRIC), "value": value,
            "unit": UNIT, "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3" if args.fp8 else "bf16", "data": "synthetic",
            "config": dict(workload_config(prob, name, world, args.bwd, args.fp8),
                           **({"launch": "one CUDA graph of the timed steps"} if args.graph else {})),
            "roofline": roofline,
            "warm_l2": {"ms_per_step": warm_ms, "value": flops / (warm_ms * 1e-3) / 1e12, "unit": UNIT,
                        "steps": warm_steps, "note": "one input set reused every step; context only"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "call": "fwd_host" if host_api else "copies + " + ("bwd" if args.bwd else "fwd_fp8"),
                    "ms_per_step": e2e_ms},
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks,
            "device_status": status_bits,
            "kernel_sha": kernel_hash(roofline["kernel"])}
    if rank == 0 and not args.no_cpu_baseline:
        v_cpu, threads, desc, _ = oracle_sample(prob, args.cpu_budget_s, backward=args.bwd)
        line["cpu_baseline"] = dict({"value": v_cpu, "unit": UNIT, "cores": threads, "kind": "oracle",
                                     "sample": desc}, **host_cpu())
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0 if status_bits == 0 else 1


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
