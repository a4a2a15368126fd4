#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step = the whole path once:
  * bf16 forward + backward (preprocess, main, dQ conversion) on
    B=1, H=32, N=8192, d=128, non-causal, 1% of key rows scaled x8;
  * FP8 (E4M3, per-tensor scales) forward on B=1, H=16, N=16384, d=128, causal.
Metric: attention TFLOP/s (forward 4*B*H*N^2*d, halved when causal; backward
2.5x the forward), whole job over all ranks.  Inputs are seeded synthetic
N(0,1) draws (no dataset involved); together they exceed the 129 MB L2, so
no flush is done between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the only reference this
method has) on a bounded sample of the same workload on the host cores.
For N > 1 (torchrun), every rank runs its own copy of the workload (weak
scaling over independent (batch, head) problems; no collective on the data
path) and rank 0 prints one JSON line.
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

from exact_attention_52_gb300.roofline import attn_bytes, attn_flops  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s on 1xGB300 (bf16, fp8 fwd) and % of dense tensor peak"
BF16 = dict(B=1, H=32, N=8192, d=128, causal=False, outlier_frac=0.01, outlier_factor=8.0)
FP8 = dict(B=1, H=16, N=16384, d=128, causal=True)
WORKLOAD = ("fwd+bwd bf16 B1 H32 N8192 d128 (1% keys x8) + fp8 fwd B1 H16 N16384 d128 causal")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
CPU_BASELINE_S = 10.0  # host seconds spent on the oracle sample of the default run
REF_BUDGET_S = 90.0  # wall time of the whole --impl reference run


def step_flops():
    fb = attn_flops(BF16["B"], BF16["H"], BF16["N"], BF16["d"], BF16["causal"])
    f8 = attn_flops(FP8["B"], FP8["H"], FP8["N"], FP8["d"], FP8["causal"])
    return {"fwd": fb, "bwd": 2.5 * fb, "fwd_fp8": f8}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_sources_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_52_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed after the capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    e = t.get(kernel_key)
    if not e or e.get("sources_sha") != kernel_sources_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clock, power and throttle-reason samples during the timed region.

    Read-only NVML queries (ctypes on the driver's libnvidia-ml) from a thread
    every ``period_s`` (5 ms), so that a region of tens of milliseconds still
    gets a dozen samples or more; the GPU is found by its PCI bus id, which
    NVML and CUDA share whatever the device numbering.  Falls back to
    ``nvidia-smi -lms 20`` when NVML cannot be opened.  Nothing is set."""

    # nvmlClocksEventReasons bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, torch_device_index, period_s=0.005):
        self.index = torch_device_index
        self.period = period_s
        self.samples = []  # (sm_mhz, max_mhz, reason bits)
        self.thread = None
        self.stop_flag = False
        self.proc = None
        self.path = None
        self.source = None

    def _bus_id(self):
        import torch
        p = torch.cuda.get_device_properties(self.index)
        try:
            return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except AttributeError:
            return None

    def _open_nvml(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        bus = self._bus_id()
        if bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        return nv, h, reasons_fn

    def start(self):
        import ctypes
        import threading
        try:
            nv, h, reasons_fn = self._open_nvml()
        except (OSError, AttributeError):
            return self._start_smi()
        self.source = "nvml"
        mx = ctypes.c_uint(0)
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM

        def loop():
            clk = ctypes.c_uint(0)
            rs = ctypes.c_ulonglong(0)
            while not self.stop_flag:
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                    r = rs.value if reasons_fn(h, ctypes.byref(rs)) == 0 else 0
                    self.samples.append((float(clk.value), float(mx.value), r))
                time.sleep(self.period)

        self.thread = threading.Thread(target=loop, daemon=True)
        self.thread.start()

    def _start_smi(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        bus = self._bus_id()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", bus or str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
            sm = [x[0] for x in self.samples]
            mx = [x[1] for x in self.samples]
            reasons = sorted({n for x in self.samples for bit, n in self.REASONS.items() if x[2] & bit})
        elif self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            sm, mx, reasons = [], [], set()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 7:
                        continue
                    try:
                        sm.append(float(parts[0]))
                        mx.append(float(parts[1]))
                    except ValueError:
                        continue
                    for n, v in zip(names, parts[3:7]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
            reasons = sorted(reasons)
        else:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "sm_min_mhz": min(sm),
                "samples": len(sm), "reasons": reasons, "source": self.source}


# ---------------------------------------------------------------------------
# CPU side: the oracle (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------


def oracle_sample_step(data, n_rows):
    """One bounded sample of the workload through the fp64 oracle: the forward
    and backward work of ``n_rows`` evenly spaced query rows of head 0 of the
    bf16 workload (non-causal, so a row subset is an exact slice of the work:
    its S, P, dP, dS and dQ rows and its rank-``n_rows`` share of dK and dV),
    plus 256 evenly spaced query rows of head 0 of the FP8 workload.  Returns
    the attention FLOPs covered (same convention as the GPU)."""
    import numpy as np

    import oracle
    q, k, v, do = data["bf16"]
    N, D = BF16["N"], BF16["d"]
    rows = np.linspace(0, N - 1, n_rows).astype(np.int64)
    s = 1.0 / math.sqrt(D)
    oracle.head_forward(q[0, 0], k[0, 0], v[0, 0], s, False, rows=rows)
    oracle.head_backward(q[0, 0][rows], k[0, 0], v[0, 0], do[0, 0][rows], s, False)
    q8, k8, v8 = data["fp8"]
    rows8 = data["fp8_rows"]
    oracle.forward(q8, k8, v8, s, FP8["causal"], heads=[(0, 0)], rows=rows8)
    f = 4.0 * n_rows * N * D * 3.5
    # causal rows i see i+1 keys: 2*(i+1)*d multiply-adds for each of S and PV
    f += sum(4.0 * (int(i) + 1) * FP8["d"] for i in rows8)
    return f


def oracle_sample_data():
    import numpy as np

    import oracle
    from exact_attention_52_gb300.inputs import make_inputs, make_inputs_fp8
    inp = make_inputs(1, 1, BF16["N"], BF16["d"], seed=0, with_grad=True,
                      outlier_frac=BF16["outlier_frac"], outlier_factor=BF16["outlier_factor"])
    bf = tuple(oracle.bf16_bits_to_f64(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    f8 = make_inputs_fp8(1, 1, FP8["N"], FP8["d"], seed=0)
    f8v = (oracle.e4m3_to_f64(f8.q8, f8.sq), oracle.e4m3_to_f64(f8.k8, f8.sk),
           oracle.e4m3_to_f64(f8.v8, f8.sv))
    rows = np.linspace(0, FP8["N"] - 1, 256).astype(np.int64)
    return {"bf16": bf, "fp8": f8v, "fp8_rows": rows}


def sample_desc(n_rows):
    return (f"fp64 oracle, explicit S and P rows: forward + backward work of {n_rows} evenly spaced "
            f"query rows of head 0 of the bf16 workload (N=8192, all keys) and 256 evenly spaced "
            f"query rows of head 0 of the FP8 workload")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    data = oracle_sample_data()
    # Size each step so that warm-up + timed steps take about REF_BUDGET_S.
    t0 = time.perf_counter()
    oracle_sample_step(data, 256)
    per_row = max((time.perf_counter() - t0) / 256, 1e-7)
    n_rows = int(min(BF16["N"], max(64, REF_BUDGET_S / (args.steps + args.warmup) / per_row)))
    for _ in range(args.warmup):
        oracle_sample_step(data, n_rows)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(args.steps):
        flops += oracle_sample_step(data, n_rows)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    desc = sample_desc(n_rows)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of per-rank timings (every rank gets the result)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_tflops(flops_per_rank, world, ms_per_step):
    """Weak scaling: every rank processes its own copy of the step's work; the
    job's throughput is the work of all ranks over the slowest rank's time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


def make_device_data(torch, dev):
    import numpy as np

    from exact_attention_52_gb300.inputs import make_inputs, make_inputs_fp8
    inp = make_inputs(BF16["B"], BF16["H"], BF16["N"], BF16["d"], seed=0, with_grad=True,
                      outlier_frac=BF16["outlier_frac"], outlier_factor=BF16["outlier_factor"])

    def host_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    h = {n: host_bf16(getattr(inp, n + "_bits")).pin_memory() for n in ("q", "k", "v", "do")}
    f8 = make_inputs_fp8(FP8["B"], FP8["H"], FP8["N"], FP8["d"], seed=0)
    for n in ("q8", "k8", "v8"):
        h[n] = torch.from_numpy(getattr(f8, n)).pin_memory()
    d = {n: t.to(dev) for n, t in h.items()}
    d["scales"] = (f8.sq, f8.sk, f8.sv)
    return h, d


def live_gemm_peaks(torch, dev, n=8192, reps=10):
    """Dense GEMM throughput of this GPU measured now, for the FP8 roofline
    denominator (no FP8 figure is in the measured-peaks file): cuBLAS through
    torch, best of ``reps`` n^3 products timed with CUDA events, 2*n^3 flops
    each.  bf16 is measured the same way, so that the two share one clock and
    method.  Returns {"fp8_tflops": .., "bf16_tflops": ..} (None where the
    product is not available)."""
    out = {"fp8_tflops": None, "bf16_tflops": None, "n": n, "reps": reps,
           "how": "torch._scaled_mm e4m3 x e4m3 -> bf16 and torch.matmul bf16, "
                  f"{n}^3, best of {reps}, CUDA events"}
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    a = torch.randn((n, n), device=dev, generator=g, dtype=torch.float32)
    b = torch.randn((n, n), device=dev, generator=g, dtype=torch.float32)

    def best(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return 2.0 * n ** 3 / (min(ts) * 1e-3) / 1e12

    try:
        ab, bb = a.to(torch.bfloat16), b.to(torch.bfloat16)
        out["bf16_tflops"] = round(best(lambda: torch.matmul(ab, bb)), 1)
        del ab, bb
    except RuntimeError:
        pass
    try:
        a8 = a.to(torch.float8_e4m3fn)
        b8 = b.to(torch.float8_e4m3fn).t()  # column-major second operand
        one = torch.ones((), device=dev, dtype=torch.float32)
        out["fp8_tflops"] = round(best(lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one,
                                                                out_dtype=torch.bfloat16)), 1)
        del a8, b8
    except (RuntimeError, AttributeError, TypeError):
        pass
    del a, b
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    from exact_attention_52_gb300 import api

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        data = oracle_sample_data()
        n_rows = BF16["N"]  # the whole of head 0 per pass
        # Passes over that sample until about 10 s of host work (at most 8 passes).
        t0 = time.perf_counter()
        f, passes = 0.0, 0
        while passes < 8 and (passes == 0 or time.perf_counter() - t0 < CPU_BASELINE_S):
            f += oracle_sample_step(data, n_rows)
            passes += 1
        dt = time.perf_counter() - t0
        cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": sample_desc(n_rows) + f" ({passes} passes, {dt:.1f} s)"}
        del data

    host, d = make_device_data(torch, dev)
    B, H, N, D = BF16["B"], BF16["H"], BF16["N"], BF16["d"]
    scale = 1.0 / math.sqrt(D)
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(o), torch.empty_like(o), torch.empty_like(o)
    ws = torch.empty(api.bwd_workspace_bytes(B, H, N, D), dtype=torch.uint8, device=dev)
    B8, H8, N8 = FP8["B"], FP8["H"], FP8["N"]
    o8 = torch.empty((B8, H8, N8, FP8["d"]), dtype=torch.bfloat16, device=dev)
    lse8 = torch.empty((B8, H8, N8), dtype=torch.float32, device=dev)
    sq, sk, sv = d["scales"]
    stream = torch.cuda.current_stream()
    KERNELS = ("fwd", "bwd_pre", "bwd_main", "bwd_dq_convert", "fwd_fp8")

    def step(ev=None):
        e = ev or [None] * 8
        if e[0] is not None:
            e[0].record(stream)
        api.fwd(d["q"], d["k"], d["v"], scale=scale, causal=BF16["causal"], o=o, lse=lse)
        api.bwd_stages(d["q"], d["k"], d["v"], o, d["do"], lse, dq, dk, dv, ws, scale,
                       BF16["causal"], events=e[1:5])
        api.fwd_fp8(d["q8"], d["k8"], d["v8"], sq, sk, sv, scale=scale, causal=FP8["causal"],
                    o=o8, lse=lse8)
        if e[5] is not None:
            e[5].record(stream)

    for _ in range(max(args.warmup, 3)):
        step()
    rc, site = api.check_device_error()
    if rc != 0:
        raise RuntimeError(f"device error {rc} at wait site {site:#x}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    rc, site = api.check_device_error()
    if rc != 0:
        raise RuntimeError(f"device error {rc} at wait site {site:#x}")
    elapsed_ms = t_start.elapsed_time(t_end)

    # per-kernel averages from the events inside the timed region
    def avg(a, b):
        return sum(evs[i][a].elapsed_time(evs[i][b]) for i in range(args.steps)) / args.steps
    k_ms = {"fwd": avg(0, 1), "bwd_pre": avg(1, 2), "bwd_main": avg(2, 3),
            "bwd_dq_convert": avg(3, 4), "fwd_fp8": avg(4, 5)}

    # End to end through the public API with host buffers: every step copies its
    # inputs from pinned host memory and reads all of its outputs back.  The copies
    # run on their own streams with double-buffered device tensors, so step k's
    # compute overlaps step k+1's inputs and step k-1's outputs (a pipelined caller);
    # the timed region spans all copies and all compute of the n steps.
    e2e = None
    if not args.no_e2e:
        ins = ("q", "k", "v", "do", "q8", "k8", "v8")
        n_out = 7
        bufs = []
        for bsel in range(2):
            din = {n: (d[n] if bsel == 0 else torch.empty_like(d[n])) for n in ins}
            dout = ([o, lse, dq, dk, dv, o8, lse8] if bsel == 0 else
                    [torch.empty_like(t) for t in (o, lse, dq, dk, dv, o8, lse8)])
            bufs.append((din, dout))
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in bufs[0][1]]
        h2d = sum(host[n].numel() * host[n].element_size() for n in ins)
        d2h = sum(t.numel() * t.element_size() for t in bufs[0][1])
        assert len(bufs[0][1]) == n_out

        def e2e_step(din, dout):
            eo, else_, edq, edk, edv, eo8, else8 = dout
            api.fwd(din["q"], din["k"], din["v"], scale=scale, causal=BF16["causal"], o=eo, lse=else_)
            api.bwd_stages(din["q"], din["k"], din["v"], eo, din["do"], else_, edq, edk, edv, ws,
                           scale, BF16["causal"])
            api.fwd_fp8(din["q8"], din["k8"], din["v8"], sq, sk, sv, scale=scale,
                        causal=FP8["causal"], o=eo8, lse=else8)

        # The first copy-in and the last copy-out overlap no compute (about 3.5 ms
        # together); 100 steps spread them to about 1 % of a step (20 steps would
        # leave 5 %), whatever the number of device-timed steps.
        n_e2e = args.e2e_steps
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(n_e2e)]
        ev_comp = [torch.cuda.Event() for _ in range(n_e2e)]
        ev_out = [torch.cuda.Event() for _ in range(n_e2e)]
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_event(a)
        s_out.wait_event(a)
        for k in range(n_e2e):
            din, dout = bufs[k % 2]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev_comp[k - 2])  # step k-2 has finished reading this buffer
                for n in ins:
                    din[n].copy_(host[n], non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if k >= 2:
                stream.wait_event(ev_out[k - 2])  # step k-2's outputs have been read back
            e2e_step(din, dout)
            ev_comp[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[k])
                for hb, t in zip(host_out, dout):
                    hb.copy_(t, non_blocking=True)
                ev_out[k].record(s_out)
        stream.wait_event(ev_out[n_e2e - 1])
        b.record(stream)
        torch.cuda.synchronize()
        rc, site = api.check_device_error()
        if rc != 0:
            raise RuntimeError(f"device error {rc} at wait site {site:#x}")
        e2e_ms = a.elapsed_time(b) / n_e2e
        e2e = {"h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pipelined": "inputs, compute and outputs of consecutive steps overlap on three streams",
               "steps": n_e2e}

    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e["ms_per_step"] if e2e else 0.0], dist,
                                        dev)
    if e2e:
        e2e["ms_per_step"] = e2e_ms
    flops = step_flops()
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tflops(sum(flops.values()), world, ms_per_step)
    total_flops = sum(flops.values()) * world

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peaks, peak_kind = load_peaks()
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # The timed region lasts tens of milliseconds at the SM clock sampled above:
    # the burst figure (a GEMM timed alone, best of 10) is the denominator; the
    # sustained one (seconds under the power cap, at a lower clock) is reported
    # beside it, labelled.
    sm_mhz = clk["sm_mhz"] if clk else None
    live = live_gemm_peaks(torch, dev) if not args.no_live_peaks else {}
    fp8_peak = live.get("fp8_tflops")
    fp8_kind = "measured live in this run (cuBLAS e4m3 GEMM)"
    if not fp8_peak:
        fp8_peak = 2.0 * burst
        fp8_kind = f"2 x {peak_kind} bf16 burst (nominal dense FP8/bf16 ratio)"
    bwd_main_flops = flops["bwd"]
    achieved = bwd_main_flops / (k_ms["bwd_main"] * 1e-3) / 1e12
    traffic = recorded_traffic("bwd_main_b1_h32_n8192_d128")
    components = {}
    for name, f, kms in (("fwd", flops["fwd"], k_ms["fwd"]),
                         ("bwd", flops["bwd"], k_ms["bwd_pre"] + k_ms["bwd_main"] + k_ms["bwd_dq_convert"]),
                         ("bwd_main", flops["bwd"], k_ms["bwd_main"]),
                         ("fwd_fp8", flops["fwd_fp8"], k_ms["fwd_fp8"])):
        tf = f / (kms * 1e-3) / 1e12
        if name == "fwd_fp8":
            c = {"ms": round(kms, 4), "tflops": round(tf, 1), "frac_of_peak": round(tf / fp8_peak, 4),
                 "peak_tflops": fp8_peak, "peak_kind": fp8_kind,
                 "frac_of_2x_bf16_burst": round(tf / (2.0 * burst), 4)}
        else:
            c = {"ms": round(kms, 4), "tflops": round(tf, 1), "frac_of_burst": round(tf / burst, 4),
                 "frac_of_sustained": round(tf / sustained, 4)}
        if sm_mhz:
            c["mcycles_at_median_sm_clock"] = round(kms * sm_mhz * 1e-3, 4)
        components[name] = c
    secondary = {}
    if world == 1 and not args.no_secondary:
        for nm in ("c1_fwd_b1_h1_n128_d64", "c2_fwd_b4_h16_n1024_d64", "c3_causal_b2_h16_n4096_d128"):
            secondary[nm] = measure_workload(nm, steps=20)[0]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "inputs 0.54 GB > 129 MB L2, no flush",
                   "parallelism": f"replicas x{world} (independent heads, no collective)"},
        "components": components,
        "secondary": secondary or None,
        "kernel_ms": {k: round(v, 4) for k, v in k_ms.items()},
        "roofline": {"kernel": "bwd_main (attn_bwd_main)", "bound": "tensor",
                     "achieved": round(achieved, 1), "peak": burst, "unit": "TFLOP/s",
                     "frac": round(achieved / burst, 4),
                     "peak_kind": f"{peak_kind} bf16 burst (GEMM timed alone; the timed region "
                                  f"is {elapsed_ms:.0f} ms at the sampled clock)",
                     "frac_of_sustained": round(achieved / sustained, 4),
                     "sustained_peak": sustained,
                     "traffic": traffic,
                     "algorithmic_bytes": attn_bytes(B, H, N, D, "bwd_main")},
        "live_gemm_peaks": live or None,
        "gpu_launches": len(KERNELS) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "e2e": None if e2e is None else {
            "value": round(total_flops / (e2e["ms_per_step"] * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
            "d2h_bytes_per_step": e2e["d2h_bytes_per_step"],
            "ms_per_step": round(e2e["ms_per_step"], 4), "pipelined": e2e["pipelined"],
            "steps": e2e["steps"]},
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


EXTRA_WORKLOADS = {
    # grouped-query attention, 4 query heads per key/value head
    "gqa_b1_h32_hk8_n8192_d128": dict(B=1, H=32, Hk=8, N=8192, d=128, causal=False),
    "gqa_causal_b2_h32_hk4_n4096_d128": dict(B=2, H=32, Hk=4, N=4096, d=128, causal=True),
    "mqa_b4_h16_hk1_n4096_d128": dict(B=4, H=16, Hk=1, N=4096, d=128, causal=False),
    # causal with one key/value head: key-tile items of up to 16 x 32 steps for 128
    # items, fewer than the CTAs (the backward deals the longest as two parts)
    "mqa_causal_b4_h16_hk1_n4096_d128": dict(B=4, H=16, Hk=1, N=4096, d=128, causal=True),
    # causal with a large batch: 512 MB of Q, dO and fp32 dQ accumulator (the backward
    # deals its key tiles in groups of heads so that the heads in flight stay in L2)
    "causal_b4_h32_n4096_d128": dict(B=4, H=32, Hk=32, N=4096, d=128, causal=True),
    # sliding window of 1024 keys to the left (and the query itself)
    "window1024_b1_h32_n8192_d128": dict(B=1, H=32, Hk=32, N=8192, d=128, causal=False,
                                         window=(1024, 0)),
    # one head, long sequence (64 CTAs without splitting): key tiles split across CTAs
    "splitkv_b1_h1_n16384_d128": dict(B=1, H=1, Hk=1, N=16384, d=128, causal=False, splitkv=True),
    # the small configurations of the parity suite: one CTA (latency), a d = 64 case
    # near the ridge point, and causal d = 128 forward + backward
    "c1_fwd_b1_h1_n128_d64": dict(B=1, H=1, Hk=1, N=128, d=64, causal=False, fwd_only=True),
    "c2_fwd_b4_h16_n1024_d64": dict(B=4, H=16, Hk=16, N=1024, d=64, causal=False, fwd_only=True),
    "c3_causal_b2_h16_n4096_d128": dict(B=2, H=16, Hk=16, N=4096, d=128, causal=True),
    # the FP8 forward of the step with one group of exponentials in eight on the FMA pipe
    "fp8_exp2_offload_b1_h16_n16384_d128_causal": dict(fp8=True),
}


def window_flops(N, d, left, right):
    """Multiply-add work of the visible (query, key) pairs, 4*d per pair."""
    import numpy as np
    i = np.arange(N)
    lo = np.zeros(N) if left < 0 else np.maximum(0, i - left)
    hi = np.full(N, N - 1) if right < 0 else np.minimum(N - 1, i + right)
    return 4.0 * d * float(np.sum(hi - lo + 1))


def measure_workload(name, steps=20, flush_bytes=512 << 20):
    """Forward (+ backward) of one of EXTRA_WORKLOADS on the current GPU.

    Device time per call between CUDA events on the launching stream, with a
    write of ``flush_bytes`` (more than the 129 MB L2) before every timed call
    so that each call reads its inputs from HBM.  Forward-only workloads also
    report the time per call of back-to-back calls (host-side argument checks
    and tensor-map encoding included) and per call replayed from a CUDA graph.
    Returns a dict of components."""
    import numpy as np
    import torch

    from exact_attention_52_gb300 import api
    from exact_attention_52_gb300.inputs import make_inputs_gqa

    w = EXTRA_WORKLOADS[name]
    B, H, Hk, N, D, causal = w["B"], w["H"], w["Hk"], w["N"], w["d"], w["causal"]
    inp = make_inputs_gqa(B, H, Hk, N, D, seed=0, with_grad=True)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v, do = (dev(x) for x in (inp.q_bits, inp.k_bits, inp.v_bits, inp.do_bits))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(api.bwd_workspace_bytes(B, H, N, D), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device="cuda")
    window = w.get("window")
    ws_split = None
    if w.get("splitkv"):
        ws_split = torch.empty(api.load_library().attn_fwd_splitkv_workspace_bytes(B, H, N, D, 0),
                               dtype=torch.uint8, device="cuda")

    def fwd_call():
        if window is not None:
            api.fwd_window(q, k, v, *window, o=o, lse=lse)
        elif ws_split is not None:
            api.fwd_splitkv(q, k, v, num_splits=0, causal=causal, o=o, lse=lse, workspace=ws_split)
        else:
            api.fwd(q, k, v, causal=causal, o=o, lse=lse)

    def second_call():
        if w.get("fwd_only"):
            return
        if window is not None:
            api.bwd_window(q, k, v, o, do, lse, *window, dq=dq, dk=dk, dv=dv, workspace=ws)
        elif ws_split is not None:
            api.fwd(q, k, v, causal=causal, o=o, lse=lse)  # single-pass forward, for comparison
        else:
            api.bwd(q, k, v, o, do, lse, causal=causal, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(3):
        fwd_call()
        second_call()
    torch.cuda.synchronize()
    t_f, t_s = [], []
    for _ in range(steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        fwd_call()
        e[1].record(stream)
        if not w.get("fwd_only"):
            flush.zero_()
            e[2].record(stream)
            second_call()
            e[3].record(stream)
        torch.cuda.synchronize()
        t_f.append(e[0].elapsed_time(e[1]))
        if not w.get("fwd_only"):
            t_s.append(e[2].elapsed_time(e[3]))
    rc, site = api.check_device_error()
    if rc != 0:
        raise RuntimeError(f"device error {rc} at wait site {site:#x}")
    fwd_ms = statistics.median(t_f)
    f = attn_flops(B, H, N, D, causal)
    if window is not None:
        f = B * H * window_flops(N, D, *window)
    peaks, kind = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tf = f / (fwd_ms * 1e-3) / 1e12
    comp = {"fwd": {"ms": round(fwd_ms, 5), "tflops": round(tf, 1),
                    "frac_of_burst": round(tf / burst, 4)}}
    if w.get("fwd_only"):
        nbytes = attn_bytes(B, H, N, D, "fwd")
        comp["fwd"]["us"] = round(fwd_ms * 1e3, 2)
        comp["fwd"]["gbs"] = round(nbytes / (fwd_ms * 1e-3) / 1e9, 1)
        comp["fwd"]["frac_of_hbm"] = round(nbytes / (fwd_ms * 1e-3) / 1e9 /
                                           float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])), 4)
        # back to back (host path included) and replayed from a CUDA graph (inputs in L2)
        n_bb = 50
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(n_bb):
            fwd_call()
        b1.record(stream)
        torch.cuda.synchronize()
        comp["fwd_back_to_back"] = {"us": round(b0.elapsed_time(b1) / n_bb * 1e3, 2), "calls": n_bb}
        per_graph, replays = 20, 50
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                fwd_call()
        graph.replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(replays):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        rc, site = api.check_device_error()
        if rc != 0:
            raise RuntimeError(f"device error {rc} at wait site {site:#x}")
        graph_ms = g0.elapsed_time(g1) / (replays * per_graph)
        comp["fwd_graph_replay"] = {"us": round(graph_ms * 1e3, 2),
                                    "tflops": round(f / (graph_ms * 1e-3) / 1e12, 1),
                                    "gbs": round(nbytes / (graph_ms * 1e-3) / 1e9, 1),
                                    "calls_per_graph": per_graph, "replays": replays}
    elif ws_split is not None:
        s_ms = statistics.median(t_s)
        comp = {"fwd_splitkv": comp["fwd"],
                "fwd_single_pass": {"ms": round(s_ms, 5), "tflops": round(f / (s_ms * 1e-3) / 1e12, 1)}}
    else:
        b_ms = statistics.median(t_s)
        tb = 2.5 * f / (b_ms * 1e-3) / 1e12
        comp["bwd"] = {"ms": round(b_ms, 5), "tflops": round(tb, 1), "frac_of_burst": round(tb / burst, 4)}
    del flush
    torch.cuda.empty_cache()
    return comp, f, kind


def run_fp8_exp2_offload(args):
    """FP8 forward of the benchmark step with and without the exponential
    offload (attn_set_exp2_offload): median device time per call, L2 flushed
    before each call."""
    import torch

    from exact_attention_52_gb300 import api
    from exact_attention_52_gb300.inputs import make_inputs_fp8
    torch.cuda.set_device(0)
    f8 = make_inputs_fp8(FP8["B"], FP8["H"], FP8["N"], FP8["d"], seed=0)
    q8, k8, v8 = (torch.from_numpy(getattr(f8, n)).cuda() for n in ("q8", "k8", "v8"))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    f = attn_flops(FP8["B"], FP8["H"], FP8["N"], FP8["d"], FP8["causal"])
    comp = {}
    for on in (False, True):
        api.set_exp2_offload(on)
        for _ in range(3):
            api.fwd_fp8(q8, k8, v8, f8.sq, f8.sk, f8.sv, causal=FP8["causal"])
        ts = []
        for _ in range(min(args.steps, 50)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            api.fwd_fp8(q8, k8, v8, f8.sq, f8.sk, f8.sv, causal=FP8["causal"])
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = statistics.median(ts)
        comp["exp2_offload" if on else "mufu_only"] = {"ms": round(ms, 5),
                                                       "tflops": round(f / (ms * 1e-3) / 1e12, 1)}
    api.set_exp2_offload(False)
    rc, site = api.check_device_error()
    if rc != 0:
        raise RuntimeError(f"device error {rc} at wait site {site:#x}")
    print(json.dumps({"metric": METRIC, "workload": args.workload, "config": FP8, "unit": "TFLOP/s",
                      "value": comp["exp2_offload"]["tflops"], "components": comp,
                      "timing": "median device time per call, L2 flushed before each call",
                      "dtype": "e4m3", "data": "synthetic"}), flush=True)
    return 0


def run_extra(args):
    """Forward (+ backward) on one of EXTRA_WORKLOADS: a secondary line; the
    default run measures the benchmark step."""
    import torch
    if args.workload == "fp8_exp2_offload_b1_h16_n16384_d128_causal":
        return run_fp8_exp2_offload(args)
    torch.cuda.set_device(0)
    comp, f, kind = measure_workload(args.workload, steps=min(args.steps, 50))
    main_ms = comp.get("fwd", comp.get("fwd_splitkv"))["ms"] + comp.get("bwd", {}).get("ms", 0.0)
    mult = 3.5 if "bwd" in comp else 1.0
    line = {"metric": METRIC, "workload": args.workload, "config": EXTRA_WORKLOADS[args.workload],
            "steps": min(args.steps, 50), "unit": "TFLOP/s",
            "value": round(mult * f / (main_ms * 1e-3) / 1e12, 2), "components": comp,
            "timing": "median device time per call between CUDA events, L2 flushed before each call",
            "peak_kind": kind, "dtype": "bf16", "data": "synthetic"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (used for profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end loop")
    ap.add_argument("--e2e-steps", type=int, default=100,
                    help="pipelined steps of the end-to-end loop (at least 2)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the small-configuration lines (C1-C3) after the timed region")
    ap.add_argument("--no-live-peaks", action="store_true",
                    help="skip the live cuBLAS GEMM peaks (FP8 roofline denominator)")
    ap.add_argument("--workload", choices=("main",) + tuple(EXTRA_WORKLOADS), default="main",
                    help="secondary workloads print their own line (not the benchmark step)")
    args = ap.parse_args()
    args.e2e_steps = max(2, args.e2e_steps)
    if args.workload != "main" and args.impl == "ours":
        return run_extra(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
