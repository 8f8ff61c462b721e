"""Benchmark of the B300 selective scan: one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one selective_scan_fwd over one batch of synthetic, seeded inputs of
the workload (default: one Mamba-130M-shaped layer, batch 8, d_inner 1536,
d_state 16, L 2048, bf16 I/O, fp32 state).  Inputs are resident in HBM; the
step rotates over enough copies of them that the data one step reads exceeds
the 126 MB L2, so no step finds the previous step's bytes in cache.

Reported:
  value       algorithmic HBM GB/s over all ranks (metric of the workload)
  roofline    the scan kernel against the slower of HBM bytes at the measured
              copy bandwidth and B*D*L*N exps at the MUFU ex2 peak
  e2e         the same metric through the C-ABI call with pinned host buffers,
              host->device inputs and device->host outputs inside the timed region
  cpu_baseline the float64 oracle on the host cores (a bounded sample)
Under torchrun every rank runs its own replica (weak scaling); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_148_b300 import inputs  # noqa: E402

METRIC = "selective_scan_fwd achieved HBM GB/s (% of peak) and (B·L) tokens/s per layer"
DEFAULT_WORKLOAD = "mamba130m_b8_d1536_n16_l2048_bf16"
L2_BYTES = 126 * 1024 * 1024
SM_COUNT_NOMINAL = 148
SM_MAX_MHZ_NOMINAL = 2032.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=float(d["hbm_gbs"]), source="measured", sm_max_mhz=float(d.get("sm_max_mhz", 2032.0)))
    return dict(hbm_gbs=6400.0, source="fallback", sm_max_mhz=SM_MAX_MHZ_NOMINAL)


def io_bytes(io):
    return 2 if io == "bf16" else 4


def scan_bytes(Bsz, Dch, L, N, io, with_z=True):
    """Algorithmic bytes of one scan: u, delta, (z) in, y out, B and C, A, D, bias, last_state."""
    s = io_bytes(io)
    return ((3 if with_z else 2) + 1) * Bsz * Dch * L * s + 2 * Bsz * N * L * s + Dch * N * 4 + 2 * Dch * 4 \
        + Bsz * Dch * N * 4


def step_bytes(Bsz, Dch, N, io):
    """Algorithmic bytes of one decode step: state in and out, u/delta/z in, y out, B, C, A, D, bias."""
    s = io_bytes(io)
    return 2 * Bsz * Dch * N * 4 + 4 * Bsz * Dch * s + 2 * Bsz * N * s + Dch * N * 4 + 2 * Dch * 4


# ----------------------------------------------------------------------------- clocks during the timed region

class _Nvml:
    """Minimal ctypes binding of libnvidia-ml (SM clock, max clock, clock-event reasons)."""
    CLOCK_SM = 1

    def __init__(self, pci_bus_id):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) != 0:
            if self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
                raise RuntimeError("no NVML device handle")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def sm_clock(self):
        v = self.ct.c_uint()
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.ct.byref(v)) == 0 else None

    def max_sm_clock(self):
        v = self.ct.c_uint()
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.ct.byref(v)) == 0 else None

    def reasons(self):
        v = self.ct.c_ulonglong()
        return v.value if self._reasons(self.h, self.ct.byref(v)) == 0 else 0


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons while the timed region runs."""

    REASONS = {
        0x0000000000000008: "hw_slowdown", 0x0000000000000020: "sw_thermal_slowdown",
        0x0000000000000040: "hw_thermal_slowdown", 0x0000000000000004: "sw_power_cap",
        0x0000000000000080: "hw_power_brake_slowdown", 0x0000000000000002: "applications_clocks_setting",
    }

    def __init__(self, pci_bus_id):
        self.samples, self.reasons, self.max_mhz, self.source = [], set(), None, None
        self._stop = threading.Event()
        self._t = None
        try:
            self.nvml = _Nvml(pci_bus_id)
            self.max_mhz = self.nvml.max_sm_clock()
            self.source = "nvml"
        except Exception as e:  # noqa: BLE001
            self.nvml = None
            self.error = str(e)

    def _sample(self):
        c = self.nvml.sm_clock()
        if c is not None:
            self.samples.append(c)
        r = self.nvml.reasons()
        for bit, name in self.REASONS.items():
            if r & bit:
                self.reasons.add(name)

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(0.001)

    def __enter__(self):
        if self.nvml is not None:
            self._sample()  # at least one sample at each end of a short timed region
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t is not None:
            self._t.join()
            self._sample()

    def summary(self):
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
               "reasons": sorted(self.reasons), "samples": len(self.samples), "source": self.source}
        if self.nvml is None:
            out["error"] = getattr(self, "error", "unavailable")
        return out


def pci_bus_id(torch):
    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    return f"{getattr(p, 'pci_domain_id', 0):08x}:{getattr(p, 'pci_bus_id', 0):02x}:{getattr(p, 'pci_device_id', 0):02x}.0"


# ----------------------------------------------------------------------------- MUFU peak

def mufu_ex2_per_clk_per_sm(m, torch):
    """ex2 per SM per clock from the MUFU microbenchmark (all SMs, 2048 threads each)."""
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    sms = props.multi_processor_count
    blocks, threads, iters = sms * 8, 256, 4096
    cycles = torch.zeros(blocks, dtype=torch.int64, device="cuda")
    sink = torch.empty(blocks * threads, dtype=torch.float32, device="cuda")
    for _ in range(2):
        m.mamba_bench_ex2(cycles, sink, iters, blocks, threads)
    torch.cuda.synchronize()
    cyc = int(cycles.max().item())
    total = blocks * threads * iters * 8
    return total / (sms * cyc), sms


# ----------------------------------------------------------------------------- oracle (CPU) timing

def time_oracle(x, budget_s=12.0):
    """Oracle over whole time rows of a growing subset of channels; returns (bytes/s, updates/s, info)."""
    import oracle
    Bsz, Dch, L, N = x.shape
    threads = oracle.num_threads()
    chans_total = Bsz * Dch

    def run(nch):
        b_idx = [c // Dch for c in range(nch)]
        d_idx = [c % Dch for c in range(nch)]
        # group by batch so each oracle call sees one batch's B and C
        t_cpu = 0.0
        for b in sorted(set(b_idx)):
            ds = [d for bb, d in zip(b_idx, d_idx) if bb == b]
            lo, hi = min(ds), max(ds) + 1
            sl = lambda a: inputs.to_f64(a[b:b + 1, lo:hi], x.io)
            args = (sl(x.u), sl(x.delta), x.A[lo:hi].astype(np.float64), inputs.to_f64(x.B[b:b + 1], x.io),
                    inputs.to_f64(x.C[b:b + 1], x.io), x.D[lo:hi].astype(np.float64), sl(x.z),
                    x.delta_bias[lo:hi].astype(np.float64))
            t0 = time.perf_counter()
            oracle.selective_scan(*args)
            t_cpu += time.perf_counter() - t0
        return t_cpu

    nch = min(chans_total, max(1, threads))
    t = run(nch)
    while t < budget_s / 4 and nch < chans_total:
        nch = min(chans_total, int(nch * max(2.0, min(8.0, budget_s / 4 / max(t, 1e-3)))))
        t = run(nch)
    frac = nch / chans_total
    bytes_s = scan_bytes(Bsz, Dch, L, N, x.io) * frac / t
    return bytes_s, nch * N * L / t, dict(channels=nch, of=chans_total, seconds=t, threads=threads)


def time_oracle_threads(x, threads, budget_s=8.0):
    """time_oracle with the oracle limited to `threads` host threads."""
    import oracle
    n0 = oracle.num_threads()
    oracle.set_num_threads(threads)
    try:
        return time_oracle(x, budget_s=budget_s)
    finally:
        oracle.set_num_threads(n0)


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(inputs.WORKLOADS) + [inputs.DECODE_WORKLOAD["name"]])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the headline workload (by default a run of the default workload at N=1 also "
                         "times every other workload into the line's 'workloads' object)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass of the scan (gradients of sum(dy * y)) on the workload")
    ap.add_argument("--flags", default="none", choices=["none", "zoh", "reverse", "zoh+reverse"],
                    help="scan flags: the exact zero-order hold and/or the reverse-time scan")
    ap.add_argument("--conv", default="none", choices=["none", "fused", "two-step"],
                    help="feed the scan through the depthwise causal conv1d + SiLU branch: fused into the scan "
                         "kernel, or as a separate convolution launch before the scan")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    import selective_state_space_148_b300 as m
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    m.lib()

    decode = args.workload == inputs.DECODE_WORKLOAD["name"]
    if decode:
        res = bench_decode(args, m, torch)
    elif args.backward:
        res = bench_backward(args, m, torch)
    else:
        res = bench_scan(args, m, torch)

    extra = None
    if world == 1 and not decode and not args.backward and args.conv == "none" and \
            args.workload == DEFAULT_WORKLOAD and not args.no_workloads:
        torch.cuda.empty_cache()
        extra = other_workloads(args, m, torch)

    # max over ranks of the timed regions; every rank ran the same per-rank workload (weak scaling)
    t_ms, res["e2e_ms"] = max_over_ranks([res["ms_per_step"], res["e2e_ms"]], dist, torch, "cuda")
    value, e2e_value = aggregate_gbs(world, res["bytes"], t_ms, res["e2e_ms"])
    peaks = measured_peaks()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not decode and args.conv == "none" and \
            not args.backward:
        bps, ups, info = time_oracle(res["inputs"])
        cpu = {"value": bps / 1e9, "unit": "GB/s", "cores": info["threads"], "kind": "oracle",
               "sample": f"float64 oracle over whole time rows of {info['channels']} of {info['of']} channels "
                         f"of {args.workload} ({info['seconds']:.1f} s); value scaled to the workload's bytes",
               "updates_per_s": ups}
        bps1, ups1, info1 = time_oracle_threads(res["inputs"], 1, budget_s=8.0)
        cpu["single_thread"] = {
            "value": bps1 / 1e9, "unit": "GB/s", "cores": 1, "updates_per_s": ups1,
            "sample": f"the same oracle on one thread: whole time rows of {info1['channels']} channels "
                      f"({info1['seconds']:.1f} s)"}

    if rank == 0:
        line = {
            "metric": ("selective_state_update achieved HBM GB/s and tokens/s" if decode else
                       "selective_scan_bwd algorithmic HBM GB/s and (B·L) tokens/s per layer" if args.backward
                       else METRIC),
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_ms, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": res["dtype"], "data": "synthetic",
            "config": res["config"],
            "pct_of_hbm_peak": round(100.0 * value / world / peaks["hbm_gbs"], 2),
            "tokens_per_s": round(world * res["tokens"] / (t_ms * 1e-3), 1),
            "roofline": res["roofline"],
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 3), "unit": "GB/s", "h2d_bytes_per_step": res["h2d"],
                    "d2h_bytes_per_step": res["d2h"], "ms_per_step": round(res["e2e_ms"], 4),
                    "tokens_per_s": round(world * res["tokens"] / (res["e2e_ms"] * 1e-3), 1)},
            "gpu_launches": res["launches"],
            "clocks": res["clocks"],
            "mufu": res.get("mufu"),
        }
        if res.get("chained") is not None:
            line["chained"] = res["chained"]
        if res.get("training_pair") is not None:
            line["training_pair"] = res["training_pair"]
        if extra is not None:
            line["workloads"] = extra
        print(json.dumps(line))
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# the other workloads timed into the default run's 'workloads' object: name -> timed steps
OTHER_SCAN_WORKLOADS = {"mamba2p8b_b4_d5120_n16_l4096_bf16": 40, "mamba2p8b_b4_d5120_n64_l4096_bf16": 12,
                        "dna_b1_d1536_n16_l1048576_bf16": 5}


def workload_entry(res):
    """The per-workload summary kept in the 'workloads' object."""
    t = res["ms_per_step"]
    e = {"ms_per_step": round(t, 6), "value": round(res["bytes"] / (t * 1e-3) / 1e9, 2), "unit": "GB/s",
         "tokens_per_s": round(res["tokens"] / (t * 1e-3), 1), "steps": res.get("steps"),
         "roofline": res["roofline"], "clocks": res["clocks"], "config": res["config"],
         "gpu_launches": res["launches"]}
    if res.get("chained") is not None:
        e["chained"] = res["chained"]
    if res.get("training_pair") is not None:
        e["training_pair"] = res["training_pair"]
    return e


def other_workloads(args, m, torch):
    """Every other workload of the benchmark, each timed in this run with its own clock record."""
    out = {}
    for name, k in OTHER_SCAN_WORKLOADS.items():
        r = bench_scan(args, m, torch, workload=name, steps=k, e2e=False, conv="none", flag_name="none")
        r["steps"] = k
        out[name] = workload_entry(r)
        del r
        torch.cuda.empty_cache()
    r = bench_decode(args, m, torch, steps=inputs.DECODE_WORKLOAD["steps"], e2e=False)
    r["steps"] = inputs.DECODE_WORKLOAD["steps"]
    out[inputs.DECODE_WORKLOAD["name"]] = workload_entry(r)
    torch.cuda.empty_cache()
    r = bench_scan(args, m, torch, workload=DEFAULT_WORKLOAD, steps=100, e2e=False, conv="fused")
    r["steps"] = 100
    out[DEFAULT_WORKLOAD + "+conv_fused"] = workload_entry(r)
    torch.cuda.empty_cache()
    for fl in ("zoh", "reverse"):
        r = bench_scan(args, m, torch, workload=DEFAULT_WORKLOAD, steps=100, e2e=False, conv="none", flag_name=fl)
        r["steps"] = 100
        out[DEFAULT_WORKLOAD + "+" + fl] = workload_entry(r)
        torch.cuda.empty_cache()
    r = bench_backward(args, m, torch, workload=DEFAULT_WORKLOAD, steps=20, e2e=False)
    r["steps"] = 20
    out[DEFAULT_WORKLOAD + "+backward"] = workload_entry(r)
    torch.cuda.empty_cache()
    return out


def pipelined_e2e(torch, steps, upload, compute, download, nbuf=2):
    """Time `steps` end-to-end steps (ms per step): step i uploads its inputs from pinned host memory into
    device buffer set i % nbuf, computes, and downloads its results, on three streams so that the upload of
    step i+1 and the download of step i-1 overlap the compute of step i.  Every step still moves all of its
    bytes inside the timed region.  upload/compute/download(k, stream) enqueue work for buffer set k."""
    main = torch.cuda.current_stream()
    up, comp, down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {n: [torch.cuda.Event() for _ in range(nbuf)] for n in ("up", "comp", "down")}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(main)
    for st in (up, comp, down):
        st.wait_stream(main)
    for i in range(steps):
        k = i % nbuf
        with torch.cuda.stream(up):
            if i >= nbuf:
                up.wait_event(ev["comp"][k])          # the compute that read buffer set k is done
            upload(k, up)
            ev["up"][k].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(ev["up"][k])
            if i >= nbuf:
                comp.wait_event(ev["down"][k])        # the results in buffer set k have been read back
            compute(k, comp)
            ev["comp"][k].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev["comp"][k])
            download(k, down)
            ev["down"][k].record(down)
    for st in (up, comp, down):
        main.wait_stream(st)
    t1.record(main)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def max_over_ranks(values, dist, torch, device):
    """Element-wise maximum over all ranks (the identity without a process group)."""
    if dist is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def aggregate_gbs(world, bytes_per_rank_step, t_ms, e2e_ms):
    """Whole-job GB/s: every rank moves bytes_per_rank_step per step; the slowest rank sets the time."""
    return (world * bytes_per_rank_step / (t_ms * 1e-3) / 1e9, world * bytes_per_rank_step / (e2e_ms * 1e-3) / 1e9)


def traffic_record(kernel_key, sources=None, kernel=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source
    (and, when `kernel` is given, on that kernel instantiation)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel_key)
    if not rec:
        return None
    if rec.get("source_sha") != kernel_source_sha(sources or SCAN_KERNEL_SOURCES):
        return None
    if kernel is not None and rec.get("kernel") != kernel:
        return None
    return rec.get("dram_bytes_per_launch")


# the sources a kernel is built from (a change to any of them voids its stored ncu record)
SCAN_KERNEL_SOURCES = ("scan_tm.cuh", "scan_tm.cu", "tcgen05.cuh", "common.cuh", "scan_kernels.cuh", "scan_fwd.cu",
                       "internal.h")
DECODE_KERNEL_SOURCES = ("state_update.cu", "common.cuh", "internal.h")


def kernel_source_sha(sources=SCAN_KERNEL_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_148_b300", "csrc")
    for f in sources:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


FLAG_BITS = {"none": 0, "zoh": 1, "reverse": 2, "zoh+reverse": 3}


def bench_scan(args, m, torch, workload=None, steps=None, e2e=True, conv=None, flag_name=None):
    workload = workload or args.workload
    steps = steps or args.steps
    conv = args.conv if conv is None else conv
    flag_name = (args.flags if flag_name is None else flag_name) if conv == "none" else "none"
    flags = FLAG_BITS[flag_name]
    x = inputs.make_workload(workload)
    Bsz, Dch, L, N = x.shape
    io = x.io
    tdt = torch.bfloat16 if io == "bf16" else torch.float32
    dev = torch.device("cuda")

    def d(a):
        if io == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    base = dict(u=d(x.u), delta=d(x.delta), z=d(x.z), B=d(x.B), C=d(x.C))
    A = torch.from_numpy(x.A).to(dev)
    D = torch.from_numpy(x.D).to(dev)
    bias = torch.from_numpy(x.delta_bias).to(dev)
    nbytes = scan_bytes(Bsz, Dch, L, N, io)
    R = max(2, math.ceil(3 * L2_BYTES / nbytes))           # rotation copies: > 3x L2 between reuses
    sets = [base] + [{k: v.clone() for k, v in base.items()} for _ in range(R - 1)]
    ys = [torch.empty_like(base["u"]) for _ in range(R)]
    hs = [torch.empty((Bsz, Dch, N), dtype=torch.float32, device=dev) for _ in range(R)]
    ws_bytes = m.mamba_scan_workspace_size(Bsz, Dch, L, N, 0, m.MAMBA_BF16 if io == "bf16" else m.MAMBA_F32)
    chunked = ws_bytes > 0
    stream = torch.cuda.current_stream()
    if conv != "none":   # s["u"] then holds x, the convolution's input
        cw, cb = (torch.from_numpy(a).to(dev) for a in inputs.conv_params(Dch, 7))
        u_tmp = torch.empty_like(base["u"])

    def run(s, y, h, st=None, ut=None):
        st = stream if st is None else st
        ut = u_tmp if ut is None and conv == "two-step" else ut
        if conv == "fused":
            m.mamba_selective_scan_fwd_conv(s["u"], cw, cb, s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, y, h,
                                            stream=st)
        elif conv == "two-step":
            m.mamba_causal_conv1d_silu(s["u"], cw, cb, 1, ut, stream=st)
            m.mamba_selective_scan_fwd(ut, s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, y, h, stream=st)
        elif flags:
            m.mamba_selective_scan_fwd_ex(s["u"], s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, y, h,
                                          flags=flags, stream=st)
        else:
            m.mamba_selective_scan_fwd(s["u"], s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, y, h, stream=st)

    def step(i):
        run(sets[i % R], ys[i % R], hs[i % R])

    mufu_per_clk, sms = mufu_ex2_per_clk_per_sm(m, torch)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(pci_bus_id(torch)) as cs:
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    t_ms = ev0.elapsed_time(ev1) / steps
    clocks = cs.summary()

    # end to end through the C ABI from pinned host buffers (uploads and downloads overlap the neighbouring
    # steps' kernels; two device buffer sets)
    e2e_ms, h2d, d2h = None, None, None
    if e2e:
        e2e_ms, h2d, d2h = scan_e2e(args, torch, base, sets, ys, hs, run, conv, tdt, Bsz, Dch, N)
    return scan_result(args, m, torch, x, workload, steps, conv, t_ms, clocks, chunked, nbytes, R, e2e_ms, h2d, d2h,
                       mufu_per_clk, sms, flag_name)


def scan_e2e(args, torch, base, sets, ys, hs, run, conv, tdt, Bsz, Dch, N):
    hsrc = {k: v.cpu().pin_memory() for k, v in base.items()}
    hy = [torch.empty(base["u"].shape, dtype=tdt).pin_memory() for _ in range(2)]
    hh = [torch.empty((Bsz, Dch, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    dsets = [sets[0], sets[1]]
    utmp = [torch.empty_like(base["u"]) for _ in range(2)] if conv == "two-step" else [None, None]

    def upload(k, st):
        for n in dsets[k]:
            dsets[k][n].copy_(hsrc[n], non_blocking=True)

    def compute(k, st):
        run(dsets[k], ys[k], hs[k], st=st, ut=utmp[k])

    def download(k, st):
        hy[k].copy_(ys[k], non_blocking=True)
        hh[k].copy_(hs[k], non_blocking=True)

    pipelined_e2e(torch, 3, upload, compute, download)   # warm-up
    e2e_ms = pipelined_e2e(torch, args.e2e_steps, upload, compute, download)
    h2d = sum(v.numel() * v.element_size() for v in hsrc.values())
    d2h = hy[0].numel() * hy[0].element_size() + hh[0].numel() * hh[0].element_size()
    return e2e_ms, h2d, d2h


def lean_warps(Bsz, Dch, S, sms):
    """The compute warps of the lean tensor-memory kernel for a plain direct bf16 scan, 0 for the regular
    form: the library's rule (csrc/scan_tm.cu, choose_lean_warps), restated to name the kernel that ran."""
    env = os.environ.get("MAMBA_TM_LEAN")
    if env == "0":
        return 0

    def waves(w):
        cw = 32 * w // S
        return -(-(Bsz * (-(-Dch // cw))) // sms)

    costs = [(waves(w) * ((w + 1 + 3) // 4), w) for w in range(8, 12)]
    regular = min(costs)[1]                   # narrowest width of least cost, as tm_launch_cost
    best, best_waves = 0, (1 << 62) if env == "1" else waves(regular)
    for w in range(12, 19):
        if waves(w) < best_waves:
            best, best_waves = w, waves(w)
    return best


def scan_result(args, m, torch, x, workload, steps, conv, t_ms, clocks, chunked, nbytes, R, e2e_ms, h2d, d2h,
                mufu_per_clk, sms, flag_name="none"):
    Bsz, Dch, L, N = x.shape
    io = x.io
    peaks = measured_peaks()
    exps = Bsz * Dch * L * N
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    mufu_units = round(mufu_per_clk)
    mufu_peak = SM_COUNT_NOMINAL * mufu_units * peaks["sm_max_mhz"] * 1e6   # ex2 per second
    t_mufu = exps / mufu_peak
    t_meas = t_ms * 1e-3
    tm = 8 < N <= 64 and (io == "bf16" or N <= 16) and os.environ.get("MAMBA_SCAN_KERNEL") != "smem"
    S = 4 if N <= 16 else 8 if N <= 32 else 16
    lean = tm and io == "bf16" and conv == "none" and flag_name == "none" and not chunked and \
        lean_warps(Bsz, Dch, S, sms) > 0
    kernel = (f"scan_tm_lean_kernel<{io},full,z,S{S},W{lean_warps(Bsz, Dch, S, sms)}>" if lean else
              f"scan_tm_kernel<{io},full,z,S{S}"
              f"{',conv' if conv == 'fused' else ''}{',flags' if flag_name != 'none' else ''}>" if tm
              else f"scan_kernel<{io},NP{1 << max(2, (N - 1).bit_length())},full>")
    traffic = traffic_record(workload, kernel=kernel)
    if t_mufu >= t_hbm:
        roof = {"bound": "alu", "achieved": round(exps / t_meas / 1e12, 4),
                "peak": round(mufu_peak / 1e12, 4), "unit": "Tex2/s", "frac": round(t_mufu / t_meas, 4),
                "traffic": traffic, "kernel": kernel,
                "peak_source": f"{SM_COUNT_NOMINAL} SMs x {mufu_units} ex2/clk/SM (microbenchmark: "
                               f"{mufu_per_clk:.2f}) x {peaks['sm_max_mhz']:.0f} MHz",
                "hbm": {"achieved": round(nbytes / t_meas / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": round(t_hbm / t_meas, 4), "peak_source": peaks["source"]}}
    else:
        roof = {"bound": "hbm", "achieved": round(nbytes / t_meas / 1e9, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(t_hbm / t_meas, 4), "traffic": traffic, "kernel": kernel,
                "peak_source": f"{peaks['source']} copy bandwidth"}
    scheme = ("two-pass" if (os.environ.get("MAMBA_CHUNKED_SCAN") == "two-pass" or not tm or flag_name != "none"
                             or conv == "fused") else "decay-truncated")
    if chunked:
        roof["note"] = (f"chunked scan ({scheme}): the step is three launches "
                        + ("(every chunk from a zero state with its end state, carry, correction of y)"
                           if scheme == "decay-truncated" else "(chunk end states, carry, rescan)")
                        + "; figures are per step")
    if conv == "two-step":
        roof["note"] = (roof.get("note", "") + "; " if "note" in roof else "") + \
            "two launches per step (convolution, then scan); figures are per step"
    return dict(ms_per_step=t_ms, bytes=nbytes, tokens=Bsz * L, dtype="f32" if io == "f32" else "bf16",
                config={"workload": workload, "batch": Bsz, "d_inner": Dch, "d_state": N, "seq_len": L,
                        "io": io, "state": "fp32", "l2": f"inputs rotate over {R} resident copies "
                                                          f"({R * nbytes / 1e6:.0f} MB > L2)",
                        "path": f"chunked ({scheme})" if chunked else "direct",
                        **({"flags": flag_name} if flag_name != "none" else {}),
                        **({"conv": conv + " (depthwise causal conv1d k=4 + SiLU feeding u)"}
                           if conv != "none" else {})},
                roofline=roof, h2d=h2d, d2h=d2h, e2e_ms=e2e_ms,
                launches=steps * ((3 if chunked else 1) + (1 if conv == "two-step" else 0)),
                clocks=clocks, inputs=x,
                mufu={"ex2_per_clk_per_sm": round(mufu_per_clk, 3), "sms": sms})


def bench_decode(args, m, torch, steps=None, e2e=True):
    steps = steps or args.steps
    cfg = inputs.DECODE_WORKLOAD
    Bsz, Dch, N, io = cfg["batch"], cfg["dim"], cfg["dstate"], cfg["io"]
    dev = torch.device("cuda")
    A, D, bias, _ = inputs.channel_params(Dch, N, cfg["seed"])
    A, D, bias = (torch.from_numpy(a).to(dev) for a in (A, D, bias))
    st0 = torch.from_numpy(inputs.make_decode_state(Bsz, Dch, N, cfg["seed"])).to(dev)
    nbytes = step_bytes(Bsz, Dch, N, io)
    R = max(2, math.ceil(3 * L2_BYTES / nbytes))
    states = [st0.clone() for _ in range(R)]
    P = 8   # distinct per-step inputs, cycled

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    steps_in = []
    for k in range(P):
        s = inputs.make_decode_step(Bsz, Dch, N, cfg["seed"], k, io)
        steps_in.append({n: d(getattr(s, n)) for n in ("u", "delta", "z", "B", "C")})
    ys = [torch.empty((Bsz, Dch), dtype=torch.bfloat16, device=dev) for _ in range(R)]
    stream = torch.cuda.current_stream()

    def step(i):
        s = steps_in[i % P]
        m.mamba_state_update(states[i % R], s["u"], s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, ys[i % R],
                             stream=stream)

    mufu_per_clk, sms = mufu_ex2_per_clk_per_sm(m, torch)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # A decode step is a ~40 us kernel: issuing it from Python once per step
    # would time the host, so the K timed steps are captured once in a CUDA
    # graph (the library launches on the caller's stream) and replayed.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(steps):
                m.mamba_state_update(states[i % R], steps_in[i % P]["u"], steps_in[i % P]["delta"], A,
                                     steps_in[i % P]["B"], steps_in[i % P]["C"], D, steps_in[i % P]["z"], bias, 1,
                                     ys[i % R], stream=cap)
    stream.wait_stream(cap)
    graph.replay()   # warm replay
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(pci_bus_id(torch)) as cs:
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    t_ms = ev0.elapsed_time(ev1) / steps
    clocks = cs.summary()

    # the same steps launched one by one from the host (no graph): what a caller that does not capture pays
    ch_steps = min(steps, 200)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    with ClockSampler(pci_bus_id(torch)) as cs2:
        ev0.record(stream)
        for i in range(ch_steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    chained_ms = ev0.elapsed_time(ev1) / ch_steps
    chained = {"ms_per_step": round(chained_ms, 6), "steps": ch_steps,
               "value": round(nbytes / (chained_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "frac": round(nbytes / (measured_peaks()["hbm_gbs"] * 1e9) / (chained_ms * 1e-3), 4),
               "clocks": cs2.summary(), "launch": "one host launch per step, chained on one stream"}
    if not e2e:
        return decode_result(args, m, torch, steps, t_ms, clocks, nbytes, R, None, None, None, mufu_per_clk, sms,
                             chained)

    # end to end: every step uploads the state and the step's inputs from pinned host memory and downloads
    # y and the new state; uploads and downloads overlap the neighbouring steps' kernels (two buffer sets)
    hst = [states[k].cpu().pin_memory() for k in range(2)]
    hin = [{k: v.cpu().pin_memory() for k, v in s.items()} for s in steps_in[:2]]
    hy = [torch.empty((Bsz, Dch), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dins = [steps_in[0], steps_in[1]]

    def upload(k, st):
        states[k].copy_(hst[k], non_blocking=True)
        for n in dins[k]:
            dins[k][n].copy_(hin[k][n], non_blocking=True)

    def compute(k, st):
        m.mamba_state_update(states[k], dins[k]["u"], dins[k]["delta"], A, dins[k]["B"], dins[k]["C"], D,
                             dins[k]["z"], bias, 1, ys[k], stream=st)

    def download(k, st):
        hy[k].copy_(ys[k], non_blocking=True)
        hst[k].copy_(states[k], non_blocking=True)

    pipelined_e2e(torch, 3, upload, compute, download)   # warm-up
    e2e_ms = pipelined_e2e(torch, args.e2e_steps, upload, compute, download)
    h2d = hst[0].numel() * 4 + sum(v.numel() * v.element_size() for v in hin[0].values())
    d2h = hy[0].numel() * 2 + hst[0].numel() * 4
    return decode_result(args, m, torch, steps, t_ms, clocks, nbytes, R, e2e_ms, h2d, d2h, mufu_per_clk, sms,
                         chained)


def decode_result(args, m, torch, steps, t_ms, clocks, nbytes, R, e2e_ms, h2d, d2h, mufu_per_clk, sms, chained):
    cfg = inputs.DECODE_WORKLOAD
    Bsz, Dch, N, io = cfg["batch"], cfg["dim"], cfg["dstate"], cfg["io"]
    peaks = measured_peaks()
    t_meas = t_ms * 1e-3
    roof = {"bound": "hbm", "achieved": round(nbytes / t_meas / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(nbytes / (peaks["hbm_gbs"] * 1e9) / t_meas, 4),
            "traffic": traffic_record(cfg["name"], DECODE_KERNEL_SOURCES), "kernel": "state_update_rows_kernel<bf16,NP16,R1,V8>",
            "peak_source": f"{peaks['source']} copy bandwidth"}
    return dict(ms_per_step=t_ms, bytes=nbytes, tokens=Bsz, dtype="bf16",
                config={"workload": cfg["name"], "batch": Bsz, "d_inner": Dch, "d_state": N, "io": io,
                        "state": "fp32", "l2": f"state rotates over {R} resident copies "
                                                f"({R * nbytes / 1e6:.0f} MB > L2)",
                        "launch": f"the {steps} timed steps replayed as one captured CUDA graph"},
                roofline=roof, h2d=h2d, d2h=d2h, e2e_ms=e2e_ms, launches=steps, clocks=clocks,
                mufu={"ex2_per_clk_per_sm": round(mufu_per_clk, 3), "sms": sms}, chained=chained)


def bwd_bytes(Bsz, Dch, L, N, io):
    """Algorithmic bytes of the backward: read u, Delta_raw, z, dy, B, C; write du, ddelta, dz (storage type)
    and dB, dC (fp32); parameters and their fp32 gradients."""
    s = io_bytes(io)
    return 7 * Bsz * Dch * L * s + 2 * Bsz * N * L * s + 2 * Bsz * N * L * 4 + 2 * Dch * N * 4 + 6 * Dch * 4


def bench_backward(args, m, torch, workload=None, steps=None, e2e=True):
    workload = workload or args.workload
    steps = steps or args.steps
    x = inputs.make_workload(workload)
    Bsz, Dch, L, N = x.shape
    io = x.io
    dev = torch.device("cuda")

    def d(a):
        if io == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    dy_host = inputs._store(np.random.default_rng(11).standard_normal(x.u.shape).astype(np.float32), io)
    t = dict(u=d(x.u), delta=d(x.delta), z=d(x.z), B=d(x.B), C=d(x.C), dy=d(dy_host))
    A, D, bias = (torch.from_numpy(a).to(dev) for a in (x.A, x.D, x.delta_bias))
    nbytes = bwd_bytes(Bsz, Dch, L, N, io)
    R = max(2, math.ceil(3 * L2_BYTES / nbytes))
    sets = [t] + [{k: v.clone() for k, v in t.items()} for _ in range(R - 1)]
    f32 = dict(dtype=torch.float32, device=dev)
    outs = [dict(du=torch.empty_like(t["u"]), dd=torch.empty_like(t["u"]), dz=torch.empty_like(t["u"]),
                 dA=torch.empty((Dch, N), **f32), dB=torch.empty((Bsz, N, L), **f32),
                 dC=torch.empty((Bsz, N, L), **f32), dD=torch.empty(Dch, **f32), db=torch.empty(Dch, **f32))
            for _ in range(R)]
    stream = torch.cuda.current_stream()

    def step(i):
        s, o = sets[i % R], outs[i % R]
        m.mamba_selective_scan_bwd(s["u"], s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, s["dy"], o["du"],
                                   o["dd"], o["dA"], o["dB"], o["dC"], o["dD"], o["dz"], o["db"], stream=stream)

    mufu_per_clk, sms = mufu_ex2_per_clk_per_sm(m, torch)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(pci_bus_id(torch)) as cs:
        ev0.record(stream)
        for i in range(steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    t_ms = ev0.elapsed_time(ev1) / steps
    clocks = cs.summary()

    # the training pair: the forward scan that saves the checkpoints, then the backward that starts from them
    ckb = m.mamba_scan_bwd_ckpt_size(Bsz, Dch, L, N)
    cks = [torch.empty(ckb // 4, **f32) for _ in range(R)]
    ys = [torch.empty_like(t["u"]) for _ in range(R)]

    def fwd_save(i):
        s = sets[i % R]
        m.mamba_selective_scan_fwd_save(s["u"], s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, ys[i % R], None,
                                        cks[i % R], stream=stream)

    def bwd_ckpt(i):
        s, o = sets[i % R], outs[i % R]
        m.mamba_selective_scan_bwd_from_ckpt(s["u"], s["delta"], A, s["B"], s["C"], D, s["z"], bias, 1, s["dy"],
                                             cks[i % R], o["du"], o["dd"], o["dA"], o["dB"], o["dC"], o["dD"], o["dz"],
                                             o["db"], stream=stream)

    def timed(fn, n):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    for i in range(R):      # every rotating set holds its own checkpoints
        fwd_save(i)
    fs_ms = timed(fwd_save, steps)
    bc_ms = timed(bwd_ckpt, steps)
    training_pair = {"fwd_save_ms": round(fs_ms, 6), "bwd_from_ckpt_ms": round(bc_ms, 6),
                     "ckpt_bytes": ckb,
                     "note": "mamba_selective_scan_fwd_save (the direct scan writing the backward's checkpoints) "
                             "and mamba_selective_scan_bwd_from_ckpt (no checkpoint sweep), each timed alone"}
    del cks, ys

    e2e_ms, h2d, d2h = None, None, None
    if e2e:
        e2e_ms, h2d, d2h = bwd_e2e(args, torch, t, sets, outs, step, stream)
    peaks = measured_peaks()
    t_meas = t_ms * 1e-3
    exps = Bsz * Dch * L * N
    mufu_units = round(mufu_per_clk)
    mufu_peak = SM_COUNT_NOMINAL * mufu_units * peaks["sm_max_mhz"] * 1e6
    roof = {"bound": "alu", "achieved": round(exps / t_meas / 1e12, 4), "peak": round(mufu_peak / 1e12, 4),
            "unit": "Tex2/s", "frac": round(exps / mufu_peak / t_meas, 4), "traffic": None,
            "kernel": f"scan_bwd_kernel<{io},NS{4 if N <= 16 else 8 if N <= 32 else 16}>",
            "peak_source": f"{SM_COUNT_NOMINAL} SMs x {mufu_units} ex2/clk/SM (microbenchmark: "
                           f"{mufu_per_clk:.2f}) x {peaks['sm_max_mhz']:.0f} MHz",
            "note": "algorithmic exps count B·D·L·N once; the kernel evaluates them three times (checkpoint "
                    "sweep, chunk recompute, reverse sweep)",
            "hbm": {"achieved": round(nbytes / t_meas / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(nbytes / (peaks["hbm_gbs"] * 1e9) / t_meas, 4)}}
    return dict(ms_per_step=t_ms, bytes=nbytes, tokens=Bsz * L, dtype="f32" if io == "f32" else "bf16",
                config={"workload": workload, "pass": "backward", "batch": Bsz, "d_inner": Dch, "d_state": N,
                        "seq_len": L, "io": io, "grads": "du, ddelta, dz (storage type); dA, dB, dC, dD, dbias fp32",
                        "l2": f"inputs rotate over {R} resident copies"},
                roofline=roof, h2d=h2d, d2h=d2h, e2e_ms=e2e_ms,
                launches=steps,  # the backward kernel (plus five cudaMemsetAsync zero fills per step)
                clocks=clocks, inputs=x, mufu={"ex2_per_clk_per_sm": round(mufu_per_clk, 3), "sms": sms},
                training_pair=training_pair)


def bwd_e2e(args, torch, t, sets, outs, step, stream):
    # end to end: inputs from pinned host memory, every gradient back to the host
    hin = {k: v.cpu().pin_memory() for k, v in t.items()}
    hout = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in outs[0].items()}

    def e2e_step(i):
        for k in t:
            sets[0][k].copy_(hin[k], non_blocking=True)
        step(0)
        for k in hout:
            hout[k].copy_(outs[0][k], non_blocking=True)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    return e2e_ms, sum(v.numel() * v.element_size() for v in hin.values()), \
        sum(v.numel() * v.element_size() for v in hout.values())


def reference_arm(args, world, rank):
    """The oracle (float64, host cores) on a bounded sample of the same workload."""
    if rank != 0:
        return
    if args.workload == inputs.DECODE_WORKLOAD["name"]:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the scan workloads only"}))
        return
    x = inputs.make_workload(args.workload)
    Bsz, Dch, L, N = x.shape
    vals = []
    info = None
    budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        bps, ups, info = time_oracle(x, budget_s=budget)
        if i >= args.warmup:
            vals.append(bps)
    v = statistics.median(vals) / 1e9
    t_ms = scan_bytes(Bsz, Dch, L, N, x.io) / (v * 1e9) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "batch": Bsz, "d_inner": Dch, "d_state": N, "seq_len": L,
                       "io": x.io},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": info["threads"], "kind": "oracle",
                             "sample": f"whole time rows of {info['channels']} of {info['of']} channels per step"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
