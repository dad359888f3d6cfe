"""Benchmark of the exact attention forward on GB300 (one JSON line on rank 0).

Default workload: one head, N_q = N_k = 8192, d = 128, non-causal, BF16
Q/K/V ~ N(0, 1), scale 1/sqrt(d) (34.4 GFLOP per step). A step is one
``fa_forward`` call through the C ABI over that batch. The K timed steps run
back to back between two CUDA events, each on the next of several copies of
the inputs, so many that together they take at least twice the L2 size (a
step's inputs have left L2 by the time their copy comes round again). Also reported: the same steps timed one by
one with L2 flushed before each ("flushed"), the end-to-end rate with host
buffers ("e2e"), and the decode workload (B=16, 32/8 heads, 8192 keys).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl fused|naive|reference]
                    [--workload NAME]

``--impl reference`` times the FP64 CPU oracle on the host cores (the only
other place this file runs the oracle besides the ``cpu_baseline`` leg).
Under torchrun (N > 1) every rank runs one independent replica of the
workload (the path needs no exchange between GPUs); rank 0 prints.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import numpy as np  # noqa: E402

from exact_tiled_attention_forward_gb300 import inputs as I  # noqa: E402
from exact_tiled_attention_forward_gb300 import replicas as R  # noqa: E402
from exact_tiled_attention_forward_gb300 import work as W  # noqa: E402

METRIC = "attention fwd TFLOP/s (prefill) & HBM GB/s (decode), % of GB300 roofline"
DEFAULT_WORKLOAD = "one_head_n8192_d128"
DECODE_WORKLOAD = "decode_b16_h32_kv8_n8192_d128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the sources each profiled kernel is built from (a summary's traffic figure is
# used only while their hash matches the one recorded with it)
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["exact_tiled_attention_forward_gb300/csrc/fa_fwd.cu",
                      "exact_tiled_attention_forward_gb300/csrc/fa_fwd_kernel.cuh",
                      "exact_tiled_attention_forward_gb300/csrc/fa_ptx.cuh"],
    "fa_fwd_tile_kernel": ["exact_tiled_attention_forward_gb300/csrc/fa_fwd_d256.cu",
                           "exact_tiled_attention_forward_gb300/csrc/fa_ptx.cuh"],
    "fa_decode_kernel": ["exact_tiled_attention_forward_gb300/csrc/fa_decode.cu",
                         "exact_tiled_attention_forward_gb300/csrc/fa_ptx.cuh"],
    "fa_bwd_kernel": ["exact_tiled_attention_forward_gb300/csrc/fa_bwd.cu",
                      "exact_tiled_attention_forward_gb300/csrc/fa_ptx.cuh"],
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "fa_fwd_kernel"):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or
    None if there is none or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    m_h = re.search(r"^kernel_source_sha256_16:\s*([0-9a-f]+)", text, re.M)
    if not m_b or not m_h or m_h.group(1) != kernel_hash(kernel):
        return None
    return float(m_b.group(1))


class ClockSampler:
    """SM clock and throttle-reason samples taken DURING the timed region.

    Reads NVML (libnvidia-ml, through ctypes) every 1 ms from a thread, so even
    a timed region of a few milliseconds gets samples; falls back to
    ``nvidia-smi -lms 200`` if NVML cannot be loaded. Read-only: no setting of
    the GPU is changed.
    """
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, bus_id: str | None, uuid: str | None):
        self.bus_id, self.uuid = bus_id, uuid
        self.samples, self.reason_bits, self.max_mhz = [], 0, None
        self.nvml = self.dev = None
        self.thread = None
        self.smi = None
        self._stop = False

    def _open_nvml(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return False
        dev = ctypes.c_void_p()
        ok = False
        if self.bus_id:
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(self.bus_id.encode(), ctypes.byref(dev)) == 0
        if not ok and self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(dev)) == 0
        if not ok:
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self.nvml, self.dev = lib, dev
        return True

    def _loop(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        get_r = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop:
            if self.nvml.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if get_r(self.dev, ctypes.byref(rs)) == 0:
                self.reason_bits |= int(rs.value)
            time.sleep(0.001)

    def start(self):
        try:
            have = self._open_nvml()
        except Exception:  # noqa: BLE001 - any NVML trouble falls back to nvidia-smi
            have = False
        if have:
            import threading
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
            return
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.smi = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=pci.bus_id,clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.smi = None

    def stop(self):
        if self.thread is not None:
            self._stop = True
            self.thread.join()
            src = "nvml, 1 ms"
        elif self.smi is not None:
            self.smi.terminate()
            self.smi.wait(timeout=5)
            self.out.close()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            bits = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
                    "sw_power_cap": 0x4}
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 7 or (self.bus_id and self.bus_id[-12:].lower() not in parts[0].lower()):
                    continue
                try:
                    self.samples.append(float(parts[1]))
                    self.max_mhz = float(parts[2])
                except ValueError:
                    continue
                for nm, val in zip(names, parts[3:7]):
                    if val.lower() == "active":
                        self.reason_bits |= bits[nm]
            os.unlink(self.path)
            src = "nvidia-smi, 200 ms"
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0, "reasons": ["unavailable"]}
        reasons = sorted(v for b, v in self.REASONS.items() if self.reason_bits & b)
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples), "reasons": reasons,
                "source": src}


def device_ids(props):
    """(PCI bus id, UUID) of a device, as NVML names them (either may be None)."""
    bus = getattr(props, "pci_bus_id", None)
    bus_id = None
    if bus is not None:
        bus_id = (f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:"
                  f"{getattr(props, 'pci_device_id', 0):02x}.0")
    uuid = getattr(props, "uuid", None)
    uuid = None if uuid is None else ("GPU-" + str(uuid) if not str(uuid).startswith("GPU-") else str(uuid))
    return bus_id, uuid


def to_device(torch, x, dev):
    """An input array on the device: FP16 values as torch.float16, BF16 bit
    patterns as torch.bfloat16, FP8 E4M3 codes as torch.uint8."""
    if x.dtype == np.float16 or x.dtype == np.uint8:
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)


def elem_dtype(torch, a):
    """Element type of O (BF16 for FP8 inputs)."""
    return torch.float16 if a.dtype == "f16" else torch.bfloat16


def forward_fn(fa, a):
    """The library's forward for the workload's input type, as fn(q, k, v, ...)."""
    if a.dtype == "e4m3":
        return lambda q, k, v, **kw: fa.fa_forward_fp8(q, k, v, a.descale, **kw)
    return fa.fa_forward


def workload_config(name: str):
    cfg = dict(I.WORKLOADS[name])
    a_flops = W.flops_pages(cfg["B"], cfg["H_q"], cfg["N_q"], cfg["N_k"], cfg["d"], cfg["causal"])
    a_bytes = W.bytes_moved(cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N_q"], cfg["N_k"], cfg["d"])
    decode = cfg["N_q"] == 1
    return cfg, a_flops, a_bytes, decode


def cpu_oracle_throughput(a, budget_s: float, max_rows: int | None = None):
    """Time the oracle on the host over query rows taken head by head (whole
    heads, or the first rows of each head once ``max_rows`` is reached), until
    ``budget_s`` has elapsed or ``max_rows`` rows are done.

    Returns (rows done, seconds, threads used, (batch, head) calls)."""
    import oracle
    B, Hq, Hkv, Nq, Nk, d = a.shape_args
    q, k, v = a.q, a.k, a.v
    if a.dtype == "e4m3":   # the FP8 oracle: the definition on code * factor
        q, k, v = (oracle.e4m3_to_f64(x) * s for x, s in zip((q, k, v), a.descale))
    t0 = time.perf_counter()
    done_rows = 0
    calls = 0
    while True:
        for b in range(B):
            for h in range(Hq):
                n = Nq if max_rows is None else min(Nq, max_rows - done_rows)
                if n <= 0:
                    break
                oracle.attention_rows(q, k, v, b, h, np.arange(n), causal=a.causal, scale=a.scale)
                done_rows += n
                calls += 1
                if time.perf_counter() - t0 >= budget_s and max_rows is None:
                    break
            else:
                continue
            break
        if max_rows is not None or time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    return done_rows, dt, cores, calls


def fused_launches_per_step(fa, cfg) -> int:
    """Kernels one fa_forward call launches (the library's own plan for it)."""
    return fa.fa_forward_plan(cfg["B"], cfg["H_q"], cfg["H_kv"], cfg["N_q"], cfg["N_k"], cfg["d"],
                              cfg["causal"])["launches"]


def hold_device(torch):
    """Queue ~100 us of device-side waiting on the current stream just before a
    timed region's start event, so the region starts with the first step's
    kernels already enqueued behind it: the host's latency to enqueue the first
    step is then not counted as device time (the steps themselves still run
    back to back, every one inside the region)."""
    torch.cuda._sleep(200_000)


def time_decode(fa, torch, dev, flush, stream, steps, warmup, world, dtype="bf16"):
    """Device time of the decode workload; GB/s of algorithmic bytes (K, V once
    per KV head, Q read, O and LSE written). Two input sets used in turn (each
    537 MB, several times L2), steps back to back between two events; also the
    same steps one at a time with L2 flushed before each ("flushed")."""
    cfg, _, a_bytes, _ = workload_config(DECODE_WORKLOAD)
    a = I.make_workload(DECODE_WORKLOAD, dtype=dtype)
    to = lambda x: to_device(torch, x, dev)
    B, Hq, Hkv, Nq, Nk, d = a.shape_args
    q, k, v = to(a.q), to(a.k), to(a.v)
    sets = [(q, k, v), (q.clone(), k.clone(), v.clone())]
    o = torch.empty((B, Hq, Nq, d), dtype=elem_dtype(torch, a), device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)

    def step(i):
        qq, kk, vv = sets[i & 1]
        fa.fa_forward(qq, kk, vv, causal=False, scale=a.scale, out=o, lse=lse)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_device(torch)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = R.slowest_rank_ms(e0.elapsed_time(e1) / steps, world, dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for f0, f1 in evs:
        flush.zero_()
        f0.record(stream)
        step(0)
        f1.record(stream)
    torch.cuda.synchronize()
    fms = R.slowest_rank_ms(sum(f0.elapsed_time(f1) for f0, f1 in evs) / steps, world, dev)
    plan = fa.fa_forward_plan(B, Hq, Hkv, Nq, Nk, d, False)
    parts = plan["ctas"] // (B * Hkv)
    split = (f"128-key chunks, {-(-((Nk + 127) // 128) // parts)} consecutive chunks per CTA, "
             f"{parts} CTAs per (batch, KV head), partials merged "
             + ("inside thread-block clusters" if plan["launches"] == 1 else "by a second kernel"))
    return {"ms": ms, "gbs": R.whole_job_rate(a_bytes / 1e9, 1, ms, world), "bytes": a_bytes, "split": split,
            "flushed_ms": fms, "flushed_gbs": R.whole_job_rate(a_bytes / 1e9, 1, fms, world),
            "launches": fused_launches_per_step(fa, cfg)}


def time_e2e(torch, fa, a, cfg, dev, stream, fn, ws, steps, warmup, world, work_per_step):
    """End-to-end rate with the step's tensors in pinned host memory.

    Fused: one ``fa_forward_host_packed`` call runs the K steps as K requests
    (each copies Q | K | V in from one pinned buffer and O | LSE out to one of two
    pinned buffers; libfa overlaps request i+1's copy in and i-1's copy out with
    request i's kernels). ``serial``: the same steps as K calls of one request
    each, nothing overlapped. Unfused: the serial form with torch copies.

    Returns (rate, ms per step, H2D bytes per step, D2H bytes per step, serial dict)."""
    B, Hq, Hkv, Nq, Nk, d = a.shape_args
    nq, nk = a.q.size, a.k.size
    el = elem_dtype(torch, a)
    hin = to_device(torch, np.concatenate([a.q.reshape(-1), a.k.reshape(-1), a.v.reshape(-1)]),
                    "cpu").pin_memory()
    o_bytes, l_bytes = B * Hq * Nq * d * 2, B * Hq * Nq * 4
    hout = [torch.empty(o_bytes + l_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]

    if ws is None and a.dtype != "e4m3":
        def run(n):
            fa.fa_forward_host_packed([hin] * n, [hout[i & 1] for i in range(n)], a.shape_args,
                                      causal=a.causal, scale=a.scale, dtype=el)
    else:
        din = torch.empty_like(hin, device=dev)
        dq, dk, dv = (din[:nq].view(B, Hq, Nq, d), din[nq:nq + nk].view(B, Hkv, Nk, d),
                      din[nq + nk:].view(B, Hkv, Nk, d))
        dout = torch.empty(o_bytes + l_bytes, dtype=torch.uint8, device=dev)
        do = dout[:o_bytes].view(el).view(B, Hq, Nq, d)
        dl = dout[o_bytes:].view(torch.float32).view(B, Hq, Nq)

        extra = {} if ws is None else {"workspace": ws}

        def run(n):
            for _ in range(n):
                din.copy_(hin, non_blocking=True)
                fn(dq, dk, dv, causal=a.causal, scale=a.scale, out=do, lse=dl, **extra)
                hout[0].copy_(dout, non_blocking=True)

    run(max(3, warmup))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws is None:
        hold_device(torch)
        e0.record(stream)
        run(steps)
        e1.record(stream)
        torch.cuda.synchronize()
        p_ms = R.slowest_rank_ms(e0.elapsed_time(e1), world, dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for x0, x1 in evs:
        x0.record(stream)
        run(1)
        x1.record(stream)
    torch.cuda.synchronize()
    s_ms = R.slowest_rank_ms(sum(x.elapsed_time(y) for x, y in evs), world, dev)
    if ws is not None:
        p_ms = s_ms
    return (R.whole_job_rate(work_per_step, steps, p_ms, world), p_ms / steps, hin.numel() * 2,
            hout[0].numel(),
            {"value": R.whole_job_rate(work_per_step, steps, s_ms, world), "ms_per_step": s_ms / steps,
             "note": "the same steps as one request per call, nothing overlapped"})


BWD_METRIC = "attention bwd TFLOP/s (10 N_q N_k d per head, halved when causal), % of GB300 roofline"


def backward_flops(cfg) -> float:
    """The backward's five products of 2 N_q N_k d each per query head (S, dP,
    dV, dK, dQ): 2.5 times the forward's count, halved when causal."""
    return 2.5 * W.flops_pages(cfg["B"], cfg["H_q"], cfg["N_q"], cfg["N_k"], cfg["d"], cfg["causal"])


def cpu_oracle_backward(a, do, budget_s: float, max_n: int = 2048):
    """The FP64 backward oracle on head 0 (and its KV head), cut to its first
    ``max_n`` query rows and keys when longer, called again until ``budget_s``
    has elapsed. Returns (FLOP/s, seconds, sample)."""
    import oracle
    n_q, n_k = min(a.N_q, max_n), min(a.N_k, max_n)
    q, k, v, g = a.q[:1, :1, :n_q], a.k[:1, :1, :n_k], a.v[:1, :1, :n_k], do[:1, :1, :n_q]
    t0 = time.perf_counter()
    calls = 0
    while calls == 0 or time.perf_counter() - t0 < budget_s:
        oracle.attention_backward(q, k, v, g, causal=a.causal, scale=a.scale)
        calls += 1
    dt = time.perf_counter() - t0
    flops = calls * 2.5 * W.flops_pages(1, 1, n_q, n_k, a.d, a.causal)
    sample = (f"{calls} calls on head 0: {n_q} query rows x {n_k} keys (of {a.N_q} x {a.N_k} in each "
              f"of {a.B * a.H_q} heads), FP64 materialised oracle, numpy/OpenBLAS")
    return flops / dt, dt, sample


def run_backward(args, rank, world, local, warmup):
    """``--pass backward``: K fa_backward steps (prep kernel + one main launch)
    back to back between two events, each on the next of several input sets
    larger than L2 together; the forward's O and LSE come from fa_forward,
    untimed. Prints one JSON line on rank 0."""
    import torch
    import exact_tiled_attention_forward_gb300 as fa
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    fa.lib()
    cfg = dict(I.WORKLOADS[args.workload])
    if cfg["N_q"] == 1:
        raise SystemExit("--pass backward takes a prefill workload")
    a = I.make_workload(args.workload, dtype=args.dtype)
    do_h = I.grad_output(a, seed=0)
    B, Hq, Hkv, Nq, Nk, d = a.shape_args
    flops = backward_flops(cfg)
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or (129 << 20))
    q, k, v, g = (to_device(torch, x, dev) for x in (a.q, a.k, a.v, do_h))
    o, lse = fa.fa_forward(q, k, v, causal=a.causal, scale=a.scale)
    set_bytes = (2 * q.numel() + 2 * k.numel() + o.numel() + g.numel()) * 2 + lse.numel() * 4
    n_sets = min(256, max(2, -(-2 * l2_bytes // set_bytes)))
    sets = []
    for _ in range(n_sets):
        sets.append(tuple(x.clone() for x in (q, k, v, o, lse, g)) +
                    (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)))

    def step(i):
        qq, kk, vv, oo, ll, gg, dq, dk, dv = sets[i % n_sets]
        fa.fa_backward(qq, kk, vv, oo, ll, gg, causal=a.causal, scale=a.scale, dq=dq, dk=dk, dv=dv)

    stream = torch.cuda.current_stream()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(*device_ids(props))
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    hold_device(torch)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = R.slowest_rank_ms(e0.elapsed_time(e1), world, dev)
    ms = total_ms / args.steps
    value = R.whole_job_rate(flops / 1e12, args.steps, total_ms, world)
    if fa.fa_device_status() != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait during the benchmark")

    # end to end: every step copies q, k, v, o, lse, dO in from pinned host memory
    # and dq, dk, dv back out, inside the timed region (nothing overlapped)
    hin = [x.cpu().pin_memory() for x in (q, k, v, o, lse, g)]
    hout = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (q, k, v)]
    dins = [torch.empty_like(x) for x in (q, k, v, o, lse, g)]
    douts = [torch.empty_like(x) for x in (q, k, v)]

    def e2e_step():
        for dx, hx in zip(dins, hin):
            dx.copy_(hx, non_blocking=True)
        fa.fa_backward(*dins, causal=a.causal, scale=a.scale, dq=douts[0], dk=douts[1], dv=douts[2])
        for hx, dx in zip(hout, douts):
            hx.copy_(dx, non_blocking=True)

    for _ in range(warmup):
        e2e_step()
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = R.slowest_rank_ms(x0.elapsed_time(x1), world, dev)
    h2d = sum(x.numel() * x.element_size() for x in hin)
    d2h = sum(x.numel() * x.element_size() for x in hout)

    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = flops / 1e12 / (ms * 1e-3)
    cpu = None
    if args.cpu_budget > 0 and world == 1:
        rate, dt, sample = cpu_oracle_backward(a, do_h, args.cpu_budget)
        cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": int(os.environ.get("OPENBLAS_NUM_THREADS", 1)),
               "kind": "oracle", "sample": f"{sample}, {dt:.1f} s"}
    line = {
        "metric": BWD_METRIC, "pass": "backward", "impl": "fused", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": args.workload, **{k2: cfg[k2] for k2 in
                   ("B", "H_q", "H_kv", "N_q", "N_k", "d", "causal")}, "scale": a.scale,
                   "l2": (f"inputs larger than L2: {n_sets} copies of q, k, v, o, lse, dO (each with "
                          f"its own dq, dk, dv) used in turn, {n_sets * set_bytes / 2**20:.0f} MiB "
                          f"against {l2_bytes / 2**20:.0f} MiB of L2; steps back to back"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic(args.workload, "fa_bwd_kernel"),
                     "peak_source": f"{peak_src} (burst)", "algorithmic_per_launch": flops,
                     "kernel": ("fa_bwd_kernel, timed together with fa_bwd_prep_kernel (the "
                                "step's other launch): a lower bound on the main kernel's rate")},
        "cpu_baseline": cpu,
        "e2e": {"value": R.whole_job_rate(flops / 1e12, args.steps, e2e_ms, world), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps,
                "note": "fa_backward with torch copies from and to pinned host memory, nothing overlapped"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


PAGED_METRIC = "paged decode HBM GB/s (K/V read once per KV head), % of GB300 roofline"


def run_paged(args, rank, world, local, warmup):
    """``--pass paged``: the decode workload (batch 16, 32 query / 8 KV heads,
    8192 keys, d = 128) with its K/V cache in shuffled 128-key pages, through
    fa_decode_paged. Two cache sets (537 MB each) used in turn, K steps back to
    back between two events; the same steps one at a time after an L2 flush;
    end to end with every input copied in from pinned host memory and O, LSE
    copied out; the contiguous layout through fa_forward beside it. One JSON
    line on rank 0."""
    import torch
    import exact_tiled_attention_forward_gb300 as fa
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    fa.lib()
    cfg = dict(I.WORKLOADS[DECODE_WORKLOAD])
    B, Hq, Hkv, Nq, Nk, d = (cfg[x] for x in ("B", "H_q", "H_kv", "N_q", "N_k", "d"))
    pin = I.make_paged(B, Hq, Hkv, Nq, [Nk] * B, d, seed=0, dtype=args.dtype)
    to = lambda x: to_device(torch, x, dev)
    table = torch.from_numpy(pin.block_table).to(dev)
    lens = torch.from_numpy(pin.seqlens).to(dev)
    q, kc, vc = to(pin.q), to(pin.k_cache), to(pin.v_cache)
    sets = [(q, kc, vc), (q.clone(), kc.clone(), vc.clone())]
    o = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    a_bytes = W.bytes_moved(B, Hq, Hkv, Nq, Nk, d) + table.numel() * 4 + lens.numel() * 4

    def step(i):
        qq, kk, vv = sets[i & 1]
        fa.fa_decode_paged(qq, kk, vv, table, lens, scale=pin.scale, out=o, lse=lse)

    stream = torch.cuda.current_stream()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(*device_ids(torch.cuda.get_device_properties(dev)))
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_device(torch)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = R.slowest_rank_ms(e0.elapsed_time(e1), world, dev)
    ms = total_ms / args.steps
    value = R.whole_job_rate(a_bytes / 1e9, args.steps, total_ms, world)
    if fa.fa_device_status() != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait during the benchmark")

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for f0, f1 in evs:
        flush.zero_()
        f0.record(stream)
        step(0)
        f1.record(stream)
    torch.cuda.synchronize()
    fms = R.slowest_rank_ms(sum(f0.elapsed_time(f1) for f0, f1 in evs), world, dev) / args.steps

    # the same keys stored contiguously, through fa_forward (the decode kernel's other addressing)
    a = I.make_workload(DECODE_WORKLOAD, dtype=args.dtype)
    csets = [tuple(to(x) for x in (a.q, a.k, a.v))]
    csets.append(tuple(x.clone() for x in csets[0]))
    del sets[1]
    for i in range(warmup):
        fa.fa_forward(*csets[i & 1], scale=a.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for i in range(args.steps):
        fa.fa_forward(*csets[i & 1], scale=a.scale, out=o, lse=lse)
    c1.record(stream)
    torch.cuda.synchronize()
    c_ms = R.slowest_rank_ms(c0.elapsed_time(c1), world, dev) / args.steps
    del csets

    # end to end: q, both caches, block table and lengths in from pinned host
    # memory, O and LSE out, every step (nothing overlapped)
    hin = [x.cpu().pin_memory() for x in (q, kc, vc, table, lens)]
    hout = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (o, lse)]
    din = [torch.empty_like(x) for x in (q, kc, vc, table, lens)]
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        for dx, hx in zip(din, hin):
            dx.copy_(hx, non_blocking=True)
        fa.fa_decode_paged(*din, scale=pin.scale, out=o, lse=lse)
        hout[0].copy_(o, non_blocking=True)
        hout[1].copy_(lse, non_blocking=True)

    for _ in range(warmup):
        e2e_step()
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = R.slowest_rank_ms(x0.elapsed_time(x1), world, dev) / e2e_steps
    h2d = sum(x.numel() * x.element_size() for x in hin)
    d2h = sum(x.numel() * x.element_size() for x in hout)

    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    peaks, peak_src = load_peaks()
    peak = float(peaks["hbm_gbs"])
    cpu = None
    if args.cpu_budget > 0 and world == 1:
        import oracle
        t0 = time.perf_counter()
        n = 0
        while n == 0 or (time.perf_counter() - t0 < args.cpu_budget and n < B):
            oracle.paged_attention_reference(pin.q[n:n + 1], pin.k_cache, pin.v_cache, pin.block_table[n:n + 1],
                                             pin.seqlens[n:n + 1], scale=pin.scale)
            n += 1
        dt = time.perf_counter() - t0
        cpu = {"value": a_bytes * n / B / 1e9 / dt, "unit": "GB/s",
               "cores": int(os.environ.get("OPENBLAS_NUM_THREADS", 1)), "kind": "oracle",
               "sample": f"{n} of {B} sequences ({n * Hq} query rows x {Nk} keys) in {dt:.1f} s, FP64 oracle"}
    line = {
        "metric": PAGED_METRIC, "pass": "paged", "impl": "fused", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD + "_paged", "B": B, "H_q": Hq, "H_kv": Hkv, "N_q": Nq,
                   "seqlens": Nk, "page_keys": I.PAGE_KEYS, "pages": int(pin.k_cache.shape[0]), "d": d,
                   "causal": False, "scale": pin.scale,
                   "l2": "inputs larger than L2: two cache sets of 537 MB used in turn, back to back",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": a_bytes / 1e9 / (ms * 1e-3), "peak": peak, "unit": "GB/s",
                     "frac": a_bytes / 1e9 / (ms * 1e-3) / peak,
                     "traffic": profiled_traffic(DECODE_WORKLOAD + "_paged", "fa_decode_kernel"),
                     "peak_source": f"{peak_src} (copy)", "algorithmic_per_launch": a_bytes,
                     "kernel": "fa_decode_kernel (paged addressing, in-cluster merge)"},
        "flushed": {"value": a_bytes / 1e9 / (fms * 1e-3), "unit": "GB/s", "ms_per_step": fms,
                    "note": "each step alone between its own events, L2 flushed before it"},
        "contiguous": {"value": a_bytes / 1e9 / (c_ms * 1e-3), "unit": "GB/s", "ms_per_step": c_ms,
                       "note": "the same keys stored contiguously, through fa_forward, same timing"},
        "cpu_baseline": cpu,
        "e2e": {"value": a_bytes / 1e9 / (e2e_ms * 1e-3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "note": "fa_decode_paged with torch copies of every input in and O, LSE out, nothing overlapped"},
        "gpu_launches": fa.fa_forward_plan(B, Hq, Hkv, Nq, Nk, d, False)["launches"] * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="fused", choices=["fused", "naive", "reference"])
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16", "e4m3"],
                    help="element type of Q, K, V (and O; BF16 O for e4m3 inputs, which run "
                         "fa_forward_fp8 with per-tensor factors); the unfused baseline is BF16 only")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--decode-steps", type=int, default=500,
                    help="timed steps of the decode workload reported beside the prefill line")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of host time for the cpu_baseline leg (0 disables it)")
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward", "paged"],
                    help="backward: time fa_backward on the workload instead; paged: the decode "
                         "workload through fa_decode_paged (fused impl only)")
    args = ap.parse_args()
    if args.impl == "naive" and args.dtype != "bf16":
        ap.error("the unfused baseline is BF16 only")
    if args.dtype == "e4m3" and args.which != "forward":
        ap.error("e4m3 inputs: forward pass only")
    if args.dtype == "e4m3":
        args.decode_steps = 0   # the secondary decode line is the BF16 decode workload
    warmup = max(3, args.warmup)

    rank, world, local = R.replica_env()
    if args.which == "backward":
        if args.impl != "fused":
            ap.error("--pass backward times the fused library path only")
        run_backward(args, rank, world, local, warmup)
        return
    if args.which == "paged":
        if args.impl != "fused":
            ap.error("--pass paged times the fused library path only")
        run_paged(args, rank, world, local, warmup)
        return
    cfg, a_flops, a_bytes, decode_cfg = workload_config(args.workload)
    unit = "GB/s" if decode_cfg else "TFLOP/s"
    work_per_step = (a_bytes / 1e9) if decode_cfg else (a_flops / 1e12)

    if args.impl == "reference":
        # The oracle on the host cores, rank 0 only; other ranks exit without work.
        if rank != 0:
            return
        a = I.make_workload(args.workload, dtype=args.dtype)
        B, Hq = cfg["B"], cfg["H_q"]
        # a bounded sample per step: about 40 s of oracle time over the whole run
        rows_sample = max(16, min(B * Hq * cfg["N_q"], 2048, (2048 * 200) // max(1, args.steps)))
        per_row = work_per_step / (B * Hq * cfg["N_q"])
        for _ in range(warmup):
            cpu_oracle_throughput(a, 0.0, rows_sample)
        times = []
        for _ in range(args.steps):
            n_rows, dt, cores, _ = cpu_oracle_throughput(a, 0.0, rows_sample)
            times.append(dt / n_rows)
        t_row = statistics.mean(times)
        value = per_row / t_row
        sample = (f"{rows_sample} query rows per step, taken head by head "
                  f"(of {B * Hq * cfg['N_q']} rows in the workload)")
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": warmup,
                "ms_per_step": t_row * rows_sample * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload, **cfg},
                "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import exact_tiled_attention_forward_gb300 as fa

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    fa.lib()

    a = I.make_workload(args.workload, dtype=args.dtype)
    B, Hq, Hkv, Nq, Nk, d = a.shape_args
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or (129 << 20))

    def to_dev(x):
        return to_device(torch, x, dev)

    q, k, v = to_dev(a.q), to_dev(a.k), to_dev(a.v)
    fn = forward_fn(fa, a) if args.impl == "fused" else fa.fa_naive_forward
    ws = None
    if args.impl == "naive":
        ws = torch.empty(fa.fa_naive_workspace_bytes(B, Hq, Nq, Nk), dtype=torch.uint8, device=dev)
    kernels_per_step = 3 if args.impl == "naive" else fused_launches_per_step(fa, cfg)

    # Input sets: copies of the same Q, K, V (and their own O, LSE), used in turn,
    # enough of them that the inputs of all sets together take at least twice
    # the L2 size: a step's inputs have left L2 by the time its set comes round again.
    set_bytes = (q.numel() + k.numel() + v.numel()) * q.element_size()
    n_sets = min(4096, max(2, -(-2 * l2_bytes // set_bytes)))
    # one copy kernel per input: [n_sets, ...] tensors whose slices are the sets
    qs, ks, vs = (x.unsqueeze(0).expand(n_sets, *x.shape).contiguous() for x in (q, k, v))
    sets = [(qs[i], ks[i], vs[i], torch.empty((B, Hq, Nq, d), dtype=elem_dtype(torch, a), device=dev),
             torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)) for i in range(n_sets)]
    del q, k, v

    def step(i):
        qq, kk, vv, oo, ll = sets[i % n_sets]
        if ws is None:
            fn(qq, kk, vv, causal=a.causal, scale=a.scale, out=oo, lse=ll)
        else:
            fn(qq, kk, vv, causal=a.causal, scale=a.scale, out=oo, lse=ll, workspace=ws)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # > 129 MB L2
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for i in range(warmup):
        step(i)
    barrier()

    sampler = ClockSampler(*device_ids(props))
    sampler.start()
    # ---- timed region: K steps back to back between two events on the launching
    # stream, each step on the next input set (inputs larger than L2)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    wall0 = time.perf_counter()
    hold_device(torch)
    e_start.record(stream)
    for i in range(args.steps):
        step(i)
    e_end.record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    total_ms = R.slowest_rank_ms(e_start.elapsed_time(e_end), world, dev)
    ms_per_step = total_ms / args.steps
    value = R.whole_job_rate(work_per_step, args.steps, total_ms, world)
    if fa.fa_device_status() != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait during the benchmark")

    # ---- flushed: every step alone between its own events, L2 flushed before it
    # (outside the events); no overlap with the step before
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier()
    for e0, e1 in fev:
        flush.zero_()
        e0.record(stream)
        step(0)
        e1.record(stream)
    barrier()
    flushed_ms = R.slowest_rank_ms(sum(e0.elapsed_time(e1) for e0, e1 in fev), world, dev)
    flushed_value = R.whole_job_rate(work_per_step, args.steps, flushed_ms, world)

    # ---- the same steps captured once into a CUDA graph and replayed: no host
    # enqueue per call, which is what bounds the smallest workloads
    graph = None
    if args.impl == "fused":
        n_cap = min(args.steps, 100)
        reps = max(1, args.steps // n_cap)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_cap):
                step(i)
        g.replay()
        barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch)
        g0.record(stream)
        for _ in range(reps):
            g.replay()
        g1.record(stream)
        barrier()
        if fa.fa_device_status() != fa.FA_OK:
            raise RuntimeError("a kernel reported a timed-out wait during the graph replays")
        g_ms = R.slowest_rank_ms(g0.elapsed_time(g1), world, dev)
        graph = {"value": R.whole_job_rate(work_per_step, n_cap * reps, g_ms, world), "unit": unit,
                 "ms_per_step": g_ms / (n_cap * reps),
                 "note": f"the same steps captured once into a CUDA graph of {n_cap} calls, replayed {reps} times"}
        del g

    # ---- end to end through the C ABI with host buffers: every step copies its
    # inputs in from pinned host memory and its O | LSE back out, inside the
    # timed region (fa_forward_host_packed; see time_e2e)
    e2e_value, e2e_ms_step, h2d, d2h, e2e_serial = time_e2e(
        torch, fa, a, cfg, dev, stream, fn, ws, args.steps, warmup, world, work_per_step)

    # ---- secondary half of the metric: decode HBM GB/s (batch 16, 32/8 heads, 8192 keys)
    decode = None
    if args.impl == "fused" and not decode_cfg and args.decode_steps > 0:
        decode = time_decode(fa, torch, dev, flush, stream, args.decode_steps, warmup, world,
                             args.dtype)

    if rank != 0:
        torch.distributed.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    if decode_cfg:
        peak = float(peaks["hbm_gbs"])
        achieved = a_bytes / 1e9 / (ms_per_step * 1e-3)
        roof = {"bound": "hbm", "unit": "GB/s"}
    else:
        # FP8 MMAs: the measured BF16 peak times the nominal FP8 / BF16 ratio (4.5 / 2.25 PF)
        peak = float(peaks["bf16_tflops"]) * (2.0 if args.dtype == "e4m3" else 1.0)
        achieved = a_flops / 1e12 / (ms_per_step * 1e-3)
        roof = {"bound": "tensor", "unit": "TFLOP/s"}
    main_kernel = "fa_fwd_tile_kernel" if d == 256 else "fa_fwd_kernel"
    traffic = (profiled_traffic(args.workload + ("_e4m3" if args.dtype == "e4m3" else ""), main_kernel)
               if args.impl == "fused" else None)
    if args.dtype == "bf16" or decode_cfg:
        peak_src_note = f"{peak_src} (burst)"
    elif args.dtype == "e4m3":
        peak_src_note = f"{peak_src} BF16 burst x nominal FP8/BF16 ratio 2 (4.5 / 2.25 PF)"
    else:
        peak_src_note = f"{peak_src} BF16 burst x nominal FP16/BF16 ratio 1 (2.25 PF both)"
    roof.update({"achieved": achieved, "peak": peak, "frac": achieved / peak,
                 "traffic": traffic,
                 "peak_source": peak_src_note,
                 "algorithmic_per_launch": a_bytes if decode_cfg else a_flops,
                 "kernel": main_kernel if args.impl == "fused" else "naive (3 kernels)"})

    cpu = None
    if args.cpu_budget > 0 and world == 1:
        per_row = work_per_step / (B * Hq * Nq)
        n_rows, dt, cores, calls = cpu_oracle_throughput(a, args.cpu_budget)
        cpu = {"value": per_row * n_rows / dt, "unit": unit, "cores": cores, "kind": "oracle",
               "sample": f"{n_rows} query rows ({calls} heads x {Nq} rows) in {dt:.1f} s, "
                         f"FP64 materialised oracle, numpy/OpenBLAS"}

    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "impl": args.impl,
        "config": {"workload": args.workload, **{k2: cfg[k2] for k2 in
                   ("B", "H_q", "H_kv", "N_q", "N_k", "d", "causal")},
                   "scale": a.scale,
                   "l2": (f"inputs larger than L2: {n_sets} copies of Q/K/V (each with its own O, "
                          f"LSE) used in turn, {n_sets * set_bytes / 2**20:.0f} MiB of inputs "
                          f"against {l2_bytes / 2**20:.0f} MiB of L2; steps back to back "
                          f"between two events"),
                   "timing": ("a ~100 us device-side wait is queued before the start event, so the "
                              "first step's kernels are already enqueued when the region starts"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms_step,
                "note": ("fa_forward_host_packed: K requests in pinned host memory; libfa copies each in "
                         "and out on its own streams through three device slots, overlapping the "
                         "neighbouring requests' kernels" if args.impl == "fused" and args.dtype != "e4m3"
                         else "torch copies around each call (pinned host buffers), nothing overlapped"),
                "serial": e2e_serial},
        "gpu_launches": kernels_per_step * args.steps,
        "graph": graph,
        "flushed": {"value": flushed_value, "unit": unit, "ms_per_step": flushed_ms / args.steps,
                    "note": ("each step alone between its own events, L2 flushed (256 MiB write) "
                             "before it, outside the events")},
        "decode": None if decode is None else {
            "workload": DECODE_WORKLOAD, "value": decode["gbs"], "unit": "GB/s",
            "split": decode["split"],
            "ms_per_step": decode["ms"], "steps": args.decode_steps,
            "l2": "inputs larger than L2: two input sets of 537 MB used in turn, back to back",
            "flushed": {"value": decode["flushed_gbs"], "unit": "GB/s",
                        "ms_per_step": decode["flushed_ms"],
                        "note": "each step alone between its own events, L2 flushed before it"},
            "roofline": {"bound": "hbm", "achieved": decode["gbs"],
                         "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": decode["gbs"] / float(peaks["hbm_gbs"]),
                         "traffic": profiled_traffic(DECODE_WORKLOAD, "fa_decode_kernel"),
                         "algorithmic_per_launch": decode["bytes"],
                         "kernel": ("fa_decode_kernel (in-cluster merge)" if decode["launches"] == 1
                                    else "fa_decode_kernel + fa_decode_merge_kernel")},
            "gpu_launches": decode["launches"] * args.decode_steps},
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
