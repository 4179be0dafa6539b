"""Throughput of the exact-attention training step on GB300.

One step = the whole hot path over one batch of the training-step workload
(bf16, B=8 H=16 N=2048 d=128, causal, scale 1/sqrt(d), seeded N(0,1) Q, K, V,
dO): the forward (O, LSE), then the backward preprocess (D, base-2 LSE), the
dK/dV kernel and the dQ kernel.  The metric counts 4 B H N^2 d FLOPs
for the forward and 2.5x that for the backward, halved for the causal mask.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch
(weak scaling over independent (batch, head) work, no collective on the data
path); the barrier and the max over ranks of the timed region stay.
``--impl reference`` times the FP64 CPU oracle on a bounded sample of the same
workload instead (rank 0 only).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("attention fwd/bwd TFLOP/s (4BHN²d, causal halved) and % of GB300 BF16 tensor "
          "peak")
B, H, N, D, CAUSAL, SEED = 8, 16, 2048, 128, True, 4
WORKLOAD = "training step fwd+bwd, bf16, B=8 H=16 N=2048 d=128, causal, scale=1/sqrt(d), seed 4"

# DRAM traffic of one launch of a kernel at this workload, read from an ncu
# capture of that kernel (dram__bytes_read.sum + dram__bytes_write.sum); valid
# only for the kernel source it was measured on (sha256 of its .cu file
# followed by the shared primitives header), else the roofline reports
# traffic as null.
CSRC = os.path.join(ROOT, "exact_io_aware_18_gb300", "csrc")
KERNEL_SRC = {"fwd_bf16": os.path.join(CSRC, "fwd_bf16_sm103.cu"),
              "bwd_dkdv_bf16": os.path.join(CSRC, "bwd_bf16_sm103.cu"),
              "bwd_dq_bf16": os.path.join(CSRC, "bwd_dq_sm103.cu")}
KERNEL_HDR = os.path.join(CSRC, "sm103_primitives.cuh")


def kernel_src_sha256(name: str) -> str:
    h = hashlib.sha256()
    for path in (KERNEL_SRC[name], KERNEL_HDR):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


KERNEL_TRAFFIC = {
    "fwd_bf16": {"bytes": 201439104 + 45610624,
                "src_sha256": "4fa05ef15dae16eef945402bf2d68bb070310270cf2644410f960675ae80837f"},
    "bwd_dkdv_bf16": {"bytes": 270648832 + 215226752,
                     "src_sha256": "56e1b2c5fc36f36544a7650bbb85c7adea8f0e3cb8e1966f72661a2b9741b0c1"},
    "bwd_dq_bf16": {"bytes": 336801024 + 108525824,
                   "src_sha256": "bd45c6dba97e1747f31ce388732ef8367b55e6e903d637375e298cc1be77c917"},
}

REFERENCE_BUDGET_S = 120.0  # wall-clock bound on the reference arm's timed steps
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Datasheet dense BF16 tensor rate of one GPU: NVIDIA quotes 36 PFLOP/s BF16
# for an 8-GPU HGX B300 board with 2:4 sparsity, i.e. 2.25 PFLOP/s dense per GPU.
NOMINAL_BF16_TFLOPS = 2250.0


def dist_env():
    """(world, rank, local rank) from the launcher's environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank: int) -> int:
    """Each rank draws its own batch (weak scaling: independent heads per rank)."""
    return SEED + rank


def max_over_ranks(torch, value: float, device, world: int) -> float:
    """The largest of every rank's value, on every rank (the slowest rank sets
    the job's time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank: float, ms_per_step: float) -> float:
    """Work of all ranks over the (max-over-ranks) time of one step."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def step_flops(b=B, h=H, n=N, d=D, causal=CAUSAL):
    fwd = 4.0 * b * h * n * n * d
    if causal:
        fwd /= 2
    return fwd, 2.5 * fwd


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.samples = []  # (t, sm, max, reasons)
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            reasons = [n for n, v in zip(self.NAMES, parts[4:8]) if v.lower() == "active"]
            self.samples.append((time.monotonic(), sm, mx, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside
        if len(used) < 3:  # a short timed region: take the samples nearest to it
            used = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:5]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({r for s in used for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in used),
                "sm_max_mhz": max(s[2] for s in used), "reasons": reasons,
                "samples": len(used), "samples_inside_timed_region": len(inside)}


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML every millisecond,
    so that even a timed region of a few milliseconds holds several samples.
    Reads only; falls back to nothing when NVML cannot be loaded."""

    # nvmlClocksEventReasons bits -> the names nvidia-smi uses
    BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, device, period_s: float = 0.001):
        self.samples = []  # (t, sm, max, reasons)
        self.period_s = period_s
        self.stop_flag = threading.Event()
        self.thread = None
        self.nvml = None
        self.handle = None
        try:
            import ctypes
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device)
            bus = None
            if all(hasattr(props, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
                bus = (f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:"
                       f"{props.pci_device_id:02X}.0").encode()
            if bus is None or nvml.nvmlDeviceGetHandleByPciBusId_v2(
                    ctypes.c_char_p(bus), ctypes.byref(handle)) != 0:
                return
            self.nvml, self.handle, self.ctypes = nvml, handle, ctypes
        except (OSError, AttributeError):
            self.nvml = None

    def _read(self):
        c = self.ctypes
        sm, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        get_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_flag.is_set():
            ok = (self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, c.byref(sm)) == 0 and
                  self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, c.byref(mx)) == 0 and
                  get_reasons(self.handle, c.byref(rs)) == 0)
            if ok:
                reasons = [n for b, n in self.BITS.items() if rs.value & b]
                self.samples.append((time.monotonic(), float(sm.value), float(mx.value), reasons))
            time.sleep(self.period_s)

    def start(self):
        if self.nvml is None:
            return False
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return True

    def stop(self):
        self.stop_flag.set()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return None
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside),
                "reasons": sorted({r for s in inside for r in s[3]}),
                "samples": len(inside), "samples_inside_timed_region": len(inside),
                "source": "NVML, 1 ms period"}


# ---------------------------------------------------------------- CPU oracle

def oracle_step_sample(x, n_heads):
    """One oracle fwd+bwd over the first n_heads heads; returns (seconds, flops)."""
    import oracle
    qs = x["q"].reshape(B * H, 1, N, D)[:n_heads].reshape(1, n_heads, N, D)
    ks = x["k"].reshape(B * H, 1, N, D)[:n_heads].reshape(1, n_heads, N, D)
    vs = x["v"].reshape(B * H, 1, N, D)[:n_heads].reshape(1, n_heads, N, D)
    dos = x["do"].reshape(B * H, 1, N, D)[:n_heads].reshape(1, n_heads, N, D)
    scale = float(np.float32(1.0 / math.sqrt(D)))
    t0 = time.perf_counter()
    oracle.attention_fwd(qs, ks, vs, CAUSAL, scale)
    oracle.attention_bwd(qs, ks, vs, dos, CAUSAL, scale, o_storage="bf16")
    dt = time.perf_counter() - t0
    f, b = step_flops(1, n_heads)
    return dt, f + b


def oracle_cores():
    import oracle
    oracle.build()
    return oracle.num_threads()


# ---------------------------------------------------------------- GPU arm

def _timed(torch, stream, fn, iters):
    """Mean device time of fn over iters back-to-back launches.  A GPU-side
    sleep queued first keeps the device busy while the host queues every
    launch, so that calls shorter than their host-side cost (argument checks,
    tensor-map encoding) are still timed on the device alone."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(4_000_000)  # about 2 ms of GPU clock cycles
    e0.record(stream)
    for _ in range(iters):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def measure_next_rows(fa, torch, q, k, v, do, stream, iters=20):
    """Rows beyond the training step, timed after (outside) its timed region on
    the same seeded inputs.  Grouped-query attention: the training-step shape
    with 4 query heads per K/V head (K, V: their first H/4 heads)."""
    import fa_inputs
    scale = fa.default_scale(D)
    peaks, _ = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    hkv = H // 4
    kg = k[:, :hkv].contiguous()
    vg = v[:, :hkv].contiguous()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(kg.shape, dtype=torch.float32, device=q.device)
    dv = torch.empty_like(dk)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, D) // 4, dtype=torch.float32,
                     device=q.device)
    f_fwd, f_bwd = step_flops()
    fwd_ms = _timed(torch, stream, lambda: fa.fa_fwd_gqa(q, kg, vg, o, lse, CAUSAL, scale,
                                                           stream), iters)
    bwd_ms = _timed(torch, stream, lambda: fa.fa_bwd_gqa(q, kg, vg, o, do, lse, dq, dk, dv,
                                                           CAUSAL, scale, ws, stream), iters)
    # The backward's first step as a launch of its own (the step-wise calls; the
    # timed step fuses it into dQ): HBM-bound, O and dO read, D and LSE2 written.
    n_pad = (N + 127) // 128 * 128
    delta = ws[:B * H * n_pad].view(B * H, n_pad)
    lse2 = ws[B * H * n_pad:].view(B * H, n_pad)
    pre_ms = _timed(torch, stream, lambda: fa.fa_bwd_preprocess(o, do, lse, delta, lse2, stream),
                    iters)
    pre_bytes = 2 * B * H * N * D * 2 + B * H * N * 4 + 2 * B * H * n_pad * 4
    # Split-KV decode: one new query per head against a long cache, grouped
    # K/V heads.  HBM-bound (K and V are read once); seeded synthetic inputs.
    db, dhq, dhkv, dnq, dnk = 4, 32, 8, 1, 16384
    gen = torch.Generator(device=q.device)
    gen.manual_seed(SEED)

    def rnd(*shape):
        return torch.randn(*shape, generator=gen, device=q.device).to(torch.bfloat16)

    dq_ = rnd(db, dhq, dnq, D)
    dk_ = rnd(db, dhkv, dnk, D)
    dv_ = rnd(db, dhkv, dnk, D)
    do_ = torch.empty_like(dq_)
    dlse = torch.empty((db, dhq, dnq), dtype=torch.float32, device=q.device)
    dws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(db, dhq, dhkv, dnq, dnk, D) // 4 + 4,
                      dtype=torch.float32, device=q.device)
    dec_ms = _timed(torch, stream, lambda: fa.fa_fwd_splitkv(dq_, dk_, dv_, do_, dlse, scale, 0,
                                                              dws, stream), iters)
    dec_bytes = (2 * db * dhkv * dnk * D * 2 + 2 * db * dhq * dnq * D * 2 + db * dhq * dnq * 4)
    dec_flops = 4.0 * db * dhq * dnq * dnk * D
    # FP8 forward with incoherent processing at the training-step shape: Q and
    # K rotated and quantised (HBM-bound), then the forward from their codes.
    signs = fa._lib._host_signs(fa_inputs.random_signs(SEED, D), D)
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=q.device)
    qs = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=q.device)
    ks = torch.empty_like(qs)
    quant_ms = _timed(torch, stream, lambda: fa.fa_fp8_quantize(q, signs, q8, qs, stream), iters)
    fa.fa_fp8_quantize(k, signs, k8, ks, stream)
    fp8_ms = _timed(torch, stream, lambda: fa.fa_fwd_fp8(q8, qs, k8, ks, v, o, lse, CAUSAL, scale,
                                                          stream), iters)
    bf16_ms = _timed(torch, stream, lambda: fa.fa_fwd(q, k, v, o, lse, CAUSAL, scale, stream),
                     iters)
    # per tensor: BF16 read, E4M3 codes and one FP32 scale per 128-row tile written
    quant_bytes = B * H * N * D * 3 + B * H * ((N + 127) // 128) * 4
    # The forward alone on the forward-only workloads (the long-sequence ones
    # carry the tensor-core target), seeded device inputs.
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    fwd_rows = {}
    for name, (fb, fh, fn, fd, fc) in (("B2_H8_N1024_d64", (2, 8, 1024, 64, False)),
                                       ("B4_H16_N4096_causal", (4, 16, 4096, 128, True)),
                                       ("B1_H16_N32768_causal", (1, 16, 32768, 128, True))):
        fq, fk, fv = rnd(fb, fh, fn, fd), rnd(fb, fh, fn, fd), rnd(fb, fh, fn, fd)
        fo = torch.empty_like(fq)
        flse = torch.empty((fb, fh, fn), dtype=torch.float32, device=q.device)
        fs = fa.default_scale(fd)
        f_ms = _timed(torch, stream, lambda: fa.fa_fwd(fq, fk, fv, fo, flse, fc, fs, stream),
                      max(3, iters // 2))
        f_tf = step_flops(fb, fh, fn, fd, fc)[0] / (f_ms * 1e-3) / 1e12
        fwd_rows[name] = {"ms": round(f_ms, 4), "tflops": round(f_tf, 2),
                          "frac_of_burst_peak": round(f_tf / burst, 4),
                          "frac_of_nominal_2250": round(f_tf / 2250.0, 4)}
        del fq, fk, fv, fo, flse
    if fa.fa_device_status(clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait in the next-row measurements")
    return {
        "forward_workloads": dict(fwd_rows, peak="bf16_tflops (burst, measured); "
                                  "nominal dense BF16 2250 TFLOP/s",
                                  flops="4 B H N^2 d, causal halved"),
        "fp8_forward": {
            "workload": f"B={B} H={H} N={N} d={D} causal: Q, K rotated by a random-sign Hadamard "
                        "transform and quantised to E4M3 per 128-row tile; S from the codes on "
                        "kind::f8f6f4; P V in BF16",
            "quantize_ms_per_tensor": round(quant_ms, 4),
            "quantize_bound": "hbm",
            "quantize_algorithmic_bytes": quant_bytes,
            "quantize_gbs": round(quant_bytes / (quant_ms * 1e-3) / 1e9, 1),
            "quantize_frac_of_hbm": round(quant_bytes / (quant_ms * 1e-3) / 1e9 / hbm, 4),
            "fwd_ms": round(fp8_ms, 4),
            "fwd_tflops": round(f_fwd / (fp8_ms * 1e-3) / 1e12, 2),
            "bf16_fwd_ms_same_inputs": round(bf16_ms, 4),
            "total_ms_quantize_q_k_and_fwd": round(2 * quant_ms + fp8_ms, 4)},
        "splitkv_decode": {
            "workload": f"B={db} Hq={dhq} Hkv={dhkv} Nq={dnq} Nk={dnk} d={D}, bf16, no mask, "
                        "library-chosen splits",
            "algorithmic_bytes_counted": "K and V read once, Q read, O and LSE written",
            "ms": round(dec_ms, 4),
            "bound": "hbm",
            "algorithmic_bytes": dec_bytes,
            "gbs": round(dec_bytes / (dec_ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(dec_bytes / (dec_ms * 1e-3) / 1e9 / hbm, 4),
            "tflops": round(dec_flops / (dec_ms * 1e-3) / 1e12, 2)},
        "bwd_preprocess_standalone": {
            "workload": f"B={B} H={H} N={N} d={D}: D = rowsum(dO o O) and LSE log2(e) as a launch "
                        "of its own (the timed step fuses it into dQ)",
            "ms": round(pre_ms, 4),
            "bound": "hbm",
            "algorithmic_bytes": pre_bytes,
            "gbs": round(pre_bytes / (pre_ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(pre_bytes / (pre_ms * 1e-3) / 1e9 / hbm, 4)},
        "gqa": {"workload": f"B={B} Hq={H} Hkv={hkv} N={N} d={D} causal, bf16",
                "fwd_ms": round(fwd_ms, 4),
                "fwd_tflops": round(f_fwd / (fwd_ms * 1e-3) / 1e12, 2),
                "bwd_ms": round(bwd_ms, 4),
                "bwd_tflops": round(f_bwd / (bwd_ms * 1e-3) / 1e12, 2),
                "flops": "4 B Hq N^2 d (causal halved), backward 2.5x"},
    }


def frac(tflops, peak):
    return round(tflops / peak, 4)


def time_training_step(fa, torch, stream, t, causal, steps, warmup):
    """Mean CUDA-event time of each kernel of the step (forward, dQ with the
    first backward step fused, dK/dV) over `steps` back-to-back steps after
    `warmup` untimed ones; t holds the step's device tensors."""
    q, k, v, do, o, lse, dq, dk, dv, delta, lse2 = t
    d = q.shape[-1]
    scale = fa.default_scale(d)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, causal, scale, stream)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_bwd_dq_preprocess(q, k, v, o, do, lse, delta, lse2, dq, causal, scale, stream)
        if ev is not None:
            ev[2].record(stream)
        fa.fa_bwd_dkdv(q, k, v, do, delta, lse2, dk, dv, causal, scale, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for i in range(steps):
        step(events[i])
    torch.cuda.synchronize()
    return tuple(statistics.mean(e[a].elapsed_time(e[a + 1]) for e in events) for a in range(3))


def measure_training_rows(fa, torch, dev, stream, steps, warmup):
    """Forward + backward at B=4 H=16 N=4096 d=128 (the shape of the N = 4096
    workload, seed 2, with dO drawn after Q, K, V), causal and not: the
    sequence length where the tensor-core targets are set.  Timed like the
    headline step; each kernel against the measured burst peak and the
    datasheet figure."""
    import fa_inputs
    b, h, n, d = 4, 16, 4096, 128
    x = fa_inputs.attention_inputs(2, b, h, n, d, "bf16")

    def put(name):
        return torch.from_numpy(x[name + "_bits"].view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v, do = (put(nm) for nm in ("q", "k", "v", "do"))
    del x
    o = torch.empty_like(q)
    lse = torch.empty((b, h, n), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty((b, h, n, d), dtype=torch.float32, device=dev) for _ in range(3))
    n_pad = (n + 127) // 128 * 128
    ws = torch.empty(fa.fa_bwd_workspace_bytes(b, h, n, d) // 4, dtype=torch.float32, device=dev)
    delta = ws[:b * h * n_pad].view(b * h, n_pad)
    lse2 = ws[b * h * n_pad:].view(b * h, n_pad)
    peaks, kind = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    rows = {}
    for causal in (True, False):
        f_fwd, f_bwd = step_flops(b, h, n, d, causal)
        fwd_ms, dq_ms, dkdv_ms = time_training_step(
            fa, torch, stream, (q, k, v, do, o, lse, dq, dk, dv, delta, lse2), causal,
            steps, warmup)
        bwd_ms = dq_ms + dkdv_ms
        tf = {"fwd": f_fwd / (fwd_ms * 1e-3) / 1e12,
              "bwd_dq": 1.5 * f_fwd / (dq_ms * 1e-3) / 1e12,
              "bwd_dkdv": 2.0 * f_fwd / (dkdv_ms * 1e-3) / 1e12,
              "bwd": f_bwd / (bwd_ms * 1e-3) / 1e12}
        rows["causal" if causal else "non_causal"] = {
            "fwd_ms": round(fwd_ms, 4), "bwd_dq_ms": round(dq_ms, 4),
            "bwd_dkdv_ms": round(dkdv_ms, 4), "bwd_ms": round(bwd_ms, 4),
            "fwd_tflops": round(tf["fwd"], 2),
            "fwd_frac_of_burst": frac(tf["fwd"], burst),
            "fwd_frac_of_nominal": frac(tf["fwd"], NOMINAL_BF16_TFLOPS),
            "bwd_tflops": round(tf["bwd"], 2),
            "bwd_frac_of_burst": frac(tf["bwd"], burst),
            "bwd_frac_of_nominal": frac(tf["bwd"], NOMINAL_BF16_TFLOPS),
            "bwd_dq_own_tflops": round(tf["bwd_dq"], 2),
            "bwd_dkdv_own_tflops": round(tf["bwd_dkdv"], 2),
        }
    if fa.fa_device_status(clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait in the N = 4096 training rows")
    return dict(rows, workload="fwd+bwd, bf16, B=4 H=16 N=4096 d=128, seed 2 (Q, K, V, dO)",
                steps=steps, warmup=warmup,
                flops="forward 4 B H N^2 d, backward 2.5x that, causal halved; each kernel's "
                      "own products: dQ 1.5x, dK/dV 2x the forward",
                peaks=f"burst bf16_tflops ({kind}) {burst}; datasheet dense BF16 "
                      f"{NOMINAL_BF16_TFLOPS}")


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import exact_io_aware_18_gb300 as fa
    import fa_inputs

    scale = fa.default_scale(D)
    x = fa_inputs.attention_inputs(rank_seed(rank), B, H, N, D, "bf16")

    def host_bf16(name):
        return torch.from_numpy(x[name + "_bits"].view(np.int16)).view(torch.bfloat16)

    hq, hk, hv, hdo = (host_bf16(n).pin_memory() for n in ("q", "k", "v", "do"))
    q, k, v, do = (t.to(dev) for t in (hq, hk, hv, hdo))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq = torch.empty((B, H, N, D), dtype=torch.float32, device=dev)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    n_pad = (N + 127) // 128 * 128
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, D) // 4, dtype=torch.float32, device=dev)
    delta = ws[:B * H * n_pad].view(B * H, n_pad)
    lse2 = ws[B * H * n_pad:].view(B * H, n_pad)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fa.fa_fwd(q, k, v, o, lse, CAUSAL, scale, stream)
        if ev is not None:
            ev[1].record(stream)
        # dQ with the first backward step fused (it writes D and LSE2), then dK/dV.
        fa.fa_bwd_dq_preprocess(q, k, v, o, do, lse, delta, lse2, dq, CAUSAL, scale, stream)
        if ev is not None:
            ev[2].record(stream)
        fa.fa_bwd_dkdv(q, k, v, do, delta, lse2, dk, dv, CAUSAL, scale, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status(clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait during warm-up")

    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_index = int(vis.split(",")[local])
        except ValueError:
            pass
    sampler = ClockSampler(gpu_index)
    sampler.start()
    fine = NvmlClockSampler(torch, dev)
    fine.start()
    time.sleep(0.3)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.monotonic()
    start.record(stream)
    for i in range(args.steps):
        step(events[i])
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.monotonic()
    if world > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(torch, start.elapsed_time(end), dev, world)
    if fa.fa_device_status(clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait in the timed region")

    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in events)
    dq_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in events)
    dkdv_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in events)

    # End to end through the public calls: every step copies its inputs in
    # from pinned host memory and its results (O, LSE, dQ, dK, dV) back.  As
    # in a training loop, the copies run on their own streams: step i+1's
    # inputs go in and step i-1's results come out while step i computes.
    # Two device buffer sets; events keep a set from being overwritten while
    # another stream still reads it.
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    hdq = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
    hdk = torch.empty_like(hdq).pin_memory()
    hdv = torch.empty_like(hdq).pin_memory()
    sets = [(q, k, v, do, o, lse, dq, dk, dv),
            tuple(torch.empty_like(t) for t in (q, k, v, do, o, lse, dq, dk, dv))]
    s_main = torch.cuda.current_stream(dev)
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        for i in range(n):
            b = i % 2
            xq, xk, xv, xdo, xo, xlse, dq_, dk_, dv_ = sets[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[b])  # step i-2 has read this set's inputs
                for dst, src in ((xq, hq), (xk, hk), (xv, hv), (xdo, hdo)):
                    dst.copy_(src, non_blocking=True)
                in_done[b].record(s_in)
            s_main.wait_event(in_done[b])
            if i >= 2:
                s_main.wait_event(out_done[b])  # step i-2's results have left this set
            fa.fa_fwd(xq, xk, xv, xo, xlse, CAUSAL, scale, stream)
            fa.fa_bwd(xq, xk, xv, xo, xdo, xlse, dq_, dk_, dv_, CAUSAL, scale, ws, stream)
            comp_done[b].record(s_main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                for dst, src in ((ho, xo), (hlse, xlse), (hdq, dq_), (hdk, dk_), (hdv, dv_)):
                    dst.copy_(src, non_blocking=True)
                out_done[b].record(s_out)
        s_main.wait_stream(s_out)

    e2e_steps = max(3, min(args.steps, 50))
    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_main)
    e2e_run(e2e_steps)
    e1.record(s_main)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(torch, e0.elapsed_time(e1) / e2e_steps, dev, world)
    sampler.stop()
    fine.stop()
    next_rows = None
    if rank == 0:
        next_rows = measure_next_rows(fa, torch, q, k, v, do, stream)
        next_rows["training_step_n4096"] = measure_training_rows(
            fa, torch, dev, stream, max(1, min(args.steps, 200)), args.warmup)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    f_fwd, f_bwd = step_flops()
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tflops(world, f_fwd + f_bwd, ms_per_step)
    peaks, peak_kind = load_peaks()
    # The timed region is a few milliseconds to a second of kernels: the
    # burst figure (a GEMM timed alone) is the denominator, not the rate a
    # GEMM settles at after seconds under the power cap.
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # Each kernel's own GEMM FLOPs per launch: the forward does 2 GEMMs per
    # (Q tile, key tile) pair, dK/dV 4 (S^T, dP^T, dV, dK), dQ 3 (S, dP, dQ;
    # S and dP recomputed).  The step metric counts 2.5x the forward for the
    # whole backward, as the workload's metric does.
    kern_flops = {"fwd_bf16": f_fwd, "bwd_dkdv_bf16": 2.0 * f_fwd, "bwd_dq_bf16": 1.5 * f_fwd}
    kern_ms = {"fwd_bf16": fwd_ms, "bwd_dkdv_bf16": dkdv_ms, "bwd_dq_bf16": dq_ms}
    dominant = max(kern_ms, key=kern_ms.get)
    achieved = kern_flops[dominant] / (kern_ms[dominant] * 1e-3) / 1e12
    traffic = None
    try:
        sha = kernel_src_sha256(dominant)
        rec = KERNEL_TRAFFIC.get(dominant)
        if rec and rec["bytes"] and rec["src_sha256"] == sha:
            traffic = rec["bytes"]
    except (OSError, KeyError):
        pass
    clocks = fine.summary(t_wall0, t_wall1) or sampler.summary(t_wall0, t_wall1)
    mhz = clocks.get("sm_mhz") or None

    # CPU baseline: the oracle as it stands on a bounded sample (whole heads).
    cores = oracle_cores()
    n_heads = max(1, min(B * H, cores))
    cpu_s, cpu_flops = oracle_step_sample(x, n_heads)

    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D, "causal": CAUSAL,
                   "l2": "inputs larger than L2: Q, K, V, dO are 4 x 64 MiB per step"},
        "roofline": {"bound": "tensor", "kernel": dominant, "achieved": round(achieved, 2),
                     "peak": peak, "peak_kind": f"bf16_tflops, burst ({peak_kind})",
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "frac_of_nominal": frac(achieved, NOMINAL_BF16_TFLOPS),
                     "nominal_peak": NOMINAL_BF16_TFLOPS,
                     "flops_counted": "the kernel's own products per launch (dK/dV: S^T, dP^T, "
                                      "dV, dK = 2x the forward; dQ: S, dP, dQ = 1.5x)",
                     "traffic": traffic},
        "cpu_baseline": {"value": round(cpu_flops / cpu_s / 1e12, 6), "unit": "TFLOP/s",
                         "cores": cores, "kind": "oracle",
                         "sample": f"{n_heads} of {B * H} heads (whole heads, fwd+bwd), "
                                   f"{cpu_s:.1f} s"},
        "e2e": {"value": round(whole_job_tflops(world, f_fwd + f_bwd, e2e_ms), 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "copies": "own streams: step i+1's inputs in and step i-1's results out "
                          "while step i computes (two device buffer sets)"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "kernels": kernel_table(fwd_ms, dq_ms, dkdv_ms, f_fwd, f_bwd, value, peak, mhz),
        "next_rows": next_rows,
    }
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def kernel_table(fwd_ms, dq_ms, dkdv_ms, f_fwd, f_bwd, step_tflops, burst, mhz):
    """Each kernel's time and rate, as fractions of the measured burst peak
    and of the datasheet figure, with time x median SM clock beside them.
    The metric's own rates: forward 4 B H N^2 d, backward 2.5x (causal
    halved); a kernel's own rate counts the products it executes."""
    def row(ms, work, **extra):
        tf = work / (ms * 1e-3) / 1e12
        r = {"ms": round(ms, 4), "tflops": round(tf, 2), "frac_of_burst": frac(tf, burst),
             "frac_of_nominal": frac(tf, NOMINAL_BF16_TFLOPS)}
        if mhz:
            r["kcycles_at_median_sm_clock"] = round(ms * mhz, 1)
        r.update(extra)
        return r

    bwd_ms = dq_ms + dkdv_ms
    return {
        "fwd": row(fwd_ms, f_fwd),
        "bwd_dq": row(dq_ms, 1.5 * f_fwd, flops="own products S, dP, dQ (1.5x the forward)",
                      includes="the first backward step: D = rowsum(dO o O), LSE log2(e)"),
        "bwd_dkdv": row(dkdv_ms, 2.0 * f_fwd, flops="own products S^T, dP^T, dV, dK (2x)"),
        "bwd": row(bwd_ms, f_bwd, flops="the metric's 2.5x the forward"),
        "bwd_total_tflops": round(f_bwd / (bwd_ms * 1e-3) / 1e12, 2),
        "step": {"tflops": round(step_tflops, 2), "frac_of_burst": frac(step_tflops, burst),
                 "frac_of_nominal": frac(step_tflops, NOMINAL_BF16_TFLOPS)},
        "peaks": {"burst_measured": burst, "nominal_dense_bf16": NOMINAL_BF16_TFLOPS},
    }


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:  # under torchrun, rank 0 alone times the oracle
        return
    import fa_inputs
    cores = oracle_cores()
    n_heads = max(1, min(B * H, cores))
    x = fa_inputs.attention_inputs(SEED, B, H, N, D, "bf16")
    # A step is the oracle on a sample of whole heads, seconds of CPU work, so
    # the run is bounded in time: the first warm-up step measures it, the rest
    # of --warmup run while they fit in a quarter of REFERENCE_BUDGET_S, and at
    # most as many timed steps as fit in REFERENCE_BUDGET_S run (never more
    # than --steps).  The line reports the counts run and requested.
    t_warm, _ = oracle_step_sample(x, n_heads)
    warmup = 1
    while warmup < args.warmup and (warmup + 1) * t_warm <= REFERENCE_BUDGET_S / 4:
        oracle_step_sample(x, n_heads)
        warmup += 1
    steps = max(1, min(args.steps, int(REFERENCE_BUDGET_S / max(t_warm, 1e-3))))
    total_s, total_f = 0.0, 0.0
    for _ in range(steps):
        s, f = oracle_step_sample(x, n_heads)
        total_s += s
        total_f += f
    value = total_f / total_s / 1e12
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "steps_requested": args.steps,
        "warmup_requested": args.warmup,
        "ms_per_step": round(1e3 * total_s / steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D, "causal": CAUSAL,
                   "l2": "CPU oracle"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{n_heads} of {B * H} heads per step (whole heads, fwd+bwd)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


CASES = ("step", "fp8_quantize", "fp8_forward", "decode")


def run_case(args):
    """One next-row workload alone (for profiling): --warmup calls, then
    --steps calls timed on the device; one JSON line with the mean time."""
    import torch

    import fa_inputs
    import exact_io_aware_18_gb300 as fa

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEED)

    def rnd(*shape):
        return torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)

    scale = fa.default_scale(D)
    if args.case == "step":
        # The training step's three kernels on seeded device inputs of the
        # training-step shape: forward, dQ with the first backward step, dK/dV.
        q, k, v, do = rnd(B, H, N, D), rnd(B, H, N, D), rnd(B, H, N, D), rnd(B, H, N, D)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        dq, dk, dv = (torch.empty((B, H, N, D), dtype=torch.float32, device=dev)
                      for _ in range(3))
        n_pad = (N + 127) // 128 * 128
        ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, D) // 4, dtype=torch.float32,
                         device=dev)
        delta = ws[:B * H * n_pad].view(B * H, n_pad)
        lse2 = ws[B * H * n_pad:].view(B * H, n_pad)
        workload = WORKLOAD + " (device-drawn inputs)"

        def fn():
            fa.fa_fwd(q, k, v, o, lse, CAUSAL, scale, stream)
            fa.fa_bwd_dq_preprocess(q, k, v, o, do, lse, delta, lse2, dq, CAUSAL, scale, stream)
            fa.fa_bwd_dkdv(q, k, v, do, delta, lse2, dk, dv, CAUSAL, scale, stream)
    elif args.case in ("fp8_quantize", "fp8_forward"):
        q, k, v = rnd(B, H, N, D), rnd(B, H, N, D), rnd(B, H, N, D)
        signs = fa._lib._host_signs(fa_inputs.random_signs(SEED, D), D)
        q8, qs = fa.fp8_quantize(q, signs, stream)
        k8, ks = fa.fp8_quantize(k, signs, stream)
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        if args.case == "fp8_quantize":
            workload = f"rotation + E4M3 quantisation of one bf16 tensor B={B} H={H} N={N} d={D}"
            fn = lambda: fa.fa_fp8_quantize(q, signs, q8, qs, stream)  # noqa: E731
        else:
            workload = f"FP8 forward B={B} H={H} N={N} d={D} causal (Q, K codes given)"
            fn = lambda: fa.fa_fwd_fp8(q8, qs, k8, ks, v, o, lse, CAUSAL, scale, stream)  # noqa: E731
    else:
        db, dhq, dhkv, dnq, dnk = 4, 32, 8, 1, 16384
        q, k, v = rnd(db, dhq, dnq, D), rnd(db, dhkv, dnk, D), rnd(db, dhkv, dnk, D)
        o = torch.empty_like(q)
        lse = torch.empty((db, dhq, dnq), dtype=torch.float32, device=dev)
        ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(db, dhq, dhkv, dnq, dnk, D) // 4 + 4,
                         dtype=torch.float32, device=dev)
        workload = f"split-KV decode B={db} Hq={dhq} Hkv={dhkv} Nq={dnq} Nk={dnk} d={D}"
        fn = lambda: fa.fa_fwd_splitkv(q, k, v, o, lse, scale, 0, ws, stream)  # noqa: E731
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ms = _timed(torch, torch.cuda.current_stream(dev), fn, args.steps)
    if fa.fa_device_status(clear=True) != fa.FA_OK:
        raise RuntimeError("a kernel reported a timed-out wait")
    print(json.dumps({"case": args.case, "workload": workload, "ms": round(ms, 4),
                      "steps": args.steps, "warmup": args.warmup}))


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--case", choices=CASES, default=None,
                   help="run one next-row workload alone (for profiling) instead of the step")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.steps < 1:
        p.error("--steps must be at least 1")
    if args.case is not None:
        run_case(args)
    elif args.impl == "reference":
        if "--steps" not in (argv or sys.argv):
            args.steps = 5
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
