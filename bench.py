"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over synthetic inputs resident in HBM:
  * fused prefill, B=4 H=16 Nq=Nk=2048 d=64 scale=1/8, non-causal, then causal
    (the headline TFLOP/s workload), and
  * split-KV decode, B=64 H=32 Nk=8192 d=128, 16 splits (split + merge kernels).
value  = prefill TFLOP/s (4*B*H*Nq*Nk*d per non-causal launch, half for causal,
         summed over both launches, divided by their device time);
decode = HBM GB/s of the decode kernels (K + V + q + o + lse bytes / time).
Every timed launch is bracketed by CUDA events on the launching stream; the
L2 (129 MB) is flushed between steps by writing a 256 MB buffer outside the
events (the prefill inputs, 67 MB, would otherwise stay L2-resident).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--prefill-workload NAME]
(the default prefill workload is the headline one; the others time the d=128
8k / 32k causal workloads through the same harness)
Under torchrun each rank runs the same per-GPU workload (weak scaling, no
data-path collective); rank 0 prints one JSON line.
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

METRIC = "attention fwd TFLOP/s (prefill) & HBM GB/s (decode) on 1 GB300, % of roofline"
PREFILL = "prefill_2k"
DECODE = "decode_8k"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


# ----------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def visible_pair_fraction(wp, causal: bool) -> float:
    """Share of the nominal (query, key) pairs a workload's key padding leaves
    visible (1.0 without padding); effective TFLOP/s = nominal x this share.
    Causal visibility is bottom-right: row i sees keys j <= i + Nk - Nq."""
    if not wp.pad_heads:
        return 1.0
    i = np.arange(wp.Nq, dtype=np.int64)
    end = np.clip(i + 1 + (wp.Nk - wp.Nq), 0, wp.Nk) if causal else np.full(wp.Nq, wp.Nk, dtype=np.int64)
    full = int(end.sum())
    padded = int(np.minimum(end, wp.pad_from).sum())
    return (wp.pad_heads * padded + (wp.H - wp.pad_heads) * full) / (wp.H * full)


def max_over_ranks(times, world: int, device):
    """Element-wise maximum of per-rank device times (seconds) over all ranks:
    the job lasts as long as its slowest rank. With world == 1 the times come
    back unchanged; otherwise every rank receives the maxima (an all-reduce on
    `device`, a CUDA device under NCCL, the CPU under gloo)."""
    import torch
    t = torch.tensor([float(x) for x in times], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_step: float, steps: int, seconds: float, world: int) -> float:
    """Whole-job throughput of `world` replicas that each process
    `units_per_step` per step for `steps` steps, the slowest taking `seconds`
    (weak scaling: every rank does the same per-rank work)."""
    return world * steps * units_per_step / seconds


def barrier(world: int):
    """Line all ranks up at the edges of a timed region (no-op for one rank)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# headers a kernel source includes besides fa_ptx.cuh and fa_common.cuh
KERNEL_HEADERS = {"decode_grouped_sm103.cu": ("decode_grouped.cuh",), "materialized_sm103.cu": ("materialized.cuh",)}


def kernel_hash(name: str) -> str:
    csrc = os.path.join(ROOT, "io_aware_exact_fa_gb300", "csrc")
    h = hashlib.sha256()
    for f in (os.path.join(csrc, name), os.path.join(csrc, "fa_ptx.cuh"), os.path.join(csrc, "fa_common.cuh"),
              *(os.path.join(csrc, x) for x in KERNEL_HEADERS.get(name, ()))):
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel source is unchanged."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    rec = json.load(open(PROFILE_TRAFFIC)).get(workload)
    if not rec or rec.get("source_hash") != kernel_hash(kernel_file):
        return None
    return rec.get("dram_bytes_per_launch")


# Clock sampler run as a separate process (no contention with the launching
# thread): NVML through ctypes, one line per sample
# "<unix time>,<sm MHz>,<max sm MHz>,<clock event reason bits>" every
# <interval> ms. argv: device (a PCI bus id "dddddddd:bb:dd.f" or an NVML
# index), interval in ms. Exits with status 3 if NVML cannot be used.
NVML_SAMPLER = r"""
import ctypes, sys, time
try:
    nv = ctypes.CDLL("libnvidia-ml.so.1")
    assert nv.nvmlInit_v2() == 0
    h = ctypes.c_void_p()
    dev = sys.argv[1]
    if ":" in dev:
        assert nv.nvmlDeviceGetHandleByPciBusId_v2(dev.encode(), ctypes.byref(h)) == 0
    else:
        assert nv.nvmlDeviceGetHandleByIndex_v2(int(dev), ctypes.byref(h)) == 0
    reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
        nv.nvmlDeviceGetCurrentClocksThrottleReasons
    mx = ctypes.c_uint()
    assert nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0
except Exception:
    sys.exit(3)
iv = float(sys.argv[2]) / 1000.0
sm, rs = ctypes.c_uint(), ctypes.c_ulonglong()
out = sys.stdout
while True:
    t = time.time()
    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and reasons_fn(h, ctypes.byref(rs)) == 0:
        out.write("%.6f,%d,%d,%d\n" % (t, sm.value, mx.value, rs.value))
        out.flush()
    time.sleep(max(0.0, iv - (time.time() - t)))
"""
# NVML clock-event reason bits and the names reported for them
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown"}


def nvml_device_id(index: int) -> str:
    """The PCI bus id NVML knows the CUDA device `index` by (CUDA_VISIBLE_DEVICES
    may renumber devices), or the index itself when torch does not say."""
    try:
        import torch
        pr = torch.cuda.get_device_properties(index)
        return "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        return str(index)


class ClockSampler:
    """Samples of the SM clock and the clock-event (throttle) reasons during
    the timed regions: NVML every 2 ms from a separate process, else
    nvidia-smi every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.t = None
        self.window = None
        self.source = None

    def start(self):
        try:
            self.proc = subprocess.Popen([sys.executable, "-c", NVML_SAMPLER, nvml_device_id(self.index), "2"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline()
            if first:
                self.source = "nvml, 2 ms"
                self._add_nvml(first)
                self.t = threading.Thread(target=self._read_nvml, daemon=True)
                self.t.start()
                return
            self.proc.wait(timeout=5)
        except (OSError, subprocess.SubprocessError):
            pass
        self.proc = None
        try:
            self.source = "nvidia-smi, 50 ms"
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _add_nvml(self, line):
        try:
            t, sm, mx, bits = line.strip().split(",")
            bits = int(bits)
        except ValueError:
            return
        names = ["Active" if bits & b else "Not Active" for b in (0x8, 0x40, 0x20, 0x4)]
        # same field order as the nvidia-smi rows: timestamp, sm, max, power, active, hw, hw_thermal, sw_thermal, sw_cap
        self.samples.append((float(t), ["", sm, mx, "", str(bits)] + names))

    def _read_nvml(self):
        for line in self.proc.stdout:
            self._add_nvml(line)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summary(self.window)

    def summary(self, window=None):
        """Median SM clock, max clock and throttle reasons seen inside ``window`` (wall-clock seconds)."""
        if self.proc is None:
            return None
        rows = list(self.samples)
        if window:
            pad = 0.004 if self.source and self.source.startswith("nvml") else 0.06
            inside = [r for r in rows if window[0] - pad <= r[0] <= window[1] + pad]
            rows = inside or rows
        if not rows:
            return None
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, f in rows:
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, val in zip(names[1:], f[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "sampler": self.source}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "" if neither says."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


def oracle_prefill_sample(w, budget_s: float):
    """Time the fp64 oracle on whole heads of the prefill workload (non-causal
    and causal alternately) until ``budget_s`` is spent; returns (flops, seconds, heads)."""
    import numpy as np
    import torch
    from io_aware_exact_fa_gb300 import workloads as W
    from oracle import attention as A
    q, k, v = W.make_qkv(1, 2, w.Nq, w.Nk, w.d, seed=0)
    qs = [q[0, h].to(torch.float64).numpy() for h in range(2)]
    ks = [k[0, h].to(torch.float64).numpy() for h in range(2)]
    vs = [v[0, h].to(torch.float64).numpy() for h in range(2)]
    per_head = 4.0 * w.Nq * w.Nk * w.d
    flops, heads, t0 = 0.0, 0, time.perf_counter()
    while True:
        causal = heads % 2 == 1
        A.attend_head(qs[heads % 2], ks[heads % 2], vs[heads % 2], w.scale, causal)
        flops += per_head / 2 if causal else per_head
        heads += 1
        el = time.perf_counter() - t0
        if el >= budget_s or heads >= 4096:
            return flops, el, heads


def run_backward(args, fa, W, wp, modes, q, k, v, lse, flush, stream, warm, world, rank, dev):
    """Time fa_bwd (prep + main + finish launches) on the prefill workload's
    inputs, once per causal mode per step, with its own events and L2 flush;
    dO is seeded N(0,1) bf16 and O, lse come from the forward pass."""
    import torch
    gen = torch.Generator().manual_seed(2000 + rank)
    dout = torch.randn(tuple(q.shape), generator=gen).to(torch.bfloat16).to(dev)
    fo = {}
    for c in modes:
        fo[c] = (torch.empty_like(q), torch.empty(tuple(lse.shape), dtype=torch.float32, device=dev))
        fa.fwd(q, k, v, scale=wp.scale, causal=c, out=fo[c][0], lse=fo[c][1])
    wsb = torch.empty(max(1, fa.bwd_workspace_size(wp.B, wp.H, wp.Nq, wp.d)), dtype=torch.uint8, device=dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))

    def backward(c):
        fa.bwd(q, k, v, fo[c][0], fo[c][1], dout, scale=wp.scale, causal=c, workspace=wsb, grads=grads)

    for _ in range(warm):
        flush.zero_()
        for c in modes:
            backward(c)
    torch.cuda.synchronize()
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("device status not OK after the backward warm-up")
    K, nm = args.steps, len(modes)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nm + 1)] for _ in range(K)]
    n0 = fa.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        for j, c in enumerate(modes):
            backward(c)
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    launches = fa.launch_count() - n0
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("device status not OK after the backward timed region")
    tm = max_over_ranks([sum(e[j].elapsed_time(e[j + 1]) for e in ev) / 1e3 for j in range(nm)], world, dev)
    fm = [wp.bwd_flops(c) for c in modes]
    ach = K * sum(fm) / sum(tm) / 1e12
    peaks = measured_peaks()
    out = {"value": whole_job_rate(sum(fm), K, sum(tm), world) / 1e12, "unit": "TFLOP/s", "ms": sum(tm) / K * 1e3,
           "gpu_launches": launches,
           "dout": "N(0,1) bf16, seeded; O and lse from fa_fwd",
           "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": ach / peaks["bf16_tflops"],
                        "traffic": recorded_traffic("backward_sm103.cu", wp.name + "_bwd"),
                        "kernel": f"fa_bwd_kernel<{wp.d}> (+ fa_bwd_prep_kernel, fa_bwd_finish_kernel)",
                        "peak_source": f"{peaks['source']} bf16 burst",
                        "flop_convention": "10*B*H*Nq*Nk*d per non-causal launch (five products), halved for causal"},
           "_window": (t0, t1)}
    for c, t, f in zip(modes, tm, fm):
        tag = "causal" if c else "noncausal"
        out["roofline"][f"ms_{tag}"] = t / K * 1e3
        out["roofline"][f"tflops_{tag}"] = K * f / t / 1e12
    return out


def e2e_prefill(fa, wp, modes, q, k, v, n_e, dev, chunk_heads=0):
    """End-to-end prefill through the host-buffer entry point fa_fwd_host.
    Each step makes one call per causal mode on pinned host q, k, v; every
    call uploads the inputs in chunks of heads, runs the fused kernel on each
    chunk and copies o and lse back to pinned host buffers, overlapping the
    copies and kernels of consecutive chunks. The modes' calls are issued as
    independent requests on one stream each (each with its own workspace), so
    one call's uploads can overlap the other's kernels and read-backs.
    Returns the seconds of the n_e steps (CUDA events: the start is recorded
    on the current stream, which both request streams wait for, and the end
    after the current stream has waited for both)."""
    import torch
    hin = [x.cpu().pin_memory() for x in (q, k, v)]
    hout = [(torch.empty(tuple(q.shape), dtype=q.dtype).pin_memory(),
             torch.empty((wp.B, wp.H, wp.Nq), dtype=torch.float32).pin_memory()) for _ in modes]
    wsb = fa.fwd_host_workspace_size(wp.B, wp.H, wp.Nq, wp.Nk, wp.d, chunk_heads)
    ws = [torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in modes]
    req = [torch.cuda.Stream() for _ in modes]
    cur = torch.cuda.current_stream()

    def step():
        for c, causal in enumerate(modes):
            fa.fwd_host(*hin, scale=wp.scale, causal=causal, chunk_heads=chunk_heads, workspace=ws[c],
                        out=hout[c][0], lse=hout[c][1], stream=req[c], sync=False)

    step()  # warm-up: creates the library's copy streams
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for s in req:
        s.wait_stream(cur)
    for _ in range(n_e):
        step()
    for s in req:
        cur.wait_stream(s)
    t1.record(cur)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / 1e3


def run_materialized(args, fa, wp, modes, q, k, v, flush, stream, warm, world, dev):
    """Time the materialising baseline (cuBLAS S = scale Q K^T in bf16, this
    library's row softmax writing P over S, cuBLAS O = P V) on the prefill
    workload's inputs, per causal mode, L2 flushed between steps."""
    import torch
    ws = torch.empty(fa.materialized_workspace_size(wp.B, wp.H, wp.Nq, wp.Nk), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(wp.B, wp.H, wp.Nq, dtype=torch.float32, device=dev)

    def call(c):
        fa.fwd_materialized(q, k, v, scale=wp.scale, causal=c, workspace=ws, out=o, lse=lse)

    for _ in range(warm):
        flush.zero_()
        for c in modes:
            call(c)
    torch.cuda.synchronize()
    K, nm = args.steps, len(modes)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nm + 1)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        for j, c in enumerate(modes):
            call(c)
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    tm = max_over_ranks([sum(e[j].elapsed_time(e[j + 1]) for e in ev) / 1e3 for j in range(nm)], world, dev)
    fm = [wp.flops(c) for c in modes]
    # the pages' count: scores written, read, probabilities written, read (2-byte), plus Q, K, V, O
    nbytes = 4 * wp.B * wp.H * wp.Nq * wp.Nk * 2 + wp.io_bytes()
    out = {"value": whole_job_rate(sum(fm), K, sum(tm), world) / 1e12, "unit": "TFLOP/s", "ms": sum(tm) / K * 1e3,
           "hbm_bytes_model_per_launch": nbytes, "fused_min_bytes_per_launch": wp.io_bytes(),
           "gbs_model": K * nm * nbytes / sum(tm) / 1e9,
           "what": "cuBLAS bf16 GEMM S = scale Q K^T -> row softmax (this library, P over S) -> cuBLAS O = P V",
           "softmax_traffic": recorded_traffic("materialized_sm103.cu", wp.name + "_materialized_softmax"),
           "_window": (t0, t1), "_t_modes": tm}
    for c, t, f in zip(modes, tm, fm):
        tag = "causal" if c else "noncausal"
        out[f"ms_{tag}"] = t / K * 1e3
        out[f"tflops_{tag}"] = K * f / t / 1e12
    return out


def grouped_decode_kernel(w):
    """The split kernel fa_decode_grouped launches for a workload: by the
    number of query rows per K/V head, (H / Hkv) * Nq, and the head dim."""
    rows = w.H // w.Hkv * w.Nq
    if w.d == 64 and rows <= 4:
        return f"fa_decode_grouped_cc_kernel<64, {1 if rows == 1 else 2 if rows == 2 else 4}>"
    if rows <= 16:
        return f"fa_decode_grouped_kt_kernel<{w.d}>"
    return f"fa_decode_grouped_kernel<{w.d}>"


def run_decode_variants(args, fa, W, stream, warm, world, rank, dev):
    """Time fa_decode_grouped on each decode-variant workload (grouped K/V
    heads, ragged lengths, 1 or 4 new tokens). Inputs are drawn on the device
    with the workload recipe; the K/V caches (2 GB) exceed L2, so no flush."""
    import torch
    peaks = measured_peaks()
    out = {"workloads": {}}
    t_first = None
    for key, w in W.DECODE_VARIANTS.items():
        if args.dv_b:
            import dataclasses
            w = dataclasses.replace(w, B=args.dv_b, name=w.name.replace("b64", f"b{args.dv_b}"))
        q, k, v, lens = W.make_decode_inputs(w, seed=3000 + rank, device="cuda")
        ws = torch.empty(fa.decode_grouped_workspace_size(w.B, w.H, w.Nq, w.d, w.num_splits), dtype=torch.uint8,
                         device=dev)
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device=dev)

        def call():
            fa.decode_grouped(q, k, v, seqlens_k=lens, scale=w.scale, num_splits=w.num_splits, workspace=ws,
                              out=o, lse=lse)

        for _ in range(warm):
            call()
        torch.cuda.synchronize()
        if fa.device_status() != fa.FA_OK:
            raise RuntimeError("device status not OK after the decode-variant warm-up")
        K = args.steps
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        t_first = t_first or t0
        n0 = fa.launch_count()
        ev[0].record(stream)
        for i in range(K):
            call()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        launches = fa.launch_count() - n0
        if fa.device_status() != fa.FA_OK:
            raise RuntimeError("device status not OK after the decode-variant timed region")
        t = max_over_ranks([ev[0].elapsed_time(ev[K]) / 1e3], world, dev)[0]
        nbytes = w.io_bytes(lens.tolist())
        ach = K * nbytes / t / 1e9
        out["workloads"][w.name] = {
            "value": whole_job_rate(nbytes, K, t, world) / 1e9, "unit": "GB/s", "ms": t / K * 1e3, "bytes": nbytes, "gpu_launches": launches,
            "config": {"B": w.B, "H": w.H, "Hkv": w.Hkv, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                       "num_splits": w.num_splits, "seqlens": f"uniform in [{w.len_lo}, {w.Nk}], seeded",
                       "mean_seqlen": float(lens.float().mean().item())},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("decode_grouped_sm103.cu", w.name),
                         "kernel": f"{grouped_decode_kernel(w)} + fa_decode_merge_kernel<{w.d}>",
                         "peak_source": f"{peaks['source']} copy",
                         "bytes_convention": "visible K and V rows read once, q and o written, lse"},
        }
        del q, k, v, ws, o, lse
        torch.cuda.empty_cache()
    out["_window"] = (t_first, time.time())
    return out


LONG_CONTEXT = ("prefill_8k", "prefill_32k", "prefill_32k_pad")


def run_long_context(args, fa, W, flush, stream, warm, world, rank, dev):
    """Time the fused prefill on the long-context workloads (B=1 H=32 N=8192
    d=128 causal; B=1 H=8 N=32768 d=128 causal, without and with key padding
    on half the heads), one launch per step with its own CUDA events; then
    the backward pass on the 8k workload. Their inputs (201 MB of q, k, v)
    exceed L2; the L2 is flushed between steps anyway, outside the events."""
    import torch
    peaks = measured_peaks()
    out = {"workloads": {}}
    K = args.steps
    for key in LONG_CONTEXT:
        w = W.WORKLOADS[key]
        q, k, v = W.make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, seed=rank, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device=dev)
        words, strides = None, (0, 0, 0)
        if w.pad_heads:
            wb = W.pack_keep_bits(W.key_padding_keep(w.B, w.H, w.Nk, w.pad_heads, w.pad_from))
            words, strides = wb.to(dev), W.mask_strides(wb)
        causal = w.causal_modes[0]

        def call():
            fa.fwd(q, k, v, scale=w.scale, causal=causal, keep_bits=words, mask_strides=strides, out=o, lse=lse)

        for _ in range(warm):
            flush.zero_()
            call()
        torch.cuda.synchronize()
        if fa.device_status() != fa.FA_OK:
            raise RuntimeError(f"device status not OK after the {w.name} warm-up")
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        n0 = fa.launch_count()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(K):
            flush.zero_()
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        t1 = time.time()
        launches = fa.launch_count() - n0
        if fa.device_status() != fa.FA_OK:
            raise RuntimeError(f"device status not OK after the {w.name} timed region")
        t = max_over_ranks([sum(a.elapsed_time(b) for a, b in ev) / 1e3], world, dev)[0]
        f = w.flops(causal)
        ach = K * f / t / 1e12
        rec = {"value": whole_job_rate(f, K, t, world) / 1e12, "unit": "TFLOP/s", "ms": t / K * 1e3,
               "gpu_launches": launches,
               "config": {"B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "scale": w.scale, "causal": causal,
                          "key_padding": ({"heads_below": w.pad_heads, "keys_from": w.pad_from}
                                          if w.pad_heads else None)},
               "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": ach / peaks["bf16_tflops"],
                            "traffic": recorded_traffic("prefill_sm103.cu", w.name),
                            "kernel": f"fa_prefill_kernel<{w.d}>", "peak_source": f"{peaks['source']} bf16 burst",
                            "flop_convention": "4*B*H*Nq*Nk*d, halved for causal (nominal: padded keys counted)"},
               "_window": (t0, t1)}
        if w.pad_heads:
            share = visible_pair_fraction(w, causal)
            rec["roofline"]["visible_pair_share"] = share
            rec["roofline"]["tflops_effective"] = ach * share
        if key == "prefill_8k" and not args.no_backward:
            rec["backward"] = run_backward(args, fa, W, w, [causal], q, k, v, lse, flush, stream, warm, world, rank,
                                           dev)
        if not w.pad_heads and not args.no_fp8:
            del q, k, v
            rec["fp8"] = run_fp8(args, fa, W, w, causal, flush, stream, warm, world, rank, dev)
        out["workloads"][w.name] = rec
        del o, lse
        torch.cuda.empty_cache()
    return out


def run_fp8(args, fa, W, w, causal, flush, stream, warm, world, rank, dev):
    """Time fa_fwd_fp8 on a workload's shape with e4m3 inputs (the same N(0,1)
    draws quantized per tensor, descale amax / 448), one launch per step, L2
    flushed between steps outside the events. The roofline peak is the fp8
    dense rate: the measured bf16 peak times the nominal fp8 / bf16 ratio 2."""
    import torch
    (q8, k8, v8), ds = W.make_qkv_fp8(w.B, w.H, w.Nq, w.Nk, w.d, seed=rank, device="cuda")
    o = torch.empty(w.B, w.H, w.Nq, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.H, w.Nq, dtype=torch.float32, device=dev)

    def call():
        fa.fwd_fp8(q8, k8, v8, *ds, scale=w.scale, causal=causal, out=o, lse=lse)

    for _ in range(warm):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError(f"device status not OK after the {w.name} fp8 warm-up")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    n0 = fa.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    launches = fa.launch_count() - n0
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError(f"device status not OK after the {w.name} fp8 timed region")
    t = max_over_ranks([sum(a.elapsed_time(b) for a, b in ev) / 1e3], world, dev)[0]
    f = w.flops(causal)
    ach = K * f / t / 1e12
    peaks = measured_peaks()
    peak = 2.0 * peaks["bf16_tflops"]
    name = w.name + "_fp8"
    return {"value": whole_job_rate(f, K, t, world) / 1e12, "unit": "TFLOP/s", "ms": t / K * 1e3,
            "gpu_launches": launches, "dtype": "e4m3 in, bf16 out",
            "inputs": "the workload's N(0,1) draws quantized per tensor to e4m3 (descale amax / 448)",
            "roofline": {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                         "traffic": recorded_traffic("prefill_sm103.cu", name),
                         "kernel": f"fa_prefill_kernel<{w.d}, e4m3>",
                         "peak_source": f"{peaks['source']} bf16 burst x 2 (nominal fp8 / bf16 dense ratio)",
                         "flop_convention": "4*B*H*Nq*Nk*d, halved for causal"},
            "_window": (t0, t1)}


# --------------------------------------------------------------- reference
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from io_aware_exact_fa_gb300 import workloads as W
    w = W.WORKLOADS[PREFILL]
    for _ in range(args.warmup):
        oracle_prefill_sample(w, 0.0)
    flops = secs = 0.0
    heads = 0
    budget = max(1.0, 60.0 / max(1, args.steps))
    for _ in range(args.steps):
        f, s, h = oracle_prefill_sample(w, budget)
        flops += f
        secs += s
        heads += h
    value = flops / secs / 1e12
    sample = f"{heads} whole heads of {w.name} (Nq=Nk={w.Nk}, d={w.d}), non-causal/causal alternating, fp64 NumPy"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "causal": [False, True], "oracle": "oracle/attention.py attend_head"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "cpu": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for cpu_baseline (0 = skip)")
    ap.add_argument("--only", default="all",
                    choices=["all", "prefill", "decode", "backward", "decode_variants", "materialized",
                             "long_context"],
                    help="run one part of the step only (small profiling runs)")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward-pass leg (timed after the step, reported under 'backward')")
    ap.add_argument("--decode-b", type=int, default=0, help="override the decode batch (profiling a small case)")
    ap.add_argument("--prefill-h", type=int, default=0, help="override the prefill heads (profiling a small case)")
    ap.add_argument("--dv-b", type=int, default=0, help="override the decode-variant batch (profiling a small case)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-fp8", action="store_true", help="skip the e4m3-input legs (the headline and long-context workloads)")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long-context prefill legs (8k and 32k, d=128; reported under 'long_context')")
    ap.add_argument("--e2e-chunk-heads", type=int, default=0,
                    help="heads per chunk of the host-buffer calls (0 = the library default, half of B*H)")
    ap.add_argument("--prefill-workload", default=PREFILL,
                    choices=["prefill_2k", "prefill_8k", "prefill_32k", "prefill_32k_pad"],
                    help="prefill workload of the step (default: the 2k / d=64 headline workload)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from io_aware_exact_fa_gb300 import build as B
    B.build()
    from io_aware_exact_fa_gb300 import fa, workloads as W

    do_p = args.only in ("all", "prefill")
    do_d = args.only in ("all", "decode")
    wp = W.WORKLOADS[args.prefill_workload]
    if args.prefill_h:
        import dataclasses
        wp = dataclasses.replace(wp, H=args.prefill_h, name=f"{wp.name}_h{args.prefill_h}")
    # the backward pass takes no key mask: it is timed on the unpadded workloads
    do_b = args.only in ("all", "backward") and not args.no_backward and not wp.pad_heads
    do_v = args.only in ("all", "decode_variants")
    do_m = args.only in ("all", "materialized") and not wp.pad_heads
    do_l = args.only in ("all", "long_context") and not args.no_long and args.prefill_workload == PREFILL \
        and not args.prefill_h
    modes = list(wp.causal_modes)
    wd = W.WORKLOADS[DECODE]
    if args.decode_b:
        import dataclasses
        wd = dataclasses.replace(wd, B=args.decode_b, name=wd.name.replace("b64", f"b{args.decode_b}"))
    if do_p or do_b or do_m:
        q, k, v = W.make_qkv(wp.B, wp.H, wp.Nq, wp.Nk, wp.d, seed=rank, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty(wp.B, wp.H, wp.Nq, dtype=torch.float32, device=dev)
        keep_words, mstrides = None, (0, 0, 0)
        if wp.pad_heads:
            words = W.pack_keep_bits(W.key_padding_keep(wp.B, wp.H, wp.Nk, wp.pad_heads, wp.pad_from))
            keep_words, mstrides = words.to(dev), W.mask_strides(words)
    if do_d:
        dq, dk, dv = W.make_qkv(wd.B, wd.H, 1, wd.Nk, wd.d, seed=1000 + rank, device="cuda")
        do = torch.empty_like(dq)
        dlse = torch.empty(wd.B, wd.H, dtype=torch.float32, device=dev)
        ws = torch.empty(fa.decode_workspace_size(wd.B, wd.H, wd.d, wd.num_splits), dtype=torch.uint8,
                         device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def prefill(causal):
        fa.fwd(q, k, v, scale=wp.scale, causal=causal, keep_bits=keep_words, mask_strides=mstrides, out=o, lse=lse)

    def decode():
        fa.decode(dq, dk, dv, scale=wd.scale, num_splits=wd.num_splits, workspace=ws, out=do, lse=dlse)

    def step_body(e):
        # events: e[0] .. e[len(modes)] bracket the prefill launches, then decode
        e[0].record(stream)
        for i, causal in enumerate(modes):
            if do_p:
                prefill(causal)
            e[i + 1].record(stream)
        if do_d:
            decode()
        e[len(modes) + 1].record(stream)

    warm = max(3, args.warmup)
    for _ in range(warm):
        flush.zero_()
        if do_p:
            for causal in modes:
                prefill(causal)
        if do_d:
            decode()
    torch.cuda.synchronize()
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("device status not OK after warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(modes) + 2)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    launches0 = fa.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(K):
        flush.zero_()                     # outside the events: evicts the prefill inputs from L2
        step_body(ev[i])
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    launches = fa.launch_count() - launches0
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("device status not OK after the timed region")
    bwd = run_backward(args, fa, W, wp, modes, q, k, v, lse, flush, stream, warm, world, rank, dev) if do_b else None
    dvar = run_decode_variants(args, fa, W, stream, warm, world, rank, dev) if do_v else None
    mat = run_materialized(args, fa, wp, modes, q, k, v, flush, stream, warm, world, dev) if do_m else None
    lng = run_long_context(args, fa, W, flush, stream, warm, world, rank, dev) if do_l else None
    # the headline workload on e4m3 inputs, both modes of the step
    pf8 = None
    if do_p and not args.no_fp8 and not wp.pad_heads:
        pf8 = {"modes": {("causal" if c else "noncausal"): run_fp8(args, fa, W, wp, c, flush, stream, warm, world,
                                                                   rank, dev) for c in modes}}
    sampler.stop()
    clocks = sampler.summary((t_wall0, t_wall1))
    if bwd is not None:
        bwd["clocks"] = sampler.summary(bwd.pop("_window"))
    if dvar is not None:
        dvar["clocks"] = sampler.summary(dvar.pop("_window"))
    if mat is not None:
        mat["clocks"] = sampler.summary(mat.pop("_window"))
    if pf8 is not None:
        for rec in pf8["modes"].values():
            rec["clocks"] = sampler.summary(rec.pop("_window"))
        fl = sum(wp.flops(c) for c in modes)
        ms = sum(r["ms"] for r in pf8["modes"].values())
        pf8["value"] = fl / (ms / 1e3) / 1e12 * world
        pf8["unit"] = "TFLOP/s"
        pf8["workload"] = wp.name + " (" + " + ".join(pf8["modes"]) + "), e4m3 inputs"
        pk = next(iter(pf8["modes"].values()))["roofline"]["peak"]
        pf8["roofline"] = {"bound": "tensor", "achieved": fl / (ms / 1e3) / 1e12, "peak": pk, "unit": "TFLOP/s",
                           "frac": fl / (ms / 1e3) / 1e12 / pk, "kernel": f"fa_prefill_kernel<{wp.d}, e4m3>",
                           "peak_source": "measured bf16 burst x 2 (nominal fp8 / bf16 dense ratio)"}
    if lng is not None:
        for rec in lng["workloads"].values():
            rec["clocks"] = sampler.summary(rec.pop("_window"))
            for sub_leg in ("backward", "fp8"):
                if sub_leg in rec:
                    rec[sub_leg]["clocks"] = sampler.summary(rec[sub_leg].pop("_window"))

    nm = len(modes)
    t_modes = [sum(e[i].elapsed_time(e[i + 1]) for e in ev) / 1e3 for i in range(nm)]
    t_d = sum(e[nm].elapsed_time(e[nm + 1]) for e in ev) / 1e3
    times = max_over_ranks(t_modes + [t_d], world, dev)
    t_modes, t_d = times[:nm], times[nm]
    f_modes = [wp.flops(c) for c in modes]
    t_p, f_p = sum(t_modes), sum(f_modes)
    peaks = measured_peaks()
    dec_bytes = wd.io_bytes()

    # ---- end to end through the public API with pinned host buffers
    e2e = dec_e2e = None
    if not args.no_e2e:
        n_e = max(3, min(K, 20))
        ee = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_e)]
        # the host-buffer entry point takes no key mask: no end-to-end leg for the padded workload
        if do_p and not wp.pad_heads:
            te_p = e2e_prefill(fa, wp, modes, q, k, v, n_e, dev, args.e2e_chunk_heads)
        if do_d:
            hdq = dq.cpu().pin_memory()
            hdo = torch.empty(do.shape, dtype=do.dtype).pin_memory()
            hdl = torch.empty(dlse.shape, dtype=dlse.dtype).pin_memory()
        torch.cuda.synchronize()
        for i in range(n_e):
            flush.zero_()
            ee[i][0].record(stream)
            ee[i][1].record(stream)
            if do_d:
                dq.copy_(hdq, non_blocking=True)
                decode()
                hdo.copy_(do, non_blocking=True)
                hdl.copy_(dlse, non_blocking=True)
            ee[i][2].record(stream)
        torch.cuda.synchronize()
        te_d = sum(e[1].elapsed_time(e[2]) for e in ee) / 1e3
        e2e_p = do_p and not wp.pad_heads
        te_p, te_d = max_over_ranks([te_p if e2e_p else 0.0, te_d], world, dev)
        if e2e_p:
            e2e = {"value": whole_job_rate(f_p, n_e, te_p, world) / 1e12, "unit": "TFLOP/s",
                   "h2d_bytes_per_step": nm * (q.numel() + k.numel() + v.numel()) * 2,
                   "d2h_bytes_per_step": nm * (o.numel() * 2 + lse.numel() * 4),
                   "steps": n_e,
                   "api": "fa_fwd_host (C ABI, host buffers), one call per causal mode",
                   "chunk_heads": args.e2e_chunk_heads or max(1, -(-wp.B * wp.H // 2)),
                   "note": "every call uploads q, k, v from pinned host memory in chunks of heads, runs the fused "
                           "kernel per chunk and reads o, lse back; copies and kernels of consecutive chunks "
                           "overlap inside the call; the two modes' calls are independent requests on one "
                           "stream each; no L2 flush (uploads land in L2)"}
        if do_d:
            dec_e2e = {"value": whole_job_rate(dec_bytes, n_e, te_d, world) / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": dq.numel() * 2, "d2h_bytes_per_step": do.numel() * 2 + dlse.numel() * 4,
                       "note": "KV cache resident on the device; q in, o and lse out per step"}

    # ---- CPU baseline: the oracle on the host cores, a bounded sample
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0 and do_p and args.prefill_workload == PREFILL:
        f, s, heads = oracle_prefill_sample(wp, args.cpu_budget)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "cpu": cpu_model(), "kind": "oracle",
               "sample": f"{heads} whole heads (1 head = {wp.Nq}x{wp.Nk}, d={wp.d}) of {wp.name}, "
                         f"non-causal/causal alternating, fp64 NumPy, {s:.1f} s"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0
    line = {
        "metric": METRIC,
        "value": whole_job_rate(f_p, K, t_p, world) / 1e12 if do_p else None,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": warm,
        "ms_per_step": (t_p + t_d) / K * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": (f"{wp.name} ({' + '.join('causal' if c else 'non-causal' for c in modes)})"
                                if do_p else "")
                   + (" + " if do_p and do_d else "") + (wd.name if do_d else ""),
                   "B": wp.B, "H": wp.H, "Nq": wp.Nq, "Nk": wp.Nk, "d": wp.d, "scale": wp.scale,
                   "causal": modes,
                   "key_padding": ({"heads_below": wp.pad_heads, "keys_from": wp.pad_from} if wp.pad_heads else None),
                   "decode": {"B": wd.B, "H": wd.H, "Nk": wd.Nk, "d": wd.d, "num_splits": wd.num_splits},
                   "l2": "flushed between steps (256 MB write outside the timed events)",
                   "parallelism": f"replicas x{world}"},
        "e2e": e2e,
        "gpu_launches": launches,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "wall_s_timed": t_wall1 - t_wall0,
    }
    if do_p:
        ach = K * f_p / t_p / 1e12
        line["roofline"] = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": ach / peaks["bf16_tflops"],
                            "traffic": recorded_traffic("prefill_sm103.cu", wp.name),
                            "kernel": f"fa_prefill_kernel<{wp.d}>", "peak_source": f"{peaks['source']} bf16 burst",
                            "flop_convention": "4*B*H*Nq*Nk*d per non-causal launch, halved for causal"}
        for c, tm, fm in zip(modes, t_modes, f_modes):
            tag = "causal" if c else "noncausal"
            line["roofline"][f"ms_{tag}"] = tm / K * 1e3
            line["roofline"][f"tflops_{tag}"] = K * fm / tm / 1e12
        if wp.pad_heads:
            # key padding: the nominal FLOPs count the padded keys as well
            share = sum(visible_pair_fraction(wp, c) * fm for c, fm in zip(modes, f_modes)) / f_p
            line["roofline"]["visible_pair_share"] = share
            line["roofline"]["tflops_effective"] = ach * share
    if do_d:
        ach = K * dec_bytes / t_d / 1e9
        line["decode"] = {"value": whole_job_rate(dec_bytes, K, t_d, world) / 1e9, "unit": "GB/s", "ms": t_d / K * 1e3, "bytes": dec_bytes,
                          "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                       "frac": ach / peaks["hbm_gbs"],
                                       "traffic": recorded_traffic("decode_sm103.cu", wd.name),
                                       "kernel": "fa_decode_split_kernel<128> + fa_decode_merge_kernel<128>",
                                       "peak_source": f"{peaks['source']} copy"},
                          "e2e": dec_e2e}
        if not do_p:
            line["value"], line["unit"] = line["decode"]["value"], "GB/s"
    if bwd is not None:
        line["backward"] = bwd
        if not do_p and not do_d:
            line["value"] = bwd["value"]
    if mat is not None:
        t_mat = mat.pop("_t_modes")
        if do_p:  # how many times faster the fused kernel ran, per mode
            mat["fused_speedup"] = {("causal" if c else "noncausal"): tmm / tm
                                    for c, tm, tmm in zip(modes, t_modes, t_mat)}
        line["materialized"] = mat
    if pf8 is not None:
        line["prefill_fp8"] = pf8
    if lng is not None:
        line["long_context"] = lng
        if not do_p and not do_d and bwd is None and dvar is None:
            first = next(iter(lng["workloads"].values()))
            line["value"], line["unit"] = first["value"], "TFLOP/s"
    if dvar is not None:
        line["decode_variants"] = dvar
        if not do_p and not do_d and bwd is None:
            first = next(iter(dvar["workloads"].values()))
            line["value"], line["unit"] = first["value"], "GB/s"
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
