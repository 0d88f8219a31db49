"""Benchmark of the sparse MoE expert block on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--fwd-only]

A step is one pass of the whole block, forward and backward (routing
histogram, permute, FC1+SwiGLU, FC2, combine, combine backward, FC2 backward
with the fused SwiGLU backward, FC1 backward, permute backward) over one
batch of seeded synthetic input resident in HBM.  The default workload is
``long_seq_train`` (T=32768 tokens = 2 x 16384, emb 2816, 128 experts,
top-8, mlp 704, router logits plus a per-expert bias): the training block
the MaxText Gemma4-26B-A4B pages measure.  Its inputs (xs 1.5 GB, wi 1 GB)
are larger than the 129 MB L2, so no L2 flush is needed between steps; a
workload whose inputs fit in L2 gets L2 flushed (a 256 MB write, not timed)
before every timed step.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica on its own tokens (weak scaling, no collective on the data path; a
max-reduction of the timings only).  ``--impl reference`` times the CPU
oracle on the host cores instead, on a bounded sample of the same workload.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_ffn_histogram_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "MoE block tokens/s (fwd+bwd)"
METRIC_FWD = "MoE block tokens/s (fwd)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_seq_train", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-mx", action="store_true",
                    help="skip the MXFP8 forward (and training step) measurements")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the timed loop over every configuration")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (small cases for profiling; not a bench line)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (small cases for profiling; not a bench line)")
    return ap.parse_args()


def selected_workload(args):
    from dataclasses import replace
    wl = WORKLOADS[args.workload]
    kw = {}
    if args.tokens is not None:
        kw["T"] = args.tokens
    if args.experts is not None:
        kw["E"] = args.experts
    if kw:
        tag = ",".join(f"{k}={v}" for k, v in kw.items())
        wl = replace(wl, name=f"{wl.name}[{tag}]", **kw)
    return wl


# ------------------------------------------------------------- distributed
def dist_setup(n):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------- roofline model
def gemm_flops(kind, R, D, F):
    return {"fc1": 4, "fc2": 2, "fc2_dlhs": 2, "fc2_drhs": 2, "fc1_dlhs": 4, "fc1_drhs": 4}[kind] * R * D * F


def hbm_bytes(kind, T, D, E, K, F):
    """Algorithmic bytes of each HBM-bound step (what the method must move):
    route reads the logits and writes ids, weights and group sizes; the
    permute/combine family moves each bf16 row once plus its index words."""
    R = T * K
    return {
        "route": 4 * T * E + 8 * T * K + 4 * E,
        "permute": 2 * T * D + 2 * R * D + 8 * T * K,
        "combine": 2 * R * D + 2 * T * D + 8 * T * K,
        "combine_bwd": 2 * T * D + 4 * R * D + 8 * T * K,
        "permute_bwd": 2 * R * D + 2 * T * D,
    }[kind]


def gemm_bytes(kind, R, D, E, F, train=True):
    z = 4 * R * F if train else 0
    return {
        "fc1": 2 * R * D + 4 * E * D * F + 2 * R * F + z,
        "fc2": 2 * R * F + 2 * E * F * D + 2 * R * D,
        "fc2_dlhs": 2 * R * D + 2 * E * F * D + 8 * R * F,
        "fc2_drhs": 2 * R * F + 2 * R * D + 2 * E * F * D,
        "fc1_dlhs": 4 * R * F + 4 * E * D * F + 2 * R * D,
        "fc1_drhs": 2 * R * D + 4 * R * F + 4 * E * D * F,
    }[kind]


# kernel names as ncu reports them, for the traffic figures under profiles/
NCU_NAME = {
    "route": "route_topk_hist", "permute": "permute_kernel", "fc1": "grouped_gemm_kernel<0>",
    "fc2": "grouped_gemm_kernel<1>", "combine": "combine_kernel", "combine_bwd": "combine_bwd_kernel",
    "fc2_dlhs": "grouped_gemm_kernel<2>", "fc2_drhs": "grouped_gemm_kernel<4>",
    "fc1_dlhs": "grouped_gemm_kernel<3>", "fc1_drhs": "grouped_gemm_kernel<5>",
    "permute_bwd": "combine_kernel",
}


# the files holding the device code behind each timed step of the bf16 block
# (a step's traffic figure under profiles/ is valid while they are unchanged)
_BASE_SOURCES = ("common.cuh", "kernels.h")
_GATHER_SOURCES = _BASE_SOURCES + ("mx_common.cuh", "permute_combine.cu")
_GEMM_SOURCES = _BASE_SOURCES + ("gemm.cu",)
STEP_SOURCES = {
    "route": _BASE_SOURCES + ("route.cu",),
    **{n: _GATHER_SOURCES for n in ("permute", "combine", "combine_bwd", "permute_bwd")},
    **{n: _GEMM_SOURCES for n in ("fc1", "fc2", "fc2_dlhs", "fc2_drhs", "fc1_dlhs", "fc1_drhs")},
}
KERNEL_SOURCES = tuple(sorted({f for v in STEP_SOURCES.values() for f in v}))


def source_hash(files=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_ffn_histogram_gb300", "csrc")
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(step: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources of that step's kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get("kernels", {}).get(workload, {}).get(step)
    if ent is None or ent.get("source_hash") != source_hash(STEP_SOURCES[step]):
        return None
    return ent.get("dram_bytes_per_launch")


def peaks():
    """Measured peaks of the GB300s: HBM copy GB/s, and cuBLAS bf16
    TF/s as a burst (near the maximum SM clock) and sustained (power-capped,
    back to back for seconds)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p["bf16_tflops_sustained"]),
                    sm_max_mhz=float(p.get("sm_max_mhz", 2070.0)), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, sm_max_mhz=2070.0,
                    source="fallback")


def tensor_peak(pk, clocks):
    """The bf16 tensor peak that matches the clocks seen while the kernels
    ran: the burst figure scaled by median SM MHz / maximum SM MHz (the
    tensor rate is proportional to the SM clock), or the sustained figure
    when no clock was sampled.  Returns (TF/s, how it was obtained)."""
    sm = clocks.get("sm_mhz") if clocks else None
    smax = (clocks.get("sm_max_mhz") if clocks else None) or pk["sm_max_mhz"]
    if sm:
        f = min(1.0, float(sm) / float(smax))
        return pk["bf16"] * f, (f"{pk['source']} bf16_tflops (burst) x median SM clock "
                                f"{sm:.0f} / {smax:.0f} MHz")
    return pk["bf16_sustained"], f"{pk['source']} bf16_tflops_sustained (no clock sampled)"


# ------------------------------------------------------------------ clocks
class NvmlSampler:
    """Samples the SM clock and the clock-event (throttle) reasons through
    NVML every few milliseconds while the timed region runs; read-only (no
    NVML call here changes a setting).  `ok` is False when NVML cannot be
    loaded, and the nvidia-smi sampler below is used instead."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev: torch.device, period_s: float = 0.004):
        import ctypes
        self.period = period_s
        self.samples = []
        self.ok = False
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            found = False
            props = torch.cuda.get_device_properties(dev)
            bus = getattr(props, "pci_bus_id", None)
            if bus is not None:
                pci = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus,
                                             getattr(props, "pci_device_id", 0))
                found = L.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(h)) == 0
            if not found:
                found = L.nvmlDeviceGetHandleByIndex_v2(dev.index or 0, ctypes.byref(h)) == 0
            if not found:
                return
            self.L, self.h, self.ct = L, h, ctypes
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = self._read() is not None
        except (OSError, AttributeError):
            self.ok = False

    def _read(self):
        c, r = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.L.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(c)) != 0:
            return None
        if self.reasons_fn(self.h, self.ct.byref(r)) != 0:
            return None
        return float(c.value), int(r.value)

    def _loop(self):
        while not self._stop:
            v = self._read()
            if v is not None:
                self.samples.append(v)
            time.sleep(self.period)

    def __enter__(self):
        import threading
        self._stop = False
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *a):
        self._stop = True
        self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"]}
        reasons = set()
        for _, bits in self.samples:
            for bit, name in self.REASONS.items():
                if bits & bit:
                    reasons.add(name)
        sm = [c for c, _ in self.samples]
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}


def clock_sampler(dev: torch.device):
    s = NvmlSampler(dev)
    return s if s.ok else ClockSampler(dev.index)


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed
    region runs (started, and seen producing samples, before the region)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.out = None
        self._thread = None
        self._active = False

    def _reader(self):
        for line in self.proc.stdout:
            if self._active:
                self.lines.append(line)
            else:
                self._seen = True

    def __enter__(self):
        import threading
        self._seen = False
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self._thread = threading.Thread(target=self._reader, daemon=True)
        self._thread.start()
        t0 = time.time()
        while not self._seen and time.time() - t0 < 5.0:
            time.sleep(0.01)
        self._active = True
        return self

    def __exit__(self, *a):
        self._active = False
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._thread is not None:
                self._thread.join(timeout=2)
        self.out = "".join(self.lines)

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- our GPU arm
class Step:
    """One forward+backward pass through the C ABI, with a CUDA event pair
    around every kernel launch (all on the one stream the block runs on)."""

    def __init__(self, wl, inp, fwd_only):
        from mixture_experts_ffn_histogram_gb300 import binding as B
        from mixture_experts_ffn_histogram_gb300.block import MoEBlock
        self.B = B
        self.wl = wl
        self.fwd_only = fwd_only
        self.blk = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=not fwd_only)
        self.inp = inp
        self.names = ["route", "permute", "fc1", "fc2", "combine"]
        if not fwd_only:
            self.names += ["combine_bwd", "fc2_dlhs", "fc2_drhs", "fc1_dlhs", "fc1_drhs", "permute_bwd"]
        # our kernels per step (the drhs schedule's counter memsets are not ours)
        self.launches_per_step = 5 + (0 if fwd_only else 6)
        self.times = {n: [] for n in self.names}
        self._ev = []

    def run(self, record=False, x=None, logits=None, dy=None):
        B, b, d, inp = self.B, self.blk, self.blk.d, self.inp
        x = inp["x"] if x is None else x
        logits = inp["logits"] if logits is None else logits
        dy = inp["dy"] if dy is None else dy
        ev = []

        def mark():
            if record:
                e = torch.cuda.Event(enable_timing=True)
                e.record()
                ev.append(e)

        if self.wl.score_mode == B.SCORE_GIVEN:
            b.ids.copy_(inp["ids"])
            b.w.copy_(inp["w"])
        mark()
        B.moe_route_histogram(logits, inp["bias"], b.mode, b.ids, b.w, b.group_sizes,
                              b.group_offsets, b.pos, b.row_src, b.status, b.ws, d)
        mark()
        B.moe_permute(x, b.pos, b.xs, d)
        mark()
        B.moe_grouped_gemm_fc1_swiglu(b.xs, inp["wi"], b.group_offsets, b.h, b.z, b.status, b.ws, d)
        mark()
        B.moe_grouped_gemm_fc2(b.h, inp["wo"], b.group_offsets, b.ys, b.status, b.ws, d)
        mark()
        B.moe_combine(b.ys, b.w, b.pos, b.out, d)
        mark()
        if not self.fwd_only:
            B.moe_combine_bwd(dy, b.ys, b.w, b.pos, b.dys, b.dw, d)
            mark()
            B.moe_grouped_gemm_fc2_bwd(b.dys, b.h, inp["wo"], b.z, b.group_offsets, b.dz, None,
                                       b.status, b.ws, d)
            mark()
            B.moe_grouped_gemm_fc2_bwd(b.dys, b.h, inp["wo"], b.z, b.group_offsets, None, b.dwo,
                                       b.status, b.ws, d)
            mark()
            B.moe_grouped_gemm_fc1_swiglu_bwd(b.dz, None, b.xs, inp["wi"], b.group_offsets, b.dxs,
                                              None, b.status, b.ws, d)
            mark()
            B.moe_grouped_gemm_fc1_swiglu_bwd(b.dz, None, b.xs, inp["wi"], b.group_offsets, None,
                                              b.dwi, b.status, b.ws, d)
            mark()
            B.moe_permute_bwd(b.dxs, b.pos, b.dx, d)
            mark()
        if record:
            self._ev.append(ev)

    def collect(self):
        torch.cuda.synchronize()
        for ev in self._ev:
            for i, n in enumerate(self.names):
                self.times[n].append(ev[i].elapsed_time(ev[i + 1]) * 1e-3)
        self._ev = []


GEMMS = ("fc1", "fc2", "fc2_dlhs", "fc2_drhs", "fc1_dlhs", "fc1_drhs")

MX_STEPS = ("route", "permute_quantize", "fc1", "fc2", "combine")


def mx_bytes(kind, T, D, E, K, F):
    """Algorithmic bytes of the MXFP8 forward's steps: e4m3 codes (1 B) plus
    one scale byte per 32 elements."""
    R = T * K
    return {
        "permute_quantize": 2 * T * D + R * D + R * D // 32 + 4 * T * K,
        "fc1": R * D + R * D // 32 + 2 * E * F * D + 2 * E * F * D // 32 + R * F + R * F // 32,
        "fc2": R * F + R * F // 32 + E * D * F + E * D * F // 32 + 2 * R * D,
    }[kind]


def measure_mx(wl, inp, steps, pk, flushed, dev):
    """The MXFP8 forward (route, permute + quantize, FC1 + SwiGLU + quantize
    h, FC2, combine) through the C ABI, weights quantized once before the
    timed loop; an event pair around every launch."""
    from mixture_experts_ffn_histogram_gb300 import binding as B
    from mixture_experts_ffn_histogram_gb300.block import MoEBlockMX
    blk = MoEBlockMX(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode)
    d = blk.d
    # the weights' quantization: one untimed call (the first call also pays
    # the one-time setup), then the median of three
    qt = {"wi": [], "wo": []}
    for rep in range(4):
        q0, q1, q2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        q0.record()
        B.moe_mx_quantize_wi(inp["wi"], blk.wiq, blk.wisc, d)
        q1.record()
        B.moe_mx_quantize_wo(inp["wo"], blk.woq, blk.wosc, d)
        q2.record()
        torch.cuda.synchronize()
        if rep > 0:
            qt["wi"].append(q0.elapsed_time(q1) * 1e3)
            qt["wo"].append(q1.elapsed_time(q2) * 1e3)
    if wl.score_mode == B.SCORE_GIVEN:
        blk.ids.copy_(inp["ids"])
        blk.w.copy_(inp["w"])

    def run(ev):
        def mark():
            if ev is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record()
                ev.append(e)
        mark()
        B.moe_route_histogram(inp.get("logits"), inp.get("bias"), blk.mode, blk.ids, blk.w,
                              blk.group_sizes, blk.group_offsets, blk.pos, blk.row_src,
                              blk.status, blk.ws, d)
        mark()
        B.moe_mx_permute_quantize(inp["x"], blk.pos, blk.group_offsets, blk.xq, blk.xsc, d)
        mark()
        B.moe_mx_grouped_gemm_fc1_swiglu(blk.xq, blk.xsc, blk.wiq, blk.wisc, blk.group_offsets,
                                         blk.hq, blk.hsc, None, blk.status, d)
        mark()
        B.moe_mx_grouped_gemm_fc2(blk.hq, blk.hsc, blk.woq, blk.wosc, blk.group_offsets, blk.ys,
                                  blk.status, d)
        mark()
        B.moe_combine(blk.ys, blk.w, blk.pos, blk.out, d)
        mark()

    for _ in range(3):
        run(None)
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flushed else None
    evs = []
    with clock_sampler(dev) as clk:
        for _ in range(steps):
            if flush is not None:
                flush.zero_()
            ev = []
            run(ev)
            evs.append(ev)
        torch.cuda.synchronize()
    clocks = clk.summary()
    if int(blk.status.item()) != 0:
        raise RuntimeError(f"device status {int(blk.status.item())} after the MX steps")
    times = {n: [ev[i].elapsed_time(ev[i + 1]) * 1e-3 for ev in evs] for i, n in enumerate(MX_STEPS)}
    step_s = sum(ev[0].elapsed_time(ev[-1]) * 1e-3 for ev in evs) / steps
    # fp8 dense peak = the clock-matched bf16 peak x 2 (nominal 4.5 / 2.25 PF)
    bf16_peak, bf16_src = tensor_peak(pk, clocks)
    fp8_peak = 2.0 * bf16_peak
    kern = {}
    for n in MX_STEPS:
        avg = sum(times[n]) / len(times[n])
        kern[n] = {"avg_us": avg * 1e6, "median_us": statistics.median(times[n]) * 1e6}
        if n in ("fc1", "fc2"):
            fl = gemm_flops(n, wl.R, wl.D, wl.F)
            kern[n]["tflops"] = fl / avg / 1e12
            kern[n]["frac_tensor"] = fl / avg / 1e12 / fp8_peak
            kern[n]["frac_hbm"] = mx_bytes(n, wl.T, wl.D, wl.E, wl.K, wl.F) / avg / 1e9 / pk["hbm"]
        elif n == "permute_quantize":
            kern[n]["frac_hbm"] = mx_bytes(n, wl.T, wl.D, wl.E, wl.K, wl.F) / avg / 1e9 / pk["hbm"]
        else:
            kern[n]["frac_hbm"] = hbm_bytes(n, wl.T, wl.D, wl.E, wl.K, wl.F) / avg / 1e9 / pk["hbm"]
    return {
        "metric": "MoE block tokens/s (fwd, MXFP8)",
        "value": wl.T / step_s,
        "unit": "tokens/s",
        "ms_per_step": step_s * 1e3,
        "steps": steps,
        "dtype": "e4m3 x e4m3 (E8M0 scales per 32), fp32 accumulation, bf16 out",
        "fp8_peak_tflops": fp8_peak,
        "fp8_peak_source": f"nominal 2 x bf16: {bf16_src}",
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "weights_quantize_us": {k: statistics.median(v) for k, v in qt.items()},
        "gpu_launches_per_step": len(MX_STEPS),
        "kernels": kern,
    }
def mx_train_work(wl, wgrad="mx"):
    """Per launch of the MXFP8 training step: (name, kind, amount) with kind
    "tensor" (FLOPs of a block-scaled GEMM), "tensor_bf16" (FLOPs of a bf16
    grouped GEMM) or "hbm" (algorithmic bytes: bf16 read once, e4m3 codes and
    one scale byte per 32 elements written once).  wgrad="bf16": the weight
    gradients on the bf16 GEMM, with xs kept in bf16 by the forward and no
    operand quantized along tokens."""
    T, D, E, K, F = wl.T, wl.D, wl.E, wl.K, wl.F
    R = T * K

    def quant(n_in, n_out):   # bf16 in, e4m3 + scales out
        return 2 * n_in + n_out + n_out // 32

    if wgrad == "bf16":
        return [
            ("quantize_wi", "hbm", quant(E * D * 2 * F, 2 * E * D * 2 * F)),
            ("quantize_wo", "hbm", quant(E * F * D, 2 * E * F * D)),
            ("route", "hbm", hbm_bytes("route", T, D, E, K, F)),
            ("permute_quantize", "hbm", mx_bytes("permute_quantize", T, D, E, K, F)),
            ("permute_xs_bf16", "hbm", hbm_bytes("permute", T, D, E, K, F)),
            ("fc1", "tensor", gemm_flops("fc1", R, D, F)),
            ("fc2", "tensor", gemm_flops("fc2", R, D, F)),
            ("combine", "hbm", hbm_bytes("combine", T, D, E, K, F)),
            ("combine_bwd_quantize", "hbm",
             hbm_bytes("combine_bwd", T, D, E, K, F) + R * D + R * D // 32),
            ("fc2_dgrad", "tensor", gemm_flops("fc2_dlhs", R, D, F)),
            ("fc2_wgrad_bf16", "tensor_bf16", gemm_flops("fc2_drhs", R, D, F)),
            ("quantize_dz_rows", "hbm", quant(R * 2 * F, R * 2 * F)),
            ("fc1_dgrad", "tensor", gemm_flops("fc1_dlhs", R, D, F)),
            ("fc1_wgrad_bf16", "tensor_bf16", gemm_flops("fc1_drhs", R, D, F)),
            ("permute_bwd", "hbm", hbm_bytes("permute_bwd", T, D, E, K, F)),
        ]
    return [   # each weight read once for its two MX copies
        ("quantize_wi", "hbm", quant(E * D * 2 * F, 2 * E * D * 2 * F)),
        ("quantize_wo", "hbm", quant(E * F * D, 2 * E * F * D)),
        ("route", "hbm", hbm_bytes("route", T, D, E, K, F)),
        ("permute_quantize", "hbm", mx_bytes("permute_quantize", T, D, E, K, F)),
        ("fc1", "tensor", gemm_flops("fc1", R, D, F)),
        ("fc2", "tensor", gemm_flops("fc2", R, D, F)),
        ("combine", "hbm", hbm_bytes("combine", T, D, E, K, F)),
        # the combine backward, writing dys also as MX codes along D
        ("combine_bwd_quantize", "hbm", hbm_bytes("combine_bwd", T, D, E, K, F) + R * D + R * D // 32),
        ("quantize_dys_tokens", "hbm", quant(R * D, R * D)),
        ("quantize_h_tokens", "hbm", quant(R * F, R * F)),
        ("fc2_dgrad", "tensor", gemm_flops("fc2_dlhs", R, D, F)),
        ("fc2_wgrad", "tensor", gemm_flops("fc2_drhs", R, D, F)),
        ("quantize_dz_rows", "hbm", quant(R * 2 * F, R * 2 * F)),
        ("quantize_dz_tokens", "hbm", quant(R * 2 * F, R * 2 * F)),
        ("quantize_x_tokens", "hbm", quant(R * D, R * D) + 4 * R),
        ("fc1_dgrad", "tensor", gemm_flops("fc1_dlhs", R, D, F)),
        ("fc1_wgrad", "tensor", gemm_flops("fc1_drhs", R, D, F)),
        ("permute_bwd", "hbm", hbm_bytes("permute_bwd", T, D, E, K, F)),
    ]


def measure_mx_train(wl, inp, steps, pk, flushed, dev, wgrad="mx"):
    """One MXFP8 training step per iteration through the C ABI: the weight
    quantizations (the weights change every step; one launch per weight
    writes its forward and dgrad copies), the MX forward
    with h and z kept in bf16, and the MX backward (see MoEBlockMX); an event
    pair around every launch.  wgrad="bf16": the weight gradients on the
    bf16 grouped GEMM instead (MoEBlockMX(wgrad="bf16"))."""
    from mixture_experts_ffn_histogram_gb300 import binding as B
    from mixture_experts_ffn_histogram_gb300.block import MoEBlockMX
    blk = MoEBlockMX(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=True, wgrad=wgrad)
    d, D, F = blk.d, wl.D, wl.F
    offs = blk.group_offsets
    if wl.score_mode == B.SCORE_GIVEN:
        blk.ids.copy_(inp["ids"])
        blk.w.copy_(inp["w"])
    wi, wo, x, dy = inp["wi"], inp["wo"], inp["x"], inp["dy"]
    calls = [
        lambda: B.moe_mx_quantize_wi(wi, blk.wiq, blk.wisc, d, wq_bwd=blk.wiq_b,
                                     wsc_bwd=blk.wisc_b),
        lambda: B.moe_mx_quantize_wo(wo, blk.woq, blk.wosc, d, wq_bwd=blk.woq_b,
                                     wsc_bwd=blk.wosc_b),
        lambda: B.moe_route_histogram(inp.get("logits"), inp.get("bias"), blk.mode, blk.ids,
                                      blk.w, blk.group_sizes, offs, blk.pos, blk.row_src,
                                      blk.status, blk.ws, d),
        lambda: B.moe_mx_permute_quantize(x, blk.pos, offs, blk.xq, blk.xsc, d),
        lambda: B.moe_mx_grouped_gemm_fc1_swiglu(blk.xq, blk.xsc, blk.wiq, blk.wisc, offs,
                                                 blk.hq, blk.hsc, blk.h, blk.status, d, z=blk.z),
        lambda: B.moe_mx_grouped_gemm_fc2(blk.hq, blk.hsc, blk.woq, blk.wosc, offs, blk.ys,
                                          blk.status, d),
        lambda: B.moe_combine(blk.ys, blk.w, blk.pos, blk.out, d),
        lambda: B.moe_mx_combine_bwd(dy, blk.ys, blk.w, blk.pos, offs, blk.dys, blk.dyq,
                                     blk.dysc, blk.dw, d),
        lambda: B.moe_mx_quantize_tokens(blk.dys, None, D, offs, blk.dyt, blk.dytsc, d),
        lambda: B.moe_mx_quantize_tokens(blk.h, None, F, offs, blk.ht, blk.htsc, d),
        lambda: B.moe_mx_grouped_gemm_fc2_bwd(blk.dyq, blk.dysc, blk.woq_b, blk.wosc_b, blk.z,
                                              None, None, None, None, offs, blk.dz, None,
                                              blk.status, d),
        lambda: B.moe_mx_grouped_gemm_fc2_bwd(None, None, None, None, None, blk.ht, blk.htsc,
                                              blk.dyt, blk.dytsc, offs, None, blk.dwo,
                                              blk.status, d),
        lambda: B.moe_mx_quantize_rows(blk.dz, 2 * F, offs, blk.dzq, blk.dzsc, d),
        lambda: B.moe_mx_quantize_tokens(blk.dz, None, 2 * F, offs, blk.dzt, blk.dztsc, d),
        lambda: B.moe_mx_quantize_tokens(x, blk.row_src, D, offs, blk.xt, blk.xtsc, d),
        lambda: B.moe_mx_grouped_gemm_fc1_bwd(blk.dzq, blk.dzsc, blk.wiq_b, blk.wisc_b, None,
                                              None, None, None, offs, blk.dxs, None, blk.status,
                                              d),
        lambda: B.moe_mx_grouped_gemm_fc1_bwd(None, None, None, None, blk.xt, blk.xtsc, blk.dzt,
                                              blk.dztsc, offs, None, blk.dwi, blk.status, d),
        lambda: B.moe_permute_bwd(blk.dxs, blk.pos, blk.dx, d),
    ]
    if wgrad == "bf16":
        calls = calls[:4] + [lambda: B.moe_permute(x, blk.pos, blk.xs, d)] + calls[4:8] + [
            calls[10],
            lambda: B.moe_grouped_gemm_fc2_bwd(blk.dys, blk.h, None, None, offs, None, blk.dwo,
                                               blk.status, blk.ws, d),
            calls[12],
            calls[15],
            lambda: B.moe_grouped_gemm_fc1_swiglu_bwd(blk.dz, None, blk.xs, None, offs, None,
                                                      blk.dwi, blk.status, blk.ws, d),
            calls[17],
        ]
    work = mx_train_work(wl, wgrad)
    assert len(work) == len(calls)

    def run(ev):
        for c in calls:
            if ev is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record()
                ev.append(e)
            c()
        if ev is not None:
            e = torch.cuda.Event(enable_timing=True)
            e.record()
            ev.append(e)

    for _ in range(3):
        run(None)
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flushed else None
    evs = []
    with clock_sampler(dev) as clk:
        for _ in range(steps):
            if flush is not None:
                flush.zero_()
            ev = []
            run(ev)
            evs.append(ev)
        torch.cuda.synchronize()
    clocks = clk.summary()
    if int(blk.status.item()) != 0:
        raise RuntimeError(f"device status {int(blk.status.item())} after the MX training steps")
    step_s = sum(ev[0].elapsed_time(ev[-1]) * 1e-3 for ev in evs) / steps
    bf16_peak, bf16_src = tensor_peak(pk, clocks)
    fp8_peak = 2.0 * bf16_peak
    kern = {}
    gemm_s = 0.0
    for i, (n, kind, amount) in enumerate(work):
        ts = [ev[i].elapsed_time(ev[i + 1]) * 1e-3 for ev in evs]
        avg = sum(ts) / len(ts)
        k = {"avg_us": avg * 1e6, "median_us": statistics.median(ts) * 1e6}
        if kind == "tensor":
            k["tflops"] = amount / avg / 1e12
            k["frac_tensor"] = amount / avg / 1e12 / fp8_peak
            gemm_s += avg
        elif kind == "tensor_bf16":
            k["tflops"] = amount / avg / 1e12
            k["frac_tensor_bf16"] = amount / avg / 1e12 / bf16_peak
        else:
            k["gbs"] = amount / avg / 1e9
            k["frac_hbm"] = amount / avg / 1e9 / pk["hbm"]
        kern[n] = k
    flops = sum(a for _, kind, a in work if kind == "tensor")
    mx_gemms = "all six GEMMs" if wgrad == "mx" else "the forward GEMMs and both dgrads"
    return {
        "metric": "MoE block tokens/s (fwd+bwd, MXFP8)" if wgrad == "mx" else
                  "MoE block tokens/s (fwd+bwd, MXFP8 forward and dgrads, bf16 weight gradients)",
        "value": wl.T / step_s,
        "unit": "tokens/s",
        "ms_per_step": step_s * 1e3,
        "steps": steps,
        "dtype": f"e4m3 x e4m3 (E8M0 scales per 32) in {mx_gemms}, fp32 accumulation, "
                 "bf16 activations and gradients between them" +
                 ("" if wgrad == "mx" else "; bf16 x bf16 weight gradients"),
        "step": "weights quantized (2 launches, both copies) + MX forward + MX backward" +
                ("" if wgrad == "mx" else " (weight gradients on the bf16 GEMM)"),
        "fp8_peak_tflops": fp8_peak,
        "fp8_peak_source": f"nominal 2 x bf16: {bf16_src}",
        "gemm_ms": gemm_s * 1e3,
        "gemm_frac_tensor": flops / gemm_s / 1e12 / fp8_peak if gemm_s > 0 else None,
        "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "gpu_launches_per_step": len(calls),
        "kernels": kern,
    }


L2_BYTES = 129 << 20


def input_footprint(inp: dict) -> int:
    """Bytes of the tensors among a step's inputs (what a step reads at least once)."""
    return sum(t.numel() * t.element_size() for t in inp.values() if isinstance(t, torch.Tensor))


def kernel_table(wl, names, times, fwd_only, pk, tpeak):
    """Per-kernel figures of a timed run and the block's roofline.

    Each kernel is held to the resource that binds it at the peaks: a GEMM
    to the tensor peak `tpeak`, or to the HBM peak when its algorithmic bytes
    take longer at the HBM peak than its FLOPs at the tensor peak (weight
    streaming at few rows per expert); the other steps to the HBM peak.  The
    block's roofline is the sum of its kernels' roofline times."""
    total = max(1e-12, sum(sum(v) for v in times.values()))
    per_kernel, roof_s = {}, 0.0
    for n in names:
        ts = times[n]
        avg = sum(ts) / len(ts)
        k = {"avg_us": avg * 1e6, "median_us": statistics.median(ts) * 1e6,
             "share": sum(ts) / total}
        if n in GEMMS:
            fl = gemm_flops(n, wl.R, wl.D, wl.F)
            by = gemm_bytes(n, wl.R, wl.D, wl.E, wl.F, not fwd_only)
            t_t, t_h = fl / (tpeak * 1e12), by / (pk["hbm"] * 1e9)
            k.update(tflops=fl / avg / 1e12, frac_tensor=fl / avg / 1e12 / tpeak,
                     hbm_gbs_algorithmic=by / avg / 1e9, frac_hbm=by / avg / 1e9 / pk["hbm"],
                     bound="hbm" if t_h > t_t else "tensor")
            t_roof = max(t_t, t_h)
        else:
            by = hbm_bytes(n, wl.T, wl.D, wl.E, wl.K, wl.F)
            t_roof = by / (pk["hbm"] * 1e9)
            k.update(gbs=by / avg / 1e9, frac_hbm=by / avg / 1e9 / pk["hbm"], bound="hbm")
        k["roofline_us"] = t_roof * 1e6
        k["frac_roofline"] = t_roof / avg
        roof_s += t_roof
        per_kernel[n] = k
    return per_kernel, roof_s


def dominant_roofline(wl, step, per_kernel, fwd_only, pk, tpeak, tpeak_src):
    """The `roofline` object: the kernel with the largest share of the step,
    its algorithmic FLOPs or bytes per launch over its mean launch time."""
    dom = max(step.names, key=lambda n: sum(step.times[n]))
    k = per_kernel[dom]
    avg = k["avg_us"] * 1e-6
    if dom in GEMMS and k["bound"] == "tensor":
        achieved = gemm_flops(dom, wl.R, wl.D, wl.F) / avg / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": tpeak,
                "unit": "TFLOP/s", "frac": achieved / tpeak, "peak_source": tpeak_src}
    else:
        by = (gemm_bytes(dom, wl.R, wl.D, wl.E, wl.F, not fwd_only) if dom in GEMMS
              else hbm_bytes(dom, wl.T, wl.D, wl.E, wl.K, wl.F))
        achieved = by / avg / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": pk["hbm"],
                "unit": "GB/s", "frac": achieved / pk["hbm"],
                "peak_source": f"{pk['source']} hbm_gbs"}
    roof["traffic"] = recorded_traffic(dom, wl.name)
    return roof


def measure_workload(wl, inp, steps, warmup, fwd_only, dev, dist=None):
    """Times `steps` block steps of `wl` after `warmup` untimed ones, with a
    CUDA event pair around every launch and the SM clock sampled throughout.
    Inputs that fit in L2 get L2 flushed (a 256 MB write, not timed) before
    every timed step.  Returns (step, elapsed seconds, clocks, flushed)."""
    step = Step(wl, inp, fwd_only)
    for _ in range(max(warmup, 3)):
        step.run()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) \
        if input_footprint(inp) < L2_BYTES else None
    with clock_sampler(dev) as clk:
        if flush is None:
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record()
            for _ in range(steps):
                step.run(record=True)
            end.record()
            torch.cuda.synchronize()
            elapsed = start.elapsed_time(end) * 1e-3
        else:
            marks = []
            for _ in range(steps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                step.run(record=True)
                b.record()
                marks.append((a, b))
            torch.cuda.synchronize()
            elapsed = sum(a.elapsed_time(b) for a, b in marks) * 1e-3
    barrier(dist)
    step.collect()
    status = int(step.blk.status.item())
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed steps of {wl.name}")
    return step, elapsed, clk.summary(), flush is not None


def measure_fused(wl, inp, steps, dev, flushed):
    """The inference forward through moe_fused_forward (routing, FC1 on rows
    gathered from x, FC2 with the weighted combine in its epilogue, the fp32
    accumulator converted to bf16), one event pair around each step."""
    from mixture_experts_ffn_histogram_gb300.block import MoEBlock
    blk = MoEBlock(wl.T, wl.D, wl.E, wl.K, wl.F, wl.score_mode, train=False, device=dev)

    def one():
        blk.forward_fused(inp["x"], inp["wi"], inp["wo"], logits=inp.get("logits"),
                          bias=inp.get("bias"), ids=inp.get("ids"), w=inp.get("w"))

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flushed else None
    marks = []
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        one()
        b.record()
        marks.append((a, b))
    torch.cuda.synchronize()
    if int(blk.status.item()) != 0:
        raise RuntimeError(f"device status {int(blk.status.item())} after the fused steps")
    step_s = sum(a.elapsed_time(b) for a, b in marks) * 1e-3 / steps
    return {"tokens_per_s": wl.T / step_s, "ms_per_step": step_s * 1e3,
            "launches_per_step": 5, "l2_flushed": flushed}


# every configuration of the block's workloads, with the pass each is quoted on
CONFIG_SWEEP = ("tiny_fwd", "token_sweep_T1024", "token_sweep_T2048", "token_sweep_T4096",
                "token_sweep_T8192", "long_seq_train", "large_expert_train", "zipf_skew_train")


def measure_configs(steps, warmup, dev, pk, skip=()):
    """Every configuration, each in its own timed loop on fresh inputs:
    tokens/s, the block roofline at the peaks (tensor peak matched to the
    clocks sampled during that loop), and per-kernel fractions."""
    res = []
    for name in CONFIG_SWEEP:
        if name in skip:
            continue
        wl = WORKLOADS[name]
        fwd_only = not wl.train
        inp = make_inputs(wl, dev, with_grad=not fwd_only)
        step, el, clocks, flushed = measure_workload(wl, inp, steps, warmup, fwd_only, dev)
        tpeak, _ = tensor_peak(pk, clocks)
        kern, roof_s = kernel_table(wl, step.names, step.times, fwd_only, pk, tpeak)
        step_s = el / steps
        res.append({
            "workload": name, "pass": "fwd" if fwd_only else "fwd+bwd",
            "T": wl.T, "D": wl.D, "E": wl.E, "K": wl.K, "F": wl.F,
            "tokens_per_s": wl.T / step_s, "ms_per_step": step_s * 1e3, "steps": steps,
            "roofline_ms": roof_s * 1e3, "roofline_frac": roof_s / step_s,
            "tensor_peak_tflops": tpeak, "l2_flushed": flushed,
            "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
            "kernels": {n: {"median_us": v["median_us"], "bound": v["bound"],
                            "frac_roofline": v["frac_roofline"]} for n, v in kern.items()},
        })
        if fwd_only:
            # the same forward through the fused entry point (no xs, no ys)
            res[-1]["fused_forward"] = measure_fused(wl, inp, steps, dev, flushed)
        del step, inp
        torch.cuda.empty_cache()
    return res


def run_ours(args, dist, rank, world):
    wl = selected_workload(args)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    from mixture_experts_ffn_histogram_gb300 import _build
    _build.build()
    from dataclasses import replace
    wl_rank = replace(wl, seed=wl.seed + rank)
    fwd_only = args.fwd_only or not wl.train
    inp = make_inputs(wl_rank, dev, with_grad=not fwd_only)
    # ---- timed region: K steps, events around every launch
    step, elapsed, clocks, flushed = measure_workload(wl_rank, inp, args.steps, args.warmup,
                                                      fwd_only, dev, dist)
    elapsed_max = max_over_ranks(dist, elapsed)
    pk = peaks()
    tpeak, tpeak_src = tensor_peak(pk, clocks)

    # ---- forward-only tokens/s, same inputs (a separate timed loop)
    fwd_tps = None
    if not fwd_only:
        fstep = Step(wl_rank, inp, True)
        for _ in range(3):
            fstep.run()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(args.steps):
            fstep.run()
        s1.record()
        torch.cuda.synchronize()
        fwd_tps = wl.T * args.steps / (s0.elapsed_time(s1) * 1e-3)
        del fstep

    # ---- the MXFP8 forward on the same inputs (a separate timed loop)
    mx = mx_train = mx_train_bw = None
    if not args.no_mx:
        mx = measure_mx(wl_rank, inp, args.steps, pk, flushed, dev)
        if not fwd_only:
            mx_train = measure_mx_train(wl_rank, inp, args.steps, pk, flushed, dev)
            mx_train_bw = measure_mx_train(wl_rank, inp, args.steps, pk, flushed, dev,
                                           wgrad="bf16")

    # ---- end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(step, inp, args, dist, fwd_only)

    T = wl.T
    value = world * T * args.steps / elapsed_max
    launches = step.launches_per_step
    per_kernel, roof_s = kernel_table(wl, step.names, step.times, fwd_only, pk, tpeak)
    roof = dominant_roofline(wl, step, per_kernel, fwd_only, pk, tpeak, tpeak_src)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, fwd_only, budget_s=20.0)
        if mx is not None:
            mx["cpu_baseline"] = mx_cpu_baseline(wl, budget_s=10.0)

    configs = None
    if rank == 0 and world == 1 and not args.no_configs and args.tokens is None \
            and args.experts is None:
        del step, inp
        torch.cuda.empty_cache()
        configs = measure_configs(min(args.steps, 10), 3, dev, pk)

    line = {
        "metric": METRIC_FWD if fwd_only else METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_max / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": wl.name, "T": wl.T, "D": wl.D, "E": wl.E, "K": wl.K, "F": wl.F,
                   "pass": "fwd" if fwd_only else "fwd+bwd",
                   "l2": "L2 flushed before each timed step (256 MB write, not timed)" if flushed
                         else "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "block_roofline": {"ms_per_step": roof_s * 1e3,
                           "frac": roof_s / (elapsed / args.steps),
                           "tensor_peak_tflops": tpeak, "tensor_peak_source": tpeak_src,
                           "hbm_peak_gbs": pk["hbm"]},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "kernels": per_kernel,
    }
    if fwd_tps is not None:
        line["fwd_tokens_per_s"] = world * fwd_tps
    if mx is not None:
        mx["value"] *= world
        line["mxfp8_forward"] = mx
    if mx_train is not None:
        mx_train["value"] *= world
        line["mxfp8_train"] = mx_train
    if mx_train_bw is not None:
        mx_train_bw["value"] *= world
        line["mxfp8_train_bf16_wgrad"] = mx_train_bw
    if configs is not None:
        line["configs"] = configs
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_e2e(step, inp, args, dist, fwd_only):
    """The same steps through the block's host-memory API (HostPipeline):
    every step's activations are copied in from pinned host memory and its
    outputs (out, and dx when training) copied back inside the timed region,
    with the copies overlapped with the kernels of neighbouring steps."""
    from mixture_experts_ffn_histogram_gb300.block import HostPipeline
    wl = step.wl
    given = step.blk.mode == step.B.SCORE_GIVEN
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    host = {"x_h": pin(inp["x"])}
    if given:
        host["ids_h"], host["w_h"] = pin(inp["ids"]), pin(inp["w"])
    else:
        host["logits_h"] = pin(inp["logits"])
    if not fwd_only:
        host["dy_h"] = pin(inp["dy"])
    out_h = torch.empty_like(step.blk.out, device="cpu").pin_memory()
    dx_h = None if fwd_only else torch.empty_like(step.blk.out, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * 2 + (dx_h.numel() * 2 if dx_h is not None else 0)
    pipe = HostPipeline(step.blk, inp["wi"], inp["wo"], inp["bias"])

    def one():
        pipe.step(out_h=out_h, dx_h=dx_h, **host)

    for _ in range(2):
        one()
    pipe.synchronize()
    torch.cuda.synchronize()
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    pipe.synchronize()
    el = max_over_ranks(dist, time.perf_counter() - t0)
    status = int(step.blk.status.item())
    if status != 0:
        raise RuntimeError(f"device status {status} after the end-to-end steps")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": world * wl.T * args.steps / el, "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "overlapped with neighbouring steps' kernels (upload, compute and "
                      "download streams)"}


# ------------------------------------------------------ oracle (CPU) arm
def _sample_workload(wl, T_sample):
    from dataclasses import replace
    return replace(wl, T=T_sample)


def _oracle_step(wl_s, inp_np, fwd_only):
    import oracle
    fwd = oracle.block_forward(inp_np, want_z=not fwd_only)
    if not fwd_only:
        oracle.block_backward(inp_np, fwd)


def _oracle_inputs(wl_s, fwd_only):
    import oracle
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    return oracle.to_numpy(make_inputs(wl_s, dev, with_grad=not fwd_only))


def cpu_baseline(wl, fwd_only, budget_s=20.0, T_sample=None):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload (the first T_sample tokens' worth of a draw with the same sizes)."""
    import oracle
    oracle.build()
    if T_sample is None:
        T_sample = 16
        probe = _oracle_inputs(_sample_workload(wl, T_sample), fwd_only)
        t0 = time.perf_counter()
        _oracle_step(None, probe, fwd_only)
        dt = time.perf_counter() - t0
        # the weight-gradient part does not shrink with T; scale the token part
        T_sample = int(max(16, min(wl.T, T_sample * budget_s / max(dt, 1e-3) / 2)))
    wl_s = _sample_workload(wl, T_sample)
    inp = _oracle_inputs(wl_s, fwd_only)
    t0 = time.perf_counter()
    _oracle_step(wl_s, inp, fwd_only)
    dt = time.perf_counter() - t0
    return {"value": T_sample / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{T_sample} of {wl.T} tokens of {wl.name} (same D,E,K,F), "
                      f"{'fwd' if fwd_only else 'fwd+bwd'}, one pass, {dt:.1f} s"}


def _oracle_mx_step(wl_s, inp, wq):
    """The oracle's MX forward of one step, the weights already quantized
    (as the GPU leg runs it): route, histogram, permute + quantize, FC1 +
    SwiGLU, quantize h, FC2, combine."""
    import oracle
    if wl_s.score_mode == oracle.GIVEN:
        ids, w = inp["ids"], inp["w"]
    else:
        ids, w = oracle.route(inp["logits"], inp["bias"], wl_s.score_mode, wl_s.T, wl_s.E, wl_s.K)
    _, off, pos, _, _ = oracle.histogram(ids, wl_s.E)
    xq, xsc = oracle.mx_quantize(oracle.bf16_to_f32(oracle.permute(inp["x"], pos)))
    h = oracle.mx_fc1_swiglu(xq, xsc, wq[0], wq[1], off)
    hq, hsc = oracle.mx_quantize(h)
    ys = oracle.mx_fc2(hq, hsc, wq[2], wq[3], off)
    oracle.combine(ys, w, pos, wl_s.T, wl_s.D)


def mx_cpu_baseline(wl, budget_s=10.0):
    """The oracle's MX forward on the host cores, on a bounded token sample of
    the workload; the weights are quantized once, outside the timing."""
    import oracle
    oracle.build()
    wl8 = _sample_workload(wl, 8)
    inp = _oracle_inputs(wl8, True)
    wq = oracle.mx_weights(inp["wi"], inp["wo"])
    t0 = time.perf_counter()
    _oracle_mx_step(wl8, inp, wq)
    dt = time.perf_counter() - t0
    T_sample = int(max(8, min(wl.T, 8 * budget_s / max(dt, 1e-3))))
    wl_s = _sample_workload(wl, T_sample)
    inp = _oracle_inputs(wl_s, True)
    t0 = time.perf_counter()
    _oracle_mx_step(wl_s, inp, wq)
    dt = time.perf_counter() - t0
    return {"value": T_sample / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{T_sample} of {wl.T} tokens of {wl.name} (same D,E,K,F), MXFP8 fwd, "
                      f"weights quantized beforehand, one pass, {dt:.1f} s"}


def run_reference(args, dist, rank, world):
    if rank != 0:
        return
    wl = selected_workload(args)
    fwd_only = args.fwd_only or not wl.train
    import oracle
    oracle.build()
    # size the per-step sample so that warmup+steps end within ~3 minutes
    steps_total = max(args.warmup, 0) + args.steps
    per_step = max(2.0, 180.0 / max(1, steps_total))
    T_sample = 8
    probe = _oracle_inputs(_sample_workload(wl, T_sample), fwd_only)
    t0 = time.perf_counter()
    _oracle_step(None, probe, fwd_only)
    dt = time.perf_counter() - t0
    T_sample = int(max(8, min(wl.T, T_sample * per_step / max(dt, 1e-3) / 2)))
    wl_s = _sample_workload(wl, T_sample)
    inp = _oracle_inputs(wl_s, fwd_only)
    for _ in range(args.warmup):
        _oracle_step(wl_s, inp, fwd_only)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(wl_s, inp, fwd_only)
    el = time.perf_counter() - t0
    value = T_sample * args.steps / el
    line = {
        "impl": "reference",
        "metric": METRIC_FWD if fwd_only else METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": wl.name, "T": wl.T, "D": wl.D, "E": wl.E, "K": wl.K, "F": wl.F,
                   "pass": "fwd" if fwd_only else "fwd+bwd", "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"{T_sample} of {wl.T} tokens per step, same D,E,K,F"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    dist, rank, world, _ = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, dist, rank, world)
        else:
            run_ours(args, dist, rank, world)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
