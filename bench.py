#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on B300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extra] [--no-cpu-baseline] [--no-e2e]
                    [--only backward|fp8]

A "step" is one launch of the hot path on one batch of the workload: by default
the causal prefill of B=4, Hq=Hkv=16, N=4096, d=128 (bf16 in, f32 accumulate,
bf16 O + f32 LSE), whose TFLOP/s is the headline value.  The same line carries
the split-KV decode workloads (million-token and batched GQA, GB/s of K/V) and
the local-window prefill as sub-objects, each with its own roofline.

Timing: W warm-up launches, then K launches bracketed by CUDA events on the
launching stream with a device synchronise (and, for N > 1, a barrier) on both
sides; the max over ranks is taken.  Every workload's inputs exceed the 126 MB
L2 (said in ``config.l2``), so no flush runs between launches.  SM clocks and
throttle reasons are polled through NVML during the timed region.

``--impl reference`` times the float64 CPU oracle (the deliberately slow
reference of this repository) on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s & decode KV GB/s on 1 B300, as % of roofline"
PKG = "exact_transformer_attention_flashattention_b300"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
NAMEPLATE_HBM_GBS = 8000.0
PLAIN_PAUSE_S = 1.5  # idle seconds before the plain-launch timing (clock recovery)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="causal_prefill_4k")
    ap.add_argument("--no-extra", action="store_true", help="skip the decode/window sub-objects")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["backward", "fp8", "decode", "prefill"], default=None,
                    help="time one extra leg of a prefill workload alone and print its object "
                         "(a small command for kernel profiles; not the benchmark line)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--extra-cpu-budget", type=float, default=4.0,
                    help="seconds of oracle work for each sub-workload's cpu_baseline")
    return ap.parse_args()


def profile_workloads():
    """Scaled shapes for ncu captures (a few GB on the device at most): the
    million-token decode with a quarter of its keys and splits."""
    from exact_transformer_attention_flashattention_b300.inputs import Workload
    return {"decode_256k": Workload("decode_256k", "decode", B=1, Hq=32, Hkv=8, N=1 << 18,
                                    d=128, seed=4, num_splits=512)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# device-code files each profiled kernel is compiled from
KERNEL_SOURCES = {
    "prefill_kernel": ("prefill.cuh", "ptx.cuh"),
    # (+ the host file that sets its tensor maps' L2 fetch granule)
    "prefill_band_kernel": ("band.cuh", "prefill.cuh", "ptx.cuh", "b300attn.cu"),
    "decode_partial_kernel": ("decode.cuh", "ptx.cuh"),
    "bwd_dkdv_kernel": ("backward.cuh", "ptx.cuh"),
    "fp8_quantize_kernel": ("fp8.cuh", "ptx.cuh"),
}


# Widest window (keys on each side) that attn_fwd sends to the band kernel.
BAND_MAX_WINDOW = 256


def prefill_kernel_name(d: int, causal: bool, window: int) -> str:
    """The kernel attn_fwd runs for a dense bf16 prefill: the band kernel for a
    short non-causal window at d = 64, prefill_kernel otherwise."""
    if d == 64 and not causal and 0 <= window <= BAND_MAX_WINDOW:
        return "prefill_band_kernel"
    return "prefill_kernel"


def kernel_source_sha(kernel: str = "prefill_kernel"):
    """Hash of the device code of `kernel` (the .cuh files it is compiled
    from); a stored ncu traffic figure is used only if it was taken from the
    same device code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, PKG, "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rows = json.load(f)
    except (OSError, ValueError):
        return None
    sha = kernel_source_sha(kernel)
    for r in rows:
        if r.get("kernel") == kernel and r.get("workload") == workload and r.get("source_sha") == sha:
            return r.get("dram_bytes_per_launch")
    return None


# ----------------------------------------------------------------- distributed
class Dist:
    """Rank bookkeeping for N independent replicas (one process per GPU, launched
    by torchrun).  The only collectives are the barrier around the timed region
    and the max of the per-rank times; the data path has none.  ``backend``
    defaults to NCCL on a GPU machine and gloo elsewhere (the CPU tests)."""

    def __init__(self, gpus: int, backend: str | None = None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cpu"
        if self.world > 1:
            import torch
            import torch.distributed as dist
            if backend is None:
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            self.device = "cuda" if backend == "nccl" else "cpu"
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------- clocks
class _Nvml:
    """Read-only NVML access: the pynvml module when it is installed, else the
    driver's libnvidia-ml.so.1 through ctypes.  Only clocks and clock-event
    reasons are read; no setting of the GPU is changed."""

    CLOCK_SM = 1

    def __init__(self, uuid: str | None, index: int):
        try:
            import pynvml
            pynvml.nvmlInit()
            self.kind = "pynvml"
            self.nv = pynvml
            h = None
            if uuid:
                try:
                    h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
                except Exception:
                    h = None
            self.h = h if h is not None else pynvml.nvmlDeviceGetHandleByIndex(index)
            self._reasons = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                pynvml.nvmlDeviceGetCurrentClocksThrottleReasons
            return
        except ImportError:
            pass
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.kind = "libnvidia-ml (ctypes)"
        self.lib = lib
        self.ct = ctypes
        h = ctypes.c_void_p()
        rc = -1
        if uuid:
            rc = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h))
        if rc != 0:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
        if rc != 0:
            raise RuntimeError(f"NVML handle lookup failed ({rc})")
        self.h = h
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons_fn = fn if fn is not None else lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self) -> int:
        if self.kind == "pynvml":
            return self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM)
        v = self.ct.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.ct.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetClockInfo failed")
        return int(v.value)

    def max_sm_mhz(self) -> int:
        if self.kind == "pynvml":
            return self.nv.nvmlDeviceGetMaxClockInfo(self.h, self.nv.NVML_CLOCK_SM)
        v = self.ct.c_uint()
        if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.ct.byref(v)) != 0:
            raise RuntimeError("nvmlDeviceGetMaxClockInfo failed")
        return int(v.value)

    def reasons(self) -> int:
        if self.kind == "pynvml":
            return int(self._reasons(self.h))
        v = self.ct.c_ulonglong()
        if self._reasons_fn(self.h, self.ct.byref(v)) != 0:
            return 0
        return int(v.value)


class ClockSampler:
    """Polls SM clock and clock-event (throttle) reasons through NVML from a
    background thread; ``window`` marks the timed region and the summary uses
    the samples taken inside it (all samples if the region was too short)."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4,
        "hw_slowdown": 0x8, "sync_boost": 0x10, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
        "display_clock_setting": 0x100,
    }

    def __init__(self, device_index: int):
        self.ok = False
        self.index = device_index
        self.samples = []  # (time, sm_mhz, reasons)
        self.t0 = self.t1 = None
        self.max_mhz = None
        self.error = None
        try:
            uuid = None
            try:  # NVML numbers all GPUs; find the one CUDA calls device_index
                import torch
                u = str(torch.cuda.get_device_properties(device_index).uuid)
                uuid = u if u.startswith("GPU-") else "GPU-" + u
            except Exception as e:
                self.error = "uuid lookup: " + repr(e)
            self.nvml = _Nvml(uuid, device_index)
            self.max_mhz = self.nvml.max_sm_mhz()
            self.ok = True
        except Exception as e:  # no NVML at all: one nvidia-smi query after the run
            self.error = repr(e)

    def _poll(self):
        while not self._stop.is_set():
            try:
                mhz = self.nvml.sm_mhz()
            except Exception:
                mhz = None
            try:
                rs = self.nvml.reasons()
            except Exception:
                rs = 0
            if mhz is not None:
                self.samples.append((time.perf_counter(), mhz, rs))
            time.sleep(0.0005)

    def _smi_fallback(self):
        """One nvidia-smi query after the run when NVML gave no samples."""
        import subprocess
        try:
            out = subprocess.run(
                ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-i", str(self.index)],
                capture_output=True, text=True, timeout=20).stdout.strip().splitlines()[0]
            sm, mx, act = [x.strip() for x in out.split(",")]
            return {"sm_mhz": float(sm), "sm_max_mhz": float(mx), "samples": 1,
                    "in_timed_region": False, "reasons_bits": act, "source": "nvidia-smi after",
                    "nvml_error": self.error}
        except Exception as e:
            return {"error": f"no clock samples (NVML: {self.error}; nvidia-smi: {e!r})"}

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stats(self, t0, t1):
        """Median SM clock and the throttle reasons seen between t0 and t1."""
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "samples": 0, "reasons": []}
        bits = 0
        for s in inside:
            bits |= s[2]
        return {"sm_mhz": float(statistics.median(s[1] for s in inside)), "samples": len(inside),
                "reasons": [n for n, bit in self.REASONS.items() if bits & bit and n != "gpu_idle"]}

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._poll, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return self._smi_fallback()
        inside = [s for s in self.samples
                  if self.t0 is not None and self.t0 <= s[0] <= self.t1]
        use = inside or self.samples
        bits = 0
        for s in use:
            bits |= s[2]
        names = [n for n, bit in self.REASONS.items() if bits & bit and n != "gpu_idle"]
        return {"sm_mhz": float(statistics.median(s[1] for s in use)),
                "sm_max_mhz": self.max_mhz, "samples": len(use),
                "in_timed_region": bool(inside), "reasons": names,
                "source": "NVML via " + self.nvml.kind}


# ----------------------------------------------------------------- timing
LAST_TIMING = {}  # how the last time_launches call timed (mode, host enqueue time per call)


def time_launches(fn, steps: int, warmup: int, dist: Dist, clocks=None, graph: bool = True):
    """Average device time of one call of ``fn`` (ms), CUDA events on the
    current stream, max over ranks.

    With ``graph`` the call is captured once in a CUDA graph (after the
    warm-up) and the timed region replays it ``steps`` times: each replay runs
    exactly the kernels of one call, without the per-call host work (argument
    checks, tensor-map encoding, ctypes), which for short kernels would
    otherwise leave the GPU idle between launches.  If capture fails the
    calls are timed as plain launches."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    run = fn
    mode = "plain launches"
    if graph:
        try:
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    fn()
            torch.cuda.current_stream().wait_stream(s)
            g.replay()
            torch.cuda.synchronize()
            run = g.replay
            mode = "cuda graph replay (one call per replay)"
        except Exception as e:  # capture not possible: time plain launches
            mode = f"plain launches (graph capture failed: {type(e).__name__})"
    dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    start.record()
    for _ in range(steps):
        run()
    end.record()
    t_enq = time.perf_counter()
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if clocks is not None:
        clocks.window(t0, t1)
    dist.barrier()
    LAST_TIMING.clear()
    LAST_TIMING.update({"mode": mode, "host_enqueue_ms_per_call": round((t_enq - t0) / steps * 1e3, 4),
                        "_t0": t0, "_t1": t1})
    return dist.max(start.elapsed_time(end) / steps)


def public_timing(t: dict) -> dict:
    return {k: v for k, v in t.items() if not k.startswith("_")}


def whole_job_rate(units_per_rank: float, world: int, ms_max: float, scale: float) -> float:
    """Aggregate throughput of all ranks: every rank processes `units_per_rank`
    units, the job takes the slowest rank's time `ms_max` (ms); `scale` converts
    units/s to the reported unit (1e12 for TFLOP/s, 1e9 for GB/s)."""
    return units_per_rank * world / (ms_max * 1e-3) / scale


def roofline(achieved, peak, unit, bound, traffic, per_launch_units, unit_name):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_per_launch": per_launch_units, "algorithmic_unit": unit_name}


# ----------------------------------------------------------------- workloads
def prefill_case(w, dev):
    import torch
    from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs
    q, k, v = (t.to(dev) for t in prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed))
    o = torch.empty(w.B, w.N, w.Hq, w.d, dtype=torch.float32 if w.o_fp32 else torch.bfloat16,
                    device=dev)
    lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device=dev)
    return q, k, v, o, lse


def bench_prefill(w, steps, warmup, dist, peaks, peak_kind, clocks=None):
    import torch
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import prefill_flops
    q, k, v, o, lse = prefill_case(w, "cuda")
    flops = prefill_flops(w.B, w.Hq, w.N, w.d, w.causal, w.window)

    def step():
        fa.attn_fwd(q, k, v, causal=w.causal, window=w.window, scale=w.scale, out=o, lse=lse)

    own = clocks is None
    if own:
        clocks = ClockSampler(torch.cuda.current_device())
    with clocks:
        ms = time_launches(step, steps, warmup, dist, clocks)
        timing = dict(LAST_TIMING)
        graph_clk = clocks.stats(timing["_t0"], timing["_t1"])
        # Plain launches, after an idle pause: a long burst of this kernel
        # draws enough power that the SM clock steps down within tens of ms,
        # so whichever of two back-to-back timings runs second would see a
        # lower clock.  The pause lets the clock return before the second one.
        time.sleep(PLAIN_PAUSE_S)
        ms_plain = time_launches(step, steps, warmup, dist, graph=False)
        plain_clk = clocks.stats(LAST_TIMING["_t0"], LAST_TIMING["_t1"])
    if not own:
        clocks.window(timing["_t0"], timing["_t1"])
    timing = public_timing(timing)
    timing["graph_clock_mhz"] = graph_clk["sm_mhz"]
    timing["plain_launch_ms"] = round(ms_plain, 5)
    timing["plain_host_enqueue_ms_per_call"] = LAST_TIMING["host_enqueue_ms_per_call"]
    timing["plain_clock_mhz"] = plain_clk["sm_mhz"]
    timing["plain_reasons"] = plain_clk["reasons"]
    assert fa.device_status() == 0, fa.last_error()
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    kname = prefill_kernel_name(w.d, w.causal, w.window)
    rf = roofline(tflops, peak, "TFLOP/s", "tensor", stored_traffic(kname, w.name), flops, "FLOP")
    rf["kernel"] = kname
    rf["peak_kind"] = f"{peak_kind} dense bf16 (burst)"
    rf["frac_of_sustained"] = round(tflops / peaks.get("bf16_tflops_sustained", peak), 4)
    io_bytes = (q.numel() + k.numel() + v.numel()) * 2 + o.numel() * o.element_size() + lse.numel() * 4
    return {"ms": ms, "tflops": tflops, "flops": flops, "roofline": rf, "io_bytes": io_bytes,
            "launches_per_step": 1, "timing": timing}


def bench_backward(w, steps, warmup, dist, peaks, peak_kind, cpu_budget=0.0):
    """The backward of the prefill workload (dQ, dK, dV from O, LSE and a random
    dO).  Algorithmic work: five products of 2*d flops per unmasked pair (S, dP,
    dV, dK, dQ), 2.5 times the forward's; the kernels recompute S and dP once
    more for the separate dQ pass, which is not counted."""
    import torch
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import prefill_flops
    q, k, v, o, lse = prefill_case(w, "cuda")
    fa.attn_fwd(q, k, v, causal=w.causal, window=w.window, scale=w.scale, out=o, lse=lse)
    g = torch.Generator("cuda").manual_seed(w.seed + 100)
    dO = torch.randn(q.shape, generator=g, device="cuda").to(torch.bfloat16)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.attn_bwd_workspace_size(w.B, w.Hq, w.N), dtype=torch.uint8, device="cuda")
    flops = 2.5 * prefill_flops(w.B, w.Hq, w.N, w.d, w.causal, w.window)

    def step():
        fa.attn_bwd(q, k, v, o, lse, dO, causal=w.causal, window=w.window, scale=w.scale,
                    dq=dq, dk=dk, dv=dv, workspace=ws)

    ms = time_launches(step, steps, warmup, dist)
    timing = public_timing(LAST_TIMING)
    assert fa.device_status() == 0, fa.last_error()
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    rf = roofline(tflops, peak, "TFLOP/s", "tensor", None, flops, "FLOP")
    rf["peak_kind"] = f"{peak_kind} dense bf16 (burst)"
    # traffic of the three launches is not one kernel's; the dK/dV kernel's own
    # DRAM bytes (ncu) are reported beside the roofline
    rf["traffic_bwd_dkdv_kernel"] = stored_traffic("bwd_dkdv_kernel", w.name + "_backward")
    res = {"value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_call": ms, "roofline": rf,
           "launches_per_call": 3, "timing": timing,
           "config": dict(workload_config(w), workload=w.name + "_backward")}
    if cpu_budget > 0 and dist.rank == 0:
        import oracle
        from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs
        qh, kh, vh = prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
        dOh = dO.cpu()
        pairs = [(i % w.B, (i * 7) % w.Hq) for i in range(w.B * w.Hq)]

        def run(i):  # Hq == Hkv: one head's gradients need that head alone
            b, h = pairs[i]
            sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
            oracle.attention_backward(qh[sl], kh[sl], vh[sl], dOh[sl], causal=w.causal,
                                      window=w.window, scale=w.scale)
        res["cpu_baseline"] = cpu_baseline_heads(
            w.name + "_backward", flops / (w.B * w.Hq), run, len(pairs), cpu_budget,
            "dQ, dK, dV of whole heads, float64 NumPy")
    return res


def bench_fp8(w, steps, warmup, dist, peaks, peak_kind):
    """FP8 (e4m3) prefill of the workload: the attention kernel alone on
    operands quantised beforehand (as a model whose previous layer writes e4m3
    would hand them over), and the quantisation of bf16 Q, K, V separately.
    Roofline: the FP8 dense tensor peak, taken as the measured bf16 peak times
    the nominal FP8/BF16 ratio (4.5 / 2.25 PFLOP/s)."""
    import torch
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import prefill_flops
    q, k, v, o, lse = prefill_case(w, "cuda")
    qz = fa.attn_fp8_quantize(q, k, v)
    ws = torch.empty(fa.attn_fp8_workspace_size(w.B, w.Hkv, w.N), dtype=torch.uint8,
                     device="cuda")
    flops = prefill_flops(w.B, w.Hq, w.N, w.d, w.causal, w.window)

    def attn():
        fa.attn_fwd_fp8(qz, causal=w.causal, window=w.window, scale=w.scale, out=o, lse=lse)

    def quant():
        fa.attn_fp8_quantize(q, k, v, out=qz, workspace=ws)

    ms = time_launches(attn, steps, warmup, dist)
    timing = public_timing(LAST_TIMING)
    ms_q = time_launches(quant, steps, warmup, dist)
    assert fa.device_status() == 0, fa.last_error()
    tflops = flops / (ms * 1e-3) / 1e12
    peak = round(peaks["bf16_tflops"] * 2.0, 1)
    rf = roofline(tflops, peak, "TFLOP/s", "tensor",
                  stored_traffic("prefill_kernel", w.name + "_fp8"), flops, "FLOP")
    rf["peak_kind"] = f"{peak_kind} dense bf16 (burst) x 2, the nominal fp8/bf16 ratio"
    q_bytes = (q.numel() + k.numel() + v.numel()) * 3  # 2 bytes read + 1 byte written each
    return {"value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_call": ms, "roofline": rf,
            "dtype": "e4m3 operands, f32 accumulate", "launches_per_call": 1, "timing": timing,
            "quantize": {"ms_per_call": round(ms_q, 5), "launches_per_call": 2,
                         "gbs": round(q_bytes / (ms_q * 1e-3) / 1e9, 1),
                         "algorithmic_bytes": q_bytes},
            "tflops_including_quantize": round(flops / ((ms + ms_q) * 1e-3) / 1e12, 2),
            "config": dict(workload_config(w), workload=w.name + "_fp8")}


def prefill_extra(w, steps, warmup, dist, peaks, peak_kind, cpu_budget=0.0):
    """A prefill workload as a sub-object: TFLOP/s with its roofline, timing,
    and the oracle on whole heads of the same inputs (the band form for a
    non-causal window, whose masked keys carry exactly zero weight)."""
    r = bench_prefill(w, steps, warmup, dist, peaks, peak_kind)
    out = {"value": round(r["tflops"], 2), "unit": "TFLOP/s", "ms_per_call": r["ms"],
           "us_per_call": round(r["ms"] * 1e3, 2), "roofline": r["roofline"],
           "timing": r["timing"], "config": workload_config(w)}
    if cpu_budget > 0 and dist.rank == 0:
        import oracle
        from exact_transformer_attention_flashattention_b300.inputs import (prefill_flops,
                                                                            prefill_inputs)
        q, k, v = prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
        pairs = [(i % w.B, (i * 7) % w.Hq) for i in range(w.B * w.Hq)]
        per_head = prefill_flops(1, 1, w.N, w.d, w.causal, w.window)
        if w.window >= 0 and not w.causal:
            run = lambda i: oracle.attention_band(q, k, v, w.window, scale=w.scale,
                                                  heads=[pairs[i]])
            what = "band form over every query row, float64 NumPy"
        else:
            run = lambda i: oracle.attention_rows(q, k, v, *pairs[i], list(range(w.N)),
                                                  causal=w.causal, window=w.window,
                                                  scale=w.scale)
            what = "every query row, float64 NumPy"
        out["cpu_baseline"] = cpu_baseline_heads(w.name, per_head, run, len(pairs), cpu_budget,
                                                 what)
    return out


def bench_paged(w, steps, warmup, dist, peaks, peak_kind, page_size=256):
    """The prefill workload with K and V in a shuffled page pool (block table),
    as an inference server keeps its cache."""
    import torch
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import prefill_flops
    q, k, v, o, lse = prefill_case(w, "cuda")
    pps = (w.N + page_size - 1) // page_size
    P = w.B * pps
    perm = torch.randperm(P, generator=torch.Generator("cpu").manual_seed(w.seed + 7))
    table = perm.view(w.B, pps).to(torch.int32).cuda()
    k_pages = torch.empty(P, page_size, w.Hkv, w.d, dtype=torch.bfloat16, device="cuda")
    v_pages = torch.empty_like(k_pages)
    k_pages[table.long()] = k.view(w.B, pps, page_size, w.Hkv, w.d)
    v_pages[table.long()] = v.view(w.B, pps, page_size, w.Hkv, w.d)
    del k, v
    flops = prefill_flops(w.B, w.Hq, w.N, w.d, w.causal, w.window)

    def step():
        fa.attn_fwd_paged(q, k_pages, v_pages, table, causal=w.causal, window=w.window,
                          scale=w.scale, out=o, lse=lse)

    ms = time_launches(step, steps, warmup, dist)
    timing = public_timing(LAST_TIMING)
    assert fa.device_status() == 0, fa.last_error()
    tflops = flops / (ms * 1e-3) / 1e12
    rf = roofline(tflops, peaks["bf16_tflops"], "TFLOP/s", "tensor", None, flops, "FLOP")
    rf["peak_kind"] = f"{peak_kind} dense bf16 (burst)"
    return {"value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_call": ms, "roofline": rf,
            "launches_per_call": 1, "timing": timing,
            "config": dict(workload_config(w), workload=w.name + "_paged", page_size=page_size,
                           pages="shuffled pool, one block-table row per sequence")}


def bench_alternating(lw, steps, warmup, dist, peaks, peak_kind, cpu_budget=0.0):
    """A stack of layers alternating global and local attention (layer l global
    when l % 3 == 0), two calls per group of three layers."""
    import torch
    from exact_transformer_attention_flashattention_b300 import alternating
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import (layer_stack_inputs,
                                                                        prefill_flops)
    host = layer_stack_inputs(lw.L, lw.B, lw.Hq, lw.Hkv, lw.N, lw.d, lw.seed)
    q, k, v = (t.cuda() for t in host)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(lw.L, lw.B, lw.Hq, lw.N, dtype=torch.float32, device="cuda")
    groups = alternating.layer_groups(lw.L, lw.global_every)
    f_glob = prefill_flops(lw.B, lw.Hq, lw.N, lw.d, False, -1)
    f_loc = prefill_flops(lw.B, lw.Hq, lw.N, lw.d, False, lw.local_window)
    n_glob = len(groups)
    flops = n_glob * f_glob + (lw.L - n_glob) * f_loc

    def step():
        alternating.alternating_attention(q, k, v, lw.global_every, lw.local_window,
                                          scale=lw.scale, out=o, lse=lse)

    ms = time_launches(step, steps, warmup, dist)
    timing = public_timing(LAST_TIMING)
    assert fa.device_status() == 0, fa.last_error()
    tflops = flops / (ms * 1e-3) / 1e12
    rf = roofline(tflops, peaks["bf16_tflops"], "TFLOP/s", "tensor", None, flops, "FLOP")
    rf["peak_kind"] = f"{peak_kind} dense bf16 (burst)"
    out = {"value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_call": ms, "roofline": rf,
           "launches_per_call": 2 * n_glob - sum(1 for _, a, e in groups if e == a),
           "timing": timing,
           "config": {"workload": lw.name, "layers": lw.L, "B": lw.B, "Hq": lw.Hq, "Hkv": lw.Hkv,
                      "N": lw.N, "d": lw.d, "global_every": lw.global_every,
                      "local_window": f"|i-j| <= {lw.local_window}", "causal": False,
                      "scale": "1/sqrt(d)", "inputs": "bf16 i.i.d. N(0,1), seeded",
                      "l2": "inputs larger than L2; no flush"}}
    if cpu_budget > 0 and dist.rank == 0:
        import oracle
        qh, kh, vh = host
        G = lw.global_every

        def run(i):  # alternate a global head and a local head of the first group
            layer = 0 if i % 2 == 0 else 1
            b, h = (i // 2) % lw.B, (i // 2) % lw.Hq
            if layer == 0:
                oracle.attention_rows(qh[0], kh[0], vh[0], b, h, list(range(lw.N)),
                                      scale=lw.scale)
            else:
                oracle.attention_band(qh[1], kh[1], vh[1], lw.local_window, scale=lw.scale,
                                      heads=[(b, h)])
        per_pair = (prefill_flops(1, 1, lw.N, lw.d, False, -1) +
                    prefill_flops(1, 1, lw.N, lw.d, False, lw.local_window)) / 2
        out["cpu_baseline"] = cpu_baseline_heads(
            lw.name, per_pair, run, lw.L * lw.B * lw.Hq, cpu_budget,
            "global and local heads alternately (local in band form), float64 NumPy")
    return out


def decode_case(w, dev, host=None):
    import torch
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import decode_inputs
    if host is None:
        host = decode_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.kv_len_lo, w.kv_len_hi)
    q, kc, vc, kv_len = host
    ws = torch.empty(fa.attn_decode_workspace_size(w.B, w.Hq, w.num_splits, w.d),
                     dtype=torch.uint8, device=dev)
    o = torch.empty(w.B, w.Hq, w.d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.Hq, dtype=torch.float32, device=dev)
    return q.to(dev), kc.to(dev), vc.to(dev), kv_len, kv_len.to(dev), ws, o, lse


def bench_decode(w, steps, warmup, dist, peaks, peak_kind, clocks=None, cpu_budget=0.0):
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import (decode_inputs,
                                                                        decode_kv_bytes)
    host = decode_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.kv_len_lo, w.kv_len_hi)
    base = cpu_baseline_decode(w, cpu_budget, host) if cpu_budget > 0 and dist.rank == 0 else None
    q, kc, vc, kv_len_host, kv_len, ws, o, lse = decode_case(w, "cuda", host)
    del host
    kv_bytes = decode_kv_bytes(kv_len_host, w.Hkv, w.d)
    m, l, po = fa.split_partials_view(ws, w.B, w.Hq, w.num_splits, w.d)

    def full():
        fa.attn_decode_splitkv(q, kc, vc, kv_len, w.num_splits, scale=w.scale, out=o, lse=lse,
                               workspace=ws)

    def partials():
        fa.attn_decode_partials(q, kc, vc, kv_len, w.num_splits, scale=w.scale, workspace=ws)

    def combine():
        fa.lse_tree_combine(m, l, po, out=o, lse=lse)

    if clocks is not None:
        with clocks:
            ms_full = time_launches(full, steps, warmup, dist, clocks)
    else:
        ms_full = time_launches(full, steps, warmup, dist)
    timing = public_timing(LAST_TIMING)
    ms_part = time_launches(partials, steps, warmup, dist)
    ms_comb = time_launches(combine, steps, warmup, dist)
    assert fa.device_status() == 0, fa.last_error()
    gbs = kv_bytes / (ms_full * 1e-3) / 1e9
    part_gbs = kv_bytes / (ms_part * 1e-3) / 1e9
    rf = roofline(part_gbs, peaks["hbm_gbs"], "GB/s", "hbm",
                  stored_traffic("decode_partial_kernel", w.name), kv_bytes, "bytes of K/V")
    rf["kernel"] = "decode_partial_kernel"
    rf["peak_kind"] = f"{peak_kind} HBM copy"
    rf["frac_of_nameplate_8tbs"] = round(part_gbs / NAMEPLATE_HBM_GBS, 4)
    res = {"workload": w.name, "value": round(gbs, 1), "unit": "GB/s", "ms_per_call": ms_full,
           "kv_bytes": kv_bytes, "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4),
           "frac_of_nameplate_8tbs": round(gbs / NAMEPLATE_HBM_GBS, 4),
           "kernels": {"decode_partial_kernel_ms": ms_part,
                       "merge_ms_in_call": round(ms_full - ms_part, 5),
                       "lse_tree_combine_alone_ms": ms_comb},
           "launches_per_call": 2, "roofline": rf, "timing": timing,
           "config": decode_config(w)}
    if base is not None:
        res["cpu_baseline"] = base
    return res


def e2e_prefill(w, steps, dist):
    """Through the public API with host buffers: pinned host -> device copies
    of q, k, v, the prefill launch, device -> pinned host copies of O and LSE,
    every step.  Steps are pipelined as a serving loop would run them: two
    device buffer sets and three streams (input copies, the kernel, result
    copies), so that step i+1's inputs cross PCIe while step i computes and
    its result comes back (PCIe moves both directions at once).  The serial
    form (copy in, compute, copy out, then the next step) is reported
    beside it."""
    import torch
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import (prefill_flops,
                                                                        prefill_inputs)
    qh, kh, vh = (t.pin_memory() for t in prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed))
    oh = torch.empty(w.B, w.N, w.Hq, w.d, dtype=torch.bfloat16).pin_memory()
    lh = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32).pin_memory()
    sets = []
    for _ in range(2):
        qd, kd, vd = (torch.empty_like(t, device="cuda") for t in (qh, kh, vh))
        sets.append((qd, kd, vd, torch.empty_like(oh, device="cuda"),
                     torch.empty_like(lh, device="cuda")))
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = oh.numel() * 2 + lh.numel() * 4
    flops = prefill_flops(w.B, w.Hq, w.N, w.d, w.causal, w.window) * dist.world

    def step_serial():
        qd, kd, vd, od, ld = sets[0]
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        fa.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale, out=od, lse=ld)
        oh.copy_(od, non_blocking=True)
        lh.copy_(ld, non_blocking=True)

    ms_serial = time_launches(step_serial, steps, 2, dist)

    s_in, s_cmp, s_out = (torch.cuda.Stream() for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "cmp", "out")}

    def run(n):
        for i in range(n):
            bset = i % 2
            qd, kd, vd, od, ld = sets[bset]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev["cmp"][bset])  # the kernel of step i-2 has read this set
                qd.copy_(qh, non_blocking=True)
                kd.copy_(kh, non_blocking=True)
                vd.copy_(vh, non_blocking=True)
                ev["in"][bset].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev["in"][bset])
                if i >= 2:
                    s_cmp.wait_event(ev["out"][bset])  # step i-2's result has left this set
                fa.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale,
                            out=od, lse=ld, stream=s_cmp)
                ev["cmp"][bset].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["cmp"][bset])
                oh.copy_(od, non_blocking=True)
                lh.copy_(ld, non_blocking=True)
                ev["out"][bset].record(s_out)

    main = torch.cuda.current_stream()
    run(2)  # warm-up
    torch.cuda.synchronize()
    dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(main)
    for st in (s_in, s_cmp, s_out):
        st.wait_event(start)
    run(steps)
    for st in (s_in, s_cmp, s_out):
        main.wait_stream(st)
    end.record(main)
    torch.cuda.synchronize()
    ms = dist.max(start.elapsed_time(end) / steps)
    # the last result copied out is the last step's output
    assert torch.equal(oh, sets[(steps - 1) % 2][3].cpu()), "pipelined copies out of order"
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "mode": "pipelined: two device buffer sets, input copies / kernel / result copies "
                    "on three streams; every step copies its own inputs in and its result out",
            "serial": {"value": round(flops / (ms_serial * 1e-3) / 1e12, 2),
                       "ms_per_step": ms_serial}}


def e2e_decode(w, steps, dist):
    """Through the public API with host buffers.  The KV cache is state that a
    decoder keeps resident in HBM, so it is copied once, outside the timed
    region; every step copies q and kv_len from pinned host memory, runs the
    decode and copies O and LSE back."""
    import torch
    from exact_transformer_attention_flashattention_b300 import binding as fa
    from exact_transformer_attention_flashattention_b300.inputs import decode_kv_bytes
    q, kc, vc, kv_len_host, kv_len, ws, o, lse = decode_case(w, "cuda")
    qh = q.cpu().pin_memory()
    lh_in = kv_len_host.pin_memory()
    oh = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def step():
        q.copy_(qh, non_blocking=True)
        kv_len.copy_(lh_in, non_blocking=True)
        fa.attn_decode_splitkv(q, kc, vc, kv_len, w.num_splits, scale=w.scale, out=o, lse=lse,
                               workspace=ws)
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)

    ms = time_launches(step, steps, 2, dist)
    gbs = decode_kv_bytes(kv_len_host, w.Hkv, w.d) * dist.world / (ms * 1e-3) / 1e9
    return {"value": round(gbs, 1), "unit": "GB/s",
            "h2d_bytes_per_step": qh.numel() * 2 + lh_in.numel() * 4,
            "d2h_bytes_per_step": oh.numel() * 2 + lh.numel() * 4, "ms_per_step": ms,
            "note": "KV cache resident in HBM; q and kv_len copied in, O and LSE copied out"}


# ----------------------------------------------------------------- CPU oracle
def oracle_prefill_sample(w, rows_per_head: int, heads, inputs=None):
    """Time the float64 oracle on `heads` (b, h) pairs, `rows_per_head` query
    rows each (rows taken from the end, the most expensive causal rows).
    Returns (seconds, algorithmic flops of the sampled rows)."""
    import numpy as np
    import oracle
    from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs
    q, k, v = inputs if inputs is not None else prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    rows = np.arange(w.N - rows_per_head, w.N)
    vis = oracle.visible(w.N, w.N, w.causal, w.window)[rows]
    flops = 4.0 * w.d * float(vis.sum()) * len(heads)
    t0 = time.perf_counter()
    for b, h in heads:
        oracle.attention_rows(q, k, v, b, h, rows, causal=w.causal, window=w.window,
                              scale=w.scale)
    return time.perf_counter() - t0, flops


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else None
    except Exception:
        return None


def cpu_baseline(w, budget_s: float):
    """The oracle as it stands on the host cores: whole heads of the workload
    until about `budget_s` seconds of work."""
    from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs
    inputs = prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    heads, secs, flops = [], 0.0, 0.0
    i = 0
    while secs < budget_s and i < w.B * w.Hq:
        hd = [(i % w.B, (i * 7) % w.Hq)]
        s, f = oracle_prefill_sample(w, w.N, hd, inputs)
        secs, flops = secs + s, flops + f
        heads += hd
        i += 1
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s",
            "cores": blas_threads() or len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{len(heads)} of {w.B * w.Hq} (batch, head) pairs of {w.name}, all "
                      f"{w.N} query rows each, float64 NumPy ({secs:.1f} s)",
            "host_cores_available": len(os.sched_getaffinity(0))}


def cpu_baseline_decode(w, budget_s: float, inputs=None):
    """The oracle decode on whole (sequence, kv head) groups (every query head
    of the group) until about `budget_s` seconds of work; GB/s of K/V rows read."""
    import oracle
    from exact_transformer_attention_flashattention_b300.inputs import decode_inputs
    if inputs is None:
        inputs = decode_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.kv_len_lo, w.kv_len_hi)
    q, kc, vc, kv_len = inputs
    G = w.Hq // w.Hkv
    secs = nbytes = 0.0
    done = 0
    for b in range(w.B):
        for hk in range(w.Hkv):
            heads = [(b, hk * G + g) for g in range(G)]
            t0 = time.perf_counter()
            oracle.decode(q, kc, vc, kv_len, scale=w.scale, heads=heads)
            secs += time.perf_counter() - t0
            nbytes += int(kv_len[b]) * w.d * 2 * 2
            done += 1
            if secs >= budget_s:
                break
        if secs >= budget_s:
            break
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s",
            "cores": blas_threads() or len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{done} of {w.B * w.Hkv} (sequence, kv head) groups of {w.name}, every "
                      f"query head of the group, float64 NumPy ({secs:.1f} s)",
            "host_cores_available": len(os.sched_getaffinity(0))}


def cpu_baseline_heads(name, flops_per_head, run_head, n_heads, budget_s: float, what: str):
    """The oracle on whole (batch, head) pairs until about `budget_s` seconds;
    `run_head(i)` computes pair i, `flops_per_head` is its algorithmic work."""
    secs = flops = 0.0
    done = 0
    while done < n_heads and (done == 0 or secs < budget_s):
        t0 = time.perf_counter()
        run_head(done)
        secs += time.perf_counter() - t0
        flops += flops_per_head
        done += 1
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s",
            "cores": blas_threads() or len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{done} of {n_heads} (batch, head) pairs of {name}, {what} ({secs:.1f} s)",
            "host_cores_available": len(os.sched_getaffinity(0))}


def run_reference(args, w, dist):
    """--impl reference: the oracle timed on bounded samples of the workload."""
    if dist.rank != 0:
        return
    if w.kind == "decode":
        per = 150.0 / max(1, args.steps + args.warmup)
        r = cpu_baseline_decode(w, per)
        line = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": dict(decode_config(w), parallelism=parallelism(dist)),
                "cpu_baseline": r,
                "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    from exact_transformer_attention_flashattention_b300.inputs import prefill_inputs
    inputs = prefill_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed)
    budget = 150.0  # seconds for the whole --warmup + --steps run
    # calibrate the rows per step so that (W + K) steps fit the budget
    t, _ = oracle_prefill_sample(w, 256, [(0, 0)], inputs)
    per_row = t / 256
    rows = int(max(16, min(w.N, budget / max(1, args.steps + args.warmup) / per_row)))
    for i in range(args.warmup):
        oracle_prefill_sample(w, rows, [(i % w.B, i % w.Hq)], inputs)
    secs = flops = 0.0
    for i in range(args.steps):
        s, f = oracle_prefill_sample(w, rows, [(i % w.B, (3 * i) % w.Hq)], inputs)
        secs, flops = secs + s, flops + f
    value = flops / secs / 1e12
    cores = blas_threads() or len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(w), parallelism=parallelism(dist)),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle",
                             "sample": f"per step: the last {rows} query rows of one (batch, "
                                       f"head) pair of {w.name}, float64 NumPy"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def summary(line):
    """One compact entry per workload of the line (value, unit, roofline
    fraction, the oracle's CPU rate), printed last so that it survives in the
    tail of the output."""
    def entry(o):
        rf = o.get("roofline", {})
        e = {"value": o.get("value"), "unit": o.get("unit"), "frac": rf.get("frac"),
             "of": rf.get("unit")}
        if "us_per_call" in o:
            e["us"] = o["us_per_call"]
        if "frac_of_hbm_peak" in o:
            e["whole_call_frac"] = o["frac_of_hbm_peak"]
        if "cpu_baseline" in o:
            e["cpu"] = o["cpu_baseline"]["value"]
        return e
    out = {line["config"]["workload"]: entry(line)}
    if "timing" in line and "plain_launch_ms" in line["timing"]:
        out[line["config"]["workload"]]["plain_launch_ms"] = line["timing"]["plain_launch_ms"]
        out[line["config"]["workload"]]["ms"] = line["ms_per_step"]
    for name, o in line.get("extra", {}).items():
        out[name] = entry(o)
    return out


def workload_config(w):
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d,
           "causal": w.causal, "window": w.window, "scale": "1/sqrt(d)",
           "o_dtype": "f32" if w.o_fp32 else "bf16", "inputs": "bf16 i.i.d. N(0,1), seeded"}
    qkv = w.B * w.N * (w.Hq + 2 * w.Hkv) * w.d * 2
    cfg["l2"] = f"inputs larger than L2 ({qkv / 2**20:.0f} MiB of Q/K/V vs 126 MB); no flush"
    return cfg


def parallelism(dist):
    return f"replicas x{dist.world}" if dist.world > 1 else "single GPU"


def decode_config(w):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Lmax": w.N, "d": w.d,
            "num_splits": w.num_splits, "chunk": 512,
            "kv_len": ("uniform [%d, %d]" % (w.kv_len_lo, w.kv_len_hi)) if w.kv_len_lo else "full",
            "inputs": "bf16 i.i.d. N(0,1), seeded",
            "l2": "inputs larger than L2 (K/V cache far above 126 MB); no flush"}


def main():
    args = parse_args()
    from exact_transformer_attention_flashattention_b300.inputs import WORKLOADS
    w = WORKLOADS[args.workload] if args.workload in WORKLOADS else \
        profile_workloads()[args.workload]
    dist = Dist(args.gpus)
    if args.impl == "reference":
        run_reference(args, w, dist)
        dist.close()
        return

    import torch
    torch.cuda.set_device(dist.local)
    from exact_transformer_attention_flashattention_b300 import binding  # noqa: F401 (loads .so)
    peaks, peak_kind = load_peaks()
    if args.only:
        if args.only == "decode":
            res = bench_decode(w, args.steps, args.warmup, dist, peaks, peak_kind)
        elif args.only == "prefill":
            res = prefill_extra(w, args.steps, args.warmup, dist, peaks, peak_kind)
        else:
            leg = bench_backward if args.only == "backward" else bench_fp8
            res = leg(w, args.steps, args.warmup, dist, peaks, peak_kind)
        if dist.rank == 0:
            print(json.dumps(res), flush=True)
        dist.close()
        return
    clocks = ClockSampler(torch.cuda.current_device())
    if w.kind == "prefill":
        main_res = bench_prefill(w, args.steps, args.warmup, dist, peaks, peak_kind, clocks)
        value = whole_job_rate(main_res["flops"], dist.world, main_res["ms"], 1e12)
        unit, ms, cfg, rf = "TFLOP/s", main_res["ms"], workload_config(w), main_res["roofline"]
        launches = args.steps * main_res["launches_per_step"]
    else:
        main_res = bench_decode(w, args.steps, args.warmup, dist, peaks, peak_kind, clocks)
        value = whole_job_rate(main_res["kv_bytes"], dist.world, main_res["ms_per_call"], 1e9)
        unit, ms, cfg, rf = "GB/s", main_res["ms_per_call"], decode_config(w), main_res["roofline"]
        launches = args.steps * main_res["launches_per_call"]
        rf = dict(rf, note="dominant kernel of the step (the split partials); the step adds "
                           "the tree combine")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": cfg, "roofline": rf, "gpu_launches": launches,
        "clocks": clocks.summary(),
    }
    if w.kind == "decode":
        line["kernels"] = main_res["kernels"]
    if "timing" in main_res:
        line["timing"] = main_res["timing"]
    line["config"]["parallelism"] = parallelism(dist)
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 10))
        line["e2e"] = e2e_prefill(w, e2e_steps, dist) if w.kind == "prefill" else \
            e2e_decode(w, e2e_steps, dist)
    if dist.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_budget) if w.kind == "prefill" else \
            cpu_baseline_decode(w, args.cpu_budget)
    if not args.no_extra:
        from exact_transformer_attention_flashattention_b300.inputs import LAYER_WORKLOADS
        budget = 0.0 if args.no_cpu_baseline else args.extra_cpu_budget
        n_ex, w_ex = max(3, min(args.steps, 100)), max(3, args.warmup)
        extra = {}
        # prefill legs first; the decode legs go last in the line
        for name in ("tiny_noncausal", "window_encoder_8k", "causal_prefill_4k"):
            if name != w.name:
                extra[name] = prefill_extra(WORKLOADS[name], n_ex, w_ex, dist, peaks, peak_kind,
                                            budget)
        if w.name == "causal_prefill_4k":
            extra["causal_prefill_4k_backward"] = bench_backward(
                w, max(3, min(args.steps, 50)), w_ex, dist, peaks, peak_kind, budget)
            extra["causal_prefill_4k_fp8"] = bench_fp8(w, n_ex, w_ex, dist, peaks, peak_kind)
            extra["causal_prefill_4k_paged"] = bench_paged(w, n_ex, w_ex, dist, peaks, peak_kind)
        lw = LAYER_WORKLOADS["modernbert_alternating_8k"]
        extra[lw.name] = bench_alternating(lw, max(3, min(args.steps, 30)), w_ex, dist, peaks,
                                           peak_kind, budget)
        for name in ("gqa_decode_batch32", "decode_1m"):
            if name != w.name:
                extra[name] = bench_decode(WORKLOADS[name], max(3, min(args.steps, 50)), w_ex,
                                           dist, peaks, peak_kind, cpu_budget=budget)
        line["extra"] = extra
        line["summary"] = summary(line)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


if __name__ == "__main__":
    main()
