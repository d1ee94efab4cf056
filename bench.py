"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--exp2-emu16 E] [--tau T] [--p-scaling 0|1|2]

A step is one attention forward (O and LSE) over the whole workload, inputs
resident in HBM (Q, K, V together exceed the 129 MB L2, so no flush is
needed). Prints one JSON line on rank 0. Under torchrun each rank runs the
same workload on its own GPU (weak scaling, no data-path collective); the
timed region is bracketed by a barrier and a device synchronisation and the
slowest rank's time is reported.

``--impl reference`` times the float64 CPU oracle instead, on a bounded sample
of the same workload per step (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import attn_inputs as I  # noqa: E402

METRIC = "attention fwd TFLOP/s on 1xGB300 and fraction of dense BF16/FP8 peak"
METRIC_BWD = "attention bwd TFLOP/s on 1xGB300 and fraction of dense BF16/FP8 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = I.NONCAUSAL_D128.name
L2_BYTES = 129 * 1024 * 1024
# sources each kernel is compiled from (a profile's traffic figure is only
# reported while these are unchanged)
KERNEL_SOURCES = {
    "bf16": ["online_softmax_fwd_gb300/csrc/fwd_bf16.cuh", "online_softmax_fwd_gb300/csrc/ptx.cuh",
             "online_softmax_fwd_gb300/csrc/exp2_fma.cuh", "online_softmax_fwd_gb300/csrc/schedule.h",
             "online_softmax_fwd_gb300/csrc/schedule.cu", "online_softmax_fwd_gb300/csrc/kernel_setup.h"],
    "bf16_2cta": ["online_softmax_fwd_gb300/csrc/fwd_bf16_2cta.cuh", "online_softmax_fwd_gb300/csrc/fwd_bf16.cuh",
                  "online_softmax_fwd_gb300/csrc/ptx.cuh", "online_softmax_fwd_gb300/csrc/schedule.h",
                  "online_softmax_fwd_gb300/csrc/schedule.cu", "online_softmax_fwd_gb300/csrc/kernel_setup.h"],
    "mxfp8": ["online_softmax_fwd_gb300/csrc/fwd_mxfp8.cuh", "online_softmax_fwd_gb300/csrc/mxfp8_common.cuh",
              "online_softmax_fwd_gb300/csrc/kernel_setup.h",
              "online_softmax_fwd_gb300/csrc/fwd_bf16.cuh", "online_softmax_fwd_gb300/csrc/ptx.cuh",
              "online_softmax_fwd_gb300/csrc/exp2_fma.cuh", "online_softmax_fwd_gb300/csrc/schedule.h",
              "online_softmax_fwd_gb300/csrc/schedule.cu"],
    "combine": ["online_softmax_fwd_gb300/csrc/combine.cu", "online_softmax_fwd_gb300/csrc/ptx.cuh"],
    "bwd": ["online_softmax_fwd_gb300/csrc/bwd_bf16.cuh", "online_softmax_fwd_gb300/csrc/bwd_common.cuh",
            "online_softmax_fwd_gb300/csrc/kernel_setup.h",
            "online_softmax_fwd_gb300/csrc/bwd_aux.cu",
            "online_softmax_fwd_gb300/csrc/fwd_bf16.cuh", "online_softmax_fwd_gb300/csrc/ptx.cuh",
            "online_softmax_fwd_gb300/csrc/exp2_fma.cuh", "online_softmax_fwd_gb300/csrc/schedule.h"],
    "bwd_mxfp8": ["online_softmax_fwd_gb300/csrc/bwd_mxfp8.cuh", "online_softmax_fwd_gb300/csrc/bwd_common.cuh",
                  "online_softmax_fwd_gb300/csrc/kernel_setup.h",
                  "online_softmax_fwd_gb300/csrc/bwd_aux.cu", "online_softmax_fwd_gb300/csrc/mxfp8_common.cuh",
                  "online_softmax_fwd_gb300/csrc/quant_mxfp8.cu", "online_softmax_fwd_gb300/csrc/fwd_bf16.cuh",
                  "online_softmax_fwd_gb300/csrc/ptx.cuh"],
}


# what the roofline's achieved figure times (CUDA events around that call)
KERNEL_NAMES = {("fwd", "bf16"): "attn_fwd_bf16_kernel", ("fwd", "mxfp8"): "attn_fwd_mxfp8_kernel",
                ("bwd", "bf16"): "attn_bwd (bwd_prep + attn_bwd_bf16_kernel + bwd_post)",
                ("bwd", "mxfp8"): "attn_bwd_mxfp8 (bwd_prep_mxfp8 + attn_bwd_mxfp8_kernel + bwd_post)"}


def kernel_sources_sha(kind: str = "bf16") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


def oracle_threads() -> tuple[int, str]:
    """Threads the float64 oracle really runs on: NumPy's BLAS pool (the
    oracle's work is NumPy matrix products), not PyTorch's intra-op pool."""
    try:
        import threadpoolctl
        for info in threadpoolctl.threadpool_info():
            if info.get("user_api") == "blas":
                return int(info["num_threads"]), f"threadpoolctl ({info.get('internal_api')})"
    except Exception:
        pass
    try:
        libs = set()
        with open("/proc/self/maps") as f:
            for line in f:
                path = line.split()[-1]
                base = os.path.basename(path).lower()
                if "blas" in base and ".so" in base:
                    libs.add(path)
        for path in sorted(libs):
            lib = ctypes.CDLL(path)
            for name in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                         "openblas_get_num_threads64_", "openblas_get_num_threads"):
                fn = getattr(lib, name, None)
                if fn is not None:
                    fn.restype = ctypes.c_int
                    return int(fn()), f"{name} ({os.path.basename(path)})"
    except Exception:
        pass
    return os.cpu_count() or 1, "os.cpu_count (BLAS pool not found)"


def profiled_traffic(workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources (else None)."""
    prof = os.path.join(ROOT, "profiles")
    text = None
    for f in sorted(os.listdir(prof) if os.path.isdir(prof) else []):
        if f.endswith(".md"):
            t = open(os.path.join(prof, f)).read()
            m = re.search(r"^workload:\s*(\S+)\s*$", t, flags=re.M)
            if m and m.group(1) == workload:
                text = t
                break
    if text is None:
        return None
    sha = re.search(r"kernel_sources_sha:\s*([0-9a-f]+)", text)
    kind = re.search(r"kernel_kind:\s*(\w+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not sha or not val or not kind or kind.group(1) not in KERNEL_SOURCES:
        return None
    if sha.group(1) != kernel_sources_sha(kind.group(1)):
        return None
    return float(val.group(1))


class ClockSampler:
    """SM clock, power and clock-event reasons sampled DURING the timed region.

    Reads NVML through ctypes (about every millisecond, so even a short timed
    region gets samples); falls back to ``nvidia-smi -lms 200`` when NVML
    cannot be loaded. Only reads; changes no GPU setting."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: torch.device):
        self.samples: list[tuple[float, float, float, int]] = []  # (t, sm MHz, W, reasons)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nv = None
        self._h = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self._uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self._uuid = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            h = ctypes.c_void_p()
            if not self._uuid or nv.nvmlDeviceGetHandleByUUID(self._uuid.encode(), ctypes.byref(h)) != 0:
                raise OSError("handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._nv, self._h, self.source = nv, h, "nvml"
        except (OSError, AttributeError):
            self.source = "nvidia-smi"

    def _nvml_loop(self):
        mhz, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            ok = self._nv.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(mhz)) == 0
            self._nv.nvmlDeviceGetPowerUsage(self._h, ctypes.byref(mw))
            self._reason_fn(self._h, ctypes.byref(rs))
            if ok:
                self.samples.append((time.time(), float(mhz.value), mw.value / 1000.0, int(rs.value)))
            time.sleep(0.001)

    def _smi_loop(self):
        fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")
        target = ["-i", self._uuid] if self._uuid else []
        try:
            self._proc = subprocess.Popen(["nvidia-smi", *target, f"--query-gpu={fields}",
                                           "--format=csv,noheader,nounits", "-lms", "200"],
                                          stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        for line in self._proc.stdout:
            f = [x.strip() for x in line.split(",")]
            try:
                self.max_mhz = float(f[1])
                self.samples.append((time.time(), float(f[0]), float(f[2]), int(f[3], 16)))
            except (ValueError, IndexError):
                pass

    def start(self):
        loop = self._nvml_loop if self.source == "nvml" else self._smi_loop
        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed_region"
        if not inside:
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest_samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no_samples"], "source": self.source}
        reasons = sorted({name for s in inside for bit, name in self.REASONS.items() if s[3] & bit})
        return {"sm_mhz": float(np.median([s[1] for s in inside])), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(s[1] for s in inside), "power_w_max": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": window, "source": self.source}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(w: I.Workload, q, k, v, seconds: float, rows_per_call: int = 512) -> dict:
    """Time the float64 oracle on consecutive row chunks of the workload's
    first heads until `seconds` have passed (at least one chunk). Returns the
    sample description and its rate in the metric's units (useful FLOP of the
    computed rows, causal rows counting only their allowed keys)."""
    from oracle.attention import attention_rows
    if w.dtype == "mxfp8":
        from oracle.mxfp8 import quantize_blocks
        prep = lambda t: quantize_blocks(I.as_f64(t))[2]
    else:
        prep = I.as_f64
    t0 = time.perf_counter()
    flops = 0.0
    rows_done = 0
    heads = 0
    for b in range(w.B):
        for h in range(w.H):
            kk, vv = prep(k[b, h]), prep(v[b, h])
            qq = prep(q[b, h])
            for r0 in range(0, w.N, rows_per_call):
                r1 = min(w.N, r0 + rows_per_call)
                idx = np.arange(r0, r1)
                attention_rows(qq[r0:r1], kk, vv, idx, w.causal, w.scale)
                keys = (idx + 1).sum() if w.causal else (r1 - r0) * w.N
                flops += 4.0 * keys * w.d
                rows_done += r1 - r0
                if time.perf_counter() - t0 >= seconds:
                    break
            heads += 1
            if time.perf_counter() - t0 >= seconds:
                break
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "seconds": dt, "rows": rows_done, "heads_touched": heads,
            "flop": flops}


def oracle_bwd_sample(w: I.Workload, q, k, v, o, do, lse, seconds: float) -> dict:
    """Time the float64 backward oracle on whole heads of the workload (at
    least one) until `seconds` have passed; useful FLOP as the metric counts
    them (10 N^2 d per head, halved for causal). MXFP8 workloads time the
    MXFP8 backward oracle on the fp32 inputs (it quantises them itself)."""
    from oracle.backward import attention_bwd_head, attention_bwd_mxfp8_head
    bwd = attention_bwd_mxfp8_head if w.dtype == "mxfp8" else attention_bwd_head
    t0 = time.perf_counter()
    heads = 0
    for b in range(w.B):
        for h in range(w.H):
            bwd(I.as_f64(q[b, h]), I.as_f64(k[b, h]), I.as_f64(v[b, h]), I.as_f64(o[b, h]),
                I.as_f64(do[b, h]), lse[b, h].double().numpy(), w.causal, w.scale)
            heads += 1
            if time.perf_counter() - t0 >= seconds:
                break
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    flops = w.flops / (w.B * w.H) * heads
    return {"value": flops / dt / 1e12, "seconds": dt, "heads_touched": heads, "flop": flops}


def bench_reference_bwd(args, w: I.Workload) -> None:
    """The reference arm of a backward workload: the float64 backward oracle on
    the workload's first head, its O and LSE from the float64 forward oracle
    (computed once, outside the timed steps)."""
    from oracle.attention import attention_fwd
    from oracle.backward import attention_bwd_head, attention_bwd_mxfp8_head
    if w.dtype == "mxfp8":
        # fp32 draws of the first head; O and LSE from the float64 forward of
        # their dequantised MXFP8 form
        from oracle.mxfp8 import quantize_blocks
        xs = I.draw_fp32(w.B, w.H, w.N, w.d, w.qk_std, w.v_std, w.seed)
        qq, kk, vv = (x[0, 0].astype(np.float64) for x in xs)
        dd = I.draw_grad(w.B, w.H, w.N, w.d, seed=w.seed + 1)[0, 0].astype(np.float64)
        qf, kf, vf = (quantize_blocks(x)[2] for x in (qq, kk, vv))
        bwd = attention_bwd_mxfp8_head
    else:
        q, k, v = (t[:1, :1] for t in I.bf16_qkv(w))
        do = I.to_bf16(I.draw_grad(w.B, w.H, w.N, w.d, seed=w.seed + 1)[:1, :1])
        qq, kk, vv, dd = (I.as_f64(t)[0, 0] for t in (q, k, v, do))
        qf, kf, vf = qq, kk, vv
        bwd = attention_bwd_head
    o, lse = attention_fwd(qf[None, None], kf[None, None], vf[None, None], w.causal, w.scale)
    o = I.as_f64(torch.from_numpy(o).to(torch.bfloat16))[0, 0]
    lse = lse.astype(np.float32).astype(np.float64)[0, 0]
    head_flop = w.flops / (w.B * w.H)

    def one_step():
        t0 = time.perf_counter()
        bwd(qq, kk, vv, o, dd, lse, w.causal, w.scale)
        return time.perf_counter() - t0
    for _ in range(args.warmup):
        one_step()
    secs = [one_step() for _ in range(args.steps)]
    value = head_flop / float(np.mean(secs)) / 1e12
    cores, cores_src = oracle_threads()
    sample = (f"float64 {'MXFP8 ' if w.dtype == 'mxfp8' else ''}backward oracle on one whole head "
              f"(N = {w.N}, d = {w.d}) of the workload per step")
    out = {"impl": "reference", "metric": METRIC_BWD, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(secs)), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {**w.describe(), "workload": w.name},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "cores_source": cores_src, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def bench_reference(args, w: I.Workload, world: int, rank: int) -> None:
    if rank != 0:
        return
    if w.direction == "bwd":
        bench_reference_bwd(args, w)
        return
    q, k, v = I.bf16_qkv(w) if w.dtype == "bf16" else tuple(torch.from_numpy(x) for x in I.draw_fp32(
        w.B, w.H, w.N, w.d, w.qk_std, w.v_std, w.seed))
    cores, cores_src = oracle_threads()
    per_step = max(1.0, args.reference_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, per_step)
    vals, secs = [], []
    for _ in range(args.steps):
        s = oracle_sample(w, q, k, v, per_step)
        vals.append(s["value"])
        secs.append(s["seconds"])
    value = float(np.mean(vals))
    sample = (f"float64 one-shot oracle on the first {s['rows']} query rows (512-row chunks, all {w.N} keys) "
              f"of the workload per step, ~{per_step:.0f} s per step")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(secs)), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {**w.describe(), "workload": w.name},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "cores_source": cores_src, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


class Bf16Step:
    """One pass of the bf16 path: attn_fwd over the resident inputs."""

    launches = 1

    def __init__(self, attn, w, dev, args):
        self.attn, self.w, self.args = attn, w, args
        self.q_h, self.k_h, self.v_h = I.bf16_qkv(w)
        self.q, self.k, self.v = (t.to(dev) for t in (self.q_h, self.k_h, self.v_h))
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        self.ptrs = tuple(t.data_ptr() for t in (self.q, self.k, self.v, self.o, self.lse))

    def run(self, sh, ev=None):
        w = self.w
        if ev:
            ev[0].record()
        if getattr(self.args, "two_cta", False):
            st = self.attn.lib().attn_fwd_2cta(*self.ptrs, w.B, w.H, w.N, w.d, int(w.causal), float(w.scale), sh)
        else:
            st = self.attn.attn_fwd_raw(*self.ptrs, w.B, w.H, w.N, w.d, int(w.causal), float(w.scale), sh,
                                        tau=self.args.tau, exp2_emu16=self.args.exp2_emu16)
        if ev:
            ev[1].record()
        if st != 0:
            raise self.attn.AttnError(st, "attn_fwd")

    def input_bytes(self):
        return 3 * self.q.numel() * 2

    def e2e(self, dev, n_steps, world):
        w = self.w
        qp, kp, vp = (t.pin_memory() for t in (self.q_h, self.k_h, self.v_h))
        o_host = torch.empty_like(qp).pin_memory()
        lse_host = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
        ws = {}
        call = lambda: self.attn.attn_fwd_from_host(qp, kp, vp, w.causal, w.scale, device=dev, o_host=o_host,
                                                    lse_host=lse_host, workspace=ws)
        for _ in range(2):
            call()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_steps):
            call()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        return {"value": w.flops * n_steps * world / dt / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": 3 * qp.numel() * 2, "d2h_bytes_per_step": o_host.numel() * 2 + lse_host.numel() * 4,
                "steps": n_steps}


class Mxfp8Step:
    """One pass of the MXFP8 path: quantise Q, K, V (fp32 resident in HBM) to
    E4M3 + E8M0 and run the block-scaled attention."""

    launches = 4

    def __init__(self, attn, w, dev, args):
        self.attn, self.w, self.args = attn, w, args
        self.xq_h, self.xk_h, self.xv_h = (torch.from_numpy(x) for x in I.draw_fp32(
            w.B, w.H, w.N, w.d, w.qk_std, w.v_std, w.seed))
        self.x = [t.to(dev) for t in (self.xq_h, self.xk_h, self.xv_h)]
        nsf = attn.mxfp8_scale_bytes(w.B, w.H, w.N, w.d)
        self.codes = [torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in self.x]
        self.sf = [torch.empty(nsf, dtype=torch.uint8, device=dev) for _ in self.x]
        self.o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        self.tau = 0.0 if args.tau_given is None else args.tau

    def run(self, sh, ev=None):
        w, L = self.w, self.attn.lib()
        for i, role in enumerate((0, 0, 1)):
            st = L.attn_mxfp8_quantize(self.x[i].data_ptr(), self.codes[i].data_ptr(), self.sf[i].data_ptr(),
                                       w.B, w.H, w.N, w.d, role, sh)
            if st != 0:
                raise self.attn.AttnError(st, "attn_mxfp8_quantize")
        if ev:
            ev[0].record()
        if getattr(self.args, "unroll_kv", False):
            st = L.attn_fwd_mxfp8_unroll_kv(self.codes[0].data_ptr(), self.sf[0].data_ptr(),
                                            self.codes[1].data_ptr(), self.sf[1].data_ptr(),
                                            self.codes[2].data_ptr(), self.sf[2].data_ptr(), self.o.data_ptr(),
                                            self.lse.data_ptr(), w.B, w.H, w.N, w.d, int(w.causal),
                                            float(w.scale), sh)
        else:
            st = L.attn_fwd_mxfp8_ex(self.codes[0].data_ptr(), self.sf[0].data_ptr(), self.codes[1].data_ptr(),
                                     self.sf[1].data_ptr(), self.codes[2].data_ptr(), self.sf[2].data_ptr(),
                                     self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H, w.N, w.d, int(w.causal),
                                     float(w.scale), float(self.tau), int(self.args.exp2_emu16),
                                     int(self.args.p_scaling), sh)
        if ev:
            ev[1].record()
        if st != 0:
            raise self.attn.AttnError(st, "attn_fwd_mxfp8")

    def input_bytes(self):
        return 3 * self.x[0].numel() * 4

    def e2e(self, dev, n_steps, world):
        w = self.w
        hp = [t.pin_memory() for t in (self.xq_h, self.xk_h, self.xv_h)]
        o_host = torch.empty(self.o.shape, dtype=torch.bfloat16).pin_memory()
        lse_host = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        sh = torch.cuda.current_stream(dev).cuda_stream

        def call():
            for d_, h_ in zip(self.x, hp):
                d_.copy_(h_, non_blocking=True)
            self.run(sh)
            o_host.copy_(self.o, non_blocking=True)
            lse_host.copy_(self.lse, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
        for _ in range(2):
            call()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_steps):
            call()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        return {"value": w.flops * n_steps * world / dt / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": sum(h.numel() * 4 for h in hp),
                "d2h_bytes_per_step": o_host.numel() * 2 + lse_host.numel() * 4, "steps": n_steps}


class BwdStep:
    """One backward pass: attn_bwd (preparation, main kernel, dQ conversion)
    over resident Q, K, V, O, dO, LSE; O and LSE come from attn_fwd once,
    before the timed region."""

    launches = 3

    def __init__(self, attn, w, dev, args):
        self.attn, self.w, self.args = attn, w, args
        self.tau = args.tau
        self.q_h, self.k_h, self.v_h = I.bf16_qkv(w)
        self.do_h = I.to_bf16(I.draw_grad(w.B, w.H, w.N, w.d, seed=w.seed + 1))
        self.q, self.k, self.v, self.do = (t.to(dev) for t in (self.q_h, self.k_h, self.v_h, self.do_h))
        self.o, self.lse = attn.attn_fwd(self.q, self.k, self.v, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize(dev)
        self.o_h, self.lse_h = self.o.cpu(), self.lse.cpu()
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        self.ws_bytes = attn.lib().attn_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.ptrs = tuple(t.data_ptr() for t in (self.q, self.k, self.v, self.o, self.do, self.lse, self.dq, self.dk,
                                                 self.dv))

    def run(self, sh, ev=None):
        w = self.w
        if ev:
            ev[0].record()
        st = self.attn.lib().attn_bwd(*self.ptrs, w.B, w.H, w.N, w.d, int(w.causal), float(w.scale),
                                      self.ws.data_ptr(), self.ws_bytes, sh)
        if ev:
            ev[1].record()
        if st != 0:
            raise self.attn.AttnError(st, "attn_bwd")

    def input_bytes(self):
        return 5 * self.q.numel() * 2

    def e2e(self, dev, n_steps, world):
        w = self.w
        src = [t.pin_memory() for t in (self.q_h, self.k_h, self.v_h, self.o_h, self.do_h, self.lse_h)]
        dst = [self.q, self.k, self.v, self.o, self.do, self.lse]
        outs = [torch.empty(self.dq.shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
        sh = torch.cuda.current_stream(dev).cuda_stream

        def call():
            for d_, h_ in zip(dst, src):
                d_.copy_(h_, non_blocking=True)
            self.run(sh)
            for h_, d_ in zip(outs, (self.dq, self.dk, self.dv)):
                h_.copy_(d_, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
        for _ in range(2):
            call()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_steps):
            call()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        return {"value": w.flops * n_steps * world / dt / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in src),
                "d2h_bytes_per_step": sum(h.numel() * 2 for h in outs), "steps": n_steps}


class BwdMxfp8Step:
    """One MXFP8 backward pass: quantise Q, K, dO (both scale layouts) and V
    (fp32, resident in HBM) to E4M3 + E8M0, then attn_bwd_mxfp8 (preparation,
    main kernel, dQ conversion). O and LSE come from the MXFP8 forward once,
    before the timed region."""

    launches = 7

    def __init__(self, attn, w, dev, args):
        self.attn, self.w, self.args = attn, w, args
        self.tau = 0.0
        L = attn.lib()
        self.xq_h, self.xk_h, self.xv_h = (torch.from_numpy(x) for x in I.draw_fp32(
            w.B, w.H, w.N, w.d, w.qk_std, w.v_std, w.seed))
        self.do_h = torch.from_numpy(I.draw_grad(w.B, w.H, w.N, w.d, seed=w.seed + 1))
        self.x = [t.to(dev) for t in (self.xq_h, self.xk_h, self.xv_h, self.do_h)]
        nsf = attn.mxfp8_scale_bytes(w.B, w.H, w.N, w.d)
        self.roles = (2, 2, 0, 2)
        self.codes = [torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in self.x]
        self.sf = [torch.empty((2 if r == 2 else 1) * nsf, dtype=torch.uint8, device=dev) for r in self.roles]
        # the forward's O and LSE (its own quantisation: Q, K role 0, V role 1)
        q8, q_sf = attn.mxfp8_quantize(self.x[0], role=0)
        k8, k_sf = attn.mxfp8_quantize(self.x[1], role=0)
        v8, v_sf = attn.mxfp8_quantize(self.x[2], role=1)
        self.o, self.lse = attn.attn_fwd_mxfp8(q8, q_sf, k8, k_sf, v8, v_sf, causal=w.causal, scale=w.scale)
        torch.cuda.synchronize(dev)
        del q8, q_sf, k8, k_sf, v8, v_sf
        self.o_h, self.lse_h = self.o.cpu(), self.lse.cpu()
        self.dq, self.dk, self.dv = (torch.empty(self.o.shape, dtype=torch.bfloat16, device=dev) for _ in range(3))
        self.ws_bytes = L.attn_bwd_workspace_bytes(w.B, w.H, w.N, w.d)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        c, f = self.codes, self.sf
        self.ptrs = tuple(t.data_ptr() for t in (c[0], f[0], c[1], f[1], c[2], f[2], self.o, c[3], f[3], self.lse,
                                                 self.dq, self.dk, self.dv))

    def run(self, sh, ev=None):
        w, L = self.w, self.attn.lib()
        for i, role in enumerate(self.roles):
            st = L.attn_mxfp8_quantize(self.x[i].data_ptr(), self.codes[i].data_ptr(), self.sf[i].data_ptr(),
                                       w.B, w.H, w.N, w.d, role, sh)
            if st != 0:
                raise self.attn.AttnError(st, "attn_mxfp8_quantize")
        if ev:
            ev[0].record()
        st = L.attn_bwd_mxfp8(*self.ptrs, w.B, w.H, w.N, w.d, int(w.causal), float(w.scale), self.ws.data_ptr(),
                              self.ws_bytes, sh)
        if ev:
            ev[1].record()
        if st != 0:
            raise self.attn.AttnError(st, "attn_bwd_mxfp8")

    def input_bytes(self):
        return 4 * self.x[0].numel() * 4 + self.o.numel() * 2

    def e2e(self, dev, n_steps, world):
        w = self.w
        src = [t.pin_memory() for t in (self.xq_h, self.xk_h, self.xv_h, self.do_h, self.o_h, self.lse_h)]
        dst = [*self.x, self.o, self.lse]
        outs = [torch.empty(self.dq.shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
        sh = torch.cuda.current_stream(dev).cuda_stream

        def call():
            for d_, h_ in zip(dst, src):
                d_.copy_(h_, non_blocking=True)
            self.run(sh)
            for h_, d_ in zip(outs, (self.dq, self.dk, self.dv)):
                h_.copy_(d_, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
        for _ in range(2):
            call()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_steps):
            call()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        return {"value": w.flops * n_steps * world / dt / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in src),
                "d2h_bytes_per_step": sum(h.numel() * 2 for h in outs), "steps": n_steps}


class CombineStep:
    """One merge (attn_combine) of `parts` partial results of a workload's
    shape, inputs resident in HBM: O parts bf16 [P,B,H,N,d] and LSE parts fp32
    [P,B,H,N], drawn on the device (N(0,1), the workload's seed)."""

    launches = 1

    def __init__(self, attn, w, dev, parts):
        self.attn, self.w, self.parts = attn, w, parts
        g = torch.Generator(device=dev).manual_seed(w.seed)
        self.o_parts = torch.randn((parts, w.B, w.H, w.N, w.d), generator=g, device=dev).to(torch.bfloat16)
        self.lse_parts = torch.randn((parts, w.B, w.H, w.N), generator=g, device=dev)
        self.o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

    def run(self, sh, ev=None):
        w = self.w
        if ev:
            ev[0].record()
        st = self.attn.lib().attn_combine(self.o_parts.data_ptr(), self.lse_parts.data_ptr(), self.parts,
                                          self.o.data_ptr(), self.lse.data_ptr(), w.B, w.H, w.N, w.d, sh)
        if ev:
            ev[1].record()
        if st != 0:
            raise self.attn.AttnError(st, "attn_combine")

    def bytes_per_launch(self):
        """Algorithmic bytes: every part's O row and LSE in, the merged ones out."""
        rows = self.w.B * self.w.H * self.w.N
        return (self.parts + 1) * rows * (2 * self.w.d + 4)

    def input_bytes(self):
        return self.o_parts.numel() * 2 + self.lse_parts.numel() * 4


def combine_name(w: I.Workload, parts: int) -> str:
    return f"combine_p{parts}_b{w.B}h{w.H}n{w.N}d{w.d}"


def combine_record(attn, w: I.Workload, parts: int, dev, world: int, steps: int, warmup: int) -> dict:
    """The merge of `parts` partial results of w's shape, timed like the
    attention steps; bandwidth against the measured HBM copy rate."""
    step = CombineStep(attn, w, dev, parts)
    flush = None
    l2_note = f"inputs larger than L2 ({step.input_bytes() / 2**20:.0f} MiB > 129 MB)"
    if step.input_bytes() <= L2_BYTES:
        scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        flush = scratch.zero_
        l2_note = "inputs fit in L2: a 258 MB buffer is written between steps; value uses the per-launch events"
    m = measure(step, dev, world, steps, warmup, flush)
    launch_mean = float(np.mean(m["launch_ms"]))
    nbytes = step.bytes_per_launch()
    hbm = measured_peaks().get("hbm_gbs")
    src = "measured hbm_gbs (copy)" if hbm else "fallback 6800 GB/s"
    hbm = hbm or 6800.0
    achieved = nbytes / (launch_mean * 1e-3) / 1e9
    name = combine_name(w, parts)
    rec = {"config": {"workload": name, "parts": parts, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                      "pass": "combine", "l2": l2_note},
           "steps": steps, "warmup": warmup,
           "value": nbytes * steps * world / (m["region_ms"] * 1e-3) / 1e9 if flush is None
           else nbytes * world / (launch_mean * 1e-3) / 1e9,
           "unit": "GB/s", "ms_per_step": m["region_ms"] / steps if flush is None else launch_mean,
           "kernel_ms": kernel_ms_of(m["launch_ms"]),
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                        "traffic": profiled_traffic(name), "peak_source": src, "bytes_per_launch": nbytes,
                        "kernel": "attn_combine_kernel"},
           "clocks": m["clocks"], "gpu_launches": steps * step.launches}
    del step
    torch.cuda.empty_cache()
    return rec


def step_class(w: I.Workload):
    if w.direction == "bwd":
        return BwdMxfp8Step if w.dtype == "mxfp8" else BwdStep
    return Mxfp8Step if w.dtype == "mxfp8" else Bf16Step


def measure(step, dev, world: int, steps: int, warmup: int, flush=None) -> dict:
    """Warm up, then time `steps` steps on the current stream: CUDA events
    around the whole region and around each step's timed kernel call, clocks
    sampled during the region, barrier + device synchronisation on both sides
    and the slowest rank's region time. ``flush`` (optional) runs between
    steps, inside the region, to evict L2 when the inputs fit in it; the
    per-launch events then still time the kernel alone."""
    import online_softmax_fwd_gb300 as attn
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    for _ in range(warmup):
        step.run(sh)
        if flush:
            flush()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(dev)
    barrier(world)
    sampler.start()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    region0.record(stream)
    for i in range(steps):
        if flush:
            flush()
        step.run(sh, evs[i])
    region1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_wall1 = time.time()
    sampler.stop()
    st = attn.device_status()
    if st != attn.Status.OK:
        raise RuntimeError(f"device status after the timed region: {st!r}")
    region_ms = region0.elapsed_time(region1)
    return {"region_ms": max_over_ranks(region_ms, world, dev), "launch_ms": [a.elapsed_time(b) for a, b in evs],
            "clocks": sampler.summary(t_wall0, t_wall1)}


def peak_for(w: I.Workload) -> tuple[float, str]:
    peaks = measured_peaks()
    bf16_peak = peaks.get("bf16_tflops")
    src = "measured bf16_tflops (burst, cuBLAS)" if bf16_peak else "fallback 1900 bf16"
    if not bf16_peak:
        bf16_peak = 1900.0
    if w.dtype == "mxfp8":
        # FP8 dense = 2 x bf16 dense (4.5 / 2.25 PFLOP/s nominal)
        return 2.0 * bf16_peak, src + " x 2 (nominal FP8/bf16 ratio)"
    return bf16_peak, src


def roofline_of(w: I.Workload, launch_ms: list[float], kernel: str | None = None, variant: str = "") -> dict:
    """Roofline of the timed kernel; ``variant`` ("_2cta", "_unroll_kv") names a
    kernel other than the workload's default, whose DRAM traffic comes from its
    own launch list (None if it has none)."""
    peak, src = peak_for(w)
    achieved = w.flops / (float(np.mean(launch_ms)) * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": profiled_traffic(w.name + variant), "peak_source": src, "flop_per_launch": w.flops,
            "kernel": kernel or KERNEL_NAMES[(w.direction, w.dtype)]}


def kernel_ms_of(launch_ms: list[float]) -> dict:
    return {"mean": float(np.mean(launch_ms)), "min": float(np.min(launch_ms)), "max": float(np.max(launch_ms)),
            "median": float(np.median(launch_ms))}


class _Opts:
    """The per-run options a step class reads, for the workload sub-records."""

    def __init__(self, base, **over):
        self.tau = base.tau if base.tau_given is not None else 8.0
        self.tau_given = base.tau_given
        self.exp2_emu16 = base.exp2_emu16
        self.p_scaling = base.p_scaling
        self.two_cta = False
        self.unroll_kv = False
        for k, v in over.items():
            setattr(self, k, v)


def sub_record(attn, w: I.Workload, dev, world: int, opts, steps: int, warmup: int) -> dict:
    """One workload of the suite: its own timed region, roofline and clocks."""
    step = step_class(w)(attn, w, dev, opts)
    flush = None
    l2_note = f"inputs larger than L2 ({step.input_bytes() / 2**20:.0f} MiB > 129 MB)"
    if step.input_bytes() <= L2_BYTES:
        scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        flush = scratch.zero_
        l2_note = ("inputs fit in L2: a 258 MB buffer is written between steps (inside the region); "
                   "value uses the per-launch CUDA events, which time the kernel alone")
    m = measure(step, dev, world, steps, warmup, flush)
    per_step_ms = m["region_ms"] / steps
    launch_mean = float(np.mean(m["launch_ms"]))
    rec = {"config": {**w.describe(), "l2": l2_note, "tau": getattr(step, "tau", opts.tau),
                      "exp2_emu16": opts.exp2_emu16},
           "steps": steps, "warmup": warmup,
           "value": w.flops * steps * world / (m["region_ms"] * 1e-3) / 1e12 if flush is None
           else w.flops * world / (launch_mean * 1e-3) / 1e12,
           "unit": UNIT, "ms_per_step": per_step_ms if flush is None else launch_mean,
           "kernel_ms": kernel_ms_of(m["launch_ms"]),
           "roofline": roofline_of(w, m["launch_ms"], "attn_fwd_bf16_2cta_kernel" if opts.two_cta else None,
                                   "_2cta" if opts.two_cta else "_unroll_kv" if opts.unroll_kv else ""),
           "clocks": m["clocks"], "gpu_launches": steps * step.launches}
    if w.dtype == "mxfp8" and w.direction == "fwd":
        rec["config"]["p_scaling"] = ["block_amax", "constant_2^-8", "constant_2^-8_e5m2"][opts.p_scaling]
        if opts.unroll_kv:
            rec["config"]["schedule"] = "unroll_kv"
        q_ms = per_step_ms - launch_mean
        rec["quantize_ms_per_step"] = q_ms
        rec["quantize_share_of_step"] = q_ms / per_step_ms
    del step
    torch.cuda.empty_cache()
    return rec


def workload_suite(attn, args, dev, world: int) -> dict:
    """Every forward workload besides the headline one, each timed on its own:
    the tiny one, the causal d = 128 one (Q, K ~ N(0, 2^2)), the causal d = 64
    one with the MUFU alone and with each software-exp2 share (the best share
    reported beside it), the headline shape on CTA pairs, the MXFP8 one with
    the quantiser's share (on both schedules), and the merge of four partial
    results of the headline shape (bandwidth against the HBM copy rate)."""
    steps, warmup = args.suite_steps, max(3, args.warmup)
    out = {}
    out[I.TINY.name] = sub_record(attn, I.TINY, dev, world, _Opts(args, exp2_emu16=0), steps, warmup)
    out[I.CAUSAL_D128_WIDE.name] = sub_record(attn, I.CAUSAL_D128_WIDE, dev, world, _Opts(args, exp2_emu16=0), steps,
                                              warmup)
    w = I.CAUSAL_D64
    mufu = sub_record(attn, w, dev, world, _Opts(args, exp2_emu16=0), steps, warmup)
    sweep = {}
    for emu in (1, 2, 3, 4):
        r = sub_record(attn, w, dev, world, _Opts(args, exp2_emu16=emu), steps, warmup)
        sweep[f"{emu}/16"] = r
    best = max(sweep, key=lambda k: sweep[k]["roofline"]["achieved"])
    mufu["software_exp2_best"] = {"share": best, **sweep[best]}
    mufu["software_exp2_sweep"] = {k: {"value": r["value"], "kernel_ms_mean": r["kernel_ms"]["mean"],
                                       "achieved": r["roofline"]["achieved"]} for k, r in sweep.items()}
    out[w.name] = mufu
    # the non-causal d = 128 workload once more on CTA pairs (attn_fwd_2cta)
    out[I.NONCAUSAL_D128.name + "_2cta"] = sub_record(attn, I.NONCAUSAL_D128, dev, world,
                                                      _Opts(args, exp2_emu16=0, two_cta=True), steps, warmup)
    out[I.MXFP8_CAUSAL.name] = sub_record(attn, I.MXFP8_CAUSAL, dev, world,
                                          _Opts(args, exp2_emu16=0, p_scaling=0), steps, warmup)
    # the merge of four partial results of the non-causal d = 128 shape (a sequence split over four ranks)
    out[combine_name(I.NONCAUSAL_D128, 4)] = combine_record(attn, I.NONCAUSAL_D128, 4, dev, world, steps, warmup)
    # the same on the unroll-KV schedule (attn_fwd_mxfp8_unroll_kv)
    out[I.MXFP8_CAUSAL.name + "_unroll_kv"] = sub_record(attn, I.MXFP8_CAUSAL, dev, world,
                                                         _Opts(args, exp2_emu16=0, p_scaling=0, unroll_kv=True),
                                                         steps, warmup)
    return out


def bench_ours(args, w: I.Workload, world: int, rank: int, local: int) -> None:
    import online_softmax_fwd_gb300 as attn
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    attn.lib()
    step = step_class(w)(attn, w, dev, args)
    m = measure(step, dev, world, args.steps, args.warmup)
    region_ms_max, launch_ms = m["region_ms"], m["launch_ms"]
    value = w.flops * args.steps * world / (region_ms_max * 1e-3) / 1e12

    e2e = None if args.no_e2e else step.e2e(dev, max(3, min(args.steps, 10)), world)
    roofline = roofline_of(w, launch_ms, "attn_fwd_bf16_2cta_kernel" if args.two_cta else None,
                           "_2cta" if args.two_cta else "_unroll_kv" if args.unroll_kv else "")

    cpu = None
    threads, threads_src = oracle_threads()
    if rank == 0 and world == 1 and not args.no_cpu_baseline and w.direction == "bwd":
        ins = ((step.xq_h, step.xk_h, step.xv_h) if w.dtype == "mxfp8" else (step.q_h, step.k_h, step.v_h))
        s = oracle_bwd_sample(w, *ins, step.o_h, step.do_h, step.lse_h, args.cpu_seconds)
        cpu = {"value": s["value"], "unit": UNIT, "cores": threads, "cores_source": threads_src, "kind": "oracle",
               "sample": f"float64 {'MXFP8 ' if w.dtype == 'mxfp8' else ''}backward oracle on the workload's first "
                         f"{s['heads_touched']} whole head(s) (O and LSE from the forward kernel), "
                         f"{s['seconds']:.1f} s"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = oracle_sample(w, *cpu_inputs(step, w), args.cpu_seconds)
        cpu = {"value": s["value"], "unit": UNIT, "cores": threads, "cores_source": threads_src, "kind": "oracle",
               "sample": f"float64 one-shot oracle on {s['rows']} query rows of the workload's first "
                         f"{s['heads_touched']} head(s) against all their keys, {s['seconds']:.1f} s"
                         + (" (inputs: the oracle's own MXFP8 quantisation, dequantised)" if w.dtype == "mxfp8" else "")}
    input_mib = step.input_bytes() / 2**20
    gpu_launches = args.steps * step.launches
    del step
    torch.cuda.empty_cache()
    suite = None
    if not args.no_suite and w.name == DEFAULT_WORKLOAD and w.direction == "fwd":
        suite = workload_suite(attn, args, dev, world)
    if rank == 0:
        out = {"metric": METRIC_BWD if w.direction == "bwd" else METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": region_ms_max / args.steps, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8" if w.dtype == "mxfp8" else "bf16",
               "data": "synthetic",
               "config": {**w.describe(), "parallelism": f"replicas{world}" if world > 1 else "single",
                          "l2": f"inputs larger than L2 ({input_mib:.0f} MiB > 129 MB)",
                          "tau": (0.0 if args.tau_given is None else args.tau) if w.dtype == "mxfp8" else args.tau,
                          "exp2_emu16": args.exp2_emu16, **({"kernel": "2cta"} if args.two_cta else {}),
                          **({"p_scaling": ["block_amax", "constant_2^-8", "constant_2^-8_e5m2"][args.p_scaling]}
                             if w.dtype == "mxfp8" and w.direction == "fwd" else
                             {"p_scaling": "constant_2^-8", "ds_blocks": "32x32"} if w.dtype == "mxfp8" else {})},
               "e2e": e2e, "gpu_launches": gpu_launches, "roofline": roofline, "cpu_baseline": cpu,
               "clocks": m["clocks"], "kernel_ms": kernel_ms_of(launch_ms),
               "host_overhead_us_per_call": 1e3 * (region_ms_max / args.steps - float(np.mean(launch_ms)))}
        if suite is not None:
            out["workloads"] = suite
        print(json.dumps(out), flush=True)


def cpu_inputs(step, w):
    """Inputs for the oracle sample: the bf16 tensors, or for MXFP8 the oracle's
    own dequantisation of the fp32 draws (per head, inside oracle_sample)."""
    if w.dtype == "mxfp8":
        return step.xq_h, step.xk_h, step.xv_h
    return step.q_h, step.k_h, step.v_h


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(I.WORKLOADS))
    ap.add_argument("--shape", default=None,
                    help="B,H,N,d[,causal[,mxfp8[,bwd]]] instead of a named workload (profiling a smaller case)")
    ap.add_argument("--qk-std", type=float, default=1.0,
                    help="standard deviation of Q and K for --shape (the causal d128 workload uses 2)")
    ap.add_argument("--combine", type=int, default=0, metavar="P",
                    help="time only attn_combine merging P partial results of the workload's shape and print its record")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--exp2-emu16", type=int, default=0)
    ap.add_argument("--tau", type=float, default=None,
                    help="rescale threshold (default 8 for bf16 P, 0 for FP8 P)")
    ap.add_argument("--p-scaling", type=int, default=0, choices=[0, 1, 2],
                    help="MXFP8 P scale: 0 one per 32 keys from the block amax, 1 the constant 2^-8, "
                         "2 the constant 2^-8 with P in E5M2")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-suite", action="store_true",
                    help="skip the other forward workloads (timed after the headline one by default)")
    ap.add_argument("--suite-steps", type=int, default=20)
    ap.add_argument("--unroll-kv", action="store_true",
                    help="MXFP8 forward on the unroll-KV schedule (attn_fwd_mxfp8_unroll_kv)")
    ap.add_argument("--two-cta", action="store_true",
                    help="bf16 d = 128 non-causal forward on CTA pairs (attn_fwd_2cta)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = I.WORKLOADS[args.workload]
    args.tau_given = args.tau
    if args.tau is None:
        args.tau = 8.0
    if args.shape:
        f = [int(x) for x in args.shape.split(",")]
        causal = bool(f[4]) if len(f) > 4 else False
        dt = "mxfp8" if len(f) > 5 and f[5] else "bf16"
        direction = "bwd" if len(f) > 6 and f[6] else "fwd"
        w = I.Workload(f"custom_b{f[0]}h{f[1]}n{f[2]}d{f[3]}{'_causal' if causal else ''}{'_mxfp8' if dt == 'mxfp8' else ''}"
                       f"{'_bwd' if direction == 'bwd' else ''}{f'_qk{args.qk_std:g}' if args.qk_std != 1.0 else ''}",
                       f[0], f[1], f[2], f[3], causal, dtype=dt, direction=direction, qk_std=args.qk_std)
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.combine:
            import online_softmax_fwd_gb300 as attn
            dev = torch.device("cuda", local)
            torch.cuda.set_device(dev)
            rec = combine_record(attn, w, args.combine, dev, world, args.steps, args.warmup)
            if rank == 0:
                print(json.dumps(rec), flush=True)
            return
        if args.impl == "reference":
            bench_reference(args, w, world, rank)
        else:
            bench_ours(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
