#!/usr/bin/env python3
"""Benchmark of the fused decoder-layer kernels on GB300: achieved HBM GB/s (and tokens/s) per step.

A step is one pass of the whole hot path over one synthetic batch: for the default workload, the
Llama-3.1-405B-shaped FP8 path (2048 tokens: add+RMSNorm -> E4M3 static, SwiGLU -> E4M3 dynamic) plus
the ragged hidden 5120 / intermediate 13824 shapes at 1, 3, 17 and 1000 tokens through all four entry
points (bf16 norm, FP8 norm, bf16 SwiGLU, FP8 SwiGLU). Every launch goes through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference] [--workload KEY]

Prints ONE JSON line on rank 0. `value` = algorithmic bytes of all steps on all ranks / device time
(max over ranks). The reference arm (--impl reference) times the CPU oracle on a bounded row sample.
Diagnostics go to stderr.
"""
from __future__ import annotations

import argparse
import ctypes
import concurrent.futures as cf
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from datetime import datetime
from typing import Dict, List, Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "achieved HBM GB/s (% of GB300 peak) and tokens/s per fused kernel vs CPU oracle"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = "llama3.1-405b_fp8_T2048+ragged"

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel, from the ncu capture
# summarised under profiles/; valid only while what the kernel and its launch shape are built from hashes to
# `src_sha256` (kernel_src_hash).
TRAFFIC: Dict[str, Dict] = {
    # profiles/swiglu_q8_dynamic_T2048_I53248.md
    "swiglu_q8_dynamic_T2048_I53248": {"bytes": 526700032, "src_sha256": "74cab478785cc9571472d05ce066d28edc4885cf97aa580d142a4528fab2d0f8"},
    # profiles/add_rmsnorm_q8_static_T1000_H5120.md
    "add_rmsnorm_q8_static_T1000_H5120": {"bytes": 20503040, "src_sha256": "713aeb9c0d1731ee9ac0e7fb9408a229094e56f2d181d344b35e6e5a800d577f"},
    # profiles/add_rmsnorm_q8_static_T2048_H16384.md
    "add_rmsnorm_q8_static_T2048_H16384": {"bytes": 174872576, "src_sha256": "713aeb9c0d1731ee9ac0e7fb9408a229094e56f2d181d344b35e6e5a800d577f"},
    # profiles/add_rmsnorm_T8192_H4096.md
    "add_rmsnorm_T8192_H4096": {"bytes": 208775424, "src_sha256": "713aeb9c0d1731ee9ac0e7fb9408a229094e56f2d181d344b35e6e5a800d577f"},
    # profiles/swiglu_T8192_I14336.md
    "swiglu_T8192_I14336": {"bytes": 657848064, "src_sha256": "74cab478785cc9571472d05ce066d28edc4885cf97aa580d142a4528fab2d0f8"},
    # profiles/swiglu_q8_dynamic_T4096_I28672.md
    "swiglu_q8_dynamic_T4096_I28672": {"bytes": 539429632, "src_sha256": "74cab478785cc9571472d05ce066d28edc4885cf97aa580d142a4528fab2d0f8"},
    # profiles/swiglu_nvfp4_T2048_I53248.md
    "swiglu_nvfp4_T2048_I53248": {"bytes": 467830272, "src_sha256": "74cab478785cc9571472d05ce066d28edc4885cf97aa580d142a4528fab2d0f8"},
    # profiles/add_rmsnorm_nvfp4_T2048_H16384.md
    "add_rmsnorm_nvfp4_T2048_H16384": {"bytes": 161357312, "src_sha256": "713aeb9c0d1731ee9ac0e7fb9408a229094e56f2d181d344b35e6e5a800d577f"},
    # profiles/allreduce_rmsnorm_q8_static_k8_T2048_H16384.md
    "allreduce_rmsnorm_q8_static_k8_T2048_H16384": {"bytes": 690852864, "src_sha256": "713aeb9c0d1731ee9ac0e7fb9408a229094e56f2d181d344b35e6e5a800d577f"},
    # profiles/allreduce_rmsnorm_k8_T2048_H16384.md
    "allreduce_rmsnorm_k8_T2048_H16384": {"bytes": 716697600, "src_sha256": "713aeb9c0d1731ee9ac0e7fb9408a229094e56f2d181d344b35e6e5a800d577f"},
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def workloads_by_key() -> Dict[str, wl.Workload]:
    ws = [wl.qwen_t16(), wl.llama3_8b_prefill(), wl.llama3_70b_fp8(), wl.llama31_405b_fp8_ragged(),
          wl.llama31_405b_tp8_allreduce_norm(), wl.llama31_405b_nvfp4()]
    ws += wl.qwen_decode_sweep()
    return {w.key: w for w in ws}


def decode_sweep_workload() -> wl.Workload:
    """All token counts of the Qwen2.5-1.5B decode sweep in one step (28 layers each)."""
    calls = []
    for w in wl.qwen_decode_sweep():
        calls += list(w.calls)
    return wl.Workload("qwen2.5-1.5b_decode_sweep", "Qwen2.5-1.5B decode sweep, T in 1..256, 28 layers",
                       tuple(calls), layers=28)


def kernel_src_hash(call) -> str:
    """sha256 over what one call's kernel and its launch shape are built from: the C-ABI header, the shared
    device headers, the planner (api.cu), the kernel's translation unit and inline body (comments and whitespace
    removed), and the packaged launch-shape tables. Unchanged when only other kernels' sources, comments or
    layout change."""
    csrc = os.path.join(ROOT, "memory_bound_decoder_gb300", "csrc")
    own = ["swiglu.cu", "swiglu_impl.cuh"] if call.kind.startswith("swiglu") else ["norm.cu", "norm_impl.cuh"]
    paths = [os.path.join(ROOT, "include", "mbd.h")] + [os.path.join(csrc, f) for f in
                                                         ["common.cuh", "launch.h", "api.cu"] + own]
    tdir = os.path.join(ROOT, "memory_bound_decoder_gb300", "tuning")
    paths += sorted(os.path.join(tdir, f) for f in os.listdir(tdir) if f.endswith(".json"))
    h = hashlib.sha256()
    for p in paths:
        with open(p, "rb") as fh:
            text = fh.read()
        if not p.endswith(".json"):   # comments and layout do not change what is built
            text = re.sub(rb"\s+", b"", re.sub(rb"/\*.*?\*/|//[^\n]*", b"", text, flags=re.S))
        h.update(os.path.basename(p).encode() + text)
    return h.hexdigest()


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------------------------------ CPU baseline

def oracle_run_call(call: wl.Call, inp) -> None:
    import oracle
    oracle.build()
    if call.kind == "allreduce_rmsnorm":
        oracle.allreduce_add_rmsnorm(inp.partials, inp.residual, inp.weight, call.eps, want_v=False)
    elif call.kind == "allreduce_rmsnorm_q8":
        oracle.allreduce_add_rmsnorm_quant_fp8(inp.partials, inp.residual, inp.weight, call.eps, call.mode,
                                               call.static_scale, want_v=False)
    elif call.kind == "add_rmsnorm":
        oracle.add_rmsnorm(inp.x, inp.residual, inp.weight, call.eps, want_v=False)
    elif call.kind == "add_rmsnorm_q8":
        oracle.add_rmsnorm_quant_fp8(inp.x, inp.residual, inp.weight, call.eps, call.mode, call.static_scale,
                                     want_v=False)
    elif call.kind == "add_rmsnorm_nvfp4":
        oracle.add_rmsnorm_quant_nvfp4(inp.x, inp.residual, inp.weight, call.eps, call.static_scale, want_v=False)
    elif call.kind == "swiglu":
        oracle.swiglu(inp.gate_up, want_h=False)
    elif call.kind == "swiglu_nvfp4":
        oracle.swiglu_quant_nvfp4(inp.gate_up, call.static_scale, want_h=False)
    else:
        oracle.swiglu_quant_fp8(inp.gate_up, call.mode, call.static_scale, want_h=False)


def _split(call: wl.Call, inp, nchunks: int):
    """Split a call's inputs into row blocks (rows are independent)."""
    T = call.T
    bounds = np.linspace(0, T, min(T, nchunks) + 1).astype(int)
    out = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            continue
        if call.kind.startswith("allreduce"):
            out.append(wl.PartialNormInputs([q[a:b] for q in inp.partials], inp.residual[a:b], inp.weight, inp.eps))
        elif call.kind.startswith("add"):
            out.append(wl.NormInputs(inp.x[a:b], inp.residual[a:b], inp.weight, inp.eps))
        else:
            out.append(wl.SwigluInputs(inp.gate_up[a:b]))
    return out


class OracleSample:
    """A bounded, evenly spaced row sample of every call of a workload, run by the oracle on all host cores."""

    def __init__(self, work: wl.Workload, frac: float, threads: int, seed: int = 0):
        import oracle
        oracle.build()
        self.work, self.threads, self.frac = work, threads, frac
        self.items = []
        self.bytes = 0
        self.rows = 0
        for ci, call in enumerate(work.calls):
            n = max(1, int(round(call.T * frac)))
            rows = np.unique(np.linspace(0, call.T - 1, n).round().astype(np.int64))
            inp = wl.inputs_for(call, seed=seed, salt=ci, rows=rows)
            sub = wl.Call(call.kind, len(rows), call.width, call.dist, call.eps, call.mode, call.static_scale,
                          call.partials)
            self.items.append((sub, _split(sub, inp, threads)))
            self.bytes += sub.algorithmic_bytes() * work.layers
            self.rows += len(rows)
        self.tokens = sum(len(np.unique(np.linspace(0, t - 1, max(1, int(round(t * frac)))).round()))
                          for t in sorted({c.T for c in work.calls}))
        self.pool = cf.ThreadPoolExecutor(max_workers=threads)

    def run(self) -> None:
        jobs = []
        for _ in range(self.work.layers):
            for call, chunks in self.items:
                for ch in chunks:
                    jobs.append(self.pool.submit(oracle_run_call, call, ch))
        for j in jobs:
            j.result()

    def describe(self) -> str:
        return (f"{self.frac:.4g} of the rows of every call, evenly spaced ({self.rows} rows, "
                f"{self.bytes / 1e6:.1f} MB algorithmic per step), fp64 C oracle, {self.threads} threads")


def calibrate_fraction(work: wl.Workload, threads: int, target_s: float) -> float:
    """Row fraction whose oracle run takes about target_s on `threads` host threads: one row of every call
    is timed on its own and scaled by that call's row count."""
    full_s = 0.0
    for ci, call in enumerate(work.calls):
        rows = np.array([0], np.int64)
        inp = wl.inputs_for(call, seed=0, salt=ci, rows=rows)
        one = wl.Call(call.kind, 1, call.width, call.dist, call.eps, call.mode, call.static_scale, call.partials)
        t = time.perf_counter()
        oracle_run_call(one, inp)
        full_s += (time.perf_counter() - t) * call.T * work.layers
    full_s /= max(1, threads)
    return float(min(1.0, max(1e-6, target_s / max(full_s, 1e-9))))


def cpu_baseline(work: wl.Workload, target_s: float = 1.0) -> Dict:
    threads = os.cpu_count() or 1
    frac = calibrate_fraction(work, threads, target_s)
    s = OracleSample(work, frac, threads)
    s.run()  # warm
    t = time.perf_counter()
    s.run()
    dt = time.perf_counter() - t
    return {"value": round(s.bytes / dt / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": s.describe(), "tokens_per_s": round(s.tokens / dt, 2), "seconds": round(dt, 3)}


# ------------------------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ["timestamp", "uuid", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid: str):
        self.uuid = uuid.lower().replace("gpu-", "")
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0: float, t1: float) -> Optional[Dict]:
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != len(self.FIELDS) or self.uuid not in parts[1].lower():
                    continue
                try:
                    ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[4], parts[6:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if t0 <= r[0] <= t1]
        basis = "inside the timed region"
        if not inside:   # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:3]
            basis = "nearest samples to a short timed region"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "basis": basis}


# ------------------------------------------------------------------------------------------------ ranks

def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank value over all ranks (the slowest rank sets the job's time); identity
    without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(bytes_per_step: int, steps: int, world: int, ms: float) -> float:
    """Whole-job GB/s: every rank processes its own full step (weak scaling), timed by the slowest rank."""
    return bytes_per_step * steps * world / (ms / 1e3) / 1e9


# ------------------------------------------------------------------------------------------------ GPU arm

class DeviceCall:
    """Device (and pinned host) buffers of one call, and the prepared C-ABI argument tuple."""

    def __init__(self, torch, mbd, call: wl.Call, inp, dev, shared_residual=None):
        self.call = call
        self.mbd = mbd
        T, W = call.T, call.width
        u16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
        self.h2d = []   # (device tensor, pinned host tensor): activation inputs copied in by the e2e leg
        self.d2h = []   # (device tensor, pinned host tensor): outputs copied back by the e2e leg
        if call.kind.startswith("allreduce"):
            self.ps = [u16(q).to(dev) for q in inp.partials]
            self.res = u16(inp.residual).to(dev)
            self.w = u16(inp.weight).to(dev)
            self.h2d += [(t, u16(q).pin_memory()) for t, q in zip(self.ps, inp.partials)]
            self.h2d.append((self.res, u16(inp.residual).pin_memory()))
            lib = mbd.get_lib()

            self._parr = (ctypes.c_void_p * len(self.ps))(*[t.data_ptr() for t in self.ps])
            if call.kind == "allreduce_rmsnorm":
                self.out = torch.empty((T, W), dtype=torch.int16, device=dev)
                self.fn = lib.mbd_fused_allreduce_add_rmsnorm
                self.args = [self.out.data_ptr(), self.res.data_ptr(), self._parr, len(self.ps), self.w.data_ptr(),
                             T, W, call.eps]
            else:
                self.out = torch.empty((T, W), dtype=torch.uint8, device=dev)
                self.scale = (torch.tensor([call.static_scale], dtype=torch.float32, device=dev)
                              if call.mode == "static" else torch.zeros((T,), dtype=torch.float32, device=dev))
                self.fn = lib.mbd_fused_allreduce_add_rmsnorm_quant_fp8
                self.args = [self.out.data_ptr(), self.res.data_ptr(), self._parr, len(self.ps), self.w.data_ptr(),
                             T, W, call.eps, mbd.MODES[call.mode], self.scale.data_ptr()]
                if call.mode == "dynamic":
                    self.d2h.append((self.scale, torch.empty_like(self.scale, device="cpu").pin_memory()))
            self.d2h.append((self.res, torch.empty_like(self.res, device="cpu").pin_memory()))
        elif call.kind.startswith("add"):
            self.x = u16(inp.x).to(dev)
            self.res = shared_residual if shared_residual is not None else u16(inp.residual).to(dev)
            self.w = u16(inp.weight).to(dev)
            self.h2d += [(self.x, u16(inp.x).pin_memory()), (self.res, u16(inp.residual).pin_memory())]
            if call.kind == "add_rmsnorm":
                self.out = torch.empty((T, W), dtype=torch.int16, device=dev)
                self.fn = mbd.get_lib().mbd_fused_add_rmsnorm
                self.args = [self.out.data_ptr(), self.res.data_ptr(), self.x.data_ptr(), self.w.data_ptr(),
                             T, W, call.eps]
            elif call.kind == "add_rmsnorm_nvfp4":
                self.out = torch.empty((T, W // 2), dtype=torch.uint8, device=dev)
                self.sf = torch.empty((T, W // 16), dtype=torch.uint8, device=dev)
                self.scale = torch.tensor([call.static_scale], dtype=torch.float32, device=dev)
                self.fn = mbd.get_lib().mbd_fused_add_rmsnorm_quant_nvfp4
                self.args = [self.out.data_ptr(), self.sf.data_ptr(), self.res.data_ptr(), self.x.data_ptr(),
                             self.w.data_ptr(), T, W, call.eps, self.scale.data_ptr()]
                self.d2h.append((self.sf, torch.empty_like(self.sf, device="cpu").pin_memory()))
            else:
                self.out = torch.empty((T, W), dtype=torch.uint8, device=dev)
                self.scale = (torch.tensor([call.static_scale], dtype=torch.float32, device=dev)
                              if call.mode == "static" else torch.zeros((T,), dtype=torch.float32, device=dev))
                self.fn = mbd.get_lib().mbd_fused_add_rmsnorm_quant_fp8
                self.args = [self.out.data_ptr(), self.res.data_ptr(), self.x.data_ptr(), self.w.data_ptr(),
                             T, W, call.eps, mbd.MODES[call.mode], self.scale.data_ptr()]
                if call.mode == "dynamic":
                    self.d2h.append((self.scale, torch.empty_like(self.scale, device="cpu").pin_memory()))
            self.d2h.append((self.res, torch.empty_like(self.res, device="cpu").pin_memory()))
        else:
            self.gu = u16(inp.gate_up).to(dev)
            self.h2d.append((self.gu, u16(inp.gate_up).pin_memory()))
            if call.kind == "swiglu":
                self.out = torch.empty((T, W), dtype=torch.int16, device=dev)
                self.fn = mbd.get_lib().mbd_swiglu
                self.args = [self.out.data_ptr(), self.gu.data_ptr(), T, W]
            elif call.kind == "swiglu_nvfp4":
                self.out = torch.empty((T, W // 2), dtype=torch.uint8, device=dev)
                self.sf = torch.empty((T, W // 16), dtype=torch.uint8, device=dev)
                self.scale = torch.tensor([call.static_scale], dtype=torch.float32, device=dev)
                self.fn = mbd.get_lib().mbd_swiglu_quant_nvfp4
                self.args = [self.out.data_ptr(), self.sf.data_ptr(), self.gu.data_ptr(), T, W, self.scale.data_ptr()]
                self.d2h.append((self.sf, torch.empty_like(self.sf, device="cpu").pin_memory()))
            else:
                self.out = torch.empty((T, W), dtype=torch.uint8, device=dev)
                self.scale = (torch.tensor([call.static_scale], dtype=torch.float32, device=dev)
                              if call.mode == "static" else torch.zeros((T,), dtype=torch.float32, device=dev))
                self.fn = mbd.get_lib().mbd_swiglu_quant_fp8
                self.args = [self.out.data_ptr(), self.gu.data_ptr(), T, W, mbd.MODES[call.mode],
                             self.scale.data_ptr()]
                if call.mode == "dynamic":
                    self.d2h.append((self.scale, torch.empty_like(self.scale, device="cpu").pin_memory()))
        self.d2h.append((self.out, torch.empty_like(self.out, device="cpu").pin_memory()))

    def bind(self, stream_handle: int):

        args = list(self.args)
        if self.call.kind in ("add_rmsnorm", "add_rmsnorm_q8"):
            args[6] = ctypes.c_float(args[6])
        elif self.call.kind.startswith("allreduce") or self.call.kind == "add_rmsnorm_nvfp4":
            args[7] = ctypes.c_float(args[7])
        self.bound = tuple(args) + (stream_handle,)

    def op(self):
        """This call as a program op (mbd_op), or None for kinds a program does not take."""
        m, c = self.mbd, self.call
        T, W = c.T, c.width
        if c.kind == "add_rmsnorm":
            return m.op_add_rmsnorm(self.out, self.res, self.x, self.w, T, W, c.eps)
        if c.kind == "add_rmsnorm_q8":
            return m.op_add_rmsnorm_quant_fp8(self.out, self.res, self.x, self.w, T, W, c.eps, c.mode, self.scale)
        if c.kind == "add_rmsnorm_nvfp4":
            return m.op_add_rmsnorm_quant_nvfp4(self.out, self.sf, self.res, self.x, self.w, T, W, c.eps, self.scale)
        if c.kind == "swiglu":
            return m.op_swiglu(self.out, self.gu, T, W)
        if c.kind == "swiglu_q8":
            return m.op_swiglu_quant_fp8(self.out, self.gu, T, W, c.mode, self.scale)
        if c.kind == "swiglu_nvfp4":
            return m.op_swiglu_quant_nvfp4(self.out, self.sf, self.gu, T, W, self.scale)
        return None

    def launch(self):
        rc = self.fn(*self.bound)
        if rc != 0:
            raise RuntimeError(f"{self.call.name}: {self.mbd.get_lib().mbd_status_string(rc).decode()}")

    def bytes_in(self):
        return sum(t.numel() * t.element_size() for t, _ in self.h2d)

    def bytes_out(self):
        return sum(t.numel() * t.element_size() for t, _ in self.d2h)


# Program variants of the library (the epilogue sets one persistent program kernel is compiled for), by call kind
# and FP8 mode: a program holds ops of one variant only.
# Epilogue class of each call kind a program can run: "bf16" and "fp8" calls may share one launch (the
# library's mixed bf16 + FP8 program variant; a static-FP8 SwiGLU runs only there), "nvfp4" calls have their
# own variant. A dynamic-FP8 norm runs in no program.
PROGRAM_CLASS = {("add_rmsnorm", None): "bf16", ("swiglu", None): "bf16",
                 ("add_rmsnorm_q8", "static"): "fp8", ("swiglu_q8", "dynamic"): "fp8", ("swiglu_q8", "static"): "fp8",
                 ("add_rmsnorm_nvfp4", None): "nvfp4", ("swiglu_nvfp4", None): "nvfp4"}
PROGRAM_MAX_NORM_WIDTH = 8192   # MBD_MAX_PROGRAM_WIDTH


class GroupCall:
    """The calls of one program launch, seen as one call (name, token count, algorithmic bytes)."""

    def __init__(self, variant: str, calls: List[wl.Call]):
        self.calls = calls
        self.kind, self.mode = "program", None
        self.name = f"program_{variant}_{len(calls)}ops_T" + "+".join(str(c.T) for c in calls)
        self.T = sum(c.T for c in calls)

    def algorithmic_bytes(self) -> int:
        return sum(c.algorithmic_bytes() for c in self.calls)


class ProgramGroup:
    """Calls of one step run as ONE launch of the library's persistent program kernel: the plan is built once,
    its schedule uploaded once to device memory, and every step launches it with one pointer
    (mbd_program_plan_launch_uploaded). Same buffers, same outputs as the calls' own launches."""

    def __init__(self, torch, mbd, variant: str, members: List[DeviceCall], dev):
        self.members, self.mbd = members, mbd
        self.call = GroupCall(variant, [d.call for d in members])
        self.plan = mbd.program_plan_build([d.op() for d in members])
        self.sched = torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device=dev)
        self.h2d = [x for d in members for x in d.h2d]
        self.d2h = [x for d in members for x in d.d2h]
        self.handle = None

    def bind(self, stream_handle: int):
        for d in self.members:
            d.bind(stream_handle)
        self.handle = stream_handle
        self.plan.upload(self.sched, stream_handle)

    def launch(self):
        lib = self.mbd.get_lib()
        rc = lib.mbd_program_plan_launch_uploaded(ctypes.addressof(self.plan.buf), self.sched.data_ptr(), self.handle)
        if rc != 0:
            raise RuntimeError(f"{self.call.name}: {lib.mbd_status_string(rc).decode()}")

    def bytes_in(self):
        return sum(t.numel() * t.element_size() for t, _ in self.h2d)

    def bytes_out(self):
        return sum(t.numel() * t.element_size() for t, _ in self.d2h)


class BatchCall:
    """The calls of one batch, seen as one call (name, token count, algorithmic bytes)."""

    def __init__(self, calls: List[wl.Call]):
        self.calls = calls
        self.kind, self.mode = "batch", None
        self.name = f"batch_{len(calls)}ops_" + "+".join(c.name for c in calls)
        self.T = sum(c.T for c in calls)

    def algorithmic_bytes(self) -> int:
        return sum(c.algorithmic_bytes() for c in self.calls)


class BatchGroup:
    """Independent calls of one step run as ONE call of mbd_run_independent: each op keeps its own single-call
    kernel and launch shape, and each launch after the first overlaps the one before it. Same buffers, same
    outputs (bit for bit) as the calls' own launches."""

    def __init__(self, mbd, members: List[DeviceCall]):
        self.members, self.mbd = members, mbd
        self.call = BatchCall([d.call for d in members])
        self.arr, self.n = mbd.program_array([d.op() for d in members])
        self.h2d = [x for d in members for x in d.h2d]
        self.d2h = [x for d in members for x in d.d2h]
        self.handle = None

    def bind(self, stream_handle: int):
        for d in self.members:
            d.bind(stream_handle)
        self.handle = stream_handle

    def launch(self):
        lib = self.mbd.get_lib()
        rc = lib.mbd_run_independent(self.arr, self.n, self.handle)
        if rc != 0:
            raise RuntimeError(f"{self.call.name}: {lib.mbd_status_string(rc).decode()}")

    def bytes_in(self):
        return sum(t.numel() * t.element_size() for t, _ in self.h2d)

    def bytes_out(self):
        return sum(t.numel() * t.element_size() for t, _ in self.d2h)


class ProgramBatchGroup:
    """A program launch and a batch as ONE call of mbd_run_independent_with_program: the program (the small,
    latency-bound calls) launches first and the batch's single calls start beside it, each overlapping the one
    before. Same buffers and outputs as the program launch followed by the calls."""

    def __init__(self, mbd, program: "ProgramGroup", batch: "BatchGroup"):
        self.mbd, self.program, self.batch = mbd, program, batch
        self.members = program.members + batch.members
        self.call = BatchCall(program.call.calls + batch.call.calls)
        self.call.name = f"{program.call.name}+{batch.call.name}"
        self.h2d = program.h2d + batch.h2d
        self.d2h = program.d2h + batch.d2h
        self.handle = None

    def bind(self, stream_handle: int):
        self.program.bind(stream_handle)
        self.batch.bind(stream_handle)
        self.handle = stream_handle

    def launch(self):
        lib = self.mbd.get_lib()
        rc = lib.mbd_run_independent_with_program(ctypes.addressof(self.program.plan.buf), self.program.sched.data_ptr(),
                                                  self.batch.arr, self.batch.n, self.handle)
        if rc != 0:
            raise RuntimeError(f"{self.call.name}: {lib.mbd_status_string(rc).decode()}")

    def bytes_in(self):
        return sum(t.numel() * t.element_size() for t, _ in self.h2d)

    def bytes_out(self):
        return sum(t.numel() * t.element_size() for t, _ in self.d2h)


def launch_groups(calls: List[wl.Call], layers: int, sms: int, max_ops: int = 128, max_batch: int = 64,
                  programs: bool = True, batches: bool = True) -> list:
    """Launch units of one step, in order: an int (the index of a call launched on its own) or (label, [indices])
    (calls run together). Only in one-layer steps, whose calls share no buffer, so that running them together,
    in any order, computes exactly what the sequence of launches does.
    - Calls with fewer tokens than the GPU has SMs are bound by launch latency, not bandwidth; those a program
      takes are gathered into program launches (at most max_ops each): the bf16 and FP8 ones together when all
      their rows fit one row per SM (one wave of the mixed variant, which runs at one CTA per SM), else one
      launch per class; NVFP4 ones in a launch of their own.
    - The call with the most algorithmic bytes keeps a launch of its own (the bench times it with CUDA events,
      which would split a batch). The other calls of at least one row per SM, if there are two or more, run as
      one batch of their own single-call launches, each overlapping the one before (label "batch",
      mbd_run_independent, at most max_batch per batch): a call of a thousand rows streams its bytes in a few
      microseconds, about as long as a launch takes to ramp up and drain.
    - Order: the largest call, then the batches, then the programs, then any other call in list order (with
      batches, the tails of the large launches overlap the next; the latency-bound programs come last).
    Without batches the units keep list order, each group where its first call stood."""
    if layers != 1:
        return list(range(len(calls)))
    cls: Dict[int, str] = {}
    for i, c in enumerate(calls):
        v = PROGRAM_CLASS.get((c.kind, c.mode if "q8" in c.kind else None))
        small = c.T < sms and not (c.kind.startswith("add") and c.width > PROGRAM_MAX_NORM_WIDTH)
        if programs and v is not None and small:
            cls[i] = v
    largest = max(range(len(calls)), key=lambda i: calls[i].algorithmic_bytes()) if calls else -1
    batch = [i for i, c in enumerate(calls) if batches and i != largest and c.T >= sms
             and not c.kind.startswith("allreduce")]
    if len(batch) >= 2:
        for i in batch:
            cls[i] = "batch"
    mixed_rows = sum(calls[i].T for i, v in cls.items() if v in ("bf16", "fp8"))
    key = {i: ("bf16+fp8" if v in ("bf16", "fp8") and mixed_rows <= sms else v) for i, v in cls.items()}
    groups: Dict[str, List[int]] = {}
    order: list = []
    for i in range(len(calls)):
        if i not in key:
            order.append(i)
            continue
        if key[i] not in groups:
            groups[key[i]] = []
            order.append(key[i])
        groups[key[i]].append(i)
    units: list = []
    for u in order:
        if isinstance(u, str):
            idx = groups[u]
            label = "+".join(sorted({cls[i] for i in idx}))   # what the launch holds
            step = max_batch if u == "batch" else max_ops
            units += [(label, idx[k:k + step]) for k in range(0, len(idx), step)]
        else:
            units.append(u)
    if "batch" in groups:
        rank = lambda u: (0 if u == largest else 3) if isinstance(u, int) else (1 if u[0] == "batch" else 2)
        units.sort(key=rank)   # stable: list order within each rank
    return units


def group_small_calls(torch, mbd, work: wl.Workload, dcalls: List[DeviceCall], sms: int, dev,
                      programs: bool = True, batches: bool = True) -> list:
    """The step's launch units (launch_groups): DeviceCalls, ProgramGroups and BatchGroups."""
    units = launch_groups([d.call for d in dcalls], work.layers, sms, mbd.MAX_PROGRAM_OPS, mbd.MAX_INDEPENDENT_OPS,
                          programs, batches)
    out = []
    for u in units:
        if isinstance(u, int):
            out.append(dcalls[u])
        elif u[0] == "batch":
            out.append(BatchGroup(mbd, [dcalls[i] for i in u[1]]))
        else:
            out.append(ProgramGroup(torch, mbd, u[0], [dcalls[i] for i in u[1]], dev))
    # one program launch and one batch: the program opens the batch (mbd_run_independent_with_program), so
    # its latency-bound rows run beside the batch's bandwidth-bound ones
    progs = [u for u in out if isinstance(u, ProgramGroup)]
    batches = [u for u in out if isinstance(u, BatchGroup)]
    if len(progs) == 1 and len(batches) == 1:
        fused = ProgramBatchGroup(mbd, progs[0], batches[0])
        out = [fused if u is batches[0] else u for u in out if u is not progs[0]]
    return out


def run_e2e(torch, dcalls: List[DeviceCall], kstream, dev, steps: int, step_bytes: int, world: int) -> Dict:
    """Time `steps` steps from pinned host memory to pinned host memory through the same C-ABI launches:
    a three-stage pipeline (H2D copy stream -> the kernel stream -> D2H copy stream) with per-call events,
    so the copy engines and the kernels of different calls overlap. A call's inputs are re-uploaded only
    after the previous step's kernel and download of that call have finished (the residual is read and
    written in place, and downloaded)."""
    steps = max(1, steps)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n = len(dcalls)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_k = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    for d in dcalls:   # one untimed round trip warms the copy paths
        with torch.cuda.stream(s_in):
            for dt_, ht in d.h2d:
                dt_.copy_(ht, non_blocking=True)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(kstream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for k in range(steps):
        for i, d in enumerate(dcalls):
            if k > 0:
                s_in.wait_event(ev_k[i])
                s_in.wait_event(ev_out[i])
            with torch.cuda.stream(s_in):
                for dt_, ht in d.h2d:
                    dt_.copy_(ht, non_blocking=True)
            ev_in[i].record(s_in)
            kstream.wait_event(ev_in[i])
            if k > 0:
                kstream.wait_event(ev_out[i])
            d.launch()
            ev_k[i].record(kstream)
            s_out.wait_event(ev_k[i])
            with torch.cuda.stream(s_out):
                for dt_, ht in d.d2h:
                    ht.copy_(dt_, non_blocking=True)
            ev_out[i].record(s_out)
    s_out.wait_event(ev_in[n - 1])
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    return {"value": round(aggregate_rate(step_bytes, steps, world, e_ms), 3), "unit": UNIT,
            "h2d_bytes_per_step": sum(d.bytes_in() for d in dcalls),
            "d2h_bytes_per_step": sum(d.bytes_out() for d in dcalls),
            "steps": steps, "ms_per_step": round(e_ms / steps, 4),
            "path": "pinned host inputs -> H2D copy stream -> C-ABI launches on the kernel stream -> D2H copy "
                    "stream of every output; per-call events pipeline the three"}


def resolve_tuning(arg: str, torch, dev) -> Optional[str]:
    """The tuning file to install: an explicit path, none, or (auto) the packaged table tuned on this GPU model
    (same name and SM count), if there is one."""
    if arg == "none":
        return None
    if arg != "auto":
        return arg
    d = os.path.join(ROOT, "memory_bound_decoder_gb300", "tuning")
    props = torch.cuda.get_device_properties(dev)
    for f in sorted(os.listdir(d)) if os.path.isdir(d) else []:
        if not f.endswith(".json"):
            continue
        with open(os.path.join(d, f)) as fh:
            meta = json.load(fh)
        if meta.get("device") == props.name and meta.get("multiprocessors") == props.multi_processor_count:
            return os.path.join(d, f)
    return None


def build_device_calls(torch, mbd, work: wl.Workload, seed: int, rank: int, dev) -> List[DeviceCall]:
    """Device buffers of every launch of one step. Layers repeat the calls with fresh inputs; in a multi-layer
    step every norm of one token count updates one shared residual, as a decoder's layers do."""
    dcalls: List[DeviceCall] = []
    residual_by_T: Dict[int, object] = {}
    for layer in range(work.layers):
        for ci, call in enumerate(work.calls):
            salt = layer * 64 + ci + 1000 * rank
            inp = wl.inputs_for(call, seed=seed, salt=salt)
            shared = None
            if work.layers > 1 and call.kind.startswith("add"):
                if call.T not in residual_by_T:
                    residual_by_T[call.T] = torch.from_numpy(inp.residual.view(np.int16)).to(dev)
                shared = residual_by_T[call.T]
            dcalls.append(DeviceCall(torch, mbd, call, inp, dev, shared))
    return dcalls


def run_decode_table(args) -> Dict:
    """Decode-step latency of the Qwen2.5-1.5B-shaped sweep (28 layers x (add + RMSNorm, add + RMSNorm,
    SwiGLU) per token count), launched three ways: one C-ABI call per op, the same calls replayed from a CUDA
    graph, programs (the 84 ops of one token count as one persistent launch, a plan built once and launched every
    step, with its schedule in the launch parameters or uploaded once to device memory), and the by-value launch
    replayed from a CUDA graph."""
    import torch
    import memory_bound_decoder_gb300 as mbd
    from memory_bound_decoder_gb300 import build as mbd_build
    mbd_build.build()
    lib = mbd.get_lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    table, modes = {}, ("calls", "graph", "program", "program_dev", "program_static", "program_graph")
    launches = {}
    tokens = tuple(int(t) for t in args.decode_tokens.split(",")) if args.decode_tokens else (1, 2, 4, 8, 32, 64, 128, 256)
    for work in wl.qwen_decode_sweep(tokens):
        T = work.calls[0].T
        dcalls = build_device_calls(torch, mbd, work, args.seed, 0, dev)
        stream = torch.cuda.Stream(device=dev)
        handle = int(stream.cuda_stream)
        for d in dcalls:
            d.bind(handle)
        ops = [d.op() for d in dcalls]
        # built once per token count (a decode loop reuses the step's program), launched every step
        t_b = time.perf_counter()
        plans = [mbd.program_plan_build(ops[i:i + mbd.MAX_PROGRAM_OPS]) for i in range(0, len(ops), mbd.MAX_PROGRAM_OPS)]
        build_us = (time.perf_counter() - t_b) * 1e6

        def run_calls():
            for d in dcalls:
                d.launch()

        plan_ptrs = [ctypes.addressof(p.buf) for p in plans]
        scheds = [torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device=dev) for _ in plans]
        for p, sc in zip(plans, scheds):
            p.upload(sc, stream)
        sched_ptrs = [sc.data_ptr() for sc in scheds]

        def run_program():
            for pp in plan_ptrs:
                rc = lib.mbd_program_plan_launch(pp, handle)
                if rc != 0:
                    raise RuntimeError(lib.mbd_status_string(rc).decode())

        with torch.cuda.stream(stream):
            run_calls()
        torch.cuda.synchronize(dev)
        def run_program_dev():
            for pp, sp in zip(plan_ptrs, sched_ptrs):
                rc = lib.mbd_program_plan_launch_uploaded(pp, sp, handle)
                if rc != 0:
                    raise RuntimeError(lib.mbd_status_string(rc).decode())

        def run_program_static():
            for pp in plan_ptrs:
                rc = lib.mbd_program_plan_launch_static(pp, handle)
                if rc != 0:
                    raise RuntimeError(lib.mbd_status_string(rc).decode())

        graphs, graph_errors = {}, {}
        for name, body in (("graph", run_calls), ("program_graph", run_program)):
            g = torch.cuda.CUDAGraph()
            try:
                with torch.cuda.graph(g, stream=stream):
                    body()
                torch.cuda.synchronize(dev)
                graphs[name] = g
            except RuntimeError as e:   # reported in the line instead of a graph time
                graph_errors[name] = str(e).splitlines()[0]
                torch.cuda.synchronize(dev)
        fns = {"calls": run_calls, "program": run_program, "program_dev": run_program_dev,
               "program_static": run_program_static}
        fns.update({k: g.replay for k, g in graphs.items()})
        row = {}
        for mode in modes:
            if mode in graph_errors:
                row[mode] = None
                row[mode + "_error"] = graph_errors[mode]
                continue
            fn = fns[mode]
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    fn()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n0 = mbd.kernel_launches()
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(args.steps):
                    fn()
                e1.record(stream)
            torch.cuda.synchronize(dev)
            launches[(T, mode)] = (mbd.kernel_launches() - n0) // args.steps if "graph" not in mode else None
            ms = e0.elapsed_time(e1) / args.steps
            row[mode] = round(ms * 1e3 / work.layers, 3)
        row["program_GBps"] = round(work.algorithmic_bytes() / (row["program"] * work.layers / 1e6) / 1e9, 1)
        row["launches_per_step"] = {"calls": launches[(T, "calls")], "graph": len(dcalls),
                                    "program": launches[(T, "program")], "program_dev": launches[(T, "program_dev")],
                                    "program_static": launches[(T, "program_static")],
                                    "program_graph": len(plans)}
        row["plan_build_us"] = round(build_us, 1)
        table[str(T)] = row
        log(f"[decode] T={T}: {row}")
        del dcalls, plans, graphs, scheds
        torch.cuda.empty_cache()
    mean_prog = statistics.mean(r["program"] for r in table.values())
    return {"metric": "decode-step latency per layer, Qwen2.5-1.5B shapes (28 layers of 2 add+RMSNorm + 1 SwiGLU)",
            "value": round(mean_prog, 3), "unit": "us/layer (mean over token counts, program launch)",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
            "data": "synthetic", "dtype": "f32",
            "config": {"workload": "qwen2.5-1.5b_decode_sweep", "hidden": 1536, "intermediate": 8960, "layers": 28,
                       "tokens": [int(t) for t in table], "modes": list(modes),
                       "l2": "decode buffers below T~64 are L2-resident between steps: these are latencies"},
            "table": table}


def prepare_step(torch, mbd, args, work: wl.Workload, rank: int, dev, props):
    """Device buffers and launch units of one step of `work`, bound to a fresh stream."""
    t_gen = time.perf_counter()
    dcalls = build_device_calls(torch, mbd, work, args.seed, rank, dev)
    n_calls = len(dcalls)
    if not (args.no_programs and args.no_batches):
        dcalls = group_small_calls(torch, mbd, work, dcalls, props.multi_processor_count, dev,
                                   programs=not args.no_programs, batches=not args.no_batches)
    log(f"[bench] rank {rank}: {work.key}: inputs for {n_calls} calls in {len(dcalls)} launch units ready in "
        f"{time.perf_counter() - t_gen:.1f}s")
    stream = torch.cuda.Stream(device=dev)
    handle = int(stream.cuda_stream)
    for d in dcalls:
        d.bind(handle)
    return dcalls, stream


def time_step(torch, mbd, dcalls, stream, steps: int, warmup: int, dev, props, rank: int, world: int) -> Dict:
    """W untimed steps, a per-unit breakdown pass (CUDA events around every launch unit, each after a read of
    twice the L2 size; untimed), then exactly `steps` timed steps between events on the launch stream (barrier
    and synchronise on both sides), with events around the roofline kernel's launch in every step and the clocks
    sampled meanwhile."""
    def step():
        for d in dcalls:
            d.launch()

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize(dev)

    # per-unit breakdown: each unit between CUDA events after a read of twice the L2 size, so that L2 holds no
    # dirty lines of an earlier kernel whose write-back the unit would pay for (as under ncu's cache control)
    l2 = int(getattr(props, "L2_cache_size", 0)) or 126 * 2 ** 20
    flush = torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)
    nb = max(3, min(20, steps))
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in dcalls]
           for _ in range(nb)]
    with torch.cuda.stream(stream):
        for k in range(nb):
            for d, (a, b) in zip(dcalls, evs[k]):
                flush.max()
                a.record(stream)
                d.launch()
                b.record(stream)
    torch.cuda.synchronize(dev)
    del flush
    per_call_ms = [statistics.median(evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(nb))
                   for i in range(len(dcalls))]
    # the roofline kernel: the slowest launch of a single call (batches and programs hold several kernels)
    singles = [i for i, d in enumerate(dcalls) if isinstance(d, DeviceCall)] or list(range(len(dcalls)))
    dom = max(singles, key=lambda i: per_call_ms[i])

    clock = ClockSampler(str(getattr(props, "uuid", ""))) if rank == 0 else None
    dom_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clock:
        clock.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches0 = mbd.kernel_launches()
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for k in range(steps):
            for i, d in enumerate(dcalls):
                if i == dom:
                    dom_ev[k][0].record(stream)
                    d.launch()
                    dom_ev[k][1].record(stream)
                else:
                    d.launch()
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    launches = mbd.kernel_launches() - launches0
    clocks = clock.stop(t0, t1) if clock else None
    return {"elapsed_ms": max_over_ranks(ev0.elapsed_time(ev1), dev), "per_call_ms": per_call_ms, "dom": dom,
            "dom_ms": statistics.mean(a.elapsed_time(b) for a, b in dom_ev), "clocks": clocks, "launches": launches}


def step_summary(work: wl.Workload, dcalls, t: Dict, steps: int, world: int) -> Dict:
    """value (GB/s), tokens/s, the roofline of the dominant kernel and the per-unit breakdown of a timed step."""
    peak, peak_kind = measured_peak()
    step_bytes = work.algorithmic_bytes()
    dcall = dcalls[t["dom"]]
    dom_bytes = dcall.call.algorithmic_bytes()
    achieved = dom_bytes / (t["dom_ms"] / 1e3) / 1e9
    tr = TRAFFIC.get(dcall.call.name)
    traffic = tr["bytes"] if tr and tr.get("src_sha256") == kernel_src_hash(dcall.call) else None
    kernels, seen = [], set()
    for d in dcalls:
        if d.call.name in seen:
            continue
        seen.add(d.call.name)
        idx = [j for j, e in enumerate(dcalls) if e.call.name == d.call.name]
        ms = statistics.mean(t["per_call_ms"][j] for j in idx)
        b = d.call.algorithmic_bytes()
        kernels.append({"call": d.call.name, "us": round(ms * 1e3, 2), "GBps": round(b / (ms / 1e3) / 1e9, 1),
                        "frac_of_measured_peak": round(b / (ms / 1e3) / 1e9 / peak, 4),
                        "tokens_per_s": round(d.call.T / (ms / 1e3), 1), "bytes": b, "launches_per_step": len(idx)})
    value = aggregate_rate(step_bytes, steps, world, t["elapsed_ms"])
    return {
        "value": round(value, 3), "ms_per_step": round(t["elapsed_ms"] / steps, 5),
        "frac_of_measured_peak": round(value / world / peak, 4),
        "tokens_per_s": round(work.tokens() * steps * world / (t["elapsed_ms"] / 1e3), 1),
        "gpu_launches": int(t["launches"]),
        "roofline": {"bound": "hbm", "kernel": dcall.call.name, "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes": dom_bytes, "us_per_launch": round(t["dom_ms"] * 1e3, 2),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "frac_of_nominal_8TBps": round(achieved / 8000.0, 4)},
        "kernels": kernels,
        "clocks": t["clocks"],
    }


def measure_configs(torch, mbd, args, dev, props, headline: Dict, head_work: wl.Workload) -> Dict:
    """One entry per named workload configuration, each with its own CUDA-event timing and clock samples:
    the Qwen2.5-1.5B 16-token layer (latency, L2 flushed before every step, and back to back), the
    Qwen2.5-1.5B decode sweep (28 layers per step as one program launch: us per layer, GB/s, tokens/s), the
    Llama-3-8B prefill and Llama-3-70B FP8 steps (GB/s, fraction of the measured copy, the dominant kernel's
    roofline, tokens/s) and the headline step."""
    peak, _ = measured_peak()
    lib = mbd.get_lib()
    l2 = int(getattr(props, "L2_cache_size", 0)) or 126 * 2 ** 20
    flush = torch.empty(4 * l2, dtype=torch.uint8, device=dev)
    out: Dict[str, Dict] = {}
    steps = args.config_steps

    # Qwen2.5-1.5B, 16 tokens: latency-bound (the step's 1 MB stays in L2 when repeated)
    work = wl.qwen_t16()
    dcalls, stream = prepare_step(torch, mbd, args, work, 0, dev, props)
    with torch.cuda.stream(stream):           # back to back, no events between the steps
        for _ in range(args.warmup):
            for d in dcalls:
                d.launch()
    torch.cuda.synchronize(dev)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        w0.record(stream)
        for _ in range(steps):
            for d in dcalls:
                d.launch()
        w1.record(stream)
    torch.cuda.synchronize(dev)
    cold = []
    clock = ClockSampler(str(getattr(props, "uuid", "")))
    clock.start()
    t0 = time.time()
    for _ in range(steps):
        with torch.cuda.stream(stream):
            flush.fill_(1)                     # evicts the step's buffers from L2 (outside the events)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for d in dcalls:
                d.launch()
            b.record(stream)
        cold.append((a, b))
    torch.cuda.synchronize(dev)
    t1 = time.time()
    cold_us = statistics.median(a.elapsed_time(b) for a, b in cold) * 1e3
    B = work.algorithmic_bytes()
    warm_us = w0.elapsed_time(w1) / steps * 1e3
    out["qwen2.5-1.5b_t16"] = {
        "calls": [c.name for c in work.calls], "launch_units": [d.call.name for d in dcalls],
        "bytes_per_step": B, "us_per_step_l2_flushed": round(cold_us, 2), "us_per_step_back_to_back": round(warm_us, 2),
        "GBps_l2_flushed": round(B / cold_us / 1e3, 1), "tokens_per_s_l2_flushed": round(16 / cold_us * 1e6, 1),
        "basis": f"median of {steps} steps, each between CUDA events after an L2 flush (an event pair adds a few "
                 f"microseconds to a launch this short); and {steps} steps back to back between one event pair",
        "clocks": clock.stop(t0, t1)}
    del dcalls
    torch.cuda.empty_cache()

    # Qwen2.5-1.5B decode sweep: 28 layers of (add+RMSNorm, add+RMSNorm, SwiGLU), one program launch per step
    rows = {}
    clock = ClockSampler(str(getattr(props, "uuid", "")))
    clock.start()
    t0 = time.time()
    for w in wl.qwen_decode_sweep():
        T = w.calls[0].T
        dc = build_device_calls(torch, mbd, w, args.seed, 0, dev)
        st = torch.cuda.Stream(device=dev)
        h = int(st.cuda_stream)
        plans = [mbd.program_plan_build([d.op() for d in dc][i:i + mbd.MAX_PROGRAM_OPS])
                 for i in range(0, len(dc), mbd.MAX_PROGRAM_OPS)]
        scheds = [torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device=dev) for _ in plans]
        for p_, sc in zip(plans, scheds):
            p_.upload(sc, h)
        pairs = [(ctypes.addressof(p_.buf), sc.data_ptr()) for p_, sc in zip(plans, scheds)]

        def launch():
            for pp, sp in pairs:
                rc = lib.mbd_program_plan_launch_uploaded(pp, sp, h)
                if rc != 0:
                    raise RuntimeError(lib.mbd_status_string(rc).decode())

        with torch.cuda.stream(st):
            for _ in range(args.warmup):
                launch()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(st):
            e0.record(st)
            for _ in range(steps):
                launch()
            e1.record(st)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / steps
        Bw = w.algorithmic_bytes()
        rows[str(T)] = {"us_per_layer": round(ms * 1e3 / w.layers, 3), "us_per_step": round(ms * 1e3, 2),
                        "GBps": round(Bw / (ms / 1e3) / 1e9, 1), "frac_of_measured_peak": round(Bw / (ms / 1e3) / 1e9 / peak, 4),
                        "tokens_per_s": round(T / (ms / 1e3), 1), "bytes_per_step": Bw, "launches_per_step": len(plans)}
        del dc, plans, scheds
        torch.cuda.empty_cache()
    t1 = time.time()
    out["qwen2.5-1.5b_decode_sweep"] = {
        "per_tokens": rows, "layers": 28, "launch": "one program launch per step (plan built once, schedule uploaded once)",
        "basis": f"{steps} steps back to back between CUDA events per token count; below ~64 tokens the step's "
                 "buffers stay in L2 between steps, so these are latencies", "clocks": clock.stop(t0, t1)}

    # bandwidth-bound configurations
    for work in (wl.llama3_8b_prefill(), wl.llama3_70b_fp8()):
        dcalls, stream = prepare_step(torch, mbd, args, work, 0, dev, props)
        t = time_step(torch, mbd, dcalls, stream, steps, args.warmup, dev, props, 0, 1)
        e = step_summary(work, dcalls, t, steps, 1)
        e.update({"calls": [c.name for c in work.calls], "bytes_per_step": work.algorithmic_bytes(),
                  "l2": "inputs larger than L2, no flush"})
        out[work.key] = e
        del dcalls
        torch.cuda.empty_cache()

    out[head_work.key] = {"see": "the line's headline (value, roofline, kernels, clocks)",
                          "value": headline["value"], "frac_of_measured_peak": headline["frac_of_measured_peak"],
                          "roofline_frac": headline["roofline"]["frac"], "tokens_per_s": headline["tokens_per_s"]}
    return out


def run_mine(args, work: wl.Workload, rank: int, world: int, local_rank: int) -> Optional[Dict]:
    import torch
    import memory_bound_decoder_gb300 as mbd
    from memory_bound_decoder_gb300 import build as mbd_build
    if rank == 0:
        mbd_build.build()
    if world > 1:
        torch.distributed.barrier()
    mbd.get_lib()
    dev = torch.device("cuda", local_rank)
    tuning = resolve_tuning(args.tuning, torch, dev)
    if tuning:
        mbd.tuning_load(tuning)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2_bytes = int(getattr(props, "L2_cache_size", 0)) or 126 * 2 ** 20

    dcalls, stream = prepare_step(torch, mbd, args, work, rank, dev, props)
    step_bytes = work.algorithmic_bytes()
    t = time_step(torch, mbd, dcalls, stream, args.steps, args.warmup, dev, props, rank, world)

    # end-to-end leg through the same public entry points: host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, dcalls, stream, dev, min(args.steps, args.e2e_steps), step_bytes, world)

    if rank != 0:
        return None
    summ = step_summary(work, dcalls, t, args.steps, world)
    tuning_desc = f"tuning table {os.path.relpath(tuning, ROOT)}" if tuning else "built-in rules"
    result = {
        "metric": METRIC, "value": summ["value"],
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": summ["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": work.key, "description": work.description,
                   "calls": [c.name for c in work.calls], "layers": work.layers, "seed": args.seed,
                   "bytes_per_step": step_bytes, "tokens_per_step": work.tokens(),
                   "io": "bf16 inputs; bf16 or E4M3 outputs; fp32 arithmetic",
                   "l2": f"inputs larger than L2: {step_bytes / 2 ** 20:.0f} MiB of distinct buffers per step "
                         f"vs {l2_bytes / 2 ** 20:.0f} MiB L2, no flush",
                   "parallelism": f"replicas x{world} (rows are independent; no collective)",
                   "launch_shapes": tuning_desc,
                   "launch_units": [d.call.name for d in dcalls],
                   "small_calls": ("the calls with fewer tokens than SMs run as program launches (bf16 and FP8 "
                                   "together while their rows fit one per SM, NVFP4 apart; --no-programs: one "
                                   "launch per call)"
                                   if any(isinstance(d, (ProgramGroup, ProgramBatchGroup)) for d in dcalls)
                                   else "one launch per call"),
                   "batches": ("the calls of at least one row per SM other than the largest run as one batch "
                               "of overlapping single-call launches (mbd_run_independent; --no-batches: one launch "
                               "unit per call)" + ("; the program launch of the small calls opens that batch "
                                                   "(mbd_run_independent_with_program)"
                                                   if any(isinstance(d, ProgramBatchGroup) for d in dcalls) else "")
                               if any(isinstance(d, (BatchGroup, ProgramBatchGroup)) for d in dcalls) else "none"),
                   "roofline_events": "CUDA events around the roofline kernel's launch in every timed step (they "
                                      "break its overlap with the launches beside it)",
                   "kernels_breakdown": "each launch unit alone between CUDA events after a read of twice the L2 "
                                        "size (no dirty lines of an earlier kernel left in L2 for it to write back), "
                                        "untimed pass before the timed region"},
        "frac_of_measured_peak": summ["frac_of_measured_peak"],
        "tokens_per_s": summ["tokens_per_s"],
        "gpu_launches": summ["gpu_launches"],
        "roofline": summ["roofline"],
        "kernels": summ["kernels"],
        "clocks": summ["clocks"],
        "e2e": e2e,
    }
    if world == 1 and not args.no_configs and work.key == DEFAULT_WORKLOAD:
        del dcalls
        torch.cuda.empty_cache()
        result["configs"] = measure_configs(torch, mbd, args, dev, props, result, work)
    return result


# ------------------------------------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="one of: " + ", ".join(list(workloads_by_key()) + ["qwen2.5-1.5b_decode_sweep"]))
    ap.add_argument("--calls", default="", help="comma-separated call names: run only these calls of the workload")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration block (default workload only: the Qwen2.5-1.5B 16-token layer and "
                         "decode sweep, Llama-3-8B prefill and Llama-3-70B FP8 steps, each timed on its own)")
    ap.add_argument("--config-steps", type=int, default=200, help="timed steps per configuration of that block")
    ap.add_argument("--no-batches", action="store_true",
                    help="no batches: every call of at least one row per SM of a one-layer step gets a launch unit of "
                         "its own (default: all but the largest run as one mbd_run_independent batch of overlapping "
                         "launches)")
    ap.add_argument("--no-programs", action="store_true",
                    help="launch every call on its own (default: the calls with fewer tokens than SMs of a one-layer "
                         "step run as program launches: bf16 and FP8 ones together while their rows fit one per SM)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=1.0, help="target wall time of the oracle sample")
    ap.add_argument("--decode-table", action="store_true",
                    help="time the Qwen decode sweep as per-op calls, a CUDA graph and programs (one JSON line)")
    ap.add_argument("--decode-tokens", default="", help="token counts of --decode-table (default 1,2,4,8,32,64,128,256)")
    ap.add_argument("--tuning", default="auto",
                    help="launch-shape table: a tuning file, 'auto' (the packaged table of this GPU model when one "
                         "exists, else the built-in rules) or 'none' (the built-in rules)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.decode_table and args.impl == "mine":
        if rank == 0:
            print(json.dumps(run_decode_table(args)), flush=True)
        return 0
    work = decode_sweep_workload() if args.workload == "qwen2.5-1.5b_decode_sweep" else workloads_by_key()[args.workload]
    if args.calls:
        keep = set(args.calls.split(","))
        sel = tuple(c for c in work.calls if c.name in keep)
        if not sel:
            ap.error(f"--calls matched nothing in {work.key}: " + ", ".join(c.name for c in work.calls))
        work = wl.Workload(work.key + "[" + args.calls + "]", work.description + " (subset)", sel, work.layers)

    if args.impl == "reference":
        if rank != 0:
            return 0
        threads = os.cpu_count() or 1
        total_steps = args.steps + args.warmup
        per_step = max(0.02, min(2.0, 150.0 / total_steps))
        frac = calibrate_fraction(work, threads, per_step)
        s = OracleSample(work, frac, threads, seed=args.seed)
        for _ in range(args.warmup):
            s.run()
        t = time.perf_counter()
        for _ in range(args.steps):
            s.run()
        dt = time.perf_counter() - t
        value = round(s.bytes * args.steps / dt / 1e9, 5)
        out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
               "data": "synthetic",
               "config": {"workload": work.key, "description": work.description,
                          "calls": [c.name for c in work.calls], "layers": work.layers, "seed": args.seed},
               "tokens_per_s": round(s.tokens * args.steps / dt, 2),
               "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": s.describe()},
               "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(out), flush=True)
        return 0

    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        res = run_mine(args, work, rank, world, local_rank)
        if rank == 0 and res is not None:
            if not args.no_cpu_baseline and world == 1:
                res["cpu_baseline"] = cpu_baseline(work, args.cpu_seconds)
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
