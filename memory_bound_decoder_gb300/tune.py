"""Launch-shape tuner: times candidate launch shapes of the single-call entry points on this GPU and writes a
shape-bucket table (mbd_tuning_entry) that memory_bound_decoder_gb300.tuning_load() installs.

The pages' form of this ("TensorRT-LLM: Compiling Inference Engines Ahead of Time", "Auto-tuning, measured"):
time every kernel variant per shape bucket once, keep the fastest in a cache file, reload it at startup.
Here the variants are launch shapes: CTAs per row (a thread-block cluster when the row is reduced), 16-byte
vectors per thread and threads per CTA. For every (entry point, FP8 mode, width) and every token count of a
grid the tuner times the built-in rules' shape and every legal candidate through the library's own tuning
hook (a one-entry table per candidate), keeps the fastest, and turns the token grid into buckets split at
the geometric midpoints between the tuned counts. Inputs rotate through enough buffer sets to exceed L2, so
each launch reads from HBM as in a model step; each timing replays the launches from a CUDA graph, so it is
device time, not the host's launch overhead.

    python -m memory_bound_decoder_gb300.tune --out tuning.json [--quick] [--shapes kind:mode:width,...]
"""
from __future__ import annotations

import argparse
import json
import math
import sys
import time

import memory_bound_decoder_gb300 as mbd

# (entry point, FP8 mode, width): the model shapes of the bench workloads (Qwen2.5-1.5B, Llama-3-8B,
# Llama-3-70B FP8, Llama-3.1-405B FP8 with its ragged tails, and the NVFP4 path).
DEFAULT_SHAPES = [
    ("add_rmsnorm", None, 1536), ("swiglu", None, 8960),
    ("add_rmsnorm", None, 4096), ("swiglu", None, 14336),
    ("add_rmsnorm_quant_fp8", "static", 8192), ("swiglu_quant_fp8", "dynamic", 28672),
    ("add_rmsnorm_quant_fp8", "static", 16384), ("swiglu_quant_fp8", "dynamic", 53248),
    ("add_rmsnorm", None, 5120), ("add_rmsnorm_quant_fp8", "static", 5120),
    ("swiglu", None, 13824), ("swiglu_quant_fp8", "dynamic", 13824),
    ("add_rmsnorm_quant_nvfp4", None, 16384), ("swiglu_quant_nvfp4", None, 53248),
]
DEFAULT_TOKENS = (1, 4, 16, 64, 256, 1024, 2048, 4096, 8192)
MAX_ELEMENTS = 1 << 28          # T x width cap per shape (keeps a buffer set near 1 GB at most)
ROTATE_BYTES = 512 << 20        # buffer sets rotated per launch: at least this much (4x L2)
CLUSTER_SIZES = range(1, 9)
STREAM_CTAS = (1, 2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64)


def cdiv(a, b):
    return -(-a // b)


def candidates(kind, mode, width):
    """Legal (ctas_per_row, vectors_per_thread, threads) shapes, deduplicated by the slices they give."""
    nvec = width // 8
    reduces = kind.startswith("add") or (kind == "swiglu_quant_fp8" and mode == "dynamic")
    pairs = kind.endswith("nvfp4")
    seen, out = set(), []
    for c in (CLUSTER_SIZES if reduces else STREAM_CTAS):
        slice_ = cdiv(nvec, c)
        if pairs and slice_ % 2:
            slice_ += 1
        real_c = cdiv(nvec, slice_)
        for v in (1, 2, 4, 8):
            th = cdiv(cdiv(slice_, v), 32) * 32
            if th > 512 or (real_c, slice_, v, th) in seen:
                continue
            seen.add((real_c, slice_, v, th))
            out.append((c, v, th))
    return out


class Call:
    """Device buffers (rotated) and one launch of an entry point on T x width."""

    def __init__(self, torch, kind, mode, T, width):
        self.kind, self.mode, self.T, self.W = kind, mode, T, width
        dev = torch.device("cuda")
        bf = torch.bfloat16
        if kind.startswith("add"):
            per = 8 * T * width
        else:
            per = 6 * T * width
        self.nsets = max(1, min(8, cdiv(ROTATE_BYTES, per)))
        self.sets = []
        for _ in range(self.nsets):
            if kind.startswith("add"):
                x = torch.randn(T, width, device=dev).to(bf)
                r = torch.randn(T, width, device=dev).to(bf)
                w = (1 + 0.1 * torch.randn(width, device=dev)).to(bf)
                self.sets.append((x, r, w))
            else:
                self.sets.append((torch.randn(T, 2 * width, device=dev).to(bf),))
        if kind in ("add_rmsnorm", "swiglu"):
            self.out = torch.empty(T, width, dtype=bf, device=dev)
        elif kind.endswith("fp8"):
            self.out = torch.empty(T, width, dtype=torch.uint8, device=dev)
        else:
            self.out = torch.empty(T, width // 2, dtype=torch.uint8, device=dev)
            self.sf = torch.empty(T, width // 16, dtype=torch.uint8, device=dev)
        n_scale = T if mode == "dynamic" else 1
        self.scale = torch.full((n_scale,), 0.03 if kind.startswith("add") else 0.17, device=dev)
        self.k = 0

    def launch(self):
        s = self.sets[self.k % self.nsets]
        self.k += 1
        T, W = self.T, self.W
        if self.kind == "add_rmsnorm":
            mbd.fused_add_rmsnorm(self.out, s[1], s[0], s[2], T, W, 1e-5)
        elif self.kind == "add_rmsnorm_quant_fp8":
            mbd.fused_add_rmsnorm_quant_fp8(self.out, s[1], s[0], s[2], T, W, 1e-5, self.mode, self.scale)
        elif self.kind == "add_rmsnorm_quant_nvfp4":
            mbd.fused_add_rmsnorm_quant_nvfp4(self.out, self.sf, s[1], s[0], s[2], T, W, 1e-5, self.scale)
        elif self.kind == "swiglu":
            mbd.swiglu(self.out, s[0], T, W)
        elif self.kind == "swiglu_quant_fp8":
            mbd.swiglu_quant_fp8(self.out, s[0], T, W, self.mode, self.scale)
        else:
            mbd.swiglu_quant_nvfp4(self.out, self.sf, s[0], T, W, self.scale)


def time_call(torch, call, reps):
    """Device time per launch: `reps` launches captured in a CUDA graph (with the table installed now) and
    replayed, so host launch overhead (several microseconds per call from Python) is not measured."""
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(reps):
            call.launch()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) * 1e3 / reps


def entry(kind, mode, t_lo, t_hi, width, shape):
    return {"kind": kind, "mode": mode, "tokens": [t_lo, t_hi], "width": [width, width],
            "ctas_per_row": shape[0], "vectors_per_thread": shape[1], "threads": shape[2]}


def tune(shapes, tokens, log=print):
    import torch
    table, evidence = [], []
    for kind, mode, width in shapes:
        rows = []
        for T in tokens:
            if T * width > MAX_ELEMENTS:
                continue
            call = Call(torch, kind, mode, T, width)
            mbd.tuning_set([])
            rules_shape = mbd.launch_shape(kind, mode, T, width)
            base = time_call(torch, call, 5)
            reps = max(5, min(400, int(2000 / max(base, 0.5))))   # about 2 ms of launches per timing
            rules_us = time_call(torch, call, reps)
            best_us, best = rules_us, rules_shape
            for cand in candidates(kind, mode, width):
                mbd.tuning_set([entry(kind, mode, T, T, width, cand)])
                got = mbd.launch_shape(kind, mode, T, width)
                if got[1:] != cand[1:]:
                    continue   # the shape does not fit this call: the rules would run instead
                us = time_call(torch, call, reps)
                if us < best_us:
                    best_us, best = us, got
            mbd.tuning_set([])
            rows.append((T, best, best_us, rules_shape, rules_us))
            log(f"[tune] {kind} {mode or ''} W={width} T={T}: rules {rules_shape} {rules_us:.2f} us, "
                f"best {best} {best_us:.2f} us ({100 * (rules_us / best_us - 1):+.1f}%)")
            del call
            torch.cuda.empty_cache()
        # buckets: each tuned count covers the token counts up to the geometric midpoints with its neighbours
        for i, (T, best, best_us, rules_shape, rules_us) in enumerate(rows):
            lo = 1 if i == 0 else math.floor(math.sqrt(rows[i - 1][0] * T)) + 1
            hi = (1 << 40) if i == len(rows) - 1 else math.floor(math.sqrt(T * rows[i + 1][0]))
            table.append(entry(kind, mode, lo, hi, width, best))
            evidence.append({"kind": kind, "mode": mode, "width": width, "tokens": T, "rules_shape": list(rules_shape),
                             "rules_us": round(rules_us, 3), "best_shape": list(best), "best_us": round(best_us, 3),
                             "gain_pct": round(100 * (rules_us / best_us - 1), 2)})
    return table, evidence


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--out", required=True, help="tuning file to write (JSON)")
    ap.add_argument("--quick", action="store_true", help="token counts 1, 64, 2048 only")
    ap.add_argument("--shapes", default="", help="kind:mode:width,... (default: the bench workloads' shapes)")
    ap.add_argument("--tokens", default="", help="comma-separated token counts of the grid")
    a = ap.parse_args()
    import torch
    from memory_bound_decoder_gb300 import build
    build.build()
    mbd.get_lib()
    shapes = DEFAULT_SHAPES
    if a.shapes:
        shapes = []
        for spec in a.shapes.split(","):
            k, m, w = spec.split(":")
            shapes.append((k, m or None, int(w)))
    tokens = tuple(int(t) for t in a.tokens.split(",")) if a.tokens else ((1, 64, 2048) if a.quick else DEFAULT_TOKENS)
    t0 = time.time()
    table, evidence = tune(shapes, tokens, log=lambda *x: print(*x, file=sys.stderr, flush=True))
    props = torch.cuda.get_device_properties(0)
    meta = {"device": props.name, "sm": f"{props.major}.{props.minor}", "multiprocessors": props.multi_processor_count,
            "generated_by": "python -m memory_bound_decoder_gb300.tune", "seconds": round(time.time() - t0, 1),
            "tokens": list(tokens), "evidence": evidence}
    mbd.tuning_save(a.out, table, meta)
    print(json.dumps({"entries": len(table), "out": a.out, "seconds": meta["seconds"]}))


if __name__ == "__main__":
    main()
