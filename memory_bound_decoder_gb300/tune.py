"""Launch-shape tuner: times candidate launch shapes of the single-call entry points on this GPU and writes a
shape-bucket table (mbd_tuning_entry) that memory_bound_decoder_gb300.tuning_load() installs.

The pages' form of this ("TensorRT-LLM: Compiling Inference Engines Ahead of Time", "Auto-tuning, measured"):
time every kernel variant per shape bucket once, keep the fastest in a cache file, reload it at startup.
Here the variants are launch shapes: CTAs per row (a thread-block cluster when the row is reduced), 16-byte
vectors per thread and threads per CTA. For every (entry point, FP8 mode, width) and every token count of a
grid the tuner times the built-in rules' shape and every legal candidate through the library's own tuning
hook (a one-entry table per candidate), keeps the fastest, and turns the token grid into buckets split at
the geometric midpoints between the tuned counts. Inputs AND outputs rotate through buffer sets whose distinct
bytes per rotation exceed three times L2 where the launch count allows, so each launch reads and writes HBM as
in a model step (decode-sized calls stay L2-resident: a graph of a few hundred of them moves a few MB); each
timing replays the launches from a CUDA graph, so it is device time, not the host's launch overhead. Where the
launch count caps the rotation below three L2 sizes (decode-sized calls), a timing whose algorithmic bytes per
second exceed 1.05 x the measured HBM copy rate is taken as L2-served: recorded in the evidence and kept out of
the ranking. With the full rotation nothing can be served from L2, and such a rate (back-to-back launches of a
streaming kernel reach a few percent above a copy kernel's) is kept and marked.

    python -m memory_bound_decoder_gb300.tune --out tuning.json [--quick] [--shapes kind:mode:width,...]
        [--hbm-gbs GBPS]
"""
from __future__ import annotations

import argparse
import json
import math
import os
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
ROTATE_L2 = 3                   # distinct bytes of one rotation of the buffer sets: at least this many L2 sizes
MAX_SETS = 400                  # at most one set per launch of a timing (reps <= 400)
HBM_SLACK = 1.05                # timings above this multiple of the measured HBM rate are L2-served
FALLBACK_HBM_GBS = 6800.0       # without a measured copy rate
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


def algorithmic_bytes(kind, mode, T, width):
    """Minimum bytes one call moves: activations in and out once, the weight and a static scale once."""
    if kind == "add_rmsnorm":
        return 8 * T * width + 2 * width
    if kind == "add_rmsnorm_quant_fp8":
        return 7 * T * width + 2 * width + (4 * T if mode == "dynamic" else 4)
    if kind == "add_rmsnorm_quant_nvfp4":
        return 6 * T * width + T * width // 2 + T * width // 16 + 2 * width + 4
    if kind == "swiglu":
        return 6 * T * width
    if kind == "swiglu_quant_fp8":
        return 5 * T * width + (4 * T if mode == "dynamic" else 4)
    return 4 * T * width + T * width // 2 + T * width // 16 + 4


class Call:
    """Rotated buffer sets (inputs and outputs) and one launch of an entry point on T x width."""

    def __init__(self, torch, kind, mode, T, width, l2_bytes):
        self.kind, self.mode, self.T, self.W = kind, mode, T, width
        dev = torch.device("cuda")
        bf = torch.bfloat16
        self.bytes = algorithmic_bytes(kind, mode, T, width)
        self.nsets = max(1, min(MAX_SETS, cdiv(ROTATE_L2 * l2_bytes, self.bytes)))
        self.sets = []
        for _ in range(self.nsets):
            st = {}
            if kind.startswith("add"):
                st["x"] = torch.randn(T, width, device=dev).to(bf)
                st["r"] = torch.randn(T, width, device=dev).to(bf)
                st["w"] = (1 + 0.1 * torch.randn(width, device=dev)).to(bf)
            else:
                st["gu"] = torch.randn(T, 2 * width, device=dev).to(bf)
            if kind in ("add_rmsnorm", "swiglu"):
                st["out"] = torch.empty(T, width, dtype=bf, device=dev)
            elif kind.endswith("fp8"):
                st["out"] = torch.empty(T, width, dtype=torch.uint8, device=dev)
            else:
                st["out"] = torch.empty(T, width // 2, dtype=torch.uint8, device=dev)
                st["sf"] = torch.empty(T, width // 16, dtype=torch.uint8, device=dev)
            n_scale = T if mode == "dynamic" else 1
            st["scale"] = torch.full((n_scale,), 0.03 if kind.startswith("add") else 0.17, device=dev)
            self.sets.append(st)
        self.k = 0

    def launch(self):
        s = self.sets[self.k % self.nsets]
        self.k += 1
        T, W = self.T, self.W
        if self.kind == "add_rmsnorm":
            mbd.fused_add_rmsnorm(s["out"], s["r"], s["x"], s["w"], T, W, 1e-5)
        elif self.kind == "add_rmsnorm_quant_fp8":
            mbd.fused_add_rmsnorm_quant_fp8(s["out"], s["r"], s["x"], s["w"], T, W, 1e-5, self.mode, s["scale"])
        elif self.kind == "add_rmsnorm_quant_nvfp4":
            mbd.fused_add_rmsnorm_quant_nvfp4(s["out"], s["sf"], s["r"], s["x"], s["w"], T, W, 1e-5, s["scale"])
        elif self.kind == "swiglu":
            mbd.swiglu(s["out"], s["gu"], T, W)
        elif self.kind == "swiglu_quant_fp8":
            mbd.swiglu_quant_fp8(s["out"], s["gu"], T, W, self.mode, s["scale"])
        else:
            mbd.swiglu_quant_nvfp4(s["out"], s["sf"], s["gu"], T, W, s["scale"])


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


def measured_hbm_gbs() -> float:
    """The measured HBM copy rate (MEASURED_PEAKS.json at the repository root, hbm_gbs), else the fallback."""
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS


def rank(rules_shape, rules_us, timed, gbps, bound, full_rotation):
    """The best shape of one point: the rules' shape unless a candidate is faster. `timed`: (shape, us) of the
    candidates that fit the call; `gbps(us)` the algorithmic rate of a timing. A timing above `bound` counts as
    L2-served, and is kept out of the ranking, where the rotation is short (below ROTATE_L2 x L2); with the full
    rotation it is kept. Returns (best shape, best us, shapes timed above the bound)."""
    best_shape, best_us = rules_shape, rules_us
    above = [list(rules_shape)] if gbps(rules_us) > bound else []
    for shape, us in timed:
        if gbps(us) > bound:
            above.append(list(shape))
            if not full_rotation:
                continue
        if us < best_us:
            best_shape, best_us = shape, us
    return best_shape, best_us, above


def tune(shapes, tokens, hbm_gbs, log=print):
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0)) or 126 * 2 ** 20
    bound = HBM_SLACK * hbm_gbs
    table, evidence = [], []
    for kind, mode, width in shapes:
        rows = []
        for T in tokens:
            if T * width > MAX_ELEMENTS:
                continue
            call = Call(torch, kind, mode, T, width, l2)
            gbps = lambda us: call.bytes / us / 1e3
            full_rotation = call.nsets * call.bytes >= ROTATE_L2 * l2
            mbd.tuning_set([])
            rules_shape = mbd.launch_shape(kind, mode, T, width)
            base = time_call(torch, call, 5)
            reps = max(5, min(MAX_SETS, int(2000 / max(base, 0.5))))   # about 2 ms of launches per timing
            rules_us = time_call(torch, call, reps)
            timed = []
            for cand in candidates(kind, mode, width):
                mbd.tuning_set([entry(kind, mode, T, T, width, cand)])
                got = mbd.launch_shape(kind, mode, T, width)
                if got[1:] != cand[1:]:
                    continue   # the shape does not fit this call: the rules would run instead
                timed.append((got, time_call(torch, call, reps)))
            mbd.tuning_set([])
            best, best_us, above = rank(rules_shape, rules_us, timed, gbps, bound, full_rotation)
            rotation_mb = call.nsets * call.bytes / 2 ** 20
            rows.append((T, best, best_us, rules_shape, rules_us, rotation_mb, above, full_rotation))
            log(f"[tune] {kind} {mode or ''} W={width} T={T}: rules {rules_shape} {rules_us:.2f} us "
                f"({gbps(rules_us):.0f} GB/s), best {best} {best_us:.2f} us ({100 * (rules_us / best_us - 1):+.1f}%), "
                f"rotation {rotation_mb:.0f} MB, {len(above)} timings above the HBM bound")
            del call
            torch.cuda.empty_cache()
        # buckets: each tuned count covers the token counts up to the geometric midpoints with its neighbours
        for i, (T, best, best_us, rules_shape, rules_us, rotation_mb, above, full_rotation) in enumerate(rows):
            lo = 1 if i == 0 else math.floor(math.sqrt(rows[i - 1][0] * T)) + 1
            hi = (1 << 40) if i == len(rows) - 1 else math.floor(math.sqrt(T * rows[i + 1][0]))
            table.append(entry(kind, mode, lo, hi, width, best))
            B = algorithmic_bytes(kind, mode, T, width)
            evidence.append({"kind": kind, "mode": mode, "width": width, "tokens": T, "rules_shape": list(rules_shape),
                             "rules_us": round(rules_us, 3), "best_shape": list(best), "best_us": round(best_us, 3),
                             "gain_pct": round(100 * (rules_us / best_us - 1), 2), "bytes": B,
                             "best_GBps": round(B / best_us / 1e3, 1), "rotation_MB": round(rotation_mb, 1),
                             "full_rotation": full_rotation, "above_hbm_bound": above})
    return table, evidence


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--out", required=True, help="tuning file to write (JSON)")
    ap.add_argument("--quick", action="store_true", help="token counts 1, 64, 2048 only")
    ap.add_argument("--shapes", default="", help="kind:mode:width,... (default: the bench workloads' shapes)")
    ap.add_argument("--tokens", default="", help="comma-separated token counts of the grid")
    ap.add_argument("--hbm-gbs", type=float, default=0.0,
                    help="HBM copy rate for the L2 check (default: MEASURED_PEAKS.json hbm_gbs, else 6800)")
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
    hbm = a.hbm_gbs or measured_hbm_gbs()
    table, evidence = tune(shapes, tokens, hbm, log=lambda *x: print(*x, file=sys.stderr, flush=True))
    props = torch.cuda.get_device_properties(0)
    meta = {"device": props.name, "sm": f"{props.major}.{props.minor}", "multiprocessors": props.multi_processor_count,
            "generated_by": "python -m memory_bound_decoder_gb300.tune", "seconds": round(time.time() - t0, 1),
            "tokens": list(tokens), "hbm_gbs": hbm, "hbm_slack": HBM_SLACK, "rotate_l2": ROTATE_L2,
            "evidence": evidence}
    mbd.tuning_save(a.out, table, meta)
    print(json.dumps({"entries": len(table), "out": a.out, "seconds": meta["seconds"]}))


if __name__ == "__main__":
    main()
