"""Seeded synthetic inputs for the decoder-layer fusions, shared by the tests, the bench and the oracle.

This module holds no arithmetic of the method itself: it only draws random numbers, rounds them to the
bf16 input type and describes the workload shapes. Both sides (the CUDA path and the CPU oracle) receive
the same bf16 bit patterns from here.

Recipe (counter-style streams: one PCG64 stream per block of ROWS_PER_BLOCK rows of each tensor, keyed by
(seed, tensor id, salt, block index), so the values do not depend on how many threads fill the tensor and
any subset of rows can be regenerated on its own):
  * activations x, residual r, gate_up: float32 draws from N(0, sigma^2); optionally each element is
    multiplied, independently with probability p, by an outlier factor k;
  * RMSNorm weight: 1 + 0.1 * N(0, 1);
  * every float32 draw is rounded to bf16 with round-to-nearest-even on its bit pattern.

The shapes stand in for the models the source pages name (Qwen2.5-1.5B, Llama-3-8B/70B, Llama-3.1-405B):
no dataset or trained weight is used.
"""
from __future__ import annotations

import os
from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np

# tensor ids for the per-tensor stream key
_TID = {"x": 1, "residual": 2, "weight": 3, "gate_up": 4}


ROWS_PER_BLOCK = 8
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import concurrent.futures as cf
        _POOL = cf.ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = u + lsb
    r += np.uint32(0x7FFF)          # finite patterns stay below 2^32 after the increment
    r >>= np.uint32(16)
    out = r.astype(np.uint16)
    nan = np.isnan(np.asarray(a, np.float32))
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _block_rng(seed: int, tensor: str, salt: int, block: int) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=int(seed), spawn_key=(_TID[tensor], int(salt), int(block)))
    return np.random.Generator(np.random.PCG64(ss))


def _fill_block(out2d, seed, tensor, salt, block, sigma, outlier_p, outlier_k, rows_lo, rows_hi):
    g = _block_rng(seed, tensor, salt, block)
    shape = (rows_hi - rows_lo, out2d.shape[1])
    v = g.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        v *= np.float32(sigma)
    if outlier_p > 0.0:
        m = g.random(size=shape, dtype=np.float32) < np.float32(outlier_p)
        v[m] *= np.float32(outlier_k)
    out2d[rows_lo:rows_hi] = f32_to_bf16_bits(v)


def normal_bf16(shape: Tuple[int, ...], seed: int, tensor: str, sigma: float = 1.0,
                outlier_p: float = 0.0, outlier_k: float = 1.0, salt: int = 0,
                rows: Optional[np.ndarray] = None) -> np.ndarray:
    """bf16 bits of N(0, sigma^2) draws, each element independently scaled by outlier_k with prob. outlier_p.
    With `rows`, only those rows of the full tensor are returned (identical to slicing the full tensor)."""
    T, W = (1, shape[0]) if len(shape) == 1 else shape
    full = np.empty((T, W), np.uint16)
    blocks = range((T + ROWS_PER_BLOCK - 1) // ROWS_PER_BLOCK)
    if rows is not None:
        rows = np.asarray(rows, np.int64)
        blocks = sorted({int(r) // ROWS_PER_BLOCK for r in rows})
    jobs = [(full, seed, tensor, salt, b, sigma, outlier_p, outlier_k, b * ROWS_PER_BLOCK,
             min(T, (b + 1) * ROWS_PER_BLOCK)) for b in blocks]
    if len(jobs) <= 2:
        for j in jobs:
            _fill_block(*j)
    else:
        list(_pool().map(lambda j: _fill_block(*j), jobs))
    if rows is not None:
        return full[rows]
    return full.reshape(shape)


def weight_bf16(hidden: int, seed: int, salt: int = 0) -> np.ndarray:
    """bf16 bits of an RMSNorm weight 1 + 0.1 * N(0, 1)."""
    g = _block_rng(seed, "weight", salt, 0)
    v = np.float32(1.0) + np.float32(0.1) * g.standard_normal(size=(hidden,), dtype=np.float32)
    return f32_to_bf16_bits(v)


@dataclass(frozen=True)
class Dist:
    sigma: float = 1.0
    outlier_p: float = 0.0
    outlier_k: float = 1.0


@dataclass
class NormInputs:
    x: np.ndarray          # [T, H] uint16 (bf16 bits)
    residual: np.ndarray   # [T, H] uint16
    weight: np.ndarray     # [H] uint16
    eps: float


@dataclass
class SwigluInputs:
    gate_up: np.ndarray    # [T, 2I] uint16: gate = columns 0..I-1, up = columns I..2I-1


def make_norm_inputs(T: int, H: int, seed: int, dist: Dist, eps: float, salt: int = 0,
                     rows: Optional[np.ndarray] = None) -> NormInputs:
    """Inputs of one fused add+RMSNorm call; with `rows`, only those rows of x and residual."""
    x = normal_bf16((T, H), seed, "x", dist.sigma, dist.outlier_p, dist.outlier_k, salt, rows)
    r = normal_bf16((T, H), seed, "residual", dist.sigma, dist.outlier_p, dist.outlier_k, salt, rows)
    w = weight_bf16(H, seed, salt)
    return NormInputs(x, r, w, float(eps))


def make_swiglu_inputs(T: int, I: int, seed: int, dist: Dist, salt: int = 0,
                       rows: Optional[np.ndarray] = None) -> SwigluInputs:
    """Inputs of one SwiGLU call; with `rows`, only those rows of gate_up."""
    return SwigluInputs(normal_bf16((T, 2 * I), seed, "gate_up", dist.sigma, dist.outlier_p,
                                    dist.outlier_k, salt, rows))


# --------------------------------------------------------------------------------------------------
# Workload descriptions. A "call" is one invocation of one entry point on one shape.
# kind: "add_rmsnorm" | "add_rmsnorm_q8" | "add_rmsnorm_nvfp4" | "swiglu" | "swiglu_q8" | "swiglu_nvfp4" |
# "allreduce_rmsnorm[_q8]"; mode: None | "static" | "dynamic" (FP8 only). static_scale is the FP8 static scale
# or the NVFP4 per-tensor scale.
# --------------------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Call:
    kind: str                  # add_rmsnorm[_q8|_nvfp4] | allreduce_rmsnorm[_q8] | swiglu[_q8|_nvfp4]
    T: int
    width: int                 # H for the norm, I for SwiGLU
    dist: Dist
    eps: float = 1e-6
    mode: Optional[str] = None
    static_scale: float = 0.05
    partials: int = 0          # allreduce_rmsnorm: number of partial activations

    @property
    def is_norm(self) -> bool:
        return self.kind.startswith("add") or self.kind.startswith("allreduce")

    @property
    def name(self) -> str:
        m = f"_{self.mode}" if self.mode else ""
        k = f"_k{self.partials}" if self.partials else ""
        w = "H" if self.is_norm else "I"
        return f"{self.kind}{m}{k}_T{self.T}_{w}{self.width}"

    def algorithmic_bytes(self) -> int:
        """Minimum HBM bytes of one call: every input read once, every output written once."""
        T, W = self.T, self.width
        if self.kind == "add_rmsnorm":
            return 8 * T * W + 2 * W
        if self.kind == "add_rmsnorm_q8":
            return 7 * T * W + 2 * W + (4 * T if self.mode == "dynamic" else 4)
        if self.kind == "allreduce_rmsnorm":       # k partials + residual in, out + residual out
            return (2 * self.partials + 6) * T * W + 2 * W
        if self.kind == "allreduce_rmsnorm_q8":
            return (2 * self.partials + 5) * T * W + 2 * W + (4 * T if self.mode == "dynamic" else 4)
        if self.kind == "add_rmsnorm_nvfp4":     # codes W/2 + block scales W/16 bytes per row, S read
            return 6 * T * W + T * W // 2 + T * W // 16 + 2 * W + 4
        if self.kind == "swiglu":
            return 6 * T * W
        if self.kind == "swiglu_q8":
            return 5 * T * W + (4 * T if self.mode == "dynamic" else 4)
        if self.kind == "swiglu_nvfp4":
            return 4 * T * W + T * W // 2 + T * W // 16 + 4
        raise ValueError(self.kind)


N01 = Dist()
C3_ACT = Dist(1.0, 0.01, 50.0)
C3_GU = Dist(float(np.sqrt(2.0)))
C5_ACT = Dist(1.0, 0.001, 100.0)


def _all_four(T: int, H: int, I: int, dist: Dist, eps: float) -> List[Call]:
    return [Call("add_rmsnorm", T, H, dist, eps), Call("add_rmsnorm_q8", T, H, dist, eps, "static"),
            Call("swiglu", T, I, dist), Call("swiglu_q8", T, I, dist, mode="dynamic")]


@dataclass(frozen=True)
class Workload:
    key: str
    description: str
    calls: Tuple[Call, ...]
    layers: int = 1            # back-to-back repeats with distinct buffers (decode sweep)

    def algorithmic_bytes(self) -> int:
        return self.layers * sum(c.algorithmic_bytes() for c in self.calls)

    def tokens(self) -> int:
        """Tokens pushed through the path per step: each distinct token count is one batch of rows
        (a decode step over all layers still moves its T tokens once)."""
        return sum(sorted({c.T for c in self.calls}))


def qwen_t16() -> Workload:
    return Workload("qwen2.5-1.5b_t16", "Qwen2.5-1.5B-shaped layer, 16 tokens",
                    (Call("add_rmsnorm", 16, 1536, N01, 1e-6), Call("swiglu", 16, 8960, N01)))


def qwen_decode_sweep(tokens: Tuple[int, ...] = (1, 2, 4, 8, 32, 64, 128, 256)) -> List[Workload]:
    out = []
    for T in tokens:
        calls = (Call("add_rmsnorm", T, 1536, N01, 1e-6), Call("add_rmsnorm", T, 1536, N01, 1e-6),
                 Call("swiglu", T, 8960, N01))
        out.append(Workload(f"qwen2.5-1.5b_decode_T{T}", f"Qwen2.5-1.5B decode, {T} tokens, 28 layers",
                            calls, layers=28))
    return out


def llama3_8b_prefill() -> Workload:
    return Workload("llama3-8b_prefill_T8192", "Llama-3-8B-shaped prefill, 8192 tokens",
                    (Call("add_rmsnorm", 8192, 4096, C3_ACT, 1e-5), Call("swiglu", 8192, 14336, C3_GU)))


def llama3_70b_fp8() -> Workload:
    return Workload("llama3-70b_fp8_T4096", "Llama-3-70B-shaped FP8 path, 4096 tokens",
                    (Call("add_rmsnorm_q8", 4096, 8192, N01, 1e-5, "static"),
                     Call("swiglu_q8", 4096, 28672, N01, mode="dynamic")))


def llama31_405b_fp8_ragged() -> Workload:
    calls = [Call("add_rmsnorm_q8", 2048, 16384, C5_ACT, 1e-5, "static"),
             Call("swiglu_q8", 2048, 53248, C5_ACT, mode="dynamic")]
    for T in (1, 3, 17, 1000):
        calls += _all_four(T, 5120, 13824, C5_ACT, 1e-5)
    return Workload("llama3.1-405b_fp8_T2048+ragged", "Llama-3.1-405B-shaped FP8 path (2048 tokens) plus "
                    "ragged 5120/13824 shapes at 1, 3, 17, 1000 tokens", tuple(calls))


# Per-tensor NVFP4 scales of the 405B-shaped C5 activations, calibrated as the tensor's amax / (6 * 448)
# (amax ~82 for the normalised rows, ~461 for the SwiGLU output at 2048 tokens): block scales then stay
# within E4M3's normal range.
NVFP4_SCALE_NORM_C5 = 0.03
NVFP4_SCALE_SWIGLU_C5 = 0.17


def llama31_405b_nvfp4() -> Workload:
    """The 405B-shaped prefill batch with the Blackwell 4-bit epilogue on both fusions."""
    return Workload("llama3.1-405b_nvfp4_T2048", "Llama-3.1-405B-shaped NVFP4 path, 2048 tokens",
                    (Call("add_rmsnorm_nvfp4", 2048, 16384, C5_ACT, 1e-5, static_scale=NVFP4_SCALE_NORM_C5),
                     Call("swiglu_nvfp4", 2048, 53248, C5_ACT, static_scale=NVFP4_SCALE_SWIGLU_C5)))


@dataclass
class PartialNormInputs:
    partials: List[np.ndarray]   # k x [T, H] uint16
    residual: np.ndarray
    weight: np.ndarray
    eps: float


def make_partial_norm_inputs(k: int, T: int, H: int, seed: int, dist: Dist, eps: float, salt: int = 0,
                             rows: Optional[np.ndarray] = None) -> PartialNormInputs:
    """k partial activations (independent streams), a residual and a weight."""
    ps = [normal_bf16((T, H), seed, "x", dist.sigma, dist.outlier_p, dist.outlier_k, salt * 16 + 1 + j, rows)
          for j in range(k)]
    r = normal_bf16((T, H), seed, "residual", dist.sigma, dist.outlier_p, dist.outlier_k, salt, rows)
    return PartialNormInputs(ps, r, weight_bf16(H, seed, salt), float(eps))


def llama31_405b_tp8_allreduce_norm() -> Workload:
    """The all-reduce half of AllReduce + RMSNorm for a Llama-3.1-405B-shaped layer split over 8
    tensor-parallel ranks: 8 partial activations per token reduced, added to the residual and normalised,
    to E4M3 with the static scale and to bf16."""
    return Workload("llama3.1-405b_tp8_allreduce_norm_T2048", "Llama-3.1-405B-shaped all-reduce half + add + "
                    "RMSNorm, 8 partials, 2048 tokens",
                    (Call("allreduce_rmsnorm_q8", 2048, 16384, C5_ACT, 1e-5, "static", partials=8),
                     Call("allreduce_rmsnorm", 2048, 16384, C5_ACT, 1e-5, partials=8)))


def inputs_for(call: Call, seed: int = 0, salt: int = 0, rows: Optional[np.ndarray] = None):
    """Seeded inputs of one call (NormInputs, PartialNormInputs or SwigluInputs), optionally only some rows."""
    if call.kind.startswith("allreduce"):
        return make_partial_norm_inputs(call.partials, call.T, call.width, seed, call.dist, call.eps, salt, rows)
    if call.kind.startswith("add"):
        return make_norm_inputs(call.T, call.width, seed, call.dist, call.eps, salt, rows)
    return make_swiglu_inputs(call.T, call.width, seed, call.dist, salt, rows)
