"""Comparison rules between the CUDA path and the oracle, and helpers that run one entry point on the GPU
with guard bands around every output.

Tolerances (stated for this library's outputs):
  * bf16 outputs: |gpu - v| <= 2^-7 * |v| + 1e-3, v the oracle's exact fp64 value;
  * the updated residual: bit-exact (it is the bf16 rounding of an exact two-term sum);
  * E4M3 codes: equal, except at most 0.1% of the elements, each of which may differ by one code step
    (adjacent magnitude; +0 and -0 are the same code);
  * dynamic scales: within 1e-6 relative (zero exactly when the oracle's is zero).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

import workloads as wl

BF16_REL = 2.0 ** -7
BF16_ABS = 1e-3
CODE_BUDGET = 1e-3
SCALE_REL = 1e-6
CANARY = 0x5A


def check_bf16(gpu_bits: np.ndarray, v: np.ndarray, what: str = "") -> float:
    g = wl.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    err = np.abs(g - v)
    bound = BF16_REL * np.abs(v) + BF16_ABS
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} bf16 outputs out of tolerance; first at {tuple(i)}: "
                             f"gpu {g[tuple(i)]!r} exact {v[tuple(i)]!r}")
    return float((err / bound).max()) if err.size else 0.0


def signed_code_index(q: np.ndarray) -> np.ndarray:
    mag = (q & 0x7F).astype(np.int32)
    return np.where(q & 0x80, -mag, mag)


def check_codes(gpu_q: np.ndarray, ref_q: np.ndarray, what: str = "") -> float:
    assert gpu_q.shape == ref_q.shape
    if gpu_q.size == 0:
        return 0.0
    assert not ((gpu_q & 0x7F) == 0x7F).any(), f"{what}: NaN code produced"
    d = np.abs(signed_code_index(gpu_q) - signed_code_index(ref_q))
    assert d.max() <= 1, f"{what}: a code differs by {int(d.max())} steps"
    frac = float((d != 0).mean())
    # the budget is a fraction of the elements; tiny tensors may carry one near-tie flip
    assert frac <= CODE_BUDGET or (d != 0).sum() <= 1, f"{what}: {frac:.2e} of codes differ (> {CODE_BUDGET})"
    return frac


def check_scales(gpu_s: np.ndarray, ref_s: np.ndarray, what: str = "") -> float:
    g = gpu_s.astype(np.float64)
    r = ref_s.astype(np.float64)
    err = np.abs(g - r)
    assert (err <= SCALE_REL * np.abs(r)).all(), f"{what}: scale rel err {float((err / np.maximum(np.abs(r), 1e-300)).max()):.3e}"
    return float((err / np.maximum(np.abs(r), 1e-300)).max()) if r.size else 0.0


# ------------------------------------------------------------------------------------------------ GPU side

class Guarded:
    """A device buffer of `n` elements of `dtype` with canary guard bands on both sides."""

    PAD_BYTES = 512

    def __init__(self, torch, n: int, dtype, device="cuda", fill: Optional[np.ndarray] = None):
        self.torch = torch
        self.itemsize = torch.empty(0, dtype=dtype).element_size()
        self.pad = self.PAD_BYTES // self.itemsize
        self.n = n
        self.raw = torch.full((n * self.itemsize + 2 * self.PAD_BYTES,), CANARY, dtype=torch.uint8, device=device)
        self.view = self.raw[self.PAD_BYTES:self.PAD_BYTES + n * self.itemsize].view(dtype)
        if fill is not None:
            self.view.copy_(torch.from_numpy(np.ascontiguousarray(fill).reshape(-1)).to(device))

    def check_guards(self, what: str = ""):
        head = self.raw[:self.PAD_BYTES]
        tail = self.raw[self.PAD_BYTES + self.n * self.itemsize:]
        assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), f"{what}: write outside the tensor"

    def numpy(self, dtype) -> np.ndarray:
        return self.view.cpu().numpy().view(dtype)


def dev_u16(torch, a: np.ndarray) -> "Guarded":
    return Guarded(torch, a.size, torch.int16, fill=a.view(np.int16))


def sample_rows(T: int, k: int, seed: int = 0) -> np.ndarray:
    """First, last and k-2 random rows (sorted, unique) of a T-row tensor."""
    if T <= k:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, T - 1), size=k - 2, replace=False)
    return np.unique(np.concatenate([[0, T - 1], mid]))
