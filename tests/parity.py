"""Comparison rules between the CUDA path and the oracle, and helpers that run one entry point on the GPU
with guard bands around every output.

Tolerances (stated for this library's outputs):
  * bf16 outputs: |gpu - v| <= 2^-7 * |v| + 1e-3, v the oracle's exact fp64 value;
  * the updated residual: bit-exact (it is the bf16 rounding of an exact two-term sum);
  * E4M3 codes: equal, except at most 0.1% of the elements (rounded down, so fewer than 1000 codes must
    all match), each of which may differ by one code step (adjacent magnitude; +0 and -0 are the same code);
  * dynamic scales: within 1e-6 relative (zero exactly when the oracle's is zero).
  * NVFP4: block scales (E4M3 codes) as E4M3 codes above; E2M1 codes of a block whose scale matches the
    oracle's: equal except at most 0.1% one step apart (+0 and -0 the same); a block whose scale is one step
    off: its codes equal the oracle's encoding of the exact values under the GPU's block scale, with the same
    budget.
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


def code_allowance(n: int) -> int:
    """How many of n codes may differ by one step: 0.1% of them, rounded down (a tensor of fewer than 1000
    codes must match exactly)."""
    return n // 1000          # CODE_BUDGET of n, rounded down


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
    n_diff = int((d != 0).sum())
    frac = n_diff / d.size
    assert n_diff <= code_allowance(d.size), f"{what}: {n_diff} of {d.size} codes differ (> {CODE_BUDGET:.1%})"
    return frac


def unpack_e2m1(q: np.ndarray) -> np.ndarray:
    """[rows, W/2] packed bytes -> [rows, W] 4-bit codes (element 2i from the low nibble of byte i)."""
    return np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[0], -1)


def check_nvfp4(q_g: np.ndarray, sf_g: np.ndarray, q_o: np.ndarray, sf_o: np.ndarray, v: np.ndarray,
                tensor_scale: float, orc, what: str = "") -> dict:
    """Compare the GPU's NVFP4 output with the oracle's (rule in the module docstring)."""
    sf_frac = check_codes(sf_g, sf_o, f"{what} block scales")
    cg, co = unpack_e2m1(q_g).astype(np.int32), unpack_e2m1(q_o).astype(np.int32)
    T, W = cg.shape
    same = np.repeat(sf_g == sf_o, 16, axis=1)
    # blocks whose scale differs: the oracle's codes under the GPU's scale (few elements; one call each)
    if (~same).any():
        S = float(np.float32(tensor_scale))
        for t, j in zip(*np.nonzero(~same)):
            sc = orc.e4m3_decode(int(sf_g[t, j // 16])) * S
            co[t, j] = 0 if sc == 0.0 else orc.e2m1_encode(float(v[t, j]) / sc)
    signed = lambda c: np.where(c & 8, -(c & 7), c & 7)
    d = np.abs(signed(cg) - signed(co))
    assert d.max(initial=0) <= 1, f"{what}: an E2M1 code differs by {int(d.max())} steps"
    # a zero keeps its sign: -0 (0x8) and +0 must match except where the step rule above allows
    bad_zero = ((cg & 7) == 0) & ((co & 7) == 0) & (cg != co)
    n_diff = int(((d != 0) | bad_zero).sum())
    frac = n_diff / d.size if d.size else 0.0
    assert n_diff <= code_allowance(d.size), f"{what}: {n_diff} of {d.size} E2M1 codes differ (> {CODE_BUDGET:.1%})"
    return {"sf_diff": sf_frac, "code_diff": frac, "blocks_rescaled": float((~same).mean()) / 1.0 if same.size else 0.0}


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
