"""Pins for the CPU oracle, independent of the oracle's own code.

Each check ties the oracle to something other than itself: library routines of PyTorch's CPU build
(bf16 and float8_e4m3fn casts, F.rms_norm and F.silu in float64), closed forms and invariants that follow
from the definitions on "TensorRT-LLM: Compiling Inference Engines Ahead of Time" ("Fusing operations,
measured") and the E4M3 format of "TensorRT-LLM" (architecture walkthrough, "Part V continued: Deep dive:
quantization co-designed with the hardware"), the golden fixtures under tests/golden/, and exact rational
arithmetic on tiny inputs. The combination is chosen so that a dropped term, a misplaced epsilon, a swapped
operand, a wrong index or a wrong rounding rule fails at least one test.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(line.split())
    return rows


def bf16_vals(bits):
    return wl.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


def torch_bf16_bits(f32):
    return torch.from_numpy(np.asarray(f32, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def torch_e4m3(f32):
    return torch.from_numpy(np.asarray(f32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ------------------------------------------------------------------------------------------------ bf16

def test_bf16_round_matches_torch_on_float32_values(orc):
    rng = np.random.default_rng(1)
    a = np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
                        (rng.random(5000).astype(np.float32) - 0.5) * np.float32(1e-38),   # subnormal range
                        np.ldexp(rng.random(3000), rng.integers(-140, 120, 3000)).astype(np.float32)])
    # exact ties: low 16 bits of the float32 pattern == 0x8000 with either parity of the kept part
    ties = (rng.integers(0x3000, 0x4F00, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    a = np.concatenate([a, ties])
    ref = torch_bf16_bits(a)
    got = np.array([orc.bf16_round(float(v)) for v in a], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_bf16_round_direct_from_double(orc):
    # 1 + 2^-8 is a tie -> even (1.0); 1 + 2^-8 + 2^-40 is above the tie -> 1 + 2^-7.
    # (A cast that goes through float32 first would give 1.0 here: rounding must be direct.)
    assert orc.bf16_round(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert orc.bf16_round(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie between odd 0x3F81 and even 0x3F82
    assert orc.bf16_round(2.0 ** -133) == 0x0001              # smallest subnormal
    assert orc.bf16_round(2.0 ** -134) == 0x0000              # tie with zero -> even
    assert orc.bf16_round(-(2.0 ** -134) * 1.5) == 0x8001
    assert orc.bf16_round(3.4e38) == 0x7F80                   # above max + half ulp -> inf
    assert orc.bf16_round(3.3895313892515355e38) == 0x7F7F    # max finite
    assert orc.bf16_round(-0.0) == 0x8000


# ------------------------------------------------------------------------------------------------ e4m3

def test_e4m3_golden_anchors(orc):
    for value, code, *_ in _golden("e4m3_anchors.txt"):
        assert orc.e4m3_encode(float(value)) == int(code, 16), value


def test_e4m3_decode_is_monotone_and_finite(orc):
    mags = [orc.e4m3_decode(c) for c in range(127)]
    assert mags[0] == 0.0 and mags[126] == 448.0
    assert all(b > a for a, b in zip(mags, mags[1:]))
    assert math.isnan(orc.e4m3_decode(0x7F)) and math.isnan(orc.e4m3_decode(0xFF))
    assert all(orc.e4m3_decode(c | 0x80) == -orc.e4m3_decode(c) for c in range(1, 127))


def test_e4m3_every_midpoint_goes_to_even_code(orc):
    mags = [Fraction(orc.e4m3_decode(c)) for c in range(127)]
    for c in range(126):
        mid = (mags[c] + mags[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        m = float(mid)
        assert Fraction(m) == mid                     # midpoints are exact in double
        assert orc.e4m3_encode(m) == even
        assert orc.e4m3_encode(-m) == 0x80 | even
        assert orc.e4m3_encode(math.nextafter(m, 0.0)) == c
        assert orc.e4m3_encode(math.nextafter(m, math.inf)) == c + 1


def test_e4m3_matches_torch_cast_in_range(orc):
    rng = np.random.default_rng(2)
    a = np.concatenate([rng.standard_normal(20000) * 40.0,
                        np.ldexp(rng.random(8000) + 0.5, rng.integers(-12, 9, 8000)) * rng.choice([-1, 1], 8000)])
    a = a.astype(np.float32)
    a = a[np.abs(a) < 464.0]        # torch's cast turns values that round past 448 into NaN; ours saturates
    ref = torch_e4m3(a)
    got = np.array([orc.e4m3_encode(float(v)) for v in a], np.uint8)
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------------------------------------------ SiLU

def test_silu_closed_forms(orc):
    for kind, g, expect in [r for r in _golden("closed_forms.txt") if r[0] == "silu"]:
        got = orc.silu(float(g))
        assert got == pytest.approx(float(expect), rel=2e-15, abs=0.0), g
    assert orc.silu(0.0) == 0.0
    assert orc.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    assert orc.silu(40.0) / 40.0 == pytest.approx(1.0, abs=1e-16)
    assert -1e-7 < orc.silu(-20.0) < 0.0


def test_silu_odd_part_identity_and_torch(orc):
    rng = np.random.default_rng(3)
    xs = rng.standard_normal(2000) * 6.0
    for x in xs:
        assert orc.silu(x) - orc.silu(-x) == pytest.approx(x, rel=1e-14, abs=1e-300)
    ref = F.silu(torch.from_numpy(xs)).numpy()
    got = np.array([orc.silu(x) for x in xs])
    np.testing.assert_allclose(got, ref, rtol=1e-15, atol=1e-300)


# ------------------------------------------------------------------------------------------------ add + RMSNorm

def test_rmsnorm_constant_row_closed_form(orc):
    for kind, c, eps, expect in [r for r in _golden("closed_forms.txt") if r[0] == "rms_const"]:
        c, eps = float(c), float(eps)
        H = 64
        x = np.full((1, H), wl.f32_to_bf16_bits(np.float32(c)), np.uint16)
        r = np.zeros((1, H), np.uint16)
        w = np.full((H,), 0x3F80, np.uint16)                     # weight 1
        res, out, v = orc.add_rmsnorm(x, r, w, eps)
        np.testing.assert_array_equal(res, x)
        np.testing.assert_allclose(v, float(expect), rtol=1e-15)
        # with a weight: every output is w_j times the same value
        wv = wl.f32_to_bf16_bits(np.linspace(0.5, 1.5, H, dtype=np.float32))
        _, _, v2 = orc.add_rmsnorm(x, r, wv, eps)
        np.testing.assert_allclose(v2[0], bf16_vals(wv) * float(expect), rtol=1e-15)


def test_rmsnorm_zero_row(orc):
    H = 32
    z = np.zeros((2, H), np.uint16)
    w = wl.weight_bf16(H, 0)
    res, out, v = orc.add_rmsnorm(z, z, w, 1e-6)
    assert not res.any() and not out.any() and not v.any()


def test_rmsnorm_norms_the_rounded_sum(orc):
    # x = 1, r = 2^-8: the exact sum is a bf16 tie and rounds to 1.0 (even); the residual written
    # and the value normalised are both the rounded sum.
    H = 8
    x = np.full((1, H), 0x3F80, np.uint16)
    r = np.full((1, H), wl.f32_to_bf16_bits(np.float32(2.0 ** -8)), np.uint16)
    w = np.full((H,), 0x3F80, np.uint16)
    res, out, v = orc.add_rmsnorm(x, r, w, 1e-6)
    assert (res == 0x3F80).all()
    np.testing.assert_allclose(v, 1.0 / math.sqrt(1.0 + float(np.float32(1e-6))), rtol=1e-15)


def test_rmsnorm_matches_torch_library(orc):
    for T, H, eps, dist in [(7, 1536, 1e-6, wl.N01), (5, 520, 1e-5, wl.C3_ACT), (3, 4096, 1e-5, wl.C5_ACT)]:
        inp = wl.make_norm_inputs(T, H, 11, dist, eps)
        res, out, v = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, eps)
        # residual: torch's bf16 add (fp32 add, RNE to bf16) is exact rounding of the exact sum
        xs = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16)
        rs = torch.from_numpy(inp.residual.view(np.int16)).view(torch.bfloat16)
        np.testing.assert_array_equal(res, (xs + rs).view(torch.int16).numpy().view(np.uint16))
        s64 = torch.from_numpy(bf16_vals(res))
        w64 = torch.from_numpy(bf16_vals(inp.weight))
        ref = F.rms_norm(s64, (H,), w64, float(np.float32(eps))).numpy()
        np.testing.assert_allclose(v, ref, rtol=1e-13, atol=1e-300)


def test_rmsnorm_unit_rms_invariant(orc):
    T, H, eps = 6, 2048, 1e-6
    inp = wl.make_norm_inputs(T, H, 5, wl.C5_ACT, eps)
    ones = np.full((H,), 0x3F80, np.uint16)
    res, _, v = orc.add_rmsnorm(inp.x, inp.residual, ones, eps)
    s = bf16_vals(res)
    ms = (s * s).mean(axis=1)
    np.testing.assert_allclose((v * v).mean(axis=1), ms / (ms + float(np.float32(eps))), rtol=1e-13)


def _exact_bf16_round(q: Fraction) -> int:
    """Independent RNE of an exact rational onto the bf16 grid (test-side, via integer arithmetic)."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** max(e - 7, -133)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = float(fl * quantum)
    return sign | int(np.array([val], np.float32).view(np.uint32)[0] >> 16)


def test_rmsnorm_brute_force_4x8(orc):
    import mpmath as mp
    mp.mp.dps = 50
    inp = wl.make_norm_inputs(4, 8, 21, wl.C3_ACT, 1e-5)
    res, out, v = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, 1e-5)
    xv, rv, wv = bf16_vals(inp.x), bf16_vals(inp.residual), bf16_vals(inp.weight)
    eps = mp.mpf(float(np.float32(1e-5)))
    for t in range(4):
        s = [Fraction(_exact_bf16_round(Fraction(xv[t, j]) + Fraction(rv[t, j]))) for j in range(8)]
        s = [Fraction(float(bf16_vals(np.array([int(b)], np.uint16))[0])) for b in
             [_exact_bf16_round(Fraction(xv[t, j]) + Fraction(rv[t, j])) for j in range(8)]]
        assert [int(b) for b in res[t]] == [_exact_bf16_round(Fraction(xv[t, j]) + Fraction(rv[t, j]))
                                            for j in range(8)]
        ms = sum(si * si for si in s) / 8
        inv = 1 / mp.sqrt(mp.mpf(ms.numerator) / ms.denominator + eps)
        for j in range(8):
            exact = mp.mpf(wv[j]) * mp.mpf(float(s[j])) * inv
            assert float(v[t, j]) == pytest.approx(float(exact), rel=1e-15, abs=1e-300)
            assert out[t, j] == _exact_bf16_round(Fraction(float(exact)))


# ------------------------------------------------------------------------------------------------ quantisation

def _near_e4m3_midpoint(x: np.ndarray, rel: float) -> np.ndarray:
    """True where |x| lies within rel (relative) of a rounding boundary of the e4m3 grid."""
    grid = np.array([float(Fraction(m)) for m in
                     [0.0] + [float(2.0 ** -9 * k) for k in range(1, 8)] +
                     [float((8 + m) * 2.0 ** (e - 10)) for e in range(1, 16) for m in range(8)][:-1]])
    mids = (grid[1:] + grid[:-1]) / 2
    a = np.abs(x)
    idx = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[idx]), np.abs(a - mids[idx - 1]))
    return d <= rel * np.maximum(a, 2.0 ** -9)


def test_quant_static_matches_torch_pipeline(orc):
    T, H, eps = 64, 512, 1e-5
    inp = wl.make_norm_inputs(T, H, 7, wl.C5_ACT, eps)
    res, q, scale, v = orc.add_rmsnorm_quant_fp8(inp.x, inp.residual, inp.weight, eps, "static", 0.05)
    assert scale[0] == np.float32(0.05)
    _, _, v_plain = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, eps)
    np.testing.assert_array_equal(v, v_plain)
    y = v / float(np.float32(0.05))
    assert (np.abs(y) > 448).any()           # the outliers saturate on purpose
    sat = np.abs(y) >= 448.0
    np.testing.assert_array_equal(q[sat] & 0x7F, 0x7E)
    ok = ~sat & ~_near_e4m3_midpoint(y, 2.0 ** -23)
    ref = torch_e4m3(y.astype(np.float32))
    np.testing.assert_array_equal(q[ok], ref[ok])


def test_quant_dynamic_invariants(orc):
    T, I = 32, 1000
    inp = wl.make_swiglu_inputs(T, I, 9, wl.C5_ACT)
    q, scale, h = orc.swiglu_quant_fp8(inp.gate_up, "dynamic")
    amax = np.abs(h).max(axis=1)
    np.testing.assert_array_equal(scale, (amax / 448.0).astype(np.float32))
    for t in range(T):
        j = int(np.argmax(np.abs(h[t])))
        assert q[t, j] == (0xFE if h[t, j] < 0 else 0x7E)
    assert ((q & 0x7F) <= 0x7E).all()
    y = h / scale.astype(np.float64)[:, None]
    ok = ~_near_e4m3_midpoint(y, 2.0 ** -23)
    np.testing.assert_array_equal(q[ok], torch_e4m3(y.astype(np.float32))[ok])


def test_quant_dynamic_zero_row_and_norm_dynamic(orc):
    gu = np.zeros((2, 64), np.uint16)
    q, scale, _ = orc.swiglu_quant_fp8(gu, "dynamic")
    assert not q.any() and not scale.any()
    inp = wl.make_norm_inputs(8, 256, 4, wl.N01, 1e-6)
    _, q, scale, v = orc.add_rmsnorm_quant_fp8(inp.x, inp.residual, inp.weight, 1e-6, "dynamic")
    np.testing.assert_array_equal(scale, (np.abs(v).max(axis=1) / 448.0).astype(np.float32))
    assert ((q & 0x7F) <= 0x7E).all() and (np.sum((q & 0x7F) == 0x7E, axis=1) >= 1).all()


# ------------------------------------------------------------------------------------------------ SwiGLU

def test_swiglu_matches_torch_library_and_layout(orc):
    for T, I, dist in [(5, 8960, wl.N01), (3, 1000, wl.C3_GU), (2, 13824, wl.C5_ACT)]:
        inp = wl.make_swiglu_inputs(T, I, 13, dist)
        out, h = orc.swiglu(inp.gate_up)
        gu = bf16_vals(inp.gate_up)
        ref = (F.silu(torch.from_numpy(gu[:, :I])) * torch.from_numpy(gu[:, I:])).numpy()
        np.testing.assert_allclose(h, ref, rtol=1e-15, atol=1e-300)
        # swapping the halves must not pass
        swapped = (F.silu(torch.from_numpy(gu[:, I:])) * torch.from_numpy(gu[:, :I])).numpy()
        assert not np.allclose(h, swapped)


def test_swiglu_brute_force_4x8(orc):
    import mpmath as mp
    mp.mp.dps = 50
    inp = wl.make_swiglu_inputs(4, 8, 17, wl.C5_ACT)
    out, h = orc.swiglu(inp.gate_up)
    gu = bf16_vals(inp.gate_up)
    for t in range(4):
        for j in range(8):
            g, u = mp.mpf(gu[t, j]), mp.mpf(gu[t, 8 + j])
            exact = g / (1 + mp.e ** (-g)) * u
            assert float(h[t, j]) == pytest.approx(float(exact), rel=1e-15, abs=1e-300)
            assert out[t, j] == _exact_bf16_round(Fraction(float(exact)))


def test_empty_and_invalid_arguments(orc):
    z = np.zeros((0, 16), np.uint16)
    res, out, v = orc.add_rmsnorm(z, z, np.zeros(16, np.uint16), 1e-6)
    assert res.shape == (0, 16)
    out, h = orc.swiglu(np.zeros((0, 32), np.uint16))
    assert out.shape == (0, 16)


# ------------------------------------------------------------------------------------------------ AllReduce half

def _partials(k, T, H, seed, dist=wl.C5_ACT):
    return [wl.normal_bf16((T, H), seed, "x", dist.sigma, dist.outlier_p, dist.outlier_k, salt=100 + j)
            for j in range(k)]


def test_allreduce_single_partial_is_the_plain_fused_norm(orc):
    inp = wl.make_norm_inputs(6, 1000, 3, wl.C5_ACT, 1e-5)
    a = orc.allreduce_add_rmsnorm([inp.x], inp.residual, inp.weight, 1e-5)
    b = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, 1e-5)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
    aq = orc.allreduce_add_rmsnorm_quant_fp8([inp.x], inp.residual, inp.weight, 1e-5, "dynamic")
    bq = orc.add_rmsnorm_quant_fp8(inp.x, inp.residual, inp.weight, 1e-5, "dynamic")
    for u, v in zip(aq, bq):
        np.testing.assert_array_equal(u, v)


def test_allreduce_sum_is_exact_and_order_free(orc):
    T, H = 5, 640
    ps = _partials(4, T, H, 9)
    r = wl.normal_bf16((T, H), 9, "residual")
    w = wl.weight_bf16(H, 9)
    res, out, v = orc.allreduce_add_rmsnorm(ps, r, w, 1e-5)
    res2, out2, v2 = orc.allreduce_add_rmsnorm(ps[::-1], r, w, 1e-5)
    np.testing.assert_array_equal(res, res2)
    np.testing.assert_array_equal(v, v2)
    # x is the exact sum rounded once (independent rational rounding), then the plain fused norm
    vals = [bf16_vals(p) for p in ps]
    x = np.empty((T, H), np.uint16)
    for t in range(T):
        for j in range(H):
            x[t, j] = _exact_bf16_round(sum(Fraction(float(a[t, j])) for a in vals))
    res3, out3, v3 = orc.add_rmsnorm(x, r, w, 1e-5)
    np.testing.assert_array_equal(res, res3)
    np.testing.assert_array_equal(v, v3)
    # and against PyTorch: where the float64 sum is exact in float32, torch's bf16 cast rounds it once
    s64 = sum(vals)
    exact32 = s64.astype(np.float32).astype(np.float64) == s64
    tx = torch.from_numpy(s64.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert exact32.mean() > 0.99
    np.testing.assert_array_equal(x[exact32], tx[exact32])


def test_allreduce_rejects_bad_partial_counts(orc):
    r = np.zeros((2, 16), np.uint16)
    w = np.zeros(16, np.uint16)
    with pytest.raises(ValueError):
        orc.allreduce_add_rmsnorm([], r, w, 1e-6)
    with pytest.raises(ValueError):
        orc.allreduce_add_rmsnorm([r] * 9, r, w, 1e-6)


# ------------------------------------------------------------------------------------------------ NVFP4

def test_e2m1_golden_anchors(orc):
    for value, code, *_ in _golden("e2m1_anchors.txt"):
        assert orc.e2m1_encode(float(value)) == int(code, 16), value


def test_e2m1_every_midpoint_and_neighbours(orc):
    mags = [orc.e2m1_decode(c) for c in range(8)]
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert all(orc.e2m1_decode(c | 8) == -mags[c] for c in range(1, 8))
    for c in range(7):
        mid = (mags[c] + mags[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert orc.e2m1_encode(mid) == even
        assert orc.e2m1_encode(-mid) == 8 | even
        assert orc.e2m1_encode(math.nextafter(mid, 0.0)) == c
        assert orc.e2m1_encode(math.nextafter(mid, math.inf)) == c + 1


def _unpack_e2m1(q):
    """Test-side unpacking of packed E2M1 codes (low nibble first) to codes and values, from the format's
    definition: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, sign in bit 3."""
    codes = np.stack([q & 0xF, q >> 4], axis=-1).reshape(q.shape[0], -1)
    mag_tab = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    return codes, np.where(codes & 8, -1.0, 1.0) * mag_tab[codes & 7]


def test_nvfp4_block_structure(orc):
    T, H, S = 6, 512, 0.02
    inp = wl.make_norm_inputs(T, H, 5, wl.C5_ACT, 1e-5)
    res, q, sf, v = orc.add_rmsnorm_quant_nvfp4(inp.x, inp.residual, inp.weight, 1e-5, S)
    res0, _, v0 = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, 1e-5)
    np.testing.assert_array_equal(res, res0)
    np.testing.assert_array_equal(v, v0)
    codes, vals = _unpack_e2m1(q)
    blk_scale = np.array([[orc.e4m3_decode(int(c)) for c in row] for row in sf]) * float(np.float32(S))
    deq = vals * np.repeat(blk_scale, 16, axis=1)
    amax = np.abs(v).reshape(T, H // 16, 16).max(axis=2)
    # the block scale is the E4M3 rounding of amax / (6 S): within one E4M3 half-step (<= 1/16 relative)
    target = amax / (6 * float(np.float32(S)))
    np.testing.assert_array_less(np.abs(blk_scale / float(np.float32(S)) - target), target / 16 + 2.0 ** -10)
    # every element sits within half an E2M1 step of its exact value (steps are <= 2 units of the block scale)
    step = np.repeat(blk_scale, 16, axis=1) * np.where(np.abs(v) / np.repeat(blk_scale, 16, axis=1) < 2, 0.5,
                                                        np.where(np.abs(v) / np.repeat(blk_scale, 16, axis=1) < 4, 1.0, 2.0))
    sat = np.abs(v) > 6 * np.repeat(blk_scale, 16, axis=1)
    assert (np.abs(deq - v)[~sat] <= step[~sat] / 2 * (1 + 1e-12)).all()
    # with a normal E4M3 block scale (relative error <= 1/16) the block maximum lands in [6/(1+1/16),
    # 6/(1-1/16)] = [5.65, 6.4], above the 4/6 midpoint: it always takes code +-6
    j = np.abs(v).reshape(T, H // 16, 16).argmax(axis=2)
    top = np.take_along_axis(codes.reshape(T, H // 16, 16), j[..., None], axis=2)[..., 0]
    normal = (sf & 0x78) != 0
    assert normal.mean() > 0.99
    assert ((top & 7) == 7)[normal].all()
    sign = np.take_along_axis(v.reshape(T, H // 16, 16), j[..., None], axis=2)[..., 0] < 0
    assert ((top >> 3) == sign)[normal].all()


def test_nvfp4_codes_vs_exact_rational(orc):
    T, I, S = 3, 64, 0.01
    inp = wl.make_swiglu_inputs(T, I, 7, wl.C5_ACT)
    q, sf, h = orc.swiglu_quant_nvfp4(inp.gate_up, S)
    Sf = Fraction(float(np.float32(S)))
    mags = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]
    for t in range(T):
        for b in range(I // 16):
            blk = [Fraction(float(x)) for x in h[t, b * 16:(b + 1) * 16]]
            amax = max(abs(x) for x in blk)
            assert sf[t, b] == orc.e4m3_encode(float(amax / (6 * Sf)))
            scale = Fraction(orc.e4m3_decode(int(sf[t, b]))) * Sf
            for j, x in enumerate(blk):
                code = (q[t, (b * 16 + j) // 2] >> (4 * (j % 2))) & 0xF
                a = abs(x) / scale
                if a >= 6:
                    want = 7
                else:
                    d = [abs(a - m) for m in mags]
                    best = min(range(8), key=lambda c: (d[c], c % 2))
                    want = best
                assert code & 7 == want
                assert (code >> 3) == (1 if x < 0 else 0)   # the sign is kept, also on a rounded zero


def test_bf16_sum_golden(orc):
    """Hand-derived exact sums (tests/golden/bf16_sums.txt): ties to even, carries into the exponent, zero sums,
    subnormals, overflow, and tiny terms that decide a tie, which a float64 accumulation loses."""
    rows = _golden("bf16_sums.txt")
    assert len(rows) >= 12
    for *addends, want in rows:
        bits = [int(a, 16) for a in addends]
        assert orc.bf16_sum(bits) == int(want, 16), addends


def _wide_bf16_sets(rng, n_sets, k):
    """bf16 addend sets with exponents spread over the whole range (normal values near 1 beside subnormals,
    huge and tiny values) and exact midpoint constructions tipped by tiny terms."""
    sets = []
    for i in range(n_sets):
        kind = i % 3 if k >= 2 else 0
        if kind == 0:      # any finite exponent field, random mantissas and signs
            e = rng.integers(0, 250, k)
            m = rng.integers(0, 128, k)
            s = rng.integers(0, 2, k)
            sets.append((s << 15) | (e << 7) | m)
        elif kind == 1:    # a value, half its bf16 ulp, and tiny terms of random sign
            e0 = int(rng.integers(40, 200))
            base = (int(rng.integers(0, 2)) << 15) | (e0 << 7) | int(rng.integers(0, 128))
            half = (base & 0x8000) | ((e0 - 8) << 7)
            tiny = [(int(rng.integers(0, 2)) << 15) | (int(rng.integers(0, max(1, e0 - 9))) << 7) | int(rng.integers(0, 128))
                    for _ in range(k - 2)]
            sets.append(np.array([base, half] + tiny))
        else:              # cancellation: x, -x and small terms
            x = int(rng.integers(0x0080, 0x7F00))
            rest = rng.integers(0, 0x7F00, k - 2) | (rng.integers(0, 2, k - 2) << 15)
            sets.append(np.array([x, x | 0x8000] + list(rest)))
    return [np.asarray(s, np.uint16) for s in sets]


def test_bf16_sum_is_the_exact_sum_rounded_once(orc):
    """Against rational arithmetic (Fractions, test-side rounding) on addend sets whose exponents span far more
    than a float64 holds."""
    rng = np.random.default_rng(2024)
    for k in (1, 2, 3, 8):
        for bits in _wide_bf16_sets(rng, 600, k):
            exact = sum((Fraction(float(v)) for v in bf16_vals(bits)), Fraction(0))
            assert orc.bf16_sum(bits) == _exact_bf16_round(exact), [hex(int(b)) for b in bits]


def test_allreduce_reduces_with_the_exact_sum(orc):
    """The all-reduce half's x is bf16_sum of the partials, element by element (wide-span partials)."""
    rng = np.random.default_rng(7)
    sets = _wide_bf16_sets(rng, 3 * 64, 8)
    ps = [np.array([s[j] for s in sets], np.uint16).reshape(3, 64) for j in range(8)]
    r = np.zeros((3, 64), np.uint16)                      # x + (+0) = x
    w = wl.weight_bf16(64, 1)
    res, _, _ = orc.allreduce_add_rmsnorm(ps, r, w, 1e-5)
    want = np.array([orc.bf16_sum(s) for s in sets], np.uint16).reshape(3, 64)
    np.testing.assert_array_equal(res, np.where(want == 0x8000, 0, want))
