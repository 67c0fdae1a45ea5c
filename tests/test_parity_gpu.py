"""Parity of the CUDA path (called through the C ABI) against the fp64 CPU oracle on the same seeded inputs.

Small and ragged shapes are compared element by element; the full-size workloads run in the same launch
configuration the bench uses and are compared on sampled rows (rows are independent, so the oracle can
compute any subset exactly). Every output sits between guard bands that must stay untouched.
"""
import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests.parity import (Guarded, check_bf16, check_codes, check_scales, dev_u16, sample_rows)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_decoder_gb300 import build
    build.build()
    orc.build()
    import memory_bound_decoder_gb300 as mbd
    mbd.get_lib()


def _mbd():
    import memory_bound_decoder_gb300 as mbd
    return mbd


# ------------------------------------------------------------------------------------------------ runners

def gpu_norm(inp, ep, mode=None, static_scale=0.05, rows=None, inplace=False, stream=None):
    """Run one norm entry point; returns (residual, out or q, scale) as numpy for `rows` (all if None)."""
    mbd = _mbd()
    T, H = inp.x.shape
    x, r, w = dev_u16(torch, inp.x), dev_u16(torch, inp.residual), dev_u16(torch, inp.weight)
    n0 = mbd.kernel_launches()
    sc = None
    if ep == "bf16":
        out = x if inplace else Guarded(torch, T * H, torch.int16)
        mbd.fused_add_rmsnorm(out.view, r.view, x.view, w.view, T, H, inp.eps, stream)
    else:
        out = Guarded(torch, T * H, torch.uint8)
        if mode == "static":
            sc = Guarded(torch, 1, torch.float32, fill=np.array([static_scale], np.float32))
        else:
            sc = Guarded(torch, max(T, 1), torch.float32)
        mbd.fused_add_rmsnorm_quant_fp8(out.view, r.view, x.view, w.view, T, H, inp.eps, mode, sc.view, stream)
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == (1 if T > 0 else 0)
    for g, name in [(x, "x"), (r, "residual"), (w, "weight"), (out, "out")] + ([(sc, "scale")] if sc else []):
        g.check_guards(name)
    if not inplace:
        np.testing.assert_array_equal(x.numpy(np.uint16), inp.x.reshape(-1), "x was modified")
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    res = r.view.view(T, H)[sel].cpu().numpy().view(np.uint16)
    if ep == "bf16":
        o = out.view.view(T, H)[sel].cpu().numpy().view(np.uint16)
        return res, o, None
    q = out.view.view(T, H)[sel].cpu().numpy()
    s = sc.view.cpu().numpy()
    if mode == "dynamic":
        s = s[:T][rows] if rows is not None else s[:T]
    return res, q, s


def gpu_swiglu(inp, ep, mode=None, static_scale=0.05, rows=None, stream=None):
    mbd = _mbd()
    T, I2 = inp.gate_up.shape
    I = I2 // 2
    gu = dev_u16(torch, inp.gate_up)
    n0 = mbd.kernel_launches()
    sc = None
    if ep == "bf16":
        out = Guarded(torch, T * I, torch.int16)
        mbd.swiglu(out.view, gu.view, T, I, stream)
    else:
        out = Guarded(torch, T * I, torch.uint8)
        if mode == "static":
            sc = Guarded(torch, 1, torch.float32, fill=np.array([static_scale], np.float32))
        else:
            sc = Guarded(torch, max(T, 1), torch.float32)
        mbd.swiglu_quant_fp8(out.view, gu.view, T, I, mode, sc.view, stream)
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == (1 if T > 0 else 0)
    for g, name in [(gu, "gate_up"), (out, "out")] + ([(sc, "scale")] if sc else []):
        g.check_guards(name)
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    if ep == "bf16":
        return out.view.view(T, I)[sel].cpu().numpy().view(np.uint16), None
    q = out.view.view(T, I)[sel].cpu().numpy()
    s = sc.view.cpu().numpy()
    if mode == "dynamic":
        s = s[:T][rows] if rows is not None else s[:T]
    return q, s


# ------------------------------------------------------------------------------------------------ checkers

def check_norm(inp, ep, mode=None, static_scale=0.05, rows=None, **kw):
    res_g, out_g, s_g = gpu_norm(inp, ep, mode, static_scale, rows, **kw)
    x, r = (inp.x, inp.residual) if rows is None else (inp.x[rows], inp.residual[rows])
    if ep == "bf16":
        res_o, out_o, v = orc.add_rmsnorm(x, r, inp.weight, inp.eps)
        np.testing.assert_array_equal(res_g, res_o, "residual must be bit-exact")
        return check_bf16(out_g, v, "add_rmsnorm")
    res_o, q_o, s_o, v = orc.add_rmsnorm_quant_fp8(x, r, inp.weight, inp.eps, mode, static_scale)
    np.testing.assert_array_equal(res_g, res_o, "residual must be bit-exact")
    if mode == "dynamic":
        check_scales(s_g, s_o, "add_rmsnorm_q8 scale")
    else:
        assert s_g[0] == np.float32(static_scale)
    return check_codes(out_g, q_o, f"add_rmsnorm_q8 {mode}")


def check_swiglu(inp, ep, mode=None, static_scale=0.05, rows=None, **kw):
    out_g, s_g = gpu_swiglu(inp, ep, mode, static_scale, rows, **kw)
    gu = inp.gate_up if rows is None else inp.gate_up[rows]
    if ep == "bf16":
        _, h = orc.swiglu(gu)
        return check_bf16(out_g, h, "swiglu")
    q_o, s_o, h = orc.swiglu_quant_fp8(gu, mode, static_scale)
    if mode == "dynamic":
        check_scales(s_g, s_o, "swiglu_q8 scale")
    return check_codes(out_g, q_o, f"swiglu_q8 {mode}")


# ------------------------------------------------------------------------------------------------ small / ragged

# The first rows use the direct (one launch wave) form; shapes with at least two units per SM use the
# persistent pipelined form: (320, 5000) ragged slices, (400, 32768) a row split over a 2-CTA cluster,
# (304, 53248) a dynamic SwiGLU row over a 4-CTA cluster, (500, 3000) ragged chunks.
NORM_SHAPES = [(16, 1536), (1, 1536), (3, 5120), (17, 5120), (7, 8), (5, 24), (33, 520), (2, 1000),
               (64, 4096), (4, 16384), (300, 1536), (2, 262144), (320, 5000), (400, 32768), (1200, 1536)]
SWIGLU_SHAPES = [(16, 8960), (1, 13824), (3, 13824), (17, 13824), (5, 8), (9, 24), (3, 1000), (2, 53248),
                 (200, 8960), (1, 262144), (400, 13824), (304, 53248), (500, 3000), (700, 256)]
EPS = [("bf16", None), ("q8", "static"), ("q8", "dynamic")]


@pytest.mark.parametrize("T,H", NORM_SHAPES)
@pytest.mark.parametrize("ep,mode", EPS)
def test_norm_small(T, H, ep, mode):
    inp = wl.make_norm_inputs(T, H, seed=T * 7 + H, dist=wl.C5_ACT, eps=1e-5)
    check_norm(inp, ep, mode, static_scale=0.05)


@pytest.mark.parametrize("T,I", SWIGLU_SHAPES)
@pytest.mark.parametrize("ep,mode", EPS)
def test_swiglu_small(T, I, ep, mode):
    inp = wl.make_swiglu_inputs(T, I, seed=T * 11 + I, dist=wl.C5_ACT)
    check_swiglu(inp, ep, mode, static_scale=0.05)


def test_swiglu_wide_streams_beyond_reduced_limit():
    inp = wl.make_swiglu_inputs(2, 300000, seed=3, dist=wl.N01)
    check_swiglu(inp, "bf16")
    check_swiglu(inp, "q8", "static", static_scale=0.01)


# C1: Qwen2.5-1.5B-shaped layer, 16 tokens (seed 0)
def test_qwen_t16_layer():
    for call in wl.qwen_t16().calls:
        inp = wl.inputs_for(call, seed=0)
        if call.kind == "add_rmsnorm":
            check_norm(inp, "bf16")
        else:
            check_swiglu(inp, "bf16")


# C2: decode sweep shapes (every layer runs the same kernels; one layer's inputs per token count)
@pytest.mark.parametrize("T", [1, 2, 4, 8, 32, 64, 128, 256])
def test_qwen_decode_sweep_shapes(T):
    inp = wl.make_norm_inputs(T, 1536, seed=T, dist=wl.N01, eps=1e-6)
    check_norm(inp, "bf16")
    check_norm(inp, "q8", "dynamic")
    gu = wl.make_swiglu_inputs(T, 8960, seed=T, dist=wl.N01)
    check_swiglu(gu, "bf16")
    check_swiglu(gu, "q8", "dynamic")


# C5 ragged part: all four entry points at 1, 3, 17, 1000 tokens, hidden 5120 / intermediate 13824
@pytest.mark.parametrize("T", [1, 3, 17, 1000])
def test_ragged_405b_tails(T):
    inp = wl.make_norm_inputs(T, 5120, seed=0, dist=wl.C5_ACT, eps=1e-5)
    check_norm(inp, "bf16")
    check_norm(inp, "q8", "static", static_scale=0.05)
    gu = wl.make_swiglu_inputs(T, 13824, seed=0, dist=wl.C5_ACT)
    check_swiglu(gu, "bf16")
    check_swiglu(gu, "q8", "dynamic")


@pytest.mark.parametrize("I,shape", [(36872, (7, 4, 192)), (81920, (8, 4, 320))])
def test_dynamic_swiglu_bulk_form(I, shape):
    """Wide dynamic-FP8 SwiGLU rows at four or more rows per SM take the bulk-copy form (slices brought into
    shared memory): 4609 vectors (the narrowest such row; clusters of 7, a ragged last slice) and 10240
    (the widest; clusters of 8, 320 threads). Sampled rows, including the first and the last."""
    mbd = _mbd()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 4 * sms + 3
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", T, I) == shape
    inp = wl.make_swiglu_inputs(T, I, seed=4, dist=wl.C5_ACT)
    check_swiglu(inp, "q8", "dynamic", rows=sample_rows(T, 16, seed=5))


# ------------------------------------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("ep,mode", [("bf16", None), ("q8", "static"), ("q8", "dynamic")])
def test_more_rows_than_one_grid_axis(ep, mode):
    """70001 rows: the launch lays rows over the grid's y and z axes (at most 65535 each), so rows past 65535
    sit in the second z plane. Every row is compared."""
    T = 70001
    check_norm(wl.make_norm_inputs(T, 64, seed=9, dist=wl.C5_ACT, eps=1e-5), ep, mode, static_scale=0.05)
    check_swiglu(wl.make_swiglu_inputs(T, 64, seed=9, dist=wl.C3_GU), ep, mode, static_scale=0.05)


def test_zero_rows_and_constant_rows():
    T, H = 4, 2048
    x = np.zeros((T, H), np.uint16)
    r = np.zeros((T, H), np.uint16)
    r[2] = wl.f32_to_bf16_bits(np.float32(3.0))          # a constant row
    r[3] = wl.f32_to_bf16_bits(np.float32(-2.0 ** -10))  # a tiny constant row: eps dominates
    inp = wl.NormInputs(x, r, wl.weight_bf16(H, 1), 1e-6)
    check_norm(inp, "bf16")
    check_norm(inp, "q8", "dynamic")
    res, q, s = gpu_norm(inp, "q8", "dynamic")
    assert s[0] == 0.0 and s[1] == 0.0 and not q[:2].any()
    gu = np.zeros((3, 2 * 512), np.uint16)
    gu[1, :512] = wl.f32_to_bf16_bits(np.float32(2.0))
    gu[1, 512:] = wl.f32_to_bf16_bits(np.float32(-1.0))
    check_swiglu(wl.SwigluInputs(gu), "q8", "dynamic")
    q, s = gpu_swiglu(wl.SwigluInputs(gu), "q8", "dynamic")
    assert s[0] == 0.0 and s[2] == 0.0 and not q[0].any() and not q[2].any()
    assert (q[1] == 0xFE).all()          # every element is the row's amax -> -448


def _residual_edge_rows(T, H, seed):
    """x and residual whose sums stress bf16(x + r): exponent spans of 0 to 40 between the addends (the fp32 sum
    is inexact beyond 15), exact midpoints of the bf16 rounding (ties to even), cancellation to zero, bf16
    subnormals (with each other and with normal values) and signed zeros, every kind in every row."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    r = rng.standard_normal((T, H))
    kind = rng.integers(0, 5, (T, H))
    xb = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(x.astype(np.float32))).astype(np.float64)
    wide = kind == 0
    r[wide] = (xb * 2.0 ** -rng.integers(0, 41, (T, H)) * rng.choice([-1.0, 1.0], (T, H)))[wide]
    tie = kind == 1
    e = np.floor(np.log2(np.maximum(np.abs(xb), 1e-30)))
    r[tie] = (np.sign(xb) * rng.choice([-1.0, 1.0], (T, H)) * 2.0 ** (e - 8))[tie]
    canc = kind == 2
    r[canc] = -xb[canc]
    sub = kind == 3
    x[sub] *= 2.0 ** -130
    r[sub] *= 2.0 ** rng.choice([-131.0, -120.0, 0.0], (T, H))[sub]
    zero = kind == 4
    x[zero] = rng.choice([0.0, -0.0], (T, H))[zero] * 1.0
    x[zero & (rng.random((T, H)) < 0.5)] = -0.0
    r[zero & (rng.random((T, H)) < 0.5)] = -0.0
    return wl.f32_to_bf16_bits(x.astype(np.float32)), wl.f32_to_bf16_bits(r.astype(np.float32))


@pytest.mark.parametrize("T,H", [(8, 5120), (6, 16384), (300, 4096)])
def test_residual_add_edges(T, H):
    """The residual s = bf16(x + r) bit-exact where the fp32 sum is inexact, lands on a rounding midpoint,
    cancels, or meets subnormals and signed zeros; the outputs within the usual tolerances."""
    xb, rb = _residual_edge_rows(T, H, seed=T + H)
    inp = wl.NormInputs(xb, rb, wl.weight_bf16(H, 3), 1e-5)
    check_norm(inp, "bf16")
    check_norm(inp, "q8", "static")
    check_norm(inp, "q8", "dynamic")


def test_static_saturation():
    inp = wl.make_norm_inputs(8, 4096, seed=2, dist=wl.C5_ACT, eps=1e-5)
    check_norm(inp, "q8", "static", static_scale=1e-3)
    _, q, _ = gpu_norm(inp, "q8", "static", static_scale=1e-3)
    assert ((q & 0x7F) == 0x7E).mean() > 0.1    # the outlier-heavy rows push many values past 448
    gu = wl.make_swiglu_inputs(8, 4096, seed=2, dist=wl.C5_ACT)
    check_swiglu(gu, "q8", "static", static_scale=1e-3)


def test_inplace_out_equals_x_and_side_stream():
    inp = wl.make_norm_inputs(37, 4096, seed=5, dist=wl.C3_ACT, eps=1e-5)
    check_norm(inp, "bf16", inplace=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        check_norm(inp, "bf16", stream=s)
        check_swiglu(wl.make_swiglu_inputs(37, 14336, seed=5, dist=wl.C3_GU), "q8", "dynamic", stream=s)


def test_zero_tokens_launches_nothing():
    mbd = _mbd()
    n0 = mbd.kernel_launches()
    mbd.fused_add_rmsnorm(None, None, None, None, 0, 4096, 1e-6)
    mbd.swiglu_quant_fp8(None, None, 0, 4096, "dynamic", None)
    assert mbd.kernel_launches() == n0


def test_repeated_calls_are_deterministic():
    inp = wl.make_swiglu_inputs(64, 28672, seed=8, dist=wl.C5_ACT)
    a = gpu_swiglu(inp, "q8", "dynamic")
    b = gpu_swiglu(inp, "q8", "dynamic")
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------------------------------------------------ full sizes

@pytest.mark.slow
def test_full_llama3_8b_prefill():
    for call in wl.llama3_8b_prefill().calls:
        inp = wl.inputs_for(call, seed=0)
        rows = sample_rows(call.T, 24, seed=1)
        if call.kind == "add_rmsnorm":
            check_norm(inp, "bf16", rows=rows)
        else:
            check_swiglu(inp, "bf16", rows=rows)


@pytest.mark.slow
def test_full_llama3_70b_fp8():
    for call in wl.llama3_70b_fp8().calls:
        inp = wl.inputs_for(call, seed=0)
        rows = sample_rows(call.T, 24, seed=2)
        if call.kind == "add_rmsnorm_q8":
            check_norm(inp, "q8", "static", call.static_scale, rows=rows)
        else:
            check_swiglu(inp, "q8", "dynamic", rows=rows)


@pytest.mark.slow
def test_full_llama31_405b_fp8():
    for call in wl.llama31_405b_fp8_ragged().calls[:2]:
        inp = wl.inputs_for(call, seed=0)
        rows = sample_rows(call.T, 16, seed=3)
        if call.kind == "add_rmsnorm_q8":
            check_norm(inp, "q8", "static", call.static_scale, rows=rows)
        else:
            check_swiglu(inp, "q8", "dynamic", rows=rows)
