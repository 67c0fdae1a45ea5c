"""Parity of the NVFP4 epilogues (fused residual add + RMSNorm, SwiGLU) against the fp64 CPU oracle.

Shapes span single-vector rows, ragged slices, rows split over a cluster (the norm), the decode-sized
single-wave launches and the 405B-shaped prefill batch the bench times (sampled rows). The tensor scales
are the calibrated ones (tensor amax / (6 * 448)) plus extremes that saturate or zero the block scales.
"""
import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests.parity import Guarded, check_nvfp4, dev_u16, sample_rows, unpack_e2m1

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


def gpu_norm_nvfp4(inp, S, rows=None, stream=None):
    mbd = _mbd()
    T, H = inp.x.shape
    x, r, w = dev_u16(torch, inp.x), dev_u16(torch, inp.residual), dev_u16(torch, inp.weight)
    q = Guarded(torch, T * H // 2, torch.uint8)
    sf = Guarded(torch, T * H // 16, torch.uint8)
    sc = Guarded(torch, 1, torch.float32, fill=np.array([S], np.float32))
    n0 = mbd.kernel_launches()
    mbd.fused_add_rmsnorm_quant_nvfp4(q.view, sf.view, r.view, x.view, w.view, T, H, inp.eps, sc.view, stream)
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == (1 if T > 0 else 0)
    for g, name in [(x, "x"), (r, "residual"), (w, "weight"), (q, "codes"), (sf, "block scales"), (sc, "scale")]:
        g.check_guards(name)
    np.testing.assert_array_equal(x.numpy(np.uint16), inp.x.reshape(-1), "x was modified")
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    res = r.view.view(T, H)[sel].cpu().numpy().view(np.uint16)
    return res, q.view.view(T, H // 2)[sel].cpu().numpy(), sf.view.view(T, H // 16)[sel].cpu().numpy()


def gpu_swiglu_nvfp4(inp, S, rows=None, stream=None):
    mbd = _mbd()
    T, I2 = inp.gate_up.shape
    I = I2 // 2
    gu = dev_u16(torch, inp.gate_up)
    q = Guarded(torch, T * I // 2, torch.uint8)
    sf = Guarded(torch, T * I // 16, torch.uint8)
    sc = Guarded(torch, 1, torch.float32, fill=np.array([S], np.float32))
    n0 = mbd.kernel_launches()
    mbd.swiglu_quant_nvfp4(q.view, sf.view, gu.view, T, I, sc.view, stream)
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == (1 if T > 0 else 0)
    for g, name in [(gu, "gate_up"), (q, "codes"), (sf, "block scales"), (sc, "scale")]:
        g.check_guards(name)
    sel = slice(None) if rows is None else torch.as_tensor(rows, device="cuda")
    return q.view.view(T, I // 2)[sel].cpu().numpy(), sf.view.view(T, I // 16)[sel].cpu().numpy()


def check_norm(inp, S, rows=None, **kw):
    res_g, q_g, sf_g = gpu_norm_nvfp4(inp, S, rows, **kw)
    x, r = (inp.x, inp.residual) if rows is None else (inp.x[rows], inp.residual[rows])
    res_o, q_o, sf_o, v = orc.add_rmsnorm_quant_nvfp4(x, r, inp.weight, inp.eps, S)
    np.testing.assert_array_equal(res_g, res_o, "residual must be bit-exact")
    return check_nvfp4(q_g, sf_g, q_o, sf_o, v, S, orc, "add_rmsnorm_nvfp4")


def check_swiglu(inp, S, rows=None, **kw):
    q_g, sf_g = gpu_swiglu_nvfp4(inp, S, rows, **kw)
    gu = inp.gate_up if rows is None else inp.gate_up[rows]
    q_o, sf_o, h = orc.swiglu_quant_nvfp4(gu, S)
    return check_nvfp4(q_g, sf_g, q_o, sf_o, h, S, orc, "swiglu_nvfp4")


# widths: one block, two vectors (one lane pair), ragged slice counts, cluster-split rows, the widest row
NORM_SHAPES = [(1, 16), (3, 48), (16, 1536), (1, 5120), (17, 5120), (33, 528), (64, 4096), (4, 16384),
               (300, 1536), (320, 5008), (400, 32768), (1200, 1536), (2, 262144), (7, 16400)]
SWIGLU_SHAPES = [(1, 16), (5, 48), (16, 8960), (1, 13824), (17, 13824), (9, 1008), (2, 53248), (200, 8960),
                 (400, 13824), (304, 53248), (500, 3008), (700, 256), (1, 262144)]


@pytest.mark.parametrize("T,H", NORM_SHAPES)
def test_norm_nvfp4_small(T, H):
    inp = wl.make_norm_inputs(T, H, seed=T * 5 + H, dist=wl.C5_ACT, eps=1e-5)
    check_norm(inp, wl.NVFP4_SCALE_NORM_C5)


@pytest.mark.parametrize("T,I", SWIGLU_SHAPES)
def test_swiglu_nvfp4_small(T, I):
    inp = wl.make_swiglu_inputs(T, I, seed=T * 13 + I, dist=wl.C5_ACT)
    check_swiglu(inp, wl.NVFP4_SCALE_SWIGLU_C5)


@pytest.mark.parametrize("T", [1, 2, 8, 64, 256])
def test_decode_sizes(T):
    check_norm(wl.make_norm_inputs(T, 1536, seed=T, dist=wl.N01, eps=1e-6), 0.003)
    check_swiglu(wl.make_swiglu_inputs(T, 8960, seed=T, dist=wl.N01), 0.01)


def test_more_rows_than_one_grid_axis():
    """70001 rows over the grid's y and z axes (rows past 65535 in the second z plane); every row compared."""
    check_norm(wl.make_norm_inputs(70001, 64, seed=9, dist=wl.C5_ACT, eps=1e-5), wl.NVFP4_SCALE_NORM_C5)
    check_swiglu(wl.make_swiglu_inputs(70001, 64, seed=9, dist=wl.C5_ACT), wl.NVFP4_SCALE_SWIGLU_C5)


def test_sign_and_zero_codes():
    """Zero rows give zero block scales and all-zero codes; negative values keep their sign bit."""
    T, H = 3, 256
    x = np.zeros((T, H), np.uint16)
    r = np.zeros((T, H), np.uint16)
    r[1] = wl.f32_to_bf16_bits(np.float32(-1.5))
    inp = wl.NormInputs(x, r, wl.f32_to_bf16_bits(np.ones(H, np.float32)), 1e-6)
    check_norm(inp, 0.01)
    _, q, sf = gpu_norm_nvfp4(inp, 0.01)
    assert not q[0].any() and not sf[0].any() and not q[2].any() and not sf[2].any()
    # row 1: v = -1 everywhere -> block scale E4M3(1 / 0.06) and every code -6 (0xF)
    assert (sf[1] == orc.e4m3_encode(1.0 / (6 * float(np.float32(0.01))))).all()
    assert (unpack_e2m1(q[1:2]) == 0xF).all()
    gu = np.zeros((2, 2 * 64), np.uint16)
    gu[1, :64] = wl.f32_to_bf16_bits(np.float32(2.0))
    gu[1, 64:] = wl.f32_to_bf16_bits(np.tile(np.float32([-1.0, 0.5, -0.25, 0.0]), 16))
    check_swiglu(wl.SwigluInputs(gu), 0.05)
    q, sf = gpu_swiglu_nvfp4(wl.SwigluInputs(gu), 0.05)
    assert not q[0].any() and not sf[0].any()


def test_block_scale_saturation_and_underflow():
    """A tiny tensor scale saturates the block scales at 448 (codes then saturate at +-6); a huge one
    rounds them to zero (codes zero)."""
    inp = wl.make_norm_inputs(8, 4096, seed=2, dist=wl.C5_ACT, eps=1e-5)
    check_norm(inp, 1e-4)
    _, q, sf = gpu_norm_nvfp4(inp, 1e-4)
    assert (sf == 0x7E).mean() > 0.5
    check_norm(inp, 1e6)
    _, q, sf = gpu_norm_nvfp4(inp, 1e6)
    assert not sf.any() and not q.any()
    gu = wl.make_swiglu_inputs(8, 4096, seed=2, dist=wl.C5_ACT)
    check_swiglu(gu, 1e-4)
    check_swiglu(gu, 1e6)


@pytest.mark.parametrize("S", [0.0, -1.0, float("nan"), float("inf"), 1e-30, 1e30])
def test_unusable_tensor_scale_gives_zeros(S):
    inp = wl.make_norm_inputs(5, 512, seed=4, dist=wl.N01, eps=1e-6)
    res, q, sf = gpu_norm_nvfp4(inp, S)
    res_o, _, _ = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, inp.eps)
    np.testing.assert_array_equal(res, res_o)
    assert not q.any() and not sf.any()
    q, sf = gpu_swiglu_nvfp4(wl.make_swiglu_inputs(5, 512, seed=4, dist=wl.N01), S)
    assert not q.any() and not sf.any()


def test_side_stream_and_determinism():
    inp = wl.make_swiglu_inputs(37, 14336, seed=5, dist=wl.C3_GU)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = gpu_swiglu_nvfp4(inp, 0.02, stream=s)
        b = gpu_swiglu_nvfp4(inp, 0.02, stream=s)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    check_swiglu(inp, 0.02)


# the 405B-shaped NVFP4 batch the bench times, in the bench's launch configuration, on sampled rows
@pytest.mark.slow
def test_full_llama31_405b_nvfp4():
    for call in wl.llama31_405b_nvfp4().calls:
        inp = wl.inputs_for(call, seed=0)
        rows = sample_rows(call.T, 16, seed=4)
        if call.is_norm:
            check_norm(inp, call.static_scale, rows=rows)
        else:
            check_swiglu(inp, call.static_scale, rows=rows)
