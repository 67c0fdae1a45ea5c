"""The launch-shape table (mbd_tuning_set) on the GPU: entry points launched with shapes the built-in rules
would not pick -- cluster sizes, vectors per thread and CTA widths from the tuner's candidate set -- must still
match the oracle, write nothing outside their outputs, and report the shape they used."""
import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests.parity import check_bf16, check_codes, check_nvfp4, check_scales
from tests.test_parity_gpu import gpu_norm, gpu_swiglu
from tests.test_nvfp4_gpu import gpu_norm_nvfp4, gpu_swiglu_nvfp4

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
    yield
    mbd.tuning_set([])


def _mbd():
    import memory_bound_decoder_gb300 as mbd
    return mbd


def force(kind, mode, T, W, shape):
    mbd = _mbd()
    mbd.tuning_set([{"kind": kind, "mode": mode, "tokens": [T, T], "width": [W, W], "ctas_per_row": shape[0],
                     "vectors_per_thread": shape[1], "threads": shape[2]}])
    got = mbd.launch_shape(kind, mode, T, W)
    assert got[1:] == tuple(shape[1:]), (kind, shape, got)
    return got


@pytest.mark.parametrize("T,H,shape", [(64, 1536, (3, 1, 64)), (200, 5120, (5, 1, 128)), (7, 16384, (8, 2, 128)),
                                       (300, 4096, (1, 8, 64)), (160, 8192, (2, 4, 128))])
def test_norm_forced_shapes(T, H, shape):
    inp = wl.make_norm_inputs(T, H, seed=T + H, dist=wl.C5_ACT, eps=1e-5)
    for kind, mode, ep in (("add_rmsnorm", None, "bf16"), ("add_rmsnorm_quant_fp8", "static", "q8"),
                           ("add_rmsnorm_quant_fp8", "dynamic", "q8")):
        force(kind, mode, T, H, shape)
        res, out, sc = gpu_norm(inp, ep, mode, static_scale=0.05)
        if ep == "bf16":
            r_o, _, v = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, inp.eps)
            np.testing.assert_array_equal(res, r_o)
            check_bf16(out, v, f"norm {shape}")
        else:
            r_o, q_o, s_o, _ = orc.add_rmsnorm_quant_fp8(inp.x, inp.residual, inp.weight, inp.eps, mode, 0.05)
            np.testing.assert_array_equal(res, r_o)
            check_codes(out, q_o, f"norm q8 {mode} {shape}")
            if mode == "dynamic":
                check_scales(sc, s_o, "norm scales")
    force("add_rmsnorm_quant_nvfp4", None, T, H, shape)
    res, q, sf = gpu_norm_nvfp4(inp, 0.03)
    r_o, q_o, sf_o, v = orc.add_rmsnorm_quant_nvfp4(inp.x, inp.residual, inp.weight, inp.eps, 0.03)
    np.testing.assert_array_equal(res, r_o)
    check_nvfp4(q, sf, q_o, sf_o, v, 0.03, orc, f"norm nvfp4 {shape}")


@pytest.mark.parametrize("T,I,shape", [(40, 8960, (5, 2, 128)), (3, 13824, (16, 1, 128)), (500, 3008, (1, 4, 96)),
                                       (257, 14336, (7, 1, 256)), (9, 53248, (8, 4, 224))])
def test_swiglu_forced_shapes(T, I, shape):
    inp = wl.make_swiglu_inputs(T, I, seed=T + I, dist=wl.C5_ACT)
    _, h = orc.swiglu(inp.gate_up)
    force("swiglu", None, T, I, shape)
    out, _ = gpu_swiglu(inp, "bf16")
    check_bf16(out, h, f"swiglu {shape}")
    force("swiglu_quant_fp8", "static", T, I, shape)
    q, _ = gpu_swiglu(inp, "q8", "static", static_scale=0.05)
    check_codes(q, orc.swiglu_quant_fp8(inp.gate_up, "static", 0.05)[0], f"swiglu q8 static {shape}")
    if shape[0] <= 8:   # the dynamic epilogue reduces over the row: one cluster at most
        force("swiglu_quant_fp8", "dynamic", T, I, shape)
        q, s = gpu_swiglu(inp, "q8", "dynamic")
        q_o, s_o, _ = orc.swiglu_quant_fp8(inp.gate_up, "dynamic")
        check_codes(q, q_o, f"swiglu q8 dynamic {shape}")
        check_scales(s, s_o, "swiglu scales")
    force("swiglu_quant_nvfp4", None, T, I, shape)
    q, sf = gpu_swiglu_nvfp4(inp, 0.17)
    q_o, sf_o, h2 = orc.swiglu_quant_nvfp4(inp.gate_up, 0.17)
    check_nvfp4(q, sf, q_o, sf_o, h2, 0.17, orc, f"swiglu nvfp4 {shape}")
    _mbd().tuning_set([])
