"""The static FP8 scale and the NVFP4 tensor scale are device inputs read after each launch's wait on the work
ahead of it in the stream: a scale that the launch before wrote (here the per-token scales of a dynamic-FP8 norm,
used as the next calls' static or tensor scale) or that the stream rewrote between two launches is the value
each launch uses. Covers the kernels that load the scale together with the weight, before the row reduction
(decode-size rows, the all-reduce half), and those that load it after the reduction (four vectors per thread).
Every launch runs back to back on one stream with a single synchronisation at the end; each launch's codes are
compared with the oracle at the scale that launch had to see. The scale buffer starts at 1.0, a value no launch
should use."""
import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests.parity import check_codes, check_nvfp4, check_scales

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS = 1e-5


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


def _dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).reshape(-1).copy()).cuda()


def _codes(t, T, W):
    return t.cpu().numpy().reshape(T, W)


@pytest.mark.parametrize("Tb,Hb,Tc,Hc", [(3, 16384, 5, 16384), (1200, 4096, 1500, 4096)])
def test_scales_written_by_the_launch_before(Tb, Hb, Tc, Hc):
    mbd = _mbd()
    h = torch.cuda.current_stream().cuda_stream
    # A: dynamic FP8 norm, writes the per-token scales S
    Ta, Ha = 4, 5120
    a = wl.make_norm_inputs(Ta, Ha, 11, wl.C5_ACT, EPS, salt=1)
    xa, ra, wa = _dev(a.x), _dev(a.residual), _dev(a.weight)
    qa = torch.empty(Ta * Ha, dtype=torch.uint8, device="cuda")
    S = torch.full((Ta,), 1.0, dtype=torch.float32, device="cuda")
    # B: static FP8 norm on scale S[0]; C: NVFP4 norm on tensor scale S[1]; D: all-reduce half on scale S[2]
    b = wl.make_norm_inputs(Tb, Hb, 12, wl.C5_ACT, EPS, salt=2)
    xb, rb, wb = _dev(b.x), _dev(b.residual), _dev(b.weight)
    qb = torch.empty(Tb * Hb, dtype=torch.uint8, device="cuda")
    c = wl.make_norm_inputs(Tc, Hc, 13, wl.C5_ACT, EPS, salt=3)
    xc, rc, wc = _dev(c.x), _dev(c.residual), _dev(c.weight)
    qc = torch.empty(Tc * Hc // 2, dtype=torch.uint8, device="cuda")
    sfc = torch.empty(Tc * Hc // 16, dtype=torch.uint8, device="cuda")
    Td, Hd, k = 3, 5120, 4
    ps = [wl.normal_bf16((Td, Hd), 14, "x", 1.0, salt=40 + j) for j in range(k)]
    rd_np, wd_np = wl.normal_bf16((Td, Hd), 14, "residual"), wl.weight_bf16(Hd, 14)
    dps, rd, wd = [_dev(p) for p in ps], _dev(rd_np), _dev(wd_np)
    qd = torch.empty(Td * Hd, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()

    mbd.fused_add_rmsnorm_quant_fp8(qa, ra, xa, wa, Ta, Ha, EPS, "dynamic", S, h)
    mbd.fused_add_rmsnorm_quant_fp8(qb, rb, xb, wb, Tb, Hb, EPS, "static", S.data_ptr(), h)
    mbd.fused_add_rmsnorm_quant_nvfp4(qc, sfc, rc, xc, wc, Tc, Hc, EPS, S.data_ptr() + 4, h)
    mbd.fused_allreduce_add_rmsnorm_quant_fp8(qd, rd, dps, wd, Td, Hd, EPS, "static", S.data_ptr() + 8, h)
    torch.cuda.synchronize()

    s_g = S.cpu().numpy()
    _, q_o, s_o, _ = orc.add_rmsnorm_quant_fp8(a.x, a.residual, a.weight, EPS, "dynamic")
    check_scales(s_g, s_o[:Ta], "dynamic scales")
    check_codes(_codes(qa, Ta, Ha), q_o, "dynamic norm")
    assert not (s_g[:3] == 1.0).any()

    _, q_o, _, _ = orc.add_rmsnorm_quant_fp8(b.x, b.residual, b.weight, EPS, "static", float(s_g[0]))
    check_codes(_codes(qb, Tb, Hb), q_o, "static norm on S[0]")

    _, q_o, sf_o, v = orc.add_rmsnorm_quant_nvfp4(c.x, c.residual, c.weight, EPS, float(s_g[1]))
    check_nvfp4(_codes(qc, Tc, Hc // 2), _codes(sfc, Tc, Hc // 16), q_o, sf_o, v, float(s_g[1]), orc,
                "NVFP4 norm on S[1]")

    _, q_o, _, _ = orc.allreduce_add_rmsnorm_quant_fp8(ps, rd_np, wd_np, EPS, "static", float(s_g[2]))
    check_codes(_codes(qd, Td, Hd), q_o, "all-reduce half on S[2]")


@pytest.mark.parametrize("T,H", [(1, 16384), (17, 5120), (1200, 4096)])
def test_static_scale_rewritten_between_launches(T, H):
    """Three launches on one residual snapshot, the scale rewritten on the stream before each."""
    mbd = _mbd()
    h = torch.cuda.current_stream().cuda_stream
    inp = wl.make_norm_inputs(T, H, 21, wl.C5_ACT, EPS)
    x, r0, w = _dev(inp.x), _dev(inp.residual), _dev(inp.weight)
    r = torch.empty_like(r0)
    sc = torch.full((1,), 1.0, dtype=torch.float32, device="cuda")
    scales = [0.05, 0.011, 0.2]
    outs = []
    for s in scales:
        r.copy_(r0)
        sc.fill_(s)
        q = torch.empty(T * H, dtype=torch.uint8, device="cuda")
        mbd.fused_add_rmsnorm_quant_fp8(q, r, x, w, T, H, EPS, "static", sc, h)
        outs.append(q)
    torch.cuda.synchronize()
    for s, q in zip(scales, outs):
        _, q_o, _, _ = orc.add_rmsnorm_quant_fp8(inp.x, inp.residual, inp.weight, EPS, "static", s)
        check_codes(_codes(q, T, H), q_o, f"static scale {s}")
