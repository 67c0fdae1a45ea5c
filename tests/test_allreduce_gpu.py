"""Parity of the all-reduce half + add + RMSNorm entry points (n partial activations summed exactly, rounded
once to bf16, then the fused norm) against the oracle, including the n = 1 identity with the plain fused
norm, in-place output, every epilogue and the direct and large-batch launch shapes."""
import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests.parity import Guarded, check_bf16, check_codes, check_scales, dev_u16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_decoder_gb300 import build
    build.build()
    orc.build()


def _mbd():
    import memory_bound_decoder_gb300 as mbd
    return mbd


def partials_for(k, T, H, seed, dist=wl.C5_ACT):
    return [wl.normal_bf16((T, H), seed, "x", dist.sigma, dist.outlier_p, dist.outlier_k, salt=100 + j)
            for j in range(k)]


def run(ps, r, w, eps, ep, mode=None, static_scale=0.05, inplace=False):
    mbd = _mbd()
    T, H = r.shape
    dps = [dev_u16(torch, p) for p in ps]
    dr, dw = dev_u16(torch, r), dev_u16(torch, w)
    sc = None
    n0 = mbd.kernel_launches()
    if ep == "bf16":
        out = dps[0] if inplace else Guarded(torch, T * H, torch.int16)
        mbd.fused_allreduce_add_rmsnorm(out.view, dr.view, [d.view for d in dps], dw.view, T, H, eps)
    else:
        out = Guarded(torch, T * H, torch.uint8)
        sc = (Guarded(torch, 1, torch.float32, fill=np.array([static_scale], np.float32)) if mode == "static"
              else Guarded(torch, T, torch.float32))
        mbd.fused_allreduce_add_rmsnorm_quant_fp8(out.view, dr.view, [d.view for d in dps], dw.view, T, H, eps,
                                                  mode, sc.view)
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == 1
    for g in dps + [dr, dw, out] + ([sc] if sc else []):
        g.check_guards()
    for d, p in zip(dps[1:] if inplace else dps, ps[1:] if inplace else ps):
        np.testing.assert_array_equal(d.numpy(np.uint16), p.reshape(-1), "a partial was modified")
    res = dr.numpy(np.uint16).reshape(T, H)
    o = out.view.cpu().numpy()
    o = o.view(np.uint16).reshape(T, H) if ep == "bf16" else o.reshape(T, H)
    s = sc.view.cpu().numpy() if sc is not None else None
    return res, o, s


CASES = [(1, 16, 5120), (2, 3, 5120), (3, 17, 1536), (4, 64, 4096), (8, 5, 520), (2, 400, 8192), (4, 1000, 5120),
         (8, 300, 16384), (3, 2, 32768)]


@pytest.mark.parametrize("k,T,H", CASES)
@pytest.mark.parametrize("ep,mode", [("bf16", None), ("q8", "static"), ("q8", "dynamic")])
def test_allreduce_parity(k, T, H, ep, mode):
    ps = partials_for(k, T, H, seed=k * 31 + T)
    r = wl.normal_bf16((T, H), k + T, "residual", 1.0, 0.001, 100.0)
    w = wl.weight_bf16(H, k)
    eps = 1e-5
    res_g, o_g, s_g = run(ps, r, w, eps, ep, mode)
    if ep == "bf16":
        res_o, _, v = orc.allreduce_add_rmsnorm(ps, r, w, eps)
        np.testing.assert_array_equal(res_g, res_o, "residual must be bit-exact")
        check_bf16(o_g, v, "allreduce_add_rmsnorm")
    else:
        res_o, q_o, s_o, _ = orc.allreduce_add_rmsnorm_quant_fp8(ps, r, w, eps, mode, 0.05)
        np.testing.assert_array_equal(res_g, res_o, "residual must be bit-exact")
        if mode == "dynamic":
            check_scales(s_g, s_o, "scale")
        check_codes(o_g, q_o, f"allreduce q8 {mode}")


def test_single_partial_equals_plain_fused_norm_on_gpu():
    mbd = _mbd()
    inp = wl.make_norm_inputs(37, 4096, 2, wl.C3_ACT, 1e-5)
    a_res, a_out, _ = run([inp.x], inp.residual, inp.weight, 1e-5, "bf16")
    x, r, w = dev_u16(torch, inp.x), dev_u16(torch, inp.residual), dev_u16(torch, inp.weight)
    out = torch.empty(37 * 4096, dtype=torch.int16, device="cuda")
    mbd.fused_add_rmsnorm(out, r.view, x.view, w.view, 37, 4096, 1e-5)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a_res, r.numpy(np.uint16).reshape(37, 4096))
    np.testing.assert_array_equal(a_out, out.cpu().numpy().view(np.uint16).reshape(37, 4096))


def test_inplace_out_is_first_partial():
    ps = partials_for(3, 33, 2048, seed=5)
    r = wl.normal_bf16((33, 2048), 5, "residual")
    w = wl.weight_bf16(2048, 5)
    res_g, o_g, _ = run(ps, r, w, 1e-6, "bf16", inplace=True)
    res_o, _, v = orc.allreduce_add_rmsnorm(ps, r, w, 1e-6)
    np.testing.assert_array_equal(res_g, res_o)
    check_bf16(o_g, v, "in place")


def _bf16(x):
    return wl.f32_to_bf16_bits(np.asarray(x, np.float32))


def _adversarial_partials(k, T, H, seed):
    """Partials whose sums stress the exactness test of the partial sum: every row mixes four constructions,
    column by column (each appears in every 32-lane warp's vectors).
      - wide spans: partial 0 scaled by 2^20, partial 1 by 2^-10 (the fp32 sum is inexact);
      - near ties tipped by tiny terms: partial 0 a bf16 value, partial 1 half its bf16 ulp (the two sum exactly
        to a rounding midpoint), the rest +-2^-(9..40) of it, so the exact sum lies just off the midpoint;
      - cancellation: partial 1 = -partial 0, the rest small;
      - zeros of either sign and bf16 subnormals."""
    rng = np.random.default_rng(seed)
    p = rng.standard_normal((k, T, H))
    kind = rng.integers(0, 4, (T, H))
    wide = kind == 0
    if k >= 2:
        p[0][wide] *= 2.0 ** 20
        p[1][wide] *= 2.0 ** -10
    tie = kind == 1
    base = wl.bf16_bits_to_f32(_bf16(p[0] * 4)).astype(np.float64)
    e = np.floor(np.log2(np.maximum(np.abs(base), 1e-30)))
    if k >= 2:
        p[0][tie] = base[tie]
        p[1][tie] = (np.sign(base) * 2.0 ** (e - 8))[tie]
        for j in range(2, k):
            p[j][tie] = (rng.choice([-1.0, 1.0], (T, H)) * 2.0 ** (e - 8 - rng.integers(1, 33, (T, H))))[tie]
    canc = kind == 2
    if k >= 2:
        p[0][canc] = wl.bf16_bits_to_f32(_bf16(p[0]))[canc]
        p[1][canc] = -p[0][canc]
        for j in range(2, k):
            p[j][canc] *= 1e-3
    odd = kind == 3
    z = rng.integers(0, 4, (k, T, H))
    for j in range(k):
        p[j][odd & (z[j] == 0)] = 0.0
        p[j][odd & (z[j] == 1)] = -0.0
        p[j][odd & (z[j] == 2)] *= 2.0 ** -130          # bf16 subnormals
    return [_bf16(p[j]) for j in range(k)]


@pytest.mark.parametrize("k,T,H", [(8, 64, 4096), (2, 33, 1536), (3, 300, 8192), (4, 5, 16384), (8, 2048, 1024)])
def test_allreduce_exactness_edges(k, T, H):
    """The reduced activation equals the bf16 rounding of the exact sum where the fp32 sum is inexact, lands on
    a rounding midpoint, cancels, or meets zeros and subnormals: the residual is compared bit for bit."""
    ps = _adversarial_partials(k, T, H, seed=k * 7 + T)
    r = wl.normal_bf16((T, H), T, "residual")
    w = wl.weight_bf16(H, k)
    res_g, o_g, _ = run(ps, r, w, 1e-5, "bf16")
    res_o, _, v = orc.allreduce_add_rmsnorm(ps, r, w, 1e-5)
    np.testing.assert_array_equal(res_g, res_o, "residual must be bit-exact")
    check_bf16(o_g, v, "allreduce_add_rmsnorm")


def test_allreduce_all_zero_partials_keep_the_sign_of_the_exact_sum():
    """Every partial -0: the exact sum is +0 (an empty sum plus -0 terms), so x = +0 and the residual keeps its
    own bits (r + 0 = r, including r = -0)."""
    T, H, k = 4, 1024, 8
    ps = [np.full((T, H), 0x8000, np.uint16) for _ in range(k)]
    r = wl.normal_bf16((T, H), 3, "residual")
    r[:, ::3] = 0x8000                                     # -0 residuals: -0 + x must give what +0 + -0 gives
    w = wl.weight_bf16(H, 1)
    res_g, _, _ = run(ps, r, w, 1e-5, "bf16")
    res_o, _, _ = orc.allreduce_add_rmsnorm(ps, r, w, 1e-5)
    np.testing.assert_array_equal(res_g, res_o)
