"""Programs (mbd_run_program): lists of fused ops in one persistent launch, checked against the fp64 oracle run
op by op in list order.

Chains (ops linked by a shared, written buffer) must keep list order per row: the decode-step layers share
one residual across all their norms, an output may feed a later op in place, and two ops writing the same
buffer must leave the later op's values. Independent ops are spread over the grid in chunks.
"""
import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests.parity import Guarded, check_bf16, check_codes, check_nvfp4, check_scales, dev_u16

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


def run(ops, guards=()):
    mbd = _mbd()
    mbd.device_error_flags(clear=True)
    n0 = mbd.kernel_launches()
    mbd.run_program(ops)
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == 1
    assert mbd.device_error_flags() == 0
    for g, name in guards:
        g.check_guards(name)


def u16(g, shape):
    return g.numpy(np.uint16).reshape(shape)


def decode_layers(T, L, H=1536, I=8960, seed=0, dist=wl.N01, eps=1e-6):
    """L layers of (add_rmsnorm, add_rmsnorm, swiglu) inputs sharing one residual, like a decode step."""
    res0 = wl.make_norm_inputs(T, H, seed, dist, eps, salt=999).residual
    layers = []
    for l in range(L):
        n1 = wl.make_norm_inputs(T, H, seed, dist, eps, salt=3 * l)
        n2 = wl.make_norm_inputs(T, H, seed, dist, eps, salt=3 * l + 1)
        gu = wl.make_swiglu_inputs(T, I, seed, dist, salt=3 * l + 2)
        layers.append((n1.x, n1.weight, n2.x, n2.weight, gu.gate_up))
    return res0, layers


@pytest.mark.parametrize("T", [1, 3, 64, 256])
def test_decode_step_bf16(T):
    """28 layers x (norm, norm, SwiGLU), all norms updating one residual: the C2 decode step."""
    mbd = _mbd()
    H, I, L, eps = 1536, 8960, 28, 1e-6
    res0, layers = decode_layers(T, L, H, I, seed=T)
    R = dev_u16(torch, res0)
    ops, keep, outs = [], [R], []
    for x1, w1, x2, w2, gu in layers:
        X1, W1, X2, W2, GU = (dev_u16(torch, a) for a in (x1, w1, x2, w2, gu))
        O1, O2 = Guarded(torch, T * H, torch.int16), Guarded(torch, T * H, torch.int16)
        Y = Guarded(torch, T * I, torch.int16)
        ops += [mbd.op_add_rmsnorm(O1.view, R.view, X1.view, W1.view, T, H, eps),
                mbd.op_add_rmsnorm(O2.view, R.view, X2.view, W2.view, T, H, eps),
                mbd.op_swiglu(Y.view, GU.view, T, I)]
        keep += [X1, W1, X2, W2, GU]
        outs.append((O1, O2, Y))
    run(ops, [(R, "residual")] + [(g, "out") for o in outs for g in o])
    r = res0
    for (x1, w1, x2, w2, gu), (O1, O2, Y) in zip(layers, outs):
        r, _, v1 = orc.add_rmsnorm(x1, r, w1, eps)
        check_bf16(u16(O1, (T, H)), v1, "layer norm 1")
        r, _, v2 = orc.add_rmsnorm(x2, r, w2, eps)
        check_bf16(u16(O2, (T, H)), v2, "layer norm 2")
        _, h = orc.swiglu(gu)
        check_bf16(u16(Y, (T, I)), h, "layer swiglu")
    np.testing.assert_array_equal(u16(R, (T, H)), r, "final residual must be bit-exact")


@pytest.mark.parametrize("T,H,I", [(1, 1536, 8960), (17, 1536, 8960), (200, 1536, 8960), (9, 4096, 13824),
                                   (3, 8192, 8192)])
def test_decode_step_fp8(T, H, I):
    """Layers of (norm -> E4M3 static, SwiGLU -> E4M3 dynamic) sharing the residual. With 1536-wide norms the
    chained norms keep the residual row in registers at 1 vector per thread, and the 8960-wide SwiGLU rows take
    the two-pass dynamic form; with 4096-wide norms (2 vectors per thread) the 13824-wide rows are held whole
    at 8 vectors per thread; 8192 at 4 vectors per thread is held in one pass."""
    mbd = _mbd()
    L, eps, S = 8, 1e-5, 0.05
    res0, layers = decode_layers(T, L, H, I, seed=T + 100, dist=wl.C5_ACT, eps=eps)
    R = dev_u16(torch, res0)
    sc = Guarded(torch, 1, torch.float32, fill=np.array([S], np.float32))
    ops, keep, outs = [], [R, sc], []
    for x1, w1, _, _, gu in layers:
        X1, W1, GU = (dev_u16(torch, a) for a in (x1, w1, gu))
        Q1 = Guarded(torch, T * H, torch.uint8)
        Q2, S2 = Guarded(torch, T * I, torch.uint8), Guarded(torch, T, torch.float32)
        ops += [mbd.op_add_rmsnorm_quant_fp8(Q1.view, R.view, X1.view, W1.view, T, H, eps, "static", sc.view),
                mbd.op_swiglu_quant_fp8(Q2.view, GU.view, T, I, "dynamic", S2.view)]
        keep += [X1, W1, GU]
        outs.append((Q1, Q2, S2))
    run(ops, [(R, "residual")] + [(g, "out") for o in outs for g in o])
    r = res0
    for (x1, w1, _, _, gu), (Q1, Q2, S2) in zip(layers, outs):
        r, q_o, _, _ = orc.add_rmsnorm_quant_fp8(x1, r, w1, eps, "static", S)
        check_codes(Q1.numpy(np.uint8).reshape(T, H), q_o, "norm e4m3")
        q_o, s_o, _ = orc.swiglu_quant_fp8(gu, "dynamic")
        check_codes(Q2.numpy(np.uint8).reshape(T, I), q_o, "swiglu e4m3")
        check_scales(S2.numpy(np.float32), s_o, "swiglu scales")
    np.testing.assert_array_equal(u16(R, (T, H)), r)


@pytest.mark.parametrize("T", [2, 33])
def test_decode_step_nvfp4(T):
    mbd = _mbd()
    H, I, L, eps, S1, S2 = 1536, 8960, 6, 1e-5, 0.03, 0.17
    res0, layers = decode_layers(T, L, H, I, seed=T + 200, dist=wl.C5_ACT, eps=eps)
    R = dev_u16(torch, res0)
    s1 = Guarded(torch, 1, torch.float32, fill=np.array([S1], np.float32))
    s2 = Guarded(torch, 1, torch.float32, fill=np.array([S2], np.float32))
    ops, keep, outs = [], [R, s1, s2], []
    for x1, w1, _, _, gu in layers:
        X1, W1, GU = (dev_u16(torch, a) for a in (x1, w1, gu))
        Q1, F1 = Guarded(torch, T * H // 2, torch.uint8), Guarded(torch, T * H // 16, torch.uint8)
        Q2, F2 = Guarded(torch, T * I // 2, torch.uint8), Guarded(torch, T * I // 16, torch.uint8)
        ops += [mbd.op_add_rmsnorm_quant_nvfp4(Q1.view, F1.view, R.view, X1.view, W1.view, T, H, eps, s1.view),
                mbd.op_swiglu_quant_nvfp4(Q2.view, F2.view, GU.view, T, I, s2.view)]
        keep += [X1, W1, GU]
        outs.append((Q1, F1, Q2, F2))
    run(ops, [(R, "residual")] + [(g, "out") for o in outs for g in o])
    r = res0
    for (x1, w1, _, _, gu), (Q1, F1, Q2, F2) in zip(layers, outs):
        r, q_o, f_o, v = orc.add_rmsnorm_quant_nvfp4(x1, r, w1, eps, S1)
        check_nvfp4(Q1.numpy(np.uint8).reshape(T, H // 2), F1.numpy(np.uint8).reshape(T, H // 16), q_o, f_o, v, S1,
                    orc, "norm nvfp4")
        q_o, f_o, h = orc.swiglu_quant_nvfp4(gu, S2)
        check_nvfp4(Q2.numpy(np.uint8).reshape(T, I // 2), F2.numpy(np.uint8).reshape(T, I // 16), q_o, f_o, h, S2,
                    orc, "swiglu nvfp4")
    np.testing.assert_array_equal(u16(R, (T, H)), r)


def test_output_feeds_next_op_in_place():
    """op 2 normalises op 1's output (same tensor): it must see op 1's values, row by row."""
    mbd = _mbd()
    T, H, eps = 40, 4096, 1e-5
    a = wl.make_norm_inputs(T, H, 1, wl.C3_ACT, eps, salt=1)
    b = wl.make_norm_inputs(T, H, 1, wl.C3_ACT, eps, salt=2)
    X0, R1, W1, R2, W2 = (dev_u16(torch, v) for v in (a.x, a.residual, a.weight, b.residual, b.weight))
    A, B = Guarded(torch, T * H, torch.int16), Guarded(torch, T * H, torch.int16)
    run([mbd.op_add_rmsnorm(A.view, R1.view, X0.view, W1.view, T, H, eps),
         mbd.op_add_rmsnorm(B.view, R2.view, A.view, W2.view, T, H, eps)], [(A, "A"), (B, "B")])
    a_gpu = u16(A, (T, H))
    r1, _, v1 = orc.add_rmsnorm(a.x, a.residual, a.weight, eps)
    check_bf16(a_gpu, v1, "op 1")
    np.testing.assert_array_equal(u16(R1, (T, H)), r1)
    r2, _, v2 = orc.add_rmsnorm(a_gpu, b.residual, b.weight, eps)   # op 2 reads op 1's rounded output
    check_bf16(u16(B, (T, H)), v2, "op 2")
    np.testing.assert_array_equal(u16(R2, (T, H)), r2)


def test_later_write_wins_across_chunks():
    """Two SwiGLUs writing one buffer form a chain: its rows are processed in 256-vector chunks, and every
    chunk must end with the second op's values."""
    mbd = _mbd()
    T, I = 9, 8960
    g1 = wl.make_swiglu_inputs(T, I, 4, wl.N01, salt=1)
    g2 = wl.make_swiglu_inputs(T, I, 4, wl.N01, salt=2)
    G1, G2 = dev_u16(torch, g1.gate_up), dev_u16(torch, g2.gate_up)
    O = Guarded(torch, T * I, torch.int16)
    n = wl.make_norm_inputs(T, 1536, 4, wl.N01, 1e-6)
    X, R, W = dev_u16(torch, n.x), dev_u16(torch, n.residual), dev_u16(torch, n.weight)
    N = Guarded(torch, T * 1536, torch.int16)
    run([mbd.op_swiglu(O.view, G1.view, T, I), mbd.op_add_rmsnorm(N.view, R.view, X.view, W.view, T, 1536, 1e-6),
         mbd.op_swiglu(O.view, G2.view, T, I)], [(O, "O"), (N, "N")])
    _, h2 = orc.swiglu(g2.gate_up)
    check_bf16(u16(O, (T, I)), h2, "second write")
    _, _, v = orc.add_rmsnorm(n.x, n.residual, n.weight, 1e-6)
    check_bf16(u16(N, (T, 1536)), v, "independent norm")


def test_independent_ops_of_mixed_shapes():
    """No shared buffers: every op is split into (row, chunk) items over the grid (2 vectors per thread here,
    set by the 4096-wide norm)."""
    mbd = _mbd()
    ops, checks, keep = [], [], []
    for k, (T, I) in enumerate([(1, 512), (5, 4096), (100, 13824), (3, 8960), (64, 256)]):
        g = wl.make_swiglu_inputs(T, I, 7, wl.C3_GU, salt=k)
        GU = dev_u16(torch, g.gate_up)
        Y = Guarded(torch, T * I, torch.int16)
        ops.append(mbd.op_swiglu(Y.view, GU.view, T, I))
        keep.append(GU)
        checks.append(("swiglu", g, Y, T, I))
    for k, (T, H) in enumerate([(1, 4096), (37, 1536), (300, 2048)]):
        n = wl.make_norm_inputs(T, H, 8, wl.C3_ACT, 1e-5, salt=k)
        X, R, W = dev_u16(torch, n.x), dev_u16(torch, n.residual), dev_u16(torch, n.weight)
        O = Guarded(torch, T * H, torch.int16)
        ops.append(mbd.op_add_rmsnorm(O.view, R.view, X.view, W.view, T, H, n.eps))
        keep += [X, W]
        checks.append(("norm", n, (O, R), T, H))
    run(ops, [(c[2], "out") for c in checks if c[0] == "swiglu"] + [(c[2][0], "out") for c in checks if c[0] == "norm"])
    for kind, inp, g, T, W in checks:
        if kind == "swiglu":
            _, h = orc.swiglu(inp.gate_up)
            check_bf16(u16(g, (T, W)), h, f"swiglu {T}x{W}")
        else:
            r, _, v = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, inp.eps)
            check_bf16(u16(g[0], (T, W)), v, f"norm {T}x{W}")
            np.testing.assert_array_equal(u16(g[1], (T, W)), r)


@pytest.mark.parametrize("I", [13824, 16384, 16400])
def test_mixed_bf16_fp8_independent_calls(I):
    """bf16 and FP8 ops in one launch (the mixed variant), as independent calls at 1, 3 and 17 tokens: norms
    5120 wide (bf16, static FP8) and SwiGLU (bf16, static FP8, dynamic FP8). A dynamic row of 13824 or 16384
    elements is held whole at 8 vectors per thread; 16400 (2050 vectors) takes the two-pass form."""
    mbd = _mbd()
    H, eps, S = 5120, 1e-5, 0.05
    sc = Guarded(torch, 1, torch.float32, fill=np.array([S], np.float32))
    ops, checks, keep, guards = [], [], [sc], []
    for k, T in enumerate([1, 3, 17]):
        for q in (False, True):
            n = wl.make_norm_inputs(T, H, 11, wl.C5_ACT, eps, salt=10 * k + int(q))
            X, R, W = dev_u16(torch, n.x), dev_u16(torch, n.residual), dev_u16(torch, n.weight)
            O = Guarded(torch, T * H, torch.uint8 if q else torch.int16)
            ops.append(mbd.op_add_rmsnorm_quant_fp8(O.view, R.view, X.view, W.view, T, H, eps, "static", sc.view)
                       if q else mbd.op_add_rmsnorm(O.view, R.view, X.view, W.view, T, H, eps))
            keep += [X, W]
            guards += [(O, "norm out"), (R, "residual")]
            checks.append(("norm", q, n, (O, R), T))
        for j, mode in enumerate((None, "static", "dynamic")):
            g = wl.make_swiglu_inputs(T, I, 11, wl.C5_ACT, salt=10 * k + 2 + j)
            GU = dev_u16(torch, g.gate_up)
            Y = Guarded(torch, T * I, torch.int16 if mode is None else torch.uint8)
            SY = sc if mode != "dynamic" else Guarded(torch, T, torch.float32)
            ops.append(mbd.op_swiglu(Y.view, GU.view, T, I) if mode is None
                       else mbd.op_swiglu_quant_fp8(Y.view, GU.view, T, I, mode, SY.view))
            keep.append(GU)
            guards.append((Y, "swiglu out"))
            if mode == "dynamic":
                guards.append((SY, "swiglu scales"))
            checks.append(("swiglu", mode, g, (Y, SY), T))
    run(ops, guards)
    for kind, mode, inp, g, T in checks:
        if kind == "norm":
            O, R = g
            if mode:
                r, q_o, _, _ = orc.add_rmsnorm_quant_fp8(inp.x, inp.residual, inp.weight, eps, "static", S)
                check_codes(O.numpy(np.uint8).reshape(T, H), q_o, f"norm e4m3 T={T}")
            else:
                r, _, v = orc.add_rmsnorm(inp.x, inp.residual, inp.weight, eps)
                check_bf16(u16(O, (T, H)), v, f"norm T={T}")
            np.testing.assert_array_equal(u16(R, (T, H)), r, f"residual T={T}")
        elif mode is None:
            _, h = orc.swiglu(inp.gate_up)
            check_bf16(u16(g[0], (T, I)), h, f"swiglu T={T}")
        else:
            q_o, s_o, _ = orc.swiglu_quant_fp8(inp.gate_up, mode, S if mode == "static" else 0.0)
            check_codes(g[0].numpy(np.uint8).reshape(T, I), q_o, f"swiglu e4m3 {mode} T={T}")
            if mode == "dynamic":
                check_scales(g[1].numpy(np.float32), s_o, f"swiglu scales T={T}")


def test_mixed_chain_across_epilogues():
    """One residual updated by a bf16 norm, then a static-FP8 norm, then a bf16 norm (a chain in the mixed
    variant), beside independent SwiGLU ops: dynamic FP8 (13824 wide, held whole at 8 vectors per thread) and
    static FP8."""
    mbd = _mbd()
    T, H, I, eps, S = 6, 4096, 13824, 1e-6, 0.05
    sc = Guarded(torch, 1, torch.float32, fill=np.array([S], np.float32))
    base = wl.make_norm_inputs(T, H, 12, wl.N01, eps, salt=0)
    R = dev_u16(torch, base.residual)
    xs = [wl.make_norm_inputs(T, H, 12, wl.N01, eps, salt=k + 1) for k in range(3)]
    ops, keep, outs = [], [R, sc], []
    for k, n in enumerate(xs):
        X, W = dev_u16(torch, n.x), dev_u16(torch, n.weight)
        O = Guarded(torch, T * H, torch.uint8 if k == 1 else torch.int16)
        ops.append(mbd.op_add_rmsnorm_quant_fp8(O.view, R.view, X.view, W.view, T, H, eps, "static", sc.view)
                   if k == 1 else mbd.op_add_rmsnorm(O.view, R.view, X.view, W.view, T, H, eps))
        keep += [X, W]
        outs.append(O)
    gd = wl.make_swiglu_inputs(T, I, 12, wl.N01, salt=7)
    gs = wl.make_swiglu_inputs(T, I, 12, wl.N01, salt=8)
    GD, GS = dev_u16(torch, gd.gate_up), dev_u16(torch, gs.gate_up)
    QD, SD = Guarded(torch, T * I, torch.uint8), Guarded(torch, T, torch.float32)
    QS = Guarded(torch, T * I, torch.uint8)
    ops += [mbd.op_swiglu_quant_fp8(QD.view, GD.view, T, I, "dynamic", SD.view),
            mbd.op_swiglu_quant_fp8(QS.view, GS.view, T, I, "static", sc.view)]
    keep += [GD, GS]
    run(ops, [(R, "residual"), (QD, "q"), (SD, "s"), (QS, "q")] + [(o, "out") for o in outs])
    r = base.residual
    for k, (n, O) in enumerate(zip(xs, outs)):
        if k == 1:
            r, q_o, _, _ = orc.add_rmsnorm_quant_fp8(n.x, r, n.weight, eps, "static", S)
            check_codes(O.numpy(np.uint8).reshape(T, H), q_o, "chained e4m3 norm")
        else:
            r, _, v = orc.add_rmsnorm(n.x, r, n.weight, eps)
            check_bf16(u16(O, (T, H)), v, f"chained norm {k}")
    np.testing.assert_array_equal(u16(R, (T, H)), r)
    q_o, s_o, _ = orc.swiglu_quant_fp8(gd.gate_up, "dynamic")
    check_codes(QD.numpy(np.uint8).reshape(T, I), q_o, "dynamic swiglu")
    check_scales(SD.numpy(np.float32), s_o, "dynamic swiglu scales")
    q_o, _, _ = orc.swiglu_quant_fp8(gs.gate_up, "static", S)
    check_codes(QS.numpy(np.uint8).reshape(T, I), q_o, "static swiglu")


def test_widest_held_rows_dynamic():
    """Norm chains and a dynamic SwiGLU at the widest row a CTA holds (8192: 4 vectors per thread)."""
    mbd = _mbd()
    T, H, eps = 5, 8192, 1e-5
    base = wl.make_norm_inputs(T, H, 9, wl.C5_ACT, eps, salt=0)
    R = dev_u16(torch, base.residual)
    sc = Guarded(torch, 1, torch.float32, fill=np.array([0.05], np.float32))
    ops, keep, outs = [], [R, sc], []
    xs = [wl.make_norm_inputs(T, H, 9, wl.C5_ACT, eps, salt=k + 1) for k in range(3)]
    for n in xs:
        X, W = dev_u16(torch, n.x), dev_u16(torch, n.weight)
        Q = Guarded(torch, T * H, torch.uint8)
        ops.append(mbd.op_add_rmsnorm_quant_fp8(Q.view, R.view, X.view, W.view, T, H, eps, "static", sc.view))
        keep += [X, W]
        outs.append(Q)
    g = wl.make_swiglu_inputs(T, 8192, 9, wl.C5_ACT)
    GU = dev_u16(torch, g.gate_up)
    QS, SS = Guarded(torch, T * 8192, torch.uint8), Guarded(torch, T, torch.float32)
    ops.append(mbd.op_swiglu_quant_fp8(QS.view, GU.view, T, 8192, "dynamic", SS.view))
    run(ops, [(R, "residual"), (QS, "q"), (SS, "s")] + [(q, "q") for q in outs])
    r = base.residual
    for n, Q in zip(xs, outs):
        r, q_o, _, _ = orc.add_rmsnorm_quant_fp8(n.x, r, n.weight, eps, "static", 0.05)
        check_codes(Q.numpy(np.uint8).reshape(T, H), q_o, "held norm")
    np.testing.assert_array_equal(u16(R, (T, H)), r)
    q_o, s_o, _ = orc.swiglu_quant_fp8(g.gate_up, "dynamic")
    check_codes(QS.numpy(np.uint8).reshape(T, 8192), q_o, "held swiglu")
    check_scales(SS.numpy(np.float32), s_o, "held swiglu scales")


def test_program_matches_single_calls():
    """The same ops as individual entry-point calls: residuals bit-identical, bf16 outputs within one ulp
    (a row reduced inside one CTA may sum in another order than a row split over a cluster)."""
    mbd = _mbd()
    T, L, H, I, eps = 17, 4, 1536, 8960, 1e-6
    res0, layers = decode_layers(T, L, H, I, seed=5)
    outs = {}
    for mode in ("calls", "program"):
        R = dev_u16(torch, res0)
        ops, keep, got = [], [R], []
        for x1, w1, x2, w2, gu in layers:
            X1, W1, X2, W2, GU = (dev_u16(torch, a) for a in (x1, w1, x2, w2, gu))
            O1, O2, Y = (torch.empty(T * n, dtype=torch.int16, device="cuda") for n in (H, H, I))
            ops += [mbd.op_add_rmsnorm(O1, R.view, X1.view, W1.view, T, H, eps),
                    mbd.op_add_rmsnorm(O2, R.view, X2.view, W2.view, T, H, eps), mbd.op_swiglu(Y, GU.view, T, I)]
            if mode == "calls":
                mbd.fused_add_rmsnorm(O1, R.view, X1.view, W1.view, T, H, eps)
                mbd.fused_add_rmsnorm(O2, R.view, X2.view, W2.view, T, H, eps)
                mbd.swiglu(Y, GU.view, T, I)
            keep += [X1, W1, X2, W2, GU]
            got += [O1, O2, Y]
        if mode == "program":
            mbd.run_program(ops)
        torch.cuda.synchronize()
        outs[mode] = (R.numpy(np.uint16), [t.cpu().numpy().view(np.uint16) for t in got])
    np.testing.assert_array_equal(outs["calls"][0], outs["program"][0])
    for a, b in zip(outs["calls"][1], outs["program"][1]):
        d = np.abs(a.astype(np.int32) - b.astype(np.int32))
        assert d.max() <= 1, "outputs differ by more than one bf16 ulp"


def test_plan_built_once_launched_twice():
    """A plan is built once and launched twice: the second launch sees the residual the first one left, as
    two decode steps through the same layers would."""
    mbd = _mbd()
    T, L, H, I, eps = 3, 4, 1536, 8960, 1e-6
    res0, layers = decode_layers(T, L, H, I, seed=11)
    R = dev_u16(torch, res0)
    ops, keep, outs = [], [R], []
    for x1, w1, x2, w2, gu in layers:
        X1, W1, X2, W2, GU = (dev_u16(torch, a) for a in (x1, w1, x2, w2, gu))
        O1, O2, Y = Guarded(torch, T * H, torch.int16), Guarded(torch, T * H, torch.int16), Guarded(torch, T * I, torch.int16)
        ops += [mbd.op_add_rmsnorm(O1.view, R.view, X1.view, W1.view, T, H, eps),
                mbd.op_add_rmsnorm(O2.view, R.view, X2.view, W2.view, T, H, eps), mbd.op_swiglu(Y.view, GU.view, T, I)]
        keep += [X1, W1, X2, W2, GU]
        outs.append((O1, O2, Y))
    plan = mbd.program_plan_build(ops)
    n0 = mbd.kernel_launches()
    plan.launch()
    plan.launch()
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == 2
    r = res0
    for step in range(2):
        for (x1, w1, x2, w2, gu), (O1, O2, Y) in zip(layers, outs):
            r, _, v1 = orc.add_rmsnorm(x1, r, w1, eps)
            r, _, v2 = orc.add_rmsnorm(x2, r, w2, eps)
            if step == 1:
                check_bf16(u16(O1, (T, H)), v1, "step 2 norm 1")
                check_bf16(u16(O2, (T, H)), v2, "step 2 norm 2")
    np.testing.assert_array_equal(u16(R, (T, H)), r, "residual after two launches")


def test_uploaded_schedule_matches_by_value_launch():
    """The same plan launched twice with its schedule by value and twice from an uploaded copy: identical bits
    (same kernel body, same schedule)."""
    mbd = _mbd()
    T, L, H, I, eps = 5, 6, 1536, 8960, 1e-6
    res0, layers = decode_layers(T, L, H, I, seed=12)
    results = []
    for mode in ("value", "uploaded"):
        R = dev_u16(torch, res0)
        ops, keep, outs = [], [R], []
        for x1, w1, x2, w2, gu in layers:
            X1, W1, X2, W2, GU = (dev_u16(torch, a) for a in (x1, w1, x2, w2, gu))
            O1, O2, Y = (torch.empty(T * n, dtype=torch.int16, device="cuda") for n in (H, H, I))
            ops += [mbd.op_add_rmsnorm(O1, R.view, X1.view, W1.view, T, H, eps),
                    mbd.op_add_rmsnorm(O2, R.view, X2.view, W2.view, T, H, eps), mbd.op_swiglu(Y, GU.view, T, I)]
            keep += [X1, W1, X2, W2, GU]
            outs += [O1, O2, Y]
        plan = mbd.program_plan_build(ops)
        if mode == "value":
            plan.launch()
            plan.launch()
        else:
            sched = torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device="cuda")
            plan.upload(sched)
            plan.launch_uploaded(sched)
            plan.launch_uploaded(sched)
        torch.cuda.synchronize()
        results.append([R.numpy(np.uint16)] + [t.cpu().numpy() for t in outs])
    for a, b in zip(*results):
        np.testing.assert_array_equal(a, b)
