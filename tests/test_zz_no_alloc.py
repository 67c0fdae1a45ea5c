"""mbd_program_plan_launch_static, the program launch that allocates nothing, for callers that cannot allocate
device memory (engines that keep nearly all HBM in their own pool, plug-in interfaces that hand a kernel only
its inputs and outputs, loops that cannot afford cudaMalloc's possible device synchronisation): its schedule
goes to a static buffer of the library instead of caller memory. Checked against the entry point it stands in for
(mbd_program_plan_upload into a caller buffer + mbd_program_plan_launch_uploaded): two consecutive calls of
each, on identical fresh inputs, give identical bits; plans may alternate through the shared buffer; the
calls take no device memory. Also checked directly against the oracle: two static launches in a row of a
decode step, the second on the residual the first left, with bf16 outputs within tolerance and the final
residual bit-exact. Collected last (file name), after every other GPU test.
"""
import numpy as np
import pytest

import workloads as wl
from tests.parity import check_bf16, dev_u16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_decoder_gb300 import build
    build.build()
    import memory_bound_decoder_gb300 as mbd
    mbd.get_lib()


def _mbd():
    import memory_bound_decoder_gb300 as mbd
    return mbd


def make_program(T, L, seed, H=1536, I=8960, eps=1e-6):
    """Decode-step layers (norm, norm, SwiGLU) sharing one residual: a chain plus independent ops."""
    mbd = _mbd()
    res0 = wl.make_norm_inputs(T, H, seed, wl.N01, eps, salt=999).residual
    R = dev_u16(torch, res0)
    ops, keep, outs = [], [R], []
    for l in range(L):
        n1 = wl.make_norm_inputs(T, H, seed, wl.N01, eps, salt=3 * l)
        n2 = wl.make_norm_inputs(T, H, seed, wl.N01, eps, salt=3 * l + 1)
        gu = wl.make_swiglu_inputs(T, I, seed, wl.N01, salt=3 * l + 2)
        X1, W1, X2, W2, GU = (dev_u16(torch, a) for a in (n1.x, n1.weight, n2.x, n2.weight, gu.gate_up))
        O1, O2, Y = (torch.empty(T * n, dtype=torch.int16, device="cuda") for n in (H, H, I))
        ops += [mbd.op_add_rmsnorm(O1, R.view, X1.view, W1.view, T, H, eps),
                mbd.op_add_rmsnorm(O2, R.view, X2.view, W2.view, T, H, eps), mbd.op_swiglu(Y, GU.view, T, I)]
        keep += [X1, W1, X2, W2, GU]
        outs += [O1, O2, Y]
    return mbd.program_plan_build(ops), (R, outs, keep)


def snapshot(state):
    R, outs, _ = state
    return [R.numpy(np.uint16)] + [t.cpu().numpy() for t in outs]


def test_two_consecutive_calls_match_the_caller_buffer_entry_point():
    mbd = _mbd()
    plan, state = make_program(T=4, L=4, seed=21)
    sched = torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device="cuda")
    plan.upload(sched)
    plan.launch_uploaded(sched)
    plan.launch_uploaded(sched)
    torch.cuda.synchronize()
    want = snapshot(state)

    plan, state = make_program(T=4, L=4, seed=21)          # identical fresh inputs
    n0 = mbd.kernel_launches()
    plan.launch_static()
    plan.launch_static()
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == 2
    for a, b in zip(want, snapshot(state)):
        np.testing.assert_array_equal(a, b)


def test_plans_alternate_through_the_static_buffer():
    """Each call copies its own schedule: A, B, A through the static buffer equals A, B, A from caller buffers."""
    mbd = _mbd()
    results = []
    for mode in ("caller", "static"):
        pa, sa = make_program(T=2, L=3, seed=31)
        pb, sb = make_program(T=7, L=2, seed=32, H=2048, I=5632)
        if mode == "caller":
            ba = torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device="cuda")
            bb = torch.empty_like(ba)
            pa.upload(ba)
            pb.upload(bb)
            pa.launch_uploaded(ba)
            pb.launch_uploaded(bb)
            pa.launch_uploaded(ba)
        else:
            pa.launch_static()
            pb.launch_static()
            pa.launch_static()
        torch.cuda.synchronize()
        results.append(snapshot(sa) + snapshot(sb))
    for a, b in zip(*results):
        np.testing.assert_array_equal(a, b)


def test_static_launches_take_no_device_memory():
    plan, state = make_program(T=3, L=2, seed=41)
    plan.launch_static()                        # first use (module and driver state settle)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    plan.launch_static()
    plan.launch_static()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == alloc0


def test_two_static_launches_match_the_oracle(orc):
    """A 28-layer decode step (norm, norm, SwiGLU per layer, one residual) launched twice in a row through the
    static buffer: each launch's outputs against the oracle run op by op, and the residual bit-exact."""
    T, L, H, I, eps, seed = 3, 28, 1536, 8960, 1e-6, 51
    plan, state = make_program(T=T, L=L, seed=seed, H=H, I=I, eps=eps)
    R, outs, _ = state
    r = wl.make_norm_inputs(T, H, seed, wl.N01, eps, salt=999).residual
    for call in range(2):
        plan.launch_static()
        torch.cuda.synchronize()
        for l in range(L):
            n1 = wl.make_norm_inputs(T, H, seed, wl.N01, eps, salt=3 * l)
            n2 = wl.make_norm_inputs(T, H, seed, wl.N01, eps, salt=3 * l + 1)
            gu = wl.make_swiglu_inputs(T, I, seed, wl.N01, salt=3 * l + 2)
            O1, O2, Y = (t.cpu().numpy().view(np.uint16) for t in outs[3 * l:3 * l + 3])
            r, _, v1 = orc.add_rmsnorm(n1.x, r, n1.weight, eps)
            check_bf16(O1.reshape(T, H), v1, f"call {call} layer {l} norm 1")
            r, _, v2 = orc.add_rmsnorm(n2.x, r, n2.weight, eps)
            check_bf16(O2.reshape(T, H), v2, f"call {call} layer {l} norm 2")
            _, h = orc.swiglu(gu.gate_up)
            check_bf16(Y.reshape(T, I), h, f"call {call} layer {l} swiglu")
        np.testing.assert_array_equal(R.numpy(np.uint16).reshape(T, H), r,
                                      f"call {call}: the residual must be bit-exact")
