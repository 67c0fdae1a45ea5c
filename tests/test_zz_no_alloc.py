"""mbd_program_plan_launch_static, the program launch that allocates nothing, for callers that cannot allocate
device memory (engines that keep nearly all HBM in their own pool, plug-in interfaces that hand a kernel only
its inputs and outputs, loops that cannot afford cudaMalloc's possible device synchronisation): its schedule
goes to a static buffer of the library instead of caller memory. Checked against the entry point it stands in for
(mbd_program_plan_upload into a caller buffer + mbd_program_plan_launch_uploaded): two consecutive calls of
each, on identical fresh inputs, give identical bits; plans may alternate through the shared buffer; and
the calls take no device memory. Collected last (file name), after every other GPU test.
"""
import numpy as np
import pytest

import workloads as wl
from tests.parity import dev_u16

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
