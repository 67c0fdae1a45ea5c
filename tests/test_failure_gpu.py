"""Failure detection on the GPU without a fault: every spin-wait in the kernels is bounded. A self-test
kernel waits on an mbarrier that nothing completes; the wait must run out after its short limit, set the
device error bit readable from the host, and leave the context usable for the next launches."""
import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests.parity import check_codes

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mbd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_decoder_gb300 import build
    build.build()
    orc.build()
    import memory_bound_decoder_gb300 as m
    m.get_lib()
    return m


def test_bounded_wait_times_out_and_reports(mbd):
    torch.cuda.synchronize()
    mbd.device_error_flags(clear=True)
    assert mbd.device_error_flags() == 0
    mbd.selftest_bounded_wait(2_000_000)            # ~1 ms of SM clock
    torch.cuda.synchronize()
    assert mbd.device_error_flags() & mbd.DEVERR_EXCHANGE_TIMEOUT
    assert mbd.device_error_flags(clear=True) & mbd.DEVERR_EXCHANGE_TIMEOUT
    assert mbd.device_error_flags() == 0

    # the context is still usable: a clustered dynamic-scale SwiGLU runs and matches the oracle
    inp = wl.make_swiglu_inputs(3, 13824, seed=1, dist=wl.C5_ACT)
    gu = torch.from_numpy(inp.gate_up.view(np.int16)).cuda()
    q = torch.empty((3, 13824), dtype=torch.uint8, device="cuda")
    sc = torch.empty((3,), dtype=torch.float32, device="cuda")
    mbd.swiglu_quant_fp8(q, gu, 3, 13824, "dynamic", sc)
    torch.cuda.synchronize()
    q_o, s_o, _ = orc.swiglu_quant_fp8(inp.gate_up, "dynamic")
    check_codes(q.cpu().numpy(), q_o, "after timeout")
    assert mbd.device_error_flags() == 0
