"""The bench's grouped step computes what its per-call step computes: the small ragged calls of the default
step, launched one by one and as one program launch (bf16 and FP8 ops together), from identical seeded inputs;
and its 1000-token calls, one by one and as one batch of overlapping launches (bit for bit).
Residuals and dynamic scales bit-identical; a norm row reduced inside one CTA (program) may sum in another
order than one split over a cluster (single call), so bf16 outputs may differ by one ulp and static-FP8
codes by one step, rarely."""
import numpy as np
import pytest

import bench
import workloads as wl

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


def _run(work, grouped):
    import memory_bound_decoder_gb300 as mbd
    dev = torch.device("cuda", 0)
    dcalls = bench.build_device_calls(torch, mbd, work, 0, 0, dev)
    units = bench.group_small_calls(torch, mbd, work, dcalls, 152, dev) if grouped else list(dcalls)
    handle = int(torch.cuda.current_stream().cuda_stream)
    for u in units:
        u.bind(handle)
    mbd.device_error_flags(clear=True)
    n0 = mbd.kernel_launches()
    for u in units:
        u.launch()
    torch.cuda.synchronize()
    launches = sum(len(u.members) if isinstance(u, bench.BatchGroup) else
                   (1 + len(u.batch.members) if isinstance(u, bench.ProgramBatchGroup) else 1) for u in units)
    assert mbd.kernel_launches() - n0 == launches
    assert mbd.device_error_flags() == 0
    outs = [(d.call, {k: getattr(d, k).cpu().numpy().copy() for k in ("out", "res", "scale") if hasattr(d, k)})
            for d in dcalls]
    return len(units), outs


def test_grouped_small_calls_match_per_call_launches():
    w = bench.workloads_by_key()[bench.DEFAULT_WORKLOAD]
    work = wl.Workload("small", "the small calls of the default step", tuple(c for c in w.calls if c.T < 152), 1)
    n_calls, ref = _run(work, grouped=False)
    n_units, got = _run(work, grouped=True)
    assert n_calls == 12 and n_units == 1
    for (call, a), (_, b) in zip(ref, got):
        if "res" in a:
            np.testing.assert_array_equal(a["res"], b["res"], f"{call.name}: residual")
        if call.mode == "dynamic":
            np.testing.assert_array_equal(a["scale"], b["scale"], f"{call.name}: dynamic scales")
        if call.kind in ("add_rmsnorm", "swiglu"):
            d = np.abs(a["out"].astype(np.int32) - b["out"].astype(np.int32))
            assert d.max() <= 1, f"{call.name}: bf16 outputs differ by more than one ulp"
        else:
            x, y = a["out"].astype(np.int32), b["out"].astype(np.int32)
            diff = x != y
            assert diff.mean() <= 1e-3, f"{call.name}: {diff.sum()} codes differ"
            assert ((x[diff] & 0x80) == (y[diff] & 0x80)).all(), f"{call.name}: sign flipped"
            assert (np.abs((x[diff] & 0x7F) - (y[diff] & 0x7F)) == 1).all(), f"{call.name}: more than one step"


def _compare(ref, got):
    """Large calls (the same single-call kernels) bit for bit; program rows within the program's rounding."""
    for (call, a), (_, b) in zip(ref, got):
        if call.T >= 152 or "res" in a:
            if call.T >= 152:
                for k in a:
                    np.testing.assert_array_equal(a[k], b[k], f"{call.name}: {k}")
                continue
            np.testing.assert_array_equal(a["res"], b["res"], f"{call.name}: residual")
        if call.mode == "dynamic":
            np.testing.assert_array_equal(a["scale"], b["scale"], f"{call.name}: dynamic scales")
        if call.kind in ("add_rmsnorm", "swiglu"):
            d = np.abs(a["out"].astype(np.int32) - b["out"].astype(np.int32))
            assert d.max() <= 1, f"{call.name}: bf16 outputs differ by more than one ulp"
        else:
            x, y = a["out"].astype(np.int32), b["out"].astype(np.int32)
            diff = x != y
            assert diff.sum() <= diff.size // 1000, f"{call.name}: {diff.sum()} codes differ"
            assert (np.abs((x[diff] & 0x7F) - (y[diff] & 0x7F)) == 1).all(), f"{call.name}: more than one step"


def test_default_step_units_match_per_call_launches():
    """The whole default step: the largest call alone, the program of the small calls opening the batch of the
    others (one mbd_run_independent_with_program call), against every call launched on its own."""
    w = bench.workloads_by_key()[bench.DEFAULT_WORKLOAD]
    n_calls, ref = _run(w, grouped=False)
    n_units, got = _run(w, grouped=True)
    assert n_calls == 18 and n_units == 2
    _compare(ref, got)


def test_batched_1000_token_calls_match_per_call_launches():
    w = bench.workloads_by_key()[bench.DEFAULT_WORKLOAD]
    work = wl.Workload("t1000", "the 1000-token calls of the default step", tuple(c for c in w.calls if c.T == 1000), 1)
    n_calls, ref = _run(work, grouped=False)
    n_units, got = _run(work, grouped=True)
    assert n_calls == 4 and n_units == 2                # the largest call alone, the other three as one batch
    for (call, a), (_, b) in zip(ref, got):
        for k in a:
            np.testing.assert_array_equal(a[k], b[k], f"{call.name}: {k}")
