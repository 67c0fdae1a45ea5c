"""mbd_run_independent: a batch of independent ops, each run by its own single-call kernel, the launches after
the first overlapping the one before. Checked bit for bit against the same ops called one after another
through their entry points (every epilogue, the launch forms a batch can take: one CTA per row, clusters,
streams, the bulk-copy dynamic SwiGLU, decode-sized rows), against the oracle for the 1000-token ragged
calls, and for stream order around the batch: a batch that reads what the kernel before it wrote, and a
kernel after it that reads what the batch wrote.
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


STATIC, NVFP4_S = 0.05, 0.03


class OpCase:
    """Inputs of one op on the device (fresh copies per run) and its outputs between guard bands."""

    def __init__(self, kind, T, W, seed, mode=None, dist=wl.N01, eps=1e-5):
        self.kind, self.mode, self.T, self.W, self.eps = kind, mode, T, W, eps
        self.norm = kind.startswith("add_rmsnorm")
        if self.norm:
            self.inp = wl.make_norm_inputs(T, W, seed, dist, eps)
        else:
            self.inp = wl.make_swiglu_inputs(T, W, seed, dist)

    def alloc(self):
        T, W, inp = self.T, self.W, self.inp
        d = {}
        if self.norm:
            d["x"], d["residual"], d["weight"] = (dev_u16(torch, a) for a in (inp.x, inp.residual, inp.weight))
        else:
            d["gate_up"] = dev_u16(torch, inp.gate_up)
        if self.kind.endswith("nvfp4"):
            d["out"] = Guarded(torch, T * W // 2, torch.uint8)
            d["sf"] = Guarded(torch, T * W // 16, torch.uint8)
            d["scale"] = Guarded(torch, 1, torch.float32, fill=np.array([NVFP4_S], np.float32))
        elif self.kind.endswith("fp8"):
            d["out"] = Guarded(torch, T * W, torch.uint8)
            d["scale"] = (Guarded(torch, 1, torch.float32, fill=np.array([STATIC], np.float32))
                          if self.mode == "static" else Guarded(torch, T, torch.float32))
        else:
            d["out"] = Guarded(torch, T * W, torch.int16)
        self.d = d
        return self

    def op(self):
        mbd, d, T, W = _mbd(), self.d, self.T, self.W
        v = lambda k: d[k].view
        if self.kind == "add_rmsnorm":
            return mbd.op_add_rmsnorm(v("out"), v("residual"), v("x"), v("weight"), T, W, self.eps)
        if self.kind == "add_rmsnorm_quant_fp8":
            return mbd.op_add_rmsnorm_quant_fp8(v("out"), v("residual"), v("x"), v("weight"), T, W, self.eps,
                                                self.mode, v("scale"))
        if self.kind == "add_rmsnorm_quant_nvfp4":
            return mbd.op_add_rmsnorm_quant_nvfp4(v("out"), v("sf"), v("residual"), v("x"), v("weight"), T, W,
                                                  self.eps, v("scale"))
        if self.kind == "swiglu":
            return mbd.op_swiglu(v("out"), v("gate_up"), T, W)
        if self.kind == "swiglu_quant_fp8":
            return mbd.op_swiglu_quant_fp8(v("out"), v("gate_up"), T, W, self.mode, v("scale"))
        return mbd.op_swiglu_quant_nvfp4(v("out"), v("sf"), v("gate_up"), T, W, v("scale"))

    def call(self):
        """The op through its own entry point."""
        mbd, d, T, W = _mbd(), self.d, self.T, self.W
        v = lambda k: d[k].view
        if self.kind == "add_rmsnorm":
            mbd.fused_add_rmsnorm(v("out"), v("residual"), v("x"), v("weight"), T, W, self.eps)
        elif self.kind == "add_rmsnorm_quant_fp8":
            mbd.fused_add_rmsnorm_quant_fp8(v("out"), v("residual"), v("x"), v("weight"), T, W, self.eps,
                                            self.mode, v("scale"))
        elif self.kind == "add_rmsnorm_quant_nvfp4":
            mbd.fused_add_rmsnorm_quant_nvfp4(v("out"), v("sf"), v("residual"), v("x"), v("weight"), T, W,
                                              self.eps, v("scale"))
        elif self.kind == "swiglu":
            mbd.swiglu(v("out"), v("gate_up"), T, W)
        elif self.kind == "swiglu_quant_fp8":
            mbd.swiglu_quant_fp8(v("out"), v("gate_up"), T, W, self.mode, v("scale"))
        else:
            mbd.swiglu_quant_nvfp4(v("out"), v("sf"), v("gate_up"), T, W, v("scale"))

    def snapshot(self):
        for name, g in self.d.items():
            g.check_guards(f"{self.kind} {name}")
        return {k: g.raw.cpu().numpy().copy() for k, g in self.d.items()}


def run_both(cases):
    """Outputs of the ops called one by one, and of the same ops (fresh inputs) as one batch."""
    mbd = _mbd()
    for c in cases:
        c.alloc()
    for c in cases:
        c.call()
    torch.cuda.synchronize()
    want = [c.snapshot() for c in cases]
    for c in cases:
        c.alloc()
    mbd.device_error_flags(clear=True)
    n0 = mbd.kernel_launches()
    mbd.run_independent([c.op() for c in cases])
    torch.cuda.synchronize()
    assert mbd.kernel_launches() - n0 == sum(1 for c in cases if c.T > 0)
    assert mbd.device_error_flags() == 0
    return want, [c.snapshot() for c in cases]


def assert_same(want, got):
    for i, (a, b) in enumerate(zip(want, got)):
        for k in a:
            np.testing.assert_array_equal(a[k], b[k], f"op {i} {k}")


def ragged_1000():
    """The four entry points at 1000 tokens, hidden 5120, inter 13824 (0.1% of values x100)."""
    return [OpCase("add_rmsnorm", 1000, 5120, 1, dist=wl.C5_ACT),
            OpCase("add_rmsnorm_quant_fp8", 1000, 5120, 2, "static", dist=wl.C5_ACT),
            OpCase("swiglu", 1000, 13824, 3, dist=wl.C5_ACT),
            OpCase("swiglu_quant_fp8", 1000, 13824, 4, "dynamic", dist=wl.C5_ACT)]


def test_ragged_1000_matches_single_calls():
    assert_same(*run_both(ragged_1000()))


BATCHES = {
    # every epilogue of both fusions, one CTA per row and streams
    "all_epilogues": [OpCase("add_rmsnorm", 700, 4096, 11), OpCase("add_rmsnorm_quant_fp8", 600, 4096, 12, "static"),
                      OpCase("add_rmsnorm_quant_fp8", 500, 2048, 13, "dynamic"),
                      OpCase("add_rmsnorm_quant_nvfp4", 400, 8192, 14, dist=wl.C5_ACT),
                      OpCase("swiglu", 300, 14336, 15), OpCase("swiglu_quant_fp8", 800, 8960, 16, "static"),
                      OpCase("swiglu_quant_fp8", 900, 13824, 17, "dynamic"),
                      OpCase("swiglu_quant_nvfp4", 256, 28672, 18, dist=wl.C5_ACT)],
    # decode-sized rows (cluster-split reductions, L2 warming before the wait) beside large batches
    "small_and_large": [OpCase("add_rmsnorm", 3, 5120, 21), OpCase("swiglu_quant_fp8", 2048, 28672, 22, "dynamic"),
                        OpCase("swiglu_quant_fp8", 17, 13824, 23, "dynamic"), OpCase("add_rmsnorm_quant_fp8", 1, 16384, 24, "dynamic"),
                        OpCase("swiglu", 5, 8960, 25), OpCase("add_rmsnorm_quant_fp8", 2048, 8192, 26, "static")],
    # the bulk-copy dynamic SwiGLU (>= 4 rows per SM, rows of 4609+ vectors) between two norms, and a zero-token op
    "bulk_form": [OpCase("add_rmsnorm", 1000, 5120, 31), OpCase("swiglu_quant_fp8", 640, 53248, 32, "dynamic", dist=wl.C5_ACT),
                  OpCase("swiglu", 0, 8960, 33), OpCase("add_rmsnorm_quant_fp8", 1000, 16384, 34, "static")],
}


@pytest.mark.parametrize("name", list(BATCHES))
def test_batch_matches_single_calls(name):
    assert_same(*run_both(BATCHES[name]))


def test_ragged_1000_against_the_oracle():
    cases = [c.alloc() for c in ragged_1000()]
    _mbd().run_independent([c.op() for c in cases])
    torch.cuda.synchronize()
    n1, q1, s1, q2 = cases
    T = 1000
    for c in cases:
        c.snapshot()                                                     # guard bands untouched
    res_o, _, v = orc.add_rmsnorm(n1.inp.x, n1.inp.residual, n1.inp.weight, n1.eps)
    np.testing.assert_array_equal(n1.d["residual"].numpy(np.uint16).reshape(T, -1), res_o)
    check_bf16(n1.d["out"].numpy(np.uint16).reshape(T, -1), v, "add_rmsnorm")
    res_o, q_o, _, _ = orc.add_rmsnorm_quant_fp8(q1.inp.x, q1.inp.residual, q1.inp.weight, q1.eps, "static", STATIC)
    np.testing.assert_array_equal(q1.d["residual"].numpy(np.uint16).reshape(T, -1), res_o)
    check_codes(q1.d["out"].numpy(np.uint8).reshape(T, -1), q_o, "add_rmsnorm_q8 static")
    _, h = orc.swiglu(s1.inp.gate_up)
    check_bf16(s1.d["out"].numpy(np.uint16).reshape(T, -1), h, "swiglu")
    q_o, s_o, _ = orc.swiglu_quant_fp8(q2.inp.gate_up, "dynamic")
    check_codes(q2.d["out"].numpy(np.uint8).reshape(T, -1), q_o, "swiglu_q8 dynamic")
    check_scales(q2.d["scale"].numpy(np.float32), s_o, "swiglu_q8 scales")


@pytest.mark.parametrize("reader_first", [False, True])
def test_stream_order_around_the_batch(reader_first):
    """A large SwiGLU writes t; in the batch, a norm reads t (as x) beside an unrelated ~80 us op, launched first
    or second; a norm after the batch reads that norm's output. Run 5 times; every result must equal the
    one-call-at-a-time sequence."""
    mbd = _mbd()
    T, W, eps = 2048, 14336, 1e-5
    gu = wl.make_swiglu_inputs(T, W, 41, wl.N01).gate_up                 # [T, 2W]: t = swiglu(gu) is [T, W]
    other = OpCase("swiglu_quant_fp8", 2048, 53248, 42, "dynamic")
    r1 = wl.make_norm_inputs(T, W, 43, wl.N01, eps)
    r2 = wl.make_norm_inputs(T, W, 44, wl.N01, eps)

    def sequence(batched):
        G = dev_u16(torch, gu)
        t = Guarded(torch, T * W, torch.int16)
        R1, W1, R2, W2 = (dev_u16(torch, a) for a in (r1.residual, r1.weight, r2.residual, r2.weight))
        o1, o2 = Guarded(torch, T * W, torch.int16), Guarded(torch, T * W, torch.int16)
        other.alloc()
        mbd.swiglu(t.view, G.view, T, W)                                          # writes t
        if batched:
            n1 = mbd.op_add_rmsnorm(o1.view, R1.view, t.view, W1.view, T, W, eps)  # reads t
            mbd.run_independent([n1, other.op()] if reader_first else [other.op(), n1])
        else:
            other.call()
            mbd.fused_add_rmsnorm(o1.view, R1.view, t.view, W1.view, T, W, eps)
        mbd.fused_add_rmsnorm(o2.view, R2.view, o1.view, W2.view, T, W, eps)      # reads o1
        torch.cuda.synchronize()
        return [g.raw.cpu().numpy().copy() for g in (t, R1, o1, R2, o2)] + list(other.snapshot().values())

    want = sequence(False)
    for _ in range(5):
        got = sequence(True)
        for a, b in zip(want, got):
            np.testing.assert_array_equal(a, b)


def _program_cases():
    """Small calls for the program (1, 3 and 17 tokens; bf16, static-FP8 and dynamic-FP8 ops) and large ones for
    the batch after it."""
    small = [OpCase("add_rmsnorm", 1, 5120, 51), OpCase("add_rmsnorm_quant_fp8", 3, 5120, 52, "static"),
             OpCase("swiglu", 17, 13824, 53), OpCase("swiglu_quant_fp8", 17, 13824, 54, "dynamic"),
             OpCase("swiglu_quant_fp8", 1, 13824, 55, "dynamic"), OpCase("add_rmsnorm", 17, 5120, 56)]
    large = [OpCase("add_rmsnorm_quant_fp8", 2048, 16384, 57, "static"), OpCase("swiglu", 1000, 13824, 58),
             OpCase("swiglu_quant_fp8", 1000, 13824, 59, "dynamic")]
    return small, large


def test_batch_with_program_matches_the_sequence():
    """The program in front of the batch, against the program launched alone and then the ops' single calls."""
    mbd = _mbd()
    small, large = _program_cases()
    results = []
    for mode in ("sequence", "batch"):
        for c in small + large:
            c.alloc()
        plan = mbd.program_plan_build([c.op() for c in small])
        sched = torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device="cuda")
        plan.upload(sched)
        mbd.device_error_flags(clear=True)
        n0 = mbd.kernel_launches()
        if mode == "sequence":
            plan.launch_uploaded(sched)
            for c in large:
                c.call()
        else:
            mbd.run_independent_with_program(plan, sched, [c.op() for c in large])
        torch.cuda.synchronize()
        assert mbd.kernel_launches() - n0 == 1 + len(large)
        assert mbd.device_error_flags() == 0
        results.append([c.snapshot() for c in small + large])
    assert_same(*results)


def test_batch_with_program_rejects_shared_memory():
    """An op that writes what the program reads (or reads what it writes) is refused before any launch."""
    mbd = _mbd()
    small, large = _program_cases()
    for c in small + large:
        c.alloc()
    plan = mbd.program_plan_build([c.op() for c in small])
    sched = torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device="cuda")
    plan.upload(sched)
    T, H = small[0].T, small[0].W
    clash = OpCase("add_rmsnorm", T, H, 60).alloc()
    clash.d["residual"] = small[0].d["residual"]        # the program's norm updates this residual
    n0 = mbd.kernel_launches()
    with pytest.raises(mbd.MbdError) as e:
        mbd.run_independent_with_program(plan, sched, [large[0].op(), clash.op()])
    assert e.value.status == mbd.ERR_INVALID_ARG
    assert mbd.kernel_launches() == n0


@pytest.mark.parametrize("reader_in_program", [False, True])
def test_stream_order_around_a_batch_with_program(reader_in_program):
    """A SwiGLU writes t; t feeds a norm in the program or in the batch beside a long op; a norm after the batch
    reads that norm's output. Five runs, each equal to the one-launch-at-a-time sequence."""
    mbd = _mbd()
    W, eps = 8192, 1e-5
    Tn = 17 if reader_in_program else 1000
    gu = wl.make_swiglu_inputs(Tn, W, 61, wl.N01).gate_up
    long_op = OpCase("swiglu_quant_fp8", 2048, 53248, 62, "dynamic")
    other_small = OpCase("swiglu", 3, 13824, 63)
    r1 = wl.make_norm_inputs(Tn, W, 64, wl.N01, eps)
    r2 = wl.make_norm_inputs(Tn, W, 65, wl.N01, eps)

    def sequence(batched):
        G = dev_u16(torch, gu)
        t = Guarded(torch, Tn * W, torch.int16)
        R1, W1, R2, W2 = (dev_u16(torch, a) for a in (r1.residual, r1.weight, r2.residual, r2.weight))
        o1, o2 = Guarded(torch, Tn * W, torch.int16), Guarded(torch, Tn * W, torch.int16)
        long_op.alloc()
        other_small.alloc()
        n1 = mbd.op_add_rmsnorm(o1.view, R1.view, t.view, W1.view, Tn, W, eps)   # reads t
        prog_ops = [other_small.op()] + ([n1] if reader_in_program else [])
        batch_ops = [long_op.op()] + ([] if reader_in_program else [n1])
        plan = mbd.program_plan_build(prog_ops)
        sched = torch.empty(mbd.program_schedule_bytes(), dtype=torch.uint8, device="cuda")
        plan.upload(sched)
        mbd.swiglu(t.view, G.view, Tn, W)                                             # writes t
        if batched:
            mbd.run_independent_with_program(plan, sched, batch_ops)
        else:
            plan.launch_uploaded(sched)
            mbd.run_independent(batch_ops[:1])
            for op in batch_ops[1:]:
                mbd.run_independent([op])
        mbd.fused_add_rmsnorm(o2.view, R2.view, o1.view, W2.view, Tn, W, eps)         # reads o1
        torch.cuda.synchronize()
        return ([g.raw.cpu().numpy().copy() for g in (t, R1, o1, R2, o2)] + list(long_op.snapshot().values())
                + list(other_small.snapshot().values()))

    want = sequence(False)
    for _ in range(5):
        got = sequence(True)
        for a, b in zip(want, got):
            np.testing.assert_array_equal(a, b)
