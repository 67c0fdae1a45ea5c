"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function the header
declares, and rejects invalid arguments before touching the device (the checks under test all fail
before any CUDA call, so fake pointer values are safe here)."""
import ctypes
import re

import pytest

import memory_bound_decoder_gb300 as mbd
from memory_bound_decoder_gb300 import build as mbd_build


@pytest.fixture(scope="module")
def lib():
    mbd_build.build()
    return mbd.get_lib()


def test_exports_every_declared_symbol(lib):
    names = mbd.header_functions()
    assert set(names) >= {"mbd_fused_add_rmsnorm", "mbd_fused_add_rmsnorm_quant_fp8", "mbd_swiglu",
                          "mbd_swiglu_quant_fp8", "mbd_status_string", "mbd_abi_version",
                          "mbd_last_cuda_error", "mbd_kernel_launches", "mbd_device_error_flags"}
    for n in names:
        assert hasattr(lib, n), n


def test_binding_names_match_header():
    for n in mbd.header_functions():
        short = n[len("mbd_"):]
        if short in ("status_string", "last_cuda_error"):
            continue
        assert hasattr(mbd, short), short


def test_version_and_status_strings(lib):
    assert lib.mbd_abi_version() == 9
    hdr = open(mbd.HEADER_PATH).read()
    assert int(re.search(r"#define MBD_ABI_VERSION (\d+)", hdr).group(1)) == 9
    for code in range(5):
        assert lib.mbd_status_string(code).decode().startswith("MBD_")
    assert lib.mbd_status_string(99) == b"unknown mbd_status"
    assert lib.mbd_last_cuda_error() == 0


A = 1 << 20   # a fake, 16-byte aligned "device pointer" (never dereferenced: validation fails first)


def _rc(fn, *args):
    with pytest.raises(mbd.MbdError) as e:
        fn(*args)
    return e.value.status


def test_zero_tokens_is_a_noop(lib):
    n0 = mbd.kernel_launches()
    mbd.fused_add_rmsnorm(None, None, None, None, 0, 4096, 1e-6)
    mbd.fused_add_rmsnorm_quant_fp8(None, None, None, None, 0, 4096, 1e-6, "dynamic", None)
    mbd.swiglu(None, None, 0, 14336)
    mbd.swiglu_quant_fp8(None, None, 0, 14336, "static", None)
    assert mbd.kernel_launches() == n0


def test_invalid_arguments(lib):
    f = mbd.fused_add_rmsnorm
    assert _rc(f, A, 2 * A, 3 * A, 4 * A, -1, 64, 1e-6) == mbd.ERR_INVALID_ARG
    assert _rc(f, A, 2 * A, 3 * A, 4 * A, 4, 0, 1e-6) == mbd.ERR_INVALID_ARG
    assert _rc(f, A, 2 * A, 3 * A, 4 * A, 4, 64, -1.0) == mbd.ERR_INVALID_ARG
    assert _rc(f, A, 2 * A, 3 * A, 4 * A, 4, 64, float("nan")) == mbd.ERR_INVALID_ARG
    assert _rc(f, None, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG
    assert _rc(f, A, 2 * A, 3 * A, None, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG
    # overlapping residual and x
    assert _rc(f, A, 2 * A, 2 * A + 64, 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG
    # out overlapping x without being equal to it
    assert _rc(f, 3 * A + 16, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG
    q = mbd.fused_add_rmsnorm_quant_fp8
    assert _rc(q, A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 7, 5 * A) == mbd.ERR_INVALID_ARG
    assert _rc(q, A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, "static", None) == mbd.ERR_INVALID_ARG
    assert _rc(q, 3 * A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, "static", 5 * A) == mbd.ERR_INVALID_ARG  # out_q == x
    s = mbd.swiglu
    assert _rc(s, A, A + 64, 4, 64) == mbd.ERR_INVALID_ARG        # out overlaps gate_up
    sq = mbd.swiglu_quant_fp8
    assert _rc(sq, A, 2 * A, 4, 64, "dynamic", A + 8) == mbd.ERR_INVALID_ARG   # scale inside out_q


def test_misaligned(lib):
    f = mbd.fused_add_rmsnorm
    assert _rc(f, A + 2, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6) == mbd.ERR_MISALIGNED
    assert _rc(f, A, 2 * A, 3 * A + 8, 4 * A, 4, 64, 1e-6) == mbd.ERR_MISALIGNED
    assert _rc(f, A, 2 * A, 3 * A, 4 * A, 4, 60, 1e-6) == mbd.ERR_MISALIGNED        # width % 8
    assert _rc(mbd.swiglu, A, 2 * A, 4, 100) == mbd.ERR_MISALIGNED
    assert _rc(mbd.swiglu_quant_fp8, A, 2 * A, 4, 64, "dynamic", 5 * A + 2) == mbd.ERR_MISALIGNED


def test_unsupported_widths(lib):
    wide = 262144 + 8
    assert _rc(mbd.fused_add_rmsnorm, A, 2 * A, 3 * A, 4 * A, 0, wide, 1e-6) == mbd.ERR_UNSUPPORTED
    assert _rc(mbd.swiglu_quant_fp8, A, 2 * A, 0, wide, "dynamic", 5 * A) == mbd.ERR_UNSUPPORTED
    # the pure streams have no such limit: zero tokens with a wide row is a no-op
    mbd.swiglu(None, None, 0, wide)
    mbd.swiglu_quant_fp8(None, None, 0, wide, "static", None)


def test_allreduce_argument_checks(lib):
    f = mbd.fused_allreduce_add_rmsnorm
    assert _rc(f, A, 2 * A, [], 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG                  # no partial
    assert _rc(f, A, 2 * A, [3 * A] * 9, 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG          # too many
    assert _rc(f, A, 2 * A, [3 * A, None], 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG        # null partial
    assert _rc(f, A, 2 * A, [3 * A, 5 * A + 8], 4 * A, 4, 64, 1e-6) == mbd.ERR_MISALIGNED    # misaligned
    assert _rc(f, A, 2 * A, [3 * A, 2 * A + 64], 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG  # overlaps residual
    assert _rc(f, A, 2 * A, [3 * A, A], 4 * A, 4, 64, 1e-6) == mbd.ERR_INVALID_ARG           # partial 1 is out
    q = mbd.fused_allreduce_add_rmsnorm_quant_fp8
    assert _rc(q, A, 2 * A, [3 * A], 4 * A, 4, 64, 1e-6, "dynamic", 3 * A + 4) == mbd.ERR_INVALID_ARG
    # the partial sums hold their accumulators in registers: at most 8 x 512 vectors per row
    assert _rc(f, A, 2 * A, [3 * A], 4 * A, 1, 32768 + 8, 1e-6) == mbd.ERR_UNSUPPORTED
    n0 = mbd.kernel_launches()
    f(None, None, [None, None], None, 0, 64, 1e-6)     # zero tokens: a no-op
    assert mbd.kernel_launches() == n0


def test_device_error_flags_rejects_null(lib):
    assert lib.mbd_device_error_flags(None, 0) == mbd.ERR_INVALID_ARG


def test_selftest_limit_validated(lib):
    assert _rc(mbd.selftest_bounded_wait, 0) == mbd.ERR_INVALID_ARG
    assert _rc(mbd.selftest_bounded_wait, (1 << 31) + 1) == mbd.ERR_INVALID_ARG


def test_raw_ctypes_signature(lib):
    # the C entry points are callable without the Python binding
    fn = lib.mbd_swiglu
    assert fn(None, None, ctypes.c_int64(0), ctypes.c_int64(64), None) == 0


def test_nvfp4_argument_checks(lib):
    n0 = mbd.kernel_launches()
    mbd.fused_add_rmsnorm_quant_nvfp4(None, None, None, None, None, 0, 4096, 1e-6, None)
    mbd.swiglu_quant_nvfp4(None, None, None, 0, 14336, None)
    assert mbd.kernel_launches() == n0
    f = mbd.fused_add_rmsnorm_quant_nvfp4
    # width a multiple of 8 but not of 16: a 16-element block would straddle rows
    assert _rc(f, A, 6 * A, 2 * A, 3 * A, 4 * A, 4, 72, 1e-6, 5 * A) == mbd.ERR_MISALIGNED
    assert _rc(f, A, None, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 5 * A) == mbd.ERR_INVALID_ARG     # no block scales
    assert _rc(f, A, 6 * A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, None) == mbd.ERR_INVALID_ARG     # no tensor scale
    assert _rc(f, A + 4, 6 * A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 5 * A) == mbd.ERR_MISALIGNED
    assert _rc(f, A, 6 * A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 5 * A + 2) == mbd.ERR_MISALIGNED
    # codes take T * H / 2 = 128 bytes: block scales starting inside them overlap
    assert _rc(f, A, A + 120, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 5 * A) == mbd.ERR_INVALID_ARG
    assert _rc(f, A, A + 128, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, A + 124) == mbd.ERR_INVALID_ARG  # scale in codes
    assert _rc(f, A, 6 * A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 6 * A + 12) == mbd.ERR_INVALID_ARG  # scale in sf
    assert _rc(f, A, 6 * A, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 2 * A + 8) == mbd.ERR_INVALID_ARG  # scale in residual
    assert _rc(f, A, 2 * A + 8, 2 * A, 3 * A, 4 * A, 4, 64, 1e-6, 5 * A) == mbd.ERR_INVALID_ARG  # sf in residual
    assert _rc(f, A, 6 * A, 2 * A, 3 * A, 4 * A, 0, 262144 + 16, 1e-6, 5 * A) == mbd.ERR_UNSUPPORTED
    s = mbd.swiglu_quant_nvfp4
    assert _rc(s, A, 6 * A, 2 * A, 4, 72, 5 * A) == mbd.ERR_MISALIGNED
    assert _rc(s, A, 2 * A + 16, 2 * A, 4, 64, 5 * A) == mbd.ERR_INVALID_ARG        # sf inside gate_up
    assert _rc(s, A, A + 64, 2 * A, 4, 64, 5 * A) == mbd.ERR_INVALID_ARG            # sf inside codes
    assert _rc(s, A, 6 * A, 2 * A, 4, 64, None) == mbd.ERR_INVALID_ARG
    # a pure stream: no width limit beyond the 2^28 sanity bound
    s(None, None, None, 0, 262144 + 16, None)


def test_program_argument_checks(lib):
    n0 = mbd.kernel_launches()
    mbd.run_program([])                                                      # empty program: nothing launched
    mbd.run_program([mbd.op_swiglu(None, None, 0, 64)])                      # zero-token ops are skipped
    assert mbd.kernel_launches() == n0
    H = 64
    norm = lambda out, res, x, T=4, H=H: mbd.op_add_rmsnorm(out, res, x, 9 * A, T, H, 1e-6)
    assert _rc(mbd.run_program, [norm(A, 2 * A, 3 * A)] * 129) == mbd.ERR_INVALID_ARG        # too many ops
    bad = norm(A, 2 * A, 3 * A)
    bad.kind = 9
    assert _rc(mbd.run_program, [bad]) == mbd.ERR_INVALID_ARG                                # unknown kind
    bad = norm(A, 2 * A, 3 * A)
    bad.reserved = 1
    assert _rc(mbd.run_program, [bad]) == mbd.ERR_INVALID_ARG
    bad = mbd.op_add_rmsnorm_quant_fp8(A, 2 * A, 3 * A, 9 * A, 4, H, 1e-6, 7, 5 * A)
    assert _rc(mbd.run_program, [bad]) == mbd.ERR_INVALID_ARG                                # unknown FP8 mode
    # each op is validated like its entry point, with the same status
    assert _rc(mbd.run_program, [norm(A + 2, 2 * A, 3 * A)]) == mbd.ERR_MISALIGNED
    assert _rc(mbd.run_program, [norm(A, 2 * A, 2 * A + 64)]) == mbd.ERR_INVALID_ARG         # x inside residual
    # a later op reading a written buffer through another pointer, or with another row layout
    a, b = norm(A, 2 * A, 3 * A), norm(4 * A, 5 * A, A + 16)
    assert _rc(mbd.run_program, [a, b]) == mbd.ERR_UNSUPPORTED
    a, b = norm(A, 2 * A, 3 * A), norm(4 * A, 5 * A, A, T=2, H=2 * H)
    assert _rc(mbd.run_program, [a, b]) == mbd.ERR_UNSUPPORTED
    # a dynamic FP8 scale written by one op and read as another op's static scale
    q1 = mbd.op_add_rmsnorm_quant_fp8(6 * A, 2 * A, 3 * A, 9 * A, 4, H, 1e-6, "dynamic", 7 * A)
    q2 = mbd.op_add_rmsnorm_quant_fp8(8 * A, 5 * A, 4 * A, 9 * A, 4, H, 1e-6, "static", 7 * A)
    assert _rc(mbd.run_program, [q1, q2]) == mbd.ERR_UNSUPPORTED
    # the weight is not a row-wise tensor: writing it in a program is rejected
    w_writer = mbd.op_add_rmsnorm(9 * A, 5 * A, 4 * A, 13 * A, 4, H, 1e-6)   # its output is the first op's weight
    assert _rc(mbd.run_program, [norm(A, 2 * A, 3 * A), w_writer]) == mbd.ERR_UNSUPPORTED
    # a row that must stay in one CTA is limited to MBD_MAX_PROGRAM_WIDTH elements
    assert _rc(mbd.run_program, [norm(A, 2 * A, 3 * A, T=1, H=8192 + 16)]) == mbd.ERR_UNSUPPORTED
    # epilogues outside the compiled sets: a dynamic-FP8 norm with a bf16 SwiGLU (the mixed bf16 + FP8 variant
    # leaves the dynamic norm out), a bf16 norm with an NVFP4 SwiGLU
    qd = mbd.op_add_rmsnorm_quant_fp8(6 * A, 2 * A, 3 * A, 9 * A, 4, H, 1e-6, "dynamic", 7 * A)
    assert _rc(mbd.run_program, [qd, mbd.op_swiglu(10 * A, 11 * A, 4, H)]) == mbd.ERR_UNSUPPORTED
    s4 = mbd.op_swiglu_quant_nvfp4(10 * A, 12 * A, 11 * A, 4, H, 13 * A)
    assert _rc(mbd.run_program, [norm(A, 2 * A, 3 * A), s4]) == mbd.ERR_UNSUPPORTED
    assert mbd.kernel_launches() == n0


def test_program_struct_layout():
    assert ctypes.sizeof(mbd.Op) == 80 and mbd.Op.out.offset == 32 and mbd.Op.scale.offset == 72


def test_program_plan_checks(lib):
    # build runs every check of mbd_run_program before touching the device
    H = 64
    a = mbd.op_add_rmsnorm(A, 2 * A, 3 * A, 9 * A, 4, H, 1e-6)
    b = mbd.op_add_rmsnorm(4 * A, 5 * A, A + 16, 9 * A, 4, H, 1e-6)
    with pytest.raises(mbd.MbdError) as e:
        mbd.program_plan_build([a, b])
    assert e.value.status == mbd.ERR_UNSUPPORTED
    with pytest.raises(mbd.MbdError) as e:
        mbd.program_plan_build([mbd.op_add_rmsnorm(A + 2, 2 * A, 3 * A, 9 * A, 4, H, 1e-6)])
    assert e.value.status == mbd.ERR_MISALIGNED
    # a plan build left unfilled (failed) cannot be launched; an empty plan launches nothing
    buf = (ctypes.c_uint64 * (mbd.PROGRAM_PLAN_BYTES // 8))()
    assert lib.mbd_program_plan_launch(ctypes.addressof(buf), None) == mbd.ERR_INVALID_ARG
    assert lib.mbd_program_plan_launch(None, None) == mbd.ERR_INVALID_ARG
    n0 = mbd.kernel_launches()
    empty = mbd.program_plan_build([mbd.op_swiglu(None, None, 0, 64)])
    empty.launch()
    assert mbd.kernel_launches() == n0


def test_program_upload_checks(lib):
    buf = (ctypes.c_uint64 * (mbd.PROGRAM_PLAN_BYTES // 8))()
    n = mbd.program_schedule_bytes()
    assert n % 256 == 0 and n >= 8192
    assert lib.mbd_program_plan_upload(ctypes.addressof(buf), A, n, None) == mbd.ERR_INVALID_ARG   # unfilled plan
    assert lib.mbd_program_plan_launch_uploaded(ctypes.addressof(buf), A, None) == mbd.ERR_INVALID_ARG
    empty = mbd.program_plan_build([])
    pp = ctypes.addressof(empty.buf)
    assert lib.mbd_program_plan_upload(pp, None, n, None) == mbd.ERR_INVALID_ARG
    assert lib.mbd_program_plan_upload(pp, A + 16, n, None) == mbd.ERR_MISALIGNED
    assert lib.mbd_program_plan_upload(pp, A, n - 256, None) == mbd.ERR_INVALID_ARG
    assert lib.mbd_program_plan_launch_uploaded(pp, A + 16, None) == mbd.ERR_MISALIGNED
    assert lib.mbd_program_plan_launch_uploaded(pp, A, None) == 0                  # nothing to do: no launch


def test_program_static_launch_checks(lib):
    buf = (ctypes.c_uint64 * (mbd.PROGRAM_PLAN_BYTES // 8))()
    assert lib.mbd_program_plan_launch_static(ctypes.addressof(buf), None) == mbd.ERR_INVALID_ARG   # unfilled
    assert lib.mbd_program_plan_launch_static(None, None) == mbd.ERR_INVALID_ARG
    n0 = mbd.kernel_launches()
    mbd.program_plan_build([]).launch_static()                                                  # nothing to do
    assert mbd.kernel_launches() == n0
    hdr = open(mbd.HEADER_PATH).read()
    assert int(re.search(r"#define MBD_STATIC_SCHEDULE_BYTES (\d+)", hdr).group(1)) >= mbd.program_schedule_bytes()


def test_tuning_table_roundtrip_and_checks(lib, tmp_path):
    mbd.tuning_set([])
    assert mbd.tuning_get() == []
    e1 = {"kind": "swiglu_quant_fp8", "mode": "dynamic", "tokens": [1024, 4096], "width": [53248, 53248],
          "ctas_per_row": 7, "vectors_per_thread": 2, "threads": 480}
    e2 = {"kind": "add_rmsnorm", "mode": None, "tokens": [0, 1 << 40], "width": [1, 1 << 20],
          "ctas_per_row": 1, "vectors_per_thread": 4, "threads": 512}
    mbd.tuning_set([e1, e2])
    assert mbd.tuning_get() == [e1, e2]
    path = str(tmp_path / "t.json")
    mbd.tuning_save(path, [e1], {"device": "test"})
    mbd.tuning_set([])
    doc = mbd.tuning_load(path)
    assert doc["device"] == "test" and mbd.tuning_get() == [e1]
    bad = [dict(e1, threads=500), dict(e1, threads=1024), dict(e1, vectors_per_thread=3), dict(e1, ctas_per_row=0),
           dict(e1, tokens=[5, 4]), dict(e1, width=[-1, 4])]
    for b in bad:
        with pytest.raises(mbd.MbdError) as e:
            mbd.tuning_set([b])
        assert e.value.status == mbd.ERR_INVALID_ARG
    assert mbd.tuning_get() == [e1]                     # a rejected table leaves the old one in place
    ent = mbd.TuningEntry(9, 0, 0, 1, 0, 1, 1, 1, 32, 0)
    assert lib.mbd_tuning_set(ctypes.byref(ent), 1) == mbd.ERR_INVALID_ARG     # unknown kind
    ent = mbd.TuningEntry(4, 5, 0, 1, 0, 1, 1, 1, 32, 0)
    assert lib.mbd_tuning_set(ctypes.byref(ent), 1) == mbd.ERR_INVALID_ARG     # unknown FP8 mode
    assert lib.mbd_tuning_set(None, 1) == mbd.ERR_INVALID_ARG
    assert lib.mbd_tuning_set(None, -1) == mbd.ERR_INVALID_ARG
    mbd.tuning_set([])


def test_launch_shape_follows_table_then_rules(lib):
    mbd.tuning_set([])
    rules = mbd.launch_shape("swiglu_quant_fp8", "dynamic", 2048, 28672)
    rules_1000 = mbd.launch_shape("swiglu_quant_fp8", "dynamic", 1000, 28672)
    assert rules[0] <= 8 and rules[2] % 32 == 0
    mbd.tuning_set([{"kind": "swiglu_quant_fp8", "mode": "dynamic", "tokens": [2000, 3000], "width": [28672, 28672],
                     "ctas_per_row": 8, "vectors_per_thread": 4, "threads": 128}])
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", 2048, 28672) == (8, 4, 128)
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", 1000, 28672) == rules_1000      # outside the bucket
    assert mbd.launch_shape("swiglu_quant_fp8", "static", 2048, 28672) != (8, 4, 128)       # other mode
    # a shape that cannot cover the row (8 CTAs x 4 x 32 threads < 3584 vectors) falls back to the rules
    mbd.tuning_set([{"kind": "swiglu_quant_fp8", "mode": "dynamic", "tokens": [1, 1 << 30], "width": [1, 1 << 30],
                     "ctas_per_row": 8, "vectors_per_thread": 4, "threads": 32}])
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", 2048, 28672) == rules
    # wide dynamic rows at >= 4 rows per SM take the bulk-copy form whatever the table says: 6656 vectors in
    # clusters of 7 (slices of 951: 256 threads x 4), 10240 in clusters of 8 (320 threads); rows of 4608
    # vectors, and fewer rows, follow the table
    mbd.tuning_set([{"kind": "swiglu_quant_fp8", "mode": "dynamic", "tokens": [1, 1 << 30], "width": [1, 1 << 30],
                     "ctas_per_row": 8, "vectors_per_thread": 2, "threads": 512}])
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", 2048, 53248) == (7, 4, 256)
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", 2048, 81920) == (8, 4, 320)
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", 2048, 36864) == (8, 2, 512)
    assert mbd.launch_shape("swiglu_quant_fp8", "dynamic", 100, 53248) == (8, 2, 512)
    # NVFP4 slices are rounded up to an even number of vectors
    mbd.tuning_set([{"kind": "swiglu_quant_nvfp4", "mode": None, "tokens": [1, 1 << 30], "width": [1, 1 << 30],
                     "ctas_per_row": 3, "vectors_per_thread": 1, "threads": 64}])
    c, v, t = mbd.launch_shape("swiglu_quant_nvfp4", None, 4, 16 * 11)   # 22 vectors: slices of 8, 3 CTAs
    assert (c, v, t) == (3, 1, 64)
    mbd.tuning_set([])
    assert lib.mbd_launch_shape(9, 0, 1, 64, None, None, None) == mbd.ERR_INVALID_ARG


def test_independent_batch_checks(lib):
    """mbd_run_independent checks every op as its entry point does, and that no op touches what another
    writes, before any launch."""
    H = 64
    n0 = mbd.kernel_launches()
    a = mbd.op_add_rmsnorm(A, 2 * A, 3 * A, 9 * A, 4, H, 1e-6)
    # two norms updating one residual are not independent (the second reads what the first writes)
    b = mbd.op_add_rmsnorm(4 * A, 2 * A, 5 * A, 9 * A, 4, H, 1e-6)
    assert _rc(mbd.run_independent, [a, b]) == mbd.ERR_INVALID_ARG
    # a SwiGLU whose input is another op's output, and one whose output lands inside another op's input
    s_in = mbd.op_swiglu(6 * A, A, 4, H // 2)
    assert _rc(mbd.run_independent, [a, s_in]) == mbd.ERR_INVALID_ARG
    s_out = mbd.op_swiglu(3 * A + 64, 7 * A, 1, 8)
    assert _rc(mbd.run_independent, [a, s_out]) == mbd.ERR_INVALID_ARG
    # a dynamic scale written by one op and read as a static scale by another
    qd = mbd.op_swiglu_quant_fp8(8 * A, 7 * A, 4, H, "dynamic", 10 * A)
    qs = mbd.op_add_rmsnorm_quant_fp8(11 * A, 12 * A, 13 * A, 9 * A, 4, H, 1e-6, "static", 10 * A + 8)
    assert _rc(mbd.run_independent, [qd, qs]) == mbd.ERR_INVALID_ARG
    # each op's own checks, with its entry point's status
    assert _rc(mbd.run_independent, [a, mbd.op_add_rmsnorm(A + 2 * 4 * H * 8, 14 * A, 15 * A + 2, 9 * A, 4, H,
                                                            1e-6)]) == mbd.ERR_MISALIGNED
    assert _rc(mbd.run_independent, [a, mbd.op_swiglu(16 * A, 17 * A, -1, H)]) == mbd.ERR_INVALID_ARG
    bad = mbd.op_swiglu(16 * A, 17 * A, 4, H)
    bad.reserved = 1
    assert _rc(mbd.run_independent, [bad]) == mbd.ERR_INVALID_ARG
    bad = mbd.op_swiglu(16 * A, 17 * A, 4, H)
    bad.kind = 9
    assert _rc(mbd.run_independent, [bad]) == mbd.ERR_INVALID_ARG
    assert _rc(mbd.run_independent, [mbd.op_swiglu(16 * A, 17 * A, 4, H)] * (mbd.MAX_INDEPENDENT_OPS + 1)) \
        == mbd.ERR_INVALID_ARG
    # ops with no tokens are skipped, and touch nothing: an empty batch launches nothing
    mbd.run_independent([])
    mbd.run_independent([mbd.op_swiglu(None, None, 0, H), mbd.op_add_rmsnorm(None, None, None, None, 0, H, 1e-6)])
    assert mbd.kernel_launches() == n0


def test_batch_with_program_checks(lib):
    """mbd_run_independent_with_program rejects a null or unfilled plan and a misaligned schedule before any
    launch; a plan with nothing to do leaves the ops' own checks."""
    H = 64
    buf = (ctypes.c_uint64 * (mbd.PROGRAM_PLAN_BYTES // 8))()
    a = mbd.op_add_rmsnorm(A, 2 * A, 3 * A, 9 * A, 4, H, 1e-6)
    arr, n = mbd.program_array([a])
    n0 = mbd.kernel_launches()
    assert lib.mbd_run_independent_with_program(None, A, arr, n, None) == mbd.ERR_INVALID_ARG
    assert lib.mbd_run_independent_with_program(ctypes.addressof(buf), A, arr, n, None) == mbd.ERR_INVALID_ARG
    empty = mbd.program_plan_build([])
    pp = ctypes.addressof(empty.buf)
    assert lib.mbd_run_independent_with_program(pp, None, arr, n, None) == mbd.ERR_INVALID_ARG
    assert lib.mbd_run_independent_with_program(pp, A + 16, arr, n, None) == mbd.ERR_MISALIGNED
    b = mbd.op_add_rmsnorm(4 * A, 2 * A, 5 * A, 9 * A, 4, H, 1e-6)   # shares the residual with a
    arr2, n2 = mbd.program_array([a, b])
    assert lib.mbd_run_independent_with_program(pp, A, arr2, n2, None) == mbd.ERR_INVALID_ARG
    assert lib.mbd_run_independent_with_program(pp, A, None, 0, None) == 0     # nothing to do at all
    assert mbd.kernel_launches() == n0
