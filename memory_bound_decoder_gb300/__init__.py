"""Python binding of libmbd, the GB300 library of memory-bound decoder-layer fusions.

Argument marshalling only: every function here converts its arguments (torch tensors or raw integer
device pointers) and calls the C entry point of the same name (without the `mbd_` prefix), which
launches one CUDA kernel. Nothing is computed in Python and there is no fallback: if libmbd.so has not
been built, the first call (or any access to `lib`) raises ImportError.

    import memory_bound_decoder_gb300 as mbd
    mbd.fused_add_rmsnorm(out, residual, x, weight, T, H, 1e-6)          # tensors on the GPU
    mbd.swiglu_quant_fp8(q, gate_up, T, I, mbd.DYNAMIC, scales)
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Any, List, Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmbd.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "mbd.h")

STATIC = 0   # MBD_SCALE_STATIC_PER_TENSOR
DYNAMIC = 1  # MBD_SCALE_DYNAMIC_PER_TOKEN
MODES = {"static": STATIC, "dynamic": DYNAMIC, STATIC: STATIC, DYNAMIC: DYNAMIC}

OK, ERR_INVALID_ARG, ERR_MISALIGNED, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3, 4


class MbdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class Op(ctypes.Structure):
    """One operation of a program (the C struct mbd_op)."""
    _fields_ = [("kind", ctypes.c_int32), ("mode", ctypes.c_int32), ("n_tokens", ctypes.c_int64),
                ("width", ctypes.c_int64), ("eps", ctypes.c_float), ("reserved", ctypes.c_int32),
                ("out", ctypes.c_void_p), ("out_sf", ctypes.c_void_p), ("residual", ctypes.c_void_p),
                ("in_", ctypes.c_void_p), ("weight", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


OP_ADD_RMSNORM = 0
OP_ADD_RMSNORM_QUANT_FP8 = 1
OP_ADD_RMSNORM_QUANT_NVFP4 = 2
OP_SWIGLU = 3
OP_SWIGLU_QUANT_FP8 = 4
OP_SWIGLU_QUANT_NVFP4 = 5
MAX_PROGRAM_OPS = 128
MAX_INDEPENDENT_OPS = 64
PROGRAM_PLAN_BYTES = 16384


class TuningEntry(ctypes.Structure):
    """One row of the launch-shape table (the C struct mbd_tuning_entry)."""
    _fields_ = [("kind", ctypes.c_int32), ("mode", ctypes.c_int32), ("tokens_min", ctypes.c_int64),
                ("tokens_max", ctypes.c_int64), ("width_min", ctypes.c_int64), ("width_max", ctypes.c_int64),
                ("ctas_per_row", ctypes.c_int32), ("vectors_per_thread", ctypes.c_int32), ("threads", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


OP_NAMES = {0: "add_rmsnorm", 1: "add_rmsnorm_quant_fp8", 2: "add_rmsnorm_quant_nvfp4", 3: "swiglu",
            4: "swiglu_quant_fp8", 5: "swiglu_quant_nvfp4"}
OP_KINDS = {v: k for k, v in OP_NAMES.items()}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with memory_bound_decoder_gb300.build.build() "
                          "(there is no non-CUDA fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, f32, cint = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    lib.mbd_abi_version.restype = cint
    lib.mbd_status_string.argtypes, lib.mbd_status_string.restype = [cint], ctypes.c_char_p
    lib.mbd_last_cuda_error.restype = cint
    lib.mbd_kernel_launches.restype = ctypes.c_uint64
    lib.mbd_device_error_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), cint]
    lib.mbd_device_error_flags.restype = cint
    lib.mbd_selftest_bounded_wait.argtypes = [ctypes.c_uint64, vp]
    lib.mbd_selftest_bounded_wait.restype = cint
    lib.mbd_fused_add_rmsnorm.argtypes = [vp, vp, vp, vp, i64, i64, f32, vp]
    lib.mbd_fused_add_rmsnorm_quant_fp8.argtypes = [vp, vp, vp, vp, i64, i64, f32, cint, vp, vp]
    lib.mbd_fused_allreduce_add_rmsnorm.argtypes = [vp, vp, ctypes.POINTER(vp), cint, vp, i64, i64, f32, vp]
    lib.mbd_fused_allreduce_add_rmsnorm_quant_fp8.argtypes = [vp, vp, ctypes.POINTER(vp), cint, vp, i64, i64, f32,
                                                              cint, vp, vp]
    lib.mbd_swiglu.argtypes = [vp, vp, i64, i64, vp]
    lib.mbd_swiglu_quant_fp8.argtypes = [vp, vp, i64, i64, cint, vp, vp]
    lib.mbd_fused_add_rmsnorm_quant_nvfp4.argtypes = [vp, vp, vp, vp, vp, i64, i64, f32, vp, vp]
    lib.mbd_swiglu_quant_nvfp4.argtypes = [vp, vp, vp, i64, i64, vp, vp]
    lib.mbd_run_program.argtypes = [ctypes.POINTER(Op), cint, vp]
    lib.mbd_run_independent.argtypes = [ctypes.POINTER(Op), cint, vp]
    lib.mbd_run_independent_with_program.argtypes = [vp, vp, ctypes.POINTER(Op), cint, vp]
    lib.mbd_program_plan_build.argtypes = [ctypes.POINTER(Op), cint, vp]
    lib.mbd_program_plan_launch.argtypes = [vp, vp]
    lib.mbd_program_schedule_bytes.restype = ctypes.c_size_t
    lib.mbd_program_plan_upload.argtypes = [vp, vp, ctypes.c_size_t, vp]
    lib.mbd_program_plan_launch_uploaded.argtypes = [vp, vp, vp]
    lib.mbd_program_plan_launch_static.argtypes = [vp, vp]
    lib.mbd_tuning_set.argtypes = [ctypes.POINTER(TuningEntry), cint]
    lib.mbd_tuning_set.restype = cint
    lib.mbd_tuning_get.argtypes = [ctypes.POINTER(TuningEntry), cint]
    lib.mbd_tuning_get.restype = cint
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.mbd_launch_shape.argtypes = [cint, cint, i64, i64, i32p, i32p, i32p]
    lib.mbd_launch_shape.restype = cint
    for fn in ("mbd_fused_add_rmsnorm", "mbd_fused_add_rmsnorm_quant_fp8", "mbd_swiglu", "mbd_swiglu_quant_fp8",
               "mbd_fused_allreduce_add_rmsnorm", "mbd_fused_allreduce_add_rmsnorm_quant_fp8",
               "mbd_fused_add_rmsnorm_quant_nvfp4", "mbd_swiglu_quant_nvfp4", "mbd_run_program",
               "mbd_run_independent", "mbd_run_independent_with_program", "mbd_program_plan_build", "mbd_program_plan_launch", "mbd_program_plan_upload",
               "mbd_program_plan_launch_uploaded", "mbd_program_plan_launch_static"):
        getattr(lib, fn).restype = cint
    return lib


_LIB: Optional[ctypes.CDLL] = None


def get_lib() -> ctypes.CDLL:
    """The loaded libmbd.so (loaded on first use; ImportError if it has not been built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load()
    return _LIB


def __getattr__(name: str):
    if name == "lib":
        return get_lib()
    raise AttributeError(name)


def header_functions() -> List[str]:
    """Names of the functions include/mbd.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mbd_[a-z0-9_]+)\s*\(", text)))


def _ptr(a: Any) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    dp = getattr(a, "data_ptr", None)
    if dp is not None:
        return int(dp())
    raise TypeError(f"expected a tensor or an integer device pointer, got {type(a).__name__}")


def _mode(mode: Any) -> int:
    """'static' / 'dynamic' or the integer enum value (passed through unchanged for the library to check)."""
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _stream(stream: Any) -> Optional[int]:
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return int(torch.cuda.current_stream().cuda_stream)
        except ImportError:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return int(getattr(stream, "cuda_stream"))


def _check(status: int, fn: str) -> None:
    if status != OK:
        lib = get_lib()
        msg = lib.mbd_status_string(status).decode()
        if status == ERR_CUDA:
            msg += f" (cudaError {lib.mbd_last_cuda_error()})"
        raise MbdError(status, f"{fn}: {msg}")


def abi_version() -> int:
    return get_lib().mbd_abi_version()


def kernel_launches() -> int:
    return int(get_lib().mbd_kernel_launches())


DEVERR_EXCHANGE_TIMEOUT = 1


def device_error_flags(clear: bool = False) -> int:
    """OR of the library's device error words on the current device (synchronous)."""
    v = ctypes.c_uint32(0)
    _check(get_lib().mbd_device_error_flags(ctypes.byref(v), int(bool(clear))), "device_error_flags")
    return int(v.value)


def selftest_bounded_wait(limit_cycles: int, stream=None) -> None:
    """Launch the self-test kernel whose wait can only time out (sets DEVERR_EXCHANGE_TIMEOUT)."""
    _check(get_lib().mbd_selftest_bounded_wait(int(limit_cycles), _stream(stream)), "selftest_bounded_wait")


def fused_add_rmsnorm(out, residual, x, weight, n_tokens: int, hidden: int, eps: float, stream=None) -> None:
    _check(get_lib().mbd_fused_add_rmsnorm(_ptr(out), _ptr(residual), _ptr(x), _ptr(weight), int(n_tokens),
                                     int(hidden), float(eps), _stream(stream)), "fused_add_rmsnorm")


def fused_add_rmsnorm_quant_fp8(out_q, residual, x, weight, n_tokens: int, hidden: int, eps: float, mode,
                                scale, stream=None) -> None:
    _check(get_lib().mbd_fused_add_rmsnorm_quant_fp8(_ptr(out_q), _ptr(residual), _ptr(x), _ptr(weight),
                                               int(n_tokens), int(hidden), float(eps), _mode(mode),
                                               _ptr(scale), _stream(stream)), "fused_add_rmsnorm_quant_fp8")


def fused_add_rmsnorm_quant_nvfp4(out_q, out_sf, residual, x, weight, n_tokens: int, hidden: int, eps: float,
                                  tensor_scale, stream=None) -> None:
    _check(get_lib().mbd_fused_add_rmsnorm_quant_nvfp4(_ptr(out_q), _ptr(out_sf), _ptr(residual), _ptr(x),
                                                       _ptr(weight), int(n_tokens), int(hidden), float(eps),
                                                       _ptr(tensor_scale), _stream(stream)),
           "fused_add_rmsnorm_quant_nvfp4")


def _ptr_array(items) -> Any:
    if items is None:
        return None
    vals = [_ptr(a) for a in items]
    return (ctypes.c_void_p * max(1, len(vals)))(*vals)


def fused_allreduce_add_rmsnorm(out, residual, partials, weight, n_tokens: int, hidden: int, eps: float,
                                stream=None) -> None:
    """`partials`: a sequence of tensors or device pointers (the C entry point gets a host pointer array)."""
    n = len(partials) if partials is not None else 0
    _check(get_lib().mbd_fused_allreduce_add_rmsnorm(_ptr(out), _ptr(residual), _ptr_array(partials), n, _ptr(weight),
                                                     int(n_tokens), int(hidden), float(eps), _stream(stream)),
           "fused_allreduce_add_rmsnorm")


def fused_allreduce_add_rmsnorm_quant_fp8(out_q, residual, partials, weight, n_tokens: int, hidden: int, eps: float,
                                          mode, scale, stream=None) -> None:
    n = len(partials) if partials is not None else 0
    _check(get_lib().mbd_fused_allreduce_add_rmsnorm_quant_fp8(_ptr(out_q), _ptr(residual), _ptr_array(partials), n,
                                                               _ptr(weight), int(n_tokens), int(hidden), float(eps),
                                                               _mode(mode), _ptr(scale), _stream(stream)),
           "fused_allreduce_add_rmsnorm_quant_fp8")


def swiglu(out, gate_up, n_tokens: int, inter: int, stream=None) -> None:
    _check(get_lib().mbd_swiglu(_ptr(out), _ptr(gate_up), int(n_tokens), int(inter), _stream(stream)), "swiglu")


def swiglu_quant_fp8(out_q, gate_up, n_tokens: int, inter: int, mode, scale, stream=None) -> None:
    _check(get_lib().mbd_swiglu_quant_fp8(_ptr(out_q), _ptr(gate_up), int(n_tokens), int(inter), _mode(mode),
                                    _ptr(scale), _stream(stream)), "swiglu_quant_fp8")


def swiglu_quant_nvfp4(out_q, out_sf, gate_up, n_tokens: int, inter: int, tensor_scale, stream=None) -> None:
    _check(get_lib().mbd_swiglu_quant_nvfp4(_ptr(out_q), _ptr(out_sf), _ptr(gate_up), int(n_tokens), int(inter),
                                            _ptr(tensor_scale), _stream(stream)), "swiglu_quant_nvfp4")


# ------------------------------------------------------------------------------------------------ programs

def op_add_rmsnorm(out, residual, x, weight, n_tokens: int, hidden: int, eps: float) -> Op:
    return Op(OP_ADD_RMSNORM, 0, int(n_tokens), int(hidden), float(eps), 0, _ptr(out), None, _ptr(residual),
              _ptr(x), _ptr(weight), None)


def op_add_rmsnorm_quant_fp8(out_q, residual, x, weight, n_tokens: int, hidden: int, eps: float, mode,
                             scale) -> Op:
    return Op(OP_ADD_RMSNORM_QUANT_FP8, _mode(mode), int(n_tokens), int(hidden), float(eps), 0, _ptr(out_q), None,
              _ptr(residual), _ptr(x), _ptr(weight), _ptr(scale))


def op_add_rmsnorm_quant_nvfp4(out_q, out_sf, residual, x, weight, n_tokens: int, hidden: int, eps: float,
                               tensor_scale) -> Op:
    return Op(OP_ADD_RMSNORM_QUANT_NVFP4, 0, int(n_tokens), int(hidden), float(eps), 0, _ptr(out_q), _ptr(out_sf),
              _ptr(residual), _ptr(x), _ptr(weight), _ptr(tensor_scale))


def op_swiglu(out, gate_up, n_tokens: int, inter: int) -> Op:
    return Op(OP_SWIGLU, 0, int(n_tokens), int(inter), 0.0, 0, _ptr(out), None, None, _ptr(gate_up), None, None)


def op_swiglu_quant_fp8(out_q, gate_up, n_tokens: int, inter: int, mode, scale) -> Op:
    return Op(OP_SWIGLU_QUANT_FP8, _mode(mode), int(n_tokens), int(inter), 0.0, 0, _ptr(out_q), None, None,
              _ptr(gate_up), None, _ptr(scale))


def op_swiglu_quant_nvfp4(out_q, out_sf, gate_up, n_tokens: int, inter: int, tensor_scale) -> Op:
    return Op(OP_SWIGLU_QUANT_NVFP4, 0, int(n_tokens), int(inter), 0.0, 0, _ptr(out_q), _ptr(out_sf), None,
              _ptr(gate_up), None, _ptr(tensor_scale))


def program_array(ops) -> Any:
    """A ctypes array of Op for mbd_run_program (keep it alive while launching it repeatedly)."""
    ops = list(ops)
    return (Op * max(1, len(ops)))(*ops), len(ops)


def run_program(ops, stream=None) -> None:
    """Run a list of Op (or a program_array result) as one persistent kernel launch."""
    arr, n = ops if isinstance(ops, tuple) else program_array(ops)
    _check(get_lib().mbd_run_program(arr if n else None, n, _stream(stream)), "run_program")


def run_independent(ops, stream=None) -> None:
    """Run a list of Op (or a program_array result) that share no written memory as their own single-call
    launches, each overlapping the one before it (mbd_run_independent)."""
    arr, n = ops if isinstance(ops, tuple) else program_array(ops)
    _check(get_lib().mbd_run_independent(arr if n else None, n, _stream(stream)), "run_independent")


def run_independent_with_program(plan, schedule, ops, stream=None) -> None:
    """A program (a built plan whose schedule was uploaded to `schedule`) launched first, then the independent ops
    of a batch, every launch after the program overlapping the one before (mbd_run_independent_with_program)."""
    arr, n = ops if isinstance(ops, tuple) else program_array(ops)
    _check(get_lib().mbd_run_independent_with_program(ctypes.addressof(plan.buf), _ptr(schedule), arr if n else None,
                                                      n, _stream(stream)), "run_independent_with_program")


class ProgramPlan:
    """A built program (the C mbd_program_plan): plain host memory, launched any number of times. Keeps the
    descriptor array alive with it (the plan itself holds only the ops' device pointers)."""

    def __init__(self, ops):
        self.buf = (ctypes.c_uint64 * (PROGRAM_PLAN_BYTES // 8))()
        self.arr, n = program_array(ops)
        _check(get_lib().mbd_program_plan_build(self.arr if n else None, n, ctypes.addressof(self.buf)),
               "program_plan_build")

    def launch(self, stream=None) -> None:
        _check(get_lib().mbd_program_plan_launch(ctypes.addressof(self.buf), _stream(stream)), "program_plan_launch")

    def upload(self, schedule, stream=None) -> None:
        """Copy the schedule into device memory `schedule` (a tensor or pointer of program_schedule_bytes())."""
        nbytes = schedule.numel() * schedule.element_size() if hasattr(schedule, "numel") else program_schedule_bytes()
        _check(get_lib().mbd_program_plan_upload(ctypes.addressof(self.buf), _ptr(schedule), nbytes, _stream(stream)),
               "program_plan_upload")

    def launch_uploaded(self, schedule, stream=None) -> None:
        _check(get_lib().mbd_program_plan_launch_uploaded(ctypes.addressof(self.buf), _ptr(schedule), _stream(stream)),
               "program_plan_launch_uploaded")

    def launch_static(self, stream=None) -> None:
        """Upload into the library's static schedule buffer and launch (allocates nothing)."""
        _check(get_lib().mbd_program_plan_launch_static(ctypes.addressof(self.buf), _stream(stream)),
               "program_plan_launch_static")


def program_schedule_bytes() -> int:
    return int(get_lib().mbd_program_schedule_bytes())


def program_plan_upload(plan: ProgramPlan, schedule, stream=None) -> None:
    plan.upload(schedule, stream)


def program_plan_launch_uploaded(plan: ProgramPlan, schedule, stream=None) -> None:
    plan.launch_uploaded(schedule, stream)


def program_plan_launch_static(plan: ProgramPlan, stream=None) -> None:
    plan.launch_static(stream)


def program_plan_build(ops) -> ProgramPlan:
    return ProgramPlan(ops)


def program_plan_launch(plan: ProgramPlan, stream=None) -> None:
    plan.launch(stream)


# ------------------------------------------------------------------------------------------------ tuning

def tuning_set(entries) -> None:
    """Install a launch-shape table (a list of TuningEntry or of dicts as in tuning files); [] clears it."""
    rows = [e if isinstance(e, TuningEntry) else _entry_from_dict(e) for e in entries]
    arr = (TuningEntry * max(1, len(rows)))(*rows)
    _check(get_lib().mbd_tuning_set(arr if rows else None, len(rows)), "tuning_set")


def launch_shape(kind, mode, n_tokens: int, width: int) -> tuple:
    """(CTAs per row, vectors per thread, threads) a call would launch with now (table, else rules)."""
    c, v, t = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    k = OP_KINDS[kind] if isinstance(kind, str) else int(kind)
    _check(get_lib().mbd_launch_shape(k, MODES[mode or "static"], int(n_tokens), int(width), ctypes.byref(c),
                                      ctypes.byref(v), ctypes.byref(t)), "launch_shape")
    return c.value, v.value, t.value


def tuning_get() -> list:
    lib = get_lib()
    n = lib.mbd_tuning_get(None, 0)
    arr = (TuningEntry * max(1, n))()
    n = lib.mbd_tuning_get(arr, n)
    return [_entry_to_dict(arr[i]) for i in range(n)]


def _entry_from_dict(d) -> TuningEntry:
    return TuningEntry(OP_KINDS[d["kind"]], MODES[d.get("mode") or "static"], int(d["tokens"][0]), int(d["tokens"][1]),
                       int(d["width"][0]), int(d["width"][1]), int(d["ctas_per_row"]), int(d["vectors_per_thread"]),
                       int(d["threads"]), 0)


def _entry_to_dict(e: TuningEntry) -> dict:
    fp8 = e.kind in (1, 4)
    return {"kind": OP_NAMES[e.kind], "mode": ("static", "dynamic")[e.mode] if fp8 else None,
            "tokens": [e.tokens_min, e.tokens_max], "width": [e.width_min, e.width_max],
            "ctas_per_row": e.ctas_per_row, "vectors_per_thread": e.vectors_per_thread, "threads": e.threads}


def tuning_save(path: str, entries, meta: Optional[dict] = None) -> None:
    import json
    doc = dict(meta or {})
    doc["entries"] = [e if isinstance(e, dict) else _entry_to_dict(e) for e in entries]
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


def tuning_load(path: str) -> dict:
    """Read a tuning file (written by memory_bound_decoder_gb300.tune) and install its table."""
    import json
    with open(path) as f:
        doc = json.load(f)
    tuning_set(doc["entries"])
    return doc
