"""CPU oracle for the decoder-layer fusions -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the bench's CPU-baseline leg may import this package. It wraps the
plain fp64 C oracle (oracle.c) through ctypes; it shares no code with the CUDA library and never imports
it. The C source cites the pages it follows; this file only marshals numpy arrays.

All functions take and return numpy arrays; bf16 tensors are uint16 bit patterns, FP8 codes uint8.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
LIB_PATH = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C11, no FMA contraction) if it is missing or stale."""
    stale = (not os.path.exists(LIB_PATH) or
             os.path.getmtime(LIB_PATH) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = LIB_PATH + ".tmp"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f64p = ctypes.POINTER(ctypes.c_double)
        f32p = ctypes.POINTER(ctypes.c_float)
        i64, f32, cint = ctypes.c_int64, ctypes.c_float, ctypes.c_int
        lib.orc_bf16_to_double.argtypes, lib.orc_bf16_to_double.restype = [ctypes.c_uint16], ctypes.c_double
        lib.orc_bf16_round.argtypes, lib.orc_bf16_round.restype = [ctypes.c_double], ctypes.c_uint16
        lib.orc_bf16_sum.argtypes, lib.orc_bf16_sum.restype = [ctypes.POINTER(ctypes.c_uint16), ctypes.c_int], ctypes.c_uint16
        lib.orc_e4m3_decode.argtypes, lib.orc_e4m3_decode.restype = [ctypes.c_uint8], ctypes.c_double
        lib.orc_e4m3_encode.argtypes, lib.orc_e4m3_encode.restype = [ctypes.c_double], ctypes.c_uint8
        lib.orc_silu.argtypes, lib.orc_silu.restype = [ctypes.c_double], ctypes.c_double
        lib.orc_e2m1_decode.argtypes, lib.orc_e2m1_decode.restype = [ctypes.c_uint8], ctypes.c_double
        lib.orc_e2m1_encode.argtypes, lib.orc_e2m1_encode.restype = [ctypes.c_double], ctypes.c_uint8
        lib.orc_add_rmsnorm_quant_nvfp4.argtypes = [u16p, u16p, u16p, i64, i64, f32, f32, u16p, u8p, u8p, f64p]
        lib.orc_swiglu_quant_nvfp4.argtypes = [u16p, i64, i64, f32, u8p, u8p, f64p]
        lib.orc_add_rmsnorm.argtypes = [u16p, u16p, u16p, i64, i64, f32, u16p, f64p, u16p]
        lib.orc_add_rmsnorm_quant_fp8.argtypes = [u16p, u16p, u16p, i64, i64, f32, cint, f32p, u16p, u8p, f64p]
        u16pp = ctypes.POINTER(u16p)
        lib.orc_allreduce_add_rmsnorm.argtypes = [u16pp, cint, u16p, u16p, i64, i64, f32, u16p, f64p, u16p]
        lib.orc_allreduce_add_rmsnorm_quant_fp8.argtypes = [u16pp, cint, u16p, u16p, i64, i64, f32, cint, f32p,
                                                            u16p, u8p, f64p]
        lib.orc_swiglu.argtypes = [u16p, i64, i64, f64p, u16p]
        lib.orc_swiglu_quant_fp8.argtypes = [u16p, i64, i64, cint, f32p, u8p, f64p]
        for fn in ("orc_add_rmsnorm", "orc_add_rmsnorm_quant_fp8", "orc_swiglu", "orc_swiglu_quant_fp8",
                   "orc_allreduce_add_rmsnorm", "orc_allreduce_add_rmsnorm_quant_fp8",
                   "orc_add_rmsnorm_quant_nvfp4", "orc_swiglu_quant_nvfp4"):
            getattr(lib, fn).restype = cint
        _lib = lib
        return lib


def _p(a: Optional[np.ndarray], ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid argument")


MODES = {"static": 0, "dynamic": 1}


def bf16_to_double(b: int) -> float:
    return _load().orc_bf16_to_double(int(b))


def bf16_round(v: float) -> int:
    return int(_load().orc_bf16_round(float(v)))


def bf16_sum(bits) -> int:
    """bf16 bits of the exact sum of up to 8 bf16 values (given as bits), rounded once; a zero sum is +0."""
    a = np.ascontiguousarray(np.asarray(bits, np.uint16).reshape(-1))
    if not 1 <= a.size <= 8:
        raise ValueError("1 to 8 addends")
    return int(_load().orc_bf16_sum(a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), int(a.size)))


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(int(code))


def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


def e2m1_decode(code: int) -> float:
    return _load().orc_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return int(_load().orc_e2m1_encode(float(v)))


def add_rmsnorm_quant_nvfp4(x, r, w, eps: float, tensor_scale: float, want_v: bool = True):
    """Returns (residual_out [T,H] u16, q packed [T,H/2] u8, sf [T,H/16] u8 E4M3, v or None)."""
    x = np.ascontiguousarray(x, np.uint16)
    r = np.ascontiguousarray(r, np.uint16)
    w = np.ascontiguousarray(w, np.uint16)
    T, H = x.shape
    res = np.empty((T, H), np.uint16)
    q = np.empty((T, H // 2), np.uint8)
    sf = np.empty((T, H // 16), np.uint8)
    v = np.empty((T, H), np.float64) if want_v else None
    u16, u8, f64 = ctypes.c_uint16, ctypes.c_uint8, ctypes.c_double
    _check(_load().orc_add_rmsnorm_quant_nvfp4(_p(x, u16), _p(r, u16), _p(w, u16), T, H, float(eps),
                                               float(tensor_scale), _p(res, u16), _p(q, u8), _p(sf, u8), _p(v, f64)),
           "add_rmsnorm_quant_nvfp4")
    return res, q, sf, v


def swiglu_quant_nvfp4(gate_up, tensor_scale: float, want_h: bool = True):
    """Returns (q packed [T,I/2] u8, sf [T,I/16] u8 E4M3, h or None)."""
    gu = np.ascontiguousarray(gate_up, np.uint16)
    T, I2 = gu.shape
    I = I2 // 2
    q = np.empty((T, I // 2), np.uint8)
    sf = np.empty((T, I // 16), np.uint8)
    h = np.empty((T, I), np.float64) if want_h else None
    _check(_load().orc_swiglu_quant_nvfp4(_p(gu, ctypes.c_uint16), T, I, float(tensor_scale), _p(q, ctypes.c_uint8),
                                          _p(sf, ctypes.c_uint8), _p(h, ctypes.c_double)), "swiglu_quant_nvfp4")
    return q, sf, h


def silu(g: float) -> float:
    return _load().orc_silu(float(g))


def add_rmsnorm(x: np.ndarray, r: np.ndarray, w: np.ndarray, eps: float,
                want_v: bool = True) -> Tuple[np.ndarray, np.ndarray, Optional[np.ndarray]]:
    """Returns (residual_out bf16 bits [T,H], out bf16 bits [T,H], v exact float64 [T,H] or None)."""
    x = np.ascontiguousarray(x, np.uint16)
    r = np.ascontiguousarray(r, np.uint16)
    w = np.ascontiguousarray(w, np.uint16)
    T, H = x.shape
    res = np.empty((T, H), np.uint16)
    out = np.empty((T, H), np.uint16)
    v = np.empty((T, H), np.float64) if want_v else None
    u16, f64 = ctypes.c_uint16, ctypes.c_double
    _check(_load().orc_add_rmsnorm(_p(x, u16), _p(r, u16), _p(w, u16), T, H, float(eps), _p(res, u16),
                                   _p(v, f64), _p(out, u16)), "add_rmsnorm")
    return res, out, v


def add_rmsnorm_quant_fp8(x: np.ndarray, r: np.ndarray, w: np.ndarray, eps: float, mode: str,
                          static_scale: float = 0.0, want_v: bool = True):
    """Returns (residual_out [T,H] u16, q [T,H] u8, scale float32 ([1] static / [T] dynamic), v or None)."""
    x = np.ascontiguousarray(x, np.uint16)
    r = np.ascontiguousarray(r, np.uint16)
    w = np.ascontiguousarray(w, np.uint16)
    T, H = x.shape
    res = np.empty((T, H), np.uint16)
    q = np.empty((T, H), np.uint8)
    scale = np.array([static_scale], np.float32) if mode == "static" else np.zeros((max(T, 1),), np.float32)
    v = np.empty((T, H), np.float64) if want_v else None
    u16, u8, f32, f64 = ctypes.c_uint16, ctypes.c_uint8, ctypes.c_float, ctypes.c_double
    _check(_load().orc_add_rmsnorm_quant_fp8(_p(x, u16), _p(r, u16), _p(w, u16), T, H, float(eps),
                                             MODES[mode], _p(scale, f32), _p(res, u16), _p(q, u8),
                                             _p(v, f64)), "add_rmsnorm_quant_fp8")
    return res, q, (scale if mode == "static" else scale[:T]), v


def _partials_arg(partials):
    arrs = [np.ascontiguousarray(p, np.uint16) for p in partials]
    u16p = ctypes.POINTER(ctypes.c_uint16)
    arr_t = u16p * len(arrs)
    return arrs, arr_t(*[a.ctypes.data_as(u16p) for a in arrs])


def allreduce_add_rmsnorm(partials, r: np.ndarray, w: np.ndarray, eps: float, want_v: bool = True):
    """x = bf16(sum of partials), then add + RMSNorm. Returns (residual_out, out, v or None)."""
    arrs, parr = _partials_arg(partials)
    r = np.ascontiguousarray(r, np.uint16)
    w = np.ascontiguousarray(w, np.uint16)
    T, H = r.shape
    res = np.empty((T, H), np.uint16)
    out = np.empty((T, H), np.uint16)
    v = np.empty((T, H), np.float64) if want_v else None
    u16, f64 = ctypes.c_uint16, ctypes.c_double
    _check(_load().orc_allreduce_add_rmsnorm(parr, len(arrs), _p(r, u16), _p(w, u16), T, H, float(eps),
                                             _p(res, u16), _p(v, f64), _p(out, u16)), "allreduce_add_rmsnorm")
    return res, out, v


def allreduce_add_rmsnorm_quant_fp8(partials, r: np.ndarray, w: np.ndarray, eps: float, mode: str,
                                    static_scale: float = 0.0, want_v: bool = True):
    """Returns (residual_out, q, scale ([1] static / [T] dynamic), v or None)."""
    arrs, parr = _partials_arg(partials)
    r = np.ascontiguousarray(r, np.uint16)
    w = np.ascontiguousarray(w, np.uint16)
    T, H = r.shape
    res = np.empty((T, H), np.uint16)
    q = np.empty((T, H), np.uint8)
    scale = np.array([static_scale], np.float32) if mode == "static" else np.zeros((max(T, 1),), np.float32)
    v = np.empty((T, H), np.float64) if want_v else None
    u16, u8, f32, f64 = ctypes.c_uint16, ctypes.c_uint8, ctypes.c_float, ctypes.c_double
    _check(_load().orc_allreduce_add_rmsnorm_quant_fp8(parr, len(arrs), _p(r, u16), _p(w, u16), T, H, float(eps),
                                                       MODES[mode], _p(scale, f32), _p(res, u16), _p(q, u8),
                                                       _p(v, f64)), "allreduce_add_rmsnorm_quant_fp8")
    return res, q, (scale if mode == "static" else scale[:T]), v


def swiglu(gate_up: np.ndarray, want_h: bool = True) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """Returns (out bf16 bits [T,I], h exact float64 [T,I] or None)."""
    gu = np.ascontiguousarray(gate_up, np.uint16)
    T, I2 = gu.shape
    I = I2 // 2
    out = np.empty((T, I), np.uint16)
    h = np.empty((T, I), np.float64) if want_h else None
    _check(_load().orc_swiglu(_p(gu, ctypes.c_uint16), T, I, _p(h, ctypes.c_double),
                              _p(out, ctypes.c_uint16)), "swiglu")
    return out, h


def swiglu_quant_fp8(gate_up: np.ndarray, mode: str, static_scale: float = 0.0, want_h: bool = True):
    """Returns (q [T,I] u8, scale float32 ([1] static / [T] dynamic), h exact float64 or None)."""
    gu = np.ascontiguousarray(gate_up, np.uint16)
    T, I2 = gu.shape
    I = I2 // 2
    q = np.empty((T, I), np.uint8)
    scale = np.array([static_scale], np.float32) if mode == "static" else np.zeros((max(T, 1),), np.float32)
    h = np.empty((T, I), np.float64) if want_h else None
    _check(_load().orc_swiglu_quant_fp8(_p(gu, ctypes.c_uint16), T, I, MODES[mode],
                                        _p(scale, ctypes.c_float), _p(q, ctypes.c_uint8),
                                        _p(h, ctypes.c_double)), "swiglu_quant_fp8")
    return q, (scale if mode == "static" else scale[:T]), h
