"""CPU oracle of the smoothed, quantized attention forward pass.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg import this package.  The CUDA library never does, and this
package imports nothing from it.

The arithmetic lives in ``sage_oracle.cpp`` (plain C++, one IEEE operation per
step, no fast-math, no FMA contraction).  This module compiles it with g++,
loads it with ctypes and wraps it for numpy arrays.  Every function works on
ONE segment (a batch entry or a packed sequence) in [H][L][D] order; callers
permute layouts before calling.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sage_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1
KEY_BLOCK = 128


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            L.oracle_padded_dim.argtypes = [I64]
            L.oracle_padded_dim.restype = I
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_value.restype = ctypes.c_float
            L.oracle_e4m3_encode_array.argtypes = [P, P, I64]
            L.oracle_e4m3_encode_array.restype = None
            L.oracle_exact_mean.argtypes = [P, I64, P]
            L.oracle_exact_mean.restype = I
            L.oracle_prologue.argtypes = [P, P, P, I, I64, I64, I64, I64, I64,
                                          P, P, P, P, P, P, P, P]
            L.oracle_prologue.restype = I
            L.oracle_attn.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64,
                                      I, ctypes.c_float, I64, I64, I64, I64, P, I]
            L.oracle_attn.restype = I
            L.oracle_attn_exact.argtypes = [P, P, P, I, I64, I64, I64, I64, I64,
                                            I, ctypes.c_double, I64, I64, I64,
                                            I64, P, I]
            L.oracle_attn_exact.restype = I
            L.oracle_fp16_encode.argtypes = [ctypes.c_float]
            L.oracle_fp16_encode.restype = ctypes.c_uint16
            L.oracle_v16.argtypes = [P, I, I64, I64, I64, P]
            L.oracle_v16.restype = I
            L.oracle_attn_pv16.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64,
                                           I, ctypes.c_float, I64, I64, I64, I64, P, I]
            L.oracle_attn_pv16.restype = I
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p)


def padded_dim(D: int) -> int:
    return int(lib().oracle_padded_dim(D))


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_value(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    L = lib()
    table = np.array([L.oracle_e4m3_value(c) for c in range(256)], dtype=np.float32)
    return table[codes]


def exact_mean(x) -> np.float32:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(1, dtype=np.float32)
    rc = lib().oracle_exact_mean(_ptr(x), x.size, _ptr(out))
    if rc:
        raise ValueError("exact sum does not fit the oracle accumulator")
    return out[0]


def prologue(q, k, v, dtype: int):
    """q [Hq,Lq,D], k/v [Hkv,Lk,D] as uint16 bit arrays of one segment."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    Hq, Lq, D = q.shape
    Hkv, Lk, _ = k.shape
    Dp = padded_dim(D)
    nkb = (Lk + KEY_BLOCK - 1) // KEY_BLOCK
    r = dict(
        q8=np.zeros((Hq, Lq, Dp), np.int8), s_q=np.zeros((Hq, Lq), np.float32),
        k_mean=np.zeros((Hkv, Dp), np.float32),
        k8=np.zeros((Hkv, Lk, Dp), np.int8), s_k=np.zeros((Hkv, nkb), np.float32),
        v_amax=np.zeros((Hkv, Dp), np.float32), s_v=np.zeros((Hkv, Dp), np.float32),
        v8=np.zeros((Hkv, Lk, Dp), np.uint8))
    rc = lib().oracle_prologue(
        _ptr(q), _ptr(k), _ptr(v), dtype, Hq, Hkv, Lq, Lk, D,
        _ptr(r["q8"]), _ptr(r["s_q"]), _ptr(r["k_mean"]), _ptr(r["k8"]),
        _ptr(r["s_k"]), _ptr(r["v_amax"]), _ptr(r["s_v"]), _ptr(r["v8"]))
    if rc:
        raise ValueError(f"oracle_prologue failed ({rc})")
    r.update(Hq=Hq, Hkv=Hkv, Lq=Lq, Lk=Lk, D=D, Dp=Dp)
    return r


def attn(pro: dict, causal: bool, sm_scale: float, heads=None, rows=None,
         nthreads: int = 0) -> np.ndarray:
    """Quantized attention from prologue outputs; [Hq,Lq,D] fp32.

    ``heads``/``rows`` are (begin, end) ranges; rows outside them stay NaN.
    """
    Hq, Lq, D = pro["Hq"], pro["Lq"], pro["D"]
    h0, h1 = heads if heads is not None else (0, Hq)
    r0, r1 = rows if rows is not None else (0, Lq)
    out = np.full((Hq, Lq, D), np.nan, dtype=np.float32)
    rc = lib().oracle_attn(
        _ptr(pro["q8"]), _ptr(pro["s_q"]), _ptr(pro["k8"]), _ptr(pro["s_k"]),
        _ptr(pro["v8"]), _ptr(pro["s_v"]), Hq, pro["Hkv"], Lq, pro["Lk"], D,
        int(bool(causal)), float(np.float32(sm_scale)), h0, h1, r0, r1,
        _ptr(out), nthreads)
    if rc:
        raise ValueError(f"oracle_attn failed ({rc})")
    return out


def fp16_encode(x) -> np.ndarray:
    """fp32 -> IEEE binary16 bits, round to nearest even (scalar loop: tests)."""
    x = np.asarray(x, dtype=np.float32)
    L = lib()
    flat = [L.oracle_fp16_encode(float(v)) for v in x.ravel()]
    return np.array(flat, dtype=np.uint16).reshape(x.shape)


def v16(v, dtype: int) -> np.ndarray:
    """V of one segment ([Hkv,Lk,D] input bits) rounded to fp16, padded to Dp:
    [Hkv,Lk,Dp] binary16 bits (the FP16-PV variant's V operand)."""
    v = np.ascontiguousarray(v, dtype=np.uint16)
    Hkv, Lk, D = v.shape
    out = np.zeros((Hkv, Lk, padded_dim(D)), dtype=np.uint16)
    rc = lib().oracle_v16(_ptr(v), dtype, Hkv, Lk, D, _ptr(out))
    if rc:
        raise ValueError(f"oracle_v16 failed ({rc})")
    return out


def attn_pv16(pro: dict, v16_bits: np.ndarray, causal: bool, sm_scale: float, heads=None,
              rows=None, nthreads: int = 0) -> np.ndarray:
    """FP16-PV variant from the prologue's Q/K operands and fp16 V; [Hq,Lq,D]
    fp32 (rows outside ``heads``/``rows`` stay NaN)."""
    Hq, Lq, D = pro["Hq"], pro["Lq"], pro["D"]
    h0, h1 = heads if heads is not None else (0, Hq)
    r0, r1 = rows if rows is not None else (0, Lq)
    v16_bits = np.ascontiguousarray(v16_bits, dtype=np.uint16)
    out = np.full((Hq, Lq, D), np.nan, dtype=np.float32)
    rc = lib().oracle_attn_pv16(
        _ptr(pro["q8"]), _ptr(pro["s_q"]), _ptr(pro["k8"]), _ptr(pro["s_k"]),
        _ptr(v16_bits), Hq, pro["Hkv"], Lq, pro["Lk"], D, int(bool(causal)),
        float(np.float32(sm_scale)), h0, h1, r0, r1, _ptr(out), nthreads)
    if rc:
        raise ValueError(f"oracle_attn_pv16 failed ({rc})")
    return out


def attn_exact(q, k, v, dtype: int, causal: bool, sm_scale: float, heads=None,
               rows=None, nthreads: int = 0) -> np.ndarray:
    """Unquantized fp64 attention of one segment; [Hq,Lq,D] float64."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    Hq, Lq, D = q.shape
    Hkv, Lk, _ = k.shape
    h0, h1 = heads if heads is not None else (0, Hq)
    r0, r1 = rows if rows is not None else (0, Lq)
    out = np.full((Hq, Lq, D), np.nan, dtype=np.float64)
    rc = lib().oracle_attn_exact(
        _ptr(q), _ptr(k), _ptr(v), dtype, Hq, Hkv, Lq, Lk, D, int(bool(causal)),
        float(sm_scale), h0, h1, r0, r1, _ptr(out), nthreads)
    if rc:
        raise ValueError(f"oracle_attn_exact failed ({rc})")
    return out
