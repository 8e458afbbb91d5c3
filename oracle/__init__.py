"""CPU oracle for the QLoRA NF4 + LoRA linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline / reference
arm may import this package.  The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``nf4_oracle.c`` (plain C loops, fp64 contractions); this module
only marshals numpy arrays through ctypes.  Every function cites the passage of the QLoRA
pages it follows in the C file's header (readings R1-R8).

Pinning status: levels, quantize, double quantization, dequantize and the LoRA
forward/backward are pinned by the not-gpu tests in ``tests/test_oracle_pins.py``
(structural invariants, brute force on small inputs, closed forms, numpy matmul special
cases and finite differences).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, f64, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        L.nf4o_levels.argtypes = [vp, vp]
        L.nf4o_levels.restype = None
        L.nf4o_bf16_rne.argtypes = [ctypes.c_float]
        L.nf4o_bf16_rne.restype = ctypes.c_uint16
        L.nf4o_num_blocks.argtypes = [i64]
        L.nf4o_num_blocks.restype = i64
        L.nf4o_num_groups.argtypes = [i64]
        L.nf4o_num_groups.restype = i64
        L.nf4o_absmax_mean.argtypes = [vp, i64]
        L.nf4o_absmax_mean.restype = ctypes.c_float
        L.nf4o_block_absmax.argtypes = [vp, i64, vp]
        L.nf4o_block_absmax.restype = None
        L.nf4o_quantize.argtypes = [vp, i64, vp, vp, vp, vp, vp, ctypes.c_int]
        L.nf4o_quantize.restype = None
        L.nf4o_dequantize.argtypes = [vp, vp, vp, ctypes.c_float, i64, vp, ctypes.c_int,
                                      ctypes.c_int]
        L.nf4o_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.nf4o_e4m3_decode.restype = f64
        L.nf4o_e4m3_encode.argtypes = [ctypes.c_float]
        L.nf4o_e4m3_encode.restype = ctypes.c_uint8
        L.nf4o_dequantize.restype = None
        L.nf4o_lora_u_rows.argtypes = [vp, vp, i64, i64, vp, i64, vp, ci]
        L.nf4o_lora_u_rows.restype = None
        L.nf4o_lora_fwd_rows.argtypes = [vp, vp, vp, vp, i64, i64, i64, f64, vp, i64, vp, vp,
                                         ci]
        L.nf4o_lora_fwd_rows.restype = None
        L.nf4o_lora_v_rows.argtypes = [vp, vp, i64, i64, vp, i64, vp, ci]
        L.nf4o_lora_v_rows.restype = None
        L.nf4o_lora_dx_rows.argtypes = [vp, vp, vp, vp, i64, i64, i64, f64, vp, i64, vp, vp,
                                        ci]
        L.nf4o_lora_dx_rows.restype = None
        L.nf4o_lora_dadb.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f64, vp, vp, ci]
        L.nf4o_lora_dadb.restype = None
        L.nf4o_bf16_rne_double.argtypes = [f64]
        L.nf4o_bf16_rne_double.restype = ctypes.c_uint16
        L.nf4o_merge.argtypes = [vp, vp, vp, i64, i64, i64, f64, vp]
        L.nf4o_dequantize_nodq.argtypes = [vp, vp, i64, vp, ci]
        L.nf4o_f16_to_double.argtypes = [ctypes.c_uint16]
        L.nf4o_f16_to_double.restype = f64
        L.nf4o_f16_rne_double.argtypes = [f64]
        L.nf4o_f16_rne_double.restype = ctypes.c_uint16
        L.nf4o_dequantize_nodq.restype = None
        L.nf4o_merge.restype = None
        L.nf4o_int4_error.argtypes = [vp, i64, vp]
        L.nf4o_int4_error.restype = None
        L.nf4o_num_threads.argtypes = []
        L.nf4o_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 inputs are passed as raw uint16 bits"
    return a


def num_threads() -> int:
    return int(lib().nf4o_num_threads())


def levels() -> tuple[np.ndarray, np.ndarray]:
    """(L[16], T[15]) fp32: NF4 levels and decision thresholds (readings R1, R2)."""
    L = np.zeros(16, np.float32)
    T = np.zeros(15, np.float32)
    lib().nf4o_levels(_p(L), _p(T))
    return L, T


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even, one element at a time through C."""
    x = np.ascontiguousarray(x, np.float32).ravel()
    f = lib().nf4o_bf16_rne
    return np.array([f(float(v)) for v in x], np.uint16)


def num_blocks(numel: int) -> int:
    return int(lib().nf4o_num_blocks(numel))


def num_groups(numel: int) -> int:
    return int(lib().nf4o_num_groups(numel))


def block_absmax(W: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W, np.float32).ravel()
    out = np.zeros(num_blocks(W.size), np.float32)
    lib().nf4o_block_absmax(_p(W), W.size, _p(out))
    return out


def absmax_mean(absmax: np.ndarray) -> np.float32:
    a = np.ascontiguousarray(absmax, np.float32)
    return np.float32(lib().nf4o_absmax_mean(_p(a), a.size))


def quantize(W: np.ndarray, fp8: bool = False) -> dict:
    """NF4 + double quantization of a fp32 tensor (flat order).  Returns a dict with
    codes (uint8), qscale (int8; E4M3 bytes when fp8, reading R15), steps (fp32), mean (fp32
    scalar), absmax (fp32)."""
    W = np.ascontiguousarray(W, np.float32).ravel()
    n = W.size
    nb, ng = num_blocks(n), num_groups(n)
    codes = np.zeros((n + 1) // 2, np.uint8)
    qscale = np.zeros(nb, np.int8)
    steps = np.zeros(ng, np.float32)
    mean = np.zeros(1, np.float32)
    absmax = np.zeros(nb, np.float32)
    lib().nf4o_quantize(_p(W), n, _p(codes), _p(qscale), _p(steps), _p(mean), _p(absmax),
                        1 if fp8 else 0)
    return {"codes": codes, "qscale": qscale, "steps": steps, "mean": mean[0],
            "absmax": absmax, "numel": n, "fp8": bool(fp8)}


def dequantize(q: dict, f16: bool = False) -> np.ndarray:
    """bf16 bits (uint16) of the dequantized weights, flat order (reading R7); binary16
    bits with f16 (reading R16)."""
    n = int(q["numel"])
    out = np.zeros(n, np.uint16)
    codes = np.ascontiguousarray(q["codes"], np.uint8)
    qscale = np.ascontiguousarray(q["qscale"], np.int8)
    steps = np.ascontiguousarray(q["steps"], np.float32)
    lib().nf4o_dequantize(_p(codes), _p(qscale), _p(steps), float(q["mean"]), n, _p(out),
                          1 if q.get("fp8") else 0, 1 if f16 else 0)
    return out


def e4m3_decode(codes) -> np.ndarray:
    f = lib().nf4o_e4m3_decode
    return np.array([f(int(c) & 0xFF) for c in np.ravel(codes)], np.float64)


def e4m3_encode(x) -> np.ndarray:
    f = lib().nf4o_e4m3_encode
    return np.array([f(float(v)) for v in np.ravel(np.asarray(x, np.float32))], np.uint8)


def _rows(rows, M):
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    return np.ascontiguousarray(rows, np.int64)


def lora_u(X, A, rows=None, f16=False):
    """U[i] = X[rows[i]] A^T in fp64.  X [M,K], A [r,K] bf16 bits (binary16 with f16)."""
    X, A = _u16(X), _u16(A)
    M, K = X.shape
    r = A.shape[0]
    rows = _rows(rows, M)
    U = np.zeros((rows.size, r), np.float64)
    lib().nf4o_lora_u_rows(_p(X), _p(A), K, r, _p(rows), rows.size, _p(U), int(f16))
    return U


def lora_fwd(X, Wd, A, B, scale, rows=None, f16=False):
    """(Y, U) for the selected rows, fp64 (reading R8).  Wd [N,K] bf16 bits; every 16-bit
    input binary16 instead with f16 (reading R16)."""
    X, Wd, A, B = _u16(X), _u16(Wd), _u16(A), _u16(B)
    M, K = X.shape
    N = Wd.shape[0]
    r = A.shape[0]
    rows = _rows(rows, M)
    Y = np.zeros((rows.size, N), np.float64)
    U = np.zeros((rows.size, r), np.float64)
    lib().nf4o_lora_fwd_rows(_p(X), _p(Wd), _p(A), _p(B), N, K, r, float(scale),
                             _p(rows), rows.size, _p(Y), _p(U), int(f16))
    return Y, U


def lora_v(dY, B, rows=None, f16=False):
    dY, B = _u16(dY), _u16(B)
    M, N = dY.shape
    r = B.shape[1]
    rows = _rows(rows, M)
    V = np.zeros((rows.size, r), np.float64)
    lib().nf4o_lora_v_rows(_p(dY), _p(B), N, r, _p(rows), rows.size, _p(V), int(f16))
    return V


def lora_dx(dY, Wd, A, B, scale, rows=None, f16=False):
    """(dX, V) for the selected rows, fp64 (reading R8; binary16 inputs with f16)."""
    dY, Wd, A, B = _u16(dY), _u16(Wd), _u16(A), _u16(B)
    M, N = dY.shape
    K = Wd.shape[1]
    r = A.shape[0]
    rows = _rows(rows, M)
    dX = np.zeros((rows.size, K), np.float64)
    V = np.zeros((rows.size, r), np.float64)
    lib().nf4o_lora_dx_rows(_p(dY), _p(Wd), _p(A), _p(B), N, K, r, float(scale),
                            _p(rows), rows.size, _p(dX), _p(V), int(f16))
    return dX, V


def lora_dadb(dY, X, A, B, scale, f16=False):
    """(dA [r,K], dB [N,r]) over all rows, fp64 (reading R8; binary16 inputs with f16)."""
    dY, X, A, B = _u16(dY), _u16(X), _u16(A), _u16(B)
    M, N = dY.shape
    K = X.shape[1]
    r = A.shape[0]
    dA = np.zeros((r, K), np.float64)
    dB = np.zeros((N, r), np.float64)
    lib().nf4o_lora_dadb(_p(dY), _p(X), _p(A), _p(B), M, N, K, r, float(scale),
                         _p(dA), _p(dB), int(f16))
    return dA, dB


def bf16_rne_double(x) -> np.ndarray:
    """fp64 -> bf16 bits, one rounding (ties to even), element by element through C."""
    x = np.ascontiguousarray(x, np.float64).ravel()
    f = lib().nf4o_bf16_rne_double
    return np.array([f(float(v)) for v in x], np.uint16)


def dequantize_nodq(q: dict, f16: bool = False) -> np.ndarray:
    """bf16 bits of the variant without double quantization: L[c] times the block's fp32
    absmax, one rounding (reading R14); binary16 bits with f16.  q is an oracle quantize()
    dict."""
    n = int(q["numel"])
    out = np.zeros(n, np.uint16)
    lib().nf4o_dequantize_nodq(_p(np.ascontiguousarray(q["codes"], np.uint8)),
                               _p(np.ascontiguousarray(q["absmax"], np.float32)), n, _p(out),
                               int(f16))
    return out


def f16_to_double(h) -> np.ndarray:
    """Values of binary16 bit patterns, element by element from the format's definition."""
    f = lib().nf4o_f16_to_double
    return np.array([f(int(v) & 0xFFFF) for v in np.ravel(h)], np.float64)


def f16_rne_double(x) -> np.ndarray:
    """fp64 -> binary16 bits, one rounding (ties to even), element by element (reading R16)."""
    f = lib().nf4o_f16_rne_double
    return np.array([f(float(v)) for v in np.ravel(x)], np.uint16)


def merge(Wd, A, B, scale) -> np.ndarray:
    """bf16 bits [N, K] of bf16(W' + scale B A) from the fp64 bracket (reading R11).
    Wd: the dequantized base as bf16 bits [N, K]; A [r, K] and B [N, r] bf16 bits."""
    Wd, A, B = _u16(Wd), _u16(A), _u16(B)
    r, K = A.shape
    N = B.shape[0]
    Wd = Wd.reshape(N, K)
    out = np.zeros((N, K), np.uint16)
    lib().nf4o_merge(_p(Wd), _p(A), _p(B), N, K, r, float(scale), _p(out))
    return out


def int4_error(W: np.ndarray) -> np.ndarray:
    """[sum w^2, sum NF4 squared error, sum INT4 squared error] in fp64 (reading R12)."""
    W = np.ascontiguousarray(W, np.float32).ravel()
    out = np.zeros(3, np.float64)
    lib().nf4o_int4_error(_p(W), W.size, _p(out))
    return out
