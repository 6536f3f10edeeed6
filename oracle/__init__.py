"""CPU oracle for the speculative-decode verify matmul -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
library never does, and this package imports nothing from the product.

Everything here is a thin ctypes/numpy wrapper over ``qmm_oracle.c``: the plain
definition of the verify product (dequantize to fp64, naive triple loop) plus
the Q4_0 / FP8 quantizers that write the synthetic weight files and the fp32
Walsh-Hadamard model.  See ``qmm_oracle.c`` for the formulas and the pages each
one follows.

Pin status (what fixes each function other than itself; see tests/test_oracle_pins.py):
  decoders (bf16, fp16, e4m3)  -- exhaustive against library casts and closed forms
  encoders (fp16, e4m3)        -- exhaustive round trips, midpoint ties, library casts
  Q4_0 quantize / dequant      -- closed form, hand blocks, top-bit-flip identity, bounds
  FP8 quantize / dequant       -- closed form, library cast, tile bounds
  FWHT (fp32 and fp64)         -- H H^T = B I, unit vectors, involution, fp64 bound, the
                                  closed-form ramp, and (B = 64, 128) the bit-exact
                                  half-size recursion that fixes the stage order
  verify product               -- M independent GEMVs, brute force vs numpy and exact
                                  rationals, one-hot and all-ones special cases
  Q8_0 quantize / dequant      -- closed form, hand blocks (tests/golden/q8_0_blocks.json),
                                  exhaustive codes x scales, quantizer bounds and ties
  greedy acceptance            -- hand-worked cases (tests/golden/greedy_accept.json),
                                  numpy's first-occurrence argmax, brute-force prefix
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

__all__ = [
    "lib", "bf16_to_f64", "f16_to_f64", "e4m3_to_f64", "f32_to_f16_rne", "f32_to_e4m3_sat",
    "fwht32_f32", "fwht32_f64", "hadamard32_act_f32", "q4_0_quantize", "q4_0_quantize_h32",
    "fwht_f32", "fwht_f64", "hadamard_act_f32", "rotate_weights_f32",
    "q4_0_dequant", "fp8_quantize", "fp8_dequant", "verify_rows",
    "num_threads", "set_num_threads", "FMT_Q4_0", "FMT_FP8", "FMT_Q8_0", "greedy_accept",
    "q8_0_quantize", "q8_0_dequant",
]

FMT_Q4_0 = 0
FMT_FP8 = 1
FMT_Q8_0 = 2

_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int


def _configure(L: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures on a loaded oracle library."""
    L.oracle_bf16_to_f64.restype = ctypes.c_double
    L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_f16_to_f64.restype = ctypes.c_double
    L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_e4m3_to_f64.restype = ctypes.c_double
    L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    L.oracle_f32_to_f16_rne.restype = ctypes.c_uint16
    L.oracle_f32_to_f16_rne.argtypes = [ctypes.c_float]
    L.oracle_f32_to_e4m3_sat.restype = ctypes.c_uint8
    L.oracle_f32_to_e4m3_sat.argtypes = [ctypes.c_float]
    L.oracle_fwht_f32.argtypes = [_P, _P, _INT]
    L.oracle_fwht_f64.argtypes = [_P, _P, _INT]
    L.oracle_hadamard_act_f32.argtypes = [_P, _I64, _INT, _I64, _INT, _P]
    L.oracle_rotate_weights_f32.argtypes = [_P, _I64, _I64, _INT, _P]
    L.oracle_q8_0_quantize.argtypes = [_P, _I64, _I64, _P]
    L.oracle_q8_0_dequant.argtypes = [_P, _I64, _I64, _P]
    L.oracle_greedy_accept.restype = _INT
    L.oracle_greedy_accept.argtypes = [_P, _I64, _INT, _I64, _P, _P, _P]
    L.oracle_fwht32_f32.argtypes = [_P, _P]
    L.oracle_fwht32_f64.argtypes = [_P, _P]
    L.oracle_hadamard32_act_f32.argtypes = [_P, _I64, _INT, _I64, _P]
    L.oracle_q4_0_quantize.argtypes = [_P, _I64, _I64, _P]
    L.oracle_q4_0_quantize_h32.argtypes = [_P, _I64, _I64, _P]
    L.oracle_q4_0_dequant.argtypes = [_P, _I64, _I64, _P]
    L.oracle_fp8_quantize.argtypes = [_P, _I64, _I64, _P, _P]
    L.oracle_fp8_dequant.argtypes = [_P, _P, _I64, _I64, _P]
    L.oracle_verify_rows.restype = _INT
    L.oracle_verify_rows.argtypes = [_INT, _P, _P, _I64, _I64, _P, _I64, _INT, _INT, _P,
                                     _I64, _P, _P]
    L.oracle_num_threads.restype = _INT
    L.oracle_set_num_threads.argtypes = [_INT]
    return L


def lib() -> ctypes.CDLL:
    """Build (if needed) and load the oracle shared library."""
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# ---------------------------------------------------------------- scalars
def bf16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16).ravel()
    f = lib().oracle_bf16_to_f64
    return np.array([f(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


def f16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16).ravel()
    f = lib().oracle_f16_to_f64
    return np.array([f(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


def e4m3_to_f64(codes) -> np.ndarray:
    b = _c(codes, np.uint8).ravel()
    f = lib().oracle_e4m3_to_f64
    return np.array([f(int(x)) for x in b], dtype=np.float64).reshape(np.shape(codes))


def f32_to_f16_rne(x) -> np.ndarray:
    v = _c(x, np.float32).ravel()
    f = lib().oracle_f32_to_f16_rne
    return np.array([f(float(t)) for t in v], dtype=np.uint16).reshape(np.shape(x))


def f32_to_e4m3_sat(x) -> np.ndarray:
    v = _c(x, np.float32).ravel()
    f = lib().oracle_f32_to_e4m3_sat
    return np.array([f(float(t)) for t in v], dtype=np.uint8).reshape(np.shape(x))


# ---------------------------------------------------------------- Hadamard
def fwht32_f32(x) -> np.ndarray:
    v = _c(x, np.float32)
    assert v.shape[-1] == 32
    flat = v.reshape(-1, 32)
    out = np.empty_like(flat)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        o = np.empty(32, np.float32)
        lib().oracle_fwht32_f32(_ptr(row), _ptr(o))
        out[i] = o
    return out.reshape(v.shape)


def fwht32_f64(x) -> np.ndarray:
    v = _c(x, np.float64)
    assert v.shape[-1] == 32
    flat = v.reshape(-1, 32)
    out = np.empty_like(flat)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        o = np.empty(32, np.float64)
        lib().oracle_fwht32_f64(_ptr(row), _ptr(o))
        out[i] = o
    return out.reshape(v.shape)


def fwht_f32(x, B: int) -> np.ndarray:
    """fp32 device model of the unnormalised B-point transform (B = 32, 64, 128)
    over the last axis."""
    v = _c(x, np.float32)
    assert B in (32, 64, 128) and v.shape[-1] == B
    flat = v.reshape(-1, B)
    out = np.empty_like(flat)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        o = np.empty(B, np.float32)
        lib().oracle_fwht_f32(_ptr(row), _ptr(o), B)
        out[i] = o
    return out.reshape(v.shape)


def fwht_f64(x, B: int) -> np.ndarray:
    v = _c(x, np.float64)
    assert B in (32, 64, 128) and v.shape[-1] == B
    flat = v.reshape(-1, B)
    out = np.empty_like(flat)
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        o = np.empty(B, np.float64)
        lib().oracle_fwht_f64(_ptr(row), _ptr(o), B)
        out[i] = o
    return out.reshape(v.shape)


def hadamard_act_f32(act_bf16: np.ndarray, B: int) -> np.ndarray:
    """fp32 device model of the B-block activation rotation: [M][K] bf16 bits -> fp32."""
    a = _c(act_bf16, np.uint16)
    M, K = a.shape
    assert B in (32, 64, 128) and K % B == 0
    out = np.empty((M, K), np.float32)
    lib().oracle_hadamard_act_f32(_ptr(a), K, M, K, B, _ptr(out))
    return out


def rotate_weights_f32(w: np.ndarray, B: int) -> np.ndarray:
    """The offline weight rotation: every B-block of a row rotated (fp32) and times 1/B."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert B in (32, 64, 128) and K % B == 0
    out = np.empty((N, K), np.float32)
    lib().oracle_rotate_weights_f32(_ptr(w), N, K, B, _ptr(out))
    return out


def hadamard32_act_f32(act_bf16: np.ndarray) -> np.ndarray:
    """fp32 device model of the activation rotation: [M][K] bf16 bits -> [M][K] fp32."""
    a = _c(act_bf16, np.uint16)
    M, K = a.shape
    assert K % 32 == 0
    out = np.empty((M, K), np.float32)
    lib().oracle_hadamard32_act_f32(_ptr(a), K, M, K, _ptr(out))
    return out


# ---------------------------------------------------------------- Q4_0
def q4_0_quantize(w: np.ndarray) -> np.ndarray:
    """[N][K] fp32 -> canonical Q4_0 bytes, shape [N][K/32][18] uint8."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    out = np.empty((N, K // 32, 18), np.uint8)
    lib().oracle_q4_0_quantize(_ptr(w), N, K, _ptr(out))
    return out


def q4_0_quantize_h32(w: np.ndarray) -> np.ndarray:
    """Rotate each 32-block by H (fp32), divide by 32, quantize to Q4_0."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    out = np.empty((N, K // 32, 18), np.uint8)
    lib().oracle_q4_0_quantize_h32(_ptr(w), N, K, _ptr(out))
    return out


def q4_0_dequant(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    b = _c(blocks, np.uint8)
    assert b.size == N * (K // 32) * 18
    out = np.empty((N, K), np.float64)
    lib().oracle_q4_0_dequant(_ptr(b), N, K, _ptr(out))
    return out


# ---------------------------------------------------------------- FP8
def q8_0_quantize(w: np.ndarray) -> np.ndarray:
    """[N][K] fp32 -> canonical Q8_0 bytes, shape [N][K/32][34] uint8."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    out = np.empty((N, K // 32, 34), np.uint8)
    lib().oracle_q8_0_quantize(_ptr(w), N, K, _ptr(out))
    return out


def q8_0_dequant(blocks: np.ndarray, N: int, K: int) -> np.ndarray:
    b = _c(blocks, np.uint8)
    out = np.empty((N, K), np.float64)
    lib().oracle_q8_0_dequant(_ptr(b), N, K, _ptr(out))
    return out


def fp8_quantize(w: np.ndarray):
    """[N][K] fp32 -> (codes [N][K] uint8, scales [ceil(N/128)][ceil(K/128)] fp32)."""
    w = _c(w, np.float32)
    N, K = w.shape
    codes = np.empty((N, K), np.uint8)
    scales = np.empty(((N + 127) // 128, (K + 127) // 128), np.float32)
    lib().oracle_fp8_quantize(_ptr(w), N, K, _ptr(codes), _ptr(scales))
    return codes, scales


def fp8_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    c = _c(codes, np.uint8)
    s = _c(scales, np.float32)
    N, K = c.shape
    out = np.empty((N, K), np.float64)
    lib().oracle_fp8_dequant(_ptr(c), _ptr(s), N, K, _ptr(out))
    return out


# ---------------------------------------------------------------- product
def _hb(hadamard) -> int:
    """Rotation block size from False / True (32) / 32 / 64 / 128."""
    if hadamard is True:
        return 32
    if not hadamard:
        return 0
    assert int(hadamard) in (32, 64, 128)
    return int(hadamard)


def verify_rows(fmt: int, wbytes: np.ndarray, scales, N: int, K: int, act_bf16: np.ndarray,
                hadamard=False, rows=None):
    """Verify product for selected weight rows (all rows when ``rows`` is None).

    Returns (out [M][len(rows)], S [M][len(rows)]) in fp64.
    """
    wb = _c(wbytes, np.uint8)
    sc = _c(scales, np.float32) if scales is not None else None
    a = _c(act_bf16, np.uint16)
    M, lda = a.shape
    if rows is None:
        r = None
        nr = N
    else:
        r = _c(rows, np.int64)
        nr = r.size
    out = np.empty((M, nr), np.float64)
    S = np.empty((M, nr), np.float64)
    rc = lib().oracle_verify_rows(fmt, _ptr(wb), _ptr(sc) if sc is not None else None, N, K,
                                  _ptr(a), lda, M, _hb(hadamard),
                                  _ptr(r) if r is not None else None, nr, _ptr(out), _ptr(S))
    if rc != 0:
        raise ValueError(f"oracle_verify_rows failed with {rc}")
    return out, S


def greedy_accept(logits: np.ndarray, tokens: np.ndarray):
    """Greedy acceptance of a verified block: (argmax [M] int32, k, next token).

    ``logits`` [M][N] fp64 scores of the M block positions; ``tokens`` [M] the
    block's input tokens (tokens[0] the last committed one).  See
    ``oracle_greedy_accept`` in qmm_oracle.c.
    """
    lg = _c(logits, np.float64)
    tk = _c(tokens, np.int32)
    M, N = lg.shape
    assert tk.shape == (M,)
    am = np.empty(M, np.int32)
    res = np.empty(2, np.int32)
    rc = lib().oracle_greedy_accept(_ptr(lg), N, M, N, _ptr(tk), _ptr(am), _ptr(res))
    if rc != 0:
        raise ValueError(f"oracle_greedy_accept failed with {rc}")
    return am, int(res[0]), int(res[1])


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))
