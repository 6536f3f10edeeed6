"""ctypes loader for ``libqmm.so`` with the C signatures of ``include/qmm.h``.

The library is built in-tree by ``build.py``.  Loading fails loudly when it is
missing: there is no CPU or PyTorch fallback for any entry point.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

QMM_OK = 0
QMM_ERR_INVALID_ARG = 1
QMM_ERR_SHAPE = 2
QMM_ERR_M_RANGE = 3
QMM_ERR_ALIGN = 4
QMM_ERR_CUDA = 5
QMM_ERR_TIMEOUT = 6
QMM_ERR_STATE = 7
QMM_ERR_DEVICE = 8

QMM_FMT_Q4_0 = 0
QMM_FMT_FP8_E4M3_B128 = 1
QMM_FMT_Q8_0 = 2
QMM_FLAG_HADAMARD32 = 1
QMM_FLAG_SIMT = 2
QMM_FLAG_TCGEN05 = 4
QMM_FLAG_HADAMARD64 = 8
QMM_FLAG_HADAMARD128 = 16


class qmm_desc(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("format", ctypes.c_uint32),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("flags", ctypes.c_uint32),
        ("weights_on_device", ctypes.c_int32),
        ("weights", ctypes.c_void_p),
        ("scales", ctypes.c_void_p),
        ("k_splits", ctypes.c_int32),
    ]


class qmm_info(ctypes.Structure):
    _fields_ = [
        ("struct_size", ctypes.c_uint32),
        ("format", ctypes.c_uint32),
        ("flags", ctypes.c_uint32),
        ("N", ctypes.c_int64),
        ("K", ctypes.c_int64),
        ("weight_bytes", ctypes.c_int64),
        ("device_weight_bytes", ctypes.c_int64),
        ("scratch_bytes", ctypes.c_int64),
        ("n_tiles", ctypes.c_int32),
        ("k_splits", ctypes.c_int32),
        ("ctas", ctypes.c_int32),
        ("stages_per_cta", ctypes.c_int32),
        ("stage_bytes", ctypes.c_int32),
        ("pipeline_depth", ctypes.c_int32),
        ("device", ctypes.c_int32),
        ("sm_count", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_U32 = ctypes.c_uint32

# name -> (restype, argtypes); every function declared in include/qmm.h
SIGNATURES = {
    "qmm_create": (_INT, [ctypes.POINTER(_P), ctypes.POINTER(qmm_desc), _P]),
    "qmm_create_rows": (_INT, [ctypes.POINTER(_P), ctypes.POINTER(qmm_desc), _I64, _I64, _P]),
    "qmm_destroy": (_INT, [_P]),
    "qmm_verify": (_INT, [_P, _P, _I64, _P, _I64, _INT, _P]),
    "qmm_verify_greedy": (_INT, [_P, _P, _I64, _P, _I64, _INT, _P, _P, _P, _P]),
    "qmm_verify_host": (_INT, [_P, _P, _I64, _P, _I64, _INT, _P]),
    "qmm_verify_noalloc": (_INT, [_P, _P, _I64, _P, _I64, _INT, _P]),
    "qmm_prefill": (_INT, [_P, _P, _I64, _P, _I64, _I64, _P, _I64, _P]),
    "qmm_prefill_workspace": (_INT, [_P, _I64, ctypes.POINTER(_I64)]),
    "qmm_sync_status": (_INT, [_P, _P]),
    "qmm_last_cuda_error": (_INT, [_P]),
    "qmm_get_info": (_INT, [_P, ctypes.POINTER(qmm_info)]),
    "qmm_strerror": (ctypes.c_char_p, [_INT]),
    "qmm_dequantize": (_INT, [_P, _P, _P]),
    "qmm_hadamard32": (_INT, [_P, _I64, _P, _INT, _I64, _P]),
    "qmm_hadamard": (_INT, [_P, _I64, _P, _INT, _I64, _INT, _P]),
    "qmm_quantize_q4_0": (_INT, [_P, _I64, _I64, _U32, _P, _P]),
    "qmm_quantize_q8_0": (_INT, [_P, _I64, _I64, _U32, _P, _P]),
    "qmm_quantize_fp8": (_INT, [_P, _I64, _I64, _U32, _P, _P, _P]),
    "qmm_debug_set_wait_limit": (_INT, [_P, _I64]),
    "qmm_debug_fail_allocs": (_INT, [_INT]),
    "qmm_debug_set_trace": (_INT, [_P, _P, _I64]),
}

QMM_TRACE_FIELDS = 16
(QMM_TR_ENTRY, QMM_TR_SMID, QMM_TR_PDL, QMM_TR_DATA, QMM_TR_LOOP, QMM_TR_EPI, QMM_TR_RED,
 QMM_TR_PART, QMM_TR_ARRIVE, QMM_TR_LAST, QMM_TR_EXIT) = range(11)

_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False, path: str | None = None) -> ctypes.CDLL:
    """Load libqmm.so (optionally building it first) and declare its signatures.

    ``path``: load that build of the library instead (a profiling variant);
    a process loads one library only."""
    global _lib
    if _lib is not None:
        if path is not None and os.path.abspath(path) != os.path.abspath(_lib._name):
            raise RuntimeError(f"libqmm already loaded from {_lib._name}")
        return _lib
    if path is None:
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(
            f"libqmm.so is not built ({path} missing); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


class QmmError(RuntimeError):
    def __init__(self, func: str, code: int):
        L = load()
        name = L.qmm_strerror(code).decode()
        super().__init__(f"{func} failed: {name} ({code})")
        self.code = code
