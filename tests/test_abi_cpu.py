"""C-ABI checks that need no GPU: the library builds, loads and exports every
function include/qmm.h declares; host-side argument validation answers before
any device work."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import speculative_decode_verification_qmm_gb300 as q
from speculative_decode_verification_qmm_gb300 import _lib, build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(qmm_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("qmm_create", "qmm_verify", "qmm_destroy", "qmm_dequantize", "qmm_hadamard32",
                     "qmm_sync_status", "qmm_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported_and_bound(L):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), f"{n} not exported by libqmm.so"
        assert n in _lib.SIGNATURES, f"{n} has no Python binding"
    assert set(_lib.SIGNATURES) == set(names)


def test_struct_layouts_match_header(L, tmp_path):
    """ctypes mirrors of qmm_desc / qmm_info have the C compiler's size and offsets."""
    fields = {"qmm_desc": [f for f, _ in _lib.qmm_desc._fields_],
              "qmm_info": [f for f, _ in _lib.qmm_info._fields_]}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "qmm.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'printf("%zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'printf("%zu\\n", offsetof({st}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    expect = []
    for st in (_lib.qmm_desc, _lib.qmm_info):
        expect.append(ctypes.sizeof(st))
        expect += [getattr(st, f).offset for f, _ in st._fields_]
    assert vals == expect


def test_strerror_names_every_code(L):
    for code, name in [(0, "QMM_OK"), (1, "QMM_ERR_INVALID_ARG"), (2, "QMM_ERR_SHAPE"),
                       (3, "QMM_ERR_M_RANGE"), (4, "QMM_ERR_ALIGN"), (5, "QMM_ERR_CUDA"),
                       (6, "QMM_ERR_TIMEOUT"), (7, "QMM_ERR_STATE"), (8, "QMM_ERR_DEVICE")]:
        assert q.qmm_strerror(code) == name
    assert q.qmm_strerror(99) == "QMM_ERR_UNKNOWN"


def test_host_validation_without_device(L):
    # all of these are decided before any CUDA call
    assert L.qmm_verify(None, None, 0, None, 0, 1, None) == q.QMM_ERR_STATE
    assert L.qmm_verify_host(None, None, 0, None, 0, 1, None) == q.QMM_ERR_STATE
    assert L.qmm_destroy(None) == q.QMM_OK
    assert L.qmm_sync_status(None, None) == q.QMM_ERR_STATE
    assert L.qmm_get_info(None, None) == q.QMM_ERR_STATE
    assert L.qmm_dequantize(None, None, None) == q.QMM_ERR_STATE
    assert L.qmm_debug_set_wait_limit(None, 5) == q.QMM_ERR_STATE
    # the prefill entry points answer on the handle first
    n = ctypes.c_int64(7)
    assert L.qmm_prefill(None, None, 0, None, 0, 64, None, 0, None) == q.QMM_ERR_STATE
    assert L.qmm_prefill_workspace(None, 64, ctypes.byref(n)) == q.QMM_ERR_STATE and n.value == 0
    assert L.qmm_prefill_workspace(None, 64, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_debug_fail_allocs(-1) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_debug_fail_allocs(0) == q.QMM_OK
    # a stale pointer that was never a live handle
    fake = ctypes.create_string_buffer(256)
    assert L.qmm_verify(ctypes.addressof(fake), None, 0, None, 0, 1, None) == q.QMM_ERR_STATE
    # qmm_create rejects bad descriptions before touching the device
    h = ctypes.c_void_p()
    assert L.qmm_create(None, None, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_create(ctypes.byref(h), None, None) == q.QMM_ERR_INVALID_ARG
    d = _lib.qmm_desc()
    d.struct_size = ctypes.sizeof(d) - 8
    w = np.zeros(18 * 8, np.uint8)
    d.weights = w.ctypes.data
    d.N, d.K = 8, 32
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.struct_size = ctypes.sizeof(d)
    d.format = 7
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.format = q.QMM_FMT_Q4_0
    d.flags = 1 << 9
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.flags = 0
    d.K = 48
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_SHAPE
    d.K = 32
    d.N = 0
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_SHAPE
    d.N = 8
    d.format = q.QMM_FMT_FP8_E4M3_B128
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG  # no scales
    s = np.zeros(1, np.float32)
    d.scales = s.ctypes.data
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_SHAPE  # N % 128
    d.flags = q.QMM_FLAG_SIMT
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.flags = q.QMM_FLAG_TCGEN05  # tcgen05 serves bf16 Q4_0 only
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.format = q.QMM_FMT_Q4_0
    d.flags = q.QMM_FLAG_TCGEN05 | q.QMM_FLAG_HADAMARD32
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.flags = q.QMM_FLAG_TCGEN05 | q.QMM_FLAG_SIMT
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    # at most one rotation; the rotation block divides K; none with tcgen05
    d.flags = q.QMM_FLAG_HADAMARD32 | q.QMM_FLAG_HADAMARD64
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.flags = q.QMM_FLAG_TCGEN05 | q.QMM_FLAG_HADAMARD128
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.flags = q.QMM_FLAG_HADAMARD64
    d.K = 96
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_SHAPE
    d.flags = q.QMM_FLAG_HADAMARD128
    d.K = 192
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_SHAPE
    d.K = 32
    d.flags = 0
    assert h.value is None
    # tool entry points validate shapes first
    assert L.qmm_quantize_q4_0(None, 4, 32, 0, None, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize_q4_0(w.ctypes.data, 4, 40, 0, w.ctypes.data, None) == q.QMM_ERR_SHAPE
    assert L.qmm_quantize_fp8(w.ctypes.data, 100, 128, 0, w.ctypes.data, s.ctypes.data, None) == q.QMM_ERR_SHAPE
    assert L.qmm_hadamard32(w.ctypes.data, 64, w.ctypes.data, 0, 64, None) == q.QMM_ERR_M_RANGE
    assert L.qmm_hadamard32(w.ctypes.data, 64, w.ctypes.data, 1, 40, None) == q.QMM_ERR_SHAPE
    assert L.qmm_hadamard(w.ctypes.data, 64, w.ctypes.data, 1, 64, 48, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_hadamard(w.ctypes.data, 96, w.ctypes.data, 1, 96, 64, None) == q.QMM_ERR_SHAPE
    assert L.qmm_hadamard(w.ctypes.data, 64, w.ctypes.data, 0, 64, 64, None) == q.QMM_ERR_M_RANGE
    H32_64 = q.QMM_FLAG_HADAMARD32 | q.QMM_FLAG_HADAMARD64
    assert L.qmm_quantize_q4_0(w.ctypes.data, 4, 64, H32_64, w.ctypes.data, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize_q4_0(w.ctypes.data, 4, 64, q.QMM_FLAG_HADAMARD128, w.ctypes.data, None) == q.QMM_ERR_SHAPE
    assert L.qmm_quantize_fp8(w.ctypes.data, 128, 128, q.QMM_FLAG_SIMT, w.ctypes.data, s.ctypes.data, None) == q.QMM_ERR_INVALID_ARG


# ---------------------------------------------------------------- input generators
def test_bf16_rounding_matches_torch():
    import torch
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(100000) * 10.0 ** rng.uniform(-5, 5, 100000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (synth.f32_to_bf16_bits(x) == ref).all()


def test_activation_recipe():
    a = synth.activations(16, 5120, 1001, outliers=True, outlier_seed=2001)
    f = synth.bf16_bits_to_f32(a)
    ch = synth.outlier_channels(5120, 2001)
    assert ch.size == 6  # ceil(0.001 * 5120)
    # the outlier columns are 20x larger on average
    big = np.abs(f[:, ch]).mean()
    small = np.abs(np.delete(f, ch, axis=1)).mean()
    assert 10 < big / small < 40
    # deterministic
    assert (synth.activations(16, 5120, 1001, outliers=True, outlier_seed=2001) == a).all()
    w = synth.weights(64, 256, 5)
    assert w.dtype == np.float32 and abs(w.std() - 0.02) < 0.002


def test_q8_0_host_validation(L):
    """Q8_0 descriptions are validated before any CUDA call: K % 32, no
    CUDA-core or tcgen05 kernel, and the quantizer's shape and flag checks."""
    h = ctypes.c_void_p()
    d = _lib.qmm_desc()
    d.struct_size = ctypes.sizeof(d)
    w = np.zeros(34 * 8, np.uint8)
    d.weights = w.ctypes.data
    d.format = q.QMM_FMT_Q8_0
    d.N, d.K = 8, 48
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_SHAPE
    d.K = 32
    d.flags = q.QMM_FLAG_SIMT
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.flags = q.QMM_FLAG_TCGEN05
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_INVALID_ARG
    d.flags = q.QMM_FLAG_HADAMARD64
    assert L.qmm_create(ctypes.byref(h), ctypes.byref(d), None) == q.QMM_ERR_SHAPE  # K % 64
    assert h.value is None
    assert L.qmm_quantize_q8_0(None, 4, 32, 0, None, None) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_quantize_q8_0(w.ctypes.data, 4, 40, 0, w.ctypes.data, None) == q.QMM_ERR_SHAPE
    assert L.qmm_quantize_q8_0(w.ctypes.data, 4, 64, q.QMM_FLAG_SIMT, w.ctypes.data, None) == q.QMM_ERR_INVALID_ARG
