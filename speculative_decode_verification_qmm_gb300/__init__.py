"""GB300-native verify matmul for speculative decoding.

Python binding of ``include/qmm.h``: the functions below keep the C names and
only marshal arguments (torch tensors -> device pointers, the current CUDA
stream); every step of the computation runs in ``libqmm.so``'s kernels.

    out[m][n] = sum_k act[m][k] * W[n][k],  1 <= M <= 16

with W in Q4_0 (32-element blocks, fp16 scale, 4-bit codes offset by 8) or
FP8 E4M3 with 128x128 fp32 scales, optionally with the 32-point Hadamard
rotation of the activations for weights rotated offline.
"""
from __future__ import annotations

import ctypes

from ._lib import (QMM_ERR_ALIGN, QMM_ERR_CUDA, QMM_ERR_DEVICE, QMM_ERR_INVALID_ARG,
                   QMM_ERR_M_RANGE, QMM_ERR_SHAPE, QMM_ERR_STATE, QMM_ERR_TIMEOUT,
                   QMM_FLAG_HADAMARD32, QMM_FLAG_HADAMARD64, QMM_FLAG_HADAMARD128, QMM_FLAG_TCGEN05, QMM_FLAG_SIMT, QMM_FMT_FP8_E4M3_B128, QMM_FMT_Q4_0, QMM_FMT_Q8_0,
                   QMM_OK, QmmError, load, qmm_desc, qmm_info)

__all__ = [
    "Matrix", "qmm_create", "qmm_create_rows", "shard_rows", "qmm_destroy", "qmm_verify", "qmm_verify_greedy", "qmm_verify_host",
    "qmm_verify_noalloc", "qmm_prefill", "qmm_prefill_workspace", "qmm_sync_status",
    "qmm_get_info", "qmm_dequantize", "qmm_hadamard32", "qmm_quantize_q4_0", "qmm_quantize_fp8",
    "qmm_debug_set_wait_limit", "qmm_debug_fail_allocs", "qmm_debug_set_trace", "qmm_strerror",
    "qmm_last_cuda_error",
    "QmmError", "load",
    "QMM_OK", "QMM_ERR_INVALID_ARG", "QMM_ERR_SHAPE", "QMM_ERR_M_RANGE", "QMM_ERR_ALIGN",
    "QMM_ERR_CUDA", "QMM_ERR_TIMEOUT", "QMM_ERR_STATE", "QMM_ERR_DEVICE",
    "QMM_FMT_Q4_0", "QMM_FMT_FP8_E4M3_B128", "QMM_FMT_Q8_0", "qmm_quantize_q8_0", "quantize_q8_0", "QMM_FLAG_HADAMARD32", "QMM_FLAG_SIMT",
    "QMM_FLAG_TCGEN05", "QMM_FLAG_HADAMARD64", "QMM_FLAG_HADAMARD128", "qmm_hadamard",
    "rotation_flag", "hadamard",
]


def _stream_ptr(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int:
    return int(t.data_ptr())


def _check(func: str, rc: int):
    if rc != QMM_OK:
        raise QmmError(func, rc)


# ------------------------------------------------------------------ raw C names
def qmm_strerror(code: int) -> str:
    return load().qmm_strerror(code).decode()


def qmm_last_cuda_error(h=None) -> int:
    return load().qmm_last_cuda_error(h)


def qmm_create(fmt: int, weights, N: int, K: int, scales=None, flags: int = 0,
               k_splits: int = 0, stream=None, rows=None) -> int:
    """Create a handle.  ``weights``/``scales`` are CUDA tensors (device) or CPU
    tensors / numpy arrays (host); returns the opaque handle as an int.
    ``rows = (n_begin, n_end)``: a handle over those rows of W only
    (qmm_create_rows)."""
    import numpy as np
    d = qmm_desc()
    d.struct_size = ctypes.sizeof(qmm_desc)
    d.format = fmt
    d.N = N
    d.K = K
    d.flags = flags
    d.k_splits = k_splits
    keep = []

    def addr(x):
        if x is None:
            return None, 0
        if isinstance(x, np.ndarray):
            a = np.ascontiguousarray(x)
            keep.append(a)
            return a.ctypes.data, 0
        t = x.contiguous()
        keep.append(t)
        return _ptr(t), int(t.is_cuda)

    d.weights, on_dev = addr(weights)
    sc, on_dev_s = addr(scales)
    d.scales = sc
    if scales is not None and on_dev_s != on_dev:
        raise ValueError("weights and scales must both be on the device or both on the host")
    d.weights_on_device = on_dev
    h = ctypes.c_void_p()
    if rows is None:
        _check("qmm_create", load().qmm_create(ctypes.byref(h), ctypes.byref(d), _stream_ptr(stream)))
    else:
        _check("qmm_create_rows", load().qmm_create_rows(ctypes.byref(h), ctypes.byref(d), int(rows[0]),
                                                         int(rows[1]), _stream_ptr(stream)))
    return h.value


def qmm_create_rows(fmt: int, weights, N: int, K: int, n_begin: int, n_end: int, scales=None,
                    flags: int = 0, k_splits: int = 0, stream=None) -> int:
    """A handle over rows [n_begin, n_end) of the N-row matrix described."""
    return qmm_create(fmt, weights, N, K, scales, flags, k_splits, stream, rows=(n_begin, n_end))


def shard_rows(N: int, G: int, g: int, align: int = 1):
    """Rows [n_begin, n_end) of shard g of G for an N-row matrix: the split
    points g N / G rounded down to a multiple of `align` (128 for FP8), the
    last shard ending at N."""
    if not (0 <= g < G):
        raise ValueError("shard index out of range")
    cut = lambda x: N if x == G else (N * x // G) // align * align
    return cut(g), cut(g + 1)


def qmm_destroy(h) -> None:
    _check("qmm_destroy", load().qmm_destroy(h))


def qmm_verify(h, act, out, M: int, stream=None) -> None:
    """act: CUDA bf16 [M, lda>=K]; out: CUDA fp32 [M, ldo>=N]; asynchronous."""
    _check("qmm_verify", load().qmm_verify(h, _ptr(act), act.stride(0), _ptr(out), out.stride(0),
                                           M, _stream_ptr(stream)))


def qmm_verify_greedy(h, act, out, M: int, tokens, argmax, accept, stream=None) -> None:
    """qmm_verify plus greedy acceptance: tokens CUDA int32 [M] (tokens[0] the
    last committed token); argmax CUDA int32 [M] and accept CUDA int32 [2]
    (accepted drafts, next token) are written; asynchronous."""
    _check("qmm_verify_greedy", load().qmm_verify_greedy(
        h, _ptr(act), act.stride(0), _ptr(out), out.stride(0), M, _ptr(tokens), _ptr(argmax),
        _ptr(accept), _stream_ptr(stream)))


def qmm_verify_host(h, act, out, M: int, stream=None) -> None:
    """act: CPU bf16 [M, K] (pinned is fastest); out: CPU fp32 [M, N]; synchronous."""
    _check("qmm_verify_host", load().qmm_verify_host(h, _ptr(act), act.stride(0), _ptr(out),
                                                     out.stride(0), M, _stream_ptr(stream)))


def qmm_verify_noalloc(h, act, out, M: int, stream=None) -> None:
    """As qmm_verify, with the working memory in the library's fixed array
    (no allocation; calls that overlap on the GPU race)."""
    _check("qmm_verify_noalloc", load().qmm_verify_noalloc(h, _ptr(act), act.stride(0), _ptr(out),
                                                           out.stride(0), M, _stream_ptr(stream)))


def qmm_prefill_workspace(h, M: int) -> int:
    """Bytes of device workspace qmm_prefill needs for M rows."""
    n = ctypes.c_int64(0)
    _check("qmm_prefill_workspace", load().qmm_prefill_workspace(h, M, ctypes.byref(n)))
    return n.value


def qmm_prefill(h, act, out, M: int, workspace, stream=None) -> None:
    """Prefill product on an FP8 handle: act CUDA bf16 [M, lda>=K], out CUDA
    fp32 [M, ldo>=N], workspace a CUDA tensor of at least
    qmm_prefill_workspace(h, M) bytes; asynchronous."""
    _check("qmm_prefill", load().qmm_prefill(
        h, _ptr(act), act.stride(0), _ptr(out), out.stride(0), M, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))


def qmm_sync_status(h, stream=None) -> int:
    return load().qmm_sync_status(h, _stream_ptr(stream))


def qmm_get_info(h) -> dict:
    info = qmm_info()
    info.struct_size = ctypes.sizeof(qmm_info)
    _check("qmm_get_info", load().qmm_get_info(h, ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in qmm_info._fields_ if name != "struct_size"}


def qmm_dequantize(h, w_out, stream=None) -> None:
    _check("qmm_dequantize", load().qmm_dequantize(h, _ptr(w_out), _stream_ptr(stream)))


def qmm_hadamard32(act, act_out, M: int, K: int, stream=None) -> None:
    _check("qmm_hadamard32", load().qmm_hadamard32(_ptr(act), act.stride(0), _ptr(act_out), M, K,
                                                   _stream_ptr(stream)))


def qmm_hadamard(act, act_out, M: int, K: int, block: int, stream=None) -> None:
    _check("qmm_hadamard", load().qmm_hadamard(_ptr(act), act.stride(0), _ptr(act_out), M, K,
                                               block, _stream_ptr(stream)))


def rotation_flag(hadamard) -> int:
    """QMM_FLAG_HADAMARD* for hadamard = False, True (32), 32, 64 or 128."""
    if hadamard is True:
        return QMM_FLAG_HADAMARD32
    if not hadamard:
        return 0
    flags = {32: QMM_FLAG_HADAMARD32, 64: QMM_FLAG_HADAMARD64, 128: QMM_FLAG_HADAMARD128}
    if int(hadamard) not in flags:
        raise ValueError(f"rotation block must be 32, 64 or 128, not {hadamard!r}")
    return flags[int(hadamard)]


def qmm_quantize_q4_0(w, blocks, flags: int = 0, stream=None) -> None:
    N, K = w.shape
    _check("qmm_quantize_q4_0", load().qmm_quantize_q4_0(_ptr(w), N, K, flags, _ptr(blocks),
                                                         _stream_ptr(stream)))


def qmm_quantize_q8_0(w, blocks, flags: int = 0, stream=None) -> None:
    N, K = w.shape
    _check("qmm_quantize_q8_0", load().qmm_quantize_q8_0(_ptr(w), N, K, flags, _ptr(blocks),
                                                         _stream_ptr(stream)))


def qmm_quantize_fp8(w, codes, scales, flags: int = 0, stream=None) -> None:
    N, K = w.shape
    _check("qmm_quantize_fp8", load().qmm_quantize_fp8(_ptr(w), N, K, flags, _ptr(codes),
                                                       _ptr(scales), _stream_ptr(stream)))


def qmm_debug_set_wait_limit(h, ns: int) -> None:
    _check("qmm_debug_set_wait_limit", load().qmm_debug_set_wait_limit(h, ns))


def qmm_debug_fail_allocs(n: int) -> None:
    _check("qmm_debug_fail_allocs", load().qmm_debug_fail_allocs(n))


def qmm_debug_set_trace(h, buf=None) -> None:
    """``buf``: a CUDA int64/uint64 tensor of stamp slots, or None to switch off
    (libraries built with QMM_TRACE only; see speculative_decode_verification_qmm_gb300.timeline)."""
    ptr, n = (None, 0) if buf is None else (_ptr(buf), buf.numel())
    _check("qmm_debug_set_trace", load().qmm_debug_set_trace(h, ptr, n))


# ------------------------------------------------------------------ convenience
def quantize_q4_0(w, hadamard=False, stream=None):
    """CUDA fp32 [N, K] -> CUDA uint8 [N, K/32, 18] Q4_0 blocks (device quantizer);
    hadamard = False, True (32), 32, 64 or 128 rotates the weights first."""
    import torch
    N, K = w.shape
    blocks = torch.empty((N, K // 32, 18), dtype=torch.uint8, device=w.device)
    qmm_quantize_q4_0(w.contiguous(), blocks, rotation_flag(hadamard), stream)
    return blocks


def quantize_q8_0(w, hadamard=False, stream=None):
    """CUDA fp32 [N, K] -> CUDA uint8 [N, K/32, 34] Q8_0 blocks (device quantizer)."""
    import torch
    N, K = w.shape
    blocks = torch.empty((N, K // 32, 34), dtype=torch.uint8, device=w.device)
    qmm_quantize_q8_0(w.contiguous(), blocks, rotation_flag(hadamard), stream)
    return blocks


def quantize_fp8(w, hadamard=False, stream=None):
    """CUDA fp32 [N, K] -> (uint8 codes [N, K], fp32 scales [N/128, K/128])."""
    import torch
    N, K = w.shape
    codes = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    scales = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    qmm_quantize_fp8(w.contiguous(), codes, scales, rotation_flag(hadamard), stream)
    return codes, scales


def hadamard(act, block: int = 32, stream=None):
    """CUDA bf16 [M, K] -> CUDA fp32 [M, K], every block-sized block rotated."""
    import torch
    M, K = act.shape
    out = torch.empty((M, K), dtype=torch.float32, device=act.device)
    qmm_hadamard(act, out, M, K, block, stream)
    return out


def hadamard32(act, stream=None):
    """CUDA bf16 [M, K] -> CUDA fp32 [M, K], every 32-block rotated."""
    import torch
    M, K = act.shape
    out = torch.empty((M, K), dtype=torch.float32, device=act.device)
    qmm_hadamard32(act, out, M, K, stream)
    return out


class Matrix:
    """One weight matrix on the device, ready for repeated verify calls."""

    def __init__(self, fmt: int, weights, N: int, K: int, scales=None, hadamard=False,
                 simt: bool = False, k_splits: int = 0, stream=None, tcgen05: bool = False,
                 rows=None):
        """``rows = (n_begin, n_end)``: the handle holds only those rows of the
        N-row matrix the arguments describe (a shard of the multi-GPU split);
        its product has n_end - n_begin columns."""
        flags = (rotation_flag(hadamard) | (QMM_FLAG_SIMT if simt else 0)
                 | (QMM_FLAG_TCGEN05 if tcgen05 else 0))
        self.N = N if rows is None else rows[1] - rows[0]
        self.K, self.fmt, self.rows = K, fmt, rows
        self.handle = qmm_create(fmt, weights, N, K, scales, flags, k_splits, stream, rows=rows)

    def verify(self, act, out=None, stream=None):
        import torch
        M = act.shape[0]
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.float32, device=act.device)
        qmm_verify(self.handle, act, out, M, stream)
        return out

    def verify_host(self, act, out=None, stream=None):
        import torch
        M = act.shape[0]
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.float32)
        qmm_verify_host(self.handle, act, out, M, stream)
        return out

    def dequantize(self, stream=None):
        import torch
        w = torch.empty((self.N, self.K), dtype=torch.float32, device="cuda")
        qmm_dequantize(self.handle, w, stream)
        return w

    def verify_greedy(self, act, tokens, out=None, stream=None):
        """(out, argmax, accept) for the drafted block; see qmm_verify_greedy."""
        import torch
        M = act.shape[0]
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.float32, device=act.device)
        argmax = torch.empty(M, dtype=torch.int32, device=act.device)
        accept = torch.empty(2, dtype=torch.int32, device=act.device)
        qmm_verify_greedy(self.handle, act, out, M, tokens, argmax, accept, stream)
        return out, argmax, accept

    def prefill(self, act, out=None, stream=None):
        """out[M, N] = act[M, K] W^T for any M (FP8 handles); the workspace is
        kept on the Matrix and grown when a call needs more."""
        import torch
        M = act.shape[0]
        if out is None:
            out = torch.empty((M, self.N), dtype=torch.float32, device=act.device)
        need = qmm_prefill_workspace(self.handle, M)
        ws = getattr(self, "_prefill_ws", None)
        if ws is None or ws.numel() < need:
            ws = torch.empty(need, dtype=torch.uint8, device=act.device)
            self._prefill_ws = ws
        qmm_prefill(self.handle, act, out, M, ws, stream)
        return out

    def info(self) -> dict:
        return qmm_get_info(self.handle)

    def sync_status(self, stream=None) -> int:
        return qmm_sync_status(self.handle, stream)

    def close(self):
        if self.handle:
            qmm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
