"""qmm_verify_noalloc: the verify product for callers that cannot have device
memory allocated for them (code captured into a CUDA graph under the global
capture mode, or hosts that own every device allocation).  It takes its working
memory from a fixed array inside the library; its results must match the
oracle (and qmm_verify) within the tolerance the other GPU tests use, on
consecutive calls and across handles of different shapes.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test.  Passes alone in a fresh process and
after the other tests (the array keeps earlier calls' contents)."""
import numpy as np
import pytest

import oracle as O
import speculative_decode_verification_qmm_gb300 as q
from speculative_decode_verification_qmm_gb300 import synth
from gpu_util import assert_within_tolerance, bf16_cuda

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _ready():
    q.load(build_if_missing=True)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


CASES = [  # (fmt, N, K, M, hadamard, k_splits)
    ("q4", 5120, 5120, 16, False, 0),
    ("q4", 424, 1376, 7, True, 3),
    ("q4", 256, 512, 1, False, 0),
    ("fp8", 384, 896, 12, False, 3),
    ("q8", 300, 1024, 5, False, 2),
]


def make(fmt, N, K, hadamard, splits, seed):
    """A handle and the oracle's view of its weights (format, bytes, scales)."""
    w = synth.weights(N, K, seed)
    if fmt == "q4":
        wb = O.q4_0_quantize_h32(w) if hadamard is True else (
            O.q4_0_quantize(O.rotate_weights_f32(w, hadamard)) if hadamard else O.q4_0_quantize(w))
        mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(wb).cuda(), N, K, hadamard=hadamard,
                       k_splits=splits)
        return mat, O.FMT_Q4_0, wb, None
    if fmt == "q8":
        wb = O.q8_0_quantize(w)
        mat = q.Matrix(q.QMM_FMT_Q8_0, torch.from_numpy(wb).cuda(), N, K, k_splits=splits)
        return mat, O.FMT_Q8_0, wb, None
    wb, sc = O.fp8_quantize(w)
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(wb).cuda(), N, K,
                   scales=torch.from_numpy(sc).cuda(), k_splits=splits)
    return mat, O.FMT_FP8, wb, sc


def noalloc_call(mat, act, M, N):
    out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    q.qmm_verify_noalloc(mat.handle, act, out, M)
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    return out.cpu().double().numpy()


@pytest.mark.parametrize("fmt,N,K,M,hadamard,splits", CASES)
def test_noalloc_matches_oracle_on_consecutive_calls(fmt, N, K, M, hadamard, splits):
    """Two calls in a row through the no-allocation entry point, each checked
    element by element against the oracle (and, as a second check, against
    the ordinary entry point at the same tolerance)."""
    mat, ofmt, wb, sc = make(fmt, N, K, hadamard, splits, 900 + N)
    a = synth.activations(M, K, 901 + K, outliers=True)
    ref, S = O.verify_rows(ofmt, wb, sc, N, K, a, hadamard=hadamard)
    act = bf16_cuda(a)
    plain = mat.verify(act).cpu().double().numpy()
    for call in range(2):
        got = noalloc_call(mat, act, M, N)
        assert_within_tolerance(got, ref, S, f"noalloc call {call} {fmt} N={N} K={K} M={M}")
        assert_within_tolerance(got, plain, S, f"noalloc vs qmm_verify, call {call}")
    mat.close()


def test_noalloc_handles_of_different_shapes_in_turn():
    """Handles of other formats and shapes one after another on the same
    stream: a 128-point rotation with a large K and several splits, an FP8
    handle with a small K and splits, a plain Q4_0 handle with splits, then the
    first again.  Whatever an earlier call left in the shared array must not
    leak into a later one; every result is checked against the oracle."""
    specs = [("q4", 640, 17408, 16, 128, 7), ("fp8", 256, 384, 3, False, 3),
             ("q4", 300, 2048, 9, False, 4), ("q4", 640, 17408, 16, 128, 7)]
    made = {}
    for i, (fmt, N, K, M, had, splits) in enumerate(specs):
        key = (fmt, N, K, had, splits)
        if key not in made:
            made[key] = make(fmt, N, K, had, splits, 960 + i)
        mat, ofmt, wb, sc = made[key]
        a = synth.activations(M, K, 970 + i, outliers=True)
        ref, S = O.verify_rows(ofmt, wb, sc, N, K, a, hadamard=had)
        got = noalloc_call(mat, bf16_cuda(a), M, N)
        assert_within_tolerance(got, ref, S, f"noalloc sequence step {i} ({fmt} N={N} K={K})")
    for mat, _, _, _ in made.values():
        mat.close()


def test_noalloc_rejects_plans_beyond_the_array():
    # the rotated activations of K = 131328 columns need more than the 4 MiB array
    N, K = 128, 131328
    blocks = q.quantize_q4_0(synth.weights_cuda(N, K, 950), hadamard=True)
    mat = q.Matrix(q.QMM_FMT_Q4_0, blocks, N, K, hadamard=True)
    act = bf16_cuda(synth.activations(4, K, 951))
    out = torch.empty((4, N), dtype=torch.float32, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.qmm_verify_noalloc(mat.handle, act, out, 4)
    assert ei.value.code == q.QMM_ERR_SHAPE
    mat.close()
