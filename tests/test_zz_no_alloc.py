"""qmm_verify_noalloc: the verify product for callers that cannot have device
memory allocated for them (code captured into a CUDA graph under the global
capture mode, or hosts that own every device allocation).  It takes its working
memory from a fixed array inside the library; its results must match
qmm_verify's within the tolerance the other GPU tests use, on consecutive calls.

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
]


@pytest.mark.parametrize("fmt,N,K,M,hadamard,splits", CASES)
def test_noalloc_matches_verify_on_consecutive_calls(fmt, N, K, M, hadamard, splits):
    w = synth.weights(N, K, 900 + N)
    a = synth.activations(M, K, 901 + K, outliers=True)
    if fmt == "q4":
        wb = O.q4_0_quantize_h32(w) if hadamard else O.q4_0_quantize(w)
        sc = None
        mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(wb).cuda(), N, K, hadamard=hadamard,
                       k_splits=splits)
        ofmt = O.FMT_Q4_0
    else:
        wb, sc = O.fp8_quantize(w)
        mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(wb).cuda(), N, K,
                       scales=torch.from_numpy(sc).cuda(), k_splits=splits)
        ofmt = O.FMT_FP8
    act = bf16_cuda(a)
    ref = mat.verify(act)
    torch.cuda.synchronize()
    ref_np = ref.cpu().double().numpy()
    _, S = O.verify_rows(ofmt, wb, sc, N, K, a, hadamard=hadamard)
    for call in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        q.qmm_verify_noalloc(mat.handle, act, out, M)
        torch.cuda.synchronize()
        assert mat.sync_status() == q.QMM_OK
        assert_within_tolerance(out.cpu().double().numpy(), ref_np, S,
                                f"noalloc call {call} {fmt} N={N} K={K} M={M}")
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
