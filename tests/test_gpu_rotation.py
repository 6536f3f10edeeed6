"""GPU parity of the 64- and 128-point Walsh-Hadamard variants.

Bit-exact: the activation rotation (qmm_hadamard) and the device quantizers
with the offline weight rotation.  Within 1e-3 * sum|a_k w_k| + 1e-6: the
verify product with rotated activations and weights, which the oracle also
checks against the un-rotated product.
"""
import numpy as np
import pytest

import oracle as O
import speculative_decode_verification_qmm_gb300 as q
from speculative_decode_verification_qmm_gb300 import synth
from gpu_util import assert_within_tolerance, bf16_cuda, f32_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    q.load(build_if_missing=True)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("B", [32, 64, 128])
@pytest.mark.parametrize("M,K,lda", [(5, 512, 512), (16, 5120, 5120), (3, 384, 392), (1, 128, 136)])
def test_hadamard_bit_exact(B, M, K, lda):
    a = synth.activations(M, K, 700 + K + B, outliers=True)
    got = q.hadamard(bf16_cuda(a, pad_to=lda), block=B).cpu().numpy()
    ref = O.hadamard_act_f32(a, B)
    assert (f32_bits(got) == f32_bits(ref)).all()


@pytest.mark.parametrize("B", [64, 128])
def test_quantize_q4_rotated_bit_exact(B):
    N, K = 96, 1024
    w = synth.weights(N, K, 710 + B)
    w[0, :B] = 0.0
    w[1, B:2 * B] = 0.5
    w[2, :B] *= 1e-6
    got = q.quantize_q4_0(torch.from_numpy(w).cuda(), hadamard=B).cpu().numpy()
    ref = O.q4_0_quantize(O.rotate_weights_f32(w, B))
    assert (got == ref).all(), f"{int((got != ref).any(axis=2).sum())} blocks differ"


@pytest.mark.parametrize("B", [64, 128])
def test_quantize_fp8_rotated_bit_exact(B):
    N, K = 256, 384
    w = synth.weights(N, K, 720 + B)
    w[:128, 128:256] = 0.0
    codes, scales = q.quantize_fp8(torch.from_numpy(w).cuda(), hadamard=B)
    rc, rs = O.fp8_quantize(O.rotate_weights_f32(w, B))
    assert (f32_bits(scales.cpu().numpy()) == f32_bits(rs)).all()
    assert (codes.cpu().numpy() == rc).all()


@pytest.mark.parametrize("B", [64, 128])
@pytest.mark.parametrize("N,K,splits", [(424, 1408, 0), (424, 1408, 3), (1000, 2560, 0), (130, 512, 2)])
@pytest.mark.parametrize("M", [1, 16])
def test_verify_q4_rotated(B, N, K, splits, M):
    w = synth.weights(N, K, 730 + N + B)
    blocks = O.q4_0_quantize(O.rotate_weights_f32(w, B))
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, hadamard=B, k_splits=splits)
    a = synth.activations(M, K, 731 + K, outliers=True)
    out = mat.verify(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    ref, S = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a, hadamard=B)
    assert_within_tolerance(out.cpu().double().numpy(), ref, S, f"q4 H{B} N={N} K={K} S={splits} M={M}")
    mat.close()


@pytest.mark.parametrize("B", [64, 128])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_verify_fp8_rotated(B, M):
    N, K = 384, 896
    w = synth.weights(N, K, 740 + B)
    codes, scales = O.fp8_quantize(O.rotate_weights_f32(w, B))
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(codes).cuda(), N, K,
                   scales=torch.from_numpy(scales).cuda(), hadamard=B)
    a = synth.activations(M, K, 741 + M, outliers=True)
    out = mat.verify(bf16_cuda(a))
    torch.cuda.synchronize()
    ref, S = O.verify_rows(O.FMT_FP8, codes, scales, N, K, a, hadamard=B)
    assert_within_tolerance(out.cpu().double().numpy(), ref, S, f"fp8 H{B} M={M}")
    mat.close()


@pytest.mark.parametrize("B", [64, 128])
def test_rotated_rows_bit_identical_for_every_M(B):
    N, K = 640, 2048
    w = synth.weights(N, K, 750 + B)
    blocks = O.q4_0_quantize(O.rotate_weights_f32(w, B))
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, hadamard=B, k_splits=4)
    act = bf16_cuda(synth.activations(16, K, 751, outliers=True))
    full = mat.verify(act).cpu().numpy()
    for M in range(1, 16):
        part = mat.verify(act[:M].contiguous()).cpu().numpy()
        assert (f32_bits(part) == f32_bits(full[:M])).all(), f"row results changed at M={M}"
    mat.close()
