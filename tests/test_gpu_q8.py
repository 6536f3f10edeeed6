"""GPU parity of the Q8_0 path (fp16 scale per 32 elements, int8 codes).

Bit-exact: the dequantization hook and the device quantizer (plain and
rotated).  Within 1e-3 * sum|a_k w_k| + 1e-6: the verify product, at sizes
spanning several tiles with ragged tails, split K, rotated activations, and
the greedy acceptance step; rows bit-identical for every M.
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


def q8_matrix(N, K, seed, hadamard=False, **kw):
    w = synth.weights(N, K, seed)
    if hadamard:
        w = O.rotate_weights_f32(w, 32 if hadamard is True else hadamard)
    blocks = O.q8_0_quantize(w)
    mat = q.Matrix(q.QMM_FMT_Q8_0, torch.from_numpy(blocks).cuda(), N, K, hadamard=hadamard, **kw)
    return mat, blocks


@pytest.mark.parametrize("N,K,splits", [(256, 512, 0), (200, 352, 0), (424, 1376, 3), (16, 32, 1),
                                        (130, 2048, 5)])
def test_dequant_q8_bit_exact(N, K, splits):
    mat, blocks = q8_matrix(N, K, 800 + N, k_splits=splits)
    got = mat.dequantize().cpu().numpy()
    ref = O.q8_0_dequant(blocks, N, K).astype(np.float32)
    assert (f32_bits(got) == f32_bits(ref)).all()
    mat.close()


@pytest.mark.parametrize("hadamard", [False, 32, 64, 128])
def test_quantize_q8_bit_exact(hadamard):
    N, K = 96, 1024
    w = synth.weights(N, K, 810)
    w[0, :32] = 0.0
    w[1, 32:64] = 0.5
    w[2, 64:96] *= 1e-6
    w[3, 96:128] = np.float32(1e6)  # the fp16 scale overflows to infinity
    # scale exactly 1 (largest magnitude 127), every other element a half: ties
    w[4, 128:160] = np.arange(32, dtype=np.float32) - np.float32(15.5)
    w[4, 128] = 127.0
    got = q.quantize_q8_0(torch.from_numpy(w).cuda(), hadamard=hadamard).cpu().numpy()
    ref = O.q8_0_quantize(O.rotate_weights_f32(w, hadamard) if hadamard else w)
    assert (got == ref).all(), f"{int((got != ref).any(axis=2).sum())} blocks differ"


@pytest.mark.parametrize("N,K,splits,hadamard", [
    (424, 1376, 0, False), (424, 1376, 3, False), (1000, 2560, 0, False), (8, 32, 0, False),
    (129, 4096, 16, False), (424, 1408, 0, 32), (1000, 2560, 2, 128), (256, 512, 2, 64),
])
@pytest.mark.parametrize("M", [1, 9, 16])
def test_verify_q8(N, K, splits, hadamard, M):
    mat, blocks = q8_matrix(N, K, 820 + N + K, hadamard=hadamard, k_splits=splits)
    a = synth.activations(M, K, 821 + K, outliers=True)
    out = mat.verify(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    ref, S = O.verify_rows(O.FMT_Q8_0, blocks, None, N, K, a, hadamard=hadamard)
    assert_within_tolerance(out.cpu().double().numpy(), ref, S,
                            f"q8 N={N} K={K} S={splits} H={hadamard} M={M}")
    mat.close()


def test_q8_rows_bit_identical_for_every_M():
    N, K = 640, 2048
    mat, _ = q8_matrix(N, K, 830, k_splits=4)
    act = bf16_cuda(synth.activations(16, K, 831, outliers=True))
    full = mat.verify(act).cpu().numpy()
    for M in range(1, 16):
        part = mat.verify(act[:M].contiguous()).cpu().numpy()
        assert (f32_bits(part) == f32_bits(full[:M])).all(), f"row results changed at M={M}"
    again = mat.verify(act).cpu().numpy()
    assert (f32_bits(again) == f32_bits(full)).all()
    mat.close()


def test_q8_full_size_sampled_rows():
    """The FP8 MLP shape in Q8_0 (N = 17408, K = 5120): every row-tile edge
    and random rows against the oracle at M = 1 and 16."""
    N, K = 17408, 5120
    w = synth.weights(N, K, 840)
    blocks = O.q8_0_quantize(w)
    del w
    mat = q.Matrix(q.QMM_FMT_Q8_0, torch.from_numpy(blocks).cuda(), N, K)
    rng = np.random.default_rng(840)
    rows = np.unique(np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128)[:64],
                                     [0, 1, N - 2, N - 1], rng.choice(N, 200, replace=False)]))
    for M in (1, 16):
        a = synth.activations(M, K, 841, outliers=True)
        out = mat.verify(bf16_cuda(a)).cpu().double().numpy()[:, rows]
        ref, S = O.verify_rows(O.FMT_Q8_0, blocks, None, N, K, a, rows=rows)
        assert_within_tolerance(out, ref, S, f"q8 full size M={M}")
    mat.close()


def test_q8_greedy_acceptance():
    N, K, M = 1000, 512, 8
    mat, blocks = q8_matrix(N, K, 850)
    a = synth.activations(M, K, 851, outliers=True)
    ref, S = O.verify_rows(O.FMT_Q8_0, blocks, None, N, K, a)
    ref_am, _, _ = O.greedy_accept(ref.astype(np.float32).astype(np.float64), np.zeros(M, np.int32))
    tokens = np.concatenate([[5], ref_am[:3], [(ref_am[3] + 1) % N], ref_am[4:7]]).astype(np.int32)
    out, am, acc = mat.verify_greedy(bf16_cuda(a), torch.from_numpy(tokens).cuda())
    torch.cuda.synchronize()
    got = out.cpu().double().numpy()
    assert_within_tolerance(got, ref, S, "q8 greedy scores")
    am = am.cpu().numpy()
    for m in range(M):
        assert got[m, am[m]] == got[m].max() and (got[m, :am[m]] < got[m, am[m]]).all()
    k = 0
    while k < M - 1 and am[k] == tokens[k + 1]:
        k += 1
    assert acc.cpu().numpy().tolist() == [k, int(am[k])]
    mat.close()
