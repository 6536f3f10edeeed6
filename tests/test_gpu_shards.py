"""The row split of the multi-GPU path, run shard after shard on one GPU.

The rows of W are independent, so a G-GPU split gives GPU g the rows
[g N / G, (g + 1) N / G) (multiples of 128 for FP8) and no reduction is needed
("r9k: a from-scratch inference engine for Qwen3.8-27B on two Radeon AI PRO
R9700", opening section, splits its model over two GPUs).  Each shard here is
a handle made by qmm_create_rows over the full weight buffers; the shards'
outputs, put side by side, must match the oracle's product of the whole matrix
element by element within 1e-3 * sum|a_k w_k| + 1e-6.
"""
import numpy as np
import pytest

import oracle as O
import speculative_decode_verification_qmm_gb300 as q
from speculative_decode_verification_qmm_gb300 import synth
from gpu_util import assert_within_tolerance, bf16_cuda

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    q.load(build_if_missing=True)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def weights_of(fmt, N, K, seed, hadamard=False):
    w = synth.weights(N, K, seed)
    if fmt == "q4":
        wb = O.q4_0_quantize_h32(w) if hadamard else O.q4_0_quantize(w)
        return q.QMM_FMT_Q4_0, O.FMT_Q4_0, wb, None
    if fmt == "q8":
        return q.QMM_FMT_Q8_0, O.FMT_Q8_0, O.q8_0_quantize(w), None
    codes, scales = O.fp8_quantize(w)
    return q.QMM_FMT_FP8_E4M3_B128, O.FMT_FP8, codes, scales


@pytest.mark.parametrize("fmt,N,K,G,hadamard,on_device", [
    ("q4", 1000, 1376, 2, False, True),
    ("q4", 1000, 1376, 3, True, True),
    ("q4", 5120, 5120, 4, False, True),
    ("q4", 777, 512, 5, False, False),
    ("q8", 600, 1024, 3, False, True),
    ("fp8", 1024, 896, 2, False, True),
    ("fp8", 1408, 512, 3, False, False),
])
@pytest.mark.parametrize("M", [1, 16])
def test_shards_side_by_side_match_the_oracle(fmt, N, K, G, hadamard, on_device, M):
    qfmt, ofmt, wb, sc = weights_of(fmt, N, K, 600 + N + G, hadamard)
    a = synth.activations(M, K, 601 + K, outliers=True)
    ref, S = O.verify_rows(ofmt, wb, sc, N, K, a, hadamard=hadamard)
    align = 128 if fmt == "fp8" else 1
    wdev = torch.from_numpy(wb).cuda() if on_device else torch.from_numpy(wb)
    sdev = None if sc is None else (torch.from_numpy(sc).cuda() if on_device else torch.from_numpy(sc))
    act = bf16_cuda(a)
    parts = []
    for g in range(G):
        n0, n1 = q.shard_rows(N, G, g, align)
        mat = q.Matrix(qfmt, wdev, N, K, scales=sdev, hadamard=hadamard, rows=(n0, n1))
        assert mat.N == n1 - n0 and mat.info()["N"] == n1 - n0
        parts.append(mat.verify(act).cpu().double().numpy())
        assert mat.sync_status() == q.QMM_OK
        mat.close()
    got = np.concatenate(parts, axis=1)
    assert got.shape == (M, N)
    assert_within_tolerance(got, ref, S, f"{fmt} N={N} K={K} G={G} M={M}")


def test_shard_argument_errors():
    N, K = 512, 256
    qfmt, _, wb, sc = weights_of("fp8", N, K, 650)
    w = torch.from_numpy(wb).cuda()
    s = torch.from_numpy(sc).cuda()
    for rows in [(0, 0), (-1, 128), (0, N + 128), (256, 128), (64, 512), (128, 200)]:
        with pytest.raises(q.QmmError) as ei:
            q.Matrix(qfmt, w, N, K, scales=s, rows=rows)
        assert ei.value.code == q.QMM_ERR_SHAPE, rows
    m = q.Matrix(qfmt, w, N, K, scales=s, rows=(128, 512))
    assert m.N == 384
    m.close()
