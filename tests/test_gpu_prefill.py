"""GPU parity of the prefill product (qmm_prefill: FP8 handles, any number of
activation rows M, tcgen05 tensor cores) against the oracle.

Within 1e-3 * sum|a_k w_k| + 1e-6 per element: every output at sizes that span
several weight tiles, activation tiles and raster groups with ragged activation
tails, the rotated variants, strided rows, and sampled outputs of the
full-size workload.  Row results do not depend on how many rows follow them.
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


def fp8_matrix(N, K, seed, hadamard=False, **kw):
    w = synth.weights(N, K, seed)
    if hadamard:
        w = O.rotate_weights_f32(w, 32 if hadamard is True else hadamard)
    codes, scales = O.fp8_quantize(w)
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(codes).cuda(), N, K,
                   scales=torch.from_numpy(scales).cuda(), hadamard=hadamard, **kw)
    return mat, codes, scales


@pytest.mark.parametrize("N,K,M,hadamard", [
    (256, 512, 200, False),    # two activation tiles, the second ragged
    (384, 1024, 1, False),     # one row
    (512, 384, 130, False),
    (1024, 2048, 300, False),  # 8 weight tiles x 2 activation tiles (192 + 108 rows)
    (2304, 256, 40, False),    # 18 weight tiles: a full raster group of 16, then one of 2
    (128, 128, 1000, False),   # one weight tile, one stage, 6 activation tiles
    (256, 640, 129, 32),
    (384, 1024, 257, 64),
    (256, 512, 128, 128),
])
def test_prefill_fp8(N, K, M, hadamard):
    mat, codes, scales = fp8_matrix(N, K, 900 + N + K, hadamard)
    a = synth.activations(M, K, 901 + M, outliers=True)
    out = mat.prefill(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    ref, S = O.verify_rows(O.FMT_FP8, codes, scales, N, K, a, hadamard=hadamard)
    assert_within_tolerance(out.cpu().double().numpy(), ref, S,
                            f"prefill N={N} K={K} M={M} H={hadamard}")
    mat.close()


def test_prefill_on_a_split_stream():
    """A handle planned with 3 K splits stores 6 stages per weight tile for
    K = 640 (5 stages of data, one of padding): the GEMM walks the 5."""
    N, K, M = 256, 640, 150
    mat, codes, scales = fp8_matrix(N, K, 960, k_splits=3)
    info = mat.info()
    assert info["k_splits"] * info["stages_per_cta"] > K // 128
    a = synth.activations(M, K, 961, outliers=True)
    out = mat.prefill(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    ref, S = O.verify_rows(O.FMT_FP8, codes, scales, N, K, a)
    assert_within_tolerance(out.cpu().double().numpy(), ref, S, "prefill, split stream")
    mat.close()


def test_prefill_many_rows():
    """70,000 prompt rows (365 activation tiles, a pre-pass of 8750 blocks)
    against one weight tile, every output compared."""
    N, K, M = 128, 256, 70_000
    mat, codes, scales = fp8_matrix(N, K, 970)
    a = synth.activations(M, K, 971, outliers=True)
    out = mat.prefill(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    ref, S = O.verify_rows(O.FMT_FP8, codes, scales, N, K, a)
    assert_within_tolerance(out.cpu().double().numpy(), ref, S, "prefill, 70k rows")
    mat.close()


def test_prefill_strided_rows_and_outputs():
    """lda > K (the padding holds NaNs that must never be read) and ldo > N
    (the columns past N stay untouched)."""
    N, K, M = 384, 512, 150
    mat, codes, scales = fp8_matrix(N, K, 910)
    a = synth.activations(M, K, 911, outliers=True)
    act = bf16_cuda(a, pad_to=K + 72)
    out_full = torch.full((M, N + 40), 7.0, dtype=torch.float32, device="cuda")
    out = out_full[:, :N]
    mat.prefill(act, out=out)
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    got = out_full.cpu().double().numpy()
    assert (got[:, N:] == 7.0).all()
    ref, S = O.verify_rows(O.FMT_FP8, codes, scales, N, K, a)
    assert_within_tolerance(got[:, :N], ref, S, "prefill strided")
    mat.close()


def test_prefill_rows_do_not_depend_on_M():
    N, K = 512, 1024
    mat, _, _ = fp8_matrix(N, K, 920)
    act = bf16_cuda(synth.activations(300, K, 921, outliers=True))
    full = mat.prefill(act).cpu().numpy()
    for M in (1, 77, 128, 191, 192, 193, 299):
        part = mat.prefill(act[:M].contiguous()).cpu().numpy()
        assert (f32_bits(part) == f32_bits(full[:M])).all(), f"row results changed at M={M}"
    mat.close()


def test_prefill_full_size_sampled():
    """The FP8 MLP weights (N = 17408, K = 5120) against 8192 prompt rows, the
    size the benchmark times: every weight-tile edge and random rows, for the
    activation-tile edges and random activation rows."""
    N, K, M = 17408, 5120, 8192
    w = synth.weights(N, K, 930)
    codes, scales = O.fp8_quantize(w)
    del w
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(codes).cuda(), N, K,
                   scales=torch.from_numpy(scales).cuda())
    a = synth.activations(M, K, 931, outliers=True)
    out = mat.prefill(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    rng = np.random.default_rng(930)
    rows = np.unique(np.concatenate([np.arange(0, N, 128)[::8], np.arange(127, N, 128)[::8],
                                     [0, 1, N - 1], rng.choice(N, 96, replace=False)]))
    ms = np.unique(np.concatenate([[0, 1, 191, 192, 383, 384, 4031, 4032, M - 1],
                                   rng.choice(M, 40, replace=False)]))
    got = out[torch.from_numpy(ms).cuda()][:, torch.from_numpy(rows).cuda()].cpu().double().numpy()
    ref, S = O.verify_rows(O.FMT_FP8, codes, scales, N, K, a[ms], rows=rows)
    assert_within_tolerance(got, ref, S, "prefill full size")
    mat.close()


def test_prefill_argument_errors():
    N, K, M = 256, 512, 64
    mat, _, _ = fp8_matrix(N, K, 940)
    w = synth.weights(N, K, 941)
    q4 = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(O.q4_0_quantize(w)).cuda(), N, K)
    L = q.load()
    s = torch.cuda.current_stream().cuda_stream
    act = bf16_cuda(synth.activations(M, K, 942))
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    need = q.qmm_prefill_workspace(mat.handle, M)
    assert need >= M * K * 2 + M * 4
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    a, o, w0 = act.data_ptr(), out.data_ptr(), ws.data_ptr()
    assert L.qmm_prefill(q4.handle, a, K, o, N, M, w0, need, s) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_prefill(mat.handle, a, K, o, N, 0, w0, need, s) == q.QMM_ERR_M_RANGE
    assert L.qmm_prefill(mat.handle, a, K, o, N, M, w0, need - 1, s) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_prefill(mat.handle, a, K, o, N, M, None, need, s) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_prefill(mat.handle, a + 2, K, o, N, M, w0, need, s) == q.QMM_ERR_ALIGN
    assert L.qmm_prefill(mat.handle, a, K, o, N, M, w0 + 16, need, s) == q.QMM_ERR_ALIGN
    assert L.qmm_prefill(mat.handle, a, K - 8, o, N, M, w0, need, s) == q.QMM_ERR_ALIGN
    assert L.qmm_prefill(mat.handle, a, K, o, N - 1, M, w0, need, s) == q.QMM_ERR_ALIGN
    with pytest.raises(q.QmmError):
        q.qmm_prefill_workspace(q4.handle, M)
    assert L.qmm_prefill(mat.handle, a, K, o, N, M, w0, need, s) == q.QMM_OK
    assert mat.sync_status() == q.QMM_OK
    mat.close()
    q4.close()


def test_prefill_timeout_path_and_recovery():
    """A wait limit of 0 makes every bounded wait of the GEMM give up at once:
    the CTAs record it, drain their copies and free tensor memory; the handle
    works again after qmm_sync_status."""
    N, K, M = 512, 1024, 200
    mat, codes, scales = fp8_matrix(N, K, 950)
    a = synth.activations(M, K, 951, outliers=True)
    act = bf16_cuda(a)
    q.qmm_debug_set_wait_limit(mat.handle, 0)
    mat.prefill(act)
    assert mat.sync_status() == q.QMM_ERR_TIMEOUT
    assert mat.sync_status() == q.QMM_OK
    q.qmm_debug_set_wait_limit(mat.handle, 2_000_000_000)
    out = mat.prefill(act)
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    ref, S = O.verify_rows(O.FMT_FP8, codes, scales, N, K, a)
    assert_within_tolerance(out.cpu().double().numpy(), ref, S, "prefill after timeout")
    mat.close()
