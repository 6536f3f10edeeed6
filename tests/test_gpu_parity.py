"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Bit-exact: dequantization, the Hadamard rotation, the device quantizers, and
row results across M.  Within 1e-3 * sum|a_k w_k| + 1e-6 per element: the
verify product, at sizes spanning several tiles with ragged tails.
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


def q4_matrix(N, K, seed, hadamard=False, **kw):
    w = synth.weights(N, K, seed)
    blocks = O.q4_0_quantize_h32(w) if hadamard else O.q4_0_quantize(w)
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, hadamard=hadamard, **kw)
    return mat, blocks


def fp8_matrix(N, K, seed, hadamard=False, **kw):
    w = synth.weights(N, K, seed)
    if hadamard:
        # the offline rotation: rotate each 32-block (fp32), divide by 32, then quantize
        r = O.fwht32_f32(w.reshape(N, K // 32, 32)).reshape(N, K) * np.float32(0.03125)
        codes, scales = O.fp8_quantize(r)
    else:
        codes, scales = O.fp8_quantize(w)
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(codes).cuda(), N, K,
                   scales=torch.from_numpy(scales).cuda(), hadamard=hadamard, **kw)
    return mat, codes, scales


def check_verify(mat, fmt, wbytes, scales, N, K, a, hadamard, rows=None, what=""):
    M = a.shape[0]
    out = mat.verify(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    got = out.cpu().double().numpy()
    ref, S = O.verify_rows(fmt, wbytes, scales, N, K, a, hadamard=hadamard, rows=rows)
    if rows is not None:
        got = got[:, rows]
    return assert_within_tolerance(got, ref, S, what)


# ---------------------------------------------------------------- bit-exact pieces
@pytest.mark.parametrize("N,K,splits", [(256, 512, 0), (200, 352, 0), (424, 1376, 3), (16, 32, 1),
                                        (130, 2048, 5)])
def test_dequant_q4_bit_exact(N, K, splits):
    mat, blocks = q4_matrix(N, K, 7 + N, k_splits=splits)
    got = mat.dequantize().cpu().numpy()
    ref = O.q4_0_dequant(blocks, N, K).astype(np.float32)
    assert (f32_bits(got) == f32_bits(ref)).all()


@pytest.mark.parametrize("N,K,splits", [(256, 384, 0), (384, 1280, 3), (128, 128, 1)])
def test_dequant_fp8_bit_exact(N, K, splits):
    mat, codes, scales = fp8_matrix(N, K, 11 + N, k_splits=splits)
    got = mat.dequantize().cpu().numpy()
    ref = O.fp8_dequant(codes, scales).astype(np.float32)
    assert (f32_bits(got) == f32_bits(ref)).all()


@pytest.mark.parametrize("M,K,lda", [(5, 512, 512), (16, 5120, 5120), (3, 96, 104), (1, 32, 40)])
def test_hadamard32_bit_exact(M, K, lda):
    a = synth.activations(M, K, 300 + K, outliers=True)
    got = q.hadamard32(bf16_cuda(a, pad_to=lda)).cpu().numpy()
    ref = O.hadamard32_act_f32(a)
    assert (f32_bits(got) == f32_bits(ref)).all()


@pytest.mark.parametrize("hadamard", [False, True])
def test_quantize_q4_bit_exact(hadamard):
    N, K = 96, 1024
    w = synth.weights(N, K, 500)
    w[0, :32] = 0.0
    w[1, 32:64] = 0.5
    w[2, 64:96] *= 1e-6
    w[3, 96 + 2], w[3, 96 + 20] = -0.3, 0.3
    w[4, :32] = np.float32(1e5)
    w[5, :32] = np.float32(6e5)  # the fp16 scale overflows to infinity
    got = q.quantize_q4_0(torch.from_numpy(w).cuda(), hadamard=hadamard).cpu().numpy()
    ref = O.q4_0_quantize_h32(w) if hadamard else O.q4_0_quantize(w)
    bad = np.argwhere((got != ref).any(axis=2))
    detail = []
    for n, b in bad[:4]:
        x = w[n, 32 * b:32 * b + 32]
        dg = np.array([got[n, b, 0] | (got[n, b, 1] << 8)], np.uint16).view(np.float16)[0]
        dr = np.array([ref[n, b, 0] | (ref[n, b, 1] << 8)], np.uint16).view(np.float16)[0]
        detail.append(f"block ({n},{b}) gpu {got[n, b].tolist()} (d {float(dg)!r}) oracle "
                      f"{ref[n, b].tolist()} (d {float(dr)!r}) x {[float(v).hex() for v in x[:4]]}")
    assert bad.size == 0, f"{len(bad)} blocks differ; " + "; ".join(detail)


@pytest.mark.parametrize("hadamard", [False, True])
def test_quantize_fp8_bit_exact(hadamard):
    N, K = 256, 384
    w = synth.weights(N, K, 600)
    w[:128, 128:256] = 0.0
    codes, scales = q.quantize_fp8(torch.from_numpy(w).cuda(), hadamard=hadamard)
    if hadamard:
        r = O.fwht32_f32(w.reshape(N, K // 32, 32)).reshape(N, K) * np.float32(0.03125)
        rc, rs = O.fp8_quantize(r)
    else:
        rc, rs = O.fp8_quantize(w)
    assert (f32_bits(scales.cpu().numpy()) == f32_bits(rs)).all()
    assert (codes.cpu().numpy() == rc).all()


# ---------------------------------------------------------------- verify product
KERNELS = {"mma": {}, "tc": {"tcgen05": True}, "simt": {"simt": True}}


@pytest.mark.parametrize("kernel", ["mma", "tc", "simt"])
@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 15, 16])
def test_verify_q4_small_config(M, kernel):
    # M rows, K = 512, N = 256 (the single-shape parity workload), seed 0
    w, a, spec = synth.workload("q4_small", M=M)
    N, K = spec["N"], spec["K"]
    blocks = O.q4_0_quantize(w)
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, **KERNELS[kernel])
    check_verify(mat, O.FMT_Q4_0, blocks, None, N, K, a, False, what=f"q4 {kernel} M={M}")


@pytest.mark.parametrize("N,K,splits,hadamard,kernel", [
    (424, 1376, 0, False, "mma"), (424, 1376, 3, False, "mma"), (424, 1376, 6, True, "mma"),
    (1000, 2560, 0, True, "mma"), (256, 512, 2, False, "simt"), (424, 1376, 3, True, "simt"),
    (8, 32, 0, False, "mma"), (1, 64, 0, False, "mma"), (129, 4096, 16, False, "mma"),
    (424, 1376, 0, False, "tc"), (424, 1376, 3, False, "tc"), (8, 32, 0, False, "tc"),
    (129, 4096, 16, False, "tc"), (1000, 2560, 5, False, "tc"),
])
@pytest.mark.parametrize("M", [1, 16])
def test_verify_q4_ragged(N, K, splits, hadamard, kernel, M):
    mat, blocks = q4_matrix(N, K, 40 + N + K, hadamard=hadamard, k_splits=splits, **KERNELS[kernel])
    a = synth.activations(M, K, 41 + K, outliers=True)
    check_verify(mat, O.FMT_Q4_0, blocks, None, N, K, a, hadamard,
                 what=f"q4 N={N} K={K} S={splits} H={hadamard} {kernel} M={M}")


@pytest.mark.parametrize("N,K,splits,hadamard", [(384, 896, 0, False), (384, 896, 3, False),
                                                 (256, 1280, 2, True), (128, 128, 1, False)])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_verify_fp8(N, K, splits, hadamard, M):
    mat, codes, scales = fp8_matrix(N, K, 70 + N, hadamard=hadamard, k_splits=splits)
    a = synth.activations(M, K, 71 + K, outliers=True)
    check_verify(mat, O.FMT_FP8, codes, scales, N, K, a, hadamard, what=f"fp8 N={N} K={K} M={M}")


@pytest.mark.parametrize("fmt,hadamard", [("q4", False), ("q4", True), ("q4tc", False),
                                          ("fp8", False)])
def test_rows_bit_identical_for_every_M(fmt, hadamard):
    N, K = 640, 2048
    if fmt.startswith("q4"):
        mat, _ = q4_matrix(N, K, 90, hadamard=hadamard, k_splits=4, tcgen05=(fmt == "q4tc"))
    else:
        mat, _, _ = fp8_matrix(N, K, 90, k_splits=4)
    a = synth.activations(16, K, 91, outliers=True)
    act = bf16_cuda(a)
    full = mat.verify(act).cpu().numpy()
    for M in range(1, 16):
        part = mat.verify(act[:M].contiguous()).cpu().numpy()
        assert (f32_bits(part) == f32_bits(full[:M])).all(), f"row results changed at M={M}"
    # and repeated calls are bit-identical (deterministic split reduction)
    again = mat.verify(act).cpu().numpy()
    assert (f32_bits(again) == f32_bits(full)).all()


def test_verify_host_buffers_match_device():
    N, K, M = 424, 1376, 11
    mat, blocks = q4_matrix(N, K, 123)
    a = synth.activations(M, K, 124, outliers=True)
    dev = mat.verify(bf16_cuda(a)).cpu().numpy()
    act_h = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    out_h = torch.empty((M, N), dtype=torch.float32).pin_memory()
    mat.verify_host(act_h, out_h)
    assert (f32_bits(out_h.numpy()) == f32_bits(dev)).all()


def test_leading_dimensions_and_untouched_memory():
    N, K, M = 300, 640, 5
    mat, blocks = q4_matrix(N, K, 130)
    a = synth.activations(M, K, 131, outliers=True)
    act = bf16_cuda(a, pad_to=K + 24)  # lda > K, padding holds NaN
    canary = 12345.0
    out_full = torch.full((M + 2, N + 36), canary, dtype=torch.float32, device="cuda")
    out = out_full[:M, :N]  # ldo = N + 36 (16-byte aligned rows: (N+36)*4 % 16 == 0)
    q.qmm_verify(mat.handle, act, out, M)
    torch.cuda.synchronize()
    full = out_full.cpu().numpy()
    assert (full[:M, N:] == canary).all() and (full[M:] == canary).all()
    ref, S = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a)
    assert_within_tolerance(full[:M, :N], ref, S, "lda/ldo")


# ---------------------------------------------------------------- full-size shapes
FULL = [
    ("q4_attn", (1, 8, 16), False),
    ("q4_attn_tc", (1, 16), False),
    ("q4_qkv", (1, 8, 16), False),
    ("q4_gateup", (16,), False),
    ("q4_down", (16,), False),
    ("q4_gateup", (16,), True),
    ("q4_down", (16,), True),
    ("q4_gateup", (16,), 128),
    ("q4_down", (16,), 128),
    ("fp8_mlp", (1, 8, 16), False),
]


@pytest.mark.parametrize("name,Ms,hadamard", FULL, ids=[f"{n}-H{h}" for n, _, h in FULL])
def test_full_size_sampled_rows(name, Ms, hadamard):
    """The workloads at full size, in the launch configuration the benchmark
    uses (planner's choice), compared on sampled rows: every row tile boundary,
    both ends, and random rows."""
    tc = name.endswith("_tc")
    spec = synth.SHAPES[name[:-3] if tc else name]
    N, K, b = spec["N"], spec["K"], spec["seed"]
    w = synth.weights(N, K, b)
    rng = np.random.default_rng(b)
    rows = np.unique(np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128)[:64],
                                     [0, 1, N - 2, N - 1], rng.choice(N, 200, replace=False)]))
    rows = rows[rows < N].astype(np.int64)
    if spec["fmt"] == "q4_0":
        if hadamard is True:
            blocks = O.q4_0_quantize_h32(w)
        elif hadamard:
            blocks = O.q4_0_quantize(O.rotate_weights_f32(w, hadamard))
        else:
            blocks = O.q4_0_quantize(w)
        del w
        mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, hadamard=hadamard,
                       tcgen05=tc)
        fmt, wb, sc = O.FMT_Q4_0, blocks, None
    else:
        codes, scales = O.fp8_quantize(w)
        del w
        mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(codes).cuda(), N, K,
                       scales=torch.from_numpy(scales).cuda())
        fmt, wb, sc = O.FMT_FP8, codes, scales
    for M in Ms:
        a = synth.activations(M, K, b + 1000, outliers=spec["outliers"], outlier_seed=b + 2000)
        check_verify(mat, fmt, wb, sc, N, K, a, hadamard, rows=rows, what=f"{name} M={M}")
    mat.close()


# ---------------------------------------------------------------- error paths
def test_error_codes():
    N, K = 256, 512
    mat, blocks = q4_matrix(N, K, 140)
    a = bf16_cuda(synth.activations(16, K, 141))
    out = torch.empty((16, N), dtype=torch.float32, device="cuda")
    L = q.load()
    s = torch.cuda.current_stream().cuda_stream
    h = mat.handle
    assert L.qmm_verify(h, a.data_ptr(), K, out.data_ptr(), N, 0, s) == q.QMM_ERR_M_RANGE
    assert L.qmm_verify(h, a.data_ptr(), K, out.data_ptr(), N, 17, s) == q.QMM_ERR_M_RANGE
    assert L.qmm_verify(h, a.data_ptr() + 2, K, out.data_ptr(), N, 4, s) == q.QMM_ERR_ALIGN
    assert L.qmm_verify(h, a.data_ptr(), K - 8, out.data_ptr(), N, 4, s) == q.QMM_ERR_ALIGN
    assert L.qmm_verify(h, a.data_ptr(), K, out.data_ptr(), N - 1, 4, s) == q.QMM_ERR_ALIGN
    assert L.qmm_verify(h, a.data_ptr(), K, out.data_ptr() + 4, N, 4, s) == q.QMM_ERR_ALIGN
    assert L.qmm_verify(h, None, K, out.data_ptr(), N, 4, s) == q.QMM_ERR_INVALID_ARG
    info = mat.info()
    assert info["N"] == N and info["K"] == K and info["weight_bytes"] == N * K // 32 * 18
    mat.close()
    assert L.qmm_verify(h, a.data_ptr(), K, out.data_ptr(), N, 4, s) == q.QMM_ERR_STATE
    assert L.qmm_destroy(h) == q.QMM_ERR_STATE


def test_injected_allocation_failure_leaks_nothing():
    N, K = 512, 1024
    blocks = torch.from_numpy(O.q4_0_quantize(synth.weights(N, K, 150))).cuda()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    for n in range(1, 64):  # fail the n-th device allocation of qmm_create, for every n
        q.qmm_debug_fail_allocs(n)
        try:
            mat = q.Matrix(q.QMM_FMT_Q4_0, blocks, N, K)
        except q.QmmError as e:
            assert e.code == q.QMM_ERR_CUDA
            failures += 1
            continue
        mat.close()  # n is past the last allocation: the hook did not fire
        break
    q.qmm_debug_fail_allocs(0)
    assert failures >= 5
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (4 << 20)
    mat = q.Matrix(q.QMM_FMT_Q4_0, blocks, N, K)  # works again
    mat.close()


@pytest.mark.parametrize("kernel", ["mma", "tc"])
def test_bounded_wait_timeout_path_and_recovery(kernel):
    """A wait limit of 0 makes every bounded device wait give up at once; the
    kernel records the timeout, drains its own copies and returns.  Nothing
    hangs; the handle works again after qmm_sync_status."""
    N, K, M = 512, 4096, 8
    mat, blocks = q4_matrix(N, K, 160, k_splits=2, **KERNELS[kernel])
    a = synth.activations(M, K, 161, outliers=True)
    act = bf16_cuda(a)
    q.qmm_debug_set_wait_limit(mat.handle, 0)
    mat.verify(act)
    assert mat.sync_status() == q.QMM_ERR_TIMEOUT
    assert mat.sync_status() == q.QMM_OK  # cleared
    q.qmm_debug_set_wait_limit(mat.handle, 2_000_000_000)
    check_verify(mat, O.FMT_Q4_0, blocks, None, N, K, a, False, what="after timeout")
