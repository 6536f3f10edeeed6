"""GPU parity of the greedy acceptance step (qmm_verify_greedy) against the oracle.

The verify product is held to the usual tolerance.  The argmax is an integer
decided by floating point: where the oracle's largest score beats every other
row by more than the two rows' tolerance bounds the GPU must pick the same row;
elsewhere its pick must be within tolerance of the maximum.  The accepted
count and the next token follow exactly from the GPU's own argmax and the
tokens, and equal the oracle's wherever the argmax is decided.
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


def block_tokens(ref_am, j, N, seed):
    """Input tokens whose drafts agree with the oracle's argmax at positions < j
    and disagree at position j (when there is one)."""
    M = ref_am.size
    rng = np.random.default_rng(seed)
    t = rng.integers(0, N, M).astype(np.int32)
    t[1:j + 1] = ref_am[:j]
    if j + 1 < M and t[j + 1] == ref_am[j]:
        t[j + 1] = (ref_am[j] + 1) % N
    return t


def check_greedy(mat, fmt, wbytes, scales, N, K, a, hadamard, j, what):
    M = a.shape[0]
    ref, S = O.verify_rows(fmt, wbytes, scales, N, K, a, hadamard=hadamard)
    tol = 1e-3 * S + 1e-6
    # the oracle's decision in the kernel's precision (fp32 scores)
    ref_am, _, _ = O.greedy_accept(ref.astype(np.float32).astype(np.float64),
                                   np.zeros(M, np.int32))
    tokens = block_tokens(ref_am, j, N, 7 + M)
    out, am, acc = mat.verify_greedy(bf16_cuda(a), torch.from_numpy(tokens).cuda())
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    got = out.cpu().double().numpy()
    assert_within_tolerance(got, ref, S, what)
    am = am.cpu().numpy()
    k, nxt = (int(v) for v in acc.cpu().numpy())
    decided = np.ones(M, bool)
    for m in range(M):
        r = ref_am[m]
        others = np.delete(np.arange(N), r)
        margin = ref[m, r] - ref[m, others] - (tol[m, r] + tol[m, others]) if N > 1 else np.ones(1)
        if (margin > 0).all():
            assert am[m] == r, f"{what}: row {m} argmax {am[m]} != {r}"
        else:
            decided[m] = False
            g = am[m]
            assert 0 <= g < N and ref[m, g] >= ref[m].max() - (tol[m, g] + tol[m, r]), what
        # the GPU's argmax is a row whose fp32 score is the largest of its own output
        assert got[m, am[m]] == got[m].max(), f"{what}: row {m} is not the max of the output"
        assert (got[m, :am[m]] < got[m, am[m]]).all(), f"{what}: row {m} is not the first max"
    # acceptance follows from the GPU's argmax exactly
    kk = 0
    while kk < M - 1 and am[kk] == tokens[kk + 1]:
        kk += 1
    assert (k, nxt) == (kk, int(am[kk])), what
    if decided.all():
        assert k == min(j, M - 1), what
    return am


def q4(N, K, seed, hadamard=False, **kw):
    w = synth.weights(N, K, seed)
    blocks = O.q4_0_quantize_h32(w) if hadamard else O.q4_0_quantize(w)
    return q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, hadamard=hadamard,
                    **kw), blocks


@pytest.mark.parametrize("variant", ["mma", "split3", "h32", "simt"])
@pytest.mark.parametrize("M,j", [(1, 0), (5, 2), (16, 15), (16, 0), (9, 4)])
def test_greedy_q4(variant, M, j):
    N, K = 1000, 512  # 8 row tiles, the last 104 rows
    kw = {"k_splits": 3} if variant == "split3" else ({"simt": True} if variant == "simt" else {})
    mat, blocks = q4(N, K, 300 + M, hadamard=(variant == "h32"), **kw)
    a = synth.activations(M, K, 301 + M, outliers=True)
    check_greedy(mat, O.FMT_Q4_0, blocks, None, N, K, a, variant == "h32", j,
                 f"greedy q4 {variant} M={M} j={j}")
    mat.close()


@pytest.mark.parametrize("M,j", [(1, 0), (8, 3), (16, 15)])
@pytest.mark.parametrize("splits", [0, 2])
def test_greedy_fp8(M, j, splits):
    N, K = 1024, 512
    w = synth.weights(N, K, 320)
    codes, scales = O.fp8_quantize(w)
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(codes).cuda(), N, K,
                   scales=torch.from_numpy(scales).cuda(), k_splits=splits)
    a = synth.activations(M, K, 321 + M, outliers=True)
    check_greedy(mat, O.FMT_FP8, codes, scales, N, K, a, False, j, f"greedy fp8 M={M} S={splits}")
    mat.close()


def test_greedy_state_resets_and_rows_do_not_depend_on_M():
    """Repeated calls on one handle with changing M: the per-handle state goes
    back to zero after every call, and the argmax of row m is the same for
    every M (the scores are bit-identical across M)."""
    N, K = 1000, 512
    mat, blocks = q4(N, K, 330, k_splits=2)
    a = synth.activations(16, K, 331, outliers=True)
    act = bf16_cuda(a)
    tok = torch.zeros(16, dtype=torch.int32, device="cuda")
    _, am16, _ = mat.verify_greedy(act, tok)
    am16 = am16.cpu().numpy()
    for M in (3, 16, 1, 11, 16):
        out, am, acc = mat.verify_greedy(act[:M].contiguous(), tok[:M].contiguous())
        torch.cuda.synchronize()
        assert (am.cpu().numpy() == am16[:M]).all(), f"argmax changed at M={M}"
    # plain verify calls in between leave the greedy state alone
    mat.verify(act)
    _, am, _ = mat.verify_greedy(act, tok)
    assert (am.cpu().numpy() == am16).all()
    assert mat.sync_status() == q.QMM_OK
    mat.close()


def test_greedy_argument_errors():
    N, K = 256, 512
    mat, _ = q4(N, K, 340)
    tc, _ = q4(N, K, 340, tcgen05=True)
    L = q.load()
    s = torch.cuda.current_stream().cuda_stream
    act = bf16_cuda(synth.activations(4, K, 341))
    out = torch.empty((4, N), dtype=torch.float32, device="cuda")
    ibuf = torch.zeros(8, dtype=torch.int32, device="cuda")
    p = ibuf.data_ptr()
    assert L.qmm_verify_greedy(mat.handle, act.data_ptr(), K, out.data_ptr(), N, 4, None, p, p + 16, s) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_verify_greedy(mat.handle, act.data_ptr(), K, out.data_ptr(), N, 4, p, p + 2, p + 16, s) == q.QMM_ERR_ALIGN
    assert L.qmm_verify_greedy(tc.handle, act.data_ptr(), K, out.data_ptr(), N, 4, p, p, p + 16, s) == q.QMM_ERR_INVALID_ARG
    assert L.qmm_verify_greedy(mat.handle, act.data_ptr(), K, out.data_ptr(), N, 17, p, p, p + 16, s) == q.QMM_ERR_M_RANGE
    mat.close()
    tc.close()


def test_greedy_full_size_output_head():
    """The output-head shape the benchmark times: N = 151,936 tokens, K = 5120
    (1187 row tiles, several waves of CTAs), every score compared."""
    spec = synth.SHAPES["q4_lmhead"]
    N, K, b = spec["N"], spec["K"], spec["seed"]
    w = synth.weights(N, K, b)
    blocks = O.q4_0_quantize(w)
    del w
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K)
    a = synth.activations(3, K, b + 1000, outliers=spec["outliers"], outlier_seed=b + 2000)
    check_greedy(mat, O.FMT_Q4_0, blocks, None, N, K, a, False, 1, "greedy output head M=3")
    mat.close()


@pytest.mark.parametrize("variant", ["mma", "split3", "simt"])
@pytest.mark.parametrize("M", [1, 6, 16])
def test_greedy_nan_scores(variant, M):
    """Non-finite scores follow the oracle's rule: a NaN ranks above every
    number and the first NaN of a row wins.  Rows 357 and 801 of W get one
    block with a NaN fp16 scale, so their scores are NaN for every drafted
    row, placed after where the finite maximum falls; one drafted row gets a
    NaN activation, so all of its scores are NaN and its argmax is 0."""
    N, K = 1000, 512
    kw = {"k_splits": 3} if variant == "split3" else ({"simt": True} if variant == "simt" else {})
    w = synth.weights(N, K, 350)
    w[:40] *= 4.0  # the largest finite scores fall in the first rows
    blocks = O.q4_0_quantize(w)
    for n, b in ((357, 5), (801, 11)):
        blocks[n, b, 0], blocks[n, b, 1] = 0x00, 0x7E  # fp16 NaN
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, **kw)
    a = synth.activations(M, K, 351 + M, outliers=True)
    nan_row = M // 2 if M > 1 else None
    if nan_row is not None:
        a[nan_row, 77] = 0x7FC0  # bf16 NaN
    ref, S = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a)
    ref_am, _, _ = O.greedy_accept(ref.astype(np.float32).astype(np.float64), np.zeros(M, np.int32))
    finite_best = np.argmax(np.where(np.isnan(ref), -np.inf, ref), axis=1)
    for m in range(M):
        assert ref_am[m] == (0 if m == nan_row else 357)
        if m != nan_row:
            assert finite_best[m] < 357  # the NaN lies after the finite maximum
    tokens = block_tokens(ref_am, M - 1, N, 352)
    out, am, acc = mat.verify_greedy(bf16_cuda(a), torch.from_numpy(tokens).cuda())
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    got = out.cpu().double().numpy()
    assert (np.isnan(got) == np.isnan(ref)).all(), "NaN positions differ from the oracle's"
    fin = ~np.isnan(ref)
    err = np.abs(got[fin] - ref[fin])
    assert (err <= 1e-3 * S[fin] + 1e-6).all(), "finite scores out of tolerance"
    am = am.cpu().numpy()
    assert (am == ref_am).all(), f"argmax {am.tolist()} != oracle {ref_am.tolist()}"
    k, nxt = (int(v) for v in acc.cpu().numpy())
    kk = 0
    while kk < M - 1 and ref_am[kk] == tokens[kk + 1]:
        kk += 1
    assert (k, nxt) == (kk, int(ref_am[kk]))
    mat.close()
