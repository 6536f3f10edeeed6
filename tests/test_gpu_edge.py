"""GPU parity on the method's own edge cases, against the oracle.

Q4_0 stores a weight as a 4-bit code offset by 8, so code 8 is the zero weight
("Qwen3.8-27B at 45.7 tok/s: DFlash2 in 1bit serve, and 4-bit activations with
a Hadamard rotation", section "Prompt processing: 4-bit activations, rotated
first"), and blocks that are almost all code 8 are ordinary in real weight
files.  The Gaussian workloads never produce them, so these tests build the
blocks by hand:

  * "spike" blocks: 31 codes at the zero weight and one extreme code (0 or 15
    for Q4_0, -127 or 127 for Q8_0) in the column where every activation row
    is 0, so the block's true contribution is exactly zero while the
    activations elsewhere are large (N(0,1) with x20 outlier channels);
  * blocks of nothing but zero weights;
  * fp16 block scales at the ends of the format: 65504, -65504, 1, the
    smallest normal 2^-14, the smallest subnormal 2^-24, and -0;
  * rows made only of such blocks, whose exact result is 0 with
    sum |a_k w_k| = 0 (so the bound is the 1e-6 absolute term alone), and rows
    that mix them with ordinary blocks.

FP8 gets the analogous tiles: zero scales, scale 1 with codes at +-448,
very large and very small fp32 scales, and tiles of zero codes with one spike.

Every output is compared element by element with the oracle at
|gpu - oracle| <= 1e-3 * sum_k |a_k w_k| + 1e-6, at M = 1, 8 and 16, with one
K split and with several.
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


# fp16 bit patterns of the edge scales
F16_EDGE = {
    "max": 0x7BFF,       # 65504
    "-max": 0xFBFF,      # -65504
    "one": 0x3C00,       # 1
    "min_normal": 0x0400,  # 2^-14
    "min_sub": 0x0001,   # 2^-24
    "-zero": 0x8000,     # -0
}
F16_TYPICAL = 0x1E66    # about 0.00625 = 0.05 / 8, a typical Q4_0 scale for N(0, 0.02)


def spike_columns(K):
    """Per 32-block the column that holds the spike (the same for every row,
    so that one zero activation column serves all rows)."""
    nb = K // 32
    return np.array([32 * b + (7 * b + 3) % 32 for b in range(nb)], np.int64)


def edge_activations(M, K, seed):
    """bf16 N(0,1) rows with x20 outlier channels, zero at every spike column
    (+0 in even rows, -0 in odd rows)."""
    a = synth.activations(M, K, seed, outliers=True)
    cols = spike_columns(K)
    for m in range(M):
        a[m, cols] = 0x0000 if m % 2 == 0 else 0x8000
    return a


def edge_row_kinds(N):
    """Row kind per output row: 0 = only zero-result blocks (spikes at the zero
    columns and all-zero blocks, edge scales), 1 = mostly those plus ordinary
    blocks, 2 = spikes at non-zero activation columns with edge scales,
    3 = ordinary random blocks with typical scales."""
    return np.array([n % 4 for n in range(N)], np.int64)


def q4_edge_blocks(N, K, seed):
    """Canonical Q4_0 blocks [N][K/32][18] built by hand (see the module doc)."""
    rng = np.random.default_rng(seed)
    nb = K // 32
    cols = spike_columns(K) - 32 * np.arange(nb)  # position inside the block
    kinds = edge_row_kinds(N)
    names = list(F16_EDGE)
    codes = np.full((N, nb, 32), 8, np.uint8)
    scale = np.zeros((N, nb), np.uint16)
    for n in range(N):
        for b in range(nb):
            kind = kinds[n]
            if kind == 1 and rng.random() < 0.25:
                kind = 3
            if kind in (0, 2):
                scale[n, b] = F16_EDGE[names[(n + b) % len(names)]]
                if rng.random() < 0.8:  # a spike; otherwise the block is all zero weights
                    j = cols[b] if kind == 0 else (cols[b] + 1 + rng.integers(0, 31)) % 32
                    codes[n, b, j] = 0 if rng.random() < 0.5 else 15
            else:
                scale[n, b] = F16_TYPICAL + rng.integers(-64, 64)
                codes[n, b] = rng.integers(0, 16, 32)
    blocks = np.zeros((N, nb, 18), np.uint8)
    blocks[:, :, 0] = scale & 0xFF
    blocks[:, :, 1] = scale >> 8
    blocks[:, :, 2:] = codes[:, :, :16] | (codes[:, :, 16:] << 4)
    return blocks


def q8_edge_blocks(N, K, seed):
    """Canonical Q8_0 blocks [N][K/32][34]: fp16 d, then 32 int8 codes."""
    rng = np.random.default_rng(seed)
    nb = K // 32
    cols = spike_columns(K) - 32 * np.arange(nb)
    kinds = edge_row_kinds(N)
    names = list(F16_EDGE)
    codes = np.zeros((N, nb, 32), np.int8)
    scale = np.zeros((N, nb), np.uint16)
    for n in range(N):
        for b in range(nb):
            kind = kinds[n]
            if kind == 1 and rng.random() < 0.25:
                kind = 3
            if kind in (0, 2):
                scale[n, b] = F16_EDGE[names[(n + b) % len(names)]]
                if rng.random() < 0.8:
                    j = cols[b] if kind == 0 else (cols[b] + 1 + rng.integers(0, 31)) % 32
                    codes[n, b, j] = -127 if rng.random() < 0.5 else 127
            else:
                scale[n, b] = 0x1A66 + rng.integers(-64, 64)  # about 0.05 / 127
                codes[n, b] = rng.integers(-127, 128, 32)
    blocks = np.zeros((N, nb, 34), np.uint8)
    blocks[:, :, 0] = scale & 0xFF
    blocks[:, :, 1] = scale >> 8
    blocks[:, :, 2:] = codes.view(np.uint8)
    return blocks


def fp8_edge(N, K, seed):
    """E4M3 codes [N][K] and fp32 tile scales [N/128][K/128]: tiles of zero codes
    with one spike per 32 columns at the zero-activation column, tiles at the
    code range ends, scale 0, and very large and very small scales."""
    rng = np.random.default_rng(seed)
    tn, tk = N // 128, K // 128
    codes = np.zeros((N, K), np.uint8)
    scales = np.zeros((tn, tk), np.float32)
    cols = spike_columns(K)
    edge_scales = [0.0, 1.0, 1e30, 1e-30, 2.0 ** -126, 3.0e-41, 0.05 / 448]
    for i in range(tn):
        for j in range(tk):
            kind = (i + 2 * j) % 4
            scales[i, j] = edge_scales[(3 * i + j) % len(edge_scales)]
            rows = slice(128 * i, 128 * i + 128)
            c = cols[(cols >= 128 * j) & (cols < 128 * j + 128)]
            if kind == 0:    # spikes at the zero columns: +-448 (0x7E / 0xFE)
                codes[rows, c] = np.where(rng.random((128, c.size)) < 0.5, 0x7E, 0xFE)
            elif kind == 1:  # random codes with the extremes sprinkled in (no NaN code)
                t = rng.integers(0, 256, (128, 128)).astype(np.uint8)
                t[(t & 0x7F) == 0x7F] = 0x7E
                codes[rows, 128 * j:128 * j + 128] = t
            elif kind == 2:  # all zero codes (+0 and -0)
                codes[rows, 128 * j:128 * j + 128] = np.where(rng.random((128, 128)) < 0.5, 0, 0x80)
            else:            # ordinary tile
                w = synth.weights(128, 128, seed + 17 * i + j)
                cq, sq = O.fp8_quantize(w)
                codes[rows, 128 * j:128 * j + 128] = cq
                scales[i, j] = sq[0, 0]
    return codes, scales


def check(mat, fmt, wbytes, scales, N, K, a, hadamard, what):
    out = mat.verify(bf16_cuda(a))
    torch.cuda.synchronize()
    assert mat.sync_status() == q.QMM_OK
    got = out.cpu().double().numpy()
    ref, S = O.verify_rows(fmt, wbytes, scales, N, K, a, hadamard=hadamard)
    assert_within_tolerance(got, ref, S, what)
    return got, ref, S


KERNEL_FLAGS = {"mma": {}, "tc": {"tcgen05": True}, "simt": {"simt": True}}


@pytest.mark.parametrize("kernel", ["mma", "tc", "simt"])
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_q4_edge_blocks(M, splits, kernel):
    N, K = 264, 1376
    blocks = q4_edge_blocks(N, K, 71)
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, k_splits=splits,
                   **KERNEL_FLAGS[kernel])
    a = edge_activations(M, K, 72)
    got, ref, S = check(mat, O.FMT_Q4_0, blocks, None, N, K, a, False,
                        f"q4 edge {kernel} S={splits} M={M}")
    # rows built only from zero-result blocks are exactly zero
    zero_rows = np.nonzero(edge_row_kinds(N) == 0)[0]
    assert (ref[:, zero_rows] == 0).all() and (S[:, zero_rows] == 0).all()
    assert (got[:, zero_rows] == 0).all(), "a row of zero weights gave a non-zero result"
    mat.close()


@pytest.mark.parametrize("rot", [32, 128])
@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_q4_edge_blocks_rotated(M, splits, rot):
    # the rotated path (f16 operands after the pre-pass) on the same blocks:
    # the weights mean H w / rot, the activations are rotated on the device
    N, K = 264, 1408
    blocks = q4_edge_blocks(N, K, 73)
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K, hadamard=rot,
                   k_splits=splits)
    a = edge_activations(M, K, 74)
    check(mat, O.FMT_Q4_0, blocks, None, N, K, a, rot, f"q4 edge H{rot} S={splits} M={M}")
    mat.close()


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_q8_edge_blocks(M, splits):
    N, K = 264, 1376
    blocks = q8_edge_blocks(N, K, 75)
    mat = q.Matrix(q.QMM_FMT_Q8_0, torch.from_numpy(blocks).cuda(), N, K, k_splits=splits)
    a = edge_activations(M, K, 76)
    got, ref, S = check(mat, O.FMT_Q8_0, blocks, None, N, K, a, False,
                        f"q8 edge S={splits} M={M}")
    zero_rows = np.nonzero(edge_row_kinds(N) == 0)[0]
    assert (ref[:, zero_rows] == 0).all() and (got[:, zero_rows] == 0).all()
    mat.close()


@pytest.mark.parametrize("splits", [1, 3])
@pytest.mark.parametrize("M", [1, 8, 16])
def test_fp8_edge_tiles(M, splits):
    N, K = 512, 896
    codes, scales = fp8_edge(N, K, 77)
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, torch.from_numpy(codes).cuda(), N, K,
                   scales=torch.from_numpy(scales).cuda(), k_splits=splits)
    a = edge_activations(M, K, 78)
    check(mat, O.FMT_FP8, codes, scales, N, K, a, False, f"fp8 edge S={splits} M={M}")
    mat.close()


def test_q4_edge_dequant_bit_exact():
    # the exact dequantization of the hand-built blocks, every scale at the format's ends
    N, K = 264, 1376
    blocks = q4_edge_blocks(N, K, 79)
    mat = q.Matrix(q.QMM_FMT_Q4_0, torch.from_numpy(blocks).cuda(), N, K)
    got = mat.dequantize().cpu().numpy()
    ref = O.q4_0_dequant(blocks, N, K).astype(np.float32)
    assert (got.view(np.uint32) == ref.view(np.uint32)).all()
    mat.close()
