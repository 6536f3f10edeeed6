"""GPU parity of the whole-model weight sweep: 64 layers, each with the four
Q4_0 matrices qkv 10240x5120, out 5120x5120, gate+up 34816x5120 and down
5120x17408 (11.60 GiB of compressed weights), one verify pass per M in
{1, 2, 4, 8, 16}, set up exactly as the benchmark sets it up.

A target forward reads all of these weights once per verified block ("Qwen3.8-
27B on the AMD R9700: up to 227 tok/s", TL;DR and "Against llama.cpp, with the
same drafter": about 13 GiB streamed per forward for 4, 8 or 16 positions).
The oracle cannot afford the full product, so every matrix of every layer is
checked on 64 sampled rows:

  * the sampled rows' fp32 weights (drawn on the device by the seeded
    generator) are copied back, quantized by the oracle and compared bit for
    bit with the device quantizer's blocks of those rows;
  * after each pass the sampled rows of every output are copied back and
    compared element by element with the oracle's product of those rows, at
    |gpu - oracle| <= 1e-3 * sum_k |a_k w_k| + 1e-6.
"""
import numpy as np
import pytest

import oracle as O
import speculative_decode_verification_qmm_gb300 as q
from speculative_decode_verification_qmm_gb300 import synth
from gpu_util import assert_within_tolerance

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROWS_PER_MATRIX = 64


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    q.load(build_if_missing=True)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def test_whole_model_sweep_sampled_rows():
    rng = np.random.default_rng(2024)
    mats = []  # (name, layer, Matrix, sampled rows, oracle blocks of those rows)
    for layer in range(synth.MODEL_LAYERS):
        for j, (name, N, K) in enumerate(synth.MODEL_LAYER):
            w = synth.weights_cuda(N, K, 4 * layer + j)
            blocks = q.quantize_q4_0(w)
            rows = np.sort(rng.choice(N, ROWS_PER_MATRIX, replace=False))
            if layer == 0:  # tile edges and both ends in the first layer
                rows = np.unique(np.concatenate([rows[:ROWS_PER_MATRIX - 6],
                                                 [0, 127, 128, N - 129, N - 2, N - 1]]))
            idx = torch.from_numpy(rows).cuda()
            w_rows = w.index_select(0, idx).cpu().numpy()
            dev_rows = blocks.index_select(0, idx).cpu().numpy()
            ref_rows = O.q4_0_quantize(w_rows)
            assert (dev_rows == ref_rows).all(), f"layer {layer} {name}: quantized blocks differ"
            del w
            mats.append((name, layer, q.Matrix(q.QMM_FMT_Q4_0, blocks, N, K), rows, ref_rows))
            del blocks
    torch.cuda.synchronize()
    acts = {}
    worst = 0.0
    for M in synth.MODEL_MS:
        outs = []
        for name, layer, mat, rows, _ in mats:
            key = (M, mat.K)
            if key not in acts:
                acts[key] = synth.activations_cuda(M, mat.K, 10_000 + mat.K, outliers=False)
            outs.append(mat.verify(acts[key]))  # one verify pass: every matrix once
        torch.cuda.synchronize()
        for (name, layer, mat, rows, ref_rows), out in zip(mats, outs):
            assert mat.sync_status() == q.QMM_OK
            a = acts[(M, mat.K)].view(torch.int16).cpu().numpy().view(np.uint16)
            got = out[:, torch.from_numpy(rows).cuda()].cpu().double().numpy()
            ref, S = O.verify_rows(O.FMT_Q4_0, ref_rows, None, rows.size, mat.K, a)
            worst = max(worst, assert_within_tolerance(got, ref, S, f"layer {layer} {name} M={M}"))
        del outs
    for _, _, mat, _, _ in mats:
        mat.close()
    assert worst <= 1.0
