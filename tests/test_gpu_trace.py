"""The per-CTA timeline hook of the verify kernel.

The product library compiles the stamps out, so qmm_debug_set_trace refuses
with QMM_ERR_STATE there.  The profiling tool builds its own variant with the
stamps (-DQMM_TRACE) and runs in a child process (a process loads one build of
the library); with --check it asserts that every CTA of every call wrote its
stamps in program order, for a split-K plan (the arrival stamp) and for one
split."""
import os
import subprocess
import sys

import pytest

import speculative_decode_verification_qmm_gb300 as q
from speculative_decode_verification_qmm_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    q.load(build_if_missing=True)
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def test_product_build_has_no_stamps():
    w = synth.weights_cuda(256, 512, 5)
    m = q.Matrix(q.QMM_FMT_Q4_0, q.quantize_q4_0(w), 256, 512)
    buf = torch.zeros(1 << 16, dtype=torch.int64, device="cuda")
    with pytest.raises(q.QmmError) as ei:
        q.qmm_debug_set_trace(m.handle, buf)
    assert ei.value.code == q.QMM_ERR_STATE
    m.close()


@pytest.mark.parametrize("splits", [0, 1])
def test_timeline_tool_stamps_in_order(splits):
    cmd = [sys.executable, "-m", "speculative_decode_verification_qmm_gb300.timeline",
           "--shape", "q4_attn", "--ms", "1,16", "--copies", "4", "--k-splits", str(splits),
           "--check"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "us per call in the graph" in r.stdout and "pdl" in r.stdout
