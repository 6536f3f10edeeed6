"""Host logic of the timeline tool (no GPU): quantiles of synthetic stamps,
the CTA-per-SM count and the program-order check."""
import numpy as np
import pytest

from speculative_decode_verification_qmm_gb300 import _lib, timeline


def stamps(ctas, base, step, last=None):
    s = np.zeros((ctas, _lib.QMM_TRACE_FIELDS), np.int64)
    order = [f for _, f in timeline.ROWS]
    for b in range(ctas):
        for i, f in enumerate(order):
            s[b, f] = base + 1000 * b + step * i
        s[b, _lib.QMM_TR_SMID] = b // 2
        s[b, _lib.QMM_TR_LAST] = 1 if last is not None and b in last else 0
    return s


def test_summary_quantiles_relative_to_previous_exit():
    st = stamps(4, 10_000, 500, last={3})
    s = timeline.summarize(st, prev_exit=9_000)
    # entry of CTA b = 10000 + 1000 b -> (1000 .. 4000 ns) after the previous exit
    assert s["entry"][0] == pytest.approx(1.0) and s["entry"][-1] == pytest.approx(4.0)
    assert s["exit"][0] == pytest.approx(1.0 + 8 * 0.5)
    assert s["ctas_per_sm"] == {2: 2}
    assert s["last"] == 1
    assert "pdl" in timeline.format_call(s)


def test_summary_skips_unwritten_stamps():
    st = stamps(3, 5_000, 100)
    st[:, _lib.QMM_TR_ARRIVE] = 0  # one split: no arrival
    s = timeline.summarize(st, prev_exit=None)
    assert "arrived" not in s and "exit" in s
    timeline.check_order(st)


def test_check_order_rejects_out_of_order_and_missing():
    st = stamps(2, 5_000, 100)
    bad = st.copy()
    bad[1, _lib.QMM_TR_DATA], bad[1, _lib.QMM_TR_PDL] = bad[1, _lib.QMM_TR_PDL], bad[1, _lib.QMM_TR_DATA]
    with pytest.raises(AssertionError):
        timeline.check_order(bad)
    bad = st.copy()
    bad[0, _lib.QMM_TR_LOOP] = 0
    bad[0, _lib.QMM_TR_RED] = 0
    with pytest.raises(AssertionError):
        timeline.check_order(bad)
