"""Per-call timeline of back-to-back verify calls (profiling tool).

    python -m speculative_decode_verification_qmm_gb300.timeline \
        [--shape q4_attn] [--ms 1,16] [--copies 12] [--k-splits 0]

Builds a variant of the library with the verify kernel's timeline stamps
compiled in (``-DQMM_TRACE``, into ``_build_trace/``; the in-tree library is
untouched), then, per M, runs ``copies`` verify calls on distinct weight copies
back to back in one CUDA graph, the way the benchmark times them, and prints:

* the graph's time per call (CUDA events, after warm-up replays);
* for the calls after the first, each stamp of every CTA (``QMM_TR_*`` in
  ``include/qmm.h``) relative to the moment the previous call's last CTA left
  the kernel: min / 10 % / median / 90 % / max over the call's CTAs.  The
  ``pdl`` row is when the kernel's wait for its predecessor returned; the rows
  after it are the activation landing, the compute, and the epilogue;
* how many SMs ran one or two CTAs of the call.

Times come from the device's global timer (ns resolution, updated about
every 32 ns on this part).  The stamps add a few stores per CTA; the
variant is a measuring instrument, not the product.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

from . import build as _build
from . import _lib

TRACE_DIR = os.path.join(_build.PKG, "_build_trace")

ROWS = (("entry", _lib.QMM_TR_ENTRY), ("pdl", _lib.QMM_TR_PDL), ("data", _lib.QMM_TR_DATA),
        ("loop end", _lib.QMM_TR_LOOP), ("all warps", _lib.QMM_TR_EPI),
        ("chunk sum", _lib.QMM_TR_RED), ("written", _lib.QMM_TR_PART),
        ("arrived", _lib.QMM_TR_ARRIVE), ("exit", _lib.QMM_TR_EXIT))


def summarize(stamps: np.ndarray, prev_exit: int | None) -> dict:
    """Quantiles (us) of each stamp of one call's CTAs, [ctas][QMM_TRACE_FIELDS]
    int64 nanoseconds, relative to ``prev_exit`` (or the call's first entry)."""
    t0 = int(stamps[:, _lib.QMM_TR_ENTRY].min()) if prev_exit is None else prev_exit
    out = {}
    for name, f in ROWS:
        col = stamps[:, f]
        col = col[col > 0]
        if col.size == 0:
            continue
        out[name] = np.quantile((col - t0) / 1e3, [0.0, 0.1, 0.5, 0.9, 1.0])
    sm = stamps[:, _lib.QMM_TR_SMID]
    per_sm = np.bincount(np.bincount(sm.astype(np.int64)))
    out["ctas_per_sm"] = {k: int(per_sm[k]) for k in range(1, per_sm.size) if per_sm[k]}
    out["last"] = int(stamps[:, _lib.QMM_TR_LAST].sum())
    return out


def check_order(stamps: np.ndarray) -> None:
    """Every CTA's stamps are in program order (the ones a call writes: the
    split-K arrival only with K splits); raises AssertionError otherwise."""
    fields = [f for _, f in ROWS]
    for b in range(stamps.shape[0]):
        seen = [int(stamps[b, f]) for f in fields if stamps[b, f] > 0]
        assert len(seen) >= len(fields) - 1, f"CTA {b}: missing stamps {stamps[b].tolist()}"
        assert seen == sorted(seen), f"CTA {b}: stamps out of order {seen}"


def format_call(s: dict) -> str:
    lines = [f"  {'stamp':10s} {'min':>7s} {'p10':>7s} {'median':>7s} {'p90':>7s} {'max':>7s}"]
    for name, _ in ROWS:
        if name in s:
            lines.append(f"  {name:10s} " + " ".join(f"{v:7.2f}" for v in s[name]))
    lines.append(f"  SMs with n CTAs of this call: {s['ctas_per_sm']}; fix-ups by the last split: {s['last']}")
    return "\n".join(lines)


def run(shape: str, Ms, copies: int, k_splits: int, shown: int, check: bool = False) -> None:
    import torch
    import speculative_decode_verification_qmm_gb300 as q
    from . import synth

    spec = synth.SHAPES[shape]
    N, K = spec["N"], spec["K"]
    mats = []
    for r in range(copies):
        w = synth.weights_cuda(N, K, 100 + r)
        if spec["fmt"] == "q4_0":
            mats.append(q.Matrix(q.QMM_FMT_Q4_0, q.quantize_q4_0(w), N, K, k_splits=k_splits))
        elif spec["fmt"] == "q8_0":
            mats.append(q.Matrix(q.QMM_FMT_Q8_0, q.quantize_q8_0(w), N, K, k_splits=k_splits))
        else:
            codes, scales = q.quantize_fp8(w)
            mats.append(q.Matrix(q.QMM_FMT_FP8_E4M3_B128, codes, N, K, scales=scales,
                                 k_splits=k_splits))
        del w
    info = mats[0].info()
    ctas = info["ctas"]
    slot = ctas * _lib.QMM_TRACE_FIELDS
    print(f"== {shape}: N={N} K={K}, {info['n_tiles']} row tiles x {info['k_splits']} K splits = "
          f"{ctas} CTAs of {info['stages_per_cta']} stages; {copies} weight copies per graph")
    for M in Ms:
        buf = torch.zeros(copies * slot, dtype=torch.int64, device="cuda")
        for r, m in enumerate(mats):
            q.qmm_debug_set_trace(m.handle, buf[r * slot:(r + 1) * slot])
        act = synth.activations_cuda(M, K, 7)
        outs = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in mats]

        def calls():
            for m, o in zip(mats, outs):
                q.qmm_verify(m.handle, act, o, M)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            calls()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls()
        for _ in range(5):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps / copies
        buf.zero_()
        g.replay()
        torch.cuda.synchronize()
        for m in mats:
            if m.sync_status() != q.QMM_OK:
                raise RuntimeError("verify call reported an error")
        st = buf.view(copies, ctas, _lib.QMM_TRACE_FIELDS).cpu().numpy()
        if check:
            for r in range(copies):
                check_order(st[r])
        print(f"-- M={M}: {us:.2f} us per call in the graph")
        gaps = []
        for r in range(1, copies):
            prev_exit = int(st[r - 1, :, _lib.QMM_TR_EXIT].max())
            s = summarize(st[r], prev_exit)
            gaps.append(s["pdl"][0])
            if r >= copies - shown:
                print(f" call {r} (times in us after call {r - 1}'s last CTA left the kernel):")
                print(format_call(s))
        print(f"  pdl release after the previous call, over calls 1..{copies - 1}: "
              f"median {np.median(gaps):.2f} us, min {np.min(gaps):.2f}, max {np.max(gaps):.2f}")
        for m in mats:
            q.qmm_debug_set_trace(m.handle, None)
    for m in mats:
        m.close()


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--shape", default="q4_attn")
    ap.add_argument("--ms", default="1,16")
    ap.add_argument("--copies", type=int, default=12)
    ap.add_argument("--k-splits", type=int, default=0)
    ap.add_argument("--shown", type=int, default=1, help="calls printed in full (the last ones)")
    ap.add_argument("--check", action="store_true",
                    help="also check that every CTA's stamps are complete and in order")
    args = ap.parse_args(argv)
    lib = _build.build(extra_flags=["-DQMM_TRACE"], out_dir=TRACE_DIR)
    _lib.load(path=lib)
    import torch
    torch.cuda.set_device(0)
    run(args.shape, [int(x) for x in args.ms.split(",")], args.copies, args.k_splits, args.shown,
        args.check)
    return 0


if __name__ == "__main__":
    sys.exit(main())
