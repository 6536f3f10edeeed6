"""Benchmark: verify-matmul weight GB/s at M = 1 / 8 / 16 drafted rows.

One "step" is one verify pass of the workload at each of M = 1, 8 and 16:
the default workload is the Q4_0 attention-projection shape (K = N = 5120),
streamed through R distinct copies of the weights whose total (R x 14.7 MB)
is well above the 129 MB L2, so every launch reads its weights from HBM.
Each M is captured as one CUDA graph of R back-to-back verify calls (the
activation pre-pass and the verify kernel per call, chained with
programmatic dependent launch) and timed with CUDA events on the launching
stream.  value = compressed weight bytes streamed per step / step time.

The default run then times the other target configurations the same way
(fewer steps) and reports each under config.per_workload with its own per-M
figures, roofline fraction, recorded DRAM traffic ratio and M=16/M=1 time
ratio: FP8 17408x5120 at M = 1/8/16, gate+up and down at M = 16 plain and
with the 32-point rotation, and the 64-layer whole-model sweep
(--no-extras skips them).

e2e is the same step through the host-buffer entry point qmm_verify_host:
every call copies its bf16 rows from pinned host memory, runs the product and
copies its fp32 result back before it returns.  e2e.graph_value is the step
as captured CUDA graphs of qmm_verify calls with torch copies around them.

Other workloads (--workload): q4_gateup, q4_down, q4_gateup_h, q4_down_h
(32-point rotation), q4_gateup_h128, q4_down_h128 (128-point rotation),
q8_mlp, q8_attn (Q8_0 at the FP8 MLP and the attention shapes),
fp8_mlp, model (64 layers x {qkv, out, gate+up, down}), q4_lmhead (the
151,936 x 5120 output head through qmm_verify_greedy: the verify product plus
the argmax and accepted-prefix step), fp8_prefill (the prompt-shaped FP8 GEMM,
qmm_prefill, at M = 512 / 2048 / 8192 rows on the FP8 MLP weights; its own
metric, TFLOP/s against the dense f16/bf16 tensor peak).

Multi-GPU (--gpus N under torchrun): the path shards into independent
problems, so every rank runs its own replica of the workload with no
collective on the data path; ranks meet only at the timing barrier and the
max-over-ranks reduction of the elapsed time ("scaling": "weak").  --shard
instead splits each matrix by rows over the ranks (qmm_create_rows) and
all-gathers every call's [M, N/G] output with NCCL ("scaling": "strong").

--impl reference times the CPU oracle (the plain fp64 triple loop) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024

WORKLOADS = {
    # name: (synth shape, hadamard, Ms)
    "q4_attn": ("q4_attn", False, (1, 8, 16)),
    "q4_gateup": ("q4_gateup", False, (16,)),
    "q4_down": ("q4_down", False, (16,)),
    "q4_gateup_h": ("q4_gateup", True, (16,)),
    "q4_down_h": ("q4_down", True, (16,)),
    "fp8_mlp": ("fp8_mlp", False, (1, 8, 16)),
    # the 128-point rotation of the activations (weights rotated offline to match)
    "q4_gateup_h128": ("q4_gateup", 128, (16,)),
    "q4_down_h128": ("q4_down", 128, (16,)),
    # Q8_0 (fp16 scale per 32 elements, int8 codes)
    "q8_mlp": ("q8_mlp", False, (1, 8, 16)),
    "q8_attn": ("q8_attn", False, (1, 8, 16)),
    # output head with the greedy acceptance step (qmm_verify_greedy)
    "q4_lmhead": ("q4_lmhead", False, (1, 8, 16)),
}


# ---------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Largest value over all ranks (x itself when there is one rank)."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int, device=None) -> float:
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def gather_shards(part, N: int, ws: int, align: int = 1):
    """All-gather the [M, N_g] outputs of the ranks' row shards into [M, N]:
    rank g computed columns shard_rows(N, ws, g, align) of the product.  The
    shards are padded to the widest one for the collective.  One rank: the
    part itself."""
    if ws <= 1:
        return part
    import torch
    import torch.distributed as dist
    from speculative_decode_verification_qmm_gb300 import shard_rows
    M = part.shape[0]
    sizes = [shard_rows(N, ws, g, align) for g in range(ws)]
    width = max(b - a for a, b in sizes)
    buf = torch.zeros((M, width), dtype=part.dtype, device=part.device)
    buf[:, :part.shape[1]] = part
    outs = [torch.empty_like(buf) for _ in range(ws)]
    dist.all_gather(outs, buf)
    return torch.cat([o[:, :b - a] for o, (a, b) in zip(outs, sizes)], dim=1)


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)
        return False

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers
def measured_peak_gbs():
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decode_verification_qmm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the verify kernel from the committed ncu summary,
    or None when it was taken on other kernel sources."""
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f)
    except Exception:
        return None
    ent = rec.get(workload)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- GPU arm
KERNEL_FLAGS = {"auto": {}, "mma": {}, "tc": {"tcgen05": True}, "simt": {"simt": True}}


def build_matrices(q, synth, shape_name, hadamard, copies, torch, seed_base=0, splits=0,
                   kernel="auto", rows=None):
    """`copies` handles of the named shape (distinct seeded weights); rows =
    (n_begin, n_end): handles over those rows only (a shard of the split)."""
    spec = synth.SHAPES[shape_name]
    kf = KERNEL_FLAGS[kernel]
    N, K = spec["N"], spec["K"]
    mats = []
    for r in range(copies):
        w = synth.weights_cuda(N, K, spec["seed"] + 7919 * r + seed_base)
        if spec["fmt"] == "q4_0":
            blocks = q.quantize_q4_0(w, hadamard=hadamard)
            del w
            mats.append(q.Matrix(q.QMM_FMT_Q4_0, blocks, N, K, hadamard=hadamard, k_splits=splits,
                                 rows=rows, **kf))
            del blocks
        elif spec["fmt"] == "q8_0":
            blocks = q.quantize_q8_0(w, hadamard=hadamard)
            del w
            mats.append(q.Matrix(q.QMM_FMT_Q8_0, blocks, N, K, hadamard=hadamard, k_splits=splits,
                                 rows=rows))
            del blocks
        else:
            codes, scales = q.quantize_fp8(w, hadamard=hadamard)
            del w
            mats.append(q.Matrix(q.QMM_FMT_FP8_E4M3_B128, codes, N, K, scales=scales,
                                 hadamard=hadamard, k_splits=splits, rows=rows))
            del codes, scales
    torch.cuda.synchronize()
    return mats, spec


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm once outside the graph
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def setup_workload(q, synth, torch, dev, args, workload):
    """Build the handles, activations and outputs of one workload (untimed).
    Returns a dict: groups [(M, [(mat, act, out)])], desc, kernel, dtype,
    greedy buffers."""
    groups = []  # list of (M, [(mat, act, out)])
    if workload == "model":
        acts = {}
        mats = []
        for layer in range(synth.MODEL_LAYERS):
            for j, (name, N, K) in enumerate(synth.MODEL_LAYER):
                w = synth.weights_cuda(N, K, 4 * layer + j)
                blocks = q.quantize_q4_0(w)
                del w
                mats.append(q.Matrix(q.QMM_FMT_Q4_0, blocks, N, K, k_splits=args.splits,
                                     **KERNEL_FLAGS[args.kernel]))
                del blocks
        torch.cuda.synchronize()
        for M in synth.MODEL_MS:
            items = []
            # one contiguous output buffer per M (the results read back per step)
            flat = torch.empty(sum(M * m.N for m in mats), dtype=torch.float32, device=dev)
            off = 0
            for m in mats:
                key = (M, m.K)
                if key not in acts:
                    acts[key] = synth.activations_cuda(M, m.K, 10_000 + m.K, outliers=False)
                out = flat[off:off + M * m.N].view(M, m.N)
                off += M * m.N
                items.append((m, acts[key], out))
            groups.append((M, items))
        per_copy = sum(m.info()["weight_bytes"] for m in mats)
        desc = (f"whole-model Q4_0 sweep: {synth.MODEL_LAYERS} layers x "
                f"{{qkv 10240x5120, out 5120x5120, gate+up 34816x5120, down 5120x17408}}, "
                f"{per_copy / 2**30:.2f} GiB compressed per pass, one pass per M")
        kernel, dtype, l2 = "verify_kernel<0", "bf16", "inputs larger than L2 (11.6 GiB per pass)"
    else:
        shape_name, hadamard, Ms = WORKLOADS[workload]
        if getattr(args, "ms", None) and workload == args.workload:
            Ms = tuple(int(x) for x in args.ms.split(","))
        spec = synth.SHAPES[shape_name]
        N, K = spec["N"], spec["K"]
        one = {"q4_0": N * K // 32 * 18, "q8_0": N * K // 32 * 34}.get(
            spec["fmt"], N * K + 4 * (N // 128) * (K // 128))
        copies = args.copies or max(2, -(-4 * L2_BYTES // one))
        mats, spec = build_matrices(q, synth, shape_name, hadamard, copies, torch,
                                    splits=args.splits, kernel=args.kernel)
        for M in Ms:
            act = synth.activations_cuda(M, K, spec["seed"] + 1000, outliers=spec["outliers"])
            outbuf = torch.empty((len(mats), M, N), dtype=torch.float32, device=dev)
            items = [(m, act, outbuf[i]) for i, m in enumerate(mats)]
            groups.append((M, items))
        fmt_name = {"q4_0": "Q4_0", "q8_0": "Q8_0"}.get(spec["fmt"], "FP8 E4M3 128x128")
        rot = f" Hadamard{32 if hadamard is True else hadamard}" if hadamard else ""
        desc = (f"{fmt_name} verify K={K} N={N}{rot}, "
                f"M={'/'.join(map(str, Ms))}, {copies} distinct weight copies "
                f"({copies * one / 1e6:.0f} MB, > 4x L2) cycled")
        kernel = "verify_kernel<" + {"q4_0": "0", "q8_0": "2"}.get(spec["fmt"], "1")
        dtype = "f16" if (hadamard or spec["fmt"] != "q4_0") else "bf16"
        l2 = "inputs larger than L2 (distinct weight copies)"
    # the greedy workload: per call the block's tokens (shared per M) and its
    # argmax [M] and accept [2] outputs, in one int32 buffer per M
    greedy = workload == "q4_lmhead"
    gbufs = {}
    if greedy:
        for M, items in groups:
            tok = torch.zeros(M, dtype=torch.int32, device=dev)
            res = torch.zeros((len(items), M + 2), dtype=torch.int32, device=dev)
            gbufs[M] = (tok, res)
    return {"name": workload, "groups": groups, "desc": desc, "kernel": kernel, "dtype": dtype,
            "l2": l2, "greedy": greedy, "gbufs": gbufs}


def make_call(q, W):
    greedy, gbufs = W["greedy"], W["gbufs"]

    def call(m, act, out, j=0):
        M = act.shape[0]
        if greedy:
            tok, res = gbufs[M]
            q.qmm_verify_greedy(m.handle, act, out, M, tok, res[j, :M], res[j, M:])
        else:
            q.qmm_verify(m.handle, act, out, M)
    return call


def time_workload(q, torch, W, steps, warmup, ws, local, dev, peak):
    """Capture one CUDA graph per M (every call of the group back to back) and
    time `steps` replays of all of them after `warmup`, with CUDA events on the
    launching stream; clocks sampled meanwhile.  Returns the per-M breakdown
    and the step totals."""
    groups = W["groups"]
    call = make_call(q, W)

    def run_group(items):
        for j, (m, act, out) in enumerate(items):
            call(m, act, out, j)

    graphs = [(M, capture(torch, lambda it=items: run_group(it)), items) for M, items in groups]
    calls_per_step = sum(len(items) for _, items in groups)
    rot_flags = q.QMM_FLAG_HADAMARD32 | q.QMM_FLAG_HADAMARD64 | q.QMM_FLAG_HADAMARD128
    # kernels per call: the verify kernel, plus the activation pre-pass on the f16 paths
    launches_per_step = sum(sum(1 + int(bool(m.info()["flags"] & rot_flags)
                                        or m.fmt != q.QMM_FMT_Q4_0)
                                for m, _, _ in items) for _, items in groups)
    bytes_per_step = sum(sum(m.info()["weight_bytes"] for m, _, _ in items) for _, items in groups)

    clocks = ClockSampler(local).__enter__()
    time.sleep(0.5)
    for _ in range(warmup):
        for _, g, _ in graphs:
            g.replay()
    torch.cuda.synchronize()
    for _, items in groups:
        for m, _, _ in items:
            rc = m.sync_status()
            if rc != q.QMM_OK:
                raise RuntimeError(f"device status after warmup: {q.qmm_strerror(rc)}")

    stream = torch.cuda.current_stream()
    barrier(ws)
    torch.cuda.synchronize()
    n_before = len(clocks.lines)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    marks = []
    ev0.record(stream)
    for _ in range(steps):
        for M, g, _ in graphs:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            marks.append((M, a, b))
    ev1.record(stream)
    torch.cuda.synchronize()
    time.sleep(0.25)
    clocks.__exit__(None, None, None)
    clocks.lines = clocks.lines[max(0, n_before - 2):]
    barrier(ws)
    total_ms = ev0.elapsed_time(ev1)
    per_m = {M: 0.0 for M, _, _ in graphs}
    per_m_samples = {M: [] for M, _, _ in graphs}
    for M, a, b in marks:
        dt = a.elapsed_time(b)
        per_m[M] += dt
        per_m_samples[M].append(dt)
    total_ms = max_over_ranks(total_ms, ws, dev)
    for _, items in groups:
        for m, _, _ in items:
            rc = m.sync_status()
            if rc != q.QMM_OK:
                raise RuntimeError(f"device status after timing: {q.qmm_strerror(rc)}")

    breakdown = {}
    for M, _, items in graphs:
        b = sum(m.info()["weight_bytes"] for m, _, _ in items)
        t = per_m[M] / steps
        xs = sorted(per_m_samples[M])
        qt = lambda f: xs[min(len(xs) - 1, int(round(f * (len(xs) - 1))))]
        med = statistics.median(xs)
        # one verify pass = one call on one matrix (the model workload: the
        # whole 64-layer sweep)
        passes = 1 if W["name"] == "model" else len(items)
        breakdown[str(M)] = {"ms": round(t, 5), "GBps": round(b / (t * 1e-3) / 1e9, 1),
                             "pct_of_peak": round(100 * b / (t * 1e-3) / 1e9 / peak, 1),
                             "ms_median": round(med, 5), "ms_p10": round(qt(0.1), 5),
                             "ms_p90": round(qt(0.9), 5),
                             "GBps_median": round(b / (med * 1e-3) / 1e9, 1),
                             "verify_passes_per_s": round(passes / (med * 1e-3), 1),
                             "us_per_call": round(t * 1e3 / len(items), 3)}
    return {"graphs": graphs, "per_M": breakdown, "total_ms": total_ms,
            "ms_per_step": total_ms / steps, "calls_per_step": calls_per_step,
            "launches_per_step": launches_per_step, "bytes_per_step": bytes_per_step,
            "clocks": clocks.summary()}


def m16_over_m1(breakdown):
    if "16" in breakdown and "1" in breakdown:
        return round(breakdown["16"]["ms"] / breakdown["1"]["ms"], 3)
    return None


# The other target configurations, timed after the headline one in the default
# run and reported under config.per_workload: FP8 at M = 1/8/16, gate+up and
# down at M = 16 plain and with the 32-point rotation, and the 64-layer sweep.
EXTRA_WORKLOADS = ("fp8_mlp", "q4_gateup", "q4_down", "q4_gateup_h", "q4_down_h", "model")


def extra_entry(q, torch, synth, dev, args, name, ws, local, peak):
    W = setup_workload(q, synth, torch, dev, args, name)
    steps = max(1, min(args.steps, 10))
    T = time_workload(q, torch, W, steps, 3, ws, local, dev, peak)
    achieved = (T["bytes_per_step"] / T["calls_per_step"]) / (T["ms_per_step"] * 1e-3 /
                                                               T["calls_per_step"]) / 1e9
    first = W["groups"][0][1][0][0]
    traffic = recorded_traffic(name)
    per_launch = T["bytes_per_step"] / T["calls_per_step"]
    entry = {"workload": W["desc"], "dtype": W["dtype"], "l2": W["l2"], "steps": steps,
             "kernel": W["kernel"],
             "plan": {k: first.info()[k] for k in
                      ("n_tiles", "k_splits", "ctas", "stages_per_cta", "pipeline_depth")},
             "per_M": T["per_M"], "GBps": round(achieved, 1),
             "roofline_frac": round(achieved / peak, 3),
             "traffic_ratio": (round(traffic / per_launch, 4) if traffic and name != "model"
                               else None),
             "m16_over_m1_time": m16_over_m1(T["per_M"]), "clocks": T["clocks"]}
    del T, W
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_gpu(args, ws, rank, local):
    import torch
    import speculative_decode_verification_qmm_gb300 as q
    from speculative_decode_verification_qmm_gb300 import synth

    torch.cuda.set_device(local)
    q.load()
    dev = torch.device("cuda", local)
    peak, peak_kind = measured_peak_gbs()

    W = setup_workload(q, synth, torch, dev, args, args.workload)
    groups = W["groups"]
    call = make_call(q, W)
    T = time_workload(q, torch, W, args.steps, args.warmup, ws, local, dev, peak)
    m_breakdown = T["per_M"]
    ms_per_step = T["ms_per_step"]
    total_bytes = sum_over_ranks(T["bytes_per_step"] * args.steps, ws, dev)
    value = total_bytes / (T["total_ms"] * 1e-3) / 1e9
    per_launch_bytes = T["bytes_per_step"] / T["calls_per_step"]
    avg_launch_s = (ms_per_step * 1e-3) / T["calls_per_step"]
    achieved = per_launch_bytes / avg_launch_s / 1e9
    stream = torch.cuda.current_stream()

    # ---- one isolated call per M after an L2 flush (a 2 x L2 buffer written
    # first; the events bracket the call only): no neighbour to overlap with
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    for M, _, items in T["graphs"]:
        m0, act0, out0 = items[0]
        iso = []
        for _ in range(5):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(m0, act0, out0)
            b.record(stream)
            torch.cuda.synchronize()
            iso.append(a.elapsed_time(b) * 1e3)
        m_breakdown[str(M)]["isolated_call_us"] = round(statistics.median(iso), 2)
    del flush

    # ---- end to end through the public host-buffer call: per step, every call
    # of the step goes through qmm_verify_host with pinned host buffers at both
    # ends (the call copies its activation rows to the device, runs the verify
    # product and copies its fp32 result back before returning).  The same step
    # run as the captured CUDA graphs with torch copies around them is reported
    # beside it (graph_value).
    e2e = None
    if not args.no_e2e:
        host_in = {}
        plan = []  # per call: (mat, pinned act, pinned out)
        for M, items in groups:
            for m, act, out in items:
                key = act.data_ptr()
                if key not in host_in:
                    host_in[key] = act.cpu().pin_memory()
                plan.append((m, host_in[key], torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()))
        h2d = sum(hi.numel() * 2 for _, hi, _ in plan)
        d2h = sum(ho.numel() * 4 for _, _, ho in plan)
        greedy = W["greedy"]

        def host_step():
            for m, hi, ho in plan:
                q.qmm_verify_host(m.handle, hi, ho, hi.shape[0])

        e2e_steps = max(1, min(args.steps, 5))

        def wall(fn):
            fn()  # warm
            barrier(ws)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(e2e_steps):
                fn()
            return max_over_ranks(time.perf_counter() - t0, ws, dev)

        e2e_bytes = sum_over_ranks(T["bytes_per_step"] * e2e_steps, ws, dev)
        e2e = {"unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps}
        if not greedy:
            el = wall(host_step)
            e2e["value"] = round(e2e_bytes / el / 1e9, 1)
            e2e["api"] = ("qmm_verify_host (host buffers): every call of the step copies its "
                          "bf16 rows from pinned host memory, runs the verify product and copies "
                          "its fp32 result back to pinned host memory before returning")
        # the graph form: per M, the activations copied in, the captured graph
        # replayed, every output copied back; one synchronize per step
        gplan = []
        for M, items in groups:
            ins = []
            for _, act, _ in items:
                if all(act.data_ptr() != d.data_ptr() for d, _ in ins):
                    ins.append((act, act.cpu().pin_memory()))
            if greedy:  # the step's result is the decision: argmax and accepted count per call
                dev_out = W["gbufs"][M][1].view(-1)
                gplan.append((ins, dev_out, torch.empty(dev_out.numel(), dtype=torch.int32).pin_memory()))
                continue
            base = items[0][2]
            n_out = sum(out.numel() for _, _, out in items)
            dev_out = torch.as_strided(base, (n_out,), (1,))  # the contiguous buffer behind the views
            gplan.append((ins, dev_out, torch.empty(n_out, dtype=torch.float32).pin_memory()))
        graph_of = {M: g for M, g, _ in T["graphs"]}

        def graph_step():
            for (M, _), (ins, dev_out, host_out) in zip(groups, gplan):
                for d, hi in ins:
                    d.copy_(hi, non_blocking=True)
                graph_of[M].replay()
                host_out.copy_(dev_out, non_blocking=True)
            torch.cuda.synchronize()

        elg = wall(graph_step)
        e2e["graph_value"] = round(e2e_bytes / elg / 1e9, 1)
        e2e["graph_api"] = ("qmm_verify captured in CUDA graphs: per step the activations are "
                            "copied from pinned host memory, the graphs replayed, all outputs "
                            "copied back to pinned host memory, one synchronize")
        if greedy:
            e2e["value"] = e2e["graph_value"]
            e2e["h2d_bytes_per_step"] = sum(hi.numel() * 2 for ins, _, _ in gplan for _, hi in ins)
            e2e["d2h_bytes_per_step"] = sum(ho.numel() * 4 for _, _, ho in gplan)
            e2e["api"] = e2e["graph_api"] + " (the step's result is the decision: argmax and k)"

    traffic = recorded_traffic(args.workload)
    first = groups[0][1][0][0]
    per_workload = {}
    gpu_launches = T["launches_per_step"] * args.steps
    main_clocks = T["clocks"]
    del T
    if args.workload == "q4_attn" and not args.no_extras:
        for name in EXTRA_WORKLOADS:
            per_workload[name] = extra_entry(q, torch, synth, dev, args, name, ws, local, peak)
    line = {
        "metric": "verify-matmul weight GB/s (% of GB300 HBM peak) at M=1/8/16 draft rows",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": W["dtype"],
        "data": "synthetic (seeded N(0,0.02) weights quantized on the device, bf16 N(0,1) "
                "activations with 0.1% x20 outlier channels)",
        "config": {"workload": W["desc"], "l2": W["l2"],
                   "plan": {k: first.info()[k] for k in
                            ("n_tiles", "k_splits", "ctas", "stages_per_cta", "pipeline_depth")},
                   "parallelism": f"replicas x{ws}", "per_M": m_breakdown,
                   "pct_of_peak": round(100 * value / ws / peak, 1),
                   "m16_over_m1_time": m16_over_m1(m_breakdown),
                   "per_workload": per_workload or None},
        "roofline": {"bound": "hbm", "kernel": W["kernel"], "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} (STREAM-style copy)", "unit": "GB/s",
                     "frac": round(achieved / peak, 3),
                     "traffic": traffic, "algorithmic_bytes_per_launch": int(per_launch_bytes),
                     "note": "verify-kernel launch duration averaged over the timed region "
                             "(back-to-back calls; any activation pre-pass included)"},
        "clocks": main_clocks,
        "e2e": e2e,
        "gpu_launches": gpu_launches,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
    return line, rank


# ---------------------------------------------------------------- row split
def run_shard(args, ws, rank, local):
    """--shard: the matrix is split by rows over the ranks (rank g holds rows
    [g N / G, (g + 1) N / G), multiples of 128 for FP8) and every verify call
    is followed by the all-gather of the [M, N / G] fp32 parts into the full
    [M, N] output (NCCL), the one exchange the split needs.  One step: at each
    M, every weight copy's call and gather.  value = compressed bytes of the
    whole matrices per step / step time (max over ranks); "scaling": "strong"
    (the total work is fixed as the ranks grow)."""
    import torch
    import speculative_decode_verification_qmm_gb300 as q
    from speculative_decode_verification_qmm_gb300 import synth

    if args.workload not in WORKLOADS or args.workload == "q4_lmhead":
        raise SystemExit("--shard takes one of the single-matrix verify workloads")
    torch.cuda.set_device(local)
    q.load()
    dev = torch.device("cuda", local)
    peak, peak_kind = measured_peak_gbs()
    shape_name, hadamard, Ms = WORKLOADS[args.workload]
    spec = synth.SHAPES[shape_name]
    N, K = spec["N"], spec["K"]
    align = 128 if spec["fmt"] == "fp8" else 1
    rows = q.shard_rows(N, ws, rank, align)
    one = {"q4_0": N * K // 32 * 18, "q8_0": N * K // 32 * 34}.get(
        spec["fmt"], N * K + 4 * (N // 128) * (K // 128))
    part_bytes = one * (rows[1] - rows[0]) / N
    copies = args.copies or max(2, int(-(-4 * L2_BYTES // part_bytes)))
    mats, _ = build_matrices(q, synth, shape_name, hadamard, copies, torch, splits=args.splits,
                             kernel=args.kernel, rows=rows)
    acts = {M: synth.activations_cuda(M, K, spec["seed"] + 1000, outliers=spec["outliers"])
            for M in Ms}
    outs = {M: [torch.empty((M, rows[1] - rows[0]), dtype=torch.float32, device=dev) for _ in mats]
            for M in Ms}

    def step_m(M):
        for m, o in zip(mats, outs[M]):
            q.qmm_verify(m.handle, acts[M], o, M)
            gather_shards(o, N, ws, align)

    clocks = ClockSampler(local).__enter__()
    time.sleep(0.5)
    for _ in range(args.warmup):
        for M in Ms:
            step_m(M)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    n_before = len(clocks.lines)
    stream = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per_m = {M: 0.0 for M in Ms}
    ev0.record(stream)
    for _ in range(args.steps):
        for M in Ms:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step_m(M)
            b.record(stream)
            torch.cuda.synchronize()
            per_m[M] += a.elapsed_time(b)
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.__exit__(None, None, None)
    clocks.lines = clocks.lines[max(0, n_before - 2):]
    barrier(ws)
    for m in mats:
        if m.sync_status() != q.QMM_OK:
            raise RuntimeError("device status after timing")
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), ws, dev)
    full_bytes = one * copies * len(Ms) * args.steps
    value = full_bytes / (total_ms * 1e-3) / 1e9
    per_M = {}
    for M in Ms:
        t = max_over_ranks(per_m[M], ws, dev) / args.steps
        per_M[str(M)] = {"ms": round(t, 5), "GBps": round(one * copies / (t * 1e-3) / 1e9, 1),
                         "us_per_call_and_gather": round(t * 1e3 / copies, 3)}
    line = {
        "metric": "verify-matmul weight GB/s (% of GB300 HBM peak) at M=1/8/16 draft rows",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
        "dtype": "f16" if (hadamard or spec["fmt"] != "q4_0") else "bf16",
        "data": "synthetic (seeded N(0,0.02) weights quantized on the device, bf16 N(0,1) "
                "activations with 0.1% x20 outlier channels)",
        "config": {"workload": f"{args.workload} split by rows over {ws} GPU(s), rows "
                               f"{rows[0]}..{rows[1]} on rank {rank}, {copies} weight copies, "
                               "NCCL all-gather of every call's [M, N/G] output",
                   "l2": "inputs larger than L2 (distinct weight copies)",
                   "parallelism": f"row split x{ws}", "per_M": per_M,
                   "pct_of_peak": round(100 * value / ws / peak, 1)},
        "roofline": None,
        "clocks": clocks.summary(),
        "e2e": None,
        "gpu_launches": copies * len(Ms) * args.steps * (1 + int(bool(hadamard) or spec["fmt"] != "q4_0")),
    }
    return line, rank


# ---------------------------------------------------------------- prefill GEMM
PREFILL_METRIC = "prefill FP8 GEMM TFLOP/s (% of GB300 dense bf16/f16 peak) at M=512/2048/8192 prompt rows"
PREFILL_MS = (512, 2048, 8192)


def measured_peak_tflops():
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_prefill(args, ws, rank, local):
    """The prefill-shaped block-scaled FP8 GEMM (qmm_prefill) on the FP8 MLP
    weights (N = 17408, K = 5120): one step = one call at each M of
    PREFILL_MS.  Every timed call is preceded by an L2 flush (a 2 x L2 buffer
    written between the events), so each call reads its operands from HBM."""
    import torch
    import speculative_decode_verification_qmm_gb300 as q
    from speculative_decode_verification_qmm_gb300 import synth

    torch.cuda.set_device(local)
    q.load()
    dev = torch.device("cuda", local)
    spec = synth.SHAPES["fp8_mlp"]
    N, K = spec["N"], spec["K"]
    w = synth.weights_cuda(N, K, spec["seed"])
    codes, scales = q.quantize_fp8(w)
    del w
    mat = q.Matrix(q.QMM_FMT_FP8_E4M3_B128, codes, N, K, scales=scales)
    del codes, scales
    Ms = PREFILL_MS
    acts = {M: synth.activations_cuda(M, K, spec["seed"] + 1000 + M, outliers=True) for M in Ms}
    outs = {M: torch.empty((M, N), dtype=torch.float32, device=dev) for M in Ms}
    ws_bytes = max(q.qmm_prefill_workspace(mat.handle, M) for M in Ms)
    wsbuf = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call(M, act=None, out=None):
        q.qmm_prefill(mat.handle, acts[M] if act is None else act, outs[M] if out is None else out,
                      M, wsbuf)

    clocks = ClockSampler(local).__enter__()
    time.sleep(0.5)
    for _ in range(args.warmup):
        for M in Ms:
            call(M)
    torch.cuda.synchronize()
    if mat.sync_status() != q.QMM_OK:
        raise RuntimeError("device status after warmup")
    barrier(ws)
    torch.cuda.synchronize()
    n_before = len(clocks.lines)
    marks = []
    for _ in range(args.steps):
        for M in Ms:
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(M)
            b.record(stream)
            marks.append((M, a, b))
    torch.cuda.synchronize()
    time.sleep(0.25)
    clocks.__exit__(None, None, None)
    clocks.lines = clocks.lines[max(0, n_before - 2):]
    barrier(ws)
    if mat.sync_status() != q.QMM_OK:
        raise RuntimeError("device status after timing")
    per_m = {M: [] for M in Ms}
    for M, a, b in marks:
        per_m[M].append(a.elapsed_time(b))
    step_ms = sum(sum(v) for v in per_m.values()) / args.steps
    step_ms = max_over_ranks(step_ms, ws, dev)
    flops_per_step = sum(2.0 * M * N * K for M in Ms)
    total_flops = sum_over_ranks(flops_per_step * args.steps, ws, dev)
    value = total_flops / (step_ms * args.steps * 1e-3) / 1e12
    peak, peak_kind = measured_peak_tflops()
    breakdown = {}
    for M in Ms:
        xs = sorted(per_m[M])
        med = statistics.median(xs)
        qt = lambda f: xs[min(len(xs) - 1, int(round(f * (len(xs) - 1))))]
        breakdown[str(M)] = {"ms_median": round(med, 4), "ms_p10": round(qt(0.1), 4),
                             "ms_p90": round(qt(0.9), 4),
                             "TFLOPs_median": round(2.0 * M * N * K / (med * 1e-3) / 1e12, 1)}
    # the dominant launch: the M = 8192 call (pre-pass + GEMM), events on its stream
    big = Ms[-1]
    big_ms = statistics.median(per_m[big])
    achieved = 2.0 * big * N * K / (big_ms * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        host_in = {M: acts[M].cpu().pin_memory() for M in Ms}
        host_out = {M: torch.empty((M, N), dtype=torch.float32).pin_memory() for M in Ms}
        h2d = sum(M * K * 2 for M in Ms)
        d2h = sum(M * N * 4 for M in Ms)

        def e2e_step():
            for M in Ms:
                acts[M].copy_(host_in[M], non_blocking=True)
                call(M)
                host_out[M].copy_(outs[M], non_blocking=True)
            torch.cuda.synchronize()

        e2e_steps = max(1, min(args.steps, 5))
        e2e_step()
        barrier(ws)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        el = max_over_ranks(time.perf_counter() - t0, ws, dev)
        e2e = {"value": round(sum_over_ranks(flops_per_step * e2e_steps, ws, dev) / el / 1e12, 1),
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps,
               "api": "qmm_prefill (device buffers): per step and M the bf16 rows are copied from "
                      "pinned host memory, the call is launched, the fp32 result is copied back "
                      "to pinned host memory; one synchronize per step"}
    traffic = recorded_traffic("fp8_prefill")
    line = {
        "metric": PREFILL_METRIC,
        "value": round(value, 1),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded N(0,0.02) weights quantized to E4M3 with 128x128 fp32 scales on "
                "the device, bf16 N(0,1) activations with 0.1% x20 outlier channels)",
        "config": {"workload": f"FP8 E4M3 128x128 prefill GEMM K={K} N={N}, "
                               f"M={'/'.join(map(str, Ms))}",
                   "l2": "L2 flushed (2 x L2 buffer written) before every timed call",
                   "parallelism": f"replicas x{ws}", "per_M": breakdown,
                   "pct_of_peak": round(100 * value / ws / peak, 1)},
        "roofline": {"bound": "tensor", "kernel": "prefill_fp8_kernel", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} (cuBLAS bf16 burst; f16 has the same "
                                                "nominal dense rate)", "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 3), "traffic": traffic,
                     "algorithmic_flops_per_launch": 2.0 * big * N * K,
                     "note": f"M = {big} call (activation pre-pass + GEMM), median CUDA-event "
                             "duration after an L2 flush"},
        "clocks": clocks.summary(),
        "e2e": e2e,
        "gpu_launches": 2 * len(Ms) * args.steps,
    }
    if rank == 0 and not args.no_cpu_baseline:
        v, cores, sample = prefill_oracle_rate(args.cpu_budget)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores,
                                "kind": "oracle", "sample": sample}
    mat.close()
    return line, rank


def prefill_oracle_rate(budget_s: float):
    """The oracle's rate (TFLOP/s) on a bounded sample of the prefill workload:
    256 prompt rows against 256 of the 17408 weight rows, K = 5120."""
    import oracle as O
    from speculative_decode_verification_qmm_gb300 import synth
    spec = synth.SHAPES["fp8_mlp"]
    K, rows_n, M = spec["K"], 256, 256
    w = synth.weights(rows_n, K, spec["seed"])
    codes, sc = O.fp8_quantize(w)
    a = synth.activations(M, K, spec["seed"] + 1000, outliers=True)
    flops, t_total, reps = 0.0, 0.0, 0
    while t_total < budget_s or reps == 0:
        t0 = time.perf_counter()
        O.verify_rows(O.FMT_FP8, codes, sc, rows_n, K, a)
        t_total += time.perf_counter() - t0
        flops += 2.0 * M * rows_n * K
        reps += 1
    sample = (f"{M} prompt rows x {rows_n} of {spec['N']} weight rows x K={K}, {reps} pass(es), "
              f"{t_total:.1f} s")
    return flops / t_total / 1e12, O.num_threads(), sample


# ---------------------------------------------------------------- CPU oracle arm
def oracle_sample_rate(budget_s: float, workload: str):
    """Time the oracle on a bounded row sample of the workload at every M of the
    step; return (GB/s of weight bytes processed, threads, sample description)."""
    import numpy as np
    import oracle as O
    from speculative_decode_verification_qmm_gb300 import synth

    if workload == "model":
        shape_name, hadamard, Ms = "q4_attn", False, synth.MODEL_MS
    else:
        shape_name, hadamard, Ms = WORKLOADS[workload]
    spec = synth.SHAPES[shape_name]
    N, K = spec["N"], spec["K"]
    rows_n = min(N, 512)
    w = synth.weights(rows_n, K, spec["seed"])
    if hadamard:  # the offline rotation of the weights (32-, 64- or 128-point)
        w = O.rotate_weights_f32(w, 32 if hadamard is True else int(hadamard))
    if spec["fmt"] == "q4_0":
        wb = O.q4_0_quantize(w)
        sc, fmt, row_bytes = None, O.FMT_Q4_0, K // 32 * 18
    elif spec["fmt"] == "q8_0":
        wb = O.q8_0_quantize(w)
        sc, fmt, row_bytes = None, O.FMT_Q8_0, K // 32 * 34
    else:
        wb, sc = O.fp8_quantize(w)
        fmt, row_bytes = O.FMT_FP8, K
    acts = {M: synth.activations(M, K, spec["seed"] + 1000, outliers=spec["outliers"],
                                 outlier_seed=spec["seed"] + 2000) for M in Ms}
    done_bytes, t_total, reps = 0, 0.0, 0
    while t_total < budget_s or reps == 0:
        for M in Ms:
            t0 = time.perf_counter()
            O.verify_rows(fmt, wb, sc, rows_n, K, acts[M], hadamard=hadamard)
            t_total += time.perf_counter() - t0
            done_bytes += rows_n * row_bytes
        reps += 1
    sample = (f"{rows_n} of {N} weight rows x K={K}, M={'/'.join(map(str, Ms))}, "
              f"{reps} pass(es), {t_total:.1f} s")
    return done_bytes / t_total / 1e9, O.num_threads(), sample


def cpu_baseline(args):
    """The oracle on all host cores (the reported baseline) and, beside it, on
    one thread with a shorter budget."""
    import oracle as O
    v, cores, sample = oracle_sample_rate(args.cpu_budget, args.workload)
    line = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": sample}
    try:
        O.set_num_threads(1)
        v1, _, sample1 = oracle_sample_rate(min(3.0, args.cpu_budget / 3), args.workload)
        line["single_thread"] = {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                                 "sample": sample1}
    finally:
        O.set_num_threads(cores)
    return line


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    if args.workload == "fp8_prefill":
        for _ in range(args.warmup):
            prefill_oracle_rate(0.0)
        vals = []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            v, cores, sample = prefill_oracle_rate(max(1.0, args.cpu_budget / max(1, args.steps)))
            vals.append(v)
        elapsed = time.perf_counter() - t0
        value = statistics.median(vals)
        return {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6),
                "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(elapsed / args.steps * 1e3, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded, same recipe as the GPU arm)",
                "config": {"workload": "fp8_prefill (CPU oracle on a bounded sample)",
                           "parallelism": "host cores"},
                "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
    for _ in range(args.warmup):
        oracle_sample_rate(0.0, args.workload)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, cores, sample = oracle_sample_rate(max(1.0, args.cpu_budget / max(1, args.steps)),
                                              args.workload)
        vals.append(v)
    elapsed = time.perf_counter() - t0
    value = statistics.median(vals)
    return {
        "impl": "reference",
        "metric": "verify-matmul weight GB/s (% of GB300 HBM peak) at M=1/8/16 draft rows",
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded, same recipe as the GPU arm)",
        "config": {"workload": f"{args.workload} (CPU oracle on a bounded row sample)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=sorted(list(WORKLOADS) + ["model", "fp8_prefill"]),
                    default="q4_attn")
    ap.add_argument("--copies", type=int, default=0, help="distinct weight copies (0: >= 4x L2)")
    ap.add_argument("--splits", type=int, default=0, help="force the K split count (0: planner)")
    ap.add_argument("--kernel", choices=sorted(KERNEL_FLAGS), default="auto",
                    help="verify kernel: auto (library default: mma.sync), tc (tcgen05, bf16 "
                         "Q4_0 only), mma (mma.sync), simt (CUDA cores, Q4_0 only)")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="default workload only: skip the other target configurations")
    ap.add_argument("--ms", default="",
                    help="comma-separated drafted-row counts to time instead of the workload's "
                         "own (for example 1,8,16 on the MLP shapes)")
    ap.add_argument("--shard", action="store_true",
                    help="split each matrix by rows over the ranks and all-gather every "
                         "call's output (strong scaling) instead of running replicas")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    ws, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0

    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.workload == "fp8_prefill":
        line, rank = run_prefill(args, ws, rank, local)
    elif args.shard:
        line, rank = run_shard(args, ws, rank, local)
    else:
        line, rank = run_gpu(args, ws, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
