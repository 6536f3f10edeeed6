"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``check_*`` function raises AssertionError when the oracle disagrees with
a closed form, a library routine, an exact rational computation, a hand-worked
golden value or a mathematical invariant.  They take the oracle module as an
argument so that tests/test_oracle_mutants.py can run the same checks against
deliberately broken builds of the oracle and show that each planted mistake is
caught.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def hadamard_matrix() -> np.ndarray:
    """Closed-form unnormalised Sylvester matrix, H[j][i] = (-1)^popcount(i & j)."""
    i = np.arange(32)
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def _same_or_both_nan(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return both_nan | eq


# ---------------------------------------------------------------- decoders
def check_bf16_decode(O):
    import torch
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_to_f64(bits)
    assert _same_or_both_nan(got, ref).all(), "bf16 decode differs from torch's cast"


def check_f16_decode(O):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = O.f16_to_f64(bits)
    assert _same_or_both_nan(got, ref).all(), "fp16 decode differs from numpy's cast"


def check_e4m3_decode(O):
    import torch
    codes = np.arange(256, dtype=np.uint8)
    got = O.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert _same_or_both_nan(got, ref).all(), "e4m3 decode differs from torch's cast"
    g = _golden("e4m3_points.json")
    for code_s, val in g["points"]:
        c = int(code_s, 16)
        v = O.e4m3_to_f64(np.array([c], np.uint8))[0]
        assert v == val and math.copysign(1, v) == math.copysign(1, val), (code_s, v, val)
    # exactly two NaN codes (S.1111.111), no infinities
    assert np.isnan(got).sum() == 2 and not np.isinf(got).any()


# ---------------------------------------------------------------- encoders
def check_f16_encode(O):
    rng = np.random.default_rng(7)
    # every fp16 value, every midpoint between neighbours, and random fp32 values
    allh = np.arange(65536, dtype=np.uint16).view(np.float16)
    fin = allh[np.isfinite(allh)].astype(np.float64)
    fin = np.unique(fin)
    mids = (fin[:-1] + fin[1:]) / 2
    xs = np.concatenate([fin, mids, rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000),
                         [70000.0, -1e30, 65519.99, 65520.0, 5.96e-8, 2.98e-8, 2.99e-8]])
    xs = xs.astype(np.float32)
    xs = xs[np.isfinite(xs)]
    with np.errstate(over="ignore"):
        ref = xs.astype(np.float16).view(np.uint16)
    got = O.f32_to_f16_rne(xs)
    bad = got != ref
    assert not bad.any(), f"fp16 RNE encode mismatch at {xs[bad][:5]}"


def check_e4m3_encode(O):
    import torch
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_to_f64(codes)
    finite = ~np.isnan(vals)
    # round trip of every finite code (the sign of zero is kept)
    rt = O.f32_to_e4m3_sat(vals[finite].astype(np.float32))
    assert (rt == codes[finite]).all(), "e4m3 round trip failed"
    # midpoints between neighbouring positive values round to the even mantissa
    pos = np.unique(vals[finite & (vals >= 0)])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    enc = O.f32_to_e4m3_sat(mids)
    assert ((enc & 1) == 0).all(), "e4m3 midpoint did not round to even"
    # in-range values against torch's cast
    rng = np.random.default_rng(11)
    xs = (rng.standard_normal(50000) * 10.0 ** rng.uniform(-4, 2.6, 50000)).astype(np.float32)
    xs = xs[np.abs(xs) <= 448]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.f32_to_e4m3_sat(xs)
    assert (got == ref).all(), "e4m3 encode differs from torch's cast"
    # saturation
    sat = O.f32_to_e4m3_sat(np.array([449.0, 1e9, -500.0, 464.0], np.float32))
    assert list(sat) == [0x7E, 0x7E, 0xFE, 0x7E]


# ---------------------------------------------------------------- Q4_0
def check_q4_0_dequant_closed_form(O):
    g = _golden("q4_0_blocks.json")
    for blk in g["blocks"]:
        b = np.array(blk["bytes"], np.uint8)
        got = O.q4_0_dequant(b, 1, 32)[0]
        assert (got == np.array(blk["values"], np.float64)).all(), blk["comment"]
    # exhaustive: every code in every nibble position for a set of scales
    for dbits in (0x3C00, 0x3800, 0xB400, 0x0000, 0x0001, 0x7BFF, 0x8001, 0x03FF):
        d = float(np.array([dbits], np.uint16).view(np.float16)[0])
        for q in range(16):
            for hi in (False, True):
                b = np.zeros(18, np.uint8)
                b[0], b[1] = dbits & 0xFF, dbits >> 8
                b[2:] = 0x88  # every other element has code 8 (value 0)
                j = 5
                b[2 + j] = (0x08 | (q << 4)) if hi else (0x80 | q)
                got = O.q4_0_dequant(b, 1, 32)[0]
                idx = j + 16 if hi else j
                assert got[idx] == d * (q - 8), (dbits, q, hi)
                mask = np.ones(32, bool)
                mask[idx] = False
                assert (got[mask] == 0).all()


def check_top_bit_flip(O):
    """Q4_0 code q with its top bit flipped, read as a 4-bit two's-complement
    integer, equals q - 8; the oracle's dequantized value is d times that."""
    for q in range(16):
        v = q ^ 8
        sext = v - 16 if v & 8 else v
        assert sext == q - 8
        b = np.zeros(18, np.uint8)
        b[0], b[1] = 0x00, 0x3C  # d = 1
        b[2:] = 0x88
        b[2] = 0x80 | q
        assert O.q4_0_dequant(b, 1, 32)[0][0] == sext


def check_q4_0_quantizer(O):
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    w[0, :32] = 0.0                       # all-zero block
    w[1, 32:64] = np.float32(0.5)         # constant block: every element is the max
    w[2, 64:96] *= 1e-6                   # tiny block (scale lands in fp16 subnormals)
    w[3, 96:128] *= 0.1                   # magnitude tie of opposite signs: the first wins
    w[3, 96 + 2] = np.float32(-0.3)
    w[3, 96 + 20] = np.float32(0.3)
    blocks = O.q4_0_quantize(w).reshape(64, 8, 18)
    deq = O.q4_0_dequant(blocks, 64, 256)
    for n in range(64):
        for b in range(8):
            x = w[n, 32 * b:32 * b + 32].astype(np.float64)
            blk = blocks[n, b]
            dbits = int(blk[0]) | (int(blk[1]) << 8)
            d = float(np.array([dbits], np.uint16).view(np.float16)[0])
            q = np.empty(32, np.int64)
            q[:16] = blk[2:] & 15
            q[16:] = blk[2:] >> 4
            amax_i = int(np.argmax(np.abs(x)))
            amax_s = x[amax_i]
            if amax_s == 0:
                assert d == 0 and (q == 8).all()
                continue
            d32 = np.float32(amax_s) / np.float32(-8.0)
            # stored d is d32 rounded to fp16
            assert abs(d - float(d32)) <= abs(float(d32)) * 2.0 ** -11 + 2.0 ** -25
            assert math.copysign(1, d) == -math.copysign(1, amax_s)
            # the signed-max element takes code 0 (value -8 d = amax up to d's rounding)
            assert q[amax_i] == 0
            # every element is within half a step, except where x/d32 > 7.5: code
            # 16 is clamped to 15, leaving x/d32 - 7 steps; plus what fp16
            # rounding of d moves a code of magnitude <= 8
            err = np.abs(deq[n, 32 * b:32 * b + 32] - x)
            t = x / float(d32)
            assert (t <= 8 + 1e-6).all() and (t >= -8 - 1e-6).all()
            step = max(abs(d), abs(float(d32)))
            slack = 8 * abs(d - float(d32)) + 1e-6 * step
            bound = np.where(t > 7.5, (t - 7) * step, step / 2) + slack
            assert (err <= bound).all()


# ---------------------------------------------------------------- FP8
def check_fp8_quantizer(O):
    import torch
    rng = np.random.default_rng(5)
    N, K = 256, 384
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[:128, 128:256] = 0.0  # an all-zero tile
    codes, scales = O.fp8_quantize(w)
    assert scales.shape == (2, 3)
    deq = O.fp8_dequant(codes, scales)
    for tn in range(2):
        for tk in range(3):
            tile = w[128 * tn:128 * tn + 128, 128 * tk:128 * tk + 128]
            c = codes[128 * tn:128 * tn + 128, 128 * tk:128 * tk + 128]
            s = scales[tn, tk]
            amax = np.abs(tile).max()
            assert s == np.float32(amax) / np.float32(448.0)
            if s == 0:
                assert (c == 0).all()
                continue
            # the max-magnitude element encodes to +-448
            i = np.unravel_index(np.argmax(np.abs(tile)), tile.shape)
            assert (c[i] & 0x7F) == 0x7E
            # codes equal torch's e4m3 cast of w / s (in range after the clamp)
            ratio = np.clip(tile / s, -448, 448).astype(np.float32)
            ref = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert (ref == c).all()
            # relative error of a normal e4m3 value <= 2^-4, absolute <= 2^-10 s below
            d = deq[128 * tn:128 * tn + 128, 128 * tk:128 * tk + 128]
            err = np.abs(d - tile)
            assert (err <= np.maximum(np.abs(tile) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-6)).all()


# ---------------------------------------------------------------- Hadamard
def check_hadamard(O):
    H = hadamard_matrix()
    assert (H @ H.T == 32 * np.eye(32, dtype=np.int64)).all()
    # the oracle's butterflies applied to unit vectors give the columns of H
    eye = np.eye(32)
    assert (O.fwht32_f64(eye) == H.T.astype(np.float64)).all()
    assert (O.fwht32_f32(eye.astype(np.float32)) == H.T.astype(np.float32)).all()
    # hand-worked golden example
    g = _golden("hadamard32_ramp.json")
    x = np.array(g["input"], np.float64)
    assert (O.fwht32_f64(x) == np.array(g["output"], np.float64)).all()
    assert (O.fwht32_f32(x.astype(np.float32)) == np.array(g["output"], np.float32)).all()
    # hand-worked fp32 case that only the stated stage order (strides 1,2,4,8,16) rounds this way
    c = g["fp32_order_case"]
    x = np.zeros(32, np.float32)
    for i, v in c["input_nonzero"]:
        x[i] = np.float32(v)
    y = O.fwht32_f32(x)
    for i, v in c["output_index_value"]:
        assert y[i] == np.float32(v), (i, y[i], v)
    # involution up to 32 (exact in fp64 for fp32-representable inputs)
    rng = np.random.default_rng(9)
    v = rng.standard_normal((200, 32)).astype(np.float32).astype(np.float64)
    assert (O.fwht32_f64(O.fwht32_f64(v)) == 32 * v).all()
    # fp32 model against a straight fp64 matrix product, within 5 * 2^-24 * sum|x|
    v32 = (rng.standard_normal((500, 32)) * 10.0 ** rng.uniform(-3, 3, (500, 1))).astype(np.float32)
    got = O.fwht32_f32(v32).astype(np.float64)
    ref = v32.astype(np.float64) @ H.T.astype(np.float64)
    bound = 5 * 2.0 ** -24 * np.abs(v32.astype(np.float64)).sum(axis=1, keepdims=True)
    assert (np.abs(got - ref) <= bound).all()


def sylvester(B: int) -> np.ndarray:
    """Closed-form unnormalised Sylvester matrix of size B, H[j][i] = (-1)^popcount(i & j)."""
    i = np.arange(B)
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


def check_hadamard_larger(O):
    """The 64- and 128-point transforms: closed forms, the involution, the fp32
    error bound, and a bit-exact recursion that fixes the stage order: with
    strides ascending, the B-point fp32 result is (A + C, A - C) in fp32 where
    A and C are the B/2-point results of the two halves (so B = 64 rests on the
    pinned 32-point transform, and B = 128 on B = 64)."""
    rng = np.random.default_rng(19)
    for B in (64, 128):
        H = sylvester(B)
        assert (H @ H.T == B * np.eye(B, dtype=np.int64)).all()
        eye = np.eye(B)
        assert (O.fwht_f64(eye, B) == H.T.astype(np.float64)).all()
        assert (O.fwht_f32(eye.astype(np.float32), B) == H.T.astype(np.float32)).all()
        # ramp x_i = i + 1: (Hx)_0 = B (B + 1) / 2, (Hx)_j = -(B / 2) j for j a
        # power of two, 0 otherwise (worked by hand from the bits of i)
        x = np.arange(1, B + 1, dtype=np.float64)
        want = np.zeros(B)
        want[0] = B * (B + 1) / 2
        for b in range(int(np.log2(B))):
            want[1 << b] = -(B / 2) * (1 << b)
        assert (O.fwht_f64(x, B) == want).all() and (O.fwht_f32(x.astype(np.float32), B) == want).all()
        v = rng.standard_normal((100, B)).astype(np.float32).astype(np.float64)
        assert (O.fwht_f64(O.fwht_f64(v, B), B) == B * v).all()
        v32 = (rng.standard_normal((300, B)) * 10.0 ** rng.uniform(-3, 3, (300, 1))).astype(np.float32)
        got = O.fwht_f32(v32, B)
        ref = v32.astype(np.float64) @ H.T.astype(np.float64)
        bound = (np.log2(B) + 1) * 2.0 ** -24 * np.abs(v32.astype(np.float64)).sum(axis=1, keepdims=True)
        assert (np.abs(got.astype(np.float64) - ref) <= bound).all()
        h = B // 2
        A = O.fwht_f32(v32[:, :h], h) if h > 32 else O.fwht32_f32(v32[:, :h])
        C = O.fwht_f32(v32[:, h:], h) if h > 32 else O.fwht32_f32(v32[:, h:])
        rec = np.concatenate([A + C, A - C], axis=1)  # fp32 adds, round to nearest even
        assert (got == rec).all(), B
        # the activation rotation and the offline weight rotation use the same model
        a = (rng.standard_normal((3, 2 * B)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        af = (a.astype(np.uint32) << 16).view(np.float32)
        assert (O.hadamard_act_f32(a, B) == O.fwht_f32(af.reshape(3, 2, B), B).reshape(3, 2 * B)).all()


def check_rotated_product(O):
    """Rotated activations times rotated (offline, /32) weights equal the
    activations times the un-rotated dequantized weights H^T deq(w')."""
    import speculative_decode_verification_qmm_gb300.synth as synth
    H = hadamard_matrix().astype(np.float64)
    N, K, M = 48, 128, 5
    w = synth.weights(N, K, 21)
    a = synth.activations(M, K, 22, outliers=True)
    blocks = O.q4_0_quantize_h32(w)
    out_rot, _ = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a, hadamard=True)
    wq = O.q4_0_dequant(blocks, N, K)
    # un-rotate the dequantized weights block by block: H^T w'_b (H symmetric)
    w_un = (wq.reshape(N, K // 32, 32) @ H).reshape(N, K)
    af = synth.bf16_bits_to_f32(a).astype(np.float64)
    ref = af @ w_un.T
    assert np.allclose(out_rot, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # and the un-rotated weights approximate w itself: H/sqrt(32) is orthogonal, so the
    # relative error equals the Q4_0 error of the rotated weights (about 10% for Gaussians)
    rel = np.linalg.norm(w_un - w) / np.linalg.norm(w)
    assert rel < 0.2, rel


# ---------------------------------------------------------------- product
def check_rotated_product_larger(O):
    """B = 64, 128: rotated activations times weights rotated offline (fp32,
    times 1/B) and quantized equal the activations times the un-rotated
    dequantized weights H^T deq(w') / (1) -- H H^T = B I and the 1/B in the
    weights cancel."""
    import speculative_decode_verification_qmm_gb300.synth as synth
    N, K, M = 40, 256, 4
    for B in (64, 128):
        H = sylvester(B).astype(np.float64)
        w = synth.weights(N, K, 23 + B)
        a = synth.activations(M, K, 24 + B, outliers=True)
        wr = O.rotate_weights_f32(w, B)
        blocks = O.q4_0_quantize(wr)
        out_rot, _ = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a, hadamard=B)
        wq = O.q4_0_dequant(blocks, N, K)
        w_un = (wq.reshape(N, K // B, B) @ H).reshape(N, K)
        af = synth.bf16_bits_to_f32(a).astype(np.float64)
        ref = af @ w_un.T
        assert np.allclose(out_rot, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        rel = np.linalg.norm(w_un - w) / np.linalg.norm(w)
        assert rel < 0.2, rel


def check_product_brute_force(O):
    import speculative_decode_verification_qmm_gb300.synth as synth
    for (M, K, N) in ((4, 32, 64), (4, 64, 32)):
        w = synth.weights(N, K, 100 + K)
        a = synth.activations(M, K, 200 + K)
        blocks = O.q4_0_quantize(w)
        out, S = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a)
        wq = O.q4_0_dequant(blocks, N, K)
        af = synth.bf16_bits_to_f32(a).astype(np.float64)
        # library matmul of the dequantized operands
        ref = af @ wq.T
        assert np.allclose(out, ref, rtol=0, atol=K * 2.0 ** -52 * S.max())
        # exact rational arithmetic
        for m in range(M):
            for n in range(N):
                ex = sum(Fraction(float(af[m, k])) * Fraction(float(wq[n, k])) for k in range(K))
                assert abs(Fraction(out[m, n]) - ex) <= Fraction(K) * Fraction(2.0 ** -53) * Fraction(S[m, n])
                sx = sum(abs(Fraction(float(af[m, k])) * Fraction(float(wq[n, k]))) for k in range(K))
                assert abs(Fraction(S[m, n]) - sx) <= Fraction(K) * Fraction(2.0 ** -53) * sx
    # FP8: one 128x128 tile, M = 4
    w = synth.weights(128, 128, 300)
    a = synth.activations(4, 128, 301, outliers=True)
    codes, scales = O.fp8_quantize(w)
    out, S = O.verify_rows(O.FMT_FP8, codes, scales, 128, 128, a)
    wq = O.fp8_dequant(codes, scales)
    af = synth.bf16_bits_to_f32(a).astype(np.float64)
    for m in range(4):
        for n in range(0, 128, 7):
            ex = sum(Fraction(float(af[m, k])) * Fraction(float(wq[n, k])) for k in range(128))
            assert abs(Fraction(out[m, n]) - ex) <= Fraction(128) * Fraction(2.0 ** -53) * Fraction(S[m, n])


def check_rows_are_independent_gemvs(O):
    import speculative_decode_verification_qmm_gb300.synth as synth
    N, K, M = 40, 256, 16
    w = synth.weights(N, K, 31)
    a = synth.activations(M, K, 32, outliers=True)
    blocks = O.q4_0_quantize(w)
    for had in (False, True):
        out, _ = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a, hadamard=had)
        for m in range(M):
            one, _ = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a[m:m + 1], hadamard=had)
            assert (one[0] == out[m]).all()
        # selected rows equal the same rows of the full product
        rows = np.array([39, 0, 17, 17, 5], np.int64)
        sel, _ = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a, hadamard=had, rows=rows)
        assert (sel == out[:, rows]).all()


def check_special_activations(O):
    import speculative_decode_verification_qmm_gb300.synth as synth
    N, K = 24, 96
    w = synth.weights(N, K, 41)
    blocks = O.q4_0_quantize(w)
    wq = O.q4_0_dequant(blocks, N, K)
    one = np.float32(1.0).view(np.uint32) >> 16
    # one-hot rows return one dequantized weight column exactly
    ks = [0, 17, 95]
    a = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        a[i, k] = one
    out, _ = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a)
    for i, k in enumerate(ks):
        assert (out[i] == wq[:, k]).all()
    # all-ones rows return exact row sums (dyadic values with few bits sum exactly)
    a = np.full((2, K), one, np.uint16)
    out, S = O.verify_rows(O.FMT_Q4_0, blocks, None, N, K, a)
    for n in range(N):
        ex = sum(Fraction(float(v)) for v in wq[n])
        assert Fraction(out[0, n]) == ex and out[1, n] == out[0, n]
        assert Fraction(S[0, n]) == sum(abs(Fraction(float(v))) for v in wq[n])


def check_hadamard_act_model(O):
    """The fp32 activation rotation equals the fp32 butterflies block by block
    and agrees with the exact fp64 rotation within the fp32 bound."""
    import speculative_decode_verification_qmm_gb300.synth as synth
    a = synth.activations(3, 128, 51, outliers=True)
    got = O.hadamard32_act_f32(a)
    af = synth.bf16_bits_to_f32(a)
    H = hadamard_matrix().astype(np.float64)
    for m in range(3):
        for b in range(4):
            blk = af[m, 32 * b:32 * b + 32]
            assert (got[m, 32 * b:32 * b + 32] == O.fwht32_f32(blk)).all()
            ref = H @ blk.astype(np.float64)
            bound = 5 * 2.0 ** -24 * np.abs(blk.astype(np.float64)).sum()
            assert (np.abs(got[m, 32 * b:32 * b + 32] - ref) <= bound).all()


# ---------------------------------------------------------------- Q8_0
def check_q8_0_dequant_closed_form(O):
    """Hand-worked blocks (tests/golden/q8_0_blocks.json), then every code
    under a few scales: w = d * (signed code)."""
    for blk in _golden("q8_0_blocks.json")["blocks"]:
        b = np.array(blk["bytes"], np.uint8).reshape(1, 1, 34)
        got = O.q8_0_dequant(b, 1, 32)[0]
        assert (got == np.array(blk["values"], np.float64)).all(), blk["name"]
    codes = np.arange(256, dtype=np.uint8)
    for d_bits in (0x3C00, 0x3800, 0xB400, 0x0001, 0x7BFF, 0x0000):
        d = float(np.array([d_bits], np.uint16).view(np.float16)[0])
        b = np.zeros((1, 8, 34), np.uint8)
        b[0, :, 0], b[0, :, 1] = d_bits & 0xFF, d_bits >> 8
        b[0, :, 2:] = codes.reshape(8, 32)
        got = O.q8_0_dequant(b, 1, 256)[0]
        assert (got == d * codes.view(np.int8).astype(np.float64)).all(), hex(d_bits)


def check_q8_0_quantizer(O):
    """Bounds and rules of the quantizer: the largest magnitude maps to +-127,
    every element is within |d| / 2 of its dequantized value (plus the fp16
    rounding of d times 127), signs survive, an all-zero block has d = 0 and
    zero codes, and halves round away from zero (checked on a block whose
    scale is exactly 1)."""
    import speculative_decode_verification_qmm_gb300.synth as synth
    w = synth.weights(64, 256, 31)
    w[0, :32] = 0.0
    b = O.q8_0_quantize(w)
    deq = O.q8_0_dequant(b, 64, 256)
    codes = b[:, :, 2:].view(np.int8).astype(np.int64)
    d = b[:, :, :2].copy().view(np.uint16)[..., 0].view(np.float16).astype(np.float64)
    x = w.reshape(64, 8, 32).astype(np.float64)
    amax = np.abs(x).max(axis=2)
    nz = amax > 0
    top = np.abs(codes)[np.arange(64)[:, None], np.arange(8)[None, :], np.abs(x).argmax(axis=2)]
    assert (top[nz] == 127).all()
    d32 = amax / 127.0
    # the stored scale is amax / 127 rounded to fp16: within half an fp16 ulp
    # (2^-11 relative for normals, 2^-25 absolute for subnormals)
    dq = 2.0 ** -11 * d32 + 2.0 ** -25
    assert (np.abs(d - d32) <= dq * (1 + 1e-6)).all()
    err = np.abs(x - deq.reshape(64, 8, 32))
    bound = d32[..., None] / 2 + dq[..., None] * 127
    assert (err <= bound * (1 + 1e-6)).all()
    assert ((np.sign(codes) == np.sign(x)) | (codes == 0)).all()
    assert (codes[~nz] == 0).all() and (d[~nz] == 0).all()
    # scale exactly 1: amax 127; 2.5 -> 3, -2.5 -> -3, 0.5 -> 1, -0.5 -> -1
    t = np.zeros((1, 32), np.float32)
    t[0, :5] = [127.0, 2.5, -2.5, 0.5, -0.5]
    c = O.q8_0_quantize(t)[0, 0, 2:7].view(np.int8).tolist()
    assert c == [127, 3, -3, 1, -1], c


def check_q8_0_product(O):
    """The Q8_0 verify product against numpy's matmul of the dequantized
    weights and against exact rationals on a small case."""
    import speculative_decode_verification_qmm_gb300.synth as synth
    N, K, M = 24, 96, 4
    w = synth.weights(N, K, 33)
    b = O.q8_0_quantize(w)
    a = synth.activations(M, K, 34, outliers=True)
    out, S = O.verify_rows(O.FMT_Q8_0, b, None, N, K, a)
    af = synth.bf16_bits_to_f32(a).astype(np.float64)
    deq = O.q8_0_dequant(b, N, K)
    ref = af @ deq.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.allclose(S, np.abs(af) @ np.abs(deq).T, rtol=1e-12)
    exact = sum(Fraction(float(af[1, k])) * Fraction(float(deq[5, k])) for k in range(K))
    assert abs(Fraction(float(out[1, 5])) - exact) <= abs(exact) * Fraction(1, 2 ** 40) + Fraction(1, 2 ** 60)


# ---------------------------------------------------------------- greedy acceptance
def check_greedy_golden(O):
    """Hand-worked blocks (tests/golden/greedy_accept.json)."""
    for case in _golden("greedy_accept.json")["cases"]:
        lg = np.array(case["logits"], np.float64)
        am, k, nxt = O.greedy_accept(lg, np.array(case["tokens"], np.int32))
        assert am.tolist() == case["argmax"], case["name"]
        assert (k, nxt) == (case["k"], case["next"]), case["name"]


def check_greedy_vs_library(O):
    """Argmax against numpy's (first occurrence of the maximum, the first NaN
    where there is one), on scores rounded coarsely so that ties are frequent; k against a brute-force count
    of the leading agreements, with drafts built to agree up to a chosen
    position."""
    rng = np.random.default_rng(11)
    for trial in range(200):
        M = int(rng.integers(1, 17))
        N = int(rng.integers(1, 40))
        lg = np.round(rng.standard_normal((M, N)) * 2.0) / 2.0
        if trial % 4 == 3:  # a few NaN scores: numpy's argmax returns the first NaN
            lg[rng.random((M, N)) < 0.1] = np.nan
        if trial % 8 == 5:  # signed zeros as the maximum: equal, the first one wins
            lg = -np.abs(lg)
            lg[rng.random((M, N)) < 0.3] = -0.0
            lg[rng.random((M, N)) < 0.3] = 0.0
        ref = np.argmax(lg, axis=1).astype(np.int32)
        j = int(rng.integers(0, M))  # drafts agree at positions < j
        tokens = rng.integers(0, N, M).astype(np.int32)
        tokens[1:j + 1] = ref[:j]
        if j + 1 < M and N > 1 and tokens[j + 1] == ref[j]:
            tokens[j + 1] = (ref[j] + 1) % N
        am, k, nxt = O.greedy_accept(lg, tokens)
        assert (am == ref).all()
        agree = (ref[:-1] == tokens[1:]) if M > 1 else np.zeros(0, bool)
        kk = int(np.cumprod(agree).sum()) if M > 1 else 0
        assert k == kk and nxt == ref[kk]
        assert k == (j if N > 1 else M - 1) or N == 1


ALL_CHECKS = [
    check_bf16_decode, check_f16_decode, check_e4m3_decode, check_f16_encode,
    check_e4m3_encode, check_q4_0_dequant_closed_form, check_top_bit_flip,
    check_q4_0_quantizer, check_fp8_quantizer, check_hadamard, check_rotated_product,
    check_product_brute_force, check_rows_are_independent_gemvs, check_special_activations,
    check_hadamard_act_model, check_greedy_golden, check_greedy_vs_library,
    check_hadamard_larger, check_rotated_product_larger, check_q8_0_dequant_closed_form,
    check_q8_0_quantizer, check_q8_0_product,
]
