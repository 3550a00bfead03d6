"""Pins for the oracle's quantiser fixes ("Decomposing MXFP4 quantization error for LLM
reinforcement learning", MBS -- macro block scaling, OF -- outlier fallback).

Each fix is pinned by hand-derived examples (tests/golden/quant_fix_examples.jsonl), by
reduction to the already-pinned row quantiser, by a closed form computed here with
Python integers, and by properties that hold for every input."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_fix_examples.jsonl")
HADS = [1, 16, 32]


def expand(lst, fill_from=None):
    """[a, b, "x31"] -> a, b and 31 copies of b; "z124" -> 124 zeros."""
    out = []
    for v in lst:
        if isinstance(v, str) and v[0] == "x":
            out += [out[-1]] * int(v[1:])
        elif isinstance(v, str) and v[0] == "z":
            out += [0] * int(v[1:])
        else:
            out.append(v)
    return out


def bf16_row(vals):
    f = np.asarray(vals, np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "example values must be exact in bf16"
    return (b >> 16).astype(np.uint16)[None, :]


def golden():
    with open(GOLDEN) as f:
        return [json.loads(line) for line in f if line.strip()]


@pytest.mark.parametrize("case", golden(), ids=lambda c: c["id"])
def test_golden_examples(case):
    x = bf16_row(expand(case["x"]))
    if case["fix"] == "of":
        c1, s1, c2, s2, bad = oracle.quantize_of(x, case["had"], case["mode"], case["alpha_log2"])
        assert bad == 0
        assert s1[0, 0] == case["q1_scale"] and s2[0, 0] == case["q2_scale"]
        assert list(oracle.unpack_codes(c1)[0]) == expand(case["q1_codes"])
        assert list(oracle.unpack_codes(c2)[0]) == expand(case["q2_codes"])
        xhat = oracle.dequant_row(c1, s1) + oracle.dequant_row(c2, s2)
        assert np.array_equal(xhat[0], np.asarray(expand(case["xhat"]), np.float64))
    else:
        codes, scales, mbs = oracle.quantize_mbs(x, case["had"], case["mode"])
        assert mbs[0, 0] == case["mbs"]
        assert list(scales[0]) == case["scales"]
        assert list(oracle.unpack_codes(codes)[0]) == expand(case["codes"])
        xhat = oracle.dequant_mbs(codes, scales, mbs)
        np.testing.assert_allclose(xhat[0], np.asarray(expand(case["xhat"])), rtol=0, atol=1e-15)
        pc, _ = oracle.quantize(x, case["had"], case["mode"], "row")
        assert list(oracle.unpack_codes(pc)[0]) == expand(case["plain_codes"])


# --------------------------------------------------------------------------- MBS
def mbs_closed_form(amax: np.float32) -> int:
    """k = floor(256 (T - f) / f) from the mantissa bits, in exact integers."""
    bits = int(np.asarray(amax, np.float32).view(np.uint32))
    if bits < 0x00800000:
        return 0
    mant = bits & 0x7FFFFF
    if mant <= 0x400000:  # f <= 1.5, T = 1.5
        return (256 * (0x400000 - mant)) // (0x800000 + mant)
    return (256 * (0x1000000 - mant)) // (0x800000 + mant)  # T = 3


def test_mbs_byte_closed_form_and_edges():
    g = np.random.default_rng(5)
    vals = list(g.standard_normal(4000).astype(np.float32) * 10.0 ** g.integers(-30, 30, 4000))
    vals += [np.float32(v) for v in (1.0, 1.5, 2.0, 3.0, 5.0, 6.0, 1e-38, 1e-45, 0.0)]
    vals += [np.nextafter(np.float32(1.5), np.float32(2)), np.nextafter(np.float32(2), np.float32(1))]
    for a in vals:
        a = np.float32(abs(a))
        k = oracle.mbs_byte(a)
        assert k == mbs_closed_form(a), a
        assert 0 <= k <= 255
        if a >= np.finfo(np.float32).tiny:
            f = Fraction(float(a)) / Fraction(2) ** (int(np.floor(np.log2(float(a)))))
            if f >= 2:  # log2 rounding guard
                f /= 2
            T = Fraction(3, 2) if f <= Fraction(3, 2) else Fraction(3)
            assert (1 + Fraction(k, 256)) * f <= T < (1 + Fraction(k + 1, 256)) * f or k == 255


def test_mbs_with_no_correction_reduces_to_plain_quantiser():
    """Macro blocks whose amax has mantissa 1.5 get k = 0: codes and scales are those of
    the plain row quantiser."""
    g = np.random.default_rng(6)
    R, C = 8, 512
    x = (g.standard_normal((R, C)) * 0.3).astype(np.float32)
    for mb in range(C // 128):
        x[:, mb * 128 + 7] = 1.5 * 2.0 ** g.integers(-3, 4, R)  # the macro max, |x| <= 1.2 elsewhere
    x[:, :] = np.clip(x, -1.2, 1.2)
    for mb in range(C // 128):
        x[:, mb * 128 + 7] = 1.5 * 2.0 ** g.integers(2, 5, R)
    xb = synth.bf16_bits(x)
    for mode in (0, 1):
        codes, scales, mbs = oracle.quantize_mbs(xb, 1, mode)
        assert np.all(mbs == 0)
        pc, ps = oracle.quantize(xb, 1, mode, "row")
        assert np.array_equal(codes, pc) and np.array_equal(scales, ps)


@pytest.mark.parametrize("had", HADS)
@pytest.mark.parametrize("mode", [0, 1])
def test_mbs_puts_the_macro_max_on_the_top_grid_point(had, mode):
    """After the prescale the macro-block maximum quantises to magnitude 6 (code 7)
    without saturating: (1 + k/256) A <= T 2^E and (1 + (k+1)/256) A > T 2^E."""
    x = synth.heavy_tailed(16, 1024, 40 + had + mode)
    codes, scales, mbs = oracle.quantize_mbs(x, had, mode)
    v = oracle.rotate_f32(synth.bf16_to_f32(x), had)
    cu = oracle.unpack_codes(codes)
    for r in range(16):
        for mb in range(1024 // 128):
            blk = v[r, mb * 128:(mb + 1) * 128]
            i = int(np.argmax(np.abs(blk)))
            if np.abs(blk[i]) < np.finfo(np.float32).tiny:
                continue
            k = int(mbs[r, mb])
            assert k == oracle.mbs_byte(np.abs(blk[i]))
            assert (cu[r, mb * 128 + i] & 7) == 7
            u = Fraction(float(np.float32(blk[i] * np.float32(1 + k / 256)))) / Fraction(2) ** (
                int(scales[r, (mb * 128 + i) // 32]) - 127)
            assert abs(u) <= 6


def test_mbs_reconstruction_beats_plain_on_the_scale_error():
    """With the macro maximum on the grid top, the MBS reconstruction error of the
    maxima is below the plain quantiser's on heavy-tailed data."""
    x = synth.heavy_tailed(64, 1024, 77)
    v = oracle.rotate_f32(synth.bf16_to_f32(x), 16).astype(np.float64)
    codes, scales, mbs = oracle.quantize_mbs(x, 16, 0)
    pc, ps = oracle.quantize(x, 16, 0, "row")
    e_mbs = np.abs(oracle.dequant_mbs(codes, scales, mbs) - v).reshape(64, 8, 128).max(axis=2)
    e_plain = np.abs(oracle.dequant_row(pc, ps) - v).reshape(64, 8, 128).max(axis=2)
    assert e_mbs.mean() < e_plain.mean()


# --------------------------------------------------------------------------- OF
@pytest.mark.parametrize("had", HADS)
@pytest.mark.parametrize("mode", [0, 1])
def test_of_first_pass_is_the_plain_quantiser_and_the_second_the_residual(had, mode):
    x = synth.heavy_tailed(32, 512, 90 + had + mode)
    c1, s1, c2, s2, bad = oracle.quantize_of(x, had, mode, 0)
    assert bad == 0
    pc, ps = oracle.quantize(x, had, mode, "row")
    assert np.array_equal(c1, pc) and np.array_equal(s1, ps)
    v = oracle.rotate_f32(synth.bf16_to_f32(x), had).astype(np.float64)
    res = v - oracle.dequant_row(c1, s1)
    assert np.array_equal(res, res.astype(np.float32).astype(np.float64))  # exact in fp32
    rc, rs = oracle.quantize_f32_rows(res.astype(np.float32), mode)
    assert np.array_equal(c2, rc) and np.array_equal(s2, rs)


@pytest.mark.parametrize("alpha_log2", [-1, -2])
def test_of_alpha_is_a_scale_byte_shift(alpha_log2):
    x = synth.heavy_tailed(32, 512, 91)
    _, _, c2a, s2a, _ = oracle.quantize_of(x, 16, 0, 0)
    _, _, c2b, s2b, _ = oracle.quantize_of(x, 16, 0, alpha_log2)
    assert np.array_equal(c2a, c2b)
    assert np.array_equal(s2b.astype(int), np.maximum(s2a.astype(int) + alpha_log2, 0))


@pytest.mark.parametrize("had", HADS)
@pytest.mark.parametrize("mode", [0, 1])
def test_of_never_increases_the_error_elementwise(had, mode):
    """|x - (q1 + alpha q2)| <= |x - q1| for alpha in {1, 1/2}: round-to-nearest on a grid
    containing 0 never moves farther than |r| from r, and the nearest nonzero grid
    value is at most 2|r| away from 0 in the direction of r."""
    x = synth.heavy_tailed(32, 1024, 92 + had + mode)
    v = oracle.rotate_f32(synth.bf16_to_f32(x), had).astype(np.float64)
    for a in (0, -1):
        c1, s1, c2, s2, _ = oracle.quantize_of(x, had, mode, a)
        q1 = oracle.dequant_row(c1, s1)
        xof = q1 + oracle.dequant_row(c2, s2)
        assert np.all(np.abs(v - xof) <= np.abs(v - q1))
    # and it recovers most of the first pass's deadzone
    dz = (q1 == 0) & (v != 0)
    assert dz.sum() > 0 and np.mean(xof[dz] != 0) > 0.5


# ---------------------------------------------------------------- GEMM over MBS operands
def test_mbs_gemm_without_correction_is_the_plain_gemm():
    """All MBS bytes zero (factor 1): the MBS GEMM is the pinned plain GEMM, exactly."""
    qa = oracle.quantize(synth.activations(64, 512, 1), 16, 0, "row")
    qb = oracle.quantize(synth.weights(48, 512, 2), 16, 0, "row")
    z_a, z_b = np.zeros((64, 4), np.uint8), np.zeros((48, 4), np.uint8)
    C, S = oracle.gemm_mbs(qa[0], qa[1], z_a, qb[0], qb[1], z_b)
    C0, S0 = oracle.gemm(*qa, *qb)
    assert np.array_equal(C, C0) and np.array_equal(S, S0)
    C1, _ = oracle.gemm_mbs(qa[0], qa[1], None, qb[0], qb[1], None)
    assert np.array_equal(C1, C0)


@pytest.mark.parametrize("which", ["both", "a", "b"])
def test_mbs_gemm_is_the_product_of_the_reconstructions(which):
    """C = x_hat_A x_hat_B^T with x_hat the MBS reconstruction dq(q) / (1 + byte/256)
    (pinned by the MBS closed-form tests above): an fp64 matmul of the reconstructions
    agrees to fp64 rounding, for one or both operands under MBS."""
    X = synth.activations(96, 640, 3)
    W = synth.weights(80, 640, 4)
    ca, sa, ma = oracle.quantize_mbs(X, 16, 0)
    cb, sb, mb = oracle.quantize_mbs(W, 16, 1)
    use_a, use_b = which in ("both", "a"), which in ("both", "b")
    if not use_a:
        ca, sa = oracle.quantize(X, 16, 0, "row")
    if not use_b:
        cb, sb = oracle.quantize(W, 16, 1, "row")
    C, S = oracle.gemm_mbs(ca, sa, ma if use_a else None, cb, sb, mb if use_b else None)
    xa = oracle.dequant_mbs(ca, sa, ma) if use_a else oracle.dequant_row(ca, sa)
    xb = oracle.dequant_mbs(cb, sb, mb) if use_b else oracle.dequant_row(cb, sb)
    ref = xa @ xb.T
    assert np.all(np.abs(C - ref) <= 1e-12 * S + 1e-300)
    assert np.allclose(S, np.abs(xa) @ np.abs(xb).T, rtol=1e-12, atol=0)
    assert (ma > 0).any() and (mb > 0).any()  # the data exercises the correction


def test_mbs_gemm_single_macro_block_by_hand():
    """K = 128, every code 1.0 (code 2) under scale byte 127 on both sides: the plain dot
    is 128; MBS bytes 128 on A (factor 1/1.5) and 64 on B (factor 1/1.25) give
    128 / (1.5 * 1.25) = 68.2666..., exactly in rationals."""
    codes = np.full((1, 64), 0x22, np.uint8)
    scales = np.full((1, 4), 127, np.uint8)
    C, S = oracle.gemm_mbs(codes, scales, np.array([[128]], np.uint8), codes, scales, np.array([[64]], np.uint8))
    want = Fraction(128) / (Fraction(3, 2) * Fraction(5, 4))
    assert abs(Fraction(float(C[0, 0])) - want) <= Fraction(1, 2 ** 45) and abs(Fraction(float(S[0, 0])) - want) <= Fraction(1, 2 ** 45)
