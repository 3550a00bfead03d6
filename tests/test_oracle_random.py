"""Pins for the oracle's randomised baselines ("Pretraining Large Language Models with
MXFP4 on Native FP4 Hardware", A.2: random sign flips before the Hadamard; the
ablation of table 1: stochastic rounding).  The random numbers are inputs (a sign
bitmask, one uniform 16-bit integer per element), so the oracle is deterministic and
is pinned by brute force over all 2^16 values, by reduction to the pinned quantiser
and by the orthogonality of the randomised rotation."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth

GRID = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
ALL_R = np.arange(65536, dtype=np.uint16)


def mean_sr_value(u: float) -> Fraction:
    """Exact mean over all 65536 random integers of the stochastically rounded u."""
    codes = [oracle.e2m1_code_sr(u, int(r)) for r in range(0, 65536, 1)]
    vals = [Fraction(oracle.e2m1_value(c)) for c in codes]
    return sum(vals, Fraction(0)) / 65536


@pytest.mark.parametrize("u", [0.125, 0.75, 1.2001953125, -2.25, 3.5, 4.5, 5.99993896484375, -0.0078125])
def test_sr_is_exactly_unbiased_over_all_random_integers(u):
    """p * 65536 is an integer for these u, so the mean over r in [0, 65536) is u exactly."""
    assert mean_sr_value(u) == Fraction(u)


def test_sr_bias_bound_for_any_u():
    g = np.random.default_rng(3)
    for u in g.uniform(-5.999, 5.999, 40).astype(np.float32):
        a = abs(float(u))
        step = 0.5 if a < 2 else (1.0 if a < 4 else 2.0)
        assert abs(mean_sr_value(float(u)) - Fraction(float(u))) <= Fraction(step) / 65536


def test_sr_leaves_grid_points_and_saturates():
    for gv in GRID:
        for s in (1, -1):
            u = s * gv
            want = oracle.e2m1_code(u)
            assert {oracle.e2m1_code_sr(u, int(r)) for r in (0, 1, 12345, 32768, 65535)} == {want}
    for u in (6.5, 7.999, -7.0):
        assert oracle.e2m1_value(oracle.e2m1_code_sr(u, 0)) == np.sign(u) * 6


def test_sr_rounds_up_with_the_stated_probability():
    # u = 2.75: lo = 2, step 1, p = 0.75 -> up for exactly 49152 of the 65536 integers
    ups = sum(oracle.e2m1_value(oracle.e2m1_code_sr(2.75, int(r))) == 3 for r in range(65536))
    assert ups == 49152


@pytest.mark.parametrize("had", [1, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_random_signs_are_the_quantiser_of_the_flipped_input(had, mode):
    """Flipping a bf16 sign is exact, so H D x quantised equals the pinned quantiser of
    the sign-flipped input."""
    g = np.random.default_rng(had + 10 * mode)
    x = synth.heavy_tailed(64, 256, 7)
    cneg = g.random(256) < 0.5
    rneg = g.random(64) < 0.5
    xr = x ^ (cneg[None, :].astype(np.uint16) << 15)
    xc = x ^ (rneg[:, None].astype(np.uint16) << 15)
    for layout, neg, flipped in (("row", cneg, xr), ("colT", rneg, xc)):
        got = oracle.quantize_rand(x, had, mode, layout, signs=oracle.pack_signs(neg))
        want = oracle.quantize(flipped, had, mode, layout)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
    none = oracle.quantize_rand(x, had, mode, "row", signs=oracle.pack_signs(np.zeros(256, bool)))
    plain = oracle.quantize(x, had, mode, "row")
    assert np.array_equal(none[0], plain[0]) and np.array_equal(none[1], plain[1])


@pytest.mark.parametrize("had", [16, 32])
def test_random_sign_rotation_cancels_in_a_dot_product(had):
    """(H D x) . (H D w) = x . w: the randomised rotation is orthogonal too."""
    g = np.random.default_rng(had)
    K = 512
    d = np.where(g.random(K) < 0.5, -1.0, 1.0)
    x, w = g.standard_normal((8, K)), g.standard_normal((8, K))
    rx, rw = oracle.rotate_f64(x * d, had), oracle.rotate_f64(w * d, had)
    np.testing.assert_allclose(rx @ rw.T, x @ w.T, rtol=0, atol=1e-12 * (np.abs(x) @ np.abs(w).T).max())


@pytest.mark.parametrize("mode", [0, 1])
def test_sr_on_grid_valued_blocks_equals_round_to_nearest(mode):
    """Blocks whose scaled values all sit on the grid quantise identically with and
    without stochastic rounding, whatever the random integers."""
    g = np.random.default_rng(mode)
    R, C = 16, 128
    vals = np.asarray(GRID, np.float32)
    x = vals[g.integers(0, 8, (R, C))] * np.where(g.random((R, C)) < 0.5, -1, 1).astype(np.float32)
    x[:, ::32] = 6.0  # amax 6 per block: scale 2^0 in both modes
    xb = synth.bf16_bits(x)
    sr = g.integers(0, 65536, (R, C)).astype(np.uint16)
    got = oracle.quantize_rand(xb, 1, mode, "row", sr=sr)
    want = oracle.quantize(xb, 1, mode, "row")
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])


def test_sr_quantiser_is_unbiased_on_a_tensor():
    """Averaged over many independent random tensors, the SR reconstruction converges to
    the rotated input (RNE keeps its fixed bias)."""
    x = synth.heavy_tailed(4, 128, 9)
    v = oracle.rotate_f32(synth.bf16_to_f32(x), 16).astype(np.float64)
    g = np.random.default_rng(11)
    acc = np.zeros_like(v)
    n = 400
    for _ in range(n):
        c, s = oracle.quantize_rand(x, 16, 1, "row", sr=g.integers(0, 65536, x.shape).astype(np.uint16))
        acc += oracle.dequant_row(c, s)
    c, s = oracle.quantize(x, 16, 1, "row")
    rne_bias = np.abs(oracle.dequant_row(c, s) - v).mean()
    sr_bias = np.abs(acc / n - v).mean()
    assert sr_bias < 0.25 * rne_bias


# ---------------------------------------------------------------- counter-based generator
def _kat():
    import json
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.jsonl")
    return [json.loads(l) for l in open(path) if l.strip()]


@pytest.mark.parametrize("case", _kat(), ids=lambda c: c["name"])
def test_philox_known_answers(oracle_mod, case):
    """The generator against the published known-answer vectors of Philox4x32-10 (a
    wrong multiplier, Weyl constant, word order or round count changes every word)."""
    h = lambda xs: [int(v, 16) for v in xs]
    assert [int(v) for v in oracle_mod.philox4x32_10(h(case["ctr"]), h(case["key"]))] == h(case["out"])


def test_philox_streams_are_balanced_and_distinct(oracle_mod):
    """Sign vectors have half their bits set, distinct seeds give distinct vectors, and
    the stochastic-rounding integers are uniform over [0, 65536): their mean and the
    counts of their top nibble are within a few standard errors of uniform."""
    a, b = oracle_mod.philox_signs(1, 1 << 16), oracle_mod.philox_signs(2, 1 << 16)
    for bits in (a, b):
        ones = int(np.unpackbits(bits).sum())
        assert abs(ones - (1 << 15)) < 5 * 128  # sd = sqrt(n)/2 = 128
    assert not np.array_equal(a, b)
    r = oracle_mod.philox_sr(7, 64, 4096, 0).astype(np.float64)
    n = r.size
    assert abs(r.mean() - 32767.5) < 5 * 65536 / np.sqrt(12 * n)
    counts = np.bincount((r.astype(np.int64) >> 12).ravel(), minlength=16)
    chi2 = ((counts - n / 16) ** 2 / (n / 16)).sum()
    assert chi2 < 50  # 15 degrees of freedom: p ~ 1e-5
    assert not np.array_equal(oracle_mod.philox_sr(7, 4, 64, 0), oracle_mod.philox_sr(7, 4, 64, 1))


def test_philox_stochastic_rounding_is_unbiased(oracle_mod):
    """With the generated integers, the mean of stochastically rounded values of one
    constant block approaches the block (the generator feeds an unbiased rounding)."""
    v = np.float32(1.3)  # between grid values 1 and 1.5 under e = 0: rounds up with p = 0.6
    x = np.full((4096, 32), v, np.float32)
    x[:, 0] = 4.0  # amax 4 -> e = 0 (floor and ceil)
    xb = synth.bf16_bits(x)
    codes, scales = oracle_mod.quantize_philox(xb, 1, 0, "row", sr_seed=99)
    vals = np.array([oracle_mod.e2m1_value(int(c)) for c in oracle_mod.unpack_codes(codes)[:, 1:].ravel()])
    want = float(synth.bf16_to_f32(synth.bf16_bits(np.array([v], np.float32)))[0])
    assert set(np.unique(vals)) <= {1.0, 1.5}
    assert abs(vals.mean() - want) < 5 * 0.5 * np.sqrt(0.24 / vals.size)
