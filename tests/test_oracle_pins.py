"""Pins of the CPU oracle to facts the pages and the mathematics fix (no GPU).

Each test checks the C oracle against something other than itself: closed forms,
brute force in exact rational arithmetic, hand-worked examples (tests/golden),
identities stated on the pages, and invariants.  A plausible slip in the oracle
(wrong sign, dropped term, wrong axis, wrong tie rule, floor/ceil confusion)
fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from mxfp4_precision_gemms_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# ---------------------------------------------------------------- independent helpers
# These are written from the format definitions, not from the oracle's code.


def sylvester_bit_formula(n):
    """H_n[i][j] = (-1)^popcount(i & j)  (closed form of the Sylvester matrix)."""
    i = np.arange(n)[:, None]
    j = np.arange(n)[None, :]
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


MIDPOINTS = [  # (midpoint between neighbouring E2M1 magnitudes, code taken on a tie)
    (Fraction(1, 4), 0), (Fraction(3, 4), 2), (Fraction(5, 4), 2), (Fraction(7, 4), 4),
    (Fraction(5, 2), 4), (Fraction(7, 2), 6), (Fraction(5), 6)]


def e2m1_code_by_thresholds(u: Fraction, negative: bool) -> int:
    """Round |u| to E2M1 by counting the midpoints it passes (ties -> even code);
    anything past the last midpoint is 6 (saturation)."""
    a = abs(u)
    code = 0
    for mid, tie_code in MIDPOINTS:
        if a > mid or (a == mid and tie_code > code):
            code += 1
    return code | (8 if negative else 0)


def e2m1_code_by_binade(u: float) -> int:
    """IEEE-style round-to-nearest-even with the E2M1 step of each binade:
    step 0.5 below 2, 1 in [2,4), 2 in [4,6]; saturate at 6."""
    a = abs(u)
    if a >= 4:
        step = 2.0
    elif a >= 2:
        step = 1.0
    else:
        step = 0.5
    q = min(np.round(a / step) * step, 6.0)  # np.round is half-to-even on the step count
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    return mags.index(q) | (8 if math.copysign(1.0, u) < 0 else 0)


def exponent_by_scan(amax: Fraction, mode: int) -> int:
    """Brute-force scan of e in [-127, 127] in exact arithmetic."""
    if amax == 0:
        return -127
    es = range(-127, 128)
    if mode == 0:  # largest e with 2^(e+2) <= amax
        ok = [e for e in es if Fraction(2) ** (e + 2) <= amax]
        return max(ok) if ok else -127
    ok = [e for e in es if 6 * Fraction(2) ** e >= amax]  # smallest e with 6*2^e >= amax
    return min(ok) if ok else 127


def f32_from_bits(b):
    return np.array([b], dtype=np.uint32).view(np.float32)[0]


# ---------------------------------------------------------------- Hadamard


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32])
def test_hadamard_is_sylvester_closed_form(oracle_mod, n):
    h = oracle_mod.hadamard_pm1(n).astype(np.int64)
    assert np.array_equal(h, sylvester_bit_formula(n))


@pytest.mark.parametrize("n", [16, 32])
def test_hadamard_orthogonal(oracle_mod, n):
    """H H^T = n I, so H / sqrt(n) is orthogonal (Pretraining ... FP4 Hardware, C)."""
    h = oracle_mod.hadamard_pm1(n).astype(np.int64)
    assert np.array_equal(h @ h.T, n * np.eye(n, dtype=np.int64))
    assert np.array_equal(h, h.T)
    hn = h / 4.0
    if n == 16:  # entries +-1/4 are exact: the identity holds exactly in fp64
        assert np.array_equal(hn @ hn.T, np.eye(16))


def test_h32_constant_is_nearest_fp32(oracle_mod):
    """The fp32 normaliser of H32 is the binary32 value nearest to 1/sqrt(32)."""
    one_hot = np.zeros(32, np.float32)
    one_hot[0] = 1.0
    c = oracle_mod.rotate_f32(one_hot, 32)
    assert np.all(c == c[0])
    cf = Fraction(float(c[0]))
    lo = Fraction(float(np.nextafter(c[0], np.float32(0))))
    hi = Fraction(float(np.nextafter(c[0], np.float32(1))))
    # midpoints bracket 1/sqrt(32): compare squares exactly
    assert ((lo + cf) / 2) ** 2 < Fraction(1, 32) < ((cf + hi) / 2) ** 2


@pytest.mark.parametrize("n", [16, 32])
def test_rotation_of_one_hot_is_hadamard_column(oracle_mod, n):
    h = sylvester_bit_formula(n)
    c = oracle_mod.rotate_f32(np.eye(n, dtype=np.float32)[0], n)[0]
    for j in range(n):
        e = np.zeros(n, np.float32)
        e[j] = 1.0
        assert np.array_equal(oracle_mod.rotate_f32(e, n), (h[:, j] * c).astype(np.float32))


def test_rotation_exact_on_small_integers(oracle_mod):
    """With small-integer inputs every fp32 partial sum is exact, so the canonical
    rotation equals the exact product H16 x / 4 bit for bit."""
    g = np.random.default_rng(1)
    x = g.integers(-1000, 1000, size=(64, 16)).astype(np.float32)
    got = oracle_mod.rotate_f32(x, 16)
    want = (x.astype(np.float64) @ sylvester_bit_formula(16).T) / 4.0
    assert np.array_equal(got.astype(np.float64), want)


def test_rotation_follows_the_sylvester_recursion(oracle_mod):
    """The canonical fp32 order is the recursion H_2n[a;b] = [H_n a + H_n b; H_n a - H_n b]:
    checked against an in-place butterfly (strides 1, 2, 4, 8) in numpy float32."""
    g = np.random.default_rng(2)
    x = synth.bf16_to_f32(synth.bf16_bits(g.standard_normal((256, 16)).astype(np.float32) * 7))
    v = x.copy()
    s = 1
    while s < 16:
        idx = np.arange(16)
        lo = idx[(idx & s) == 0]
        a, b = v[:, lo].copy(), v[:, lo + s].copy()
        v[:, lo] = a + b
        v[:, lo + s] = a - b
        s *= 2
    v = v * np.float32(0.25)
    assert np.array_equal(oracle_mod.rotate_f32(x, 16), v)


def test_rotation_close_to_exact(oracle_mod):
    g = np.random.default_rng(3)
    for n in (16, 32):
        x = synth.bf16_to_f32(synth.bf16_bits(g.standard_normal((512, n)).astype(np.float32)))
        got = oracle_mod.rotate_f32(x, n).astype(np.float64)
        want = oracle_mod.rotate_f64(x.astype(np.float64), n)
        bound = (math.log2(n) + 2) * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True)
        assert np.all(np.abs(got - want) <= bound)


# ---------------------------------------------------------------- cancellation (C.1 - C.3)


def _rot_rows(oracle_mod, a, n):
    return oracle_mod.rotate_f64(a, n)


@pytest.mark.parametrize("n", [16, 32])
def test_cancellation_identities(oracle_mod, n):
    """Rotating each operand along its GEMM's contraction leaves the product unchanged:
    Y = (XH)(WH)^T = XW^T, dX = (dY H)(W^T H)^T = dY W, dW = (dY^T H)(X^T H)^T = dY^T X."""
    M, N, K = 256, 512, 512
    X, W, dY = (synth.bf16_to_f32(a).astype(np.float64) for a in synth.linear_inputs(M, N, K, 0))
    # Fprop: contraction K
    Y = _rot_rows(oracle_mod, X, n) @ _rot_rows(oracle_mod, W, n).T
    tolY = 1e-12 * (np.abs(X) @ np.abs(W).T)
    assert np.all(np.abs(Y - X @ W.T) <= tolY)
    # Dgrad: contraction N
    dX = _rot_rows(oracle_mod, dY, n) @ _rot_rows(oracle_mod, np.ascontiguousarray(W.T), n).T
    assert np.all(np.abs(dX - dY @ W) <= 1e-12 * (np.abs(dY) @ np.abs(W)))
    # Wgrad: contraction M
    dW = _rot_rows(oracle_mod, np.ascontiguousarray(dY.T), n) @ _rot_rows(oracle_mod, np.ascontiguousarray(X.T), n).T
    assert np.all(np.abs(dW - dY.T @ X) <= 1e-12 * (np.abs(dY.T) @ np.abs(X)))
    # a rotation along the wrong axis does not cancel
    bad = _rot_rows(oracle_mod, X, n) @ W.T
    assert np.max(np.abs(bad - X @ W.T)) > 1e-3 * np.max(np.abs(X @ W.T))


# ---------------------------------------------------------------- E2M1 rounding


def all_finite_bf16():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_to_f32(b)
    return f[np.isfinite(f)]


def test_e2m1_rounding_exhaustive_bf16(oracle_mod):
    """Every finite bf16 value as u: oracle code == midpoint count == binade RNE."""
    vals = all_finite_bf16()
    for u in vals:
        u = float(u)
        c = oracle_mod.e2m1_code(u)
        neg = math.copysign(1.0, u) < 0
        assert c == e2m1_code_by_thresholds(Fraction(u), neg), u
        if abs(u) <= 64:
            assert c == e2m1_code_by_binade(u), u


def test_e2m1_values(oracle_mod):
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for c in range(16):
        assert oracle_mod.e2m1_value(c) == (-1 if c & 8 else 1) * mags[c & 7]
        assert oracle_mod.e2m1_code(oracle_mod.e2m1_value(c)) == (c if c != 8 else 8)


# ---------------------------------------------------------------- E8M0 scale


def _scale_cases():
    pos = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)  # positive finite bf16 incl. subnormals
    bf = synth.bf16_to_f32(pos)
    g = np.random.default_rng(4)
    rnd = g.integers(1, 0x7F800000, size=4000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    specials = []
    for E in (-130, -127, -126, -125, -2, 0, 1, 5, 100, 126, 127):
        for m in (1.0, 1.25, 1.5, np.nextafter(np.float32(1.5), np.float32(2)), 1.75, np.nextafter(np.float32(2), np.float32(1))):
            v = np.float32(np.ldexp(np.float64(m), E))
            if np.isfinite(v) and v > 0:
                specials.append(v)
    return np.concatenate([bf, rnd, np.array(specials, np.float32)])


@pytest.mark.parametrize("mode", [0, 1])
def test_scale_by_bruteforce_scan(oracle_mod, mode):
    cases = _scale_cases()
    for a in cases[:: 3 if mode == 0 else 3]:
        assert oracle_mod.shared_exponent(float(a), mode) == exponent_by_scan(Fraction(float(a)), mode), a
    assert oracle_mod.shared_exponent(0.0, mode) == -127


def test_scale_floor_vs_ceil_relation(oracle_mod):
    """Ceiling exponent = floor exponent when the mantissa of amax is <= 1.5, else one more."""
    for m, E in [(1.0, 3), (1.5, 3), (1.5000001, 3), (1.99, -7), (1.25, 20)]:
        a = float(np.float32(m * 2.0 ** E))
        f = oracle_mod.shared_exponent(a, 0)
        c = oracle_mod.shared_exponent(a, 1)
        mant = a / 2.0 ** math.floor(math.log2(a))
        assert c == f + (1 if mant > 1.5 else 0)


# ---------------------------------------------------------------- hand-worked examples


def load_golden():
    with open(os.path.join(GOLDEN, "quant_examples.jsonl")) as f:
        return [json.loads(l) for l in f if l.strip()]


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c["name"])
def test_hand_worked_examples(oracle_mod, case):
    x = np.zeros(32, np.float32)
    x[: len(case["x"])] = case["x"]
    xb = synth.bf16_bits(x)
    codes, scales = oracle_mod.quantize_vec(xb, case["had"], case["mode"])
    want = np.zeros(32, np.uint8)
    want[: len(case["codes"])] = case["codes"]
    assert int(scales[0]) == case["scale"]
    assert np.array_equal(oracle_mod.unpack_codes(codes), want)


def test_h16_all_ones_roundtrip(oracle_mod):
    """Dequantise + inverse rotation of the all-ones block gives the ones back exactly."""
    xb = synth.bf16_bits(np.ones((1, 32), np.float32))
    codes, scales = oracle_mod.quantize(xb, 16, 0, "row")
    dq = oracle_mod.dequant_row(codes, scales)
    back = oracle_mod.rotate_f64(dq, 16)  # H16/4 is its own inverse
    assert np.array_equal(back, np.ones((1, 32)))


# ---------------------------------------------------------------- layouts


def test_layouts_consistent(oracle_mod):
    x = synth.heavy_tailed(64, 96, 7)
    for had in (1, 16, 32):
        for mode in (0, 1):
            cr, sr = oracle_mod.quantize(x, had, mode, "row")
            for r in range(0, 64, 13):
                cv, sv = oracle_mod.quantize_vec(x[r], had, mode)
                assert np.array_equal(cr[r], cv) and np.array_equal(sr[r], sv)
            ct, st = oracle_mod.quantize(x, had, mode, "colT")
            cr2, sr2 = oracle_mod.quantize(np.ascontiguousarray(x.T), had, mode, "row")
            assert np.array_equal(ct, cr2) and np.array_equal(st, sr2)
            c2, s2 = oracle_mod.quantize(x, had, mode, "2d")
            # the 2D scale is the row scale of the row with the largest block amax
            assert np.array_equal(s2, sr.reshape(2, 32, 3).max(axis=1))


def codes_2d_independent(oracle_mod, xb, had, mode):
    """The 32x32 2D layout rebuilt from pinned pieces, not from the oracle's 2D code:
    rotation along the columns by the canonical fp32 rotation (pinned above), one
    exponent per 32x32 tile by the brute-force scan over the tile's amax, and every
    element rounded by counting E2M1 midpoints in exact rationals.
    Returns per-element codes [R, C] and the scale bytes [R/32, C/32]."""
    R, C = xb.shape
    v = oracle_mod.rotate_f32(synth.bf16_to_f32(xb), had)
    codes = np.zeros((R, C), np.uint8)
    scales = np.zeros((R // 32, C // 32), np.uint8)
    for tr in range(R // 32):
        for tc in range(C // 32):
            tile = v[32 * tr:32 * tr + 32, 32 * tc:32 * tc + 32]
            e = exponent_by_scan(Fraction(float(np.abs(tile).max())), mode)
            scales[tr, tc] = e + 127
            step = Fraction(2) ** e
            for i in range(32):
                for j in range(32):
                    val = float(tile[i, j])
                    codes[32 * tr + i, 32 * tc + j] = e2m1_code_by_thresholds(Fraction(val) / step,
                                                                              math.copysign(1.0, val) < 0)
    return codes, scales


@pytest.mark.parametrize("had", [1, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_2d_codes_by_tile_exponent(oracle_mod, had, mode):
    """2D codes and bytes equal the independent rebuild on heavy-tailed data, and the
    data is such that quantising each row segment with its own exponent (a plausible
    slip) would change codes: the per-row copy differs from the 2D copy."""
    xb = synth.heavy_tailed(64, 96, 17)
    c2, s2 = oracle_mod.quantize(xb, had, mode, "2d")
    want_c, want_s = codes_2d_independent(oracle_mod, xb, had, mode)
    assert np.array_equal(s2, want_s)
    assert np.array_equal(oracle_mod.unpack_codes(c2), want_c)
    cr, _ = oracle_mod.quantize(xb, had, mode, "row")
    assert (oracle_mod.unpack_codes(cr) != want_c).sum() > 100


def load_golden_2d():
    with open(os.path.join(GOLDEN, "quant_2d_examples.jsonl")) as f:
        return [json.loads(l) for l in f if l.strip()]


@pytest.mark.parametrize("case", load_golden_2d(), ids=lambda c: c["name"])
def test_hand_worked_2d_examples(oracle_mod, case):
    """Hand-worked 32x32 tiles (tests/golden/quant_2d_examples.jsonl, each with its why)."""
    x = np.array([case["x_row0"]] + [case["x_other_rows"]] * 31, np.float32)
    want = np.array([case["codes_row0"]] + [case["codes_other_rows"]] * 31, np.uint8)
    codes, scales = oracle_mod.quantize(synth.bf16_bits(x), case["had"], case["mode"], "2d")
    assert scales.shape == (1, 1) and int(scales[0, 0]) == case["scale"]
    assert np.array_equal(oracle_mod.unpack_codes(codes), want)
    # the independent rebuild agrees with the hand-worked values too
    ic, isc = codes_2d_independent(oracle_mod, synth.bf16_bits(x), case["had"], case["mode"])
    assert int(isc[0, 0]) == case["scale"] and np.array_equal(ic, want)


# ---------------------------------------------------------------- error decomposition


def _q_star(x, amax):
    """Ideal-scale quantiser Q*: s* = amax / 6, Q*(x) = s* * RNE_grid(x / s*)."""
    s = amax / 6
    out = []
    for v in x:
        c = e2m1_code_by_thresholds(v / s, v < 0) if s != 0 else 0
        mag = [0, Fraction(1, 2), 1, Fraction(3, 2), 2, 3, 4, 6][c & 7]
        out.append((-mag if c & 8 else mag) * s)
    return out


def _decompose(oracle_mod, block_bf16, mode):
    codes, scales = oracle_mod.quantize_vec(block_bf16, 1, mode)
    e = int(scales[0]) - 127
    x = [Fraction(float(v)) for v in synth.bf16_to_f32(block_bf16)]
    q = [Fraction(oracle_mod.e2m1_value(int(c))) * Fraction(2) ** e for c in oracle_mod.unpack_codes(codes)]
    amax = max(abs(v) for v in x)
    qs = _q_star(x, amax)
    dz = [abs(v) < amax / 24 for v in x]
    e_scale = [a - b for a, b in zip(q, qs)]
    e_dz = [(b - v) if d else Fraction(0) for b, v, d in zip(qs, x, dz)]
    e_grid = [Fraction(0) if d else (b - v) for b, v, d in zip(qs, x, dz)]
    e_tot = [a - v for a, v in zip(q, x)]
    return e_scale, e_dz, e_grid, e_tot


def _dot(a, b):
    return sum(x * y for x, y in zip(a, b))


def test_deadzone_orthogonality_ceil(oracle_mod):
    """Property 1 (Decomposing MXFP4 quantization error): under the ceiling scale the
    deadzone error is pointwise orthogonal to the scale and grid errors, and the MSE
    splits with one cross term, exactly."""
    g = np.random.default_rng(5)
    for t in range(60):
        blk = g.standard_t(3, size=32).astype(np.float32) * np.float32(10 ** g.uniform(-3, 2))
        blk[g.integers(0, 32)] *= np.float32(30)
        b = synth.bf16_bits(blk)
        es, edz, eg, e = _decompose(oracle_mod, b, 1)
        assert all(a * c == 0 for a, c in zip(edz, es))
        assert _dot(edz, eg) == 0
        assert _dot(e, e) == _dot(es, es) + _dot(edz, edz) + _dot(eg, eg) + 2 * _dot(es, eg)


def test_deadzone_orthogonality_fails_for_floor_scale(oracle_mod):
    """Contrast: the OCP floor scale lies below amax/6 when the mantissa of amax
    exceeds 1.5, so the lemma's premise s_b >= s*_b fails.  With amax = 1.9, the
    floor scale is 2^-2 = 0.25 < s* = 0.3167; x = 0.07 lies in the deadzone of Q*
    (|x| < 1.9/24) but Q(x) = 0.125, so e_DZ * e_scale != 0 in every such block."""
    g = np.random.default_rng(6)
    for t in range(50):
        blk = (g.standard_normal(32) * 0.01).astype(np.float32)
        blk[0] = np.float32(1.9)
        blk[1] = np.float32(0.07)
        es, edz, eg, e = _decompose(oracle_mod, synth.bf16_bits(blk), 0)
        assert es[1] * edz[1] != 0
        # the split itself stays exact: e = e_scale + e_dz + e_grid
        assert all(a == b + c + d for a, b, c, d in zip(e, es, edz, eg))
        # and under the ceiling scale the same block satisfies the lemma
        es, edz, eg, e = _decompose(oracle_mod, synth.bf16_bits(blk), 1)
        assert all(a * c == 0 for a, c in zip(edz, es))


def test_ceiling_scale_bias_is_one_over_ln2(oracle_mod):
    """Scale bias (Decomposing MXFP4 quantization error): with the ceiling scale,
    s_b / s*_b = 2^delta, delta ~ U[0,1) when log2 amax has a uniform fractional part,
    so its mean is 1/ln 2 ~ 1.443 (the '~44%' bias)."""
    g = np.random.default_rng(7)
    amax = (2.0 ** (g.uniform(0, 1, 200000) + g.integers(-20, 20, 200000))).astype(np.float32)
    ratios = np.array([2.0 ** oracle_mod.shared_exponent(float(a), 1) * 6.0 / float(a) for a in amax[:20000]])
    assert np.all(ratios >= 1.0) and np.all(ratios < 2.0)
    assert abs(ratios.mean() - 1 / math.log(2)) < 0.01 * (1 / math.log(2))


# ---------------------------------------------------------------- GEMM


def test_gemm_single_block_by_hand(oracle_mod):
    """K = 32: C = 2^(ea+eb) * sum_k qa_k qb_k."""
    qa = np.array([2] * 16 + [10] * 16, np.uint8)   # +1 x16, -1 x16
    qb = np.array([7] * 8 + [5] * 8 + [4] * 8 + [15] * 8, np.uint8)  # 6, 3, 2, -6
    pack = lambda q: (q[0::2] | (q[1::2] << 4)).astype(np.uint8)[None, :]
    ca, cb = pack(qa), pack(qb)
    sa = np.array([[127 + 3]], np.uint8)
    sb = np.array([[127 - 5]], np.uint8)
    C, S = oracle_mod.gemm(ca, sa, cb, sb)
    dot = 8 * 6 + 8 * 3 - 8 * 2 - 8 * (-6)
    absd = 8 * 6 + 8 * 3 + 8 * 2 + 8 * 6
    assert C[0, 0] == dot * 2.0 ** (3 - 5)
    assert S[0, 0] == absd * 2.0 ** (3 - 5)


def test_gemm_equals_dequantised_matmul(oracle_mod):
    """Integer-exact block sums == fp64 matmul of the dequantised operands."""
    X, W, _ = synth.linear_inputs(64, 96, 256, 11)
    ca, sa = oracle_mod.quantize(X, 16, 0, "row")
    cb, sb = oracle_mod.quantize(W, 16, 0, "row")
    C, S = oracle_mod.gemm(ca, sa, cb, sb)
    A = oracle_mod.dequant_row(ca, sa)
    B = oracle_mod.dequant_row(cb, sb)
    assert np.allclose(C, A @ B.T, rtol=0, atol=1e-13 * np.max(np.abs(A) @ np.abs(B).T))
    assert np.allclose(S, np.abs(A) @ np.abs(B).T, rtol=1e-14, atol=0)
    Cp, Sp = oracle_mod.dot_pairs(ca[[3, 5]], sa[[3, 5]], cb[[7, 0]], sb[[7, 0]])
    assert Cp[0] == C[3, 7] and Cp[1] == C[5, 0] and Sp[0] == S[3, 7]


def test_linear_samples_match_full(oracle_mod):
    X, W, dY = synth.linear_inputs(64, 64, 96, 12)
    for had in (16, 32):
        Y, _ = oracle_mod.fprop(X, W, had, 0)
        dX, _ = oracle_mod.dgrad(dY, W, had, 1)
        dW, _ = oracle_mod.wgrad(dY, X, had, 0)
        rows, cols = [0, 5, 63], [1, 63, 7]
        assert np.array_equal(oracle_mod.fprop_sample(X, W, had, 0, rows, cols)[0], Y[rows, cols])
        assert np.array_equal(oracle_mod.dgrad_sample(dY, W, had, 1, rows, [1, 95, 7])[0], dX[rows, [1, 95, 7]])
        assert np.array_equal(oracle_mod.wgrad_sample(dY, X, had, 0, rows, [1, 95, 7])[0], dW[rows, [1, 95, 7]])


def test_linear_close_to_exact(oracle_mod):
    """The quantised linear GEMMs approximate the exact products; error is reported for
    none / H16 / H32 (the pages' claim that H16 helps on outlier data is not pinned)."""
    X, W, dY = synth.linear_inputs(256, 512, 512, 0)
    Xf, Wf, dYf = (synth.bf16_to_f32(a).astype(np.float64) for a in (X, W, dY))
    exact = {"fprop": Xf @ Wf.T, "dgrad": dYf @ Wf, "wgrad": dYf.T @ Xf}
    for had in (1, 16, 32):
        got = {"fprop": oracle_mod.fprop(X, W, had, 0)[0], "dgrad": oracle_mod.dgrad(dY, W, had, 0)[0],
               "wgrad": oracle_mod.wgrad(dY, X, had, 0)[0]}
        for k in got:
            rel = np.linalg.norm(got[k] - exact[k]) / np.linalg.norm(exact[k])
            assert rel < 0.35, (had, k, rel)


# ---------------------------------------------------------------- error decomposition sums


def test_error_decomposition_sums_match_exact_rationals(oracle_mod):
    """The fp64 sums of the oracle's decomposition equal the exact rational sums of the
    component definitions (computed here from the oracle's codes with Fractions), and
    satisfy the MSE identity with one cross term under the ceiling scale."""
    g = np.random.default_rng(11)
    blk = (g.standard_t(3, size=(4, 64)) * 0.3).astype(np.float32)
    blk[0, 3] *= 40
    xb = synth.bf16_bits(blk)
    d = oracle_mod.error_decomposition(xb, 1, 1)
    tot = {"e2": 0, "scale2": 0, "dz2": 0, "grid2": 0, "scale_grid": 0, "n_deadzone": 0}
    for r in range(4):
        for b in range(2):
            es, edz, eg, e = _decompose(oracle_mod, np.ascontiguousarray(xb[r, 32 * b:32 * b + 32]), 1)
            tot["e2"] += _dot(e, e)
            tot["scale2"] += _dot(es, es)
            tot["dz2"] += _dot(edz, edz)
            tot["grid2"] += _dot(eg, eg)
            tot["scale_grid"] += _dot(es, eg)
            amax = max(abs(Fraction(float(v))) for v in synth.bf16_to_f32(xb[r, 32 * b:32 * b + 32]))
            tot["n_deadzone"] += sum(abs(Fraction(float(v))) < amax / 24 for v in synth.bf16_to_f32(xb[r, 32 * b:32 * b + 32]))
    for k, v in tot.items():
        assert abs(d[k] - float(v)) <= 1e-12 * max(1.0, abs(float(v))), (k, d[k], float(v))
    assert d["n"] == 256
    assert abs(d["e2"] - (d["scale2"] + d["dz2"] + d["grid2"] + 2 * d["scale_grid"])) <= 1e-12 * d["e2"]


def test_error_decomposition_h16_reduces_error_on_outliers(oracle_mod):
    """Reported, not a pin of the pages' numbers: on outlier-heavy activations the
    rotation lowers the total MXFP4 error."""
    X = synth.activations(256, 512, 0)
    none = oracle_mod.error_decomposition(X, 1, 1)
    h16 = oracle_mod.error_decomposition(X, 16, 1)
    assert h16["e2"] < none["e2"]


# ----------------------------------------------------------------- canonical vs exact rotation
def _bf16_bits(vals):
    f = np.asarray(vals, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "values must be exact in bf16"
    return (bits >> 16).astype(np.uint16)


def test_rotation_divergence_is_zero_without_rotation(oracle_mod):
    """With no rotation the exact and the canonical values are the same bf16 inputs, so
    the exact-rotation quantiser must agree with the canonical one on every block."""
    X, W, dY = synth.linear_inputs(256, 512, 512, 0)
    for a in (X, W, dY):
        for mode in (0, 1):
            d = oracle_mod.rotation_divergence(a, oracle_mod.HAD_NONE, mode)
            assert d["blocks_differ"] == 0 and d["bytes_differ"] == 0 and d["blocks"] == a.size // 32


@pytest.mark.parametrize("mode", [0, 1])
def test_rotation_divergence_detects_fp32_rounding(oracle_mod, mode):
    """Hand-worked block [5*2^22, 1, 0, ...] under H16 (normalised by 1/4, exact).  In
    fp32 the butterfly sums 5*2^22 +- 1 are ties (ulp 2 at 2^24) that round to the even
    neighbour 5*2^22, so every canonical value is 5*2^20, the amax is 5*2^20 = 1.25 * 2^22
    and e = 20 in both scale modes: u = 5, a tie between 4 and 6, rounds to 4.  Exactly,
    the eight values (5*2^22 + 1)/4 give u = 5 + 2^-22, which rounds to 6, with the same
    byte.  So exactly one block differs, and not in its byte."""
    blk = np.zeros(64, np.float32)
    blk[0], blk[1] = 5.0 * 2.0 ** 22, 1.0
    x = _bf16_bits(blk).reshape(1, 64)
    d = oracle_mod.rotation_divergence(x, oracle_mod.HAD_16, mode)
    assert d == {"blocks_differ": 1, "bytes_differ": 0, "blocks": 2}
    # the canonical codes are the tie's even choice (4 -> code 6) on all 16 rotated values
    codes, scales = oracle_mod.quantize(x, oracle_mod.HAD_16, mode, "row")
    assert int(scales[0, 0]) == 127 + 20
    assert np.all(oracle_mod.unpack_codes(codes)[0, :16] % 8 == 6)
    # without the rotation the block is quantised from the same values on both sides
    assert oracle_mod.rotation_divergence(x, oracle_mod.HAD_NONE, mode)["blocks_differ"] == 0


def test_rotation_divergence_on_workload_data(oracle_mod):
    """Report (a diagnostic, not a failure): on the correctness and sweep workloads the
    canonical fp32 order changes the quantised result of at most a handful of blocks in
    a million."""
    X, W, dY = synth.linear_inputs(256, 512, 512, 0)
    xs = synth.heavy_tailed(1024, 4096, 1000)
    for a in (X, W, dY, xs):
        for had in (oracle_mod.HAD_16, oracle_mod.HAD_32):
            for mode in (0, 1):
                d = oracle_mod.rotation_divergence(a, had, mode)
                print(f"rotation divergence {a.shape} H{had} mode {mode}: {d}")
                assert d["blocks_differ"] <= max(1, d["blocks"] // 100000)


def test_oracle_refuses_library_rotation_codes(oracle_mod):
    """The oracle takes the Hadamard block size (1, 16, 32); the library's 0 for "no
    rotation", or any other value, is refused before the C code runs, as is a scale rule
    other than 0 or 1."""
    x = synth.activations(32, 64, 1)
    for bad in (0, 8, 64):
        with pytest.raises(ValueError):
            oracle_mod.quantize(x, bad, 0, "row")
        with pytest.raises(ValueError):
            oracle_mod.rotate_f32(np.zeros((1, 32), np.float32), bad)
    with pytest.raises(ValueError):
        oracle_mod.quantize(x, 16, 2, "row")
    c, s = oracle_mod.quantize(x, 1, 0, "row")  # 1 = no rotation is accepted
    assert c.shape == (32, 32) and s.shape == (32, 2)
