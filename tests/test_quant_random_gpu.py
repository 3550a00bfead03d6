"""GPU randomised quantiser baselines vs the CPU oracle ("Pretraining Large Language
Models with MXFP4 on Native FP4 Hardware", A.2 random sign flips; stochastic
rounding): with the same sign bitmasks and random integers, codes and E8M0 bytes are
bit-exact."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import ORACLE_HAD, gpu_ready

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return gpu_ready()


def same(got, want, what):
    if not np.array_equal(got, want):
        i = np.argwhere(got != want)[:4]
        raise AssertionError(f"{what} differ at {i.tolist()}: gpu {got[tuple(i[0])]} oracle {want[tuple(i[0])]} "
                             f"({int((got != want).sum())} of {got.size})")


def dev(torch, a):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if a.dtype == np.uint16 else a.dtype))
    return t.cuda()


@pytest.mark.parametrize("shape", [(64, 256), (96, 160), (192, 1056), (32, 32), (128, 384)])
@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("opts", ["signs", "sr", "both"])
def test_randomised_bit_exact(torch, shape, had, mode, opts):
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = shape
    g = np.random.default_rng(R * 7 + C + had + mode)
    xb = synth.heavy_tailed(R, C, 700 + R + C + had)
    cs = oracle.pack_signs(g.random(C) < 0.5) if opts != "sr" else None
    rs = oracle.pack_signs(g.random(R) < 0.5) if opts != "sr" else None
    srr = g.integers(0, 65536, (R, C)).astype(np.uint16) if opts != "signs" else None
    src = g.integers(0, 65536, (C, R)).astype(np.uint16) if opts != "signs" else None
    layouts = mx.LAYOUT_ROW | mx.LAYOUT_COLT
    out = mx.rotate_quantize_rand(mx.bf16_tensor(xb), had=had, mode=mode, layouts=layouts,
                                  col_signs=None if cs is None else dev(torch, cs),
                                  row_signs=None if rs is None else dev(torch, rs),
                                  sr_row=None if srr is None else dev(torch, srr),
                                  sr_colT=None if src is None else dev(torch, src), sf_layout=mx.SF_MMA)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for key, signs, sr in (("row", cs, srr), ("colT", rs, src)):
        wc, ws = oracle.quantize_rand(xb, ORACLE_HAD[had], mode, key, signs=signs, sr=sr)
        what = f"{key} {shape} had={had} mode={mode} {opts}"
        same(out[key].plain_scales(), ws, what + " scales")
        same(out[key].codes.cpu().numpy(), wc, what + " codes")


@pytest.mark.parametrize("had", [16, 32])
def test_randomised_row_only_ragged_rows(torch, had):
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = 200, 1056
    g = np.random.default_rng(had)
    xb = synth.heavy_tailed(R, C, 800 + had)
    cs = oracle.pack_signs(g.random(C) < 0.5)
    srr = g.integers(0, 65536, (R, C)).astype(np.uint16)
    out = mx.rotate_quantize_rand(mx.bf16_tensor(xb), had=had, mode=1, layouts=mx.LAYOUT_ROW, col_signs=dev(torch, cs),
                                  sr_row=dev(torch, srr), sf_layout=mx.SF_PLAIN)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    wc, ws = oracle.quantize_rand(xb, ORACLE_HAD[had], 1, "row", signs=cs, sr=srr)
    same(out["row"].plain_scales(), ws, "row scales")
    same(out["row"].codes.cpu().numpy(), wc, "row codes")


def test_random_signs_cancel_in_the_gemm(torch):
    """Fprop with the same random column signs on X and W: Y = X W^T within the GEMM
    tolerance of the oracle's quantised product, and close to the bf16 product."""
    from mxfp4_precision_gemms_gb300 import binding as mx
    from tests.gpu_util import assert_within

    X, W, _ = synth.linear_inputs(256, 384, 1024, 21)
    signs = oracle.pack_signs(np.random.default_rng(4).random(1024) < 0.5)
    sd = dev(torch, signs)
    qx = mx.rotate_quantize_rand(mx.bf16_tensor(X), had=16, col_signs=sd)["row"]
    qw = mx.rotate_quantize_rand(mx.bf16_tensor(W), had=16, col_signs=sd)["row"]
    Y = mx.gemm(qx, qw)
    torch.cuda.synchronize()
    cx, sx = oracle.quantize_rand(X, 16, 0, "row", signs=signs)
    cw, sw = oracle.quantize_rand(W, 16, 0, "row", signs=signs)
    want, S = oracle.gemm(cx, sx, cw, sw)
    got = Y.double().cpu().numpy()
    assert_within(got, want, S, what="random-sign Fprop")
    exact = synth.bf16_to_f32(X).astype(np.float64) @ synth.bf16_to_f32(W).astype(np.float64).T
    assert np.linalg.norm(got - exact) < 0.2 * np.linalg.norm(exact)


def test_sr_argument_checks(torch):
    from mxfp4_precision_gemms_gb300 import binding as mx

    x = mx.bf16_tensor(synth.heavy_tailed(64, 128, 1))
    r = dev(torch, np.zeros((64, 128), np.uint16))
    with pytest.raises(RuntimeError):  # SR for the row copy only, both layouts requested
        mx.rotate_quantize_rand(x, layouts=mx.LAYOUT_ROW | mx.LAYOUT_COLT, sr_row=r)
    with pytest.raises(RuntimeError):  # 2D layout with an option
        mx.rotate_quantize_rand(x, layouts=mx.LAYOUT_2D, sr_row=r)


@pytest.mark.parametrize("pad,offset", [(8, 0), (0, 8)])
def test_randomised_strided_inputs(torch, pad, offset):
    """Random signs and stochastic rounding on both copies, x read through a view with
    leading dimension C + pad starting `offset` elements into a larger buffer."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = 128, 384
    g = np.random.default_rng(31 + pad + offset)
    xb = synth.heavy_tailed(R, C, 950 + pad + offset)
    big = torch.zeros((R + 1) * (C + pad) + offset, dtype=torch.bfloat16, device="cuda")
    x = big[offset:offset + R * (C + pad)].view(R, C + pad)[:, :C]
    x.copy_(mx.bf16_tensor(xb))
    cs = oracle.pack_signs(g.random(C) < 0.5)
    rs = oracle.pack_signs(g.random(R) < 0.5)
    srr = g.integers(0, 65536, (R, C)).astype(np.uint16)
    src = g.integers(0, 65536, (C, R)).astype(np.uint16)
    out = mx.rotate_quantize_rand(x, had=16, mode=0, layouts=mx.LAYOUT_ROW | mx.LAYOUT_COLT,
                                  col_signs=dev(torch, cs), row_signs=dev(torch, rs), sr_row=dev(torch, srr),
                                  sr_colT=dev(torch, src), sf_layout=mx.SF_MMA)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for key, signs, sr in (("row", cs, srr), ("colT", rs, src)):
        wc, ws = oracle.quantize_rand(xb, ORACLE_HAD[16], 0, key, signs=signs, sr=sr)
        same(out[key].plain_scales(), ws, f"{key} strided scales")
        same(out[key].codes.cpu().numpy(), wc, f"{key} strided codes")


# ---------------------------------------------------------------- in-kernel Philox4x32-10
@pytest.mark.parametrize("shape", [(64, 256), (96, 160), (192, 1056), (32, 32), (256, 512)])
@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("opts", ["signs", "sr", "both"])
def test_philox_generated_bit_exact(torch, shape, had, mode, opts):
    """Random signs and stochastic rounding drawn in the kernel from Philox4x32-10:
    codes and bytes bit-exact with the oracle, which draws the same numbers from its own
    generator (pinned to the published known-answer vectors) and runs the pinned
    randomised quantiser; and byte-identical to the array-input kernel given those
    numbers."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = shape
    xb = synth.heavy_tailed(R, C, 900 + R + C + had)
    seeds = dict(col_sign_seed=0x1234_5678_9ABC_DEF0 + had if opts != "sr" else None,
                 row_sign_seed=(7 << 40) + mode if opts != "sr" else None,
                 sr_seed=0xFEED_0000_0000_0001 + R if opts != "signs" else None)
    layouts = mx.LAYOUT_ROW | mx.LAYOUT_COLT
    x = mx.bf16_tensor(xb)
    out = mx.rotate_quantize_philox(x, had=had, mode=mode, layouts=layouts, **seeds)
    cs = None if seeds["col_sign_seed"] is None else oracle.philox_signs(seeds["col_sign_seed"], C)
    rs = None if seeds["row_sign_seed"] is None else oracle.philox_signs(seeds["row_sign_seed"], R)
    srr = None if seeds["sr_seed"] is None else oracle.philox_sr(seeds["sr_seed"], R, C, 0)
    src = None if seeds["sr_seed"] is None else oracle.philox_sr(seeds["sr_seed"], C, R, 1)
    arr = mx.rotate_quantize_rand(x, had=had, mode=mode, layouts=layouts,
                                  col_signs=None if cs is None else dev(torch, cs),
                                  row_signs=None if rs is None else dev(torch, rs),
                                  sr_row=None if srr is None else dev(torch, srr),
                                  sr_colT=None if src is None else dev(torch, src))
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for key in ("row", "colT"):
        wc, ws = oracle.quantize_philox(xb, ORACLE_HAD[had], mode, key, **seeds)
        what = f"philox {key} {shape} had={had} mode={mode} {opts}"
        same(out[key].plain_scales(), ws, what + " scales")
        same(out[key].codes.cpu().numpy(), wc, what + " codes")
        assert torch.equal(out[key].codes, arr[key].codes) and torch.equal(out[key].scales, arr[key].scales)


def test_philox_signs_cancel_in_the_gemm(torch):
    """X and W quantised with the same Philox sign vector over K (one seed): the Fprop
    GEMM of the two copies is within tolerance of the oracle's product of the same
    codes, and close to the bf16 product (the signs cancel like the rotation)."""
    from mxfp4_precision_gemms_gb300 import binding as mx
    from tests.gpu_util import assert_within

    X, W, _ = synth.linear_inputs(256, 384, 1024, 31)
    qx = mx.rotate_quantize_philox(mx.bf16_tensor(X), had=16, col_sign_seed=2024, sr_seed=5)["row"]
    qw = mx.rotate_quantize_philox(mx.bf16_tensor(W), had=16, col_sign_seed=2024, sr_seed=6)["row"]
    Y = mx.gemm(qx, qw)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    cx, sx = oracle.quantize_philox(X, 16, 0, "row", col_sign_seed=2024, sr_seed=5)
    cw, sw = oracle.quantize_philox(W, 16, 0, "row", col_sign_seed=2024, sr_seed=6)
    want, S = oracle.gemm(cx, sx, cw, sw)
    assert_within(Y.double().cpu().numpy(), want, S, what="philox-signed fprop")
    dense = synth.bf16_to_f32(X).astype(np.float64) @ synth.bf16_to_f32(W).astype(np.float64).T
    rel = np.linalg.norm(Y.double().cpu().numpy() - dense) / np.linalg.norm(dense)
    assert rel < 0.25, rel
