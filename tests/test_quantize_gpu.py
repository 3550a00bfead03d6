"""GPU rotate+quantise vs the CPU oracle: packed codes and E8M0 bytes bit-exact.

Inputs are the seeded synthetic recipes (config-0 linear-layer tensors, config-1
heavy-tailed sweep tensors), ragged shapes and exhaustive bf16 sweeps."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import ORACLE_HAD, gpu_ready

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return gpu_ready()


def gpu_quantize(torch, xbits, had, mode, layouts, sf):
    from mxfp4_precision_gemms_gb300 import binding as mx

    x = mx.bf16_tensor(xbits)
    outs = mx.rotate_quantize(x, had=had, mode=mode, layouts=layouts, sf_layout=sf)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return {k: (v.codes.cpu().numpy(), v.plain_scales()) for k, v in outs.items()}


def check(torch, xbits, had, mode, layouts, sf, what=""):
    from mxfp4_precision_gemms_gb300 import binding as mx

    got = gpu_quantize(torch, xbits, had, mode, layouts, sf)
    names = {mx.LAYOUT_ROW: "row", mx.LAYOUT_COLT: "colT", mx.LAYOUT_2D: "2d"}
    for bit, key in names.items():
        if not layouts & bit:
            continue
        want_c, want_s = oracle.quantize(xbits, ORACLE_HAD[had], mode, key)
        gc, gs = got[key]
        if not np.array_equal(gs, want_s):
            i = np.argwhere(gs != want_s)[:4]
            raise AssertionError(f"{what} {key} scales differ at {i.tolist()}: gpu {gs[tuple(i[0])]} "
                                 f"oracle {want_s[tuple(i[0])]} ({int((gs != want_s).sum())} bytes)")
        if not np.array_equal(gc, want_c):
            i = np.argwhere(gc != want_c)[:4]
            raise AssertionError(f"{what} {key} codes differ at {i.tolist()}: gpu {gc[tuple(i[0])]:#04x} "
                                 f"oracle {want_c[tuple(i[0])]:#04x} ({int((gc != want_c).sum())} bytes)")


@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("sf", [0, 1])
def test_config0_linear_tensors(torch, had, mode, sf):
    X, W, dY = synth.linear_inputs(256, 512, 512, 0)
    for name, t in (("X", X), ("W", W), ("dY", dY)):
        check(torch, t, had, mode, 1 | 2, sf, f"{name} had={had} mode={mode}")
        check(torch, t, had, mode, 1, sf, f"{name} row-only")
        check(torch, t, had, mode, 2, sf, f"{name} colT-only")


@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_config0_2d(torch, had, mode):
    X, W, dY = synth.linear_inputs(256, 512, 512, 0)
    for t in (X, dY):
        check(torch, t, had, mode, 4, 0, "2d")


@pytest.mark.parametrize("shape", [(96, 160), (33, 96), (1, 32), (160, 224), (64, 32), (320, 1056)])
def test_ragged_shapes(torch, shape):
    R, C = shape
    x = synth.heavy_tailed(R, C, 1000 + R + C)
    for had in (0, 16, 32):
        for sf in (0, 1):
            check(torch, x, had, 1, 1, sf, f"ragged {shape} row")
            if R % 32 == 0:
                check(torch, x, had, 0, 1 | 2, sf, f"ragged {shape} row+colT")
        if R % 32 == 0:
            check(torch, x, had, 0, 4, 0, f"ragged {shape} 2d")


def _finite_bf16_patterns():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    e = (b >> 7) & 0xFF
    return b[e != 0xFF]


@pytest.mark.parametrize("mode", [0, 1])
def test_exhaustive_bf16_consecutive_blocks(torch, mode):
    """All finite bf16 patterns, 32 consecutive patterns per block."""
    p = _finite_bf16_patterns()
    p = p[: (p.size // 32) * 32].reshape(-1, 32)
    rows = (p.shape[0] // 32) * 32
    check(torch, np.ascontiguousarray(p[:rows]), 0, mode, 1 | 2, 1, "consecutive")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("had", [0, 16])
def test_exhaustive_bf16_under_fixed_scale(torch, mode, had):
    """Every finite bf16 pattern with |x| <= 4*2^e quantised in blocks whose amax is
    4*2^e, for several e: exercises every rounding tie and the deadzone."""
    vals = synth.bf16_to_f32(_finite_bf16_patterns())
    blocks = []
    g = np.random.default_rng(9)
    for e in (-128, -100, -3, 0, 7, 90):
        anchor = np.float32(4.0 * 2.0 ** e)
        sel = _finite_bf16_patterns()[np.abs(vals) <= anchor]
        sel = sel[g.permutation(sel.size)]
        n = (sel.size // 31) * 31
        body = sel[:n].reshape(-1, 31)
        a = np.full((body.shape[0], 1), synth.bf16_bits(np.array([anchor]))[0], np.uint16)
        blocks.append(np.concatenate([a, body], axis=1))
    x = np.concatenate(blocks)
    x = np.ascontiguousarray(x[: (x.shape[0] // 32) * 32])
    check(torch, x, had, mode, 1 | 2, 1, f"fixed-scale e sweep had={had}")


@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_config1_4096(torch, had, mode):
    x = synth.heavy_tailed(4096, 4096, 1000)
    check(torch, x, had, mode, 1 | 2, 1, "4096^2 row+colT")
    check(torch, x, had, mode, 4, 0, "4096^2 2d")


@pytest.fixture(scope="module")
def x_8192x14336():
    return synth.heavy_tailed(8192, 14336, 1001)


@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_config1_8192x14336(torch, x_8192x14336, had, mode):
    """The whole config-1 sweep at its full size, every kernel instance the benchmark's
    sweep times: the row + transposed pass and the row-only and transposed-only passes
    (scales in the GEMM's order), and the 2D pass (plain scales)."""
    x = x_8192x14336
    what = f"8192x14336 had={had} mode={mode}"
    check(torch, x, had, mode, 1 | 2, 1, what + " row+colT")
    check(torch, x, had, mode, 1, 1, what + " row")
    check(torch, x, had, mode, 2, 1, what + " colT")
    check(torch, x, had, mode, 4, 0, what + " 2d")


def test_empty_input(torch):
    from mxfp4_precision_gemms_gb300 import binding as mx

    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    outs = mx.rotate_quantize(x, layouts=1 | 2)
    assert outs["row"].rows == 0


@pytest.mark.parametrize("layouts", [1, 2, 3, 4])
@pytest.mark.parametrize("pad,offset", [(8, 0), (0, 8), (16, 0), (24, 16)])
def test_strided_and_offset_inputs(torch, layouts, pad, offset):
    """x as a view into a larger bf16 buffer: leading dimension C + pad and a start
    offset of `offset` elements (16-byte granules).  Rows that start on a 32-byte
    boundary take the kernel's 32-byte loads, the others its 16-byte loads; both must
    give the oracle's bytes for the same values."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = 320, 1056
    xbits = synth.heavy_tailed(R, C, 77 + pad + offset)
    big = torch.zeros((R + 1) * (C + pad) + offset, dtype=torch.bfloat16, device="cuda")
    view = big[offset:offset + R * (C + pad)].view(R, C + pad)[:, :C]
    view.copy_(mx.bf16_tensor(xbits))
    assert view.stride(0) == C + pad and view.data_ptr() % 16 == 0
    outs = mx.rotate_quantize(view, had=16, mode=0, layouts=layouts, sf_layout=0)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    names = {mx.LAYOUT_ROW: "row", mx.LAYOUT_COLT: "colT", mx.LAYOUT_2D: "2d"}
    for bit, key in names.items():
        if not layouts & bit:
            continue
        want_c, want_s = oracle.quantize(xbits, ORACLE_HAD[16], 0, key)
        gc, gs = outs[key].codes.cpu().numpy(), outs[key].plain_scales()
        assert np.array_equal(gs, want_s), f"{key} scales, pad {pad} offset {offset}"
        assert np.array_equal(gc, want_c), f"{key} codes, pad {pad} offset {offset}"


@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("layouts", [1, 2, 3])
def test_pair_launch_equals_two_calls_and_the_oracle(torch, had, mode, layouts):
    """mxfp4_rotate_quantize_pair (two matrices with the same columns in one launch):
    every output byte-identical to two separate rotate_quantize calls, bit-exact with the
    oracle, for row counts that end mid-tile on either side and plain and MMA scales."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    names = {mx.LAYOUT_ROW: "row", mx.LAYOUT_COLT: "colT"}
    for (ra, rb, c), seed in (((256, 512, 512), 1), ((96, 160, 256), 2), ((224, 32, 384), 3)):
        A = synth.activations(ra, c, seed)
        B = synth.weights(rb, c, seed + 100)
        for sf in (0, 1):
            a, b = mx.bf16_tensor(A), mx.bf16_tensor(B)
            pa, pb = mx.rotate_quantize_pair(a, b, had=had, mode=mode, layouts=layouts, sf_layout=sf)
            sa = mx.rotate_quantize(a, had=had, mode=mode, layouts=layouts, sf_layout=sf)
            sb = mx.rotate_quantize(b, had=had, mode=mode, layouts=layouts, sf_layout=sf)
            torch.cuda.synchronize()
            assert mx.device_status() == 0
            for bit, key in names.items():
                if not layouts & bit:
                    continue
                for got, ref, bits in ((pa, sa, A), (pb, sb, B)):
                    assert torch.equal(got[key].codes, ref[key].codes), f"{key} codes {ra}/{rb}x{c}"
                    assert torch.equal(got[key].scales, ref[key].scales), f"{key} scales {ra}/{rb}x{c}"
                    assert got[key].had == had and got[key].mode == mode
                    want_c, want_s = oracle.quantize(bits, ORACLE_HAD[had], mode, key)
                    assert np.array_equal(got[key].codes.cpu().numpy(), want_c)
                    assert np.array_equal(got[key].plain_scales(), want_s)


def test_pair_launch_rejects_mismatched_columns(torch):
    from mxfp4_precision_gemms_gb300 import binding as mx

    a = mx.bf16_tensor(synth.activations(64, 256, 1))
    b = mx.bf16_tensor(synth.activations(64, 512, 2))
    with pytest.raises(ValueError):
        mx.rotate_quantize_pair(a, b)


def _random_quant_cases(count, seed):
    g = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        R = int(g.integers(1, 60)) * 32      # rows in whole blocks (the transposed and 2D copies need it)
        C = int(g.integers(1, 90)) * 32
        lay = int(g.choice([1, 2, 3, 4]))
        sf = 0 if lay == 4 else int(g.integers(0, 2))
        out.append((R, C, int(g.choice([0, 16, 32])), int(g.integers(0, 2)), lay, sf))
    return out


@pytest.mark.parametrize("R,C,had,mode,layouts,sf", _random_quant_cases(24, 2027))
def test_random_shapes_bit_exact(torch, R, C, had, mode, layouts, sf):
    """Seeded random shapes, rotations, scale rules, layouts and scale orders: codes and
    scale bytes bit-exact against the oracle."""
    x = synth.heavy_tailed(R, C, R * 7 + C)
    check(torch, x, had, mode, layouts, sf, f"{R}x{C} had={had} mode={mode} layouts={layouts} sf={sf}")
