"""GPU quantiser fixes vs the CPU oracle ("Decomposing MXFP4 quantization error for LLM
reinforcement learning", OF and MBS): codes, E8M0 bytes and MBS bytes bit-exact; the
GEMM over an OF operand (two accumulating MXFP4 GEMMs) within the GEMM tolerance."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import ORACLE_HAD, assert_within, gpu_ready

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return gpu_ready()


def same(got, want, what):
    if not np.array_equal(got, want):
        i = np.argwhere(got != want)[:4]
        raise AssertionError(f"{what} differ at {i.tolist()}: gpu {got[tuple(i[0])]} oracle {want[tuple(i[0])]} "
                             f"({int((got != want).sum())} of {got.size})")


SHAPES = [(64, 256), (96, 160), (200, 1056), (1, 32), (130, 384)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_of_bit_exact(torch, shape, had, mode):
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = shape
    xb = synth.heavy_tailed(R, C, 500 + R + C + had + mode)
    for alpha_log2, sf in ((0, mx.SF_PLAIN), (-1, mx.SF_MMA)):
        q1, q2 = mx.rotate_quantize_of(mx.bf16_tensor(xb), had=had, mode=mode, alpha_log2=alpha_log2, sf_layout=sf)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        c1, s1, c2, s2, bad = oracle.quantize_of(xb, ORACLE_HAD[had], mode, alpha_log2)
        assert bad == 0
        what = f"OF {shape} had={had} mode={mode} alpha_log2={alpha_log2}"
        same(q1.plain_scales(), s1, what + " q1 scales")
        same(q1.codes.cpu().numpy(), c1, what + " q1 codes")
        same(q2.plain_scales(), s2, what + " q2 scales")
        same(q2.codes.cpu().numpy(), c2, what + " q2 codes")


@pytest.mark.parametrize("shape", [(64, 256), (96, 128), (200, 1024), (1, 128), (130, 384)])
@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_mbs_bit_exact(torch, shape, had, mode):
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = shape
    xb = synth.heavy_tailed(R, C, 600 + R + C + had + mode)
    for sf in (mx.SF_PLAIN, mx.SF_MMA):
        q, mbs = mx.rotate_quantize_mbs(mx.bf16_tensor(xb), had=had, mode=mode, sf_layout=sf)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        codes, scales, kb = oracle.quantize_mbs(xb, ORACLE_HAD[had], mode)
        what = f"MBS {shape} had={had} mode={mode} sf={sf}"
        same(mbs.cpu().numpy(), kb, what + " mbs bytes")
        same(q.plain_scales(), scales, what + " scales")
        same(q.codes.cpu().numpy(), codes, what + " codes")


def test_fixes_on_linear_activations_at_scale(torch):
    """Config-2 sized activations (8192 x 4096, 1% outlier channels), H16, floor: every
    byte of both fixes against the oracle."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    xb = synth.activations(8192, 4096, 7)
    x = mx.bf16_tensor(xb)
    q1, q2 = mx.rotate_quantize_of(x, had=16, mode=0, alpha_log2=-1, sf_layout=mx.SF_MMA)
    q, mbs = mx.rotate_quantize_mbs(x, had=16, mode=0, sf_layout=mx.SF_MMA)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    c1, s1, c2, s2, _ = oracle.quantize_of(xb, 16, 0, -1)
    same(q1.codes.cpu().numpy(), c1, "OF q1 codes")
    same(q1.plain_scales(), s1, "OF q1 scales")
    same(q2.codes.cpu().numpy(), c2, "OF q2 codes")
    same(q2.plain_scales(), s2, "OF q2 scales")
    codes, scales, kb = oracle.quantize_mbs(xb, 16, 0)
    same(mbs.cpu().numpy(), kb, "MBS bytes")
    same(q.plain_scales(), scales, "MBS scales")
    same(q.codes.cpu().numpy(), codes, "MBS codes")


def test_gemm_over_an_of_operand(torch):
    """Y = X_OF W^T as GEMM(q1, Wq) + GEMM(q2, Wq) (fp32, accumulate): within the GEMM
    tolerance of the oracle's dq(q1) Wq^T + dq(q2) Wq^T."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    X, W, _ = synth.linear_inputs(384, 512, 1024, 8)
    q1, q2 = mx.rotate_quantize_of(mx.bf16_tensor(X), had=16, mode=0, alpha_log2=-1)
    wq = mx.rotate_quantize(mx.bf16_tensor(W), had=16, mode=0, layouts=mx.LAYOUT_ROW)["row"]
    Y = mx.gemm(q1, wq)
    mx.gemm(q2, wq, accumulate=True, out=Y)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    c1, s1, c2, s2, _ = oracle.quantize_of(X, 16, 0, -1)
    cw, sw = oracle.quantize(W, 16, 0, "row")
    C1, S1 = oracle.gemm(c1, s1, cw, sw)
    C2, S2 = oracle.gemm(c2, s2, cw, sw)
    assert_within(Y.double().cpu().numpy(), C1 + C2, S1 + S2, what="OF GEMM")
    # the OF operand is closer to the rotated X than the plain one
    v = oracle.rotate_f32(synth.bf16_to_f32(X), 16).astype(np.float64)
    err_of = np.abs(oracle.dequant_row(c1, s1) + oracle.dequant_row(c2, s2) - v).sum()
    err_q = np.abs(oracle.dequant_row(c1, s1) - v).sum()
    assert err_of < err_q


def test_fix_argument_checks(torch):
    from mxfp4_precision_gemms_gb300 import binding as mx

    x = mx.bf16_tensor(synth.heavy_tailed(64, 96, 1))
    with pytest.raises(RuntimeError):
        mx.rotate_quantize_mbs(x)  # cols % 128 != 0
    with pytest.raises(RuntimeError):
        mx.rotate_quantize_of(x, alpha_log2=1)
    e = mx.bf16_tensor(np.zeros((0, 128), np.uint16))
    q, mbs = mx.rotate_quantize_mbs(e)
    assert q.rows == 0 and mbs.numel() == 0


def _strided(torch, xb, pad, offset):
    """x's values in a view with leading dimension C + pad, starting `offset` elements
    into a larger buffer."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = xb.shape
    big = torch.zeros((R + 1) * (C + pad) + offset, dtype=torch.bfloat16, device="cuda")
    view = big[offset:offset + R * (C + pad)].view(R, C + pad)[:, :C]
    view.copy_(mx.bf16_tensor(xb))
    return view


@pytest.mark.parametrize("pad,offset", [(8, 0), (0, 8), (136, 24)])
def test_of_and_mbs_strided_inputs(torch, pad, offset):
    """OF and MBS read x through its leading dimension and start address: a view into a
    larger buffer gives the oracle's bytes for the same values."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    R, C = 130, 384
    xb = synth.heavy_tailed(R, C, 900 + pad + offset)
    x = _strided(torch, xb, pad, offset)
    q1, q2 = mx.rotate_quantize_of(x, had=16, mode=0, alpha_log2=-1, sf_layout=mx.SF_PLAIN)
    q, mbs = mx.rotate_quantize_mbs(x, had=16, mode=1, sf_layout=mx.SF_PLAIN)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    c1, s1, c2, s2, bad = oracle.quantize_of(xb, ORACLE_HAD[16], 0, -1)
    assert bad == 0
    same(q1.plain_scales(), s1, "OF q1 scales")
    same(q1.codes.cpu().numpy(), c1, "OF q1 codes")
    same(q2.plain_scales(), s2, "OF q2 scales")
    same(q2.codes.cpu().numpy(), c2, "OF q2 codes")
    c, s, m = oracle.quantize_mbs(xb, ORACLE_HAD[16], 1)
    same(q.plain_scales(), s, "MBS scales")
    same(q.codes.cpu().numpy(), c, "MBS codes")
    same(mbs.cpu().numpy(), m, "MBS bytes")


# ---------------------------------------------------------------- GEMM over MBS operands
def _mbs_operands(mx, X, W, which, had=16, mode=0):
    """GPU MBS (or plain) copies of X and W and the oracle's own copies of the same."""
    xa, xb = mx.bf16_tensor(X), mx.bf16_tensor(W)
    out = []
    for x, bits, use in ((xa, X, which in ("both", "a")), (xb, W, which in ("both", "b"))):
        if use:
            q, m = mx.rotate_quantize_mbs(x, had=had, mode=mode)
            oc, os_, om = oracle.quantize_mbs(bits, had, mode)
        else:
            q, m = mx.rotate_quantize(x, had=had, mode=mode, layouts=mx.LAYOUT_ROW)["row"], None
            (oc, os_), om = oracle.quantize(bits, had, mode, "row"), None
        out.append((q, m, oc, os_, om))
    return out


@pytest.mark.parametrize("shape", [(256, 256, 512), (200, 136, 384), (384, 520, 1024)])
@pytest.mark.parametrize("which", ["both", "a", "b"])
def test_gemm_over_mbs_operands(torch, shape, which):
    """C = x_hat_A x_hat_B^T with each 128-element macro block's partial product scaled by
    its postscale factors: within the GEMM tolerance of the oracle's fp64 MBS GEMM, for
    ragged shapes (an odd number of macro blocks: K = 384), fp32 and bf16 output, and
    accumulation."""
    from mxfp4_precision_gemms_gb300 import binding as mx
    from tests.gpu_util import assert_within

    M, N, K = shape
    X, W, _ = synth.linear_inputs(M, N, K, 90 + M)
    (qa, ma, ca, sa, oma), (qb, mb, cb, sb, omb) = _mbs_operands(mx, X, W, which)
    want, S = oracle.gemm_mbs(ca, sa, oma, cb, sb, omb)
    C = mx.gemm_mbs(qa, ma, qb, mb)
    Cb = mx.gemm_mbs(qa, ma, qb, mb, out_dtype=mx.OUT_BF16)
    Cacc = torch.full((M, N), -1.5, dtype=torch.float32, device="cuda")
    mx.gemm_mbs(qa, ma, qb, mb, accumulate=True, out=Cacc)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert_within(C.double().cpu().numpy(), want, S, what=f"mbs gemm {shape} {which}")
    assert_within(Cb.double().cpu().numpy(), want, S, bf16=True, what=f"mbs gemm bf16 {shape} {which}")
    assert_within(Cacc.double().cpu().numpy(), want - 1.5, S, what=f"mbs gemm accumulate {shape} {which}")
    if which == "both":  # the correction is not a no-op on this data
        plain, _ = oracle.gemm(ca, sa, cb, sb)
        assert np.abs(plain - want).max() > 1e-3 * np.abs(want).max()


def test_gemm_over_mbs_operands_full_size_sampled(torch):
    """An o-projection-sized Fprop (8192 x 4096 x 4096) over MBS activations and weights:
    every output row and column sampled (first, last and random 64) against the oracle."""
    from mxfp4_precision_gemms_gb300 import binding as mx
    from tests.gpu_util import assert_within

    M, N, K = 8192, 4096, 4096
    X, W, _ = synth.linear_inputs(M, N, K, 2011)
    (qa, ma, ca, sa, oma), (qb, mb, cb, sb, omb) = _mbs_operands(mx, X, W, "both")
    C = mx.gemm_mbs(qa, ma, qb, mb, out_dtype=mx.OUT_BF16)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    g = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(M - 64, M), g.integers(0, M, 64)]))
    cols = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N), g.integers(0, N, 64)]))
    want, S = oracle.gemm_mbs(ca[rows], sa[rows], oma[rows], cb[cols], sb[cols], omb[cols])
    got = C[torch.as_tensor(rows, device="cuda")][:, torch.as_tensor(cols, device="cuda")]
    assert_within(got.double().cpu().numpy(), want, S, bf16=True, what="mbs gemm 8192x4096x4096")


def test_gemm_mbs_rejects_k_beyond_its_macro_blocks(torch):
    from mxfp4_precision_gemms_gb300 import binding as mx

    q = mx.rotate_quantize(mx.bf16_tensor(synth.activations(128, 320, 1)), layouts=mx.LAYOUT_ROW)["row"]
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.gemm_mbs(q, None, q, None)  # K = 320 is not a multiple of 128
    assert e.value.status == 2
