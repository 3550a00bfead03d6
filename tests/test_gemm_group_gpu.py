"""Grouped GEMM (mxfp4_gemm_group): several problems in one persistent launch.  Every
output must equal the same problem launched on its own (bit for bit where the single
launch also takes the CTA-pair kernel, M and N > 128) and lie within the 1e-5 *
sum|a||b| tolerance of the oracle, including narrow and ragged problems."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import assert_within, gpu_ready, sample_pairs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return gpu_ready()


def _q(mx, bits, layout=1):
    return mx.rotate_quantize(mx.bf16_tensor(bits), had=16, mode=0, layouts=layout)


def test_backward_pair_matches_separate_launches(torch):
    """Dgrad and Wgrad of one linear layer (the backward pair) in one launch."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    M, N, K = 1024, 768, 512
    X, W, dY = synth.linear_inputs(M, N, K, 40)
    dq = _q(mx, dY, 3)
    wT = _q(mx, W, 2)["colT"]
    xT = _q(mx, X, 2)["colT"]
    dx, dw = mx.gemm_group([(dq["row"], wT, mx.OUT_BF16, False, None), (dq["colT"], xT, mx.OUT_F32, False, None)])
    dx1 = mx.gemm(dq["row"], wT, mx.OUT_BF16)
    dw1 = mx.gemm(dq["colT"], xT, mx.OUT_F32)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(dx, dx1) and torch.equal(dw, dw1)
    want, S = oracle.dgrad(dY, W, 16, 0)
    assert_within(dx.double().cpu().numpy(), want, S, bf16=True, what="grouped dgrad")
    want, S = oracle.wgrad(dY, X, 16, 0)
    assert_within(dw.double().cpu().numpy(), want, S, what="grouped wgrad")


def test_qkv_projections_share_one_launch(torch):
    """q, k, v Fprop (N = 1024 for k and v: narrower than one tile pair row on its own
    in the single-CTA kernel) in one launch, against separate launches and the oracle."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    M, K = 512, 1024
    X = synth.activations(M, K, 41)
    xq = _q(mx, X)["row"]
    Ws = [synth.weights(N, K, 42 + i) for i, N in enumerate((512, 256, 256))]
    wqs = [_q(mx, w)["row"] for w in Ws]
    ys = mx.gemm_group([(xq, wq, mx.OUT_F32, False, None) for wq in wqs])
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for y, w in zip(ys, Ws):
        want, S = oracle.fprop(X, w, 16, 0)
        assert_within(y.double().cpu().numpy(), want, S, what=f"grouped q/k/v N={w.shape[0]}")
        assert torch.equal(y, mx.gemm(xq, _q(mx, w)["row"], mx.OUT_F32))


def test_mixed_group_with_ragged_and_accumulating_problems(torch):
    """Four problems of different K, ragged M and N and an accumulating one (ordered by
    the library longest-contraction first; outputs come back in the caller's order)."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    shapes = [(300, 200, 256), (640, 512, 2048), (136, 520, 512), (256, 384, 1024)]
    ops, wants = [], []
    for i, (M, N, K) in enumerate(shapes):
        qa = oracle.quantize(synth.activations(M, K, 50 + i), 16, 0, "row")
        qb = oracle.quantize(synth.weights(N, K, 60 + i), 16, 0, "row")
        A, B = mx.qtensor_from_host(*qa, had=16), mx.qtensor_from_host(*qb, had=16)
        acc = i == 3
        out = torch.full((M, N), 0.5, dtype=torch.float32, device="cuda") if acc else None
        ops.append((A, B, mx.OUT_F32, acc, out))
        want, S = oracle.gemm(*qa, *qb)
        wants.append((want + (0.5 if acc else 0.0), S))
    outs = mx.gemm_group(ops)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for (M, N, K), out, (want, S) in zip(shapes, outs, wants):
        assert out.shape == (M, N)
        assert_within(out.double().cpu().numpy(), want, S, what=f"group {M}x{N}x{K}")


def test_full_size_backward_pair_sampled(torch):
    """The o-projection's backward pair at T = 8192 (dX 8192 x 4096 x 4096 bf16, dW 4096 x
    4096 x 8192 fp32) in one launch: sampled outputs against the oracle and equal to
    separate launches."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    T, N, K = 8192, 4096, 4096
    X, W, dY = synth.linear_inputs(T, N, K, 2010)
    dq = _q(mx, dY, 3)
    wT = _q(mx, W, 2)["colT"]
    xT = _q(mx, X, 2)["colT"]
    dx, dw = mx.gemm_group([(dq["row"], wT, mx.OUT_BF16, False, None), (dq["colT"], xT, mx.OUT_F32, False, None)])
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(dx, mx.gemm(dq["row"], wT, mx.OUT_BF16))
    assert torch.equal(dw, mx.gemm(dq["colT"], xT, mx.OUT_F32))
    r, c = sample_pairs(T, K, 48, 3)
    want, S = oracle.dgrad_sample(dY, W, 16, 0, r, c)
    assert_within(dx[r, c].double().cpu().numpy(), want, S, bf16=True, what="grouped dgrad T=8192")
    r, c = sample_pairs(N, K, 48, 4)
    want, S = oracle.wgrad_sample(dY, X, 16, 0, r, c)
    assert_within(dw[r, c].double().cpu().numpy(), want, S, what="grouped wgrad T=8192")


@pytest.mark.parametrize("had,mode", [(16, 0), (32, 1)])
def test_linear_backward_equals_dgrad_plus_wgrad(torch, had, mode):
    """mxfp4_linear_backward (one dY quantisation, one grouped launch) gives the same dX
    and dW bytes as mxfp4_linear_dgrad + mxfp4_linear_wgrad, and adds to dW under
    accumulate."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    M, N, K = 512, 384, 640
    X, W, dY = synth.linear_inputs(M, N, K, 70)
    x, w, dy = (mx.bf16_tensor(a) for a in (X, W, dY))
    cfg = mx.Config(had=had, mode=mode, out_dtype=mx.OUT_BF16)
    _, xT, wT = mx.linear_fprop(x, w, cfg)
    dx_ref, dyT = mx.linear_dgrad(dy, wT, cfg)
    dw_ref = mx.linear_wgrad(dyT, xT, mx.Config(had=had, mode=mode, out_dtype=mx.OUT_F32))
    dx, dw = mx.linear_backward(dy, wT, xT, cfg)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    assert torch.equal(dx, dx_ref) and torch.equal(dw, dw_ref)
    acc = mx.Config(had=had, mode=mode, out_dtype=mx.OUT_BF16, accumulate=1)
    dw2 = torch.full_like(dw_ref, 0.25)
    mx.linear_backward(dy, wT, xT, acc, dw=dw2)
    torch.cuda.synchronize()
    want, S = oracle.wgrad(dY, X, {0: 1, 16: 16, 32: 32}[had], mode)
    assert_within(dw2.double().cpu().numpy(), want + 0.25, S, what="backward dW accumulate")


def test_group_with_narrow_problems(torch):
    """Problems with M <= 128 or N <= 128 (which a single launch would give the single-CTA
    kernel) run on the pair kernel inside a group: half-empty tiles are zero-filled on load
    and clipped on store.  Outputs within tolerance, and no byte outside them is written."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    shapes = [(64, 512, 512), (1024, 96, 256), (96, 64, 1024), (512, 384, 768)]
    ops, wants, guards = [], [], []
    for i, (M, N, K) in enumerate(shapes):
        qa = oracle.quantize(synth.activations(M, K, 80 + i), 16, 0, "row")
        qb = oracle.quantize(synth.weights(N, K, 90 + i), 16, 0, "row")
        A, B = mx.qtensor_from_host(*qa, had=16), mx.qtensor_from_host(*qb, had=16)
        # C inside a larger buffer with ldc = N + 8: the padding columns must stay untouched
        buf = torch.full((M, N + 8), 3.25, dtype=torch.float32, device="cuda")
        ops.append((A, B, mx.OUT_F32, False, buf[:, :N]))
        wants.append(oracle.gemm(*qa, *qb))
        guards.append(buf)
    mx.gemm_group(ops)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for (M, N, K), buf, (want, S) in zip(shapes, guards, wants):
        assert_within(buf[:, :N].double().cpu().numpy(), want, S, what=f"narrow group {M}x{N}x{K}")
        assert torch.all(buf[:, N:] == 3.25), f"{M}x{N}x{K}: padding written"


def test_eight_problem_group(torch):
    """The largest group (8 problems): contractions from 256 to 2048, ragged shapes,
    problems whose tiles walk M fastest (more column than row tiles) and N fastest, bf16
    and fp32 outputs.  Each output equals its own launch bit for bit and the oracle
    within tolerance."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    shapes = [(256, 1024, 512), (1024, 256, 512), (384, 384, 1024), (512, 768, 256), (300, 648, 768),
              (640, 296, 256), (256, 256, 2048), (768, 1280, 512)]
    ops, refs = [], []
    for i, (M, N, K) in enumerate(shapes):
        qa = oracle.quantize(synth.activations(M, K, 70 + i), 16, 0, "row")
        qb = oracle.quantize(synth.weights(N, K, 80 + i), 16, 0, "row")
        A, B = mx.qtensor_from_host(*qa, had=16), mx.qtensor_from_host(*qb, had=16)
        od = mx.OUT_BF16 if i % 2 else mx.OUT_F32
        ops.append((A, B, od, False, None))
        refs.append((qa, qb, od))
    outs = mx.gemm_group(ops)
    singles = [mx.gemm(A, B, od) for A, B, od, _, _ in ops]
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for (M, N, K), out, one, (qa, qb, od) in zip(shapes, outs, singles, refs):
        assert torch.equal(out, one), f"group vs single launch {M}x{N}x{K}"
        want, S = oracle.gemm(*qa, *qb)
        assert_within(out.double().cpu().numpy(), want, S, bf16=od == mx.OUT_BF16, what=f"group of 8 {M}x{N}x{K}")
