"""GPU block-scaled MXFP4 GEMM vs the CPU oracle.

Operands are quantised by the oracle on the CPU and uploaded, so these tests check
the GEMM alone: |C_gpu - C_oracle| <= 1e-5 * sum_k |dq a_k| |dq b_k| per element
(plus 2^-8 |C| for bf16 output, the rounding of the output itself)."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import ORACLE_HAD, assert_within, gpu_ready

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return gpu_ready()


def oracle_operands(M, N, K, seed, had=16, mode=0):
    X, W, _ = synth.linear_inputs(M, N, K, seed)
    return oracle.quantize(X, had, mode, "row"), oracle.quantize(W, had, mode, "row")


def run(torch, qa, qb, out_dtype=0, accumulate=False, init=None):
    from mxfp4_precision_gemms_gb300 import binding as mx

    A = mx.qtensor_from_host(*qa)
    B = mx.qtensor_from_host(*qb)
    out = None
    if init is not None:
        out = torch.from_numpy(init).cuda()
    C = mx.gemm(A, B, out_dtype=out_dtype, accumulate=accumulate, out=out)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return C.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("N", [128, 256])
def test_single_block_scales(torch, N):
    """K = 32: every output is 2^(ea+eb) * sum qa*qb; rows use distinct scales, so a
    wrong scale-factor placement shows up as an exact power-of-two error (N = 256 covers
    the second 128-row group of B's scales in a 256-wide tile)."""
    M, K = 128, 32
    g = np.random.default_rng(0)
    ca = g.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = (120 + (np.arange(M) % 13)).astype(np.uint8)[:, None]
    sb = (112 + (np.arange(N) % 29)).astype(np.uint8)[:, None]
    want, S = oracle.gemm(ca, sa, cb, sb)
    got = run(torch, (ca, sa), (cb, sb))
    assert_within(got, want, S, what="single block")


def test_single_block_scales_pair(torch):
    """CTA-pair tiles (M, N > 128): every row of A and of B has its own scale in each of
    the two K blocks, so a scale read from the wrong CTA, row group or block gives an
    exact power-of-two error in that quadrant of the 256 x 256 tile."""
    M, N, K = 512, 512, 64
    g = np.random.default_rng(1)
    ca = g.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = (110 + (np.arange(M)[:, None] * 7 + np.arange(K // 32)[None, :] * 3) % 23).astype(np.uint8)
    sb = (105 + (np.arange(N)[:, None] * 5 + np.arange(K // 32)[None, :] * 11) % 31).astype(np.uint8)
    want, S = oracle.gemm(ca, sa, cb, sb)
    got = run(torch, (ca, sa), (cb, sb))
    assert_within(got, want, S, what="pair single block")


@pytest.mark.parametrize("shape", [(128, 128, 256), (256, 512, 512), (128, 128, 2048), (384, 256, 1024),
                                   (300, 520, 768)])
def test_aligned_shapes(torch, shape):
    M, N, K = shape
    qa, qb = oracle_operands(M, N, K, 10)
    want, S = oracle.gemm(*qa, *qb)
    assert_within(run(torch, qa, qb), want, S, what=f"{shape}")


@pytest.mark.parametrize("shape", [(200, 136, 96), (1, 8, 32), (130, 264, 1056), (77, 1000, 288), (256, 40, 4128)])
def test_ragged_shapes(torch, shape):
    M, N, K = shape
    qa, qb = oracle_operands(M, N, K, 11, had=32, mode=1)
    want, S = oracle.gemm(*qa, *qb)
    assert_within(run(torch, qa, qb), want, S, what=f"{shape}")


def test_bf16_output(torch):
    qa, qb = oracle_operands(256, 384, 768, 12)
    want, S = oracle.gemm(*qa, *qb)
    assert_within(run(torch, qa, qb, out_dtype=1), want, S, bf16=True, what="bf16 out")


def test_accumulate(torch):
    qa, qb = oracle_operands(256, 256, 512, 13)
    want, S = oracle.gemm(*qa, *qb)
    init = np.random.default_rng(1).standard_normal((256, 256)).astype(np.float32)
    got = run(torch, qa, qb, accumulate=True, init=init)
    # the fp32 add of the old value rounds once more: allow 2^-23 (|init| + |C|)
    assert_within(got - init.astype(np.float64), want, S + 0.02 * (np.abs(init) + np.abs(want)), what="accumulate")


def test_extreme_scales(torch):
    """Scale bytes near both ends of the E8M0 range used by the quantiser."""
    M, N, K = 128, 128, 256
    g = np.random.default_rng(3)
    ca = g.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = g.integers(100, 154, size=(M, K // 32), dtype=np.uint8)
    sb = g.integers(100, 154, size=(N, K // 32), dtype=np.uint8)
    want, S = oracle.gemm(ca, sa, cb, sb)
    assert_within(run(torch, (ca, sa), (cb, sb)), want, S, what="wide scales")


def test_many_tiles_narrow_n(torch):
    """N <= 128 selects the 128-wide tiles with two TMEM accumulators; ~300 tiles make
    every persistent CTA alternate between them (and the M tail is ragged)."""
    M, N, K = 37984 + 40, 96, 512
    qa, qb = oracle_operands(M, N, K, 14)
    want, S = oracle.gemm(*qa, *qb)
    assert_within(run(torch, qa, qb), want, S, what="many tiles, N=96")
    assert_within(run(torch, qa, qb, out_dtype=1), want, S, bf16=True, what="many tiles, N=96, bf16")


def test_back_to_back_accumulate_chain(torch):
    """GEMMs overlap the previous kernel's drain (programmatic dependent launch) and wait
    for it before touching memory: C = A1 B1^T, then C += A2 B2^T launched right after
    on the same stream (CTA-pair tiles), must equal the sum of the two products."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    M, N, K = 1024, 768, 512
    qa1, qb1 = oracle_operands(M, N, K, 15)
    qa2, qb2 = oracle_operands(M, N, K, 16)
    w1, S1 = oracle.gemm(*qa1, *qb1)
    w2, S2 = oracle.gemm(*qa2, *qb2)
    A1, B1, A2, B2 = (mx.qtensor_from_host(*q) for q in (qa1, qb1, qa2, qb2))
    C = mx.gemm(A1, B1, out_dtype=mx.OUT_F32)
    for _ in range(3):  # the accumulating launches follow one another with no sync between
        C = mx.gemm(A2, B2, out_dtype=mx.OUT_F32, accumulate=True, out=C)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    got = C.double().cpu().numpy()
    # each fp32 add of the running value rounds once more: allow 2^-22 of the magnitudes
    assert_within(got, w1 + 3 * w2, S1 + 3 * S2 + 2.4e-7 * (np.abs(w1) + 3 * np.abs(w2)) / 1e-5,
                  what="accumulate chain")


@pytest.mark.parametrize("shape", [(544, 20000, 256), (20000, 544, 256)])
def test_many_waves_both_tile_orders(torch, shape):
    """More column tiles than row tiles (3 x 79: tiles walk M fastest) and the transpose
    (79 x 3: N fastest), both with ragged edges and about three tiles per CTA pair, so
    every pair wraps around the walked dimension several times."""
    M, N, K = shape
    qa, qb = oracle_operands(M, N, K, 15)
    want, S = oracle.gemm(*qa, *qb)
    assert_within(run(torch, qa, qb), want, S, what=f"{shape}")
    assert_within(run(torch, qa, qb, out_dtype=1), want, S, bf16=True, what=f"{shape} bf16")


def _random_shapes(count, seed):
    g = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        M = int(g.integers(1, 1400))
        N = int(g.integers(1, 180)) * 8      # the output's row pitch is a multiple of 8
        K = int(g.integers(1, 80)) * 32      # contraction in whole 32-element blocks
        out.append((M, N, K, int(g.choice([0, 16, 32])), int(g.integers(0, 2)), int(g.integers(0, 2))))
    return out


@pytest.mark.parametrize("M,N,K,had,mode,out_dtype", _random_shapes(24, 2026))
def test_random_shapes(torch, M, N, K, had, mode, out_dtype):
    """Seeded random shapes (ragged M, N and K in 32-element blocks; both kernels; every
    rotation and scale rule; fp32 and bf16 out) against the oracle."""
    qa, qb = oracle_operands(M, N, K, M + N + K, had=ORACLE_HAD[had], mode=mode)
    want, S = oracle.gemm(*qa, *qb)
    assert_within(run(torch, qa, qb, out_dtype=out_dtype), want, S, bf16=out_dtype == 1,
                  what=f"{M}x{N}x{K} had={had} mode={mode} out={out_dtype}")
