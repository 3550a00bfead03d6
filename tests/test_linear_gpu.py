"""End-to-end H16/H32 + MXFP4 linear layer through the C ABI vs the CPU oracle:
Fprop Y = X W^T, Dgrad dX = dY W, Wgrad dW = dY^T X, each operand rotated along the
GEMM's contraction and quantised ("Pretraining ... Native FP4 Hardware", C.1-C.3).

Small configs are compared element by element; the Llama-3.1-8B-shaped configs
(T = 8192, and the T = 32768 Wgrad stress case) on sampled outputs, which the
oracle computes one by one from the rows/columns involved, plus tile edges."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import ORACLE_HAD, assert_within, gpu_ready, sample_pairs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return gpu_ready()


def run_linear(torch, X, W, dY, had, mode, out_dtype=0):
    from mxfp4_precision_gemms_gb300 import binding as mx

    x, w, dy = (mx.bf16_tensor(a) for a in (X, W, dY))
    cfg = mx.Config(had=had, mode=mode, out_dtype=out_dtype)
    y, xT, wT = mx.linear_fprop(x, w, cfg)
    dx, dyT = mx.linear_dgrad(dy, wT, cfg)
    wcfg = mx.Config(had=had, mode=mode, out_dtype=mx.OUT_F32)
    dw = mx.linear_wgrad(dyT, xT, wcfg)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    return y, dx, dw, xT, wT, dyT


@pytest.mark.parametrize("had", [16, 32, 0])
@pytest.mark.parametrize("mode", [0, 1])
def test_config0_full(torch, had, mode):
    X, W, dY = synth.linear_inputs(256, 512, 512, 0)
    y, dx, dw, xT, wT, dyT = run_linear(torch, X, W, dY, had, mode)
    h = ORACLE_HAD[had]
    for name, got, (want, S) in (("fprop", y, oracle.fprop(X, W, h, mode)), ("dgrad", dx, oracle.dgrad(dY, W, h, mode)),
                                 ("wgrad", dw, oracle.wgrad(dY, X, h, mode))):
        assert_within(got.double().cpu().numpy(), want, S, what=f"{name} had={had} mode={mode}")
    # the saved transposed operands are bit-exact with the oracle's column layout
    for q, src in ((xT, X), (wT, W), (dyT, dY)):
        c, s = oracle.quantize(src, h, mode, "colT")
        assert np.array_equal(q.codes.cpu().numpy(), c)
        assert np.array_equal(q.plain_scales(), s)


def test_config0_bf16_out(torch):
    X, W, dY = synth.linear_inputs(256, 512, 512, 0)
    y, dx, dw, *_ = run_linear(torch, X, W, dY, 16, 0, out_dtype=1)
    want, S = oracle.fprop(X, W, 16, 0)
    assert_within(y.double().cpu().numpy(), want, S, bf16=True, what="fprop bf16")
    want, S = oracle.dgrad(dY, W, 16, 0)
    assert_within(dx.double().cpu().numpy(), want, S, bf16=True, what="dgrad bf16")


@pytest.mark.parametrize("MNK", [(160, 96, 224), (32, 32, 32), (96, 1056, 64)])
def test_ragged_full(torch, MNK):
    M, N, K = MNK
    X, W, dY = synth.linear_inputs(M, N, K, 5)
    y, dx, dw, *_ = run_linear(torch, X, W, dY, 16, 0)
    for name, got, (want, S) in (("fprop", y, oracle.fprop(X, W, 16, 0)), ("dgrad", dx, oracle.dgrad(dY, W, 16, 0)),
                                 ("wgrad", dw, oracle.wgrad(dY, X, 16, 0))):
        assert_within(got.double().cpu().numpy(), want, S, what=f"{name} {MNK}")


def _sampled_checks(torch, X, W, dY, had, mode, y, dx, dw, n=256, seed=0):
    M, K = X.shape
    N = W.shape[0]
    h = ORACLE_HAD[had]
    r, c = sample_pairs(M, N, n, seed)
    want, S = oracle.fprop_sample(X, W, h, mode, r, c)
    assert_within(y[r, c].double().cpu().numpy(), want, S, bf16=y.dtype != torch.float32, what="fprop sampled")
    r, c = sample_pairs(M, K, n, seed + 1)
    want, S = oracle.dgrad_sample(dY, W, h, mode, r, c)
    assert_within(dx[r, c].double().cpu().numpy(), want, S, bf16=dx.dtype != torch.float32, what="dgrad sampled")
    r, c = sample_pairs(N, K, n // 4, seed + 2)
    want, S = oracle.wgrad_sample(dY, X, h, mode, r, c)
    assert_within(dw[r, c].double().cpu().numpy(), want, S, what="wgrad sampled")


@pytest.mark.parametrize("name,N,K", [("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 14336, 4096),
                                    ("down", 4096, 14336), ("k", 1024, 4096)])
def test_llama8b_linears_sampled(torch, name, N, K):
    """Config 2 shapes at T = 8192 in the launch configuration the benchmark times
    (bf16 Fprop/Dgrad outputs, fp32 Wgrad)."""
    T = 8192
    X, W, dY = synth.linear_inputs(T, N, K, 2000)
    y, dx, dw, *_ = run_linear(torch, X, W, dY, 16, 0, out_dtype=1)
    _sampled_checks(torch, X, W, dY, 16, 0, y, dx, dw)


@pytest.mark.parametrize("had,mode", [(32, 0), (0, 0), (16, 1)])
def test_llama8b_qkv_other_rotations_sampled(torch, had, mode):
    """The QKV linear at T = 8192 under H32 and without rotation (the H32 leg of the
    benchmark), and under H16 with the ceiling scale."""
    T, N, K = 8192, 6144, 4096
    X, W, dY = synth.linear_inputs(T, N, K, 2000)
    y, dx, dw, *_ = run_linear(torch, X, W, dY, had, mode, out_dtype=1)
    _sampled_checks(torch, X, W, dY, had, mode, y, dx, dw, n=128, seed=had + mode)


@pytest.mark.parametrize("had", [16, 32, 0])
def test_wgrad_stress_sampled(torch, had):
    """Config 3: dW = dY^T X over T = 32768 tokens, dY [32768, 4096], X [32768, 14336]."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    T, N, K = 32768, 4096, 14336
    X = synth.activations(T, K, 3000)
    dY = synth.output_grads(T, N, 3002)
    x, dy = mx.bf16_tensor(X), mx.bf16_tensor(dY)
    xT = mx.rotate_quantize(x, had=had, mode=0, layouts=mx.LAYOUT_COLT)["colT"]
    dyT = mx.rotate_quantize(dy, had=had, mode=0, layouts=mx.LAYOUT_COLT)["colT"]
    dw = mx.linear_wgrad(dyT, xT, mx.Config(had=had))
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    r, c = sample_pairs(N, K, 48, 7, edge=2)
    want, S = oracle.wgrad_sample(dY, X, ORACLE_HAD[had], 0, r, c)
    assert_within(dw[r, c].double().cpu().numpy(), want, S, what=f"wgrad T=32768 had={had}")


def test_cuda_graph_replay_matches_eager(torch):
    """Every launch of the linear-layer API can be held in a CUDA graph: no host syncs,
    no allocations once buffers exist, per-device launch settings cached on first use.
    Fprop, Dgrad and Wgrad captured once and replayed twice (ragged M, the CTA-pair GEMM
    and the single-CTA one) give the same bytes as eager calls."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    M, N, K = 640, 384, 128  # Dgrad and Wgrad outputs 128 wide: the single-CTA GEMM
    X, W, dY = synth.linear_inputs(M, N, K, 21)
    x, w, dy = (mx.bf16_tensor(a) for a in (X, W, dY))
    cfg = mx.Config(had=16, mode=0, out_dtype=mx.OUT_BF16)
    wcfg = mx.Config(had=16, mode=0, out_dtype=mx.OUT_F32)
    ws = mx.Workspace()

    def buffers():
        return {"y": torch.empty((M, N), dtype=torch.bfloat16, device="cuda"),
                "dx": torch.empty((M, K), dtype=torch.bfloat16, device="cuda"),
                "dw": torch.empty((N, K), dtype=torch.float32, device="cuda"),
                "xT": mx.empty_qtensor(K, M, mx.LAYOUT_COLT, mx.SF_MMA),
                "wT": mx.empty_qtensor(K, N, mx.LAYOUT_COLT, mx.SF_MMA),
                "dyT": mx.empty_qtensor(N, M, mx.LAYOUT_COLT, mx.SF_MMA)}

    def step(b):
        mx.linear_fprop(x, w, cfg, y=b["y"], xT=b["xT"], wT=b["wT"], ws=ws)
        mx.linear_dgrad(dy, b["wT"], cfg, dx=b["dx"], dyT=b["dyT"], ws=ws)
        mx.linear_wgrad(b["dyT"], b["xT"], wcfg, dw=b["dw"])

    eager, cap = buffers(), buffers()
    step(eager)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(cap)
    torch.cuda.synchronize()
    for _ in range(2):
        for k in ("y", "dx", "dw"):
            cap[k].zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for k in ("y", "dx", "dw"):
        assert torch.equal(eager[k], cap[k]), k
    for k in ("xT", "wT", "dyT"):
        assert torch.equal(eager[k].codes, cap[k].codes) and torch.equal(eager[k].scales, cap[k].scales), k


def test_decoder_block_sampled(torch):
    """The Llama-3.1-8B-shaped decoder block (q, k, v, o, gate, up, down at T = 8192,
    H16, OCP floor) exactly as the benchmark times it -- the 20-launch grouped graph,
    activations quantised once and shared by the linears that read them -- against the
    oracle on sampled Y, dX and dW of every linear, from the same seeded inputs."""
    import importlib.util
    import os

    from mxfp4_precision_gemms_gb300 import binding as mx

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_block_mod", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dev = torch.device("cuda", 0)
    groups = bench.make_block_groups(dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        bench.run_block_grouped(groups)
    graph.replay()
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    T = bench.T_TOKENS
    for gi, (inp, lins) in enumerate(groups):
        X = synth.activations(T, inp.K, bench.BLOCK_SEED + 100 * gi)
        for j, L in enumerate(lins):
            s = bench.BLOCK_SEED + 100 * gi + 10 * (j + 1)
            W, dY = synth.weights(L.N, L.K, s + 1), synth.output_grads(T, L.N, s + 2)
            _sampled_checks(torch, X, W, dY, 16, 0, L.y, L.dx, L.dw, n=96, seed=gi * 10 + j)
