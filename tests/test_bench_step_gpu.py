"""The benchmark's timed steps as CUDA graphs must give byte-identical outputs to the
same work issued launch by launch on one stream, with every quantised operand and every
output cleared in between (so a launch that ran before its producer would read zeros):
the headline step (per linear: X and W quantised in one launch, Fprop, the dY
quantisation, Dgrad and Wgrad in one grouped launch), its two-branch form with separate
launches, and the decoder block.  The headline step's graph is also checked against the
oracle on sampled outputs and on every output of the tile-edge rows and columns."""
import importlib.util
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_step_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.gpu
def test_two_branch_graph_step_matches_serial_launches():
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300 import synth

    bench = _bench()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    layers = [bench.Layer(n, N, K, 2000 + 10 * i, dev) for i, (n, N, K) in enumerate(synth.LLAMA8B_LINEARS)]

    def quantised(L):
        return [L.xq, L.wq, L.dyq, L.xT, L.wT, L.dyT]

    bench.run_step(layers, pair=False, group=False)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    want = [[t.clone() for t in (L.y, L.dx, L.dw)] + [b.clone() for q in quantised(L) for b in (q.codes, q.scales)]
            for L in layers]

    for L in layers:
        for t in (L.y, L.dx, L.dw):
            t.zero_()
        for q in quantised(L):
            q.codes.zero_()
            q.scales.zero_()
    torch.cuda.synchronize()

    for pair, group in ((True, True), (False, False)):
        for L in layers:
            for t in (L.y, L.dx, L.dw):
                t.zero_()
            for q in quantised(L):
                q.codes.zero_()
                q.scales.zero_()
        torch.cuda.synchronize()
        side, aux = torch.cuda.Stream(), torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            bench.run_step(layers, aux=aux, pair=pair, group=group)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        for L, w in zip(layers, want):
            got = [L.y, L.dx, L.dw] + [b for q in quantised(L) for b in (q.codes, q.scales)]
            for i, (a, b) in enumerate(zip(got, w)):
                assert torch.equal(a, b), f"{L.name}: tensor {i} differs (graph pair={pair} group={group})"


@pytest.mark.gpu
def test_decoder_block_graph_matches_serial_launches():
    """The decoder block's graph (activations quantised once and shared by the linears
    that read them; quantisations two matrices per launch; each activation's Fprops in
    one grouped GEMM launch and its Dgrads and Wgrads in another) gives the same bytes as
    every launch issued separately, one after another on one stream, outputs and
    quantised copies cleared in between."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx

    bench = _bench()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    groups = bench.make_block_groups(dev)
    outs = lambda: [t for _, lins in groups for L in lins for t in (L.y, L.dx, L.dw)]
    bench.run_block(groups)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    want = [t.clone() for t in outs()]
    for t in outs():
        t.zero_()
    for inp, lins in groups:
        for q in [inp.xq, inp.xT] + [q for L in lins for q in (L.wq, L.wT, L.dyq, L.dyT)]:
            q.codes.zero_()
            q.scales.zero_()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        bench.run_block_grouped(groups)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    for i, (a, b) in enumerate(zip(outs(), want)):
        assert torch.equal(a, b), f"output {i} differs between the grouped block graph and separate launches"


def _edges(n, w=128):
    return np.unique(np.r_[np.arange(min(w, n)), np.arange(max(0, n - w), n)])


@pytest.mark.gpu
def test_headline_step_vs_oracle():
    """The benchmark's timed step exactly as timed (the CUDA graph of 16 launches: per
    linear the X+W pair quantisation, Fprop, the dY quantisation, Dgrad and Wgrad in one
    grouped launch) at T = 8192 on the four Llama-3.1-8B linears, against the oracle:
    1024 random outputs of each of the 12 GEMMs, plus every output in the first and last
    128 rows and columns (the tile edges), within 1e-5 * sum|a||b| (+ the bf16 rounding
    of Y and dX)."""
    import torch

    import oracle
    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300 import synth
    from tests.gpu_util import assert_within, sample_pairs

    bench = _bench()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    layers = [bench.Layer(n, N, K, 2000 + 10 * i, dev) for i, (n, N, K) in enumerate(synth.LLAMA8B_LINEARS)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        bench.run_step(layers)
    graph.replay()
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    h, mode, M = 16, 0, bench.T_TOKENS
    for i, L in enumerate(layers):
        X, W, dY = synth.linear_inputs(M, L.N, L.K, 2000 + 10 * i)
        y, dx, dw = (t.double().cpu().numpy() for t in (L.y, L.dx, L.dw))
        rm, rn, rk = _edges(M), _edges(L.N), _edges(L.K)
        q = lambda a, lay: oracle.quantize(np.ascontiguousarray(a), h, mode, lay)
        # Fprop Y [M, N]: X row copy x W row copy
        xr, wr = q(X, "row"), q(W, "row")
        want, S = oracle.gemm(*q(X[rm], "row"), *wr)
        assert_within(y[rm], want, S, bf16=True, what=f"{L.name} fprop edge rows")
        want, S = oracle.gemm(*xr, *q(W[rn], "row"))
        assert_within(y[:, rn], want, S, bf16=True, what=f"{L.name} fprop edge cols")
        r, c = sample_pairs(M, L.N, 1024, 10 * i, edge=0)
        want, S = oracle.fprop_sample(X, W, h, mode, r, c)
        assert_within(y[r, c], want, S, bf16=True, what=f"{L.name} fprop sampled")
        del xr, wr
        # Dgrad dX [M, K]: dY row copy x W column copy
        dyr, wT = q(dY, "row"), q(W, "colT")
        want, S = oracle.gemm(*q(dY[rm], "row"), *wT)
        assert_within(dx[rm], want, S, bf16=True, what=f"{L.name} dgrad edge rows")
        want, S = oracle.gemm(*dyr, *q(W[:, rk], "colT"))
        assert_within(dx[:, rk], want, S, bf16=True, what=f"{L.name} dgrad edge cols")
        r, c = sample_pairs(M, L.K, 1024, 10 * i + 1, edge=0)
        want, S = oracle.dgrad_sample(dY, W, h, mode, r, c)
        assert_within(dx[r, c], want, S, bf16=True, what=f"{L.name} dgrad sampled")
        del dyr, wT
        # Wgrad dW [N, K]: dY column copy x X column copy (contraction over tokens)
        dyT, xT = q(dY, "colT"), q(X, "colT")
        want, S = oracle.gemm(*q(dY[:, rn], "colT"), *xT)
        assert_within(dw[rn], want, S, what=f"{L.name} wgrad edge rows")
        want, S = oracle.gemm(*dyT, *q(X[:, rk], "colT"))
        assert_within(dw[:, rk], want, S, what=f"{L.name} wgrad edge cols")
        r, c = sample_pairs(L.N, L.K, 1024, 10 * i + 2, edge=0)
        want, S = oracle.wgrad_sample(dY, X, h, mode, r, c)
        assert_within(dw[r, c], want, S, what=f"{L.name} wgrad sampled")
