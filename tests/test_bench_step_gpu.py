"""The benchmark's timed step as a two-branch CUDA graph: each linear layer's X and W
quantisations run on two streams before Fprop, and its Dgrad and Wgrad GEMMs on two
streams after the dY quantisation.  Replaying that graph must give byte-identical outputs
to the same 24 launches issued one after another on a single stream, with every
quantised operand and every output cleared in between (so a launch that ran before its
producer would read zeros)."""
import importlib.util
import os

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

    bench.run_step(layers)
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

    side, aux = torch.cuda.Stream(), torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        bench.run_step(layers, aux=aux)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert mx.device_status() == 0

    for L, w in zip(layers, want):
        got = [L.y, L.dx, L.dw] + [b for q in quantised(L) for b in (q.codes, q.scales)]
        for i, (a, b) in enumerate(zip(got, w)):
            assert torch.equal(a, b), f"{L.name}: tensor {i} differs between the two-branch graph and serial launches"
