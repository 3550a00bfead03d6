"""The benchmark's timed steps as CUDA graphs must give byte-identical outputs to the
same work issued launch by launch on one stream, with every quantised operand and every
output cleared in between (so a launch that ran before its producer would read zeros):
the headline step (per linear: X and W quantised in one launch, Fprop, the dY
quantisation, Dgrad and Wgrad in one grouped launch), its two-branch form with separate
launches, and the decoder block."""
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
