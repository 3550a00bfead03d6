"""The Fprop entry point that allocates nothing (mxfp4_linear_fprop_noalloc).

It serves callers that cannot allocate device memory themselves -- plugins whose
host framework owns all device memory, or loops that must not call cudaMalloc --
by running Fprop on a fixed scratch area inside the library.  Here it is called
through the C ABI twice in a row (different inputs, so stale scratch from the
first call would show) and compared with mxfp4_linear_fprop using a caller
workspace: both run the same kernels, so Y and all four saved arrays (codes and
scales of X^T and W^T) must match byte for byte; Y is also within the 1e-5 *
sum|a||b| tolerance of the oracle, as in the other GPU tests.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import assert_within, gpu_ready

pytestmark = pytest.mark.gpu


def test_noalloc_fprop_matches_workspace_fprop():
    torch = gpu_ready()
    from mxfp4_precision_gemms_gb300 import binding as mx

    L = mx.lib()
    assert L.mxfp4_noalloc_scratch_bytes() == 64 << 20
    M, N, K = 256, 512, 512
    for call, seed in enumerate((0, 7)):
        X, W, _ = synth.linear_inputs(M, N, K, seed)
        x, w = mx.bf16_tensor(X), mx.bf16_tensor(W)
        cfg = mx.Config(had=mx.HAD_16, mode=mx.SCALE_FLOOR, out_dtype=mx.OUT_F32)
        y_ref, xT_ref, wT_ref = mx.linear_fprop(x, w, cfg)

        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        xT = mx.empty_qtensor(K, M, mx.LAYOUT_COLT, mx.SF_MMA)
        wT = mx.empty_qtensor(K, N, mx.LAYOUT_COLT, mx.SF_MMA)
        cx, cw, cc = xT.c(), wT.c(), cfg.c()
        st = L.mxfp4_linear_fprop_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()), M, N, K,
                                          ctypes.byref(cc), ctypes.c_void_p(y.data_ptr()), ctypes.byref(cx),
                                          ctypes.byref(cw), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, L.mxfp4_last_error()
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        want, S = oracle.fprop(X, W, 16, 0)
        assert torch.equal(y, y_ref), f"noalloc call {call}: Y differs from the workspace path"
        assert_within(y.double().cpu().numpy(), want, S, what=f"noalloc call {call}")
        for name, got, ref in (("xT codes", xT.codes, xT_ref.codes), ("xT scales", xT.scales, xT_ref.scales),
                               ("wT codes", wT.codes, wT_ref.codes), ("wT scales", wT.scales, wT_ref.scales)):
            assert np.array_equal(got.cpu().numpy(), ref.cpu().numpy()), f"noalloc call {call}: {name}"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    gpu_ready()
    from mxfp4_precision_gemms_gb300 import binding as mx

    L = mx.lib()
    cc = mx.Config().c()
    P = ctypes.c_void_p
    # down-proj Fprop at T = 8192 needs about 93 MB of scratch: refused before any launch
    st = L.mxfp4_linear_fprop_noalloc(P(0x1000), P(0x2000), 8192, 4096, 14336, ctypes.byref(cc), P(0x3000), None,
                                      None, None)
    assert st == 4
    assert b"scratch" in L.mxfp4_last_error()
