"""A rejected linear-layer call launches nothing: the workspace, the saved transposed
copies and the output keep every byte they held before the call.  (The CPU tests show
that the checks come before the first CUDA call; this shows it on the device.)"""
import ctypes

import pytest

from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import gpu_ready

pytestmark = pytest.mark.gpu


def _sentinels(torch, *tensors):
    for t in tensors:
        t.fill_(0xA5 if t.dtype == torch.uint8 else 7.0)
    return [t.clone() for t in tensors]


def _unchanged(torch, tensors, before):
    torch.cuda.synchronize()
    for t, b in zip(tensors, before):
        assert torch.equal(t, b)


def test_rejected_fprop_leaves_every_buffer_untouched():
    torch = gpu_ready()
    from mxfp4_precision_gemms_gb300 import binding as mx

    L = mx.lib()
    M, N, K = 256, 256, 512
    X, W, _ = synth.linear_inputs(M, N, K, 0)
    x = mx.bf16_tensor(X)
    wbuf = torch.empty(N * K + 4, dtype=torch.bfloat16, device="cuda")
    wbuf[4:].copy_(mx.bf16_tensor(W).reshape(-1))
    cfg = mx.Config(had=mx.HAD_16, mode=mx.SCALE_FLOOR, out_dtype=mx.OUT_F32)
    nb = mx.workspace_bytes(mx.OP_FPROP, M, N, K, cfg)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    xT = mx.empty_qtensor(K, M, mx.LAYOUT_COLT, mx.SF_MMA)
    wT = mx.empty_qtensor(K, N, mx.LAYOUT_COLT, mx.SF_MMA)
    bufs = [ws, y, xT.codes, xT.scales, wT.codes, wT.scales]
    before = _sentinels(torch, *bufs)
    cc, cx, cw = cfg.c(), xT.c(), wT.c()
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    # W 8 bytes past a 16-byte boundary: X is valid and would have been quantised first
    st = L.mxfp4_linear_fprop(P(x.data_ptr()), P(wbuf[4:].data_ptr()), M, N, K, ctypes.byref(cc), P(y.data_ptr()),
                              ctypes.byref(cx), ctypes.byref(cw), P(ws.data_ptr()), nb, stream)
    assert st == 3, L.mxfp4_last_error()
    _unchanged(torch, bufs, before)
    # a W^T copy that needs N % 32 == 0 with N = 240: rejected before X's pass as well
    st = L.mxfp4_linear_fprop(P(x.data_ptr()), P(wbuf.data_ptr()), M, 240, K, ctypes.byref(cc), P(y.data_ptr()),
                              ctypes.byref(cx), ctypes.byref(cw), P(ws.data_ptr()), nb, stream)
    assert st == 2, L.mxfp4_last_error()
    _unchanged(torch, bufs, before)
    assert mx.device_status() == 0


def test_rejected_dgrad_and_wgrad_leave_every_buffer_untouched():
    torch = gpu_ready()
    from mxfp4_precision_gemms_gb300 import binding as mx

    L = mx.lib()
    M, N, K = 256, 256, 512
    _, W, dY = synth.linear_inputs(M, N, K, 1)
    dy = mx.bf16_tensor(dY)
    # W^T quantised under H32, used in an H16 layer: the rotations would not cancel
    wT32 = mx.rotate_quantize(mx.bf16_tensor(W), had=mx.HAD_32, layouts=mx.LAYOUT_COLT)["colT"]
    cfg = mx.Config(had=mx.HAD_16, mode=mx.SCALE_FLOOR, out_dtype=mx.OUT_F32)
    nb = mx.workspace_bytes(mx.OP_DGRAD, M, N, K, cfg)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    dx = torch.empty((M, K), dtype=torch.float32, device="cuda")
    dyT = mx.empty_qtensor(N, M, mx.LAYOUT_COLT, mx.SF_MMA)
    bufs = [ws, dx, dyT.codes, dyT.scales]
    before = _sentinels(torch, *bufs)
    torch.cuda.synchronize()
    with pytest.raises(mx.Mxfp4Error) as e:
        mx.linear_dgrad(dy, wT32, cfg, dx=dx, dyT=dyT, ws=_FixedWorkspace(ws))
    assert e.value.status == 1 and "had" in str(e.value)
    _unchanged(torch, bufs, before)
    # Wgrad over an H16 dY^T and an H32 X^T
    xT32 = mx.rotate_quantize(mx.bf16_tensor(synth.activations(M, K, 2)), had=mx.HAD_32,
                              layouts=mx.LAYOUT_COLT)["colT"]
    dyT16 = mx.rotate_quantize(dy, had=mx.HAD_16, layouts=mx.LAYOUT_COLT)["colT"]
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    (dw_before,) = _sentinels(torch, dw)
    with pytest.raises(mx.Mxfp4Error):
        mx.linear_wgrad(dyT16, xT32, mx.Config(had=mx.HAD_16), dw=dw)
    with pytest.raises(mx.Mxfp4Error):
        mx.gemm(dyT16, xT32, out=dw)
    _unchanged(torch, [dw], [dw_before])
    assert mx.device_status() == 0


class _FixedWorkspace:
    """Hands out one given buffer (so the test can watch its bytes)."""

    def __init__(self, buf):
        self.buf = buf

    def get(self, nbytes, device):
        assert nbytes <= self.buf.numel()
        return self.buf[:nbytes]
