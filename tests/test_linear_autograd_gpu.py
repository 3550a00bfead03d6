"""The autograd linear layer (mxfp4_precision_gemms_gb300.linear): its forward output and
both gradients must be byte-identical to the three linear-layer calls made directly,
for a 3-D activation (batch x tokens x features) and for both scale modes."""
import pytest

from mxfp4_precision_gemms_gb300 import synth


@pytest.mark.gpu
@pytest.mark.parametrize("had,mode", [(16, 0), (32, 1), (0, 0)])
def test_autograd_linear_matches_direct_calls(had, mode):
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300.linear import mxfp4_linear

    M, N, K = 256, 512, 512
    X, W, dY = synth.linear_inputs(M, N, K, 0)
    x = mx.bf16_tensor(X)
    w = mx.bf16_tensor(W)
    dy = mx.bf16_tensor(dY)

    xa = x.clone().reshape(2, M // 2, K).requires_grad_(True)
    wa = w.clone().requires_grad_(True)
    y = mxfp4_linear(xa, wa, had=had, mode=mode)
    assert y.shape == (2, M // 2, N) and y.dtype == torch.bfloat16
    y.backward(dy.reshape(2, M // 2, N))
    torch.cuda.synchronize()
    assert mx.device_status() == 0

    cfg = mx.Config(had=had, mode=mode, out_dtype=mx.OUT_BF16)
    y_ref, xT, wT = mx.linear_fprop(x, w, cfg)
    dx_ref, dyT = mx.linear_dgrad(dy, wT, cfg)
    dw_ref = mx.linear_wgrad(dyT, xT, mx.Config(had=had, mode=mode, out_dtype=mx.OUT_F32))
    torch.cuda.synchronize()
    assert torch.equal(y.reshape(M, N), y_ref)
    assert torch.equal(xa.grad.reshape(M, K), dx_ref)
    assert wa.grad.dtype == torch.bfloat16
    assert torch.equal(wa.grad, dw_ref.to(torch.bfloat16))
    # and the layer is the linear map it claims to be, to MXFP4 accuracy
    dense = (x.float() @ w.float().t())
    rel = ((y_ref.float() - dense).norm() / dense.norm()).item()
    assert rel < 0.2, rel
