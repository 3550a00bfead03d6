"""Failure detection without a GPU fault: a GEMM whose first K stage is never loaded
(host-side fault injection) must end its bounded waits, report MXFP4_ERR_TIMEOUT
through the status word, and leave the context usable for the next call."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import assert_within, gpu_ready

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [256, 128])  # CTA-pair kernel, single-CTA kernel
def test_bounded_wait_timeout_is_reported(M):
    torch = gpu_ready()
    from mxfp4_precision_gemms_gb300 import binding as mx

    X, W, _ = synth.linear_inputs(M, 256, 1024, 21)
    qa, qb = oracle.quantize(X, 16, 0, "row"), oracle.quantize(W, 16, 0, "row")
    A, B = mx.qtensor_from_host(*qa), mx.qtensor_from_host(*qb)
    assert mx.device_status() == 0
    mx.set_wait_limit_ns(50_000_000)  # 50 ms
    try:
        mx.lib().mxfp4_test_inject_gemm_fault(1)
        mx.gemm(A, B)
        assert mx.device_status() == 6  # MXFP4_ERR_TIMEOUT
        assert b"wait" in mx.lib().mxfp4_last_error()
        assert mx.device_status() == 0  # cleared by the read
    finally:
        mx.lib().mxfp4_test_inject_gemm_fault(0)
        mx.set_wait_limit_ns(0)
    # the context is still usable and the next GEMM is correct
    C = mx.gemm(A, B)
    assert mx.device_status() == 0
    want, S = oracle.gemm(*qa, *qb)
    assert_within(C.double().cpu().numpy(), want, S, what="after timeout")
