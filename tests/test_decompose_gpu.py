"""GPU error-decomposition measurement vs the CPU oracle ("Decomposing MXFP4
quantization error ...", core insight): every per-element error term is computed in the
same arithmetic on both sides, so the sums agree up to fp64 summation order."""
import numpy as np
import pytest

import oracle
from mxfp4_precision_gemms_gb300 import synth
from tests.gpu_util import ORACLE_HAD, gpu_ready

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("had", [0, 16, 32])
@pytest.mark.parametrize("mode", [0, 1])
def test_decomposition_matches_oracle(had, mode):
    gpu_ready()
    from mxfp4_precision_gemms_gb300 import binding as mx

    for name, x in (("X", synth.activations(256, 512, 0)), ("sweep", synth.heavy_tailed(512, 1024, 1000)),
                    ("W", synth.weights(512, 512, 1))):
        got = mx.error_decomposition(mx.bf16_tensor(x), had=had, mode=mode)
        want = oracle.error_decomposition(x, ORACLE_HAD[had], mode)
        for k in mx.DECOMP_KEYS:
            assert abs(got[k] - want[k]) <= 1e-11 * max(abs(want[k]), 1e-300) + 1e-300, (name, k, got[k], want[k])
        if mode == 1:
            assert abs(got["e2"] - (got["scale2"] + got["dz2"] + got["grid2"] + 2 * got["scale_grid"])) <= 1e-10 * got["e2"]
