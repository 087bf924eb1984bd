"""SR toy (a reconstruction; parity unpinned, see sr_toy.py): with decaying
steps, round-to-nearest BF16 stalls short of the target, every
stochastically rounded run converges, close to the FP32 step count on average
and with a spread of run lengths above it."""
import numpy as np
import pytest

import sr_toy as T

pytestmark = pytest.mark.gpu


def test_sr_toy(cuda_device):
    t32 = T.fp32_steps()
    assert 0 < t32 < T.STEPS
    rn = T.bf16_steps(cuda_device, 0, runs=1)
    assert rn[0] < 0                                     # RN stalls: updates fall below half an ulp
    sr = T.bf16_steps(cuda_device, 1)
    assert np.all(sr > 0)                                # every SR run converges
    assert abs(sr.mean() - t32) < 0.1 * t32              # unbiased steps: near the FP32 count on average
    assert sr.max() > 1.1 * t32 and sr.std() > 0        # and a tail of slower runs
