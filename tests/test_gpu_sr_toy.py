"""SR toy (a reconstruction; parity unpinned, see sr_toy.py): with decaying
steps, round-to-nearest BF16 never moves, every stochastically rounded run
converges, slower than FP32 on average, and single runs take many times the
FP32 step count -- the outcomes the pages report for their toy."""
import numpy as np
import pytest

import sr_toy as T

pytestmark = pytest.mark.gpu


def test_sr_toy(cuda_device):
    t32 = T.fp32_steps()
    assert 0 < t32 < 20_000
    rn = T.bf16_steps(cuda_device, 0, runs=1)
    assert rn[0] < 0                                     # RN stalls: every update is below half a spacing
    sr = T.bf16_steps(cuda_device, 1)
    assert np.all(sr > 0)                                # every SR run converges
    assert sr.mean() > 1.2 * t32                         # slower than FP32 on average
    assert sr.max() > 4 * t32                            # with single runs far slower still
    assert np.median(sr) < sr.mean()                     # a right-skewed spread of run lengths
