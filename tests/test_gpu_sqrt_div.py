"""The packed square root and division the AdamW steps use where they are
exact (Markstein's correction with y = RN(1/d), "Computation of elementary
functions on the IBM RISC System/6000 processor", 1990; the reciprocal square
root with one Newton-Raphson correction) against CUDA's IEEE reciprocal,
division and square root, on the device: y for every positive normal d with a
normal reciprocal, seeded pseudo-random quotients spanning the bounds inside
which the steps take the packed path, and the square root of every normal
v >= 2^-100."""
import pytest
import torch

import bit_blockwise_adamw_gb300 as q8

pytestmark = pytest.mark.gpu


def test_sqrt_div_selftest(cuda_device):
    counts = torch.zeros(6, dtype=torch.int64, device=cuda_device)
    q8.q8_selftest_sqrt_div(counts)
    bad_y, checked, bad_q, pairs, bad_s, checked_v = (int(x) for x in counts.cpu())
    assert checked == 0x7E800000 - 0x00800000
    assert bad_y == 0
    assert pairs == 2 * 2 * checked
    assert bad_q == 0
    assert checked_v == 0x7F800000 - 0x0D800000
    assert bad_s == 0
