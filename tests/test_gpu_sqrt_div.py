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
    counts = torch.zeros(8, dtype=torch.int64, device=cuda_device)
    q8.q8_selftest_sqrt_div(counts)
    bad_y, checked, bad_q, pairs, bad_s, checked_v, err_s, err_r = (int(x) for x in counts.cpu())
    assert checked == 0x7E800000 - 0x00800000
    assert bad_y == 0
    assert pairs == 2 * 2 * checked
    assert bad_q == 0
    assert checked_v == 0x7F800000 - 0x0D800000
    assert bad_s == 0


def test_fast_mode_approximations_within_bound(cuda_device):
    """The fast mode's approximate square root and reciprocal are each within
    2^-21 relative error over every normal input: the bound its per-thread
    cancellation check is derived from (with a factor of two to spare)."""
    import math
    import struct
    counts = torch.zeros(8, dtype=torch.int64, device=cuda_device)
    q8.q8_selftest_sqrt_div(counts)
    as_float = lambda b: struct.unpack("<f", struct.pack("<I", int(b)))[0]
    err_s, err_r = as_float(counts[6].item()), as_float(counts[7].item())
    print("largest relative error: sqrt.approx.ftz %.3g (2^%.2f), rcp.approx.ftz %.3g (2^%.2f)" % (
        err_s, math.log2(err_s), err_r, math.log2(err_r)))
    assert 0.0 < err_s <= 2.0 ** -21
    assert 0.0 < err_r <= 2.0 ** -21
