"""Accumulated-update study, RN against SR ("Stochastic rounding support for
8-bit optimizers", activity: compare both roundings with a higher-precision
reference, accumulated-update tests, several seeds; "Stochastic rounding of
AdamW momentums": weight decay lost in bf16).

Runs the library's steps (8-bit, fp32-state and bf16-state AdamW, each with
sr = 0 and sr = 1) against a float64 AdamW for 1000 steps and three seeds per
regime; the study and its metrics are described in rounding_study.py.
"""
import pytest

import rounding_study as S

pytestmark = pytest.mark.gpu

STEPS = 1000
SEEDS = (1, 2, 3)


def _final(regime, seed, device):
    return S.run(regime, seed, STEPS, device)[STEPS]


@pytest.mark.parametrize("seed", SEEDS)
def test_sub_ulp_updates_vanish_under_rn_and_survive_under_sr(cuda_device, seed):
    res = _final("sub-ulp", seed, cuda_device)
    for arm in S.ARMS:
        rn, sr = res[(arm, "RN")], res[(arm, "SR")]
        # RN: only parameters near zero (where an update reaches half an ulp) move
        assert rn["realised"] < 0.15 and rn["unmoved"] > 0.75, (arm, rn)
        # SR: unbiased, so the whole accumulated update arrives; the 8-bit state
        # adds its own small deficit (requantized second moments)
        lo = 0.95 if arm == "8bit" else 0.98
        assert lo < sr["realised"] < 1.02, (arm, sr)
        assert sr["rel_err"] < 0.3 and sr["rel_err"] < rn["rel_err"] / 3, (arm, sr, rn)
        assert sr["unmoved"] < 0.05, (arm, sr)


@pytest.mark.parametrize("seed", SEEDS)
def test_weight_decay_is_lost_under_rn_and_kept_under_sr(cuda_device, seed):
    res = _final("decay-only", seed, cuda_device)
    for arm in S.ARMS:
        rn, sr = res[(arm, "RN")], res[(arm, "SR")]
        # a 1e-5 relative shrink never reaches half a bf16 ulp: RN keeps every bit
        assert rn["realised"] == 0.0 and rn["unmoved"] == 1.0, (arm, rn)
        assert 0.93 < sr["realised"] < 1.07, (arm, sr)


@pytest.mark.parametrize("seed", SEEDS)
def test_growing_weights_stall_rn_but_not_sr(cuda_device, seed):
    res = _final("growing", seed, cuda_device)
    for arm in S.ARMS:
        rn, sr = res[(arm, "RN")], res[(arm, "SR")]
        lo = 0.95 if arm == "8bit" else 0.98
        assert lo < sr["realised"] < 1.02 and sr["rel_err"] < 0.08, (arm, sr)
        # once the weights have grown, RN drops the (now sub-ulp) updates
        assert rn["realised"] < 0.8 and rn["rel_err"] > 4 * sr["rel_err"], (arm, rn, sr)


@pytest.mark.parametrize("seed", SEEDS)
def test_noise_both_track_and_rn_has_less_variance(cuda_device, seed):
    res = _final("noise", seed, cuda_device)
    for arm in S.ARMS:
        rn, sr = res[(arm, "RN")], res[(arm, "SR")]
        for m in (rn, sr):
            assert 0.97 < m["realised"] < 1.03 and m["rel_err"] < 0.1, (arm, m)
        # with updates near or above an ulp, SR's extra variance costs more
        # than RN's rounding error
        assert rn["rel_err"] < sr["rel_err"], (arm, rn, sr)
