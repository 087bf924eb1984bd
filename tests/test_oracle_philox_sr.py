"""Pins for the oracle's Philox4x32-10 stream and its fp32 -> bf16 rounding.

Philox4x32-10 is the generator of Salmon et al., "Parallel Random Numbers: As
Easy as 1, 2, 3" (SC'11).  It is pinned against cuRAND's host-side generator of
the same name, an independent implementation that runs on the CPU: output word
4*j + i of that generator with seed s and offset 2^50*w1 + 2^18*w0 is word i of
Philox(counter = (w0, w1, j, 0), key = (s & 0xffffffff, s >> 32)).

Stochastic rounding ("Stochastic rounding support for 8-bit optimizers",
feature request: round up or down with a chance set by the rounding error) is
pinned by its exact expectation over all 2^16 random values, by exactness on
bf16 values, by a statistical test over the oracle's own Philox stream and by
the weight-decay survival case ("[Feat]: Stochastic rounding of AdamW
momentums", the linked decay-with-bf16 bug).
"""
import ctypes
import ctypes.util
import glob
import os
from fractions import Fraction as Fr

import numpy as np
import pytest
import torch

import oracle as o


def _load_curand():
    names = [ctypes.util.find_library("curand")]
    for root in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        names += sorted(glob.glob(os.path.join(root, "lib64", "libcurand.so*")))
    for n in names:
        if not n:
            continue
        try:
            return ctypes.CDLL(n)
        except OSError:
            continue
    pytest.skip("libcurand not found")


CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def curand_host_words(seed, offset, n):
    lib = _load_curand()
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
        return out
    finally:
        lib.curandDestroyGenerator(gen)


@pytest.mark.parametrize("seed", [0, 1, 0x123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_block_matches_curand_host(seed):
    key = (seed & 0xFFFFFFFF, seed >> 32)
    words = curand_host_words(seed, 0, 4 * 64)
    for j in range(64):
        assert np.array_equal(o.philox4x32_10((0, 0, j, 0), key), words[4 * j:4 * j + 4]), j
    # counter word 0 (steps of 2^18 outputs) and word 1 (steps of 2^50 outputs)
    for w0, w1, j in [(1, 0, 0), (3, 0, 5), (0, 1, 0), (2, 1, 7), (0x1234, 3, 11)]:
        got = curand_host_words(seed, (w1 << 50) + (w0 << 18) + 4 * j, 4)
        assert np.array_equal(o.philox4x32_10((w0, w1, j, 0), key), got), (w0, w1, j)


def test_r16_layout():
    # element E takes half (E & 1) of word (E >> 1) & 3 of the call for E >> 3
    seed, step, stream = 0xDEADBEEF01234567, 17, 2
    key = (seed & 0xFFFFFFFF, seed >> 32)
    for E in [0, 1, 2, 7, 8, 1000, (1 << 35) + 9, (1 << 40) + 3]:
        g = E >> 3
        w = o.philox4x32_10((g & 0xFFFFFFFF, stream, step, g >> 32), key)
        word = int(w[(E >> 1) & 3])
        want = (word >> 16) if (E & 1) else (word & 0xFFFF)
        assert o.r16(seed, step, stream, E) == want
    fill = o.philox_fill(seed, step, stream, 12345, 100)
    assert [o.r16(seed, step, stream, 12345 + i) for i in range(100)] == list(fill)


def test_r16_statistics():
    r = o.philox_fill(0, 1, 0, 0, 10_000_000).astype(np.float64)
    n = r.size
    sd = np.sqrt((65536.0 ** 2 - 1) / 12)
    assert abs(r.mean() - 32767.5) < 4 * sd / np.sqrt(n)
    # each of the 16 bits is set half the time
    ri = r.astype(np.uint32)
    for b in range(16):
        p = ((ri >> b) & 1).mean()
        assert abs(p - 0.5) < 4 * 0.5 / np.sqrt(n)
    # byte histogram chi-square (255 dof): mean 255, sd ~22.6
    hist = np.bincount((ri & 0xFF), minlength=256)
    chi2 = ((hist - n / 256) ** 2 / (n / 256)).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)
    # different streams and steps give different sequences
    a = o.philox_fill(0, 1, 1, 0, 64)
    b = o.philox_fill(0, 2, 0, 0, 64)
    assert not np.array_equal(a, r[:64].astype(np.uint16)) and not np.array_equal(b, a)


def _f32_from_bf16(h):
    return np.array([h << 16], np.uint32).view(np.float32)[0]


SR_VALUES = [1.0, -1.0, 1.0 + 2 ** -10, -(1.0 + 3 * 2 ** -12), 0.3, -0.3, 3.0e-39,
             -7.1e-40, 1e-30, 65504.1, 3.3e38, 1.17549435e-38, 2.5e-5]


@pytest.mark.parametrize("x", SR_VALUES)
def test_sr_exact_expectation(x):
    """Over all 2^16 random values the mean of SR(x) is x exactly."""
    x = np.float32(x)
    outs = np.array([o.sr_bf16(x, r) for r in range(0, 65536, 1)], np.uint32)
    vals, counts = np.unique(outs, return_counts=True)
    assert vals.size <= 2
    mean = sum(Fr(float(_f32_from_bf16(int(v)))) * int(c) for v, c in zip(vals, counts)) / 65536
    assert mean == Fr(float(x))


def test_sr_is_identity_on_bf16_values():
    rng = np.random.default_rng(3)
    hs = np.concatenate([rng.integers(0, 0x7F80, 200), rng.integers(0x8000, 0xFF80, 200),
                         [0, 0x8000, 0x7F7F, 0xFF7F, 0x0001, 0x8001, 0x7F80, 0xFF80]])
    for h in hs:
        x = _f32_from_bf16(int(h))
        for r in (0, 1, 0x7FFF, 0x8000, 0xFFFF, int(rng.integers(0, 65536))):
            assert o.sr_bf16(x, r) == h


def test_sr_nan_and_rne_against_torch():
    assert o.sr_bf16(np.float32("nan"), 0xFFFF) == 0x7FC0
    assert o.rne_bf16(np.float32("nan")) == 0x7FC0
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([o.rne_bf16(v) for v in x[:20000]], np.uint16)
    assert np.array_equal(got, want[:20000])


def test_sr_unbiased_over_philox_stream():
    """Mean of SR over 1e5 Philox draws lies within 3 sigma of x."""
    n = 100_000
    r = o.philox_fill(12345, 3, 0, 0, n)
    for x in (np.float32(1.0 + 2 ** -9), np.float32(-0.123456), np.float32(7.77e-6)):
        bits = int(np.array([x], np.float32).view(np.uint32)[0])
        lo = _f32_from_bf16(bits >> 16)
        hi = _f32_from_bf16((bits >> 16) + 1)
        ulp = abs(float(hi) - float(lo))
        p = (float(x) - float(lo)) / (float(hi) - float(lo))
        vals = np.array([_f32_from_bf16(o.sr_bf16(x, int(ri))) for ri in r], np.float64)
        sigma = ulp * np.sqrt(p * (1 - p) / n)
        assert abs(vals.mean() - float(x)) <= 3 * sigma + 1e-12


def test_weight_decay_survives_with_sr_only():
    """p = 1, g = 0, lr*wd = 1e-5: round-to-nearest never moves p; SR decays it
    in expectation as decay^steps."""
    n, steps = 4000, 1000
    one = np.full(n, 0x3F80, np.uint16)
    hp = o.hparams(lr=1e-3, weight_decay=1e-2, seed=9)
    st_sr = o.State8.zeros(one.copy(), np.zeros(n, np.uint16))
    st_rn = o.State8.zeros(one.copy(), np.zeros(n, np.uint16))
    for t in range(1, steps + 1):
        hp.step = t
        hp.sr = 1
        o.adamw8bit_sr_step([st_sr], hp)
        hp.sr = 0
        o.adamw8bit_sr_step([st_rn], hp)
    assert np.all(st_rn.param == 0x3F80)
    decay = float(o.step_scalars(hp).decay)
    expect = decay ** steps
    vals = (st_sr.param.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # each step rounds down with chance <= 1e-5 / 2^-8 < 0.003 (ulp 2^-8 below
    # 1), so the per-element variance is below steps * ulp^2 * 0.003
    sigma = np.sqrt(steps * (2.0 ** -8) ** 2 * 0.003 / n)
    assert abs(vals.mean() - expect) < 3 * sigma
    assert vals.mean() < 0.995


# An independent restatement of Philox4x32-10 in numpy uint32/uint64
# arithmetic, written from Salmon et al. (SC'11), section 4: each of the ten
# rounds multiplies counter words 0 and 2 by the two round multipliers,
# crosses the halves of the products with words 1 and 3 and the round key,
# and the key is bumped by the two Weyl constants between rounds.  Vectorised
# over many counters; used to pin counter word 3, which cuRAND's offset
# cannot reach (it is non-zero only past 2^35 elements).
_PHILOX_M = (np.uint64(0xD2511F53), np.uint64(0xCD9E8D57))
_PHILOX_W = (0x9E3779B9, 0xBB67AE85)


def _philox_numpy(ctr, key):
    c = [np.asarray(ctr[:, i], np.uint64) for i in range(4)]
    k0, k1 = int(key[0]), int(key[1])
    mask = np.uint64(0xFFFFFFFF)
    for _ in range(10):
        p0 = _PHILOX_M[0] * c[0]
        p1 = _PHILOX_M[1] * c[2]
        c = [(p1 >> np.uint64(32)) ^ c[1] ^ np.uint64(k0), p1 & mask,
             (p0 >> np.uint64(32)) ^ c[3] ^ np.uint64(k1), p0 & mask]
        k0 = (k0 + _PHILOX_W[0]) & 0xFFFFFFFF
        k1 = (k1 + _PHILOX_W[1]) & 0xFFFFFFFF
    return np.stack([x.astype(np.uint32) for x in c], axis=1)


def test_philox_numpy_restatement_agrees_with_curand():
    """The restatement above is itself right where cuRAND reaches (words 0-2)."""
    seed = 0x0123456789ABCDEF
    key = (seed & 0xFFFFFFFF, seed >> 32)
    ctr = np.array([[0, 0, j, 0] for j in range(32)], np.uint64)
    want = curand_host_words(seed, 0, 4 * 32).reshape(32, 4)
    assert np.array_equal(_philox_numpy(ctr, key), want)


@pytest.mark.parametrize("seed", [0, 0xFFFFFFFFFFFFFFFF, 0x9E3779B97F4A7C15])
def test_philox_word3_against_numpy_restatement(seed):
    rng = np.random.default_rng(seed & 0xFFFF)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint64)
    ctr = rng.integers(0, 2 ** 32, (300, 4), dtype=np.uint64)
    ctr[:100, 3] = rng.integers(1, 16, 100)          # small non-zero word 3 (E just past 2^35)
    ctr[100:110, 3] = 0xFFFFFFFF
    want = _philox_numpy(ctr, key)
    for i in range(ctr.shape[0]):
        assert np.array_equal(o.philox4x32_10(ctr[i].astype(np.uint32), key.astype(np.uint32)), want[i]), i


def test_r16_past_2_35_against_numpy_restatement():
    """Draws of elements E >= 2^35, where the high half of E/8 is counter word 3."""
    seed, step, stream = 0xC0FFEE0012345678, 123456, 1
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint64)
    Es = [(1 << 35) + i for i in range(40)] + [(1 << 40) + 7, (1 << 45) + 12345, (1 << 61) + 3]
    ctr = np.array([[(E >> 3) & 0xFFFFFFFF, stream, step, E >> 35] for E in Es], np.uint64)
    words = _philox_numpy(ctr, key)
    for E, w in zip(Es, words):
        word = int(w[(E >> 1) & 3])
        want = (word >> 16) if (E & 1) else (word & 0xFFFF)
        assert o.r16(seed, step, stream, E) == want, E


@pytest.mark.parametrize("x", [1.0 + 2 ** -9, -0.123456, 7.77e-6, 3.0e-39])
def test_sr_unbiased_over_philox_seeds(x):
    """SR of a fixed x at one element, over 10^5 distinct Philox seeds: the
    mean lies within 3 sigma of x (sigma = ulp * sqrt(p (1 - p) / n), p the
    chance of rounding up)."""
    n = 100_000
    x = np.float32(x)
    bits = int(np.array([x], np.float32).view(np.uint32)[0])
    lo = float(_f32_from_bf16(bits >> 16))
    hi = float(_f32_from_bf16((bits >> 16) + 1))
    p = (float(x) - lo) / (hi - lo)
    up = 0
    E = 987654321
    for seed in range(1, n + 1):
        h = o.sr_bf16(x, o.r16(seed * 0x9E3779B97F4A7C15 & 0xFFFFFFFFFFFFFFFF, 5, 0, E))
        assert h in (bits >> 16, (bits >> 16) + 1)
        up += h != (bits >> 16)
    mean = lo + (hi - lo) * up / n
    sigma = abs(hi - lo) * np.sqrt(p * (1 - p) / n)
    assert abs(mean - float(x)) <= 3 * sigma
