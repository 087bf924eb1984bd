"""Pins for the oracle's one-state optimizers with 8-bit blockwise state and
SR parameter write: SGD with momentum ("8-bit Optimizers via Block-wise
Quantization", introduction: Adam and Momentum states) and Lion ("Stochastic
rounding support for 8-bit optimizers", motivation: 8-bit Lion).  Formulas
follow the published definitions (PyTorch SGD with momentum; Chen et al. 2023,
Lion, Algorithm 2); each check uses exact rationals or a closed form.
"""
from fractions import Fraction as Fr

import numpy as np
import pytest

import oracle as o

MOM, LION = o.MOMENTUM, o.LION


def rn32(q):
    """Nearest float32 to the exact rational q (ties to even)."""
    x = np.float32(float(q))
    cands = [np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))]
    return np.float32(min(cands, key=lambda c: (abs(Fr(float(c)) - q),
                                                int(np.array([c], np.float32).view(np.uint32)[0]) & 1)))


F = lambda z: Fr(float(z))


def test_lion_against_exact_rationals():
    rng = np.random.default_rng(1)
    hp = o.hparams(lr=3e-4, beta1=0.9, beta2=0.99, weight_decay=0.1)
    s = o.step_scalars1(LION, hp)
    for _ in range(3000):
        g = np.float32(rng.standard_normal() * 10.0 ** rng.uniform(-6, 0))
        p = np.float32(rng.standard_normal() * 0.05)
        m = np.float32(rng.standard_normal() * 10.0 ** rng.uniform(-6, 0))
        pn, mn = o.onestate_element(LION, s, g, p, m)
        c = rn32(F(s.a) * F(m) + F(np.float32(s.oma) * g))
        u = np.sign(c)
        pd = np.float32(p * np.float32(s.decay))
        assert pn == rn32(F(s.lr_neg) * F(u) + F(pd))
        assert mn == rn32(F(s.b) * F(m) + F(np.float32(s.omb) * g))


def test_lion_step_is_sign_times_lr():
    """From zero state the update is exactly lr * sign(g) after the decay:
    |p_new - RN(p*decay)| is lr rounded once."""
    hp = o.hparams(lr=2 ** -10, beta1=0.9, beta2=0.99, weight_decay=0.0)
    s = o.step_scalars1(LION, hp)
    for g in (1e-9, -3.0, 0.5, -1e-30):
        pn, mn = o.onestate_element(LION, s, g, 1.0, 0.0)
        assert pn == np.float32(1.0 - np.sign(g) * 2 ** -10)
    pn, mn = o.onestate_element(LION, s, 0.0, 1.0, 0.0)         # sign(0) = 0
    assert pn == 1.0 and mn == 0.0


def test_momentum_against_exact_rationals():
    rng = np.random.default_rng(2)
    hp = o.hparams(lr=1e-2, beta1=0.9, weight_decay=5e-4)
    s = o.step_scalars1(MOM, hp)
    for _ in range(3000):
        g = np.float32(rng.standard_normal() * 10.0 ** rng.uniform(-6, 0))
        p = np.float32(rng.standard_normal() * 0.05)
        m = np.float32(rng.standard_normal() * 10.0 ** rng.uniform(-6, 0))
        pn, mn = o.onestate_element(MOM, s, g, p, m)
        d = rn32(F(s.wd) * F(p) + F(g))
        assert mn == rn32(F(s.a) * F(m) + F(d))
        assert pn == rn32(F(s.lr_neg) * F(mn) + F(p))


def test_momentum_closed_form_geometric_sum():
    """Constant gradient, no decay: m_t = g (1 - mu^t) / (1 - mu)."""
    hp = o.hparams(lr=0.0, beta1=0.9, weight_decay=0.0)
    s = o.step_scalars1(MOM, hp)
    m, g = np.float32(0), np.float32(0.001)
    for t in range(1, 60):
        _, m = o.onestate_element(MOM, s, g, 1.0, m)
        exact = 0.001 * (1 - np.float32(0.9).astype(np.float64) ** t) / (1 - np.float32(0.9).astype(np.float64))
        assert abs(float(m) - exact) <= 2e-6 * exact * t


def test_hand_worked_cases():
    # momentum: mu = 1/2, lr = 1/4, wd = 1/8, p = 1, g = 1/2, m = 1:
    # d = 1/8 + 1/2 = 5/8, m = 1/2 + 5/8 = 9/8, p = 1 - 9/32 = 23/32
    s = o.step_scalars1(MOM, o.hparams(lr=0.25, beta1=0.5, weight_decay=0.125))
    assert o.onestate_element(MOM, s, 0.5, 1.0, 1.0) == (np.float32(23 / 32), np.float32(9 / 8))
    # lion: b1 = 1/2, b2 = 3/4, lr = 1/8, wd = 1 (decay 7/8), p = 1, g = -1, m = 1/4:
    # c = 1/8 - 1/2 < 0 -> u = -1, p = 7/8 + 1/8 = 1, m = 3/16 - 1/4 = -1/16
    s = o.step_scalars1(LION, o.hparams(lr=0.125, beta1=0.5, beta2=0.75, weight_decay=1.0))
    assert o.onestate_element(LION, s, -1.0, 1.0, 0.25) == (np.float32(1.0), np.float32(-1 / 16))


def _bf16(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("opt", [MOM, LION])
def test_eight_bit_equals_fp32_state_at_step_one(opt):
    rng = np.random.default_rng(3)
    n = 2 * 2048 + 77
    p = _bf16(rng.standard_normal(n) * 0.02)
    g = _bf16(rng.standard_normal(n) * 1e-3)
    a = o.zeros_onestate(p.copy(), g, eight_bit=True)
    b = o.zeros_onestate(p.copy(), g, eight_bit=False)
    hp = o.hparams(lr=1e-3, beta1=0.9, beta2=0.99, weight_decay=0.01, step=1, seed=4)
    o.onestate8bit_tensor(opt, a, 0, hp)
    o.onestate32_tensor(opt, b, 0, hp)
    assert np.array_equal(a.param, b.param)
    mq = o.dequantize(o.SIGNED, a.m_codes, a.m_absmax)
    M = np.repeat(a.m_absmax, 2048)[:n]
    assert np.all(np.abs(mq - b.m32) <= M * (0.9 / 64 / 2 + 2 ** -22))


@pytest.mark.parametrize("opt", [MOM, LION])
def test_list_routing_and_offsets(opt):
    rng = np.random.default_rng(5)
    sizes = [5000, 100, 2048 * 3]
    params = [_bf16(rng.standard_normal(n) * 0.02) for n in sizes]
    grads = [_bf16(rng.standard_normal(n) * 1e-3) for n in sizes]
    hp = o.hparams(lr=1e-3, beta1=0.9, beta2=0.99, weight_decay=0.01, step=2, seed=6)
    whole = [o.zeros_onestate(p.copy(), g) for p, g in zip(params, grads)]
    o.onestate_sr_step(opt, whole, hp)
    offs = [0, 5000, 5100]
    parts = [o.zeros_onestate(p.copy(), g, philox_offset=off) for p, g, off in zip(params, grads, offs)]
    for st in parts:
        o.onestate_sr_step(opt, [st], hp)
    for a, b in zip(whole, parts):
        assert np.array_equal(a.param, b.param)


@pytest.mark.parametrize("opt", [MOM, LION])
def test_eight_bit_step_is_the_composition_of_its_pinned_parts(opt):
    """At a later step (nonzero 8-bit state, partial last block): dequantize,
    the element update, blockwise requantization of the new m and the
    stochastically rounded parameter write with the element's stream-0 draw."""
    rng = np.random.default_rng(23)
    n = 2 * 2048 + 555
    p = _bf16(rng.standard_normal(n) * 0.02)
    g = _bf16(rng.standard_normal(n) * 1e-3)
    mc, ma = o.quantize(o.SIGNED, (rng.standard_normal(n) * 1e-3).astype(np.float32))
    hp = o.hparams(lr=1e-3, beta1=0.9, beta2=0.99, weight_decay=0.01, step=5, seed=17)
    E0 = 4242
    st = o.State8(p.copy(), g, m_codes=mc.copy(), m_absmax=ma.copy())
    o.onestate8bit_tensor(opt, st, E0, hp)
    s = o.step_scalars1(opt, hp)
    m = o.dequantize(o.SIGNED, mc, ma)
    pf = np.zeros(n, np.float32)
    for i in range(n):
        pf[i], m[i] = o.onestate_element(opt, s, o.bf16_to_f32(g[i]), o.bf16_to_f32(p[i]), m[i])
    want_mc, want_ma = o.quantize(o.SIGNED, m)
    want_p = np.array([o.sr_bf16(pf[i], o.r16(17, 5, 0, E0 + i)) for i in range(n)], np.uint16)
    assert np.array_equal(st.param, want_p)
    assert np.array_equal(st.m_codes, want_mc)
    assert np.array_equal(st.m_absmax.view(np.uint32), want_ma.view(np.uint32))
