"""Pins for the oracle's fp32 AdamW element update and its whole-step plumbing.

AdamW with decoupled weight decay is named on "Stochastic Rounding for LLM
Training: Theory and Practice" (TL;DR); the update runs in 32 bit ("8-bit
Optimizers via Block-wise Quantization", method bullets) with the add and
divide in fp32 ("[Feat]: Stochastic rounding of AdamW momentums").  The update
is pinned by hand-worked exact cases, by the bias-correction closed form at
step 1 and by a 60-digit evaluation of the textbook formula
p*(1 - lr*wd) - lr * mhat / (sqrt(vhat) + eps).
"""
from fractions import Fraction as Fr

import mpmath
import numpy as np
import pytest

import oracle as o

mpmath.mp.dps = 60


def ulp(x):
    x = abs(np.float32(x))
    return float(np.nextafter(x, np.float32(np.inf)) - x) if x > 0 else 2.0 ** -149


def exact_adamw(g, p, m, v, lr, b1, b2, eps, wd, t):
    """Textbook AdamW in 60-digit arithmetic (bias-corrected moments)."""
    g, p, m, v = (mpmath.mpf(float(z)) for z in (g, p, m, v))
    lr, b1, b2, eps, wd = (mpmath.mpf(z) for z in (lr, b1, b2, eps, wd))
    m_new = b1 * m + (1 - b1) * g
    v_new = b2 * v + (1 - b2) * g * g
    mhat = m_new / (1 - b1 ** t)
    vhat = v_new / (1 - b2 ** t)
    p_new = p * (1 - lr * wd) - lr * mhat / (mpmath.sqrt(vhat) + eps)
    return p_new, m_new, v_new


def test_hand_worked_exact_case():
    # b1 = 1/2, b2 = 3/4, lr = 1/2, eps = 0, wd = 0, t = 1, g = p = 1, zero state:
    # m = 1/2, v = 1/4, a_t = lr*sqrt(1/4)/(1/2) = 1/2, sqrt(v) = 1/2, m/den = 1,
    # p = 1 - 1/2 = 1/2 -- every intermediate is a short binary fraction.
    hp = o.hparams(lr=0.5, beta1=0.5, beta2=0.75, eps=0.0, weight_decay=0.0, step=1)
    s = o.step_scalars(hp)
    assert (s.step_size, s.eps_t, s.decay) == (0.5, 0.0, 1.0)
    pn, mn, vn = o.adamw_element(s, 1.0, 1.0, 0.0, 0.0)
    assert (pn, mn, vn) == (0.5, 0.5, 0.25)
    # t = 2 from (m, v) = (1/2, 1/4) with g = -1, p = 1/2, wd = 1/4:
    # m = -1/4, v = 7/16, bc1 = 3/4, bc2 = 7/16, a_t = (1/2)(sqrt(7)/4)/(3/4),
    # m/den = (-1/4)/(sqrt(7)/4) = -1/sqrt(7), so p = 1/2*(1 - 1/8) + 1/6 = 0.60416...
    hp = o.hparams(lr=0.5, beta1=0.5, beta2=0.75, eps=0.0, weight_decay=0.25, step=2)
    s = o.step_scalars(hp)
    pn, mn, vn = o.adamw_element(s, -1.0, 0.5, 0.5, 0.25)
    assert mn == -0.25 and vn == 0.4375
    assert abs(float(pn) - (0.4375 + 1.0 / 6.0)) <= 2 * ulp(pn)


def test_step_one_closed_form():
    """From zero state at t = 1: mhat = g and sqrt(vhat) = |g|, so
    p1 = p*(1 - lr*wd) - lr*g/(|g| + eps)."""
    rng = np.random.default_rng(1)
    hp = o.hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1)
    s = o.step_scalars(hp)
    for _ in range(2000):
        g = np.float32(rng.standard_normal() * 10.0 ** rng.uniform(-9, 1))
        p = np.float32(rng.standard_normal() * 0.02)
        pn, mn, vn = o.adamw_element(s, g, p, 0.0, 0.0)
        want = float(p) * (1 - 1e-5) - 1e-3 * float(g) / (abs(float(g)) + 1e-8)
        assert abs(float(pn) - want) <= 4 * ulp(max(abs(want), 1e-3)), (g, p)
    # zero gradient: only the decay acts
    pn, _, _ = o.adamw_element(s, 0.0, 0.75, 0.0, 0.0)
    assert pn == np.float32(0.75) * s.decay


@pytest.mark.parametrize("t", [1, 2, 10, 1000, 100000])
def test_against_high_precision_textbook(t):
    rng = np.random.default_rng(t)
    lr, b1, b2, eps, wd = 6e-4, 0.9, 0.999, 1e-8, 0.1
    hp = o.hparams(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd, step=t)
    s = o.step_scalars(hp)
    for _ in range(1500):
        scale = 10.0 ** rng.uniform(-10, 0)        # includes the eps-dominated regime
        g = np.float32(rng.standard_normal() * scale)
        m = np.float32(rng.standard_normal() * scale * 0.3)
        v = np.float32(abs(rng.standard_normal()) * scale * scale)
        p = np.float32(rng.standard_normal() * 0.05)
        pn, mn, vn = o.adamw_element(s, g, p, m, v)
        ep, em, ev = exact_adamw(g, p, m, v, lr, b1, b2, eps, wd, t)
        # moments: two products and a sum, each rounded once (+ rounded betas)
        assert abs(float(mn) - float(em)) <= 3 * ulp(max(abs(float(em)), abs(float(m)), abs(float(g)) * 0.1))
        assert abs(float(vn) - float(ev)) <= 3 * ulp(max(float(ev), float(v)))
        # parameter: a few ulps of the update term plus one of p
        upd = abs(float(ep) - float(p) * (1 - lr * wd))
        tol = 8 * ulp(max(upd, 1e-30)) + 2 * ulp(p)
        assert abs(float(pn) - float(ep)) <= tol, (t, g, m, v, p)


def test_scalars_match_definition():
    hp = o.hparams(lr=1.2e-3, beta1=0.9, beta2=0.95, eps=1e-6, weight_decay=0.1, step=7)
    s = o.step_scalars(hp)
    bc1 = 1 - mpmath.mpf(0.9) ** 7
    bc2 = 1 - mpmath.mpf(0.95) ** 7
    assert abs(float(s.step_size) - float(mpmath.mpf(1.2e-3) * mpmath.sqrt(bc2) / bc1)) <= ulp(s.step_size)
    assert abs(float(s.eps_t) - float(mpmath.mpf(1e-6) * mpmath.sqrt(bc2))) <= ulp(s.eps_t)
    assert s.decay == np.float32(1 - 1.2e-4)
    assert s.omb1 == np.float32(0.1) and s.omb2 == np.float32(0.05)


def _bf16(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _tensor(rng, n):
    return _bf16(rng.standard_normal(n) * 0.02), _bf16(rng.standard_normal(n) * 1e-3)


def test_eight_bit_path_matches_fp32_path_at_step_one():
    """From zero state, the stored moments are exactly zero on both paths, so
    step 1 gives identical parameters; the requantized moments then lie within
    the round-trip bound of the fp32 moments."""
    rng = np.random.default_rng(2)
    n = 3 * 2048 + 100
    p, g = _tensor(rng, n)
    a = o.State8.zeros(p.copy(), g)
    b = o.State8(p.copy(), g, m32=np.zeros(n, np.float32), v32=np.zeros(n, np.float32))
    hp = o.hparams(step=1, seed=5)
    o.adamw8bit_tensor(a, 0, hp)
    o.adamw32_tensor(b, 0, hp)
    assert np.array_equal(a.param, b.param)
    mq = o.dequantize(o.SIGNED, a.m_codes, a.m_absmax)
    vq = o.dequantize(o.UNSIGNED, a.v_codes, a.v_absmax)
    M = np.repeat(a.m_absmax, 2048)[:n]
    V = np.repeat(a.v_absmax, 2048)[:n]
    assert np.all(np.abs(mq - b.m32) <= M * (0.9 / 64 / 2 + 2 ** -22))
    assert np.all(np.abs(vq - b.v32) <= V * (0.9 / 128 / 2 + 2 ** -22))
    assert np.all(a.m_absmax == np.array([np.abs(b.m32[i:i + 2048]).max() for i in range(0, n, 2048)]))


def test_resume_and_split_invariance():
    rng = np.random.default_rng(3)
    sizes = [5000, 300, 4096, 2048 * 3 + 7, 1]
    params = [_tensor(rng, n) for n in sizes]
    grads = [[_bf16(rng.standard_normal(n) * 1e-3) for n in sizes] for _ in range(10)]

    def run(states, steps, split=False):
        for t in steps:
            for st, g in zip(states, grads[t - 1]):
                st.grad = g
            hp = o.hparams(step=t, seed=77)
            if split:
                offs = np.concatenate([[0], np.cumsum(sizes)[:-1]])
                for st, off in zip(states, offs):
                    st.philox_offset = int(off)
                o.adamw8bit_sr_step(states[:2], hp)
                o.adamw8bit_sr_step(states[2:], hp)
            else:
                o.adamw8bit_sr_step(states, hp)

    full = [o.State8.zeros(p.copy(), g) for p, g in params]
    run(full, range(1, 11))
    half = [o.State8.zeros(p.copy(), g) for p, g in params]
    run(half, range(1, 6))
    run(half, range(6, 11), split=True)
    for a, b in zip(full, half):
        assert np.array_equal(a.param, b.param)
        if a.m_codes is not None:
            assert np.array_equal(a.m_codes, b.m_codes) and np.array_equal(a.v_absmax, b.v_absmax)
        else:
            assert np.array_equal(a.m32, b.m32)


def test_small_tensor_routing_and_offsets():
    """Tensors below 4096 elements keep fp32 state; the Philox offset of each
    tensor is the running element count (checked through the SR draw)."""
    rng = np.random.default_rng(4)
    p1, g1 = _tensor(rng, 4095)
    p2, g2 = _tensor(rng, 4096)
    a = o.State8.zeros(p1.copy(), g1)
    b = o.State8.zeros(p2.copy(), g2)
    assert a.m32 is not None and b.m_codes is not None
    hp = o.hparams(step=3, seed=123)
    o.adamw8bit_sr_step([a, b], hp)
    # redo tensor b alone with the explicit offset 4095: same bits
    c = o.State8.zeros(p2.copy(), g2, philox_offset=4095)
    o.adamw8bit_sr_step([c], hp)
    assert np.array_equal(b.param, c.param)
    d = o.State8.zeros(p2.copy(), g2, philox_offset=0)
    o.adamw8bit_sr_step([d], hp)
    assert not np.array_equal(b.param, d.param)


def test_bf16_state_variant():
    """BF16 state: fp32 maths, three independent SR streams; the expectation of
    the stored moments equals the fp32 moments (SR is unbiased)."""
    rng = np.random.default_rng(6)
    n = 20000
    p, g = _tensor(rng, n)
    m0 = _bf16(rng.standard_normal(n) * 1e-4)
    v0 = _bf16(np.abs(rng.standard_normal(n)) * 1e-8)
    hp = o.hparams(lr=1.2e-3, weight_decay=0.1, step=4, seed=8)
    st = o.State16(p.copy(), g, m0.copy(), v0.copy())
    o.adamw_bf16_sr_step([st], hp)
    s = o.step_scalars(hp)
    f = lambda h: (h.astype(np.uint32) << 16).view(np.float32)
    for i in range(0, n, 997):
        pn, mn, vn = o.adamw_element(s, f(g[i:i + 1])[0], f(p[i:i + 1])[0], f(m0[i:i + 1])[0], f(v0[i:i + 1])[0])
        for got, want in ((st.param[i], pn), (st.m[i], mn), (st.v[i], vn)):
            lo = int(np.array([want], np.float32).view(np.uint32)[0] >> 16)
            assert got in (lo, lo + 1)
    assert np.all(f(st.v) >= 0)


def _round_f32(q):
    """Nearest float32 to the exact rational q (ties to even)."""
    x = np.float32(float(q))
    cands = [np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Fr(float(c)) - q), int(np.array([c], np.float32).view(np.uint32)[0]) & 1))
    return np.float32(best)


def test_multiply_adds_are_fused():
    """Each multiply-add of the update rounds once (fmaf): checked against
    exact rational arithmetic on inputs where fused and unfused differ."""
    rng = np.random.default_rng(9)
    hp = o.hparams(lr=6e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, step=3)
    s = o.step_scalars(hp)
    fused_differs = 0
    for _ in range(3000):
        g = np.float32(rng.standard_normal() * 1e-3)
        p = np.float32(rng.standard_normal() * 0.02)
        m = np.float32(rng.standard_normal() * 3e-4)
        v = np.float32(abs(rng.standard_normal()) * 1e-6)
        pn, mn, vn = o.adamw_element(s, g, p, m, v)
        f = lambda z: Fr(float(z))
        want_m = _round_f32(f(s.b1) * f(m) + f(np.float32(s.omb1) * g))
        want_v = _round_f32(f(s.b2) * f(v) + f(np.float32(s.omb2) * np.float32(g * g)))
        assert mn == want_m and vn == want_v
        ratio = np.float32(mn / np.float32(np.float32(np.sqrt(vn)) + np.float32(s.eps_t)))
        want_p = _round_f32(-f(s.step_size) * f(ratio) + f(np.float32(p * np.float32(s.decay))))
        assert pn == want_p
        unfused = np.float32(np.float32(p * np.float32(s.decay)) - np.float32(np.float32(s.step_size) * ratio))
        fused_differs += int(unfused != pn)
    assert fused_differs > 0          # the cases do tell the two readings apart


def test_eight_bit_step_is_the_composition_of_its_pinned_parts():
    """At a later step (nonzero 8-bit state, partial last block), the 8-bit
    tensor step equals, element by element: dequantize the codes ([BW] method
    bullets: lookup table times block absmax), the fp32 AdamW element update,
    blockwise requantization of the new m and v, and the stochastically
    rounded parameter write with the element's own Philox draw -- each part
    pinned separately in this directory."""
    rng = np.random.default_rng(21)
    n = 2 * 2048 + 333
    p = (np.asarray(rng.standard_normal(n) * 0.02, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    g = (np.asarray(rng.standard_normal(n) * 1e-3, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    m0 = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v0 = (rng.random(n) * 1e-8).astype(np.float32)
    mc, ma = o.quantize(o.SIGNED, m0)
    vc, va = o.quantize(o.UNSIGNED, v0)
    hp = o.hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=7, seed=13)
    E0 = 12345
    st = o.State8(p.copy(), g, mc.copy(), vc.copy(), ma.copy(), va.copy())
    o.adamw8bit_tensor(st, E0, hp)

    s = o.step_scalars(hp)
    m = o.dequantize(o.SIGNED, mc, ma)
    v = o.dequantize(o.UNSIGNED, vc, va)
    pf = np.zeros(n, np.float32)
    for i in range(n):
        pf[i], m[i], v[i] = o.adamw_element(s, o.bf16_to_f32(g[i]), o.bf16_to_f32(p[i]), m[i], v[i])
    want_mc, want_ma = o.quantize(o.SIGNED, m)
    want_vc, want_va = o.quantize(o.UNSIGNED, v)
    want_p = np.array([o.sr_bf16(pf[i], o.r16(13, 7, 0, E0 + i)) for i in range(n)], np.uint16)
    assert np.array_equal(st.param, want_p)
    assert np.array_equal(st.m_codes, want_mc) and np.array_equal(st.v_codes, want_vc)
    assert np.array_equal(st.m_absmax.view(np.uint32), want_ma.view(np.uint32))
    assert np.array_equal(st.v_absmax.view(np.uint32), want_va.view(np.uint32))


def test_bf16_step_is_the_composition_of_its_pinned_parts():
    """BF16 state at a later step: every element equals the fp32 element
    update followed by stochastic rounding of p, m and v with the draws of
    Philox streams 0, 1 and 2 at that element ("Stochastic rounding of AdamW
    momentums": fp32 maths, stochastically rounded write-back)."""
    rng = np.random.default_rng(22)
    n = 3000
    p, g = _tensor(rng, n)
    m0 = _bf16(rng.standard_normal(n) * 1e-4)
    v0 = _bf16(np.abs(rng.standard_normal(n)) * 1e-8)
    hp = o.hparams(lr=1.2e-3, weight_decay=0.1, step=9, seed=31)
    E0 = 777
    st = o.State16(p.copy(), g, m0.copy(), v0.copy(), philox_offset=E0)
    o.adamw_bf16_sr_step([st], hp)
    s = o.step_scalars(hp)
    for i in range(n):
        pn, mn, vn = o.adamw_element(s, o.bf16_to_f32(g[i]), o.bf16_to_f32(p[i]), o.bf16_to_f32(m0[i]),
                                     o.bf16_to_f32(v0[i]))
        assert st.param[i] == o.sr_bf16(pn, o.r16(31, 9, 0, E0 + i))
        assert st.m[i] == o.sr_bf16(mn, o.r16(31, 9, 1, E0 + i))
        assert st.v[i] == o.sr_bf16(vn, o.r16(31, 9, 2, E0 + i))
