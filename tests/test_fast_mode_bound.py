"""The rounding lemma behind the fast mode's one-ulp guarantee, checked on the
host (no GPU).

The fast mode computes the parameter update P from an approximate quotient
and redoes an element on the exact path unless |P| >= |q| * a_t * 2^-9.  Past
that bound its P and the exact P differ by at most 2^-9 of their magnitude,
with the same sign.  The lemma: two such fp32 values, rounded to bf16 with the
same 16-bit stochastic-rounding draw (bits + r, keep the top half) or to
nearest even, land at most one bf16 ulp apart.  Checked here on random pairs
spread over the whole exponent range, on pairs placed at binade edges and at
the largest allowed distance, and with every draw for a few fixed pairs.
The quotient bound the cancellation check rests on (within 2^-19 of the
correctly rounded quotient) is checked by emulation too.
"""
import numpy as np


def _sr(bits, r):
    return ((bits.astype(np.uint64) + r.astype(np.uint64)) >> 16).astype(np.int64)


def _rne(bits):
    b = bits.astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.int64)


def _pairs(rng, n):
    """fp32 pairs (a, b) of the same sign with |a - b| <= 2^-9 * min(|a|, |b|)."""
    e = rng.integers(-120, 120, n)
    a = (rng.uniform(1.0, 2.0, n) * np.exp2(e.astype(np.float64))).astype(np.float32)
    rel = rng.uniform(-1.0, 1.0, n) * 2.0 ** -9 * (1.0 - 2.0 ** -20)
    b = (a.astype(np.float64) * (1.0 + rel)).astype(np.float32)
    # keep only pairs that meet the bound after the cast to fp32
    lo = np.minimum(np.abs(a), np.abs(b)).astype(np.float64)
    ok = np.abs(a.astype(np.float64) - b.astype(np.float64)) <= 2.0 ** -9 * lo
    sign = np.where(rng.integers(0, 2, n) == 1, -1.0, 1.0).astype(np.float32)
    return (a * sign)[ok], (b * sign)[ok]


def _check(a, b, r):
    ba, bb = a.view(np.uint32), b.view(np.uint32)
    # same sign: the bf16 results are ordered like their magnitudes' bit patterns
    assert np.all((ba >> 31) == (bb >> 31))
    assert np.abs(_sr(ba, r) - _sr(bb, r)).max() <= 1
    assert np.abs(_rne(ba) - _rne(bb)).max() <= 1


def test_random_pairs_round_within_one_ulp():
    rng = np.random.default_rng(11)
    a, b = _pairs(rng, 2_000_000)
    r = rng.integers(0, 1 << 16, a.size).astype(np.uint32)
    _check(a, b, r)


def test_pairs_at_binade_edges_and_the_largest_distance():
    rng = np.random.default_rng(12)
    e = rng.integers(-120, 120, 200_000).astype(np.float64)
    # a just below a power of two, b pushed across it by the largest allowed amount
    a = (np.exp2(e) * (1.0 - 2.0 ** -24)).astype(np.float32)
    b = (a.astype(np.float64) * (1.0 + 2.0 ** -9 * (1.0 - 2.0 ** -20))).astype(np.float32)
    keep = np.abs(a.astype(np.float64) - b.astype(np.float64)) <= 2.0 ** -9 * np.minimum(a, b)
    a, b = a[keep], b[keep]
    r = rng.integers(0, 1 << 16, a.size).astype(np.uint32)
    _check(a, b, r)
    _check(-a, -b, r)


def test_every_draw_for_fixed_pairs():
    r = np.arange(1 << 16, dtype=np.uint32)
    for x in (1.0, 1.9999999, 3.0e-5, 6.1e-5, 2.0 ** -126 * 1.5, 1.0e30):
        a = np.full(r.size, x, np.float32)
        b = (a.astype(np.float64) * (1.0 + 2.0 ** -9 * (1.0 - 2.0 ** -20))).astype(np.float32)
        _check(a, b, r)
        _check(b, a, r)


def test_the_bound_is_needed():
    """At a relative distance of 2^-6 (eight times the bound) some draw puts
    the two results two or more ulps apart: the check above can fail."""
    r = np.arange(1 << 16, dtype=np.uint32)
    a = np.full(r.size, 1.3, np.float32)
    b = (a.astype(np.float64) * (1.0 + 2.0 ** -6)).astype(np.float32)
    assert np.abs(_sr(a.view(np.uint32), r) - _sr(b.view(np.uint32), r)).max() >= 2


def test_quotient_error_bound():
    """The other half of the argument: with the approximate square root and
    reciprocal each within 2^-21 relative error (the device self-test measures
    about 2^-23.3), and the packed add and multiply rounded to fp32, the fast
    quotient m * rcp(sqrt(v) + eps_t) lies within 2^-19 of the correctly rounded
    m / (sqrt(v) + eps_t).  Emulated in float64 with the roundings to fp32 at
    the same places, the approximation errors at their extremes."""
    rng = np.random.default_rng(13)
    n = 2_000_000
    f32 = lambda x: np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
    v = f32(np.exp2(rng.uniform(-126, 120, n)))
    m = f32(np.exp2(rng.uniform(-120, 60, n)) * np.where(rng.integers(0, 2, n) == 1, -1.0, 1.0))
    eps = f32(np.exp2(rng.uniform(-36, 20, n)))
    exact = f32(m / f32(f32(np.sqrt(v)) + eps))
    es = rng.choice([-1.0, 1.0], n) * 2.0 ** -21
    er = rng.choice([-1.0, 1.0], n) * 2.0 ** -21
    s_a = f32(np.sqrt(v) * (1.0 + es))
    d_a = f32(s_a + eps)
    y_a = f32((1.0 / d_a) * (1.0 + er))
    fast = f32(m * y_a)
    ok = np.isfinite(exact) & (np.abs(exact) >= 2.0 ** -126)    # normal quotients
    rel = np.abs(fast[ok] - exact[ok]) / np.abs(exact[ok])
    assert rel.max() <= 2.0 ** -19
