"""Pins for the oracle's codebooks, thresholds and blockwise (de)quantization.

The pages ("8-bit Optimizers via Block-wise Quantization", innovations list and
method bullets) fix: a dynamic-tree code, a signed and a unipolar variant,
2048-element blocks normalised by their absmax, a binary search to an 8-bit
index and a lookup-times-absmax dequantization.  Each test below checks the
oracle against a different computation of the same fact.
"""
from fractions import Fraction as Fr

import numpy as np
import pytest

import oracle as o

S, U = o.SIGNED, o.UNSIGNED


def decode_dynamic_tree(byte, signed):
    """Value of one dynamic-tree bit pattern, decoded bit by bit (exact rational).

    Signed: bit 7 is the sign and bits 6..0 the tree; unsigned: all 8 bits are
    the tree.  In the tree, the leading zero bits count the decade e, the first
    one bit is the indicator and the f bits below it are the linear fraction k.
    """
    width = 7 if signed else 8
    negative = signed and (byte >> 7) & 1
    body = byte & ((1 << width) - 1)
    if body == 0:
        return Fr(0)
    e = width - body.bit_length()           # leading zeros inside the tree
    f = body.bit_length() - 1               # bits below the indicator
    k = body & ((1 << f) - 1)
    frac = Fr(1, 10) + Fr(9, 10) * Fr(k + 1, 2 ** f)
    value = frac / Fr(10) ** e
    return -value if negative else value


def to_f32(q):
    # the reading rounds the exact value to double, then once to float
    return np.float32(float(q))


@pytest.mark.parametrize("signed", [True, False])
def test_codebook_equals_sorted_bit_decode(signed):
    kind = S if signed else U
    table = o.codebook(kind)
    values = sorted({decode_dynamic_tree(b, signed) for b in range(256)})
    decoded = np.array([to_f32(v) for v in values], np.float32)
    if signed:
        assert len(values) == 255           # +0 and -0 collapse
        assert np.array_equal(table[:255], decoded)
        assert table[255] == np.float32(1.0)  # pad, a duplicate of the top code
    else:
        assert len(values) == 256
        assert np.array_equal(table, decoded)


def test_codebook_structure():
    cs, cu = o.codebook(S), o.codebook(U)
    assert cs[0] == -1 and cs[127] == 0 and cs[254] == 1 and cs[255] == 1
    assert cu[0] == 0 and cu[255] == 1
    assert cu[1] == np.float32(1e-7) and cs[128] == np.float32(1e-6)
    assert cs[129] == np.float32(5.5e-6)      # decade 1e-5 with one fraction bit: 0.55e-5
    assert np.all(np.diff(cs[:255]) > 0) and np.all(np.diff(cu) > 0)
    # odd symmetry of the signed book
    assert np.array_equal(cs[:127][::-1], -cs[128:255])
    # 0.1 + 0.9/64, the first fraction step of the top signed decade
    assert cs[128 + 127 - 64] == np.float32(0.1140625)


@pytest.mark.parametrize("kind,width", [(S, 7), (U, 8)])
def test_codes_per_decade_and_even_spacing(kind, width):
    table = o.codebook(kind).astype(np.float64)
    pos = table[table > 0]
    if kind == S:
        pos = pos[:-1]                       # drop the pad
    for e in range(width):
        f = width - 1 - e
        hi, lo = 10.0 ** -e, 10.0 ** -(e + 1)
        dec = pos[(pos > lo * (1 + 1e-6)) & (pos <= hi * (1 + 1e-6))]
        assert dec.size == 2 ** f, (e, dec.size)
        gap = 0.9 * hi / 2 ** f
        assert np.allclose(np.diff(dec), gap, rtol=1e-5, atol=0)
        assert abs(dec[-1] - hi) <= 1e-7 * hi


@pytest.mark.parametrize("kind", [S, U])
def test_midpoints_are_nearest_float_to_exact_midpoint(kind):
    c = o.codebook(kind)
    mid = o.midpoints(kind)
    for j in range(255):
        mu = (Fr(float(c[j])) + Fr(float(c[j + 1]))) / 2
        m = mid[j]
        err = abs(Fr(float(m)) - mu)
        for nb in (np.nextafter(m, np.float32(-2)), np.nextafter(m, np.float32(2))):
            assert err <= abs(Fr(float(nb)) - mu), j
        if c[j] != c[j + 1]:
            assert c[j] < m <= c[j + 1] or c[j] <= m < c[j + 1]


def _dense_inputs(kind):
    """Every 97th float of [0, 1] and its negative, all floats within 64 ulps of
    every threshold, and the special values."""
    bits = np.arange(0, 0x3F800001, 97, dtype=np.uint32)
    x = bits.view(np.float32)
    mid = o.midpoints(kind)
    mag = np.abs(mid).view(np.uint32).astype(np.int64)
    offs = np.arange(-64, 65, dtype=np.int64)
    near_bits = np.clip(mag[:, None] + offs[None, :], 0, 0x3F800000).astype(np.uint32)
    near = near_bits.view(np.float32) * np.sign(mid)[:, None].astype(np.float32)
    special = np.array([0.0, -0.0, 1.0, -1.0, 1e-45, -1e-45], np.float32)
    return np.concatenate([x, -x, near.ravel(), special]).astype(np.float32)


@pytest.mark.parametrize("kind", [S, U])
def test_search_equals_library_searchsorted(kind):
    x = _dense_inputs(kind)
    mid = o.midpoints(kind)
    got = o.search_many(kind, x).astype(np.int64)
    want = np.searchsorted(mid, x, side="left")      # count of thresholds < x
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], want[bad[:5]])


def _nearest_linear(table, x):
    """Brute force: index of the nearest code by exact distance, first on ties."""
    out = np.empty(x.size, np.int64)
    t = table.astype(np.float64)
    for s in range(0, x.size, 8192):
        d = np.abs(x[s:s + 8192].astype(np.float64)[:, None] - t[None, :])
        out[s:s + 8192] = np.argmin(d, axis=1)
    return out


@pytest.mark.parametrize("kind", [S, U])
def test_search_against_brute_force_nearest(kind):
    rng = np.random.default_rng(7)
    lo = -1.0 if kind == S else 0.0
    mid = o.midpoints(kind)
    table = o.codebook(kind)
    x = np.concatenate([
        rng.uniform(lo, 1.0, 200_000).astype(np.float32),
        (np.sign(rng.uniform(lo, 1.0, 100_000)) * 10.0 ** rng.uniform(-8, 0, 100_000)).astype(np.float32),
        _dense_inputs(kind)[-(255 * 129 + 6):],       # the near-threshold set
    ])
    if kind == U:
        x = x[x >= 0]
    got = o.search_many(kind, x).astype(np.int64)
    want = _nearest_linear(table, x)
    bad = np.nonzero(got != want)[0]
    # The count rule and exact-nearest differ only where x is a threshold that
    # rounding moved above the exact midpoint: there the count rule keeps the
    # lower code.
    for i in bad:
        j = got[i]
        assert want[i] == j + 1 and x[i] == mid[j], (x[i], got[i], want[i])
        mu = (Fr(float(table[j])) + Fr(float(table[j + 1]))) / 2
        assert Fr(float(mid[j])) > mu
    assert bad.size <= 255


def test_search_extremes():
    assert o.search(S, 1.0) == 254 and o.search(S, -1.0) == 0
    assert o.search(S, 0.0) == 127 and o.search(S, -0.0) == 127
    assert o.search(U, 0.0) == 0 and o.search(U, 1.0) == 255
    assert o.zero_code(S) == 127 and o.zero_code(U) == 0


def _blocks(rng, n):
    base = rng.standard_normal(n).astype(np.float32) * 1e-3
    outl = rng.random(n) < 0.001
    base[outl] *= 100
    logn = (rng.standard_normal(n) * 2).astype(np.float32)
    return [base, np.exp(logn).astype(np.float32) * 1e-6, np.abs(base), (base ** 2).astype(np.float32)]


@pytest.mark.parametrize("kind", [S, U])
def test_round_trip_bound(kind):
    rng = np.random.default_rng(11)
    table = o.codebook(kind)
    gaps = np.diff(table.astype(np.float64))
    maxgap = gaps.max()
    for x in _blocks(rng, 3 * 2048 + 333):
        if kind == U:
            x = np.abs(x)
        codes, absmax = o.quantize(kind, x)
        y = o.dequantize(kind, codes, absmax)
        M = np.repeat(absmax, 2048)[: x.size].astype(np.float64)
        err = np.abs(y.astype(np.float64) - x.astype(np.float64))
        assert np.all(err <= M * (maxgap / 2 + 2.0 ** -22))
        # per-block absmax is the library max of |x| over each block
        for b in range(absmax.size):
            assert absmax[b] == np.abs(x[b * 2048:(b + 1) * 2048]).max()
        # the absmax element maps to +-1 exactly
        for b in range(absmax.size):
            blk = x[b * 2048:(b + 1) * 2048]
            i = int(np.argmax(np.abs(blk)))
            assert y[b * 2048 + i] == blk[i]


@pytest.mark.parametrize("kind", [S, U])
def test_codes_times_power_of_two_round_trip_exactly(kind):
    table = o.codebook(kind)
    n = 2048
    codes = np.arange(n) % 255
    for M in (1.0, 0.25, 2.0 ** -20, 2.0 ** 10):
        x = (table[codes] * np.float32(M)).astype(np.float32)
        x[0] = np.float32(M)                 # make the block absmax exactly M
        q, a = o.quantize(kind, x)
        assert a[0] == np.float32(M)
        assert np.array_equal(o.dequantize(kind, q, a), x)


@pytest.mark.parametrize("kind", [S, U])
def test_degenerate_blocks(kind):
    z = np.zeros(2048 + 5, np.float32)
    q, a = o.quantize(kind, z)
    assert np.all(q == o.zero_code(kind)) and np.all(a == 0)
    assert np.all(o.dequantize(kind, q, a) == 0)
    one = np.full(7, 0.5, np.float32)
    q, a = o.quantize(kind, one)
    assert a[0] == np.float32(0.5) and np.all(o.dequantize(kind, q, a) == one)
    q, a = o.quantize(kind, np.array([3.0], np.float32))
    assert q[0] == 255 - (1 if kind == S else 0) and a[0] == 3.0
