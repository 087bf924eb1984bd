"""GPU parity of the codebooks, blockwise quantize / dequantize and the Philox
stream against the oracle, bit for bit, through the C ABI."""
import numpy as np
import pytest
import torch

import bit_blockwise_adamw_gb300 as q8
import oracle as o

pytestmark = pytest.mark.gpu

KINDS = [q8.SIGNED, q8.UNSIGNED]


@pytest.mark.parametrize("kind", KINDS)
def test_device_codebook_bit_exact(cuda_device, kind):
    """Dequantizing every code with absmax 1 reads the device table."""
    codes = torch.arange(256, dtype=torch.uint8, device=cuda_device).repeat(8)
    absmax = torch.ones(1, dtype=torch.float32, device=cuda_device)
    x = torch.empty(codes.numel(), dtype=torch.float32, device=cuda_device)
    q8.q8_blockwise_dequantize(codes, absmax, x, kind)
    got = x.cpu().numpy()[:256]
    assert np.array_equal(got.view(np.uint32), o.codebook(kind).view(np.uint32))


def _sweep(kind, stride):
    """Every `stride`-th float of [0, 1] (and the negatives for the signed
    book) plus every float within 64 ulps of a threshold, packed into
    2048-blocks whose first element is 1.0, so each block's absmax is 1 and
    the normalised value is the float itself."""
    bits = np.arange(0, 0x3F800001, stride, dtype=np.uint32)
    vals = [bits.view(np.float32)]
    if kind == q8.SIGNED:
        vals.append(-bits.view(np.float32))
    mid = o.midpoints(kind)
    mag = np.abs(mid).view(np.uint32).astype(np.int64)
    near = np.clip(mag[:, None] + np.arange(-64, 65)[None, :], 0, 0x3F800000).astype(np.uint32)
    vals.append((near.view(np.float32) * np.sign(mid)[:, None].astype(np.float32)).ravel())
    v = np.concatenate(vals).astype(np.float32)
    per = 2047
    nb = (v.size + per - 1) // per
    body = np.zeros(nb * per, np.float32)
    body[:v.size] = v
    x = np.empty((nb, 2048), np.float32)
    x[:, 0] = 1.0
    x[:, 1:] = body.reshape(nb, per)
    assert np.array_equal(x[:, 1:].reshape(-1)[:v.size], v)
    return x.reshape(-1)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("lead", [1.0, 0.75])
def test_quantize_dense_sweep(cuda_device, kind, lead):
    """Every 13th float of [0, 1] (both signs for the signed book) and every
    float near a threshold, quantized in blocks whose first element is `lead`
    (with 1.0 every block's absmax is 1 and the normalised value is the float
    itself; with 0.75 most blocks normalise by another absmax)."""
    x = _sweep(kind, 13)
    x[::2048] = lead
    xd = torch.from_numpy(x).to(cuda_device)
    codes = torch.empty(x.size, dtype=torch.uint8, device=cuda_device)
    absmax = torch.empty(x.size // 2048, dtype=torch.float32, device=cuda_device)
    q8.q8_blockwise_quantize(xd, codes, absmax, kind)
    want_c, want_a = o.quantize(kind, x)
    got_c = codes.cpu().numpy()
    bad = np.nonzero(got_c != want_c)[0]
    assert bad.size == 0, (x[bad[:5]], got_c[bad[:5]], want_c[bad[:5]])
    assert np.array_equal(absmax.cpu().numpy(), want_a)


def _inputs(rng, n, kind, dist):
    if dist == "normal":
        x = rng.standard_normal(n) * 1e-3
    elif dist == "outliers":
        x = rng.standard_normal(n) * 1e-4
        x[rng.random(n) < 1e-3] *= 1000
    elif dist == "lognormal":
        x = np.exp(rng.standard_normal(n) * 3) * 1e-6 * np.sign(rng.standard_normal(n))
    elif dist == "zeros":
        x = np.zeros(n)
    else:   # constant
        x = np.full(n, -0.375)
    if kind == q8.UNSIGNED:
        x = np.abs(x)
    return x.astype(np.float32)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [1, 7, 8, 2047, 2048, 2049, 4096 + 3, 10 * 2048 + 5, 1 << 20])
@pytest.mark.parametrize("dist", ["normal", "outliers", "lognormal", "zeros", "const"])
def test_quantize_dequantize_parity(cuda_device, kind, n, dist):
    rng = np.random.default_rng(n * 31 + kind)
    x = _inputs(rng, n, kind, dist)
    xd = torch.from_numpy(x).to(cuda_device)
    nb = (n + 2047) // 2048
    codes = torch.empty(n, dtype=torch.uint8, device=cuda_device)
    absmax = torch.empty(nb, dtype=torch.float32, device=cuda_device)
    q8.q8_blockwise_quantize(xd, codes, absmax, kind)
    want_c, want_a = o.quantize(kind, x)
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(absmax.cpu().numpy().view(np.uint32), want_a.view(np.uint32))
    y = torch.empty(n, dtype=torch.float32, device=cuda_device)
    q8.q8_blockwise_dequantize(codes, absmax, y, kind)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), o.dequantize(kind, want_c, want_a).view(np.uint32))


def test_unsigned_negative_inputs(cuda_device):
    x = np.array([-1.0, -0.0, 0.5, -3e-9, 2.0] + [0.0] * 3, np.float32)
    xd = torch.from_numpy(x).to(cuda_device)
    codes = torch.empty(8, dtype=torch.uint8, device=cuda_device)
    absmax = torch.empty(1, dtype=torch.float32, device=cuda_device)
    q8.q8_blockwise_quantize(xd, codes, absmax, q8.UNSIGNED)
    want_c, want_a = o.quantize(o.UNSIGNED, x)
    assert np.array_equal(codes.cpu().numpy(), want_c) and absmax.item() == want_a[0]


@pytest.mark.parametrize("seed", [0, 1, 0xDEADBEEFCAFEF00D])
@pytest.mark.parametrize("step,sid", [(1, 0), (7, 1), (123456, 2), (0x7FFFFFFF, 0)])
@pytest.mark.parametrize("offset,n", [(0, 1), (0, 4096), (3, 1000), (8, 17), (5, 100_000),
                                      ((1 << 35) + 3, 5000), ((1 << 40) + 7, 33)])
def test_philox_fill_bit_exact(cuda_device, seed, step, sid, offset, n):
    out = torch.empty(n, dtype=torch.int16, device=cuda_device)
    q8.q8_philox_fill(seed, step, sid, offset, out)
    got = out.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, o.philox_fill(seed, step, sid, offset, n))


def test_empty_calls(cuda_device):
    e = torch.empty(0, dtype=torch.float32, device=cuda_device)
    c = torch.empty(0, dtype=torch.uint8, device=cuda_device)
    a = torch.empty(0, dtype=torch.float32, device=cuda_device)
    q8.q8_blockwise_quantize(e, c, a, q8.SIGNED)
    q8.q8_blockwise_dequantize(c, a, e, q8.SIGNED)
    q8.q8_philox_fill(0, 1, 0, 0, torch.empty(0, dtype=torch.int16, device=cuda_device))
    torch.cuda.synchronize()
