"""The C-ABI library: it builds, loads, exports every entry point that
include/q8adamw.h declares, and rejects bad arguments on the host before any
launch.  No GPU is needed: nothing here computes on a device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import bit_blockwise_adamw_gb300 as q8
from bit_blockwise_adamw_gb300 import _binding as B
import oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\([^;{]*\)\s*;", text, flags=re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    from bit_blockwise_adamw_gb300 import build
    build.build()
    return q8.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names == set(B.EXPORTS), names ^ set(B.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version(lib):
    assert q8.q8_abi_version() == 5


@pytest.mark.parametrize("kind", [q8.SIGNED, q8.UNSIGNED])
def test_host_codebook_bit_exact_with_oracle(lib, kind):
    assert np.array_equal(q8.q8_codebook_init(kind).view(np.uint32), o.codebook(kind).view(np.uint32))


def _t8(**kw):
    base = dict(param=0x1000, grad=0x2000, numel=8192, philox_offset=-1, m_codes=0x3000,
                v_codes=0x4000, m_absmax=0x5000, v_absmax=0x6000, m32=None, v32=None)
    base.update(kw)
    return B._Tensor8(**base)


def _call8(lib, tensors, hp=None, n=None):
    arr = (B._Tensor8 * len(tensors))(*tensors)
    hp = hp if hp is not None else q8.hparams()
    return lib.adamw8bit_sr_step(arr, len(tensors) if n is None else n, C.byref(hp), None)


@pytest.mark.parametrize("field,value,code", [
    ("param", None, -1), ("grad", None, -1), ("m_codes", None, -1), ("v_absmax", None, -1),
    ("param", 0x1002, -3), ("grad", 0x2008, -3), ("m_codes", 0x3004, -3), ("m_absmax", 0x5002, -3),
    ("numel", -1, -2), ("numel", 1 << 40, -2), ("philox_offset", (1 << 62), -2),
])
def test_step8_rejects_bad_tensor(lib, field, value, code):
    assert _call8(lib, [_t8(), _t8(**{field: value})]) == code
    assert "tensor 1" in q8.q8_last_error()


def test_state_picks_the_path(lib):
    no8 = dict(m_codes=None, v_codes=None, m_absmax=None, v_absmax=None)
    assert _call8(lib, [_t8(numel=100, **no8)]) == -1                       # no state at all
    assert _call8(lib, [_t8(numel=100, m32=0x7000, v32=0x7004, **no8)]) == -3
    assert _call8(lib, [_t8(numel=5000, m32=0x7000, v32=0x7010, **no8)]) == -2   # fp32 state is for < 4096
    assert _call8(lib, [_t8(numel=100, m32=0x7000, v32=0x7010)]) == -4      # both kinds of state


@pytest.mark.parametrize("field,value", [
    ("step", 0), ("step", 1 << 31), ("beta1", 1.0), ("beta2", -0.1), ("lr", float("nan")),
    ("eps", -1.0), ("weight_decay", float("inf")), ("sr", 2), ("exact", 2), ("exact", -1)])
def test_step8_rejects_bad_hparams(lib, field, value):
    hp = q8.hparams()
    setattr(hp, field, value)
    assert _call8(lib, [_t8()], hp) == -4


def test_step8_null_arguments(lib):
    assert lib.adamw8bit_sr_step(None, 1, C.byref(q8.hparams()), None) == -1
    assert lib.adamw8bit_sr_step(None, 1, None, None) == -1
    assert lib.adamw8bit_sr_step(None, -1, C.byref(q8.hparams()), None) == -2
    assert lib.adamw8bit_sr_step(None, 0, C.byref(q8.hparams()), None) == 0


def test_bf16_step_validation(lib):
    t = B._Tensor16(0x1000, 0x2000, 0x3000, 0x4000, 100, -1)
    bad = B._Tensor16(0x1000, 0x2000, 0x3008, 0x4000, 100, -1)
    arr = (B._Tensor16 * 2)(t, bad)
    assert lib.adamw_bf16_sr_step(arr, 2, C.byref(q8.hparams()), None) == -3
    arr = (B._Tensor16 * 1)(B._Tensor16(0x1000, None, 0x3000, 0x4000, 100, -1))
    assert lib.adamw_bf16_sr_step(arr, 1, C.byref(q8.hparams()), None) == -1


def test_codec_validation(lib):
    assert lib.q8_blockwise_quantize(0x1000, 0x2000, 0x3000, 10, 2, None) == -4
    assert lib.q8_blockwise_quantize(0x1004, 0x2000, 0x3000, 10, 0, None) == -3
    assert lib.q8_blockwise_dequantize(0x1000, None, 0x3000, 10, 0, None) == -1
    assert lib.q8_blockwise_quantize(None, None, None, 0, 0, None) == 0
    assert lib.q8_blockwise_quantize(0x1000, 0x2000, 0x3000, -5, 0, None) == -2
    assert lib.q8_philox_fill(0, 1, 0, 0, 10, 0x1001, None) == -3
    assert lib.q8_selftest_sqrt_div(None, None) == -1
    assert lib.q8_selftest_sqrt_div(0x1004, None) == -3
    assert lib.q8_codebook_init(0, None) == -1
    assert lib.q8_codebook_init(7, (C.c_float * 256)()) == -4


def test_onestate_validation(lib):
    def t1(**kw):
        return _t8(v_codes=None, v_absmax=None, **kw)
    good = B.MomentumHParams(1e-2, 0.9, 0.0, 1, 0, 1)
    arr = (B._Tensor8 * 1)(_t8())                      # carries a second moment
    assert lib.momentum8bit_sr_step(arr, 1, C.byref(good), None) == -4
    arr = (B._Tensor8 * 1)(t1(m_absmax=None))
    assert lib.momentum8bit_sr_step(arr, 1, C.byref(good), None) == -1
    arr = (B._Tensor8 * 1)(t1(m_codes=0x3008))
    assert lib.momentum8bit_sr_step(arr, 1, C.byref(good), None) == -3
    for bad in (B.MomentumHParams(1e-2, 1.0, 0.0, 1, 0, 1), B.MomentumHParams(-1.0, 0.9, 0.0, 1, 0, 1),
                B.MomentumHParams(1e-2, 0.9, 0.0, 0, 0, 1)):
        assert lib.momentum8bit_sr_step(arr, 1, C.byref(bad), None) == -4
    lion_bad = B.LionHParams(1e-4, 0.9, 1.5, 0.0, 1, 0, 1)
    assert lib.lion8bit_sr_step((B._Tensor8 * 1)(t1()), 1, C.byref(lion_bad), None) == -4
    assert lib.lion8bit_sr_step(None, 0, C.byref(B.LionHParams(1e-4, 0.9, 0.99, 0.0, 1, 0, 1)), None) == 0
