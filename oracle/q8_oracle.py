"""ctypes/numpy wrapper around the C oracle (test infrastructure only).

Arrays are numpy: bf16 values travel as their uint16 bit patterns.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

SIGNED, UNSIGNED = 0, 1
BLOCK = 2048
SMALL = 4096

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.q8o_codebook.argtypes = [C.c_int, P]
        L.q8o_midpoints.argtypes = [C.c_int, P]
        L.q8o_zero_code.argtypes = [C.c_int]
        L.q8o_zero_code.restype = C.c_int
        L.q8o_search.argtypes = [C.c_int, C.c_float]
        L.q8o_search.restype = C.c_int
        L.q8o_search_many.argtypes = [C.c_int, P, C.c_int64, P]
        L.q8o_quantize.argtypes = [C.c_int, P, C.c_int64, P, P]
        L.q8o_dequantize.argtypes = [C.c_int, P, P, C.c_int64, P]
        L.q8o_philox4x32_10.argtypes = [P, P, P]
        L.q8o_r16.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint64]
        L.q8o_r16.restype = C.c_uint16
        L.q8o_philox_fill.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint64, C.c_int64, P]
        L.q8o_sr_bf16.argtypes = [C.c_float, C.c_uint16]
        L.q8o_sr_bf16.restype = C.c_uint16
        L.q8o_rne_bf16.argtypes = [C.c_float]
        L.q8o_rne_bf16.restype = C.c_uint16
        L.q8o_bf16_to_f32.argtypes = [C.c_uint16]
        L.q8o_bf16_to_f32.restype = C.c_float
        L.q8o_step_scalars.argtypes = [C.POINTER(HParams), C.POINTER(Scalars)]
        L.q8o_adamw_element.argtypes = [C.POINTER(Scalars), C.c_float, C.c_float,
                                        C.POINTER(C.c_float), C.POINTER(C.c_float)]
        L.q8o_adamw_element.restype = C.c_float
        L.q8o_adamw8bit_tensor.argtypes = [C.POINTER(Tensor8), C.c_uint64, C.POINTER(HParams)]
        L.q8o_adamw32_tensor.argtypes = [C.POINTER(Tensor8), C.c_uint64, C.POINTER(HParams)]
        L.q8o_adamw_bf16_tensor.argtypes = [C.POINTER(Tensor16), C.c_uint64, C.POINTER(HParams)]
        L.q8o_adamw8bit_sr_step.argtypes = [C.POINTER(Tensor8), C.c_int, C.POINTER(HParams)]
        L.q8o_adamw_bf16_sr_step.argtypes = [C.POINTER(Tensor16), C.c_int, C.POINTER(HParams)]
        L.q8o_step_scalars1.argtypes = [C.c_int, C.POINTER(HParams), C.POINTER(Scalars1)]
        L.q8o_onestate_element.argtypes = [C.c_int, C.POINTER(Scalars1), C.c_float, C.c_float,
                                           C.POINTER(C.c_float)]
        L.q8o_onestate_element.restype = C.c_float
        L.q8o_onestate8bit_tensor.argtypes = [C.c_int, C.POINTER(Tensor8), C.c_uint64, C.POINTER(HParams)]
        L.q8o_onestate32_tensor.argtypes = [C.c_int, C.POINTER(Tensor8), C.c_uint64, C.POINTER(HParams)]
        L.q8o_onestate_sr_step.argtypes = [C.c_int, C.POINTER(Tensor8), C.c_int, C.POINTER(HParams)]
        _lib = L
    return _lib


class HParams(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double),
                ("step", C.c_int64), ("seed", C.c_uint64), ("sr", C.c_int32)]


class Scalars(C.Structure):
    _fields_ = [(n, C.c_float) for n in
                ("b1", "omb1", "b2", "omb2", "eps_t", "step_size", "decay")]


class Scalars1(C.Structure):
    _fields_ = [(n, C.c_float) for n in ("lr_neg", "a", "oma", "b", "omb", "decay", "wd")]


MOMENTUM, LION = 0, 1


class Tensor8(C.Structure):
    _fields_ = [("param", C.c_void_p), ("grad", C.c_void_p), ("numel", C.c_int64),
                ("philox_offset", C.c_int64), ("m_codes", C.c_void_p), ("v_codes", C.c_void_p),
                ("m_absmax", C.c_void_p), ("v_absmax", C.c_void_p),
                ("m32", C.c_void_p), ("v32", C.c_void_p)]


class Tensor16(C.Structure):
    _fields_ = [("param", C.c_void_p), ("grad", C.c_void_p), ("m", C.c_void_p),
                ("v", C.c_void_p), ("numel", C.c_int64), ("philox_offset", C.c_int64)]


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
            step=1, seed=0, sr=1):
    return HParams(lr, beta1, beta2, eps, weight_decay, step, seed, sr)


def codebook(kind):
    out = np.zeros(256, np.float32)
    lib().q8o_codebook(kind, _ptr(out))
    return out


def midpoints(kind):
    out = np.zeros(255, np.float32)
    lib().q8o_midpoints(kind, _ptr(out))
    return out


def zero_code(kind):
    return lib().q8o_zero_code(kind)


def search(kind, x):
    return lib().q8o_search(kind, float(np.float32(x)))


def search_many(kind, x):
    x = np.ascontiguousarray(x, np.float32)
    out = np.zeros(x.size, np.uint8)
    lib().q8o_search_many(kind, _ptr(x), x.size, _ptr(out))
    return out


def quantize(kind, x):
    x = np.ascontiguousarray(x, np.float32)
    n = x.size
    codes = np.zeros(n, np.uint8)
    absmax = np.zeros((n + BLOCK - 1) // BLOCK, np.float32)
    lib().q8o_quantize(kind, _ptr(x), n, _ptr(codes), _ptr(absmax))
    return codes, absmax


def dequantize(kind, codes, absmax):
    codes = np.ascontiguousarray(codes, np.uint8)
    absmax = np.ascontiguousarray(absmax, np.float32)
    out = np.zeros(codes.size, np.float32)
    lib().q8o_dequantize(kind, _ptr(codes), _ptr(absmax), codes.size, _ptr(out))
    return out


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, np.uint32).copy()
    k = np.asarray(key, np.uint32).copy()
    out = np.zeros(4, np.uint32)
    lib().q8o_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def r16(seed, step, stream, E):
    return lib().q8o_r16(seed, step, stream, E)


def philox_fill(seed, step, stream, offset, n):
    out = np.zeros(n, np.uint16)
    lib().q8o_philox_fill(seed, step, stream, offset, n, _ptr(out))
    return out


def sr_bf16(x, r):
    return lib().q8o_sr_bf16(float(np.float32(x)), int(r))


def rne_bf16(x):
    return lib().q8o_rne_bf16(float(np.float32(x)))


def bf16_to_f32(h):
    return np.float32(lib().q8o_bf16_to_f32(int(h)))


def step_scalars(hp):
    s = Scalars()
    lib().q8o_step_scalars(C.byref(hp), C.byref(s))
    return s


def adamw_element(s, g, p, m, v):
    """One fp32 AdamW element update; returns (p_new, m_new, v_new) as float32."""
    mm = C.c_float(float(np.float32(m)))
    vv = C.c_float(float(np.float32(v)))
    pn = lib().q8o_adamw_element(C.byref(s), float(np.float32(g)), float(np.float32(p)),
                                 C.byref(mm), C.byref(vv))
    return np.float32(pn), np.float32(mm.value), np.float32(vv.value)


class State8:
    """Host copy of one tensor's optimizer state for the 8-bit (or fp32) path."""

    def __init__(self, param, grad, m_codes=None, v_codes=None, m_absmax=None,
                 v_absmax=None, m32=None, v32=None, philox_offset=-1):
        self.param = np.ascontiguousarray(param, np.uint16)
        self.grad = np.ascontiguousarray(grad, np.uint16)
        self.m_codes = None if m_codes is None else np.ascontiguousarray(m_codes, np.uint8)
        self.v_codes = None if v_codes is None else np.ascontiguousarray(v_codes, np.uint8)
        self.m_absmax = None if m_absmax is None else np.ascontiguousarray(m_absmax, np.float32)
        self.v_absmax = None if v_absmax is None else np.ascontiguousarray(v_absmax, np.float32)
        self.m32 = None if m32 is None else np.ascontiguousarray(m32, np.float32)
        self.v32 = None if v32 is None else np.ascontiguousarray(v32, np.float32)
        self.philox_offset = philox_offset

    @classmethod
    def zeros(cls, param, grad, philox_offset=-1, eight_bit=None):
        """Fresh state; the 8-bit layout when eight_bit (default: numel >= 4096)."""
        n = param.size
        if eight_bit is None:
            eight_bit = n >= SMALL
        if eight_bit:
            nb = (n + BLOCK - 1) // BLOCK
            return cls(param, grad, np.full(n, zero_code(SIGNED), np.uint8),
                       np.full(n, zero_code(UNSIGNED), np.uint8),
                       np.zeros(nb, np.float32), np.zeros(nb, np.float32),
                       philox_offset=philox_offset)
        return cls(param, grad, m32=np.zeros(n, np.float32), v32=np.zeros(n, np.float32),
                   philox_offset=philox_offset)

    def struct(self):
        return Tensor8(_ptr(self.param), _ptr(self.grad), self.param.size, self.philox_offset,
                       _ptr(self.m_codes), _ptr(self.v_codes), _ptr(self.m_absmax),
                       _ptr(self.v_absmax), _ptr(self.m32), _ptr(self.v32))


class State16:
    """Host copy of one tensor's state for the BF16-state path."""

    def __init__(self, param, grad, m, v, philox_offset=-1):
        self.param = np.ascontiguousarray(param, np.uint16)
        self.grad = np.ascontiguousarray(grad, np.uint16)
        self.m = np.ascontiguousarray(m, np.uint16)
        self.v = np.ascontiguousarray(v, np.uint16)
        self.philox_offset = philox_offset

    def struct(self):
        return Tensor16(_ptr(self.param), _ptr(self.grad), _ptr(self.m), _ptr(self.v),
                        self.param.size, self.philox_offset)


def adamw8bit_sr_step(states, hp):
    """Whole-list 8-bit step (routing by size, running Philox offsets)."""
    arr = (Tensor8 * len(states))(*[s.struct() for s in states])
    lib().q8o_adamw8bit_sr_step(arr, len(states), C.byref(hp))


def adamw8bit_tensor(state, E0, hp):
    """8-bit path on one tensor (or a block-aligned slice) with explicit offset."""
    if state.m_codes is None or state.v_codes is None or state.m_absmax is None or state.v_absmax is None:
        raise ValueError("adamw8bit_tensor needs the 8-bit state arrays")
    if state.m_absmax.size < (state.param.size + BLOCK - 1) // BLOCK:
        raise ValueError("absmax arrays are too short")
    t = state.struct()
    lib().q8o_adamw8bit_tensor(C.byref(t), E0, C.byref(hp))


def adamw32_tensor(state, E0, hp):
    if state.m32 is None or state.v32 is None:
        raise ValueError("adamw32_tensor needs m32 and v32")
    t = state.struct()
    lib().q8o_adamw32_tensor(C.byref(t), E0, C.byref(hp))


def adamw_bf16_sr_step(states, hp):
    arr = (Tensor16 * len(states))(*[s.struct() for s in states])
    lib().q8o_adamw_bf16_sr_step(arr, len(states), C.byref(hp))


def adamw_bf16_tensor(state, E0, hp):
    t = state.struct()
    lib().q8o_adamw_bf16_tensor(C.byref(t), E0, C.byref(hp))


def lib_path():
    return os.path.abspath(_build.LIB)


def step_scalars1(opt, hp):
    s = Scalars1()
    lib().q8o_step_scalars1(opt, C.byref(hp), C.byref(s))
    return s


def onestate_element(opt, s, g, p, m):
    """One element of Momentum / Lion; returns (p_new, m_new) as float32."""
    mm = C.c_float(float(np.float32(m)))
    pn = lib().q8o_onestate_element(opt, C.byref(s), float(np.float32(g)), float(np.float32(p)), C.byref(mm))
    return np.float32(pn), np.float32(mm.value)


def onestate_sr_step(opt, states, hp):
    """Momentum / Lion step over a list of State8 (m only; v fields unused)."""
    arr = (Tensor8 * len(states))(*[s.struct() for s in states])
    lib().q8o_onestate_sr_step(opt, arr, len(states), C.byref(hp))


def onestate8bit_tensor(opt, state, E0, hp):
    if state.m_codes is None or state.m_absmax is None:
        raise ValueError("onestate8bit_tensor needs m_codes and m_absmax")
    t = state.struct()
    lib().q8o_onestate8bit_tensor(opt, C.byref(t), E0, C.byref(hp))


def onestate32_tensor(opt, state, E0, hp):
    if state.m32 is None:
        raise ValueError("onestate32_tensor needs m32")
    t = state.struct()
    lib().q8o_onestate32_tensor(opt, C.byref(t), E0, C.byref(hp))


def zeros_onestate(param, grad, philox_offset=-1, eight_bit=None):
    """Fresh one-state (m only) state."""
    n = param.size
    if eight_bit is None:
        eight_bit = n >= SMALL
    if eight_bit:
        nb = (n + BLOCK - 1) // BLOCK
        return State8(param, grad, m_codes=np.full(n, zero_code(SIGNED), np.uint8),
                      m_absmax=np.zeros(nb, np.float32), philox_offset=philox_offset)
    return State8(param, grad, m32=np.zeros(n, np.float32), philox_offset=philox_offset)
