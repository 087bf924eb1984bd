"""ctypes binding of libq8adamw.so: argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/q8adamw.h) and takes torch tensors that already live on a CUDA device;
all work runs in the library's kernels.  A missing library is an error: there
is no fallback path.
"""
import ctypes as C
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np
import torch

from . import build as _build

SIGNED, UNSIGNED = 0, 1
BLOCK = 2048
SMALL_NUMEL = 4096
MAX_STEP = 0x7FFFFFFF

Q8_OK = 0
_STATUS = {-1: "Q8_ERR_NULL", -2: "Q8_ERR_SIZE", -3: "Q8_ERR_ALIGN", -4: "Q8_ERR_ARG", -5: "Q8_ERR_CUDA"}

# every symbol the header declares
EXPORTS = ("q8_codebook_init", "q8_blockwise_quantize", "q8_blockwise_dequantize",
           "adamw8bit_sr_step", "adamw_bf16_sr_step", "momentum8bit_sr_step", "lion8bit_sr_step",
           "q8_philox_fill", "q8_selftest_sqrt_div", "q8_prepare_device", "q8_last_error", "q8_abi_version")


class Q8Error(RuntimeError):
    """A non-zero status from the library, with its message."""

    def __init__(self, fn, code, msg):
        super().__init__("%s failed: %s (%d): %s" % (fn, _STATUS.get(code, "?"), code, msg))
        self.code = code


class HParams(C.Structure):
    """q8_adamw_hparams."""
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double),
                ("step", C.c_int64), ("seed", C.c_uint64), ("sr", C.c_int32), ("exact", C.c_int32)]


class MomentumHParams(C.Structure):
    """q8_momentum_hparams."""
    _fields_ = [("lr", C.c_double), ("momentum", C.c_double), ("weight_decay", C.c_double),
                ("step", C.c_int64), ("seed", C.c_uint64), ("sr", C.c_int32)]


class LionHParams(C.Structure):
    """q8_lion_hparams."""
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("weight_decay", C.c_double), ("step", C.c_int64), ("seed", C.c_uint64), ("sr", C.c_int32)]


class _Tensor8(C.Structure):
    _fields_ = [("param", C.c_void_p), ("grad", C.c_void_p), ("numel", C.c_int64),
                ("philox_offset", C.c_int64), ("m_codes", C.c_void_p), ("v_codes", C.c_void_p),
                ("m_absmax", C.c_void_p), ("v_absmax", C.c_void_p),
                ("m32", C.c_void_p), ("v32", C.c_void_p)]


class _Tensor16(C.Structure):
    _fields_ = [("param", C.c_void_p), ("grad", C.c_void_p), ("m", C.c_void_p),
                ("v", C.c_void_p), ("numel", C.c_int64), ("philox_offset", C.c_int64)]


_lib = None


def library_path():
    return _build.LIB


def load_library(path: Optional[str] = None):
    """Load (once) and type the shared library; raise if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError("libq8adamw.so is not built (%s); run bit_blockwise_adamw_gb300.build.build()" % path)
    L = C.CDLL(path)
    P, S = C.c_void_p, C.c_void_p
    L.q8_codebook_init.argtypes = [C.c_int, P]
    L.q8_blockwise_quantize.argtypes = [P, P, P, C.c_int64, C.c_int, S]
    L.q8_blockwise_dequantize.argtypes = [P, P, P, C.c_int64, C.c_int, S]
    L.adamw8bit_sr_step.argtypes = [C.POINTER(_Tensor8), C.c_int, C.POINTER(HParams), S]
    L.adamw_bf16_sr_step.argtypes = [C.POINTER(_Tensor16), C.c_int, C.POINTER(HParams), S]
    L.momentum8bit_sr_step.argtypes = [C.POINTER(_Tensor8), C.c_int, C.POINTER(MomentumHParams), S]
    L.lion8bit_sr_step.argtypes = [C.POINTER(_Tensor8), C.c_int, C.POINTER(LionHParams), S]
    L.q8_philox_fill.argtypes = [C.c_uint64, C.c_uint32, C.c_uint32, C.c_uint64, C.c_int64, P, S]
    L.q8_selftest_sqrt_div.argtypes = [P, S]
    L.q8_prepare_device.argtypes = []
    L.q8_last_error.argtypes = []
    L.q8_last_error.restype = C.c_char_p
    L.q8_abi_version.argtypes = []
    for name in EXPORTS:
        if name not in ("q8_last_error",):
            getattr(L, name).restype = C.c_int
    _lib = L
    return L


def _check(fn, rc):
    if rc != Q8_OK:
        raise Q8Error(fn, rc, load_library().q8_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def hparams(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1, seed=0, sr=1, exact=0):
    """q8_adamw_hparams; exact=0 is the fast mode (approximate square root and
    reciprocal in the parameter update of full blocks), exact=1 the bit-exact one."""
    return HParams(lr, beta1, beta2, eps, weight_decay, step, seed, sr, int(exact))


def momentum_hparams(lr=1e-2, momentum=0.9, weight_decay=0.0, step=1, seed=0, sr=1):
    return MomentumHParams(lr, momentum, weight_decay, step, seed, sr)


def lion_hparams(lr=1e-4, beta1=0.9, beta2=0.99, weight_decay=0.0, step=1, seed=0, sr=1):
    return LionHParams(lr, beta1, beta2, weight_decay, step, seed, sr)


# ---------------------------------------------------------------- entry points

def q8_abi_version() -> int:
    return load_library().q8_abi_version()


def q8_last_error() -> str:
    return load_library().q8_last_error().decode()


def q8_prepare_device() -> None:
    _check("q8_prepare_device", load_library().q8_prepare_device())


def q8_codebook_init(kind: int) -> np.ndarray:
    out = np.zeros(256, np.float32)
    _check("q8_codebook_init", load_library().q8_codebook_init(kind, out.ctypes.data))
    return out


def q8_blockwise_quantize(x: torch.Tensor, codes: torch.Tensor, absmax: torch.Tensor, kind: int,
                          stream=None) -> None:
    assert x.dtype == torch.float32 and codes.dtype == torch.uint8 and absmax.dtype == torch.float32
    n = x.numel()
    assert codes.numel() >= n and absmax.numel() >= (n + BLOCK - 1) // BLOCK
    _check("q8_blockwise_quantize", load_library().q8_blockwise_quantize(
        _ptr(x), _ptr(codes), _ptr(absmax), n, kind, _stream(stream)))


def q8_blockwise_dequantize(codes: torch.Tensor, absmax: torch.Tensor, x: torch.Tensor, kind: int,
                            stream=None) -> None:
    assert x.dtype == torch.float32 and codes.dtype == torch.uint8 and absmax.dtype == torch.float32
    n = x.numel()
    assert codes.numel() >= n and absmax.numel() >= (n + BLOCK - 1) // BLOCK
    _check("q8_blockwise_dequantize", load_library().q8_blockwise_dequantize(
        _ptr(codes), _ptr(absmax), _ptr(x), n, kind, _stream(stream)))


def q8_philox_fill(seed: int, step: int, stream_id: int, offset: int, out: torch.Tensor,
                   stream=None) -> None:
    assert out.element_size() == 2, "out holds 16-bit draws (int16 or uint16)"
    _check("q8_philox_fill", load_library().q8_philox_fill(
        seed, step, stream_id, offset, out.numel(), _ptr(out), _stream(stream)))


def q8_selftest_sqrt_div(counts: torch.Tensor, stream=None) -> None:
    """Device self-test of the packed square root and division; counts:
    int64[8] on the GPU (reciprocal mismatches, d values checked, quotient
    mismatches, pairs checked, square-root mismatches, v values checked, and
    the largest relative errors of the fast mode's approximate square root and
    reciprocal as float bit patterns)."""
    assert counts.dtype == torch.int64 and counts.numel() >= 8 and counts.is_contiguous()
    _check("q8_selftest_sqrt_div", load_library().q8_selftest_sqrt_div(_ptr(counts), _stream(stream)))


@dataclass
class Tensor8:
    """One tensor of the 8-bit step: bf16 param/grad plus its optimizer state
    (uint8 codes + float32 block absmax when numel >= 4096, else float32
    m32/v32).  philox_offset < 0 means the running element count."""
    param: torch.Tensor
    grad: torch.Tensor
    m_codes: Optional[torch.Tensor] = None
    v_codes: Optional[torch.Tensor] = None
    m_absmax: Optional[torch.Tensor] = None
    v_absmax: Optional[torch.Tensor] = None
    m32: Optional[torch.Tensor] = None
    v32: Optional[torch.Tensor] = None
    philox_offset: int = -1

    @classmethod
    def zeros_like(cls, param: torch.Tensor, grad: Optional[torch.Tensor] = None, philox_offset=-1,
                   moments: int = 2):
        """Fresh (all-zero) state for `param` on its device: first and second
        moment (AdamW) or, with moments=1, the first only (Momentum, Lion)."""
        n = param.numel()
        dev = param.device
        two = moments == 2
        if n >= SMALL_NUMEL:
            nb = (n + BLOCK - 1) // BLOCK
            return cls(param, grad, torch.full((n,), 127, dtype=torch.uint8, device=dev),
                       torch.zeros(n, dtype=torch.uint8, device=dev) if two else None,
                       torch.zeros(nb, dtype=torch.float32, device=dev),
                       torch.zeros(nb, dtype=torch.float32, device=dev) if two else None,
                       philox_offset=philox_offset)
        return cls(param, grad, m32=torch.zeros(n, dtype=torch.float32, device=dev),
                   v32=torch.zeros(n, dtype=torch.float32, device=dev) if two else None,
                   philox_offset=philox_offset)

    def slice(self, start: int, count: int, philox_offset: int):
        """Block-aligned slice [start, start + count) of this tensor with the
        given global Philox offset (the 8-bit state stays on the 8-bit path)."""
        assert self.m_codes is not None, "slices are taken of 8-bit state"
        assert start % BLOCK == 0 and 0 <= start and start + count <= self.param.numel()
        b0, b1 = start // BLOCK, (start + count + BLOCK - 1) // BLOCK
        sl = slice(start, start + count)
        opt = lambda t, s: None if t is None else t[s]
        return Tensor8(self.param[sl], opt(self.grad, sl), self.m_codes[sl], opt(self.v_codes, sl),
                       self.m_absmax[b0:b1], opt(self.v_absmax, slice(b0, b1)), philox_offset=philox_offset)

    def _struct(self):
        assert self.param.dtype == torch.bfloat16 and self.grad.dtype == torch.bfloat16
        assert self.grad.numel() == self.param.numel()
        return _Tensor8(_ptr(self.param), _ptr(self.grad), self.param.numel(), self.philox_offset,
                        _ptr(self.m_codes), _ptr(self.v_codes), _ptr(self.m_absmax),
                        _ptr(self.v_absmax), _ptr(self.m32), _ptr(self.v32))


@dataclass
class Tensor16:
    """One tensor of the BF16-state step (all bf16)."""
    param: torch.Tensor
    grad: torch.Tensor
    m: torch.Tensor
    v: torch.Tensor
    philox_offset: int = -1

    def _struct(self):
        for t in (self.param, self.grad, self.m, self.v):
            assert t.dtype == torch.bfloat16 and t.numel() == self.param.numel()
        return _Tensor16(_ptr(self.param), _ptr(self.grad), _ptr(self.m), _ptr(self.v),
                         self.param.numel(), self.philox_offset)


def pack_tensor8(tensors: Sequence[Tensor8]):
    """ctypes array for adamw8bit_sr_step (keep it to re-issue the same list)."""
    return (_Tensor8 * len(tensors))(*[t._struct() for t in tensors])


def pack_tensor16(tensors: Sequence[Tensor16]):
    return (_Tensor16 * len(tensors))(*[t._struct() for t in tensors])


def adamw8bit_sr_step(tensors, hp: HParams, stream=None) -> None:
    """Fused 8-bit blockwise AdamW + SR step over a list of Tensor8 (or a list
    already packed by pack_tensor8)."""
    arr = tensors if isinstance(tensors, C.Array) else pack_tensor8(tensors)
    _check("adamw8bit_sr_step", load_library().adamw8bit_sr_step(arr, len(arr), C.byref(hp), _stream(stream)))


def adamw_bf16_sr_step(tensors, hp: HParams, stream=None) -> None:
    """BF16-state AdamW + SR step over a list of Tensor16 (or a packed list)."""
    arr = tensors if isinstance(tensors, C.Array) else pack_tensor16(tensors)
    _check("adamw_bf16_sr_step", load_library().adamw_bf16_sr_step(arr, len(arr), C.byref(hp), _stream(stream)))


def momentum8bit_sr_step(tensors, hp: MomentumHParams, stream=None) -> None:
    """8-bit SGD-with-momentum step with SR parameter write over a list of
    Tensor8 holding first-moment state only (see Tensor8.zeros_like(moments=1))."""
    arr = tensors if isinstance(tensors, C.Array) else pack_tensor8(tensors)
    _check("momentum8bit_sr_step", load_library().momentum8bit_sr_step(arr, len(arr), C.byref(hp), _stream(stream)))


def lion8bit_sr_step(tensors, hp: LionHParams, stream=None) -> None:
    """8-bit Lion step with SR parameter write (first-moment state only)."""
    arr = tensors if isinstance(tensors, C.Array) else pack_tensor8(tensors)
    _check("lion8bit_sr_step", load_library().lion8bit_sr_step(arr, len(arr), C.byref(hp), _stream(stream)))
