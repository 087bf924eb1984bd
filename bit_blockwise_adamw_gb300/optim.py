"""torch.optim front end for the library's steps ("8-bit Optimizers via
Block-wise Quantization", applications: plug-and-play with PyTorch).

Each optimizer keeps its state in ordinary tensors (so `state_dict()` saves
and restores it) and issues one library call per parameter group and step.
Parameters must be contiguous bf16 CUDA tensors with bf16 gradients.  Every
parameter is given a fixed global Philox offset when it is first seen (the
running element count in group order), so the stochastic-rounding draws of
an element depend only on (seed, step, element) and a restored optimizer
continues bit for bit.

The descriptor table a step passes to the library is built once per group
(state pointers do not move); each step only refreshes its param and grad
pointers.
"""
import numpy as np
import torch

from . import _binding as B

_T8_FIELDS = [f[0] for f in B._Tensor8._fields_]
_T16_FIELDS = [f[0] for f in B._Tensor16._fields_]


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def _check_param(p):
    if p.dtype != torch.bfloat16 or not p.is_cuda or not p.is_contiguous():
        raise ValueError("parameters must be contiguous bf16 CUDA tensors")
    g = p.grad
    if g.dtype != torch.bfloat16 or not g.is_contiguous() or g.shape != p.shape or g.device != p.device:
        raise ValueError("gradients must be contiguous bf16 tensors shaped like their parameters")
    return g


class _Table:
    """A group's packed descriptors: an int64 table whose rows have the
    layout of the library's tensor struct (all fields 8 bytes), viewed as a
    ctypes array without a copy."""

    def __init__(self, params, rows, struct, fields):
        self.params = list(params)
        self.np = np.array([[row[f] for f in fields] for row in rows], dtype=np.int64).reshape(len(rows),
                                                                                            len(fields))
        self.c = (struct * len(rows)).from_buffer(self.np)

    def matches(self, params):
        return len(params) == len(self.params) and all(a is b for a, b in zip(params, self.params))

    def refresh(self):
        for i, p in enumerate(self.params):
            g = _check_param(p)
            self.np[i, 0] = p.data_ptr()
            self.np[i, 1] = g.data_ptr()
        return self.c


class _FrontEnd(torch.optim.Optimizer):
    """Philox offset bookkeeping, the cached descriptor tables and a
    state_dict round trip that keeps each state tensor's dtype (torch.optim
    casts floating-point state to the parameter's dtype on load, which would
    turn uint8 codes and float32 absmax into bf16)."""

    def __init__(self, params, defaults):
        super().__init__(params, defaults)
        self._next_offset = 0
        self._tables = {}
        # the library's one-time per-device set-up (tables, launch
        # configurations) now, so that no step synchronises or does set-up
        # (a step may then be captured in a CUDA graph)
        devices = {p.device for g in self.param_groups for p in g["params"] if p.is_cuda}
        for dev in devices:
            with torch.cuda.device(dev):
                B.q8_prepare_device()

    def _offset(self, p, state):
        if "philox_offset" not in state:
            state["philox_offset"] = self._next_offset
            self._next_offset += p.numel()
        return int(state["philox_offset"])

    def load_state_dict(self, state_dict):
        saved = state_dict["state"]
        ids = [i for g in state_dict["param_groups"] for i in g["params"]]
        params = [p for g in self.param_groups for p in g["params"]]
        super().load_state_dict(state_dict)
        for i, p in zip(ids, params):
            for k, v in saved.get(i, {}).items():
                if torch.is_tensor(v):
                    self.state[p][k] = v.to(device=p.device).clone()
        used = [int(s["philox_offset"]) + p.numel() for p, s in self.state.items() if "philox_offset" in s]
        self._next_offset = max(used, default=0)
        self._tables = {}

    def _table(self, gi, params):
        t = self._tables.get(gi)
        if t is None or not t.matches(params):
            t = _Table(params, [self._row(p) for p in params], *self._struct)
            self._tables[gi] = t
        return t.refresh()

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for gi, group in enumerate(self.param_groups):
            params = [p for p in group["params"] if p.grad is not None]
            if not params:
                continue
            arr = self._table(gi, params)
            group["step"] = group.get("step", 0) + 1
            self._run(group, arr)
        return loss


class _Q8Optimizer(_FrontEnd):
    moments = 2
    _struct = (B._Tensor8, _T8_FIELDS)

    def _row(self, p):
        _check_param(p)
        state = self.state[p]
        off = self._offset(p, state)
        if "m_codes" not in state and "m32" not in state:
            t = B.Tensor8.zeros_like(p.detach(), moments=self.moments)
            for k in ("m_codes", "v_codes", "m_absmax", "v_absmax", "m32", "v32"):
                if getattr(t, k) is not None:
                    state[k] = getattr(t, k)
        row = {k: _ptr(state.get(k)) for k in ("m_codes", "v_codes", "m_absmax", "v_absmax", "m32", "v32")}
        row.update(param=p.data_ptr(), grad=p.grad.data_ptr(), numel=p.numel(), philox_offset=off)
        return row


class AdamW8bitSR(_Q8Optimizer):
    """AdamW with 8-bit blockwise m, v and stochastically rounded bf16 params
    (adamw8bit_sr_step).  Parameters below 4096 elements keep fp32 state.
    exact=True asks for the bit-exact mode (correctly rounded square root and
    division); the default fast mode differs from it by at most one bf16 ulp
    on rare parameters, never in the state."""

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=1e-2, seed=0,
                 stochastic_rounding=True, exact=False):
        super().__init__(params, dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding), exact=int(exact)))

    def _run(self, group, arr):
        b1, b2 = group["betas"]
        B.adamw8bit_sr_step(arr, B.hparams(lr=group["lr"], beta1=b1, beta2=b2, eps=group["eps"],
                                           weight_decay=group["weight_decay"], step=group["step"],
                                           seed=group["seed"], sr=group["sr"], exact=group.get("exact", 0)))


class Momentum8bitSR(_Q8Optimizer):
    """SGD with momentum, 8-bit blockwise momentum buffer, SR bf16 params."""
    moments = 1

    def __init__(self, params, lr=1e-2, momentum=0.9, weight_decay=0.0, seed=0, stochastic_rounding=True):
        super().__init__(params, dict(lr=lr, momentum=momentum, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding)))

    def _run(self, group, arr):
        B.momentum8bit_sr_step(arr, B.momentum_hparams(lr=group["lr"], momentum=group["momentum"],
                                                       weight_decay=group["weight_decay"],
                                                       step=group["step"], seed=group["seed"], sr=group["sr"]))


class Lion8bitSR(_Q8Optimizer):
    """Lion with an 8-bit blockwise momentum, SR bf16 params."""
    moments = 1

    def __init__(self, params, lr=1e-4, betas=(0.9, 0.99), weight_decay=0.0, seed=0, stochastic_rounding=True):
        super().__init__(params, dict(lr=lr, betas=betas, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding)))

    def _run(self, group, arr):
        b1, b2 = group["betas"]
        B.lion8bit_sr_step(arr, B.lion_hparams(lr=group["lr"], beta1=b1, beta2=b2,
                                               weight_decay=group["weight_decay"], step=group["step"],
                                               seed=group["seed"], sr=group["sr"]))


class AdamWBF16SR(_FrontEnd):
    """BF16-state AdamW with stochastic rounding of params and both moments
    (adamw_bf16_sr_step)."""
    _struct = (B._Tensor16, _T16_FIELDS)

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=1e-2, seed=0,
                 stochastic_rounding=True, exact=False):
        super().__init__(params, dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding), exact=int(exact)))

    def _row(self, p):
        _check_param(p)
        st = self.state[p]
        off = self._offset(p, st)
        if "m" not in st:
            st["m"] = torch.zeros_like(p)
            st["v"] = torch.zeros_like(p)
        return dict(param=p.data_ptr(), grad=p.grad.data_ptr(), m=st["m"].data_ptr(), v=st["v"].data_ptr(),
                    numel=p.numel(), philox_offset=off)

    def _run(self, group, arr):
        b1, b2 = group["betas"]
        B.adamw_bf16_sr_step(arr, B.hparams(lr=group["lr"], beta1=b1, beta2=b2, eps=group["eps"],
                                            weight_decay=group["weight_decay"], step=group["step"],
                                            seed=group["seed"], sr=group["sr"], exact=group.get("exact", 0)))
