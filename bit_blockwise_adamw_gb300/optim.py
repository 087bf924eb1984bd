"""torch.optim front end for the library's steps ("8-bit Optimizers via
Block-wise Quantization", applications: plug-and-play with PyTorch).

Each optimizer keeps its state in ordinary tensors (so `state_dict()` saves
and restores it) and issues one library call per parameter group and step.
Parameters must be contiguous bf16 CUDA tensors with bf16 gradients.  Every
parameter is given a fixed global Philox offset when it is first seen (the
running element count in group order), so the stochastic-rounding draws of
an element depend only on (seed, step, element) and a restored optimizer
continues bit for bit.
"""
import torch

from . import _binding as B


class _FrontEnd(torch.optim.Optimizer):
    """Philox offset bookkeeping and a state_dict round trip that keeps each
    state tensor's dtype (torch.optim casts floating-point state to the
    parameter's dtype on load, which would turn uint8 codes and float32
    absmax into bf16)."""

    def __init__(self, params, defaults):
        super().__init__(params, defaults)
        self._next_offset = 0

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


class _Q8Optimizer(_FrontEnd):
    moments = 2

    def _tensor8(self, p):
        if p.dtype != torch.bfloat16 or not p.is_cuda or not p.is_contiguous():
            raise ValueError("parameters must be contiguous bf16 CUDA tensors")
        state = self.state[p]
        off = self._offset(p, state)
        if "m_codes" not in state and "m32" not in state:
            t = B.Tensor8.zeros_like(p.detach(), moments=self.moments)
            for k in ("m_codes", "v_codes", "m_absmax", "v_absmax", "m32", "v32"):
                if getattr(t, k) is not None:
                    state[k] = getattr(t, k)
        return B.Tensor8(p.detach(), p.grad.detach(), state.get("m_codes"), state.get("v_codes"),
                         state.get("m_absmax"), state.get("v_absmax"), state.get("m32"), state.get("v32"),
                         philox_offset=off)

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for group in self.param_groups:
            tensors = [self._tensor8(p) for p in group["params"] if p.grad is not None]
            if not tensors:
                continue
            group["step"] = group.get("step", 0) + 1
            self._run(group, tensors)
        return loss


class AdamW8bitSR(_Q8Optimizer):
    """AdamW with 8-bit blockwise m, v and stochastically rounded bf16 params
    (adamw8bit_sr_step).  Parameters below 4096 elements keep fp32 state."""

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=1e-2, seed=0,
                 stochastic_rounding=True):
        super().__init__(params, dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding)))

    def _run(self, group, tensors):
        b1, b2 = group["betas"]
        B.adamw8bit_sr_step(tensors, B.hparams(lr=group["lr"], beta1=b1, beta2=b2, eps=group["eps"],
                                               weight_decay=group["weight_decay"], step=group["step"],
                                               seed=group["seed"], sr=group["sr"]))


class Momentum8bitSR(_Q8Optimizer):
    """SGD with momentum, 8-bit blockwise momentum buffer, SR bf16 params."""
    moments = 1

    def __init__(self, params, lr=1e-2, momentum=0.9, weight_decay=0.0, seed=0, stochastic_rounding=True):
        super().__init__(params, dict(lr=lr, momentum=momentum, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding)))

    def _run(self, group, tensors):
        B.momentum8bit_sr_step(tensors, B.momentum_hparams(lr=group["lr"], momentum=group["momentum"],
                                                           weight_decay=group["weight_decay"],
                                                           step=group["step"], seed=group["seed"], sr=group["sr"]))


class Lion8bitSR(_Q8Optimizer):
    """Lion with an 8-bit blockwise momentum, SR bf16 params."""
    moments = 1

    def __init__(self, params, lr=1e-4, betas=(0.9, 0.99), weight_decay=0.0, seed=0, stochastic_rounding=True):
        super().__init__(params, dict(lr=lr, betas=betas, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding)))

    def _run(self, group, tensors):
        b1, b2 = group["betas"]
        B.lion8bit_sr_step(tensors, B.lion_hparams(lr=group["lr"], beta1=b1, beta2=b2,
                                                   weight_decay=group["weight_decay"], step=group["step"],
                                                   seed=group["seed"], sr=group["sr"]))


class AdamWBF16SR(_FrontEnd):
    """BF16-state AdamW with stochastic rounding of params and both moments
    (adamw_bf16_sr_step)."""

    def __init__(self, params, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=1e-2, seed=0,
                 stochastic_rounding=True):
        super().__init__(params, dict(lr=lr, betas=betas, eps=eps, weight_decay=weight_decay, seed=seed,
                                      sr=int(stochastic_rounding)))

    @torch.no_grad()
    def step(self, closure=None):
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        for group in self.param_groups:
            tensors = []
            for p in group["params"]:
                if p.grad is None:
                    continue
                st = self.state[p]
                off = self._offset(p, st)
                if "m" not in st:
                    st["m"] = torch.zeros_like(p)
                    st["v"] = torch.zeros_like(p)
                tensors.append(B.Tensor16(p.detach(), p.grad.detach(), st["m"], st["v"], off))
            if not tensors:
                continue
            group["step"] = group.get("step", 0) + 1
            b1, b2 = group["betas"]
            B.adamw_bf16_sr_step(tensors, B.hparams(lr=group["lr"], beta1=b1, beta2=b2, eps=group["eps"],
                                                    weight_decay=group["weight_decay"], step=group["step"],
                                                    seed=group["seed"], sr=group["sr"]))
        return loss
