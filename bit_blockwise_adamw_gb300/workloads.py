"""Synthetic, seeded workloads shaped like the models the pages train.

This module holds shapes, hyper-parameters and random-number recipes only --
none of the optimizer's arithmetic.  The tests feed the same generated
tensors to the CUDA path and to the oracle; the benchmark times the step on
them.  Nothing here reads a dataset or a checkpoint: parameters are a fresh
N(0, 0.02) draw (LayerNorm gains 1, biases 0) and gradients are Gaussian
draws with the outlier and scale structure stated per workload.

Shapes: GPT-2 350M ("Stochastic Rounding for LLM Training: Theory and
Practice", Figure 4), GPT-2 XL 1.5B (the 1.5B language model of "8-bit
Optimizers via Block-wise Quantization", results), GPT-Neo 6.7B and 2.7B
(the same LLM-training page, Figures 5 and 6).
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

BLOCK = 2048
SMALL_NUMEL = 4096


@dataclass(frozen=True)
class TensorSpec:
    name: str
    numel: int
    kind: str            # "weight" | "gain" | "bias"


@dataclass
class Workload:
    name: str
    tensors: List[TensorSpec]
    steps: int
    hp: Dict[str, float]
    grad_std: float
    outlier_rate: float = 0.0
    outlier_factor: float = 1.0
    lognormal_sigma: float = 0.0      # per-tensor scale exp(sigma * z), z ~ N(0, 1)
    state: str = "8bit"               # "8bit" | "bf16"
    data_seed: int = 1000
    philox_seed: int = 0
    note: str = ""
    extra: Dict[str, object] = field(default_factory=dict)

    @property
    def numel(self) -> int:
        return sum(t.numel for t in self.tensors)

    def blocks(self) -> int:
        return sum((t.numel + BLOCK - 1) // BLOCK for t in self.tensors if t.numel >= SMALL_NUMEL)

    def small_tensors(self) -> List[int]:
        return [i for i, t in enumerate(self.tensors) if t.numel < SMALL_NUMEL]


def _gpt2(L, d, ffn, vocab=50257, ctx=1024):
    ts = [TensorSpec("wte", vocab * d, "weight"), TensorSpec("wpe", ctx * d, "weight")]
    for i in range(L):
        p = "h%d." % i
        ts += [TensorSpec(p + "ln_1.g", d, "gain"), TensorSpec(p + "ln_1.b", d, "bias"),
               TensorSpec(p + "attn.qkv.W", d * 3 * d, "weight"), TensorSpec(p + "attn.qkv.b", 3 * d, "bias"),
               TensorSpec(p + "attn.out.W", d * d, "weight"), TensorSpec(p + "attn.out.b", d, "bias"),
               TensorSpec(p + "ln_2.g", d, "gain"), TensorSpec(p + "ln_2.b", d, "bias"),
               TensorSpec(p + "mlp.fc1.W", d * ffn, "weight"), TensorSpec(p + "mlp.fc1.b", ffn, "bias"),
               TensorSpec(p + "mlp.fc2.W", ffn * d, "weight"), TensorSpec(p + "mlp.fc2.b", d, "bias")]
    ts += [TensorSpec("ln_f.g", d, "gain"), TensorSpec("ln_f.b", d, "bias")]
    return ts


def _gptneo(L, d, ffn, vocab=50257, ctx=2048):
    ts = [TensorSpec("wte", vocab * d, "weight"), TensorSpec("wpe", ctx * d, "weight")]
    for i in range(L):
        p = "h%d." % i
        ts += [TensorSpec(p + "ln_1.g", d, "gain"), TensorSpec(p + "ln_1.b", d, "bias"),
               TensorSpec(p + "attn.q.W", d * d, "weight"), TensorSpec(p + "attn.k.W", d * d, "weight"),
               TensorSpec(p + "attn.v.W", d * d, "weight"), TensorSpec(p + "attn.out.W", d * d, "weight"),
               TensorSpec(p + "attn.out.b", d, "bias"),
               TensorSpec(p + "ln_2.g", d, "gain"), TensorSpec(p + "ln_2.b", d, "bias"),
               TensorSpec(p + "mlp.fc1.W", d * ffn, "weight"), TensorSpec(p + "mlp.fc1.b", ffn, "bias"),
               TensorSpec(p + "mlp.fc2.W", ffn * d, "weight"), TensorSpec(p + "mlp.fc2.b", d, "bias")]
    ts += [TensorSpec("ln_f.g", d, "gain"), TensorSpec("ln_f.b", d, "bias")]
    return ts


_HP1 = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)

WORKLOADS: Dict[str, Workload] = {
    "flat-1m": Workload(
        "flat-1m", [TensorSpec("flat", 1 << 20, "weight")], steps=10, hp=dict(_HP1),
        grad_std=1e-3, outlier_rate=1e-3, outlier_factor=100.0, data_seed=1000,
        note="one flat tensor of 1,048,576 params (512 blocks of 2048)"),
    "gpt2-350m": Workload(
        "gpt2-350m", _gpt2(24, 1024, 4096), steps=100, hp=dict(_HP1), grad_std=1e-3, data_seed=1001,
        note="GPT-2 350M tensor list: 24 layers, d=1024, ffn 4096, vocab 50257, ctx 1024"),
    "gpt2-xl-1.5b": Workload(
        "gpt2-xl-1.5b", _gpt2(48, 1600, 6400), steps=20, hp=dict(_HP1), grad_std=1e-3,
        lognormal_sigma=1.0, data_seed=1002,
        note="GPT-2 XL 1.5B tensor list: 48 layers, d=1600, ffn 6400, vocab 50257, ctx 1024"),
    "gptneo-6.7b": Workload(
        "gptneo-6.7b", _gptneo(32, 4096, 16384), steps=10,
        hp=dict(lr=6e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1),
        grad_std=1e-4, outlier_rate=1e-4, outlier_factor=1000.0, data_seed=1003,
        note="GPT-Neo 6.7B tensor list: 32 layers, d=4096, ffn 16384, vocab 50257, ctx 2048"),
    "gptneo-2.7b-bf16": Workload(
        "gptneo-2.7b-bf16", _gptneo(32, 2560, 10240), steps=20,
        hp=dict(lr=1.2e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1),
        grad_std=1e-4, state="bf16", data_seed=1004,
        note="GPT-Neo 2.7B tensor list on the BF16-state variant: 32 layers, d=2560, ffn 10240"),
}

ORDER = ["flat-1m", "gpt2-350m", "gpt2-xl-1.5b", "gptneo-6.7b", "gptneo-2.7b-bf16"]


def custom(name: str, sizes: List[int], steps: int = 3, grad_std: float = 1e-3, **kw) -> Workload:
    """A small ad-hoc list (for edge cases): weights of the given sizes."""
    hp = dict(_HP1)
    hp.update(kw.pop("hp", {}))
    return Workload(name, [TensorSpec("t%d" % i, n, "weight") for i, n in enumerate(sizes)],
                    steps=steps, hp=hp, grad_std=grad_std, **kw)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def init_params(wl: Workload, device) -> List[torch.Tensor]:
    """bf16 parameters: weights ~ N(0, 0.02) (rounded to nearest), gains 1, biases 0."""
    g = _gen(device, wl.data_seed)
    out = []
    for t in wl.tensors:
        if t.kind == "gain":
            out.append(torch.ones(t.numel, dtype=torch.bfloat16, device=device))
        elif t.kind == "bias":
            out.append(torch.zeros(t.numel, dtype=torch.bfloat16, device=device))
        else:
            x = torch.randn(t.numel, generator=g, device=device, dtype=torch.float32)
            out.append(x.mul_(0.02).to(torch.bfloat16))
    return out


def grad_seed(wl: Workload, step: int) -> int:
    return wl.data_seed * 1_000_003 + step


def make_grads(wl: Workload, step: int, device, out: Optional[List[torch.Tensor]] = None) -> List[torch.Tensor]:
    """Fresh bf16 gradients for `step`: N(0, grad_std), times a per-tensor
    lognormal scale if set, with a Bernoulli(outlier_rate) mask scaled by
    outlier_factor.  Written into `out` when given."""
    g = _gen(device, grad_seed(wl, step))
    scales = None
    if wl.lognormal_sigma > 0:
        z = torch.randn(len(wl.tensors), generator=_gen("cpu", wl.data_seed + 7), dtype=torch.float64)
        scales = torch.exp(wl.lognormal_sigma * z).tolist()
    res = []
    for i, t in enumerate(wl.tensors):
        x = torch.randn(t.numel, generator=g, device=device, dtype=torch.float32)
        std = wl.grad_std * (scales[i] if scales else 1.0)
        x.mul_(std)
        if wl.outlier_rate > 0:
            mask = torch.rand(t.numel, generator=g, device=device) < wl.outlier_rate
            x[mask] *= wl.outlier_factor
            del mask
        if out is not None:
            out[i].copy_(x)
            res.append(out[i])
        else:
            res.append(x.to(torch.bfloat16))
        del x
    return res


def philox_offsets(wl: Workload) -> List[int]:
    """Global Philox index of element 0 of each tensor (running element count)."""
    offs, run = [], 0
    for t in wl.tensors:
        offs.append(run)
        run += t.numel
    return offs


def sample_blocks(wl: Workload, fraction: float, seed: int = 0):
    """Blocks whose trajectories the oracle replays: the first and last block
    of every 8-bit tensor plus a seeded fraction of the rest.  Returns a list
    of (tensor index, block index)."""
    g = torch.Generator()
    g.manual_seed(seed)
    picks = []
    for i, t in enumerate(wl.tensors):
        if t.numel < SMALL_NUMEL and wl.state == "8bit":
            continue
        nb = (t.numel + BLOCK - 1) // BLOCK
        chosen = {0, nb - 1}
        if nb > 2 and fraction > 0:
            k = int(round((nb - 2) * fraction))
            if k:
                chosen |= set((torch.randperm(nb - 2, generator=g)[:k] + 1).tolist())
        picks += [(i, b) for b in sorted(chosen)]
    return picks
