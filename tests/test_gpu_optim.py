"""The torch.optim front end: the same bits as direct library calls, and a
state_dict round trip that continues bit for bit."""
import copy

import pytest
import torch

import bit_blockwise_adamw_gb300 as q8
from bit_blockwise_adamw_gb300 import optim

pytestmark = pytest.mark.gpu


def _params(dev, seed=0):
    g = torch.Generator(device=dev).manual_seed(seed)
    shapes = [(300, 64), (64,), (4096,), (1000, 7)]
    return [torch.nn.Parameter((torch.randn(s, generator=g, device=dev) * 0.02).to(torch.bfloat16)) for s in shapes]


def _grads(params, step, dev):
    g = torch.Generator(device=dev).manual_seed(1000 + step)
    for p in params:
        p.grad = (torch.randn(p.shape, generator=g, device=dev) * 1e-3).to(torch.bfloat16)


def test_adamw_front_end_equals_direct_calls(cuda_device):
    a = _params(cuda_device)
    b = [torch.nn.Parameter(p.detach().clone()) for p in a]
    opt = optim.AdamW8bitSR(a, lr=1e-3, weight_decay=0.01, seed=5)
    states = [q8.Tensor8.zeros_like(p.detach()) for p in b]
    offs, run = [], 0
    for p in b:
        offs.append(run)
        run += p.numel()
    for step in range(1, 4):
        _grads(a, step, cuda_device)
        _grads(b, step, cuda_device)
        opt.step()
        for s, p, off in zip(states, b, offs):
            s.param, s.grad, s.philox_offset = p.detach(), p.grad.detach(), off
        q8.adamw8bit_sr_step(states, q8.hparams(lr=1e-3, weight_decay=0.01, step=step, seed=5))
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.detach(), y.detach())


@pytest.mark.parametrize("cls", [optim.AdamW8bitSR, optim.Momentum8bitSR, optim.Lion8bitSR, optim.AdamWBF16SR])
def test_state_dict_resume(cuda_device, cls):
    a = _params(cuda_device)
    opt = cls(a, seed=7)
    for step in range(1, 4):
        _grads(a, step, cuda_device)
        opt.step()
    saved_params = [p.detach().clone() for p in a]
    saved = copy.deepcopy(opt.state_dict())
    for step in range(4, 7):
        _grads(a, step, cuda_device)
        opt.step()
    b = [torch.nn.Parameter(p.clone()) for p in saved_params]
    opt2 = cls(b, seed=7)
    opt2.load_state_dict(saved)
    for step in range(4, 7):
        _grads(b, step, cuda_device)
        opt2.step()
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.detach(), y.detach())


def test_param_groups_and_missing_grads(cuda_device):
    """Two groups with their own lr, one parameter without a gradient in one
    step: each group equals direct calls with its own hyper-parameters and a
    parameter without a gradient is left alone (its Philox offset stays
    reserved)."""
    a = _params(cuda_device)
    b = [torch.nn.Parameter(p.detach().clone()) for p in a]
    opt = optim.AdamW8bitSR([{"params": a[:2], "lr": 1e-3}, {"params": a[2:], "lr": 3e-4}], seed=2)
    states = [q8.Tensor8.zeros_like(p.detach()) for p in b]
    offs = [0, a[0].numel(), a[0].numel() + a[1].numel(), a[0].numel() + a[1].numel() + a[2].numel()]
    for step in range(1, 3):
        _grads(a, step, cuda_device)
        _grads(b, step, cuda_device)
        if step == 2:
            a[3].grad = None
        opt.step()
        for s, p, off in zip(states, b, offs):
            s.param, s.grad, s.philox_offset = p.detach(), p.grad.detach(), off
        q8.adamw8bit_sr_step(states[:2], q8.hparams(lr=1e-3, weight_decay=0.01, step=step, seed=2))
        q8.adamw8bit_sr_step(states[2:] if step == 1 else states[2:3],
                             q8.hparams(lr=3e-4, weight_decay=0.01, step=step, seed=2))
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.detach(), y.detach())


@pytest.mark.parametrize("cls", [optim.AdamW8bitSR, optim.Lion8bitSR, optim.AdamWBF16SR])
def test_front_end_trains_a_linear_model(cuda_device, cls):
    """End to end through torch.optim: a bf16 linear layer fitted to a fixed
    random linear map; the loss falls by more than 10x."""
    g = torch.Generator(device=cuda_device).manual_seed(3)
    target = torch.randn(64, 256, generator=g, device=cuda_device) / 16
    model = torch.nn.Linear(256, 64, bias=True, dtype=torch.bfloat16, device=cuda_device)
    lr = 1e-3 if cls is optim.Lion8bitSR else 3e-3
    opt = cls(model.parameters(), lr=lr, weight_decay=0.0, seed=1)
    x = torch.randn(512, 256, generator=g, device=cuda_device)
    y = x @ target.T
    losses = []
    for _ in range(300):
        opt.zero_grad(set_to_none=True)
        loss = (model(x.to(torch.bfloat16)).float() - y).square().mean()
        loss.backward()
        opt.step()
        losses.append(float(loss.detach()))
    assert losses[-1] < losses[0] / 10, (losses[0], losses[-1])
