"""GPU parity of the 8-bit Momentum and 8-bit Lion steps (SR parameter write)
against the oracle, bit for bit, through the C ABI."""
import numpy as np
import pytest
import torch

import bit_blockwise_adamw_gb300 as q8
from bit_blockwise_adamw_gb300 import workloads as W
import oracle as o

from parity import SampledRun, compare_slice8, host_slice8, oracle_pool, shift16, u16

pytestmark = pytest.mark.gpu

OPTS = {"momentum": (o.MOMENTUM, q8.momentum8bit_sr_step), "lion": (o.LION, q8.lion8bit_sr_step)}


def _hp(name, step, sr, wd=0.01):
    if name == "momentum":
        return (q8.momentum_hparams(lr=1e-2, momentum=0.9, weight_decay=wd, step=step, seed=3, sr=sr),
                o.hparams(lr=1e-2, beta1=0.9, weight_decay=wd, step=step, seed=3, sr=sr))
    return (q8.lion_hparams(lr=1e-4, beta1=0.9, beta2=0.99, weight_decay=wd, step=step, seed=3, sr=sr),
            o.hparams(lr=1e-4, beta1=0.9, beta2=0.99, weight_decay=wd, step=step, seed=3, sr=sr))


def _run(name, wl, device, steps, sr=1, offsets=None, grad_hook=None, wd=0.01, shifted=()):
    opt, fn = OPTS[name]
    params = W.init_params(wl, device)
    params = [shift16(p) if i in shifted else p for i, p in enumerate(params)]
    offsets = offsets or [-1] * len(params)
    gpu = [q8.Tensor8.zeros_like(p, None, philox_offset=off, moments=1) for p, off in zip(params, offsets)]
    host = [o.zeros_onestate(u16(p), np.zeros(p.numel(), np.uint16), philox_offset=off)
            for p, off in zip(params, offsets)]
    for step in range(1, steps + 1):
        grads = W.make_grads(wl, step, device)
        grads = [shift16(g) if i in shifted else g for i, g in enumerate(grads)]
        if grad_hook:
            grad_hook(step, grads)
        for a, b, g in zip(gpu, host, grads):
            a.grad = g
            b.grad = u16(g)
        hg, hh = _hp(name, step, sr, wd)
        fn(gpu, hg)
        o.onestate_sr_step(opt, host, hh)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(gpu, host)):
            where = "%s tensor %d step %d" % (name, i, step)
            np.testing.assert_array_equal(u16(a.param), b.param, err_msg="param " + where)
            if b.m_codes is not None:
                np.testing.assert_array_equal(a.m_codes.cpu().numpy(), b.m_codes, err_msg="codes " + where)
                np.testing.assert_array_equal(a.m_absmax.cpu().numpy().view(np.uint32),
                                              b.m_absmax.view(np.uint32), err_msg="absmax " + where)
            else:
                np.testing.assert_array_equal(a.m32.cpu().numpy().view(np.uint32), b.m32.view(np.uint32),
                                              err_msg="m32 " + where)


@pytest.mark.parametrize("name", ["momentum", "lion"])
@pytest.mark.parametrize("sr", [1, 0])
def test_flat_full_parity(cuda_device, name, sr):
    wl = W.custom("flat", [1 << 20], steps=6, outlier_rate=1e-3, outlier_factor=100.0, data_seed=90)
    _run(name, wl, cuda_device, 6, sr=sr)


@pytest.mark.parametrize("name", ["momentum", "lion"])
def test_edge_sizes(cuda_device, name):
    wl = W.custom("edges", [1, 7, 2047, 2048, 4095, 4096, 4097, 3 * 2048 + 1, 65536 + 24, 0, 300],
                  steps=4, data_seed=91)
    _run(name, wl, cuda_device, 4)


@pytest.mark.parametrize("name", ["momentum", "lion"])
def test_zero_gradient_blocks(cuda_device, name):
    """Blocks with an all-zero first moment (absmax 0, zero code 127); no
    weight decay, which momentum would otherwise add to the gradient."""
    wl = W.custom("zeros", [4 * 2048, 2048 * 3 + 100, 5000], steps=4, data_seed=94)

    def hook(step, grads):
        grads[0][2048:4096].zero_()
        grads[1][3 * 2048:].zero_()
        grads[2].zero_()
    _run(name, wl, cuda_device, 4, grad_hook=hook, wd=0.0)


@pytest.mark.parametrize("name", ["momentum", "lion"])
def test_misaligned_offsets(cuda_device, name):
    wl = W.custom("offs", [5000, 2048 * 3 + 5, 700], steps=3, data_seed=92)
    _run(name, wl, cuda_device, 3, offsets=[3, (1 << 33) + 5, 11])


@pytest.mark.parametrize("name", ["momentum", "lion"])
@pytest.mark.parametrize("shifted", [(0, 1, 2), (1,)], ids=["all", "one"])
def test_grad_and_param_16_byte_aligned(cuda_device, name, shifted):
    """Grad and param arrays 16-byte but not 32-byte aligned: 16-byte accesses
    instead of 32-byte ones, the same results."""
    wl = W.custom("shift16", [2048 * 30, 2048 * 5 + 9, 3000], steps=3, data_seed=94)
    _run(name, wl, cuda_device, 3, shifted=shifted)


@pytest.mark.parametrize("name", ["momentum", "lion"])
def test_model_shaped_list(cuda_device, name):
    """A GPT-2-shaped list of two layers (weights, biases, LayerNorm gains)."""
    from bit_blockwise_adamw_gb300.workloads import _gpt2
    wl = W.Workload("gpt2-2l", _gpt2(2, 256, 1024, vocab=1000, ctx=128), steps=3,
                    hp={}, grad_std=1e-3, data_seed=93)
    _run(name, wl, cuda_device, 3)


@pytest.mark.parametrize("name", ["momentum", "lion"])
def test_sharded_step_equals_unsharded(cuda_device, name):
    """Three data-parallel ranks emulated in sequence on one GPU, each updating
    only its block-aligned slices with global Philox offsets.  After every
    rank's call the oracle replays that rank's slices (one-state tensor step
    with the slice's absmax sub-array and global offset) and the rank's params,
    codes and absmax must equal it bit for bit; the union also equals the
    unsharded one-state step."""
    from bit_blockwise_adamw_gb300 import sharding
    opt, fn = OPTS[name]
    wl = W.custom("shard1", [2048 * 20 + 7, 300, 4096, 2048 * 9, 65536 + 24], steps=3, data_seed=95)
    params = W.init_params(wl, cuda_device)
    whole = [q8.Tensor8.zeros_like(p.clone(), None, moments=1) for p in params]
    split = [q8.Tensor8.zeros_like(p.clone(), None, moments=1) for p in params]
    host = [o.zeros_onestate(u16(p), np.zeros(p.numel(), np.uint16)) for p in params]
    plan = sharding.plan([p.numel() for p in params], 3)
    for step in range(1, 4):
        grads = W.make_grads(wl, step, cuda_device)
        for a, b, c, g in zip(whole, split, host, grads):
            a.grad = g
            b.grad = g
            c.grad[:] = u16(g)
        hg, hh = _hp(name, step, 1)
        fn(whole, hg)
        for rank in range(3):
            fn(sharding.shard(split, 3, rank), hg)
            for sl in plan[rank]:
                hs = host_slice8(host[sl.tensor], sl)
                if hs.m_codes is not None:
                    o.onestate8bit_tensor(opt, hs, sl.philox_offset, hh)
                else:
                    o.onestate32_tensor(opt, hs, sl.philox_offset, hh)
            torch.cuda.synchronize()
            for sl in plan[rank]:
                compare_slice8(split[sl.tensor], host[sl.tensor], sl,
                               "%s rank %d, tensor %d, step %d" % (name, rank, sl.tensor, step))
    torch.cuda.synchronize()
    for a, b in zip(whole, split):
        assert torch.equal(a.param, b.param)
        if a.m_codes is not None:
            assert torch.equal(a.m_codes, b.m_codes) and torch.equal(a.m_absmax, b.m_absmax)
        else:
            assert torch.equal(a.m32, b.m32)


@pytest.fixture(scope="module")
def pool():
    p = oracle_pool()
    yield p
    p.close()
    p.join()


@pytest.mark.parametrize("name", ["momentum", "lion"])
def test_full_size_sampled_parity_gptneo67b(cuda_device, pool, name):
    """The GPT-Neo 6.7B list at full size, launched as the benchmark launches
    it (one call per step, the bench's hyper-parameters): a seeded sample of
    blocks plus the first and last block of every tensor, replayed by the
    oracle over three steps, bit for bit."""
    run = SampledRun(W.WORKLOADS["gptneo-6.7b"], cuda_device, 0.002, steps=3, opt=OPTS[name][0])
    run.run()
    assert run.check(pool) > 0
