"""GPU parity of the fused steps against the oracle, through the C ABI.

Small cases compare every element after every step; the full-size workloads
(the model-shaped tensor lists at their real sizes, launched exactly as the
benchmark launches them) compare a seeded sample of 2048-blocks, every small
tensor and the first and last block of every tensor, replayed by the oracle
over all steps.  The bar is bit-exact parameters, codes, absmax and fp32
state (the method has one correct answer once its readings are fixed).
"""
import numpy as np
import pytest
import torch

import bit_blockwise_adamw_gb300 as q8
from bit_blockwise_adamw_gb300 import workloads as W
import oracle as o

from parity import (ParamTolerance, SampledRun, compare_slice8, compare_state8, gpu_states8, host_slice8,
                    host_states8, hp_for, oracle_pool, shift16, u16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pool():
    p = oracle_pool()
    yield p
    p.close()
    p.join()


def _run_full(wl, device, steps=None, sr=1, offsets=None, split=None, grad_hook=None, param_hook=None, shifted=(),
              exact=True, expect_bitexact=False):
    """Run `wl` on both sides for `steps`, comparing everything after each step
    (`grad_hook(step, grads)` may edit the step's gradients in place first,
    `param_hook(params)` the initial parameters; the params and grads of the
    tensors in `shifted` sit 16 bytes past a 32-byte boundary).  exact=False
    runs the fast mode and holds the parameters of each step to its tolerance,
    then gives the GPU the oracle's parameters, so that every step starts from
    identical inputs (expect_bitexact: the fast mode must be bit-exact here)."""
    steps = steps or wl.steps
    params = W.init_params(wl, device)
    params = [shift16(p) if i in shifted else p for i, p in enumerate(params)]
    if param_hook:
        param_hook(params)
    gpu = gpu_states8(params, offsets)
    host = host_states8([u16(p) for p in params], offsets)
    for step in range(1, steps + 1):
        grads = W.make_grads(wl, step, device)
        grads = [shift16(g) if i in shifted else g for i, g in enumerate(grads)]
        if grad_hook:
            grad_hook(step, grads)
        for g_gpu, g_host, gr in zip(gpu, host, grads):
            g_gpu.grad = gr
            g_host.grad = u16(gr)
        h = hp_for(wl, step, sr)
        if split:
            q8.adamw8bit_sr_step(gpu[:split], q8.hparams(**h, exact=int(exact)))
            q8.adamw8bit_sr_step(gpu[split:], q8.hparams(**h, exact=int(exact)))
        else:
            q8.adamw8bit_sr_step(gpu, q8.hparams(**h, exact=int(exact)))
        o.adamw8bit_sr_step(host, o.hparams(**h))
        torch.cuda.synchronize()
        tol = None if exact or expect_bitexact else ParamTolerance()
        for i, (a, b) in enumerate(zip(gpu, host)):
            compare_state8(a, b, "tensor %d step %d" % (i, step), tol)
        if tol is not None:
            tol.check()
            for a, b in zip(gpu, host):             # identical inputs for the next step
                a.param.copy_(torch.from_numpy(b.param.view(np.int16)).view(torch.bfloat16).to(a.param.device))
    return gpu, host


MODES = [True, False]
MODE_IDS = ["exact", "fast"]


@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("sr", [1, 0])
def test_flat_1m_full_parity(cuda_device, sr, exact):
    """1,048,576 params, 512 blocks, 10 steps, every element every step, in
    the bit-exact and the fast mode."""
    _run_full(W.WORKLOADS["flat-1m"], cuda_device, sr=sr, exact=exact)


EDGE_SIZES = [1, 7, 8, 9, 2047, 2048, 4095, 4096, 4097, 3 * 2048 + 1, 12345, 65536 + 24, 0, 300]


@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("sr", [1, 0])
def test_edge_sizes_mixed_paths(cuda_device, sr, exact):
    """Ragged tails, partial blocks, the 4095/4096 routing edge and an empty
    tensor in one list, 4 steps, both rounding modes."""
    wl = W.custom("edges", EDGE_SIZES, steps=4, outlier_rate=0.01, outlier_factor=50.0, data_seed=77)
    _run_full(wl, cuda_device, sr=sr, exact=exact)


@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("sr", [1, 0])
def test_nonfinite_parameters(cuda_device, sr, exact):
    """NaN, +inf and -inf parameters (finite gradients) in full blocks, a
    partial block and the fp32-state path: the step keeps the infinities and
    writes the quiet NaN 0x7FC0, as the oracle does, in both modes (the fast
    mode sends a NaN to its IEEE fallback; its one-ulp tolerance admits no other
    pattern for a NaN or an infinity)."""
    wl = W.custom("nonfinite", [2048 * 4, 2048 * 2 + 100, 3000], steps=3, data_seed=97)

    def params_hook(params):
        for p in params:
            w = p.view(torch.int16)
            w[5::97] = 0x7FC0                      # NaN
            w[11::89] = 0x7F80                     # +inf
            w[17::83] = -128                       # -inf (0xFF80)
    gpu, host = _run_full(wl, cuda_device, sr=sr, param_hook=params_hook, exact=exact)
    for t in host:
        assert int((t.param == 0x7FC0).sum()) > 0 and int((t.param == 0x7F80).sum()) > 0


@pytest.mark.parametrize("hp", [dict(eps=0.0), dict(eps=1e-12), dict(lr=10.0, weight_decay=0.0)],
                         ids=["eps_zero", "eps_below_2^-36", "step_size_above_1"])
def test_fast_mode_outside_its_range_is_exact(cuda_device, hp):
    """The fast mode applies only for eps_t in [2^-36, 2^20] and a_t <= 1;
    outside that range a call with exact=0 takes the exact path, bit for bit."""
    wl = W.custom("fastrange", [2048 * 6, 2048 * 2 + 7, 5000], steps=3, data_seed=96, hp=hp)
    _run_full(wl, cuda_device, exact=False, expect_bitexact=True)


@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
def test_zero_gradient_blocks(cuda_device, exact):
    """Blocks whose moments are all zero (absmax 0, zero codes 127 and 0):
    zero gradients from the first step in some blocks, a whole tensor and a
    partial last block, and zero gradients again after nonzero steps, where the
    moments decay but stay nonzero."""
    wl = W.custom("zeros", [4 * 2048, 2048 * 3 + 100, 5000, 4096], steps=5, data_seed=79)

    def hook(step, grads):
        grads[0][2048:4096].zero_()                     # one full block, every step
        grads[1][3 * 2048:].zero_()                     # the partial last block
        grads[2].zero_()                                # a whole tensor
        if step >= 3:
            grads[3].zero_()                            # zero after nonzero steps
    _run_full(wl, cuda_device, grad_hook=hook, exact=exact)


@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
def test_negative_zero_moments_and_params(cuda_device, exact):
    """Signed zeros through the whole step, with beta1 = 0 so that the new
    first moment is 0*m + g.  Elements 0 mod 4 get a -0 gradient every step:
    their m is +0 (+0 + -0), so where the parameter starts at -0 (every third
    element) the update is -0*decay - a*(+0/d) = -0, kept step after step.
    Elements 2 mod 4 get a -0 gradient on even steps: where the old m was
    negative the new m is -0, which must take the zero code 127 like +0 and
    the IEEE quotient -0/d = -0.  8-bit blocks, a partial block and the
    fp32-state path."""
    wl = W.custom("negzero", [4 * 2048, 2048 * 2 + 300, 3000], steps=4, data_seed=95, hp={"beta1": 0.0})

    def params_hook(params):
        for p in params:
            p.view(torch.int16)[::3] = -32768               # bf16 -0 (0x8000)

    def hook(step, grads):
        for g in grads:
            g.view(torch.int16)[::4] = -32768
            if step % 2 == 0:
                g.view(torch.int16)[2::4] = -32768
    gpu, host = _run_full(wl, cuda_device, grad_hook=hook, param_hook=params_hook, exact=exact)
    # the cases are live: -0 parameters survive, and zero codes sit in blocks
    # whose absmax is nonzero
    for t in host:
        assert int((t.param == 0x8000).sum()) > 0
    assert bool((gpu[0].m_codes == 127).any()) and bool((gpu[0].m_absmax > 0).all())


def test_explicit_misaligned_offsets(cuda_device):
    """Philox offsets that are not multiples of 8 (draws span two counters)."""
    sizes = [5000, 4099, 700, 2048 * 5 + 3]
    wl = W.custom("offsets", sizes, steps=3, data_seed=78)
    _run_full(wl, cuda_device, offsets=[3, 1 << 33, 12345677, 7])


@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("sr", [1, 0])
@pytest.mark.parametrize("shifted", [(0, 1, 2, 3), (2,)], ids=["all", "one"])
def test_grad_and_param_16_byte_aligned(cuda_device, sr, shifted, exact):
    """Grad and param arrays 16-byte but not 32-byte aligned (all of them, or
    one tensor of the list): the launch then moves grad and param with 16-byte
    accesses instead of 32-byte ones; the results are the oracle's all the same."""
    sizes = [2048 * 40, 2048 * 7 + 5, 5000, 1000]
    wl = W.custom("shift16", sizes, steps=3, data_seed=83, grad_std=1e-3)
    _run_full(wl, cuda_device, sr=sr, shifted=shifted, exact=exact)


def test_split_list_equals_whole_list(cuda_device):
    """Splitting a list with explicit global offsets gives the same bits as one call."""
    sizes = [8192, 3000, 2048 * 7 + 11, 4096]
    wl = W.custom("split", sizes, steps=3, data_seed=79)
    offs = W.philox_offsets(wl)
    a, _ = _run_full(wl, cuda_device)
    b, _ = _run_full(wl, cuda_device, offsets=offs, split=2)
    for x, y in zip(a, b):
        assert torch.equal(x.param, y.param)


def test_resume_equals_continuous(cuda_device):
    """5 + 5 steps with the state round-tripped through host memory equals 10 steps."""
    wl = W.custom("resume", [2048 * 9 + 5, 1000], steps=10, data_seed=80)
    params = W.init_params(wl, cuda_device)
    ref = gpu_states8([p.clone() for p in params])
    res = gpu_states8([p.clone() for p in params])
    for step in range(1, 11):
        grads = W.make_grads(wl, step, cuda_device)
        h = q8.hparams(**hp_for(wl, step))
        for s, g in zip(ref, grads):
            s.grad = g
        q8.adamw8bit_sr_step(ref, h)
        for s, g in zip(res, grads):
            s.grad = g
        q8.adamw8bit_sr_step(res, h)
        if step == 5:   # checkpoint: copy everything to the host and back
            for s in res:
                for f in ("param", "m_codes", "v_codes", "m_absmax", "v_absmax", "m32", "v32"):
                    t = getattr(s, f)
                    if t is not None:
                        t.copy_(t.cpu().to(cuda_device))
    torch.cuda.synchronize()
    for a, b in zip(ref, res):
        assert torch.equal(a.param, b.param)


def test_many_tensors_take_several_launches(cuda_device):
    """More tensors than one launch carries (448 per launch)."""
    sizes = [4096 + 8 * (i % 5) for i in range(500)] + [100 + i for i in range(460)]
    wl = W.custom("many", sizes, steps=2, data_seed=81)
    _run_full(wl, cuda_device)


def _run_bf16(wl, device, steps, offsets=None, sr=1, exact=True):
    params = W.init_params(wl, device)
    offsets = offsets or [-1] * len(params)
    gpu = [q8.Tensor16(p, None, torch.zeros_like(p), torch.zeros_like(p), off) for p, off in zip(params, offsets)]
    host = [o.State16(u16(p), np.zeros(p.numel(), np.uint16), np.zeros(p.numel(), np.uint16),
                      np.zeros(p.numel(), np.uint16), off) for p, off in zip(params, offsets)]
    for step in range(1, steps + 1):
        grads = W.make_grads(wl, step, device)
        for a, b, g in zip(gpu, host, grads):
            a.grad = g
            b.grad = u16(g)
        h = hp_for(wl, step, sr)
        q8.adamw_bf16_sr_step(gpu, q8.hparams(**h, exact=int(exact)))
        o.adamw_bf16_sr_step(host, o.hparams(**h))
        torch.cuda.synchronize()
        tol = None if exact else ParamTolerance()
        for i, (a, b) in enumerate(zip(gpu, host)):
            for name, x, y in (("param", a.param, b.param), ("m", a.m, b.m), ("v", a.v, b.v)):
                where = "%s tensor %d step %d" % (name, i, step)
                if tol is not None and name == "param":
                    tol.add(u16(x), y, where)
                else:
                    np.testing.assert_array_equal(u16(x), y, err_msg=where)
        if tol is not None:
            tol.check()
            for a, b in zip(gpu, host):             # identical inputs for the next step
                a.param.copy_(torch.from_numpy(b.param.view(np.int16)).view(torch.bfloat16).to(a.param.device))


@pytest.mark.parametrize("sr", [1, 0])
@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
def test_bf16_state_full_parity(cuda_device, sr, exact):
    wl = W.custom("bf16", [1, 7, 2048, 2049, 5000, 1 << 18, 0, 333], steps=5, data_seed=82,
                  hp=dict(lr=1.2e-3, weight_decay=0.1), grad_std=1e-4)
    _run_bf16(wl, cuda_device, 5, sr=sr, exact=exact)


def test_bf16_state_misaligned_offsets(cuda_device):
    wl = W.custom("bf16off", [1000, 4099, 2048 * 3 + 5], steps=3, data_seed=83)
    _run_bf16(wl, cuda_device, 3, offsets=[5, (1 << 34) + 1, 77])


def test_empty_list_and_zero_tensor(cuda_device):
    q8.adamw8bit_sr_step([], q8.hparams())
    q8.adamw_bf16_sr_step([], q8.hparams())
    p = torch.zeros(0, dtype=torch.bfloat16, device=cuda_device)
    q8.adamw8bit_sr_step([q8.Tensor8(p, p, m32=torch.zeros(0, device=cuda_device),
                                     v32=torch.zeros(0, device=cuda_device))], q8.hparams())
    torch.cuda.synchronize()


def test_bad_arguments_raise(cuda_device):
    p = torch.zeros(8192, dtype=torch.bfloat16, device=cuda_device)
    st = q8.Tensor8.zeros_like(p, p.clone())
    with pytest.raises(q8.Q8Error):
        q8.adamw8bit_sr_step([st], q8.hparams(step=0))
    st.param = p[1:4097]                       # misaligned view
    st.grad = p[1:4097]
    with pytest.raises(q8.Q8Error):
        q8.adamw8bit_sr_step([st], q8.hparams())


# ---------------------------------------------------------------- full size

FULL = [("gpt2-350m", 0.01), ("gpt2-xl-1.5b", 0.005), ("gptneo-6.7b", 0.003), ("gptneo-2.7b-bf16", 0.003)]


@pytest.mark.parametrize("exact", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("name,fraction", FULL)
def test_full_size_sampled_parity(cuda_device, pool, name, fraction, exact):
    """The five configurations at full size over all their steps, launched as
    the benchmark launches them: sampled blocks replayed by the oracle.  In the
    fast mode (each side on its own trajectory) codes, absmax and BF16 moments
    stay bit-exact and at least 99.9 % of the sampled parameters too; the
    one-ulp bound of a single step is tested from identical inputs in
    test_gpu_fast_mode.py and in the small cases above."""
    wl = W.WORKLOADS[name]
    run = SampledRun(wl, cuda_device, fraction, exact=exact)
    run.run()
    compared = run.check(pool)
    assert compared > 0
    if run.tol is not None:
        print("%s fast mode: %d of %d sampled parameters differ from the oracle (largest distance %d ulp)" % (
            name, run.tol.diff, run.tol.n, run.tol.max_ulps))


@pytest.mark.parametrize("state", ["8bit", "bf16"])
def test_tensor_beyond_2_31_elements(cuda_device, pool, state):
    """One tensor of 2^31 + 6221 elements (more elements than a signed 32-bit
    index reaches, with a partial last block) after a small one: the blocks on
    both sides of element 2^31, the first and the last, and a seeded sample,
    replayed by the oracle over two steps."""
    n = (1 << 31) + 3 * 2048 + 77
    wl = W.custom("huge-" + state, [5000, n], steps=2, data_seed=85, state=state)
    edge = (1 << 31) // 2048
    run = SampledRun(wl, cuda_device, 2e-6, extra_blocks=[(1, edge - 1), (1, edge), (1, edge + 1)])
    run.run()
    assert run.check(pool) > 0


@pytest.mark.parametrize("world", [2, 3, 8])
def test_sharded_step_equals_unsharded(cuda_device, world):
    """N data-parallel ranks emulated in sequence on one GPU: each updates only
    its block-aligned slices (global Philox offsets).  After every rank's call
    the oracle replays that rank's slices from the same inputs (its 8-bit
    tensor step on the slice, with the slice's absmax sub-arrays and global
    offset) and the rank's params, codes and absmax must equal it bit for bit;
    after every step the union also equals the unsharded CUDA step."""
    from bit_blockwise_adamw_gb300 import sharding
    wl = W.custom("shard", [2048 * 50 + 7, 300, 4096, 2048 * 9, 1000, 65536 + 24], steps=3, data_seed=84)
    params = W.init_params(wl, cuda_device)
    whole = gpu_states8([p.clone() for p in params])
    split = gpu_states8([p.clone() for p in params])
    host = host_states8([u16(p) for p in params])
    plan = sharding.plan([p.numel() for p in params], world)
    for step in range(1, 4):
        grads = W.make_grads(wl, step, cuda_device)
        hd = hp_for(wl, step)
        h = q8.hparams(**hd, exact=1)
        for a, b, c, g in zip(whole, split, host, grads):
            a.grad = g
            b.grad = g
            c.grad[:] = u16(g)
        q8.adamw8bit_sr_step(whole, h)
        for rank in range(world):
            q8.adamw8bit_sr_step(sharding.shard(split, world, rank), h)
            for sl in plan[rank]:
                hs = host_slice8(host[sl.tensor], sl)
                if hs.m_codes is not None:
                    o.adamw8bit_tensor(hs, sl.philox_offset, o.hparams(**hd))
                else:
                    o.adamw32_tensor(hs, sl.philox_offset, o.hparams(**hd))
            torch.cuda.synchronize()
            for sl in plan[rank]:
                compare_slice8(split[sl.tensor], host[sl.tensor], sl,
                               "rank %d of %d, tensor %d, step %d" % (rank, world, sl.tensor, step))
    torch.cuda.synchronize()
    for a, b in zip(whole, split):
        assert torch.equal(a.param, b.param)
        if a.m_codes is not None:
            assert torch.equal(a.m_codes, b.m_codes) and torch.equal(a.v_codes, b.v_codes)
            assert torch.equal(a.m_absmax, b.m_absmax) and torch.equal(a.v_absmax, b.v_absmax)
        else:
            assert torch.equal(a.m32, b.m32) and torch.equal(a.v32, b.v32)


@pytest.mark.parametrize("world", [3, 8])
def test_sharded_fast_step_equals_unsharded(cuda_device, world):
    """The fast mode shards like the bit-exact one: each element's result
    depends only on that element (and the cancellation check on its own pair),
    so N ranks' block-aligned slices with global Philox offsets give the
    unsharded fast step's bits."""
    from bit_blockwise_adamw_gb300 import sharding
    wl = W.custom("shard", [2048 * 50 + 7, 300, 4096, 2048 * 9, 1000, 65536 + 24], steps=3, data_seed=84)
    params = W.init_params(wl, cuda_device)
    whole = gpu_states8([p.clone() for p in params])
    split = gpu_states8([p.clone() for p in params])
    for step in range(1, 4):
        grads = W.make_grads(wl, step, cuda_device)
        h = q8.hparams(**hp_for(wl, step), exact=0)
        for a, b, g in zip(whole, split, grads):
            a.grad = g
            b.grad = g
        q8.adamw8bit_sr_step(whole, h)
        for rank in range(world):
            q8.adamw8bit_sr_step(sharding.shard(split, world, rank), h)
        torch.cuda.synchronize()
        for a, b in zip(whole, split):
            for f in ("param", "m_codes", "v_codes", "m_absmax", "v_absmax", "m32", "v32"):
                x, y = getattr(a, f), getattr(b, f)
                assert x is None or torch.equal(x.view(torch.uint8), y.view(torch.uint8)), (f, step)


def test_packed_sqrt_division_guard_boundaries(cuda_device):
    """Blocks whose moments straddle the bounds of the packed exact square root
    and division (|m| around 2^-90 and 2^26, v around 2^-100 and 2^40), so that
    within one warp some threads take the packed path and others the IEEE one;
    every result equals the oracle's, which uses IEEE sqrt and division only."""
    blocks = [(2.0 ** 27, 1.0), (2.0 ** 25, 2.0 ** 41), (2.0 ** -80, 1e-6), (1e-3, 2.0 ** -95),
              (2.0 ** -88, 2.0 ** -98), (3.0, 2.0 ** 39), (1e-4, 1e-9), (2.0 ** 20, 2.0 ** 39.9)]
    nb = len(blocks)
    n = nb * 2048
    rng = np.random.default_rng(86)
    p = (np.asarray(rng.standard_normal(n) * 0.02, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    mc = rng.integers(0, 255, n).astype(np.uint8)
    vc = rng.integers(0, 256, n).astype(np.uint8)
    ma = np.array([b[0] for b in blocks], np.float32)
    va = np.array([b[1] for b in blocks], np.float32)
    host = o.State8(p.copy(), np.zeros(n, np.uint16), mc.copy(), vc.copy(), ma.copy(), va.copy())
    dev = cuda_device
    gpu = q8.Tensor8(torch.from_numpy(p.view(np.int16)).to(dev).view(torch.bfloat16),
                     torch.zeros(n, dtype=torch.bfloat16, device=dev),
                     torch.from_numpy(mc).to(dev), torch.from_numpy(vc).to(dev),
                     torch.from_numpy(ma).to(dev), torch.from_numpy(va).to(dev))
    for step in range(1, 4):
        g = (np.asarray(rng.standard_normal(n) * 10.0 ** rng.uniform(-12, 2, n), np.float32)
             .view(np.uint32) >> 16).astype(np.uint16)
        host.grad = g
        gpu.grad = torch.from_numpy(g.view(np.int16)).to(dev).view(torch.bfloat16)
        h = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=step, seed=21, sr=1)
        q8.adamw8bit_sr_step([gpu], q8.hparams(**h, exact=1))
        o.adamw8bit_sr_step([host], o.hparams(**h))
        torch.cuda.synchronize()
        compare_state8(gpu, host, "step %d" % step)


def test_bf16_state_guard_boundaries(cuda_device):
    """BF16 state with moments spread over the bounds of the packed exact
    square root and division (|m| from 2^-100 to 2^30, v from 2^-110 to 2^45,
    zeros included): both paths agree with the oracle bit for bit."""
    n = 64 * 1024 + 40
    rng = np.random.default_rng(87)

    def bf(x):
        return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    p = bf(rng.standard_normal(n) * 0.02)
    m = bf(rng.choice([-1.0, 1.0], n) * 2.0 ** rng.uniform(-100, 30, n))
    v = bf(2.0 ** rng.uniform(-110, 45, n))
    m[::97] = 0
    v[::89] = 0
    host = o.State16(p.copy(), np.zeros(n, np.uint16), m.copy(), v.copy())
    dev = cuda_device
    t = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    gpu = q8.Tensor16(t(p), t(np.zeros(n, np.uint16)), t(m), t(v))
    for step in range(1, 4):
        g = bf(rng.standard_normal(n) * 10.0 ** rng.uniform(-12, 2, n))
        host.grad = g
        gpu.grad = t(g)
        h = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=step, seed=22, sr=1)
        q8.adamw_bf16_sr_step([gpu], q8.hparams(**h, exact=1))
        o.adamw_bf16_sr_step([host], o.hparams(**h))
        torch.cuda.synchronize()
        for name, a, b in (("param", gpu.param, host.param), ("m", gpu.m, host.m), ("v", gpu.v, host.v)):
            np.testing.assert_array_equal(u16(a), b, err_msg="%s step %d" % (name, step))
