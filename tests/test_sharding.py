"""Sharded (data-parallel) step: the block-aligned partition covers every
element exactly once with global Philox offsets, and ranks that update only
their slices reproduce the unsharded step bit for bit ("Stochastic Rounding
for LLM Training: Theory and Practice", TL;DR: SR in distributed settings with
shared randomness).  The multi-process checks run as world-size-2 gloo groups
on the CPU, each rank stepping its shard with the oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

from bit_blockwise_adamw_gb300 import sharding as S
import oracle as o

SIZES = [50257 * 8, 300, 4096, 2048 * 7 + 5, 1, 4095, 12345, 8192, 0, 2049]


@pytest.mark.parametrize("world", [1, 2, 3, 5, 8, 64])
def test_plan_covers_each_element_once(world):
    shards = S.plan(SIZES, world)
    assert len(shards) == world
    seen = [np.zeros(n, np.int32) for n in SIZES]
    offs = np.concatenate([[0], np.cumsum(SIZES)[:-1]])
    for rank, slices in enumerate(shards):
        for s in slices:
            n = SIZES[s.tensor]
            seen[s.tensor][s.start:s.start + s.count] += 1
            assert s.philox_offset == offs[s.tensor] + s.start
            if n >= 4096:
                assert s.start % 2048 == 0
                assert s.count % 2048 == 0 or s.start + s.count == n
            else:
                assert s.start == 0 and s.count == n
    assert all(np.all(x == 1) for x in seen)


def test_plan_is_balanced():
    sizes = [2048 * 1000 + 17] * 7 + [1000] * 30
    total = sum(sizes)
    for world in (2, 4, 8):
        loads = [sum(s.count for s in sl) for sl in S.plan(sizes, world)]
        assert sum(loads) == total
        assert max(loads) - min(loads) <= 3 * 2048


def _bf16(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _data(step):
    rng = np.random.default_rng(100 + step)
    params = [_bf16(np.random.default_rng(7).standard_normal(n) * 0.02) for n in SIZES]
    grads = [_bf16(rng.standard_normal(n) * 1e-3) for n in SIZES]
    return params, grads


def _oracle_slices(states, slices):
    out = []
    for s in slices:
        st = states[s.tensor]
        sl = slice(s.start, s.start + s.count)
        if st.m_codes is not None:
            b0, b1 = s.start // 2048, (s.start + s.count + 2047) // 2048
            out.append(o.State8(st.param[sl], st.grad[sl], st.m_codes[sl], st.v_codes[sl],
                                st.m_absmax[b0:b1], st.v_absmax[b0:b1], philox_offset=s.philox_offset))
        else:
            out.append(o.State8(st.param, st.grad, m32=st.m32, v32=st.v32, philox_offset=s.philox_offset))
    return out


def _run(world, rank, steps=3):
    params, _ = _data(0)
    states = [o.State8.zeros(p.copy(), np.zeros_like(p)) for p in params]
    slices = S.plan(SIZES, world)[rank]
    for t in range(1, steps + 1):
        _, grads = _data(t)
        for st, g in zip(states, grads):
            st.grad = g
        mine = _oracle_slices(states, slices)
        o.adamw8bit_sr_step(mine, o.hparams(step=t, seed=11))
        # write the slices back (they are copies: numpy slicing of a 1-D
        # contiguous array is a view, but ascontiguousarray may copy absmax)
        for s, m in zip(slices, mine):
            st = states[s.tensor]
            sl = slice(s.start, s.start + s.count)
            st.param[sl] = m.param
            if st.m_codes is not None:
                b0, b1 = s.start // 2048, (s.start + s.count + 2047) // 2048
                st.m_codes[sl], st.v_codes[sl] = m.m_codes, m.v_codes
                st.m_absmax[b0:b1], st.v_absmax[b0:b1] = m.m_absmax, m.v_absmax
            else:
                st.m32[:], st.v32[:] = m.m32, m.v32
    return states, slices


def test_single_process_shards_equal_unsharded():
    whole, _ = _run(1, 0)
    for world in (2, 3):
        parts = [_run(world, r) for r in range(world)]
        for r, (states, slices) in enumerate(parts):
            for s in slices:
                sl = slice(s.start, s.start + s.count)
                assert np.array_equal(states[s.tensor].param[sl], whole[s.tensor].param[sl])


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _gloo_worker(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        states, slices = _run(world, rank)
        # gather every rank's updated parameter slices on every rank
        mine = [(s.tensor, s.start, states[s.tensor].param[s.start:s.start + s.count].tolist()) for s in slices]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            full = [np.zeros(n, np.uint16) for n in SIZES]
            for part in gathered:
                for t, start, vals in part:
                    full[t][start:start + len(vals)] = vals
            np.savez(os.path.join(result_dir, "sharded.npz"), *full)
        # replicas (each rank steps the whole list) must agree bit for bit
        rep, _ = _run(1, 0)
        digest = torch.tensor([int(np.bitwise_xor.reduce(np.concatenate([s.param for s in rep]).astype(np.int64)))])
        all_d = [torch.zeros_like(digest) for _ in range(world)]
        dist.all_gather(all_d, digest)
        assert all(int(d) == int(digest) for d in all_d)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_sharded_step(tmp_path):
    world = 2
    tmp.spawn(_gloo_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    whole, _ = _run(1, 0)
    got = np.load(os.path.join(tmp_path, "sharded.npz"))
    for i, st in enumerate(whole):
        assert np.array_equal(got["arr_%d" % i], st.param)


def _gather_worker(rank, world, port):
    """Each rank keeps the optimizer state of its own slices only, steps them
    with the oracle, and all-gathers the updated parameters every step: all
    ranks end with the unsharded step's parameters."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        params, _ = _data(0)
        views = [torch.from_numpy(p.view(np.int16)).view(torch.bfloat16) for p in params]
        states = [o.State8.zeros(p, np.zeros_like(p)) for p in params]     # full-size, only own slices used
        slices = S.plan(SIZES, world)[rank]
        for t in range(1, 4):
            _, grads = _data(t)
            for st, g in zip(states, grads):
                st.grad = g
            mine = _oracle_slices(states, slices)
            o.adamw8bit_sr_step(mine, o.hparams(step=t, seed=11))
            for s, m in zip(slices, mine):
                st = states[s.tensor]
                sl = slice(s.start, s.start + s.count)
                st.param[sl] = m.param
                if st.m_codes is not None:
                    b0, b1 = s.start // 2048, (s.start + s.count + 2047) // 2048
                    st.m_codes[sl], st.v_codes[sl] = m.m_codes, m.v_codes
                    st.m_absmax[b0:b1], st.v_absmax[b0:b1] = m.m_absmax, m.v_absmax
                else:
                    st.m32[:], st.v32[:] = m.m32, m.v32
            S.gather_params(views, world, rank)                       # st.param shares memory with views
        whole, _ = _run(1, 0)
        for st, w in zip(states, whole):
            assert np.array_equal(st.param, w.param)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_gloo_three_ranks_sharded_step_with_param_all_gather():
    tmp.spawn(_gather_worker, args=(3, _free_port()), nprocs=3, join=True)
