"""Block-aligned partition of a tensor list across data-parallel ranks.

"Stochastic Rounding for LLM Training: Theory and Practice" (TL;DR and
abstract) carries SR into distributed training with shared randomness.  Here
every 2048-element block's update depends only on its own inputs and on Philox
draws keyed by the global element index, so a list can be cut at block
boundaries: each rank updates its own slices (with their global Philox
offsets) and the union of the ranks' results is bit-identical to one
unsharded step.  Replicas that each update the whole list draw the same bits
and stay identical without any exchange.

This module is host-side planning plus the one exchange a sharded
(ZeRO-style) data-parallel step needs afterwards: `gather_params` brings every
rank's updated parameter slices to all ranks with one all-gather of a flat
buffer (2 bytes per parameter).  The step itself runs in the library.
"""
from dataclasses import dataclass
from typing import List, Sequence

import torch

BLOCK = 2048
SMALL_NUMEL = 4096


@dataclass(frozen=True)
class Slice:
    tensor: int          # index of the tensor in the list
    start: int           # first element of the slice (a multiple of 2048)
    count: int           # number of elements
    philox_offset: int   # global Philox index of the slice's first element


def _ceil_block(x: int) -> int:
    return -(-x // BLOCK) * BLOCK


def plan(numels: Sequence[int], world: int) -> List[List[Slice]]:
    """Slices each rank updates.  The list is laid end to end (global element
    index = running sum of numel); rank r owns the units that start inside
    [r*total/world, (r+1)*total/world), where a unit is a 2048-block of a
    tensor with at least 4096 elements, or a whole smaller tensor (whose
    fp32 state is not cut).  Consecutive units of one tensor form one slice."""
    if world < 1:
        raise ValueError("world must be >= 1")
    total = sum(numels)
    bounds = [r * total // world for r in range(world + 1)]
    out: List[List[Slice]] = [[] for _ in range(world)]
    g = 0
    for i, n in enumerate(numels):
        if n <= 0:
            continue
        if n < SMALL_NUMEL:
            r = next(r for r in range(world) if bounds[r] <= g < bounds[r + 1])
            out[r].append(Slice(i, 0, n, g))
        else:
            for r in range(world):
                first = _ceil_block(max(0, bounds[r] - g))
                last = min(n, _ceil_block(max(0, bounds[r + 1] - g)))
                if first < last:
                    out[r].append(Slice(i, first, last - first, g + first))
        g += n
    return out


def shard(tensors, world: int, rank: int):
    """This rank's share of a list of Tensor8: block-aligned slices of the
    8-bit tensors and whole small tensors, each with its global offset."""
    numels = [t.param.numel() for t in tensors]
    out = []
    for s in plan(numels, world)[rank]:
        t = tensors[s.tensor]
        if t.m_codes is not None:
            out.append(t.slice(s.start, s.count, s.philox_offset))
        else:
            out.append(type(t)(t.param, t.grad, m32=t.m32, v32=t.v32, philox_offset=s.philox_offset))
    return out


def gather_params(params: Sequence[torch.Tensor], world: int, rank: int, group=None) -> None:
    """After each rank has stepped its `plan(...)[rank]` slices of `params`
    (1-D bf16 tensors, one per list entry, on this rank's device), copy every
    rank's updated slices into every rank's `params`: each rank packs its
    slices end to end into one buffer, padded to the longest rank's length,
    and one all_gather of int32 words over `group` (torch.distributed: NCCL on
    GPUs, gloo on the CPU) exchanges them.  In place; returns when done."""
    import torch.distributed as dist
    shards = plan([p.numel() for p in params], world)
    sizes = [sum(s.count for s in sl) for sl in shards]
    width = max(sizes) if sizes else 0
    if width == 0:
        return
    width += width & 1                  # exchanged as int32 words (gloo has no int16)
    dev = params[0].device
    mine = torch.zeros(width, dtype=torch.int16, device=dev)
    at = 0
    for s in shards[rank]:
        mine[at:at + s.count] = params[s.tensor].view(torch.int16)[s.start:s.start + s.count]
        at += s.count
    bufs = [torch.empty(width, dtype=torch.int16, device=dev) for _ in range(world)]
    dist.all_gather([b.view(torch.int32) for b in bufs], mine.view(torch.int32), group=group)
    for r, sl in enumerate(shards):
        if r == rank:
            continue
        at = 0
        for s in sl:
            params[s.tensor].view(torch.int16)[s.start:s.start + s.count] = bufs[r][at:at + s.count]
            at += s.count
