"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, replay the same inputs through the oracle, compare element by
element.  Inputs come from bit_blockwise_adamw_gb300.workloads (seeded torch
generators); no expected value is taken from the CUDA path."""
import multiprocessing as mp

import numpy as np
import torch

import bit_blockwise_adamw_gb300 as q8
from bit_blockwise_adamw_gb300 import workloads as W
import oracle as o

BLOCK = 2048


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def hp_for(wl, step, sr=1):
    h = wl.hp
    return dict(lr=h["lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["eps"],
                weight_decay=h["weight_decay"], step=step, seed=wl.philox_seed, sr=sr)


def shift16(t):
    """A copy of the 1-D tensor t whose data starts 16 bytes past a 32-byte
    boundary (allowed by the ABI's 16-byte rule, but not 32-byte aligned)."""
    buf = torch.empty(t.numel() + 16 // t.element_size(), dtype=t.dtype, device=t.device)
    v = buf[16 // t.element_size():]
    v.copy_(t)
    assert v.data_ptr() % 32 == 16
    return v


def gpu_states8(params, offsets=None):
    offsets = offsets or [-1] * len(params)
    return [q8.Tensor8.zeros_like(p, None, philox_offset=off) for p, off in zip(params, offsets)]


def host_states8(params_host, offsets=None):
    offsets = offsets or [-1] * len(params_host)
    return [o.State8.zeros(p.copy(), np.zeros_like(p), philox_offset=off)
            for p, off in zip(params_host, offsets)]


# The fast mode (exact=0: approximate square root and reciprocal in the
# parameter update) against the oracle, at the tolerance the target states
# for floating-point results: BF16 parameters bit-exact on at least 99.9 % of
# elements and within one BF16 ulp on the rest, for a step from identical
# inputs.  Codes, absmax, fp32 state and BF16 moments do not depend on the
# approximation and stay bit-exact.  Along a whole run a parameter that once
# differed by an ulp keeps that small absolute offset, which a later update
# that nearly cancels it can make many ulps of the small result; whole runs
# are therefore held to the share alone (ParamTolerance(ulps=None)).
PARAM_EXACT_SHARE = 0.999


def bf16_ulps(a, b):
    """Distance between arrays of BF16 bit patterns in units in the last
    place, along the ordered line of BF16 values (+0 and -0 coincide)."""
    def key(x):
        x = np.asarray(x).astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(key(a) - key(b))


class ParamTolerance:
    """Tally of the BF16 parameters compared in the fast mode: every one within
    `ulps` of the oracle's (no bound for ulps=None), and (check()) at most
    0.1 % of them different."""

    def __init__(self, ulps=1):
        self.ulps = ulps
        self.n = 0
        self.diff = 0
        self.max_ulps = 0

    def add(self, got, want, where=""):
        d = bf16_ulps(got, want)
        self.n += d.size
        self.diff += int(np.count_nonzero(d))
        if d.size:
            worst = int(d.max())
            self.max_ulps = max(self.max_ulps, worst)
            assert self.ulps is None or worst <= self.ulps, \
                "param %s: %d ulps from the oracle at %d" % (where, worst, int(d.argmax()))

    def check(self):
        assert self.diff <= (1.0 - PARAM_EXACT_SHARE) * self.n, \
            "%d of %d parameters differ from the oracle" % (self.diff, self.n)


def compare_state8(gpu, host, where="", tol=None):
    """Comparison of one tensor's parameters and state: bit-exact, or with
    the parameters tallied in `tol` (a ParamTolerance) for the fast mode."""
    if tol is None:
        np.testing.assert_array_equal(u16(gpu.param), host.param, err_msg="param " + where)
    else:
        tol.add(u16(gpu.param), host.param, where)
    if host.m_codes is not None:
        np.testing.assert_array_equal(gpu.m_codes.cpu().numpy(), host.m_codes, err_msg="m codes " + where)
        np.testing.assert_array_equal(gpu.v_codes.cpu().numpy(), host.v_codes, err_msg="v codes " + where)
        np.testing.assert_array_equal(gpu.m_absmax.cpu().numpy().view(np.uint32),
                                      host.m_absmax.view(np.uint32), err_msg="m absmax " + where)
        np.testing.assert_array_equal(gpu.v_absmax.cpu().numpy().view(np.uint32),
                                      host.v_absmax.view(np.uint32), err_msg="v absmax " + where)
    else:
        np.testing.assert_array_equal(gpu.m32.cpu().numpy().view(np.uint32), host.m32.view(np.uint32),
                                      err_msg="m32 " + where)
        np.testing.assert_array_equal(gpu.v32.cpu().numpy().view(np.uint32), host.v32.view(np.uint32),
                                      err_msg="v32 " + where)


def host_slice8(state, sl):
    """Views into a host State8 for one sharding.Slice (block-aligned slice of
    an 8-bit tensor, or a whole small tensor), so that the oracle's in-place
    update of the slice writes into the full host arrays."""
    a, b = sl.start, sl.start + sl.count
    if state.m_codes is None:
        return o.State8(state.param, state.grad, m32=state.m32, v32=state.v32, philox_offset=sl.philox_offset)
    b0, b1 = a // BLOCK, (b + BLOCK - 1) // BLOCK
    opt = lambda x, lo, hi: None if x is None else x[lo:hi]
    return o.State8(state.param[a:b], state.grad[a:b], state.m_codes[a:b], opt(state.v_codes, a, b),
                    state.m_absmax[b0:b1], opt(state.v_absmax, b0, b1), philox_offset=sl.philox_offset)


def compare_slice8(gpu, host, sl, where=""):
    """Bit-exact comparison of one rank's slice (params, codes, absmax or fp32 state)."""
    a, b = sl.start, sl.start + sl.count
    np.testing.assert_array_equal(u16(gpu.param[a:b]), host.param[a:b], err_msg="param " + where)
    if host.m_codes is None:
        np.testing.assert_array_equal(gpu.m32.cpu().numpy().view(np.uint32), host.m32.view(np.uint32),
                                      err_msg="m32 " + where)
        if host.v32 is not None:
            np.testing.assert_array_equal(gpu.v32.cpu().numpy().view(np.uint32), host.v32.view(np.uint32),
                                          err_msg="v32 " + where)
        return
    b0, b1 = a // BLOCK, (b + BLOCK - 1) // BLOCK
    np.testing.assert_array_equal(gpu.m_codes[a:b].cpu().numpy(), host.m_codes[a:b], err_msg="m codes " + where)
    np.testing.assert_array_equal(gpu.m_absmax[b0:b1].cpu().numpy().view(np.uint32),
                                  host.m_absmax[b0:b1].view(np.uint32), err_msg="m absmax " + where)
    if host.v_codes is not None:
        np.testing.assert_array_equal(gpu.v_codes[a:b].cpu().numpy(), host.v_codes[a:b], err_msg="v codes " + where)
        np.testing.assert_array_equal(gpu.v_absmax[b0:b1].cpu().numpy().view(np.uint32),
                                      host.v_absmax[b0:b1].view(np.uint32), err_msg="v absmax " + where)


# ---------------------------------------------------------------- sampled replay
# Each 2048-block's trajectory depends only on its own inputs, so the oracle
# can replay any chosen blocks over all steps.  Workers are started with
# "spawn" (a forked child of a CUDA process can hang).

def _replay8(job):
    """Oracle replay of one 8-bit block: job = (param0, grads[steps], E0, hps)."""
    p0, grads, e0, hps = job
    st = o.State8(p0.copy(), grads[0], np.full(p0.size, o.zero_code(o.SIGNED), np.uint8),
                  np.full(p0.size, o.zero_code(o.UNSIGNED), np.uint8),
                  np.zeros(1, np.float32), np.zeros(1, np.float32))
    for g, h in zip(grads, hps):
        st.grad = g
        o.adamw8bit_tensor(st, e0, o.hparams(**h))
    return st.param, st.m_codes, st.v_codes, st.m_absmax, st.v_absmax


def _replay32(job):
    p0, grads, e0, hps = job
    n = p0.size
    st = o.State8(p0.copy(), grads[0], m32=np.zeros(n, np.float32), v32=np.zeros(n, np.float32))
    for g, h in zip(grads, hps):
        st.grad = g
        o.adamw32_tensor(st, e0, o.hparams(**h))
    return st.param, st.m32, st.v32


def _replay16(job):
    p0, grads, e0, hps = job
    n = p0.size
    st = o.State16(p0.copy(), grads[0], np.zeros(n, np.uint16), np.zeros(n, np.uint16))
    for g, h in zip(grads, hps):
        st.grad = g
        o.adamw_bf16_tensor(st, e0, o.hparams(**h))
    return st.param, st.m, st.v


def _replay1(job):
    """Oracle replay of one block of a one-state step (8-bit m), or of a whole
    small tensor (fp32 m): job = (param0, grads[steps], E0, (opt, hps, eight_bit))."""
    p0, grads, e0, (opt, hps, eight_bit) = job
    st = o.zeros_onestate(p0.copy(), grads[0], eight_bit=eight_bit)
    if eight_bit:
        st.m_absmax = np.zeros(1, np.float32)
    for g, h in zip(grads, hps):
        st.grad = g
        if eight_bit:
            o.onestate8bit_tensor(opt, st, e0, o.hparams(**h))
        else:
            o.onestate32_tensor(opt, st, e0, o.hparams(**h))
    return (st.param, st.m_codes, st.m_absmax) if eight_bit else (st.param, st.m32)


def onestate_hp(opt, wl, step, sr=1):
    """Hyper-parameters of the one-state steps on a workload, as the bench
    times them: Momentum with momentum beta1; Lion with lr/10, beta1 and 0.99;
    the workload's weight decay.  Returned as oracle keyword arguments."""
    h = wl.hp
    if opt == o.MOMENTUM:
        return dict(lr=h["lr"], beta1=h["beta1"], weight_decay=h["weight_decay"], step=step,
                    seed=wl.philox_seed, sr=sr)
    return dict(lr=h["lr"] / 10, beta1=h["beta1"], beta2=0.99, weight_decay=h["weight_decay"], step=step,
                seed=wl.philox_seed, sr=sr)


def oracle_pool(processes=None):
    return mp.get_context("spawn").Pool(processes)


class SampledRun:
    """Run a full-size workload on the GPU while recording the inputs of the
    sampled blocks (and of every small tensor) for an oracle replay."""

    def __init__(self, wl, device, fraction, steps=None, extra_blocks=(), opt=None, exact=True):
        self.wl = wl
        self.exact = exact              # AdamW: the bit-exact mode, or the fast one
        self.tol = None
        self.opt = opt                  # None: AdamW; o.MOMENTUM or o.LION: the one-state step
        self.steps = steps or wl.steps
        self.device = device
        self.picks = sorted(set(W.sample_blocks(wl, fraction)) | set(extra_blocks))
        self.small = wl.small_tensors() if wl.state == "8bit" else []
        self.offsets = W.philox_offsets(wl)
        self.by_tensor = {}
        for i, b in self.picks:
            self.by_tensor.setdefault(i, []).append(b)

    def _gather(self, tensors, conv):
        """Host copies of the sampled blocks of per-element tensors, batched
        into one gather and one copy per tensor."""
        out = {}
        for i, blocks in self.by_tensor.items():
            t = tensors[i]
            nfull = t.numel() // BLOCK
            full = [b for b in blocks if b < nfull]
            if full:
                idx = torch.tensor(full, device=t.device)
                rows = conv(t[:nfull * BLOCK].view(nfull, BLOCK)[idx])
                for j, b in enumerate(full):
                    out[(i, b)] = rows[j]
            for b in blocks:
                if b >= nfull:
                    out[(i, b)] = conv(t[b * BLOCK:])
        return out

    def _slices(self, tensors):
        out = self._gather(tensors, u16)
        for i in self.small:
            out[(i, -1)] = u16(tensors[i])
        return out

    def run(self):
        wl, dev = self.wl, self.device
        params = W.init_params(wl, dev)
        self.p0 = self._slices(params)
        self.grads = []
        self.hps = []
        if self.opt is not None:
            states = [q8.Tensor8.zeros_like(p, None, moments=1) for p in params]
        elif wl.state == "8bit":
            states = gpu_states8(params)
        else:
            states = [q8.Tensor16(p, None, torch.zeros_like(p), torch.zeros_like(p)) for p in params]
        packed = None
        for step in range(1, self.steps + 1):
            grads = W.make_grads(wl, step, dev)
            for s, g in zip(states, grads):
                s.grad = g
            packed = q8.pack_tensor8(states) if wl.state == "8bit" else q8.pack_tensor16(states)
            h = hp_for(wl, step) if self.opt is None else onestate_hp(self.opt, wl, step)
            if self.opt == o.MOMENTUM:
                q8.momentum8bit_sr_step(packed, q8.momentum_hparams(
                    lr=h["lr"], momentum=h["beta1"], weight_decay=h["weight_decay"], step=step, seed=h["seed"]))
            elif self.opt == o.LION:
                q8.lion8bit_sr_step(packed, q8.lion_hparams(
                    lr=h["lr"], beta1=h["beta1"], beta2=h["beta2"], weight_decay=h["weight_decay"], step=step,
                    seed=h["seed"]))
            elif wl.state == "8bit":
                q8.adamw8bit_sr_step(packed, q8.hparams(**h, exact=int(self.exact)))
            else:
                q8.adamw_bf16_sr_step(packed, q8.hparams(**h, exact=int(self.exact)))
            self.grads.append(self._slices(grads))
            self.hps.append(h)
            del grads
        torch.cuda.synchronize()
        self.final = {}
        npy = lambda t: t.cpu().numpy()
        fp = self._gather([s.param for s in states], u16)
        if self.opt is not None:
            fm = self._gather([s.m_codes if s.m_codes is not None else s.param for s in states], npy)
            for i, b in self.picks:
                self.final[(i, b)] = (fp[(i, b)], fm[(i, b)], npy(states[i].m_absmax[b:b + 1]))
            for i in self.small:
                self.final[(i, -1)] = (u16(states[i].param), states[i].m32.cpu().numpy())
        elif wl.state == "8bit":
            fm = self._gather([s.m_codes if s.m_codes is not None else s.param for s in states], npy)
            fv = self._gather([s.v_codes if s.v_codes is not None else s.param for s in states], npy)
            for i, b in self.picks:
                s = states[i]
                self.final[(i, b)] = (fp[(i, b)], fm[(i, b)], fv[(i, b)],
                                      npy(s.m_absmax[b:b + 1]), npy(s.v_absmax[b:b + 1]))
        else:
            fm = self._gather([s.m for s in states], u16)
            fv = self._gather([s.v for s in states], u16)
            for k in self.picks:
                self.final[k] = (fp[k], fm[k], fv[k])
        for i in self.small if self.opt is None else []:
            s = states[i]
            self.final[(i, -1)] = (u16(s.param), s.m32.cpu().numpy(), s.v32.cpu().numpy())
        del states, params
        torch.cuda.empty_cache()

    def jobs(self):
        keys = list(self.picks) + [(i, -1) for i in self.small]
        out = []
        for k in keys:
            i, b = k
            e0 = self.offsets[i] + (b * BLOCK if b >= 0 else 0)
            extra = self.hps if self.opt is None else (self.opt, self.hps, b >= 0)
            out.append((k, (self.p0[k], [g[k] for g in self.grads], e0, extra)))
        return out

    def check(self, pool):
        """Replay every sampled block on the oracle; return the number of
        elements compared.  Raises on the first mismatch."""
        jobs = self.jobs()
        fns = []
        for k, job in jobs:
            if self.opt is not None:
                fns.append(_replay1)
            elif k[1] == -1:
                fns.append(_replay32)
            elif self.wl.state == "8bit":
                fns.append(_replay8)
            else:
                fns.append(_replay16)
        results = [pool.apply_async(f, (job,)) for f, (_, job) in zip(fns, jobs)]
        compared = 0
        tol = None if self.exact or self.opt is not None else ParamTolerance(ulps=None)
        for (k, _), r in zip(jobs, results):
            want = r.get()
            got = self.final[k]
            names = ("param", "m", "v", "m_absmax", "v_absmax") if self.opt is None else ("param", "m", "m_absmax")
            for name, gv, wv in zip(names, got, want):
                gv = np.asarray(gv)
                wv = np.asarray(wv)
                if tol is not None and name == "param":
                    tol.add(gv, wv, "tensor %d block %d" % k)
                    continue
                if gv.dtype == np.float32:
                    gv, wv = gv.view(np.uint32), wv.view(np.uint32)
                if not np.array_equal(gv, wv):
                    bad = np.nonzero(gv != wv)[0]
                    raise AssertionError("%s mismatch in tensor %d block %d: %d of %d differ, first at %d "
                                         "(gpu %r oracle %r)" % (name, k[0], k[1], bad.size, gv.size,
                                                                  bad[0], gv[bad[0]], wv[bad[0]]))
            compared += got[0].size
        if tol is not None:
            tol.check()
            self.tol = tol
        return compared
