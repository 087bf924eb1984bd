#!/usr/bin/env python
"""Benchmark of the fused 8-bit blockwise AdamW + stochastic-rounding step.

One "step" is one adamw8bit_sr_step call over the whole tensor list of the
workload (default: the GPT-Neo 6.7B-shaped list, 6,658,011,136 bf16 params,
8-bit m/v with per-2048 absmax), with every input resident in HBM.  Inputs
(66.6 GB of traffic per step) are far larger than the 129 MB L2, so no flush
is needed between steps.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain C restatement of the method,
single-threaded) on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fused AdamW8bit+SR step: Gparams/s and HBM GB/s (% of peak), 1 GB300"
UNIT = "Gparams/s"
BLOCK = 2048
NOMINAL_HBM_GBS = 7900.0          # NVIDIA's HBM3e figure for GB300, for context only


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gptneo-6.7b")
    ap.add_argument("--flat", type=int, default=0,
                    help="replace the workload by one flat tensor of this many params (profiling)")
    ap.add_argument("--flat-state", default="8bit", choices=["8bit", "bf16"],
                    help="optimizer state of the --flat tensor")
    ap.add_argument("--rounding", default="stochastic", choices=["stochastic", "nearest"],
                    help="bf16 writes: stochastic rounding (the method) or round-to-nearest-even")
    ap.add_argument("--optimizer", default="adamw", choices=["adamw", "momentum", "lion"],
                    help="8-bit-state optimizer of the step (adamw is the headline)")
    ap.add_argument("--exact", action="store_true",
                    help="AdamW in the bit-exact mode (correctly rounded square root and division) instead of "
                         "the fast mode; the other mode is timed in the secondary entries either way")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the BF16-state, Momentum and Lion timings that follow the headline")
    ap.add_argument("--secondary-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-blocks", type=int, default=100000,
                    help="2048-blocks in the oracle's single-core timed sample (about 20 s on one core)")
    ap.add_argument("--cpu-blocks-per-proc", type=int, default=6000,
                    help="2048-blocks per process in the oracle's block-parallel timing")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def workload(args):
    from bit_blockwise_adamw_gb300 import workloads as W
    if args.flat:
        return W.custom("flat-%d-%s" % (args.flat, args.flat_state), [args.flat], steps=args.steps,
                        grad_std=1e-4, outlier_rate=1e-4, outlier_factor=1000.0,
                        hp=dict(lr=6e-4, weight_decay=0.1), data_seed=1003, state=args.flat_state)
    return W.WORKLOADS[args.workload]


def algorithmic_bytes(wl, moments=2):
    """Bytes the step must move: 8-bit path 10 B/param (grad 2, param 2+2,
    codes 1+1 each way) + 16 B per block (two absmax read and written);
    fp32-state path 22 B/param; BF16-state path 14 B/param.  With one moment
    (Momentum, Lion): 8 B/param + 8 B/block, fp32 state 14 B/param."""
    total = 0
    for t in wl.tensors:
        if wl.state == "bf16":
            total += 14 * t.numel
        elif t.numel >= 4096:
            total += (6 + 2 * moments) * t.numel + 8 * moments * ((t.numel + BLOCK - 1) // BLOCK)
        else:
            total += (6 + 8 * moments) * t.numel
    return total


def launches_per_step(wl):
    """Kernel launches of one step: one per chunk of up to 448 tensors, plus,
    on the 8-bit path, one tail launch for a chunk holding a tensor whose
    length is not a multiple of 2048."""
    per = 448
    if wl.state == "bf16":
        return (len(wl.tensors) + per - 1) // per
    big = [t.numel for t in wl.tensors if t.numel >= 4096]
    n_small = sum(1 for t in wl.tensors if 0 < t.numel < 4096)
    chunks = [big[i:i + per] for i in range(0, len(big), per)]
    tails = sum(1 for c in chunks if any(n % BLOCK for n in c))
    return len(chunks) + tails + (n_small + per - 1) // per


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        busy = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(busy or sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def traffic_per_launch(kernel, units):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    scaled to `units` params, or None if the kernel source changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    h = hashlib.sha256()
    for rel in d["sources"]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != d["sources_sha256"]:
        return None
    return d["dram_bytes_per_param"] * units


# ---------------------------------------------------------------- CPU oracle

def sample_runs(wl, nblocks, rng, run_blocks=512):
    """The oracle sample's layout: (tensor index, first block, blocks) runs of
    consecutive full 2048-blocks, tensors drawn in proportion to their size
    among those on the 8-bit path (all of them for BF16 state), `nblocks`
    blocks in all."""
    bigs = [i for i, t in enumerate(wl.tensors) if t.numel >= 4096 or wl.state == "bf16"]
    sizes = np.array([wl.tensors[i].numel for i in bigs], np.float64)
    runs, left = [], nblocks
    while left > 0:
        i = bigs[rng.choice(len(bigs), p=sizes / sizes.sum())]
        full = max(1, wl.tensors[i].numel // BLOCK)
        n = min(run_blocks, left, full)
        runs.append((i, int(rng.integers(0, full - n + 1)), n))
        left -= n
    return runs


def _oracle_sample(wl, nblocks, seed, run_blocks=512):
    """A seeded sample of the workload's 2048-blocks as oracle states, in runs
    of up to `run_blocks` consecutive full blocks of one tensor (so that the
    oracle's per-call set-up, its codebooks and midpoints, weighs as little as
    in a whole-tensor call), and a function that runs one step of the oracle
    over them with each run's global Philox offset; returns (params, run)."""
    import oracle as o
    from bit_blockwise_adamw_gb300 import workloads as W
    rng = np.random.default_rng(seed)
    offs = W.philox_offsets(wl)
    # inputs of the sample: N(0, 0.02) params and the workload's grad law
    gen = torch.Generator().manual_seed(seed)

    def bits(x):
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    h = dict(wl.hp)
    hp = o.hparams(lr=h["lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["eps"],
                   weight_decay=h["weight_decay"], step=1, seed=wl.philox_seed)
    states, e0 = [], []
    for i, b0, n in sample_runs(wl, nblocks, rng, run_blocks):
        p = bits(torch.randn(n * BLOCK, generator=gen) * 0.02)
        g = bits(torch.randn(n * BLOCK, generator=gen) * wl.grad_std)
        if wl.state == "bf16":
            z = np.zeros(n * BLOCK, np.uint16)
            states.append(o.State16(p, g, z, z.copy()))
        else:
            states.append(o.State8.zeros(p, g, eight_bit=True))
        e0.append(offs[i] + b0 * BLOCK)
    one = o.adamw_bf16_tensor if wl.state == "bf16" else o.adamw8bit_tensor

    def run():
        for st, e in zip(states, e0):
            one(st, e, hp)
    return nblocks * BLOCK, run


def oracle_flat1m_time(device):
    """Time the oracle (single-threaded C) over the whole flat 1,048,576-param
    workload, all its steps (fresh gradients each step, made on the GPU and
    copied to the host before the clock starts); returns (param-steps, seconds)."""
    import oracle as o
    from bit_blockwise_adamw_gb300 import workloads as W
    wl = W.WORKLOADS["flat-1m"]
    params = [p.view(torch.int16).cpu().numpy().view(np.uint16) for p in W.init_params(wl, device)]
    grads = [[g.view(torch.int16).cpu().numpy().view(np.uint16) for g in W.make_grads(wl, t, device)]
             for t in range(1, wl.steps + 1)]
    states = [o.State8.zeros(p.copy(), np.zeros_like(p)) for p in params]
    h = dict(wl.hp)
    dt = 0.0
    for t in range(1, wl.steps + 1):
        for st, g in zip(states, grads[t - 1]):
            st.grad = g
        hp = o.hparams(lr=h["lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["eps"],
                       weight_decay=h["weight_decay"], step=t, seed=wl.philox_seed)
        t0 = time.perf_counter()
        o.adamw8bit_sr_step(states, hp)
        dt += time.perf_counter() - t0
    return sum(p.size for p in params) * wl.steps, dt


def oracle_sample_time(wl, nblocks, seed=0):
    """Time the oracle (single-threaded C) on a seeded sample of the
    workload's 2048-blocks for one step; returns (params, seconds)."""
    n, run = _oracle_sample(wl, nblocks, seed)
    t0 = time.perf_counter()
    run()
    return n, time.perf_counter() - t0


def _oracle_proc(wl, nblocks, seed, barrier, results):
    """One process of the block-parallel timing: build its own seeded share of
    the sample, wait for the others, then time its oracle calls."""
    n, run = _oracle_sample(wl, nblocks, seed)
    barrier.wait()
    t0 = time.perf_counter()
    run()
    results.put((n, t0, time.perf_counter()))


def oracle_parallel_time(wl, nblocks_per_proc, procs):
    """The same oracle, block-parallel: `procs` spawned processes (blocks are
    independent), each with its own seeded sample, started together.
    Returns (params, wall seconds from the first start to the last end)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(procs), ctx.Queue()
    ps = [ctx.Process(target=_oracle_proc, args=(wl, nblocks_per_proc, 100 + i, barrier, results))
          for i in range(procs)]
    for q in ps:
        q.start()
    got = [results.get(timeout=600) for _ in ps]
    for q in ps:
        q.join()
    return sum(r[0] for r in got), max(r[2] for r in got) - min(r[1] for r in got)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = workload(args)
    # each step: a bounded sample of the workload (bounded so K+W steps stay within minutes)
    nblocks = max(64, min(args.cpu_blocks, 2000))
    times = []
    units = 0
    for i in range(args.warmup + args.steps):
        n, dt = oracle_sample_time(wl, nblocks, seed=i)
        if i >= args.warmup:
            times.append(dt)
            units += n
    total = sum(times)
    value = units / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": wl.name, "sample_blocks_per_step": nblocks},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "%d seeded 2048-blocks of %s per step in runs of up to 512 consecutive blocks, one step each" % (nblocks, wl.name)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # one rank per node compiles (a no-op when the library is current); the
    # others wait for it instead of racing on the same build directory
    from bit_blockwise_adamw_gb300 import build as B
    if local == 0:
        B.build()
    barrier()
    import bit_blockwise_adamw_gb300 as q8
    from bit_blockwise_adamw_gb300 import workloads as W

    wl = workload(args)
    q8.q8_prepare_device()
    params = W.init_params(wl, device)
    grads = W.make_grads(wl, 1, device)
    moments = 2 if args.optimizer == "adamw" else 1
    if wl.state == "bf16":
        states = [q8.Tensor16(p, g, torch.zeros_like(p), torch.zeros_like(p)) for p, g in zip(params, grads)]
        packed = q8.pack_tensor16(states)
        step_fn = q8.adamw_bf16_sr_step
    else:
        states = [q8.Tensor8.zeros_like(p, g, moments=moments) for p, g in zip(params, grads)]
        packed = q8.pack_tensor8(states)
        step_fn = {"adamw": q8.adamw8bit_sr_step, "momentum": q8.momentum8bit_sr_step,
                   "lion": q8.lion8bit_sr_step}[args.optimizer]
    numel = wl.numel
    h = dict(wl.hp)

    sr = 1 if args.rounding == "stochastic" else 0

    def hp(t):
        if args.optimizer == "momentum":
            return q8.momentum_hparams(lr=h["lr"], momentum=h["beta1"], weight_decay=h["weight_decay"],
                                       step=t, seed=wl.philox_seed, sr=sr)
        if args.optimizer == "lion":
            return q8.lion_hparams(lr=h["lr"], beta1=h["beta1"], beta2=0.99, weight_decay=h["weight_decay"],
                                   step=t, seed=wl.philox_seed, sr=sr)
        return q8.hparams(lr=h["lr"], beta1=h["beta1"], beta2=h["beta2"], eps=h["eps"],
                          weight_decay=h["weight_decay"], step=t, seed=wl.philox_seed, sr=sr,
                          exact=int(args.exact))

    stream = torch.cuda.current_stream(device)
    t = 0
    for _ in range(args.warmup):
        t += 1
        step_fn(packed, hp(t), stream)
    torch.cuda.synchronize(device)

    # timed region: K steps, one event pair per step on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize(device)
    start.record(stream)
    for k in range(args.steps):
        t += 1
        ev[k][0].record(stream)
        step_fn(packed, hp(t), stream)
        ev[k][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    clock_info = clocks.stop()
    total_ms = start.elapsed_time(stop)
    per = [a.elapsed_time(b) for a, b in ev]
    if world > 1:
        tt = torch.tensor([total_ms], device=device)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(tt.item())
    ms_per_step = total_ms / args.steps
    value = world * numel * args.steps / (total_ms / 1e3) / 1e9

    # roofline of the dominant kernel (the fused step kernel: one launch per step here)
    peak, peak_kind = load_peaks()
    abytes = algorithmic_bytes(wl, moments)
    nl = launches_per_step(wl)
    mean_ms = statistics.mean(per)
    achieved = abytes / (mean_ms / 1e3) / 1e9
    kernel = "step16_kernel" if wl.state == "bf16" else ("step8_kernel" if moments == 2 else "step1_kernel")
    traffic = traffic_per_launch(kernel, numel / nl) if nl == 1 else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": kernel,
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                "algorithmic_bytes_per_launch": abytes / nl, "peak_source": peak_kind,
                "median_ms_per_step": statistics.median(per), "min_ms_per_step": min(per)}

    # the other steps of the path, timed the same way in the same run: the
    # BF16-state step on its GPT-Neo 2.7B list, 8-bit Momentum and Lion on the
    # headline's 6.7B list (their one state is the headline's m codes)
    secondary = None
    if not args.no_secondary and not args.flat and args.workload == "gptneo-6.7b" and args.optimizer == "adamw":
        secondary = run_secondary(args, wl, states, peak, device, world, barrier)

    # end to end through the public API: grads in from pinned host memory,
    # step, updated params back to pinned host memory, every step
    e2e = None
    if not args.no_e2e and args.optimizer == "adamw":
        e2e = run_e2e(args, wl, states, step_fn, hp, t, device, world, barrier)
        t += args.e2e_steps + 3

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and args.optimizer == "adamw":
        n, dt = oracle_sample_time(wl, args.cpu_blocks)
        cpu = {"value": n / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "%d seeded 2048-blocks (%d params) of %s in runs of up to 512 consecutive blocks, one step, single-threaded C oracle"
                         % (args.cpu_blocks, n, wl.name)}
        n, dt = oracle_flat1m_time(device)
        cpu["flat_1m"] = {"value": n / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
                          "sample": "the whole flat-1m workload (1,048,576 params), all %d steps, single-threaded C oracle"
                                    % (n // 1048576)}
        procs = len(os.sched_getaffinity(0))
        if procs > 1:
            per = max(1, args.cpu_blocks_per_proc)
            n, dt = oracle_parallel_time(wl, per, procs)
            cpu["block_parallel"] = {
                "value": n / dt / 1e9, "unit": UNIT, "cores": procs, "kind": "oracle",
                "sample": "%d processes x %d seeded 2048-blocks (%d params) of %s in runs of up to 512 consecutive blocks, one step each, started together"
                          % (procs, per, n, wl.name)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "storage_dtype": "bf16+u8" if wl.state == "8bit" else "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "optimizer": args.optimizer, "rounding": args.rounding,
                       "mode": ("exact" if args.exact else "fast") if args.optimizer == "adamw" else "exact",
                       "params": numel, "tensors": len(wl.tensors),
                       "blocks": wl.blocks(), "state": wl.state,
                       "bytes_per_step": abytes, "gbs": abytes / (ms_per_step / 1e3) / 1e9,
                       "l2": "inputs larger than L2 (%.1f GB moved per step, no flush)" % (abytes / 1e9),
                       "parallelism": "replicas x%d (each GPU steps its own full list)" % world},
            "roofline": roofline, "secondary": secondary, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": nl * args.steps, "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _time_steps(fn, steps, warmup, stream, device, barrier):
    """Warm-up, then `steps` calls of fn(t) with one event pair per call on
    the launching stream; returns the per-call milliseconds."""
    t = 0
    for _ in range(warmup):
        t += 1
        fn(t)
    torch.cuda.synchronize(device)
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for k in range(steps):
        t += 1
        ev[k][0].record(stream)
        fn(t)
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    barrier()
    return [a.elapsed_time(b) for a, b in ev]


def run_secondary(args, wl8, states8, peak, device, world, barrier):
    """The headline's 8-bit AdamW step in its other mode (bit-exact or fast),
    BF16-state AdamW on the GPT-Neo 2.7B list (in both modes), 8-bit
    Momentum and 8-bit Lion on the 6.7B list (using the headline's parameters,
    gradients and state), each with the headline's warm-up and events, one
    launch per step.  Per entry: ms/step, Gparams/s, algorithmic GB/s and the
    fraction of the measured HBM peak."""
    import bit_blockwise_adamw_gb300 as q8
    from bit_blockwise_adamw_gb300 import workloads as W
    stream = torch.cuda.current_stream(device)
    out = {}
    h8 = dict(wl8.hp)

    def entry(name, wl, kernel, moments, per, nl):
        ms = statistics.mean(per)
        ab = algorithmic_bytes(wl, moments)
        gbs = ab / (ms / 1e3) / 1e9
        out[name] = {"workload": wl.name, "kernel": kernel, "ms_per_step": ms,
                     "median_ms_per_step": statistics.median(per), "steps": len(per),
                     "value": world * wl.numel / (ms / 1e3) / 1e9, "unit": UNIT,
                     "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
                     "algorithmic_bytes_per_launch": ab / nl,
                     "traffic": traffic_per_launch(kernel, wl.numel / nl) if nl == 1 else None}

    # the headline step in the other mode, on the headline's state
    other = 0 if args.exact else 1
    packed8 = q8.pack_tensor8(states8)
    per = _time_steps(lambda t: q8.adamw8bit_sr_step(packed8, q8.hparams(
        lr=h8["lr"], beta1=h8["beta1"], beta2=h8["beta2"], eps=h8["eps"], weight_decay=h8["weight_decay"],
        step=t, seed=wl8.philox_seed, exact=other), stream), args.secondary_steps, args.warmup, stream, device,
        barrier)
    entry("adamw8bit_exact" if other else "adamw8bit_fast", wl8, "step8_kernel", 2, per, launches_per_step(wl8))
    del packed8

    # one-state steps on the 6.7B list: the m codes and absmax of the headline state
    one = [q8.Tensor8(s.param, s.grad, m_codes=s.m_codes, m_absmax=s.m_absmax) for s in states8]
    packed1 = q8.pack_tensor8(one)
    nl1 = launches_per_step(wl8)
    per = _time_steps(lambda t: q8.momentum8bit_sr_step(packed1, q8.momentum_hparams(
        lr=h8["lr"], momentum=h8["beta1"], weight_decay=h8["weight_decay"], step=t, seed=wl8.philox_seed), stream),
        args.secondary_steps, args.warmup, stream, device, barrier)
    entry("momentum8bit", wl8, "step1_kernel", 1, per, nl1)
    per = _time_steps(lambda t: q8.lion8bit_sr_step(packed1, q8.lion_hparams(
        lr=h8["lr"] / 10, beta1=h8["beta1"], beta2=0.99, weight_decay=h8["weight_decay"], step=t,
        seed=wl8.philox_seed), stream), args.secondary_steps, args.warmup, stream, device, barrier)
    entry("lion8bit", wl8, "step1_kernel", 1, per, nl1)
    del one, packed1

    # the BF16-state step on its own (GPT-Neo 2.7B) list
    wl16 = W.WORKLOADS["gptneo-2.7b-bf16"]
    p16 = W.init_params(wl16, device)
    g16 = W.make_grads(wl16, 1, device)
    st16 = [q8.Tensor16(p, g, torch.zeros_like(p), torch.zeros_like(p)) for p, g in zip(p16, g16)]
    packed16 = q8.pack_tensor16(st16)
    h16 = dict(wl16.hp)
    per = _time_steps(lambda t: q8.adamw_bf16_sr_step(packed16, q8.hparams(
        lr=h16["lr"], beta1=h16["beta1"], beta2=h16["beta2"], eps=h16["eps"], weight_decay=h16["weight_decay"],
        step=t, seed=wl16.philox_seed, exact=int(args.exact)), stream), args.secondary_steps, args.warmup, stream,
        device, barrier)
    entry("adamw_bf16", wl16, "step16_kernel", 2, per, launches_per_step(wl16))
    per = _time_steps(lambda t: q8.adamw_bf16_sr_step(packed16, q8.hparams(
        lr=h16["lr"], beta1=h16["beta1"], beta2=h16["beta2"], eps=h16["eps"], weight_decay=h16["weight_decay"],
        step=t, seed=wl16.philox_seed, exact=other), stream), args.secondary_steps, args.warmup, stream,
        device, barrier)
    entry("adamw_bf16_exact" if other else "adamw_bf16_fast", wl16, "step16_kernel", 2, per, launches_per_step(wl16))
    del st16, packed16, p16, g16
    torch.cuda.empty_cache()
    return out


def run_e2e(args, wl, states, step_fn, hp, t, device, world, barrier):
    """Per step: H2D copy of this step's grads from pinned host memory, the
    step through the C ABI, D2H copy of the updated params into pinned host
    memory.  The list is cut into chunks (explicit Philox offsets keep the
    bits identical to one call) so the copies of one chunk overlap the step
    of another.  Two copy schedules: "duplex" (H2D and D2H on their own
    streams, running at once) and "serial" (both in order on one copy stream,
    one chunk's grads ahead of the compute stream).  Which is faster depends
    on the host link: concurrent H2D + D2H reached 343 GB/s on one GB300 machine
    and 99 GB/s on another, against about 200 GB/s one direction at a time.
    Two untimed steps of each pick the schedule for the timed steps."""
    import bit_blockwise_adamw_gb300 as q8
    from bit_blockwise_adamw_gb300 import workloads as W
    offs = W.philox_offsets(wl)
    for s, off in zip(states, offs):
        s.philox_offset = off
    nchunks = min(8, len(states))
    bounds = np.linspace(0, len(states), nchunks + 1).astype(int)
    chunks = [list(range(bounds[c], bounds[c + 1])) for c in range(nchunks) if bounds[c + 1] > bounds[c]]
    host_g = [torch.empty(s.param.numel(), dtype=torch.bfloat16, pin_memory=True) for s in states]
    host_p = [torch.empty(s.param.numel(), dtype=torch.bfloat16, pin_memory=True) for s in states]
    for hg, s in zip(host_g, states):
        hg.copy_(s.grad)
    packs = [(q8.pack_tensor16 if wl.state == "bf16" else q8.pack_tensor8)([states[i] for i in c]) for c in chunks]
    s_in, s_out, s_cmp = (torch.cuda.Stream(device) for _ in range(3))

    def record(stream):
        e = torch.cuda.Event()
        e.record(stream)
        return e

    def grads_in(c, stream):
        with torch.cuda.stream(stream):
            for i in chunks[c]:
                states[i].grad.copy_(host_g[i], non_blocking=True)
        return record(stream)

    def params_out(c, stream):
        with torch.cuda.stream(stream):
            for i in chunks[c]:
                host_p[i].copy_(states[i].param, non_blocking=True)

    def step_serial(tt):
        e_in = grads_in(0, s_in)
        for c, pk in enumerate(packs):
            s_cmp.wait_event(e_in)
            step_fn(pk, hp(tt), s_cmp)
            e_c = record(s_cmp)
            if c + 1 < len(packs):
                e_in = grads_in(c + 1, s_in)
            s_in.wait_event(e_c)
            params_out(c, s_in)

    done_cmp = [None] * len(packs)              # per chunk, from the previous step
    done_out = [None] * len(packs)

    def step_duplex(tt):
        for c, pk in enumerate(packs):
            if done_cmp[c] is not None:
                s_in.wait_event(done_cmp[c])    # the last step has read these grads
            e_in = grads_in(c, s_in)
            s_cmp.wait_event(e_in)
            if done_out[c] is not None:
                s_cmp.wait_event(done_out[c])   # the last step's params are out
            step_fn(pk, hp(tt), s_cmp)
            done_cmp[c] = record(s_cmp)
            s_out.wait_event(done_cmp[c])
            params_out(c, s_out)
            done_out[c] = record(s_out)

    def timed(fn, first, k):
        torch.cuda.synchronize(device)
        barrier()
        t0 = time.perf_counter()
        for j in range(k):
            fn(first + j)
        torch.cuda.synchronize(device)
        barrier()
        return time.perf_counter() - t0

    # Each trial runs two back-to-back steps, so that the copies of one step
    # overlap those of the next as in the timed run (a single step from idle
    # never runs both directions at once for long).
    tt = t + 1
    timed(step_duplex, tt, 1)                  # warm-up
    d_duplex = timed(step_duplex, tt + 1, 2) / 2
    d_serial = timed(step_serial, tt + 3, 2) / 2
    if world > 1:
        tt2 = torch.tensor([d_duplex, d_serial], device=device)
        torch.distributed.all_reduce(tt2, op=torch.distributed.ReduceOp.MAX)
        d_duplex, d_serial = (float(x) for x in tt2.tolist())
    mode, fn = ("duplex", step_duplex) if d_duplex <= d_serial else ("serial", step_serial)
    dt = timed(fn, tt + 5, args.e2e_steps)
    if world > 1:
        tt3 = torch.tensor([dt], device=device)
        torch.distributed.all_reduce(tt3, op=torch.distributed.ReduceOp.MAX)
        dt = float(tt3.item())
    nb = 2 * wl.numel
    for s in states:
        s.philox_offset = -1
    return {"value": world * wl.numel * args.e2e_steps / dt / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": nb, "d2h_bytes_per_step": nb, "steps": args.e2e_steps,
            "ms_per_step": 1e3 * dt / args.e2e_steps, "schedule": mode,
            "trial_ms": {"duplex": 1e3 * d_duplex, "serial": 1e3 * d_serial},
            "note": "pinned host grads in, params out, %d chunks, %s copy schedule" % (len(chunks), mode)}


if __name__ == "__main__":
    sys.exit(main())
