"""Steps issued from two host threads at once, in a fresh process.

The library keeps per-device state that its first call on a device sets up
(the staged tables and each kernel's persistent grid size).  Here two
threads make their first calls at the same moment, each on its own CUDA
stream and its own tensor list (8-bit AdamW with partial blocks and
fp32-state tensors; BF16-state AdamW; 8-bit Lion), for three steps, and every
result is compared bit for bit with the oracle.  The work runs in a child
process so that the library's caches start cold whatever ran before.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
import numpy as np, torch
import bit_blockwise_adamw_gb300 as q8
from bit_blockwise_adamw_gb300 import workloads as W
import oracle as o
from parity import compare_state8, gpu_states8, host_states8, hp_for, u16

dev = torch.device("cuda:0")
torch.cuda.init()
STEPS = 3
start = threading.Barrier(2)
errors = []

def adamw8(seed, sizes, out):
    wl = W.custom("t%d" % seed, sizes, steps=STEPS, outlier_rate=1e-3, outlier_factor=100.0, data_seed=seed)
    params = W.init_params(wl, dev)
    gpu = gpu_states8(params)
    host = host_states8([u16(p) for p in params])
    stream = torch.cuda.Stream(dev)
    grads = [W.make_grads(wl, t, dev) for t in range(1, STEPS + 1)]
    torch.cuda.synchronize()
    start.wait()
    for t in range(1, STEPS + 1):
        for a, g in zip(gpu, grads[t - 1]):
            a.grad = g
        q8.adamw8bit_sr_step(gpu, q8.hparams(**hp_for(wl, t), exact=1), stream)
    stream.synchronize()
    for t in range(1, STEPS + 1):
        for b, g in zip(host, grads[t - 1]):
            b.grad = u16(g)
        o.adamw8bit_sr_step(host, o.hparams(**hp_for(wl, t)))
    out.append((gpu, host))

def other(seed, out):
    # BF16-state AdamW and 8-bit Lion, each through its own launcher
    n = 2048 * 37 + 100
    wl = W.custom("u%d" % seed, [n], steps=STEPS, data_seed=seed)
    p = W.init_params(wl, dev)[0]
    t16 = q8.Tensor16(p.clone(), None, torch.zeros_like(p), torch.zeros_like(p))
    s16 = o.State16(u16(p), np.zeros(n, np.uint16), np.zeros(n, np.uint16), np.zeros(n, np.uint16))
    t1 = q8.Tensor8.zeros_like(p.clone(), None, moments=1)
    s1 = o.zeros_onestate(u16(p), np.zeros(n, np.uint16))
    stream = torch.cuda.Stream(dev)
    grads = [W.make_grads(wl, t, dev)[0] for t in range(1, STEPS + 1)]
    torch.cuda.synchronize()
    start.wait()
    for t in range(1, STEPS + 1):
        t16.grad = grads[t - 1]
        t1.grad = grads[t - 1]
        q8.adamw_bf16_sr_step([t16], q8.hparams(**hp_for(wl, t), exact=1), stream)
        q8.lion8bit_sr_step([t1], q8.lion_hparams(lr=1e-4, weight_decay=0.1, step=t, seed=3), stream)
    stream.synchronize()
    for t in range(1, STEPS + 1):
        s16.grad = u16(grads[t - 1])
        s1.grad = u16(grads[t - 1])
        o.adamw_bf16_sr_step([s16], o.hparams(**hp_for(wl, t)))
        o.onestate_sr_step(o.LION, [s1], o.hparams(lr=1e-4, beta1=0.9, beta2=0.99, weight_decay=0.1, step=t, seed=3))
    out.append((t16, s16, t1, s1))

def guard(fn, *args):
    try:
        fn(*args)
    except BaseException as e:  # reported by the parent
        errors.append(repr(e))
        try:
            start.abort()
        except Exception:
            pass

which = sys.argv[1]
ra, rb = [], []
if which == "same":
    ths = [threading.Thread(target=guard, args=(adamw8, 11, [2048 * 50 + 5, 1000, 4096 * 3], ra)),
           threading.Thread(target=guard, args=(adamw8, 12, [2048 * 70, 3000, 2048 * 9 + 1], rb))]
else:
    ths = [threading.Thread(target=guard, args=(adamw8, 13, [2048 * 40 + 9, 77, 2048 * 12], ra)),
           threading.Thread(target=guard, args=(other, 14, rb))]
for th in ths:
    th.start()
for th in ths:
    th.join()
if errors:
    print("ERRORS", errors)
    sys.exit(1)
for gpu, host in [ra[0]] + ([rb[0]] if which == "same" else []):
    for i, (a, b) in enumerate(zip(gpu, host)):
        compare_state8(a, b, "tensor %d" % i)
if which != "same":
    t16, s16, t1, s1 = rb[0]
    assert np.array_equal(u16(t16.param), s16.param) and np.array_equal(u16(t16.m), s16.m)
    assert np.array_equal(u16(t16.v), s16.v)
    assert np.array_equal(u16(t1.param), s1.param) and np.array_equal(t1.m_codes.cpu().numpy(), s1.m_codes)
print("OK")
"""


@pytest.mark.parametrize("which", ["same", "mixed"])
def test_two_host_threads_first_calls(which):
    """Two threads' first calls race on the per-device set-up; both results
    must equal the oracle's."""
    pytest.importorskip("torch")
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests"), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", CHILD, which], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
