"""A step captured in a CUDA graph right after q8_prepare_device().

q8_prepare_device() uploads the tables and caches every kernel's launch
configuration, so that no later call does any set-up.  In a fresh process
(cold caches), the first 8-bit AdamW, BF16-state and Lion steps are captured
in one CUDA graph, the graph is replayed, and the results must equal the
same steps run eagerly on copies of the same inputs, bit for bit.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
import bit_blockwise_adamw_gb300 as q8
from bit_blockwise_adamw_gb300 import workloads as W

dev = torch.device("cuda:0")
q8.q8_prepare_device()
wl = W.custom("graph", [2048 * 30 + 5, 1000, 4096], steps=1, outlier_rate=1e-3, outlier_factor=100.0, data_seed=21)
params = W.init_params(wl, dev)
grads = W.make_grads(wl, 1, dev)

def states8(ps):
    return [q8.Tensor8.zeros_like(p.clone(), g) for p, g in zip(ps, grads)]

def states16(p, g):
    return [q8.Tensor16(p.clone(), g, torch.zeros_like(p), torch.zeros_like(p))]

def states1(p, g):
    return [q8.Tensor8.zeros_like(p.clone(), g, moments=1)]

hp = q8.hparams(lr=1e-3, weight_decay=0.1, step=1, seed=5)
hl = q8.lion_hparams(lr=1e-4, weight_decay=0.1, step=1, seed=5)
cap8, eag8 = states8(params), states8(params)
cap16, eag16 = states16(params[0], grads[0]), states16(params[0], grads[0])
cap1, eag1 = states1(params[0], grads[0]), states1(params[0], grads[0])
torch.cuda.synchronize()

g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):
    q8.adamw8bit_sr_step(cap8, hp)
    q8.adamw_bf16_sr_step(cap16, hp)
    q8.lion8bit_sr_step(cap1, hl)
g.replay()
q8.adamw8bit_sr_step(eag8, hp)
q8.adamw_bf16_sr_step(eag16, hp)
q8.lion8bit_sr_step(eag1, hl)
torch.cuda.synchronize()

def same(a, b):
    return a is None and b is None or torch.equal(a.view(torch.uint8), b.view(torch.uint8))

for a, b in zip(cap8 + cap1, eag8 + eag1):
    for f in ("param", "m_codes", "v_codes", "m_absmax", "v_absmax", "m32", "v32"):
        assert same(getattr(a, f), getattr(b, f)), f
for a, b in zip(cap16, eag16):
    for f in ("param", "m", "v"):
        assert same(getattr(a, f), getattr(b, f)), f
assert not torch.equal(cap8[0].param, params[0])      # the replay did update the parameters
print("OK")
"""


def test_step_captured_after_prepare_matches_eager():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([ROOT, env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
