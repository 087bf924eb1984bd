"""Host-side logic of bench.py (no GPU): the algorithmic byte model, the
launch count per step, the oracle sample's layout and timing and the reference
arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
from bit_blockwise_adamw_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _blocks(wl):
    return sum((t.numel + 2047) // 2048 for t in wl.tensors if t.numel >= 4096)


@pytest.mark.parametrize("name", ["gptneo-6.7b", "gpt2-350m", "gpt2-xl-1.5b", "flat-1m"])
def test_byte_model(name):
    """8-bit path: grad 2 + param 2+2 + one code byte each way per moment,
    plus 4 B of absmax each way per moment per block; fp32-state tensors
    (n < 4096): 2 + 2+2 + 8 per moment."""
    wl = W.WORKLOADS[name]
    small = sum(t.numel for t in wl.tensors if t.numel < 4096)
    big = wl.numel - small
    assert bench.algorithmic_bytes(wl, 2) == 10 * big + 16 * _blocks(wl) + 22 * small
    assert bench.algorithmic_bytes(wl, 1) == 8 * big + 8 * _blocks(wl) + 14 * small


def test_byte_model_headline_figures():
    assert bench.algorithmic_bytes(W.WORKLOADS["gptneo-6.7b"], 2) == 66_632_127_072
    assert bench.algorithmic_bytes(W.WORKLOADS["gptneo-2.7b-bf16"]) == 14 * 2_651_307_520


def test_launches_per_step():
    assert bench.launches_per_step(W.WORKLOADS["gptneo-6.7b"]) == 1          # 420 tensors, no partial block
    assert bench.launches_per_step(W.WORKLOADS["gpt2-xl-1.5b"]) == 3         # main + tail + small tensors
    assert bench.launches_per_step(W.WORKLOADS["gptneo-2.7b-bf16"]) == 1
    wl = W.custom("many", [4096] * 500, steps=1)
    assert bench.launches_per_step(wl) == 2                                 # 448 + 52 tensors


def test_block_parallel_oracle_timing():
    wl = W.WORKLOADS["gptneo-6.7b"]
    n, dt = bench.oracle_parallel_time(wl, 16, 2)
    assert n == 2 * 16 * 2048 and dt > 0


@pytest.mark.parametrize("name", ["gptneo-6.7b", "gpt2-350m", "gptneo-2.7b-bf16"])
def test_oracle_sample_runs(name):
    """The oracle's timed sample: runs of consecutive full blocks inside one
    tensor each, only tensors on the 8-bit path, the requested block count."""
    wl = W.WORKLOADS[name]
    runs = bench.sample_runs(wl, 5000, np.random.default_rng(3), 512)
    assert sum(n for _, _, n in runs) == 5000
    for i, b0, n in runs:
        t = wl.tensors[i]
        assert 1 <= n <= 512 and b0 >= 0 and (b0 + n) * 2048 <= max(t.numel, 2048)
        assert t.numel >= 4096 or wl.state == "bf16"
    assert len({i for i, _, _ in runs}) > 5


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0", "--cpu-blocks", "64"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "Gparams/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
