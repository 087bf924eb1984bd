"""Accumulated-update study: round-to-nearest (RN) against stochastic rounding
(SR) of the bf16 writes, both measured against a float64 AdamW that keeps
float64 parameters and moments.

Pages: "Stochastic rounding support for 8-bit optimizers" (activity: the
proposed evaluation compares nearest and stochastic rounding with a
higher-precision reference through accumulated-update tests over several
seeds) and "Stochastic rounding of AdamW momentums" (bf16 moment accumulation
losing precision; the linked report that weight decay has no effect with bf16
parameters).

Three arms run the library's own steps through the C ABI on the same bf16
gradients:
  8bit  one 65,536-element tensor, 8-bit blockwise m and v (adamw8bit_sr_step)
  fp32  sixteen 4,095-element tensors, fp32 m and v (same call, small path)
  bf16  one 65,536-element tensor, bf16 m and v (adamw_bf16_sr_step)
each twice, sr = 0 (RN) and sr = 1 (SR).  The reference is the textbook
AdamW with decoupled weight decay and bias correction, in float64, started
from the same bf16 parameters.

Gradients are synthetic: g = scale * (mu + xi), mu a fixed per-element mean
(signal * N(0, 1)), xi fresh N(0, 1) every step, rounded to bf16 (RNE).
Parameters start at N(0, 0.02^2) rounded to bf16.

Reported per arm and rounding, for the accumulated update D = p_t - p_0
against the reference's R = p_ref_t - p_0:
  realised  <D, R> / <R, R>   (1 = the reference's update, 0 = none of it)
  rel_err   |D - R| / |R|
  unmoved   share of the elements with R != 0 whose bf16 parameter ends
            where it started

Regimes:
  sub-ulp     lr 1e-5, no decay: every update is far below half a bf16 ulp
  decay-only  zero gradient, lr 1e-3, weight decay 1e-2 (a 1e-5 shrink a step)
  growing     lr 1e-3, weight decay 1e-2, a steady gradient mean: updates
              start at a few ulps of the initial weights, and as the weights
              grow the same updates fall below half an ulp
  noise       lr 1e-3, zero-mean gradient: the weights random-walk and stay
              small, so updates stay near or above an ulp

`PYTHONPATH=. python tests/rounding_study.py` prints the table (needs a GPU).
"""
import argparse
import time

import numpy as np
import torch

import bit_blockwise_adamw_gb300 as q8

B1, B2, EPS = 0.9, 0.999, 1e-8
REGIMES = {
    "sub-ulp": dict(lr=1e-5, wd=0.0, scale=1e-3, signal=0.3),
    "decay-only": dict(lr=1e-3, wd=1e-2, scale=0.0, signal=0.0),
    "growing": dict(lr=1e-3, wd=1e-2, scale=1e-3, signal=0.3),
    "noise": dict(lr=1e-3, wd=0.0, scale=1e-3, signal=0.0),
}
ARMS = {"8bit": [65536], "fp32": [4095] * 16, "bf16": [65536]}
ROUNDINGS = {"RN": 0, "SR": 1}


def bf16_bits(x32):
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x32, np.float32).view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> 16) & np.uint32(1))) >> 16).astype(np.uint16)


def bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Layout:
    """All arms' tensors in one flat bf16 buffer; every tensor starts on a
    16-byte boundary (a multiple of 8 elements)."""

    def __init__(self):
        self.segments = []          # (arm, start, n)
        off = 0
        for arm, sizes in ARMS.items():
            for n in sizes:
                self.segments.append((arm, off, n))
                off += (n + 7) // 8 * 8
        self.total = off
        self.mask = {arm: np.zeros(off, bool) for arm in ARMS}
        for arm, s, n in self.segments:
            self.mask[arm][s:s + n] = True


class Reference:
    """Float64 AdamW (decoupled decay, bias-corrected moments)."""

    def __init__(self, p0, lr, wd):
        self.p, self.m, self.v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
        self.lr, self.wd = lr, wd

    def step(self, g, t):
        self.m = B1 * self.m + (1 - B1) * g
        self.v = B2 * self.v + (1 - B2) * g * g
        mhat = self.m / (1 - B1 ** t)
        vhat = self.v / (1 - B2 ** t)
        self.p = self.p * (1 - self.lr * self.wd) - self.lr * mhat / (np.sqrt(vhat) + EPS)


def metrics(d, r):
    rr = float(np.dot(r, r))
    if rr == 0.0:
        return dict(realised=float("nan"), rel_err=float("nan"), unmoved=float("nan"))
    moved = r != 0
    return dict(realised=float(np.dot(d, r)) / rr,
                rel_err=float(np.linalg.norm(d - r)) / np.sqrt(rr),
                unmoved=float(np.count_nonzero((d == 0) & moved)) / max(int(np.count_nonzero(moved)), 1))


def run(regime, seed, steps, device, every=None, exact=1):
    """One regime and seed.  Returns {step: {(arm, rounding): metrics}} at the
    checkpoints (every `every` steps, and the last)."""
    cfg = REGIMES[regime]
    lay = Layout()
    rng = np.random.default_rng(1000 + seed)
    p0_bits = np.zeros(lay.total, np.uint16)
    mu = np.zeros(lay.total, np.float32)
    for arm, s, n in lay.segments:
        p0_bits[s:s + n] = bf16_bits((rng.standard_normal(n) * 0.02).astype(np.float32))
        mu[s:s + n] = rng.standard_normal(n).astype(np.float32) * cfg["signal"]
    valid = np.zeros(lay.total, bool)
    for arm in ARMS:
        valid |= lay.mask[arm]
    p0 = bf16_value(p0_bits)
    ref = Reference(p0, cfg["lr"], cfg["wd"])

    host_g = torch.empty(lay.total, dtype=torch.int16).pin_memory()
    grad = torch.zeros(lay.total, dtype=torch.bfloat16, device=device)
    params, lists8, lists16 = {}, {}, {}
    for name in ROUNDINGS:
        flat = torch.from_numpy(p0_bits.view(np.int16)).to(device).view(torch.bfloat16)
        params[name] = flat
        t8, t16 = [], []
        for arm, s, n in lay.segments:
            pv, gv = flat[s:s + n], grad[s:s + n]
            if arm == "bf16":
                t16.append(q8.Tensor16(pv, gv, torch.zeros_like(pv), torch.zeros_like(pv)))
            else:
                t8.append(q8.Tensor8.zeros_like(pv, gv))
        lists8[name], lists16[name] = t8, t16

    out = {}
    for t in range(1, steps + 1):
        if cfg["scale"] > 0:
            xi = rng.standard_normal(lay.total, dtype=np.float32)
            gb = bf16_bits(np.float32(cfg["scale"]) * (mu + xi))
            gb[~valid] = 0
        else:
            gb = np.zeros(lay.total, np.uint16)
        host_g.numpy()[:] = gb.view(np.int16)
        grad.view(torch.int16).copy_(host_g)
        for name, sr in ROUNDINGS.items():
            hp = q8.hparams(exact=exact, lr=cfg["lr"], beta1=B1, beta2=B2, eps=EPS, weight_decay=cfg["wd"],
                            step=t, seed=seed, sr=sr)
            q8.adamw8bit_sr_step(lists8[name], hp)
            q8.adamw_bf16_sr_step(lists16[name], hp)
        ref.step(bf16_value(gb), t)
        if (every and t % every == 0) or t == steps:
            torch.cuda.synchronize()
            r = ref.p - p0
            row = {}
            for name in ROUNDINGS:
                bits = params[name].view(torch.int16).cpu().numpy().view(np.uint16)
                d = bf16_value(bits) - p0
                for arm in ARMS:
                    k = lay.mask[arm]
                    row[(arm, name)] = metrics(d[k], r[k])
            out[t] = row
    return out


def table(results, steps):
    """Markdown: per regime, arm and rounding, mean [min, max] over seeds of
    the final checkpoint's metrics."""
    lines = ["| regime | arm | rounding | realised | rel_err | unmoved |", "|---|---|---|---|---|---|"]
    for regime, per_seed in results.items():
        for arm in ARMS:
            for name in ROUNDINGS:
                vals = [per_seed[s][steps][(arm, name)] for s in per_seed]
                cells = []
                for key in ("realised", "rel_err", "unmoved"):
                    xs = np.array([v[key] for v in vals])
                    cells.append("%.3f [%.3f, %.3f]" % (xs.mean(), xs.min(), xs.max()))
                lines.append("| %s | %s | %s | %s |" % (regime, arm, name, " | ".join(cells)))
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--seeds", type=int, default=3)
    ap.add_argument("--every", type=int, default=500)
    ap.add_argument("--regimes", nargs="*", default=list(REGIMES))
    ap.add_argument("--fast", action="store_true", help="the AdamW steps in the fast mode (default: bit-exact)")
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    results = {}
    t0 = time.time()
    for regime in a.regimes:
        results[regime] = {}
        for seed in range(1, a.seeds + 1):
            results[regime][seed] = run(regime, seed, a.steps, dev, a.every, exact=0 if a.fast else 1)
            for t, row in results[regime][seed].items():
                print("%s seed %d step %d: %s" % (regime, seed, t, "; ".join(
                    "%s/%s %.3f %.3f" % (arm, name, m["realised"], m["rel_err"]) for (arm, name), m in row.items())),
                      flush=True)
    print()
    print("%d steps, seeds 1..%d, %s mode, %.0f s" % (a.steps, a.seeds, "fast" if a.fast else "bit-exact",
                                                     time.time() - t0))
    print(table(results, a.steps))


if __name__ == "__main__":
    main()
