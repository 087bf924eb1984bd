"""SR toy: a one-dimensional descent with decaying steps, BF16 iterates
written with stochastic rounding against FP32 iterates ("Stochastic Rounding
for LLM Training: Theory and Practice", Figures 2-3: with decaying updates SR
can take longer to converge than FP32 on average, and single runs take much
longer still).  The pages give neither the objective nor the schedule, so
this is a reconstruction and its numbers are not comparable to the figure's:
parity unpinned.

Reading: minimise f(x) = |x - 1| by gradient descent with the step
lr_t = C * t^-0.7 (decaying, and below one bf16 spacing from the first step),
from x_0 = 1 + 6 * 2^-7, six bf16 spacings above the minimum (in [1, 2) the
spacing is 2^-7); converged once |x - 1| <= 0.001, which in bf16 means x = 1
exactly.  The gradient sign(x - 1) does not shrink as x nears the minimum,
so FP32 moves by exactly lr_t a step, while a stochastically rounded iterate
moves by whole spacings, each step with chance lr_t / 2^-7: its progress is a
count of rare jumps whose rate decays with t, unbiased, but with a
right-skewed time to the sixth jump.  Round-to-nearest never moves (every
update is below half a spacing).

The BF16 arms run the library's 8-bit Momentum step with momentum 0 (plain
SGD; 100 elements, so the fp32-state path, and the elements are 100
independent runs because each draws its own Philox stream); the gradient of
each run is the bf16 sign of its current iterate minus 1.  The FP32 arm is
the same recursion in float32 on the host.

`PYTHONPATH=. python tests/sr_toy.py` prints the summary (needs a GPU).
"""
import numpy as np
import torch

import bit_blockwise_adamw_gb300 as q8

RUNS, STEPS = 100, 300_000
C, POWER = 0.00116, 0.7
X_STAR = 1.0
X0 = 1.0 + 6 * 2.0 ** -7
TOL = 0.001


def lr(t):
    return C * t ** -POWER


def fp32_steps():
    x, xs = np.float32(X0), np.float32(X_STAR)
    for t in range(1, STEPS + 1):
        x = np.float32(x - np.float32(lr(t)) * np.float32(np.sign(x - xs)))
        if abs(x - xs) <= TOL:
            return t
    return -1


def bf16_steps(device, sr, runs=RUNS, seed=0):
    """Steps to convergence of each run (-1: not within STEPS)."""
    p = torch.full((runs,), X0, dtype=torch.bfloat16, device=device)
    st = q8.Tensor8.zeros_like(p, torch.empty_like(p), moments=1)
    done = torch.full((runs,), -1, dtype=torch.int64, device=device)
    for t in range(1, STEPS + 1):
        st.grad.copy_(torch.sign(p.float() - X_STAR))
        q8.momentum8bit_sr_step([st], q8.momentum_hparams(lr=lr(t), momentum=0.0, weight_decay=0.0, step=t,
                                                          seed=seed, sr=sr))
        hit = (done < 0) & ((p.float() - X_STAR).abs() <= TOL)
        done[hit] = t
        if t % 1000 == 0 and bool((done >= 0).all()):
            break
        if sr == 0 and t == 20_000:
            break
    return done.cpu().numpy()


def main():
    dev = torch.device("cuda", 0)
    t32 = fp32_steps()
    sr = bf16_steps(dev, 1)
    rn = bf16_steps(dev, 0, runs=1)
    ok = sr[sr > 0]
    print("FP32: %d steps" % t32)
    print("BF16+SR: %d/%d runs converged; mean %.0f, median %.0f, min %d, max %d steps"
          % (len(ok), RUNS, ok.mean(), np.median(ok), ok.min(), ok.max()))
    print("BF16+RN: %s" % ("converged in %d steps" % rn[0] if rn[0] > 0 else "not converged"))


if __name__ == "__main__":
    main()
