"""SR toy: gradient descent on a one-dimensional quadratic with decaying
steps, BF16 iterates written with stochastic rounding against FP32 iterates
("Stochastic Rounding for LLM Training: Theory and Practice", Figures 2-3:
with decaying updates SR converges more slowly on average than FP32 and
single runs have a long tail).  The pages give neither the objective nor the
schedule, so this is a reconstruction and its numbers are not comparable to
the figure's: parity unpinned.

Reading: f(x) = x^2 / 2 from x_0 = 1, plain gradient descent
x <- x - lr_t * x with lr_t = 0.05 * t^-0.7, converged once |x| <= 0.1.
The BF16 arms run the library's 8-bit Momentum step with momentum 0 (plain
SGD; 100 elements, so the fp32-state path, and the elements are 100
independent runs because each draws its own Philox stream); the gradient is
the current bf16 iterate itself.  The FP32 arm is the same recursion in
float32 on the host.

`PYTHONPATH=. python tests/sr_toy.py` prints the summary (needs a GPU).
"""
import numpy as np
import torch

import bit_blockwise_adamw_gb300 as q8

RUNS, STEPS, TOL, X0 = 100, 20000, 0.1, 1.0


def lr(t):
    return 0.05 * t ** -0.7


def fp32_steps():
    x = np.float32(X0)
    for t in range(1, STEPS + 1):
        x = np.float32(x - np.float32(lr(t)) * x)
        if abs(x) <= TOL:
            return t
    return -1


def bf16_steps(device, sr, runs=RUNS, seed=0):
    """Steps to convergence of each run (-1: not within STEPS)."""
    p = torch.full((runs,), X0, dtype=torch.bfloat16, device=device)
    st = q8.Tensor8.zeros_like(p, torch.empty_like(p), moments=1)
    done = torch.full((runs,), -1, dtype=torch.int64, device=device)
    for t in range(1, STEPS + 1):
        st.grad.copy_(p)
        q8.momentum8bit_sr_step([st], q8.momentum_hparams(lr=lr(t), momentum=0.0, weight_decay=0.0, step=t,
                                                          seed=seed, sr=sr))
        hit = (done < 0) & (p.float().abs() <= TOL)
        done[hit] = t
        if t % 1000 == 0 and bool((done >= 0).all()):
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
    print("BF16+RN: %s" % ("converged in %d steps" % rn[0] if rn[0] > 0 else "not converged in %d steps" % STEPS))


if __name__ == "__main__":
    main()
