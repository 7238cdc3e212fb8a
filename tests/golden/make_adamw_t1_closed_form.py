"""Writes adamw_t1_closed_form.txt: AdamW's first step from m = v = 0 in
closed form, evaluated in exact rational arithmetic (no oracle, no CUDA).

At t = 1 the bias-corrected moments are m_hat = g and v_hat = g*g, so with
decoupled weight decay scaled by lr the step is
    theta_1 = theta_0 - lr * (g / (|g| + eps) + wd * theta_0)
for lr = 1e-3, eps = 1e-8, wd = 0.1 (beta1 and beta2 cancel at t = 1).
Reading of "A4 — Multi-GPU with NCCL and ZeRO-1", Part 4 (AdamW on the owned
shard); the hyperparameters are the tiny workload's.

    python tests/golden/make_adamw_t1_closed_form.py > tests/golden/adamw_t1_closed_form.txt
"""
from fractions import Fraction as F

LR, EPS, WD = F(1, 1000), F(1, 10 ** 8), F(1, 10)
CASES = [(F(1, 2), F(1)), (F(1, 2), F(-1)), (F(-1, 4), F(1, 1000)), (F(0), F(0)), (F(1), F(0))]


def theta1(theta0: F, g: F) -> F:
    return theta0 - LR * (g / (abs(g) + EPS) + WD * theta0)


def lines() -> list[str]:
    out = [
        "# AdamW at its first step from m = v = 0 (bias-corrected moments give",
        "# m_hat = g and v_hat = g*g), decoupled weight decay scaled by lr:",
        "#   theta_1 = theta_0 - lr * ( g / (|g| + eps) + wd * theta_0 )",
        "# lr = 1e-3, eps = 1e-8, wd = 0.1 (beta1 = 0.9, beta2 = 0.999 cancel at t = 1),",
        "# evaluated exactly by make_adamw_t1_closed_form.py.  Readings: \"A4 — Multi-GPU",
        "# with NCCL and ZeRO-1\", Part 4 (AdamW on the owned shard); hyperparameters of",
        "# the tiny workload.",
        "# theta_0 g theta_1",
    ]
    for t0, g in CASES:
        out.append(f"{float(t0)!r} {float(g)!r} {float(theta1(t0, g))!r}")
    return out


if __name__ == "__main__":
    print("\n".join(lines()))
