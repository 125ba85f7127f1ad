"""CPU oracle of the optimizer step: AdamW over flat float arrays, in float64.

TEST INFRASTRUCTURE ONLY (same rule as the rest of ``oracle``): only
``tests/`` and ``bench.py``'s CPU legs may use it; it shares no code with
``layer_streamed_gb300``.

Follows "MegaTrain: Full Precision Training of 100B+ Parameter Large Language
Models on a Single GPU", section 方法步骤详情, stage 4 (the CPU optimizer update
theta <- AdamUpdate(theta, grad, m, v) applied to the host-resident master
weights after the gradients have streamed back). The pages name Adam without
its formula; the update written here is Adam with bias correction and
decoupled weight decay (AdamW, Loshchilov and Hutter, "Decoupled Weight Decay
Regularization", 2019), which is Adam when weight_decay = 0:

    m_t  = beta1 m_{t-1} + (1 - beta1) g
    v_t  = beta2 v_{t-1} + (1 - beta2) g^2
    m^   = m_t / (1 - beta1^t),   v^ = v_t / (1 - beta2^t)
    theta_t = theta_{t-1} - lr (m^ / (sqrt(v^) + eps) + weight_decay theta_{t-1})
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class AdamW:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0


def adamw_step(opt: AdamW, step: int, theta, m, v, g):
    """One update at step number `step` (1-based). Returns new (theta, m, v)
    as float64 arrays; the inputs are not modified."""
    if step < 1:
        raise ValueError("step numbers start at 1")
    theta = np.asarray(theta, np.float64)
    g = np.asarray(g, np.float64)
    m = opt.beta1 * np.asarray(m, np.float64) + (1.0 - opt.beta1) * g
    v = opt.beta2 * np.asarray(v, np.float64) + (1.0 - opt.beta2) * g * g
    m_hat = m / (1.0 - opt.beta1 ** step)
    v_hat = v / (1.0 - opt.beta2 ** step)
    theta = theta - opt.lr * (m_hat / (np.sqrt(v_hat) + opt.eps) + opt.weight_decay * theta)
    return theta, m, v
