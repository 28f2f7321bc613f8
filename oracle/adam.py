"""Plain fp64 Adam step: the oracle for the host optimizer.

TEST INFRASTRUCTURE.  Only the tests may import this module; the library
never does and shares no code with it.

The pages put the optimizer state at 12 bytes per parameter -- the fp32
master weight, the first moment and the second moment (gpu_zero_sharding,
"The architecture: every piece explained") -- and run the elementwise update
on the CPU beside that state, since its arithmetic intensity (about 12 FLOPs
over 24 bytes) fails the FLOPs-per-byte test at every tier
(tm_zero_infinity, "Applying the test: which state can live where").  They
name Adam but write no formula; this is the textbook step (Kingma & Ba, with
bias correction) with decoupled weight decay (Loshchilov & Hutter), written
out in float64 one line per equation:
    m_t   = beta1 m_{t-1} + (1 - beta1) g
    v_t   = beta2 v_{t-1} + (1 - beta2) g^2
    mhat  = m_t / (1 - beta1^t)
    vhat  = v_t / (1 - beta2^t)
    p_t   = p_{t-1} - lr mhat / (sqrt(vhat) + eps) - lr wd p_{t-1}
"""
from __future__ import annotations

import numpy as np


def adam_step(p, m, v, g, t: int, lr: float, beta1: float, beta2: float, eps: float, wd: float = 0.0):
    """One step; returns (p_t, m_t, v_t) as float64 arrays."""
    p = np.asarray(p, np.float64)
    m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    m_t = beta1 * m + (1.0 - beta1) * g
    v_t = beta2 * v + (1.0 - beta2) * g * g
    mhat = m_t / (1.0 - beta1 ** t)
    vhat = v_t / (1.0 - beta2 ** t)
    p_t = p - lr * mhat / (np.sqrt(vhat) + eps) - lr * wd * p
    return p_t, m_t, v_t
