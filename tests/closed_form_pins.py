"""Pins of the closed forms (``oracle/closed_forms.py``) that do not retype them.

Each ``pin_*(cf)`` takes a closed-forms module (the real one, or a copy with a
planted mistake) and raises AssertionError when it disagrees with:
  * brute force: the multiply-adds of the plain definitions of Y, dX and dW,
    counted one by one on tiny shapes (2 FLOPs each);
  * the schedule model (``schedule_sim``): the bytes its transfers move, and
    its makespan, which no schedule can beat and which a deep ring with
    ample staging approaches, in each of the three regimes;
  * the pages' own efficiency rule (tm_zero_infinity, "The honest cost"),
    which the golden worked numbers pin separately.
"""
from __future__ import annotations

import itertools

import schedule_sim as S


def _count_macs(T: int, K: int, M: int) -> tuple[int, int, int]:
    """Multiply-adds of Y = X W, dX = dY W^T and dW = X^T dY, one per innermost
    iteration of each definition."""
    y = dx = dw = 0
    for _t, _m, _k in itertools.product(range(T), range(M), range(K)):
        y += 1
    for _t, _k, _m in itertools.product(range(T), range(K), range(M)):
        dx += 1
    for _k, _m, _t in itertools.product(range(K), range(M), range(T)):
        dw += 1
    return y, dx, dw


def pin_flops_brute_force(cf):
    for T, K, M in [(1, 1, 1), (2, 3, 5), (3, 4, 7), (5, 2, 6)]:
        y, dx, dw = _count_macs(T, K, M)
        assert cf.linear_flops_forward(T, K, M) == 2 * y, (T, K, M)
        assert cf.linear_flops_backward(T, K, M) == 2 * (dx + dw), (T, K, M)


def pin_bytes_from_schedule(cf):
    for T, K, M, N, d in [(64, 128, 512, 4, 1), (32, 96, 768, 3, 2), (16, 64, 640, 5, 0)]:
        r = S.simulate(T, K, M, N, d, 1e12, 1e10, 1e10, steps=3)
        assert cf.linear_h2d_bytes_fwd_bwd(K, M) * 3 == r["h2d_bytes"], (K, M)
        assert cf.linear_d2h_bytes_fwd_bwd(K, M) * 3 == r["d2h_bytes"], (K, M)
        assert cf.linear_flops_forward(T, K, M) * 3 + cf.linear_flops_backward(T, K, M) * 3 == r["flops"]


# (T, K, M, R, B_h2d, B_d2h) with the regime that binds: the GPT-scale layer
# on a fast link (compute), a small batch (host->device), a slow
# device->host direction (device->host).
REGIMES = [
    ("tensor", (8192, 1024, 4096, 1.5e15, 2e11, 1.8e11)),
    ("h2d", (256, 1024, 4096, 1.5e15, 2e11, 1.8e11)),
    ("d2h", (4096, 1024, 4096, 1.5e15, 2e11, 1.5e10)),
]


def _regime_terms(cf, T, K, M, R, bh, bd):
    flops = cf.linear_flops_forward(T, K, M) + cf.linear_flops_backward(T, K, M)
    return {"tensor": flops / R, "h2d": cf.linear_h2d_bytes_fwd_bwd(K, M) / bh,
            "d2h": cf.linear_d2h_bytes_fwd_bwd(K, M) / bd}


def pin_roofline_against_schedule(cf):
    """roofline_seconds is a lower bound of the modelled step, and the model
    with a deep ring and ample staging reaches it within 1 %, in every regime."""
    for name, (T, K, M, R, bh, bd) in REGIMES:
        steps, N = 60, 16
        bound = cf.roofline_seconds(T, K, M, R, bh, bd)
        deep = S.simulate(T, K, M, N, N - 1, R, bh, bd, steps, staging=4 * N)["seconds"] / steps
        shallow = S.simulate(T, K, M, N, 1, R, bh, bd, steps, staging=2)["seconds"] / steps
        assert bound <= deep * (1 + 1e-12) and bound <= shallow * (1 + 1e-12), (name, bound, deep, shallow)
        assert deep <= 1.01 * bound, (name, bound, deep)
        terms = _regime_terms(cf, T, K, M, R, bh, bd)
        assert max(terms, key=terms.get) == name, (name, terms)


def pin_link_bound_efficiency_is_the_pages_rule(cf):
    """Below the crossover the step's efficiency against compute alone is
    ait / (R / BW) with ait = 6TKM / 4KM over the host->device link
    (tm_zero_infinity, "The honest cost"); above it, 1."""
    K, M, R, B = 1024, 4096, 1.5e15, 2e11
    for T in (128, 512, 2048, 8192, 65536):
        t = cf.roofline_seconds(T, K, M, R, B, 10 * B)
        compute = (cf.linear_flops_forward(T, K, M) + cf.linear_flops_backward(T, K, M)) / R
        ait = (cf.linear_flops_forward(T, K, M) + cf.linear_flops_backward(T, K, M)) / \
            cf.linear_h2d_bytes_fwd_bwd(K, M)
        eff = cf.efficiency(ait, R, B)
        assert abs(compute / t - eff) <= 1e-12 * max(1.0, eff), (T, compute / t, eff)


ALL_PINS = [pin_flops_brute_force, pin_bytes_from_schedule, pin_roofline_against_schedule,
            pin_link_bound_efficiency_is_the_pages_rule]
