"""The CPU oracle against facts that do not come from it (see oracle_pins)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import closed_forms as CF
from oracle import oracle as O
import oracle_pins as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_worked_numbers.json")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_brute_force_several_seeds(oracle_lib):
    for seed in range(10, 14):
        P.pin_brute_force(oracle_lib, seed=seed, T=3 + seed % 3, K=5 + seed, M=4 + 2 * (seed % 4))


def test_oracle_thread_count_does_not_change_results(oracle_lib):
    rng = np.random.default_rng(9)
    X = P.random_bf16(rng, (33, 70))
    W = P.random_bf16(rng, (70, 45), 0.1)
    dY = P.random_bf16(rng, (33, 45))
    base = O.max_threads()
    try:
        O.set_threads(1)
        ref = (O.forward(X, W), *O.backward(X, W, dY))
        O.set_threads(max(2, base))
        got = (O.forward(X, W), *O.backward(X, W, dY))
    finally:
        O.set_threads(base)
    for a, b in zip(ref, got):
        assert np.array_equal(a, b)


def test_distribution_sanity(oracle_lib):
    """With X, dY ~ N(0,1) and W ~ N(0, 1/K): Y ~ N(0,1), dX ~ N(0, M/K),
    dW ~ N(0, T).  A coarse check (5 %) that catches scale mistakes."""
    rng = np.random.default_rng(11)
    T, K, M = 64, 256, 384
    X = P.random_bf16(rng, (T, K))
    W = P.random_bf16(rng, (K, M), 1 / math.sqrt(K))
    dY = P.random_bf16(rng, (T, M))
    Y = O.forward(X, W)
    dX, dW = O.backward(X, W, dY)
    assert abs(Y.std() - 1.0) < 0.05
    assert abs(dX.std() - math.sqrt(M / K)) < 0.05 * math.sqrt(M / K)
    assert abs(dW.std() - math.sqrt(T)) < 0.05 * math.sqrt(T)


def test_sampled_input_validation(oracle_lib):
    X = np.zeros((4, 8), np.uint16)
    W = np.zeros((8, 16), np.uint16)
    with pytest.raises(IndexError):
        O.sample_y(X, W, [4], [0])
    with pytest.raises(TypeError):
        O.forward(X.astype(np.int32), W)


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["entries"]


def _eval(fn, args):
    if fn == "mul":
        return args["a"] * args["b"]
    if fn == "div":
        return args["a"] / args["b"]
    return getattr(CF, fn)(**args)


@pytest.mark.parametrize("entry", _golden(), ids=lambda e: e["id"])
def test_closed_form_matches_pages(entry):
    got = _eval(entry["fn"], entry["args"])
    want = entry["value"]
    if entry["rel_tol"] == 0:
        assert got == want, (entry["id"], got, want)
    else:
        assert abs(got - want) <= entry["rel_tol"] * abs(want), (entry["id"], got, want)


def test_closed_forms_consistency():
    # forward 2P and backward 4P per token; three GEMMs of 2TKM each.
    assert CF.linear_flops_forward(3, 5, 7) * 2 == CF.linear_flops_backward(3, 5, 7)
    # fwd+bwd ait over the host->device link is 6TKM / 4KM = 1.5 T.
    T, K, M = 8192, 8192, 32768
    a = CF.ait(CF.linear_flops_forward(T, K, M) + CF.linear_flops_backward(T, K, M),
               CF.linear_h2d_bytes_fwd_bwd(K, M))
    assert a == 1.5 * T
    # efficiency saturates at 1 exactly at the machine balance.
    assert CF.efficiency(63, 125e12, 2e12) == 1.0
    assert CF.efficiency(31.25, 125e12, 2e12) == pytest.approx(0.5)
    assert CF.tier_hidden(62.5, 125e12, 2e12) and not CF.tier_hidden(62.4, 125e12, 2e12)
    # ring: d tiles ahead plus the one computing; capped at N tiles.
    assert CF.ring_bytes(1024, 4096, 4, 1) == 2 * 1024 * 1024 * 2
    assert CF.ring_bytes(1024, 4096, 4, 9) == 4 * 1024 * 1024 * 2
    assert CF.roofline_seconds(T, K, M, 1.0e15, 1e12, 1e12) == pytest.approx(6 * T * K * M / 1e15)
