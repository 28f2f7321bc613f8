"""Checks that pin the CPU oracle to facts that do not come from the oracle.

Each ``pin_*`` function takes an oracle library handle (``oracle.load()`` or a
deliberately broken build of the same source) and raises AssertionError when
the oracle disagrees with an independent fact:

* exact rational brute force (Python ``fractions``) within the fp32 summation
  error bound  |fl(sum) - sum| <= gamma_{n} * sum |terms|,  gamma_n = n u / (1 - n u),
  u = 2^-24 (a textbook bound for recursive summation);
* an all-integer case, which fp32 evaluates exactly, against numpy's int64
  matrix product;
* identity weights (K = M, W = I): Y = X and dX = dY exactly;
* the concatenation property of output-dimension tiling (pwwt.cn/news/5430303,
  关键技术一 核心思想; tm_zero_infinity, "Memory-centric tiling"): the product
  with one column block of W equals that block of the full product;
* the adjoint identity <Y, dY> = <X, dX> = <W, dW> (all equal
  sum_{t,k,m} X[t,k] W[k,m] dY[t,m]);
* sampled entries equal full-tensor entries, for both W storage layouts;
* fp32 -> bf16 rounding against torch's conversion and hand-made ties;
* chains of two operators with one identity matrix, where the composition
  reduces to single products and one rounding.

Shapes are chosen with T, K, M pairwise distinct so that a transposed operand
or a swapped index changes the answer.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from oracle import oracle as O

U32 = 2.0 ** -24


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp64 -> bf16 bits, via fp32 (exact for the small
    integers and bf16-representable values the pins use)."""
    f = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def random_bf16(rng: np.random.Generator, shape, std=1.0) -> np.ndarray:
    return f64_to_bf16_bits(rng.standard_normal(shape) * std)


def gamma(n: int) -> float:
    return n * U32 / (1 - n * U32)


def _exact_dot(a_bits, b_bits) -> tuple[Fraction, float]:
    a = bf16_bits_to_f64(a_bits)
    b = bf16_bits_to_f64(b_bits)
    terms = [Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a, b)]
    return sum(terms, Fraction(0)), float(sum(abs(t) for t in terms))


def _check_close_exact(got: float, exact: Fraction, abs_terms: float, n: int, what: str):
    assert np.isfinite(got), f"{what}: oracle value {got} is not finite"
    err = abs(Fraction(float(got)) - exact)
    bound = Fraction(gamma(n) * abs_terms) + Fraction(1, 1 << 140)
    assert err <= bound, f"{what}: |oracle - exact| = {float(err):.3e} > bound {float(bound):.3e}"


def pin_brute_force(lib, seed=0, T=5, K=11, M=7):
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    W = random_bf16(rng, (K, M), 1 / np.sqrt(K))
    dY = random_bf16(rng, (T, M))
    Y = O.forward(X, W, lib)
    dX, dW = O.backward(X, W, dY, lib)
    for t in range(T):
        for m in range(M):
            ex, s = _exact_dot(X[t, :], W[:, m])
            _check_close_exact(Y[t, m], ex, s, K, f"Y[{t},{m}]")
    for t in range(T):
        for k in range(K):
            ex, s = _exact_dot(dY[t, :], W[k, :])
            _check_close_exact(dX[t, k], ex, s, M, f"dX[{t},{k}]")
    for k in range(K):
        for m in range(M):
            ex, s = _exact_dot(X[:, k], dY[:, m])
            _check_close_exact(dW[k, m], ex, s, T, f"dW[{k},{m}]")


def ternary(rng, shape) -> np.ndarray:
    return rng.integers(-1, 2, shape).astype(np.int64)


def pin_integer_exact(lib, seed=1, T=128, K=96, M=160):
    """Entries in {-1,0,1}: every partial sum is an integer of magnitude at
    most max(T,K,M) < 2^24, so the fp32 oracle must equal the integer product."""
    rng = np.random.default_rng(seed)
    Xi, Wi, dYi = ternary(rng, (T, K)), ternary(rng, (K, M)), ternary(rng, (T, M))
    X, W, dY = (f64_to_bf16_bits(a.astype(np.float64)) for a in (Xi, Wi, dYi))
    Y = O.forward(X, W, lib)
    dX, dW = O.backward(X, W, dY, lib)
    assert np.array_equal(Y.astype(np.int64), Xi @ Wi) and np.all(Y == np.round(Y)), "Y integer case"
    assert np.array_equal(dX.astype(np.int64), dYi @ Wi.T) and np.all(dX == np.round(dX)), "dX integer case"
    assert np.array_equal(dW.astype(np.int64), Xi.T @ dYi) and np.all(dW == np.round(dW)), "dW integer case"


def pin_identity(lib, seed=2, T=9, K=24):
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    dY = random_bf16(rng, (T, K))
    W = f64_to_bf16_bits(np.eye(K))
    Y = O.forward(X, W, lib)
    dX, dW = O.backward(X, W, dY, lib)
    assert np.array_equal(Y.astype(np.float64), bf16_bits_to_f64(X)), "identity: Y != X"
    assert np.array_equal(dX.astype(np.float64), bf16_bits_to_f64(dY)), "identity: dX != dY"
    ref = bf16_bits_to_f64(X).T @ bf16_bits_to_f64(dY)
    bound = gamma(T) * (np.abs(bf16_bits_to_f64(X)).T @ np.abs(bf16_bits_to_f64(dY))) + 1e-30
    assert np.all(np.abs(dW - ref) <= bound), "identity: dW != X^T dY"


def pin_concatenation(lib, seed=3, T=6, K=10, M=12, N=3):
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    W = random_bf16(rng, (K, M), 1 / np.sqrt(K))
    Y = O.forward(X, W, lib)
    Mi = M // N
    for i in range(N):
        Wi = np.ascontiguousarray(W[:, i * Mi:(i + 1) * Mi])
        Yi = O.forward(X, Wi, lib)
        assert np.array_equal(Yi, Y[:, i * Mi:(i + 1) * Mi]), f"tile {i} != column block {i}"


def pin_adjoint(lib, seed=4, T=24, K=40, M=56):
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    W = random_bf16(rng, (K, M), 1 / np.sqrt(K))
    dY = random_bf16(rng, (T, M))
    Y = O.forward(X, W, lib).astype(np.float64)
    dX, dW = (a.astype(np.float64) for a in O.backward(X, W, dY, lib))
    x, w, dy = bf16_bits_to_f64(X), bf16_bits_to_f64(W), bf16_bits_to_f64(dY)
    a = float(np.sum(Y * dy))
    b = float(np.sum(x * dX))
    c = float(np.sum(w * dW))
    scale = float(np.sum(np.abs(x) @ np.abs(w) * np.abs(dy)))
    tol = 4 * gamma(max(T, K, M)) * scale
    assert abs(a - b) <= tol and abs(a - c) <= tol, f"adjoint: {a} {b} {c} (tol {tol})"


def pin_sampled(lib, seed=5, T=7, K=12, M=20, N=4):
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    W = random_bf16(rng, (K, M), 1 / np.sqrt(K))
    dY = random_bf16(rng, (T, M))
    Y = O.forward(X, W, lib)
    dX, dW = O.backward(X, W, dY, lib)
    Wt = np.ascontiguousarray(W.reshape(K, N, M // N).transpose(1, 0, 2))
    r, c = np.meshgrid(np.arange(T), np.arange(M), indexing="ij")
    for Ws in (W, Wt):
        assert np.array_equal(O.sample_y(X, Ws, r.ravel(), c.ravel(), lib), Y.ravel()), "sample_y"
    r, c = np.meshgrid(np.arange(T), np.arange(K), indexing="ij")
    for Ws in (W, Wt):
        assert np.array_equal(O.sample_dx(dY, Ws, r.ravel(), c.ravel(), lib), dX.ravel()), "sample_dx"
    r, c = np.meshgrid(np.arange(K), np.arange(M), indexing="ij")
    assert np.array_equal(O.sample_dw(X, dY, r.ravel(), c.ravel(), lib), dW.ravel()), "sample_dw"


def pin_sampled_brute_force(lib, seed=6, T=9, K=13, M=16, N=4):
    """The sampled entry points against exact rational brute force on their
    own (a mistake shared by full and sampled code is caught here too)."""
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    W = random_bf16(rng, (K, M), 1 / np.sqrt(K))
    dY = random_bf16(rng, (T, M))
    Wt = np.ascontiguousarray(W.reshape(K, N, M // N).transpose(1, 0, 2))
    rows = rng.integers(0, T, 12)
    cols = rng.integers(0, M, 12)
    got = O.sample_y(X, Wt, rows, cols, lib)
    for j, (t, m) in enumerate(zip(rows, cols)):
        ex, s = _exact_dot(X[t, :], W[:, m])
        _check_close_exact(got[j], ex, s, K, f"sample_y[{t},{m}]")
    cols_k = rng.integers(0, K, 12)
    got = O.sample_dx(dY, Wt, rows, cols_k, lib)
    for j, (t, k) in enumerate(zip(rows, cols_k)):
        ex, s = _exact_dot(dY[t, :], W[k, :])
        _check_close_exact(got[j], ex, s, M, f"sample_dx[{t},{k}]")
    rows_k = rng.integers(0, K, 12)
    got = O.sample_dw(X, dY, rows_k, cols, lib)
    for j, (k, m) in enumerate(zip(rows_k, cols)):
        ex, s = _exact_dot(X[:, k], dY[:, m])
        _check_close_exact(got[j], ex, s, T, f"sample_dw[{k},{m}]")


def pin_round_bf16(lib):
    """fp32 -> bf16 round-to-nearest-even against torch's conversion (an
    independent library routine) for every sign / exponent / kept-fraction
    pattern with the dropped half at and around the rounding boundaries, and
    hand-made ties that must go to the even neighbour."""
    import torch
    hi = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    f = (hi[:, None] | lows[None, :]).ravel().view(np.float32)
    got = O.round_bf16(f, lib)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan]), "round_bf16 differs from torch on finite / infinite values"
    assert np.all(np.isnan(bf16_bits_to_f64(got[nan]))), "round_bf16 lost a NaN"
    ties = {1 + 2.0 ** -8: 0x3F80, 1 + 3 * 2.0 ** -8: 0x3F82, -(1 + 2.0 ** -8): 0xBF80,
            1 + 2.0 ** -8 + 2.0 ** -20: 0x3F81, 3.4028234663852886e38: 0x7F80, 2.0 ** -133: 0x0001,
            2.0 ** -134: 0x0000, 3 * 2.0 ** -134: 0x0002}
    got = O.round_bf16(np.array(list(ties), np.float32), lib)
    assert list(got) == list(ties.values()), f"round_bf16 ties: {[hex(v) for v in got]}"


def _eye_bits(n):
    return f64_to_bf16_bits(np.eye(n))


def pin_chain_identity_first(lib, seed=8, T=7, K=12, M=20):
    """Chain (I, W1): the first operator passes X through exactly, so Y_1 is
    the single product, dX_0 is the bf16 rounding of dX_1 (operator 1's dX)
    and dW_0 = X^T.bf16(dX_1)."""
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    W1 = random_bf16(rng, (K, M), 1 / np.sqrt(K))
    dY = random_bf16(rng, (T, M))
    ys = O.chain_forward(X, [_eye_bits(K), W1], lib)
    assert np.array_equal(ys[0].astype(np.float64), bf16_bits_to_f64(X)), "chain (I, W): Y_0 != X"
    assert np.array_equal(ys[1], O.forward(X, W1, lib)), "chain (I, W): Y_1 != X.W"
    dx, dws = O.chain_backward(X, [_eye_bits(K), W1], dY, lib)
    dx1 = O.backward_dx(dY, W1, lib)
    dy0 = O.round_bf16(dx1, lib)
    assert np.array_equal(dx.astype(np.float64), bf16_bits_to_f64(dy0)), "chain (I, W): dX_0 != bf16(dX_1)"
    assert not np.array_equal(dx, dx1), "chain (I, W): the dY between operators was not rounded"
    assert np.array_equal(dws[1], O.backward_dw(X, dY, lib)), "chain (I, W): dW_1"
    assert np.array_equal(dws[0], O.backward_dw(X, dy0, lib)), "chain (I, W): dW_0"


def pin_chain_identity_last(lib, seed=9, T=9, K=14, M=22):
    """Chain (W0, I): Y_1 is the bf16 rounding of Y_0, dX_1 = dY exactly, so
    dX_0 = dY.W0^T and dW_1 = bf16(Y_0)^T.dY."""
    rng = np.random.default_rng(seed)
    X = random_bf16(rng, (T, K))
    W0 = random_bf16(rng, (K, M), 1 / np.sqrt(K))
    dY = random_bf16(rng, (T, M))
    ys = O.chain_forward(X, [W0, _eye_bits(M)], lib)
    y0 = O.round_bf16(ys[0], lib)
    assert np.array_equal(ys[1].astype(np.float64), bf16_bits_to_f64(y0)), "chain (W, I): Y_1 != bf16(Y_0)"
    dx, dws = O.chain_backward(X, [W0, _eye_bits(M)], dY, lib)
    assert np.array_equal(dx, O.backward_dx(dY, W0, lib)), "chain (W, I): dX_0 != dY.W0^T"
    assert np.array_equal(dws[0], O.backward_dw(X, dY, lib)), "chain (W, I): dW_0"
    assert np.array_equal(dws[1], O.backward_dw(y0, dY, lib)), "chain (W, I): dW_1"


ALL_PINS = [pin_brute_force, pin_integer_exact, pin_identity, pin_concatenation,
            pin_adjoint, pin_sampled, pin_sampled_brute_force, pin_round_bf16,
            pin_chain_identity_first, pin_chain_identity_last]
