"""Comparison rules for GPU outputs against the CPU oracle.

Two bars, both asserted:
* the stated tolerance: max |gpu - oracle| <= 2e-2 * max |oracle| per tensor;
* a per-element bound derived from the arithmetic.  The GPU and the oracle
  both accumulate exact bf16 x bf16 products in fp32, in different orders, so
  each is within gamma_n * S of the exact sum (S = sum of |terms|, gamma_n =
  n u / (1 - n u), u = 2^-24).  bf16 outputs are then rounded to nearest even
  (relative error <= 2^-9).  The bound used is
      |gpu - oracle| <= 2^-8 |oracle| + 4 gamma_n S   (bf16 outputs)
      |gpu - oracle| <= 4 gamma_n S                   (fp32 outputs)
  with a factor 2 of slack on the accumulation term for tensor-core
  accumulation that truncates instead of rounding.
"""
from __future__ import annotations

import numpy as np

STATED_REL_TOL = 2e-2


def gamma(n: int) -> float:
    u = 2.0 ** -24
    return n * u / (1 - n * u)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check(name: str, got: np.ndarray, ref: np.ndarray, S: np.ndarray | None, n: int, bf16_out: bool):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite GPU values"
    err = np.abs(got - ref)
    max_ref = float(np.max(np.abs(ref))) if ref.size else 0.0
    assert float(err.max(initial=0.0)) <= STATED_REL_TOL * max_ref + 1e-30, \
        f"{name}: max err {err.max():.3e} > {STATED_REL_TOL} * {max_ref:.3e}"
    if S is not None:
        bound = (2.0 ** -8 * np.abs(ref) if bf16_out else 0.0) + 4 * gamma(n) * np.asarray(S, np.float64) + 1e-30
        bad = err > bound
        if bad.any():
            i = int(np.flatnonzero(bad.ravel())[0])
            raise AssertionError(f"{name}: {int(bad.sum())} entries beyond the element bound; first flat "
                                 f"index {i}: gpu {got.ravel()[i]!r} oracle {ref.ravel()[i]!r} "
                                 f"bound {np.broadcast_to(bound, err.shape).ravel()[i]:.3e}")
    return float(err.max(initial=0.0)), max_ref
