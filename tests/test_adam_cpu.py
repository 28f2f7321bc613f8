"""The host optimizer's Adam update (CPU code in the library) against the
fp64 oracle, and the oracle against closed forms of the update."""
import ctypes

import numpy as np
import pytest

from oracle import adam as A
from oracle import oracle as O

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def test_oracle_first_step_is_lr_times_normalised_gradient():
    """From zero moments, bias correction gives mhat = g and vhat = g^2, so the
    first step moves each weight by lr g / (|g| + eps)."""
    rng = np.random.default_rng(0)
    p, g = rng.standard_normal(1000), rng.standard_normal(1000)
    pt, mt, vt = A.adam_step(p, 0 * p, 0 * p, g, 1, **HP)
    assert np.allclose(pt, p - HP["lr"] * g / (np.abs(g) + HP["eps"]), rtol=0, atol=1e-15)
    assert np.allclose(mt, (1 - HP["beta1"]) * g) and np.allclose(vt, (1 - HP["beta2"]) * g * g)


def test_oracle_constant_gradient_moves_linearly():
    """With the same gradient every step, the bias-corrected moments stay g and
    g^2 exactly, so t steps move each weight by t lr g / (|g| + eps)."""
    rng = np.random.default_rng(1)
    p0, g = rng.standard_normal(500), rng.standard_normal(500)
    p, m, v = p0, 0 * p0, 0 * p0
    for t in range(1, 8):
        p, m, v = A.adam_step(p, m, v, g, t, **HP)
    assert np.allclose(p, p0 - 7 * HP["lr"] * g / (np.abs(g) + HP["eps"]), rtol=0, atol=1e-12)


def test_oracle_weight_decay_alone_shrinks_geometrically():
    p0 = np.linspace(-2, 2, 101)
    p, m, v = p0, 0 * p0, 0 * p0
    for t in range(1, 4):
        p, m, v = A.adam_step(p, m, v, 0 * p0, t, lr=0.1, beta1=0.9, beta2=0.99, eps=1e-8, wd=0.5)
    assert np.allclose(p, p0 * (1 - 0.05) ** 3, rtol=1e-14, atol=0)


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    from offload_streamed_gb300 import _build
    _build.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def _run_lib(tl, cfg, step, p, m, v, g_bits, acc=None):
    p, m, v = (np.array(a, np.float32) for a in (p, m, v))
    w = np.zeros(p.shape, np.uint16)
    g_bits = np.ascontiguousarray(g_bits, np.uint16)
    accp = 0
    if acc is not None:
        acc = np.ascontiguousarray(acc, np.float32)
        accp = acc.ctypes.data
    tl.tiled_linear_adam_update(cfg, step, p.size, p.ctypes.data, m.ctypes.data, v.ctypes.data, accp,
                                g_bits.ctypes.data, w.ctypes.data)
    return p, m, v, w


@pytest.mark.parametrize("step,wd,use_acc", [(1, 0.0, False), (3, 0.0, False), (7, 0.01, True), (50, 0.1, False)])
def test_library_update_matches_oracle(tl, step, wd, use_acc):
    rng = np.random.default_rng(step)
    n = 4099
    p = rng.standard_normal(n).astype(np.float32)
    m = (0.01 * rng.standard_normal(n)).astype(np.float32)
    v = (1e-4 * rng.random(n) + 1e-6).astype(np.float32)
    g_bits = O.round_bf16(rng.standard_normal(n).astype(np.float32) * np.float32(0.03))
    acc = (0.02 * rng.standard_normal(n)).astype(np.float32) if use_acc else None
    cfg = tl.adam_config(lr=2e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd)
    P, Mm, V, W = _run_lib(tl, cfg, step, p, m, v, g_bits, acc)
    g = (g_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if use_acc:
        g = g + acc.astype(np.float64)
    pr, mr, vr = A.adam_step(p, m, v, g, step, lr=2e-3, beta1=0.9, beta2=0.95, eps=1e-8, wd=wd)
    # fp32 evaluation of a few operations per element: a few ulps of each
    # term, the update term carrying at most ~1e-5 relative error
    u = 2.0 ** -24
    assert np.all(np.abs(Mm - mr) <= 8 * u * (np.abs(m) + np.abs(g)) + 1e-30)
    assert np.all(np.abs(V - vr) <= 8 * u * (np.abs(v) + g * g) + 1e-30)
    assert np.all(np.abs(P - pr) <= 8 * u * np.abs(p) + 1e-5 * 2e-3 * (1 + np.abs(mr) / np.sqrt(np.abs(vr) + 1e-30)))
    # the bf16 weights are the new master rounded to nearest even
    assert np.array_equal(W, O.round_bf16(P))


def test_library_update_rejects_bad_arguments(tl):
    lib = tl.load()
    cfg = tl.adam_config()
    x = np.zeros(8, np.float32)
    h = np.zeros(8, np.uint16)
    args = (x.ctypes.data, x.ctypes.data, x.ctypes.data, None, h.ctypes.data, h.ctypes.data)
    assert lib.tiled_linear_adam_update(ctypes.byref(cfg), 0, 8, *args) == tl.TL_ERR_INVALID   # step < 1
    bad = tl.adam_config(beta1=1.0)
    assert lib.tiled_linear_adam_update(ctypes.byref(bad), 1, 8, *args) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_adam_update(ctypes.byref(cfg), 1, 8, None, *args[1:]) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_adam_update(ctypes.byref(cfg), 1, 0, *args) == tl.TL_OK
    assert lib.tiled_linear_optimizer_step(None) == tl.TL_ERR_STATE
    assert lib.tiled_linear_optimizer_destroy(None) == tl.TL_OK
