"""The closed forms against brute force, the schedule model and the pages'
efficiency rule; planted mistakes in a copy of them must be caught; the
benchmark's accounting (``offload_streamed_gb300.roofline``) must agree with
them and with the model."""
import importlib.util
import os

import pytest

import closed_form_pins as P
import schedule_sim as S
from oracle import closed_forms as CF
from offload_streamed_gb300 import roofline as RL

SRC = os.path.join(os.path.dirname(CF.__file__), "closed_forms.py")


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_closed_form_pin(pin):
    pin(CF)


MUTANTS = {
    "h2d_fetched_once": ("    return 2 * linear_weight_bytes(K, M)", "    return linear_weight_bytes(K, M)"),
    "d2h_written_twice": ('    """dW (2 bytes per weight) is written back once per step."""\n'
                          "    return linear_weight_bytes(K, M)",
                          '    """dW (2 bytes per weight) is written back once per step."""\n'
                          "    return 2 * linear_weight_bytes(K, M)"),
    "roofline_swaps_links": ("    return max(flops / R, linear_h2d_bytes_fwd_bwd(K, M) / B_h2d,\n"
                             "               linear_d2h_bytes_fwd_bwd(K, M) / B_d2h)",
                             "    return max(flops / R, linear_h2d_bytes_fwd_bwd(K, M) / B_d2h,\n"
                             "               linear_d2h_bytes_fwd_bwd(K, M) / B_h2d)"),
    "roofline_drops_d2h": ("    return max(flops / R, linear_h2d_bytes_fwd_bwd(K, M) / B_h2d,\n"
                           "               linear_d2h_bytes_fwd_bwd(K, M) / B_d2h)",
                           "    return max(flops / R, linear_h2d_bytes_fwd_bwd(K, M) / B_h2d)"),
    "roofline_min_not_max": ("    return max(flops / R, linear_h2d_bytes_fwd_bwd(K, M) / B_h2d,",
                             "    return min(flops / R, linear_h2d_bytes_fwd_bwd(K, M) / B_h2d,"),
    "backward_flops_halved": ("    return 4 * T * K * M", "    return 2 * T * K * M"),
    "forward_flops_halved": ("def linear_flops_forward(T: int, K: int, M: int) -> int:\n    return 2 * T * K * M",
                             "def linear_flops_forward(T: int, K: int, M: int) -> int:\n    return T * K * M"),
    "efficiency_inverted": ("    return min(1.0, ait_value / machine_balance(R, BW))",
                            "    return min(1.0, machine_balance(R, BW) / ait_value)"),
}


def _load_copy(path):
    spec = importlib.util.spec_from_file_location("closed_forms_mutant", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_closed_form_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "closed_forms_mutant.py"
    path.write_text(src.replace(old, new))
    mod = _load_copy(str(path))
    failures = []
    for pin in P.ALL_PINS:
        try:
            pin(mod)
        except AssertionError as e:
            failures.append(f"{pin.__name__}: {str(e)[:80]}")
    assert failures, f"no pin caught mutant {name}"


SHAPES = [(256, 1024, 4096), (8192, 8192, 32768), (4096, 25600, 102400), (2048, 65536, 262144),
          (65536, 16384, 65536), (1, 8, 8)]


@pytest.mark.parametrize("T,K,M", SHAPES)
def test_bench_accounting_matches_closed_forms(T, K, M):
    assert RL.step_flops(T, K, M) == CF.linear_flops_forward(T, K, M) + CF.linear_flops_backward(T, K, M)
    assert RL.step_h2d_bytes(K, M) == CF.linear_h2d_bytes_fwd_bwd(K, M)
    assert RL.step_d2h_bytes(K, M) == CF.linear_d2h_bytes_fwd_bwd(K, M)
    assert RL.ait_h2d(T) == CF.ait(RL.step_flops(T, K, M), CF.linear_h2d_bytes_fwd_bwd(K, M))
    for R, bh, bd in [(1.936e15, 2.1e11, 1.9e11), (1.936e15, 2e9, 1.9e11), (1e12, 2.1e11, 1e8)]:
        t, bound = RL.step_bound(T, K, M, R, bh, bd)
        assert t == pytest.approx(CF.roofline_seconds(T, K, M, R, bh, bd), rel=1e-15)
        assert bound in ("tensor", "h2d", "d2h")
    # the crossover is where compute and the host->device link take equally long
    R, bh = 1.936e15, 2.1e11
    Tx = RL.crossover_tokens(R, bh)
    assert CF.linear_flops_forward(Tx, K, M) * 3 / R == pytest.approx(CF.linear_h2d_bytes_fwd_bwd(K, M) / bh)


@pytest.mark.parametrize("T,R,bh,bd", [(8192, 1.5e15, 2e11, 1.8e11), (256, 1.5e15, 2e11, 1.8e11),
                                        (4096, 1.5e15, 2e11, 1.5e10)])
def test_phase_bound_matches_phase_serial_schedule(T, R, bh, bd):
    """Forward and backward summed separately: the schedule model with a
    barrier between phases, a deep ring and ample staging reaches it within 1 %."""
    K, M, N, steps = 1024, 4096 * 8, 128, 4
    t_f, t_b = RL.phase_bound(T, K, M, R, bh, bh, bd)
    sim = S.simulate(T, K, M, N, N - 1, R, bh, bd, steps, staging=4 * N, phase_barrier=True)["seconds"] / steps
    assert t_f + t_b <= sim * (1 + 1e-12)
    assert sim <= 1.01 * (t_f + t_b), (sim, t_f + t_b)
    assert t_f + t_b >= RL.step_bound(T, K, M, R, bh, bd)[0] * (1 - 1e-12)


@pytest.mark.parametrize("h,d,bh,bd,bb", [(5e9, 2e9, 2.1e11, 1.9e11, 1.7e11), (1e9, 3e9, 2.1e11, 1.9e11, 1.7e11),
                                         (4e9, 4e9, 2e11, 2e11, 1.2e11), (3e9, 0.0, 2e11, 1e11, 1e11)])
def test_link_seconds_is_the_best_time_sharing_schedule(h, d, bh, bd, bb):
    """Brute force over schedules that spend t_c with both directions running
    (B_bidir each), t_h with host->device alone and t_d with device->host
    alone: the least t_c + t_h + t_d that moves both amounts."""
    best = float("inf")
    top = min(h, d) / bb
    for j in range(2001):
        t_c = top * j / 2000
        t = t_c + max(0.0, h - bb * t_c) / bh + max(0.0, d - bb * t_c) / bd
        best = min(best, t)
    assert RL.link_seconds(h, d, bh, bd, bb) == pytest.approx(best, rel=1e-9)


def test_e2e_bound():
    T, K, M, R = 2048, 65536, 262144, 1.936e15
    bh, bd, bb = 2.1e11, 1.92e11, 1.7e11
    w = 2.0 * K * M
    # no activations: the per-phase bound's link time (W in alone, then W in and dW out together)
    t_f, t_b = RL.phase_bound(T, K, M, R, bh, bb, bb)
    assert RL.e2e_bound(T, K, M, R, 0.0, 0.0, bh, bd, bb) == pytest.approx(t_f + t_b, rel=1e-12)
    # activations: X, dY in and Y, dX (fp32) out, each byte at the rate of the direction it shares
    a_in, a_out = 2.0 * T * (K + M), 2.0 * T * M + 4.0 * T * K
    t = RL.e2e_bound(T, K, M, R, a_in, a_out, bh, bd, bb)
    assert t == pytest.approx((w + a_out) / bb + (2 * w + a_in - w - a_out) / bh, rel=1e-12)
    # compute-bound: the FLOPs at R
    assert RL.e2e_bound(65536, 1024, 1024, 1e12, 1.0, 1.0, bh, bd, bb) == pytest.approx(
        RL.step_flops(65536, 1024, 1024) / 1e12)


def test_gemm_accounting():
    # one tile GEMM of each kind does a third of the tile's step FLOPs
    T, K, M, N = 8192, 8192, 32768, 8
    n = M // N
    assert 3 * N * RL.gemm_flops(T, K, n) == RL.step_flops(T, K, M)
    # operands once, outputs once; dX's fp32 read-modify-write, or its write alone
    assert RL.gemm_bytes("fwd", T, K, n) == 2 * T * K + 2 * K * n + 2 * T * n
    assert RL.gemm_bytes("dx", T, K, 2 * n) - RL.gemm_bytes("dx", T, K, 2 * n, accumulate=False) == 4 * T * K
    with pytest.raises(ValueError):
        RL.gemm_bytes("other", 1, 1, 1)
