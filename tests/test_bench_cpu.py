"""Host logic of bench.py that needs no GPU: the timeline summary's interval
arithmetic, the dX tile-group rule the resident reference follows, and the
extension guard."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _ev(kind, tile, a, b):
    return {"kind": kind, "tile": tile, "start_ms": a, "end_ms": b}


def test_timeline_summary_by_hand():
    tr = [_ev("fwd_gemm", 0, 1.0, 3.0), _ev("h2d", 0, 0.0, 1.0), _ev("h2d", 1, 1.0, 2.0), _ev("d2h", 1, 1.5, 2.5)]
    s = bench.timeline_summary(tr)
    assert s["span_ms"] == 3.0
    assert s["gemm_busy_pct"] == pytest.approx(66.7, abs=0.05)
    assert s["h2d_busy_pct"] == pytest.approx(66.7, abs=0.05)
    assert s["d2h_busy_pct"] == pytest.approx(33.3, abs=0.05)
    assert s["both_links_under_gemm_pct"] == pytest.approx(16.7, abs=0.05)  # [1.5, 2] under [1, 3]
    assert s["copy_outside_gemm_pct"] == pytest.approx(33.3, abs=0.05)    # [0, 1]
    assert s["copies_started_before_the_call"] == 0


def test_timeline_summary_clips_copies_before_the_call():
    """A copy fetched under the previous call counts from the call's start."""
    tr = [_ev("fwd_gemm", 0, 0.0, 2.0), _ev("h2d", 0, -1.0, 0.5), _ev("h2d", 1, -3.0, -2.0)]
    s = bench.timeline_summary(tr)
    assert s["span_ms"] == 2.0
    assert s["h2d_busy_pct"] == pytest.approx(25.0)
    assert s["copy_outside_gemm_pct"] == 0.0
    assert s["copies_started_before_the_call"] == 2
    assert bench.timeline_summary([]) == {}


def test_union_and_overlap():
    assert bench._union([(3, 4), (0, 1), (0.5, 2), (2, 2.5)]) == [[0, 2.5], [3, 4]]
    assert bench._overlap([[0, 2], [3, 5]], [[1, 4]]) == pytest.approx(2.0)
    assert bench._overlap([], [[0, 1]]) == 0.0


@pytest.mark.parametrize("d,N,Mi,g", [(2, 8, 4096, 2), (2, 8, 1024, 2), (3, 16, 1024, 3), (4, 16, 1024, 4),
                                      (9, 16, 256, 4), (0, 8, 4096, 1), (1, 4, 256, 1), (1, 16, 6400, 1),
                                      (5, 1, 4096, 1), (2, 8, 100, 1), (4, 8, 8192, 2), (3, 3, 1024, 2)])
def test_dx_group_rule(d, N, Mi, g):
    """max(2, ceil(8192 / Mi)) bounded by d, N and 4 (d clamped to N - 1);
    one tile when the ring holds at most two tiles or Mi is not a multiple
    of 64."""
    assert bench.dx_group(d, N, Mi) == g


class _OneRank:
    world = 1


class _TwoRanks:
    world = 2


def test_extension_guard_reports_host_failures_on_one_rank():
    def fails():
        raise OSError(22, "direct I/O not supported")
    out = bench._extension(fails, _OneRank())
    assert "unavailable" in out and "OSError" in out["unavailable"]
    assert bench._extension(lambda: {"value": 1.0}, _OneRank()) == {"value": 1.0}


def test_extension_guard_reraises_with_several_ranks_and_on_cuda_errors():
    from offload_streamed_gb300 import tiled_linear as tl

    def io():
        raise OSError(5, "I/O error")
    with pytest.raises(OSError):
        bench._extension(io, _TwoRanks())

    def cuda():
        raise tl.TiledLinearError(tl.TL_ERR_CUDA, "x")
    with pytest.raises(tl.TiledLinearError):
        bench._extension(cuda, _OneRank())


def test_block_sizes():
    """Per-config blocks: at least the given counts, and at least 0.3 s of
    timed steps after 0.15 s of warm-up."""
    assert bench.block_sizes(8.0, 6, 2) == (38, 19)        # an 8 ms step: 0.3 s and 0.15 s decide
    assert bench.block_sizes(250.0, 6, 2) == (6, 2)        # a 250 ms step: the minimum counts decide
    assert bench.block_sizes(0.0, 6, 2) == (300, 150)      # a zero reading counts as 1 ms
    s, w = bench.block_sizes(23.0, 6, 2)
    assert s * 23.0 >= 300.0 and w * 23.0 >= 150.0 and (s - 1) * 23.0 < 300.0
