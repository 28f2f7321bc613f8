"""The launch and copy timeline (tiled_linear_get_trace) of real calls, and
the pipeline's ordering rules checked on it: a GEMM starts after its tile has
landed, no more tiles are in flight than the ring has slots, launches on the
caller's stream do not overlap, a dW write-back starts after its GEMM, and a
dX launch starts after the last tile of its group has landed."""
import pytest
import torch

from offload_streamed_gb300 import inputs as I

pytestmark = pytest.mark.gpu

EPS = 1e-3  # ms: events of different streams read one device clock


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def _op(tl, K, M, N, d):
    w, dw = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, 1)
    return tl.TiledLinear(K, M, N, d, w, dw, tile_major=True), (w, dw)


def _by(trace, kind):
    return {e["tile"]: e for e in trace if e["kind"] == kind}


def _steps(op, T, K, M, calls=2):
    x, dy = I.make_x(T, K, 2).cuda(), I.make_dy(T, M, 3).cuda()
    for _ in range(calls):
        op.forward(x)
        op.backward(x, dy)
    torch.cuda.synchronize()


@pytest.mark.parametrize("N,d", [(8, 2), (5, 1), (6, 3)])
def test_forward_and_backward_timelines_follow_the_pipeline(tl, N, d):
    T, K, Mi = 256, 512, 512
    M = N * Mi
    op, bufs = _op(tl, K, M, N, d)
    _steps(op, T, K, M)
    fwd, bwd = op.trace(False), op.trace(True)
    # forward: one GEMM and one copy per tile
    g, h = _by(fwd, "fwd_gemm"), _by(fwd, "h2d")
    assert sorted(g) == list(range(N)) and sorted(h) == list(range(N))
    for e in fwd:
        assert e["end_ms"] >= e["start_ms"]
        if e["kind"] == "fwd_gemm":  # a copy may run ahead of the call (it waits only for its slot)
            assert e["start_ms"] >= -EPS
    for i in range(N):
        assert g[i]["start_ms"] >= h[i]["end_ms"] - EPS, i  # the GEMM waits for its tile
        if i:
            assert g[i]["start_ms"] >= g[i - 1]["end_ms"] - EPS  # one stream: no overlap
    # in flight (copy started, GEMM not done) never more than the forward's slots:
    # d + 1 ring slots plus the two dW staging slots it borrows
    slots = d + 1 + min(2, N)
    for i in range(N):
        t = h[i]["start_ms"] + EPS
        assert sum(1 for j in range(N) if h[j]["start_ms"] <= t < g[j]["end_ms"]) <= slots, i
    # backward: dW and write-back per tile, dX per group, copies descending
    dwg, dxg, bh, bd = (_by(bwd, k) for k in ("dw_gemm", "dx_gemm", "h2d", "d2h"))
    assert sorted(dwg) == sorted(bd) == sorted(bh) == list(range(N))
    st = op.stats()
    assert len(dxg) == st["bwd_launches"] - N
    for i in range(N):
        assert bd[i]["start_ms"] >= dwg[i]["end_ms"] - EPS, i  # the write-back waits for its dW
    for i, e in dxg.items():
        assert e["start_ms"] >= bh[i]["end_ms"] - EPS, i  # the group's lowest tile lands last
    gemms = [e for e in bwd if e["kind"] in ("dw_gemm", "dx_gemm")]
    for a, b in zip(gemms, gemms[1:]):
        assert b["start_ms"] >= a["end_ms"] - EPS
    assert op.close() == tl.TL_OK
    for b in bufs:
        b.close()


def test_reused_tiles_have_no_copy(tl):
    T, K, M, N, d = 128, 512, 4096, 8, 2
    op, bufs = _op(tl, K, M, N, d)
    op.set_tile_reuse(True)
    _steps(op, T, K, M)
    bh = _by(op.trace(True), "h2d")
    assert sorted(bh) == list(range(N - (d + 1)))  # the forward's last d+1 tiles stayed in the ring
    assert op.close() == tl.TL_OK
    for b in bufs:
        b.close()


def test_no_timed_call_gives_an_empty_trace(tl):
    op, bufs = _op(tl, 256, 1024, 2, 1)
    assert op.trace(False) == [] and op.trace(True) == []
    assert op.close() == tl.TL_OK
    for b in bufs:
        b.close()
