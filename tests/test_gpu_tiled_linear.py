"""The streamed tiled linear operator end to end through the C ABI (host W in
pinned memory, depth-d ring, copy streams) against the CPU oracle."""
import math

import numpy as np
import pytest
import torch

from offload_streamed_gb300 import inputs as I
from oracle import oracle as O
from gpu_check import bf16_bits_to_f64, check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


class Run:
    pass


def make_op(tl, K, M, N, d, w, dw, tile_major=True):
    return tl.TiledLinear(K, M, N, d, w, dw, tile_major=tile_major)


def run_op(tl, T, K, M, N, d, tile_major=True, seed=0, kind="normal", calls=1, stream=None,
           reuse=False, extra_backward=False):
    r = Run()
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, tile_major, seed, kind=kind)
    dw.tensor.view(torch.int16).fill_(0x7FC0)  # NaN: catches tiles never written
    x = I.make_x(T, K, seed, kind=kind)
    dy = I.make_dy(T, M, seed, kind=kind)
    op = make_op(tl, K, M, N, d, w, dw, tile_major=tile_major)
    if reuse:
        op.set_tile_reuse(True)
    xd, dyd = x.cuda(), dy.cuda()
    s = stream or torch.cuda.current_stream()
    with torch.cuda.stream(s):
        for _ in range(calls):
            y = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
            dx = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
            op.forward(xd, y, stream=s)
            op.backward(xd, dyd, dx, stream=s)
            if extra_backward:  # a second backward with no forward between
                dx.fill_(float("nan"))
                op.backward(xd, dyd, dx, stream=s)
    s.synchronize()
    r.stats = op.stats()
    r.y = y.cpu()
    r.dx = dx.cpu()
    r.dw = I.w_logical(dw.tensor, K, M, N, tile_major).clone()
    r.x, r.dy = x, dy
    r.W = I.w_logical(w.tensor, K, M, N, tile_major).contiguous().clone()
    assert op.close() == tl.TL_OK
    w.close()
    dw.close()
    return r


def oracle_check(r, T, K, M):
    xb, wb, dyb = I.bits(r.x), I.bits(r.W), I.bits(r.dy)
    xa, wa, dya = (np.abs(bf16_bits_to_f64(b)) for b in (xb, wb, dyb))
    check("Y", r.y.float().numpy(), O.forward(xb, wb), xa @ wa, K, True)
    dX, dW = O.backward(xb, wb, dyb)
    check("dX", r.dx.numpy(), dX, dya @ wa.T, M, False)
    check("dW", r.dw.float().numpy(), dW, xa.T @ dya, T, True)


@pytest.mark.parametrize("tile_major", [True, False], ids=["tilemajor", "rowmajor"])
def test_tiny_config_full_parity(tl, tile_major):
    """X [256,1024], W [1024,4096] in N=4 tiles, dY [256,4096], d=1."""
    T, K, M, N, d = 256, 1024, 4096, 4, 1
    r = run_op(tl, T, K, M, N, d, tile_major=tile_major)
    oracle_check(r, T, K, M)
    st = r.stats
    # one dW launch per tile, one dX launch per group of tiles
    g = dx_group(d, N, M // N)
    assert st["fwd_launches"] == N and st["bwd_launches"] == N + (N + g - 1) // g
    assert st["staging_slots"] == 2
    assert st["fwd_h2d_bytes"] == K * M * 2 and st["bwd_h2d_bytes"] == K * M * 2
    assert st["bwd_d2h_bytes"] == K * M * 2
    assert st["depth"] == d


def test_integer_exact(tl):
    """X, W, dY in {-1,0,1}, T = K = 128, M = 1024, N = 4: every GPU output
    equals the integer product exactly."""
    T, K, M, N = 128, 128, 1024, 4
    r = run_op(tl, T, K, M, N, 1, kind="ternary", seed=3)
    xi = r.x.float().numpy().astype(np.int64)
    wi = r.W.float().numpy().astype(np.int64)
    dyi = r.dy.float().numpy().astype(np.int64)
    assert np.array_equal(r.y.float().numpy().astype(np.int64), xi @ wi)
    assert np.array_equal(r.dx.numpy().astype(np.int64), dyi @ wi.T)
    assert np.array_equal(r.dw.float().numpy().astype(np.int64), xi.T @ dyi)


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                       b.contiguous().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


def dx_group(depth, N, Mi):
    """Tiles per dX accumulation group for the depth a call ran with (from its
    stats): the engine reduces dX over groups of
    min(max(2, ceil(8192 / Mi)), depth, N, 4) tiles whenever the ring holds
    more than two (depth >= 2) and the tile width is a multiple of 64;
    otherwise one tile at a time."""
    if not (depth >= 2 and N >= 2 and Mi % 64 == 0):
        return 1
    return min(max(2, -(-8192 // Mi)), depth, N, 4)


def test_schedule_does_not_change_results(tl):
    """Depth, host layout and repeated calls change only the schedule: Y and dW
    are bit-identical for every schedule; dX (an fp32 sum whose grouping is
    part of the schedule) is bit-identical among schedules with the same dX
    grouping and matches the oracle for every one."""
    T, K, M, N = 200, 264, 2048, 8
    base = {g: run_op(tl, T, K, M, N, g if g > 1 else 0, tile_major=True, seed=7) for g in (1, 2, 3, 4)}
    for g, r in base.items():
        assert dx_group(r.stats["depth"], N, M // N) == g
        oracle_check(r, T, K, M)
    for d, tm, calls in [(0, True, 1), (2, True, 1), (3, False, 1), (7, True, 2), (12, False, 1), (-1, True, 3),
                         (1, True, 1), (0, False, 2), (5, True, 1), (-1, False, 2)]:
        r = run_op(tl, T, K, M, N, d, tile_major=tm, seed=7, calls=calls)
        ref = base[dx_group(r.stats["depth"], N, M // N)]
        assert _same(r.y, ref.y), (d, tm)
        assert _same(r.dw, ref.dw), (d, tm)
        assert _same(r.dx, ref.dx), (d, tm)


def test_dx_grouping_matches_oracle_for_odd_tile_counts(tl):
    """N odd: the last dX group holds a single tile."""
    T, K, M = 160, 512, 5 * 512
    for d in (1, 2, 4):
        r = run_op(tl, T, K, M, 5, d, seed=13)
        oracle_check(r, T, K, M)


def test_tiled_forward_bit_exact_vs_untiled(tl):
    """The same logical W split into N = 1, 2, 4, 16 tiles: Y is bit-identical
    to the untiled (N = 1) product, and so is dW (each dW column is reduced
    over T by one CTA either way); dX sums its tiles in a different order and
    is only close."""
    T, K, M = 320, 512, 4096
    w16 = run_op(tl, T, K, M, 16, 1, seed=12)
    outs = {N: run_with_logical_w(tl, w16.W, w16.x, w16.dy, N) for N in (1, 2, 4, 16)}
    for N in (2, 4, 16):
        assert _same(outs[N][0], outs[1][0]), N
        assert _same(outs[N][2], outs[1][2]), N
        dx1 = outs[1][1].numpy()
        assert np.allclose(outs[N][1].numpy(), dx1, rtol=1e-4, atol=1e-4 * np.abs(dx1).max())
    assert _same(outs[16][0], w16.y)


def run_with_logical_w(tl, W, x, dy, N, d=1):
    K, M = W.shape
    T = x.shape[0]
    Mi = M // N
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    w.tensor.view(N, K, Mi).copy_(W.view(K, N, Mi).permute(1, 0, 2))
    op = tl.TiledLinear(K, M, N, d, w, dw, tile_major=True)
    xd, dyd = x.cuda(), dy.cuda()
    y = op.forward(xd)
    dx = op.backward(xd, dyd)
    torch.cuda.synchronize()
    out = (y.cpu(), dx.cpu(), I.w_logical(dw.tensor, K, M, N, True).clone())
    op.close()
    w.close()
    dw.close()
    return out


@pytest.mark.parametrize("T", [1, 129, 383])
def test_ragged_token_counts(tl, T):
    K, M, N = 256, 1536, 3
    r = run_op(tl, T, K, M, N, 1, seed=T)
    oracle_check(r, T, K, M)


@pytest.mark.parametrize("K,M,N", [(264, 1200, 3), (520, 776, 1), (264, 960, 3)])
def test_ragged_tile_width_runs_per_tile(tl, K, M, N):
    """Tile widths that are not a multiple of 256 run one launch per tile;
    a width of 320 (five 64-deep K-blocks) still pairs the dX tiles."""
    T = 150
    r = run_op(tl, T, K, M, N, 1, seed=K)
    oracle_check(r, T, K, M)


def test_zero_tokens(tl):
    """T = 0: forward does nothing; backward writes dW = 0 (an empty sum)."""
    K, M, N = 64, 512, 2
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, 0)
    dw.tensor.view(torch.int16).fill_(0x7FC0)
    op = tl.TiledLinear(K, M, N, 1, w, dw)
    x = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    dy = torch.empty(0, M, dtype=torch.bfloat16, device="cuda")
    op.forward(x)
    op.backward(x, dy)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw.tensor.float()) == 0
    op.close()
    w.close()
    dw.close()


def test_side_stream_and_default_stream(tl):
    T, K, M, N = 128, 256, 1024, 4
    side = torch.cuda.Stream()
    a = run_op(tl, T, K, M, N, 1, seed=5, stream=side)
    b = run_op(tl, T, K, M, N, 1, seed=5)
    assert _same(a.y, b.y) and _same(a.dx, b.dx) and _same(a.dw, b.dw)


def test_stats_are_consistent(tl):
    T, K, M, N = 512, 1024, 8192, 8
    r = run_op(tl, T, K, M, N, 2, seed=1, calls=2)
    st = r.stats
    assert st["fwd_valid"] == 1 and st["bwd_valid"] == 1
    assert st["n_tiles"] == N and st["depth"] == 2
    assert st["fwd_calls"] == 2 and st["bwd_calls"] == 2
    for k in ("fwd_total_ms", "fwd_gemm_ms", "fwd_h2d_ms", "bwd_total_ms", "bwd_gemm_ms", "bwd_h2d_ms",
              "bwd_d2h_ms"):
        assert st[k] > 0, k
    assert st["bwd_launches"] == N + (N + 1) // 2  # d = 2: pairs
    assert st["bwd_dw_gemm_ms"] > 0 and st["bwd_dx_gemm_ms"] > 0
    assert abs(st["bwd_dw_gemm_ms"] + st["bwd_dx_gemm_ms"] - st["bwd_gemm_ms"]) < 1e-3
    assert 0 < st["fwd_h2d_max_ms"] <= st["fwd_h2d_ms"] + 1e-3
    assert st["fwd_gemm_ms"] <= st["fwd_total_ms"] + 1e-3
    assert st["bwd_gemm_ms"] <= st["bwd_total_ms"] + 1e-3


def test_auto_depth_picks_within_ring(tl):
    """With room for every tile, the default stall allowance (50 ms, far more
    than these tiles' GEMMs take) keeps every tile in the ring, and every
    staging slot is used; results match the oracle."""
    T, K, M, N = 256, 1024, 8192, 8
    r = run_op(tl, T, K, M, N, -1, seed=2, calls=2)
    assert r.stats["depth"] == N - 1 and r.stats["staging_slots"] == N
    oracle_check(r, T, K, M)


def _auto_op(tl, K, M, N, seed, **kw):
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed)
    return tl.TiledLinear(K, M, N, -1, w, dw, **kw), w, dw


def test_auto_depth_rule_and_workspace_bound(tl):
    """Without a stall allowance the rule d = ceil(t_fetch / t_layer) is
    applied to the first forward's slowest copy and mean GEMM time (recorded
    in the stats); the smallest workspace allowed gives d = 1 and two staging
    slots."""
    T, K, M, N = 512, 2048, 8 * 1024, 8
    x = I.make_x(T, K, 4).cuda()
    op, w, dw = _auto_op(tl, K, M, N, 4)
    op.set_stall_allowance(0.0)
    y1 = op.forward(x)
    st1 = op.stats()
    y2 = op.forward(x)  # the depth is chosen before this call
    torch.cuda.synchronize()
    st = op.stats()
    t_layer = st1["fwd_gemm_ms"] / N
    want = max(1, min(N - 1, math.ceil(st1["fwd_h2d_max_ms"] / t_layer)))
    assert st["depth"] == want, (st1, st)
    assert _same(y1.cpu(), y2.cpu())
    with pytest.raises(tl.TiledLinearError):
        op.set_stall_allowance(-1.0)
    op.close()
    least = tl.tiled_linear_workspace_bytes(K, M, N, 1)
    small, w2, dw2 = _auto_op(tl, K, M, N, 4, auto_workspace_bytes=least)
    y3 = small.forward(x)
    small.forward(x)
    torch.cuda.synchronize()
    st = small.stats()
    assert st["depth"] == 1 and st["staging_slots"] == 2
    assert _same(y3.cpu(), y1.cpu())
    small.close()
    for b in (w, dw, w2, dw2):
        b.close()


def test_not_pinned_is_rejected(tl):
    K, M, N = 64, 256, 2
    w = torch.zeros(K * M, dtype=torch.bfloat16)  # pageable host memory
    dw = tl.PinnedBuffer(K * M)
    ws = torch.empty(tl.tiled_linear_workspace_bytes(K, M, N, 1), dtype=torch.uint8, device="cuda")
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.tiled_linear_create(K, M, N, 1, w.data_ptr(), dw.ptr, ws.data_ptr(), ws.numel(), 0)
    assert ei.value.status == tl.TL_ERR_NOT_PINNED
    dw.close()


def test_host_workspace_is_rejected(tl):
    K, M, N = 64, 256, 2
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    nb = tl.tiled_linear_workspace_bytes(K, M, N, 1)
    ws = tl.PinnedBuffer(nb, dtype=torch.uint8)
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.tiled_linear_create(K, M, N, 1, w.ptr, dw.ptr, ws.ptr, nb, 0)
    assert ei.value.status == tl.TL_ERR_WORKSPACE
    for b in (w, dw, ws):
        b.close()


@pytest.mark.parametrize("N,d,calls", [(8, 2, 2), (5, 1, 2), (4, 0, 2), (3, 7, 1), (6, 3, 3), (8, -1, 3)])
def test_tile_reuse_is_bit_identical_and_skips_fetches(tl, N, d, calls):
    """With tile reuse on, the backward takes the last min(d+1, N) tiles from
    the ring instead of fetching them again: same bits, fewer H2D bytes."""
    T, K, Mi = 192, 512, 512
    M = N * Mi
    ref = run_op(tl, T, K, M, N, d, seed=21, calls=calls)
    r = run_op(tl, T, K, M, N, d, seed=21, calls=calls, reuse=True)
    assert _same(r.y, ref.y) and _same(r.dw, ref.dw) and _same(r.dx, ref.dx)
    oracle_check(r, T, K, M)
    want = min(r.stats["depth"] + 1, N)
    assert r.stats["bwd_reused_tiles"] == want
    assert r.stats["bwd_h2d_bytes"] == (N - want) * K * Mi * 2
    assert ref.stats["bwd_reused_tiles"] == 0 and ref.stats["bwd_h2d_bytes"] == N * K * Mi * 2


def test_tile_reuse_after_a_backward_refetches(tl):
    """After a backward the ring holds the first tiles, not the ones a
    backward starts with: the next backward fetches everything again."""
    T, K, M, N = 160, 512, 4 * 512, 4
    ref = run_op(tl, T, K, M, N, 1, seed=5, calls=2, extra_backward=True)
    r = run_op(tl, T, K, M, N, 1, seed=5, calls=2, reuse=True, extra_backward=True)
    assert _same(r.y, ref.y) and _same(r.dw, ref.dw) and _same(r.dx, ref.dx)
    assert r.stats["bwd_reused_tiles"] == 0
    oracle_check(r, T, K, M)


def test_sampled_timing_counts_and_results(tl):
    """Timing every third call: all calls counted, three of seven timed, the
    results unchanged."""
    T, K, M, N = 128, 512, 2048, 4
    ref = run_op(tl, T, K, M, N, 1, seed=3, calls=1)
    w, dw = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, 3)
    op = make_op(tl, K, M, N, 1, w, dw)
    op.set_timing(3)
    xd, dyd = ref.x.cuda(), ref.dy.cuda()
    for _ in range(7):
        y = op.forward(xd)
        dx = op.backward(xd, dyd)
    torch.cuda.synchronize()
    st = op.stats()
    assert st["fwd_calls"] == 7 and st["bwd_calls"] == 7
    assert st["fwd_timed_calls"] == 3 and st["bwd_timed_calls"] == 3 and st["timing_every"] == 3
    assert st["fwd_gemm_ms"] > 0 and st["sum_fwd_gemm_ms"] > 0
    assert _same(y.cpu(), ref.y) and _same(dx.cpu(), ref.dx)
    with pytest.raises(tl.TiledLinearError) as ei:
        op.set_timing(0)
    assert ei.value.status == tl.TL_ERR_INVALID
    assert op.close() == tl.TL_OK
    w.close()
    dw.close()
