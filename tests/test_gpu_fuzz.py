"""Seeded random schedules against the oracle: operator shapes, tile counts,
ring depths, host layouts, repeated calls, tile reuse and chains drawn at
random (small sizes, so the oracle runs in full).  Catches scheduling slips
(slot order, dX pairing, reuse prefixes, operator boundaries) that a fixed
list of shapes could miss."""
import numpy as np
import pytest
import torch

from offload_streamed_gb300 import inputs as I
from oracle import oracle as O
from gpu_check import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def _draw(rng):
    N = int(rng.integers(1, 7))
    Mi = 8 * int(rng.integers(1, 49))          # 8 .. 384, ragged against 64 and 256
    K = 8 * int(rng.integers(1, 65))           # 8 .. 512
    T = int(rng.integers(1, 300))
    d = int(rng.integers(-1, N + 2))
    return T, K, N * Mi, N, d


@pytest.mark.parametrize("seed", range(24))
def test_random_single_operator_schedules(tl, seed):
    rng = np.random.default_rng(1000 + seed)
    T, K, M, N, d = _draw(rng)
    tile_major = bool(rng.integers(0, 2))
    reuse = bool(rng.integers(0, 2)) and tile_major
    calls = int(rng.integers(1, 4))
    w, dw = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, tile_major, seed)
    dw.tensor.view(torch.int16).fill_(0x7FC0)
    op = tl.TiledLinear(K, M, N, d, w, dw, tile_major=tile_major)
    op.set_tile_reuse(reuse)
    x, dy = I.make_x(T, K, seed), I.make_dy(T, M, seed)
    xd, dyd = x.cuda(), dy.cuda()
    for _ in range(calls):
        y = op.forward(xd)
        dx = op.backward(xd, dyd)
    torch.cuda.synchronize()
    xb, dyb = I.bits(x), I.bits(dy)
    wb = I.bits(I.w_logical(w.tensor, K, M, N, tile_major).contiguous())
    case = f"T={T} K={K} M={M} N={N} d={d} tm={tile_major} reuse={reuse} calls={calls}"
    check("Y " + case, y.cpu().float().numpy(), O.forward(xb, wb), None, K, True)
    rdx, rdw = O.backward(xb, wb, dyb)
    check("dX " + case, dx.cpu().numpy(), rdx, None, M, False)
    check("dW " + case, I.w_logical(dw.tensor, K, M, N, tile_major).float().numpy(), rdw, None, T, True)
    assert op.close() == tl.TL_OK
    w.close()
    dw.close()


@pytest.mark.parametrize("seed", range(10))
def test_random_chains(tl, seed):
    rng = np.random.default_rng(2000 + seed)
    L = int(rng.integers(1, 4))
    n = [int(rng.integers(1, 5)) for _ in range(L)]
    dims = [8 * int(rng.integers(2, 49))]
    for l in range(L):
        dims.append(n[l] * 8 * int(rng.integers(1, 33)))
    T = int(rng.integers(1, 200))
    d = int(rng.integers(0, sum(n) + 1))
    reuse = bool(rng.integers(0, 2))
    w, dw = [], []
    for l in range(L):
        K, M = dims[l], dims[l + 1]
        wb, dwb = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
        I.fill_w_host(wb.tensor, K, M, n[l], True, seed + 7 * l)
        w.append(wb)
        dw.append(dwb)
    ch = tl.TiledLinearChain(dims, n, d, w, dw)
    ch.set_tile_reuse(reuse)
    x, dy = I.make_x(T, dims[0], seed), I.make_dy(T, dims[-1], seed)
    xd, dyd = x.cuda(), dy.cuda()
    for _ in range(2):
        ys = ch.forward(xd)
        dx = ch.backward(xd, ys, dyd)
    torch.cuda.synchronize()
    Wb = [I.bits(I.w_logical(w[l].tensor, dims[l], dims[l + 1], n[l], True).contiguous()) for l in range(L)]
    ry = O.chain_forward(I.bits(x), Wb)
    rdx, rdw = O.chain_backward(I.bits(x), Wb, I.bits(dy))
    case = f"T={T} dims={dims} n={n} d={d} reuse={reuse}"
    for l in range(L):
        check(f"Y_{l} " + case, ys[l].cpu().float().numpy(), ry[l], None, dims[l], True)
        check(f"dW_{l} " + case, I.w_logical(dw[l].tensor, dims[l], dims[l + 1], n[l], True).float().numpy(),
              rdw[l], None, T, True)
    check("dX " + case, dx.cpu().numpy(), rdx, None, dims[1], False)
    assert ch.close() == tl.TL_OK
    for b in w + dw:
        b.close()


@pytest.mark.parametrize("seed", range(6))
def test_random_file_tier(tl, tmp_path, seed):
    """Random shapes, depths, host slots, I/O threads, reuse and call counts
    through the file tier: bit-identical to the host-memory path (which the
    cases above check against the oracle)."""
    rng = np.random.default_rng(3000 + seed)
    N = int(rng.integers(1, 7))
    Mi = 8 * int(rng.integers(1, 49))
    K = 256 * int(rng.integers(1, 4))          # K * Mi * 2 bytes: a multiple of 4096 for direct I/O
    M, T = N * Mi, int(rng.integers(1, 300))
    d = int(rng.integers(-1, N + 2))
    slots, io = int(rng.integers(2, 6)), int(rng.integers(1, 5))
    reuse, calls = bool(rng.integers(0, 2)), int(rng.integers(1, 4))
    w, dw = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed)
    w.tensor.view(torch.int16).numpy().tofile(tmp_path / "w.bin")
    x, dy = I.make_x(T, K, seed).cuda(), I.make_dy(T, M, seed).cuda()
    ops = [tl.TiledLinear(K, M, N, d, w, dw, tile_major=True),
           tl.TiledLinearFile(K, M, N, d, tmp_path / "w.bin", tmp_path / "dw.bin", host_slots=slots, io_threads=io)]
    outs = []
    for op in ops:
        op.set_tile_reuse(reuse)
        for _ in range(calls):
            y = op.forward(x)
            dx = op.backward(x, dy)
        torch.cuda.synchronize()
        outs.append((y.cpu().view(torch.int16), dx.cpu().view(torch.int32)))
    ops[1].sync()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1]), (T, K, M, N, d, slots, io)
    assert np.array_equal(np.fromfile(tmp_path / "dw.bin", dtype=np.int16), dw.tensor.view(torch.int16).numpy())
    for op in ops:
        assert op.close() == tl.TL_OK
    w.close()
    dw.close()
