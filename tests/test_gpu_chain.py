"""Chains of tiled linear operators (one ring and one prefetcher over several
layers, e.g. the FFN's up- and down-projection) through the C ABI, against
the CPU oracle's chain and against the single-operator calls on the GPU."""
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


def run_chain(tl, T, dims, n_tiles, d, seed=0, kind="normal", calls=1, reuse=False):
    L = len(n_tiles)
    r = Run()
    w, dw = [], []
    for l in range(L):
        K, M, N = dims[l], dims[l + 1], n_tiles[l]
        wb, dwb = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
        I.fill_w_host(wb.tensor, K, M, N, True, seed + 17 * l, kind=kind)
        dwb.tensor.view(torch.int16).fill_(0x7FC0)  # NaN: catches tiles never written
        w.append(wb)
        dw.append(dwb)
    x = I.make_x(T, dims[0], seed, kind=kind)
    dy = I.make_dy(T, dims[-1], seed, kind=kind)
    ch = tl.TiledLinearChain(dims, n_tiles, d, w, dw)
    if reuse:
        ch.set_tile_reuse(True)
    xd, dyd = x.cuda(), dy.cuda()
    for _ in range(calls):
        ys = ch.forward(xd)
        dx = torch.full((T, dims[0]), float("nan"), dtype=torch.float32, device="cuda")
        ch.backward(xd, ys, dyd, dx)
    torch.cuda.synchronize()
    r.stats = ch.stats()
    r.ys = [y.cpu() for y in ys]
    r.dx = dx.cpu()
    r.W = [I.w_logical(w[l].tensor, dims[l], dims[l + 1], n_tiles[l], True).contiguous().clone() for l in range(L)]
    r.dW = [I.w_logical(dw[l].tensor, dims[l], dims[l + 1], n_tiles[l], True).contiguous().clone()
            for l in range(L)]
    r.x, r.dy = x, dy
    assert ch.close() == tl.TL_OK
    for b in w + dw:
        b.close()
    return r


def _same(a, b):
    view = torch.int16 if a.dtype == torch.bfloat16 else torch.int32
    return torch.equal(a.contiguous().view(view), b.contiguous().view(view))


def test_chain_integer_exact(tl):
    """Ternary inputs keep every value of the chain an integer that bf16 and
    fp32 hold exactly (|Y_0| <= 8, |Y_1|, |dX_0|, |dW| <= 256): the GPU chain
    equals the oracle's bit for bit, including the fp32 -> bf16 handover."""
    T, dims, n = 32, [8, 16, 8], [2, 1]
    r = run_chain(tl, T, dims, n, 1, seed=3, kind="ternary")
    Wb = [I.bits(w) for w in r.W]
    ys = O.chain_forward(I.bits(r.x), Wb)
    dx, dws = O.chain_backward(I.bits(r.x), Wb, I.bits(r.dy))
    for l in range(2):
        assert np.array_equal(r.ys[l].float().numpy(), ys[l]), l
        assert np.array_equal(r.dW[l].float().numpy(), dws[l]), l
    assert np.array_equal(r.dx.numpy(), dx)


@pytest.mark.parametrize("T,dims,n,d", [(160, [256, 1024, 256], [4, 2], 1),
                                        (96, [128, 512, 256, 384], [2, 2, 3], 2),
                                        (129, [264, 1056, 264], [4, 1], 0)])
def test_chain_matches_oracle(tl, T, dims, n, d):
    r = run_chain(tl, T, dims, n, d, seed=T)
    Wb = [I.bits(w) for w in r.W]
    xb, dyb = I.bits(r.x), I.bits(r.dy)
    ys = O.chain_forward(xb, Wb)
    dx, dws = O.chain_backward(xb, Wb, dyb)
    xa, wa = np.abs(bf16_bits_to_f64(xb)), np.abs(bf16_bits_to_f64(Wb[0]))
    # the first operator sees the same inputs as the oracle: the element bound applies
    check("Y_0", r.ys[0].float().numpy(), ys[0], xa @ wa, dims[0], True)
    # later ones take bf16-rounded intermediates that may differ by one bf16
    # step where the two fp32 sums straddle a rounding boundary: stated bar
    for l in range(1, len(n)):
        check(f"Y_{l}", r.ys[l].float().numpy(), ys[l], None, dims[l], True)
    for l in range(len(n)):
        check(f"dW_{l}", r.dW[l].float().numpy(), dws[l], None, T, True)
    check("dX_0", r.dx.numpy(), dx, None, dims[1], False)
    assert r.stats["n_tiles"] == sum(n)


@pytest.mark.parametrize("T,dims,n,d", [(200, [256, 768, 512], [3, 2], 1),
                                        (136, [192, 512, 320, 384], [2, 5, 3], 2),
                                        (64, [128, 256, 384, 128, 256], [1, 3, 2, 2], 1)])
def test_chain_composes_the_single_operator_calls(tl, T, dims, n, d):
    """The chain's results are the single-operator calls applied in turn, bit
    for bit: operator l on the chain's own Y_{l-1}, and operator l's backward
    on bf16 of operator l+1's dX.  With three or more operators the middle
    ones read one dY buffer and write the other."""
    r = run_chain(tl, T, dims, n, d, seed=11)
    L = len(n)
    ops, bufs = [], []
    for l in range(L):
        K, M = dims[l], dims[l + 1]
        wb, dwb = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
        wb.tensor.view(n[l], K, M // n[l]).copy_(r.W[l].view(K, n[l], M // n[l]).permute(1, 0, 2))
        bufs += [wb, dwb]
        ops.append((tl.TiledLinear(K, M, n[l], d, wb, dwb, tile_major=True), dwb))
    xs = [r.x.cuda()] + [y.cuda() for y in r.ys[:-1]]
    for l in range(L):
        assert _same(ops[l][0].forward(xs[l]).cpu(), r.ys[l]), l
    g = r.dy.cuda()
    for l in range(L - 1, -1, -1):
        dx = ops[l][0].backward(xs[l], g)
        g = dx.to(torch.bfloat16)
    torch.cuda.synchronize()
    assert _same(dx.cpu(), r.dx)
    for l in range(L):
        K, M = dims[l], dims[l + 1]
        assert _same(I.w_logical(ops[l][1].tensor, K, M, n[l], True), r.dW[l]), l
        assert ops[l][0].close() == tl.TL_OK
    for b in bufs:
        b.close()


def test_chain_of_one_equals_the_single_operator(tl):
    T, K, M, N, d = 150, 512, 2048, 4, 1
    r = run_chain(tl, T, [K, M], [N], d, seed=2)
    w, dw = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    w.tensor.view(N, K, M // N).copy_(r.W[0].view(K, N, M // N).permute(1, 0, 2))
    op = tl.TiledLinear(K, M, N, d, w, dw, tile_major=True)
    x, dy = r.x.cuda(), r.dy.cuda()
    y = op.forward(x)
    dx = op.backward(x, dy)
    torch.cuda.synchronize()
    assert _same(y.cpu(), r.ys[0]) and _same(dx.cpu(), r.dx)
    assert _same(I.w_logical(dw.tensor, K, M, N, True), r.dW[0])
    assert op.close() == tl.TL_OK
    w.close()
    dw.close()


@pytest.mark.parametrize("d", [1, 2, 5])
def test_chain_tile_reuse(tl, d):
    """Reuse crosses the operator boundary: the backward starts with the last
    operator's last tiles, which the forward left in the ring."""
    T, dims, n = 128, [256, 512, 256], [2, 2]
    ref = run_chain(tl, T, dims, n, d, seed=9, calls=2)
    r = run_chain(tl, T, dims, n, d, seed=9, calls=2, reuse=True)
    for l in range(2):
        assert _same(r.ys[l], ref.ys[l]) and _same(r.dW[l], ref.dW[l])
    assert _same(r.dx, ref.dx)
    want = min(r.stats["depth"] + 1, sum(n))
    assert r.stats["bwd_reused_tiles"] == want
    tb = [dims[l] * (dims[l + 1] // n[l]) * 2 for l in range(2)]
    tiles = [tb[1]] * n[1] + [tb[0]] * n[0]  # backward order
    assert r.stats["bwd_h2d_bytes"] == sum(tiles[want:])


def test_chain_argument_errors(tl):
    dims, n = [256, 512, 256], [2, 2]
    w = [tl.PinnedBuffer(256 * 512) for _ in range(2)]
    dw = [tl.PinnedBuffer(256 * 512) for _ in range(2)]
    ch = tl.TiledLinearChain(dims, n, 1, w, dw)
    x = torch.zeros(64, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tl.TiledLinearError) as ei:  # single-operator call on a chain
        tl.tiled_linear_forward(ch.handle, 64, x.data_ptr(), x.data_ptr(), 0)
    assert ei.value.status == tl.TL_ERR_INVALID
    ys = ch.forward(x)
    dx = torch.empty(64, 256, dtype=torch.float32, device="cuda")
    need = tl.tiled_linear_chain_scratch_bytes(64, 2, dims)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.tiled_linear_chain_backward(ch.handle, 64, x.data_ptr(), [y.data_ptr() for y in ys], x.data_ptr(),
                                       dx.data_ptr(), small.data_ptr(), small.numel(), 0)
    assert ei.value.status == tl.TL_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert ch.close() == tl.TL_OK
    op = tl.TiledLinear(256, 512, 2, 1, w[0], dw[0])
    with pytest.raises(tl.TiledLinearError) as ei:  # chain call on a single-operator handle
        tl.tiled_linear_chain_forward(op.handle, 64, x.data_ptr(), [ys[0].data_ptr()], 0)
    assert ei.value.status == tl.TL_ERR_INVALID
    assert op.close() == tl.TL_OK
    for b in w + dw:
        b.close()
