"""The host optimizer attached to a streamed layer: its overlapped per-tile
Adam steps give the same bits as the synchronous update after each backward
(tiled_linear_adam_update, checked against the fp64 oracle on the CPU), for
a single operator, with gradient accumulation, with tile reuse and for a
chain."""
import numpy as np
import pytest
import torch

from offload_streamed_gb300 import inputs as I

pytestmark = pytest.mark.gpu

LR, B1, B2, EPS, WD = 1e-3, 0.9, 0.95, 1e-8, 0.01


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def _bufs(tl, K, M, N, seed):
    w, dw = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed)
    dw.tensor.zero_()
    return w, dw


def _data(T, K, M, seed, steps):
    return [(I.make_x(T, K, seed + 100 * s).cuda(), I.make_dy(T, M, seed + 100 * s).cuda()) for s in range(steps)]


def _manual(tl, cfg, step, master, m, v, dw, w, acc=None):
    tl.tiled_linear_adam_update(cfg, step, master.size, master.ctypes.data, m.ctypes.data, v.ctypes.data,
                                acc.ctypes.data if acc is not None else 0, dw.ptr, w.ptr)


def _same_host(a, b):
    return np.array_equal(a.tensor.view(torch.int16).numpy(), b.tensor.view(torch.int16).numpy())


@pytest.mark.parametrize("reuse", [False, True], ids=["refetch", "reuse"])
def test_overlapped_steps_match_the_synchronous_update(tl, reuse):
    T, K, M, N, d, steps = 192, 512, 2048, 4, 1, 3
    cfg = tl.adam_config(LR, B1, B2, EPS, WD, threads=4)
    data = _data(T, K, M, 5, steps)
    # overlapped: the optimizer runs while the next calls are queued
    wa, dwa = _bufs(tl, K, M, N, 5)
    op = tl.TiledLinear(K, M, N, d, wa, dwa)
    op.set_tile_reuse(reuse)
    opt = tl.HostAdam(op, LR, B1, B2, EPS, WD, threads=4)
    for x, dy in data:
        ya = op.forward(x)
        op.backward(x, dy)
        opt.step()
    opt.wait()
    torch.cuda.synchronize()
    assert opt.stats()["steps"] == steps
    # synchronous reference
    wb, dwb = _bufs(tl, K, M, N, 5)
    ref = tl.TiledLinear(K, M, N, d, wb, dwb)
    master = wb.tensor.float().numpy().copy()
    m, v = np.zeros_like(master), np.zeros_like(master)
    for s, (x, dy) in enumerate(data):
        yb = ref.forward(x)
        ref.backward(x, dy)
        torch.cuda.synchronize()
        _manual(tl, cfg, s + 1, master, m, v, dwb, wb)
    assert torch.equal(ya.cpu().view(torch.int16), yb.cpu().view(torch.int16))
    assert _same_host(wa, wb) and _same_host(dwa, dwb)
    assert np.array_equal(opt.master[0].numpy(), master)
    assert np.array_equal(opt.m[0].numpy(), m) and np.array_equal(opt.v[0].numpy(), v)
    assert opt.close() == tl.TL_OK
    for o in (op, ref):
        assert o.close() == tl.TL_OK
    for b in (wa, dwa, wb, dwb):
        b.close()


def test_gradient_accumulation_then_step(tl):
    """Two micro-batches per step: accumulate the first backward's dW in fp32,
    step with the second one's added."""
    T, K, M, N, d = 128, 256, 1024, 2, 1
    cfg = tl.adam_config(LR, B1, B2, EPS, WD, threads=2)
    data = _data(T, K, M, 7, 4)
    wa, dwa = _bufs(tl, K, M, N, 7)
    op = tl.TiledLinear(K, M, N, d, wa, dwa)
    opt = tl.HostAdam(op, LR, B1, B2, EPS, WD, threads=2, accumulate=True)
    for s in range(2):
        for j, (x, dy) in enumerate(data[2 * s:2 * s + 2]):
            op.forward(x)
            op.backward(x, dy)
            if j == 0:
                opt.accumulate()
            else:
                opt.step()
    opt.wait()
    wb, dwb = _bufs(tl, K, M, N, 7)
    ref = tl.TiledLinear(K, M, N, d, wb, dwb)
    master = wb.tensor.float().numpy().copy()
    m, v = np.zeros_like(master), np.zeros_like(master)
    for s in range(2):
        for j, (x, dy) in enumerate(data[2 * s:2 * s + 2]):
            ref.forward(x)
            ref.backward(x, dy)
            torch.cuda.synchronize()
            if j == 0:
                acc = dwb.tensor.float().numpy().copy()
            else:
                _manual(tl, cfg, s + 1, master, m, v, dwb, wb, acc)
    assert _same_host(wa, wb)
    assert np.array_equal(opt.master[0].numpy(), master)
    assert np.array_equal(opt.m[0].numpy(), m) and np.array_equal(opt.v[0].numpy(), v)
    for o in (opt, op, ref):
        assert o.close() == tl.TL_OK
    for b in (wa, dwa, wb, dwb):
        b.close()


def test_chain_optimizer(tl):
    T, dims, n, d = 96, [256, 512, 256], [2, 2], 1
    cfg = tl.adam_config(LR, B1, B2, EPS, 0.0, threads=3)
    xs = [I.make_x(T, 256, 30 + s).cuda() for s in range(2)]
    dys = [I.make_dy(T, 256, 30 + s).cuda() for s in range(2)]

    def bufs():
        out = []
        for l in range(2):
            out.append(_bufs(tl, dims[l], dims[l + 1], n[l], 40 + l))
        return [b[0] for b in out], [b[1] for b in out]

    wa, dwa = bufs()
    ch = tl.TiledLinearChain(dims, n, d, wa, dwa)
    opt = tl.HostAdam(ch, LR, B1, B2, EPS, 0.0, threads=3)
    for x, dy in zip(xs, dys):
        ys = ch.forward(x)
        ch.backward(x, ys, dy)
        opt.step()
    opt.wait()
    wb, dwb = bufs()
    ref = tl.TiledLinearChain(dims, n, d, wb, dwb)
    masters = [w.tensor.float().numpy().copy() for w in wb]
    ms = [np.zeros_like(a) for a in masters]
    vs = [np.zeros_like(a) for a in masters]
    for s, (x, dy) in enumerate(zip(xs, dys)):
        ys = ref.forward(x)
        ref.backward(x, ys, dy)
        torch.cuda.synchronize()
        for l in range(2):
            _manual(tl, cfg, s + 1, masters[l], ms[l], vs[l], dwb[l], wb[l])
    for l in range(2):
        assert _same_host(wa[l], wb[l])
        assert np.array_equal(opt.master[l].numpy(), masters[l])
    for o in (opt, ch, ref):
        assert o.close() == tl.TL_OK
    for b in wa + dwa + wb + dwb:
        b.close()


def test_optimizer_state_errors_and_destroy_order(tl):
    K, M, N = 256, 512, 2
    w, dw = _bufs(tl, K, M, N, 1)
    op = tl.TiledLinear(K, M, N, 1, w, dw)
    opt = tl.HostAdam(op)
    with pytest.raises(tl.TiledLinearError) as ei:  # no backward yet
        opt.step()
    assert ei.value.status == tl.TL_ERR_STATE
    with pytest.raises(tl.TiledLinearError) as ei:  # no accumulator
        x = torch.zeros(64, K, dtype=torch.bfloat16, device="cuda")
        op.forward(x)
        op.backward(x, torch.zeros(64, M, dtype=torch.bfloat16, device="cuda"))
        opt.accumulate()
    assert ei.value.status == tl.TL_ERR_INVALID
    opt.step()
    with pytest.raises(tl.TiledLinearError) as ei:  # a second optimizer on the same handle
        tl.HostAdam(op)
    assert ei.value.status == tl.TL_ERR_STATE
    # destroying the handle first detaches the optimizer; its own destroy then only frees it
    assert op.close() == tl.TL_OK
    assert opt.close() == tl.TL_OK
    w.close()
    dw.close()
