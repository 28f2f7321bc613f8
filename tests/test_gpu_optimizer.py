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


# ---- against the fp64 Adam oracle, after real GPU backward calls ---------------

def _bits_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _check_adam_state(name, prev, new, g, step, wd):
    """The library's state after one step against oracle/adam.py applied to
    its state before the step and the gradient it read; the bounds are
    those of the CPU test of the update (fp32 evaluation of a few operations
    per element)."""
    from oracle import adam as A
    from oracle import oracle as O
    p0, m0, v0 = (np.asarray(a, np.float64) for a in prev)
    P, Mm, V, W = new
    pr, mr, vr = A.adam_step(p0, m0, v0, g, step, lr=LR, beta1=B1, beta2=B2, eps=EPS, wd=wd)
    u = 2.0 ** -24
    assert np.all(np.abs(Mm - mr) <= 8 * u * (np.abs(m0) + np.abs(g)) + 1e-30), name
    assert np.all(np.abs(V - vr) <= 8 * u * (np.abs(v0) + g * g) + 1e-30), name
    assert np.all(np.abs(P - pr) <= 8 * u * np.abs(p0) + 1e-5 * LR * (1 + np.abs(mr) / np.sqrt(np.abs(vr) + 1e-30))), name
    # the weights the next pass streams are the new master rounded to nearest even
    assert np.array_equal(W, O.round_bf16(np.asarray(P, np.float32))), name


def _oracle_checked_dw(name, dw_bits_logical, X, dY, element_bound=True):
    """The GPU's dW (bf16, logical [K, M]) against the oracle's X^T dY: the
    stated tolerance, and the per-element bound when the GPU read exactly
    these X and dY."""
    from gpu_check import check
    from oracle import oracle as O
    xb, dyb = I.bits(X), I.bits(dY)
    S = np.abs(_bits_f64(xb)).T @ np.abs(_bits_f64(dyb)) if element_bound else None
    check(name, _bits_f64(dw_bits_logical), O.backward_dw(xb, dyb), S, X.shape[0], True)


def test_steps_after_gpu_backward_match_the_adam_oracle(tl):
    """Three training steps of one operator (row-major host W, N = 4 tiles of
    strided columns): each step's dW from the GPU meets the oracle, the host
    optimizer's new master / m / v meet the fp64 Adam oracle applied to the
    state before the step and that dW, W is the new master rounded, and the
    next forward streams the updated W (Y meets the oracle on it)."""
    from gpu_check import check
    from oracle import oracle as O
    T, K, M, N, d, steps = 160, 384, 1536, 4, 1, 3
    w, dw = tl.PinnedBuffer(K * M), tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, False, 17)
    op = tl.TiledLinear(K, M, N, d, w, dw, tile_major=False)
    opt = tl.HostAdam(op, LR, B1, B2, EPS, WD, threads=3)
    for s in range(steps):
        x, dy = I.make_x(T, K, 60 + s), I.make_dy(T, M, 60 + s)
        prev = [t.numpy().copy() for t in (opt.master[0], opt.m[0], opt.v[0])]
        wb = I.bits(w.tensor).reshape(K, M).copy()
        y = op.forward(x.cuda())
        op.backward(x.cuda(), dy.cuda())
        opt.step()
        opt.wait()
        torch.cuda.synchronize()
        xb = I.bits(x)
        check(f"Y step {s}", y.float().cpu().numpy(), O.forward(xb, wb),
              np.abs(_bits_f64(xb)) @ np.abs(_bits_f64(wb)), K, True)
        g_bits = I.bits(dw.tensor).reshape(K, M)
        _oracle_checked_dw(f"dW step {s}", g_bits, x, dy)
        new = (opt.master[0].numpy(), opt.m[0].numpy(), opt.v[0].numpy(), I.bits(w.tensor))
        _check_adam_state(f"step {s}", [a.reshape(-1) for a in prev], new, _bits_f64(g_bits).reshape(-1),
                          s + 1, WD)
    for o in (opt, op):
        assert o.close() == tl.TL_OK
    w.close()
    dw.close()


def test_chain_steps_match_the_adam_oracle(tl):
    """Two steps of a two-operator chain (tile-major, different tile shapes
    per operator): each operator's state follows the oracle from its own dW,
    so the optimizer's per-operator offsets and tile order are right."""
    from oracle import oracle as O
    T, dims, n, d = 128, [256, 768, 384], [3, 2], 1
    ws, dws = [], []
    for l in range(2):
        w, dw = _bufs(tl, dims[l], dims[l + 1], n[l], 70 + l)
        ws.append(w)
        dws.append(dw)
    ch = tl.TiledLinearChain(dims, n, d, ws, dws)
    opt = tl.HostAdam(ch, LR, B1, B2, EPS, 0.0, threads=2)
    for s in range(2):
        x, dy = I.make_x(T, dims[0], 80 + s), I.make_dy(T, dims[2], 80 + s)
        prev = [[t.numpy().copy() for t in (opt.master[l], opt.m[l], opt.v[l])] for l in range(2)]
        xd = x.cuda()
        ys = ch.forward(xd)
        ch.backward(xd, ys, dy.cuda())
        opt.step()
        opt.wait()
        torch.cuda.synchronize()
        # operator 1's input is the GPU's bf16 Y of operator 0; its dY is the
        # bf16 of operator 1's dX (the chain's reading); dW_l = X_l^T dY_l
        y0 = ys[0].cpu()
        for l in range(2):
            K, M, N = dims[l], dims[l + 1], n[l]
            g_logical = I.bits(I.w_logical(dws[l].tensor, K, M, N, True).contiguous())
            if l == 1:
                _oracle_checked_dw(f"chain dW1 step {s}", g_logical, y0, dy)
            else:
                # dY_0 = bf16(dY . W_1^T) with the W_1 the step streamed (the
                # rounded master before the update); the GPU rounds its own
                # fp32 dX_1, which may differ from the oracle's in the last
                # bit here and there, so only the stated tolerance applies
                w1_before = O.round_bf16(prev[1][0].astype(np.float32)).reshape(n[1], dims[1], dims[2] // n[1])
                w1_before = np.ascontiguousarray(w1_before.transpose(1, 0, 2).reshape(dims[1], dims[2]))
                dy0 = O.round_bf16(O.backward_dx(I.bits(dy), w1_before))
                dy0_t = torch.from_numpy(dy0.view(np.int16)).view(torch.bfloat16)
                _oracle_checked_dw(f"chain dW0 step {s}", g_logical, x, dy0_t, element_bound=False)
            new = (opt.master[l].numpy(), opt.m[l].numpy(), opt.v[l].numpy(), I.bits(ws[l].tensor))
            g = _bits_f64(I.bits(dws[l].tensor))
            _check_adam_state(f"chain op {l} step {s}", prev[l], new, g, s + 1, 0.0)
    for o in (opt, ch):
        assert o.close() == tl.TL_OK
    for b in ws + dws:
        b.close()
