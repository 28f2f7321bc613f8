"""The kernels' failure path, made to run on purpose without faulting or
hanging anything: a forward GEMM whose loads are withheld must give up its
bounded wait within the limit, report the error bit, free its tensor memory
and leave the device usable; a handle whose error word is set reports
TL_ERR_TIMEOUT once and is then sticky-failed."""
import time

import numpy as np
import pytest
import torch

from offload_streamed_gb300 import inputs as I
from oracle import oracle as O
from gpu_check import check

pytestmark = pytest.mark.gpu

ERR_MMA_WAIT_FULL = 2


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def test_bounded_wait_runs_out_and_reports(tl):
    scratch = torch.full((1 << 17,), 0x55, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    tl.tiled_linear_selftest_timeout(scratch.data_ptr(), scratch.numel(), 50_000_000, stream.cuda_stream)
    stream.synchronize()
    elapsed = time.perf_counter() - t0
    word = int(scratch[:4].view(torch.int32).item())
    assert word & ERR_MMA_WAIT_FULL, word
    assert elapsed < 5.0, elapsed
    # nothing past the error word and the tile counter was written
    assert torch.all(scratch[8:] == 0x55)
    # the context is still usable: a normal GEMM right after is correct
    T, K, n = 256, 192, 512
    x = I.make_x(T, K, 1)
    w = I.make_w_tile(K, n, 0, 2)
    xd, wd = x.cuda(), w.cuda()
    y = torch.empty(T, n, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    tl.tiled_linear_gemm_forward(T, K, n, xd.data_ptr(), K, wd.data_ptr(), n, y.data_ptr(), n,
                                 err.data_ptr(), stream.cuda_stream)
    stream.synchronize()
    assert int(err[0].item()) == 0
    check("Y after self-test", y.float().cpu().numpy(), O.forward(I.bits(x), I.bits(w)), None, K, True)


def test_handle_turns_sticky_after_a_timeout(tl):
    K, M, N = 256, 1024, 4
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, 0)
    op = tl.TiledLinear(K, M, N, 1, w, dw)
    stream = torch.cuda.current_stream()
    x = I.make_x(64, K, 0).cuda()
    op.forward(x)
    stream.synchronize()
    assert op.stats()["fwd_valid"] == 1
    # the handle's kernels report timeouts through the first word of its
    # workspace; run the failing self-test against that word
    tl.tiled_linear_selftest_timeout(op.workspace.data_ptr(), op.workspace.numel(), 20_000_000,
                                     stream.cuda_stream)
    stream.synchronize()
    with pytest.raises(tl.TiledLinearError) as ei:
        op.stats()
    assert ei.value.status == tl.TL_ERR_TIMEOUT
    with pytest.raises(tl.TiledLinearError) as ei:
        op.forward(x)
    assert ei.value.status == tl.TL_ERR_STATE
    assert "timed out" in tl.tiled_linear_last_error(op.handle)
    assert op.close() == tl.TL_ERR_TIMEOUT
    w.close()
    dw.close()
