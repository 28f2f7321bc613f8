"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (tile-major pinned host W, the configured N and d).

The oracle evaluates 4096 seeded (row, col) entries per output tensor plus the
first / last column of every tile crossed with the first / last row, one
entry at a time (each entry is the same ascending fp32 sum as the full
oracle).  Forward Y is also compared bit for bit with the untiled product
(one resident GEMM over the whole W), which the tiled path must reproduce
exactly."""
import numpy as np
import pytest
import torch

from offload_streamed_gb300 import inputs as I
from oracle import oracle as O
from gpu_check import check

pytestmark = pytest.mark.gpu

NSAMPLE = 4096


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def _sampled_parity(T, K, M, N, x_bits, dy_bits, w_tm, y, dx, dw_tm, seed):
    """w_tm / dw_tm: numpy uint16 [N, K, Mi] views of the pinned host buffers."""
    Mi = M // N
    r, c = I.sample_indices(T, M, NSAMPLE, seed, 0, col_block=Mi)
    got = y[torch.as_tensor(r, device=y.device), torch.as_tensor(c, device=y.device)].float().cpu().numpy()
    check("Y sampled", got, O.sample_y(x_bits, w_tm, r, c), None, K, True)
    r, c = I.sample_indices(T, K, NSAMPLE, seed, 1, col_block=None)
    got = dx[torch.as_tensor(r, device=dx.device), torch.as_tensor(c, device=dx.device)].cpu().numpy()
    check("dX sampled", got, O.sample_dx(dy_bits, w_tm, r, c), None, M, False)
    r, c = I.sample_indices(K, M, NSAMPLE, seed, 2, col_block=Mi)
    blk, col = c // Mi, c % Mi
    got_bits = dw_tm[blk, r, col]
    got = (got_bits.astype(np.uint32) << 16).view(np.float32)
    check("dW sampled", got, O.sample_dw(x_bits, dy_bits, r, c), None, T, True)


def _dx_group(d, N, Mi):
    """Tiles per dX group for depth d (the engine's rule)."""
    d = min(d, N - 1)
    if not (d >= 2 and N >= 2 and Mi % 64 == 0):
        return 1
    return min(max(2, -(-8192 // Mi)), d, N, 4)


def _run_config(tl, T, K, M, N, depths, seed=0, untiled=True):
    Mi = M // N
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed, device="cuda")
    x = I.make_x(T, K, seed, device="cuda")
    dy = I.make_dy(T, M, seed, device="cuda")
    x_bits, dy_bits = I.bits(x.cpu()), I.bits(dy.cpu())
    w_tm = I.bits(w.tensor).reshape(N, K, Mi)
    dw_tm = dw.tensor.view(torch.int16).numpy().view(np.uint16).reshape(N, K, Mi)
    first = None
    for d in depths:
        dw.tensor.view(torch.int16).fill_(0x7FC0)
        op = tl.TiledLinear(K, M, N, d, w, dw, tile_major=True)
        y = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
        dx = torch.empty(T, K, dtype=torch.float32, device="cuda")
        op.forward(x, y)
        op.backward(x, dy, dx)
        torch.cuda.synchronize()
        assert op.close() == tl.TL_OK
        if first is None:
            _sampled_parity(T, K, M, N, x_bits, dy_bits, w_tm, y, dx, dw_tm, seed)
            first = (y, dx, dw.tensor.clone(), _dx_group(d, N, Mi))
        else:  # another depth: only the schedule changed
            assert torch.equal(y.view(torch.int16), first[0].view(torch.int16)), d
            assert torch.equal(dw.tensor.view(torch.int16), first[2].view(torch.int16)), d
            if _dx_group(d, N, Mi) == first[3]:
                assert torch.equal(dx.view(torch.int32), first[1].view(torch.int32)), d
            else:  # dX sums its tiles in other groups: check it against the oracle
                r, c = I.sample_indices(T, K, NSAMPLE, seed, 1, col_block=None)
                got = dx[torch.as_tensor(r, device=dx.device), torch.as_tensor(c, device=dx.device)].cpu().numpy()
                check(f"dX sampled (d={d})", got, O.sample_dx(dy_bits, w_tm, r, c), None, M, False)
    if untiled:
        # untiled product: one resident GEMM over the whole logical W [K, M]
        w_dev = w.tensor.view(N, K, Mi).to("cuda").permute(1, 0, 2).reshape(K, M).contiguous()
        y_full = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(2, dtype=torch.int32, device="cuda")
        tl.tiled_linear_gemm_forward(T, K, M, x.data_ptr(), K, w_dev.data_ptr(), M, y_full.data_ptr(), M,
                                     err.data_ptr(), torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert int(err[0].item()) == 0
        assert torch.equal(y_full.view(torch.int16), first[0].view(torch.int16))
        del w_dev, y_full
    w.close()
    dw.close()
    torch.cuda.empty_cache()


def test_gpt_scale_ffn_up_proj(tl):
    """X [8192, 8192], W [8192, 32768], N = 8 tiles of 4096, d = 2."""
    _run_config(tl, 8192, 8192, 32768, 8, depths=(2, 1))


def test_1t_width_ffn(tl):
    """X [4096, 25600], W [25600, 102400] (5.2 GB), N = 16 tiles of 6400, d in {1, 2, 3}."""
    _run_config(tl, 4096, 25600, 102400, 16, depths=(1, 2, 3))


def test_64k_hidden_ffn(tl):
    """X [2048, 65536], W [65536, 262144] (32 GiB + 32 GiB dW pinned), N = 16 tiles of 16384, d = 2."""
    _run_config(tl, 2048, 65536, 262144, 16, depths=(2,))


@pytest.mark.parametrize("T,d", [(512, 4), (65536, 1)])
def test_ait_sweep_points(tl, T, d):
    """K = 16384, M = 65536, N = 16 tiles of 4096: the sweep's smallest and
    largest token counts.  At T = 65536 the untiled check holds X (2 GiB), W
    (2 GiB) and two Y of 8 GiB on the device besides the run's dY and dX."""
    _run_config(tl, T, 16384, 65536, 16, depths=(d,))
