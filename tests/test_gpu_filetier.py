"""The file tier (tiled_linear_create_file): W and dW in files, read and
written with direct I/O through pinned host slots.  The data source changes,
the arithmetic does not, so every result must equal the host-memory path's
bit for bit; and that path equals the CPU oracle (checked here once more on
a small case)."""
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


def _w_file(tl, path, K, M, N, seed, kind="normal"):
    w = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed, kind=kind)
    w.tensor.view(torch.int16).numpy().tofile(path)
    return w


def _bits(a):
    return a.contiguous().view(torch.int16) if a.dtype == torch.bfloat16 else a.contiguous().view(torch.int32)


def _run(op, x, dy, calls):
    for _ in range(calls):
        y = op.forward(x)
        dx = op.backward(x, dy)
    torch.cuda.synchronize()
    return y.cpu(), dx.cpu()


@pytest.mark.parametrize("K,M,N,d,slots,io,T", [
    (512, 2048, 4, 1, 2, 1, 200),      # 512 KiB tiles, the smallest ring and host ring
    (512, 2048, 4, 2, 3, 4, 129),      # ragged T
    (8192, 4096, 2, 1, 2, 4, 256),     # 32 MiB tiles: two 16 MiB requests each, over four threads
    (1024, 6144, 6, 3, 4, 2, 64),
])
def test_file_tier_equals_the_host_memory_path(tl, tmp_path, K, M, N, d, slots, io, T):
    w = _w_file(tl, tmp_path / "w.bin", K, M, N, seed=K + N)
    x = I.make_x(T, K, 3).cuda()
    dy = I.make_dy(T, M, 4).cuda()
    # reference: pinned host memory
    dw_ref = tl.PinnedBuffer(K * M)
    ref = tl.TiledLinear(K, M, N, d, w, dw_ref, tile_major=True)
    y_ref, dx_ref = _run(ref, x, dy, 2)
    # file tier, two calls (the second reuses the host slots)
    (tmp_path / "dw.bin").write_bytes(b"\xff" * 4096)  # stale, short: extended and overwritten
    op = tl.TiledLinearFile(K, M, N, d, tmp_path / "w.bin", tmp_path / "dw.bin", host_slots=slots, io_threads=io)
    y, dx = _run(op, x, dy, 2)
    op.sync()
    assert torch.equal(_bits(y), _bits(y_ref))
    assert torch.equal(_bits(dx), _bits(dx_ref))
    dw_file = np.fromfile(tmp_path / "dw.bin", dtype=np.int16)
    assert dw_file.size == K * M
    assert np.array_equal(dw_file, dw_ref.tensor.view(torch.int16).numpy())
    fs = op.file_stats()
    tb = K * (M // N) * 2
    assert fs["read_bytes"] == 2 * 2 * N * tb  # two calls of forward + backward, every tile fetched
    assert fs["write_bytes"] == 2 * N * tb
    assert fs["host_slots"] == slots and fs["io_threads"] == io
    st = op.stats()
    assert st["staging_slots"] == min(2, N) and st["fwd_h2d_bytes"] == N * tb
    for o in (op, ref):
        assert o.close() == tl.TL_OK
    w.close()
    dw_ref.close()


def test_file_tier_matches_the_oracle(tl, tmp_path):
    T, K, M, N, d = 96, 256, 1024, 4, 1
    w = _w_file(tl, tmp_path / "w.bin", K, M, N, seed=5)
    W = I.w_logical(w.tensor, K, M, N, True).contiguous()
    xh, dyh = I.make_x(T, K, 6), I.make_dy(T, M, 7)
    op = tl.TiledLinearFile(K, M, N, d, tmp_path / "w.bin", tmp_path / "dw.bin")
    y = op.forward(xh.cuda())
    dx = op.backward(xh.cuda(), dyh.cuda())
    op.sync()
    xb, wb, dyb = I.bits(xh), I.bits(W), I.bits(dyh)
    xa, wa, dya = (np.abs(bf16_bits_to_f64(b)) for b in (xb, wb, dyb))
    check("Y", y.float().cpu().numpy(), O.forward(xb, wb), xa @ wa, K, True)
    dx_o, dw_o = O.backward(xb, wb, dyb)
    check("dX", dx.cpu().numpy(), dx_o, dya @ wa.T, M, False)
    dw = torch.from_numpy(np.fromfile(tmp_path / "dw.bin", dtype=np.int16)).view(torch.bfloat16)
    dw = I.w_logical(dw, K, M, N, True).float().numpy()
    check("dW", dw, dw_o, xa.T @ dya, T, True)
    assert op.close() == tl.TL_OK
    w.close()


def test_file_tier_tile_reuse_reads_less(tl, tmp_path):
    T, K, M, N, d = 128, 512, 4096, 8, 2
    w = _w_file(tl, tmp_path / "w.bin", K, M, N, seed=9)
    x, dy = I.make_x(T, K, 1).cuda(), I.make_dy(T, M, 2).cuda()
    plain = tl.TiledLinearFile(K, M, N, d, tmp_path / "w.bin", tmp_path / "dw0.bin")
    y0, dx0 = _run(plain, x, dy, 1)
    plain.sync()
    op = tl.TiledLinearFile(K, M, N, d, tmp_path / "w.bin", tmp_path / "dw1.bin")
    op.set_tile_reuse(True)
    y1, dx1 = _run(op, x, dy, 1)
    op.sync()
    assert torch.equal(_bits(y0), _bits(y1)) and torch.equal(_bits(dx0), _bits(dx1))
    assert np.array_equal(np.fromfile(tmp_path / "dw0.bin", dtype=np.int16),
                          np.fromfile(tmp_path / "dw1.bin", dtype=np.int16))
    tb = K * (M // N) * 2
    reused = op.stats()["bwd_reused_tiles"]
    assert reused == d + 1
    assert op.file_stats()["read_bytes"] == (2 * N - reused) * tb
    for o in (plain, op):
        assert o.close() == tl.TL_OK
    w.close()


def test_file_tier_empty_backward_writes_zero(tl, tmp_path):
    K, M, N = 256, 1024, 2
    w = _w_file(tl, tmp_path / "w.bin", K, M, N, seed=3)
    (tmp_path / "dw.bin").write_bytes(b"\x7f" * (K * M * 2))
    op = tl.TiledLinearFile(K, M, N, 1, tmp_path / "w.bin", tmp_path / "dw.bin")
    x = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    op.backward(x, torch.empty(0, M, dtype=torch.bfloat16, device="cuda"),
                torch.empty(0, K, dtype=torch.float32, device="cuda"))
    op.sync()
    assert not np.fromfile(tmp_path / "dw.bin", dtype=np.int16).any()
    assert op.close() == tl.TL_OK
    w.close()


def test_file_tier_io_errors_and_exclusions(tl, tmp_path):
    K, M, N = 256, 1024, 2
    (tmp_path / "short.bin").write_bytes(b"\0" * (K * M * 2 - 4096))  # one page short of N tiles
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.TiledLinearFile(K, M, N, 1, tmp_path / "short.bin", tmp_path / "dw.bin")
    assert ei.value.status == tl.TL_ERR_IO and "shorter" in str(ei.value)
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.TiledLinearFile(K, M, N, 1, tmp_path / "missing.bin", tmp_path / "dw.bin")
    assert ei.value.status == tl.TL_ERR_IO
    w = _w_file(tl, tmp_path / "w.bin", K, M, N, seed=1)
    with pytest.raises(tl.TiledLinearError) as ei:  # the dW file's directory does not exist
        tl.TiledLinearFile(K, M, N, 1, tmp_path / "w.bin", tmp_path / "no_such_dir" / "dw.bin")
    assert ei.value.status == tl.TL_ERR_IO
    op = tl.TiledLinearFile(K, M, N, 1, tmp_path / "w.bin", tmp_path / "dw.bin")
    with pytest.raises(tl.TiledLinearError) as ei:  # the host optimizer needs W in host memory
        tl.tiled_linear_optimizer_create(op.handle, tl.adam_config(1e-3, 0.9, 0.95, 1e-8, 0.0), [0], [0], [0])
    assert ei.value.status == tl.TL_ERR_INVALID and "host memory" in str(ei.value)
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.HostAdam(op)
    assert ei.value.status == tl.TL_ERR_INVALID
    plain = tl.TiledLinear(K, M, N, 1, w, tl.PinnedBuffer(K * M))
    with pytest.raises(tl.TiledLinearError) as ei:  # no file tier on a host-memory handle
        tl.tiled_linear_file_sync(plain.handle)
    assert ei.value.status == tl.TL_ERR_INVALID
    for o in (op, plain):
        assert o.close() == tl.TL_OK
    w.close()
