"""The allocation-free forward (tiled_linear_forward_static) against the
handle-based forward and the CPU oracle.

It is for callers that cannot allocate device memory (for example a plug-in
inside a framework whose allocator owns the whole GPU, or a service that
forbids allocation after start-up): its scratch lives in a static device array
inside the library.  Two calls in a row, with different activations, must
each match tiled_linear_forward on the same host weights bit for bit, and the
oracle within the stated tolerance, so the array's left-over contents from the
first call cannot leak into the second.  A tile just under the array's limit
checks the slot's bounds.  This file is collected last so that a
stop-at-first-failure run has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_check import bf16_bits_to_f64, check
from offload_streamed_gb300 import inputs as I
from oracle import oracle as O

pytestmark = pytest.mark.gpu

STATED_REL_TOL = 2e-2


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def _static_forward(tl, lib, T, K, M, N, w, x, status, stream):
    y = torch.full((T, M), float("nan"), dtype=torch.bfloat16, device="cuda")
    status.tensor.fill_(-1)
    rc = lib.tiled_linear_forward_static(T, K, M, N, w.ptr, x.data_ptr(), y.data_ptr(), status.ptr,
                                         stream.cuda_stream)
    assert rc == tl.TL_OK, f"status {rc}: {tl.tiled_linear_last_error(None)}"
    stream.synchronize()
    assert int(status.tensor.item()) == 0, f"timeout word {int(status.tensor.item())}"
    return y


def test_forward_static_matches_forward_twice(tl):
    T, K, M, N = 256, 1024, 4096, 4  # one tile = 2 MiB, well inside the static slot
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed=4)
    status = tl.PinnedBuffer(1, dtype=torch.int32)
    op = tl.TiledLinear(K, M, N, 1, w, dw, tile_major=True)
    lib = tl.load()
    stream = torch.cuda.current_stream()
    wl = I.bits(I.w_logical(w.tensor, K, M, N, True).contiguous())
    for call, seed in enumerate((21, 22)):
        x = I.make_x(T, K, seed)
        xd = x.cuda()
        y_ref = op.forward(xd)
        y = _static_forward(tl, lib, T, K, M, N, w, xd, status, stream)
        got, ref = y.float().cpu().numpy(), y_ref.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - ref)) <= STATED_REL_TOL * np.max(np.abs(ref))
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), f"call {call}: not bit-identical"
        xb = I.bits(x)
        check(f"Y (call {call})", got, O.forward(xb, wl),
              np.abs(bf16_bits_to_f64(xb)) @ np.abs(bf16_bits_to_f64(wl)), K, True)
    op.close()
    for b in (w, dw, status):
        b.close()


def test_forward_static_tile_at_the_limit(tl):
    """K = 2048, M/N = 8184: one tile is 33,521,664 bytes, 32,512 below the
    static slot's 32 MiB - 256 B.  Y on a ragged T against the oracle at
    sampled entries (every tile's edge columns included) and bit for bit
    against the handle forward, two calls in a row."""
    T, K, Mi, N = 300, 2048, 8184, 2
    M = Mi * N
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed=8)
    status = tl.PinnedBuffer(1, dtype=torch.int32)
    op = tl.TiledLinear(K, M, N, 1, w, dw, tile_major=True)
    lib = tl.load()
    stream = torch.cuda.current_stream()
    wt = I.bits(w.tensor).reshape(N, K, Mi)  # the oracle reads the tile-major storage as it is
    for seed in (31, 32):
        x = I.make_x(T, K, seed)
        xd = x.cuda()
        y = _static_forward(tl, lib, T, K, M, N, w, xd, status, stream)
        y_ref = op.forward(xd)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        rows, cols = I.sample_indices(T, M, 4096, seed, 0, col_block=Mi)
        want = O.sample_y(I.bits(x), wt, rows, cols)
        got = y.float().cpu().numpy()[rows, cols]
        err = float(np.max(np.abs(got.astype(np.float64) - want)))
        assert np.all(np.isfinite(got)) and err <= STATED_REL_TOL * float(np.max(np.abs(want))), err
    op.close()
    for b in (w, dw, status):
        b.close()


def test_forward_static_rejects_oversized_tile(tl):
    lib = tl.load()
    status = tl.PinnedBuffer(1, dtype=torch.int32)
    # one tile of 8192 x 4096 bf16 = 64 MiB > the 32 MiB static slot
    rc = lib.tiled_linear_forward_static(16, 8192, 8192, 2, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                         ctypes.c_void_p(16), status.ptr, None)
    assert rc == tl.TL_ERR_WORKSPACE
    assert "static slot" in tl.tiled_linear_last_error(None)
    rc = lib.tiled_linear_forward_static(16, 12, 64, 1, None, None, None, status.ptr, None)
    assert rc == tl.TL_ERR_INVALID
    # the status word is required: without it a kernel timeout would go unseen
    rc = lib.tiled_linear_forward_static(16, 64, 64, 1, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                         ctypes.c_void_p(16), None, None)
    assert rc == tl.TL_ERR_INVALID
    status.close()
