"""The allocation-free forward (tiled_linear_forward_static) against the
handle-based forward.

It is for callers that cannot allocate device memory (for example a plug-in
inside a framework whose allocator owns the whole GPU): its scratch lives in a
static device array inside the library.  Two calls in a row, with different
activations, must each match tiled_linear_forward on the same host weights --
bit for bit, and within the stated tolerance -- so the array's left-over
contents from the first call cannot leak into the second.  This file is
collected last so that a stop-at-first-failure run has already run every
other test."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

STATED_REL_TOL = 2e-2


@pytest.fixture(scope="module")
def tl():
    import __graft_entry__ as g
    g.build()
    from offload_streamed_gb300 import tiled_linear
    return tiled_linear


def test_forward_static_matches_forward_twice(tl):
    from offload_streamed_gb300 import inputs as I
    T, K, M, N = 256, 1024, 4096, 4  # one tile = 2 MiB, well inside the static slot
    w = tl.PinnedBuffer(K * M)
    dw = tl.PinnedBuffer(K * M)
    I.fill_w_host(w.tensor, K, M, N, True, seed=4)
    status = tl.PinnedBuffer(1, dtype=torch.int32)
    op = tl.TiledLinear(K, M, N, 1, w, dw, tile_major=True)
    lib = tl.load()
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((21, 22)):
        x = I.make_x(T, K, seed).cuda()
        y_ref = op.forward(x)
        y = torch.full((T, M), float("nan"), dtype=torch.bfloat16, device="cuda")
        status.tensor.fill_(-1)
        rc = lib.tiled_linear_forward_static(T, K, M, N, w.ptr, x.data_ptr(), y.data_ptr(),
                                             status.ptr, stream.cuda_stream)
        assert rc == tl.TL_OK, f"call {call}: status {rc}"
        stream.synchronize()
        assert int(status.tensor.item()) == 0, f"call {call}: timeout word {int(status.tensor.item())}"
        got, ref = y.float().cpu().numpy(), y_ref.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert np.max(np.abs(got - ref)) <= STATED_REL_TOL * np.max(np.abs(ref))
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), f"call {call}: not bit-identical"
    op.close()
    for b in (w, dw, status):
        b.close()


def test_forward_static_rejects_oversized_tile(tl):
    lib = tl.load()
    # one tile of 8192 x 4096 bf16 = 64 MiB > the 32 MiB static slot
    rc = lib.tiled_linear_forward_static(16, 8192, 8192, 2, ctypes.c_void_p(16), ctypes.c_void_p(16),
                                         ctypes.c_void_p(16), None, None)
    assert rc == tl.TL_ERR_WORKSPACE
    rc = lib.tiled_linear_forward_static(16, 12, 64, 1, None, None, None, None, None)
    assert rc == tl.TL_ERR_INVALID
