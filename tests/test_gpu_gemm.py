"""The three tile GEMMs (tcgen05 kernels) on device-resident operands,
called through the C ABI, against the CPU oracle.  Shapes span several
128 x 256 output tiles and 64-deep K-blocks with ragged tails in every
dimension, plus degenerate sizes and an exact integer case."""
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


def _dev(t):
    return t.cuda()


def _bits(t):
    return I.bits(t.cpu())


def _err_word():
    return torch.zeros(2, dtype=torch.int32, device="cuda")


SHAPES = [(128, 64, 256), (300, 520, 776), (1, 8, 8), (517, 1032, 264), (256, 1024, 1024),
          (64, 200, 40), (129, 72, 264)]


@pytest.mark.parametrize("T,K,n", SHAPES)
def test_gemm_forward(tl, T, K, n):
    x = I.make_x(T, K, seed=T)
    w = I.make_w_tile(K, n, 0, seed=K)
    y = torch.empty(T, n, dtype=torch.bfloat16, device="cuda")
    err = _err_word()
    s = torch.cuda.current_stream()
    xd, wd = _dev(x), _dev(w)  # keep the device copies alive until the kernel is done
    tl.tiled_linear_gemm_forward(T, K, n, xd.data_ptr(), K, wd.data_ptr(), n,
                                 y.data_ptr(), n, err.data_ptr(), s.cuda_stream)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert int(err[1].item()) == 0  # the dynamic schedule's tile counter is left at zero
    xb, wb = _bits(x), _bits(w)
    ref = O.forward(xb, wb)
    S = np.abs(bf16_bits_to_f64(xb)) @ np.abs(bf16_bits_to_f64(wb))
    check("Y", y.float().cpu().numpy(), ref, S, K, bf16_out=True)


@pytest.mark.parametrize("T,K,n", SHAPES)
def test_gemm_dw(tl, T, K, n):
    x = I.make_x(T, K, seed=T + 1)
    dy = I.make_dy(T, n, seed=n + 1)
    dw = torch.empty(K, n, dtype=torch.bfloat16, device="cuda")
    err = _err_word()
    xd, dyd = _dev(x), _dev(dy)
    tl.tiled_linear_gemm_dw(T, K, n, xd.data_ptr(), K, dyd.data_ptr(), n, dw.data_ptr(), n,
                            err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    xb, dyb = _bits(x), _bits(dy)
    ref = O.backward_dw(xb, dyb)
    S = np.abs(bf16_bits_to_f64(xb)).T @ np.abs(bf16_bits_to_f64(dyb))
    check("dW", dw.float().cpu().numpy(), ref, S, T, bf16_out=True)


@pytest.mark.parametrize("T,K,n", SHAPES)
def test_gemm_dx_store_then_accumulate(tl, T, K, n):
    dy = I.make_dy(T, n, seed=T + 2)
    w = I.make_w_tile(K, n, 3, seed=K + 2)
    dx = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    err = _err_word()
    dyd, wd = _dev(dy), _dev(w)
    st = torch.cuda.current_stream().cuda_stream
    # dx = dy . w^T  (overwrite: the NaN fill must disappear)
    tl.tiled_linear_gemm_dx(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, dx.data_ptr(), K, 0,
                            err.data_ptr(), st)
    torch.cuda.synchronize()
    first = dx.cpu().numpy().copy()
    # dx += dy . w^T
    tl.tiled_linear_gemm_dx(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, dx.data_ptr(), K, 1,
                            err.data_ptr(), st)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    dyb, wb = _bits(dy), _bits(w)
    ref = O.backward_dx(dyb, wb)
    S = np.abs(bf16_bits_to_f64(dyb)) @ np.abs(bf16_bits_to_f64(wb)).T
    check("dX", first, ref, S, n, bf16_out=False)
    # accumulation adds exactly the same fp32 tile: 2 * first (exact doubling)
    assert np.array_equal(dx.cpu().numpy(), first + first)


def test_gemm_dx_accumulate_is_an_fp32_add(tl):
    """dX (+)= dY . W^T adds each new value to the old one as one IEEE fp32
    addition: round to nearest, ties to even, subnormals kept.  dY selects
    one column of W per row, so every new value is a single exact product;
    the old values are chosen so that the sums hit ties at 2^24 and land on
    or start from subnormals."""
    T, K, n = 256, 64, 64
    rng = np.random.default_rng(3)
    dy = torch.zeros(T, n, dtype=torch.float32)
    dy[torch.arange(T), torch.arange(T) % n] = 1.0
    w = torch.tensor(rng.integers(-8, 9, size=(K, n)), dtype=torch.float32)
    w[0], w[1], w[2], w[3] = 1.0, 3.0, 0.0, -(2.0 ** -126)
    old = rng.integers(-100, 101, size=(T, K)).astype(np.float32)
    old[:, 0] = old[:, 1] = np.float32(2.0 ** 24)   # + 1 and + 3: ties, to even
    old[:, 2] = np.float32(2.0 ** -130)             # + 0: a subnormal survives
    old[:, 3] = np.float32(1.5 * 2.0 ** -126)       # - 2^-126: a subnormal result
    dyb, wb = dy.bfloat16(), w.bfloat16()
    assert torch.equal(wb.float(), w) and torch.equal(dyb.float(), dy)
    dyd, wd = _dev(dyb), _dev(wb)
    dx = torch.from_numpy(old.copy()).cuda()
    err = _err_word()
    st = torch.cuda.current_stream().cuda_stream
    tl.tiled_linear_gemm_dx(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, dx.data_ptr(), K, 1, err.data_ptr(), st)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    new = w.numpy()[:, np.arange(T) % n].T.astype(np.float32)  # [T, K]: the one product of each entry
    want = old + new  # numpy: IEEE fp32 addition
    got = dx.cpu().numpy()
    assert want[0, 0] == np.float32(2.0 ** 24) and want[0, 1] == np.float32(2.0 ** 24 + 4)
    assert want[0, 3] == np.float32(2.0 ** -127) and want[0, 2] == np.float32(2.0 ** -130)
    assert np.array_equal(got.view(np.int32), want.view(np.int32))


@pytest.mark.parametrize("T,K,n", SHAPES)
def test_gemm_dx_bf16_is_accumulate_then_round(tl, T, K, n):
    """dX rounded to bf16 after adding an fp32 addend (a strided one here) is,
    bit for bit, the fp32 accumulate into a copy of the addend followed by
    torch's round to nearest even; with no addend it is the rounded plain
    product, which also matches the oracle.  Ragged rows and a partial last
    64-column chunk take the epilogue's bounded loads."""
    dy = I.make_dy(T, n, seed=T + 5)
    w = I.make_w_tile(K, n, 1, seed=K + 5)
    ld_add = K + 8
    addend = torch.randn(T, ld_add, generator=torch.Generator().manual_seed(T * K)).cuda()
    dyd, wd = _dev(dy), _dev(w)
    st = torch.cuda.current_stream().cuda_stream
    err = _err_word()
    out = torch.full((T, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    tl.tiled_linear_gemm_dx_bf16(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, addend.data_ptr(), ld_add,
                                 out.data_ptr(), K, err.data_ptr(), st)
    acc = addend[:, :K].contiguous()
    tl.tiled_linear_gemm_dx(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, acc.data_ptr(), K, 1, err.data_ptr(), st)
    plain_bf16 = torch.full((T, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    tl.tiled_linear_gemm_dx_bf16(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, None, 0,
                                 plain_bf16.data_ptr(), K, err.data_ptr(), st)
    plain = torch.empty(T, K, dtype=torch.float32, device="cuda")
    tl.tiled_linear_gemm_dx(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, plain.data_ptr(), K, 0, err.data_ptr(), st)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0 and int(err[1].item()) == 0
    assert torch.equal(out.view(torch.int16), acc.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(plain_bf16.view(torch.int16), plain.to(torch.bfloat16).view(torch.int16))
    dyb, wb = _bits(dy), _bits(w)
    S = np.abs(bf16_bits_to_f64(dyb)) @ np.abs(bf16_bits_to_f64(wb)).T
    check("dX bf16", plain_bf16.float().cpu().numpy(), O.backward_dx(dyb, wb), S, n, bf16_out=True)


def test_gemm_integer_exact(tl):
    """Entries in {-1, 0, 1}: every partial sum is a small integer, exact in
    fp32 and (|values| <= 256) in bf16, so the GPU must equal the integer
    product bit for bit."""
    T, K, n = 256, 192, 512
    x = I.make_x(T, K, 5, kind="ternary")
    w = I.make_w_tile(K, n, 0, 6, kind="ternary")
    dy = I.make_dy(T, n, 7, kind="ternary")
    xi = x.float().numpy().astype(np.int64)
    wi = w.float().numpy().astype(np.int64)
    dyi = dy.float().numpy().astype(np.int64)
    err = _err_word()
    st = torch.cuda.current_stream().cuda_stream
    xd, wd, dyd = _dev(x), _dev(w), _dev(dy)
    y = torch.empty(T, n, dtype=torch.bfloat16, device="cuda")
    dw = torch.empty(K, n, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty(T, K, dtype=torch.float32, device="cuda")
    tl.tiled_linear_gemm_forward(T, K, n, xd.data_ptr(), K, wd.data_ptr(), n, y.data_ptr(), n, err.data_ptr(), st)
    tl.tiled_linear_gemm_dw(T, K, n, xd.data_ptr(), K, dyd.data_ptr(), n, dw.data_ptr(), n, err.data_ptr(), st)
    tl.tiled_linear_gemm_dx(T, K, n, dyd.data_ptr(), n, wd.data_ptr(), n, dx.data_ptr(), K, 0, err.data_ptr(), st)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert np.array_equal(y.float().cpu().numpy().astype(np.int64), xi @ wi)
    assert np.array_equal(dw.float().cpu().numpy().astype(np.int64), xi.T @ dyi)
    assert np.array_equal(dx.cpu().numpy().astype(np.int64), dyi @ wi.T)


def test_gemm_persistent_many_tiles(tl):
    """More output tiles than SMs (each CTA loops over several tiles and both
    TMEM accumulators); checked on sampled entries."""
    T, K, n = 4096, 512, 2560
    x = I.make_x(T, K, 21, device="cuda")
    w = I.make_w_tile(K, n, 0, 22, device="cuda")
    y = torch.empty(T, n, dtype=torch.bfloat16, device="cuda")
    err = _err_word()
    tl.tiled_linear_gemm_forward(T, K, n, x.data_ptr(), K, w.data_ptr(), n, y.data_ptr(), n,
                                 err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    rows, cols = I.sample_indices(T, n, 4096, 0, 0, col_block=256)
    xb, wb = I.bits(x.cpu()), I.bits(w.cpu())
    ref = O.sample_y(xb, wb, rows, cols)
    got = y.float().cpu().numpy()[rows, cols]
    xa, wa = np.abs(bf16_bits_to_f64(xb)), np.abs(bf16_bits_to_f64(wb))
    S = np.einsum("ik,ki->i", xa[rows], wa[:, cols])
    check("Y sampled", got, ref, S, K, bf16_out=True)


def test_gemm_bit_exact_column_slices(tl):
    """A column block computed alone equals the same block of the wide
    product bit for bit (no shape-dependent reduction split)."""
    T, K, M, N = 384, 640, 2048, 4
    x = I.make_x(T, K, 31, device="cuda")
    w = torch.cat([I.make_w_tile(K, M // N, i, 32, device="cuda") for i in range(N)], dim=1).contiguous()
    err = _err_word()
    st = torch.cuda.current_stream().cuda_stream
    y_full = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
    tl.tiled_linear_gemm_forward(T, K, M, x.data_ptr(), K, w.data_ptr(), M, y_full.data_ptr(), M, err.data_ptr(), st)
    Mi = M // N
    y_tiles = torch.empty(T, M, dtype=torch.bfloat16, device="cuda")
    for i in range(N):
        wi = w[:, i * Mi:(i + 1) * Mi].contiguous()
        tl.tiled_linear_gemm_forward(T, K, Mi, x.data_ptr(), K, wi.data_ptr(), Mi,
                                     y_tiles[:, i * Mi:].data_ptr(), M, err.data_ptr(), st)
        torch.cuda.synchronize()
    assert int(err[0].item()) == 0
    assert torch.equal(y_full.view(torch.int16), y_tiles.view(torch.int16))
