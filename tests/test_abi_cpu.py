"""The C-ABI library without a GPU: it loads, exports every declared entry
point, sizes workspaces as the closed forms say, and rejects bad arguments
before touching CUDA."""
import ctypes
import os
import re

import pytest

from oracle import closed_forms as CF

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_FILE = os.path.join(ROOT, "include", "tiled_linear.h")
HEADER = 4096  # workspace header: the kernels' error word and tile counter


@pytest.fixture(scope="module")
def tl():
    from offload_streamed_gb300 import _build
    _build.build()
    from offload_streamed_gb300 import tiled_linear
    tiled_linear.load()
    return tiled_linear


def declared_functions():
    src = open(HEADER_FILE).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tiled_linear_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tiled_linear_create", "tiled_linear_forward", "tiled_linear_backward",
                     "tiled_linear_destroy", "tiled_linear_workspace_bytes",
                     "tiled_linear_last_error", "tiled_linear_get_stats"):
        assert required in names


def test_library_exports_every_declared_symbol(tl):
    lib = ctypes.CDLL(tl.lib_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_has_the_same_names(tl):
    for n in declared_functions():
        assert callable(getattr(tl, n, None)), n


def test_version(tl):
    assert "sm_103a" in tl.tiled_linear_version()


@pytest.mark.parametrize("K,M,N,d", [(1024, 4096, 4, 1), (8192, 32768, 8, 2), (25600, 102400, 16, 3),
                                     (65536, 262144, 16, 2), (16384, 65536, 16, 4), (64, 64, 1, 0),
                                     (1024, 4096, 4, 9)])
def test_workspace_bytes_matches_closed_form(tl, K, M, N, d):
    tile = CF.tile_bytes(K, M, N)
    tile_al = (tile + 255) // 256 * 256
    ring = CF.ring_bytes(K, M, N, d) // tile * tile_al
    staging = min(2, N) * tile_al
    assert tl.tiled_linear_workspace_bytes(K, M, N, d) == HEADER + ring + staging


def test_workspace_bytes_auto_depth(tl):
    """Automatic depth sizes for the most a handle can use: N ring slots (every
    tile resident, d = N - 1) and N staging slots."""
    tile = CF.tile_bytes(1024, 4096, 4)
    assert tl.tiled_linear_workspace_bytes(1024, 4096, 4, -1) == HEADER + (4 + 4) * tile
    assert tl.tiled_linear_workspace_bytes(1024, 4096 * 4, 16, -1) == HEADER + (16 + 16) * tile
    assert tl.tiled_linear_workspace_bytes(1024, 4096, 1, -1) == HEADER + (1 + 1) * 4 * tile


def test_auto_depth_accepts_a_smaller_workspace(tl):
    """Create with d = -1 refuses less than two ring slots and min(2, N)
    staging slots (the d = 1 workspace), and accepts that much."""
    K, M, N = 64, 64 * 8, 8
    least = tl.tiled_linear_workspace_bytes(K, M, N, 1)
    assert least < tl.tiled_linear_workspace_bytes(K, M, N, -1)
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.tiled_linear_create(K, M, N, -1, 16, 16, 256, least - 1, 0)
    assert ei.value.status == tl.TL_ERR_WORKSPACE
    assert str(least) in tl.tiled_linear_last_error(None)


@pytest.mark.parametrize("K,M,N,d", [(0, 64, 1, 0), (12, 64, 1, 0), (64, 65, 1, 0), (64, 64, 3, 0),
                                     (64, 100, 2, 0), (64, 64, 0, 0), (64, 64, 1, -2)])
def test_invalid_shapes(tl, K, M, N, d):
    assert tl.tiled_linear_workspace_bytes(K, M, N, d) == 0
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.tiled_linear_create(K, M, N, d, 16, 16, 256, 1 << 30, 0)
    assert ei.value.status == tl.TL_ERR_INVALID
    assert tl.tiled_linear_last_error(None)


def test_null_pointers_and_small_workspace(tl):
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.tiled_linear_create(64, 64, 1, 0, 0, 16, 256, 1 << 20, 0)
    assert ei.value.status == tl.TL_ERR_INVALID
    need = tl.tiled_linear_workspace_bytes(64, 64, 1, 0)
    with pytest.raises(tl.TiledLinearError) as ei:
        tl.tiled_linear_create(64, 64, 1, 0, 16, 16, 256, need - 1, 0)
    assert ei.value.status == tl.TL_ERR_WORKSPACE
    with pytest.raises(tl.TiledLinearError) as ei:  # misaligned workspace
        tl.tiled_linear_create(64, 64, 1, 0, 16, 16, 256 + 16, need, 0)
    assert ei.value.status == tl.TL_ERR_WORKSPACE


def test_null_handle_calls(tl):
    lib = tl.load()
    assert lib.tiled_linear_forward(None, 1, None, None, None) == tl.TL_ERR_STATE
    assert lib.tiled_linear_backward(None, 1, None, None, None, None) == tl.TL_ERR_STATE
    assert lib.tiled_linear_destroy(None) == tl.TL_OK
    assert lib.tiled_linear_get_stats(None, None) == tl.TL_ERR_INVALID


def test_resident_gemm_argument_checks(tl):
    lib = tl.load()
    # sizes < 1, null pointers and unaligned leading dimensions are refused
    # before any CUDA call
    assert lib.tiled_linear_gemm_forward(0, 64, 64, 256, 64, 256, 64, 256, 64, 256, None) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_gemm_forward(64, 64, 64, None, 64, 256, 64, 256, 64, 256, None) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_gemm_dw(64, 64, 64, 256, 60, 256, 64, 256, 64, 256, None) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_gemm_dx(64, 64, 64, 256, 64, 256, 64, 256, 32, 0, 256, None) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_gemm_dx(64, 64, 64, 258, 64, 256, 64, 256, 64, 0, 256, None) == tl.TL_ERR_INVALID
    # the bf16 dX: a misaligned addend, an addend row shorter than K or not a
    # multiple of 8 elements
    dxb = lib.tiled_linear_gemm_dx_bf16
    assert dxb(64, 64, 64, 256, 64, 256, 64, 264, 64, 256, 64, 256, None) == tl.TL_ERR_INVALID
    assert dxb(64, 64, 64, 256, 64, 256, 64, 256, 56, 256, 64, 256, None) == tl.TL_ERR_INVALID
    assert dxb(64, 64, 64, 256, 64, 256, 64, 256, 68, 256, 64, 256, None) == tl.TL_ERR_INVALID
    assert dxb(64, 64, 64, None, 64, 256, 64, None, 0, 256, 64, 256, None) == tl.TL_ERR_INVALID


def test_trace_argument_checks(tl):
    lib = tl.load()
    n = ctypes.c_int32(5)
    assert lib.tiled_linear_get_trace(None, 0, None, 0, ctypes.byref(n)) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_get_trace(256, 0, None, 0, None) == tl.TL_ERR_INVALID  # null count
    assert lib.tiled_linear_get_trace(256, 0, None, -1, ctypes.byref(n)) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_get_trace(256, 0, None, 4, ctypes.byref(n)) == tl.TL_ERR_INVALID  # null out


def test_null_handle_tile_reuse(tl):
    assert tl.load().tiled_linear_set_tile_reuse(None, 1) == tl.TL_ERR_STATE
    assert tl.load().tiled_linear_set_stall_allowance(None, 1.0) == tl.TL_ERR_STATE


def test_forward_static_argument_checks(tl):
    """The allocation-free forward refuses bad shapes, oversized tiles and a
    missing status word before any CUDA call, and keeps the reason where
    tiled_linear_last_error(NULL) finds it."""
    lib = tl.load()
    st = ctypes.c_void_p(16)
    assert lib.tiled_linear_forward_static(16, 12, 64, 1, None, None, None, st, None) == tl.TL_ERR_INVALID
    assert "K % 8" in tl.tiled_linear_last_error(None)
    assert lib.tiled_linear_forward_static(1 << 30, 64, 64, 1, None, None, None, st, None) == tl.TL_ERR_INVALID
    assert lib.tiled_linear_forward_static(16, 1 << 30, 64, 1, None, None, None, st, None) == tl.TL_ERR_INVALID
    # one tile of 8192 x 4096 bf16 = 64 MiB > the 32 MiB static slot
    assert lib.tiled_linear_forward_static(16, 8192, 8192, 2, None, None, None, st, None) == tl.TL_ERR_WORKSPACE
    assert "static slot" in tl.tiled_linear_last_error(None)
    # K * (M/N) * 2 would overflow 64 bits if multiplied first
    assert lib.tiled_linear_forward_static(16, (1 << 30) - 8, (1 << 30) - 8, 1, None, None, None, st, None) \
        == tl.TL_ERR_WORKSPACE
    # the largest tile that fits: 2048 x 8184 bf16 = 32 MiB - 32,768 bytes
    assert lib.tiled_linear_forward_static(16, 2048, 8184, 1, 16, 16, 16, None, None) == tl.TL_ERR_INVALID
    assert "status_host" in tl.tiled_linear_last_error(None)
    assert lib.tiled_linear_forward_static(16, 2048, 8192, 1, 16, 16, 16, st, None) == tl.TL_ERR_WORKSPACE


@pytest.mark.parametrize("struct", ["tl_stats", "tl_file_stats", "tl_adam_config", "tl_trace_event"])
def test_stats_struct_layout_matches_the_header(tl, tmp_path, struct):
    """The binding's structs mirror the C structs field by field: a C program
    built against include/tiled_linear.h prints sizeof and every offsetof."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    cls = getattr(tl, struct)
    fields = [name for name, _ in cls._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"tiled_linear.h\"\nint main(void) {\n"
                   f"  printf(\"%zu\\n\", sizeof({struct}));\n"
                   + "".join(f"  printf(\"%zu\\n\", offsetof({struct}, {f}));\n" for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(cls)
    assert out[1:] == [getattr(cls, f).offset for f in fields]


def test_file_tier_argument_checks(tl, tmp_path):
    """Paths, slot and thread counts and the direct-I/O tile size are refused
    before any CUDA call or file access."""
    lib = tl.load()
    w, dw = str(tmp_path / "w.bin").encode(), str(tmp_path / "dw.bin").encode()
    h = ctypes.c_void_p()
    K, M, N = 256, 1024, 4  # tile = 256 * 256 * 2 bytes, a multiple of 4096
    args = lambda **kw: dict(dict(w=w, dw=dw, slots=4, io=2, K=K, M=M, N=N), **kw)
    def create(a):
        return lib.tiled_linear_create_file(ctypes.byref(h), a["K"], a["M"], a["N"], 1, a["w"], a["dw"],
                                            a["slots"], a["io"], 256, 1 << 30, 0)
    assert create(args(w=None)) == tl.TL_ERR_INVALID
    assert create(args(dw=b"")) == tl.TL_ERR_INVALID
    assert create(args(slots=1)) == tl.TL_ERR_INVALID
    assert create(args(slots=65)) == tl.TL_ERR_INVALID
    assert create(args(io=0)) == tl.TL_ERR_INVALID
    assert create(args(K=8, M=64, N=8)) == tl.TL_ERR_INVALID  # 128-byte tiles: no direct I/O
    assert create(args(K=256, M=1000, N=4)) == tl.TL_ERR_INVALID  # tile width 250: not a multiple of 8
    assert h.value is None
    assert lib.tiled_linear_file_sync(None) == tl.TL_ERR_STATE
    assert lib.tiled_linear_file_stats(None, None) == tl.TL_ERR_INVALID
    assert not (tmp_path / "dw.bin").exists()  # nothing was opened


def test_chain_workspace_and_scratch_bytes(tl):
    """Ring slots are sized for the chain's largest tile; d counts tiles over
    all operators; one operator gives the single-operator figure."""
    mib = 1 << 20
    # GPT-scale FFN: up 8192 -> 32768 and down 32768 -> 8192, 8 tiles each (64 MiB tiles)
    assert tl.tiled_linear_chain_workspace_bytes(2, [8192, 32768, 8192], [8, 8], 2) == HEADER + (3 + 2) * 64 * mib
    # tiles of 2 MiB and 4 MiB: five tiles, d = 1 -> 2 ring slots + 2 staging slots of 4 MiB
    assert tl.tiled_linear_chain_workspace_bytes(2, [1024, 4096, 512], [4, 1], 1) == HEADER + 4 * 4 * mib
    for K, M, N, d in [(1024, 4096, 4, 1), (512, 1536, 3, -1), (264, 1200, 3, 0)]:
        assert tl.tiled_linear_chain_workspace_bytes(1, [K, M], [N], d) == tl.tiled_linear_workspace_bytes(K, M, N, d)
    assert tl.tiled_linear_chain_workspace_bytes(2, [1024, 4096, 500], [4, 3], 1) == 0  # 500 % 3
    assert tl.tiled_linear_chain_workspace_bytes(0, [1024], [], 1) == 0
    # fp32 dX and one bf16 dY buffer; two dY buffers from three operators on
    assert tl.tiled_linear_chain_scratch_bytes(100, 2, [64, 256, 64]) == 100 * 256 * 4 + 100 * 256 * 2
    assert tl.tiled_linear_chain_scratch_bytes(100, 3, [64, 256, 128, 64]) == 100 * 256 * 4 + 2 * 100 * 256 * 2
    assert tl.tiled_linear_chain_scratch_bytes(100, 1, [64, 256]) == 0


def test_chain_create_argument_checks(tl):
    lib = tl.load()
    h = ctypes.c_void_p()
    dims = (ctypes.c_int64 * 3)(256, 512, 256)
    n = (ctypes.c_int32 * 2)(2, 2)
    ptrs = (ctypes.c_void_p * 2)(16, 16)
    # mismatched operator count / null arrays / bad shapes are refused before any CUDA call
    assert lib.tiled_linear_chain_create(ctypes.byref(h), 0, dims, n, 1, ptrs, ptrs, 256, 1 << 30, 0) == \
        tl.TL_ERR_INVALID
    assert lib.tiled_linear_chain_create(ctypes.byref(h), 2, dims, n, 1, None, ptrs, 256, 1 << 30, 0) == \
        tl.TL_ERR_INVALID
    bad = (ctypes.c_int32 * 2)(3, 2)  # 512 % 3
    assert lib.tiled_linear_chain_create(ctypes.byref(h), 2, dims, bad, 1, ptrs, ptrs, 256, 1 << 30, 0) == \
        tl.TL_ERR_INVALID
    assert h.value is None
    assert lib.tiled_linear_chain_forward(None, 1, None, None, None) == tl.TL_ERR_STATE
    assert lib.tiled_linear_chain_backward(None, 1, None, None, None, None, None, 0, None) == tl.TL_ERR_STATE
