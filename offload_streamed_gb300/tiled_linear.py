"""Python binding of ``libtiled_linear.so`` (the C ABI in ``include/tiled_linear.h``).

Argument marshalling only: every step of the forward / backward path runs in
the library's CUDA kernels and copy streams.  There is no fallback: if the
shared library is missing or fails to load, every entry point raises.

Module-level functions carry the C names and take plain integers (pointers,
sizes, stream handles).  ``TiledLinear`` and ``PinnedBuffer`` wrap them for
PyTorch callers: PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

(TL_OK, TL_ERR_INVALID, TL_ERR_NOT_PINNED, TL_ERR_WORKSPACE, TL_ERR_CUDA, TL_ERR_TIMEOUT, TL_ERR_STATE,
 TL_ERR_IO) = range(8)
STATUS_NAMES = {0: "TL_OK", 1: "TL_ERR_INVALID", 2: "TL_ERR_NOT_PINNED", 3: "TL_ERR_WORKSPACE",
                4: "TL_ERR_CUDA", 5: "TL_ERR_TIMEOUT", 6: "TL_ERR_STATE", 7: "TL_ERR_IO"}


class TiledLinearError(RuntimeError):
    def __init__(self, status: int, where: str, message: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}"
                         + (f" ({message})" if message else ""))


class tl_stats(ctypes.Structure):
    _fields_ = [
        ("n_tiles", ctypes.c_int32), ("depth", ctypes.c_int32),
        ("fwd_valid", ctypes.c_int32), ("bwd_valid", ctypes.c_int32),
        ("fwd_total_ms", ctypes.c_float), ("fwd_gemm_ms", ctypes.c_float), ("fwd_h2d_ms", ctypes.c_float),
        ("bwd_total_ms", ctypes.c_float), ("bwd_dw_gemm_ms", ctypes.c_float),
        ("bwd_dx_gemm_ms", ctypes.c_float), ("bwd_h2d_ms", ctypes.c_float), ("bwd_d2h_ms", ctypes.c_float),
        ("fwd_wait_ms", ctypes.c_float), ("bwd_wait_ms", ctypes.c_float),
        ("fwd_h2d_bytes", ctypes.c_int64), ("bwd_h2d_bytes", ctypes.c_int64), ("bwd_d2h_bytes", ctypes.c_int64),
        ("fwd_launches", ctypes.c_int32), ("bwd_launches", ctypes.c_int32),
        ("fwd_calls", ctypes.c_int64), ("bwd_calls", ctypes.c_int64),
        ("sum_fwd_total_ms", ctypes.c_double), ("sum_fwd_gemm_ms", ctypes.c_double),
        ("sum_fwd_h2d_ms", ctypes.c_double), ("sum_bwd_total_ms", ctypes.c_double),
        ("sum_bwd_dw_gemm_ms", ctypes.c_double), ("sum_bwd_dx_gemm_ms", ctypes.c_double),
        ("sum_bwd_h2d_ms", ctypes.c_double), ("sum_bwd_d2h_ms", ctypes.c_double),
        ("sum_bwd_gemm_ms", ctypes.c_double), ("bwd_gemm_ms", ctypes.c_float), ("staging_slots", ctypes.c_int32),
        ("bwd_reused_tiles", ctypes.c_int32),
        ("fwd_timed_calls", ctypes.c_int64), ("bwd_timed_calls", ctypes.c_int64), ("timing_every", ctypes.c_int32),
        ("fwd_h2d_max_ms", ctypes.c_float),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class tl_file_stats(ctypes.Structure):
    _fields_ = [("read_bytes", ctypes.c_int64), ("write_bytes", ctypes.c_int64),
                ("read_seconds", ctypes.c_double), ("write_seconds", ctypes.c_double),
                ("fetch_wait_seconds", ctypes.c_double), ("writeback_wait_seconds", ctypes.c_double),
                ("host_slots", ctypes.c_int32), ("io_threads", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


TL_TRACE_FWD_GEMM, TL_TRACE_DW_GEMM, TL_TRACE_DX_GEMM, TL_TRACE_H2D, TL_TRACE_D2H = range(5)
TRACE_KINDS = {0: "fwd_gemm", 1: "dw_gemm", 2: "dx_gemm", 3: "h2d", 4: "d2h"}


class tl_trace_event(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("tile", ctypes.c_int32),
                ("start_ms", ctypes.c_float), ("end_ms", ctypes.c_float)]


class tl_adam_config(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("threads", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return _build.LIB


def load():
    """Load the shared library (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(path)
        i64, i32, sz, vp, st = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
        L.tiled_linear_workspace_bytes.argtypes = [i64, i64, i32, i32]
        L.tiled_linear_workspace_bytes.restype = sz
        for name in ("tiled_linear_create", "tiled_linear_create_tilemajor"):
            fn = getattr(L, name)
            fn.argtypes = [ctypes.POINTER(vp), i64, i64, i32, i32, vp, vp, vp, sz, ctypes.c_int]
            fn.restype = st
        L.tiled_linear_create_file.argtypes = [ctypes.POINTER(vp), i64, i64, i32, i32, ctypes.c_char_p,
                                               ctypes.c_char_p, i32, i32, vp, sz, ctypes.c_int]
        L.tiled_linear_create_file.restype = st
        L.tiled_linear_file_sync.argtypes = [vp]
        L.tiled_linear_file_sync.restype = st
        L.tiled_linear_file_stats.argtypes = [vp, vp]
        L.tiled_linear_file_stats.restype = st
        L.tiled_linear_forward.argtypes = [vp, i64, vp, vp, vp]
        L.tiled_linear_forward.restype = st
        L.tiled_linear_backward.argtypes = [vp, i64, vp, vp, vp, vp]
        L.tiled_linear_backward.restype = st
        L.tiled_linear_destroy.argtypes = [vp]
        L.tiled_linear_destroy.restype = st
        L.tiled_linear_last_error.argtypes = [vp]
        L.tiled_linear_last_error.restype = ctypes.c_char_p
        L.tiled_linear_get_stats.argtypes = [vp, vp]
        L.tiled_linear_get_stats.restype = st
        L.tiled_linear_get_trace.argtypes = [vp, i32, vp, i32, ctypes.POINTER(i32)]
        L.tiled_linear_get_trace.restype = st
        L.tiled_linear_reset_stats.argtypes = [vp]
        L.tiled_linear_reset_stats.restype = st
        L.tiled_linear_set_tile_reuse.argtypes = [vp, i32]
        L.tiled_linear_set_tile_reuse.restype = st
        L.tiled_linear_set_timing.argtypes = [vp, i32]
        L.tiled_linear_set_timing.restype = st
        L.tiled_linear_set_stall_allowance.argtypes = [vp, ctypes.c_double]
        L.tiled_linear_set_stall_allowance.restype = st
        L.tiled_linear_adam_update.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, vp]
        L.tiled_linear_adam_update.restype = st
        L.tiled_linear_optimizer_create.argtypes = [ctypes.POINTER(vp), vp, vp, vp, vp, vp, vp]
        L.tiled_linear_optimizer_create.restype = st
        for name in ("tiled_linear_optimizer_accumulate", "tiled_linear_optimizer_step",
                     "tiled_linear_optimizer_wait", "tiled_linear_optimizer_destroy"):
            getattr(L, name).argtypes = [vp]
            getattr(L, name).restype = st
        L.tiled_linear_optimizer_stats.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]
        L.tiled_linear_optimizer_stats.restype = st
        L.tiled_linear_chain_workspace_bytes.argtypes = [i32, vp, vp, i32]
        L.tiled_linear_chain_workspace_bytes.restype = sz
        L.tiled_linear_chain_create.argtypes = [ctypes.POINTER(vp), i32, vp, vp, i32, vp, vp, vp, sz, ctypes.c_int]
        L.tiled_linear_chain_create.restype = st
        L.tiled_linear_chain_forward.argtypes = [vp, i64, vp, vp, vp]
        L.tiled_linear_chain_forward.restype = st
        L.tiled_linear_chain_scratch_bytes.argtypes = [i64, i32, vp]
        L.tiled_linear_chain_scratch_bytes.restype = sz
        L.tiled_linear_chain_backward.argtypes = [vp, i64, vp, vp, vp, vp, vp, sz, vp]
        L.tiled_linear_chain_backward.restype = st
        L.tiled_linear_gemm_forward.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, vp]
        L.tiled_linear_gemm_forward.restype = st
        L.tiled_linear_gemm_dw.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, vp]
        L.tiled_linear_gemm_dw.restype = st
        L.tiled_linear_gemm_dx.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, i32, vp, vp]
        L.tiled_linear_gemm_dx.restype = st
        L.tiled_linear_gemm_dx_bf16.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp, vp]
        L.tiled_linear_gemm_dx_bf16.restype = st
        L.tiled_linear_selftest_timeout.argtypes = [vp, sz, i64, vp]
        L.tiled_linear_selftest_timeout.restype = st
        L.tiled_linear_forward_static.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, vp]
        L.tiled_linear_forward_static.restype = st
        L.tiled_linear_host_alloc.argtypes = [sz, ctypes.POINTER(vp)]
        L.tiled_linear_host_alloc.restype = st
        L.tiled_linear_host_free.argtypes = [vp]
        L.tiled_linear_host_free.restype = st
        L.tiled_linear_version.restype = ctypes.c_char_p
        _lib = L
        return L


def _check(status: int, where: str, handle=None):
    if status != TL_OK:
        raise TiledLinearError(status, where, tiled_linear_last_error(handle))


# --- the C ABI, name for name ----------------------------------------------

def tiled_linear_workspace_bytes(K: int, M: int, N: int, d: int) -> int:
    return int(load().tiled_linear_workspace_bytes(K, M, N, d))


def tiled_linear_create(K, M, N, d, w_host, dw_host, workspace_dev, workspace_bytes, device,
                        tile_major: bool = False) -> int:
    """Returns the handle (an integer).  ``tile_major`` selects
    ``tiled_linear_create_tilemajor``."""
    h = ctypes.c_void_p()
    fn = load().tiled_linear_create_tilemajor if tile_major else load().tiled_linear_create
    _check(fn(ctypes.byref(h), K, M, N, d, w_host, dw_host, workspace_dev, workspace_bytes, device),
           "tiled_linear_create")
    return h.value


def tiled_linear_create_tilemajor(K, M, N, d, w_host, dw_host, workspace_dev, workspace_bytes,
                                  device) -> int:
    return tiled_linear_create(K, M, N, d, w_host, dw_host, workspace_dev, workspace_bytes, device,
                               tile_major=True)


def tiled_linear_create_file(K, M, N, d, w_path: str, dw_path: str, host_slots: int, io_threads: int,
                             workspace_dev, workspace_bytes, device) -> int:
    """W and dW in files (tile-major), streamed through pinned host slots."""
    h = ctypes.c_void_p()
    _check(load().tiled_linear_create_file(ctypes.byref(h), K, M, N, d, os.fsencode(w_path), os.fsencode(dw_path),
                                           host_slots, io_threads, workspace_dev, workspace_bytes, device),
           "tiled_linear_create_file")
    return h.value


def tiled_linear_file_sync(h: int) -> None:
    _check(load().tiled_linear_file_sync(h), "tiled_linear_file_sync", h)


def tiled_linear_file_stats(h: int) -> dict:
    s = tl_file_stats()
    _check(load().tiled_linear_file_stats(h, ctypes.byref(s)), "tiled_linear_file_stats", h)
    return s.as_dict()


def tiled_linear_forward(h: int, T: int, x_dev: int, y_dev: int, stream: int) -> None:
    _check(load().tiled_linear_forward(h, T, x_dev, y_dev, stream), "tiled_linear_forward", h)


def tiled_linear_backward(h: int, T: int, x_dev: int, dy_dev: int, dx_dev: int, stream: int) -> None:
    _check(load().tiled_linear_backward(h, T, x_dev, dy_dev, dx_dev, stream), "tiled_linear_backward", h)


def tiled_linear_destroy(h: int) -> int:
    return int(load().tiled_linear_destroy(h))


def tiled_linear_last_error(h=None) -> str:
    msg = load().tiled_linear_last_error(h)
    return msg.decode(errors="replace") if msg else ""


def tiled_linear_get_stats(h: int) -> dict:
    s = tl_stats()
    _check(load().tiled_linear_get_stats(h, ctypes.byref(s)), "tiled_linear_get_stats", h)
    return s.as_dict()


def tiled_linear_get_trace(h: int, backward: bool) -> list:
    """The last timed forward / backward call's launches and copies: a list of
    {"kind", "tile", "start_ms", "end_ms"} (see include/tiled_linear.h)."""
    n = ctypes.c_int32(0)
    _check(load().tiled_linear_get_trace(h, 1 if backward else 0, None, 0, ctypes.byref(n)),
           "tiled_linear_get_trace", h)
    buf = (tl_trace_event * max(n.value, 1))()
    _check(load().tiled_linear_get_trace(h, 1 if backward else 0, buf, n.value, ctypes.byref(n)),
           "tiled_linear_get_trace", h)
    return [{"kind": TRACE_KINDS[e.kind], "tile": e.tile, "start_ms": e.start_ms, "end_ms": e.end_ms}
            for e in buf[:n.value]]


def tiled_linear_reset_stats(h: int) -> None:
    _check(load().tiled_linear_reset_stats(h), "tiled_linear_reset_stats", h)


def tiled_linear_set_timing(h: int, every: int) -> None:
    _check(load().tiled_linear_set_timing(h, int(every)), "tiled_linear_set_timing", h)


def tiled_linear_set_tile_reuse(h: int, enable: bool) -> None:
    _check(load().tiled_linear_set_tile_reuse(h, 1 if enable else 0), "tiled_linear_set_tile_reuse", h)


def tiled_linear_set_stall_allowance(h: int, ms: float) -> None:
    _check(load().tiled_linear_set_stall_allowance(h, float(ms)), "tiled_linear_set_stall_allowance", h)


def _i64s(v):
    return (ctypes.c_int64 * len(v))(*[int(a) for a in v])


def _i32s(v):
    return (ctypes.c_int32 * len(v))(*[int(a) for a in v])


def _ptrs(v):
    return (ctypes.c_void_p * len(v))(*[int(a) if a else None for a in v])


def tiled_linear_chain_workspace_bytes(L: int, dims, n_tiles, d: int) -> int:
    return int(load().tiled_linear_chain_workspace_bytes(L, _i64s(dims), _i32s(n_tiles), d))


def tiled_linear_chain_create(L, dims, n_tiles, d, w_hosts, dw_hosts, workspace_dev, workspace_bytes,
                              device) -> int:
    h = ctypes.c_void_p()
    _check(load().tiled_linear_chain_create(ctypes.byref(h), L, _i64s(dims), _i32s(n_tiles), d,
                                            _ptrs(w_hosts), _ptrs(dw_hosts), workspace_dev, workspace_bytes,
                                            device), "tiled_linear_chain_create")
    return h.value


def tiled_linear_chain_forward(h: int, T: int, x_dev: int, y_devs, stream: int) -> None:
    _check(load().tiled_linear_chain_forward(h, T, x_dev, _ptrs(y_devs), stream), "tiled_linear_chain_forward", h)


def tiled_linear_chain_scratch_bytes(T: int, L: int, dims) -> int:
    return int(load().tiled_linear_chain_scratch_bytes(T, L, _i64s(dims)))


def tiled_linear_chain_backward(h: int, T: int, x_dev: int, y_devs, dy_dev: int, dx_dev: int, scratch_dev: int,
                                scratch_bytes: int, stream: int) -> None:
    _check(load().tiled_linear_chain_backward(h, T, x_dev, _ptrs(y_devs) if y_devs is not None else None, dy_dev,
                                              dx_dev, scratch_dev, scratch_bytes, stream),
           "tiled_linear_chain_backward", h)


def adam_config(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, threads=0) -> tl_adam_config:
    return tl_adam_config(lr, beta1, beta2, eps, weight_decay, threads)


def tiled_linear_adam_update(cfg: tl_adam_config, step: int, n: int, master: int, m: int, v: int, grad_acc: int,
                             grad_bf16: int, w_bf16: int) -> None:
    _check(load().tiled_linear_adam_update(ctypes.byref(cfg), step, n, master, m, v, grad_acc or None, grad_bf16,
                                           w_bf16), "tiled_linear_adam_update")


def tiled_linear_optimizer_create(h: int, cfg: tl_adam_config, masters, ms, vs, accs=None) -> int:
    o = ctypes.c_void_p()
    _check(load().tiled_linear_optimizer_create(ctypes.byref(o), h, ctypes.byref(cfg), _ptrs(masters), _ptrs(ms),
                                                _ptrs(vs), _ptrs(accs) if accs else None),
           "tiled_linear_optimizer_create", h)
    return o.value


def tiled_linear_optimizer_accumulate(o: int, h=None) -> None:
    _check(load().tiled_linear_optimizer_accumulate(o), "tiled_linear_optimizer_accumulate", h)


def tiled_linear_optimizer_step(o: int, h=None) -> None:
    _check(load().tiled_linear_optimizer_step(o), "tiled_linear_optimizer_step", h)


def tiled_linear_optimizer_wait(o: int, h=None) -> None:
    _check(load().tiled_linear_optimizer_wait(o), "tiled_linear_optimizer_wait", h)


def tiled_linear_optimizer_stats(o: int) -> tuple:
    steps, busy = ctypes.c_int64(), ctypes.c_double()
    _check(load().tiled_linear_optimizer_stats(o, ctypes.byref(steps), ctypes.byref(busy)),
           "tiled_linear_optimizer_stats")
    return steps.value, busy.value


def tiled_linear_optimizer_destroy(o: int) -> int:
    return int(load().tiled_linear_optimizer_destroy(o))


def tiled_linear_gemm_forward(T, K, n, x, ldx, w, ldw, y, ldy, err, stream) -> None:
    _check(load().tiled_linear_gemm_forward(T, K, n, x, ldx, w, ldw, y, ldy, err, stream),
           "tiled_linear_gemm_forward")


def tiled_linear_gemm_dw(T, K, n, x, ldx, dy, lddy, dw, lddw, err, stream) -> None:
    _check(load().tiled_linear_gemm_dw(T, K, n, x, ldx, dy, lddy, dw, lddw, err, stream),
           "tiled_linear_gemm_dw")


def tiled_linear_gemm_dx(T, K, n, dy, lddy, w, ldw, dx, lddx, accumulate, err, stream) -> None:
    _check(load().tiled_linear_gemm_dx(T, K, n, dy, lddy, w, ldw, dx, lddx, int(accumulate), err, stream),
           "tiled_linear_gemm_dx")


def tiled_linear_gemm_dx_bf16(T, K, n, dy, lddy, w, ldw, addend, ld_add, dx, lddx, err, stream) -> None:
    _check(load().tiled_linear_gemm_dx_bf16(T, K, n, dy, lddy, w, ldw, addend, ld_add, dx, lddx, err, stream),
           "tiled_linear_gemm_dx_bf16")


def tiled_linear_selftest_timeout(scratch_dev: int, scratch_bytes: int, timeout_ns: int, stream: int) -> None:
    """Run the kernels' failure path once (see the header); the error bits
    land in the first int32 of scratch_dev."""
    _check(load().tiled_linear_selftest_timeout(scratch_dev, scratch_bytes, timeout_ns, stream),
           "tiled_linear_selftest_timeout")


def tiled_linear_forward_static(T, K, M, N, w_host, x_dev, y_dev, status_host, stream) -> None:
    """Forward with no device allocation (scratch in a static device array);
    see the header for its limit and ordering rules."""
    st = load().tiled_linear_forward_static(T, K, M, N, w_host, x_dev, y_dev, status_host, stream)
    if st != TL_OK:
        raise TiledLinearError(st, "tiled_linear_forward_static")


def tiled_linear_host_alloc(nbytes: int) -> int:
    p = ctypes.c_void_p()
    _check(load().tiled_linear_host_alloc(nbytes, ctypes.byref(p)), "tiled_linear_host_alloc")
    return p.value


def tiled_linear_host_free(p: int) -> None:
    _check(load().tiled_linear_host_free(p), "tiled_linear_host_free")


def tiled_linear_version() -> str:
    return load().tiled_linear_version().decode()


# --- PyTorch convenience wrappers --------------------------------------------

def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def host_tensor(ptr: int, numel: int, dtype=None):
    """Wrap ``numel`` elements of host memory at ``ptr`` as a CPU tensor (no
    copy; the memory stays owned by whoever allocated it)."""
    import torch
    dtype = dtype or torch.bfloat16
    itemsize = torch.empty((), dtype=dtype).element_size()
    buf = (ctypes.c_uint8 * (numel * itemsize)).from_address(ptr)
    return torch.frombuffer(buf, dtype=torch.uint8).view(dtype)


class PinnedBuffer:
    """Page-locked host memory from ``tiled_linear_host_alloc``, viewed as a
    CPU tensor of ``dtype``.  Freed by ``close()`` (or garbage collection)."""

    def __init__(self, numel: int, dtype=None):
        import torch
        self.dtype = dtype or torch.bfloat16
        self.numel = int(numel)
        itemsize = torch.empty((), dtype=self.dtype).element_size()
        self.nbytes = self.numel * itemsize
        self.ptr = tiled_linear_host_alloc(max(self.nbytes, 16))
        self.tensor = host_tensor(self.ptr, self.numel, self.dtype)

    def close(self):
        if self.ptr:
            self.tensor = None
            tiled_linear_host_free(self.ptr)
            self.ptr = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class TiledLinear:
    """Y = X.W with W [K, M] in pinned host memory, streamed in N output tiles
    through a depth-d device ring (see ``include/tiled_linear.h``).

    w_host / dw_host: pinned host buffers (``PinnedBuffer`` or a pinned CPU
    tensor) of K*M bf16 each, tile-major [N][K][M/N] when ``tile_major`` else
    row-major [K][M].  The workspace is a device uint8 tensor owned here.

    d = -1 (automatic depth): the workspace holds as many ring and staging
    slots as ``auto_workspace_bytes`` allows (default: half of the device's
    free memory), at most N of each."""

    def __init__(self, K: int, M: int, N: int, d: int, w_host, dw_host, *, tile_major: bool = True,
                 device=None, auto_workspace_bytes: int | None = None):
        import torch
        self.K, self.M, self.N, self.d = int(K), int(M), int(N), int(d)
        self.Mi = self.M // self.N
        self.tile_major = bool(tile_major)
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        wb = tiled_linear_workspace_bytes(self.K, self.M, self.N, self.d)
        if wb == 0:
            raise TiledLinearError(TL_ERR_INVALID, "tiled_linear_workspace_bytes",
                                   f"invalid shape K={K} M={M} N={N} d={d}")
        if self.d < 0:
            least = tiled_linear_workspace_bytes(self.K, self.M, self.N, min(1, self.N - 1))
            budget = auto_workspace_bytes
            if budget is None:
                budget = torch.cuda.mem_get_info(self.device)[0] // 2
            wb = max(least, min(wb, int(budget)))
        self.workspace = torch.empty(wb, dtype=torch.uint8, device=self.device)
        self._w, self._dw = w_host, dw_host
        wp = w_host.ptr if isinstance(w_host, PinnedBuffer) else w_host.data_ptr()
        dwp = dw_host.ptr if isinstance(dw_host, PinnedBuffer) else dw_host.data_ptr()
        self.handle = tiled_linear_create(self.K, self.M, self.N, self.d, wp, dwp,
                                          self.workspace.data_ptr(), wb, self.device.index,
                                          tile_major=self.tile_major)

    def forward(self, x, y=None, stream=None):
        import torch
        T = x.shape[0]
        if y is None:
            y = torch.empty(T, self.M, dtype=torch.bfloat16, device=self.device)
        tiled_linear_forward(self.handle, T, x.data_ptr(), y.data_ptr(), _stream_handle(stream))
        return y

    def backward(self, x, dy, dx=None, stream=None):
        import torch
        T = x.shape[0]
        if dx is None:
            dx = torch.empty(T, self.K, dtype=torch.float32, device=self.device)
        tiled_linear_backward(self.handle, T, x.data_ptr(), dy.data_ptr(), dx.data_ptr(),
                              _stream_handle(stream))
        return dx

    def stats(self) -> dict:
        return tiled_linear_get_stats(self.handle)

    def reset_stats(self) -> None:
        tiled_linear_reset_stats(self.handle)

    def trace(self, backward: bool) -> list:
        """Launch and copy timeline of the last timed forward / backward call."""
        return tiled_linear_get_trace(self.handle, backward)

    def set_tile_reuse(self, enable: bool = True) -> None:
        """Let backward calls take the tiles still resident from the calls
        before them (W must not change in between)."""
        tiled_linear_set_tile_reuse(self.handle, enable)

    def set_timing(self, every: int) -> None:
        """Record per-launch / per-copy timing events on every `every`-th call."""
        tiled_linear_set_timing(self.handle, every)

    def set_stall_allowance(self, ms: float) -> None:
        """Automatic depth: host-link stall (ms) the ring is sized to ride out."""
        tiled_linear_set_stall_allowance(self.handle, ms)

    def close(self) -> int:
        st = TL_OK
        if self.handle:
            st = tiled_linear_destroy(self.handle)
            self.handle = 0
        return st

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class TiledLinearFile(TiledLinear):
    """A ``TiledLinear`` whose W and dW live in files (tile-major [N][K][M/N]
    bf16), one storage tier below host memory: reader threads stream the
    tiles into pinned host slots with direct I/O, ahead of the host->device
    copies, and writer threads store dW.  ``sync()`` waits until the dW of the
    backward calls made so far is in ``dw_path``."""

    def __init__(self, K: int, M: int, N: int, d: int, w_path: str, dw_path: str, *, host_slots: int = 4,
                 io_threads: int = 4, device=None):
        import torch
        self.K, self.M, self.N, self.d = int(K), int(M), int(N), int(d)
        self.Mi = self.M // self.N
        self.tile_major = True
        self.w_path, self.dw_path = str(w_path), str(dw_path)
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        self.handle = 0
        wb = tiled_linear_workspace_bytes(self.K, self.M, self.N, self.d)
        if wb == 0:
            raise TiledLinearError(TL_ERR_INVALID, "tiled_linear_workspace_bytes",
                                   f"invalid shape K={K} M={M} N={N} d={d}")
        self.workspace = torch.empty(wb, dtype=torch.uint8, device=self.device)
        self.handle = tiled_linear_create_file(self.K, self.M, self.N, self.d, self.w_path, self.dw_path,
                                               int(host_slots), int(io_threads), self.workspace.data_ptr(), wb,
                                               self.device.index)

    def sync(self) -> None:
        """Wait for the device, then for the writers: dW is in ``dw_path``."""
        import torch
        torch.cuda.synchronize(self.device)
        tiled_linear_file_sync(self.handle)

    def file_stats(self) -> dict:
        return tiled_linear_file_stats(self.handle)


class TiledLinearChain:
    """A chain of tiled linear operators (see the chain section of
    ``include/tiled_linear.h``): operator l maps dims[l] -> dims[l+1] with its
    W_l in n_tiles[l] column tiles, tile-major in pinned host memory.  One
    ring and one prefetcher serve the whole chain."""

    def __init__(self, dims, n_tiles, d: int, w_hosts, dw_hosts, device=None):
        import torch
        self.dims = [int(v) for v in dims]
        self.n_tiles = [int(v) for v in n_tiles]
        self.L = len(self.n_tiles)
        if len(self.dims) != self.L + 1:
            raise ValueError("dims needs one entry more than n_tiles")
        self.d = int(d)
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        wb = tiled_linear_chain_workspace_bytes(self.L, self.dims, self.n_tiles, self.d)
        if wb == 0:
            raise TiledLinearError(TL_ERR_INVALID, "tiled_linear_chain_workspace_bytes",
                                   f"invalid chain dims={self.dims} n_tiles={self.n_tiles} d={d}")
        self.workspace = torch.empty(wb, dtype=torch.uint8, device=self.device)
        self._w, self._dw = list(w_hosts), list(dw_hosts)
        ptr = lambda b: b.ptr if isinstance(b, PinnedBuffer) else b.data_ptr()
        self.handle = tiled_linear_chain_create(self.L, self.dims, self.n_tiles, self.d,
                                                [ptr(b) for b in self._w], [ptr(b) for b in self._dw],
                                                self.workspace.data_ptr(), wb, self.device.index)
        self._scratch = None

    def forward(self, x, ys=None, stream=None):
        """Returns the list of every operator's output (keep it for backward)."""
        import torch
        T = x.shape[0]
        if ys is None:
            ys = [torch.empty(T, self.dims[l + 1], dtype=torch.bfloat16, device=self.device)
                  for l in range(self.L)]
        tiled_linear_chain_forward(self.handle, T, x.data_ptr(), [y.data_ptr() for y in ys],
                                   _stream_handle(stream))
        return ys

    def backward(self, x, ys, dy, dx=None, stream=None):
        import torch
        T = x.shape[0]
        if dx is None:
            dx = torch.empty(T, self.dims[0], dtype=torch.float32, device=self.device)
        need = tiled_linear_chain_scratch_bytes(T, self.L, self.dims)
        if need and (self._scratch is None or self._scratch.numel() < need):
            self._scratch = torch.empty(need, dtype=torch.uint8, device=self.device)
        sp = self._scratch.data_ptr() if need else 0
        tiled_linear_chain_backward(self.handle, T, x.data_ptr(), [y.data_ptr() for y in ys] if ys else None,
                                    dy.data_ptr(), dx.data_ptr(), sp, need, _stream_handle(stream))
        return dx

    def stats(self) -> dict:
        return tiled_linear_get_stats(self.handle)

    def reset_stats(self) -> None:
        tiled_linear_reset_stats(self.handle)

    def trace(self, backward: bool) -> list:
        """Launch and copy timeline of the last timed forward / backward call."""
        return tiled_linear_get_trace(self.handle, backward)

    def set_tile_reuse(self, enable: bool = True) -> None:
        tiled_linear_set_tile_reuse(self.handle, enable)

    def close(self) -> int:
        st = TL_OK
        if self.handle:
            st = tiled_linear_destroy(self.handle)
            self.handle = 0
        return st

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostAdam:
    """The Adam step on the host CPU for a ``TiledLinear`` or
    ``TiledLinearChain`` (see the optimizer section of
    ``include/tiled_linear.h``).  Keeps fp32 master weights (initialised from
    the op's host W), first and second moments, and optionally an fp32
    gradient accumulator, in the layout of each operator's host W.  After a
    backward call, ``step()`` (or ``accumulate()``) returns at once; the update
    overlaps the GPU, and the op's next calls wait for the tiles they read."""

    def __init__(self, op, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, threads=0,
                 accumulate=False):
        import torch
        self.op = op
        self.handle = 0
        if getattr(op, "_w", None) is None:
            raise TiledLinearError(TL_ERR_INVALID, "HostAdam", "the host optimizer needs W and dW in host memory")
        ws = op._w if isinstance(op._w, list) else [op._w]
        hosts = [b.tensor if isinstance(b, PinnedBuffer) else b for b in ws]
        self.master = [h.view(-1).float() for h in hosts]
        self.m = [torch.zeros_like(a) for a in self.master]
        self.v = [torch.zeros_like(a) for a in self.master]
        self.acc = [torch.zeros_like(a) for a in self.master] if accumulate else None
        self.cfg = adam_config(lr, beta1, beta2, eps, weight_decay, threads)
        ptr = lambda ts: [t.data_ptr() for t in ts]
        self.handle = tiled_linear_optimizer_create(op.handle, self.cfg, ptr(self.master), ptr(self.m), ptr(self.v),
                                                    ptr(self.acc) if self.acc else None)

    def step(self) -> None:
        tiled_linear_optimizer_step(self.handle, self.op.handle)

    def accumulate(self) -> None:
        tiled_linear_optimizer_accumulate(self.handle, self.op.handle)

    def wait(self) -> None:
        tiled_linear_optimizer_wait(self.handle, self.op.handle)

    def stats(self) -> dict:
        steps, busy = tiled_linear_optimizer_stats(self.handle)
        return {"steps": steps, "busy_seconds": busy}

    def close(self) -> int:
        st = TL_OK
        if self.handle:
            st = tiled_linear_optimizer_destroy(self.handle)
            self.handle = 0
        return st

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
