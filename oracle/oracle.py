"""Python front of the CPU oracle for the streamed tiled linear operator.

TEST INFRASTRUCTURE.  Only the tests, the smoke check in ``__graft_entry__``
and the CPU-baseline / reference legs of ``bench.py`` may import this module.
The library under ``offload_streamed_gb300`` never does, and shares no code
with it.

The arithmetic lives in ``oracle.c`` (plain fp32 triple loops over bf16 bit
patterns, ascending summation order); this file only compiles it with gcc and
marshals numpy arrays.  Inputs are ``np.uint16`` arrays holding bf16 bits,
row-major and C-contiguous:  X [T,K], W [K,M], dY [T,M].  Outputs are fp32.

Definitions (see the header of ``oracle.c`` for the passages they follow):
    Y[t,m]  = sum_k X[t,k] W[k,m]
    dX[t,k] = sum_m dY[t,m] W[k,m]
    dW[k,m] = sum_t X[t,k] dY[t,m]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile ``src`` with gcc into the shared library ``out`` (if stale)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src], check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and type the oracle library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        lib = ctypes.CDLL(path or build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        for name in ("oracle_forward", "oracle_backward_dx", "oracle_backward_dw"):
            fn = getattr(lib, name)
            fn.argtypes = [i64, i64, i64, p, p, p]
            fn.restype = None
        for name in ("oracle_sample_y", "oracle_sample_dx"):
            fn = getattr(lib, name)
            fn.argtypes = [i64, i64, i64, i64, p, p, i64, p, p, p]
            fn.restype = None
        lib.oracle_sample_dw.argtypes = [i64, i64, i64, p, p, i64, p, p, p]
        lib.oracle_sample_dw.restype = None
        lib.oracle_round_bf16.argtypes = [i64, p, p]
        lib.oracle_round_bf16.restype = None
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        if path is None:
            _lib = lib
        return lib


def _bits(a: np.ndarray, shape: tuple[int, int], name: str) -> np.ndarray:
    if a.dtype != np.uint16:
        raise TypeError(f"{name} must hold bf16 bits as np.uint16, got {a.dtype}")
    if tuple(a.shape) != shape:
        raise ValueError(f"{name} has shape {a.shape}, expected {shape}")
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def set_threads(n: int) -> None:
    load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(load().oracle_max_threads())


def forward(X: np.ndarray, W: np.ndarray, lib=None) -> np.ndarray:
    """Untiled Y = X.W in fp32 (ascending k)."""
    T, K = X.shape
    M = W.shape[1]
    X = _bits(X, (T, K), "X")
    W = _bits(W, (K, M), "W")
    Y = np.empty((T, M), np.float32)
    (lib or load()).oracle_forward(T, K, M, _ptr(X), _ptr(W), _ptr(Y))
    return Y


def backward_dx(dY: np.ndarray, W: np.ndarray, lib=None) -> np.ndarray:
    """dX = dY.W^T in fp32 (ascending m)."""
    T, M = dY.shape
    K = W.shape[0]
    dY = _bits(dY, (T, M), "dY")
    W = _bits(W, (K, M), "W")
    dX = np.empty((T, K), np.float32)
    (lib or load()).oracle_backward_dx(T, K, M, _ptr(dY), _ptr(W), _ptr(dX))
    return dX


def backward_dw(X: np.ndarray, dY: np.ndarray, lib=None) -> np.ndarray:
    """dW = X^T.dY in fp32 (ascending t)."""
    T, K = X.shape
    M = dY.shape[1]
    X = _bits(X, (T, K), "X")
    dY = _bits(dY, (T, M), "dY")
    dW = np.empty((K, M), np.float32)
    (lib or load()).oracle_backward_dw(T, K, M, _ptr(X), _ptr(dY), _ptr(dW))
    return dW


def backward(X, W, dY, lib=None):
    return backward_dx(dY, W, lib), backward_dw(X, dY, lib)


def round_bf16(a: np.ndarray, lib=None) -> np.ndarray:
    """bf16 bits (np.uint16) of the fp32 array ``a`` rounded to nearest, ties
    to even (NaN stays NaN)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    (lib or load()).oracle_round_bf16(a.size, _ptr(a), _ptr(out))
    return out


def chain_forward(X: np.ndarray, Ws, lib=None) -> list:
    """Operators in sequence: Y_0 = X.W_0, Y_l = bf16(Y_{l-1}).W_l.  Returns the
    fp32 Y_l of every operator (each from the bf16-rounded input before it)."""
    ys, x = [], X
    for W in Ws:
        y = forward(x, W, lib)
        ys.append(y)
        x = round_bf16(y, lib)
    return ys


def chain_backward(X: np.ndarray, Ws, dY: np.ndarray, lib=None):
    """Backward through chain_forward's operators, last to first: operator l
    takes dY_l (dY for the last, bf16(dX_{l+1}) before it) and its input X_l
    (X, then bf16(Y_{l-1})); dX_l = dY_l.W_l^T, dW_l = X_l^T.dY_l.  Returns
    (dX_0 in fp32, [dW_0, ..., dW_{L-1}] in fp32)."""
    xs, x = [], X
    for W in Ws[:-1]:
        xs.append(x)
        x = round_bf16(forward(x, W, lib), lib)
    xs.append(x)
    dws = [None] * len(Ws)
    dy = dY
    dx = None
    for l in range(len(Ws) - 1, -1, -1):
        dx = backward_dx(dy, Ws[l], lib)
        dws[l] = backward_dw(xs[l], dy, lib)
        if l > 0:
            dy = round_bf16(dx, lib)
    return dx, dws


def _idx(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _w_storage(W: np.ndarray) -> tuple[np.ndarray, int, int, int]:
    """Accept W row-major [K, M], or stored tile by tile as [N, K, C] (N column
    blocks of C columns each).  Returns (W, K, M, C); C = M when row-major."""
    if W.ndim == 2:
        K, M = W.shape
        return _bits(W, (K, M), "W"), K, M, M
    if W.ndim == 3:
        N, K, C = W.shape
        return _bits(W, (N, K, C), "W"), K, N * C, C
    raise ValueError("W must be [K, M] or [N, K, M/N]")


def sample_y(X, W, rows, cols, lib=None) -> np.ndarray:
    """Y at the entries (rows[i] = t, cols[i] = m); equals ``forward`` bit for
    bit.  W is [K, M] row-major, or tile-major [N, K, M/N]."""
    T, K = X.shape
    Ws, KW, M, C = _w_storage(W)
    if KW != K:
        raise ValueError("X and W disagree on K")
    rows, cols = _idx(rows), _idx(cols)
    _check_idx(rows, T, cols, M)
    out = np.empty(rows.shape[0], np.float32)
    (lib or load()).oracle_sample_y(T, K, M, C, _ptr(_bits(X, (T, K), "X")),
                                    _ptr(Ws), rows.shape[0],
                                    _ptr(rows), _ptr(cols), _ptr(out))
    return out


def sample_dx(dY, W, rows, cols, lib=None) -> np.ndarray:
    """dX at the entries (rows[i] = t, cols[i] = k).  W as in ``sample_y``."""
    T, M = dY.shape
    Ws, K, MW, C = _w_storage(W)
    if MW != M:
        raise ValueError("dY and W disagree on M")
    rows, cols = _idx(rows), _idx(cols)
    _check_idx(rows, T, cols, K)
    out = np.empty(rows.shape[0], np.float32)
    (lib or load()).oracle_sample_dx(T, K, M, C, _ptr(_bits(dY, (T, M), "dY")),
                                     _ptr(Ws), rows.shape[0],
                                     _ptr(rows), _ptr(cols), _ptr(out))
    return out


def sample_dw(X, dY, rows, cols, lib=None) -> np.ndarray:
    """dW at the entries (rows[i] = k, cols[i] = m)."""
    T, K = X.shape
    M = dY.shape[1]
    rows, cols = _idx(rows), _idx(cols)
    _check_idx(rows, K, cols, M)
    out = np.empty(rows.shape[0], np.float32)
    (lib or load()).oracle_sample_dw(T, K, M, _ptr(_bits(X, (T, K), "X")),
                                     _ptr(_bits(dY, (T, M), "dY")), rows.shape[0],
                                     _ptr(rows), _ptr(cols), _ptr(out))
    return out


def _check_idx(rows, nrows, cols, ncols):
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and of equal length")
    if rows.size and (rows.min() < 0 or rows.max() >= nrows
                      or cols.min() < 0 or cols.max() >= ncols):
        raise IndexError("sample index out of range")
