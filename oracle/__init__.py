"""CPU oracle for the sum-reduction library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The library (``libtcr``) never does,
and this package imports nothing from it: the two share no code.

The arithmetic lives in ``tcr_oracle.c`` (plain C, binary32 additions with
no contraction, an exact fixed-point accumulator for the exact sum); this
module only compiles it with gcc and marshals numpy arrays through ctypes.

Functions (sources are cited in ``tcr_oracle.c``):

``exact_sum``          exact sum rounded once to binary64, and sum of |x|
                       ("GPU Tensor Cores for fast Arithmetic Reductions",
                       Abstract: the arithmetic reduction of n numbers).
``fixed_order``        balanced binary32 tree over index order, -0.0 pad
                       ("Taming Bitwise Behavior in GPU Kernels with Tensor
                       Core", Abstract: balanced-tree reduction order).
``shuffle_tree``       declared order of the conventional reduction
                       (grid-stride accumulation, warp butterfly, block tree,
                       grid tree).
``blocked_order``      runs of 2^c inputs added left to right, then the
                       balanced tree over the runs (a second declared order
                       of the fixed-order mode).
``mean_var``           per-row mean and variance from a row's sum and sum
                       of squares (declared binary32 formula).
``gemm_f64``, ``gemm_splitk``
                       C = A W^T in binary64, and the declared split-K order
                       (balanced tree over once-rounded split partials).
``*_sq``, ``exact_sum_squares``
                       the same over the leaves x_i^2 (sum of squares).
``*_rows``             the same, one result per row.

Inputs are binary16 / bfloat16 patterns (uint16, or float16 arrays) or
binary32 values (float32 or uint32 patterns, dtype ``F32``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tcr_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

F16 = 0
BF16 = 1
F32 = 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``tcr_oracle.c`` into ``_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = f"{_LIB}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.c_void_p      # 16-bit or (binary32) 32-bit patterns
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            sz, i = ctypes.c_size_t, ctypes.c_int
            lib.oracle_exact_sum.argtypes = [u16p, sz, i, i, f64p, f64p]
            lib.oracle_exact_sum.restype = None
            lib.oracle_exact_sum_rows.argtypes = [u16p, sz, sz, i, i, f64p, f64p]
            lib.oracle_exact_sum_rows.restype = None
            lib.oracle_fixed_order_f32.argtypes = [u16p, sz, i, i]
            lib.oracle_fixed_order_f32.restype = ctypes.c_float
            lib.oracle_exact_sum_squares.argtypes = [u16p, sz, i, i, f64p, f64p]
            lib.oracle_exact_sum_squares.restype = None
            lib.oracle_exact_sum_squares_rows.argtypes = [u16p, sz, sz, i, i, f64p, f64p]
            lib.oracle_exact_sum_squares_rows.restype = None
            lib.oracle_fixed_order_sq_f32.argtypes = [u16p, sz, i, i]
            lib.oracle_fixed_order_sq_f32.restype = ctypes.c_float
            lib.oracle_shuffle_tree_sq_f32.argtypes = [u16p, sz, i, i, i, i]
            lib.oracle_shuffle_tree_sq_f32.restype = ctypes.c_float
            lib.oracle_fixed_order_rows_f32.argtypes = [u16p, sz, sz, i, i, i, f32p]
            lib.oracle_fixed_order_rows_f32.restype = None
            lib.oracle_shuffle_tree_f32.argtypes = [u16p, sz, i, i, i, i]
            lib.oracle_shuffle_tree_f32.restype = ctypes.c_float
            lib.oracle_shuffle_tree_rows_f32.argtypes = [u16p, sz, sz, i, i, i, i, i, f32p]
            lib.oracle_shuffle_tree_rows_f32.restype = None
            lib.oracle_blocked_order_f32.argtypes = [u16p, sz, i, i, i]
            lib.oracle_blocked_order_f32.restype = ctypes.c_float
            lib.oracle_blocked_order_rows_f32.argtypes = [u16p, sz, sz, i, i, i, f32p]
            lib.oracle_blocked_order_rows_f32.restype = None
            lib.oracle_mean_var_f32.argtypes = [f32p, f32p, sz, sz, f32p, f32p]
            lib.oracle_mean_var_f32.restype = None
            lib.oracle_gemm_f64.argtypes = [u16p, u16p, sz, sz, sz, i, i, f64p, f64p]
            lib.oracle_gemm_f64.restype = None
            lib.oracle_gemm_splitk_f32.argtypes = [u16p, u16p, sz, sz, sz, i, i, sz, i, f32p]
            lib.oracle_gemm_splitk_f32.restype = None
            lib.oracle_leaves_f32.argtypes = [u16p, sz, i, f32p]
            lib.oracle_leaves_f32.restype = None
            _lib = lib
    return _lib


def _bits(x, dtype: int) -> np.ndarray:
    """The raw patterns of ``x``, C-contiguous: uint16 for F16 / BF16,
    uint32 for F32."""
    a = np.asarray(x)
    if dtype == F32:
        if a.dtype == np.float32:
            a = a.view(np.uint32)
        if a.dtype != np.uint32:
            raise TypeError(f"binary32 oracle inputs are float32 or uint32 patterns, got {a.dtype}")
    else:
        if a.dtype == np.float16:
            a = a.view(np.uint16)
        if a.dtype != np.uint16:
            raise TypeError(f"16-bit oracle inputs are uint16 patterns, got {a.dtype}")
    return np.ascontiguousarray(a)


def _u16p(a):
    return ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def exact_sum(x, dtype: int, threads: int | None = None) -> tuple[float, float]:
    """(exact sum rounded to binary64, exact sum of |x| rounded to binary64)."""
    a = _bits(x, dtype).reshape(-1)
    s, m = ctypes.c_double(), ctypes.c_double()
    _load().oracle_exact_sum(_u16p(a), a.size, dtype, threads or default_threads(),
                             ctypes.byref(s), ctypes.byref(m))
    return s.value, m.value


def exact_sum_squares(x, dtype: int, threads: int | None = None) -> tuple[float, float]:
    """(exact sum of x_i^2 rounded to binary64, the same value)."""
    a = _bits(x, dtype).reshape(-1)
    s, m = ctypes.c_double(), ctypes.c_double()
    _load().oracle_exact_sum_squares(_u16p(a), a.size, dtype, threads or default_threads(),
                                     ctypes.byref(s), ctypes.byref(m))
    return s.value, m.value


def exact_sum_rows(x, dtype: int, threads: int | None = None, squares: bool = False):
    a = _bits(x, dtype)
    rows, cols = a.shape
    s = np.empty(rows, np.float64)
    m = np.empty(rows, np.float64)
    fn = _load().oracle_exact_sum_squares_rows if squares else _load().oracle_exact_sum_rows
    fn(
        _u16p(a), rows, cols, dtype, threads or default_threads(),
        s.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        m.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return s, m


def fixed_order(x, dtype: int, threads: int | None = None) -> np.float32:
    a = _bits(x, dtype).reshape(-1)
    return np.float32(_load().oracle_fixed_order_f32(_u16p(a), a.size, dtype,
                                                     threads or default_threads()))


def fixed_order_sq(x, dtype: int, threads: int | None = None) -> np.float32:
    """Balanced binary32 tree over the leaves x_i^2."""
    a = _bits(x, dtype).reshape(-1)
    return np.float32(_load().oracle_fixed_order_sq_f32(_u16p(a), a.size, dtype,
                                                        threads or default_threads()))


def fixed_order_rows(x, dtype: int, threads: int | None = None,
                     squares: bool = False) -> np.ndarray:
    a = _bits(x, dtype)
    rows, cols = a.shape
    out = np.empty(rows, np.float32)
    _load().oracle_fixed_order_rows_f32(_u16p(a), rows, cols, dtype, 1 if squares else 0,
                                        threads or default_threads(),
                                        out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return out


def shuffle_tree(x, dtype: int, team_threads: int, team_blocks: int,
                 threads: int | None = None) -> np.float32:
    a = _bits(x, dtype).reshape(-1)
    return np.float32(_load().oracle_shuffle_tree_f32(
        _u16p(a), a.size, dtype, team_threads, team_blocks, threads or default_threads()))


def shuffle_tree_sq(x, dtype: int, team_threads: int, team_blocks: int,
                    threads: int | None = None) -> np.float32:
    """The declared SHUFFLE_TREE order over the leaves x_i^2."""
    a = _bits(x, dtype).reshape(-1)
    return np.float32(_load().oracle_shuffle_tree_sq_f32(
        _u16p(a), a.size, dtype, team_threads, team_blocks, threads or default_threads()))


def shuffle_tree_rows(x, dtype: int, team_threads: int, team_blocks: int,
                      threads: int | None = None, squares: bool = False) -> np.ndarray:
    a = _bits(x, dtype)
    rows, cols = a.shape
    out = np.empty(rows, np.float32)
    _load().oracle_shuffle_tree_rows_f32(_u16p(a), rows, cols, dtype, 1 if squares else 0,
                                         team_threads,
                                         team_blocks, threads or default_threads(),
                                         out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return out


def blocked_order(x, dtype: int, run_log2: int, threads: int | None = None) -> np.float32:
    """Runs of 2^run_log2 inputs summed left to right, then the balanced tree
    over the run values (-0.0 pad)."""
    a = _bits(x, dtype).reshape(-1)
    return np.float32(_load().oracle_blocked_order_f32(_u16p(a), a.size, dtype, run_log2,
                                                       threads or default_threads()))


def blocked_order_rows(x, dtype: int, run_log2: int, threads: int | None = None) -> np.ndarray:
    a = _bits(x, dtype)
    rows, cols = a.shape
    out = np.empty(rows, np.float32)
    _load().oracle_blocked_order_rows_f32(_u16p(a), rows, cols, dtype, run_log2,
                                          threads or default_threads(),
                                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return out


def mean_var(s1, s2, cols: int) -> tuple[np.ndarray, np.ndarray]:
    """Per-row mean and variance from the row sums s1 and sums of squares s2
    (binary32, the declared formula of ``oracle_mean_var_f32``)."""
    a = np.ascontiguousarray(s1, np.float32).reshape(-1)
    b = np.ascontiguousarray(s2, np.float32).reshape(-1)
    m = np.empty(a.size, np.float32)
    v = np.empty(a.size, np.float32)
    fp = ctypes.POINTER(ctypes.c_float)
    _load().oracle_mean_var_f32(a.ctypes.data_as(fp), b.ctypes.data_as(fp), a.size, cols,
                                m.ctypes.data_as(fp), v.ctypes.data_as(fp))
    return m, v


def gemm_f64(A, W, dtype: int, threads: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """(A @ W.T as binary64 sums of exact products, the same sum of |products|);
    A is M x K, W is N x K, 16-bit patterns."""
    a, w = _bits(A, dtype), _bits(W, dtype)
    M, K = a.shape
    N = w.shape[0]
    out = np.empty((M, N), np.float64)
    aout = np.empty((M, N), np.float64)
    fp = ctypes.POINTER(ctypes.c_double)
    _load().oracle_gemm_f64(_u16p(a), _u16p(w), M, N, K, dtype, threads or default_threads(),
                            out.ctypes.data_as(fp), aout.ctypes.data_as(fp))
    return out, aout


def gemm_splitk(A, W, dtype: int, splits: int, k_split: int, threads: int | None = None) -> np.ndarray:
    """The declared split-K order over exactly summed, once-rounded partials."""
    a, w = _bits(A, dtype), _bits(W, dtype)
    M, K = a.shape
    N = w.shape[0]
    out = np.empty((M, N), np.float32)
    _load().oracle_gemm_splitk_f32(_u16p(a), _u16p(w), M, N, K, dtype, splits, k_split,
                                   threads or default_threads(),
                                   out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return out


def leaves(x, dtype: int) -> np.ndarray:
    a = _bits(x, dtype).reshape(-1)
    out = np.empty(a.size, np.float32)
    _load().oracle_leaves_f32(_u16p(a), a.size, dtype,
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return out
