"""tcr: tensor-core and fixed-order sum reduction on one GB300 GPU.

A thin ctypes binding of ``libtcr.so`` (``include/tcr.h``), with the C
names.  It only marshals arguments: every step of every reduction runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.

    import torch
    import arithmetic_reduction_tensor_gb300 as tcr
    x = torch.randn(1 << 20, device="cuda", dtype=torch.float16)
    s = tcr.tcr_reduce_sum(x, tcr.Mode(tcr.FIXED_ORDER))        # 1-element fp32
    r = tcr.tcr_reduce_rows(x.view(1024, 1024), tcr.Mode(tcr.MMA_CHAIN, R=4))

The library must have been built (``python -m arithmetic_reduction_tensor_gb300.build``
or ``__graft_entry__.build()``); without it every call raises -- there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

__all__ = [
    "MMA_CHAIN", "SHUFFLE_TREE", "FIXED_ORDER", "MMA_CHAIN_TMEM", "F16", "BF16", "F32",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA",
    "ORDER_TENSOR_CORE", "ORDER_GRID_STRIDE", "ORDER_BALANCED_TREE", "ORDER_BLOCKED_TREE",
    "tcr_mode", "tcr_order_desc", "Mode", "TcrError", "c_api",
    "tcr_reduce_sum", "tcr_reduce_rows", "tcr_reduce_sum_squares", "tcr_reduce_rows_sum_squares",
    "tcr_reduce_rows_moments", "tcr_reduce_rows_mean_var",
    "tcr_order_descriptor", "tcr_order_equivalent", "tcr_status_string", "tcr_device_faults",
    "FAULT_PIPELINE_WAIT", "tcr_gemm_desc", "tcr_gemm_descriptor", "tcr_gemm_splitk",
    "tcr_reduce_sum_noalloc", "tcr_read_probe",
]

MMA_CHAIN, SHUFFLE_TREE, FIXED_ORDER, MMA_CHAIN_TMEM = 0, 1, 2, 3
F16, BF16, F32 = 0, 1, 2
DTYPE_NAMES = {F16: "f16", BF16: "bf16", F32: "f32"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3
ORDER_TENSOR_CORE, ORDER_GRID_STRIDE, ORDER_BALANCED_TREE, ORDER_BLOCKED_TREE = 0, 1, 2, 3

KIND_NAMES = {MMA_CHAIN: "MMA_CHAIN", SHUFFLE_TREE: "SHUFFLE_TREE", FIXED_ORDER: "FIXED_ORDER",
              MMA_CHAIN_TMEM: "MMA_CHAIN_TMEM"}


class tcr_mode(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("R", ctypes.c_int),
                ("block_threads", ctypes.c_int), ("dtype", ctypes.c_int),
                ("run_log2", ctypes.c_int)]

    def __repr__(self):
        return (f"Mode({KIND_NAMES.get(self.kind, self.kind)}, R={self.R}, "
                f"block_threads={self.block_threads}, "
                f"dtype={DTYPE_NAMES.get(self.dtype, self.dtype)}, run_log2={self.run_log2})")


class tcr_order_desc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("order", ctypes.c_int),
                ("segment_len", ctypes.c_size_t), ("segments", ctypes.c_size_t),
                ("vector_len", ctypes.c_int), ("team_threads", ctypes.c_int),
                ("team_blocks", ctypes.c_int), ("chain_R", ctypes.c_int),
                ("pad_negative_zero", ctypes.c_int), ("launch_grid", ctypes.c_int),
                ("launch_block", ctypes.c_int), ("chunk_log2", ctypes.c_int),
                ("partials", ctypes.c_size_t), ("launches", ctypes.c_int),
                ("dtype", ctypes.c_int), ("run_log2", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class tcr_gemm_desc(ctypes.Structure):
    _fields_ = [("M", ctypes.c_size_t), ("N", ctypes.c_size_t), ("K", ctypes.c_size_t),
                ("dtype", ctypes.c_int), ("splits", ctypes.c_int), ("k_split", ctypes.c_size_t),
                ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("combine_order", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
                ("launch_grid", ctypes.c_int), ("launch_block", ctypes.c_int),
                ("launches", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def Mode(kind: int, R: int = 0, block_threads: int = 0, dtype: int = F16,
         run_log2: int = 0) -> tcr_mode:
    """A ``tcr_mode`` (R is used by MMA_CHAIN only, 0 meaning the default;
    run_log2 by FIXED_ORDER only: runs of 2^run_log2 inputs added left to
    right, then the balanced tree)."""
    return tcr_mode(kind, R, block_threads, dtype, run_log2)


class TcrError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tcr_status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def c_api() -> ctypes.CDLL:
    """The loaded ``libtcr.so`` with the C signatures of ``include/tcr.h``."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libtcr is not built ({LIB_PATH} missing); run "
                    "`python -m arithmetic_reduction_tensor_gb300.build` -- there is no fallback")
            lib = ctypes.CDLL(LIB_PATH)
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            lib.tcr_reduce_sum.argtypes = [vp, sz, vp, tcr_mode, vp]
            lib.tcr_reduce_sum.restype = ctypes.c_int
            lib.tcr_reduce_rows.argtypes = [vp, sz, sz, vp, tcr_mode, vp]
            lib.tcr_reduce_rows.restype = ctypes.c_int
            lib.tcr_reduce_sum_squares.argtypes = [vp, sz, vp, tcr_mode, vp]
            lib.tcr_reduce_sum_squares.restype = ctypes.c_int
            lib.tcr_reduce_rows_sum_squares.argtypes = [vp, sz, sz, vp, tcr_mode, vp]
            lib.tcr_reduce_rows_sum_squares.restype = ctypes.c_int
            lib.tcr_reduce_rows_moments.argtypes = [vp, sz, sz, vp, vp, tcr_mode, vp]
            lib.tcr_reduce_rows_moments.restype = ctypes.c_int
            lib.tcr_reduce_rows_mean_var.argtypes = [vp, sz, sz, vp, vp, tcr_mode, vp]
            lib.tcr_reduce_rows_mean_var.restype = ctypes.c_int
            lib.tcr_order_descriptor.argtypes = [sz, sz, sz, tcr_mode, ctypes.POINTER(tcr_order_desc)]
            lib.tcr_order_descriptor.restype = ctypes.c_int
            lib.tcr_order_equivalent.argtypes = [ctypes.POINTER(tcr_order_desc),
                                                 ctypes.POINTER(tcr_order_desc),
                                                 ctypes.POINTER(ctypes.c_int)]
            lib.tcr_order_equivalent.restype = ctypes.c_int
            lib.tcr_gemm_descriptor.argtypes = [sz, sz, sz, ctypes.c_int, ctypes.c_int,
                                                ctypes.POINTER(tcr_gemm_desc)]
            lib.tcr_gemm_descriptor.restype = ctypes.c_int
            lib.tcr_gemm_splitk.argtypes = [vp, vp, vp, sz, sz, sz, ctypes.c_int, ctypes.c_int, vp]
            lib.tcr_gemm_splitk.restype = ctypes.c_int
            lib.tcr_device_faults.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]
            lib.tcr_device_faults.restype = ctypes.c_int
            lib.tcr_reduce_sum_noalloc.argtypes = [vp, sz, vp, tcr_mode, vp]
            lib.tcr_reduce_sum_noalloc.restype = ctypes.c_int
            lib.tcr_read_probe.argtypes = [vp, sz, vp, ctypes.c_int, ctypes.c_int, vp]
            lib.tcr_read_probe.restype = ctypes.c_int
            lib.tcr_status_string.argtypes = [ctypes.c_int]
            lib.tcr_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def tcr_status_string(status: int) -> str:
    return c_api().tcr_status_string(status).decode()


FAULT_PIPELINE_WAIT = 1


def tcr_device_faults(clear: bool = False) -> int:
    """The current device's fault word (``tcr_device_faults``); synchronous."""
    v = ctypes.c_uint(0)
    st = c_api().tcr_device_faults(ctypes.byref(v), 1 if clear else 0)
    if st != OK:
        raise TcrError(st, "tcr_device_faults")
    return v.value


# ------------------------------------------------------------------ torch

def _dtype_code(t, mode: tcr_mode) -> int:
    import torch
    if t.dtype == torch.float16:
        code = F16
    elif t.dtype == torch.bfloat16:
        code = BF16
    elif t.dtype == torch.float32:
        code = F32
    elif t.dtype in (torch.int16, torch.uint16):
        if mode.dtype not in (F16, BF16):
            raise ValueError("16-bit patterns need mode.dtype F16 or BF16")
        return mode.dtype          # raw 16-bit patterns: the mode says what they are
    elif t.dtype in (torch.int32, torch.uint32):
        if mode.dtype != F32:
            raise ValueError("32-bit patterns need mode.dtype F32")
        return F32
    else:
        raise TypeError("inputs must be float16, bfloat16, float32 or their raw patterns, "
                        f"got {t.dtype}")
    if mode.dtype != code:
        raise ValueError(f"mode.dtype {mode.dtype} does not match tensor dtype {t.dtype}")
    return code


def _stream_handle(device, stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_out(out, device, count: int):
    import torch
    if out is None:
        return torch.empty(max(count, 1), dtype=torch.float32, device=device)
    if out.dtype != torch.float32 or out.device != device or not out.is_contiguous() or out.numel() < count:
        raise ValueError("out must be a contiguous float32 tensor on the input's device "
                         f"with at least {count} elements")
    return out


def _sum_call(name, x, mode, out, stream):
    import torch
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    m = tcr_mode(mode.kind, mode.R, mode.block_threads, _dtype_code(x, mode), mode.run_log2)
    out = _check_out(out, x.device, 1)
    with torch.cuda.device(x.device):
        st = getattr(c_api(), name)(x.data_ptr() if x.numel() else None, x.numel(),
                                    out.data_ptr(), m, _stream_handle(x.device, stream))
    if st != OK:
        raise TcrError(st, name)
    return out


def _rows_call(name, x, mode, out, stream):
    import torch
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be a contiguous 2-D CUDA tensor")
    rows, cols = x.shape
    m = tcr_mode(mode.kind, mode.R, mode.block_threads, _dtype_code(x, mode), mode.run_log2)
    out = _check_out(out, x.device, rows)
    with torch.cuda.device(x.device):
        st = getattr(c_api(), name)(x.data_ptr() if x.numel() else None, rows, cols,
                                    out.data_ptr(), m, _stream_handle(x.device, stream))
    if st != OK:
        raise TcrError(st, name)
    return out[:rows] if rows else out[:0]


def tcr_reduce_sum(x, mode: tcr_mode, out=None, stream=None):
    """out[0] = sum of the contiguous CUDA tensor ``x`` (``tcr_reduce_sum``)."""
    return _sum_call("tcr_reduce_sum", x, mode, out, stream)


def tcr_reduce_rows(x, mode: tcr_mode, out=None, stream=None):
    """out[r] = sum of row r of the contiguous 2-D CUDA tensor ``x`` (``tcr_reduce_rows``)."""
    return _rows_call("tcr_reduce_rows", x, mode, out, stream)


def tcr_reduce_sum_noalloc(x, mode: tcr_mode, out=None, stream=None):
    """``tcr_reduce_sum`` without device allocation (``tcr_reduce_sum_noalloc``:
    FIXED_ORDER and MMA_CHAIN; the partials live in the library's fixed
    device array).  A new ``out`` is allocated here by torch when none is
    given: callers that must not allocate pass their own."""
    return _sum_call("tcr_reduce_sum_noalloc", x, mode, out, stream)


def tcr_read_probe(x, ctas_per_sm: int = 0, block_threads: int = 0, out=None, stream=None):
    """Stream the bytes of the contiguous CUDA tensor ``x`` in and XOR their
    32-bit words into ``out`` (``tcr_read_probe``, a measurement aid: the
    read ceiling of the GPU).  Returns ``out`` (an int32 tensor of one)."""
    import torch
    if not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA tensor")
    nbytes = x.numel() * x.element_size()
    if out is None:
        out = torch.empty(1, dtype=torch.int32, device=x.device)
    with torch.cuda.device(x.device):
        st = c_api().tcr_read_probe(x.data_ptr() if nbytes else None, nbytes, out.data_ptr(),
                                    ctas_per_sm, block_threads, _stream_handle(x.device, stream))
    if st != OK:
        raise TcrError(st, "tcr_read_probe")
    return out


def tcr_reduce_sum_squares(x, mode: tcr_mode, out=None, stream=None):
    """out[0] = sum of x_i^2 (``tcr_reduce_sum_squares``)."""
    return _sum_call("tcr_reduce_sum_squares", x, mode, out, stream)


def tcr_reduce_rows_sum_squares(x, mode: tcr_mode, out=None, stream=None):
    """out[r] = sum of the squares of row r (``tcr_reduce_rows_sum_squares``)."""
    return _rows_call("tcr_reduce_rows_sum_squares", x, mode, out, stream)


def _rows_pair_call(name, x, mode, out_a, out_b, stream):
    import torch
    if not x.is_cuda or not x.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be a contiguous 2-D CUDA tensor")
    rows, cols = x.shape
    m = tcr_mode(mode.kind, mode.R, mode.block_threads, _dtype_code(x, mode), mode.run_log2)
    out_a = _check_out(out_a, x.device, rows)
    out_b = _check_out(out_b, x.device, rows)
    with torch.cuda.device(x.device):
        st = getattr(c_api(), name)(x.data_ptr() if x.numel() else None, rows, cols,
                                    out_a.data_ptr(), out_b.data_ptr(), m,
                                    _stream_handle(x.device, stream))
    if st != OK:
        raise TcrError(st, name)
    return (out_a[:rows], out_b[:rows]) if rows else (out_a[:0], out_b[:0])


def tcr_reduce_rows_moments(x, mode: tcr_mode, sums=None, sums_of_squares=None, stream=None):
    """(sums, sums of squares) of the rows of ``x`` in one pass
    (``tcr_reduce_rows_moments``)."""
    return _rows_pair_call("tcr_reduce_rows_moments", x, mode, sums, sums_of_squares, stream)


def tcr_reduce_rows_mean_var(x, mode: tcr_mode, mean=None, var=None, stream=None):
    """(mean, population variance) of the rows of ``x`` in one pass
    (``tcr_reduce_rows_mean_var``)."""
    return _rows_pair_call("tcr_reduce_rows_mean_var", x, mode, mean, var, stream)


def _descriptor(n, rows, cols, mode) -> tcr_order_desc:
    d = tcr_order_desc()
    st = c_api().tcr_order_descriptor(n, rows, cols, mode if mode is not None else Mode(FIXED_ORDER),
                                      ctypes.byref(d))
    if st != OK:
        raise TcrError(st, "tcr_order_descriptor")
    return d


def tcr_order_descriptor(n: int = 0, rows: int = 0, cols: int = 0,
                         mode: tcr_mode | None = None) -> dict:
    """The declared order and launch plan of a call (``tcr_order_descriptor``)."""
    return _descriptor(n, rows, cols, mode).as_dict()


def tcr_order_equivalent(call_a: dict, call_b: dict) -> bool:
    """Whether two calls, each given as the keyword arguments of
    ``tcr_order_descriptor`` (n / rows / cols / mode), are in one
    bit-equivalence class (``tcr_order_equivalent``)."""
    a = _descriptor(call_a.get("n", 0), call_a.get("rows", 0), call_a.get("cols", 0), call_a.get("mode"))
    b = _descriptor(call_b.get("n", 0), call_b.get("rows", 0), call_b.get("cols", 0), call_b.get("mode"))
    eq = ctypes.c_int(0)
    st = c_api().tcr_order_equivalent(ctypes.byref(a), ctypes.byref(b), ctypes.byref(eq))
    if st != OK:
        raise TcrError(st, "tcr_order_equivalent")
    return bool(eq.value)


# ------------------------------------------------------------------ GEMM

def tcr_gemm_descriptor(M: int, N: int, K: int, splits: int = 0, dtype: int = F16) -> dict:
    """The K partition and launch plan of a split-K GEMM (``tcr_gemm_descriptor``)."""
    d = tcr_gemm_desc()
    st = c_api().tcr_gemm_descriptor(M, N, K, splits, dtype, ctypes.byref(d))
    if st != OK:
        raise TcrError(st, "tcr_gemm_descriptor")
    return d.as_dict()


def tcr_gemm_splitk(A, W, splits: int = 0, out=None, stream=None, dtype: int | None = None):
    """C = A @ W.T in binary32 with the declared split-K combine
    (``tcr_gemm_splitk``); A is M x K, W is N x K, both contiguous CUDA
    tensors of float16 or bfloat16 (or raw 16-bit patterns with ``dtype``)."""
    import torch
    if not (A.is_cuda and W.is_cuda and A.is_contiguous() and W.is_contiguous()
            and A.dim() == 2 and W.dim() == 2):
        raise ValueError("A and W must be contiguous 2-D CUDA tensors")
    if A.shape[1] != W.shape[1]:
        raise ValueError(f"inner dimensions differ: {tuple(A.shape)} vs {tuple(W.shape)}")
    if A.dtype != W.dtype:
        raise ValueError("A and W must have the same dtype")
    if dtype is None:
        if A.dtype == torch.float16:
            dtype = F16
        elif A.dtype == torch.bfloat16:
            dtype = BF16
        else:
            raise TypeError(f"A must be float16 or bfloat16 (or pass dtype), got {A.dtype}")
    M, K = A.shape
    N = W.shape[0]
    if out is None:
        out = torch.empty(M, N, dtype=torch.float32, device=A.device)
    if out.dtype != torch.float32 or not out.is_contiguous() or out.numel() < M * N:
        raise ValueError("out must be a contiguous float32 tensor with M * N elements")
    with torch.cuda.device(A.device):
        st = c_api().tcr_gemm_splitk(A.data_ptr() if A.numel() else None,
                                     W.data_ptr() if W.numel() else None, out.data_ptr(),
                                     M, N, K, splits, dtype, _stream_handle(A.device, stream))
    if st != OK:
        raise TcrError(st, "tcr_gemm_splitk")
    return out
