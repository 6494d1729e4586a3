"""tcr_reduce_sum_noalloc through the C ABI: the same results as
tcr_reduce_sum, on two calls in a row, checked against the oracle too, and
no device memory taken after the first call on a device.

This file is collected last so that, should it fail, a run stopping at the
first failure has already run every other test.  It builds what it needs
itself and passes alone in a fresh process as well as after the others.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library
from tests import spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)
    lib = tcr.c_api()
    f = lib.tcr_reduce_sum_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, tcr.tcr_mode, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return lib


def _call(fn, x, out, mode, n=None):
    return fn(x.data_ptr(), x.numel() if n is None else n, out.data_ptr(), mode,
              torch.cuda.current_stream().cuda_stream)


def _dev(bits):
    return torch.from_numpy(bits.view(np.float32 if bits.dtype == np.uint32 else np.int16)).cuda()


SIZES = [1, 1000, 65537, (1 << 22) + 5, 1 << 26]


@pytest.mark.parametrize("dtype", [tcr.F16, tcr.BF16, tcr.F32])
@pytest.mark.parametrize("kind", [tcr.FIXED_ORDER, tcr.MMA_CHAIN])
@pytest.mark.parametrize("n", SIZES)
def test_no_alloc_matches_allocating_entry_point_twice(lib, dtype, kind, n):
    bits = synth.generate(n, "uniform_pm1", dtype, seed=n + 1)
    x = _dev(bits)
    mode = tcr.Mode(kind, dtype=dtype)
    ref = torch.full((1,), 5.0, device="cuda")
    assert _call(lib.tcr_reduce_sum, x, ref, mode) == tcr.OK
    outs = [torch.full((1,), 7.0, device="cuda") for _ in range(2)]
    for o in outs:                            # two calls in a row, same stream
        assert _call(lib.tcr_reduce_sum_noalloc, x, o, mode) == tcr.OK
    torch.cuda.synchronize()
    r = ref.cpu().numpy()
    exact, abs_sum = oracle.exact_sum(bits, dtype)
    fixed = oracle.fixed_order(bits, dtype) if kind == tcr.FIXED_ORDER else None
    for o in outs:
        g = o.cpu().numpy()
        # one plan function serves both entry points: the same kernels and
        # work split, so the same bits in every mode
        assert g.tobytes() == r.tobytes()
        if kind == tcr.FIXED_ORDER:
            assert g.tobytes() == np.float32(fixed).tobytes()    # the declared tree
        else:
            assert abs(float(g[0]) - exact) <= spec.mma_tolerance(abs_sum)


@pytest.mark.parametrize("R,block", [(1, 32), (5, 1024), (8, 128)])
def test_no_alloc_chain_lengths_and_blocks(lib, R, block):
    n = (1 << 24) + 3
    bits = synth.generate(n, "normal", tcr.F16, seed=R)
    x = _dev(bits)
    mode = tcr.Mode(tcr.MMA_CHAIN, R=R, block_threads=block)
    ref, o = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    assert _call(lib.tcr_reduce_sum, x, ref, mode) == tcr.OK
    assert _call(lib.tcr_reduce_sum_noalloc, x, o, mode) == tcr.OK
    torch.cuda.synchronize()
    assert o.cpu().numpy().tobytes() == ref.cpu().numpy().tobytes()
    exact, abs_sum = oracle.exact_sum(bits, tcr.F16)
    assert abs(float(o.item()) - exact) <= spec.mma_tolerance(abs_sum)


def test_no_alloc_misaligned_base(lib):
    bits = synth.generate((1 << 22) + 9, "normal", tcr.F16, seed=77)
    x = _dev(bits)[1:]
    for kind in (tcr.FIXED_ORDER, tcr.MMA_CHAIN):
        ref, o = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
        assert _call(lib.tcr_reduce_sum, x, ref, tcr.Mode(kind)) == tcr.OK
        assert _call(lib.tcr_reduce_sum_noalloc, x, o, tcr.Mode(kind)) == tcr.OK
        torch.cuda.synchronize()
        assert o.cpu().numpy().tobytes() == ref.cpu().numpy().tobytes()
    fixed = torch.zeros(1, device="cuda")
    assert _call(lib.tcr_reduce_sum_noalloc, x, fixed, tcr.Mode(tcr.FIXED_ORDER)) == tcr.OK
    torch.cuda.synchronize()
    assert fixed.cpu().numpy().tobytes() == np.float32(oracle.fixed_order(bits[1:], tcr.F16)).tobytes()


def test_no_alloc_after_a_larger_call_and_limits(lib):
    big = _dev(synth.generate(1 << 24, "normal", tcr.F16, seed=3))
    bits = synth.generate(300_001, "normal", tcr.F16, seed=4)
    small = _dev(bits)
    o = torch.zeros(1, device="cuda")
    mode = tcr.Mode(tcr.FIXED_ORDER)
    assert _call(lib.tcr_reduce_sum_noalloc, big, o, mode) == tcr.OK
    assert _call(lib.tcr_reduce_sum_noalloc, small, o, mode) == tcr.OK
    torch.cuda.synchronize()
    assert o.cpu().numpy()[0] == oracle.fixed_order(bits, tcr.F16)
    # beyond the array: rejected before any GPU work
    too_many = 65536 * (1 << 16) + 1
    assert _call(lib.tcr_reduce_sum_noalloc, small, o, mode, n=too_many) == tcr.ERR_UNSUPPORTED


def test_no_alloc_status_codes_follow_tcr_reduce_sum(lib):
    x = torch.zeros(100, dtype=torch.float16, device="cuda")
    o = torch.zeros(1, device="cuda")
    f = lib.tcr_reduce_sum_noalloc
    # well-formed requests this entry point does not serve
    for m in (tcr.Mode(tcr.SHUFFLE_TREE), tcr.Mode(tcr.MMA_CHAIN_TMEM),
              tcr.Mode(tcr.FIXED_ORDER, run_log2=4)):
        assert _call(lib.tcr_reduce_sum, x, o, m) == tcr.OK
        assert _call(f, x, o, m) == tcr.ERR_UNSUPPORTED
    # malformed ones: the same answer as tcr_reduce_sum
    bad = [tcr.Mode(tcr.MMA_CHAIN, run_log2=3), tcr.Mode(tcr.MMA_CHAIN, R=9),
           tcr.Mode(tcr.FIXED_ORDER, block_threads=48), tcr.Mode(7), tcr.Mode(tcr.FIXED_ORDER, dtype=5)]
    for m in bad:
        assert _call(lib.tcr_reduce_sum, x, o, m) == tcr.ERR_INVALID_ARG
        assert _call(f, x, o, m) == tcr.ERR_INVALID_ARG
    odd = x.view(torch.uint8)[1:].data_ptr()      # not aligned to its element
    stream = torch.cuda.current_stream().cuda_stream
    assert f(odd, 10, o.data_ptr(), tcr.Mode(tcr.FIXED_ORDER), stream) == tcr.ERR_INVALID_ARG
    assert f(x.data_ptr(), 10, None, tcr.Mode(tcr.FIXED_ORDER), stream) == tcr.ERR_INVALID_ARG


def test_no_alloc_works_where_allocation_fails(lib):
    # TCR_FAULT_INJECT=alloc makes the stream-ordered pool path of
    # tcr_reduce_sum fail; the entry point without allocation is untouched
    bits = synth.generate((1 << 22) + 5, "normal", tcr.F16, seed=21)
    x = _dev(bits)
    ref, o = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    for kind in (tcr.FIXED_ORDER, tcr.MMA_CHAIN):
        assert _call(lib.tcr_reduce_sum, x, ref, tcr.Mode(kind)) == tcr.OK
        os.environ["TCR_FAULT_INJECT"] = "alloc"
        try:
            assert _call(lib.tcr_reduce_sum, x, o, tcr.Mode(kind)) == tcr.ERR_CUDA
            assert _call(lib.tcr_reduce_sum_noalloc, x, o, tcr.Mode(kind)) == tcr.OK
        finally:
            del os.environ["TCR_FAULT_INJECT"]
        torch.cuda.synchronize()
        assert o.cpu().numpy().tobytes() == ref.cpu().numpy().tobytes()


def test_no_alloc_takes_no_device_memory_after_its_first_call(lib):
    # every kernel variant the entry point can launch (input types,
    # alignments, chain lengths, with and without a combine) after one
    # first call: the device's free memory does not move
    inputs = []
    for dt in (tcr.F16, tcr.BF16, tcr.F32):
        t = _dev(synth.generate((1 << 21) + 3, "normal", dt, seed=dt))
        inputs += [t, t[1:], t[:1000]]
    o = torch.zeros(1, device="cuda")
    modes = [tcr.Mode(tcr.FIXED_ORDER, dtype=dt) for dt in (tcr.F16, tcr.BF16, tcr.F32)]
    modes += [tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=dt) for dt in (tcr.F16, tcr.BF16, tcr.F32)
              for R in range(1, 9)]
    assert _call(lib.tcr_reduce_sum_noalloc, inputs[0], o, modes[0]) == tcr.OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for m in modes:
        for t in inputs:
            if (t.dtype == torch.float32) != (m.dtype == tcr.F32):
                continue
            assert _call(lib.tcr_reduce_sum_noalloc, t, o, m) == tcr.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
