"""tcr_reduce_sum_noalloc through the C ABI: the same results as
tcr_reduce_sum, on two calls in a row, without any device allocation.

This file is collected last so that, should it fail, a run stopping at the
first failure has already run every other test.  It builds what it needs
itself and passes alone in a fresh process as well as after the others.
"""
import ctypes

import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library

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


def _call(fn, x, out, mode):
    return fn(x.data_ptr(), x.numel(), out.data_ptr(), mode,
              torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("kind", [tcr.FIXED_ORDER, tcr.MMA_CHAIN])
@pytest.mark.parametrize("n", [1, 1000, 65537, (1 << 22) + 5, 1 << 26])
def test_no_alloc_matches_allocating_entry_point_twice(lib, kind, n):
    bits = synth.generate(n, "uniform_pm1", tcr.F16, seed=n + 1)
    x = torch.from_numpy(bits.view(np.int16)).cuda()
    mode = tcr.Mode(kind)
    ref = torch.full((1,), 5.0, device="cuda")
    assert _call(lib.tcr_reduce_sum, x, ref, mode) == tcr.OK
    outs = [torch.full((1,), 7.0, device="cuda") for _ in range(2)]
    for o in outs:                            # two calls in a row, same stream
        assert _call(lib.tcr_reduce_sum_noalloc, x, o, mode) == tcr.OK
    torch.cuda.synchronize()
    r = ref.cpu().numpy()
    _, abs_sum = oracle.exact_sum(bits, tcr.F16)
    tol = 2.0 ** -20 * abs_sum + 1e-6
    for o in outs:
        g = o.cpu().numpy()
        if kind == tcr.FIXED_ORDER:
            assert g.tobytes() == r.tobytes()          # the fixed order is bit-exact
        else:
            assert abs(float(g[0]) - float(r[0])) <= tol


def test_no_alloc_after_a_larger_call_and_limits(lib):
    big = torch.from_numpy(synth.generate(1 << 24, "normal", tcr.F16, seed=3).view(np.int16)).cuda()
    bits = synth.generate(300_001, "normal", tcr.F16, seed=4)
    small = torch.from_numpy(bits.view(np.int16)).cuda()
    o = torch.zeros(1, device="cuda")
    mode = tcr.Mode(tcr.FIXED_ORDER)
    assert _call(lib.tcr_reduce_sum_noalloc, big, o, mode) == tcr.OK
    assert _call(lib.tcr_reduce_sum_noalloc, small, o, mode) == tcr.OK
    torch.cuda.synchronize()
    assert o.cpu().numpy()[0] == oracle.fixed_order(bits, tcr.F16)
    # beyond the array: rejected before any GPU work
    too_many = 65536 * (1 << 16) + 1
    st = lib.tcr_reduce_sum_noalloc(small.data_ptr(), too_many, o.data_ptr(), mode, None)
    assert st == tcr.ERR_UNSUPPORTED
    st = lib.tcr_reduce_sum_noalloc(small.data_ptr(), 10, o.data_ptr(), tcr.Mode(tcr.SHUFFLE_TREE), None)
    assert st == tcr.ERR_UNSUPPORTED


@pytest.mark.parametrize("kind", [tcr.FIXED_ORDER, tcr.MMA_CHAIN])
@pytest.mark.parametrize("n", [3, 4097, (1 << 22) + 5])
def test_no_alloc_binary32(lib, kind, n):
    bits = synth.generate(n, "normal", tcr.F32, seed=n)
    x = torch.from_numpy(bits.view(np.float32)).cuda()
    mode = tcr.Mode(kind, dtype=tcr.F32)
    ref = torch.full((1,), 5.0, device="cuda")
    assert _call(lib.tcr_reduce_sum, x, ref, mode) == tcr.OK
    o = torch.full((1,), 7.0, device="cuda")
    assert _call(lib.tcr_reduce_sum_noalloc, x, o, mode) == tcr.OK
    torch.cuda.synchronize()
    # the same kernels and work split as the allocating call: the same bits
    assert o.cpu().numpy().tobytes() == ref.cpu().numpy().tobytes()
    if kind == tcr.FIXED_ORDER:
        assert o.cpu().numpy()[0] == oracle.fixed_order(bits, tcr.F32)


def test_no_alloc_refuses_the_blocked_order(lib):
    x = torch.zeros(100, dtype=torch.float16, device="cuda")
    o = torch.zeros(1, device="cuda")
    m = tcr.Mode(tcr.FIXED_ORDER, run_log2=4)
    assert lib.tcr_reduce_sum_noalloc(x.data_ptr(), 100, o.data_ptr(), m, None) == tcr.ERR_UNSUPPORTED
