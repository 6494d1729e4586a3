"""Failure detection on the GPU without a GPU fault.

Every mbarrier wait of the tcgen05 kernels (the MMA_CHAIN_TMEM reductions
and the split-K GEMM) gives up after about a second.
A host-side injection (TCR_FAULT_INJECT=stall) makes the MMA issuer
withhold its first chain, so the epilogue's wait runs out its limit: the
kernel must raise the device fault word, drain its copies and MMAs, free
its tensor memory and return NaN -- and the context must stay usable.
"""
import time

import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def test_wait_limit_reports_nan_and_fault_word_then_recovers(monkeypatch):
    n = (1 << 22) + 77
    bits = synth.generate(n, "uniform01", tcr.F16, seed=21)
    x = torch.from_numpy(bits.view(np.int16)).cuda()
    rows, cols = 1000, 4096
    rbits = synth.generate(rows * cols, "uniform01", tcr.F16, seed=22).reshape(rows, cols)
    xr = torch.from_numpy(rbits.reshape(-1).view(np.int16)).cuda().view(rows, cols)
    mode = tcr.Mode(tcr.MMA_CHAIN_TMEM)
    torch.cuda.synchronize()
    tcr.tcr_device_faults(clear=True)

    monkeypatch.setenv("TCR_FAULT_INJECT", "stall")
    t0 = time.time()
    s = tcr.tcr_reduce_sum(x, mode)
    r = tcr.tcr_reduce_rows(xr, mode)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    monkeypatch.delenv("TCR_FAULT_INJECT")
    assert np.isnan(s.item())
    assert np.isnan(r.cpu().numpy()).any()
    assert tcr.tcr_device_faults(clear=True) & tcr.FAULT_PIPELINE_WAIT
    assert elapsed < 20          # each stalled launch ends after about a second

    # the context still works, the word stays clear, results are right again
    s = tcr.tcr_reduce_sum(x, mode).item()
    exact, abs_sum = oracle.exact_sum(bits, tcr.F16)
    assert abs(s - exact) <= 2.0 ** -20 * abs_sum + 1e-6
    got = tcr.tcr_reduce_rows(xr, mode).cpu().numpy().astype(np.float64)
    es, ea = oracle.exact_sum_rows(rbits, tcr.F16)
    assert np.all(np.abs(got - es) <= 2.0 ** -20 * ea + 1e-6)
    torch.cuda.synchronize()
    assert tcr.tcr_device_faults() == 0


@pytest.mark.parametrize("kernel", ["pair", "one_sm"])
def test_gemm_wait_limit_reports_nan_and_fault_word_then_recovers(monkeypatch, kernel):
    if kernel == "one_sm":
        monkeypatch.setenv("TCR_GEMM_ONE_SM", "1")
    M, N, K = 512, 768, 1024
    ab = synth.generate(M * K, "normal", tcr.BF16, seed=23).reshape(M, K)
    wb = synth.generate(N * K, "normal", tcr.BF16, seed=24).reshape(N, K)
    A = torch.from_numpy(ab.view(np.int16)).cuda().view(torch.bfloat16)
    W = torch.from_numpy(wb.view(np.int16)).cuda().view(torch.bfloat16)
    torch.cuda.synchronize()
    tcr.tcr_device_faults(clear=True)
    monkeypatch.setenv("TCR_FAULT_INJECT", "stall")
    t0 = time.time()
    C = tcr.tcr_gemm_splitk(A, W, splits=2)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    monkeypatch.delenv("TCR_FAULT_INJECT")
    assert np.isnan(C.cpu().numpy()).any()
    assert tcr.tcr_device_faults(clear=True) & tcr.FAULT_PIPELINE_WAIT
    assert elapsed < 20
    # healthy again: within the bound of the oracle's binary64 product
    C = tcr.tcr_gemm_splitk(A, W, splits=2).cpu().numpy().astype(np.float64)
    c64, a64 = oracle.gemm_f64(ab, wb, tcr.BF16)
    d = tcr.tcr_gemm_descriptor(M, N, K, 2, tcr.BF16)
    bound = (2.0 ** -22 * d["k_split"] / 16 + 2.0 ** -24) * a64 + 1e-30
    assert np.all(np.abs(C - c64) <= bound)
    torch.cuda.synchronize()
    assert tcr.tcr_device_faults() == 0
