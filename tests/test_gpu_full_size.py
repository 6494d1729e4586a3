"""The later paths at full size: the blocked order on the 2^30-input sum, the
fused row moments on the 65536 x 4096 rows, binary32 at 2^29, the 2^30 sum
seen as short rows (packed kernels) and from a misaligned base, and large
split-K GEMMs on sampled elements (the oracle computes those one by one)."""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library
from tests import spec
from tests.test_oracle import exact_partials_operands

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F16, BF16, F32 = tcr.F16, tcr.BF16, tcr.F32


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def same_bits(a, b):
    a = np.asarray(a, np.float32).reshape(-1)
    b = np.asarray(b, np.float32).reshape(-1)
    nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan]) and \
        np.array_equal(np.isnan(a), np.isnan(b))


@pytest.fixture(scope="module")
def sum_2p30():
    x = synth.generate(1 << 30, "uniform_pm1", F16, seed=4)
    return x, torch.from_numpy(x.view(np.int16)).cuda()


@pytest.mark.parametrize("c", [3, 4, 10])
def test_blocked_order_on_the_2p30_sum(sum_2p30, c):
    x, t = sum_2p30
    got = np.float32(tcr.tcr_reduce_sum(t, tcr.Mode(tcr.FIXED_ORDER, run_log2=c)).cpu().numpy()[0])
    assert same_bits(got, oracle.blocked_order(x, F16, c))


@pytest.mark.parametrize("cols", [64, 100])
def test_the_2p30_sum_as_short_rows(sum_2p30, cols):
    # every row of the full input through the packed kernels (rows of 100 are
    # not 16-byte aligned); the oracle's row emulation runs on all of them
    x, t = sum_2p30
    rows = (1 << 30) // cols
    xr = x[:rows * cols].reshape(rows, cols)
    tr = t[:rows * cols].view(rows, cols)
    got = tcr.tcr_reduce_rows(tr, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()
    assert same_bits(got, oracle.fixed_order_rows(xr, F16))
    got = tcr.tcr_reduce_rows(tr, tcr.Mode(tcr.SHUFFLE_TREE)).cpu().numpy()
    assert same_bits(got, oracle.shuffle_tree_rows(xr, F16, *spec.shuffle_team(cols)))
    e, a = oracle.exact_sum_rows(xr, F16)
    got = tcr.tcr_reduce_rows(tr, tcr.Mode(tcr.MMA_CHAIN)).cpu().numpy()
    assert np.all(np.abs(got - e) <= spec.mma_tolerance(a))


def test_the_2p30_sum_from_a_misaligned_base(sum_2p30):
    x, t = sum_2p30
    xs, ts = x[1:], t[1:]
    assert same_bits(tcr.tcr_reduce_sum(ts, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy(),
                     oracle.fixed_order(xs, F16))
    assert same_bits(tcr.tcr_reduce_sum(ts, tcr.Mode(tcr.SHUFFLE_TREE)).cpu().numpy(),
                     oracle.shuffle_tree(xs, F16, *spec.shuffle_team(xs.size)))


def test_moments_on_the_65536x4096_rows():
    rows, cols = 65536, 4096
    x = synth.generate(rows * cols, "normal", F16, seed=2).reshape(rows, cols)
    t = torch.from_numpy(x.reshape(-1).view(np.int16)).cuda().view(rows, cols)
    f1 = oracle.fixed_order_rows(x, F16)
    f2 = oracle.fixed_order_rows(x, F16, squares=True)
    s1, s2 = tcr.tcr_reduce_rows_moments(t, tcr.Mode(tcr.FIXED_ORDER))
    assert same_bits(s1.cpu().numpy(), f1) and same_bits(s2.cpu().numpy(), f2)
    m, v = tcr.tcr_reduce_rows_mean_var(t, tcr.Mode(tcr.SHUFFLE_TREE))
    bt, g = spec.shuffle_team(cols)
    om, ov = oracle.mean_var(oracle.shuffle_tree_rows(x, F16, bt, g),
                             oracle.shuffle_tree_rows(x, F16, bt, g, squares=True), cols)
    assert same_bits(m.cpu().numpy(), om) and same_bits(v.cpu().numpy(), ov)


def test_binary32_sum_2p29_every_mode():
    n = 1 << 29
    x = synth.generate(n, "uniform_pm1", F32, seed=4)
    t = torch.from_numpy(x.view(np.float32)).cuda()
    m = tcr.Mode(tcr.FIXED_ORDER, dtype=F32)
    assert same_bits(tcr.tcr_reduce_sum(t, m).cpu().numpy(), oracle.fixed_order(x, F32))
    m = tcr.Mode(tcr.SHUFFLE_TREE, dtype=F32)
    assert same_bits(tcr.tcr_reduce_sum(t, m).cpu().numpy(),
                     oracle.shuffle_tree(x, F32, *spec.shuffle_team(n, 0, F32)))
    exact, abs_sum = oracle.exact_sum(x, F32)
    got = float(tcr.tcr_reduce_sum(t, tcr.Mode(tcr.MMA_CHAIN, dtype=F32)).cpu().numpy()[0])
    assert abs(got - exact) <= spec.mma_tolerance(abs_sum)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_large_gemm_sampled(dtype):
    M = N = K = 8192
    gen = np.random.default_rng(90)
    A = synth.generate(M * K, "normal", dtype, seed=91).reshape(M, K)
    W = synth.generate(N * K, "normal", dtype, seed=92).reshape(N, K)
    ta = torch.from_numpy(A.view(np.int16)).cuda().view(M, K)
    tw = torch.from_numpy(W.view(np.int16)).cuda().view(N, K)
    dt = torch.float16 if dtype == F16 else torch.bfloat16
    for S in (0, 8):
        d = tcr.tcr_gemm_descriptor(M, N, K, S, dtype)
        C = tcr.tcr_gemm_splitk(ta.view(dt), tw.view(dt), splits=S).cpu().numpy()
        ri = np.sort(gen.choice(M, 48, replace=False))
        cj = np.sort(gen.choice(N, 48, replace=False))
        c, a = oracle.gemm_f64(A[ri], W[cj], dtype)
        got = C[np.ix_(ri, cj)].astype(np.float64)
        assert np.all(np.abs(got - c) <= spec.gemm_bound(d["k_split"], d["splits"], a))


def test_large_exact_partials_gemm_sampled():
    M, N, K, S = 3000, 2500, 4096, 8
    scales = (0, 3, 24, 9, 17, 11, 22, 5)
    A, W = exact_partials_operands(M, N, K, K // S, scales, BF16, seed=93)
    ta = torch.from_numpy(A.view(np.int16)).cuda().view(M, K).view(torch.bfloat16)
    tw = torch.from_numpy(W.view(np.int16)).cuda().view(N, K).view(torch.bfloat16)
    C = tcr.tcr_gemm_splitk(ta, tw, splits=S).cpu().numpy()
    gen = np.random.default_rng(94)
    ri = np.sort(gen.choice(M, 64, replace=False))
    cj = np.sort(gen.choice(N, 64, replace=False))
    ref = oracle.gemm_splitk(A[ri], W[cj], BF16, S, K // S)
    assert same_bits(C[np.ix_(ri, cj)], ref)
