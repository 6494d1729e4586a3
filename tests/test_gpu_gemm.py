"""GPU parity for the split-K GEMM with the declared K-partition combine.

With exact-partials operands (small integers, one power-of-two scale per
split) every split's partial is exact on the tensor core and in the oracle,
so only the declared combine rounds: C must equal the oracle bit for bit.
General operands: within the bound stated in include/tcr.h of the binary64
product, and bit-identical from call to call.
"""
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

F16, BF16 = tcr.F16, tcr.BF16
TORCH_DT = {F16: torch.float16, BF16: torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


@pytest.fixture(autouse=True, params=["pair", "one_sm"])
def gemm_kernel(request, monkeypatch):
    # every test on both kernels: CTA pairs (the default where pairs can be
    # scheduled) and one SM per tile (TCR_GEMM_ONE_SM)
    if request.param == "one_sm":
        monkeypatch.setenv("TCR_GEMM_ONE_SM", "1")
    return request.param


def dev(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(TORCH_DT[dtype])


def gemm(A, W, dtype, splits=0):
    return tcr.tcr_gemm_splitk(dev(A, dtype), dev(W, dtype), splits=splits).cpu().numpy()


def same_bits(a, b):
    a = np.asarray(a, np.float32).reshape(-1)
    b = np.asarray(b, np.float32).reshape(-1)
    nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan]) and \
        np.array_equal(np.isnan(a), np.isnan(b))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("shape,S,scales", [
    ((128, 128, 256), 4, (0, 24, 24, 24)),
    ((200, 300, 320), 5, (0, 13, 24, 7, 20)),
    ((7, 9, 192), 3, (3, 0, 17)),
    ((384, 256, 1024), 8, (0, 5, 10, 15, 20, 23, 2, 9)),
])
def test_exact_partials_bit_exact(dtype, shape, S, scales):
    M, N, K = shape
    d = tcr.tcr_gemm_descriptor(M, N, K, S, dtype)
    assert (d["splits"], d["k_split"]) == spec.gemm_splits(M, N, K, S) == (S, K // S)
    A, W = exact_partials_operands(M, N, K, d["k_split"], scales, dtype, seed=M + N + K)
    got = gemm(A, W, dtype, S)
    assert same_bits(got, oracle.gemm_splitk(A, W, dtype, S, d["k_split"]))


def test_the_combine_is_the_declared_tree():
    # P = (1, t, t, t) with t = 2^-24: the tree gives 1 + 2^-23, not 1
    A = np.full((1, 256), 0x3C00, np.uint16)
    W = np.zeros((1, 256), np.uint16)
    W[0, 0] = 0x3C00
    W[0, 64] = W[0, 128] = W[0, 192] = 0x0001
    assert gemm(A, W, F16, 4)[0, 0] == np.float32(1 + 2.0 ** -23)
    assert gemm(A, W, F16, 1)[0, 0] in (np.float32(1 + 2.0 ** -23), np.float32(1 + 2.0 ** -22),
                                        np.float32(1.0))


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("shape,S", [
    ((256, 384, 1024), 0), ((1000, 64, 4096), 0), ((129, 257, 200), 0), ((77, 131, 40), 0),
    ((1, 1, 8), 0), ((1, 640, 1024), 3), ((640, 1, 1024), 16), ((2048, 2048, 512), 0),
])
def test_general_within_bound(dtype, shape, S):
    M, N, K = shape
    A = synth.generate(M * K, "normal", dtype, seed=M + 1).reshape(M, K)
    W = synth.generate(N * K, "normal", dtype, seed=N + 2).reshape(N, K)
    d = tcr.tcr_gemm_descriptor(M, N, K, S, dtype)
    assert (d["splits"], d["k_split"]) == spec.gemm_splits(M, N, K, S)
    got = gemm(A, W, dtype, S).astype(np.float64)
    c, a = oracle.gemm_f64(A, W, dtype)
    tol = spec.gemm_bound(d["k_split"], d["splits"], a)
    assert np.all(np.abs(got - c) <= tol), float(np.max(np.abs(got - c) / tol))


def test_bits_repeat_and_do_not_depend_on_the_stream():
    M, N, K = 300, 500, 2048
    A = synth.generate(M * K, "uniform_pm1", BF16, seed=80).reshape(M, K)
    W = synth.generate(N * K, "uniform_pm1", BF16, seed=81).reshape(N, K)
    ta, tw = dev(A, BF16), dev(W, BF16)
    first = tcr.tcr_gemm_splitk(ta, tw, splits=6).cpu().numpy()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        again = tcr.tcr_gemm_splitk(ta, tw, splits=6, stream=s)
    s.synchronize()
    assert same_bits(again.cpu().numpy(), first)
    for _ in range(3):
        assert same_bits(tcr.tcr_gemm_splitk(ta, tw, splits=6).cpu().numpy(), first)
    # another split is another declared order: other bits, the same bound
    other = tcr.tcr_gemm_splitk(ta, tw, splits=2).cpu().numpy()
    assert not same_bits(other, first)


def test_degenerate_and_rejected():
    A = torch.zeros(3, 0, dtype=torch.float16, device="cuda")
    W = torch.zeros(5, 0, dtype=torch.float16, device="cuda")
    out = torch.full((3, 5), 7.0, device="cuda")
    tcr.tcr_gemm_splitk(A, W, out=out)
    assert np.all(out.cpu().numpy() == 0.0)
    with pytest.raises(tcr.TcrError):
        tcr.tcr_gemm_splitk(torch.zeros(4, 12, dtype=torch.float16, device="cuda"),
                            torch.zeros(4, 12, dtype=torch.float16, device="cuda"))   # K % 8 != 0
    with pytest.raises(tcr.TcrError):
        tcr.tcr_gemm_splitk(torch.zeros(4, 16, dtype=torch.float16, device="cuda"),
                            torch.zeros(4, 16, dtype=torch.float16, device="cuda"), splits=65)
    assert tcr.tcr_device_faults() == 0


def test_descriptor_reports_the_kernel(gemm_kernel):
    # a GB300 schedules CTA pairs: 256 x 256 tiles, two CTAs per pair; on
    # request one SM per 128 x 256 tile
    d = tcr.tcr_gemm_descriptor(4096, 4096, 4096, 0, BF16)
    if gemm_kernel == "pair":
        assert (d["tile_m"], d["tile_n"]) == (256, 256)
        assert d["launch_grid"] % 2 == 0 and 2 <= d["launch_grid"] <= 152
    else:
        assert (d["tile_m"], d["tile_n"]) == (128, 256)
        assert d["launch_grid"] <= 152
