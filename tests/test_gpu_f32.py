"""GPU parity for binary32 inputs: every mode of libtcr against the CPU oracle.

A binary32 vector is 16 bytes = 4 inputs, so a warp load covers 128 inputs
and a warp group 1024.  FIXED_ORDER and SHUFFLE_TREE must equal the
oracle's emulation bit for bit; MMA_CHAIN (three bfloat16 parts per input on
the tensor cores) must be within |gpu - exact| <= 2^-20 * sum|x_i| + 1e-6.
"""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library
from tests import spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32 = tcr.F32


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def dev(bits):
    """binary32 patterns (uint32) to a CUDA float32 tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint32).view(np.float32)).to("cuda")


def gpu_sum(bits, mode, squares=False):
    f = tcr.tcr_reduce_sum_squares if squares else tcr.tcr_reduce_sum
    return np.float32(f(dev(bits), mode).cpu().numpy()[0])


def gpu_rows(bits2d, mode, squares=False):
    f = tcr.tcr_reduce_rows_sum_squares if squares else tcr.tcr_reduce_rows
    return f(dev(bits2d), mode).cpu().numpy()


def same_bits(a, b):
    a = np.asarray(a, np.float32).reshape(-1)
    b = np.asarray(b, np.float32).reshape(-1)
    nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan]) and \
        np.array_equal(np.isnan(a), np.isnan(b))


def assert_within_mma_tolerance(got, exact, abs_sum):
    got = np.asarray(got, np.float64)
    err = np.abs(got - np.asarray(exact))
    tol = spec.mma_tolerance(np.asarray(abs_sum))
    assert np.all(err <= tol), f"error {np.max(err)} exceeds tolerance (ratio {np.max(err / tol)})"


def inputs(n, dist="normal", seed=None):
    return synth.generate(n, dist, F32, seed=n if seed is None else seed)


def wide_inputs(n, seed):
    """normal values times 2^e, e uniform in [-20, 10]: 30 binades."""
    z = synth.as_float(synth.generate(n, "normal", F32, seed=seed), F32)
    p = synth.as_float(synth.generate(n, "pow2", F32, seed=seed + 1), F32)
    return (z * np.abs(p)).astype(np.float32).view(np.uint32)


SIZES = [1, 3, 4, 5, 127, 128, 129, 1023, 1024, 1025, 4095, 4096, 4097, 8191, 8192, 8193,
         65537, 1_000_003, (1 << 22) + 13]


# ------------------------------------------------------------ ordered modes

@pytest.mark.parametrize("n", SIZES)
def test_fixed_order_sum_bit_exact(n):
    x = inputs(n)
    assert same_bits(gpu_sum(x, tcr.Mode(tcr.FIXED_ORDER, dtype=F32)), oracle.fixed_order(x, F32))
    assert same_bits(gpu_sum(x, tcr.Mode(tcr.FIXED_ORDER, dtype=F32), squares=True),
                     oracle.fixed_order_sq(x, F32))


@pytest.mark.parametrize("n", [4097, 1_000_003])
def test_fixed_order_is_one_class_over_block_sizes(n):
    x = inputs(n, "uniform_pm1")
    ref = oracle.fixed_order(x, F32)
    for block in (32, 64, 128, 256, 512, 1024):
        assert same_bits(gpu_sum(x, tcr.Mode(tcr.FIXED_ORDER, block_threads=block, dtype=F32)), ref)


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("block", [0, 128, 1024])
def test_shuffle_tree_sum_bit_exact(n, block):
    x = inputs(n, "uniform01")
    m = tcr.Mode(tcr.SHUFFLE_TREE, block_threads=block, dtype=F32)
    bt, g = spec.shuffle_team(n, block, F32)
    d = tcr.tcr_order_descriptor(n=n, mode=m)
    assert (d["team_threads"], d["team_blocks"], d["vector_len"]) == (bt, g, 4)
    assert same_bits(gpu_sum(x, m), oracle.shuffle_tree(x, F32, bt, g))
    assert same_bits(gpu_sum(x, m, squares=True), oracle.shuffle_tree_sq(x, F32, bt, g))


def test_binary32_holding_16_bit_values_gives_the_16_bit_fixed_order_bits():
    h = synth.generate(1_000_003, "normal", tcr.F16, seed=77)
    w = synth.as_float(h, tcr.F16).view(np.uint32)
    got32 = gpu_sum(w, tcr.Mode(tcr.FIXED_ORDER, dtype=F32))
    t16 = torch.from_numpy(h.view(np.int16)).to("cuda")
    got16 = np.float32(tcr.tcr_reduce_sum(t16, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()[0])
    assert same_bits(got32, got16)


# ------------------------------------------------------------ MMA_CHAIN

@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("R", [1, 4, 8])
def test_mma_chain_sum_within_tolerance(n, R):
    for dist in ("normal", "uniform01"):
        x = inputs(n, dist)
        exact, abs_sum = oracle.exact_sum(x, F32)
        assert_within_mma_tolerance(gpu_sum(x, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=F32)),
                                    exact, abs_sum)
    x = wide_inputs(n, seed=n + 5)
    exact, abs_sum = oracle.exact_sum(x, F32)
    assert_within_mma_tolerance(gpu_sum(x, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=F32)), exact, abs_sum)


@pytest.mark.parametrize("n", [1, 129, 4097, 1_000_003])
@pytest.mark.parametrize("R", [1, 4, 8])
def test_mma_chain_sum_squares_within_tolerance(n, R):
    x = inputs(n)
    s, _ = oracle.exact_sum_squares(x, F32)
    for kind in (tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM):
        assert_within_mma_tolerance(gpu_sum(x, tcr.Mode(kind, R=R, dtype=F32), squares=True), s, s)


@pytest.mark.parametrize("n,R", [(256, 1), (256, 4), (2048, 4), (2048, 8), (4096, 1), (4096, 4)])
def test_mma_chain_keeps_all_three_parts(n, R):
    # c = 1 + 2^-8 + 2^-16 splits into hi = 1, mid = 2^-8, lo = 2^-16; every
    # partial sum of these n copies is exact in binary32, so the result must
    # be n * c exactly -- a split into two parts would lose n * 2^-16
    c = np.float32(1 + 2.0 ** -8 + 2.0 ** -16)
    x = np.full(n, c, np.float32).view(np.uint32)
    got = gpu_sum(x, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=F32))
    assert got == np.float32(n * (1 + 2.0 ** -8 + 2.0 ** -16))


def test_mma_chain_tmem_binary32_runs_the_split_kernel():
    x = inputs(3_000_001)
    a = gpu_sum(x, tcr.Mode(tcr.MMA_CHAIN_TMEM, dtype=F32))
    b = gpu_sum(x, tcr.Mode(tcr.MMA_CHAIN, dtype=F32))
    assert same_bits(a, b)


def test_mma_chain_is_run_to_run_stable():
    x = wide_inputs(5_000_011, seed=9)
    m = tcr.Mode(tcr.MMA_CHAIN, dtype=F32)
    first = gpu_sum(x, m)
    for _ in range(3):
        assert same_bits(gpu_sum(x, m), first)


def test_mma_chain_extremes_split_without_overflow():
    # the largest binary32 values round to infinity in bfloat16 under round
    # to nearest; the split rounds toward zero, so +-max cancel exactly
    fmax = 0x7F7FFFFF
    x = np.zeros(5000, np.uint32)
    x[10], x[4000], x[4999] = fmax, fmax | 0x80000000, np.float32(1.5).view(np.uint32)
    got = gpu_sum(x, tcr.Mode(tcr.MMA_CHAIN, dtype=F32))
    assert got == np.float32(1.5)
    # subnormals and tiny normals: within the absolute term of the bound
    tiny = np.arange(1, 10_001, dtype=np.uint32)            # 1..10000 * 2^-149
    tiny[::2] |= np.uint32(0x80000000)
    tiny[::3] += np.uint32(0x00800000)                      # some normal values near 2^-126
    exact, abs_sum = oracle.exact_sum(tiny, F32)
    assert_within_mma_tolerance(gpu_sum(tiny, tcr.Mode(tcr.MMA_CHAIN, dtype=F32)), exact, abs_sum)


# ------------------------------------------------------------ every mode

KINDS = [tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM]


@pytest.mark.parametrize("kind", KINDS)
def test_non_finite_inputs(kind):
    x = inputs(100_000)
    m = tcr.Mode(kind, dtype=F32)
    cases = ((0x7F800000, np.inf), (0xFF800000, -np.inf), (0x7FC00000, np.nan),
             (0x7F800001, np.nan), (0xFFFFFFFF, np.nan))
    for pattern, expect in cases:
        y = x.copy()
        y[12345] = pattern
        got = gpu_sum(y, m)
        assert np.isnan(got) if np.isnan(expect) else got == expect, hex(pattern)
    y = x.copy()
    y[1], y[99_999] = 0x7F800000, 0xFF800000
    assert np.isnan(gpu_sum(y, m))
    # squares: -inf squared is +inf
    y = x.copy()
    y[7] = 0xFF800000
    assert gpu_sum(y, m, squares=True) == np.inf


@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("kind", KINDS)
def test_misaligned_base_pointer(offset, kind):
    n = 300_007
    x = inputs(n + offset, "uniform_pm1")
    t = dev(x)[offset:]
    xs = x[offset:]
    m = tcr.Mode(kind, dtype=F32)
    got = np.float32(tcr.tcr_reduce_sum(t, m).cpu().numpy()[0])
    if kind == tcr.FIXED_ORDER:
        assert same_bits(got, oracle.fixed_order(xs, F32))
    elif kind == tcr.SHUFFLE_TREE:
        assert same_bits(got, oracle.shuffle_tree(xs, F32, *spec.shuffle_team(n, 0, F32)))
    else:
        assert_within_mma_tolerance(got, *oracle.exact_sum(xs, F32))


ROW_SHAPES = [(1, 1), (3, 5), (1000, 4096), (333, 4095), (64, 8192), (50, 8193), (4, 1_000_003)]


@pytest.mark.parametrize("shape", ROW_SHAPES)
def test_rows_all_modes(shape):
    rows, cols = shape
    x = inputs(rows * cols, seed=rows + cols).reshape(rows, cols)
    for squares in (False, True):
        got = gpu_rows(x, tcr.Mode(tcr.FIXED_ORDER, dtype=F32), squares)
        assert same_bits(got, oracle.fixed_order_rows(x, F32, squares=squares))
        bt, g = spec.shuffle_team(cols, 0, F32)
        got = gpu_rows(x, tcr.Mode(tcr.SHUFFLE_TREE, dtype=F32), squares)
        assert same_bits(got, oracle.shuffle_tree_rows(x, F32, bt, g, squares=squares))
        s, a = oracle.exact_sum_rows(x, F32, squares=squares)
        for kind in (tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM):
            assert_within_mma_tolerance(gpu_rows(x, tcr.Mode(kind, dtype=F32), squares), s, a)


def test_rows_are_batch_invariant():
    cols = 3001
    x = inputs(40 * cols, seed=5).reshape(40, cols)
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        m = tcr.Mode(kind, dtype=F32)
        whole = gpu_rows(x, m)
        for r in (0, 17, 39):
            assert same_bits(gpu_rows(x[r:r + 1], m), whole[r])
            assert same_bits(gpu_sum(x[r], m), whole[r])


def test_float32_tensor_and_raw_patterns_agree():
    x = inputs(100_003)
    as_float = tcr.tcr_reduce_sum(dev(x), tcr.Mode(tcr.FIXED_ORDER, dtype=F32))
    raw = torch.from_numpy(x.view(np.int32)).to("cuda")
    as_bits = tcr.tcr_reduce_sum(raw, tcr.Mode(tcr.FIXED_ORDER, dtype=F32))
    assert same_bits(as_float.cpu().numpy(), as_bits.cpu().numpy())
    with pytest.raises(ValueError):
        tcr.tcr_reduce_sum(dev(x), tcr.Mode(tcr.FIXED_ORDER, dtype=tcr.F16))
