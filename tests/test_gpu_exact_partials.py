"""MMA_CHAIN bit for bit at full size, on inputs whose partial sums are all exact.

The tolerance |gpu - exact| <= 2^-20 * sum|x| + 1e-6 that bounds MMA_CHAIN on
general inputs is about 512 on the 2^30-input sum: it cannot see a dropped or
repeated warp load.  These tests feed inputs on which no addition rounds, so
the tensor-core path must return the exact sum itself:

* the tensor core rounds an MMA's result (toward zero) only when the exact
  value does not fit binary32, and every CUDA-core addition rounds only then
  too ("GPU Tensor Cores for fast Arithmetic Reductions", Abstract: the chain
  sub-results are kept and reduced in 32-bit floating point);
* ``exact_int`` inputs (synth) are integers; each 16-byte vector sums to
  exactly +-1 and opens with a pair (a, -a) that shares one 32-bit register,
  so every partial a kernel forms is an integer far below 2^24 and the exact
  total is a small integer.  Dropping or repeating any one vector moves the
  total by 1, which binary32 represents: any such slip fails these tests;
* all-ones inputs must give n exactly (n a power of two here), and +-1
  inputs give a sum of squares of exactly n.

Sizes are the benchmark's workloads (2^30 sum, 65536 x 4096 rows, 2^29
bfloat16 and binary32 sums), the 64-bit offset case (2^32 + 1000 inputs),
misaligned bases and ragged tails.
"""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F16, BF16, F32 = tcr.F16, tcr.BF16, tcr.F32
MMA, TMEM, FIXED, SHUFFLE = tcr.MMA_CHAIN, tcr.MMA_CHAIN_TMEM, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def to_dev(bits):
    if bits.dtype == np.uint32:
        return torch.from_numpy(bits.view(np.float32)).cuda()
    return torch.from_numpy(bits.view(np.int16)).cuda()


def exact_f32(bits, dtype):
    """The exact sum, checked to be an integer that binary32 holds exactly."""
    e, _ = oracle.exact_sum(bits, dtype)
    assert e == np.round(e) and abs(e) < 2 ** 24
    return np.float32(e)


def exact_rows_f32(bits2d, dtype, squares=False):
    e, _ = oracle.exact_sum_rows(bits2d, dtype, squares=squares)
    assert np.all(e == np.round(e)) and np.all(np.abs(e) < 2 ** 24)
    return e.astype(np.float32)


def sum_bits(t, mode, squares=False):
    f = tcr.tcr_reduce_sum_squares if squares else tcr.tcr_reduce_sum
    return f(t, mode).cpu().numpy().view(np.uint32)[0]


def rows_bits(t, mode, squares=False):
    f = tcr.tcr_reduce_rows_sum_squares if squares else tcr.tcr_reduce_rows
    return f(t, mode).cpu().numpy().view(np.uint32)


def bits_of(v):
    return np.asarray(v, np.float32).view(np.uint32)


# every MMA_CHAIN configuration a caller can pick on a sum (chain length x
# block size), and the tcgen05 kind by chain length
MMA_CONFIGS = [(R, b) for R in (1, 4, 5, 8) for b in (32, 256, 1024)] + [(0, 0)]
TMEM_R = (0, 1, 3, 5, 8)


@pytest.fixture(scope="module")
def sum_2p30():
    x = synth.generate(1 << 30, "exact_int", F16, seed=11)
    return x, to_dev(x), exact_f32(x, F16)


def test_2p30_sum_every_chain_and_block(sum_2p30):
    x, t, e = sum_2p30
    for R, b in MMA_CONFIGS:
        assert sum_bits(t, tcr.Mode(MMA, R=R, block_threads=b)) == bits_of(e), (R, b)
    for R in TMEM_R:
        assert sum_bits(t, tcr.Mode(TMEM, R=R)) == bits_of(e), R
    # the ordered modes meet no rounding either
    assert sum_bits(t, tcr.Mode(FIXED)) == bits_of(e)
    assert sum_bits(t, tcr.Mode(SHUFFLE)) == bits_of(e)


@pytest.mark.parametrize("lo,hi", [(1, 1 << 30), (0, (1 << 30) - 3), (3, (1 << 30) - 1001),
                                   (8, (1 << 30) - 8)])
def test_2p30_sum_misaligned_and_ragged(sum_2p30, lo, hi):
    # a base 2 or 6 bytes past a 16-byte boundary takes the realigning loads
    # (the tcgen05 kind then runs the mma.sync kernel); ragged tails end
    # inside a vector, a group and a tile
    x, t, _ = sum_2p30
    xs, ts = x[lo:hi], t[lo:hi]
    e = exact_f32(xs, F16)
    for R, b in ((4, 256), (1, 1024), (8, 32), (0, 0)):
        assert sum_bits(ts, tcr.Mode(MMA, R=R, block_threads=b)) == bits_of(e), (lo, hi, R, b)
    for R in (0, 5):
        assert sum_bits(ts, tcr.Mode(TMEM, R=R)) == bits_of(e), (lo, hi, R)


def test_2p30_all_ones_gives_n():
    n = 1 << 30
    t = torch.full((n,), 1.0, dtype=torch.float16, device="cuda").view(torch.int16)
    for R, b in ((4, 256), (1, 1024), (5, 32)):
        assert sum_bits(t, tcr.Mode(MMA, R=R, block_threads=b)) == bits_of(n)
    for R in (0, 3):
        assert sum_bits(t, tcr.Mode(TMEM, R=R)) == bits_of(n)
    # +-1: every square is 1, the sum of squares is n on the A * A^T path
    signs = synth.generate(n, "uniform_pm1", F16, seed=12) & np.uint16(0x8000)
    pm1 = to_dev(signs | np.uint16(0x3C00))
    for kind in (MMA, TMEM):
        assert sum_bits(pm1, tcr.Mode(kind), squares=True) == bits_of(n)


def test_past_2p32_inputs():
    """2^32 + 1000 inputs: every index and byte offset runs past 32 bits."""
    n = (1 << 32) + 1000
    x = synth.generate(n, "exact_int", F16, seed=13)
    t = to_dev(x)
    e = exact_f32(x, F16)
    for R, b in ((4, 256), (1, 1024), (8, 32)):
        assert sum_bits(t, tcr.Mode(MMA, R=R, block_threads=b)) == bits_of(e), (R, b)
    assert sum_bits(t, tcr.Mode(TMEM)) == bits_of(e)
    # from a misaligned base, through the realigning loads
    e1 = exact_f32(x[1:], F16)
    assert sum_bits(t[1:], tcr.Mode(MMA)) == bits_of(e1)
    # as 65536 rows of 65536 (rows through the chunked kernels, row offsets
    # past 2^32 bytes)
    rows, cols = 65536, 65536
    xr = x[:rows * cols].reshape(rows, cols)
    er = exact_rows_f32(xr, F16)
    for kind in (MMA, TMEM):
        assert np.array_equal(rows_bits(t[:rows * cols].view(rows, cols), tcr.Mode(kind)),
                              bits_of(er)), kind


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_65536x4096_rows(dtype):
    rows, cols = 65536, 4096
    x = synth.generate(rows * cols, "exact_int", dtype, seed=14).reshape(rows, cols)
    t = to_dev(x.reshape(-1)).view(rows, cols)
    e = bits_of(exact_rows_f32(x, dtype))
    for R in (0, 1, 4, 5, 8):
        assert np.array_equal(rows_bits(t, tcr.Mode(MMA, R=R, dtype=dtype)), e), R
    for R in (0, 1, 3, 5, 8):
        assert np.array_equal(rows_bits(t, tcr.Mode(TMEM, R=R, dtype=dtype)), e), R
    # rows from a base one input past a boundary: every row misaligned
    xm = x.reshape(-1)[1:1 + (rows - 1) * cols].reshape(rows - 1, cols)
    tm = t.view(-1)[1:1 + (rows - 1) * cols].view(rows - 1, cols)
    em = bits_of(exact_rows_f32(xm, dtype))
    for kind in (MMA, TMEM):
        assert np.array_equal(rows_bits(tm, tcr.Mode(kind, dtype=dtype)), em), kind


@pytest.mark.parametrize("cols", [64, 100, 1000, 12288, 40000])
def test_rows_every_width_path(cols):
    # packed short rows (64, 100 not 16-byte aligned), the tcgen05 rows
    # kernel's two-group instance (1000), one warp per row (12288) and the
    # chunked kernels with a combine (40000)
    rows = max(3, (1 << 26) // cols)
    x = synth.generate(rows * cols, "exact_int", F16, seed=cols).reshape(rows, cols)
    t = to_dev(x.reshape(-1)).view(rows, cols)
    e = bits_of(exact_rows_f32(x, F16))
    for kind in (MMA, TMEM):
        for R in (0, 1, 5):
            assert np.array_equal(rows_bits(t, tcr.Mode(kind, R=R)), e), (kind, R)


def test_2p29_bfloat16_sum():
    x = synth.generate(1 << 29, "exact_int", BF16, seed=15)
    t = to_dev(x)
    e = exact_f32(x, BF16)
    for R, b in MMA_CONFIGS:
        assert sum_bits(t, tcr.Mode(MMA, R=R, block_threads=b, dtype=BF16)) == bits_of(e), (R, b)
    for R in TMEM_R:
        assert sum_bits(t, tcr.Mode(TMEM, R=R, dtype=BF16)) == bits_of(e), R


def test_2p29_binary32_sum_through_the_split():
    # the a's carry 20 significant bits: hi, mid and lo of the three-way
    # bfloat16 split are all in use
    x = synth.generate(1 << 29, "exact_int", F32, seed=16)
    t = to_dev(x)
    e = exact_f32(x, F32)
    for R, b in MMA_CONFIGS:
        assert sum_bits(t, tcr.Mode(MMA, R=R, block_threads=b, dtype=F32)) == bits_of(e), (R, b)
    assert sum_bits(t, tcr.Mode(TMEM, dtype=F32)) == bits_of(e)
    # ragged tail (the last vector cut short)
    e2 = exact_f32(x[:-3], F32)
    assert sum_bits(t[:-3], tcr.Mode(MMA, dtype=F32)) == bits_of(e2)
    rows, cols = 65536, 2048
    xr = x[:rows * cols].reshape(rows, cols)
    er = bits_of(exact_rows_f32(xr, F32))
    for R in (0, 1, 8):
        assert np.array_equal(rows_bits(t[:rows * cols].view(rows, cols), tcr.Mode(MMA, R=R, dtype=F32)), er)


@pytest.mark.parametrize("dtype", [F16, BF16, F32])
def test_sum_of_squares_exact(dtype):
    # +-1 and 0 (the signs of exact_int inputs): every square is 0 or 1 and
    # the total stays below 2^24, so a dropped or repeated vector holding a
    # nonzero input changes it
    n = (1 << 23) + 5
    v = np.sign(synth.as_float(synth.generate(n, "exact_int", dtype, seed=17), dtype).astype(np.float64))
    if dtype == F32:
        x = v.astype(np.float32).view(np.uint32)
    elif dtype == F16:
        x = v.astype(np.float16).view(np.uint16)
    else:
        x = (v.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    t = to_dev(x)
    e, _ = oracle.exact_sum_squares(x, dtype)
    assert e < 2 ** 24
    for R, b in ((4, 256), (1, 1024), (8, 32)):
        assert sum_bits(t, tcr.Mode(MMA, R=R, block_threads=b, dtype=dtype), squares=True) == bits_of(e)
    rows, cols = 2048, 4096
    xr = x[:rows * cols].reshape(rows, cols)
    er = bits_of(exact_rows_f32(xr, dtype, squares=True))
    tr = t[:rows * cols].view(rows, cols)
    for R in (0, 1, 8):
        assert np.array_equal(rows_bits(tr, tcr.Mode(MMA, R=R, dtype=dtype), squares=True), er)


# The tcgen05 rows kernel for rows of 1024 k columns (k a divisor or a
# multiple of 16) reads the matrix as a flat array: a row is 8 k TMEM lanes
# inside one warp (k = 1, 2, 4), two or four warps (k = 8, 16), or all 128
# lanes over several stages (k = 32, 48, 64), or chunks of 65536 columns
# with partials and the rows combine (k = 80, 128).  Row counts that leave a
# partial last unit.
FLAT_SHAPES = [(65, 1024), (33, 2048), (17, 4096), (9, 8192), (5, 16384), (3, 32768),
               (2, 49152), (3, 65536), (2, 81920), (2, 131072)]


@pytest.mark.parametrize("dtype", [F16, BF16])
@pytest.mark.parametrize("shape", FLAT_SHAPES)
def test_flat_tcgen05_rows_every_lane_layout(dtype, shape):
    rows, cols = shape
    x = synth.generate(rows * cols, "exact_int", dtype, seed=cols + rows).reshape(rows, cols)
    t = to_dev(x.reshape(-1)).view(rows, cols)
    e = bits_of(exact_rows_f32(x, dtype))
    for R in (0, 1, 3, 5, 8):
        assert np.array_equal(rows_bits(t, tcr.Mode(TMEM, R=R, dtype=dtype)), e), (shape, R)
    # a single row alone gives its bits (no dependence on the row count)
    assert np.array_equal(rows_bits(t[rows - 1:rows], tcr.Mode(TMEM, dtype=dtype)), e[rows - 1:rows])
