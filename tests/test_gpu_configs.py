"""Parity at the full workload sizes, in the launch configuration the
benchmark times (default block size and chain length unless the workload
names others).

  sum of 2^20 binary16 values, U[-1,1], seed 0     MMA_CHAIN(R=4), FIXED_ORDER
  sum of 2^28 binary16 values, U[0,1), seed 1      MMA_CHAIN R x block sweep, SHUFFLE_TREE,
                                                   MMA_CHAIN_TMEM by R
  65536 x 4096 binary16 rows, N(0,1), seed 2       all three modes and MMA_CHAIN_TMEM
  sum of 2^29 bfloat16 values +-2^e, seed 3        MMA_CHAIN (both kinds) against the exact sum
  sum of 2^30 binary16 values, U[-1,1], seed 4     FIXED_ORDER, 10 runs, bit-exact; MMA_CHAIN
                                                   (both kinds), SHUFFLE_TREE
"""
import numpy as np
import pytest

import oracle
import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300 import synth
from arithmetic_reduction_tensor_gb300.build import build_library
from tests import spec
from tests.test_gpu_parity import assert_within_mma_tolerance, same_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F16, BF16 = tcr.F16, tcr.BF16


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_library()
    torch.cuda.set_device(0)


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).to("cuda")


def run_sum(t, mode):
    return np.float32(tcr.tcr_reduce_sum(t, mode).cpu().numpy()[0])


def test_sum_2p20_f16():
    x = synth.generate(1 << 20, "uniform_pm1", F16, seed=0)
    t = to_dev(x)
    assert same_bits(run_sum(t, tcr.Mode(tcr.FIXED_ORDER)), oracle.fixed_order(x, F16))
    assert_within_mma_tolerance(run_sum(t, tcr.Mode(tcr.MMA_CHAIN, R=4)), *oracle.exact_sum(x, F16))


def test_sum_2p28_f16_sweep_and_shuffle():
    x = synth.generate(1 << 28, "uniform01", F16, seed=1)
    t = to_dev(x)
    exact, abs_sum = oracle.exact_sum(x, F16)
    for R in (1, 2, 4, 5):
        for block in (32, 128, 256, 1024):
            got = run_sum(t, tcr.Mode(tcr.MMA_CHAIN, R=R, block_threads=block))
            assert_within_mma_tolerance(got, exact, abs_sum)
    for R in (1, 2, 3, 4, 5, 8):
        assert_within_mma_tolerance(run_sum(t, tcr.Mode(tcr.MMA_CHAIN_TMEM, R=R)), exact, abs_sum)
    bt, g = spec.shuffle_team(x.size)
    assert same_bits(run_sum(t, tcr.Mode(tcr.SHUFFLE_TREE)), oracle.shuffle_tree(x, F16, bt, g))
    assert same_bits(run_sum(t, tcr.Mode(tcr.FIXED_ORDER)), oracle.fixed_order(x, F16))


def test_rows_65536x4096_f16():
    rows, cols = 65536, 4096
    x = synth.generate(rows * cols, "normal", F16, seed=2).reshape(rows, cols)
    t = to_dev(x.reshape(-1)).view(rows, cols)
    got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()
    assert same_bits(got, oracle.fixed_order_rows(x, F16))
    got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.SHUFFLE_TREE)).cpu().numpy()
    assert same_bits(got, oracle.shuffle_tree_rows(x, F16, *spec.shuffle_team(cols)))
    s, a = oracle.exact_sum_rows(x, F16)
    for R in (0, 1, 4):
        got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.MMA_CHAIN, R=R)).cpu().numpy()
        assert_within_mma_tolerance(got, s, a)
    # the tcgen05 kernel as the bench times it (R = 4), and chains that end with their stage
    for R in (0, 3, 5, 8):
        got = tcr.tcr_reduce_rows(t, tcr.Mode(tcr.MMA_CHAIN_TMEM, R=R)).cpu().numpy()
        assert_within_mma_tolerance(got, s, a)


def test_sum_2p29_bf16_cancellation():
    x = synth.generate(1 << 29, "pow2", BF16, seed=3)
    t = to_dev(x)
    exact, abs_sum = oracle.exact_sum(x, BF16)
    for R in (0, 1, 4, 5, 8):
        assert_within_mma_tolerance(run_sum(t, tcr.Mode(tcr.MMA_CHAIN, R=R, dtype=BF16)), exact, abs_sum)
    for R in (0, 3, 5):
        assert_within_mma_tolerance(run_sum(t, tcr.Mode(tcr.MMA_CHAIN_TMEM, R=R, dtype=BF16)), exact, abs_sum)
    assert same_bits(run_sum(t, tcr.Mode(tcr.FIXED_ORDER, dtype=BF16)), oracle.fixed_order(x, BF16))


def test_sum_2p30_f16_fixed_order_ten_runs():
    x = synth.generate(1 << 30, "uniform_pm1", F16, seed=4)
    t = to_dev(x)
    ref = oracle.fixed_order(x, F16)
    outs = torch.empty(10, dtype=torch.float32, device="cuda")
    for i in range(10):
        tcr.tcr_reduce_sum(t, tcr.Mode(tcr.FIXED_ORDER), out=outs[i:i + 1])
    got = outs.cpu().numpy()
    assert same_bits(got, np.full(10, ref, np.float32))
    exact, abs_sum = oracle.exact_sum(x, F16)
    assert_within_mma_tolerance(run_sum(t, tcr.Mode(tcr.MMA_CHAIN)), exact, abs_sum)
    assert_within_mma_tolerance(run_sum(t, tcr.Mode(tcr.MMA_CHAIN_TMEM)), exact, abs_sum)
    assert same_bits(run_sum(t, tcr.Mode(tcr.SHUFFLE_TREE)),
                     oracle.shuffle_tree(x, F16, *spec.shuffle_team(x.size)))


def test_sum_past_2p32_inputs():
    """The largest case: 2^32 + 1000 binary16 inputs (8 GiB), so every index
    and pointer offset of the kernels runs past 32 bits."""
    n = (1 << 32) + 1000
    x = synth.generate(n, "uniform_pm1", F16, seed=5)
    t = to_dev(x)
    assert same_bits(run_sum(t, tcr.Mode(tcr.FIXED_ORDER)), oracle.fixed_order(x, F16))
    assert same_bits(run_sum(t, tcr.Mode(tcr.SHUFFLE_TREE)),
                     oracle.shuffle_tree(x, F16, *spec.shuffle_team(n)))
    exact, abs_sum = oracle.exact_sum(x, F16)
    assert_within_mma_tolerance(run_sum(t, tcr.Mode(tcr.MMA_CHAIN)), exact, abs_sum)
    # the first 2^32 inputs as 65536 rows of 65536: long rows through the
    # chunked kernels, row offsets past 2^32 bytes
    rows, cols = 65536, 65536
    xr = t[:rows * cols].view(rows, cols)
    got = tcr.tcr_reduce_rows(xr, tcr.Mode(tcr.FIXED_ORDER)).cpu().numpy()
    sel = [0, 1, 32768, 65534, 65535]
    ref = np.array([oracle.fixed_order(x[r * cols:(r + 1) * cols], F16, threads=1) for r in sel])
    assert same_bits(got[sel], ref)
