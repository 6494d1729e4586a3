"""The C ABI without a GPU: the library loads, exports every entry point
``include/tcr.h`` declares, rejects bad arguments before any GPU work and
describes the declared orders."""
import ctypes
import os
import re
import subprocess

import pytest

import arithmetic_reduction_tensor_gb300 as tcr
from arithmetic_reduction_tensor_gb300.build import build_library, LIB_PATH
from tests import spec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_library()
    return tcr.c_api()


def declared_entry_points():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"TCR_API\s+[\w\s\*]+?\b(tcr_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("tcr_reduce_sum", "tcr_reduce_rows", "tcr_order_descriptor", "tcr_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (tcr_\w+)", out))
    assert set(declared_entry_points()) <= exported
    # nothing else of ours leaks out of the shared object
    assert {s for s in exported if s.startswith("tcr")} == set(declared_entry_points())
    for n in declared_entry_points():
        assert hasattr(lib, n)


def test_status_strings(lib):
    for st in range(4):
        assert isinstance(tcr.tcr_status_string(st), str) and tcr.tcr_status_string(st)
    assert tcr.tcr_status_string(99) == "unknown status"


FAKE = 0x7F0000000000      # never dereferenced: every case below fails validation


@pytest.mark.parametrize("args", [
    # (x, n, out, mode)
    (FAKE, 10, None, tcr.Mode(tcr.FIXED_ORDER)),                 # out NULL
    (FAKE, 10, FAKE + 2, tcr.Mode(tcr.FIXED_ORDER)),             # out misaligned
    (None, 10, FAKE, tcr.Mode(tcr.FIXED_ORDER)),                 # x NULL with n > 0
    (FAKE + 1, 10, FAKE, tcr.Mode(tcr.FIXED_ORDER)),             # x not 2-byte aligned
    (FAKE, 1 << 40, FAKE, tcr.Mode(tcr.FIXED_ORDER)),            # n too large
    (FAKE, 10, FAKE, tcr.Mode(7)),                               # unknown kind
    (FAKE, 10, FAKE, tcr.Mode(tcr.FIXED_ORDER, dtype=5)),        # unknown dtype
    (FAKE, 10, FAKE, tcr.Mode(tcr.FIXED_ORDER, dtype=3)),
    (FAKE + 2, 10, FAKE, tcr.Mode(tcr.FIXED_ORDER, dtype=tcr.F32)),   # binary32 not 4-byte aligned
    (FAKE + 2, 10, FAKE, tcr.Mode(tcr.MMA_CHAIN, dtype=tcr.F32)),
    (FAKE, 10, FAKE, tcr.Mode(tcr.MMA_CHAIN, R=9)),              # R out of range
    (FAKE, 10, FAKE, tcr.Mode(tcr.MMA_CHAIN, R=-1)),
    (FAKE, 10, FAKE, tcr.Mode(tcr.SHUFFLE_TREE, block_threads=48)),   # not a power of two
    (FAKE, 10, FAKE, tcr.Mode(tcr.SHUFFLE_TREE, block_threads=2048)),
    (FAKE, 10, FAKE, tcr.Mode(tcr.SHUFFLE_TREE, block_threads=16)),
])
def test_sum_rejects_bad_arguments_before_gpu_work(lib, args):
    x, n, out, mode = args
    assert lib.tcr_reduce_sum(x, n, out, mode, None) == tcr.ERR_INVALID_ARG
    # the entry point without allocation checks its arguments the same way
    f = lib.tcr_reduce_sum_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, tcr.tcr_mode, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(x, n, out, mode, None) == tcr.ERR_INVALID_ARG


@pytest.mark.parametrize("mode", [tcr.Mode(tcr.SHUFFLE_TREE), tcr.Mode(tcr.MMA_CHAIN_TMEM),
                                  tcr.Mode(tcr.FIXED_ORDER, run_log2=3)])
def test_noalloc_refuses_what_it_does_not_serve_before_gpu_work(lib, mode):
    f = lib.tcr_reduce_sum_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, tcr.tcr_mode, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(FAKE, 10, FAKE, mode, None) == tcr.ERR_UNSUPPORTED
    # more chunks than its fixed array holds: 65536 chunks of 2^16 inputs (8
    # warps of 2^13) at 256 threads
    assert f(FAKE, 65536 * 8192 * 8 + 1, FAKE, tcr.Mode(tcr.FIXED_ORDER), None) == tcr.ERR_UNSUPPORTED


def test_rows_rejects_bad_arguments(lib):
    m = tcr.Mode(tcr.FIXED_ORDER)
    assert lib.tcr_reduce_rows(FAKE, 1 << 21, 1 << 21, FAKE, m, None) == tcr.ERR_INVALID_ARG
    assert lib.tcr_reduce_rows(FAKE, 1 << 40, 1 << 40, FAKE, m, None) == tcr.ERR_INVALID_ARG
    assert lib.tcr_reduce_rows(FAKE, 3, 5, None, m, None) == tcr.ERR_INVALID_ARG
    assert lib.tcr_reduce_rows(FAKE, 3, 5, FAKE, tcr.Mode(tcr.MMA_CHAIN, R=11), None) == \
        tcr.ERR_INVALID_ARG
    # no rows: nothing to do, any pointers
    assert lib.tcr_reduce_rows(None, 0, 5, None, m, None) == tcr.OK


def test_descriptor_rejects_bad_arguments(lib):
    d = tcr.tcr_order_desc()
    assert lib.tcr_order_descriptor(10, 0, 0, tcr.Mode(9), ctypes.byref(d)) == tcr.ERR_INVALID_ARG
    assert lib.tcr_order_descriptor(10, 0, 0, tcr.Mode(0), None) == tcr.ERR_INVALID_ARG
    assert lib.tcr_order_descriptor(1 << 40, 0, 0, tcr.Mode(0), ctypes.byref(d)) == \
        tcr.ERR_INVALID_ARG


@pytest.mark.parametrize("L", [1, 100, 4096, 4097, 8192, 8193, 10_000, 1 << 20, 1 << 28, 1 << 30])
@pytest.mark.parametrize("block", [0, 32, 128, 1024])
@pytest.mark.parametrize("dtype", [tcr.F16, tcr.BF16, tcr.F32])
def test_shuffle_descriptor_matches_the_declared_rule(lib, L, block, dtype):
    m = tcr.Mode(tcr.SHUFFLE_TREE, block_threads=block, dtype=dtype)
    bt, g = spec.shuffle_team(L, block, dtype)
    for d in (tcr.tcr_order_descriptor(n=L, mode=m), tcr.tcr_order_descriptor(rows=3, cols=L, mode=m)):
        assert d["order"] == tcr.ORDER_GRID_STRIDE
        assert (d["team_threads"], d["team_blocks"]) == (bt, g)
        assert d["vector_len"] == spec.vector_len(dtype) and d["pad_negative_zero"] == 1
        assert d["dtype"] == dtype
        assert d["partials"] == (0 if g == 1 else d["segments"] * g)


def test_short_rows_are_packed(lib):
    # rows of at most 128 vectors share a warp group: 256 / 2^v rows per warp
    # (2^v vector slots per row, at least 4 for MMA_CHAIN), 8 warps per CTA,
    # one launch, no scratch; longer rows take one warp each.  (Without a
    # device the plan assumes 152 SMs and one resident CTA per SM.)
    def grid(rows, cols, kind, dtype=tcr.F16):
        d = tcr.tcr_order_descriptor(rows=rows, cols=cols, mode=tcr.Mode(kind, dtype=dtype))
        assert (d["launch_block"], d["launches"], d["partials"]) == (256, 1, 0)
        return d["launch_grid"]

    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
        assert grid(1000, 64, kind) == 4              # 8 vectors: 32 rows a warp
        assert grid(1000, 65, kind) == 8              # 9 vectors: 16 rows a warp
        assert grid(1000, 1024, kind) == 63           # 128 vectors: 2 rows a warp
        assert grid(1000, 1025, kind) == 125          # one warp per row
        assert grid(10 ** 6, 100, kind) == 8 * 152    # at most eight waves
    # rows that are not whole vectors pack the same way
    assert grid(1000, 255, tcr.FIXED_ORDER) == 16     # 32 vectors: 8 rows a warp
    assert grid(1000, 1020, tcr.SHUFFLE_TREE) == 63   # 128 vectors: 2 rows a warp
    assert grid(1000, 8, tcr.FIXED_ORDER) == 1        # one vector: 256 rows a warp
    assert grid(1000, 8, tcr.MMA_CHAIN) == 2          # one lane quad: 64 rows a warp
    assert grid(1000, 64, tcr.FIXED_ORDER, tcr.F32) == 8
    assert grid(1000, 512, tcr.SHUFFLE_TREE, tcr.F32) == 63
    assert grid(1000, 513, tcr.SHUFFLE_TREE, tcr.F32) == 125
    # binary32 MMA_CHAIN (the three-way split) packs the same way
    assert grid(1000, 64, tcr.MMA_CHAIN, tcr.F32) == 8
    assert grid(1000, 8, tcr.MMA_CHAIN, tcr.F32) == 2     # two vectors: one lane quad each


def test_binary32_descriptors(lib):
    # a warp span is 16 KiB: 2^13 16-bit inputs, 2^12 binary32 inputs (at a
    # length where no CTA size is shrunk)
    for blk in (32, 256, 1024):
        d16 = tcr.tcr_order_descriptor(n=1 << 28, mode=tcr.Mode(tcr.FIXED_ORDER, block_threads=blk))
        d32 = tcr.tcr_order_descriptor(
            n=1 << 28, mode=tcr.Mode(tcr.FIXED_ORDER, block_threads=blk, dtype=tcr.F32))
        assert d32["chunk_log2"] == d16["chunk_log2"] - 1
        assert d32["partials"] == 2 * d16["partials"]
    # rows of up to 32 KiB take one warp each: 16384 16-bit or 8192 binary32 inputs
    # (at 32 threads a chunked row is 2^12-input chunks, so 8193 makes 3 --
    # 300 work units, fewer than two per SM, so the spans halve: 5 per row)
    m = tcr.Mode(tcr.FIXED_ORDER, block_threads=32, dtype=tcr.F32)
    d = tcr.tcr_order_descriptor(rows=100, cols=8192, mode=m)
    assert d["partials"] == 0 and d["launch_block"] == 256
    d = tcr.tcr_order_descriptor(rows=100, cols=8193, mode=m)
    assert d["partials"] == 500 and d["launch_block"] == 32 and d["chunk_log2"] == 11
    d = tcr.tcr_order_descriptor(rows=200, cols=8193, mode=m)
    assert d["partials"] == 600 and d["chunk_log2"] == 12
    # the tcgen05 kind reduces binary32 inputs with the mma.sync split kernel
    d = tcr.tcr_order_descriptor(n=1 << 24, mode=tcr.Mode(tcr.MMA_CHAIN_TMEM, dtype=tcr.F32))
    dm = tcr.tcr_order_descriptor(n=1 << 24, mode=tcr.Mode(tcr.MMA_CHAIN, dtype=tcr.F32))
    assert (d["launch_block"], d["chunk_log2"], d["partials"]) == \
        (dm["launch_block"], dm["chunk_log2"], dm["partials"])


def test_equivalence_needs_the_same_input_type(lib):
    for kind in (tcr.FIXED_ORDER, tcr.SHUFFLE_TREE, tcr.MMA_CHAIN):
        a = {"n": 100_000, "mode": tcr.Mode(kind)}
        assert tcr.tcr_order_equivalent(a, a)
        assert not tcr.tcr_order_equivalent(a, {"n": 100_000, "mode": tcr.Mode(kind, dtype=tcr.F32)})
    f32 = tcr.Mode(tcr.SHUFFLE_TREE, dtype=tcr.F32)
    # 3000 binary32 inputs are 750 vectors: every team of at least 750
    # threads holds at most one vector per thread
    assert tcr.tcr_order_equivalent(
        {"n": 3000, "mode": tcr.Mode(tcr.SHUFFLE_TREE, block_threads=1024, dtype=tcr.F32)},
        {"n": 3000, "mode": f32})


def test_fixed_descriptor_is_the_balanced_tree(lib):
    for blk in (32, 256, 1024):
        d = tcr.tcr_order_descriptor(n=(1 << 30) + 5, mode=tcr.Mode(tcr.FIXED_ORDER, block_threads=blk))
        assert d["order"] == tcr.ORDER_BALANCED_TREE and d["segments"] == 1
        assert d["chunk_log2"] == 13 + {32: 0, 256: 3, 1024: 5}[blk]
        assert d["partials"] == -(-((1 << 30) + 5) // (1 << d["chunk_log2"]))
        assert d["launches"] == 2


def test_warp_stream_kernels_launch_one_cta_per_unit(lib):
    # The chunked sums, the one-warp rows, the blocked order and the
    # SHUFFLE_TREE block team launch every work unit as its own CTA (the
    # block scheduler balances the SMs; the bits do not depend on the grid):
    # launch_grid equals the partials of a sum, one CTA per 8 rows of the
    # one-warp rows kernels; packed short rows take at most eight waves.
    for kind in (tcr.MMA_CHAIN, tcr.FIXED_ORDER, tcr.SHUFFLE_TREE):
        d = tcr.tcr_order_descriptor(n=1 << 30, mode=tcr.Mode(kind))
        assert d["launch_grid"] == d["partials"] > 152 * 8
        d = tcr.tcr_order_descriptor(rows=65536, cols=4096, mode=tcr.Mode(kind))
        assert (d["launch_grid"], d["launch_block"], d["partials"]) == (65536 // 8, 256, 0)
    # the declared SHUFFLE_TREE team of a 2^30 sum: about 16 vectors per
    # thread, no cap at one wave of resident blocks
    d = tcr.tcr_order_descriptor(n=1 << 30, mode=tcr.Mode(tcr.SHUFFLE_TREE))
    assert (d["team_threads"], d["team_blocks"]) == (256, (1 << 27) // (256 * 16))
    # blocked order: a sum's chunks, and rows of at most 16 runs, 8 warp rounds a CTA
    d = tcr.tcr_order_descriptor(n=1 << 30, mode=tcr.Mode(tcr.FIXED_ORDER, run_log2=8))
    assert d["launch_grid"] == d["partials"]
    d = tcr.tcr_order_descriptor(rows=65536, cols=4096, mode=tcr.Mode(tcr.FIXED_ORDER, run_log2=8))
    assert d["launch_grid"] == 65536 // 2 // 8 and d["partials"] == 0


def test_mma_descriptor_defaults_R_by_block(lib):
    for blk in (32, 64, 128, 256, 512, 1024):
        d = tcr.tcr_order_descriptor(n=1 << 20, mode=tcr.Mode(tcr.MMA_CHAIN, block_threads=blk))
        assert d["chain_R"] == spec.default_R(blk)
        assert d["order"] == tcr.ORDER_TENSOR_CORE
    d = tcr.tcr_order_descriptor(n=1 << 20, mode=tcr.Mode(tcr.MMA_CHAIN, R=5))
    assert d["chain_R"] == 5


def test_rows_descriptor_short_rows_need_no_scratch(lib):
    for kind in (tcr.FIXED_ORDER, tcr.MMA_CHAIN, tcr.SHUFFLE_TREE):
        d = tcr.tcr_order_descriptor(rows=65536, cols=4096, mode=tcr.Mode(kind))
        assert d["partials"] == 0 and d["launches"] == 1 and d["segments"] == 65536


def test_device_faults_rejects_null(lib):
    assert lib.tcr_device_faults(None, 0) == tcr.ERR_INVALID_ARG


def test_python_binding_fails_loudly_without_cuda_tensors():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        tcr.tcr_reduce_sum(torch.zeros(4, dtype=torch.float16), tcr.Mode(tcr.FIXED_ORDER))


def test_blocked_order_arguments(lib):
    ok = tcr.Mode(tcr.FIXED_ORDER, run_log2=4)
    d = tcr.tcr_order_desc()
    assert lib.tcr_order_descriptor(1000, 0, 0, ok, ctypes.byref(d)) == tcr.OK
    for bad in (tcr.Mode(tcr.FIXED_ORDER, run_log2=17), tcr.Mode(tcr.FIXED_ORDER, run_log2=-1),
                tcr.Mode(tcr.MMA_CHAIN, run_log2=3), tcr.Mode(tcr.SHUFFLE_TREE, run_log2=2)):
        assert lib.tcr_order_descriptor(1000, 0, 0, bad, ctypes.byref(d)) == tcr.ERR_INVALID_ARG
        assert lib.tcr_reduce_sum(FAKE, 10, FAKE, bad, None) == tcr.ERR_INVALID_ARG
    # sums of squares have no blocked order: refused before any GPU work
    assert lib.tcr_reduce_sum_squares(FAKE, 10, FAKE, ok, None) == tcr.ERR_UNSUPPORTED
    assert lib.tcr_reduce_rows_sum_squares(FAKE, 3, 10, FAKE, ok, None) == tcr.ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", [tcr.F16, tcr.F32])
def test_blocked_order_descriptors(lib, dtype):
    V = spec.vector_len(dtype)
    for c in range(0, 17):
        d = tcr.tcr_order_descriptor(n=1 << 28, mode=tcr.Mode(tcr.FIXED_ORDER, run_log2=c, dtype=dtype))
        assert d["order"] == (tcr.ORDER_BLOCKED_TREE if c else tcr.ORDER_BALANCED_TREE)
        assert d["run_log2"] == c
        if (1 << c) > V:
            # a warp span holds whole rounds of 32 runs: chunk >= 32 runs
            assert d["chunk_log2"] >= c + 5
            assert d["launch_block"] <= 256
        else:
            assert d["chunk_log2"] == spec.span_log2(dtype) + 3     # the tree's chunk at 256 threads
        assert d["partials"] == -(-(1 << 28) // (1 << d["chunk_log2"]))


def test_blocked_order_equivalence(lib):
    def m(c, **kw):
        return {"n": 100_000, "mode": tcr.Mode(tcr.FIXED_ORDER, run_log2=c, **kw)}
    assert tcr.tcr_order_equivalent(m(0), m(1))                  # runs of two are the pairs
    assert not tcr.tcr_order_equivalent(m(0), m(2))
    assert not tcr.tcr_order_equivalent(m(5), m(6))
    assert tcr.tcr_order_equivalent(m(5), m(5, block_threads=32))    # the CTA size never matters
    assert tcr.tcr_order_equivalent(m(16), m(16, block_threads=1024))
    # one run covering the segment (2^17 > 100 000): every longer run is the same sum
    short = {"n": 1000, "mode": tcr.Mode(tcr.FIXED_ORDER, run_log2=10)}
    longer = {"n": 1000, "mode": tcr.Mode(tcr.FIXED_ORDER, run_log2=16)}
    assert tcr.tcr_order_equivalent(short, longer)
    assert not tcr.tcr_order_equivalent(short, {"n": 1000, "mode": tcr.Mode(tcr.FIXED_ORDER, run_log2=9)})


def test_moments_reject_bad_arguments(lib):
    m = tcr.Mode(tcr.FIXED_ORDER)
    for fn in (lib.tcr_reduce_rows_moments, lib.tcr_reduce_rows_mean_var):
        assert fn(FAKE, 3, 5, FAKE, None, m, None) == tcr.ERR_INVALID_ARG        # second output NULL
        assert fn(FAKE, 3, 5, None, FAKE, m, None) == tcr.ERR_INVALID_ARG
        assert fn(FAKE, 3, 5, FAKE, FAKE + 2, m, None) == tcr.ERR_INVALID_ARG    # misaligned output
        assert fn(FAKE + 1, 3, 5, FAKE, FAKE, m, None) == tcr.ERR_INVALID_ARG    # misaligned input
        assert fn(FAKE, 3, 5, FAKE, FAKE, tcr.Mode(tcr.MMA_CHAIN, R=9), None) == tcr.ERR_INVALID_ARG
        assert fn(FAKE, 1 << 21, 1 << 21, FAKE, FAKE, m, None) == tcr.ERR_INVALID_ARG
        assert fn(FAKE, 3, 5, FAKE, FAKE, tcr.Mode(tcr.FIXED_ORDER, run_log2=2), None) == \
            tcr.ERR_UNSUPPORTED
        assert fn(None, 0, 5, None, None, m, None) == tcr.OK                    # no rows


def test_gemm_descriptor_rule(lib):
    for (M, N, K, S) in ((4096, 4096, 4096, 0), (1024, 1024, 8192, 0), (100, 100, 64, 0),
                         (128, 128, 1000, 0), (64, 64, 8, 5), (2048, 2048, 512, 64)):
        d = tcr.tcr_gemm_descriptor(M, N, K, S)
        assert (d["splits"], d["k_split"]) == spec.gemm_splits(M, N, K, S)
        assert d["combine_order"] == tcr.ORDER_BALANCED_TREE
        assert d["workspace_bytes"] == (d["splits"] * M * N * 4 if d["splits"] > 1 else 0)
        assert d["launches"] == (2 if d["splits"] > 1 else 1)
    bad = tcr.tcr_gemm_desc()
    for args in ((64, 64, 12, 0, 0), (64, 64, 64, 65, 0), (64, 64, 64, -1, 0), (64, 64, 64, 0, 2),
                 (1 << 31, 64, 64, 0, 0)):
        assert lib.tcr_gemm_descriptor(*args, ctypes.byref(bad)) == tcr.ERR_INVALID_ARG
    assert lib.tcr_gemm_splitk(FAKE, FAKE, FAKE, 8, 8, 12, 0, 0, None) == tcr.ERR_INVALID_ARG
    assert lib.tcr_gemm_splitk(FAKE + 8, FAKE, FAKE, 8, 8, 16, 0, 0, None) == tcr.ERR_INVALID_ARG
    assert lib.tcr_gemm_splitk(FAKE, FAKE, FAKE + 2, 8, 8, 16, 0, 0, None) == tcr.ERR_INVALID_ARG



def test_small_inputs_get_smaller_ctas(lib):
    # FIXED_ORDER (bits independent of the CTA size) and default-size MMA_CHAIN:
    # a sum of at most 2^17 inputs is one CTA (spans of one 2^11-input group,
    # two above 2^16 inputs; as few warps as cover it), one launch; larger
    # ones halve the CTA, from the requested (or default 256) size, then the
    # warp span (2^13 inputs down to one group), until there are 2 x 152
    # work units of span x warps inputs or neither can shrink; a caller's
    # MMA_CHAIN block size is kept
    def expected(n, blk):
        if n <= 1 << 17:
            span = 12 if n > 1 << 16 else 11
            warps = 1
            while warps << span < n:
                warps *= 2
            return 32 * warps, span + warps.bit_length() - 1
        span = 13
        while -(-n // ((1 << span) * (blk // 32))) < 304:
            if blk > 32:
                blk //= 2
            elif span > 11:
                span -= 1
            else:
                break
        return blk, span + (blk // 32).bit_length() - 1
    for n in (1, 5000, 1 << 14, 1 << 17, (1 << 17) + 1, 1 << 20, 1 << 22, 1 << 24, 1 << 26, 1 << 30):
        for m, start in ((tcr.Mode(tcr.FIXED_ORDER), 256),
                         (tcr.Mode(tcr.FIXED_ORDER, block_threads=1024), 1024),
                         (tcr.Mode(tcr.MMA_CHAIN), 256)):
            d = tcr.tcr_order_descriptor(n=n, mode=m)
            assert (d["launch_block"], d["chunk_log2"]) == expected(n, start), (n, m)
    d = tcr.tcr_order_descriptor(n=1 << 20, mode=tcr.Mode(tcr.FIXED_ORDER))
    assert (d["launch_block"], d["chunk_log2"], d["partials"]) == (32, 11, 512)
    d = tcr.tcr_order_descriptor(n=1 << 14, mode=tcr.Mode(tcr.MMA_CHAIN))
    assert (d["launch_block"], d["chunk_log2"], d["partials"], d["launches"]) == (256, 14, 0, 1)
    d = tcr.tcr_order_descriptor(n=100_000, mode=tcr.Mode(tcr.FIXED_ORDER))
    assert (d["launch_block"], d["chunk_log2"], d["partials"], d["launches"]) == (1024, 17, 0, 1)
    d = tcr.tcr_order_descriptor(n=1 << 20, mode=tcr.Mode(tcr.MMA_CHAIN, block_threads=256))
    assert (d["launch_block"], d["chunk_log2"]) == (256, 16)


def test_tcgen05_units_shrink_for_small_inputs(lib):
    # the tcgen05 sum's work unit is 2^16 inputs (one unit, one launch, up to
    # 2^16 inputs), above that halved while it leaves fewer than 152 / 2
    # units, down to one 2048-input tile
    def expected(n):
        l = 16
        while n > 1 << 16 and l > 11 and -(-n // (1 << l)) < 76:
            l -= 1
        return l, -(-n // (1 << l))
    for n in (1, 2048, 1 << 16, (1 << 16) + 1, 100_000, 1 << 20, 1 << 24, 1 << 26, 1 << 30):
        d = tcr.tcr_order_descriptor(n=n, mode=tcr.Mode(tcr.MMA_CHAIN_TMEM))
        l, units = expected(n)
        assert d["chunk_log2"] == l, n
        assert d["partials"] == (units if units > 1 else 0), n
    assert tcr.tcr_order_descriptor(n=1 << 20, mode=tcr.Mode(tcr.MMA_CHAIN_TMEM))["chunk_log2"] == 13
    assert tcr.tcr_order_descriptor(n=1 << 30, mode=tcr.Mode(tcr.MMA_CHAIN_TMEM))["chunk_log2"] == 16


def test_tmem_rows_plan(lib):
    # the tcgen05 rows kernels (192 threads).  Rows of 1024 k columns, k a
    # divisor or a multiple of 16, are read as one flat array: a unit is
    # 65536 / cols whole rows (65536 inputs) or a 65536-column chunk of a
    # longer row (per-row partials and a combine), one CTA per unit.  Other
    # rows: units of 16 rows x the whole row up to 8192 columns (32 rows for
    # rows of 768..1024 inputs), longer rows in 8192-column chunks, at most
    # one CTA per SM.  Rows under 768 inputs and rows that are not whole
    # 16-byte vectors go to the mma.sync kernels.  (Without a device the
    # plan assumes 152 SMs.)
    def plan(rows, cols):
        d = tcr.tcr_order_descriptor(rows=rows, cols=cols, mode=tcr.Mode(tcr.MMA_CHAIN_TMEM))
        return d["launch_block"], d["launch_grid"], d["partials"], d["launches"]

    assert plan(1000, 4096) == (192, 63, 0, 1)              # 63 units of 16 rows
    assert plan(65536, 4096) == (192, 4096, 0, 1)           # one CTA per unit
    assert plan(65, 1024) == (192, 2, 0, 1)                 # 64 rows a unit
    assert plan(10, 16384) == (192, 3, 0, 1)                # 4 rows a unit
    assert plan(9, 49152) == (192, 9, 0, 1)                 # a row a unit
    assert plan(100, 131072) == (192, 200, 200, 2)          # 2 chunks per row
    assert plan(3000, 768) == (192, 94, 0, 1)               # two row groups per unit
    assert plan(3000, 3072) == (192, 152, 0, 1)             # 3 groups a row: 16-row tiles
    assert plan(100, 20000) == (192, 21, 300, 2)            # 3 chunks per row
    assert plan(100, 512)[0] == 256                         # packed mma.sync rows
    assert plan(1000, 4100)[0] == 256                       # not whole vectors
