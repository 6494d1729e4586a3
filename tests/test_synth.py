"""The seeded input generator: determinism and its SplitMix64 definition."""
import numpy as np

from arithmetic_reduction_tensor_gb300 import synth

MASK = (1 << 64) - 1


def splitmix64_stream(state, count):
    """SplitMix64 as published: state += gamma, then the output mix."""
    out = []
    for _ in range(count):
        state = (state + 0x9E3779B97F4A7C15) & MASK
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def test_words_are_a_splitmix64_stream():
    for seed in (0, 1, 4):
        start_state = ((seed << 40) * 0x9E3779B97F4A7C15) & MASK
        ref = splitmix64_stream(start_state, 50)
        assert [int(w) for w in synth._words(seed, 0, 50)] == ref


def test_slices_are_independent_of_chunking():
    full = synth.generate(3 * (1 << 22) + 77, "normal", synth.F16, seed=2, threads=3)
    part = synth.generate(1000, "normal", synth.F16, seed=2, start=(1 << 22) - 501)
    assert np.array_equal(full[(1 << 22) - 501:(1 << 22) + 499], part)


def test_distributions_have_the_stated_ranges():
    u = synth.as_float(synth.generate(1 << 18, "uniform_pm1", synth.F16, seed=0), synth.F16)
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 0.01
    u = synth.as_float(synth.generate(1 << 18, "uniform01", synth.F16, seed=1), synth.F16)
    assert u.min() >= 0 and u.max() <= 1 and abs(u.mean() - 0.5) < 0.01
    z = synth.as_float(synth.generate(1 << 18, "normal", synth.F16, seed=2), synth.F16)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    for dt in (synth.F16, synth.BF16):
        p = synth.as_float(synth.generate(1 << 18, "pow2", dt, seed=3), dt)
        e = np.log2(np.abs(p))
        assert np.all(e == np.round(e)) and e.min() == -20 and e.max() == 10


def test_binary32_patterns_round_the_same_binary64_values():
    # the binary32 stream is the binary64 values of the 16-bit streams,
    # rounded once to binary32 instead of to 16 bits
    for dist in ("uniform_pm1", "uniform01", "normal"):
        b32 = synth.generate(4096, dist, synth.F32, seed=5)
        assert b32.dtype == np.uint32
        f32 = b32.view(np.float32)
        f16 = synth.as_float(synth.generate(4096, dist, synth.F16, seed=5), synth.F16)
        via32 = f32.astype(np.float16).astype(np.float32)
        # rounding twice (64 -> 32 -> 16) may differ from once only where the
        # binary32 value lies exactly halfway between two binary16 values
        differ = via32 != f16
        assert differ.sum() <= 4
        lo = np.minimum(via32, f16)[differ].astype(np.float64)
        hi = np.maximum(via32, f16)[differ].astype(np.float64)
        assert np.array_equal(f32[differ].astype(np.float64), (lo + hi) / 2)
    p = synth.as_float(synth.generate(1 << 16, "pow2", synth.F32, seed=3), synth.F32)
    p16 = synth.as_float(synth.generate(1 << 16, "pow2", synth.F16, seed=3), synth.F16)
    assert np.array_equal(p, p16)


def test_exact_int_vectors_sum_to_one_and_open_with_a_pair():
    for dt, V, lo, hi in ((synth.F16, 8, 1024, 2047), (synth.BF16, 8, 128, 255 << 8),
                          (synth.F32, 4, 1 << 19, (1 << 20) - 1)):
        b = synth.generate(3 * (1 << 22) + 5 * V, "exact_int", dt, seed=7)
        f = synth.as_float(b, dt).astype(np.float64).reshape(-1, V)
        assert np.all(f == np.round(f))                 # integers, exact in the type
        assert set(np.unique(f.sum(axis=1))) == {-1.0, 1.0}
        assert np.array_equal(f[:, 1], -f[:, 0])
        a = np.abs(f[:, 0])
        assert a.min() >= lo and a.max() <= hi
        assert np.all(np.abs(f[:, 2:V - 1]) <= 4)
        # slices that start inside a vector give the same elements
        part = synth.generate(1001, "exact_int", dt, seed=7, start=(1 << 22) - 3)
        assert np.array_equal(part, b[(1 << 22) - 3:(1 << 22) + 998])


def test_exact_int_split_parts_all_in_use():
    # the binary32 a's have 20 significant bits: truncated to bfloat16 (hi)
    # they leave a residual whose top 8 bits (mid) and the rest (lo) are both
    # nonzero for most a (lo for about 4 in 5)
    b = synth.generate(1 << 16, "exact_int", synth.F32, seed=8).reshape(-1, 4)[:, 0]
    hi = b & np.uint32(0xFFFF0000)
    r = b.view(np.float32).astype(np.float64) - hi.view(np.float32).astype(np.float64)
    mid = (np.abs(r).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    lo = np.abs(r) - mid
    assert np.mean(r != 0) > 0.99 and np.mean(lo != 0) > 0.75


def test_exact_int_dropping_or_repeating_a_vector_changes_the_sum():
    import oracle
    b = synth.generate(1 << 16, "exact_int", synth.F16, seed=9)
    total, _ = oracle.exact_sum(b, synth.F16)
    rng = np.random.default_rng(0)
    for v in rng.integers(0, (1 << 16) // 8, 20):
        dropped = np.concatenate([b[:8 * v], b[8 * v + 8:]])
        repeated = np.concatenate([b[:8 * v + 8], b[8 * v:]])
        assert abs(oracle.exact_sum(dropped, synth.F16)[0] - total) == 1
        assert abs(oracle.exact_sum(repeated, synth.F16)[0] - total) == 1
