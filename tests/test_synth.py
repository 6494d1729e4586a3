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
