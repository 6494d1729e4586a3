"""Seeded synthetic inputs for the reduction tests and benchmark.

This module holds no reduction arithmetic: it only turns (seed, index) into
input patterns (16-bit for binary16 / bfloat16, 32-bit for binary32).  Both the CPU oracle side and the GPU side of every
test consume the same bytes produced here.

Generator (counter based, so any slice can be produced independently):

* word(i) = mix(((seed << 40) + i + 1) * GAMMA mod 2^64), where GAMMA =
  0x9E3779B97F4A7C15 and ``mix`` is the SplitMix64 output function of Steele,
  Lea and Flood, "Fast splittable pseudorandom number generators" (OOPSLA
  2014): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
  z *= 0x94D049BB133111EB; z ^= z >> 31.  word(i) is the (i+1)-th output of
  a SplitMix64 stream whose state starts at (seed << 40) * GAMMA.
* u(i) = (word(i) >> 11) * 2^-53, uniform on [0, 1).

Distributions (the workload recipes of the benchmark configurations):

``uniform_pm1``  2 u(i) - 1, uniform on [-1, 1)
``uniform01``    u(i), uniform on [0, 1)
``normal``       Box-Muller on the pair (u(2k), u(2k+1)):
                 r = sqrt(-2 ln(1 - u(2k))), t = 2 pi u(2k+1);
                 element 2k = r cos t, element 2k+1 = r sin t
``pow2``         sign = bit 63 of word(i); e = -20 + (low 32 bits mod 31);
                 the value is sign * 2^e (exact in every storage type)
``exact_int``    integers built per 16-byte vector (V = 8 inputs of 16 bits,
                 V = 4 of binary32; vector v holds elements V v .. V v + V - 1,
                 each drawing on its own word w = word(i), h = w >> 32):
                 element 0 is a = +-A (sign: bit 63 of w), element 1 is -a;
                 elements 2 .. V - 2 are (h mod 9) - 4; element V - 1 is
                 s - (the sum of elements 2 .. V - 2), s = +1 if bit 63 of
                 its word is set, else -1.  A is 1024 + (h mod 1024) for
                 binary16 (11 significant bits), (128 + (h mod 128)) *
                 2^((h >> 8) mod 9) for bfloat16, and 2^19 + (h mod 2^19)
                 for binary32 (20 significant bits, so a three-way bfloat16
                 split of it has all three parts).  Every vector sums to
                 exactly +-1, so the total is a small integer, dropping or
                 repeating any one vector changes it, and a partial sum that
                 keeps each aligned pair (a, -a) together is an integer far
                 below 2^24: binary32 adds it without rounding in any order.

Rounding to the storage type: binary16 and binary32 take the binary64 value
rounded to nearest even in one step (numpy's casts); bfloat16 takes the
binary64 value rounded to binary32 and then to bfloat16, nearest even at
each step.  ``pow2`` values are exact and need no rounding.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

F16 = 0
BF16 = 1
F32 = 2

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

DISTRIBUTIONS = ("uniform_pm1", "uniform01", "normal", "pow2", "exact_int")


def _words(seed: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    idx += np.uint64((seed << 40) & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        z = idx * GAMMA
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def _uniform(seed: int, start: int, count: int) -> np.ndarray:
    # (word >> 11) < 2^53 fits int64, whose conversion to float64 is exact
    top = (_words(seed, start, count) >> np.uint64(11)).view(np.int64)
    return top.astype(np.float64) * (2.0 ** -53)


def _to_bits(v: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return v.astype(np.float32).view(np.uint32)
    if dtype == F16:
        return v.astype(np.float16).view(np.uint16)
    f = v.astype(np.float32).view(np.uint32)
    # round-to-nearest-even from binary32 to bfloat16 on the bit pattern
    rounded = (f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def _chunk(dist: str, dtype: int, seed: int, start: int, count: int) -> np.ndarray:
    if dist == "uniform_pm1":
        return _to_bits(2.0 * _uniform(seed, start, count) - 1.0, dtype)
    if dist == "uniform01":
        return _to_bits(_uniform(seed, start, count), dtype)
    if dist == "normal":
        # pairs (2k, 2k+1); start is even for every chunk but possibly the caller's
        p0 = start - (start & 1)
        cnt = count + (start & 1)
        cnt += cnt & 1
        u = _uniform(seed, p0, cnt)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = 2.0 * np.pi * u2
        z = np.empty(cnt, np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        return _to_bits(z[start - p0:start - p0 + count], dtype)
    if dist == "pow2":
        w = _words(seed, start, count)
        sign = (w >> np.uint64(63)).astype(np.uint16)
        e = ((w & np.uint64(0xFFFFFFFF)) % np.uint64(31)).astype(np.int32) - 20
        if dtype == F32:
            return ((sign.astype(np.uint32) << np.uint32(31))
                    | ((e + 127).astype(np.uint32) << np.uint32(23)))
        if dtype == BF16:
            return (sign << np.uint16(15)) | ((e + 127).astype(np.uint16) << np.uint16(7))
        # binary16: 2^e is normal for e >= -14 (biased exponent e + 15) and
        # subnormal below (fraction bit e + 24 set)
        normal = (np.maximum(e + 15, 0).astype(np.uint16) << np.uint16(10))
        subnormal = np.left_shift(np.uint16(1), np.clip(e + 24, 0, 15).astype(np.uint16))
        mag = np.where(e >= -14, normal, subnormal).astype(np.uint16)
        return (sign << np.uint16(15)) | mag
    if dist == "exact_int":
        return _exact_int(dtype, seed, start, count)
    raise ValueError(f"unknown distribution {dist!r}")


def _exact_int(dtype: int, seed: int, start: int, count: int) -> np.ndarray:
    V = 4 if dtype == F32 else 8
    p0 = start - start % V                      # whole vectors around the slice
    nv = (start + count - p0 + V - 1) // V
    w = _words(seed, p0, nv * V).reshape(nv, V)
    h = (w >> np.uint64(32)).astype(np.int64)
    neg = (w >> np.uint64(63)).astype(bool)
    v = np.empty((nv, V), np.int64)
    if dtype == F16:
        A = 1024 + h[:, 0] % 1024
    elif dtype == BF16:
        A = (128 + h[:, 0] % 128) << ((h[:, 0] >> 8) % 9)
    else:
        A = (1 << 19) + h[:, 0] % (1 << 19)
    v[:, 0] = np.where(neg[:, 0], -A, A)
    v[:, 1] = -v[:, 0]
    v[:, 2:V - 1] = h[:, 2:V - 1] % 9 - 4
    s = np.where(neg[:, V - 1], 1, -1)
    v[:, V - 1] = s - v[:, 2:V - 1].sum(axis=1)
    flat = v.reshape(-1)[start - p0:start - p0 + count]
    # every value is an integer exact in the storage type: the casts are exact
    return _to_bits(flat.astype(np.float64), dtype)


def generate(n: int, dist: str, dtype: int = F16, seed: int = 0, start: int = 0,
             threads: int | None = None) -> np.ndarray:
    """The patterns of elements ``start .. start+n-1``: uint16 for F16 and
    BF16, uint32 for F32."""
    out = np.empty(n, np.uint32 if dtype == F32 else np.uint16)
    if n == 0:
        return out
    starts = list(range(0, n, _CHUNK))
    nt = threads or max(1, min(len(starts), len(os.sched_getaffinity(0))))

    def work(off: int) -> None:
        c = min(_CHUNK, n - off)
        out[off:off + c] = _chunk(dist, dtype, seed, start + off, c)

    if nt == 1 or len(starts) == 1:
        for off in starts:
            work(off)
    else:
        with ThreadPoolExecutor(nt) as ex:
            list(ex.map(work, starts))
    return out


def as_float(bits: np.ndarray, dtype: int) -> np.ndarray:
    """binary32 view of the patterns, for display and host-side checks."""
    if dtype == F32:
        return bits.view(np.float32)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
