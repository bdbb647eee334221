"""Counter-based random numbers for the synthetic inputs (host side).

Every random input of the paged-attention workloads is a pure function of
(seed, stream, index), so any element (one page of a 5 GB cache, say) can be
regenerated on its own, on the host or on the device, without producing the
rest.  The mixing function is SplitMix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014; constants as in
Vigna's public-domain reference implementation):

    z  = x + 0x9E3779B97F4A7C15
    z  = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z  = (z ^ (z >> 27)) * 0x94D049BB133111EB
    out = z ^ (z >> 31)                      (all arithmetic mod 2^64)

Counter scheme used here:

    key(seed, stream) = splitmix64(splitmix64(seed) ^ stream)
    u64(seed, stream, i) = splitmix64(key ^ i)

Derived draws:
    uniform integer in [lo, hi]:  lo + ((u64 >> 32) * (hi - lo + 1)) >> 32
    uniform real in [0, 1):       (u64 >> 11) * 2^-53
    standard normal (index i):    Box-Muller on the pair (2i, 2i+1),
                                  sqrt(-2 ln(1 - r0)) * cos(2 pi r1)

The device generator in ``synth/csrc/synth_gen.cu`` implements the integer
draw with the same formulas, so its bytes equal these bit for bit.  Normal
draws come from the threaded host library ``synth/csrc/synth_host.c`` (the same
formulas in C, built next to this package) when it is present; its values and
the numpy expression ``normal_np`` below agree to within two ulps (the two
libraries' log1p / cos differ in the last bits), and every input of one run
comes from the same one of the two.

This module holds no attention arithmetic; it is shared by the oracle tests,
the CUDA parity tests and the benchmark as the single source of inputs.
"""
from __future__ import annotations

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)


def splitmix64(x):
    """SplitMix64 finaliser applied elementwise to uint64 input (wraps mod 2^64)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    """Per-(seed, stream) key: splitmix64(splitmix64(seed) ^ stream)."""
    s = splitmix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF))
    return np.uint64(splitmix64(s ^ np.uint64(stream)))


def u64(seed: int, stream: int, idx) -> np.ndarray:
    """Raw 64-bit draws for counters ``idx`` (any integer array)."""
    key = stream_key(seed, stream)
    i = np.asarray(idx, dtype=np.uint64)
    return splitmix64(i ^ key)


def uniform_int(seed: int, stream: int, idx, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on [lo, hi] (multiply-shift on the top 32 bits)."""
    n = np.uint64(hi - lo + 1)
    hi32 = u64(seed, stream, idx) >> np.uint64(32)
    with np.errstate(over="ignore"):
        v = (hi32 * n) >> np.uint64(32)
    return v.astype(np.int64) + lo


def uniform_i8_bytes(seed: int, stream: int, start: int, count: int, lo: int, hi: int) -> np.ndarray:
    """uniform_int draws for counters start .. start+count-1 as two's-complement
    bytes (uint8); the threaded C generator when built (integer arithmetic:
    the same bytes), else numpy."""
    import os
    lib = _host_lib()
    if lib is not None and count > 0 and -128 <= lo <= hi <= 127:
        out = np.empty(count, dtype=np.uint8)
        lib.synth_uniform_i8(seed & 0xFFFFFFFFFFFFFFFF, stream, start, count, lo, hi, out.ctypes.data,
                             min(32, os.cpu_count() or 1))
        return out
    v = uniform_int(seed, stream, np.arange(start, start + count, dtype=np.uint64), lo, hi)
    return np.asarray(v, dtype=np.int64).astype(np.int8).view(np.uint8)


def uniform01(seed: int, stream: int, idx) -> np.ndarray:
    """Reals uniform on [0, 1) with 53 random bits (float64)."""
    return (u64(seed, stream, idx) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform_real(seed: int, stream: int, idx, a: float, b: float) -> np.ndarray:
    return a + (b - a) * uniform01(seed, stream, idx)


def normal_np(seed: int, stream: int, idx) -> np.ndarray:
    """Standard normal draws by Box-Muller on the counter pair (2i, 2i+1)."""
    i = np.asarray(idx, dtype=np.uint64)
    r0 = uniform01(seed, stream, i * np.uint64(2))
    r1 = uniform01(seed, stream, i * np.uint64(2) + np.uint64(1))
    return np.sqrt(-2.0 * np.log1p(-r0)) * np.cos(2.0 * np.pi * r1)


_HOST = None


def _host_lib():
    """The threaded C generator, or None when it has not been built."""
    global _HOST
    if _HOST is None:
        import ctypes
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa_synth_host.so")
        if not os.path.exists(path):
            return None
        lib = ctypes.CDLL(path)
        lib.synth_normal.argtypes = [ctypes.c_uint64] * 4 + [ctypes.c_void_p, ctypes.c_int]
        lib.synth_normal.restype = ctypes.c_int
        lib.synth_uniform_i8.argtypes = [ctypes.c_uint64] * 4 + [ctypes.c_int32, ctypes.c_int32,
                                                                 ctypes.c_void_p, ctypes.c_int]
        lib.synth_uniform_i8.restype = ctypes.c_int
        _HOST = lib
    return _HOST


def normal(seed: int, stream: int, idx) -> np.ndarray:
    """Standard normal draws by Box-Muller on the counter pair (2i, 2i+1).

    Contiguous counter ranges go through the threaded C generator when it is
    built; anything else (or no library) through ``normal_np``."""
    import os
    i = np.asarray(idx, dtype=np.uint64)
    lib = _host_lib()
    if lib is not None and i.ndim == 1 and i.size > 0:
        start = int(i[0])
        if int(i[-1]) - start == i.size - 1 and (i.size < 3 or np.all(np.diff(i) == 1)):
            out = np.empty(i.size, dtype=np.float64)
            lib.synth_normal(seed & 0xFFFFFFFFFFFFFFFF, stream, start, i.size, out.ctypes.data,
                             min(32, os.cpu_count() or 1))
            return out
    return normal_np(seed, stream, i)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of 0..n-1 driven by the counter stream.

    Step k (k = n-1 down to 1) swaps position k with position
    uniform_int(counter = n-1-k, lo = 0, hi = k).
    """
    perm = np.arange(n, dtype=np.int64)
    if n <= 1:
        return perm
    ks = np.arange(n - 1, 0, -1, dtype=np.int64)
    hi32 = (u64(seed, stream, np.arange(n - 1, dtype=np.uint64)) >> np.uint64(32))
    with np.errstate(over="ignore"):
        js = ((hi32 * (ks + 1).astype(np.uint64)) >> np.uint64(32)).astype(np.int64)
    for k, j in zip(ks.tolist(), js.tolist()):
        perm[k], perm[j] = perm[j], perm[k]
    return perm
