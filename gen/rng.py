"""Counter-based random numbers: SplitMix64 output mixing over (seed, stream, index).

Every value is a pure function of (seed, stream, index), so any element of any
tensor can be regenerated on its own, in any order, on any machine.

Definition (SplitMix64 finaliser, Steele, Lea and Flood 2014, with Vigna's
constants):

    mix(z)   = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^ (z >> 31)
    key      = mix(seed ^ (stream * 0xD1B54A32D192ED03))
    x(index) = mix(key + (index + 1) * 0x9E3779B97F4A7C15)      (all mod 2**64)

    uniform  = (x >> 11) * 2**-53                                in [0, 1)
    normal i = sqrt(-2 ln(1 - u(2i))) * cos(2 pi u(2i+1))        (Box-Muller)
"""
import numpy as np

_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_STREAM = np.uint64(0xD1B54A32D192ED03)


def _mix(z):
    z = z ^ (z >> np.uint64(30))
    z = z * _M1
    z = z ^ (z >> np.uint64(27))
    z = z * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_stream(seed, stream, index):
    """Raw 64-bit words for the given indices (uint64 array or scalar)."""
    with np.errstate(over="ignore"):
        s = np.array([seed], dtype=np.uint64) ^ (np.array([stream], dtype=np.uint64) * _STREAM)
        key = _mix(s)[0]
        idx = np.asarray(index, dtype=np.uint64)
        return _mix(key + (idx + np.uint64(1)) * _GOLDEN)


def uniform(seed, stream, n, offset=0):
    """n doubles in [0, 1) for indices offset .. offset+n-1."""
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    x = splitmix64_stream(seed, stream, idx)
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


_CHUNK = 1 << 20


def normal(seed, stream, n, sigma=1.0, offset=0):
    """n standard normals (times sigma) in double, Box-Muller over index pairs
    offset .. offset+n-1. Large requests are computed in chunks on a thread
    pool (numpy releases the GIL); every value depends on its index only, so
    the result is the same as in one piece."""
    if n > 2 * _CHUNK:
        from concurrent.futures import ThreadPoolExecutor
        import os
        out = np.empty(n, dtype=np.float64)

        def fill(lo):
            hi = min(n, lo + _CHUNK)
            out[lo:hi] = normal(seed, stream, hi - lo, sigma, offset + lo)
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(0, n, _CHUNK)))
        return out
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        u1 = (splitmix64_stream(seed, stream, idx * np.uint64(2)) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u2 = (splitmix64_stream(seed, stream, idx * np.uint64(2) + np.uint64(1)) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log1p(-u1))
    return sigma * r * np.cos(2.0 * np.pi * u2)
