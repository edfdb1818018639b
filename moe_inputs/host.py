"""Host (numpy) twin of the seeded input generator.

The generator is counter based, so any element of any tensor can be drawn on its own, and
it uses only IEEE-754 basic operations (+, -, *, /, sqrt) plus exact bit manipulation.
The CUDA twin in ``csrc/gen.cu`` performs the same operations in the same order with
explicitly rounded intrinsics, so both produce bit-identical tensors.  This module holds
no arithmetic of the MoE layer itself.

Recipe for element ``i`` (flat row-major index) of tensor ``tid`` under ``seed``:

* splitmix64 (Steele, Lea & Flood 2014; Vigna's constants): ``mix64`` finaliser,
  stream key ``key = mix64(mix64((seed+1)*G) ^ ((tid+1)*G))``, word ``n`` of the stream is
  ``mix64(key + (n+1)*G)`` with ``G = 0x9E3779B97F4A7C15`` (all mod 2**64).
* uniform ``U = (word >> 11) * 2**-53`` in [0, 1).
* normal: Marsaglia & Bray's polar method.  Attempt ``a`` (0..63) draws words
  ``n = 2*(64*i + a)`` and ``n+1``, ``u = 2U-1``, ``v = 2U-1``, ``s = u*u + v*v``; the first
  attempt with ``0 < s < 1`` gives ``z = u * sqrt(-2 ln(s) / s)``.
* ``ln`` is computed here (not by a libm): ``s = m * 2**e`` by frexp, ``m`` moved into
  [1/sqrt2, sqrt2), then ``ln m = 2 atanh(t)``, ``t = (m-1)/(m+1)``, summed as the odd power
  series of atanh (Abramowitz & Stegun 4.1.27) with 13 terms in Horner form, plus ``e*ln2``.
* value ``z * std`` in fp64, rounded to fp32 (round to nearest even), then for bf16
  tensors rounded again from fp32 to bf16 (round to nearest even).
* uniform(lo, hi) tensors: ``lo + (hi - lo) * U`` in fp64, rounded to fp32.
"""
import numpy as np

_MASK = (1 << 64) - 1
_G = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

LN2 = float.fromhex("0x1.62e42fefa39efp-1")         # ln 2 rounded to nearest double
SQRT_HALF = float.fromhex("0x1.6a09e667f3bcdp-1")   # 1/sqrt(2) rounded to nearest double
N_ATANH = 12                                         # highest power index of the series
ATANH_COEF = [1.0 / (2 * n + 1) for n in range(N_ATANH + 1)]
MAX_ATTEMPTS = 64


def _mix64_int(z):
    z &= _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def stream_key(seed, tid):
    k0 = _mix64_int(((seed + 1) * _G) & _MASK)
    return _mix64_int(k0 ^ (((tid + 1) * _G) & _MASK))


def _mix64(z):
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def words(key, n):
    """Stream words ``n`` (uint64 array) of the stream with the given key."""
    n = np.asarray(n, dtype=np.uint64)
    return _mix64(np.uint64(key) + (n + np.uint64(1)) * np.uint64(_G))


def unit(w):
    """53-bit uniform in [0, 1) from a uint64 word."""
    return (w >> np.uint64(11)).astype(np.float64) * float.fromhex("0x1p-53")


def ln_series(s):
    """Natural log of positive fp64 values using only basic IEEE operations."""
    s = np.asarray(s, dtype=np.float64)
    m, e = np.frexp(s)
    small = m < SQRT_HALF
    m = np.where(small, m * 2.0, m)
    e = np.where(small, e - 1, e)
    t = (m - 1.0) / (m + 1.0)
    w = t * t
    p = np.full_like(t, ATANH_COEF[N_ATANH])
    for n in range(N_ATANH - 1, -1, -1):
        p = p * w + ATANH_COEF[n]
    return e.astype(np.float64) * LN2 + (2.0 * t) * p


def normal_f64(idx, seed, tid):
    """Standard normal fp64 values for the flat element indices ``idx``."""
    idx = np.asarray(idx, dtype=np.uint64).ravel()
    key = stream_key(seed, tid)
    out = np.zeros(idx.shape, dtype=np.float64)
    pending = np.arange(idx.size)
    for a in range(MAX_ATTEMPTS):
        if pending.size == 0:
            break
        n1 = (idx[pending] * np.uint64(MAX_ATTEMPTS) + np.uint64(a)) * np.uint64(2)
        u = 2.0 * unit(words(key, n1)) - 1.0
        v = 2.0 * unit(words(key, n1 + np.uint64(1))) - 1.0
        s = u * u + v * v
        ok = (s < 1.0) & (s > 0.0)
        sel = pending[ok]
        uo, so = u[ok], s[ok]
        out[sel] = uo * np.sqrt((-2.0 * ln_series(so)) / so)
        pending = pending[~ok]
    return out


def f32_to_bf16_bits(f):
    """Round fp32 to bf16 (nearest even); returns uint16 bit patterns."""
    b = np.asarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal(idx, seed, tid, std, dtype):
    """Element values: fp32 array, or uint16 bf16 bit patterns for dtype 'bf16'."""
    v = (normal_f64(idx, seed, tid) * float(std)).astype(np.float32)
    return f32_to_bf16_bits(v) if dtype == "bf16" else v


def uniform_f32(idx, seed, tid, lo, hi):
    idx = np.asarray(idx, dtype=np.uint64).ravel()
    u = unit(words(stream_key(seed, tid), idx))
    return (lo + (hi - lo) * u).astype(np.float32)


def tensor_normal(shape, seed, tid, std, dtype):
    n = int(np.prod(shape))
    return normal(np.arange(n, dtype=np.uint64), seed, tid, std, dtype).reshape(shape)


def zipf_offsets(E, seed, s, scale):
    """Per-expert additive logit offsets ``scale * ln(r**-s)`` over a seeded permutation.

    Rank ``r`` (1-based) goes to expert ``perm[r-1]``; ``perm`` is a Fisher-Yates shuffle
    drawn from the stream of ``TID_ZIPF_PERM``.  Returns fp32 offsets indexed by expert.
    """
    from .configs import TID_ZIPF_PERM
    key = stream_key(seed, TID_ZIPF_PERM)
    perm = list(range(E))
    for i in range(E - 1, 0, -1):
        u = float(unit(words(key, np.array([i], dtype=np.uint64)))[0])
        j = int(u * (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    ranks = np.arange(1, E + 1, dtype=np.float64)
    off = scale * (-s * ln_series(ranks))
    out = np.zeros(E, dtype=np.float64)
    for r in range(E):
        out[perm[r]] = off[r]
    return out.astype(np.float32), perm
