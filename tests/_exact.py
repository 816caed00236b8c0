"""Exact arithmetic for pinning the oracle: rationals, and rounding to a
storage dtype by brute force (search of the sorted list of every finite value
of the format), written from the IEEE-754 definitions alone.

Nothing here is shared with the oracle or the CUDA library.
"""
from __future__ import annotations

import bisect
from decimal import Decimal, getcontext
from fractions import Fraction
from functools import lru_cache

import numpy as np

getcontext().prec = 80


def bf16_value(bits: int) -> Fraction:
    """Exact value of a bf16 bit pattern (1 sign, 8 exponent, 7 fraction bits).
    Raises for inf/NaN patterns."""
    s, e, f = (bits >> 15) & 1, (bits >> 7) & 0xFF, bits & 0x7F
    if e == 0xFF:
        raise ValueError("not finite")
    v = Fraction(f, 1 << 133) if e == 0 else Fraction(128 + f) * Fraction(2) ** (e - 134)
    return -v if s else v


def fp16_value(bits: int) -> Fraction:
    """Exact value of a binary16 bit pattern (1, 5, 10)."""
    s, e, f = (bits >> 15) & 1, (bits >> 10) & 0x1F, bits & 0x3FF
    if e == 0x1F:
        raise ValueError("not finite")
    v = Fraction(f, 1 << 24) if e == 0 else Fraction(1024 + f) * Fraction(2) ** (e - 25)
    return -v if s else v


@lru_cache(maxsize=None)
def _grid(dtype: str):
    """Sorted (values, bits) of every finite non-negative value of the format."""
    value = bf16_value if dtype == "bf16" else fp16_value
    top = 0x7F80 if dtype == "bf16" else 0x7C00
    bits = list(range(0, top))
    vals = [value(b) for b in bits]
    return vals, bits


def round_to(q: Fraction, dtype: str) -> int:
    """Bit pattern of the value of `dtype` nearest to q, ties to the even bit
    pattern (IEEE round-to-nearest-even).  q must be inside the finite range."""
    if dtype == "fp32":
        return round_to_fp32(q)
    vals, bits = _grid(dtype)
    a = abs(q)
    i = bisect.bisect_left(vals, a)
    if i == len(vals):
        raise OverflowError
    if vals[i] == a:
        k = bits[i]
    else:
        lo, hi = i - 1, i
        dlo, dhi = a - vals[lo], vals[hi] - a
        if dlo < dhi or (dlo == dhi and bits[lo] % 2 == 0):
            k = bits[lo]
        else:
            k = bits[hi]
    if q < 0:
        k |= 0x8000
    return k


def round_to_fp32(q: Fraction) -> int:
    """Bit pattern (as uint32) of the float32 nearest to q, ties to even:
    the candidates are the float32 next to float(q) and its two neighbours,
    compared by exact distance."""
    c = np.float32(float(q))
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = None
    for x in cands:
        if not np.isfinite(x):
            continue
        d = abs(Fraction(float(x)) - q)
        b = int(np.array([x], dtype=np.float32).view(np.uint32)[0])
        key = (d, b % 2)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def value_of(bits: int, dtype: str) -> Fraction:
    if dtype == "bf16":
        return bf16_value(bits)
    if dtype == "fp16":
        return fp16_value(bits)
    return Fraction(float(np.array([bits], dtype=np.uint32).view(np.float32)[0]))


def ulp_distance(a_bits: int, b_bits: int, dtype: str) -> int:
    """Distance between two finite patterns along the ordered line of values."""
    width = 32 if dtype == "fp32" else 16
    sign = 1 << (width - 1)

    def ordered(b):
        return -(b & (sign - 1)) if b & sign else b

    return abs(ordered(a_bits) - ordered(b_bits))


def ulp_at(q: Fraction, dtype: str) -> Fraction:
    """Spacing of the dtype's values at magnitude |q| (the larger spacing at a
    power of two)."""
    mant = {"bf16": 8, "fp16": 11, "fp32": 24}[dtype]
    emin = {"bf16": -126, "fp16": -14, "fp32": -126}[dtype]
    a = abs(q)
    if a == 0:
        return Fraction(2) ** (emin - mant + 1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    return Fraction(2) ** (e - mant + 1)


def sqrt_fraction(q: Fraction) -> Fraction:
    """sqrt(q) to 80 significant decimal digits, as an exact Fraction of that
    decimal."""
    d = (Decimal(q.numerator) / Decimal(q.denominator)).sqrt()
    return Fraction(d)


def words(t) -> list:
    """Storage words of a torch tensor / numpy array as Python ints
    (uint16 for 2-byte dtypes, uint32 for fp32)."""
    import torch
    if isinstance(t, torch.Tensor):
        t = t.contiguous()
        if t.element_size() == 2:
            return [int(v) & 0xFFFF for v in t.view(torch.int16).reshape(-1).tolist()]
        return [int(v) & 0xFFFFFFFF for v in t.view(torch.int32).reshape(-1).tolist()]
    a = np.ascontiguousarray(t)
    if a.dtype.itemsize == 2:
        return [int(v) for v in a.view(np.uint16).reshape(-1)]
    return [int(v) for v in a.view(np.uint32).reshape(-1)]
