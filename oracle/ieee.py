"""IEEE-754 binary16 and bfloat16 <-> fp64, written from the format definitions.

Part of the CPU oracle (test infrastructure; see oracle/__init__.py).

binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits (the upper half of binary32).

A finite value with biased exponent e and fraction f is
    (-1)^s * (2^p + f) * 2^(e - bias - p)     if e > 0   (normal)
    (-1)^s * f         * 2^(1 - bias - p)     if e == 0  (subnormal)
with p the number of fraction bits; e == all-ones encodes inf (f == 0) or NaN.

Encoding rounds to nearest, ties to even, on the integer significand of the
target format: the value divided by the quantum of its binade is rounded to an
integer; a carry out of the significand moves to the next binade by ordinary
integer addition on the bit pattern; results at or above 2^emax * (2 - 2^-p)
rounded up become inf.
"""
from __future__ import annotations

import numpy as np

FORMATS = {
    # name: (exponent bits, fraction bits, bias)
    "f16": (5, 10, 15),
    "bf16": (8, 7, 127),
}


def _fmt(dtype: str):
    try:
        return FORMATS[dtype]
    except KeyError:
        raise ValueError(f"unknown dtype {dtype!r}") from None


def t_decode(bits, dtype: str) -> np.ndarray:
    """16-bit patterns -> exact fp64 values (every binary16/bfloat16 value is exact in fp64)."""
    eb, p, bias = _fmt(dtype)
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> p) & ((1 << eb) - 1)
    f = (b & ((1 << p) - 1)).astype(np.float64)
    emax = (1 << eb) - 1
    normal = sign * np.ldexp((1 << p) + f, (e - bias - p).astype(np.int64))
    sub = sign * np.ldexp(f, np.full(e.shape, 1 - bias - p, dtype=np.int64))
    special = np.where(f == 0, sign * np.inf, np.nan)
    out = np.where(e == 0, sub, np.where(e == emax, special, normal))
    return out.astype(np.float64)


def t_encode_rne(x, dtype: str) -> np.ndarray:
    """fp64 values -> 16-bit patterns, rounded to nearest with ties to even (one rounding)."""
    eb, p, bias = _fmt(dtype)
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.int64)
    sign_bit = np.signbit(x).astype(np.int64) << 15
    a = np.abs(x)
    emax_field = (1 << eb) - 1
    nan = np.isnan(x)
    inf = np.isinf(a)
    finite = ~(nan | inf)
    nz = finite & (a > 0)
    if np.any(nz):
        av = a[nz]
        # binade exponent: av = m * 2^E with m in [0.5, 1)  =>  floor(log2 av) = E - 1
        _, E = np.frexp(av)
        e_unb = E.astype(np.int64) - 1
        emin = 1 - bias                      # smallest normal exponent
        e_unb = np.maximum(e_unb, emin)      # subnormals share the quantum of the smallest binade
        quantum_exp = e_unb - p
        sig = np.ldexp(av, -quantum_exp)     # exact: scaling by a power of two
        r = np.rint(sig).astype(np.int64)    # round half to even (IEEE default rounding)
        normal_binade = (E.astype(np.int64) - 1) >= emin
        # normal: (biased exponent << p) + (r - 2^p); subnormal: r (exponent field 0)
        bits = np.where(normal_binade, ((e_unb + bias) << p) + (r - (1 << p)), r)
        bits = np.where(bits >= (emax_field << p), emax_field << p, bits)   # overflow -> inf
        out[nz] = bits
    out[inf] = emax_field << p
    out[nan] = (emax_field << p) | (1 << (p - 1))     # quiet NaN
    out = out | sign_bit
    return (out & 0xFFFF).astype(np.uint16)


def t_unit_roundoff(dtype: str) -> float:
    """u = 2^-(p+1): the largest relative rounding error for normal results."""
    _, p, _ = _fmt(dtype)
    return 2.0 ** -(p + 1)


def t_min_subnormal(dtype: str) -> float:
    eb, p, bias = _fmt(dtype)
    return 2.0 ** (1 - bias - p)
