"""Brute-force exact checker in rational arithmetic, for tiny problems. Test infrastructure only.

Independent of oracle/w4a16.py and oracle/ieee.py: it decodes 16-bit floats from
their bit fields with Python integers and Fractions, extracts nibbles with
integer shifts, and sums products exactly. Pure-Python loops: use it only for
problems with a few thousand multiply-adds.

Semantics restated from the PR #40977 report, key source snippets (the test
reference): W = (raw - zero_point) * scale with scale and zero point repeated
group_size times along K; out = A @ W (+ bias).
"""
from __future__ import annotations

from fractions import Fraction

_FIELDS = {"f16": (5, 10, 15), "bf16": (8, 7, 127)}


def decode(bits: int, dtype: str) -> Fraction:
    eb, p, bias = _FIELDS[dtype]
    bits = int(bits) & 0xFFFF
    s = -1 if bits >> 15 else 1
    e = (bits >> p) & ((1 << eb) - 1)
    f = bits & ((1 << p) - 1)
    if e == (1 << eb) - 1:
        raise ValueError("inf/nan has no rational value")
    if e == 0:
        return s * Fraction(f) * Fraction(2) ** (1 - bias - p)
    return s * Fraction((1 << p) + f) * Fraction(2) ** (e - bias - p)


def nibble(word: int, j: int) -> int:
    return ((int(word) & 0xFFFFFFFF) >> (4 * j)) & 0xF


def weight(b_q, scales, qzeros, G, zp_bias, dtype, k, n) -> Fraction:
    q = nibble(b_q[k][n // 8], n % 8)
    g = k // G
    zp = zp_bias if qzeros is None else nibble(qzeros[g][n // 8], n % 8)
    return (q - zp) * decode(scales[g][n], dtype)


def gemm(a, b_q, scales, qzeros, G, zp_bias, bias, dtype):
    """list-of-lists of Fractions [M][N]."""
    M = len(a)
    K = len(b_q)
    N = len(b_q[0]) * 8 if K else 0
    W = [[weight(b_q, scales, qzeros, G, zp_bias, dtype, k, n) for n in range(N)] for k in range(K)]
    out = []
    for m in range(M):
        Am = [decode(a[m][k], dtype) for k in range(K)]
        row = []
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Am[k] * W[k][n]
            if bias is not None:
                acc += decode(bias[n], dtype)
            row.append(acc)
        out.append(row)
    return out


def round_rne(x: Fraction, dtype: str) -> int:
    """Exact RNE of a rational to the 16-bit format (finite results only), by integer search."""
    eb, p, bias = _FIELDS[dtype]
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    if a == 0:
        return sign
    # binade: largest e with 2^e <= a
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, 1 - bias)
    quantum = Fraction(2) ** (e - p)
    sig = a / quantum
    lo = sig.numerator // sig.denominator
    rem = sig - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    if e == 1 - bias and lo < (1 << p):
        bits = lo
    else:
        bits = ((e + bias) << p) + (lo - (1 << p))
    if bits >= ((1 << eb) - 1) << p:
        bits = ((1 << eb) - 1) << p
    return sign | bits
