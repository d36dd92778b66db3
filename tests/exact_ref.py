"""Exact and arbitrary-precision references used to pin the oracle.

Nothing here shares code with the oracle (``oracle/mbglu_oracle.c``) or with
the CUDA library.  bf16 rounding is done by brute force: the full sorted list
of finite bf16 values is searched for the two neighbours of an exact rational,
and the nearer one wins, ties going to the pattern with an even last bit --
the IEEE 754 round-to-nearest-even definition, stated without bit tricks.
SiLU is evaluated with mpmath at 120 bits.
"""
from __future__ import annotations

import bisect
import functools
import struct
from fractions import Fraction

import numpy as np

POS_INF_BITS = 0x7F80


def bf16_bits_to_fraction(b: int) -> Fraction:
    f = struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0]
    return Fraction(f)


@functools.lru_cache(maxsize=1)
def _positive_table():
    # finite non-negative bf16 patterns 0x0000 .. 0x7F7F, ascending in value
    vals = [bf16_bits_to_fraction(b) for b in range(0x0000, 0x7F80)]
    for a, b in zip(vals, vals[1:]):
        assert a < b
    return vals


def rne_bf16(q) -> int:
    """Nearest bf16 to the exact value q (Fraction/int/float), ties to even."""
    q = Fraction(q)
    if q == 0:
        return 0
    neg = q < 0
    a = -q if neg else q
    table = _positive_table()
    top = table[-1]
    if a > top:
        # beyond the largest finite value: compare with the midpoint to 2^128
        mid = (top + Fraction(2) ** 128) / 2
        if a < mid:
            bits = len(table) - 1
        else:  # at or above the midpoint: 0x7F7F is odd, so the tie goes up
            bits = POS_INF_BITS
    else:
        i = bisect.bisect_left(table, a)
        if table[i] == a:
            bits = i
        else:
            lo, hi = i - 1, i
            dlo, dhi = a - table[lo], table[hi] - a
            if dlo < dhi:
                bits = lo
            elif dhi < dlo:
                bits = hi
            else:
                bits = lo if lo % 2 == 0 else hi
    return (0x8000 | bits) if neg else bits


def mp():
    import mpmath
    mpmath.mp.prec = 120
    return mpmath


def mpf_to_fraction(x) -> Fraction:
    """Exact value of a finite mpf.  Magnitudes below 2^-300 (which every
    bf16 rounding sends to zero) are returned as +-2^-300 so that the
    Fraction stays small."""
    sign, man, exp, bc = x._mpf_     # value = (-1)^sign * man * 2^exp
    man, exp = int(man), int(exp)
    if man and exp + int(bc) < -300:
        man, exp = 1, -300
    if sign:
        man = -man
    return Fraction(man) * Fraction(2) ** exp if exp >= 0 else Fraction(man, 2 ** (-exp))


def fraction_to_mpf(q):
    m = mp()
    q = Fraction(q)
    return m.mpf(q.numerator) / m.mpf(q.denominator)


def silu_exact(q) -> Fraction:
    """SiLU(q) = q / (1 + e^-q) at 120 bits, as a Fraction."""
    m = mp()
    x = fraction_to_mpf(q)
    return mpf_to_fraction(x / (1 + m.exp(-x)))


def glu_exact(h_bits, g_bits, u_bits, mode):
    """Exact-rational dot products, 120-bit SiLU, brute-force bf16 rounding."""
    h = [[bf16_bits_to_fraction(v) for v in row] for row in np.asarray(h_bits)]
    G_rows = [[bf16_bits_to_fraction(v) for v in row] for row in np.asarray(g_bits)]
    U_rows = [[bf16_bits_to_fraction(v) for v in row] for row in np.asarray(u_bits)]
    M, N = len(h), len(G_rows)
    out = np.zeros((M, N), dtype=np.uint16)
    Gx = [[None] * N for _ in range(M)]
    Ux = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            G = sum((a * b for a, b in zip(h[m], G_rows[n])), Fraction(0))
            U = sum((a * b for a, b in zip(h[m], U_rows[n])), Fraction(0))
            Gx[m][n], Ux[m][n] = G, U
            if mode == "fused":
                out[m, n] = rne_bf16(silu_exact(G) * U)
            else:
                gb = bf16_bits_to_fraction(rne_bf16(G))
                ub = bf16_bits_to_fraction(rne_bf16(U))
                sb = bf16_bits_to_fraction(rne_bf16(silu_exact(gb)))
                out[m, n] = rne_bf16(sb * ub)
    return out, Gx, Ux


def rmsnorm_exact_row(x_bits, r_bits, w_bits, eps32: float):
    """(s, h) of one row: exact residual sum, 120-bit norm, brute-force rounding."""
    m = mp()
    s = [rne_bf16(bf16_bits_to_fraction(int(a)) + bf16_bits_to_fraction(int(b))) for a, b in zip(x_bits, r_bits)]
    sv = [bf16_bits_to_fraction(v) for v in s]
    var = sum((v * v for v in sv), Fraction(0)) / len(sv)
    denom = m.sqrt(fraction_to_mpf(var + Fraction(eps32)))
    h = []
    for v, wb in zip(sv, w_bits):
        val = fraction_to_mpf(v) / denom * fraction_to_mpf(1 + bf16_bits_to_fraction(int(wb)))
        h.append(rne_bf16(mpf_to_fraction(val)))
    return s, h
