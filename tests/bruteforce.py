"""Exact pure-Python brute force used to pin the oracle (tests only).

Everything here works on ``fractions.Fraction`` values, enumerates the E4M3
code space instead of searching a table, and rounds to float32 with integer
arithmetic, so it shares no numerics with the numpy oracle. It is slow and is
only run on tiny inputs.
"""
from __future__ import annotations

import math
from fractions import Fraction

E4M3_MAX = Fraction(448)


def e4m3_value(code: int) -> Fraction | None:
    """Exact value of an E4M3 code from its bit fields (None for NaN)."""
    if code & 0x7F == 0x7F:
        return None
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 0:
        mag = Fraction(m, 8) * Fraction(1, 2 ** 6)
    else:
        mag = (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))
    return -mag if code & 0x80 else mag


_NONNEG = [(c, e4m3_value(c)) for c in range(0x7F)]


def encode(x: float) -> int:
    """Nearest finite E4M3 value by exhaustive search (ties to the even code);
    anything above 448 is nearest to 448, which is saturation. Sign kept."""
    neg = math.copysign(1.0, x) < 0
    a = abs(Fraction(x))
    best_c, best_d = None, None
    for c, v in _NONNEG:
        d = abs(a - v)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best_c, best_d = c, d
    return best_c | (0x80 if neg else 0)


def round_to_f32(r: Fraction) -> Fraction:
    """Round an exact rational to the nearest float32 (ties to even), returned
    exactly. Subnormals included; no overflow handling (not needed here)."""
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * quantum


def scale_of(amax: Fraction, pow2: bool) -> Fraction:
    if pow2:
        p = -126
        while amax > E4M3_MAX * Fraction(2) ** p:
            p += 1
        return Fraction(2) ** p
    s = round_to_f32(amax / E4M3_MAX)
    return max(s, Fraction(2) ** -126)


def quant_tile(xs: list[float], pow2: bool) -> tuple[list[int], Fraction]:
    """Codes and scale of one tile of float32 values: enc(RN32(x * RN32(1/s)))."""
    amax = max(abs(Fraction(x)) for x in xs)
    s = scale_of(amax, pow2)
    f = round_to_f32(1 / s)  # quantization factor RN32(1/s)
    codes = []
    for x in xs:
        q = round_to_f32(Fraction(x) * f)
        # the sign of a quotient that rounds to zero is the sign of x
        codes.append(encode(math.copysign(float(q), x) if q == 0 else float(q)))
    return codes, s


def gemm_exact(qa, sa, qb, sb, scale_b="128x128"):
    """Exact rational block-scaled GEMM: sum_kb P_kb * sa * sb, together with
    sum_kb |P_kb * sa * sb| (the scale of the rounding error of any evaluation)."""
    M, K = len(qa), len(qa[0])
    N = len(qb)
    out = [[Fraction(0)] * N for _ in range(M)]
    mag = [[Fraction(0)] * N for _ in range(M)]
    for kb in range(K // 128):
        for i in range(M):
            for j in range(N):
                p = sum(e4m3_value(qa[i][k]) * e4m3_value(qb[j][k])
                        for k in range(kb * 128, kb * 128 + 128))
                sbv = sb[kb][j // 128] if scale_b == "128x128" else sb[kb][j]
                term = p * Fraction(float(sa[kb][i])) * Fraction(float(sbv))
                out[i][j] += term
                mag[i][j] += abs(term)
    return out, mag
