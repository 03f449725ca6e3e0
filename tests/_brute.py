"""Brute force in exact rational arithmetic (Python ``fractions``), used to pin the
oracle on tiny inputs.  Shares nothing with the oracle's C code: every value is
an exact rational, and rounding to a binary format is done on rationals.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

GROUP = 128


def half_bits_to_fraction(bits: int) -> Fraction:
    """Exact value of an IEEE binary16 bit pattern (finite values only)."""
    sign = -1 if (bits >> 15) & 1 else 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    assert e != 31, "inf/nan not expected"
    if e == 0:
        v = Fraction(f, 1 << 24)
    else:
        v = Fraction(1024 + f) * (Fraction(2) ** (e - 25))
    return sign * v


def float32_to_fraction(v) -> Fraction:
    return Fraction(float(np.float32(v)))


def _floor_log2(a: Fraction) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # adjust so that 2**e <= a < 2**(e+1)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_half_even_int(a: Fraction) -> int:
    """Nearest integer to a, ties to even."""
    fl = a.numerator // a.denominator
    rem = a - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def round_to_binary(x: Fraction, p: int, emin: int, emax: int):
    """Round x to the binary format with p significand bits (implicit bit included),
    minimum normal exponent emin and maximum exponent emax; ties to even.
    Returns a Fraction, or float('inf') / -inf on overflow."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = max(_floor_log2(a), emin)
    quantum = Fraction(2) ** (e - p + 1)
    n = round_half_even_int(a / quantum)
    r = n * quantum
    max_finite = (Fraction(2) - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if r > max_finite:
        return float("inf") * sign
    return sign * r


def to_half(x: Fraction):
    return round_to_binary(x, 11, -14, 15)


def to_float32(x: Fraction):
    return round_to_binary(x, 24, -126, 127)


def fraction_to_half_bits(v) -> int:
    """binary16 bit pattern of an exactly representable value (or +-inf)."""
    if v == float("inf"):
        return 0x7C00
    if v == float("-inf"):
        return 0xFC00
    return int(np.array([float(v)], dtype=np.float64).astype(np.float16).view(np.uint16)[0])


def quant_act_int8(xbits: np.ndarray):
    """Exact per-token quantizer: s = fp32(amax/127), q = clamp(rne(fp32(x/s)), -127, 127)."""
    M, K = xbits.shape
    q = np.zeros((M, K), np.int64)
    s = np.zeros((M,), np.float64)
    for m in range(M):
        vals = [half_bits_to_fraction(int(b)) for b in xbits[m]]
        amax = max(abs(v) for v in vals)
        if amax == 0:
            continue
        sm = to_float32(amax / 127)
        s[m] = float(sm)
        for k, v in enumerate(vals):
            t = to_float32(v / sm)
            r = round_half_even_int(t)
            q[m, k] = max(-127, min(127, r))
    return q, s


def gemm_wxa16(xbits: np.ndarray, codes: np.ndarray, sbits: np.ndarray) -> np.ndarray:
    """Exact y = fp16(sum_g s[n,g] sum_k x[m,k] q[n,k]) as binary16 bit patterns."""
    M, K = xbits.shape
    N = codes.shape[0]
    G = K // GROUP
    xf = [[half_bits_to_fraction(int(b)) for b in row] for row in xbits]
    sf = [[half_bits_to_fraction(int(b)) for b in row] for row in sbits]
    y = np.zeros((M, N), np.uint16)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for g in range(G):
                inner = Fraction(0)
                for k in range(g * GROUP, (g + 1) * GROUP):
                    c = int(codes[n, k])
                    if c:
                        inner += xf[m][k] * c
                acc += sf[n][g] * inner
            y[m, n] = fraction_to_half_bits(to_half(acc))
    return y


def gemm_w4a8(qa: np.ndarray, sx: np.ndarray, codes: np.ndarray, sbits: np.ndarray) -> np.ndarray:
    """Exact y = fp16(sx[m] * sum_g s[n,g] * sum_k qa[m,k] q[n,k]) as binary16 bits."""
    M, K = qa.shape
    N = codes.shape[0]
    G = K // GROUP
    sf = [[half_bits_to_fraction(int(b)) for b in row] for row in sbits]
    y = np.zeros((M, N), np.uint16)
    qa64 = qa.astype(np.int64)
    c64 = codes.astype(np.int64)
    for m in range(M):
        sm = float32_to_fraction(sx[m])
        for n in range(N):
            acc = Fraction(0)
            for g in range(G):
                inner = int(np.dot(qa64[m, g * GROUP:(g + 1) * GROUP], c64[n, g * GROUP:(g + 1) * GROUP]))
                acc += sf[n][g] * inner
            y[m, n] = fraction_to_half_bits(to_half(sm * acc))
    return y


def embed_w8(ids, codes: np.ndarray, sbits: np.ndarray) -> np.ndarray:
    """Exact out[t,k] = fp16(codes[ids[t],k] * scale[ids[t],k/128]) as binary16 bits."""
    T = len(ids)
    D = codes.shape[1]
    out = np.zeros((T, D), np.uint16)
    for t, v in enumerate(ids):
        for k in range(D):
            sb = int(sbits[v, k // GROUP])
            c = int(codes[v, k])
            p = c * half_bits_to_fraction(sb)
            if p == 0:
                # IEEE: the sign of a zero product is the XOR of the operands' signs
                # (an integer code 0 is +0)
                out[t, k] = 0x8000 if ((c < 0) != bool(sb & 0x8000)) else 0
            else:
                out[t, k] = fraction_to_half_bits(to_half(p))
    return out


def topk(vals: np.ndarray, k: int):
    """Indices of the k largest values, largest first, ties to the smaller index."""
    order = sorted(range(len(vals)), key=lambda i: (-float(vals[i]), i))
    return order[:k]
