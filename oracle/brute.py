"""Exact rational brute force (pure Python, ``fractions.Fraction``) for tiny
inputs.  Used only to pin the NumPy oracle: every rounding decision here is
made on the exact real value, straight from the definitions (nearest grid
value, ties to the even code, saturation), with no float arithmetic except
the one binary32 multiply that the activation path specifies."""
from __future__ import annotations

import struct
from fractions import Fraction


def f32(x: float) -> float:
    """Round a Python float to binary32 (round to nearest even)."""
    return struct.unpack("<f", struct.pack("<f", x))[0]


def e2m1_value(code: int) -> Fraction:
    sign = -1 if code & 8 else 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = Fraction(m, 2)
    else:
        mag = Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return sign * mag


def e4m3_value(b: int) -> Fraction:
    sign = -1 if b & 0x80 else 1
    e = (b >> 3) & 0xF
    m = b & 7
    if e == 0xF and m == 7:
        raise ValueError("NaN")
    if e == 0:
        mag = Fraction(m, 8) * Fraction(1, 64)
    else:
        mag = (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return sign * mag


E2M1_POS = [(c, e2m1_value(c)) for c in range(8)]
E4M3_POS = [(b, e4m3_value(b)) for b in range(0x7F)]


def nearest_even(value: Fraction, grid):
    """Code of the grid entry nearest to |value| (ties: even code; beyond the
    largest entry: the largest).  ``grid`` is [(code, magnitude)] ascending."""
    a = abs(value)
    if a >= grid[-1][1]:
        return grid[-1][0]
    best = None
    for code, mag in grid:
        d = abs(a - mag)
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    return best[1]


def rne_e2m1(value: Fraction, negative: bool) -> int:
    return nearest_even(value, E2M1_POS) | (8 if negative else 0)


def rne_e4m3(value: Fraction) -> int:
    return nearest_even(value, E4M3_POS)


def quantize_act_row(x_row, inv_lambda):
    """One activation row (floats exactly bf16) -> (codes, scale bytes)."""
    xhat = [f32(float(x) * float(il)) for x, il in zip(x_row, inv_lambda)]
    codes, scales = [], []
    for b in range(0, len(xhat), 16):
        blk = xhat[b:b + 16]
        amax = max(abs(Fraction(v)) for v in blk)
        s_code = rne_e4m3(amax / 6)
        s = e4m3_value(s_code)
        scales.append(s_code)
        for v in blk:
            if s == 0:
                codes.append(0)
            else:
                neg = struct.pack("<f", v)[3] & 0x80 != 0
                codes.append(rne_e2m1(Fraction(v) / s, neg))
    return codes, scales


def quantize_weight_col(r_col, s_T: Fraction):
    """One output channel of the residual (floats) -> (codes, scale bytes)."""
    codes, scales = [], []
    for b in range(0, len(r_col), 16):
        blk = [Fraction(v) for v in r_col[b:b + 16]]
        amax = max(abs(v) for v in blk)
        s_code = rne_e4m3(amax / (6 * s_T))
        s = e4m3_value(s_code)
        scales.append(s_code)
        for v, raw in zip(blk, r_col[b:b + 16]):
            if s == 0:
                codes.append(0)
            else:
                neg = struct.pack("<d", raw)[7] & 0x80 != 0
                codes.append(rne_e2m1(v / (s * s_T), neg))
    return codes, scales


def gemm_exact(a_codes, a_scales, w_codes, w_scales, s_T, lora_act, L2, bias):
    """Exact Y (Fractions) from unpacked codes and unswizzled scales; every
    product and sum is rational."""
    M = len(a_codes)
    N = len(w_codes)
    K = len(a_codes[0]) if M else 0
    adec = [[e2m1_value(a_codes[m][k]) * e4m3_value(a_scales[m][k // 16]) for k in range(K)]
            for m in range(M)]
    wdec = [[e2m1_value(w_codes[n][k]) * e4m3_value(w_scales[n][k // 16]) for k in range(K)]
            for n in range(N)]
    r = len(L2)
    Y = []
    for m in range(M):
        row = []
        for n in range(N):
            acc = sum((adec[m][k] * wdec[n][k] for k in range(K)), Fraction(0))
            y = Fraction(s_T) * acc
            for i in range(r):
                y += Fraction(lora_act[m][i]) * Fraction(L2[i][n])
            if bias is not None:
                y += Fraction(bias[n])
            row.append(y)
        Y.append(row)
    return Y


# ---------------------------------------------------------------- INT4 variant
def round_binary(value: Fraction, mant_bits: int, emin: int = -126) -> Fraction:
    """Nearest number with ``mant_bits`` significant bits, exponent >= emin
    (below it: the fixed subnormal spacing 2^(emin - mant_bits + 1)), ties to
    an even last digit.  binary32: (24, -126); bfloat16: (8, -126).  No
    overflow (the callers' values stay far below the largest finite one)."""
    if value == 0:
        return Fraction(0)
    a = abs(value)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, emin) - (mant_bits - 1))
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * quantum
    return -r if value < 0 else r


def round_half_even_int(value: Fraction) -> int:
    fl = value.numerator // value.denominator
    rem = value - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def int4_codes(values, s: Fraction):
    """Symmetric 4-bit integer codes of exact values under scale s (0 -> 0)."""
    if s == 0:
        return [0] * len(values)
    return [max(-8, min(7, round_half_even_int(v / s))) for v in values]


def int4_act_row(x_row, inv_lambda):
    """One activation row (floats exactly bf16) -> (codes, scales as
    Fractions): x_hat = fl32(x inv), s = bf16(fl32(amax / 7)) per 64 k."""
    xhat = [Fraction(f32(float(x) * float(il))) for x, il in zip(x_row, inv_lambda)]
    codes, scales = [], []
    for g in range(0, len(xhat), 64):
        blk = xhat[g:g + 64]
        amax = max(abs(v) for v in blk)
        s = round_binary(round_binary(amax / 7, 24), 8)
        scales.append(s)
        codes += int4_codes(blk, s)
    return codes, scales


def int4_weight_col(r_col):
    """One output channel of the float64 residual -> (codes, scales):
    s = bf16(amax / 7) of the exact quotient per 64 k."""
    vals = [Fraction(v) for v in r_col]
    codes, scales = [], []
    for g in range(0, len(vals), 64):
        blk = vals[g:g + 64]
        s = round_binary(max(abs(v) for v in blk) / 7, 8)
        scales.append(s)
        codes += int4_codes(blk, s)
    return codes, scales


def int4_gemm_exact(a_codes, a_scales, w_codes, w_scales, lora_act, L2, bias):
    """Exact Y of the INT4 layer from codes and group scales (Fractions or
    floats); L2 is [r][N]."""
    M, N = len(a_codes), len(w_codes)
    K = len(a_codes[0]) if M else 0
    Y = []
    for m in range(M):
        row = []
        for n in range(N):
            y = Fraction(0)
            for g in range(K // 64):
                isum = sum(int(a_codes[m][k]) * int(w_codes[n][k]) for k in range(64 * g, 64 * g + 64))
                y += Fraction(a_scales[m][g]) * Fraction(w_scales[n][g]) * isum
            for i in range(len(L2)):
                y += Fraction(lora_act[m][i]) * Fraction(L2[i][n])
            if bias is not None:
                y += Fraction(bias[n])
            row.append(y)
        Y.append(row)
    return Y
