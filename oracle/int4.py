"""Oracle of the SVDQuant W4A4 linear layer, INT4 variant.  Test
infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use it.

What the pages fix ([dothoosh], kernel-family list: svdq_w4a4 comes in INT4
and NVFP4 variants; hardware list: INT4 serves Turing, Ampere and Ada, NVFP4
Blackwell; "quantization_config" block: compute dtype bfloat16, and the one
int4 group size it prints, 64): the same SVDQuant layer -- smoothing, a
16-bit low-rank branch, a 4-bit residual, 4-bit activations -- with the
4-bit values integers instead of e2m1.

Readings of what the pages leave open (each used below):
  I1  groups of 64 consecutive k, for the weight residual (per output
      channel) and for the activations (per row).
  I2  codes are signed 4-bit integers, two's complement in a nibble; the
      scale is symmetric: s = RNE_bf16(amax / 7) (the scale is kept in the
      compute dtype), code q = clamp(RNE(v / s), -8, 7) with ties to even.
      A group whose scale is 0 or not finite gets all codes 0.  Since
      s >= amax/7 (1 - 2^-9), |v / s| < 7.02 and -8 never occurs.
  I3  activations: x_hat = fl32(x * inv_lambda) as in the NVFP4 variant (R7);
      the scale quotient is the binary32 one, s = RNE_bf16(fl32(amax / 7))
      (what one writes in fp32 arithmetic; for amax below 7 * 2^-126 it can
      differ from the exact quotient's rounding, so the definition names it).
      The code quotient x_hat / s is rounded from the exact real quotient
      (equal to rounding the binary32 quotient: it lies more than half a
      binary32 ulp from any half-integer it is not equal to).
  I4  weights: smoothing, low rank and residual exactly as the NVFP4 variant
      (R1-R4); s_w = RNE_bf16(amax_R / 7) and q = clamp(RNE(R / s_w), -8, 7)
      from float64 quotients (R is float64; a float64 quotient of a 53-bit
      numerator by 7 or by an 8-bit scale cannot be rounded across a bf16 or
      half-integer midpoint that the exact quotient does not sit on).  No
      tensor scale: bf16 scales have the range.
  I5  Y = sum_g s_x[m,g] s_w[n,g] sum_{k in g} q_x q_w + lora_act L2 + b,
      float64, unrounded; the device rounds once to bf16.  The low-rank
      branch is that of the NVFP4 variant with L2 unscaled.
Layouts: codes [rows][K/2] bytes, element 2i of a row in the low nibble of
byte i; scales [rows][K/64] bf16, row-major.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_bits, round_to_bf16
from .svdq import (
    lora_down,
    lowrank_factors,
    residual,
    smooth_activations,
    smoothing_inv_lambda,
)

GROUP = 64
QMAX = 7.0
QMIN = -8.0


def _codes_from_quotient(q: np.ndarray) -> np.ndarray:
    """Round-half-even to an integer, clamp to [-8, 7] (float64 in, int8 out)."""
    return np.clip(np.rint(q), QMIN, QMAX).astype(np.int8)


def _quantize_groups(V: np.ndarray, S: np.ndarray) -> np.ndarray:
    """codes of the float64 values V [rows][K] under the group scales S
    [rows][K/64] (reading I2: scale 0 or non-finite -> codes 0)."""
    rows, K = V.shape
    blocks = V.reshape(rows, K // GROUP, GROUP)
    s = S[..., None]
    ok = np.broadcast_to((s > 0) & np.isfinite(s), blocks.shape)
    codes = np.zeros(blocks.shape, dtype=np.int8)
    codes[ok] = _codes_from_quotient(blocks[ok] / np.broadcast_to(s, blocks.shape)[ok])
    return codes.reshape(rows, K)


def quantize_activations(X: np.ndarray, inv_lambda: np.ndarray):
    """Readings I1-I3.  X: [M, K] bf16 values.  Returns (x_hat float32,
    codes [M][K] int8 in [-8, 7], scales [M][K/64] float64 bf16 values)."""
    xhat = smooth_activations(X, inv_lambda)
    M, K = xhat.shape
    if M == 0:
        return xhat, np.zeros((0, K), np.int8), np.zeros((0, K // GROUP))
    amax = np.max(np.abs(xhat.reshape(M, K // GROUP, GROUP)), axis=2).astype(np.float32)
    quot32 = (amax / np.float32(QMAX)).astype(np.float32)   # binary32 division
    scales = round_to_bf16(quot32.astype(np.float64))
    codes = _quantize_groups(xhat.astype(np.float64), scales)
    return xhat, codes, scales


def quantize_weight_residual(R: np.ndarray):
    """Reading I4.  R is [K, N] float64; returns (codes [N][K] int8,
    scales [N][K/64] float64 bf16 values)."""
    Rt = np.ascontiguousarray(np.asarray(R, dtype=np.float64).T)
    N, K = Rt.shape
    amax = np.max(np.abs(Rt.reshape(N, K // GROUP, GROUP)), axis=2)
    scales = round_to_bf16(amax / QMAX)
    return _quantize_groups(Rt, scales), scales


def pack_weights(W: np.ndarray, x_absmax, rank: int, lowrank=None):
    """Offline packing, INT4 variant (readings R1-R4 of the NVFP4 variant
    for the factors and the residual, I4 for its quantization).  W: [N, K]
    float32; x_absmax: [K] or None (no smoothing)."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    inv = np.ones(K, dtype=np.float32) if x_absmax is None else smoothing_inv_lambda(x_absmax, W)
    inv64 = inv.astype(np.float64)
    if lowrank is None:
        L1, L2 = lowrank_factors(W.T.astype(np.float64) / inv64[:, None], rank)
    else:
        L1, L2 = lowrank
    L1s = round_to_bf16(inv64[:, None] * L1)
    L2 = round_to_bf16(L2)
    R = residual(W, inv, L1s, L2)
    codes, scales = quantize_weight_residual(R)
    return {"N": N, "K": K, "rank": rank, "inv_lambda": inv, "L1s": L1s, "L2": L2, "R": R,
            "w_codes": codes, "w_scales": scales}


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 values q * s of codes [rows][K] under group scales [rows][K/64]."""
    return codes.astype(np.float64) * np.repeat(np.asarray(scales, np.float64), GROUP, axis=1)


def gemm_reference(a_codes, a_scales, w_codes, w_scales, lora_act, L2, bias):
    """Reading I5: the dequantized product plus the low-rank and bias terms,
    float64, unrounded.  L2 is [r][N]."""
    Y = dequantize(a_codes, a_scales) @ dequantize(w_codes, w_scales).T
    if lora_act is not None and np.asarray(lora_act).shape[1] > 0:
        Y = Y + np.asarray(lora_act, np.float64) @ np.asarray(L2, np.float64)
    if bias is not None:
        Y = Y + np.asarray(bias, np.float64)[None, :]
    return Y


def linear_forward(X: np.ndarray, packed: dict, bias):
    """The whole INT4 layer for bf16 X [M, K]: every intermediate the device
    produces, plus Y (float64)."""
    xhat, a_codes, a_scales = quantize_activations(X, packed["inv_lambda"])
    lora = lora_down(X, packed["L1s"])
    Y = gemm_reference(a_codes, a_scales, packed["w_codes"], packed["w_scales"], lora,
                       packed["L2"], bias)
    return {"x_hat": xhat, "a_codes": a_codes, "a_scales": a_scales, "lora_act": lora, "Y": Y}


def naive_w4a4(X: np.ndarray, W: np.ndarray, bias):
    """The same INT4 rules with no smoothing and no low-rank branch."""
    return linear_forward(X, pack_weights(W, None, 0), bias)["Y"]


# ---------------------------------------------------------------- byte layouts
def pack_codes(codes: np.ndarray) -> np.ndarray:
    """int8 codes [rows][K] -> [rows][K/2] bytes, element 2i in the low nibble."""
    u = (np.asarray(codes, np.int16) & 0xF).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[rows][K/2] bytes -> int8 codes [rows][K] (two's complement nibbles)."""
    p = np.asarray(packed, np.uint8)
    lo = (p & 0xF).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    out = np.empty((p.shape[0], p.shape[1] * 2), np.int16)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return np.where(out >= 8, out - 16, out).astype(np.int8)


def scale_bits(scales: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of the group scales."""
    return bf16_bits(scales)
