"""Oracle of the AWQ W4A16 linear (4-bit weights, 16-bit activations).

The pages ([dothoosh], "two kernel families" list and "quantization_config"
block; [hamidun-ar], "What are Nunchaku and SVDQuant") say only that awq_w4a16
keeps 16-bit activations and 4-bit weights with group size 64, and that it
serves the precision-sensitive, memory-bound modulation layers
(adaLN_modulation.1).  Readings:
  A1  plain asymmetric group quantization along K, group 64, per output
      channel (the activation-aware scale search of AWQ is not described):
      s = fp16((max - min) / 15), z = fp16(-min / s),
      q = clamp(RNE(w / s + z), 0, 15), all in float64 before the fp16
      roundings; a group with max == min, or with s rounding to 0, uses
      s = 1, z = fp16(-min).  z is clamped to the finite fp16 range.
  A2  dequantized weight w' = (q - z) s, with s and z as stored (fp16);
      Y = X w'^T + b, returned unrounded in float64.
  A3  layout: qweight [N][K/2] bytes, even k in the low nibble; scales and
      zeros [N][K/64] fp16.
"""
from __future__ import annotations

import numpy as np

from .formats import round_to_f16, f16_bits
from .layout import pack_nibbles, unpack_nibbles

F16_MAX = 65504.0


def awq_pack(W: np.ndarray, group_size: int = 64):
    W = np.asarray(W, dtype=np.float32).astype(np.float64)
    N, K = W.shape
    if K % group_size:
        raise ValueError("K must be a multiple of the group size")
    G = W.reshape(N, K // group_size, group_size)
    mx = G.max(axis=2)
    mn = G.min(axis=2)
    s = round_to_f16((mx - mn) / 15.0)
    degenerate = (mx == mn) | (s == 0.0)
    s = np.where(degenerate, 1.0, s)
    z = round_to_f16(np.clip(-mn / s, -F16_MAX, F16_MAX))
    q = np.clip(np.rint(G / s[..., None] + z[..., None]), 0, 15).astype(np.uint8)
    q = q.reshape(N, K)
    return {"q": q, "qweight": pack_nibbles(q), "scales": s, "zeros": z,
            "scales_bits": f16_bits(s), "zeros_bits": f16_bits(z),
            "group_size": group_size}


def awq_dequant(qweight: np.ndarray, scales: np.ndarray, zeros: np.ndarray,
                group_size: int = 64) -> np.ndarray:
    q = unpack_nibbles(qweight).astype(np.float64)
    s = np.repeat(np.asarray(scales, dtype=np.float64), group_size, axis=1)
    z = np.repeat(np.asarray(zeros, dtype=np.float64), group_size, axis=1)
    return (q - z) * s


def awq_linear(X: np.ndarray, qweight, scales, zeros, bias, group_size: int = 64):
    """Reading A2: Y = X ((q - z) s)^T + b in float64."""
    Wd = awq_dequant(qweight, scales, zeros, group_size)
    Y = np.asarray(X, dtype=np.float64) @ Wd.T
    if bias is not None:
        Y = Y + np.asarray(bias, dtype=np.float64)[None, :]
    return Y
