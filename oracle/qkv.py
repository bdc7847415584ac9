"""Oracle of the fused QKV epilogue: per-head RMS normalization of Q and K and
the rotary position embedding, applied to the output of the fused QKV
projection (an SVDQ W4A4 linear with N = 3 H D).

TEST INFRASTRUCTURE, NOT PRODUCT CODE (see the package docstring).

What the pages fix ([dothoosh], the paragraphs on structural rewrites): the
full engine merges the attention block's three projections to_q, to_k, to_v
into one quantized module, joined along the output dimension in the order Q,
K, V; its fused operator then takes the QKV projection, the normalization of Q
and K and the rotary embeddings in one step, where the default path runs them
one after another: the separate projections, the split into heads, norm_q and
norm_k, then the rotary embeddings.

Readings (the pages give no formula):
  Q1  layout: columns [0, HD) are Q, [HD, 2HD) K, [2HD, 3HD) V; head h of Q
      (of K) is its columns hD .. hD + D - 1; D = 128 (hidden size 3072 =
      24 heads x 128).
  Q2  normalization: RMS normalization over the D channels of one head of one
      token, n = y / sqrt(mean(y^2) + eps) * w, eps = 1e-6, with one learned
      weight vector w[D] for Q and one for K.
  Q3  rotary embedding, after the normalization (the pages' order), on the
      channel pairs (2i, 2i+1) of a head:
      (a, b) -> (a cos(theta) - b sin(theta), a sin(theta) + b cos(theta)),
      theta = theta[m][i] per token m and pair i, the same for every head; the
      caller supplies cos and sin (token positions are the model's business).
  Q4  precision: the input is the projection's bf16 output Y_b (bias
      included); normalization and rotation are exact here and the device
      rounds once to bf16 at the end; V is Y_b itself.
"""
from __future__ import annotations

import numpy as np

HEAD_DIM = 128
RMS_EPS = 1e-6


def _heads(y: np.ndarray, head_dim: int) -> np.ndarray:
    y = np.asarray(y, dtype=np.float64)
    M, C = y.shape
    assert C % head_dim == 0 and head_dim % 2 == 0
    return y.reshape(M, C // head_dim, head_dim)


def rms_norm_heads(y: np.ndarray, w: np.ndarray, head_dim: int = HEAD_DIM,
                   eps: float = RMS_EPS) -> np.ndarray:
    """Reading Q2: every head of every token divided by the root of its mean
    square (+ eps), times the per-channel weight w [head_dim]; float64."""
    h = _heads(y, head_dim)
    rms = np.sqrt(np.mean(h * h, axis=2, keepdims=True) + eps)
    out = h / rms * np.asarray(w, dtype=np.float64)[None, None, :]
    return out.reshape(y.shape)


def rope_pairs(x: np.ndarray, cos: np.ndarray, sin: np.ndarray,
               head_dim: int = HEAD_DIM) -> np.ndarray:
    """Reading Q3: rotation of the channel pairs (2i, 2i+1) of every head of
    token m by the angle whose cosine and sine are cos[m][i], sin[m][i]."""
    h = _heads(x, head_dim)
    c = np.asarray(cos, dtype=np.float64)[:, None, :]
    s = np.asarray(sin, dtype=np.float64)[:, None, :]
    a, b = h[:, :, 0::2], h[:, :, 1::2]
    out = np.empty_like(h)
    out[:, :, 0::2] = a * c - b * s
    out[:, :, 1::2] = a * s + b * c
    return out.reshape(np.asarray(x).shape)


def qkv_norm_rope(y_b: np.ndarray, w_q: np.ndarray, w_k: np.ndarray, cos: np.ndarray,
                  sin: np.ndarray, head_dim: int = HEAD_DIM,
                  eps: float = RMS_EPS) -> np.ndarray:
    """Readings Q1-Q4 together: Q and K normalized then rotated, V passed
    through; float64, unrounded ([M, 3 H D])."""
    y_b = np.asarray(y_b, dtype=np.float64)
    M, N = y_b.shape
    assert N % (3 * head_dim) == 0
    hd = N // 3
    out = y_b.copy()
    out[:, :hd] = rope_pairs(rms_norm_heads(y_b[:, :hd], w_q, head_dim, eps), cos, sin,
                             head_dim)
    out[:, hd:2 * hd] = rope_pairs(rms_norm_heads(y_b[:, hd:2 * hd], w_k, head_dim, eps),
                                   cos, sin, head_dim)
    return out
