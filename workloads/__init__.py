"""Seeded synthetic inputs for the SVDQ W4A4 linear and the AWQ W4A16 GEMV.

This module is the only code shared by the CUDA path's tests/benchmark and
the CPU oracle.  It draws random tensors and converts them to the storage
formats of the inputs (bfloat16 activations and bias, float32 weights); it
holds none of the layer's arithmetic.

The pages' workload (a FLUX / ERNIE-Image class diffusion transformer at
1024x1024, i.e. 64x64 = 4096 latent patch tokens, hidden size 3072, heavy
outlier channels in the activations) is not available as weights; these
tensors stand in for it with its shapes and the stated statistics:

  * activations X ~ N(0, 1), with a few "outlier" input channels multiplied
    by a large factor (1% of channels x50; the tiny case: 4 channels x40);
  * weights W = N(0, 0.02^2) noise + a planted low-rank part
    sum_i (3/i) a_i b_i^T whose singular vectors come from the QR factors of
    Gaussian matrices (rank 32; the tiny case rank 4, spectral norm 3);
  * bias ~ N(0, 0.01^2), stored as bfloat16;
  * AWQ modulation weights W ~ N(0, 0.02^2), 57 independent blocks sharing
    one conditioning vector X ~ N(0, 1).

Every tensor draws from its own child stream of ``SeedSequence(seed)``.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """float32 -> nearest bfloat16 (ties to even), returned as float32 values
    (storage-format conversion of a generated input)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32)


def bf16_bits_of(x_bf16_values: np.ndarray) -> np.ndarray:
    """uint16 storage of float32 values that are already bfloat16."""
    x = np.ascontiguousarray(x_bf16_values, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@dataclass(frozen=True)
class SVDQCase:
    name: str
    M: int
    K: int
    N: int
    rank: int
    seed: int
    outlier_channels: int
    outlier_scale: float
    planted_rank: int
    planted_norm: float = 3.0


# The workloads: a tiny parity case and the diffusion-transformer linears.
CASES = {
    "tiny": SVDQCase("tiny", 128, 256, 256, 16, 0, 4, 40.0, 4),
    "attn_out": SVDQCase("attn_out", 4096, 3072, 3072, 32, 1, 31, 50.0, 32),
    "qkv": SVDQCase("qkv", 4608, 3072, 9216, 32, 2, 31, 50.0, 32),
    "fc1": SVDQCase("fc1", 4096, 3072, 12288, 32, 3, 31, 50.0, 32),
    "fc1_b4": SVDQCase("fc1_b4", 16384, 3072, 12288, 32, 3, 31, 50.0, 32),
    # fc2's activations are GELU(fc1 output), produced by the caller; only its
    # weights and bias come from here (its own child streams of seed 3).
    "fc2": SVDQCase("fc2", 4096, 12288, 3072, 32, 3, 0, 1.0, 32),
    "fc2_b4": SVDQCase("fc2_b4", 16384, 12288, 3072, 32, 3, 0, 1.0, 32),
}


def custom_case(M, K, N, rank, seed=0, outlier_channels=None, outlier_scale=50.0,
                planted_rank=None, name="custom") -> SVDQCase:
    if outlier_channels is None:
        outlier_channels = max(1, round(0.01 * K))
    if planted_rank is None:
        planted_rank = min(32, K, N)
    return SVDQCase(name, M, K, N, rank, seed, outlier_channels, outlier_scale, planted_rank)


def _streams(seed: int, n: int, offset: int = 0):
    ss = np.random.SeedSequence(seed)
    kids = ss.spawn(n + offset)
    return [np.random.default_rng(k) for k in kids[offset:]]


def make_activations(case: SVDQCase, M: int | None = None) -> np.ndarray:
    """X [M, K] as float32 values that are exactly bfloat16."""
    M = case.M if M is None else M
    rng_x, rng_o = _streams(case.seed, 2)
    X = rng_x.standard_normal((M, case.K), dtype=np.float32)
    if case.outlier_channels:
        ch = rng_o.choice(case.K, case.outlier_channels, replace=False)
        X[:, ch] *= np.float32(case.outlier_scale)
    return to_bf16_values(X)


def make_weights(case: SVDQCase, stream_offset: int = 0):
    """(W [N, K] float32, bias [N] float32 values exactly bfloat16)."""
    off = 2 + stream_offset
    rng_w, rng_a, rng_b, rng_bias = _streams(case.seed, 4, off)
    W = rng_w.standard_normal((case.N, case.K), dtype=np.float32) * np.float32(0.02)
    p = min(case.planted_rank, case.N, case.K)
    if p:
        A, _ = np.linalg.qr(rng_a.standard_normal((case.N, p)))
        B, _ = np.linalg.qr(rng_b.standard_normal((case.K, p)))
        sig = case.planted_norm / np.arange(1, p + 1)
        W = (W.astype(np.float64) + (A * sig[None, :]) @ B.T).astype(np.float32)
    bias = to_bf16_values(rng_bias.standard_normal(case.N, dtype=np.float32) * np.float32(0.01))
    return W, bias


def make_fc2_weights(case: SVDQCase):
    """fc2 of the MLP pair: streams after fc1's four."""
    return make_weights(case, stream_offset=4)


# ---------------------------------------------------------------------------
# AWQ W4A16 modulation GEMV
# ---------------------------------------------------------------------------

AWQ_K = 3072
AWQ_N = 6 * 3072
AWQ_BLOCKS = 57
AWQ_SEED = 4


def make_awq_activations(M: int, K: int = AWQ_K, seed: int = AWQ_SEED) -> np.ndarray:
    (rng,) = _streams(seed, 1)
    return to_bf16_values(rng.standard_normal((M, K), dtype=np.float32))


def make_awq_weights(block: int, N: int = AWQ_N, K: int = AWQ_K, seed: int = AWQ_SEED):
    """(W [N, K] float32 ~ N(0, 0.02^2), bias [N] bf16 values ~ N(0, 0.01^2))
    of modulation block ``block`` (its own child streams)."""
    rng_w, rng_b = _streams(seed, 2, 1 + 2 * block)
    W = rng_w.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    bias = to_bf16_values(rng_b.standard_normal(N, dtype=np.float32) * np.float32(0.01))
    return W, bias


# ---------------------------------------------------------------------------
# Fused QKV epilogue (normalization of Q and K, rotary embedding)
# ---------------------------------------------------------------------------

QKV_TEXT_TOKENS = 512           # the qkv case: 512 text tokens, then 64 x 64 image patches
QKV_GRID = (64, 64)
ROPE_AXES = (16, 56, 56)        # channels of a 128-wide head given to each position axis
ROPE_BASE = 10000.0
QKV_NORM_SEED = 5


def rope_positions(n_text: int = QKV_TEXT_TOKENS, grid=QKV_GRID) -> np.ndarray:
    """[M, 3] integer positions of the tokens: the text tokens first, all at
    (0, 0, 0), then the image patches in row-major order at (0, row, col)."""
    gh, gw = grid
    img = np.zeros((gh * gw, 3), dtype=np.int64)
    img[:, 1] = np.repeat(np.arange(gh), gw)
    img[:, 2] = np.tile(np.arange(gw), gh)
    return np.concatenate([np.zeros((n_text, 3), dtype=np.int64), img])


def make_rope_tables(positions: np.ndarray, axes=ROPE_AXES, base: float = ROPE_BASE):
    """(cos, sin) [M, sum(axes)/2] float32 rotary tables (input data of the
    fused epilogue): the channel pairs of a head are split over the position
    axes in order, and pair j of an axis with d channels turns by
    position * base^(-2j/d) (the rotary embedding's frequency ladder, per axis)."""
    positions = np.asarray(positions, dtype=np.float64)
    angles = []
    for a, d in enumerate(axes):
        freq = base ** (-np.arange(0, d, 2, dtype=np.float64) / d)
        angles.append(positions[:, a:a + 1] * freq[None, :])
    theta = np.concatenate(angles, axis=1)
    return np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)


def make_qk_norm_weights(head_dim: int = 128, seed: int = QKV_NORM_SEED):
    """(w_q, w_k) [head_dim] bf16 values ~ 1 + N(0, 0.1^2): the learned scales
    of the Q and K normalizations."""
    rq, rk = _streams(seed, 2)
    return tuple(to_bf16_values(1.0 + 0.1 * r.standard_normal(head_dim, dtype=np.float32))
                 for r in (rq, rk))
