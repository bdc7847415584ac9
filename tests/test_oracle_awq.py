"""Pins of the AWQ W4A16 oracle (CPU only): round trip of exactly
representable groups, the asymmetric quantizer's error bound, degenerate
groups, and an exact rational brute-force GEMV."""
from fractions import Fraction

import numpy as np

import workloads
from oracle import awq, formats, layout


def test_representable_groups_roundtrip():
    rng = np.random.default_rng(0)
    N, K = 8, 256
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    q[:, ::64] = 0
    q[:, 1::64] = 15                         # every group spans the full 0..15 range
    s = formats.round_to_f16(np.exp2(rng.uniform(-9, -4, (N, K // 64))))
    z = rng.integers(0, 16, (N, K // 64)).astype(np.float64)
    W = (q - np.repeat(z, 64, axis=1)) * np.repeat(s, 64, axis=1)
    assert np.array_equal(W.astype(np.float32).astype(np.float64), W)
    p = awq.awq_pack(W.astype(np.float32))
    assert np.array_equal(p["q"], q)
    assert np.array_equal(p["scales"], s)
    assert np.array_equal(p["zeros"], z)


def test_dequant_error_bound():
    W = np.random.default_rng(1).standard_normal((64, 512)).astype(np.float32) * 0.02
    p = awq.awq_pack(W)
    Wd = awq.awq_dequant(p["qweight"], p["scales"], p["zeros"])
    s = np.repeat(p["scales"], 64, axis=1)
    # |w - (q - z) s| <= s/2 (rounding) + s * |z - fp16(z)| + slack for the
    # fp16 rounding of s (relative 2^-11 over at most 15 steps)
    err = np.abs(W - Wd)
    assert np.all(err <= s * (0.5 + 2.0 ** -11 * 16) + s * 2.0 ** -7)
    assert np.mean(err / s) < 0.3


def test_degenerate_groups():
    W = np.zeros((2, 128), dtype=np.float32)
    W[1, 64:] = 0.75
    p = awq.awq_pack(W)
    assert p["scales"].tolist() == [[1.0, 1.0], [1.0, 1.0]]
    Wd = awq.awq_dequant(p["qweight"], p["scales"], p["zeros"])
    assert np.array_equal(Wd, W.astype(np.float64))


def test_nibble_layout():
    W = np.zeros((1, 64), dtype=np.float32)
    W[0, 0] = -1.0
    W[0, 1] = 1.0
    p = awq.awq_pack(W)
    # min -1, max 1: s = fp16(2/15), z = fp16(1/s); k=0 -> code 0, k=1 -> code 15
    assert p["qweight"][0, 0] == (0 | (15 << 4))


def test_gemv_brute_force():
    rng = np.random.default_rng(2)
    M, N, K = 3, 5, 128
    X = workloads.to_bf16_values(rng.standard_normal((M, K)).astype(np.float32))
    W = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    b = workloads.to_bf16_values(rng.standard_normal(N).astype(np.float32) * 0.01)
    p = awq.awq_pack(W)
    Y = awq.awq_linear(X, p["qweight"], p["scales"], p["zeros"], b)
    q = layout.unpack_nibbles(p["qweight"])
    for m in range(M):
        for n in range(N):
            exact = Fraction(float(b[n]))
            for k in range(K):
                g = k // 64
                exact += Fraction(float(X[m, k])) * (int(q[n, k]) - Fraction(p["zeros"][n, g])) \
                    * Fraction(p["scales"][n, g])
            assert abs(float(exact) - Y[m, n]) <= 1e-14 * max(1.0, abs(float(exact)))
