"""Pins of the fused-QKV-epilogue oracle (oracle/qkv.py) against things other
than itself: a library routine (torch's RMS normalization in float64), complex
multiplication for the rotation, invariants of both steps, and a worked
example computed by hand that also fixes the order of the two steps."""
import numpy as np
import pytest
import torch

import workloads
from oracle import qkv


def _rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------- RMS normalization
def test_rms_norm_matches_torch_float64():
    y = _rng(1).standard_normal((37, 4 * 128)) * 3.0
    w = 1.0 + 0.1 * _rng(2).standard_normal(128)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(y.reshape(37, 4, 128)), (128,),
                                       weight=torch.from_numpy(w), eps=1e-6)
    got = qkv.rms_norm_heads(y, w, 128, 1e-6)
    assert np.max(np.abs(got - ref.numpy().reshape(37, 512))) < 1e-13


def test_rms_norm_invariants():
    y = _rng(3).standard_normal((9, 3 * 64)) * 5.0
    ones = np.ones(64)
    n = qkv.rms_norm_heads(y, ones, 64, 0.0).reshape(9, 3, 64)
    assert np.allclose(np.sqrt(np.mean(n * n, axis=2)), 1.0, rtol=0, atol=1e-13)  # unit RMS
    # scale invariance per head (eps = 0): each head scaled by its own positive factor
    c = np.repeat(np.array([0.5, 7.0, 1e-3]), 64)[None, :]
    assert np.allclose(qkv.rms_norm_heads(y * c, ones, 64, 0.0), n.reshape(9, -1), atol=1e-12)
    # a constant head a * 1 with eps: a / sqrt(a^2 + eps) * w
    a, eps = 0.01, 1e-6
    w = np.arange(1, 65, dtype=np.float64)
    got = qkv.rms_norm_heads(np.full((1, 64), a), w, 64, eps)[0]
    assert np.allclose(got, a / np.sqrt(a * a + eps) * w, rtol=1e-14, atol=0)
    # heads are independent: changing head 1 leaves heads 0 and 2
    y2 = y.copy()
    y2[:, 64:128] *= -3.0
    n2 = qkv.rms_norm_heads(y2, ones, 64, 0.0)
    assert np.array_equal(n2[:, :64], n.reshape(9, -1)[:, :64])
    assert np.array_equal(n2[:, 128:], n.reshape(9, -1)[:, 128:])


# --------------------------------------------------------------------------- rotary embedding
def test_rope_is_complex_multiplication():
    M, H, D = 11, 3, 16
    x = _rng(4).standard_normal((M, H * D))
    theta = _rng(5).uniform(-7, 7, (M, D // 2))
    got = qkv.rope_pairs(x, np.cos(theta), np.sin(theta), D).reshape(M, H, D)
    z = x.reshape(M, H, D)[:, :, 0::2] + 1j * x.reshape(M, H, D)[:, :, 1::2]
    zr = z * np.exp(1j * theta)[:, None, :]
    assert np.max(np.abs(got[:, :, 0::2] - zr.real)) < 1e-14
    assert np.max(np.abs(got[:, :, 1::2] - zr.imag)) < 1e-14


def test_rope_invariants():
    M, D = 6, 8
    x = _rng(6).standard_normal((M, 2 * D))
    theta = _rng(7).uniform(-3, 3, (M, D // 2))
    r = qkv.rope_pairs(x, np.cos(theta), np.sin(theta), D)
    pair_norm = lambda v: np.hypot(v[:, 0::2], v[:, 1::2])  # noqa: E731
    assert np.allclose(pair_norm(r), pair_norm(x), rtol=1e-14)            # rotations keep norms
    back = qkv.rope_pairs(r, np.cos(-theta), np.sin(-theta), D)
    assert np.allclose(back, x, atol=1e-14)                               # turn back by -theta
    zero = np.zeros_like(theta)
    assert np.array_equal(qkv.rope_pairs(x, np.cos(zero), np.sin(zero), D), x)  # theta = 0


def test_rope_relative_position_property():
    """With angles linear in the position (the workload's tables), the dot
    product of a rotated query and a rotated key depends only on the
    difference of their positions."""
    pos = np.array([[0, 3, 5], [0, 10, 1], [0, 3 + 4, 5 - 2], [0, 10 + 4, 1 - 2]])
    cos, sin = workloads.make_rope_tables(pos)
    q, k = _rng(8).standard_normal((2, 128))
    Q = qkv.rope_pairs(np.stack([q, q, q, q]), cos.astype(np.float64), sin.astype(np.float64))
    K = qkv.rope_pairs(np.stack([k, k, k, k]), cos.astype(np.float64), sin.astype(np.float64))
    # tables are float32 samples of cos and sin: agreement to float32 rounding
    assert abs(Q[0] @ K[1] - Q[2] @ K[3]) < 1e-5 * np.abs(q).sum() * np.abs(k).sum() / 16


def test_rope_tables_of_the_workload():
    pos = workloads.rope_positions()
    assert pos.shape == (4608, 3)
    assert np.all(pos[:512] == 0)
    assert tuple(pos[512 + 64 * 5 + 7]) == (0, 5, 7)
    cos, sin = workloads.make_rope_tables(pos)
    assert cos.shape == (4608, 64) and sin.dtype == np.float32
    assert np.all(cos[:512] == 1.0) and np.all(sin[:512] == 0.0)      # text tokens: no turn
    # patch (5, 7): axis 1 pair 0 turns by 5 radians, axis 2 pair 0 by 7
    assert sin[512 + 64 * 5 + 7, 8] == np.float32(np.sin(5.0))
    assert cos[512 + 64 * 5 + 7, 8 + 28] == np.float32(np.cos(7.0))


# --------------------------------------------------------------------------- the composite
def test_worked_example_by_hand():
    """One token, head_dim 4, one head each of Q, K, V, eps = 0.
    Q head (3, 4, 0, 0): mean square 25/4, RMS 2.5, normalized (1.2, 1.6, 0, 0),
    times w_q = (1, 2, 1, 1): (1.2, 3.2, 0, 0); pair 0 turned by 90 degrees
    (a, b) -> (-b, a): (-3.2, 1.2, 0, 0).  (Rotating first would give
    (-4, 3) -> (-1.6, 1.2) -> (-1.6, 2.4): the order matters.)
    K head (0, 0, 1, 1): RMS sqrt(1/2), normalized (0, 0, sqrt 2, sqrt 2), times
    w_k = 1; pair 1 turned by 180 degrees: (0, 0, -sqrt 2, -sqrt 2).
    V head passes unchanged."""
    y = np.array([[3.0, 4.0, 0.0, 0.0, 0.0, 0.0, 1.0, 1.0, 9.0, -8.0, 7.0, 0.5]])
    cos = np.array([[0.0, -1.0]])
    sin = np.array([[1.0, 0.0]])
    out = qkv.qkv_norm_rope(y, np.array([1.0, 2.0, 1.0, 1.0]), np.ones(4), cos, sin,
                            head_dim=4, eps=0.0)
    r2 = np.sqrt(2.0)
    want = [-3.2, 1.2, 0.0, 0.0, 0.0, 0.0, -r2, -r2, 9.0, -8.0, 7.0, 0.5]
    assert np.allclose(out[0], want, rtol=0, atol=1e-15)


def test_composite_is_norm_then_rope_on_q_and_k_only():
    M, H, D = 5, 2, 8
    y = _rng(9).standard_normal((M, 3 * H * D)) * 4.0
    w_q, w_k = 1.0 + 0.1 * _rng(10).standard_normal((2, D))
    theta = _rng(11).uniform(-3, 3, (M, D // 2))
    c, s = np.cos(theta), np.sin(theta)
    out = qkv.qkv_norm_rope(y, w_q, w_k, c, s, head_dim=D)
    hd = H * D
    assert np.array_equal(out[:, 2 * hd:], y[:, 2 * hd:])
    assert np.allclose(out[:, :hd], qkv.rope_pairs(qkv.rms_norm_heads(y[:, :hd], w_q, D), c, s, D))
    assert np.allclose(out[:, hd:2 * hd],
                       qkv.rope_pairs(qkv.rms_norm_heads(y[:, hd:2 * hd], w_k, D), c, s, D))
    # K uses w_k, not w_q
    assert not np.allclose(out[:, hd:2 * hd],
                           qkv.rope_pairs(qkv.rms_norm_heads(y[:, hd:2 * hd], w_q, D), c, s, D))


@pytest.mark.parametrize("mistake", ["rope_first", "no_eps", "mean_abs", "sin_sign"])
def test_worked_example_catches_plausible_mistakes(mistake):
    """Each plausible slip in the composite changes the hand-worked output."""
    y = np.array([[3.0, 4.0, 0.0, 0.0, 0.0, 0.0, 1.0, 1.0, 9.0, -8.0, 7.0, 0.5]])
    cos, sin = np.array([[0.0, -1.0]]), np.array([[1.0, 0.0]])
    w_q, w_k = np.array([1.0, 2.0, 1.0, 1.0]), np.ones(4)
    good = qkv.qkv_norm_rope(y, w_q, w_k, cos, sin, head_dim=4, eps=1e-2)
    q = y[:, :4]
    if mistake == "rope_first":
        bad = qkv.rms_norm_heads(qkv.rope_pairs(q, cos, sin, 4), w_q, 4, 1e-2)
    elif mistake == "no_eps":
        bad = qkv.rope_pairs(qkv.rms_norm_heads(q, w_q, 4, 0.0), cos, sin, 4)
    elif mistake == "mean_abs":
        bad = qkv.rope_pairs(q / (np.mean(np.abs(q)) + 1e-2) * w_q, cos, sin, 4)
    else:  # the pair turned the other way (a swapped pair or a sign slip)
        bad = qkv.rope_pairs(qkv.rms_norm_heads(q, w_q, 4, 1e-2), cos, -sin, 4)
    assert not np.allclose(good[:, :4], bad, atol=1e-6)
