"""Pins of the INT4-variant oracle (CPU only).

Each check ties oracle/int4.py to something other than itself:
  * exact rational brute force of every rounding decision (binary32 quotient,
    bf16 scale, half-even integer codes) and of Y on small inputs;
  * hand-worked groups: scales that are powers of two, ties, clamping, zero,
    infinite and subnormal groups;
  * the byte layout against hand-packed bytes;
  * exactly representable operands reproduce the integer product exactly;
  * the method's purpose: SVDQ beats plain INT4 W4A4 on outlier-heavy inputs.
"""
from fractions import Fraction

import numpy as np
import pytest

import workloads
from oracle import brute, int4, svdq


def _row(vals, K=64):
    x = np.zeros((1, K), np.float32)
    x[0, :len(vals)] = vals
    return x


# --------------------------------------------------------------------------- hand cases
def test_power_of_two_scale_and_ties():
    # amax 7 -> s = 1 exactly: codes are the values rounded half to even
    vals = [7.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, -7.0, 6.5, 5.5, 0.25]
    _, codes, scales = int4.quantize_activations(_row(vals), np.ones(64, np.float32))
    assert scales[0, 0] == 1.0
    assert codes[0, :len(vals)].tolist() == [7, 2, 4, -2, 0, 2, 0, -7, 6, 6, 0]
    # amax 14 -> s = 2
    _, codes, scales = int4.quantize_activations(_row([14.0, 5.0, -3.0]), np.ones(64, np.float32))
    assert scales[0, 0] == 2.0 and codes[0, :3].tolist() == [7, 2, -2]


def test_scale_is_bf16_of_binary32_quotient():
    # amax 1 -> 1/7 = 0.142857...: binary32 quotient, then nearest bf16 (8 bits)
    _, codes, scales = int4.quantize_activations(_row([1.0, -0.5]), np.ones(64, np.float32))
    s = float(brute.round_binary(brute.round_binary(Fraction(1, 7), 24), 8))
    assert scales[0, 0] == s == 0.142578125
    # 1 / s = 7.0137 -> 7 ; -0.5 / s = -3.5068 -> -4
    assert codes[0, :2].tolist() == [7, -4]


def test_codes_never_minus_eight_and_error_within_half_scale():
    rng = np.random.default_rng(3)
    X = (rng.standard_normal((64, 512)) * np.exp(rng.uniform(-8, 8, (64, 1)))).astype(np.float32)
    X = X.astype(np.float64)
    from oracle.formats import round_to_bf16
    X = round_to_bf16(X).astype(np.float32)
    xhat, codes, scales = int4.quantize_activations(X, np.ones(512, np.float32))
    assert codes.min() >= -7 and codes.max() <= 7
    err = np.abs(xhat.astype(np.float64) - int4.dequantize(codes, scales))
    assert np.all(err <= np.repeat(scales, 64, axis=1) / 2)


def test_degenerate_groups():
    inv = np.ones(192, np.float32)
    X = np.zeros((1, 192), np.float32)
    X[0, 64] = np.inf          # group 1: infinite scale -> codes 0
    X[0, 65] = 3.0
    X[0, 128] = 2.0 ** -140    # group 2: scale rounds to 0 -> codes 0
    _, codes, scales = int4.quantize_activations(X, inv)
    assert scales[0].tolist()[0] == 0.0 and np.isinf(scales[0, 1]) and scales[0, 2] == 0.0
    assert not codes.any()


def test_subnormal_groups_follow_the_binary32_definition():
    """Below 7 * 2^-126 the binary32 quotient is itself rounded; the oracle
    must agree with the brute force that rounds it the same way, including on
    the amax values where that differs from the exact quotient's rounding."""
    amaxes = [np.float32(2.0 ** -130) * np.float32(1 + i / 64) for i in range(64)]
    amaxes += [np.float32(np.ldexp(1.0 + j / 8.0, -149 + e)) for e in (0, 3, 9, 17) for j in range(8)]
    # amax / 7 within half a binary32 subnormal step of a bf16 midpoint
    # (2j + 1) 2^-134 without sitting on it: the two roundings part there
    amaxes += [np.float32(np.ldexp(7.0 * (2 * j + 1) * 2 ** 15 + d, -149))
               for j in (0, 1, 5) for d in (-3, -2, -1, 1, 2, 3)]
    differs = 0
    for a in amaxes:
        _, codes, scales = int4.quantize_activations(_row([a, a / 3]), np.ones(64, np.float32))
        c, s = brute.int4_act_row(_row([a, a / 3])[0].tolist(), [1.0] * 64)
        assert scales[0, 0] == float(s[0]) and codes[0].tolist() == c
        differs += brute.round_binary(Fraction(float(a)) / 7, 8) != s[0]
    assert differs > 0  # the cases exist, so the definition matters


def test_weight_scale_is_bf16_of_exact_quotient():
    R = np.zeros((64, 1))
    R[0, 0] = 1.0
    R[1, 0] = -0.75
    codes, scales = int4.quantize_weight_residual(R)
    assert scales[0, 0] == 0.142578125 and codes[0, :2].tolist() == [7, -5]


# --------------------------------------------------------------------------- layout
def test_code_bytes():
    codes = np.array([[-1, 3, 7, -8, 0, -7]], np.int8)
    packed = int4.pack_codes(codes)
    assert packed.tolist() == [[0x3F, 0x87, 0x90]]
    assert np.array_equal(int4.unpack_codes(packed), codes)


# --------------------------------------------------------------------------- brute force
@pytest.fixture(scope="module")
def small():
    case = workloads.custom_case(48, 256, 40, 8, seed=11, outlier_channels=3,
                                 outlier_scale=40.0, planted_rank=8)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = int4.pack_weights(W, svdq.calib_absmax(X), case.rank)
    return case, X, W, b, packed, int4.linear_forward(X, packed, b)


def test_small_activation_quantization_brute_force(small):
    case, X, W, b, packed, out = small
    for m in range(0, case.M, 5):
        codes, scales = brute.int4_act_row(X[m].tolist(), packed["inv_lambda"].tolist())
        assert codes == out["a_codes"][m].tolist()
        assert [float(s) for s in scales] == out["a_scales"][m].tolist()


def test_small_weight_quantization_brute_force(small):
    case, X, W, b, packed, out = small
    for n in range(0, case.N, 3):
        codes, scales = brute.int4_weight_col(packed["R"][:, n].tolist())
        assert codes == packed["w_codes"][n].tolist()
        assert [float(s) for s in scales] == packed["w_scales"][n].tolist()


def test_small_gemm_brute_force(small):
    case, X, W, b, packed, out = small
    rows, cols = [0, 13, 47], [0, 9, 39]
    Yx = brute.int4_gemm_exact(out["a_codes"][rows].tolist(), out["a_scales"][rows].tolist(),
                               packed["w_codes"][cols].tolist(), packed["w_scales"][cols].tolist(),
                               out["lora_act"][rows].tolist(), packed["L2"][:, cols].tolist(),
                               b[cols].tolist())
    scale = np.max(np.abs(out["Y"]))
    for i, m in enumerate(rows):
        for j, n in enumerate(cols):
            assert abs(float(Yx[i][j]) - out["Y"][m, n]) <= 1e-13 * scale


def test_representable_operands_give_exact_integer_product():
    """Codes and power-of-two scales chosen directly: Y is the integer dot
    product times the scale product, exactly."""
    rng = np.random.default_rng(5)
    M, N, K = 5, 7, 192
    a = rng.integers(-7, 8, (M, K)).astype(np.int8)
    w = rng.integers(-7, 8, (N, K)).astype(np.int8)
    sa = np.ldexp(1.0, rng.integers(-6, 6, (M, K // 64)))
    sw = np.ldexp(1.0, rng.integers(-6, 6, (N, K // 64)))
    Y = int4.gemm_reference(a, sa, w, sw, None, None, None)
    for m in range(M):
        for n in range(N):
            want = sum(int(a[m, k]) * int(w[n, k]) * sa[m, k // 64] * sw[n, k // 64]
                       for k in range(K))
            assert Y[m, n] == want


# --------------------------------------------------------------------------- the method's purpose
def test_int4_svdq_beats_naive_int4_on_outliers():
    case = workloads.custom_case(256, 512, 384, 32, seed=7, outlier_channels=5,
                                 outlier_scale=50.0, planted_rank=32)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    exact = X.astype(np.float64) @ W.T.astype(np.float64) + b
    nrm = np.linalg.norm(exact)
    e_svdq = np.linalg.norm(int4.linear_forward(
        X, int4.pack_weights(W, svdq.calib_absmax(X), 32), b)["Y"] - exact) / nrm
    e_naive = np.linalg.norm(int4.naive_w4a4(X, W, b) - exact) / nrm
    assert e_svdq < 0.5 * e_naive
