"""Pins of the SVDQ W4A4 oracle (CPU only).

Each check ties the oracle to something other than itself:
  * the full-rank identity: with rank = min(K, N) and unrounded factors the
    layer reduces to the plain product X W^T + b (a textbook matmul);
  * exactly representable operands (rank 0, no smoothing) reproduce X W^T + b
    exactly through the 4-bit path;
  * exact rational brute force of every rounding decision and of Y on the
    tiny workload;
  * Eckart-Young: the low-rank factors reach the optimal tail norm given by
    LAPACK's singular values;
  * hand-computed layout offsets and smoothing factors;
  * the method's purpose: SVDQ beats plain W4A4 on outlier-heavy inputs.
"""
import os

import numpy as np
import pytest

import workloads
from oracle import brute, formats, layout, svdq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------- layout
def test_scale_layout_worked_offsets():
    with open(os.path.join(GOLDEN, "sf_layout.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for C, r, c, off in rows:
        assert int(layout.sf_offset(int(r), int(c), int(C))) == int(off)


@pytest.mark.parametrize("rows,C", [(128, 4), (200, 8), (384, 48), (5, 16)])
def test_scale_layout_is_a_bijection(rows, C):
    r, c = np.meshgrid(np.arange(layout.sf_padded_rows(rows)), np.arange(C), indexing="ij")
    off = layout.sf_offset(r, c, C).reshape(-1)
    assert np.array_equal(np.sort(off), np.arange(layout.sf_padded_rows(rows) * C))
    s = np.random.default_rng(0).integers(0, 127, (rows, C), dtype=np.uint8)
    assert np.array_equal(layout.sf_unswizzle(layout.sf_swizzle(s), rows, C), s)


def test_nibble_order():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    assert layout.pack_nibbles(codes).tolist() == [[0x21, 0x43]]
    assert np.array_equal(layout.unpack_nibbles(layout.pack_nibbles(codes)), codes)


# --------------------------------------------------------------------------- smoothing
def test_smoothing_hand_cases():
    # lambda = sqrt(xmax / wmax); 1 when either maximum is 0; clamped to 2^+-20
    W = np.array([[1.0, -2.0, 0.0, 1e-30, 1.0],
                  [-0.5, 1.0, 0.0, 0.0, 4.0]], dtype=np.float32)
    xm = np.array([4.0, 8.0, 3.0, 1e30, 0.0], dtype=np.float32)
    inv = svdq.smoothing_inv_lambda(xm, W)
    # ch0: sqrt(4/1)=2 -> 0.5; ch1: sqrt(8/2)=2 -> 0.5; ch2: w=0 -> 1;
    # ch3: sqrt(1e60) clamps to 2^20; ch4: x=0 -> 1
    assert inv.tolist() == [0.5, 0.5, 1.0, 2.0 ** -20, 1.0]


def test_calib_absmax():
    X = np.array([[1.0, -3.0], [-2.0, 0.5]], dtype=np.float32)
    assert svdq.calib_absmax(X).tolist() == [2.0, 3.0]


# --------------------------------------------------------------------------- low rank
@pytest.mark.parametrize("K,N,r", [(64, 48, 8), (40, 96, 5)])
def test_lowrank_reaches_eckart_young_tail(K, N, r):
    A = np.random.default_rng(1).standard_normal((K, N))
    L1, L2 = svdq.lowrank_factors(A, r)
    s = np.linalg.svd(A, compute_uv=False)
    tail = np.sqrt(np.sum(s[r:] ** 2))
    assert abs(np.linalg.norm(A - L1 @ L2) - tail) <= 1e-10 * tail


def test_lowrank_gram_path_matches_svd_path():
    # the large-matrix path (Gram eigenvectors) on a matrix above its threshold
    rng = np.random.default_rng(2)
    K, N, r = 1100, 4000, 6
    A = rng.standard_normal((K, N)) * 0.05
    A += (rng.standard_normal((K, r)) * np.arange(r, 0, -1)) @ rng.standard_normal((r, N))
    L1, L2 = svdq.lowrank_factors(A, r)
    s = np.linalg.svd(A, compute_uv=False)
    tail = np.sqrt(np.sum(s[r:] ** 2))
    assert abs(np.linalg.norm(A - L1 @ L2) - tail) <= 1e-8 * tail
    # and the other orientation
    L1t, L2t = svdq.lowrank_factors(A.T, r)
    assert abs(np.linalg.norm(A.T - L1t @ L2t) - tail) <= 1e-8 * tail


# --------------------------------------------------------------------------- residual, tensor scale
def test_tensor_scale_is_smallest_sufficient_power_of_two():
    for e in (-20, -3, 0, 5):
        p = 2.0 ** e
        assert svdq.tensor_scale(np.array([2688.0 * p])) == p
        assert svdq.tensor_scale(np.array([np.nextafter(2688.0 * p, np.inf)])) == 2 * p
        assert svdq.tensor_scale(np.array([2688.0 * p * 0.75])) == p
    assert svdq.tensor_scale(np.zeros(3)) == 1.0


def test_residual_reconstructs_weight_through_smoothing():
    rng = np.random.default_rng(3)
    N, K, r = 24, 32, 4
    W = rng.standard_normal((N, K)).astype(np.float32)
    inv = np.exp2(rng.integers(-3, 3, K)).astype(np.float32) * np.float32(1.25)
    L1s = formats.round_to_bf16(rng.standard_normal((K, r)))
    L2 = formats.round_to_bf16(rng.standard_normal((r, N)))
    R = svdq.residual(W, inv, L1s, L2)
    X = rng.standard_normal((7, K))
    lhs = (X * inv.astype(np.float64)) @ R + X @ L1s @ L2
    assert np.allclose(lhs, X @ W.T.astype(np.float64), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- identities of the layer
@pytest.mark.parametrize("N,K", [(32, 32), (48, 32), (32, 64), (64, 128)])
def test_full_rank_layer_is_plain_matmul(N, K):
    """rank = min(K, N) with unrounded factors: R vanishes (up to float64
    rounding) and the layer returns X W^T + b."""
    rng = np.random.default_rng(4)
    W = rng.standard_normal((N, K)).astype(np.float32)
    X = workloads.to_bf16_values(rng.standard_normal((16, K)).astype(np.float32) * 3)
    b = rng.standard_normal(N)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), min(N, K), factor_rounding="none")
    W_hat = W.T.astype(np.float64) / packed["inv_lambda"].astype(np.float64)[:, None]
    assert np.max(np.abs(packed["R"])) <= 1e-12 * np.max(np.abs(W_hat))
    Y = svdq.linear_forward(X, packed, b)["Y"]
    ref = X.astype(np.float64) @ W.T.astype(np.float64) + b
    assert np.max(np.abs(Y - ref)) <= 1e-12 * np.max(np.abs(ref))


def _representable(rng, rows, K, scale_bytes):
    """rows x K values code * scale, each 16-block holding a +-6 so that its
    amax/6 is exactly the block's scale."""
    codes = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    codes[:, ::16] = np.where(rng.random((rows, K // 16)) < 0.5, 7, 15)
    sc = rng.choice(scale_bytes, (rows, K // 16)).astype(np.uint8)
    vals = formats.e2m1_decode(codes) * np.repeat(formats.e4m3_decode(sc), 16, axis=1)
    return codes, sc, vals


def test_representable_activations_roundtrip():
    rng = np.random.default_rng(5)
    codes, sc, vals = _representable(rng, 40, 128, np.arange(1, 0x7F))
    # x_hat = x exactly when inv_lambda is a power of two: scale X by 2^-e
    inv = np.exp2(rng.integers(-2, 3, 128)).astype(np.float32)
    X = (vals / inv.astype(np.float64)[None, :]).astype(np.float32)
    # keep X bf16: e2m1 x e4m3 x 2^e has at most 6 significant bits
    assert np.array_equal(workloads.to_bf16_values(X), X)
    _, q, s = svdq.quantize_activations(X, inv)
    # -0 codes (value 0 with sign) come back as +0 only if the input was +0
    want = np.where(formats.e2m1_decode(codes) == 0, np.where(np.signbit(vals), 8, 0), codes)
    assert np.array_equal(s, sc)
    assert np.array_equal(q, want)


def test_representable_weights_give_exact_plain_product():
    """rank 0, lambda = 1, W = code * scale * s_T with s_T reached exactly:
    the 4-bit path reproduces X W^T + b exactly (compared in Fractions)."""
    rng = np.random.default_rng(6)
    N, K, M = 16, 64, 6
    wc, ws, wv = _representable(rng, N, K, np.arange(0x30, 0x70))
    ws[0, 0] = 0x7E  # one block scale 448 with a +-6 in it: max|R| = 2688 s_T
    wv = formats.e2m1_decode(wc) * np.repeat(formats.e4m3_decode(ws), 16, axis=1)
    s_T = 2.0 ** -12
    W = (wv * s_T).astype(np.float32)
    assert np.array_equal(W.astype(np.float64), wv * s_T)
    ac, asc, av = _representable(rng, M, K, np.arange(0x20, 0x60))
    X = av.astype(np.float32)
    # x_absmax equal to the weight column maxima makes lambda = 1
    xm = np.max(np.abs(W), axis=0)
    packed = svdq.pack_weights(W, xm, 0)
    assert np.all(packed["inv_lambda"] == 1.0)
    assert packed["s_T"] == s_T
    b = workloads.to_bf16_values(rng.standard_normal(N).astype(np.float32))
    out = svdq.linear_forward(X, packed, b)
    from fractions import Fraction
    for m in range(M):
        for n in range(N):
            want = sum(Fraction(float(X[m, k])) * Fraction(float(W[n, k])) for k in range(K)) \
                + Fraction(float(b[n]))
            assert Fraction(out["Y"][m, n]) == want


# --------------------------------------------------------------------------- brute force, tiny workload
@pytest.fixture(scope="module")
def tiny():
    case = workloads.CASES["tiny"]
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), case.rank)
    out = svdq.linear_forward(X, packed, b)
    return case, X, W, b, packed, out


def test_tiny_activation_quantization_brute_force(tiny):
    case, X, W, b, packed, out = tiny
    inv = packed["inv_lambda"]
    for m in range(0, case.M, 7):
        codes, scales = brute.quantize_act_row(X[m].tolist(), inv.tolist())
        assert codes == out["a_codes"][m].tolist()
        assert scales == out["a_scales"][m].tolist()


def test_tiny_weight_quantization_brute_force(tiny):
    case, X, W, b, packed, out = tiny
    from fractions import Fraction
    R = packed["R"]
    for n in range(0, case.N, 5):
        codes, scales = brute.quantize_weight_col(R[:, n].tolist(), Fraction(packed["s_T"]))
        assert codes == packed["w_codes"][n].tolist()
        assert scales == packed["w_scales"][n].tolist()


def test_tiny_gemm_brute_force(tiny):
    """Y from the codes in exact rationals equals the oracle's float64 Y to
    float64 rounding (relative 1e-13)."""
    case, X, W, b, packed, out = tiny
    rows = [0, 17, 127]
    cols = [0, 5, 100, 255]
    Yx = brute.gemm_exact(out["a_codes"][rows].tolist(), out["a_scales"][rows].tolist(),
                          packed["w_codes"][cols].tolist(), packed["w_scales"][cols].tolist(),
                          packed["s_T"], out["lora_act"][rows].tolist(),
                          packed["L2"][:, cols].tolist(), b[cols].tolist())
    scale = np.max(np.abs(out["Y"]))
    for i, m in enumerate(rows):
        for j, n in enumerate(cols):
            assert abs(float(Yx[i][j]) - out["Y"][m, n]) <= 1e-13 * scale


def test_tiny_lora_is_rounded_exact_sum(tiny):
    case, X, W, b, packed, out = tiny
    from fractions import Fraction
    for m in (0, 64):
        for i in (0, 7, 15):
            exact = sum(Fraction(float(X[m, k])) * Fraction(float(packed["L1s"][k, i]))
                        for k in range(case.K))
            # nearest bf16 of the exact sum
            r = formats.round_to_bf16(np.array([float(exact)]))[0]
            assert out["lora_act"][m, i] == r


def test_tiny_weights_are_bf16_and_residual_small(tiny):
    case, X, W, b, packed, out = tiny
    formats.bf16_bits(packed["L1s"])
    formats.bf16_bits(packed["L2"])
    W_hat = W.T.astype(np.float64) / packed["inv_lambda"].astype(np.float64)[:, None]
    assert np.linalg.norm(packed["R"]) < np.linalg.norm(W_hat)


# --------------------------------------------------------------------------- the method's purpose
def test_svdq_beats_naive_w4a4_on_outliers():
    case = workloads.custom_case(256, 512, 384, 32, seed=7, outlier_channels=5,
                                 outlier_scale=50.0, planted_rank=32)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    exact = X.astype(np.float64) @ W.T.astype(np.float64) + b
    nrm = np.linalg.norm(exact)
    e_svdq = np.linalg.norm(svdq.linear_forward(
        X, svdq.pack_weights(W, svdq.calib_absmax(X), 32), b)["Y"] - exact) / nrm
    e_smooth = np.linalg.norm(svdq.linear_forward(
        X, svdq.pack_weights(W, svdq.calib_absmax(X), 0), b)["Y"] - exact) / nrm
    e_naive = np.linalg.norm(svdq.naive_w4a4(X, W, b) - exact) / nrm
    assert e_svdq < e_smooth < e_naive
    assert e_svdq < 0.5 * e_naive


# --------------------------------------------------------------------------- GELU glue
def test_gelu_tanh_identities():
    from scipy.special import erf
    y = np.linspace(-8, 8, 2001)
    g = svdq.gelu_tanh(y)
    exact_erf = 0.5 * y * (1 + erf(y / np.sqrt(2)))
    assert np.max(np.abs(g - exact_erf)) < 1e-3       # the tanh form approximates erf-GELU
    # x Phi(x) structure: g(y) - g(-y) = y for the tanh form too
    assert np.max(np.abs(g - svdq.gelu_tanh(-y) - y)) < 1e-12
    assert svdq.gelu_tanh_bf16(np.array([0.0]))[0] == 0.0
    big = np.array([30.0, -30.0])
    assert svdq.gelu_tanh_bf16(big).tolist() == [30.0, -0.0]


def test_gelu_tanh_matches_library_and_taylor():
    """The constants of the tanh form: torch's own tanh-approximated GELU in
    float64 (a library routine, not this code) agrees to rounding; and both
    GELU forms share the expansion y/2 + y^2/sqrt(2 pi) + O(y^4), which fixes
    the sqrt(2/pi) factor independently of any implementation."""
    import torch
    y = np.concatenate([np.linspace(-12, 12, 4801), [1e-30, -1e-30, 1e3, -1e3]])
    ref = torch.nn.functional.gelu(torch.from_numpy(y), approximate="tanh").numpy()
    assert np.max(np.abs(svdq.gelu_tanh(y) - ref) / (1.0 + np.abs(y))) < 1e-14
    # (g(h) - h/2) / h^2 = c/2 + (c a - c^3/3) h^2 / 2 + ..., |that h^2 term| < 0.07 h^2
    for h in (1e-3, 1e-4):
        second = (svdq.gelu_tanh(np.array([h]))[0] - h / 2) / h ** 2
        assert abs(second - 1 / np.sqrt(2 * np.pi)) < h ** 2
