"""Oracle of the SVDQuant W4A4 linear layer, NVFP4 variant.

What the pages fix ([dothoosh], SVDQuant and fused-kernel paragraphs;
[hamidun-ar] "What are Nunchaku and SVDQuant"; [nextgz] "Why is W4A4
different from weight-only backends?"):
  * both weights and activations of the heavy linears go to 4 bit (W4A4);
  * activation outliers are migrated into the weights (smoothing);
  * the hardest part of each weight matrix is kept as a small 16-bit
    low-rank branch; the residual is quantized to 4 bit;
  * the low-rank down projection runs with the activation quantization, the
    low-rank up projection with the 4-bit product;
  * NVFP4, group size 16, rank 32, compute dtype bfloat16 ("quantization_config"
    block of [dothoosh]).

The layer therefore computes
    Y = Q4(X_hat) . Q4(R) * s_T  +  (X . L1s) . L2  +  b
with X_hat = X diag(inv_lambda).

Readings of what the pages leave open (each used below):
  R1  lambda_j = sqrt(max|X_j| / max|W_j|) over calibration rows and output
      channels; lambda_j = 1 if either maximum is 0; clamped to [2^-20, 2^20];
      stored as inv_lambda = fl32(1/lambda) (float64 division, one rounding).
  R2  low rank: top-r SVD of W_hat^T = diag(1/inv_lambda) W^T (K x N);
      L1 = U_r Sigma_r, L2 = V_r^T.
  R3  the down projection uses L1s = bf16(inv_lambda (.) L1) on the raw bf16
      X (so X . L1s approximates X_hat . L1); L2 is stored as bf16(L2).
  R4  the residual is taken against the factors exactly as the device uses
      them:  R[k,n] = (W[n,k] - sum_i L1s[k,i] L2[i,n]) / inv_lambda[k],
      float64, the sum over i in increasing order, products exact (bf16 x bf16),
      one rounding per addition, then one subtraction and one division.  Then
      X_hat R + X L1s L2 = X W^T exactly in real arithmetic.
  R5  weight tensor scale s_T = the smallest power of two p with
      6 * 448 * p >= max|R|; s_T = 1 if R == 0.
  R6  weight block scale s_b = RNE_e4m3(amax_b / (6 s_T)) over 16 consecutive
      k of one output channel; codes q = RNE_e2m1(R / (s_b s_T)); a block with
      s_b = 0 gets all codes +0.
  R7  activations have no tensor scale: x_hat = fl32(x * inv_lambda_j) (one
      binary32 multiply); s = RNE_e4m3(amax/6) over 16 consecutive k; codes
      q = RNE_e2m1(x_hat / s) with the sign bit of x_hat; s = 0 gives codes +0.
  R8  lora_act = RNE_bf16(sum_k x_k L1s[k,i]) of the exact sum.
  R9  Y is returned unrounded (float64); the device rounds once to bf16.
Quotients in R6/R7 are rounded from the exact real quotient.  A float64
division followed by rounding to the coarse grid gives the same result:
the float64 quotient of a 24-bit numerator cannot land on a grid midpoint
unless the real quotient is exactly that midpoint.
"""
from __future__ import annotations

import numpy as np

from .formats import (
    e2m1_decode,
    e4m3_decode,
    rne_e2m1,
    rne_e4m3,
    round_to_bf16,
    bf16_bits,
)
from .layout import pack_nibbles, sf_swizzle

LAMBDA_MIN = 2.0 ** -20
LAMBDA_MAX = 2.0 ** 20
E2M1_MAX = 6.0
E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# offline: calibration, smoothing, low rank, residual quantization
# ---------------------------------------------------------------------------


def calib_absmax(X: np.ndarray) -> np.ndarray:
    """max_m |X[m, j]| per input channel, as float32 (exact)."""
    X = np.asarray(X, dtype=np.float32)
    if X.shape[0] == 0:
        return np.zeros(X.shape[1], dtype=np.float32)
    return np.max(np.abs(X), axis=0).astype(np.float32)


def smoothing_inv_lambda(x_absmax: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Reading R1 of the smoothing step ([dothoosh], SVDQuant paragraph: the
    activation outliers are moved into the weights)."""
    xm = np.asarray(x_absmax, dtype=np.float32).astype(np.float64)
    wm = np.max(np.abs(np.asarray(W, dtype=np.float32)), axis=0).astype(np.float64)
    lam = np.ones_like(xm)
    ok = (xm > 0) & (wm > 0)
    lam[ok] = np.sqrt(xm[ok] / wm[ok])
    lam = np.clip(lam, LAMBDA_MIN, LAMBDA_MAX)
    return (1.0 / lam).astype(np.float32)


def lowrank_factors(A: np.ndarray, r: int):
    """Reading R2: best rank-r factors of A (K x N) by SVD, L1 = U_r S_r,
    L2 = V_r^T.  Uses LAPACK's SVD for moderate sizes and the eigenvectors of
    the smaller Gram matrix otherwise (same subspace, exact up to rounding)."""
    A = np.asarray(A, dtype=np.float64)
    K, N = A.shape
    if r == 0:
        return np.zeros((K, 0)), np.zeros((0, N))
    if K * N <= 4 * 1024 * 1024:
        U, S, Vt = np.linalg.svd(A, full_matrices=False)
        return U[:, :r] * S[:r][None, :], Vt[:r, :].copy()
    if K <= N:
        G = A @ A.T
        w, V = np.linalg.eigh(G)
        idx = np.argsort(w)[::-1][:r]
        U = V[:, idx]
        L2 = U.T @ A                       # = S_r V_r^T
        S = np.sqrt(np.maximum(w[idx], 0.0))
        safe = np.where(S > 0, S, 1.0)
        return U * S[None, :], L2 / safe[:, None]
    G = A.T @ A
    w, V = np.linalg.eigh(G)
    idx = np.argsort(w)[::-1][:r]
    Vr = V[:, idx]
    return A @ Vr, Vr.T.copy()


def residual(W: np.ndarray, inv_lambda: np.ndarray, L1s: np.ndarray, L2: np.ndarray) -> np.ndarray:
    """Reading R4, evaluated in the stated order.  Returns R as [K, N] float64."""
    W = np.asarray(W, dtype=np.float32).astype(np.float64)
    N, K = W.shape
    acc = np.zeros((K, N), dtype=np.float64)
    for i in range(L1s.shape[1]):
        acc += np.outer(L1s[:, i], L2[i, :])
    inv = np.asarray(inv_lambda, dtype=np.float32).astype(np.float64)
    return (W.T - acc) / inv[:, None]


def tensor_scale(R: np.ndarray) -> float:
    """Reading R5: smallest power of two p with 2688 p >= max|R| (exact
    comparisons on powers of two)."""
    amax = float(np.max(np.abs(R))) if R.size else 0.0
    if amax == 0.0:
        return 1.0
    bound = E2M1_MAX * E4M3_MAX
    e = int(np.ceil(np.log2(amax / bound)))
    while bound * 2.0 ** e < amax:
        e += 1
    while bound * 2.0 ** (e - 1) >= amax:
        e -= 1
    return float(2.0 ** e)


def quantize_weight_residual(R: np.ndarray, s_T: float):
    """Reading R6.  R is [K, N]; returns (codes [N][K] uint8 4-bit,
    scales [N][K/16] e4m3 bytes)."""
    Rt = np.asarray(R, dtype=np.float64).T
    N, K = Rt.shape
    blocks = Rt.reshape(N, K // 16, 16)
    amax = np.max(np.abs(blocks), axis=2)
    s_code = rne_e4m3(amax / (E2M1_MAX * s_T))
    s = e4m3_decode(s_code)
    scale = (s * s_T)[..., None]
    codes = np.zeros(blocks.shape, dtype=np.uint8)
    nz = np.broadcast_to(scale > 0, blocks.shape)
    codes[nz] = rne_e2m1(blocks[nz] / np.broadcast_to(scale, blocks.shape)[nz])
    return codes.reshape(N, K), s_code


def pack_weights(W: np.ndarray, x_absmax, rank: int, factor_rounding: str = "bf16",
                 lowrank=None):
    """Offline weight packing (readings R1-R6).

    W: [N, K] float32 (nn.Linear layout).  x_absmax: [K] calibration maxima,
    or None for no smoothing (inv_lambda = 1).  factor_rounding: "bf16" (the
    layer) or "none" (float64 factors, used to pin the full-rank identity).
    lowrank: optional precomputed (L1, L2) float64 factors of W_hat^T.
    """
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if x_absmax is None:
        inv = np.ones(K, dtype=np.float32)
    else:
        inv = smoothing_inv_lambda(x_absmax, W)
    inv64 = inv.astype(np.float64)
    W_hat_T = W.T.astype(np.float64) / inv64[:, None]
    if lowrank is None:
        L1, L2 = lowrank_factors(W_hat_T, rank)
    else:
        L1, L2 = lowrank
    L1s = inv64[:, None] * L1
    if factor_rounding == "bf16":
        L1s = round_to_bf16(L1s)
        L2 = round_to_bf16(L2)
    elif factor_rounding != "none":
        raise ValueError(factor_rounding)
    R = residual(W, inv, L1s, L2)
    s_T = tensor_scale(R)
    codes, s_code = quantize_weight_residual(R, s_T)
    return {
        "N": N, "K": K, "rank": rank,
        "inv_lambda": inv,
        "L1": L1, "L2_exact": L2 if factor_rounding == "none" else None,
        "L1s": L1s, "L2": L2,
        "R": R, "s_T": s_T,
        "w_codes": codes, "w_scales": s_code,
        "w_codes_packed": pack_nibbles(codes),
        "w_scales_swizzled": sf_swizzle(s_code) if K % 64 == 0 else None,
        "factor_rounding": factor_rounding,
    }


def device_factor_bits(packed):
    """bf16 bit patterns of L1s [K][r] and L2 [r][N] (bf16 mode only)."""
    return bf16_bits(packed["L1s"]), bf16_bits(packed["L2"])


# ---------------------------------------------------------------------------
# per forward: activation quantization + low-rank down projection, GEMM
# ---------------------------------------------------------------------------


def smooth_activations(X: np.ndarray, inv_lambda: np.ndarray) -> np.ndarray:
    """x_hat = fl32(x * inv_lambda_j): one binary32 multiply (reading R7)."""
    X = np.asarray(X, dtype=np.float32)
    return (X * np.asarray(inv_lambda, dtype=np.float32)[None, :]).astype(np.float32)


def quantize_activations(X: np.ndarray, inv_lambda: np.ndarray):
    """Reading R7.  X: [M, K] values exactly representable in bf16.
    Returns (x_hat float32, codes [M][K] uint8, scales [M][K/16] e4m3 bytes)."""
    xhat = smooth_activations(X, inv_lambda)
    M, K = xhat.shape
    blocks = xhat.astype(np.float64).reshape(M, K // 16, 16)
    amax = np.max(np.abs(blocks), axis=2) if M else np.zeros((0, K // 16))
    s_code = rne_e4m3(amax / E2M1_MAX)
    s = e4m3_decode(s_code)[..., None]
    codes = np.zeros(blocks.shape, dtype=np.uint8)
    nz = np.broadcast_to(s > 0, blocks.shape)
    codes[nz] = rne_e2m1(blocks[nz] / np.broadcast_to(s, blocks.shape)[nz])
    return xhat, codes.reshape(M, K), s_code


def lora_down(X: np.ndarray, L1s: np.ndarray, rounding: str = "bf16") -> np.ndarray:
    """Reading R8: lora_act = RNE_bf16(X . L1s) of the float64 product."""
    out = np.asarray(X, dtype=np.float64) @ np.asarray(L1s, dtype=np.float64)
    return round_to_bf16(out) if rounding == "bf16" else out


def gemm_reference(a_codes, a_scales, w_codes, w_scales, s_T, lora_act, L2, bias):
    """Y = s_T * dec(A) dec(W)^T + lora_act L2 + b, float64, unrounded (R9).
    a_codes [M][K], a_scales [M][K/16], w_codes [N][K], w_scales [N][K/16]
    (unpacked 4-bit codes, unswizzled scales)."""
    A = e2m1_decode(a_codes) * np.repeat(e4m3_decode(a_scales), 16, axis=1)
    Wd = e2m1_decode(w_codes) * np.repeat(e4m3_decode(w_scales), 16, axis=1)
    Y = float(s_T) * (A @ Wd.T)
    if lora_act is not None and np.asarray(lora_act).shape[1] > 0:
        Y = Y + np.asarray(lora_act, dtype=np.float64) @ np.asarray(L2, dtype=np.float64)
    if bias is not None:
        Y = Y + np.asarray(bias, dtype=np.float64)[None, :]
    return Y


def linear_forward(X: np.ndarray, packed: dict, bias):
    """The whole layer for bf16 X [M, K]; returns a dict of every
    intermediate the device produces plus Y (float64)."""
    xhat, a_codes, a_scales = quantize_activations(X, packed["inv_lambda"])
    rounding = "bf16" if packed["factor_rounding"] == "bf16" else "none"
    lora = lora_down(X, packed["L1s"], rounding)
    Y = gemm_reference(a_codes, a_scales, packed["w_codes"], packed["w_scales"],
                       packed["s_T"], lora, packed["L2"], bias)
    return {"x_hat": xhat, "a_codes": a_codes, "a_scales": a_scales,
            "a_codes_packed": pack_nibbles(a_codes) if X.shape[0] else
            np.zeros((0, X.shape[1] // 2), np.uint8),
            "a_scales_swizzled": sf_swizzle(a_scales) if X.shape[1] % 64 == 0 else None,
            "lora_act": lora, "Y": Y}


def naive_w4a4(X: np.ndarray, W: np.ndarray, bias):
    """Same NVFP4 rules with no smoothing and no low-rank branch (the baseline
    of the quality comparison)."""
    packed = pack_weights(W, None, 0)
    return linear_forward(X, packed, bias)["Y"]


def gelu_tanh(y: np.ndarray) -> np.ndarray:
    """GELU in its tanh form, float64 (libm tanh): the glue between the MLP
    pair's fc1 and fc2 ([dothoosh] names GELU/MLP kernels of the full engine)."""
    y = np.asarray(y, dtype=np.float64)
    c = np.sqrt(2.0 / np.pi)
    return 0.5 * y * (1.0 + np.tanh(c * (y + 0.044715 * y ** 3)))


def gelu_tanh_bf16(y: np.ndarray) -> np.ndarray:
    """GELU (tanh form) of the bf16 fc1 output, rounded to bf16: fc2's input."""
    return round_to_bf16(gelu_tanh(y))
