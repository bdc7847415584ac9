"""svdq_gemm_w4a4_qkv: the fused Q|K|V projection with the per-head RMS
normalization of Q and K and the rotary embedding in the GEMM's epilogue,
against the oracle (oracle/qkv.py).

As for the GELU epilogue, the plain GEMM on the same operands returns the
exact bf16 Y_b the fused epilogue starts from (fixed accumulation order); Y_b
is checked against the oracle's forward, and the V columns of the fused output
must equal it bit for bit.  A Q or K pair (o0, o1) must be the bf16 rounding of
the oracle's float64 result G from Y_b, the same bf16 weights and the same
fp32 cos/sin values (and eps as the fp32 value the kernel receives):

    |o - G| <= ulp_bf16/2 + 2^-16 (|n0| + |n1|)

with (n0, n1) the oracle's normalized pair before the rotation:
  - ulp/2 (of the larger of |o|, |G|): the final rounding;
  - 2^-16 (|n0| + |n1|): the fp32 evaluation.  The sum of 128 squares in two
    sequential halves has relative error <= 65 * 2^-24; the scaled mean plus
    eps one rounding; rsqrtf at most 2 ulp; so 1/rms is within 2^-18.5 and
    n = (y * rs) * w within 2^-18.3 of the exact value.  The rotation adds two
    roundings, and its error is bounded by the pair's norm, not by |o| (o can
    cancel).  The total is below 2^-17.9 (|n0| + |n1|).

Where G is farther from a bf16 rounding boundary than that error, o is exactly
RNE_bf16(G): the tests require that of all but 1% of the Q and K elements."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, qkv, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import (assert_y_close, dev_bf16, dev_f32, half_ulp_bf16, host_bf16,
                      lora_rounding_slack, oracle_weight_operands)

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))  # the value the kernel receives


def _run(X, w, rank, norm_q, norm_k, cos, sin):
    """(Y_b, QKV) from one activation quantization, the plain GEMM and the
    fused QKV GEMM on the same operands."""
    M, K = X.shape
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(dev_bf16(X), w["inv_lambda"], w["L1s"], rank,
                                                dev_status=status)
    args = (codes, scales, w["w_codes"], w["w_scales"], w["s_T"], lora, w["L2"], w["bias"])
    Y = lib.svdq_gemm_w4a4(*args, M, w["N"], K, rank, dev_status=status)
    out = lib.svdq_gemm_w4a4_qkv(*args, dev_bf16(norm_q), dev_bf16(norm_k), dev_f32(cos),
                                 dev_f32(sin), M, w["N"], K, rank, eps=EPS, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return host_bf16(Y), host_bf16(out)


def assert_qkv_of(out: np.ndarray, y_b: np.ndarray, norm_q, norm_k, cos, sin, what: str):
    M, N = y_b.shape
    hd = N // 3
    assert np.array_equal(out[:, 2 * hd:], y_b[:, 2 * hd:]), f"{what}: V columns differ from Y_b"
    G = qkv.qkv_norm_rope(y_b, norm_q, norm_k, cos, sin, eps=EPS)
    off = 0.0
    for lo, w in ((0, norm_q), (hd, norm_k)):
        o, g = out[:, lo:lo + hd], G[:, lo:lo + hd]
        n = qkv.rms_norm_heads(y_b[:, lo:lo + hd], w, eps=EPS)
        pair = np.abs(n[:, 0::2]) + np.abs(n[:, 1::2])
        pair = np.repeat(pair, 2, axis=1)
        bound = half_ulp_bf16(np.maximum(np.abs(o), np.abs(g))) + 2.0 ** -16 * pair
        excess = np.abs(o - g) - bound
        k = int(np.argmax(excess))
        assert excess.flat[k] <= 0, (
            f"{what}: column {lo + k % hd} row {k // hd}: {o.flat[k]!r} vs {g.flat[k]!r} "
            f"(bound {bound.flat[k]:.3e})")
        off += float(np.mean(o != formats.round_to_bf16(g))) / 2
    assert off < 0.01, f"{what}: {off:.3e} of the Q, K elements differ from RNE(oracle)"
    return off


def _norm_weights(seed):
    rng = np.random.default_rng(seed)
    return tuple(workloads.to_bf16_values(1.0 + 0.1 * rng.standard_normal(128).astype(np.float32))
                 for _ in range(2))


def test_qkv_epilogue_small_ragged():
    """M = 200 (ragged last tile), K = 512, N = 768 (two heads each of Q, K, V),
    rank 32; random angles in [-pi, pi]."""
    case = workloads.custom_case(200, 512, 768, 32, seed=61)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), case.rank)
    ref = svdq.linear_forward(X, packed, b)
    nq, nk = _norm_weights(62)
    theta = np.random.default_rng(63).uniform(-np.pi, np.pi, (case.M, 64))
    cos, sin = np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)
    y_b, out = _run(X, oracle_weight_operands(packed, b), case.rank, nq, nk, cos, sin)
    assert_y_close(y_b, ref["Y"], "Y_b", lora_rounding_slack(X, packed["L1s"], packed["L2"]))
    assert_qkv_of(out, y_b, nq, nk, cos, sin, "small")


def test_qkv_epilogue_full_size():
    """The QKV workload at full size (M = 4608: 512 text + 4096 image tokens,
    K = 3072, N = 9216 = 3 x 24 heads x 128, rank 32) with the rotary tables of
    the tokens' positions, in the launch configuration of the plain GEMM: Y_b
    against the oracle on 256 sampled rows, the fused output on every element."""
    case = workloads.CASES["qkv"]
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), case.rank)
    nq, nk = workloads.make_qk_norm_weights()
    cos, sin = workloads.make_rope_tables(workloads.rope_positions())
    y_b, out = _run(X, oracle_weight_operands(packed, b), case.rank, nq, nk, cos, sin)
    rows = np.sort(np.random.default_rng(64).choice(case.M, 256, replace=False))
    ref = svdq.linear_forward(X[rows], packed, b)
    assert_y_close(y_b[rows], ref["Y"], "Y_b (sampled rows)",
                   lora_rounding_slack(X[rows], packed["L1s"], packed["L2"]))
    assert_qkv_of(out, y_b, nq, nk, cos, sin, "qkv full size")


def test_qkv_epilogue_zero_heads_and_identity_rotation():
    """Degenerate inputs: X = 0 with no bias gives Y_b = 0, so every head has
    mean square 0 and the output must be exactly 0 (y * rsqrt(eps) = 0); with
    angle 0 and unit weights the Q and K heads are plainly RMS-normalized."""
    case = workloads.custom_case(128, 256, 768, 16, seed=65)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), case.rank)
    w = oracle_weight_operands(packed, None)
    ones = np.ones(128, dtype=np.float32)
    cos, sin = np.ones((case.M, 64), np.float32), np.zeros((case.M, 64), np.float32)
    y0, out0 = _run(np.zeros_like(X), w, case.rank, ones, ones, cos, sin)
    assert np.all(y0 == 0) and np.all(out0 == 0)
    y_b, out = _run(X, w, case.rank, ones, ones, cos, sin)
    assert_qkv_of(out, y_b, ones, ones, cos, sin, "identity rotation")
