"""svdq_gemm_w4a4_gelu_quant: the first MLP linear with GELU and the second
linear's activation side (smoothing, NVFP4 quantization, low-rank down
projection) fused into its epilogue, against the oracle.

H is the bf16 GELU output; svdq_gemm_w4a4_gelu computes the same H (its
parity with the oracle is tested on its own), so the fused call must write it
bit for bit.  Its quantization is row-local and exact: a2_codes and a2_scales
must equal the oracle's quantize_activations of that H with the second
layer's inv_lambda, bit for bit.

lora_act2 = bf16(sum_n H[m][n] L1s2[n][i]) is accumulated in fp32 by the
tensor cores, 16 MMAs of depth 16 per 256-column tile, over each CTA pair's
run of tiles of one 256-row block; the (few) run sums of a row are then added
in a fixed order.  Each MMA adds its 16 exact products to the accumulator with
an error of at most a few fp32 roundings, and each addition of a run sum one
rounding, all relative to at most sum_n |H L1s2| = mag, so the device sum lies
within (N/16 * 2^-21 + 2^-23 * (number of runs)) * mag of the exact one; the
test allows (N/16 * 2^-21 + 2^-20) * mag.  After the final rounding,
lora_act2 is within one bf16 ulp of the oracle's rounded exact sum plus that
allowance."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, layout, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import (dev_bf16, dev_bits16, dev_f32, host_bf16, oracle_weight_operands,
                      scales_from_device)

pytestmark = pytest.mark.gpu


def _second_layer(rng, N, rank2, h_absmax_scale=1.0):
    """inv_lambda2 [N] and L1s2 [N][rank2] (bf16 values) of a second layer with
    K2 = N: smoothing factors spread over [2^-3, 2^3], factor entries ~N(0, 0.05)."""
    inv2 = np.exp2(rng.uniform(-3.0, 3.0, N)).astype(np.float32) * np.float32(h_absmax_scale)
    L1s2 = formats.round_to_bf16(rng.standard_normal((N, rank2)) * 0.05)
    return inv2, L1s2


def _first_layer(case):
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), case.rank)
    return X, oracle_weight_operands(packed, b)


def _run(X_dev, w, rank, inv2_d, l1s2_d, rank2, write_h=True):
    """(a2_codes, a2_scales, lora_act2, H_fused or None, H of svdq_gemm_w4a4_gelu)."""
    M, K = X_dev.shape
    N = w["N"]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(X_dev, w["inv_lambda"], w["L1s"], rank,
                                                dev_status=status)
    args = (codes, scales, w["w_codes"], w["w_scales"], w["s_T"], lora, w["L2"], w["bias"])
    H_ref = lib.svdq_gemm_w4a4_gelu(*args, M, N, K, rank, dev_status=status)
    H = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda") if write_h else None
    c2, s2, l2 = lib.svdq_gemm_w4a4_gelu_quant(*args, inv2_d, l1s2_d, rank2, M, N, K, rank, H=H,
                                               dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return c2, s2, l2, H, H_ref


def _check_lora2(lora2: np.ndarray, h: np.ndarray, L1s2: np.ndarray):
    N = h.shape[1]
    ref = svdq.lora_down(h, L1s2)
    diff = np.abs(lora2 - ref)
    ulp = 2 * np.maximum(np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 9), 2.0 ** -133)
    mag = np.abs(h) @ np.abs(np.asarray(L1s2, dtype=np.float64))
    allow = ulp + (N // 16 * 2.0 ** -21 + 2.0 ** -20) * mag
    assert np.all(diff <= allow), f"lora_act2 error {np.max(diff / allow):.2f} x the allowance"
    return float(np.mean(diff > 0))


def _check_quant(c2, s2, h, inv2, rows=None):
    M, N = h.shape
    rows = np.arange(M) if rows is None else rows
    _, c_ref, s_ref = svdq.quantize_activations(h[rows], inv2)
    codes = c2.cpu().numpy()
    assert np.array_equal(codes[rows], layout.pack_nibbles(c_ref)), "a2_codes differ"
    scales = scales_from_device(s2, M, N)
    assert np.array_equal(scales[rows], s_ref), "a2_scales differ"


@pytest.mark.parametrize("M,K,N,rank,rank2,seed", [
    (128, 256, 256, 16, 32, 1),     # one tile
    (333, 640, 512, 32, 64, 2),     # ragged M, two n tiles, rank2 64
    (200, 512, 768, 64, 32, 3),     # rank 64, three n tiles
    (1, 256, 256, 16, 64, 4),       # a single row
    (520, 384, 1024, 32, 32, 5),    # five m tiles, four n tiles, ragged
    (2048, 256, 4096, 16, 32, 6),   # more tiles than CTA pairs: segments of 1-2 tiles
    (40000, 256, 256, 16, 32, 7),   # one n tile: 2-3 single-tile segments per pair
    (2560, 256, 4096, 32, 64, 8),   # rank2 64 with multi-tile segments
])
def test_gelu_quant_parity(M, K, N, rank, rank2, seed):
    case = workloads.custom_case(M, K, N, rank, seed=seed)
    X, w = _first_layer(case)
    inv2, L1s2 = _second_layer(np.random.default_rng(seed + 1000), N, rank2)
    inv2_d, l1s2_d = dev_f32(inv2), dev_bits16(formats.bf16_bits(L1s2).T.copy())
    c2, s2, l2, H, H_ref = _run(dev_bf16(X), w, rank, inv2_d, l1s2_d, rank2)
    assert torch.equal(H.view(torch.int16), H_ref.view(torch.int16)), "H differs from the GELU GEMM"
    h = host_bf16(H_ref)
    _check_quant(c2, s2, h, inv2)
    _check_lora2(host_bf16(l2), h, L1s2)


def test_gelu_quant_without_h_and_repeatable():
    """H = NULL writes nothing else differently; two calls agree bit for bit."""
    M, K, N, rank, rank2 = 300, 512, 768, 32, 32
    case = workloads.custom_case(M, K, N, rank, seed=9)
    X, w = _first_layer(case)
    inv2, L1s2 = _second_layer(np.random.default_rng(9), N, rank2)
    inv2_d, l1s2_d = dev_f32(inv2), dev_bits16(formats.bf16_bits(L1s2).T.copy())
    Xd = dev_bf16(X)
    a = _run(Xd, w, rank, inv2_d, l1s2_d, rank2, write_h=True)
    b = _run(Xd, w, rank, inv2_d, l1s2_d, rank2, write_h=False)
    c = _run(Xd, w, rank, inv2_d, l1s2_d, rank2, write_h=False)
    assert torch.equal(a[0], b[0]) and torch.equal(b[0], c[0]), "a2_codes"
    # (the scale tiles' padding rows past M are not written)
    sa, sb, sc = (scales_from_device(x[1], M, N) for x in (a, b, c))
    assert np.array_equal(sa, sb) and np.array_equal(sb, sc), "a2_scales"
    la, lb, lc = (x[2].view(torch.int16) for x in (a, b, c))
    assert torch.equal(la, lb) and torch.equal(lb, lc), "lora_act2"
    _check_quant(b[0], b[1], host_bf16(a[4]), inv2)


def test_gelu_quant_scratch_check_and_empty():
    case = workloads.custom_case(128, 256, 256, 16, seed=11)
    X, w = _first_layer(case)
    inv2, L1s2 = _second_layer(np.random.default_rng(11), 256, 32)
    inv2_d, l1s2_d = dev_f32(inv2), dev_bits16(formats.bf16_bits(L1s2).T.copy())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(dev_bf16(X), w["inv_lambda"], w["L1s"], 16,
                                                dev_status=status)
    args = (codes, scales, w["w_codes"], w["w_scales"], w["s_T"], lora, w["L2"], w["bias"],
            inv2_d, l1s2_d, 32)
    short = torch.empty(lib.gelu_quant_scratch_bytes(128, 256, 32) - 16, dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(lib.SvdqError, match="SHAPE"):
        lib.svdq_gemm_w4a4_gelu_quant(*args, 128, 256, 256, 16, scratch=short)
    with pytest.raises(lib.SvdqError, match="RANK"):
        lib.svdq_gemm_w4a4_gelu_quant(*args[:-1], 16, 128, 256, 256, 16)
    e = torch.empty((0, 256), dtype=torch.uint8, device="cuda")
    c2, s2, l2 = lib.svdq_gemm_w4a4_gelu_quant(e, e, w["w_codes"], w["w_scales"], w["s_T"], e,
                                               w["L2"], w["bias"], inv2_d, l1s2_d, 32, 0, 256,
                                               256, 16)
    torch.cuda.synchronize()
    assert tuple(c2.shape) == (0, 128) and tuple(l2.shape) == (0, 32)


def test_gelu_quant_mlp_full_size():
    """fc1 of the MLP pair at full size (M = 4096, K = 3072, N = 12288, r = 32)
    with fc2's activation side fused (K2 = 12288, rank2 = 32), in the launch
    configuration the benchmark times: every row's codes and scales equal
    svdq_quantize_act's on the same H (itself bit-exact to the oracle), 256
    sampled rows are checked against the oracle directly, and lora_act2 on
    those rows against the oracle's exact sum."""
    c1 = workloads.CASES["fc1"]
    X1, w1 = _first_layer(c1)
    c2 = workloads.CASES["fc2"]
    W2, _ = workloads.make_fc2_weights(c2)
    M, N = c1.M, c1.N
    # fc2's smoothing from a calibration of H (as its packer would see it)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(dev_bf16(X1), w1["inv_lambda"], w1["L1s"],
                                                c1.rank, dev_status=status)
    args = (codes, scales, w1["w_codes"], w1["w_scales"], w1["s_T"], lora, w1["L2"], w1["bias"])
    H_ref = lib.svdq_gemm_w4a4_gelu(*args, M, N, c1.K, c1.rank, dev_status=status)
    h = host_bf16(H_ref)
    p2 = svdq.pack_weights(W2, svdq.calib_absmax(h), c2.rank)
    w2 = oracle_weight_operands(p2)
    a2c, a2s, l2 = lib.svdq_gemm_w4a4_gelu_quant(*args, w2["inv_lambda"], w2["L1s"], c2.rank, M,
                                                 N, c1.K, c1.rank, dev_status=status)
    uc, us, _ = lib.svdq_quantize_act(H_ref, w2["inv_lambda"], w2["L1s"], c2.rank,
                                      dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(a2c, uc), "a2_codes differ from svdq_quantize_act on H"
    assert torch.equal(a2s, us), "a2_scales differ from svdq_quantize_act on H"
    rows = np.sort(np.random.default_rng(61).choice(M, 256, replace=False))
    _check_quant(a2c, a2s, h, p2["inv_lambda"], rows)
    _check_lora2(host_bf16(l2)[rows], h[rows], p2["L1s"])


def test_mlp_layer_fused_against_oracle_and_unfused():
    """SVDQMLP (the user-level path: K1, the fused GELU + quantization GEMM,
    fc2's GEMM) on weights packed by svdq_pack_weights, fc2 calibrated on H:
    the fused and the unfused (H written, then fc2's own K1) outputs each
    against the oracle's fc2 forward of the device's H on those packed
    weights."""
    from test_gpu_linear import _oracle_view_of_product_packing
    from gpu_util import assert_y_close, lora_rounding_slack

    M, K, N1, N2, r = 300, 256, 512, 256, 32
    c1 = workloads.custom_case(M, K, N1, r, seed=41)
    X = workloads.make_activations(c1)
    W1, b1 = workloads.make_weights(c1)
    W2, b2 = workloads.make_weights(workloads.custom_case(M, N1, N2, r, seed=42))
    fc1 = lib.SVDQLinear.from_float(W1, lib.svdq_calib_absmax(workloads.bf16_bits_of(X)), r,
                                    bias_bf16_bits=workloads.bf16_bits_of(b1))
    Xd = dev_bf16(X)
    h = host_bf16(fc1(Xd, gelu=True))
    p2 = lib.svdq_pack_weights(W2, lib.svdq_calib_absmax(workloads.bf16_bits_of(h)), r)
    fc2 = lib.SVDQLinear(p2, workloads.bf16_bits_of(b2))
    mlp = lib.SVDQMLP(fc1, fc2)
    y_fused = host_bf16(mlp(Xd))
    y_unfused = host_bf16(mlp(Xd, fused=False))
    view = _oracle_view_of_product_packing(p2)
    ref = svdq.linear_forward(h, view, b2)["Y"]
    slack = lora_rounding_slack(h, view["L1s"], view["L2"])
    assert_y_close(y_fused, ref, "MLP fused (fc2 Y)", slack)
    assert_y_close(y_unfused, ref, "MLP unfused (fc2 Y)", slack)
