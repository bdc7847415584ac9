"""The whole SVDQ linear on the GPU (svdq_quantize_act -> svdq_gemm_w4a4)
against the oracle's forward on the same packed weights, for the diffusion
transformer workloads; and the product packer's weights through the device
path against the unquantized float64 product (quality: SVDQ beats plain
W4A4 on outlier-heavy inputs)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, layout, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import (assert_y_close, dev_bf16, host_bf16, lora_rounding_slack,
                      oracle_weight_operands)

pytestmark = pytest.mark.gpu


def _device_forward(X, w, rank):
    M, K = X.shape
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(dev_bf16(X), w["inv_lambda"], w["L1s"], rank,
                                                dev_status=status)
    Y = lib.svdq_gemm_w4a4(codes, scales, w["w_codes"], w["w_scales"], w["s_T"], lora, w["L2"],
                           w["bias"], M, w["N"], K, rank, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return Y, codes, scales, lora


def _slack(X, packed):
    return lora_rounding_slack(X, packed["L1s"], packed["L2"])


def _oracle_case(case, X=None, W=None, b=None):
    if X is None:
        X = workloads.make_activations(case)
    if W is None:
        W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), case.rank)
    return X, W, b, packed, svdq.linear_forward(X, packed, b)


@pytest.mark.parametrize("name", ["tiny", "attn_out", "qkv"])
def test_linear_parity(name):
    case = workloads.CASES[name]
    X, W, b, packed, out = _oracle_case(case)
    Y, codes, _, _ = _device_forward(X, oracle_weight_operands(packed, b), case.rank)
    assert np.array_equal(codes.cpu().numpy(), out["a_codes_packed"])
    assert_y_close(host_bf16(Y), out["Y"], name, _slack(X, packed))


def test_linear_ragged():
    case = workloads.custom_case(333, 640, 384, 32, seed=21)
    X, W, b, packed, out = _oracle_case(case)
    Y, _, _, _ = _device_forward(X, oracle_weight_operands(packed, b), 32)
    assert_y_close(host_bf16(Y), out["Y"], "ragged", _slack(X, packed))


def test_mlp_pair_fc1_gelu_fc2():
    """fc1 (4096 x 3072 -> 12288), GELU (tanh) on fc1's oracle output rounded
    to bf16, fc2 (12288 -> 3072); fc2's own smoothing comes from its input."""
    c1 = workloads.CASES["fc1"]
    X1, W1, b1, p1, o1 = _oracle_case(c1)
    Y1, _, _, _ = _device_forward(X1, oracle_weight_operands(p1, b1), c1.rank)
    assert_y_close(host_bf16(Y1), o1["Y"], "fc1", _slack(X1, p1))
    X2 = svdq.gelu_tanh_bf16(formats.round_to_bf16(o1["Y"])).astype(np.float32)
    c2 = workloads.CASES["fc2"]
    W2, b2 = workloads.make_fc2_weights(c2)
    _, _, _, p2, o2 = _oracle_case(c2, X2, W2, b2)
    Y2, _, _, _ = _device_forward(X2, oracle_weight_operands(p2, b2), c2.rank)
    assert_y_close(host_bf16(Y2), o2["Y"], "fc2", _slack(X2, p2))


def _oracle_view_of_product_packing(p):
    """The oracle's packed-weight dict for weights packed by svdq_pack_weights:
    its smoothing, bf16 factors (L2 = L2s^T s_T, exact), codes and scales."""
    N, K = p["N"], p["K"]
    return {"N": N, "K": K, "rank": p["rank"], "inv_lambda": p["inv_lambda"],
            "L1s": formats.bf16_from_bits(p["L1s"]).T,
            "L2": formats.bf16_from_bits(p["L2s"]).T * p["w_tensor_scale"],
            "s_T": p["w_tensor_scale"],
            "w_codes": layout.unpack_nibbles(p["w_codes"]).reshape(N, K),
            "w_scales": layout.sf_unswizzle(p["w_scales"], N, K // 16),
            "factor_rounding": "bf16"}


def test_product_packer_parity_attn_out():
    """The attention out-projection (M = 4096, K = N = 3072, rank 32) with the
    weights packed by svdq_pack_weights (not the oracle): the device forward
    against the oracle's forward on those same packed weights, every code
    and every output."""
    case = workloads.CASES["attn_out"]
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    p = lib.svdq_pack_weights(W, lib.svdq_calib_absmax(workloads.bf16_bits_of(X)), case.rank)
    view = _oracle_view_of_product_packing(p)
    out = svdq.linear_forward(X, view, b)
    layer = lib.SVDQLinear(p, workloads.bf16_bits_of(b))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(dev_bf16(X), layer.inv_lambda, layer.L1s,
                                                case.rank, dev_status=status)
    Y = lib.svdq_gemm_w4a4(codes, scales, layer.w_codes, layer.w_scales, layer.w_tensor_scale,
                           lora, layer.L2s, layer.bias, case.M, case.N, case.K, case.rank,
                           dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(codes.cpu().numpy(), layout.pack_nibbles(out["a_codes"]))
    assert_y_close(host_bf16(Y), out["Y"], "attn_out, product packer",
                   lora_rounding_slack(X, view["L1s"], view["L2"]))


def test_product_packer_quality_through_device():
    """Weights packed by svdq_pack_weights, run through the device path: the
    error against float64 X W^T + b is below plain W4A4's (oracle) and within
    10% of the oracle's own SVDQ error."""
    case = workloads.custom_case(1024, 1024, 1024, 32, seed=31, outlier_scale=50.0)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    exact = X.astype(np.float64) @ W.T.astype(np.float64) + b
    layer = lib.SVDQLinear.from_float(W, lib.svdq_calib_absmax(workloads.bf16_bits_of(X)), 32,
                                      workloads.bf16_bits_of(b))
    y = host_bf16(layer(dev_bf16(X)))
    nrm = np.linalg.norm(exact)
    e_dev = np.linalg.norm(y - exact) / nrm
    e_naive = np.linalg.norm(svdq.naive_w4a4(X, W, b) - exact) / nrm
    e_oracle = np.linalg.norm(_oracle_case(case, X, W, b)[4]["Y"] - exact) / nrm
    assert e_dev < 0.5 * e_naive, (e_dev, e_naive)
    assert e_dev < 1.1 * e_oracle + 2e-3, (e_dev, e_oracle)


def test_mlp_pair_batch4_sampled_rows():
    """The MLP pair at a batch of 4 images (M = 16384): fc1's codes on every
    row and its Y in full; fc2 (input GELU of fc1's oracle output, smoothing
    from all of it) checked on 512 sampled rows (quantization is row-local, so
    the oracle's rows are exact)."""
    c1 = workloads.CASES["fc1_b4"]
    X1, W1, b1, p1, o1 = _oracle_case(c1)
    Y1, codes1, _, _ = _device_forward(X1, oracle_weight_operands(p1, b1), c1.rank)
    assert np.array_equal(codes1.cpu().numpy(), o1["a_codes_packed"])
    assert_y_close(host_bf16(Y1), o1["Y"], "fc1 batch 4", _slack(X1, p1))
    del Y1, codes1
    X2 = svdq.gelu_tanh_bf16(formats.round_to_bf16(o1["Y"])).astype(np.float32)
    del o1
    c2 = workloads.CASES["fc2_b4"]
    W2, b2 = workloads.make_fc2_weights(c2)
    p2 = svdq.pack_weights(W2, svdq.calib_absmax(X2), c2.rank)
    Y2, codes2, _, _ = _device_forward(X2, oracle_weight_operands(p2, b2), c2.rank)
    rows = np.sort(np.random.default_rng(41).choice(c2.M, 512, replace=False))
    o2 = svdq.linear_forward(X2[rows], p2, b2)
    assert np.array_equal(codes2.cpu().numpy()[rows], o2["a_codes_packed"])
    assert_y_close(host_bf16(Y2)[rows], o2["Y"], "fc2 batch 4 (sampled rows)",
                   _slack(X2[rows], p2))
