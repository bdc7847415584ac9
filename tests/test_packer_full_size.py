"""svdq_pack_weights at the diffusion transformer's full weight sizes (slow,
CPU; run with -m slow): the attention out-projection (3072 x 3072) and the
MLP's first linear (12288 x 3072), rank 32; svdq_pack_weights_int4 at the
attention out-projection.

* Codes, block scales and tensor scale are bit-exact against the oracle's
  quantization of the residual the packer's own bf16 factors leave.
* The packer's truncated SVD (randomized subspace iteration and a Jacobi SVD
  of the projection) is near-optimal: its residual is within 1e-3 (relative)
  of the residual left by LAPACK's exact top-r factors, the Eckart-Young
  optimum (both with the factors rounded to bf16)."""
import numpy as np
import pytest

import workloads
from oracle import formats, layout, svdq

import bit_w4a4_diffusion_quantize_b300 as lib

pytestmark = pytest.mark.slow


@pytest.mark.parametrize("name", ["attn_out", "fc1"])
def test_packer_full_size(name):
    case = workloads.CASES[name]
    X = workloads.make_activations(case)
    W, _ = workloads.make_weights(case)
    xm = svdq.calib_absmax(X)
    p = lib.svdq_pack_weights(W, xm, case.rank)
    assert np.array_equal(p["inv_lambda"], svdq.smoothing_inv_lambda(xm, W))
    L1s = formats.bf16_from_bits(p["L1s"]).T
    L2 = formats.bf16_from_bits(p["L2s"]).T * p["w_tensor_scale"]
    R = svdq.residual(W, p["inv_lambda"], L1s, L2)
    sT = svdq.tensor_scale(R)
    codes, sc = svdq.quantize_weight_residual(R, sT)
    assert p["w_tensor_scale"] == sT
    assert np.array_equal(p["w_codes"], layout.pack_nibbles(codes))
    assert np.array_equal(p["w_scales"], layout.sf_swizzle(sc))
    ref = svdq.pack_weights(W, xm, case.rank)
    assert np.linalg.norm(R) <= (1.0 + 1e-3) * np.linalg.norm(ref["R"])


def test_int4_packer_attn_out_full_size():
    """svdq_pack_weights_int4 at the attention out-projection (3072 x 3072,
    rank 32): codes and bf16 group scales bit-exact against the INT4 oracle's
    quantization of the residual the packer's own factors leave, the factors
    those of the NVFP4 packer (the same steps), and the residual within 1e-3
    of the LAPACK-optimal one."""
    from oracle import int4
    case = workloads.CASES["attn_out"]
    X = workloads.make_activations(case)
    W, _ = workloads.make_weights(case)
    xm = svdq.calib_absmax(X)
    p = lib.svdq_pack_weights_int4(W, xm, case.rank)
    assert np.array_equal(p["inv_lambda"], svdq.smoothing_inv_lambda(xm, W))
    L1s = formats.bf16_from_bits(p["L1s"]).T
    L2 = formats.bf16_from_bits(p["L2"]).T
    R = svdq.residual(W, p["inv_lambda"], L1s, L2)
    codes, scales = int4.quantize_weight_residual(R)
    assert np.array_equal(p["w_codes"], int4.pack_codes(codes))
    assert np.array_equal(p["w_scales"], formats.bf16_bits(scales))
    ref = int4.pack_weights(W, xm, case.rank)
    assert np.linalg.norm(R) <= (1.0 + 1e-3) * np.linalg.norm(ref["R"])
