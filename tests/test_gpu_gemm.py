"""svdq_gemm_w4a4 on the GPU against the oracle.  The GEMM gets the oracle's
own operands (activation codes/scales/lora from the oracle's quantizer,
weights from the oracle's packing), so this isolates the tcgen05 product,
the block-scale handling, the rank-r term and the epilogue."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import (assert_y_close, dev_bf16, dev_bits16, dev_u8, host_bf16,
                      oracle_weight_operands)

pytestmark = pytest.mark.gpu


def _gemm_case(case, M=None, rows=None):
    X = workloads.make_activations(case, M)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), case.rank)
    out = svdq.linear_forward(X, packed, b)
    w = oracle_weight_operands(packed, b)
    Mx = X.shape[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = lib.svdq_gemm_w4a4(dev_u8(out["a_codes_packed"]), dev_u8(out["a_scales_swizzled"]),
                           w["w_codes"], w["w_scales"], w["s_T"],
                           dev_bits16(formats.bf16_bits(out["lora_act"])), w["L2"], w["bias"],
                           Mx, case.N, case.K, case.rank, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return host_bf16(Y), out["Y"]


@pytest.mark.parametrize("M,K,N,rank", [
    (128, 256, 256, 16),    # the tiny workload's shape
    (200, 512, 384, 32),    # ragged M, N not a multiple of 256 (128-wide tiles)
    (130, 384, 512, 32),    # K not a multiple of 256 (half k tile at the end)
    (64, 256, 256, 64),     # rank 64
    (1, 128, 128, 16),      # one row, smallest K and N
    (513, 1024, 768, 32),   # several tiles in both directions
])
def test_gemm_parity(M, K, N, rank):
    case = workloads.custom_case(M, K, N, rank, seed=M + N + K, planted_rank=min(8, rank))
    y, ref = _gemm_case(case)
    assert_y_close(y, ref)


def test_gemm_tiny_workload():
    y, ref = _gemm_case(workloads.CASES["tiny"])
    assert_y_close(y, ref)


def test_gemm_attn_out_full_size():
    """Attention out-projection, M = 4096, K = N = 3072, rank 32: every output."""
    y, ref = _gemm_case(workloads.CASES["attn_out"])
    assert_y_close(y, ref)


def test_gemm_without_bias():
    case = workloads.custom_case(100, 256, 256, 16, seed=11)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), 16)
    out = svdq.linear_forward(X, packed, None)
    w = oracle_weight_operands(packed, None)
    Y = lib.svdq_gemm_w4a4(dev_u8(out["a_codes_packed"]), dev_u8(out["a_scales_swizzled"]),
                           w["w_codes"], w["w_scales"], w["s_T"],
                           dev_bits16(formats.bf16_bits(out["lora_act"])), w["L2"], None,
                           100, 256, 256, 16)
    torch.cuda.synchronize()
    assert_y_close(host_bf16(Y), out["Y"])


def test_gemm_exact_operands_reproduce_plain_product():
    """Representable operands (rank-0 residual path exercised through a zero
    rank-16 branch): the device must reproduce X W^T exactly up to the final
    bf16 rounding."""
    rng = np.random.default_rng(12)
    M, K, N = 128, 256, 256
    # codes of 0, +-1, +-2, +-4 and power-of-two scales: every product is a
    # signed power of two in [2^-2, 2^8], so any fp32 summation order is exact
    pow2_codes = np.array([0, 2, 4, 6, 8, 10, 12, 14], dtype=np.uint8)
    a_codes = rng.choice(pow2_codes, (M, K))
    w_codes = rng.choice(pow2_codes, (N, K))
    a_sc = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), (M, K // 16))
    w_sc = rng.choice(np.array([0x30, 0x38, 0x40], np.uint8), (N, K // 16))
    s_T = 2.0 ** -6
    lora = np.zeros((M, 16))
    L2 = np.zeros((16, N))
    ref = svdq.gemm_reference(a_codes, a_sc, w_codes, w_sc, s_T, lora, L2, None)
    from oracle import layout
    Y = lib.svdq_gemm_w4a4(dev_u8(layout.pack_nibbles(a_codes)), dev_u8(layout.sf_swizzle(a_sc)),
                           dev_u8(layout.pack_nibbles(w_codes)), dev_u8(layout.sf_swizzle(w_sc)),
                           s_T, dev_bf16(lora.astype(np.float32)),
                           dev_bf16(L2.T.copy().astype(np.float32)), None, M, N, K, 16)
    torch.cuda.synchronize()
    y = host_bf16(Y)
    # exact products of few-bit values: fp32 accumulation is exact here too
    assert np.array_equal(y, formats.round_to_bf16(ref))
