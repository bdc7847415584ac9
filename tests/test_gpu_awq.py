"""awq_gemv_w4a16 on the GPU against the oracle (same packed weights), for
the adaLN modulation GEMV (K = 3072, N = 6 x 3072, M in 1..8) and ragged
shapes."""
import numpy as np
import pytest
import torch

import workloads
from oracle import awq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import assert_y_close, dev_bf16, dev_bits16, dev_u8, host_bf16

pytestmark = pytest.mark.gpu


def _run(X, p, b):
    Y = lib.awq_gemv_w4a16(dev_bf16(X), dev_u8(p["qweight"]),
                           dev_bits16(p["scales_bits"], torch.float16),
                           dev_bits16(p["zeros_bits"], torch.float16),
                           dev_bf16(b) if b is not None else None)
    torch.cuda.synchronize()
    return host_bf16(Y)


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_awq_modulation_full_size(M):
    X = workloads.make_awq_activations(M)
    W, b = workloads.make_awq_weights(0)
    p = awq.awq_pack(W)
    assert_y_close(_run(X, p, b), awq.awq_linear(X, p["qweight"], p["scales"], p["zeros"], b))


# K covers every kernel variant: up to 1, 2, 3, 4 groups per compute warp with
# 12 compute warps, and 16 compute warps above K = 3072
@pytest.mark.parametrize("M,N,K", [(3, 200, 128), (1, 24, 64), (7, 1000, 640), (5, 4096, 192),
                                   (8, 72, 1280), (6, 40, 960), (4, 136, 2048), (2, 1008, 4096),
                                   (1, 56, 3584)])
def test_awq_ragged(M, N, K):
    rng = np.random.default_rng(M * N + K)
    X = workloads.to_bf16_values(rng.standard_normal((M, K)).astype(np.float32))
    W = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    b = workloads.to_bf16_values(rng.standard_normal(N).astype(np.float32) * 0.01)
    p = awq.awq_pack(W)
    assert_y_close(_run(X, p, b), awq.awq_linear(X, p["qweight"], p["scales"], p["zeros"], b))
    assert_y_close(_run(X, p, None), awq.awq_linear(X, p["qweight"], p["scales"], p["zeros"], None))


def test_awq_product_packer_through_device():
    X = workloads.make_awq_activations(4)
    W, b = workloads.make_awq_weights(3)
    layer = lib.AWQLinear.from_float(W, workloads.bf16_bits_of(b))
    y = host_bf16(layer(dev_bf16(X)))
    p = awq.awq_pack(W)
    assert_y_close(y, awq.awq_linear(X, p["qweight"], p["scales"], p["zeros"], b))
