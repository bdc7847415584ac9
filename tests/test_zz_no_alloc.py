"""svdq_gemm_w4a4_gelu_quant_static (the fused fc1 GELU + quantization call
with the library's static device scratch instead of caller scratch) against
svdq_gemm_w4a4_gelu_quant on the same operands: two calls in a row, each
matching the caller-scratch call (codes and scales bit for bit, lora_act2
within the tolerance of the fused call's own parity test; the two run the same
kernels, so in practice bit for bit), and no change in the device's free
memory across the static calls.

This file is collected last: the static scratch is state shared by every call
on the device, and the test must pass both alone and after the others."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import (dev_bf16, dev_bits16, dev_f32, host_bf16, oracle_weight_operands,
                      scales_from_device)

pytestmark = pytest.mark.gpu


def _lora_allow(h: np.ndarray, L1s2: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """The fused call's lora_act2 allowance (tests/test_gpu_gelu_quant.py)."""
    ulp = 2 * np.maximum(np.ldexp(1.0, np.frexp(np.abs(ref))[1] - 9), 2.0 ** -133)
    mag = np.abs(h) @ np.abs(np.asarray(L1s2, dtype=np.float64))
    return ulp + (h.shape[1] // 16 * 2.0 ** -21 + 2.0 ** -20) * mag


@pytest.mark.parametrize("M,K,N,rank,rank2,seed", [
    (2048, 256, 4096, 16, 32, 31),   # multi-tile segments
    (333, 512, 768, 32, 64, 32),     # ragged M, rank2 64
])
def test_static_scratch_matches_caller_scratch(M, K, N, rank, rank2, seed):
    case = workloads.custom_case(M, K, N, rank, seed=seed)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    w = oracle_weight_operands(svdq.pack_weights(W, svdq.calib_absmax(X), rank), b)
    rng = np.random.default_rng(seed)
    inv2 = np.exp2(rng.uniform(-3.0, 3.0, N)).astype(np.float32)
    L1s2 = formats.round_to_bf16(rng.standard_normal((N, rank2)) * 0.05)
    inv2_d, l1s2_d = dev_f32(inv2), dev_bits16(formats.bf16_bits(L1s2).T.copy())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(dev_bf16(X), w["inv_lambda"], w["L1s"], rank,
                                                dev_status=status)
    args = (codes, scales, w["w_codes"], w["w_scales"], w["s_T"], lora, w["L2"], w["bias"],
            inv2_d, l1s2_d, rank2, M, N, K, rank)
    H = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ref = lib.svdq_gemm_w4a4_gelu_quant(*args, H=H, dev_status=status)
    # every output buffer of the static calls exists before the first of them
    outs = [(torch.empty_like(ref[0]), torch.empty_like(ref[1]), torch.empty_like(ref[2]))
            for _ in range(2)]
    torch.cuda.synchronize()
    h = host_bf16(H)
    lref = svdq.lora_down(h, L1s2)
    allow = _lora_allow(h, L1s2, lref)
    ref_s = lib.scale_bytes(M, N)
    free_before = None
    for i, (c2, s2, l2) in enumerate(outs):
        lib.svdq_gemm_w4a4_gelu_quant_static(*args, c2, s2, l2, dev_status=status)
        torch.cuda.synchronize()
        free = torch.cuda.mem_get_info()[0]
        if free_before is None:
            free_before = free  # after the first call's set-up
        else:
            assert free == free_before, "device memory changed across static calls"
        assert int(status.item()) == 0
        assert torch.equal(c2, ref[0]), f"call {i}: a2_codes"
        # (scale tiles: rows past M are written by neither call)
        assert np.array_equal(scales_from_device(s2, M, N),
                              scales_from_device(ref[1], M, N)), f"call {i}: a2_scales"
        assert ref_s == s2.numel()
        l_dev = host_bf16(l2)
        assert np.all(np.abs(l_dev - lref) <= allow), f"call {i}: lora_act2 beyond its allowance"
        assert np.all(np.abs(l_dev - host_bf16(ref[2])) <= allow), f"call {i}: lora_act2"


def test_static_scratch_refuses_rows_beyond_its_size():
    """M above the static scratch's row limit is refused before any launch."""
    e = torch.empty(16, dtype=torch.uint8, device="cuda")
    b16 = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    f32 = torch.empty(16, dtype=torch.float32, device="cuda")
    raw = lib.raw_lib()
    P = lambda t: t.data_ptr()  # noqa: E731
    for rank2, m_max in ((32, 98304), (64, 32768)):
        st = raw.svdq_gemm_w4a4_gelu_quant_static(
            P(e), P(e), P(e), P(e), 2.0 ** -8, P(b16), P(b16), None, P(f32), P(b16), rank2,
            P(e), P(e), P(b16), None, m_max + 1, 256, 256, 16, None, None)
        assert st == -2, (rank2, st)
