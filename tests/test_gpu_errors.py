"""Device-side error behaviour through the C ABI: the compute-capability
check (forced with the library's test hook svdq_test_set_hooks: a reported
capability of 9.0), pointer alignment checks on real device buffers, empty
inputs, and the bounded pipeline waits of the GEMM (forced with the same hook:
the loader issues nothing, the waits run out after 100 ms, the kernel reports
SVDQ_DEV_TIMEOUT through dev_status and returns; the context stays usable).
No test here faults or hangs the GPU."""
import ctypes
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import formats, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import (assert_y_close, dev_bf16, dev_bits16, dev_u8, host_bf16,
                      oracle_weight_operands)

pytestmark = pytest.mark.gpu


def _small_problem():
    case = workloads.custom_case(64, 256, 256, 16, seed=41)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = svdq.pack_weights(W, svdq.calib_absmax(X), 16)
    out = svdq.linear_forward(X, packed, b)
    return case, X, b, packed, out, oracle_weight_operands(packed, b)


def test_device_is_supported():
    assert lib.check_device() == 0


def test_fake_capability_is_refused():
    case, X, b, packed, out, w = _small_problem()
    lib.test_set_hooks(fake_compute_capability=90)
    try:
        assert lib.check_device() == -4
        with pytest.raises(lib.SvdqError) as e:
            lib.svdq_quantize_act(dev_bf16(X), w["inv_lambda"], w["L1s"], 16)
        assert e.value.status == -4
        Xa = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(lib.SvdqError) as e:
            lib.awq_gemv_w4a16(Xa, torch.zeros((64, 128), dtype=torch.uint8, device="cuda"),
                               torch.zeros((64, 4), dtype=torch.float16, device="cuda"),
                               torch.zeros((64, 4), dtype=torch.float16, device="cuda"), None)
        assert e.value.status == -4
    finally:
        lib.test_set_hooks()
    assert lib.check_device() == 0


def test_misaligned_device_buffers_are_refused():
    case, X, b, packed, out, w = _small_problem()
    Xd = dev_bf16(X)
    big = torch.zeros(Xd.numel() + 8, dtype=torch.bfloat16, device="cuda")
    shifted = big[1:1 + Xd.numel()].view(64, 256)   # 2-byte offset
    with pytest.raises(lib.SvdqError) as e:
        lib.svdq_quantize_act(shifted, w["inv_lambda"], w["L1s"], 16)
    assert e.value.status == -3


def test_dev_status_stays_clear_and_empty_input_is_a_no_op():
    case, X, b, packed, out, w = _small_problem()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(dev_bf16(X), w["inv_lambda"], w["L1s"], 16,
                                                dev_status=status)
    Y = lib.svdq_gemm_w4a4(codes, scales, w["w_codes"], w["w_scales"], w["s_T"], lora, w["L2"],
                           w["bias"], 64, 256, 256, 16, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_y_close(host_bf16(Y), out["Y"])
    Y0 = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    lib.svdq_gemm_w4a4(codes, scales, w["w_codes"], w["w_scales"], w["s_T"], lora, w["L2"],
                       None, 0, 256, 256, 16, Y=Y0)


def test_gemm_pipeline_wait_times_out_cleanly():
    case, X, b, packed, out, w = _small_problem()
    a_codes = dev_u8(out["a_codes_packed"])
    a_scales = dev_u8(out["a_scales_swizzled"])
    lora = dev_bits16(formats.bf16_bits(out["lora_act"]))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.test_set_hooks(gemm_stall=1)
    try:
        lib.svdq_gemm_w4a4(a_codes, a_scales, w["w_codes"], w["w_scales"], w["s_T"], lora,
                           w["L2"], w["bias"], 64, 256, 256, 16, dev_status=status)
        torch.cuda.synchronize()
    finally:
        lib.test_set_hooks()
    assert int(status.item()) == lib.DEV_TIMEOUT
    # the context is intact: the same call now completes and is correct
    status.zero_()
    Y = lib.svdq_gemm_w4a4(a_codes, a_scales, w["w_codes"], w["w_scales"], w["s_T"], lora,
                           w["L2"], w["bias"], 64, 256, 256, 16, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_y_close(host_bf16(Y), out["Y"])
