"""libsvdq on the CPU: the library loads and exports every symbol the C
headers declare; host-detectable argument errors of the device calls; the
host packers against the oracle (bit-exact where the result is unique,
validity where it is not: the SVD factors are unique only up to rotation and
rounding, so the packed codes are checked to be exactly the quantization of
the residual of the packer's own factors)."""
import ctypes
import functools
import glob
import os
import re

import numpy as np
import pytest
import torch

import workloads
from oracle import awq, formats, int4, layout, svdq

import bit_w4a4_diffusion_quantize_b300 as lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HAS_GPU = torch.cuda.is_available()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert {"svdq_pack_weights", "svdq_quantize_act", "svdq_gemm_w4a4", "svdq_gemm_w4a4_gelu",
            "svdq_gemm_w4a4_qkv", "svdq_gemm_w4a4_gelu_quant", "awq_gemv_w4a16",
            "awq_pack_weights", "svdq_calib_absmax", "svdq_check_device",
            "svdq_status_string", "svdq_pack_weights_int4", "svdq_quantize_act_int4",
            "svdq_gemm_w4a4_int4"} <= names
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_quant_sweep_argument_errors():
    raw = lib.raw_lib()
    assert raw.svdq_test_quant_sweep(2, ALIGNED, None) == -7
    assert raw.svdq_test_quant_sweep(0, None, None) == -1
    assert raw.svdq_test_quant_sweep(0, MISALIGNED, None) == -3


def test_test_hooks_refuse_bad_values_and_reset():
    raw = lib.raw_lib()
    assert raw.svdq_test_set_hooks(-1, 0) == -7
    assert raw.svdq_test_set_hooks(0, 2) == -7
    assert raw.svdq_test_set_hooks(0, 0) == 0


def test_status_strings():
    for st in range(-8, 1):
        s = lib.raw_lib().svdq_status_string(st).decode()
        assert s.startswith(lib.status_name(st))


def test_check_device_status_is_defined():
    st = lib.check_device()
    if HAS_GPU:
        assert st in (0, -4)
    else:
        assert st == -5  # no device to query


# ------------------------------------------------------------- argument errors
P = ctypes.c_void_p
ALIGNED = P(0x10000)      # never dereferenced: every case below fails validation
MISALIGNED = P(0x10008)


def _qa(X=ALIGNED, inv=ALIGNED, l1=ALIGNED, M=64, K=256, r=32, codes=ALIGNED, sc=ALIGNED,
        lora=ALIGNED):
    return lib.raw_lib().svdq_quantize_act(X, inv, l1, M, K, r, codes, sc, lora, None, None)


def _gemm(M=64, N=256, K=256, r=32, sT=2.0 ** -10, Y=ALIGNED, a=ALIGNED, bias=None,
          fn="svdq_gemm_w4a4"):
    return getattr(lib.raw_lib(), fn)(a, ALIGNED, ALIGNED, ALIGNED, ctypes.c_float(sT),
                                      ALIGNED, ALIGNED, bias, Y, M, N, K, r, None, None)


def _qkv(M=64, N=768, K=256, r=32, eps=1e-6, nq=ALIGNED, cos=ALIGNED):
    return lib.raw_lib().svdq_gemm_w4a4_qkv(ALIGNED, ALIGNED, ALIGNED, ALIGNED,
                                            ctypes.c_float(2.0 ** -10), ALIGNED, ALIGNED, None,
                                            nq, ALIGNED, cos, ALIGNED, ctypes.c_float(eps),
                                            ALIGNED, M, N, K, r, None, None)


def _gq(M=64, N=256, K=256, r=32, r2=32, scratch_bytes=None, H=None, inv2=ALIGNED,
        scratch=ALIGNED, lora2=ALIGNED):
    if scratch_bytes is None:
        scratch_bytes = lib.gelu_quant_scratch_bytes(M, N, r2)
    return lib.raw_lib().svdq_gemm_w4a4_gelu_quant(
        ALIGNED, ALIGNED, ALIGNED, ALIGNED, ctypes.c_float(2.0 ** -10), ALIGNED, ALIGNED, None,
        inv2, ALIGNED, r2, ALIGNED, ALIGNED, lora2, H, scratch, scratch_bytes, M, N, K, r, None,
        None)


def _awq(M=1, N=64, K=256, g=64, X=ALIGNED):
    return lib.raw_lib().awq_gemv_w4a16(X, ALIGNED, ALIGNED, ALIGNED, None, ALIGNED, M, N, K, g,
                                        None, None)


def test_quantize_act_argument_errors():
    assert _qa(K=200) == -2 and _qa(K=0) == -2 and _qa(M=-1) == -2
    assert _qa(r=8) == -6 and _qa(r=48) == -6
    assert _qa(X=P(0)) == -1 and _qa(lora=P(0)) == -1
    assert _qa(X=MISALIGNED) == -3 and _qa(sc=MISALIGNED) == -3
    assert _qa(M=0, X=P(0)) == 0  # empty input: nothing to do


@pytest.mark.parametrize("fn", ["svdq_gemm_w4a4", "svdq_gemm_w4a4_gelu"])
def test_gemm_argument_errors(fn):
    g = functools.partial(_gemm, fn=fn)
    assert g(N=200) == -2 and g(K=200) == -2 and g(M=-3) == -2
    assert g(r=24) == -6
    assert g(sT=3.0) == -7 and g(sT=float("inf")) == -7 and g(sT=0.0) == -7
    assert g(sT=2.0 ** -101) == -7 and g(sT=2.0 ** 101) == -7
    assert g(Y=P(0)) == -1
    assert g(a=MISALIGNED) == -3 and g(bias=MISALIGNED) == -3
    assert g(M=0, Y=P(0)) == 0


def test_qkv_argument_errors():
    assert _qkv(N=512) == -2 and _qkv(N=1152) == -2      # not whole pairs of 128-wide heads
    assert _qkv(r=8) == -6
    assert _qkv(eps=-1e-6) == -7 and _qkv(eps=float("nan")) == -7 and _qkv(eps=float("inf")) == -7
    assert _qkv(eps=0.0) == -7   # an all-zero head would give 0 * rsqrt(0) = NaN
    assert _qkv(nq=P(0)) == -1 and _qkv(cos=P(0)) == -1
    assert _qkv(cos=MISALIGNED) == -3 and _qkv(nq=MISALIGNED) == -3
    assert _qkv(M=0, nq=P(0)) == 0


def test_gelu_quant_argument_errors():
    assert _gq(N=128) == -2 and _gq(N=384) == -2   # whole 256-column tiles only
    assert _gq(K=200) == -2 and _gq(M=-1) == -2
    assert _gq(r=8) == -6 and _gq(r2=16) == -6 and _gq(r2=48) == -6
    assert _gq(inv2=P(0)) == -1 and _gq(scratch=P(0)) == -1 and _gq(lora2=P(0)) == -1
    assert _gq(scratch_bytes=lib.gelu_quant_scratch_bytes(64, 256, 32) - 1) == -2
    assert _gq(M=300, N=512, r2=64,
               scratch_bytes=lib.gelu_quant_scratch_bytes(300, 512, 64) - 16) == -2
    assert lib.gelu_quant_scratch_bytes(4096, 12288, 32) == (128 + 16) * 256 * 32 * 4
    assert _gq(inv2=MISALIGNED) == -3 and _gq(H=MISALIGNED) == -3
    assert _gq(M=0, inv2=P(0), scratch_bytes=0) == 0


def test_gelu_quant_static_argument_errors():
    raw = lib.raw_lib()

    def call(M=64, N=256, r2=32):
        return raw.svdq_gemm_w4a4_gelu_quant_static(
            ALIGNED, ALIGNED, ALIGNED, ALIGNED, ctypes.c_float(2.0 ** -10), ALIGNED, ALIGNED,
            None, ALIGNED, ALIGNED, r2, ALIGNED, ALIGNED, ALIGNED, None, M, N, 256, 32, None,
            None)
    assert call(N=384) == -2 and call(M=-1) == -2 and call(r2=16) == -6
    assert call(M=98304) != -2 and call(M=98305) == -2            # rank2 32: row limit
    assert call(M=32768, r2=64) != -2 and call(M=32769, r2=64) == -2
    assert call(M=0) == 0


def _qa4(X=ALIGNED, M=64, K=256, r=32, sc=ALIGNED, lora=ALIGNED):
    return lib.raw_lib().svdq_quantize_act_int4(X, ALIGNED, ALIGNED, M, K, r, ALIGNED, sc, lora,
                                                None, None)


def _g4(M=64, N=256, K=256, r=32, Y=ALIGNED, a=ALIGNED, sw=ALIGNED, bias=None):
    return lib.raw_lib().svdq_gemm_w4a4_int4(a, ALIGNED, ALIGNED, sw, ALIGNED, ALIGNED, bias, Y,
                                             M, N, K, r, None, None)


def test_int4_argument_errors():
    assert _qa4(K=192) == -2 and _qa4(M=-1) == -2 and _qa4(r=8) == -6
    assert _qa4(X=P(0)) == -1 and _qa4(sc=MISALIGNED) == -3 and _qa4(M=0, X=P(0)) == 0
    assert _g4(N=192) == -2 and _g4(K=64) == -2 and _g4(M=-1) == -2 and _g4(r=48) == -6
    assert _g4(Y=P(0)) == -1 and _g4(sw=P(0)) == -1
    assert _g4(a=MISALIGNED) == -3 and _g4(bias=MISALIGNED) == -3
    assert _g4(M=0, Y=P(0)) == 0


def test_awq_argument_errors():
    assert _awq(M=0) == -2 and _awq(M=9) == -2 and _awq(g=128) == -2
    assert _awq(N=0) == -2 and _awq(N=12) == -2 and _awq(K=4224) == -2
    assert _awq(K=96) == -2  # K % 64 != 0
    assert _awq(X=P(0)) == -1 and _awq(X=MISALIGNED) == -3


@pytest.mark.skipif(HAS_GPU, reason="valid arguments would launch on a real device")
def test_device_calls_without_device_report_cuda_error():
    assert _qa() == -5 and _gemm() == -5 and _awq() == -5
    assert _qa4() == -5 and _g4() == -5
    assert _gemm(fn="svdq_gemm_w4a4_gelu") == -5 and _qkv() == -5 and _gq() == -5
    assert _gq(H=ALIGNED) == -5


# ------------------------------------------------------------- host packers
def test_calib_absmax_matches_oracle():
    case = workloads.CASES["tiny"]
    X = workloads.make_activations(case)
    got = lib.svdq_calib_absmax(workloads.bf16_bits_of(X))
    assert np.array_equal(got, svdq.calib_absmax(X))
    assert np.array_equal(lib.svdq_calib_absmax(np.zeros((0, 128), np.uint16)), np.zeros(128))


def _packer_case(case):
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    xm = svdq.calib_absmax(X)
    return X, W, xm, lib.svdq_pack_weights(W, xm, case.rank)


@pytest.mark.parametrize("case", [
    workloads.CASES["tiny"],                                 # direct Jacobi SVD path
    workloads.custom_case(256, 512, 384, 32, seed=3),        # randomized subspace path
    workloads.custom_case(64, 384, 640, 16, seed=4),         # N > K
], ids=lambda c: f"{c.name}-{c.N}x{c.K}-r{c.rank}")
def test_packer_matches_oracle(case):
    X, W, xm, p = _packer_case(case)
    # unique parts: smoothing factors
    assert np.array_equal(p["inv_lambda"], svdq.smoothing_inv_lambda(xm, W))
    # factors are bf16; the residual of the packer's own factors, quantized by
    # the oracle, must equal the packer's codes, scales and tensor scale
    L1s = formats.bf16_from_bits(p["L1s"]).T
    L2 = formats.bf16_from_bits(p["L2s"]).T * p["w_tensor_scale"]
    R = svdq.residual(W, p["inv_lambda"], L1s, L2)
    sT = svdq.tensor_scale(R)
    codes, sc = svdq.quantize_weight_residual(R, sT)
    assert p["w_tensor_scale"] == sT
    assert np.array_equal(p["w_codes"], layout.pack_nibbles(codes))
    assert np.array_equal(p["w_scales"], layout.sf_swizzle(sc))
    # the low-rank branch is near-optimal: residual within 1% of the residual
    # left by LAPACK's exact top-r factors (both with bf16 factors)
    ref = svdq.pack_weights(W, xm, case.rank)
    assert np.linalg.norm(R) <= 1.01 * np.linalg.norm(ref["R"])


def test_packer_full_rank_leaves_rounding_residual():
    case = workloads.custom_case(32, 128, 128, 128, seed=6, outlier_channels=2,
                                 planted_rank=8)
    X, W, xm, p = _packer_case(case)
    L1s = formats.bf16_from_bits(p["L1s"]).T
    L2 = formats.bf16_from_bits(p["L2s"]).T * p["w_tensor_scale"]
    W_hat = W.T.astype(np.float64) / p["inv_lambda"].astype(np.float64)[:, None]
    R = svdq.residual(W, p["inv_lambda"], L1s, L2)
    # only the bf16 rounding of the factors is left
    assert np.linalg.norm(R) <= 2.0 ** -7 * np.linalg.norm(W_hat)


@pytest.mark.parametrize("case", [
    workloads.CASES["tiny"],                                 # direct Jacobi SVD path
    workloads.custom_case(256, 512, 384, 32, seed=3),        # randomized subspace path
], ids=lambda c: f"{c.name}-{c.N}x{c.K}-r{c.rank}")
def test_int4_packer_matches_oracle(case):
    """svdq_pack_weights_int4: the same smoothing as the oracle; codes and
    scales equal to the oracle's INT4 quantization of the residual of the
    packer's own factors; the factors those of the NVFP4 packer (same
    steps); the residual near the LAPACK-optimal one."""
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    xm = svdq.calib_absmax(X)
    p = lib.svdq_pack_weights_int4(W, xm, case.rank)
    assert np.array_equal(p["inv_lambda"], svdq.smoothing_inv_lambda(xm, W))
    L1s = formats.bf16_from_bits(p["L1s"]).T
    L2 = formats.bf16_from_bits(p["L2"]).T
    R = svdq.residual(W, p["inv_lambda"], L1s, L2)
    codes, scales = int4.quantize_weight_residual(R)
    assert np.array_equal(p["w_codes"], int4.pack_codes(codes))
    assert np.array_equal(p["w_scales"], formats.bf16_bits(scales))
    q = lib.svdq_pack_weights(W, xm, case.rank)
    assert np.array_equal(p["L1s"], q["L1s"])
    ref = int4.pack_weights(W, xm, case.rank)
    assert np.linalg.norm(R) <= 1.01 * np.linalg.norm(ref["R"])


def test_int4_packer_argument_errors():
    W = np.zeros((128, 128), np.float32)
    xm = np.ones(128, np.float32)
    for args, st in (((np.zeros((100, 128), np.float32), xm, 16), -2), ((W, xm, 0), -6),
                     ((np.full((128, 128), np.nan, np.float32), xm, 16), -7)):
        with pytest.raises(lib.SvdqError) as e:
            lib.svdq_pack_weights_int4(*args)
        assert e.value.status == st


def test_packer_argument_errors():
    W = np.zeros((128, 128), np.float32)
    xm = np.ones(128, np.float32)
    with pytest.raises(lib.SvdqError) as e:
        lib.svdq_pack_weights(np.zeros((100, 128), np.float32), xm, 16)
    assert e.value.status == -2
    with pytest.raises(lib.SvdqError) as e:
        lib.svdq_pack_weights(W, xm, 0)
    assert e.value.status == -6
    with pytest.raises(lib.SvdqError) as e:
        lib.svdq_pack_weights(W, xm, 129)
    assert e.value.status == -6
    Wn = W.copy()
    Wn[3, 5] = np.nan
    with pytest.raises(lib.SvdqError) as e:
        lib.svdq_pack_weights(Wn, xm, 16)
    assert e.value.status == -7


def test_packer_zero_weight():
    p = lib.svdq_pack_weights(np.zeros((128, 128), np.float32), np.ones(128, np.float32), 16)
    assert p["w_tensor_scale"] == 1.0
    assert not p["w_codes"].any() and not p["w_scales"].any()


@pytest.mark.parametrize("N,K", [(64, 128), (37, 192), (1, 64)])
def test_awq_packer_matches_oracle(N, K):
    rng = np.random.default_rng(N + K)
    W = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    W[0, :64] = 0.5           # a constant group
    if N > 1:
        W[1, 64:128 if K >= 128 else 64] = 0.0
    q, s, z = lib.awq_pack_weights(W)
    o = awq.awq_pack(W)
    assert np.array_equal(q, o["qweight"])
    assert np.array_equal(s, o["scales_bits"])
    assert np.array_equal(z, o["zeros_bits"])


def test_awq_packer_errors():
    with pytest.raises(lib.SvdqError):
        lib.awq_pack_weights(np.zeros((4, 100), np.float32))
    with pytest.raises(lib.SvdqError):
        lib.awq_pack_weights(np.full((4, 64), np.inf, np.float32))


# ------------------------------------------------------------- binding buffer checks
def test_binding_refuses_short_or_mistyped_buffers():
    """The binding's size guard (a short buffer would be overrun on the device):
    element width and element count, checked on host tensors without a call."""
    from bit_w4a4_diffusion_quantize_b300 import _lib as b
    b._need(torch.zeros(8, dtype=torch.int16), "x", 8, 2)
    b._need(torch.zeros(8, dtype=torch.bfloat16), "x", 8, 2)
    b._need(None, "bias", 8, 2)                                   # nullable
    b._need(torch.zeros(0, dtype=torch.uint8), "lora", 0, 2)      # nothing touched: no check
    with pytest.raises(ValueError, match="8 elements needed"):
        b._need(torch.zeros(7, dtype=torch.int16), "x", 8, 2)
    with pytest.raises(ValueError, match="16-bit elements expected"):
        b._need(torch.zeros(8, dtype=torch.float32), "x", 8, 2)
    with pytest.raises(ValueError, match="8-bit elements expected"):
        b._need(torch.zeros(8, dtype=torch.int16), "codes", 8, 1)
