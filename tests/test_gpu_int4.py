"""The INT4 variant on the GPU against the oracle (oracle/int4.py):
svdq_quantize_act_int4's codes and bf16 scales bit-exact (random rows with
outlier channels, and hand-built groups: ties, clamping, zero, infinite and
subnormal groups, the amax values where the binary32 quotient's rounding
decides the scale); lora_act within the allowance of the NVFP4 activation
test; svdq_gemm_w4a4_int4 on the oracle's operands within the output
tolerance of tests/gpu_util.py, bit-exact on exactly representable operands;
the layer end to end from the product packer."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, int4, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import assert_y_close, dev_bf16, dev_bits16, dev_f32, dev_u8, host_bf16

pytestmark = pytest.mark.gpu


def _quant(X, inv, L1s_Kr, rank):
    M, K = X.shape
    Xd = dev_bf16(X) if M else torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    l1 = dev_bits16(formats.bf16_bits(L1s_Kr).T.copy())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act_int4(Xd, dev_f32(inv), l1, rank,
                                                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return (codes.cpu().numpy(), scales.view(torch.int16).cpu().numpy().view(np.uint16),
            host_bf16(lora) if M else np.zeros((0, rank)))


def _check_quant(X, inv, L1s, rank, lora_rows=None):
    M, K = X.shape
    codes, sbits, lora = _quant(X, inv, L1s, rank)
    _, c_ref, s_ref = int4.quantize_activations(X, inv)
    assert np.array_equal(codes, int4.pack_codes(c_ref)), "codes differ"
    ref_bits = (np.asarray(s_ref, np.float64).astype(np.float32).view(np.uint32) >> 16)
    assert np.array_equal(sbits, ref_bits.astype(np.uint16)), "scales differ"
    rows = np.arange(M) if lora_rows is None else lora_rows
    if len(rows):
        l_ref = svdq.lora_down(X[rows], L1s)
        diff = np.abs(lora[rows] - l_ref)
        ulp = 2 * np.maximum(np.ldexp(1.0, np.frexp(np.abs(l_ref))[1] - 9), 2.0 ** -133)
        allow = ulp + 2.0 ** -20 * (np.abs(X[rows].astype(np.float64)) @ np.abs(L1s))
        assert np.all(diff <= allow), f"lora error {np.max(diff / allow):.2f} x the allowance"


def _inputs(M, K, rank, seed):
    case = workloads.custom_case(M, K, 256, rank, seed=seed)
    X = workloads.make_activations(case)
    W, _ = workloads.make_weights(case)
    inv = svdq.smoothing_inv_lambda(svdq.calib_absmax(X), W)
    rng = np.random.default_rng(seed + 100)
    L1s = formats.round_to_bf16(rng.standard_normal((K, rank)) * 0.05)
    return X, inv, L1s


@pytest.mark.parametrize("M,K,rank", [
    (128, 256, 16), (77, 256, 32), (1, 128, 16), (130, 384, 64), (513, 1024, 32),
])
def test_quantize_act_int4_parity(M, K, rank):
    X, inv, L1s = _inputs(M, K, rank, seed=M + K)
    _check_quant(X, inv, L1s, rank)


def test_quantize_act_int4_attn_out_full_size():
    X, inv, L1s = _inputs(4096, 3072, 32, seed=31)
    _check_quant(X, inv, L1s, 32, lora_rows=np.arange(0, 4096, 16))


def test_quantize_act_int4_ties_zero_inf_tiny():
    """Hand-built rows (inv_lambda = 1, two groups each): power-of-two scales
    (amax 7 * 2^e) with values at every half-integer tie, a zero row, a row
    with an infinity, and tiny and subnormal groups (scaled by 2^64 inside
    the kernel)."""
    rng = np.random.default_rng(9)
    ties = np.concatenate([np.arange(-7, 7) + 0.5, np.arange(-7, 8),
                           np.linspace(-6.75, 6.75, 35)])
    rows = []
    for e in (-3, 0, 5):
        rows.append(np.concatenate([ties * 2.0 ** e, -ties[::-1] * 2.0 ** e]))
    rows.append(np.zeros(128))
    g = rng.uniform(-1, 1, 128)
    g[3] = np.inf
    rows.append(g)
    for e in (-140, -133, -130, -126, -120, -100, -70):
        rows.append(rng.uniform(-1, 1, 128) * 2.0 ** e)
    X = formats.round_to_bf16(np.array(rows)).astype(np.float32)
    X = np.concatenate([X, -X], axis=0)
    inv = np.ones(128, np.float32)
    L1s = formats.round_to_bf16(rng.standard_normal((128, 16)) * 0.05)
    finite = np.nonzero(np.all(np.isfinite(X), axis=1))[0]
    _check_quant(X, inv, L1s, 16, lora_rows=finite)


def test_quantize_act_int4_binary32_quotient_cases():
    """Group maxima placed through inv_lambda (x = 1 at column r, inv[r] =
    the wanted x_hat): amax / 7 one binary32 step either side of, or exactly
    on, a bf16 midpoint (the scale's rounding is decided by the binary32
    quotient), and subnormal amax where the binary32 quotient's own rounding
    lands on a bf16 midpoint that the exact quotient misses.  A second
    element of each row (column r + 32, x_hat = -amax / 3) checks a code."""
    targets = []
    for j in range(9):
        m = (1.0 + (2 * j + 1) / 256.0) * 2.0 ** (3 * j - 14)   # a bf16 midpoint
        a = np.float32(7.0 * m)                                  # exact (12 bits)
        targets += [a, np.nextafter(a, np.float32(np.inf)), np.nextafter(a, np.float32(0))]
    targets += [np.float32(np.ldexp(7.0 * 3 * 2 ** 15 + d, -149)) for d in (-2, -1, 1, 2)]
    M = len(targets)
    assert M <= 32
    X = np.zeros((M, 128), np.float32)
    inv = np.ones(128, np.float32)
    rng = np.random.default_rng(4)
    for r, a in enumerate(targets):
        X[r, r] = 1.0
        X[r, r + 32] = 1.0
    inv[:M] = np.array(targets, np.float32)
    # column r + 32 holds -amax_r / 3 for row r (no other row has a 1 there)
    inv[32:32 + M] = (-np.array(targets, np.float32) / np.float32(3)).astype(np.float32)
    X[:, 64:] = formats.round_to_bf16(rng.standard_normal((M, 64))).astype(np.float32)
    L1s = formats.round_to_bf16(rng.standard_normal((128, 16)) * 0.05)
    _check_quant(X, inv, L1s, 16)


def test_quantize_act_int4_empty():
    codes, sbits, lora = _quant(np.zeros((0, 128), np.float32), np.ones(128, np.float32),
                                np.zeros((128, 16)), 16)
    assert codes.shape == (0, 64) and sbits.shape == (0, 2)


# --------------------------------------------------------------------------- GEMM
def _gemm(out, packed, b, M, N, K, rank, bias=True):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = lib.svdq_gemm_w4a4_int4(
        dev_u8(int4.pack_codes(out["a_codes"])), dev_bits16(int4.scale_bits(out["a_scales"])),
        dev_u8(int4.pack_codes(packed["w_codes"])),
        dev_bits16(int4.scale_bits(packed["w_scales"])),
        dev_bits16(formats.bf16_bits(out["lora_act"])),
        dev_bits16(formats.bf16_bits(packed["L2"]).T.copy()),
        dev_bf16(b) if bias else None, M, N, K, rank, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status set"
    return host_bf16(Y)


def _gemm_case(M, K, N, rank, seed, bias=True, rows=None):
    case = workloads.custom_case(M, K, N, rank, seed=seed, planted_rank=min(8, rank))
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    packed = int4.pack_weights(W, svdq.calib_absmax(X), rank)
    out = int4.linear_forward(X, packed, b if bias else None)
    y = _gemm(out, packed, b, M, N, K, rank, bias)
    return y, out["Y"]


@pytest.mark.parametrize("M,K,N,rank", [
    (128, 256, 256, 16), (200, 512, 384, 32), (64, 256, 128, 64), (1, 128, 128, 16),
    (513, 1024, 768, 32),
])
def test_gemm_int4_parity(M, K, N, rank):
    y, ref = _gemm_case(M, K, N, rank, seed=M + N + K)
    assert_y_close(y, ref, "Y int4")


def test_gemm_int4_without_bias():
    y, ref = _gemm_case(100, 256, 256, 16, seed=11, bias=False)
    assert_y_close(y, ref, "Y int4")


def test_gemm_int4_attn_out_full_size():
    """Attention out-projection shape, M = 4096, K = N = 3072, rank 32: every
    output (the oracle's operands)."""
    y, ref = _gemm_case(4096, 3072, 3072, 32, seed=31)
    assert_y_close(y, ref, "Y int4 attn_out")


def test_gemm_int4_exact_operands():
    """Codes and power-of-two scales chosen directly, no low-rank term: every
    group sum is an integer and every scaled partial a dyadic number well
    inside fp32, so Y is exact before its one rounding: bit-exact."""
    rng = np.random.default_rng(12)
    M, K, N, r = 200, 512, 256, 16
    a = rng.integers(-7, 8, (M, K)).astype(np.int8)
    w = rng.integers(-7, 8, (N, K)).astype(np.int8)
    sa = np.ldexp(1.0, rng.integers(-4, 4, (M, K // 64)))
    sw = np.ldexp(1.0, rng.integers(-4, 4, (N, K // 64)))
    ref = int4.gemm_reference(a, sa, w, sw, None, None, None)
    out = {"a_codes": a, "a_scales": sa, "lora_act": np.zeros((M, r))}
    packed = {"w_codes": w, "w_scales": sw, "L2": np.zeros((r, N))}
    y = _gemm(out, packed, None, M, N, K, r, bias=False)
    assert np.array_equal(y, formats.round_to_bf16(ref))


def test_gemm_int4_empty():
    e = torch.empty(0, dtype=torch.uint8, device="cuda")
    b = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    Y = lib.svdq_gemm_w4a4_int4(e, b, e, b, b, b, None, 0, 128, 128, 16)
    assert Y.shape == (0, 128)


# --------------------------------------------------------------------------- the layer
def test_int4_layer_from_product_packer():
    """SVDQLinearInt4 packed by svdq_pack_weights_int4: the device layer
    against the oracle's forward on the same packed weights, and SVDQ below
    plain INT4 W4A4 in error against the fp64 product."""
    case = workloads.custom_case(512, 1024, 768, 32, seed=7, outlier_channels=8,
                                 outlier_scale=50.0, planted_rank=32)
    X = workloads.make_activations(case)
    W, b = workloads.make_weights(case)
    xm = svdq.calib_absmax(X)
    p = lib.svdq_pack_weights_int4(W, xm, 32)
    layer = lib.SVDQLinearInt4(p, workloads.bf16_bits_of(b))
    y = host_bf16(layer(dev_bf16(X)))
    torch.cuda.synchronize()
    packed = {"inv_lambda": p["inv_lambda"], "L1s": formats.bf16_from_bits(p["L1s"]).T,
              "L2": formats.bf16_from_bits(p["L2"]).T,
              "w_codes": int4.unpack_codes(p["w_codes"]),
              "w_scales": formats.bf16_from_bits(p["w_scales"])}
    ref = int4.linear_forward(X, packed, b)["Y"]
    assert_y_close(y, ref, "Y int4 layer")
    exact = X.astype(np.float64) @ W.T.astype(np.float64) + b
    e_dev = np.linalg.norm(y - exact) / np.linalg.norm(exact)
    e_naive = np.linalg.norm(int4.naive_w4a4(X, W, b) - exact) / np.linalg.norm(exact)
    assert e_dev < 0.5 * e_naive
