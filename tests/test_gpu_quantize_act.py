"""svdq_quantize_act on the GPU against the oracle: e4m3 scales and e2m1
codes bit-exact; lora_act within one bf16 ulp of the oracle's rounded exact
sum plus the fp32 accumulation allowance 2^-20 * sum_k |x_k L1s[k,i]| (the
tensor cores accumulate in fp32 in their own order; where the sum cancels,
that error is measured against the size of the terms, not of the result)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import formats, layout, svdq

import bit_w4a4_diffusion_quantize_b300 as lib
from gpu_util import dev_bf16, dev_bits16, dev_f32, host_bf16, scales_from_device

pytestmark = pytest.mark.gpu


def _run(X, inv, L1s_Kr, rank):
    """X float32 bf16 values [M,K], inv fp32 [K], L1s float values [K][r]."""
    M, K = X.shape
    Xd = dev_bf16(X) if M else torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    l1 = dev_bits16(formats.bf16_bits(L1s_Kr).T.copy())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales, lora = lib.svdq_quantize_act(Xd, dev_f32(inv), l1, rank, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return codes.cpu().numpy(), scales, host_bf16(lora) if M else np.zeros((0, rank))


def _check(X, inv, L1s, rank, lora_rows=None):
    M, K = X.shape
    codes, scales, lora = _run(X, inv, L1s, rank)
    _, c_ref, s_ref = svdq.quantize_activations(X, inv)
    assert np.array_equal(codes, layout.pack_nibbles(c_ref)), "codes differ"
    assert np.array_equal(scales_from_device(scales, M, K), s_ref), "scales differ"
    rows = np.arange(M) if lora_rows is None else lora_rows
    l_ref = svdq.lora_down(X[rows], L1s)
    diff = np.abs(lora[rows] - l_ref)
    ulp = 2 * np.maximum(np.ldexp(1.0, np.frexp(np.abs(l_ref))[1] - 9), 2.0 ** -133)
    mag = np.abs(X[rows].astype(np.float64)) @ np.abs(L1s)
    allow = ulp + 2.0 ** -20 * mag
    assert np.all(diff <= allow), f"lora error {np.max(diff / allow):.2f} x the allowance"
    return np.mean(diff > 0)


def _case_inputs(case, M=None):
    X = workloads.make_activations(case, M)
    W, _ = workloads.make_weights(case)
    inv = svdq.smoothing_inv_lambda(svdq.calib_absmax(X), W)
    rng = np.random.default_rng(case.seed + 100)
    L1s = formats.round_to_bf16(rng.standard_normal((case.K, case.rank)) * 0.05)
    return X, inv, L1s


@pytest.mark.parametrize("M,K,rank", [
    (128, 256, 16),   # the tiny workload
    (77, 256, 32),    # ragged rows (not a multiple of 16)
    (1, 128, 16),     # single row, smallest K
    (130, 384, 64),   # K not a multiple of 256, rank 64
    (300, 640, 32),   # several row tiles, ragged
    (5000, 512, 32),  # enough rows for the two-tile-per-warp variant
])
def test_quantize_act_parity(M, K, rank):
    case = workloads.custom_case(M, K, 128, rank, seed=M + K, planted_rank=4)
    X, inv, L1s = _case_inputs(case)
    _check(X, inv, L1s, rank)


def test_quantize_act_tiny_workload():
    case = workloads.CASES["tiny"]
    X, inv, L1s = _case_inputs(case)
    _check(X, inv, L1s, case.rank)


def test_quantize_act_attn_out_full_size():
    """The attention out-projection workload (4096 x 3072, rank 32): every code
    and scale; lora on 256 sampled rows."""
    case = workloads.CASES["attn_out"]
    X, inv, L1s = _case_inputs(case)
    rows = np.random.default_rng(0).choice(case.M, 256, replace=False)
    _check(X, inv, L1s, case.rank, lora_rows=rows)


def test_quantize_act_every_midpoint_of_every_scale():
    """For each finite positive e4m3 scale s and each e2m1 midpoint m, x_hat
    equal to m*s and to its two float32 neighbours (ties and near-ties of the
    quotient rounding), with the block's amax fixing the scale exactly."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    cols_inv = []
    for b in range(1, 0x7F):
        s = formats.E4M3_TABLE[b]
        targets = []
        for m in mids:
            t = np.float32(m * s)
            targets += [t, np.nextafter(t, np.float32(0)), np.nextafter(t, np.float32(np.inf))]
        for blk in range(2):
            block = [np.float32(6 * s)] + targets[15 * blk:15 * blk + 15]
            block += [np.float32(0.0)] * (16 - len(block))
            cols_inv += block
    K = ((len(cols_inv) + 127) // 128) * 128
    inv = np.zeros(K, dtype=np.float32)
    inv[:len(cols_inv)] = np.array(cols_inv, dtype=np.float32)
    # rows: x = +1, -1, +2, -0.5 (x_hat = x * inv exactly), and a row of -0.0
    X = np.array([[1.0], [-1.0], [2.0], [-0.5], [-0.0]], dtype=np.float32) * np.ones((1, K),
                                                                                    np.float32)
    L1s = np.zeros((K, 16))
    _check(X, inv, L1s, 16)


def test_quantize_act_special_values():
    """Zero blocks (scale 0), -0.0, tiny blocks with subnormal e4m3 scales,
    huge blocks whose scale saturates at 448, an infinite element, and
    arbitrary (non power of two) smoothing factors."""
    K = 256
    rng = np.random.default_rng(7)
    X = workloads.to_bf16_values(rng.standard_normal((40, K)).astype(np.float32))
    X[0, :] = 0.0
    X[1, :16] = -0.0
    X[2, :] = workloads.to_bf16_values(X[2] * np.float32(1e-3))     # subnormal scales
    X[3, :] = workloads.to_bf16_values(X[3] * np.float32(1e4))      # scale saturates at 448
    X[4, 16:32] = workloads.to_bf16_values(np.full(16, 3e38, np.float32))
    X[5, 5] = np.inf
    X[6, 40] = -np.inf
    X[7, :] = workloads.to_bf16_values(X[7] * np.float32(1e-20))    # underflowing block scale
    inv = (rng.uniform(0.3, 3.0, K)).astype(np.float32)
    L1s = formats.round_to_bf16(rng.standard_normal((K, 32)) * 0.05)
    with np.errstate(over="ignore", invalid="ignore"):
        finite_rows = np.where(np.all(np.isfinite(X * inv), axis=1))[0]
        _check(X, inv, L1s, 32, lora_rows=finite_rows)


def test_quantize_act_empty():
    codes, scales, lora = _run(np.zeros((0, 128), np.float32), np.ones(128, np.float32),
                               np.zeros((128, 16)), 16)
    assert codes.shape == (0, 64)


def test_quantize_act_repeatable():
    case = workloads.custom_case(200, 512, 128, 32, seed=3)
    X, inv, L1s = _case_inputs(case)
    a = _run(X, inv, L1s, 32)
    b = _run(X, inv, L1s, 32)
    assert np.array_equal(a[0], b[0])
    # padding rows of the scale tiles are never written: compare the real rows
    assert np.array_equal(scales_from_device(a[1], 200, 512), scales_from_device(b[1], 200, 512))
    assert np.array_equal(a[2], b[2])


@pytest.mark.parametrize("which", [0, 1], ids=["scales_all_fp32", "codes_every_scale"])
def test_exact_quotient_rounding_exhaustive(which):
    """The library's division-free rounding (shared by svdq_quantize_act and
    the fused GELU + quantization epilogue) against IEEE division followed by
    the same RNE conversion -- the exact rounding of the quotient -- over every
    finite fp32 amax (scale bytes), and over every e4m3 scale with every fp32
    value in the top 8 binades below its block amax, both signs (codes)."""
    count, first, checked = lib.test_quant_sweep(which)
    assert checked == (0x7F800000 if which == 0 else 126 * -(-(1 << 26) // 7)), checked
    assert count == 0, f"{count} blocks differ; smallest fp32 pattern {first:#010x}"
