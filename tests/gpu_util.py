"""Helpers of the GPU parity tests: moving oracle/workload arrays to the
device in the layouts of include/svdq.h, and the output tolerance.

Output tolerance (float outputs): the device rounds Y once to bf16 and
accumulates in fp32 on tensor cores; the oracle returns Y unrounded in fp64.
Relative Frobenius error <= 2e-3, and elementwise
|Y_dev - Y_ref| <= 1e-2 * rms(Y_ref) + ulp_bf16(Y_ref)/2 (the half-ulp term
covers the final bf16 rounding of large outputs) + the lora rounding slack.

Lora rounding slack: lora_act is stored in bf16 by both sides, rounded from
the exact sum by the oracle and from an fp32 tensor-core sum by the device.
Where the exact sum lies within the fp32 accumulation allowance
2^-20 * sum_k |x_k L1s[k,i]| of a bf16 rounding boundary, either neighbour is a
correct result, and the two choices differ in Y by |delta lora_i| * |L2[i,n]|
(up to 0.15 at the diffusion-transformer scales: |lora| reaches 512, where one
bf16 step is 4).  The slack adds that difference for exactly those (row, i)
pairs; it is computed from the oracle's values alone."""
from __future__ import annotations

import numpy as np
import torch

from oracle import formats, layout

REL_FRO_TOL = 2e-3
ABS_RMS_TOL = 1e-2

# One record per output check: the unmodified figures and how many elements
# needed each widening of the 1e-2 * rms(Y) bound (printed at the end of the
# test session by conftest.py).
TOLERANCE_LOG = []


def dev_bf16(values_f32: np.ndarray) -> torch.Tensor:
    """float32 values that are exactly bf16 -> CUDA bf16 tensor."""
    bits = formats.bf16_bits(np.asarray(values_f32, dtype=np.float64))
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def dev_bits16(bits: np.ndarray, dtype=torch.bfloat16) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda().view(
        dtype)


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_bf16(t: torch.Tensor) -> np.ndarray:
    """CUDA bf16 tensor -> float64 values."""
    bits = t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return formats.bf16_from_bits(bits)


def half_ulp_bf16(y: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(y, dtype=np.float64))
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))
    return np.ldexp(1.0, e - 9)  # ulp = 2^(e-1-7); half of it


def lora_rounding_slack(X: np.ndarray, L1s: np.ndarray, L2: np.ndarray):
    """(rows, slack[len(rows), N]): the Y slack of the rows that hold an
    ambiguous lora_act rounding (see the module docstring)."""
    X = np.asarray(X, dtype=np.float64)
    L1s = np.asarray(L1s, dtype=np.float64)
    exact = X @ L1s
    ref = formats.round_to_bf16(exact)
    allow = 2.0 ** -20 * (np.abs(X) @ np.abs(L1s))
    amb = np.maximum(np.abs(formats.round_to_bf16(exact + allow) - ref),
                     np.abs(formats.round_to_bf16(exact - allow) - ref))
    rows = np.nonzero(np.any(amb > 0, axis=1))[0]
    return rows, amb[rows] @ np.abs(np.asarray(L2, dtype=np.float64))


def assert_y_close(y_dev: np.ndarray, y_ref: np.ndarray, what: str = "Y", slack=None):
    """slack: None or (rows, extra[len(rows), N]) added to the elementwise
    bound of those rows (lora_rounding_slack)."""
    y_dev = np.asarray(y_dev, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y_dev.shape == y_ref.shape
    assert np.all(np.isfinite(y_dev)), f"{what}: non-finite device output"
    err = y_dev - y_ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-300)
    rms = np.sqrt(np.mean(y_ref ** 2)) if y_ref.size else 0.0
    bound = ABS_RMS_TOL * rms + half_ulp_bf16(y_ref)
    if slack is not None and len(slack[0]):
        bound[slack[0]] += slack[1]
    worst = np.max(np.abs(err) - bound) if err.size else -1.0
    aerr = np.abs(err)
    base = ABS_RMS_TOL * rms
    TOLERANCE_LOG.append({
        "what": what, "elements": int(err.size), "rel_fro": float(rel),
        "max_abs_over_rms": float(aerr.max() / rms) if err.size and rms > 0 else 0.0,
        # beyond 1e-2 rms: admitted by the half-ulp term (or the slack)
        "needed_half_ulp": int(np.count_nonzero(aerr > base)),
        # beyond 1e-2 rms + half ulp: admitted by the lora rounding slack
        "needed_lora_slack": int(np.count_nonzero(aerr > base + half_ulp_bf16(y_ref))),
    })
    assert rel <= REL_FRO_TOL, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO_TOL}"
    assert worst <= 0, (f"{what}: elementwise error exceeds 1e-2*rms + ulp/2 by {worst:.3e} "
                        f"(max |err| {np.max(np.abs(err)):.3e}, rms {rms:.3e})")
    return rel


def oracle_weight_operands(packed: dict, bias_values=None) -> dict:
    """Device buffers of the weight side from the oracle's packing."""
    K, N = packed["K"], packed["N"]
    out = {
        "inv_lambda": dev_f32(packed["inv_lambda"]),
        "L1s": dev_bits16(formats.bf16_bits(packed["L1s"]).T.copy()),     # [r][K]
        # [N][r], divided by the power-of-two tensor scale (exact)
        "L2": dev_bits16(formats.bf16_bits(packed["L2"].T / packed["s_T"])),
        "w_codes": dev_u8(packed["w_codes_packed"]),
        "w_scales": dev_u8(packed["w_scales_swizzled"]),
        "s_T": float(packed["s_T"]),
        "bias": dev_bf16(bias_values) if bias_values is not None else None,
        "K": K, "N": N, "rank": packed["rank"],
    }
    return out


def scales_from_device(a_scales: torch.Tensor, rows: int, K: int) -> np.ndarray:
    return layout.sf_unswizzle(a_scales.cpu().numpy(), rows, K // 16)
