"""ctypes binding of libsvdq (include/svdq.h): argument marshalling only.

Device calls take torch CUDA tensors (PyTorch provides device memory and
streams); host calls take NumPy arrays.  Outputs that are not passed in are
allocated here with torch/NumPy; every computation happens in the library.
A missing library raises ImportError: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsvdq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python -m bit_w4a4_diffusion_quantize_b300.build` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

_c_p = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_f32 = ctypes.c_float

STATUS = {
    0: "SVDQ_OK", -1: "SVDQ_ERR_NULL", -2: "SVDQ_ERR_SHAPE", -3: "SVDQ_ERR_ALIGN",
    -4: "SVDQ_ERR_UNSUPPORTED_ARCH", -5: "SVDQ_ERR_CUDA", -6: "SVDQ_ERR_RANK",
    -7: "SVDQ_ERR_VALUE", -8: "SVDQ_ERR_NOMEM",
}
DEV_OK = 0
DEV_TIMEOUT = 1

_SIGS = {
    "svdq_status_string": (ctypes.c_char_p, [_i32]),
    "svdq_check_device": (_i32, []),
    "svdq_calib_absmax": (_i32, [_c_p, _i64, _i64, _c_p]),
    "svdq_pack_weights": (_i32, [_c_p, _i32, _i32, _c_p, _i32, _c_p, _c_p, _c_p, _c_p, _c_p,
                                 _c_p]),
    "awq_pack_weights": (_i32, [_c_p, _i32, _i32, _i32, _c_p, _c_p, _c_p]),
    "svdq_pack_weights_int4": (_i32, [_c_p, _i32, _i32, _c_p, _i32, _c_p, _c_p, _c_p, _c_p,
                                      _c_p]),
    "svdq_quantize_act_int4": (_i32, [_c_p, _c_p, _c_p, _i32, _i32, _i32, _c_p, _c_p, _c_p,
                                      _c_p, _c_p]),
    "svdq_gemm_w4a4_int4": (_i32, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _i32, _i32,
                                   _i32, _i32, _c_p, _c_p]),
    "svdq_quantize_act": (_i32, [_c_p, _c_p, _c_p, _i32, _i32, _i32, _c_p, _c_p, _c_p, _c_p,
                                 _c_p]),
    "svdq_gemm_w4a4": (_i32, [_c_p, _c_p, _c_p, _c_p, _f32, _c_p, _c_p, _c_p, _c_p, _i32,
                              _i32, _i32, _i32, _c_p, _c_p]),
    "svdq_gemm_w4a4_gelu": (_i32, [_c_p, _c_p, _c_p, _c_p, _f32, _c_p, _c_p, _c_p, _c_p,
                                   _i32, _i32, _i32, _i32, _c_p, _c_p]),
    "svdq_gemm_w4a4_qkv": (_i32, [_c_p, _c_p, _c_p, _c_p, _f32, _c_p, _c_p, _c_p, _c_p, _c_p,
                                  _c_p, _c_p, _f32, _c_p, _i32, _i32, _i32, _i32, _c_p, _c_p]),
    "svdq_gemm_w4a4_gelu_quant": (_i32, [_c_p, _c_p, _c_p, _c_p, _f32, _c_p, _c_p, _c_p,
                                         _c_p, _c_p, _i32, _c_p, _c_p, _c_p, _c_p, _c_p,
                                         ctypes.c_size_t, _i32, _i32, _i32, _i32, _c_p, _c_p]),
    "svdq_gemm_w4a4_gelu_quant_static": (_i32, [_c_p, _c_p, _c_p, _c_p, _f32, _c_p, _c_p,
                                                _c_p, _c_p, _c_p, _i32, _c_p, _c_p, _c_p, _c_p,
                                                _i32, _i32, _i32, _i32, _c_p, _c_p]),
    "awq_gemv_w4a16": (_i32, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _i32, _i32, _i32, _i32,
                              _c_p, _c_p]),
    "svdq_bench_mma_rate": (_i32, [_i32, _i32, _i32, _i32, _c_p, _c_p]),
    "svdq_test_set_hooks": (_i32, [_i32, _i32]),
    "svdq_test_quant_sweep": (_i32, [_i32, _c_p, _c_p]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class SvdqError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        msg = _lib.svdq_status_string(status)
        super().__init__(f"{call}: {msg.decode() if msg else STATUS.get(status, status)}")


def _check(status: int, call: str):
    if status != 0:
        raise SvdqError(status, call)


def status_name(status: int) -> str:
    return STATUS.get(status, str(status))


def raw_lib():
    """The ctypes handle (for tests that call the C ABI directly)."""
    return _lib


# --------------------------------------------------------------------------- sizes
def code_bytes(rows: int, K: int) -> int:
    return rows * K // 2


def scale_bytes(rows: int, K: int) -> int:
    return ((rows + 127) // 128) * 128 * (K // 16)


def int4_scale_bytes(rows: int, K: int) -> int:
    """Bytes of an INT4-variant scale buffer: [rows][K/64] bf16."""
    return rows * (K // 64) * 2


def gelu_quant_scratch_bytes(M: int, N: int, rank2: int) -> int:
    """Scratch svdq_gemm_w4a4_gelu_quant needs (SVDQ_GELU_QUANT_SCRATCH_BYTES)."""
    return (128 + (M + 255) // 256) * 256 * rank2 * 4


# --------------------------------------------------------------------------- host calls
def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def check_device() -> int:
    """Status of svdq_check_device (0 when the current device is CC 10.3)."""
    return int(_lib.svdq_check_device())


def svdq_calib_absmax(X_bf16_bits: np.ndarray) -> np.ndarray:
    X = np.ascontiguousarray(X_bf16_bits, dtype=np.uint16)
    M, K = X.shape
    out = np.zeros(K, dtype=np.float32)
    _check(_lib.svdq_calib_absmax(_np_ptr(X), M, K, _np_ptr(out)), "svdq_calib_absmax")
    return out


def svdq_pack_weights(W: np.ndarray, x_absmax: np.ndarray, rank: int) -> dict:
    """Offline packing of an nn.Linear weight W [N, K] (float32).  Returns the
    device-side buffers as NumPy arrays: inv_lambda [K] fp32, L1s [rank, K]
    and L2s [N, rank] bf16 bits (L2s = L2^T / s_T), w_codes [N, K/2],
    w_scales (tile layout), w_tensor_scale."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    xm = np.ascontiguousarray(x_absmax, dtype=np.float32)
    N, K = W.shape
    r = max(int(rank), 0)
    inv = np.zeros(K, dtype=np.float32)
    L1s = np.zeros((r, K), dtype=np.uint16)
    L2s = np.zeros((N, r), dtype=np.uint16)
    codes = np.zeros((N, K // 2), dtype=np.uint8)
    scales = np.zeros(scale_bytes(N, K), dtype=np.uint8)
    sT = np.zeros(1, dtype=np.float32)
    st = _lib.svdq_pack_weights(_np_ptr(W), N, K, _np_ptr(xm), int(rank), _np_ptr(inv),
                                _np_ptr(L1s), _np_ptr(L2s), _np_ptr(codes), _np_ptr(scales),
                                _np_ptr(sT))
    _check(st, "svdq_pack_weights")
    return {"N": N, "K": K, "rank": int(rank), "inv_lambda": inv, "L1s": L1s, "L2s": L2s,
            "w_codes": codes, "w_scales": scales, "w_tensor_scale": float(sT[0])}


def svdq_pack_weights_int4(W: np.ndarray, x_absmax: np.ndarray, rank: int) -> dict:
    """Offline packing, INT4 variant, of an nn.Linear weight W [N, K]
    (float32).  Returns inv_lambda [K] fp32, L1s [rank, K] and L2 [N, rank]
    bf16 bits, w_codes [N, K/2] and w_scales [N, K/64] bf16 bits."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    xm = np.ascontiguousarray(x_absmax, dtype=np.float32)
    N, K = W.shape
    r = max(int(rank), 0)
    inv = np.zeros(K, dtype=np.float32)
    L1s = np.zeros((r, K), dtype=np.uint16)
    L2 = np.zeros((N, r), dtype=np.uint16)
    codes = np.zeros((N, K // 2), dtype=np.uint8)
    scales = np.zeros((N, K // 64), dtype=np.uint16)
    st = _lib.svdq_pack_weights_int4(_np_ptr(W), N, K, _np_ptr(xm), int(rank), _np_ptr(inv),
                                     _np_ptr(L1s), _np_ptr(L2), _np_ptr(codes), _np_ptr(scales))
    _check(st, "svdq_pack_weights_int4")
    return {"N": N, "K": K, "rank": int(rank), "inv_lambda": inv, "L1s": L1s, "L2": L2,
            "w_codes": codes, "w_scales": scales}


def awq_pack_weights(W: np.ndarray, group_size: int = 64):
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    G = K // 64 if group_size == 64 and K % 64 == 0 else 1
    q = np.zeros((N, K // 2), dtype=np.uint8)
    s = np.zeros((N, G), dtype=np.uint16)
    z = np.zeros((N, G), dtype=np.uint16)
    _check(_lib.awq_pack_weights(_np_ptr(W), N, K, int(group_size), _np_ptr(q), _np_ptr(s),
                                 _np_ptr(z)), "awq_pack_weights")
    return q, s, z


# --------------------------------------------------------------------------- device calls
def _torch():
    import torch
    return torch


def _dptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_cuda(t, name):
    if t is not None:
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (the library reads raw row-major memory)")
        cur = _torch().cuda.current_device()
        if t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}; the library runs on the current device "
                             f"(cuda:{cur})")


_WIDTH = {1: "8-bit", 2: "16-bit", 4: "32-bit"}


def _need(t, name: str, elems: int, size: int):
    """The kernels read or write `elems` elements of `size` bytes through t's
    pointer: refuse a tensor of another element width or fewer elements (a
    short buffer would be overrun on the device).  An empty need checks
    nothing (no byte of t is touched)."""
    if t is None or elems <= 0:
        return
    if t.element_size() != size:
        raise ValueError(f"{name}: {_WIDTH[size]} elements expected, got {t.dtype}")
    if t.numel() < elems:
        raise ValueError(f"{name}: {elems} elements needed, the tensor holds {t.numel()}")


def svdq_quantize_act(X, inv_lambda, L1s, rank: int, a_codes=None, a_scales=None,
                      lora_act=None, dev_status=None, stream=None):
    """X: CUDA bf16 (or int16/uint16 bits) [M, K]; inv_lambda fp32 [K];
    L1s bf16 bits [rank, K].  Returns (a_codes, a_scales, lora_act)."""
    torch = _torch()
    for t, n in ((X, "X"), (inv_lambda, "inv_lambda"), (L1s, "L1s"), (a_codes, "a_codes"),
                 (a_scales, "a_scales"), (lora_act, "lora_act"), (dev_status, "dev_status")):
        _check_cuda(t, n)
    M, K = X.shape
    dev = X.device
    if a_codes is None:
        a_codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    if a_scales is None:
        a_scales = torch.empty(scale_bytes(M, K), dtype=torch.uint8, device=dev)
    if lora_act is None:
        lora_act = torch.empty((M, rank), dtype=torch.bfloat16, device=dev)
    if M > 0:
        for t, n, e, z in ((X, "X", M * K, 2), (inv_lambda, "inv_lambda", K, 4),
                           (L1s, "L1s", rank * K, 2), (a_codes, "a_codes", code_bytes(M, K), 1),
                           (a_scales, "a_scales", scale_bytes(M, K), 1),
                           (lora_act, "lora_act", M * rank, 2), (dev_status, "dev_status", 1, 4)):
            _need(t, n, e, z)
    st = _lib.svdq_quantize_act(_dptr(X), _dptr(inv_lambda), _dptr(L1s), M, K, int(rank),
                                _dptr(a_codes), _dptr(a_scales), _dptr(lora_act),
                                _dptr(dev_status), _stream_ptr(stream))
    _check(st, "svdq_quantize_act")
    return a_codes, a_scales, lora_act


def svdq_quantize_act_int4(X, inv_lambda, L1s, rank: int, a_codes=None, a_scales=None,
                           lora_act=None, dev_status=None, stream=None):
    """INT4 variant.  X: CUDA bf16 [M, K]; inv_lambda fp32 [K]; L1s bf16
    bits [rank, K].  Returns (a_codes [M, K/2] uint8, a_scales [M, K/64]
    bf16, lora_act [M, rank] bf16)."""
    torch = _torch()
    for t, n in ((X, "X"), (inv_lambda, "inv_lambda"), (L1s, "L1s"), (a_codes, "a_codes"),
                 (a_scales, "a_scales"), (lora_act, "lora_act"), (dev_status, "dev_status")):
        _check_cuda(t, n)
    M, K = X.shape
    dev = X.device
    if a_codes is None:
        a_codes = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    if a_scales is None:
        a_scales = torch.empty((M, K // 64), dtype=torch.bfloat16, device=dev)
    if lora_act is None:
        lora_act = torch.empty((M, rank), dtype=torch.bfloat16, device=dev)
    if M > 0:
        for t, n, e, z in ((X, "X", M * K, 2), (inv_lambda, "inv_lambda", K, 4),
                           (L1s, "L1s", rank * K, 2), (a_codes, "a_codes", code_bytes(M, K), 1),
                           (a_scales, "a_scales", M * (K // 64), 2),
                           (lora_act, "lora_act", M * rank, 2), (dev_status, "dev_status", 1, 4)):
            _need(t, n, e, z)
    st = _lib.svdq_quantize_act_int4(_dptr(X), _dptr(inv_lambda), _dptr(L1s), M, K, int(rank),
                                     _dptr(a_codes), _dptr(a_scales), _dptr(lora_act),
                                     _dptr(dev_status), _stream_ptr(stream))
    _check(st, "svdq_quantize_act_int4")
    return a_codes, a_scales, lora_act


def svdq_gemm_w4a4_int4(a_codes, a_scales, w_codes, w_scales, lora_act, L2, bias, M: int,
                        N: int, K: int, rank: int, Y=None, dev_status=None, stream=None):
    """INT4 variant.  a_scales [M, K/64] and w_scales [N, K/64] bf16, L2
    [N, rank] bf16.  Returns Y [M, N] bf16 (CUDA)."""
    torch = _torch()
    for t, n in ((a_codes, "a_codes"), (a_scales, "a_scales"), (w_codes, "w_codes"),
                 (w_scales, "w_scales"), (lora_act, "lora_act"), (L2, "L2"), (bias, "bias"),
                 (Y, "Y"), (dev_status, "dev_status")):
        _check_cuda(t, n)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    if M > 0:
        for t, n, e, z in ((a_codes, "a_codes", code_bytes(M, K), 1),
                           (a_scales, "a_scales", M * (K // 64), 2),
                           (w_codes, "w_codes", code_bytes(N, K), 1),
                           (w_scales, "w_scales", N * (K // 64), 2),
                           (lora_act, "lora_act", M * rank, 2), (L2, "L2", N * rank, 2),
                           (bias, "bias", N, 2), (Y, "Y", M * N, 2),
                           (dev_status, "dev_status", 1, 4)):
            _need(t, n, e, z)
    st = _lib.svdq_gemm_w4a4_int4(_dptr(a_codes), _dptr(a_scales), _dptr(w_codes),
                                  _dptr(w_scales), _dptr(lora_act), _dptr(L2), _dptr(bias),
                                  _dptr(Y), int(M), int(N), int(K), int(rank),
                                  _dptr(dev_status), _stream_ptr(stream))
    _check(st, "svdq_gemm_w4a4_int4")
    return Y


def _gemm(name, a_codes, a_scales, w_codes, w_scales, w_tensor_scale, lora_act, L2s, bias, M,
          N, K, rank, Y, dev_status, stream):
    torch = _torch()
    for t, n in ((a_codes, "a_codes"), (a_scales, "a_scales"), (w_codes, "w_codes"),
                 (w_scales, "w_scales"), (lora_act, "lora_act"), (L2s, "L2s"), (bias, "bias"),
                 (Y, "Y"), (dev_status, "dev_status")):
        _check_cuda(t, n)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    if M > 0:
        for t, n, e, z in ((a_codes, "a_codes", code_bytes(M, K), 1),
                           (a_scales, "a_scales", scale_bytes(M, K), 1),
                           (w_codes, "w_codes", code_bytes(N, K), 1),
                           (w_scales, "w_scales", scale_bytes(N, K), 1),
                           (lora_act, "lora_act", M * rank, 2), (L2s, "L2s", N * rank, 2),
                           (bias, "bias", N, 2), (Y, "Y", M * N, 2),
                           (dev_status, "dev_status", 1, 4)):
            _need(t, n, e, z)
    st = getattr(_lib, name)(_dptr(a_codes), _dptr(a_scales), _dptr(w_codes), _dptr(w_scales),
                             float(w_tensor_scale), _dptr(lora_act), _dptr(L2s), _dptr(bias),
                             _dptr(Y), int(M), int(N), int(K), int(rank), _dptr(dev_status),
                             _stream_ptr(stream))
    _check(st, name)
    return Y


def svdq_gemm_w4a4(a_codes, a_scales, w_codes, w_scales, w_tensor_scale: float, lora_act, L2s,
                   bias, M: int, N: int, K: int, rank: int, Y=None, dev_status=None,
                   stream=None):
    """L2s: [N, rank] bf16 = L2^T / s_T.  Returns Y [M, N] bf16 (CUDA)."""
    return _gemm("svdq_gemm_w4a4", a_codes, a_scales, w_codes, w_scales, w_tensor_scale,
                 lora_act, L2s, bias, M, N, K, rank, Y, dev_status, stream)


def svdq_gemm_w4a4_gelu(a_codes, a_scales, w_codes, w_scales, w_tensor_scale: float, lora_act,
                        L2s, bias, M: int, N: int, K: int, rank: int, H=None, dev_status=None,
                        stream=None):
    """svdq_gemm_w4a4 followed by GELU (tanh form) in its epilogue: returns
    H = bf16(gelu_tanh(Y)) [M, N] (CUDA)."""
    return _gemm("svdq_gemm_w4a4_gelu", a_codes, a_scales, w_codes, w_scales, w_tensor_scale,
                 lora_act, L2s, bias, M, N, K, rank, H, dev_status, stream)


def svdq_gemm_w4a4_qkv(a_codes, a_scales, w_codes, w_scales, w_tensor_scale: float, lora_act,
                       L2s, bias, norm_q, norm_k, rope_cos, rope_sin, M: int, N: int, K: int,
                       rank: int, eps: float = 1e-6, QKV=None, dev_status=None, stream=None):
    """svdq_gemm_w4a4 of a fused Q|K|V projection (N = 3 x heads x 128) with the
    per-head RMS normalization of Q and K (weights norm_q, norm_k: [128] bf16)
    and the rotary embedding (rope_cos, rope_sin: [M, 64] fp32) in its
    epilogue.  Returns QKV [M, N] bf16 (CUDA)."""
    torch = _torch()
    for t, n in ((a_codes, "a_codes"), (a_scales, "a_scales"), (w_codes, "w_codes"),
                 (w_scales, "w_scales"), (lora_act, "lora_act"), (L2s, "L2s"), (bias, "bias"),
                 (norm_q, "norm_q"), (norm_k, "norm_k"), (rope_cos, "rope_cos"),
                 (rope_sin, "rope_sin"), (QKV, "QKV"), (dev_status, "dev_status")):
        _check_cuda(t, n)
    if QKV is None:
        QKV = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    if M > 0:
        for t, n, e, z in ((a_codes, "a_codes", code_bytes(M, K), 1),
                           (a_scales, "a_scales", scale_bytes(M, K), 1),
                           (w_codes, "w_codes", code_bytes(N, K), 1),
                           (w_scales, "w_scales", scale_bytes(N, K), 1),
                           (lora_act, "lora_act", M * rank, 2), (L2s, "L2s", N * rank, 2),
                           (bias, "bias", N, 2), (norm_q, "norm_q", 128, 2),
                           (norm_k, "norm_k", 128, 2), (rope_cos, "rope_cos", M * 64, 4),
                           (rope_sin, "rope_sin", M * 64, 4), (QKV, "QKV", M * N, 2),
                           (dev_status, "dev_status", 1, 4)):
            _need(t, n, e, z)
    st = _lib.svdq_gemm_w4a4_qkv(_dptr(a_codes), _dptr(a_scales), _dptr(w_codes),
                                 _dptr(w_scales), float(w_tensor_scale), _dptr(lora_act),
                                 _dptr(L2s), _dptr(bias), _dptr(norm_q), _dptr(norm_k),
                                 _dptr(rope_cos), _dptr(rope_sin), float(eps), _dptr(QKV),
                                 int(M), int(N), int(K), int(rank), _dptr(dev_status),
                                 _stream_ptr(stream))
    _check(st, "svdq_gemm_w4a4_qkv")
    return QKV


def svdq_gemm_w4a4_gelu_quant(a_codes, a_scales, w_codes, w_scales, w_tensor_scale: float,
                              lora_act, L2s, bias, inv_lambda2, L1s2, rank2: int, M: int, N: int,
                              K: int, rank: int, a2_codes=None, a2_scales=None, lora_act2=None,
                              H=None, scratch=None, dev_status=None, stream=None):
    """svdq_gemm_w4a4_gelu with the next SVDQ linear's activation side fused:
    returns (a2_codes, a2_scales, lora_act2) of H = bf16(gelu_tanh(Y)) for the
    layer with inv_lambda2 [N] fp32 and L1s2 bf16 bits [rank2, N]; H [M, N]
    bf16 is written only when passed.  `scratch` (uint8/float, CUDA) holds at
    least gelu_quant_scratch_bytes(M, N, rank2) bytes (allocated if None)."""
    torch = _torch()
    for t, n in ((a_codes, "a_codes"), (a_scales, "a_scales"), (w_codes, "w_codes"),
                 (w_scales, "w_scales"), (lora_act, "lora_act"), (L2s, "L2s"), (bias, "bias"),
                 (inv_lambda2, "inv_lambda2"), (L1s2, "L1s2"), (a2_codes, "a2_codes"),
                 (a2_scales, "a2_scales"), (lora_act2, "lora_act2"), (H, "H"),
                 (scratch, "scratch"), (dev_status, "dev_status")):
        _check_cuda(t, n)
    dev = a_codes.device
    if a2_codes is None:
        a2_codes = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    if a2_scales is None:
        a2_scales = torch.empty(scale_bytes(M, N), dtype=torch.uint8, device=dev)
    if lora_act2 is None:
        lora_act2 = torch.empty((M, rank2), dtype=torch.bfloat16, device=dev)
    need = gelu_quant_scratch_bytes(M, N, rank2)
    if scratch is None:
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if M > 0:
        for t, n, e, z in ((a_codes, "a_codes", code_bytes(M, K), 1),
                           (a_scales, "a_scales", scale_bytes(M, K), 1),
                           (w_codes, "w_codes", code_bytes(N, K), 1),
                           (w_scales, "w_scales", scale_bytes(N, K), 1),
                           (lora_act, "lora_act", M * rank, 2), (L2s, "L2s", N * rank, 2),
                           (bias, "bias", N, 2), (inv_lambda2, "inv_lambda2", N, 4),
                           (L1s2, "L1s2", rank2 * N, 2),
                           (a2_codes, "a2_codes", code_bytes(M, N), 1),
                           (a2_scales, "a2_scales", scale_bytes(M, N), 1),
                           (lora_act2, "lora_act2", M * rank2, 2), (H, "H", M * N, 2),
                           (dev_status, "dev_status", 1, 4)):
            _need(t, n, e, z)
    scratch_bytes = scratch.numel() * scratch.element_size()
    st = _lib.svdq_gemm_w4a4_gelu_quant(
        _dptr(a_codes), _dptr(a_scales), _dptr(w_codes), _dptr(w_scales), float(w_tensor_scale),
        _dptr(lora_act), _dptr(L2s), _dptr(bias), _dptr(inv_lambda2), _dptr(L1s2), int(rank2),
        _dptr(a2_codes), _dptr(a2_scales), _dptr(lora_act2), _dptr(H), _dptr(scratch),
        int(scratch_bytes), int(M), int(N), int(K), int(rank), _dptr(dev_status),
        _stream_ptr(stream))
    _check(st, "svdq_gemm_w4a4_gelu_quant")
    return a2_codes, a2_scales, lora_act2


GELU_QUANT_STATIC_SCRATCH_BYTES = 16 << 20


def svdq_gemm_w4a4_gelu_quant_static(a_codes, a_scales, w_codes, w_scales,
                                     w_tensor_scale: float, lora_act, L2s, bias, inv_lambda2,
                                     L1s2, rank2: int, M: int, N: int, K: int, rank: int,
                                     a2_codes, a2_scales, lora_act2, H=None, dev_status=None,
                                     stream=None):
    """svdq_gemm_w4a4_gelu_quant with the library's static device scratch
    (include/svdq.h): nothing is allocated, here or in the library, so every
    output must be passed.  Calls on one device must not overlap in time."""
    for t, n in ((a_codes, "a_codes"), (a_scales, "a_scales"), (w_codes, "w_codes"),
                 (w_scales, "w_scales"), (lora_act, "lora_act"), (L2s, "L2s"), (bias, "bias"),
                 (inv_lambda2, "inv_lambda2"), (L1s2, "L1s2"), (a2_codes, "a2_codes"),
                 (a2_scales, "a2_scales"), (lora_act2, "lora_act2"), (H, "H"),
                 (dev_status, "dev_status")):
        _check_cuda(t, n)
    if M > 0:
        for t, n, e, z in ((a_codes, "a_codes", code_bytes(M, K), 1),
                           (a_scales, "a_scales", scale_bytes(M, K), 1),
                           (w_codes, "w_codes", code_bytes(N, K), 1),
                           (w_scales, "w_scales", scale_bytes(N, K), 1),
                           (lora_act, "lora_act", M * rank, 2), (L2s, "L2s", N * rank, 2),
                           (bias, "bias", N, 2), (inv_lambda2, "inv_lambda2", N, 4),
                           (L1s2, "L1s2", rank2 * N, 2),
                           (a2_codes, "a2_codes", code_bytes(M, N), 1),
                           (a2_scales, "a2_scales", scale_bytes(M, N), 1),
                           (lora_act2, "lora_act2", M * rank2, 2), (H, "H", M * N, 2),
                           (dev_status, "dev_status", 1, 4)):
            if t is None and n not in ("bias", "H", "dev_status"):
                raise ValueError(f"{n}: required (this call allocates nothing)")
            _need(t, n, e, z)
    if gelu_quant_scratch_bytes(M, N, rank2) > GELU_QUANT_STATIC_SCRATCH_BYTES and rank2 in (32, 64):
        raise SvdqError(-2, f"svdq_gemm_w4a4_gelu_quant_static: M = {M} needs "
                            f"{gelu_quant_scratch_bytes(M, N, rank2)} bytes of scratch, the "
                            f"static scratch holds {GELU_QUANT_STATIC_SCRATCH_BYTES}")
    st = _lib.svdq_gemm_w4a4_gelu_quant_static(
        _dptr(a_codes), _dptr(a_scales), _dptr(w_codes), _dptr(w_scales), float(w_tensor_scale),
        _dptr(lora_act), _dptr(L2s), _dptr(bias), _dptr(inv_lambda2), _dptr(L1s2), int(rank2),
        _dptr(a2_codes), _dptr(a2_scales), _dptr(lora_act2), _dptr(H), int(M), int(N), int(K),
        int(rank), _dptr(dev_status), _stream_ptr(stream))
    _check(st, "svdq_gemm_w4a4_gelu_quant_static")
    return a2_codes, a2_scales, lora_act2


def awq_gemv_w4a16(X, qweight, scales, zeros, bias, group_size: int = 64, Y=None,
                   dev_status=None, stream=None):
    """X: CUDA bf16 [M, K] (M <= 8); returns Y [M, N] bf16."""
    torch = _torch()
    for t, n in ((X, "X"), (qweight, "qweight"), (scales, "scales"), (zeros, "zeros"),
                 (bias, "bias"), (Y, "Y"), (dev_status, "dev_status")):
        _check_cuda(t, n)
    M, K = X.shape
    N = qweight.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    groups = K // group_size if group_size > 0 else 0
    for t, n, e, z in ((X, "X", M * K, 2), (qweight, "qweight", N * K // 2, 1),
                       (scales, "scales", N * groups, 2), (zeros, "zeros", N * groups, 2),
                       (bias, "bias", N, 2), (Y, "Y", M * N, 2), (dev_status, "dev_status", 1, 4)):
        _need(t, n, e, z)
    st = _lib.awq_gemv_w4a16(_dptr(X), _dptr(qweight), _dptr(scales), _dptr(zeros), _dptr(bias),
                             _dptr(Y), int(M), int(N), int(K), int(group_size),
                             _dptr(dev_status), _stream_ptr(stream))
    _check(st, "awq_gemv_w4a16")
    return Y


def bench_mma_rate(mode: int, n: int, iters: int, ctas: int, dev_status=None, stream=None):
    """Launch the tensor-core rate kernel (include/svdq_bench.h); time it with
    CUDA events on `stream`."""
    _check(_lib.svdq_bench_mma_rate(int(mode), int(n), int(iters), int(ctas), _dptr(dev_status),
                                    _stream_ptr(stream)), "svdq_bench_mma_rate")


def test_set_hooks(fake_compute_capability: int = 0, gemm_stall: int = 0):
    """Test hooks of the library (include/svdq_test.h): a compute capability to
    report instead of the device's (10 * major + minor, 0 = off) and a GEMM
    loader that issues nothing (1), so that its bounded waits run out."""
    _check(_lib.svdq_test_set_hooks(int(fake_compute_capability), int(gemm_stall)),
           "svdq_test_set_hooks")


def test_quant_sweep(which: int, stream=None):
    """Run the exhaustive rounding check (include/svdq_test.h); returns
    (mismatching blocks, smallest mismatching fp32 bit pattern or None,
    blocks checked)."""
    torch = _torch()
    out = torch.tensor([0, -1, 0, 0], dtype=torch.int64, device="cuda")
    _check(_lib.svdq_test_quant_sweep(int(which), _dptr(out), _stream_ptr(stream)),
           "svdq_test_quant_sweep")
    torch.cuda.synchronize()
    count, first, checked, _ = (int(v) for v in out.cpu().tolist())
    return count, (None if count == 0 else first & 0xFFFFFFFF), checked
