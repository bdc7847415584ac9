"""Layer-level wrappers: a packed SVDQ W4A4 linear (NVFP4, or the INT4
variant) and an AWQ W4A16 linear
holding their device buffers.  ``forward`` is the per-call path a user runs
(two library calls for SVDQ: svdq_quantize_act then svdq_gemm_w4a4; one for
AWQ).  Pure marshalling: buffers are torch tensors, all arithmetic is in
libsvdq."""
from __future__ import annotations

import numpy as np

from . import _lib


class SVDQLinear:
    """Y = svdq_gemm_w4a4(svdq_quantize_act(X)) for a weight packed once by
    svdq_pack_weights (or given as already packed buffers)."""

    def __init__(self, packed: dict, bias_bf16_bits=None, device="cuda"):
        import torch

        self.N, self.K, self.rank = packed["N"], packed["K"], packed["rank"]
        dev = torch.device(device)

        def t(a, dtype):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dtype)

        self.inv_lambda = t(packed["inv_lambda"].astype(np.float32), torch.float32)
        self.L1s = t(packed["L1s"].astype(np.uint16).view(np.int16), torch.bfloat16)
        self.L2s = t(packed["L2s"].astype(np.uint16).view(np.int16), torch.bfloat16)
        self.w_codes = t(packed["w_codes"].astype(np.uint8), torch.uint8)
        self.w_scales = t(packed["w_scales"].astype(np.uint8), torch.uint8)
        self.w_tensor_scale = float(packed["w_tensor_scale"])
        self.bias = None
        if bias_bf16_bits is not None:
            self.bias = t(np.asarray(bias_bf16_bits, dtype=np.uint16).view(np.int16),
                          torch.bfloat16)

    @classmethod
    def from_float(cls, W: np.ndarray, x_absmax: np.ndarray, rank: int, bias_bf16_bits=None,
                   device="cuda"):
        return cls(_lib.svdq_pack_weights(W, x_absmax, rank), bias_bf16_bits, device)

    def forward(self, X, out=None, act_buffers=None, dev_status=None, stream=None,
                gelu=False):
        """gelu=True returns bf16(gelu_tanh(Y)) (svdq_gemm_w4a4_gelu): the
        first linear of a transformer MLP with its activation fused."""
        M = X.shape[0]
        bufs = act_buffers or (None, None, None)
        a_codes, a_scales, lora = _lib.svdq_quantize_act(
            X, self.inv_lambda, self.L1s, self.rank, *bufs, dev_status=dev_status,
            stream=stream)
        gemm = _lib.svdq_gemm_w4a4_gelu if gelu else _lib.svdq_gemm_w4a4
        return gemm(a_codes, a_scales, self.w_codes, self.w_scales, self.w_tensor_scale, lora,
                    self.L2s, self.bias, M, self.N, self.K, self.rank, out,
                    dev_status=dev_status, stream=stream)

    __call__ = forward


class SVDQLinearInt4:
    """The INT4 variant: Y = svdq_gemm_w4a4_int4(svdq_quantize_act_int4(X))
    for a weight packed once by svdq_pack_weights_int4."""

    def __init__(self, packed: dict, bias_bf16_bits=None, device="cuda"):
        import torch

        self.N, self.K, self.rank = packed["N"], packed["K"], packed["rank"]
        dev = torch.device(device)

        def t(a, dtype):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(dtype)

        def bf16(a):
            return t(np.asarray(a, dtype=np.uint16).view(np.int16), torch.bfloat16)

        self.inv_lambda = t(packed["inv_lambda"].astype(np.float32), torch.float32)
        self.L1s, self.L2 = bf16(packed["L1s"]), bf16(packed["L2"])
        self.w_codes = t(packed["w_codes"].astype(np.uint8), torch.uint8)
        self.w_scales = bf16(packed["w_scales"])
        self.bias = None if bias_bf16_bits is None else bf16(bias_bf16_bits)

    @classmethod
    def from_float(cls, W: np.ndarray, x_absmax: np.ndarray, rank: int, bias_bf16_bits=None,
                   device="cuda"):
        return cls(_lib.svdq_pack_weights_int4(W, x_absmax, rank), bias_bf16_bits, device)

    def forward(self, X, out=None, act_buffers=None, dev_status=None, stream=None):
        M = X.shape[0]
        bufs = act_buffers or (None, None, None)
        a_codes, a_scales, lora = _lib.svdq_quantize_act_int4(
            X, self.inv_lambda, self.L1s, self.rank, *bufs, dev_status=dev_status,
            stream=stream)
        return _lib.svdq_gemm_w4a4_int4(a_codes, a_scales, self.w_codes, self.w_scales, lora,
                                        self.L2, self.bias, M, self.N, self.K, self.rank, out,
                                        dev_status=dev_status, stream=stream)

    __call__ = forward


class SVDQMLP:
    """Y2 = fc2(gelu_tanh(fc1(X))) for two SVDQ linears, fc1.N == fc2.K.  The
    fused path is three library calls: svdq_quantize_act (fc1's activation
    side), svdq_gemm_w4a4_gelu_quant (fc1 with GELU and fc2's activation side
    in its epilogue: H is never written) and svdq_gemm_w4a4 (fc2).
    fused=False runs fc1 with the GELU epilogue, writes H, and runs fc2 on it
    (the four-call path), for comparison."""

    def __init__(self, fc1: SVDQLinear, fc2: SVDQLinear):
        if fc1.N != fc2.K:
            raise ValueError(f"fc1.N = {fc1.N} must equal fc2.K = {fc2.K}")
        self.fc1, self.fc2 = fc1, fc2
        self._scratch = None

    def _scratch_for(self, M, device):
        import torch

        need = _lib.gelu_quant_scratch_bytes(M, self.fc1.N, self.fc2.rank)
        if self._scratch is None or self._scratch.numel() < need or \
                self._scratch.device != device:
            self._scratch = torch.empty(need, dtype=torch.uint8, device=device)
        return self._scratch

    def forward(self, X, out=None, fused=True, dev_status=None, stream=None):
        fc1, fc2 = self.fc1, self.fc2
        M = X.shape[0]
        if not fused:
            H = fc1(X, gelu=True, dev_status=dev_status, stream=stream)
            return fc2(H, out=out, dev_status=dev_status, stream=stream)
        a_codes, a_scales, lora = _lib.svdq_quantize_act(
            X, fc1.inv_lambda, fc1.L1s, fc1.rank, dev_status=dev_status, stream=stream)
        a2_codes, a2_scales, lora2 = _lib.svdq_gemm_w4a4_gelu_quant(
            a_codes, a_scales, fc1.w_codes, fc1.w_scales, fc1.w_tensor_scale, lora, fc1.L2s,
            fc1.bias, fc2.inv_lambda, fc2.L1s, fc2.rank, M, fc1.N, fc1.K, fc1.rank,
            scratch=self._scratch_for(M, X.device), dev_status=dev_status, stream=stream)
        return _lib.svdq_gemm_w4a4(a2_codes, a2_scales, fc2.w_codes, fc2.w_scales,
                                   fc2.w_tensor_scale, lora2, fc2.L2s, fc2.bias, M, fc2.N,
                                   fc2.K, fc2.rank, out, dev_status=dev_status, stream=stream)

    __call__ = forward


class AWQLinear:
    """Y = awq_gemv_w4a16(X) for a weight packed by awq_pack_weights."""

    def __init__(self, qweight, scales, zeros, bias_bf16_bits=None, device="cuda"):
        import torch

        dev = torch.device(device)
        self.qweight = torch.from_numpy(np.ascontiguousarray(qweight)).to(dev)
        self.scales = torch.from_numpy(np.ascontiguousarray(scales).view(np.int16)).to(dev)
        self.zeros = torch.from_numpy(np.ascontiguousarray(zeros).view(np.int16)).to(dev)
        self.bias = None
        if bias_bf16_bits is not None:
            self.bias = torch.from_numpy(
                np.asarray(bias_bf16_bits, dtype=np.uint16).view(np.int16)).to(dev).view(
                    torch.bfloat16)
        self.N = self.qweight.shape[0]

    @classmethod
    def from_float(cls, W: np.ndarray, bias_bf16_bits=None, device="cuda"):
        q, s, z = _lib.awq_pack_weights(W, 64)
        return cls(q, s, z, bias_bf16_bits, device)

    def forward(self, X, out=None, stream=None):
        return _lib.awq_gemv_w4a16(X, self.qweight, self.scales, self.zeros, self.bias, 64,
                                   Y=out, stream=stream)

    __call__ = forward
