"""SVDQuant W4A4 linear layer (NVFP4, and the INT4 variant) and AWQ W4A16 GEMV
for NVIDIA B300.

The compute lives in ``libsvdq.so`` (C ABI, ``include/svdq.h``): hand-written
sm_103a kernels for the per-forward path and C++ host packers for the
offline weight preparation.  This package is the thin Python binding.

Attributes load the library on first use (so that ``build`` can run before
it exists); any use without a built library raises ImportError.
"""
import importlib

_LIB_NAMES = {
    "DEV_OK", "DEV_TIMEOUT", "LIB_PATH", "SvdqError", "awq_gemv_w4a16", "awq_pack_weights",
    "bench_mma_rate", "check_device", "code_bytes", "raw_lib", "scale_bytes", "status_name",
    "svdq_calib_absmax", "svdq_gemm_w4a4", "svdq_gemm_w4a4_gelu", "svdq_gemm_w4a4_qkv",
    "svdq_gemm_w4a4_gelu_quant", "gelu_quant_scratch_bytes", "svdq_pack_weights",
    "svdq_gemm_w4a4_gelu_quant_static", "GELU_QUANT_STATIC_SCRATCH_BYTES",
    "svdq_quantize_act", "test_set_hooks", "test_quant_sweep",
    "svdq_pack_weights_int4", "svdq_quantize_act_int4", "svdq_gemm_w4a4_int4",
    "int4_scale_bytes",
}
_LAYER_NAMES = {"SVDQLinear", "SVDQLinearInt4", "SVDQMLP", "AWQLinear"}

__all__ = sorted(_LIB_NAMES | _LAYER_NAMES)


def __getattr__(name):
    if name in _LIB_NAMES:
        return getattr(importlib.import_module("._lib", __name__), name)
    if name in _LAYER_NAMES:
        return getattr(importlib.import_module(".layer", __name__), name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
