"""SVDQuant W4A4 (NVFP4) linear layer and AWQ W4A16 GEMV for NVIDIA B300.

The compute lives in ``libsvdq.so`` (C ABI, ``include/svdq.h``): hand-written
sm_103a kernels for the per-forward path and C++ host packers for the
offline weight preparation.  This package is the thin Python binding.
"""
from ._lib import (  # noqa: F401
    DEV_OK,
    DEV_TIMEOUT,
    LIB_PATH,
    SvdqError,
    awq_gemv_w4a16,
    awq_pack_weights,
    check_device,
    code_bytes,
    raw_lib,
    scale_bytes,
    status_name,
    svdq_calib_absmax,
    svdq_gemm_w4a4,
    svdq_pack_weights,
    svdq_quantize_act,
)
from .layer import SVDQLinear, AWQLinear  # noqa: F401
