/*
 * svdq_test.h -- test hooks of libsvdq (not part of the layer; the pages
 * have no counterpart).
 *
 * svdq_test_set_hooks lets a test exercise two error paths that a healthy
 * B300 never takes, without faulting or hanging the GPU:
 *   fake_compute_capability  10 * major + minor of a capability the device
 *                            calls then report instead of the device's own
 *                            (so 90 makes every device call return
 *                            SVDQ_ERR_UNSUPPORTED_ARCH); 0 turns it off.
 *   gemm_stall               1: the loader of svdq_gemm_w4a4 (and of its
 *                            variants) issues no copy, so the kernel's bounded
 *                            pipeline waits run out after 100 ms, it writes
 *                            SVDQ_DEV_TIMEOUT to dev_status and returns; 0 off.
 * The settings are process-wide and hold until the next call.  Both are off
 * at load.  Errors: SVDQ_ERR_VALUE (negative capability, stall not 0 or 1).
 */
#ifndef SVDQ_TEST_H_
#define SVDQ_TEST_H_

#include "svdq.h"

#ifdef __cplusplus
extern "C" {
#endif

svdq_status svdq_test_set_hooks(int fake_compute_capability, int gemm_stall);

/* Exhaustive check of the activation quantization's division-free rounding
 * (the routine svdq_quantize_act and the GELU + quantization epilogue share)
 * against IEEE division followed by the same round-to-nearest-even
 * conversion, which equals the exact rounding of the quotient (a correctly
 * rounded fp32 quotient of a 24-bit value by 6 or by an e4m3 scale lands on an
 * e4m3 / e2m1 rounding midpoint only when the exact quotient is that
 * midpoint):
 *   which 0  every finite non-negative fp32 value as a block's amax: its scale
 *            byte RNE_e4m3(amax / 6);
 *   which 1  every positive finite e4m3 scale s, the block amax 6 s, and every
 *            fp32 value of magnitude in [6 s 2^-8, 6 s) with both signs: its
 *            code RNE_e2m1(x / s) (and the block's scale byte).
 * dev_out: device, 16-byte aligned, three u64: the caller sets [0] = 0,
 * [1] = ~0 and [2] = 0; the kernel adds 1 to [0] per mismatching block,
 * lowers [1] to the smallest mismatching fp32 bit pattern and adds the number
 * of blocks it checked to [2] (0x7F800000 for which 0; 126 x
 * ceil(2^26 / 7) for which 1).  Asynchronous on `stream`.
 * Errors: SVDQ_ERR_VALUE (which), SVDQ_ERR_NULL, SVDQ_ERR_ALIGN,
 * SVDQ_ERR_UNSUPPORTED_ARCH, SVDQ_ERR_CUDA. */
svdq_status svdq_test_quant_sweep(int which, unsigned long long* dev_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SVDQ_TEST_H_ */
