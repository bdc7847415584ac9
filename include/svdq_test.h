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

#ifdef __cplusplus
}
#endif

#endif /* SVDQ_TEST_H_ */
