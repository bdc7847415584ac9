/*
 * svdq_bench.h -- measurement entry point of libsvdq (not part of the layer).
 *
 * The roofline of svdq_gemm_w4a4 needs the tensor cores' own NVFP4 rate on
 * the device at hand.  svdq_bench_mma_rate launches `ctas` CTAs (one per SM
 * when ctas = number of SMs); each issues `iters` tcgen05 MMAs (M = 128,
 * N = n) back to back on operands resident in shared memory, accumulating in
 * tensor memory, then waits for them.  There is no global-memory traffic; the
 * caller times the launch (CUDA events on `stream`) and divides the work,
 * 2 * 128 * n * K_mma * iters * ctas flops, by the time.
 *
 *   mode 0: kind::mxf4nvf4 block-scaled NVFP4, K_mma = 64
 *   mode 1: kind::f16 (bf16 inputs, fp32 accumulate), K_mma = 16
 *   mode 2: mode 0 plus the tcgen05.cp copies of the block-scale chunks
 *           (1 + n/128 of them) before every MMA, as the GEMM issues them
 *
 * n in {128, 256}; iters >= 1; ctas >= 1.  dev_status (nullable device int)
 * receives SVDQ_DEV_TIMEOUT if the completion wait exceeds its bound.
 * Errors: SVDQ_ERR_SHAPE, SVDQ_ERR_UNSUPPORTED_ARCH, SVDQ_ERR_CUDA.
 * The pages have no counterpart: this is instrumentation for the roofline.
 */
#ifndef SVDQ_BENCH_H_
#define SVDQ_BENCH_H_

#include "svdq.h"

#ifdef __cplusplus
extern "C" {
#endif

svdq_status svdq_bench_mma_rate(int mode, int n, int iters, int ctas, int* dev_status,
                                void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SVDQ_BENCH_H_ */
