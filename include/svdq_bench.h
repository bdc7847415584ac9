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
 *   mode 3: mode 0 on CTA pairs (tcgen05 cta_group::2: clusters of two CTAs,
 *           one M = 256 MMA over the two SMs, issued by the even CTA)
 *   mode 4: mode 1 on CTA pairs (cta_group::2, M = 256)
 *   mode 5: mode 0 with consecutive MMAs alternating between two
 *           accumulators (n = 128 only)
 *   mode 6: mode 3 with the same alternation (n = 128 only)
 *   mode 7: the legacy warp-level MMA (mma.sync m16n8k16, f16 inputs, fp32
 *           accumulate; operands in registers, 8 warps per CTA, 16
 *           independent accumulators per warp), K_mma = 16, n = 128 only:
 *           128 such MMAs per CTA and iteration
 * For modes 3, 4 and 6 the work is 2 * 256 * n * K_mma * iters * ctas / 2
 * flops, the same total as the formula above.
 *
 * n in {128, 256}; iters >= 1; ctas >= 1 (even for modes 3, 4 and 6).  dev_status (nullable device int)
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
