// Tensor-core rate measurement for the roofline of svdq_gemm_w4a4: every CTA
// (one per SM) issues `iters` tcgen05 MMAs back to back on operands resident
// in shared memory (zeros), accumulating into one TMEM accumulator, and waits
// for completion.  No global memory traffic; the host times the launch.
//
// mode 0: kind::mxf4nvf4 block-scaled NVFP4 (M=128, N=n, K=64, ue4m3 scales)
// mode 1: kind::f16 bf16 (M=128, N=n, K=16)
// mode 2: mode 0 plus the tcgen05.cp of the scale chunks before every MMA
//         (as the GEMM issues them)
// mode 3: kind::mxf4nvf4 on CTA pairs (cta_group::2, M=256 over two SMs,
//         N=n, K=64): clusters of two CTAs, the even one issues
// mode 4: kind::f16 bf16 on CTA pairs (cta_group::2, M=256, N=n, K=16)
// mode 5: mode 0 with consecutive MMAs alternating between two accumulators
//         (n = 128: columns 0 and 128)
// mode 6: mode 3 with the same alternation (n = 128)
// mode 7: the legacy warp-level MMA, mma.sync m16n8k16 f16 with fp32
//         accumulation (n = 128): 8 warps per CTA, each issuing 16
//         independent MMAs per iteration, operands in registers
#include <cstdint>

#include "../../include/svdq_bench.h"
#include "device_common.cuh"

namespace svdq {
namespace {

constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads, 1)
    k_mma_rate(int mode, int n, int iters, int* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // A 128 x 128 B, B n x 128 B (128B swizzle), scales 4 KB, barrier, tmem slot
  uint8_t* A = smem;
  uint8_t* B = smem + 16384;
  uint8_t* SF = B + 32768;
  uint64_t* bar = reinterpret_cast<uint64_t*>(SF + 4096);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(SF + 4096 + 8);
  for (int i = threadIdx.x; i < (16384 + 32768 + 4096) / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (threadIdx.x == 0) {
    const uint32_t a = smem_u32(A), b = smem_u32(B), sf = smem_u32(SF);
    const uint32_t idesc_nvf4 =
        (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const uint32_t idesc_bf16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    const uint32_t sfa = tmem + 256, sfb = tmem + 256 + 4;
    for (int i = 0; i < iters; ++i) {
      const uint32_t koff = (uint32_t)(i & 3) * 32;
      if (mode == 1) {
        tc_mma_bf16(tmem, smem_desc(a + koff, 16, 1024, kSwizzle128B),
                    smem_desc(b + koff, 16, 1024, kSwizzle128B), idesc_bf16, i > 0 ? 1u : 0u);
      } else {
        if (mode == 2) {
          tc_cp_32x128b_warpx4(sfa, smem_desc(sf, 128, 128, kSwizzleNone));
          for (int h = 0; h < n / 128; ++h)
            tc_cp_32x128b_warpx4(sfb + 4 * h, smem_desc(sf + 512 * (h + 1), 128, 128,
                                                        kSwizzleNone));
        }
        const uint32_t d = mode == 5 ? tmem + (uint32_t)(i & 1) * 128u : tmem;
        tc_mma_nvf4(d, smem_desc(a + koff, 16, 1024, kSwizzle128B),
                    smem_desc(b + koff, 16, 1024, kSwizzle128B), idesc_nvf4, sfa, sfb,
                    i > (mode == 5 ? 1 : 0) ? 1u : 0u);
      }
    }
    tc_commit(bar);
    mbar_wait(bar, 0, dev_status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


// modes 3 and 4: clusters of two CTAs; the pair allocates TMEM collectively,
// the even CTA issues M=256 MMAs whose accumulator rows 128-255 live in the
// odd CTA's TMEM and whose B operand is split between the two shared memories
__global__ void __launch_bounds__(kThreads, 1)
    k_mma_rate_pair(int mode, int n, int iters, int* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* A = smem;
  uint8_t* B = smem + 16384;
  uint64_t* bar = reinterpret_cast<uint64_t*>(B + 32768 + 4096);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(B + 32768 + 4096 + 8);
  for (int i = threadIdx.x; i < (16384 + 32768 + 4096) / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  const int warp = threadIdx.x >> 5;
  const uint32_t crank = cluster_ctarank();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  cluster_sync();  // both CTAs resident before the collective allocation
  if (warp == 0) tmem_alloc_pair(tslot, 512);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (crank == 0 && threadIdx.x == 0) {
    const uint32_t a = smem_u32(A), b = smem_u32(B);
    const uint32_t idesc_nvf4 =
        (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
    const uint32_t idesc_bf16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(n >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
    const uint32_t sfa = tmem + 256, sfb = tmem + 256 + 4;
    for (int i = 0; i < iters; ++i) {
      const uint32_t koff = (uint32_t)(i & 3) * 32;
      if (mode == 4)
        tc_mma_bf16_pair(tmem, smem_desc(a + koff, 16, 1024, kSwizzle128B),
                         smem_desc(b + koff, 16, 1024, kSwizzle128B), idesc_bf16,
                         i > 0 ? 1u : 0u);
      else
        tc_mma_nvf4_pair(mode == 6 ? tmem + (uint32_t)(i & 1) * 128u : tmem,
                         smem_desc(a + koff, 16, 1024, kSwizzle128B),
                         smem_desc(b + koff, 16, 1024, kSwizzle128B), idesc_nvf4, sfa, sfb,
                         i > (mode == 6 ? 1 : 0) ? 1u : 0u);
    }
    tc_commit_pair(cluster_map(smem_u32(bar), 0));
    mbar_wait(bar, 0, dev_status);
  }
  tc_fence_before();
  cluster_sync();  // the pair's MMAs are complete before either CTA frees TMEM
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// mode 7: 8 warps x 16 accumulators; 128 m16n8k16 MMAs per CTA and iteration
// (2 * 16 * 8 * 16 * 128 = 2 * 128 * 128 * 16 flops, the formula with n = 128,
// K_mma = 16).  Operands: f16 1.0 (0x3C00) and 2.0 (0x4000).  The accumulators
// feed a store under a condition the compiler cannot decide (iters < 0; the
// host rejects it), so that no MMA is dead code.
__global__ void __launch_bounds__(256, 1) k_mma_rate_warp(int iters, int* dev_status) {
  const uint32_t a0 = 0x3C004000u, a1 = 0x40003C00u, a2 = 0x3C003C00u, a3 = 0x40004000u,
                 b0 = 0x3C003C00u, b1 = 0x40003C00u;
  float d[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int c = 0; c < 4; ++c) d[j][c] = 0.0f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
          "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
          : "+f"(d[j][0]), "+f"(d[j][1]), "+f"(d[j][2]), "+f"(d[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  float s = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) s += d[j][0] + d[j][1] + d[j][2] + d[j][3];
  if (iters < 0 && dev_status) *dev_status = (int)s;
}

}  // namespace
}  // namespace svdq

extern "C" svdq_status svdq_bench_mma_rate(int mode, int n, int iters, int ctas,
                                           int* dev_status, void* stream) {
  if (mode < 0 || mode > 7 || (n != 128 && n != 256) || iters < 1 || ctas < 1)
    return SVDQ_ERR_SHAPE;
  if (mode == 7 && n != 128) return SVDQ_ERR_SHAPE;
  const bool pair = mode == 3 || mode == 4 || mode == 6;
  if (pair && ctas % 2 != 0) return SVDQ_ERR_SHAPE;  // whole CTA pairs
  if (mode >= 5 && n != 128) return SVDQ_ERR_SHAPE;  // two accumulators of 128 columns
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return SVDQ_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return SVDQ_ERR_UNSUPPORTED_ARCH;
  if (mode == 7) {
    svdq::k_mma_rate_warp<<<ctas, 256, 0, static_cast<cudaStream_t>(stream)>>>(iters,
                                                                              dev_status);
    return cudaGetLastError() == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
  }
  const int smem = 16384 + 32768 + 4096 + 64 + 1024;
  if (pair) {
    if (cudaFuncSetAttribute(svdq::k_mma_rate_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return SVDQ_ERR_CUDA;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(svdq::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, svdq::k_mma_rate_pair, mode, n, iters, dev_status) !=
        cudaSuccess)
      return SVDQ_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
  }
  if (cudaFuncSetAttribute(svdq::k_mma_rate, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return SVDQ_ERR_CUDA;
  svdq::k_mma_rate<<<ctas, svdq::kThreads, smem, static_cast<cudaStream_t>(stream)>>>(
      mode, n, iters, dev_status);
  return cudaGetLastError() == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
}
