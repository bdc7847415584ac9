// Exhaustive checks of the activation quantization's division-free rounding
// (act_quant.cuh, shared by svdq_quantize_act and the GEMM's GELU +
// quantization epilogue) against IEEE division followed by the same
// round-to-nearest-even conversion.
//
// For a divisor d with few significant bits (6, or an e4m3 scale s) and a
// 24-bit x, the correctly rounded fp32 quotient fl32(x/d) lands on an e2m1 or
// e4m3 rounding midpoint only if x/d is that midpoint exactly (x != m d
// differs from m d by at least one ulp of x, i.e. by more than half an fp32
// ulp of the quotient), so RNE(fl32(x/d)) is the exact rounding of x/d --
// what the oracle computes in rational arithmetic.  The kernels here run the
// library's own routine (quant_block16) on blocks whose inputs are chosen so
// that one element or the block amax takes every value of a range, and count
// where it disagrees with RNE(fl32(x/d)).
#include <cstdint>

#include "../../include/svdq_test.h"
#include "act_quant.cuh"
#include "device_common.cuh"

namespace svdq {

namespace {

constexpr uint32_t kOneBf16x2 = 0x3F803F80u;  // bf16 {1.0, 1.0}: x_hat = inv exactly

SVDQ_DEVINL void build_table(float2* tab) {
  for (int c = threadIdx.x; c < 128; c += blockDim.x)
    tab[c] = c == 0 || c == 127 ? make_float2(0.0f, 0.0f) : recip2(e4m3_to_f32(c));
}

SVDQ_DEVINL void report(unsigned long long* out, uint32_t pattern) {
  atomicAdd(&out[0], 1ull);
  atomicMin(&out[1], (unsigned long long)pattern);
}

// every finite non-negative fp32 value as a block amax: its scale byte
__global__ void __launch_bounds__(256) k_sweep_scales(unsigned long long* out) {
  __shared__ float2 tab[128];
  build_table(tab);
  __syncthreads();
  const float2 r6 = recip2(6.0f);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = kOneBf16x2;
  const uint32_t stride = gridDim.x * blockDim.x;
  unsigned long long checked = 0;
  for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < 0x7F800000u; u += stride) {
    float inv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) inv[i] = 0.0f;
    inv[0] = __uint_as_float(u);
    uint2 codes;
    uint32_t sb;
    quant_block16(w, inv, r6, tab, codes, sb);
    const uint32_t ref = f32_to_e4m3_sat(__fdiv_rn(__uint_as_float(u), 6.0f));
    if (sb != ref) report(out, u);
    ++checked;
  }
  atomicAdd(&out[2], checked);
}

// every positive finite e4m3 scale s (blockIdx.y + 1): a block whose amax is
// 6 s (so its scale is s), and in its other elements every fp32 value of
// magnitude in [6 s 2^-8, 6 s), with both signs: their codes
__global__ void __launch_bounds__(256) k_sweep_codes(unsigned long long* out) {
  __shared__ float2 tab[128];
  build_table(tab);
  __syncthreads();
  const float2 r6 = recip2(6.0f);
  const uint32_t sc = blockIdx.y + 1;  // 1 .. 126
  const float s = e4m3_to_f32(sc);
  const float amax = 6.0f * s;  // exact: s has at most 4 significant bits
  const uint32_t hi = __float_as_uint(amax);
  const uint32_t lo = hi - (8u << 23);  // 8 binades below
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = kOneBf16x2;
  const uint32_t stride = gridDim.x * blockDim.x * 7u;
  unsigned long long checked = 0;
  for (uint32_t u0 = lo + 7u * (blockIdx.x * blockDim.x + threadIdx.x); u0 < hi; u0 += stride) {
    // element 0: amax; elements 1..7: u0 .. u0 + 6; 8..14: their negatives; 15: 0
    float inv[16];
    inv[0] = amax;
#pragma unroll
    for (int i = 0; i < 7; ++i) {
      const uint32_t u = min(u0 + (uint32_t)i, hi - 1u);
      inv[1 + i] = __uint_as_float(u);
      inv[8 + i] = -__uint_as_float(u);
    }
    inv[15] = 0.0f;
    uint2 codes;
    uint32_t sb;
    quant_block16(w, inv, r6, tab, codes, sb);
    float q[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) q[i] = __fdiv_rn(inv[i], s);
    const uint32_t rx = f32x8_to_e2m1x8(q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]);
    const uint32_t ry = f32x8_to_e2m1x8(q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]);
    if (sb != sc || codes.x != rx || codes.y != ry) report(out, u0);
    ++checked;
  }
  atomicAdd(&out[2], checked);
}

}  // namespace

}  // namespace svdq

extern "C" svdq_status svdq_test_quant_sweep(int which, unsigned long long* dev_out,
                                             void* stream) {
  if (which != 0 && which != 1) return SVDQ_ERR_VALUE;
  if (!dev_out) return SVDQ_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(dev_out) & 15u) != 0) return SVDQ_ERR_ALIGN;
  int dev = 0, ma = 0, mi = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return SVDQ_ERR_CUDA;
  }
  if (ma != 10 || mi != 3) return SVDQ_ERR_UNSUPPORTED_ARCH;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (which == 0)
    svdq::k_sweep_scales<<<4096, 256, 0, st>>>(dev_out);
  else
    svdq::k_sweep_codes<<<dim3(256, 126), 256, 0, st>>>(dev_out);
  return cudaGetLastError() == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
}
