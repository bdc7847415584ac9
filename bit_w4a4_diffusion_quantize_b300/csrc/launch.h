// Internal launchers of libsvdq's kernels (called by the C ABI in capi.cu
// after argument validation).  All launches are asynchronous on `stream`.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace svdq {

cudaError_t launch_quantize_act(const uint16_t* X, const float* inv_lambda, const uint16_t* L1s,
                                int M, int K, int rank, uint8_t* a_codes, uint8_t* a_scales,
                                uint16_t* lora_act, int* dev_status, cudaStream_t stream,
                                int num_sms);

// Tensor maps of the packed 4-bit codes (built by the caller on the host).
struct GemmMaps {
  CUtensorMap a_codes;  // [M][K/2] bytes, box 128 x 128 rows, 128B swizzle
  CUtensorMap w_codes;  // [N][K/2] bytes, box 128 x BN rows, 128B swizzle
};

cudaError_t launch_gemm_w4a4(const GemmMaps& maps, int block_n, const uint8_t* a_scales,
                             const uint8_t* w_scales, float w_tensor_scale,
                             const uint16_t* lora_act, const uint16_t* L2,
                             const uint16_t* bias, uint16_t* Y, int M, int N, int K, int rank,
                             int* dev_status, int test_stall, cudaStream_t stream);

cudaError_t launch_awq_gemv(const uint16_t* X, const uint8_t* qweight, const uint16_t* scales,
                            const uint16_t* zeros, const uint16_t* bias, uint16_t* Y, int M,
                            int N, int K, cudaStream_t stream, int num_sms);

}  // namespace svdq
