// Internal launchers of libsvdq's kernels (called by the C ABI in capi.cu
// after argument validation).  All launches are asynchronous on `stream`.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace svdq {

// tm_x: X [M][K] bf16, box 64 x 32 rows, 128B swizzle; tm_l1s: L1s [rank][K]
// bf16, box 64 x rank rows, 128B swizzle (both built on the host per call)
cudaError_t launch_quantize_act(const CUtensorMap& tm_x, const CUtensorMap& tm_l1s,
                                const float* inv_lambda, int M, int K, int rank,
                                uint8_t* a_codes, uint8_t* a_scales, uint16_t* lora_act,
                                int* dev_status, cudaStream_t stream, bool int4);

// INT4 variant's GEMM (gemm_int4.cu): grid N/128 x ceil(M/128)
cudaError_t launch_gemm_int4(const uint8_t* a_codes, const uint16_t* a_scales,
                             const uint8_t* w_codes, const uint16_t* w_scales,
                             const uint16_t* lora_act, const uint16_t* L2, const uint16_t* bias,
                             uint16_t* Y, int M, int N, int K, int rank, int* dev_status,
                             cudaStream_t stream);

// Tensor maps of svdq_gemm_w4a4 (and of its GELU and QKV variants).  The
// kernel runs on CTA pairs: each CTA loads its own 128 A rows and one half
// (BN/2 rows) of the tile's W and L2s rows.
struct GemmMaps {
  CUtensorMap a_codes;  // [M][K/2] bytes: box 128 x 128 rows, 128B swizzle
  CUtensorMap w_codes;  // [N][K/2] bytes: box 128 x BN/2 rows (one CTA's half), 128B swizzle
  CUtensorMap lora;     // lora_act [M][rank] bf16: box rank x 128 rows, swizzle = 2*rank bytes
  CUtensorMap l2s;      // L2s [N][rank] bf16: box rank x BN/2 rows, same swizzle
  CUtensorMap y;        // Y [M][N] bf16: box BN/4 x 32 rows, swizzle = BN/2 bytes (stores)
  CUtensorMap l1s2;     // GELU + quantization only: the next layer's L1s [rank2][N] bf16,
                        // box 64 x rank2/2 rows, 128B swizzle
};

// What svdq_gemm_w4a4's epilogue does after y = s_T * acc + bias is rounded to
// bf16: nothing; GELU (tanh form); per-head RMS normalization and rotary
// embedding of the Q and K column blocks (fused QKV projection, block_n 256);
// GELU, then the next layer's activation quantization of the result (block_n
// 256).
enum class GemmEpilogue { kPlain, kGelu, kQkv, kGeluQuant };

// Operands of the GELU + quantization epilogue (all null for the others): the
// GELU output H [M][N] is quantized as the next linear's input X2 (K2 = N).
struct GeluQuantEpilogue {
  const float* inv_lambda2;  // [N] the next layer's smoothing
  uint8_t* a2_codes;         // [M][N/2] e2m1 codes of H
  uint8_t* a2_scales;        // scale tiles of H (rows M, K2 = N)
  float* partial;            // scratch: [128 + ceil(M/256)][256][rank2] segment sums
  uint16_t* h_out;           // [M][N] bf16 H, or null (H is not written)
  uint16_t* lora2;           // [M][rank2] bf16 down projection (a second kernel adds the
                             // segment sums)
  int rank2;                 // 32 or 64
  size_t scratch_bytes;      // bytes at `partial`
};

// Operands of the QKV epilogue (all null / zero for the others).
struct QkvEpilogue {
  const uint16_t* norm_q;  // [128] bf16 weights of the Q normalization
  const uint16_t* norm_k;  // [128] bf16 weights of the K normalization
  const float* rope_cos;   // [M][64] fp32, per token and channel pair
  const float* rope_sin;   // [M][64] fp32
  float eps;               // added to the mean square
  int hd;                  // columns of each of Q, K, V: N / 3 (a multiple of 256)
};

cudaError_t launch_gemm_w4a4(const GemmMaps& maps, int block_n, const uint8_t* a_scales,
                             const uint8_t* w_scales, float w_tensor_scale, const uint16_t* bias,
                             uint16_t* Y, int M, int N, int K, int rank, GemmEpilogue epi,
                             const QkvEpilogue& qe, const GeluQuantEpilogue& gq,
                             int* dev_status, int test_stall, int num_sms, cudaStream_t stream);

// Largest K the AWQ GEMV stages in shared memory.
int awq_max_k();

// qweight [N][K/2] bytes (16-byte aligned).
cudaError_t launch_awq_gemv(const uint8_t* qweight, const uint16_t* X, const uint16_t* scales,
                            const uint16_t* zeros, const uint16_t* bias, uint16_t* Y, int M,
                            int N, int K, int* dev_status, cudaStream_t stream, int num_sms);

}  // namespace svdq
