// svdq_quantize_act: the activation side of the SVDQ W4A4 linear in one pass
// over X (dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion
// models", fused-kernel paragraph: the low-rank down projection is fused with
// the quantization kernel).
//
//   lora_act[m][i] = bf16( sum_k X[m][k] L1s[i][k] )      tensor cores, fp32 acc
//   x_hat          = fl32( X[m][k] * inv_lambda[k] )
//   scale byte     = RNE_e4m3( amax16(x_hat) / 6 )        IEEE fp32 division
//   code nibble    = RNE_e2m1( x_hat / s )                exact quotient rounding
//
// Work split.  A CTA owns 16*MT consecutive rows (MT m16 tiles) and all of K;
// its 8 warps split K into contiguous ranges of 64-wide steps.  In one step a
// thread (quad lane t, group g) holds 16 consecutive k of rows g, g+8 (+16,
// +24): exactly one 16-element quantization block per row, read with 128-bit
// loads.  The same registers are the A fragments of the m16n8k16 MMAs of the
// down projection; the k order inside an MMA is permuted, and the B fragments
// (L1s rows, k contiguous) are read with the same permutation, so no data is
// moved between lanes.  Partial lora sums of the 8 warps are added in a fixed
// order through shared memory, then rounded once to bf16.
//
// Quotient x_hat / s.  s is an e4m3 value (4 significant bits).  With
// r_hi = RD(1/s) and r_lo = RN((1 - r_hi s) / s) (the residual 1 - r_hi s is
// exact through one fma), y = RN(x r_hi + RN(x r_lo)) differs from the exact
// quotient by less than 2^-46 of it.  The exact quotient is either an e2m1
// midpoint m itself or more than 0.53 ulp(m) away from it (x_hat has 24
// significant bits, m*s at most 7), so y rounds to the same e2m1 code as the
// exact quotient.  r_hi rounds down so that r_lo >= 0 and y keeps the sign of
// x_hat even for -0.  Blocks whose amax is infinite take IEEE division.
#include <cstdint>

#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// quantize one 16-element block held by one thread (8 bf16x2 words)
SVDQ_DEVINL void quant_block16(const uint32_t (&w)[8], const float (&inv)[16], uint2& codes,
                               uint32_t& sbyte) {
  float xh[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    xh[2 * i] = __fmul_rn(bf16lo_to_f32(w[i]), inv[2 * i]);
    xh[2 * i + 1] = __fmul_rn(bf16hi_to_f32(w[i]), inv[2 * i + 1]);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(xh[i]));
  sbyte = f32_to_e4m3_sat(__fdiv_rn(amax, 6.0f));
  const float s = e4m3_to_f32(sbyte);
  float y[16];
  if (s == 0.0f) {
    codes = make_uint2(0u, 0u);
    return;
  }
  if (!(amax <= 3.402823466e38f)) {  // infinite block: plain IEEE division
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __fdiv_rn(xh[i], s);
  } else {
    const float r_hi = __frcp_rd(s);
    const float r_lo = __fdiv_rn(__fmaf_rn(-r_hi, s, 1.0f), s);
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = __fmaf_rn(xh[i], r_hi, __fmul_rn(xh[i], r_lo));
  }
  codes.x = f32x8_to_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
  codes.y = f32x8_to_e2m1x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
}

SVDQ_DEVINL void unpack8(const uint4& a, const uint4& b, uint32_t (&w)[8]) {
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

template <int RANK, int MT>
__global__ void __launch_bounds__(kThreads, 1)
    k_quantize_act(const uint16_t* __restrict__ X, const float* __restrict__ inv_lambda,
                   const uint16_t* __restrict__ L1s, int M, int K,
                   uint8_t* __restrict__ a_codes, uint8_t* __restrict__ a_scales,
                   uint16_t* __restrict__ lora_act) {
  constexpr int NT = RANK / 8;        // n8 tiles of the down projection
  constexpr int ROWS = 16 * MT;       // rows of this CTA
  constexpr int NR = 2 * MT;          // rows per thread: g, g+8, g+16, g+24
  extern __shared__ float red[];      // [kWarps][ROWS][RANK]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int m0 = blockIdx.x * ROWS;
  const int steps = K >> 6;
  const int s_begin = (warp * steps) / kWarps, s_end = ((warp + 1) * steps) / kWarps;
  const size_t rowpitch = (size_t)K;   // bf16 elements
  const int C4 = K >> 6;               // 4-column scale groups per row

  int rows[NR];
  bool ok[NR];
#pragma unroll
  for (int j = 0; j < NR; ++j) {
    rows[j] = m0 + g + 8 * j;
    ok[j] = rows[j] < M;
  }

  float acc[MT][NT][4];
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][n][c] = 0.0f;

  for (int st = s_begin; st < s_end; ++st) {
    const int k0 = st * 64 + 16 * t;
    // ---- loads: X (read once), inv_lambda and L1s (shared by all CTAs)
    uint32_t xw[NR][8];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (ok[j]) {
        const uint16_t* p = X + (size_t)rows[j] * rowpitch + k0;
        lo = ld_stream_v4(p);
        hi = ld_stream_v4(p + 8);
      }
      unpack8(lo, hi, xw[j]);
    }
    float inv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = ld_keep_f4(inv_lambda + k0 + 4 * q);
      inv[4 * q] = v.x; inv[4 * q + 1] = v.y; inv[4 * q + 2] = v.z; inv[4 * q + 3] = v.w;
    }
    uint32_t bw[NT][8];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const uint16_t* p = L1s + (size_t)(g + 8 * n) * K + k0;
      unpack8(ld_keep_v4(p), ld_keep_v4(p + 8), bw[n]);
    }
    // ---- down projection: 4 k16 sub-steps x NT n-tiles x MT m-tiles
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4)
#pragma unroll
      for (int a = 0; a < MT; ++a)
#pragma unroll
        for (int n = 0; n < NT; ++n)
          mma_bf16_16816(acc[a][n], xw[2 * a][2 * j4], xw[2 * a + 1][2 * j4],
                         xw[2 * a][2 * j4 + 1], xw[2 * a + 1][2 * j4 + 1], bw[n][2 * j4],
                         bw[n][2 * j4 + 1]);
    // ---- quantization: one block per row
    uint32_t sw[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      uint2 codes;
      uint32_t sb;
      quant_block16(xw[j], inv, codes, sb);
      if (ok[j])
        *reinterpret_cast<uint2*>(a_codes + (size_t)rows[j] * (K >> 1) + (k0 >> 1)) = codes;
      // gather the 4 scale bytes of this row's 64-wide step across the quad
      uint32_t word = sb << (8 * t);
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 1);
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 2);
      sw[j] = word;
    }
    // lane t of the quad writes the scale word of row j == t (tile layout:
    // tile (r/128, c/4) of 512 bytes; entry (r%32)*16 + ((r/32)%4)*4 + c%4)
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      if (j == t && ok[j]) {
        const int r = rows[j];
        const size_t off = ((size_t)(r >> 7) * C4 + st) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
        *reinterpret_cast<uint32_t*>(a_scales + off) = sw[j];
      }
    }
  }

  // ---- reduce the warps' partial lora sums in a fixed order, round once
#pragma unroll
  for (int a = 0; a < MT; ++a)
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int col = 8 * n + 2 * t;
      float* base = red + ((size_t)warp * ROWS + 16 * a + g) * RANK + col;
      base[0] = acc[a][n][0];
      base[1] = acc[a][n][1];
      base[8 * RANK] = acc[a][n][2];
      base[8 * RANK + 1] = acc[a][n][3];
    }
  __syncthreads();
  for (int idx = threadIdx.x; idx < ROWS * RANK; idx += kThreads) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[(size_t)w * ROWS * RANK + idx];
    const int r = m0 + idx / RANK;
    if (r < M) lora_act[(size_t)m0 * RANK + idx] = f32_to_bf16_rn(s);
  }
}

template <int RANK, int MT>
cudaError_t launch_t(const uint16_t* X, const float* inv_lambda, const uint16_t* L1s, int M,
                     int K, uint8_t* a_codes, uint8_t* a_scales, uint16_t* lora_act,
                     cudaStream_t stream) {
  constexpr int ROWS = 16 * MT;
  const size_t smem = (size_t)kWarps * ROWS * RANK * sizeof(float);
  auto kern = k_quantize_act<RANK, MT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int grid = (M + ROWS - 1) / ROWS;
  kern<<<grid, kThreads, smem, stream>>>(X, inv_lambda, L1s, M, K, a_codes, a_scales, lora_act);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_act(const uint16_t* X, const float* inv_lambda, const uint16_t* L1s,
                                int M, int K, int rank, uint8_t* a_codes, uint8_t* a_scales,
                                uint16_t* lora_act, int* /*dev_status*/, cudaStream_t stream,
                                int num_sms) {
  // two m16 tiles per warp halve the L1s traffic when there are enough rows
  // to keep every SM busy; otherwise one tile per warp
  const bool wide = (M + 31) / 32 >= num_sms;
  switch (rank) {
    case 16:
      return wide ? launch_t<16, 2>(X, inv_lambda, L1s, M, K, a_codes, a_scales, lora_act, stream)
                  : launch_t<16, 1>(X, inv_lambda, L1s, M, K, a_codes, a_scales, lora_act, stream);
    case 32:
      return wide ? launch_t<32, 2>(X, inv_lambda, L1s, M, K, a_codes, a_scales, lora_act, stream)
                  : launch_t<32, 1>(X, inv_lambda, L1s, M, K, a_codes, a_scales, lora_act, stream);
    case 64:
      return wide ? launch_t<64, 2>(X, inv_lambda, L1s, M, K, a_codes, a_scales, lora_act, stream)
                  : launch_t<64, 1>(X, inv_lambda, L1s, M, K, a_codes, a_scales, lora_act, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace svdq
