// awq_gemv_w4a16: 4-bit weights x bf16 activations for the small-M
// modulation layers (dothoosh.com, "How Nunchaku Lite halves the VRAM of
// diffusion models", kernel-family list: awq_w4a16 serves the memory-bound
// adaLN modulation projections; config block: int4, group_size 64).
//
//   Y[m][n] = bf16( sum_g s[n][g] * ( sum_{k in g} q[n][k] x[m][k]
//                                     - z[n][g] * sum_{k in g} x[m][k] ) + bias[n] )
//
// which equals sum_k x (q - z) s.  The inner sums run on tensor cores
// (m16n8k16, bf16 in, fp32 out) with the codes q as exact bf16 integers: the
// 16 weight rows of a warp tile are the MMA's M, the (up to 8) activation rows
// its N.  Per 64-group the fp32 partial sums get the scale and zero point;
// sum_{k in g} x[m][k] is computed once per CTA.  The weights stream from HBM
// exactly once (128-bit-sector-aligned 8-byte loads, prefetched one step
// ahead); X is staged in shared memory in the k order the MMA fragments use.
//
// Code -> bf16: OR-ing a nibble into the mantissa of 128.0 (0x4300) gives the
// bf16 value 128 + q exactly; subtracting 128 (bf16x2) leaves q exactly.
#include <cstdint>
#include <cuda_bf16.h>

#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

// nibbles at bit s and s+16 of w -> bf16x2 {q_lo, q_hi}
SVDQ_DEVINL uint32_t nib2_to_bf16x2(uint32_t w, int s) {
  const uint32_t v = ((w >> s) & 0x000F000Fu) | 0x43004300u;  // {128+q, 128+q'}
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                                   __floats2bfloat162_rn(128.0f, 128.0f));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// k (within a thread's 16) of the two elements of fragment pair p (0..7):
// word p/4, nibbles p%4 and p%4+4
SVDQ_DEVINL int pair_k(int p, int hi) { return 8 * (p >> 2) + (p & 3) + 4 * hi; }

struct Step {     // one 2-group (128-k) step of one thread: rows r8 and r8+8
  uint2 c[2][2];  // [row][group] 8 bytes of codes (16 nibbles)
  uint32_t s[2], z[2];  // [row] fp16 pairs: groups g, g+1
};

SVDQ_DEVINL void load_step(Step& st, const uint8_t* __restrict__ qw, const uint16_t* __restrict__ sc,
                           const uint16_t* __restrict__ zr, const int (&row)[2], const bool (&ok)[2],
                           int step, int K, int G, int t) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (ok[i]) {
      const uint8_t* p = qw + (size_t)row[i] * (K >> 1) + step * 64 + 8 * t;
      st.c[i][0] = *reinterpret_cast<const uint2*>(p);
      st.c[i][1] = *reinterpret_cast<const uint2*>(p + 32);
      st.s[i] = *reinterpret_cast<const uint32_t*>(sc + (size_t)row[i] * G + 2 * step);
      st.z[i] = *reinterpret_cast<const uint32_t*>(zr + (size_t)row[i] * G + 2 * step);
    } else {
      st.c[i][0] = st.c[i][1] = make_uint2(0, 0);
      st.s[i] = st.z[i] = 0u;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    k_awq_gemv(const uint16_t* __restrict__ X, const uint8_t* __restrict__ qw,
               const uint16_t* __restrict__ sc, const uint16_t* __restrict__ zr,
               const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K) {
  extern __shared__ uint32_t xs[];  // [G][32 lanes][8 words] then sx [G][8]
  const int G = K >> 6;
  float* sx = reinterpret_cast<float*>(xs + (size_t)G * 256);

  // ---- stage X in fragment order: word (g, lane, p) = {x[r8][k_lo], x[r8][k_hi]}
  for (int idx = threadIdx.x; idx < G * 256; idx += kThreads) {
    const int g = idx >> 8, ln = (idx >> 3) & 31, p = idx & 7;
    const int m = ln >> 2, t = ln & 3;
    uint32_t w = 0;
    if (m < M) {
      const uint16_t* xr = X + (size_t)m * K + g * 64 + 16 * t;
      w = (uint32_t)xr[pair_k(p, 0)] | ((uint32_t)xr[pair_k(p, 1)] << 16);
    }
    xs[idx] = w;
  }
  for (int idx = threadIdx.x; idx < G * 8; idx += kThreads) {
    const int g = idx >> 3, m = idx & 7;
    float s = 0.0f;
    if (m < M) {
      const uint16_t* xr = X + (size_t)m * K + g * 64;
      for (int k = 0; k < 64; ++k) s += __uint_as_float((uint32_t)xr[k] << 16);
    }
    sx[idx] = s;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r8 = lane >> 2, t = lane & 3;
  const int steps = K >> 7;  // 2-group steps
  const int tiles = (N + 15) >> 4;
  for (int tile = blockIdx.x * kWarps + warp; tile < tiles; tile += gridDim.x * kWarps) {
    const int n0 = tile * 16;
    const int row[2] = {n0 + r8, n0 + r8 + 8};
    const bool ok[2] = {row[0] < N, row[1] < N};
    float y[4] = {0.f, 0.f, 0.f, 0.f};  // (row r8, m 2t), (r8, 2t+1), (r8+8, 2t), (r8+8, 2t+1)
    Step cur, nxt;
    load_step(cur, qw, sc, zr, row, ok, 0, K, G, t);
    for (int st = 0; st < steps; ++st) {
      if (st + 1 < steps) load_step(nxt, qw, sc, zr, row, ok, st + 1, K, G, t);
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int g = 2 * st + gg;
        const uint4* xf = reinterpret_cast<const uint4*>(xs + ((size_t)g * 32 + lane) * 8);
        const uint4 xb0 = xf[0], xb1 = xf[1];
        const uint32_t b[8] = {xb0.x, xb0.y, xb0.z, xb0.w, xb1.x, xb1.y, xb1.z, xb1.w};
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        const uint2 ca = cur.c[0][gg], cb = cur.c[1][gg];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // pairs p = 2j, 2j+1 -> word (2j)/4, nibble shifts 4*(p%4)
          const int p0 = 2 * j, p1 = 2 * j + 1;
          const uint32_t wa0 = (p0 >> 2) ? ca.y : ca.x, wa1 = (p1 >> 2) ? ca.y : ca.x;
          const uint32_t wb0 = (p0 >> 2) ? cb.y : cb.x, wb1 = (p1 >> 2) ? cb.y : cb.x;
          mma_bf16_16816(d, nib2_to_bf16x2(wa0, 4 * (p0 & 3)), nib2_to_bf16x2(wb0, 4 * (p0 & 3)),
                         nib2_to_bf16x2(wa1, 4 * (p1 & 3)), nib2_to_bf16x2(wb1, 4 * (p1 & 3)),
                         b[p0], b[p1]);
        }
        // scale / zero point of rows r8, r8+8 for group g
        const float s0 = __half2float(__ushort_as_half((uint16_t)(cur.s[0] >> (16 * gg))));
        const float z0 = __half2float(__ushort_as_half((uint16_t)(cur.z[0] >> (16 * gg))));
        const float s1 = __half2float(__ushort_as_half((uint16_t)(cur.s[1] >> (16 * gg))));
        const float z1 = __half2float(__ushort_as_half((uint16_t)(cur.z[1] >> (16 * gg))));
        const float sxa = sx[g * 8 + 2 * t], sxb = sx[g * 8 + 2 * t + 1];
        y[0] = __fmaf_rn(s0, __fmaf_rn(-z0, sxa, d[0]), y[0]);
        y[1] = __fmaf_rn(s0, __fmaf_rn(-z0, sxb, d[1]), y[1]);
        y[2] = __fmaf_rn(s1, __fmaf_rn(-z1, sxa, d[2]), y[2]);
        y[3] = __fmaf_rn(s1, __fmaf_rn(-z1, sxb, d[3]), y[3]);
      }
      cur = nxt;
    }
    // ---- bias, round, store Y[m][n]
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (!ok[i]) continue;
      const float bv = bias ? __uint_as_float((uint32_t)bias[row[i]] << 16) : 0.0f;
      const int m0 = 2 * t;
      if (m0 < M) Y[(size_t)m0 * N + row[i]] = f32_to_bf16_rn(y[2 * i] + bv);
      if (m0 + 1 < M) Y[(size_t)(m0 + 1) * N + row[i]] = f32_to_bf16_rn(y[2 * i + 1] + bv);
    }
  }
}

}  // namespace

cudaError_t launch_awq_gemv(const uint16_t* X, const uint8_t* qweight, const uint16_t* scales,
                            const uint16_t* zeros, const uint16_t* bias, uint16_t* Y, int M,
                            int N, int K, cudaStream_t stream, int num_sms) {
  const int G = K >> 6;
  const size_t smem = (size_t)G * 256 * sizeof(uint32_t) + (size_t)G * 8 * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_awq_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int tiles = (N + 15) / 16;
  int grid = 2 * num_sms;
  if (grid * kWarps > tiles) grid = (tiles + kWarps - 1) / kWarps;
  k_awq_gemv<<<grid, kThreads, smem, stream>>>(X, qweight, scales, zeros, bias, Y, M, N, K);
  return cudaGetLastError();
}

}  // namespace svdq
