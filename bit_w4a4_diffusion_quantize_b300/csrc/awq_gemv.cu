// awq_gemv_w4a16: 4-bit weights x bf16 activations for the small-M
// modulation layers (dothoosh.com, "How Nunchaku Lite halves the VRAM of
// diffusion models", kernel-family list: awq_w4a16 serves the memory-bound
// adaLN modulation projections; config block: int4, group_size 64).
//
//   Y[m][n] = bf16( sum_g s[n][g] * ( sum_{k in g} q[n][k] x[m][k]
//                                     - z[n][g] * sum_{k in g} x[m][k] ) + bias[n] )
//
// which equals sum_k x (q - z) s.  The inner sums run on tensor cores
// (m16n8k16, bf16 in, fp32 out) with the codes q as exact bf16 integers.  The
// activations (M <= 8 rows, zero-padded to the MMA's 16) are the A operand
// and stay in registers for the whole kernel: each warp owns a fixed range of
// K groups; the weights are the B operand, 8 output channels per MMA.  Per
// 64-group the fp32 partial sums get the scale and zero point;
// sum_{k in g} x[m][k] is formed once per warp.
//
// Streaming.  The weights are read exactly once.  A persistent CTA walks its
// 16-row tiles; one thread streams each tile (16 x K/2 bytes of codes as
// 128-byte-wide TMA boxes with the 128-byte swizzle, plus the tile's fp16
// scales and zeros as plain bulk copies) into a shared-memory ring of up to
// 6 tiles.  The 8 warps split each tile's K groups; their fp32 partials are
// added in a fixed order through shared memory.
//
// The k order inside an MMA is permuted: a thread feeds 16 consecutive k of a
// group, paired as (k, k+4) within each 8, the pairing in which two nibbles
// of a 32-bit code word become one bf16x2 register: OR-ing a nibble into the
// mantissa of 128.0 (0x4300) gives the bf16 value 128 + q exactly, and
// subtracting 128 leaves q exactly.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxStages = 6;
constexpr int kGpw = 8;  // K groups per warp at most (K <= 8 * 8 * 64 = 4096)
constexpr int kSmemBudget = 224 * 1024;

// nibbles at bit s and s+16 of w -> bf16x2 {q_lo, q_hi}
SVDQ_DEVINL uint32_t nib2_to_bf16x2(uint32_t w, int s) {
  const uint32_t v = ((w >> s) & 0x000F000Fu) | 0x43004300u;  // {128+q, 128+q'}
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&v),
                                   __floats2bfloat162_rn(128.0f, 128.0f));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// bf16 element e (0..15) of the 8 words w
SVDQ_DEVINL uint32_t elem(const uint32_t (&w)[8], int e) {
  return (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
}

struct AwqLayout {
  int G, boxes, code_bytes, sz_bytes, stage_bytes, stages, off_red, off_bar, smem;
};

__host__ __device__ inline AwqLayout awq_layout(int K) {
  AwqLayout L;
  L.G = K / 64;
  L.boxes = (K / 2 + 127) / 128;       // 128-byte boxes per row
  L.code_bytes = L.boxes * 16 * 128;   // 16 rows per tile
  L.sz_bytes = 16 * L.G * 2;           // fp16 scales (and as much for zeros)
  L.stage_bytes = (L.code_bytes + 2 * L.sz_bytes + 1023) / 1024 * 1024;
  const int red = 2 * kWarps * 16 * 8 * 4;
  int st = (kSmemBudget - red - 128 - 1024) / L.stage_bytes;
  L.stages = st > kMaxStages ? kMaxStages : st;
  L.off_red = L.stages * L.stage_bytes;
  L.off_bar = L.off_red + red;
  L.smem = L.off_bar + 128 + 1024;
  return L;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_awq_gemv(const __grid_constant__ CUtensorMap tm_q, const uint16_t* __restrict__ X,
               const uint16_t* __restrict__ sc, const uint16_t* __restrict__ zr,
               const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K,
               int* dev_status, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const AwqLayout L = awq_layout(K);
  const int G = L.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, t = lane & 3;  // MMA row (activation m / weight row), quad lane
  float* red = reinterpret_cast<float*>(smem + L.off_red);  // [2][warps][16 rows][8 m]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(smem + L.off_bar + 120);

  const int tiles = (N + 15) >> 4;
  const int my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int stages = L.stages;

  // ---- producer: one thread streams this CTA's tiles into the ring
  auto issue = [&](int j) {
    const int slot = j % stages;
    const int n0 = (blockIdx.x + j * gridDim.x) * 16;
    uint8_t* st = smem + slot * L.stage_bytes;
    const int rows = min(16, N - n0);
    mbar_arrive_expect_tx(&full[slot], (uint32_t)(L.code_bytes + 2 * rows * G * 2));
    for (int b = 0; b < L.boxes; ++b) tma_load_2d(st + b * 2048, &tm_q, &full[slot], b * 128, n0);
    bulk_load(st + L.code_bytes, sc + (size_t)n0 * G, (uint32_t)(rows * G * 2), &full[slot]);
    bulk_load(st + L.code_bytes + L.sz_bytes, zr + (size_t)n0 * G, (uint32_t)(rows * G * 2),
              &full[slot]);
  };
  int issued = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    for (; issued < min(stages, my_tiles); ++issued) issue(issued);
  }

  // ---- this warp's activation fragments: groups [g_begin, g_end), row m = r,
  // 16 consecutive k (16t .. 16t+15) paired (e, e+4) within each 8
  const int g_begin = (warp * G) / kWarps, ng = ((warp + 1) * G) / kWarps - g_begin;
  uint32_t afr[kGpw][8];
  float sxr[kGpw];
#pragma unroll
  for (int gi = 0; gi < kGpw; ++gi) {
    uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (gi < ng && r < M) {
      const uint16_t* xp = X + (size_t)r * K + (g_begin + gi) * 64 + 16 * t;
      const uint4 lo = ld_keep_v4(xp), hi = ld_keep_v4(xp + 8);
      w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
      w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
    }
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int e = 8 * (p >> 2) + (p & 3);
      afr[gi][p] = elem(w, e) | (elem(w, e + 4) << 16);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += bf16lo_to_f32(w[i]) + bf16hi_to_f32(w[i]);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
    sxr[gi] = s;  // sum over the group's 64 k of row m = r
  }
  __syncthreads();

  for (int j = 0; j < my_tiles; ++j) {
    const int slot = j % stages;
    const int n0 = (blockIdx.x + j * gridDim.x) * 16;
    const bool ok = mbar_wait(&full[slot], (uint32_t)(j / stages) & 1u, dev_status, wait_ns);
    if (!ok) *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;  // CTA-uniform
    const uint8_t* st = smem + slot * L.stage_bytes;
    const uint16_t* ss = reinterpret_cast<const uint16_t*>(st + L.code_bytes);
    const uint16_t* zz = reinterpret_cast<const uint16_t*>(st + L.code_bytes + L.sz_bytes);
    float y[2][2] = {{0.f, 0.f}, {0.f, 0.f}};  // [half][c]: m = r, weight row 8h + 2t + c
#pragma unroll
    for (int gi = 0; gi < kGpw; ++gi) {
      if (gi >= ng) break;
      const int g = g_begin + gi;
      const int chunk = ((2 * (g & 3) + (t >> 1)) ^ r) << 4;
      const uint8_t* box = st + (g >> 2) * 2048 + chunk + (t & 1) * 8;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint2 cw = *reinterpret_cast<const uint2*>(box + (8 * h + r) * 128);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int p0 = 2 * jj, p1 = 2 * jj + 1;
          const uint32_t b0 = nib2_to_bf16x2((p0 >> 2) ? cw.y : cw.x, 4 * (p0 & 3));
          const uint32_t b1 = nib2_to_bf16x2((p1 >> 2) ? cw.y : cw.x, 4 * (p1 & 3));
          mma_bf16_16816(d, afr[gi][p0], 0u, afr[gi][p1], 0u, b0, b1);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int row = 8 * h + 2 * t + c;
          const float s = __half2float(__ushort_as_half(ss[row * G + g]));
          const float z = __half2float(__ushort_as_half(zz[row * G + g]));
          y[h][c] = __fmaf_rn(s, __fmaf_rn(-z, sxr[gi], d[c]), y[h][c]);
        }
      }
    }
    float* rb = red + (size_t)(j & 1) * kWarps * 128;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int c = 0; c < 2; ++c) rb[(warp * 16 + 8 * h + 2 * t + c) * 8 + r] = y[h][c];
    __syncthreads();  // stage `slot` fully read; partials complete
    if (threadIdx.x == 0 && issued < my_tiles) {
      fence_proxy_async_smem();
      issue(issued);
      ++issued;
    }
    if (threadIdx.x < 128) {
      const int row = threadIdx.x >> 3, m = threadIdx.x & 7;
      if (m < M && n0 + row < N) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += rb[(w * 16 + row) * 8 + m];
        if (bias) s += __uint_as_float((uint32_t)bias[n0 + row] << 16);
        Y[(size_t)m * N + n0 + row] = f32_to_bf16_rn(s);
      }
    }
  }
  if (threadIdx.x == 0 && *abort_flag) {  // let issued copies land before exiting
    for (int j = max(0, issued - stages); j < issued; ++j)
      mbar_wait(&full[j % stages], (uint32_t)(j / stages) & 1u, nullptr, wait_ns);
  }
}

}  // namespace

int awq_max_k() { return kWarps * kGpw * 64; }

cudaError_t launch_awq_gemv(const CUtensorMap& tm_q, const uint16_t* X, const uint16_t* scales,
                            const uint16_t* zeros, const uint16_t* bias, uint16_t* Y, int M,
                            int N, int K, int* dev_status, cudaStream_t stream, int num_sms) {
  const AwqLayout L = awq_layout(K);
  if (L.stages < 2 || K > awq_max_k()) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(k_awq_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize, L.smem);
  if (e != cudaSuccess) return e;
  const int tiles = (N + 15) / 16;
  const int grid = tiles < num_sms ? tiles : num_sms;
  k_awq_gemv<<<grid, kThreads, L.smem, stream>>>(tm_q, X, scales, zeros, bias, Y, M, N, K,
                                                 dev_status, kWaitTimeoutNs);
  return cudaGetLastError();
}

}  // namespace svdq
