// svdq_gemm_w4a4_int4: the 4-bit GEMM of the INT4 variant of the SVDQ W4A4
// linear (dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion
// models", kernel-family list: svdq_w4a4 comes in INT4 and NVFP4 variants;
// hardware list: INT4 is the format of the pre-Blackwell GPUs).
//
//   Y[m][n] = bf16( sum_g sx[m][g] sw[n][g] sum_{k in g} qx[m][k] qw[n][k]
//                   + sum_i lora_act[m][i] L2[n][i] + bias[n] )
//
// groups g of 64 consecutive k, codes signed 4-bit integers, scales bf16.
// B300's tensor cores have no integer 4-bit path (and a slow 8-bit one), so
// this variant runs on the warp-level f16 MMA: every code -8..7 is exactly an
// f16 value, the m16n8k16 MMAs of one group accumulate its integer sum
// exactly in fp32 (|sum| <= 64 * 64), and the group's sum is added to the
// accumulator with one fma by the product sx * sw (exact: two 8-bit
// significands).  The low-rank up projection runs as bf16 m16n8k16 MMAs into
// the same accumulators, then the bias; Y is rounded once.
//
// CTA tile 128 x 128, 16 warps of 32 x 32 (four per scheduler, at most 128
// registers each); k tiles of 128 (two groups) stream through a 3-stage
// cp.async ring (codes 64 bytes per row, scales 4 bytes per row).  Each k
// tile's codes are converted once per CTA into f16 tiles (rows of 256 bytes,
// the 16-byte pieces of each 128-byte half XOR-ed by row % 8, read with
// ldmatrix), keeping the k order.
#include <cstdint>

#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 128;
constexpr int kThreads = 512;
constexpr int kStages = 3;
constexpr int kNibBytes = kBK / 2;                    // code bytes per row per k tile
constexpr int kStageA = 0;                            // [128][64] codes
constexpr int kStageB = kStageA + kBM * kNibBytes;    // [128][64] codes
constexpr int kStageSA = kStageB + kBN * kNibBytes;   // [128][2] bf16 scales
constexpr int kStageSB = kStageSA + kBM * 4;          // [128][2] bf16 scales
constexpr int kStageBytes = kStageSB + kBN * 4;
constexpr int kF16Row = kBK * 2;                      // bytes of a converted row
constexpr int kE4A = kStages * kStageBytes;           // [128][128] f16
constexpr int kE4B = kE4A + kBM * kF16Row;
constexpr int kSmemBytes = kE4B + kBN * kF16Row;
static_assert(kStageBytes % 16 == 0 && kE4A % 128 == 0, "alignment");

SVDQ_DEVINL uint32_t lds32(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}
SVDQ_DEVINL uint32_t lds16(const uint8_t* p) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(smem_u32(p)));
  return v;
}
SVDQ_DEVINL void sts128v(uint8_t* p, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
SVDQ_DEVINL void ldsm_x4(const uint8_t* p, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                         uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
// D[16x8] += A[16x16] B[16x8], f16 inputs, fp32 accumulate
SVDQ_DEVINL void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
      "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
SVDQ_DEVINL uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
SVDQ_DEVINL uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// eight two's-complement nibbles (element i at bits 4i..4i+3) -> eight f16
// values of the same integers, element i in half i of the 16 bytes: v + 8 is
// the nibble with its top bit flipped; the f16 with bits 0x6400 | (v + 8) is
// 1024 + v + 8, and subtracting 1032 leaves v exactly
SVDQ_DEVINL uint4 nib8_to_f16(uint32_t w) {
  const uint32_t u = w ^ 0x88888888u;
  const uint32_t t0 = u & 0x0F0F0F0Fu;         // v0, v2, v4, v6 (+ 8), one per byte
  const uint32_t t1 = (u >> 4) & 0x0F0F0F0Fu;  // v1, v3, v5, v7 (+ 8)
  const uint32_t lo = prmt(t0, t1, 0x5140u);   // v0, v1, v2, v3
  const uint32_t hi = prmt(t0, t1, 0x7362u);   // v4, v5, v6, v7
  constexpr uint32_t kHigh = 0x64646464u, kOff = 0x64086408u;  // f16 1032 twice
  return make_uint4(hsub2(prmt(lo, kHigh, 0x4140u), kOff), hsub2(prmt(lo, kHigh, 0x4342u), kOff),
                    hsub2(prmt(hi, kHigh, 0x4140u), kOff), hsub2(prmt(hi, kHigh, 0x4342u), kOff));
}
// byte offset of 16-byte piece c (0..15) of row r in a converted tile
SVDQ_DEVINL int f16_piece(int r, int c) { return r * kF16Row + (((c & 8) | ((c ^ r) & 7)) << 4); }

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_int4(const uint8_t* __restrict__ a_codes, const uint16_t* __restrict__ a_scales,
                const uint8_t* __restrict__ w_codes, const uint16_t* __restrict__ w_scales,
                const uint16_t* __restrict__ lora_act, const uint16_t* __restrict__ L2,
                const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K,
                int rank) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int wm = warp >> 2, wn = warp & 3;  // warp tile rows wm*32, cols wn*32
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int G = K >> 6, KT = K / kBK;
  const size_t row_bytes = (size_t)K / 2;

  grid_dep_launch();
  grid_dep_wait();  // the previous kernel's outputs (the activation codes) are complete

  // asynchronous copies of k tile kt into stage kt % kStages (one commit
  // group per tile, empty past the last, so that group counting is uniform)
  auto load = [&](int kt) {
    if (kt < KT) {
      uint8_t* st = smem + (kt % kStages) * kStageBytes;
      {
        const int r = tid >> 2, c = tid & 3;  // 128 rows x 4 pieces of 16 bytes
        const int ar = m0 + r;
        cp_async16_cg(st + kStageA + r * kNibBytes + c * 16,
                      a_codes + (size_t)min(ar, M - 1) * row_bytes + kt * kNibBytes + c * 16,
                      ar < M ? 16 : 0);
        cp_async16_cg(st + kStageB + r * kNibBytes + c * 16,
                      w_codes + (size_t)(n0 + r) * row_bytes + kt * kNibBytes + c * 16, 16);
      }
      if (tid < kBM) {
        const int ar = m0 + tid;
        cp_async<4>(st + kStageSA + tid * 4, a_scales + (size_t)min(ar, M - 1) * G + kt * 2,
                    ar < M ? 4 : 0);
      } else if (tid < kBM + kBN) {
        const int r = tid - kBM;
        cp_async<4>(st + kStageSB + r * 4, w_scales + (size_t)(n0 + r) * G + kt * 2, 4);
      }
    }
    cp_async_commit();
  };

  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][j][c] = 0.0f;

  uint8_t* e4a = smem + kE4A;  // converted A tile (f16)
  uint8_t* e4b = smem + kE4B;  // converted B tile (f16)
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) load(s);
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<kStages - 2>();  // this thread's copies of tile kt landed
    __syncthreads();  // ... and every thread's; every warp is done with the f16 tiles
    const uint8_t* st = smem + (kt % kStages) * kStageBytes;
    // codes -> f16 tiles: 2 x 128 rows x 16 words of 8 codes (one 16-byte
    // piece each)
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
      const int idx = tid + kThreads * i;        // 0 .. 4095
      const int half = idx >> 11, q = idx & 2047;  // A or B; word q of the tile
      const int r = q >> 4, wd = q & 15;
      const uint32_t w = lds32(st + (half ? kStageB : kStageA) + r * kNibBytes + wd * 4);
      sts128v((half ? e4b : e4a) + f16_piece(r, wd), nib8_to_f16(w));
    }
    __syncthreads();
    load(kt + kStages - 1);  // into the stage of tile kt - 1, converted last iteration

#pragma unroll
    for (int h = 0; h < 2; ++h) {  // the two groups of the k tile
      float part[2][4][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int c = 0; c < 4; ++c) part[i][j][c] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int c0 = h * 8 + kk * 2;  // first 16-byte piece of this k16 step
        uint32_t a[2][4], b[4][2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = wm * 32 + 16 * i + (lane & 7) + ((lane >> 3) & 1) * 8;
          ldsm_x4(e4a + f16_piece(r, c0 + (lane >> 4)), a[i][0], a[i][1], a[i][2], a[i][3]);
        }
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          const int r = wn * 32 + 16 * jp + (lane & 7) + (lane >> 4) * 8;
          ldsm_x4(e4b + f16_piece(r, c0 + ((lane >> 3) & 1)), b[2 * jp][0], b[2 * jp][1],
                  b[2 * jp + 1][0], b[2 * jp + 1][1]);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) mma_f16_16816(part[i][j], a[i], b[j][0], b[j][1]);
      }
      // acc += part * (sx sw): the scale product is exact, one rounding per fma
      float2 sw[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = wn * 32 + 8 * j + 2 * t;
        sw[j] = make_float2(__uint_as_float(lds16(st + kStageSB + c * 4 + h * 2) << 16),
                            __uint_as_float(lds16(st + kStageSB + (c + 1) * 4 + h * 2) << 16));
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = wm * 32 + 16 * i + g;
        const float sa = __uint_as_float(lds16(st + kStageSA + r * 4 + h * 2) << 16);
        const float sb = __uint_as_float(lds16(st + kStageSA + (r + 8) * 4 + h * 2) << 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 pa = mul2_rn(make_float2(sa, sa), sw[j]);
          const float2 pb = mul2_rn(make_float2(sb, sb), sw[j]);
          const float2 lo = fma2_rn(make_float2(part[i][j][0], part[i][j][1]), pa,
                                    make_float2(acc[i][j][0], acc[i][j][1]));
          const float2 hi = fma2_rn(make_float2(part[i][j][2], part[i][j][3]), pb,
                                    make_float2(acc[i][j][2], acc[i][j][3]));
          acc[i][j][0] = lo.x; acc[i][j][1] = lo.y;
          acc[i][j][2] = hi.x; acc[i][j][3] = hi.y;
        }
      }
    }
  }
  cp_async_wait<0>();  // nothing may land in shared memory after the CTA exits

  // ---- low-rank up projection (bf16 MMAs into the accumulators), bias, Y
  auto ld32 = [](const uint16_t* p) { return __ldg(reinterpret_cast<const uint32_t*>(p)); };
  for (int k16 = 0; k16 < rank; k16 += 16) {
    uint32_t b[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint16_t* p = L2 + (size_t)(n0 + wn * 32 + 8 * j + g) * rank + k16 + 2 * t;
      b[j][0] = ld32(p);
      b[j][1] = ld32(p + 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r0 = m0 + wm * 32 + 16 * i + g, r1 = r0 + 8;
      const uint16_t* p0 = lora_act + (size_t)min(r0, M - 1) * rank + k16 + 2 * t;
      const uint16_t* p1 = lora_act + (size_t)min(r1, M - 1) * rank + k16 + 2 * t;
      const uint32_t a0 = r0 < M ? ld32(p0) : 0u, a2 = r0 < M ? ld32(p0 + 8) : 0u;
      const uint32_t a1 = r1 < M ? ld32(p1) : 0u, a3 = r1 < M ? ld32(p1 + 8) : 0u;
#pragma unroll
      for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[i][j], a0, a1, a2, a3, b[j][0], b[j][1]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = n0 + wn * 32 + 8 * j + 2 * t;
    float b0 = 0.0f, b1 = 0.0f;
    if (bias) {
      const uint32_t bw = ld32(bias + c);
      b0 = bf16lo_to_f32(bw);
      b1 = bf16hi_to_f32(bw);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r0 = m0 + wm * 32 + 16 * i + g;
      if (r0 < M)
        *reinterpret_cast<uint32_t*>(Y + (size_t)r0 * N + c) =
            (uint32_t)f32_to_bf16_rn(acc[i][j][0] + b0) |
            ((uint32_t)f32_to_bf16_rn(acc[i][j][1] + b1) << 16);
      if (r0 + 8 < M)
        *reinterpret_cast<uint32_t*>(Y + (size_t)(r0 + 8) * N + c) =
            (uint32_t)f32_to_bf16_rn(acc[i][j][2] + b0) |
            ((uint32_t)f32_to_bf16_rn(acc[i][j][3] + b1) << 16);
    }
  }
}

}  // namespace

cudaError_t launch_gemm_int4(const uint8_t* a_codes, const uint16_t* a_scales,
                             const uint8_t* w_codes, const uint16_t* w_scales,
                             const uint16_t* lora_act, const uint16_t* L2, const uint16_t* bias,
                             uint16_t* Y, int M, int N, int K, int rank, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(k_gemm_int4, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(N / kBN), (unsigned)((M + kBM - 1) / kBM), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_gemm_int4, a_codes, a_scales, w_codes, w_scales, lora_act, L2,
                         bias, Y, M, N, K, rank);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace svdq
