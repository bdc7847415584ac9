// svdq_gemm_w4a4_int4: the 4-bit GEMM of the INT4 variant of the SVDQ W4A4
// linear (dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion
// models", kernel-family list: svdq_w4a4 comes in INT4 and NVFP4 variants;
// hardware list: INT4 is the format of the pre-Blackwell GPUs).
//
//   Y[m][n] = bf16( sum_g sx[m][g] sw[n][g] sum_{k in g} qx[m][k] qw[n][k]
//                   + sum_i lora_act[m][i] L2[n][i] + bias[n] )
//
// groups g of 64 consecutive k, codes signed 4-bit integers, scales bf16.
// B300's tensor cores have no integer 4-bit path, but every code -8..7 is an
// exact f16 value: per group, tcgen05 kind::f16 MMAs (M = 128, N = 128,
// K = 4 x 16) of the f16 code tiles give the group's integer sum exactly in
// fp32 (|sum| <= 64 * 64) in a TMEM partial, and the epilogue warps add it to
// their register accumulators with one fma by the product sx * sw (exact: two
// 8-bit significands).  The low-rank term is one more "group": bf16 MMAs of
// lora_act and L2 into a partial, added with unit scales.  Y is rounded once.
//
// One CTA per 128 x 128 output tile; warp roles:
//   warps 0-3   converters: each thread owns row c of the A tile and row c of
//               the W tile; it copies their codes and scale words kRing groups
//               ahead into a ring in shared memory (cp.async: a thread reads
//               back only its own bytes, so no CTA barrier), and per group
//               writes the 64 codes of both rows as f16 into a 128-byte row of
//               an operand tile (128B swizzle, K-major: the tcgen05 layout)
//               and the rows' two scales; the rows of lora_act and L2 go
//               straight into bf16 operand tiles at the start;
//   warps 4-11  epilogue: lane quarter warp % 4, 64 columns each; per group
//               read the TMEM partial, fma it into 64 fp32 accumulators;
//   warp 12     TMEM allocation and the MMA issue (one lane).
// Four operand-tile buffers and four TMEM partials (128 columns each) let the
// conversion, the MMAs and the epilogue of different groups overlap with
// slack for the hand-over latencies; the group scales sit in an 8-deep ring
// (a converter writes scale slot g % 8 only after the MMAs of group g - 4,
// which waited for the epilogue of group g - 8 to finish with that slot).
// Every wait is bounded and reports SVDQ_DEV_TIMEOUT through the status word.
#include <cstdint>

#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int kBM = 128, kBN = 128;
constexpr int kConvWarps = 4, kEpiWarps = 8;
constexpr int kMmaWarp = kConvWarps + kEpiWarps;  // warp 12
constexpr int kThreads = 32 * (kMmaWarp + 1);     // 416
constexpr int kTileBytes = 128 * 128;             // 128 rows x 128 bytes (64 f16)
constexpr int kBuf = 4;                           // operand-tile buffers and TMEM partials
constexpr int kScaleSlots = 2 * kBuf;             // depth of the group-scale ring
constexpr int kRing = 5;                          // groups of codes in flight per thread
constexpr int kSlotBytes = 2 * 128 * 32 + 2 * 128 * 4;  // codes of A and W rows, scale words
constexpr int kOffA = 0;                          // [kBuf] A tiles
constexpr int kOffB = kOffA + kBuf * kTileBytes;  // [kBuf] W tiles
constexpr int kOffLR = kOffB + kBuf * kTileBytes; // lora_act rows (bf16 operand tile)
constexpr int kOffLW = kOffLR + kTileBytes;       // L2 rows (bf16 operand tile)
constexpr int kOffRing = kOffLW + kTileBytes;     // [kRing] slots of codes and scale words
constexpr int kOffSX = kOffRing + kRing * kSlotBytes;    // [slots][128] fp32 activation scales
constexpr int kOffSW = kOffSX + kScaleSlots * 128 * 4;   // [slots][128] fp32 weight scales
constexpr int kOffBar = kOffSW + kScaleSlots * 128 * 4;  // 4 x kBuf mbarriers
constexpr int kOffMisc = kOffBar + 4 * kBuf * 8;         // TMEM base, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + slack for the 1024-byte base alignment
constexpr uint32_t kTmemCols = 128 * kBuf;        // kBuf partials of 128 columns
static_assert(kSmemBytes <= 227 * 1024 && kTmemCols <= 512, "shared and tensor memory");
// instruction descriptors, kind::f16: D fp32, K-major A and B, N = 128, M = 128;
// A and B f16 (format 0) for the code tiles, bf16 (format 1) for the low rank
constexpr uint32_t kIdescF16 =
    (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
constexpr uint32_t kIdescBF16 = kIdescF16 | (1u << 7) | (1u << 10);

SVDQ_DEVINL void sts128v(uint8_t* p, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
SVDQ_DEVINL float4 lds128f(const float* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p)));
  return v;
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
// byte offset of 16-byte piece p (0..7) of row r in an operand tile (128B
// swizzle: pieces XOR-ed by r % 8 within each 1024-byte group of 8 rows)
SVDQ_DEVINL int tile_piece(int r, int p) { return r * 128 + ((p ^ (r & 7)) << 4); }

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_int4(const uint8_t* __restrict__ a_codes, const uint16_t* __restrict__ a_scales,
                const uint8_t* __restrict__ w_codes, const uint16_t* __restrict__ w_scales,
                const uint16_t* __restrict__ lora_act, const uint16_t* __restrict__ L2,
                const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K,
                int rank, int* dev_status, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int G = K >> 6;  // code groups; "group" G is the low-rank term
  uint64_t* f16_full = reinterpret_cast<uint64_t*>(smem + kOffBar);  // [kBuf] count 128
  uint64_t* f16_empty = f16_full + kBuf;                              // [kBuf] MMA commit
  uint64_t* part_full = f16_full + 2 * kBuf;                          // [kBuf] MMA commit
  uint64_t* part_empty = f16_full + 3 * kBuf;                         // [kBuf] count kEpiWarps
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const float* sx_ring = reinterpret_cast<const float*>(smem + kOffSX);
  const float* sw_ring = reinterpret_cast<const float*>(smem + kOffSW);

  if (threadIdx.x == 0) {
    for (int b = 0; b < kBuf; ++b) {
      mbar_init(&f16_full[b], 32 * kConvWarps);
      mbar_init(&f16_empty[b], 1);
      mbar_init(&part_full[b], 1);
      mbar_init(&part_empty[b], kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tslot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  grid_dep_launch();
  grid_dep_wait();  // the previous kernel's outputs (the activation side) are complete

  if (warp < kConvWarps) {
    // ---------------------------------------------------------------- converters
    const int c = threadIdx.x;  // row of the A tile and of the W tile
    const int ar = m0 + c;
    const bool arow = ar < M;
    const size_t row_bytes = (size_t)K / 2;
    const uint8_t* ap = a_codes + (size_t)(arow ? ar : M - 1) * row_bytes;
    const uint8_t* wp = w_codes + (size_t)(n0 + c) * row_bytes;
    // the low-rank rows first (their own commit group): piece p of row c at
    // its swizzled place in the bf16 operand tiles
    for (int p = 0; p < rank / 8; ++p) {
      cp_async16_cg(smem + kOffLR + tile_piece(c, p),
                    lora_act + (size_t)(arow ? ar : M - 1) * rank + 8 * p, arow ? 16 : 0);
      cp_async16_cg(smem + kOffLW + tile_piece(c, p), L2 + (size_t)(n0 + c) * rank + 8 * p, 16);
    }
    cp_async_commit();
    // codes and scale words of group g into ring slot g % kRing (one commit
    // group per group, empty past the last).  Scale element i sits in the
    // 4-byte word at i & ~1: G is even, so a row's word holds groups g & ~1
    // and g | 1, and the word never passes the end of the array.
    auto fetch = [&](int g) {
      if (g < G) {
        uint8_t* slot = smem + kOffRing + (g % kRing) * kSlotBytes;
        cp_async16_cg(slot + c * 32, ap + (size_t)g * 32, arow ? 16 : 0);
        cp_async16_cg(slot + c * 32 + 16, ap + (size_t)g * 32 + 16, arow ? 16 : 0);
        cp_async16_cg(slot + 4096 + c * 32, wp + (size_t)g * 32, 16);
        cp_async16_cg(slot + 4096 + c * 32 + 16, wp + (size_t)g * 32 + 16, 16);
        cp_async<4>(slot + 8192 + c * 4,
                    a_scales + (((size_t)(arow ? ar : M - 1) * G + g) & ~(size_t)1),
                    arow ? 4 : 0);
        cp_async<4>(slot + 8704 + c * 4, w_scales + (((size_t)(n0 + c) * G + g) & ~(size_t)1),
                    4);
      }
      cp_async_commit();
    };
#pragma unroll 1
    for (int s = 0; s < kRing - 1; ++s) fetch(s);
    for (int g = 0; g <= G; ++g) {
      const int b = g % kBuf;
      fetch(g + kRing - 1);  // into the slot of group g - 1, read last iteration
      if (!mbar_wait(&f16_empty[b], (((uint32_t)g / kBuf) & 1u) ^ 1u, dev_status, wait_ns))
        *abort_flag = 1;
      if (*abort_flag) break;
      cp_async_wait<kRing - 1>();  // the low-rank rows and this thread's copies of group g
      float* sx = reinterpret_cast<float*>(smem + kOffSX) + (g % kScaleSlots) * 128;
      float* sw = reinterpret_cast<float*>(smem + kOffSW) + (g % kScaleSlots) * 128;
      if (g < G) {
        const uint8_t* slot = smem + kOffRing + (g % kRing) * kSlotBytes;
        uint8_t* ta = smem + kOffA + b * kTileBytes;
        uint8_t* tw = smem + kOffB + b * kTileBytes;
        const uint4 a0 = lds128(slot + c * 32), a1 = lds128(slot + c * 32 + 16);
        const uint4 w0 = lds128(slot + 4096 + c * 32), w1 = lds128(slot + 4096 + c * 32 + 16);
        const uint32_t a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          sts128v(ta + tile_piece(c, p), nib8_to_f16(a[p]));
          sts128v(tw + tile_piece(c, p), nib8_to_f16(w[p]));
        }
        const uint32_t sh = (uint32_t)(g & 1) * 16;  // the group's half of the scale word
        const uint32_t sa = *reinterpret_cast<const uint32_t*>(slot + 8192 + c * 4);
        const uint32_t sb = *reinterpret_cast<const uint32_t*>(slot + 8704 + c * 4);
        sx[c] = arow ? __uint_as_float(((sa >> sh) & 0xFFFFu) << 16) : 0.0f;
        sw[c] = __uint_as_float(((sb >> sh) & 0xFFFFu) << 16);
      } else {
        sx[c] = 1.0f;  // the low-rank term: unit scales
        sw[c] = 1.0f;
      }
      fence_proxy_async_smem();  // the tiles are read by the tensor cores (async proxy)
      mbar_arrive(&f16_full[b]);
    }
    cp_async_wait<0>();  // nothing may land in shared memory after the CTA exits
  } else if (warp < kMmaWarp) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int col0 = ((warp - kConvWarps) >> 2) * 64;  // its 64 columns of the tile
    const int row = 32 * q + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
    for (int g = 0; g <= G; ++g) {
      const int b = g % kBuf;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&part_full[b], ((uint32_t)g / kBuf) & 1u,
                                             dev_status, wait_ns)))
        *abort_flag = 1;
      if (*abort_flag) break;
      tc_fence_after();
      const float* sx = sx_ring + (g % kScaleSlots) * 128;
      const float* sw = sw_ring + (g % kScaleSlots) * 128 + col0;
      const float s_row = sx[row];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_base + (uint32_t)(b * 128 + col0 + 32 * h), v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 s4 = lds128f(sw + 32 * h + j);
          // acc += partial * (sx * sw): the scale product is exact, one rounding
          const float2 p01 = mul2_rn(make_float2(s_row, s_row), make_float2(s4.x, s4.y));
          const float2 p23 = mul2_rn(make_float2(s_row, s_row), make_float2(s4.z, s4.w));
          const float2 a01 = fma2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])),
                                     p01, make_float2(acc[32 * h + j], acc[32 * h + j + 1]));
          const float2 a23 = fma2_rn(make_float2(__uint_as_float(v[j + 2]),
                                                 __uint_as_float(v[j + 3])),
                                     p23, make_float2(acc[32 * h + j + 2], acc[32 * h + j + 3]));
          acc[32 * h + j] = a01.x;
          acc[32 * h + j + 1] = a01.y;
          acc[32 * h + j + 2] = a23.x;
          acc[32 * h + j + 3] = a23.y;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&part_empty[b]);  // partial b and the group's scales are read
    }
    // bias, one rounding to bf16, Y (64 consecutive columns of one row)
    const int r = m0 + row;
    if (!*abort_flag && r < M) {
      uint16_t* yp = Y + (size_t)r * N + n0 + col0;
#pragma unroll
      for (int j = 0; j < 64; j += 8) {
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float b0 = 0.0f, b1 = 0.0f;
          if (bias) {
            const uint32_t bw = __ldg(reinterpret_cast<const uint32_t*>(bias + n0 + col0 + j) + e);
            b0 = bf16lo_to_f32(bw);
            b1 = bf16hi_to_f32(bw);
          }
          o[e] = (uint32_t)f32_to_bf16_rn(acc[j + 2 * e] + b0) |
                 ((uint32_t)f32_to_bf16_rn(acc[j + 2 * e + 1] + b1) << 16);
        }
        *reinterpret_cast<uint4*>(yp + j) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  } else {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      int issued = 0;
      for (int g = 0; g <= G; ++g) {
        const int b = g % kBuf;
        const uint32_t ph = ((uint32_t)g / kBuf) & 1u;
        if (!mbar_wait(&f16_full[b], ph, dev_status, wait_ns) ||
            !mbar_wait(&part_empty[b], ph ^ 1u, dev_status, wait_ns))
          *abort_flag = 1;
        if (*abort_flag) break;
        tc_fence_after();
        const bool low_rank = g == G;
        const uint32_t a0 = smem_u32(smem + (low_rank ? kOffLR : kOffA + b * kTileBytes));
        const uint32_t w0 = smem_u32(smem + (low_rank ? kOffLW : kOffB + b * kTileBytes));
        const int ksteps = low_rank ? rank / 16 : 4;
        for (int kk = 0; kk < ksteps; ++kk)
          tc_mma_bf16(tmem + (uint32_t)(b * 128),
                      smem_desc(a0 + 32u * kk, 16, 1024, kSwizzle128B),
                      smem_desc(w0 + 32u * kk, 16, 1024, kSwizzle128B),
                      low_rank ? kIdescBF16 : kIdescF16, kk > 0 ? 1u : 0u);
        tc_commit(&part_full[b]);
        tc_commit(&f16_empty[b]);
        issued = g + 1;
      }
      // every issued MMA has completed before the TMEM is released (commits
      // complete in order)
      if (issued > 0) {
        const int g = issued - 1;
        mbar_wait(&part_full[g % kBuf], ((uint32_t)g / kBuf) & 1u, nullptr, wait_ns);
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_gemm_int4(const uint8_t* a_codes, const uint16_t* a_scales,
                             const uint8_t* w_codes, const uint16_t* w_scales,
                             const uint16_t* lora_act, const uint16_t* L2, const uint16_t* bias,
                             uint16_t* Y, int M, int N, int K, int rank, int* dev_status,
                             cudaStream_t stream) {
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
                         bias, Y, M, N, K, rank, dev_status, (uint64_t)kWaitTimeoutNs);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace svdq
