// svdq_gemm_w4a4: the 4-bit product of the SVDQ W4A4 linear with the
// low-rank up projection and the bias fused into it (dothoosh.com, "How
// Nunchaku Lite halves the VRAM of diffusion models", fused-kernel paragraph:
// the up projection is fused with the 4-bit compute kernel).
//
//   acc  = sum_k dec(a)[m][k] dec(w)[n][k]            tcgen05 kind::mxf4nvf4,
//          + sum_i lora[m][i] (L2[i][n] / s_T)          then kind::f16 (bf16),
//                                                     one fp32 TMEM accumulator
//   Y    = bf16( s_T * acc + bias[n] )
//
// One CTA computes one 128 x BN tile of Y (BN = 256, or 128 when N is not a
// multiple of 256).  Warp roles:
//   warp 0     one lane issues TMA: A/B code tiles (128-byte rows, 128B
//              swizzle) and the block-scale chunks (plain bulk copies: the
//              scale layout is already the tensor core's) into a STAGES-deep
//              ring, completion on `full[s]`;
//   warp 1     allocates TMEM; one lane copies the scales of each stage into
//              TMEM (tcgen05.cp) and issues the MMAs; tcgen05.commit frees a
//              stage (`empty[s]`) and finally signals `acc_full`;
//   warps 2-5  stage the rank-r operands (lora rows, L2 scaled by 1/s_T and
//              transposed to K-major) into shared memory while the main loop
//              runs, then read the accumulator from TMEM (one row per thread)
//              and write bf16 Y.
// Dividing L2 by s_T is exact because s_T is a power of two, so the rank-r
// term can share the fp32 accumulator with the 4-bit product.
//
// Block scales in TMEM.  Per 64-wide K step, the 128 x 4 scale chunk of A
// (512 bytes, row r at byte (r%32)*16 + (r/32)*4) is copied with
// tcgen05.cp.32x128b.warpx4 to 4 columns (lane l, column j holding rows
// l%32 + 32j); B's BN rows take BN/32 columns the same way.
//
// Every wait is bounded: on timeout the kernel reports SVDQ_DEV_TIMEOUT,
// stops issuing work, lets the copies and MMAs in flight land, frees TMEM and
// returns.
#include <cstdint>

#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int BM = 128;
constexpr int BK_BYTES = 128;     // one k tile: 256 fp4 values per row
constexpr int KB_PER_TILE = 4;    // 64-wide MMA steps per k tile
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int BN, int RANK>
struct Cfg {
  static constexpr int STAGES = (BN == 256) ? 3 : 5;
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = BN * BK_BYTES;
  static constexpr int SFA_BYTES = KB_PER_TILE * 512;
  static constexpr int SFB_BYTES = KB_PER_TILE * 512 * (BN / 128);
  static constexpr int LROW = RANK * 2;  // bytes of one rank-r row (bf16)
  static constexpr int LA_BYTES = BM * LROW;
  static constexpr int LB_BYTES = BN * LROW;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_LA = align_up(OFF_SFB + STAGES * SFB_BYTES, 1024);
  static constexpr int OFF_LB = align_up(OFF_LA + LA_BYTES, 1024);
  static constexpr int OFF_BIAS = OFF_LB + LB_BYTES;
  static constexpr int OFF_BAR = align_up(OFF_BIAS + BN * 4, 8);
  static constexpr int NUM_BARS = 2 * STAGES + 2;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + base alignment slack
  // TMEM columns: accumulator [0, BN), then per stage the scales of A and B
  static constexpr int SF_COLS_A = 4 * KB_PER_TILE;
  static constexpr int SF_COLS_B = 4 * KB_PER_TILE * (BN / 128);
  static constexpr int SF_STAGE_COLS = SF_COLS_A + SF_COLS_B;
  static constexpr int SF_BASE = BN;
  static_assert(SF_BASE + STAGES * SF_STAGE_COLS <= (int)TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  // swizzle of the rank-r operands: one row of LROW bytes is one swizzle span
  static constexpr SmemLayout LSW =
      LROW == 128 ? kSwizzle128B : (LROW == 64 ? kSwizzle64B : kSwizzle32B);
  // instruction descriptors (kind::mxf4nvf4: E2M1 x E2M1, UE4M3 scales, K-major,
  // M = 128, N = BN; kind::f16: bf16 x bf16 -> f32)
  static constexpr uint32_t IDESC_NVF4 = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                         ((uint32_t)(BM >> 4) << 24);
  static constexpr uint32_t IDESC_BF16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};

// byte offset of 16-byte chunk c of row `row` in a K-major tile whose rows
// are `rowbytes` long and one swizzle span wide (32/64/128B swizzle)
SVDQ_DEVINL uint32_t swz_off(int row, int c, int rowbytes) {
  const int mask = rowbytes / 16 - 1;
  return (uint32_t)(row * rowbytes + ((c ^ ((row * rowbytes >> 7) & mask)) << 4));
}

template <int BN, int RANK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_w4a4(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const uint8_t* __restrict__ a_scales, const uint8_t* __restrict__ w_scales,
                float s_T, const uint16_t* __restrict__ lora_act,
                const uint16_t* __restrict__ L2, const uint16_t* __restrict__ bias,
                uint16_t* __restrict__ Y, int M, int N, int K, int* dev_status,
                int test_stall, uint64_t wait_ns) {
  using C = Cfg<BN, RANK>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* lora_full = empty + STAGES;
  uint64_t* acc_full = lora_full + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);  // [0] tmem, [1] abort
  float* bias_f = reinterpret_cast<float*>(smem + C::OFF_BIAS);
  volatile uint32_t* abort_flag = &misc[1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.y, n_tile = blockIdx.x;
  const int m0 = m_tile * BM, n0 = n_tile * BN;
  const int kb_total = K >> 6;                   // 64-wide steps
  const int k_tiles = (kb_total + KB_PER_TILE - 1) / KB_PER_TILE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(lora_full, 128);
    mbar_init(acc_full, 1);
    misc[1] = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
  }
  if (warp == 1) tmem_alloc(&misc[0], TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  int issued = 0;  // k tiles whose loads the producer lane has issued
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // test_stall (host test hook): issue nothing, so the consumer's bounded
      // wait runs out and the timeout path is exercised
      for (int kt = 0; kt < (test_stall ? 0 : k_tiles); ++kt) {
        const int s = kt % STAGES;
        const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
        if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1u, dev_status, wait_ns)) {
          *abort_flag = 1;
          break;
        }
        const int nkb = min(KB_PER_TILE, kb_total - kt * KB_PER_TILE);
        const uint32_t bytes =
            (uint32_t)(C::A_BYTES + C::B_BYTES + nkb * 512 * (1 + BN / 128));
        mbar_arrive_expect_tx(&full[s], bytes);
        tma_load_2d(smem + C::OFF_A + s * C::A_BYTES, &tm_a, &full[s], kt * BK_BYTES, m0);
        tma_load_2d(smem + C::OFF_B + s * C::B_BYTES, &tm_b, &full[s], kt * BK_BYTES, n0);
        bulk_load(smem + C::OFF_SFA + s * C::SFA_BYTES,
                  a_scales + ((size_t)m_tile * kb_total + (size_t)kt * KB_PER_TILE) * 512,
                  (uint32_t)nkb * 512u, &full[s]);
#pragma unroll
        for (int h = 0; h < BN / 128; ++h)
          bulk_load(smem + C::OFF_SFB + s * C::SFB_BYTES + h * KB_PER_TILE * 512,
                    w_scales +
                        ((size_t)(n0 / 128 + h) * kb_total + (size_t)kt * KB_PER_TILE) * 512,
                    (uint32_t)nkb * 512u, &full[s]);
        ++issued;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int kt = 0; kt < k_tiles; ++kt) {
        const int s = kt % STAGES;
        const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
        if (*abort_flag || !mbar_wait(&full[s], ph, dev_status, wait_ns)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const int nkb = min(KB_PER_TILE, kb_total - kt * KB_PER_TILE);
        const uint32_t a_base = smem_u32(smem + C::OFF_A + s * C::A_BYTES);
        const uint32_t b_base = smem_u32(smem + C::OFF_B + s * C::B_BYTES);
        const uint32_t sfa = smem_u32(smem + C::OFF_SFA + s * C::SFA_BYTES);
        const uint32_t sfb = smem_u32(smem + C::OFF_SFB + s * C::SFB_BYTES);
        const uint32_t sf_col = (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS);
        for (int kb = 0; kb < nkb; ++kb) {
          tc_cp_32x128b_warpx4(tmem + sf_col + kb * 4,
                               smem_desc(sfa + kb * 512, 128, 128, kSwizzleNone));
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tc_cp_32x128b_warpx4(
                tmem + sf_col + C::SF_COLS_A + kb * 4 * (BN / 128) + h * 4,
                smem_desc(sfb + h * KB_PER_TILE * 512 + kb * 512, 128, 128, kSwizzleNone));
        }
        for (int kb = 0; kb < nkb; ++kb) {
          tc_mma_nvf4(tmem, smem_desc(a_base + kb * 32, 16, 1024, kSwizzle128B),
                      smem_desc(b_base + kb * 32, 16, 1024, kSwizzle128B), C::IDESC_NVF4,
                      tmem + sf_col + kb * 4, tmem + sf_col + C::SF_COLS_A + kb * 4 * (BN / 128),
                      (kt | kb) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[s]);
      }
      if (ok) {
        if (!mbar_wait(lora_full, 0, dev_status, wait_ns)) {
          *abort_flag = 1;
        } else {
          tc_fence_after();
          const uint32_t la = smem_u32(smem + C::OFF_LA), lb = smem_u32(smem + C::OFF_LB);
#pragma unroll
          for (int kk = 0; kk < RANK / 16; ++kk)
            tc_mma_bf16(tmem, smem_desc(la + kk * 32, 16, 8 * C::LROW, C::LSW),
                        smem_desc(lb + kk * 32, 16, 8 * C::LROW, C::LSW), C::IDESC_BF16, 1u);
        }
      }
      tc_commit(acc_full);  // fires once every MMA issued above has completed
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int et = threadIdx.x - 64;  // 0..127
    // (1) rank-r operands into shared memory, K-major, swizzled
    {
      uint8_t* la = smem + C::OFF_LA;
      const int row = m0 + et;
#pragma unroll
      for (int c = 0; c < C::LROW / 16; ++c) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < M) v = ld_keep_v4(lora_act + (size_t)row * RANK + c * 8);
        *reinterpret_cast<uint4*>(la + swz_off(et, c, C::LROW)) = v;
      }
      uint8_t* lb = smem + C::OFF_LB;
      const float inv_sT = 1.0f / s_T;  // exact: s_T is a power of two
#pragma unroll
      for (int h = 0; h < BN / 128; ++h) {
        const int nl = et + 128 * h;
        const uint16_t* src = L2 + n0 + nl;
#pragma unroll
        for (int c = 0; c < C::LROW / 16; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float lo = __uint_as_float((uint32_t)src[(size_t)(8 * c + 2 * p) * N] << 16);
            const float hi =
                __uint_as_float((uint32_t)src[(size_t)(8 * c + 2 * p + 1) * N] << 16);
            w[p] = (uint32_t)f32_to_bf16_rn(lo * inv_sT) |
                   ((uint32_t)f32_to_bf16_rn(hi * inv_sT) << 16);
          }
          *reinterpret_cast<uint4*>(lb + swz_off(nl, c, C::LROW)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        bias_f[nl] = bias ? __uint_as_float((uint32_t)bias[n0 + nl] << 16) : 0.0f;
      }
      fence_proxy_async_smem();
      mbar_arrive(lora_full);
      asm volatile("bar.sync 1, 128;" ::: "memory");  // bias_f visible to all epilogue warps
    }
    // (2) accumulator -> Y
    if (mbar_wait(acc_full, 0, dev_status, wait_ns) && !*abort_flag) {
      tc_fence_after();
      const int q = warp & 3;  // TMEM lane quarter this warp may access
      const int row = m0 + q * 32 + lane;
      uint16_t* yrow = Y + (size_t)row * N + n0;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(c * 32), v);
        tmem_ld_wait();
        if (row < M) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float y0 = __fmaf_rn(s_T, __uint_as_float(v[2 * j]), bias_f[c * 32 + 2 * j]);
            const float y1 =
                __fmaf_rn(s_T, __uint_as_float(v[2 * j + 1]), bias_f[c * 32 + 2 * j + 1]);
            pk[j] = (uint32_t)f32_to_bf16_rn(y0) | ((uint32_t)f32_to_bf16_rn(y1) << 16);
          }
          uint4* dst = reinterpret_cast<uint4*>(yrow + c * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // an aborted tile: the last STAGES loads may still be landing; the CTA
    // must not exit before they complete
    for (int kt = max(0, issued - STAGES); kt < issued; ++kt)
      mbar_wait(&full[kt % STAGES], (uint32_t)(kt / STAGES) & 1u, nullptr, wait_ns);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int BN, int RANK>
cudaError_t launch_t(const GemmMaps& maps, const uint8_t* a_scales, const uint8_t* w_scales,
                     float s_T, const uint16_t* lora_act, const uint16_t* L2,
                     const uint16_t* bias, uint16_t* Y, int M, int N, int K, int* dev_status,
                     int test_stall, cudaStream_t stream) {
  using C = Cfg<BN, RANK>;
  auto kern = k_gemm_w4a4<BN, RANK>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(N / BN, (M + BM - 1) / BM);
  kern<<<grid, NUM_THREADS, C::SMEM_BYTES, stream>>>(maps.a_codes, maps.w_codes, a_scales,
                                                     w_scales, s_T, lora_act, L2, bias, Y, M, N,
                                                     K, dev_status, test_stall,
                                                     test_stall ? 100000000ull : kWaitTimeoutNs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_w4a4(const GemmMaps& maps, int block_n, const uint8_t* a_scales,
                             const uint8_t* w_scales, float w_tensor_scale,
                             const uint16_t* lora_act, const uint16_t* L2,
                             const uint16_t* bias, uint16_t* Y, int M, int N, int K, int rank,
                             int* dev_status, int test_stall, cudaStream_t stream) {
#define SVDQ_GEMM_CASE(BN_, R_)                                                               \
  if (block_n == BN_ && rank == R_)                                                           \
    return launch_t<BN_, R_>(maps, a_scales, w_scales, w_tensor_scale, lora_act, L2, bias, Y, \
                             M, N, K, dev_status, test_stall, stream);
  SVDQ_GEMM_CASE(256, 16)
  SVDQ_GEMM_CASE(256, 32)
  SVDQ_GEMM_CASE(256, 64)
  SVDQ_GEMM_CASE(128, 16)
  SVDQ_GEMM_CASE(128, 32)
  SVDQ_GEMM_CASE(128, 64)
#undef SVDQ_GEMM_CASE
  return cudaErrorInvalidValue;
}

}  // namespace svdq
