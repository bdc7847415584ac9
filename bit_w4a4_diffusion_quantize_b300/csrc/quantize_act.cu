// svdq_quantize_act: the activation side of the SVDQ W4A4 linear in one pass
// over X (dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion
// models", fused-kernel paragraph: the low-rank down projection is fused with
// the quantization kernel).
//
//   lora_act[m][i] = bf16( sum_k X[m][k] L1s[i][k] )      tensor cores, fp32 acc
//   x_hat          = fl32( X[m][k] * inv_lambda[k] )
//   scale byte     = RNE_e4m3( amax16(x_hat) / 6 )        exact quotient rounding
//   code nibble    = RNE_e2m1( x_hat / s )                exact quotient rounding
//
// Work split.  A CTA owns 32 consecutive rows (two m16 tiles) and all of K;
// K is split into 8 contiguous ranges of 64-wide steps, each streamed through
// its own TMA ring in shared memory: per step a 32 x 64 bf16 tile of X, the
// rank x 64 slice of L1s (both with the 128-byte swizzle, so the fragment
// reads below are free of bank conflicts) and the 64 matching floats of
// inv_lambda, landing on one mbarrier.  Two warps share a ring, one per m
// tile (16 warps per CTA); a slot is refilled once both have read it.  In one
// step a thread (quad lane t, group g) holds 16 consecutive k of rows g and
// g+8 of its m tile: exactly one 16-element quantization block per row.  The
// same registers are the A fragments of the m16n8k16 MMAs of the down
// projection; the k order inside an MMA is permuted, and the B fragments (L1s
// rows, k contiguous) use the same permutation.  Partial lora sums of the 8 K
// ranges are added in a fixed order through shared memory, then rounded once.
//
// Exact quotients without division.  For a divisor d with few significant
// bits (6 for the scale, an e4m3 value s for the codes), take r_hi = RD(1/d)
// and r_lo = RN((1 - r_hi d) / d) (the residual 1 - r_hi d is exact through
// one fma).  Then y = RN(x r_hi + RN(x r_lo)) differs from x/d by less than
// 2^-46 of it.  An exact quotient of a 24-bit x is either a grid midpoint m
// itself or more than half an ulp of m away from it (for d = s, x_hat/s vs the
// e2m1 midpoints: at least 0.53 ulp(m); for d = 6, amax/6 vs the e4m3
// midpoints: at least 0.66 ulp(m)), so y rounds (RNE, satfinite) to the same
// grid point as the exact quotient.  r_hi rounds down so that r_lo >= 0 and y
// keeps the sign of x_hat even for -0.  The reciprocal pairs of the 127
// positive e4m3 values are tabulated per CTA.  A block holding +-inf gets
// s = 448 (saturated), r_lo > 0, so inf stays inf and saturates to +-6, which
// is the exact rounding too.  A block whose s is 0 is masked to codes +0.
#include <cstdint>

#include "act_quant.cuh"
#include "device_common.cuh"
#include "int4_quant.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int kRanges = 8;               // K ranges (TMA rings) per CTA
constexpr int kWarps = 2 * kRanges;      // two warps (m tiles) per range
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 32;  // rows per CTA (two m16 tiles)
constexpr int kSmemBudget = 222 * 1024;

template <int RANK>
struct QCfg {
  static constexpr int NT = RANK / 8;            // n8 tiles of the down projection
  static constexpr int X_BYTES = kRows * 128;    // 32 rows x 64 bf16
  static constexpr int L_BYTES = RANK * 128;     // RANK rows x 64 bf16 of L1s
  static constexpr int INV_BYTES = 64 * 4;
  static constexpr int TX_BYTES = X_BYTES + L_BYTES + INV_BYTES;
  static constexpr int STAGE_ALL = kRanges * (X_BYTES + L_BYTES + INV_BYTES);
  static constexpr int FIXED = 128 * 8 + kRanges * 8 * 8;  // reciprocal table, barriers
  static constexpr int STAGES = (kSmemBudget - FIXED) / STAGE_ALL > 4
                                    ? 4 : (kSmemBudget - FIXED) / STAGE_ALL;
  static constexpr int OFF_X = 0;                                    // [ranges][stages] tiles
  static constexpr int OFF_L = OFF_X + kRanges * STAGES * X_BYTES;   // [ranges][stages] slices
  static constexpr int OFF_INV = OFF_L + kRanges * STAGES * L_BYTES;
  static constexpr int OFF_TAB = OFF_INV + kRanges * STAGES * INV_BYTES;  // [128] float2
  static constexpr int OFF_BAR = OFF_TAB + 128 * 8;  // [ranges][4] full, [ranges][4] empty
  // the lora partials [ranges][32 rows][RANK] fp32 reuse the X ring afterwards
  static constexpr int RED_BYTES = kRanges * kRows * RANK * 4;
  static_assert(RED_BYTES <= OFF_L, "reduction buffer fits the X ring");
  static_assert(STAGES >= 2 && STAGES <= 4, "pipeline depth");
  static constexpr int SMEM_BYTES = OFF_BAR + kRanges * 8 * 8 + 1024;  // + alignment slack
};

SVDQ_DEVINL float4 lds128f(const uint8_t* p) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// 16 bf16 of row `row` of a 128-byte-swizzled tile, chunks 2t and 2t+1
SVDQ_DEVINL void load_row16(const uint8_t* tile, int row, int t, uint32_t (&w)[8]) {
  const int sw = row & 7;
  const uint4 lo = lds128(tile + row * 128 + (((2 * t) ^ sw) << 4));
  const uint4 hi = lds128(tile + row * 128 + (((2 * t + 1) ^ sw) << 4));
  w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
  w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
}

#ifdef SVDQ_QUANT_TRACE
// timeline instrumentation, compiled only into instrumented builds: the first
// 8 CTAs stamp %globaltimer at fixed slots (256 per CTA)
__device__ unsigned long long* g_quant_trace = nullptr;
#define SVDQ_QTR(slot, idx)                                                        \
  do {                                                                             \
    if (g_quant_trace && blockIdx.x < 8 && (idx) < 16)                             \
      g_quant_trace[blockIdx.x * 256 + (slot) + (idx)] = globaltimer_ns();         \
  } while (0)
#else
#define SVDQ_QTR(slot, idx) \
  do {                      \
  } while (0)
#endif

// INT4: the INT4 variant's quantization (64-element groups over the quad,
// bf16 scales [M][K/64] row-major); the rest of the kernel is shared.
template <int RANK, bool INT4>
__global__ void __launch_bounds__(kThreads, 1)
    k_quantize_act(const __grid_constant__ CUtensorMap tm_x,
                   const __grid_constant__ CUtensorMap tm_l1s, const float* __restrict__ inv_lambda,
                   int M, int K, uint8_t* __restrict__ a_codes, uint8_t* __restrict__ a_scales,
                   uint16_t* __restrict__ lora_act, int* dev_status, uint64_t wait_ns) {
  using C = QCfg<RANK>;
  constexpr int NT = C::NT;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kr = warp % kRanges, mt = warp / kRanges;  // K range, m tile
  const int g = lane >> 2, t = lane & 3;
  const int m0 = blockIdx.x * kRows;
  const int steps = K >> 6;
  const int s_begin = (kr * steps) / kRanges;
  const int nst = ((kr + 1) * steps) / kRanges - s_begin;
  uint8_t* xring = smem + C::OFF_X + kr * S * C::X_BYTES;
  uint8_t* lring = smem + C::OFF_L + kr * S * C::L_BYTES;
  uint8_t* iring = smem + C::OFF_INV + kr * S * C::INV_BYTES;
  float2* tab = reinterpret_cast<float2*>(smem + C::OFF_TAB);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR) + kr * 8;
  uint64_t* empty = full + 4;  // both warps of the range have read the slot
  const int C4 = K >> 6;       // 4-column scale groups per row
  const bool producer = mt == 0 && lane == 0;
  // rows of this thread: g and g + 8 of its m tile
  const int rowA = m0 + 16 * mt + g, rowB = rowA + 8;

  if (threadIdx.x == 0) SVDQ_QTR(0, 0);
  if (producer) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
    }
    fence_mbar_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_l1s);
  }
  int issued = 0;  // producer lane only
  auto issue = [&](int i) {
    const int slot = i % S;
    const int k0 = (s_begin + i) * 64;
    mbar_arrive_expect_tx(&full[slot], (uint32_t)C::TX_BYTES);
    tma_load_2d(xring + slot * C::X_BYTES, &tm_x, &full[slot], k0, m0);
    tma_load_2d(lring + slot * C::L_BYTES, &tm_l1s, &full[slot], k0, 0);
    bulk_load(iring + slot * C::INV_BYTES, inv_lambda + k0, (uint32_t)C::INV_BYTES, &full[slot]);
  };
  // two-term reciprocals of the 127 positive e4m3 values (code 0: zeros)
  if (threadIdx.x < 128)
    tab[threadIdx.x] = threadIdx.x == 0 || threadIdx.x == 127
                           ? make_float2(0.0f, 0.0f)
                           : recip2(e4m3_to_f32(threadIdx.x));
  const float2 r6 = recip2(6.0f);
  __syncthreads();  // barriers initialised, table written
  grid_dep_launch();
  grid_dep_wait();  // the previous kernel's outputs (X among them) are complete
  if (producer)
    for (; issued < min(S, nst); ++issued) issue(issued);
  if (threadIdx.x == 0) SVDQ_QTR(1, 0);

  float acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[n][c] = 0.0f;

  int consumed = 0;
  bool aborted = false;
  for (int i = 0; i < nst; ++i) {
    const int slot = i % S;
    const int step = s_begin + i;
    const int k0 = step * 64 + 16 * t;
    const uint32_t ph = (uint32_t)(i / S) & 1u;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[slot], ph, dev_status, wait_ns))) {
      aborted = true;  // warp-uniform abort on timeout
      break;
    }
    if (lane == 0 && warp == 0) SVDQ_QTR(16, i);
    if (lane == 0 && warp == kWarps - 1) SVDQ_QTR(48, i);
    const uint8_t* xt = xring + slot * C::X_BYTES;
    const uint8_t* lt = lring + slot * C::L_BYTES;
    uint32_t xa[8], xb[8];
    load_row16(xt, 16 * mt + g, t, xa);
    load_row16(xt, 16 * mt + g + 8, t, xb);
    uint32_t bfr[NT][8];
#pragma unroll
    for (int n = 0; n < NT; ++n) load_row16(lt, g + 8 * n, t, bfr[n]);
    float inv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 v = lds128f(iring + slot * C::INV_BYTES + 64 * t + 16 * q);
      inv[4 * q] = v.x; inv[4 * q + 1] = v.y; inv[4 * q + 2] = v.z; inv[4 * q + 3] = v.w;
    }
    __syncwarp();
    consumed = i + 1;
    if (lane == 0) mbar_arrive(&empty[slot]);  // this warp is done reading the slot
    if (producer && issued < nst) {
      // refill once the other m tile's warp has read it too
      if (mbar_wait(&empty[slot], ph, dev_status, wait_ns)) {
        fence_proxy_async_smem();
        issue(issued);
        ++issued;
      }
    }
    // ---- down projection: NT n tiles x 4 k16 sub-steps
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int j4 = 0; j4 < 4; ++j4)
        mma_bf16_16816(acc[n], xa[2 * j4], xb[2 * j4], xa[2 * j4 + 1], xb[2 * j4 + 1],
                       bfr[n][2 * j4], bfr[n][2 * j4 + 1]);
    // ---- quantization: one block per row
    uint2 ca, cb;
    uint32_t sa, sb;
    if constexpr (INT4) {
      quant_group64_int4(xa, inv, ca, sa);
      quant_group64_int4(xb, inv, cb, sb);
    } else {
      quant_block16(xa, inv, r6, tab, ca, sa);
      quant_block16(xb, inv, r6, tab, cb, sb);
    }
    if (rowA < M) *reinterpret_cast<uint2*>(a_codes + (size_t)rowA * (K >> 1) + (k0 >> 1)) = ca;
    if (rowB < M) *reinterpret_cast<uint2*>(a_codes + (size_t)rowB * (K >> 1) + (k0 >> 1)) = cb;
    if constexpr (INT4) {
      // the row's 64-group scale (every lane of the quad holds it): lane
      // t = 0 writes row g's, lane t = 1 row g+8's
      if (t < 2) {
        const int r = t == 0 ? rowA : rowB;
        if (r < M)
          reinterpret_cast<uint16_t*>(a_scales)[(size_t)r * (K >> 6) + step] =
              (uint16_t)(t == 0 ? sa : sb);
      }
      if (lane == 0 && warp == 0) SVDQ_QTR(32, i);
      if (lane == 0 && warp == kWarps - 1) SVDQ_QTR(64, i);
      continue;
    }
    // gather the 4 scale bytes of each row's 64-wide step across the quad;
    // lane t = 0 writes row g's word, lane t = 1 row g+8's (tile layout:
    // tile (r/128, c/4) of 512 bytes; entry (r%32)*16 + ((r/32)%4)*4 + c%4)
    uint32_t wa = sa << (8 * t), wb = sb << (8 * t);
    wa |= __shfl_xor_sync(0xFFFFFFFFu, wa, 1);
    wa |= __shfl_xor_sync(0xFFFFFFFFu, wa, 2);
    wb |= __shfl_xor_sync(0xFFFFFFFFu, wb, 1);
    wb |= __shfl_xor_sync(0xFFFFFFFFu, wb, 2);
    if (t < 2) {
      const int r = t == 0 ? rowA : rowB;
      if (r < M) {
        const size_t off =
            ((size_t)(r >> 7) * C4 + step) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
        *reinterpret_cast<uint32_t*>(a_scales + off) = t == 0 ? wa : wb;
      }
    }
    if (lane == 0 && warp == 0) SVDQ_QTR(32, i);
    if (lane == 0 && warp == kWarps - 1) SVDQ_QTR(64, i);
  }
  if (producer && (aborted || consumed < nst || issued < nst)) {
    // timed out: let every copy already issued land before the CTA exits
    for (int i = consumed; i < issued; ++i)
      mbar_wait(&full[i % S], (uint32_t)(i / S) & 1u, nullptr, wait_ns);
  }

  // ---- reduce the K ranges' partial lora sums in a fixed order, round once
  // (the buffer reuses the X ring: every warp is done with it after the barrier)
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem + C::OFF_X);
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int col = 8 * n + 2 * t;
    float* base = red + ((size_t)kr * kRows + 16 * mt + g) * RANK + col;
    base[0] = acc[n][0];
    base[1] = acc[n][1];
    base[8 * RANK] = acc[n][2];
    base[8 * RANK + 1] = acc[n][3];
  }
  __syncthreads();
  if (threadIdx.x == 0) SVDQ_QTR(2, 0);
  for (int idx = threadIdx.x; idx < kRows * RANK; idx += kThreads) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kRanges; ++w) s += red[(size_t)w * kRows * RANK + idx];
    const int rr = m0 + idx / RANK;
    if (rr < M) lora_act[(size_t)m0 * RANK + idx] = f32_to_bf16_rn(s);
  }
}

template <int RANK, bool INT4>
cudaError_t launch_t(const CUtensorMap& tm_x, const CUtensorMap& tm_l1s, const float* inv_lambda,
                     int M, int K, uint8_t* a_codes, uint8_t* a_scales, uint16_t* lora_act,
                     int* dev_status, cudaStream_t stream) {
  using C = QCfg<RANK>;
  auto kern = k_quantize_act<RANK, INT4>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((M + kRows - 1) / kRows, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, tm_x, tm_l1s, inv_lambda, M, K, a_codes, a_scales, lora_act,
                         dev_status, (uint64_t)kWaitTimeoutNs);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_act(const CUtensorMap& tm_x, const CUtensorMap& tm_l1s,
                                const float* inv_lambda, int M, int K, int rank,
                                uint8_t* a_codes, uint8_t* a_scales, uint16_t* lora_act,
                                int* dev_status, cudaStream_t stream, bool int4) {
#define SVDQ_QA_CASE(R_)                                                                  \
  case R_:                                                                                \
    return int4 ? launch_t<R_, true>(tm_x, tm_l1s, inv_lambda, M, K, a_codes, a_scales,  \
                                     lora_act, dev_status, stream)                        \
                : launch_t<R_, false>(tm_x, tm_l1s, inv_lambda, M, K, a_codes, a_scales, \
                                      lora_act, dev_status, stream);
  switch (rank) {
    SVDQ_QA_CASE(16)
    SVDQ_QA_CASE(32)
    SVDQ_QA_CASE(64)
    default:
      return cudaErrorInvalidValue;
  }
#undef SVDQ_QA_CASE
}

}  // namespace svdq

#ifdef SVDQ_QUANT_TRACE
// instrumented builds only: where the first 8 CTAs write their timeline
// (256 x u64 per CTA), or nullptr to stop
extern "C" int svdq_quant_trace_set(unsigned long long* p) {
  return (int)cudaMemcpyToSymbol(svdq::g_quant_trace, &p, sizeof(p));
}
#endif
