// awq_gemv_w4a16: 4-bit weights x bf16 activations for the small-M
// modulation layers (dothoosh.com, "How Nunchaku Lite halves the VRAM of
// diffusion models", kernel-family list: awq_w4a16 serves the memory-bound
// adaLN modulation projections; config block: int4, group_size 64).
//
//   Y[m][n] = bf16( sum_g s[n][g] * ( sum_{k in g} (128 + q[n][k]) x[m][k]
//                                     - (128 + z[n][g]) * sum_{k in g} x[m][k] )
//                   + bias[n] )
//
// which equals sum_k x (q - z) s.  The inner sums run on tensor cores
// (m16n8k16, bf16 in, fp32 out).  The weights are the A operand: 16 rows of a
// tile by 16 k per MMA, every code fed as the exact bf16 value 128 + q (a
// nibble OR-ed into the mantissa of 128.0, 0x4300: one shift and one logic op
// per pair of codes); the constant 128 is folded into the zero point.  The
// activations (M <= 8 rows) are the B operand (N = 8 of the MMA, nothing
// wasted) and stay in registers for the whole kernel: each compute warp of a
// CTA owns a fixed range of at most 4 K groups.  Per 64-group the fp32 sums
// get scale and zero point; sum_{k in g} x[m][k] is formed once per warp.
//
// Streaming.  The weights are read exactly once, by the compute warps
// themselves, kStages tiles ahead of their math with per-thread asynchronous
// copies (cp.async): a warp copies its span of each of the tile's 16 code rows
// (32 bytes per group) in 16-byte pieces, 8 consecutive lanes per 128-byte
// line, into its own shared-memory area (rows of 128 bytes, pieces XOR-ed by
// row % 8, so the fragment reads are conflict-free); each lane also copies
// the scale and zero words of its group.  A lane waits for its own copies and
// the warp synchronises: no CTA-wide barrier.  (Copying 8-byte pieces of 8
// rows per instruction instead left the stream at a third of HBM rate.)  Scale and zero values reach the lanes that need
// them through quad shuffles.  A persistent CTA walks tiles
// blockIdx.x + j * gridDim.x.  The warps leave their fp32 partials in a ring
// of reduction buffers (no CTA-wide barrier); a reduction warp adds the
// partials and the bias in a fixed order and writes Y.
//
// The k order inside an MMA is permuted: a lane feeds 16 consecutive k of a
// group (two 32-bit code words per weight row), paired as (k, k+4) within
// each 8 -- the pairing in which two nibbles of a code word become one bf16x2
// register -- and the activation fragments use the same permutation.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

// compute warps per CTA: CW (12, or 16 when K > 3072), each owning at most
// 4 K groups (one lane of a quad loads the scale words of one group); plus
// one reduction warp
constexpr int kRed = 4;  // reduction buffers (tiles whose partials may be in flight)
constexpr int kStages = 4;  // tiles in flight per lane (cp.async groups)

// nibbles at bit s and s+16 of w -> bf16x2 {128 + q_lo, 128 + q_hi} (exact)
SVDQ_DEVINL uint32_t nib2_biased(uint32_t w, int s) {
  return ((w >> s) & 0x000F000Fu) | 0x43004300u;
}

// bf16 element e (0..15) of the 8 words w
SVDQ_DEVINL uint32_t elem(const uint32_t (&w)[8], int e) {
  return (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
}

SVDQ_DEVINL uint32_t ld_stream_u16(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// shared memory of one warp for one tile: its 16 code rows (128 bytes each,
// 16-byte pieces XOR-ed by row % 8), then per lane the 4-byte words holding the
// scale of group t of rows r, r + 8 (8 bytes), then the same for the zeros
// (lanes t < groups; the fp16 value is the half picked by the index parity)
constexpr int kWarpCodeBytes = 16 * 128;
constexpr int kWarpStageBytes = kWarpCodeBytes + 2 * 32 * 8;
template <int GPW, int CW>
constexpr int awq_smem_bytes() {
  return kStages * CW * kWarpStageBytes;
}

#ifdef SVDQ_AWQ_TRACE
// timeline instrumentation, compiled only into instrumented builds: the first
// 8 CTAs stamp %globaltimer at fixed slots (512 per CTA)
__device__ unsigned long long* g_awq_trace = nullptr;
#define SVDQ_ATR(slot, idx)                                                          \
  do {                                                                               \
    if (g_awq_trace && blockIdx.x < 8 && (idx) < 32)                                 \
      g_awq_trace[blockIdx.x * 512 + (slot) + (idx)] = globaltimer_ns();             \
  } while (0)
#else
#define SVDQ_ATR(slot, idx) \
  do {                      \
  } while (0)
#endif

// GPW: K groups per compute warp at most (ceil(G / CW), 1..4)
template <int GPW, int CW>
__global__ void __launch_bounds__(32 * (CW + 1), 1)
    k_awq_gemv(const uint8_t* __restrict__ qw, const uint16_t* __restrict__ X,
               const uint16_t* __restrict__ sc, const uint16_t* __restrict__ zr,
               const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K,
               int* dev_status, uint64_t wait_ns) {
  static_assert(GPW >= 1 && GPW <= 4, "a quad loads the scale words of at most 4 groups");
  extern __shared__ __align__(128) uint8_t slots[];  // [stage][warp] kWarpStageBytes
  __shared__ __align__(16) float red[kRed][CW][16 * 8];  // [buffer][warp][row * 8 + m]
  __shared__ __align__(8) uint64_t red_full[kRed];        // count CW
  __shared__ __align__(8) uint64_t red_empty[kRed];       // count 1
  __shared__ volatile uint32_t abort_flag;
  const int G = K / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, t = lane & 3;  // MMA group (weight row r / activation m) and quad lane

  const int tiles = (N + 15) >> 4;
  const int my_tiles = blockIdx.x < tiles ? (tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int b = 0; b < kRed; ++b) {
      mbar_init(&red_full[b], CW);
      mbar_init(&red_empty[b], 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  // The weights of this CTA's first tiles are read-only operands: ask L2 for
  // them now (hints only, no data comes back), before the wait for the
  // previous kernel, so that the stream from HBM starts with the launch and
  // the first loads find L2 lines.  (Asking for all of the CTA's tiles at
  // once measured slower: 14.4 against 13.8 us per 57-block launch.)
  constexpr int kPrefetchTiles = 2;
  if (threadIdx.x == 32 * CW) {
    const size_t row_bytes = (size_t)K / 2;
    for (int j = 0; j < my_tiles && j < kPrefetchTiles; ++j) {
      const int n0 = (blockIdx.x + j * gridDim.x) * 16;
      const int rows = min(16, N - n0);
      bulk_prefetch_l2(qw + (size_t)n0 * row_bytes, (uint32_t)(rows * row_bytes));
      const uint32_t gb = (uint32_t)(rows * G * 2) & ~15u;  // whole 16-byte pieces
      if (gb) {
        bulk_prefetch_l2(sc + (size_t)n0 * G, gb);
        bulk_prefetch_l2(zr + (size_t)n0 * G, gb);
      }
    }
  }
  __syncthreads();
  grid_dep_launch();
  grid_dep_wait();  // the previous kernel's outputs (X among them) are complete

  if (warp == CW) {
    // ---------------------------------------------------------- reduction warp
    // the bias values of tile j are fetched three tiles ahead (a register
    // ring), so that their memory latency stays off this warp's path
    auto load_bias = [&](int j, uint32_t (&bv)[4]) {
      const int n0 = (blockIdx.x + j * gridDim.x) * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = (lane + 32 * i) >> 3;
        bv[i] = (bias && j < my_tiles && n0 + row < N) ? ld_stream_u16(bias + n0 + row) : 0u;
      }
    };
    uint32_t bv[4], bv1[4], bv2[4];
    load_bias(0, bv);
    load_bias(1, bv1);
    load_bias(2, bv2);
    for (int j = 0; j < my_tiles; ++j) {
      const int b = j % kRed;
      const int n0 = (blockIdx.x + j * gridDim.x) * 16;
      const bool ok =
          mbar_wait(&red_full[b], (uint32_t)(j / kRed) & 1u, dev_status, wait_ns) && !abort_flag;
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        abort_flag = 1;
        break;
      }
      if (lane == 0) SVDQ_ATR(32, j);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = lane + 32 * i, row = idx >> 3, m = idx & 7;
        if (m < M && n0 + row < N) {
          float s = 0.0f;
#pragma unroll
          for (int w = 0; w < CW; ++w) s += red[b][w][idx];
          s += __uint_as_float(bv[i] << 16);
          Y[(size_t)m * N + n0 + row] = f32_to_bf16_rn(s);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bv[i] = bv1[i];
        bv1[i] = bv2[i];
      }
      load_bias(j + 3, bv2);
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_empty[b]);
      if (lane == 0) SVDQ_ATR(64, j);
    }
    return;
  }

  // ---------------------------------------------------------------- compute warps
  if (lane == 0 && warp == 0) SVDQ_ATR(1, 0);
  // activation fragments of this warp's groups [g_begin, g_begin + ng): lane
  // (r, t) holds x[m = r][64 g + 16 t .. + 15] as the B operand of the 4 MMAs
  // of a group: MMA v takes k pairs (e, e + 4) and (e + 1, e + 5), e = 8 (v/2) + 2 (v%2)
  const int g_begin = (warp * G) / CW, ng = ((warp + 1) * G) / CW - g_begin;
  uint32_t bfr[GPW][8];
  float sx[GPW][2];  // sum over the group's 64 k of x[m] for m = 2t, 2t + 1
#pragma unroll
  for (int gi = 0; gi < GPW; ++gi) {
    uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (gi < ng && r < M) {
      const uint16_t* xp = X + (size_t)r * K + (g_begin + gi) * 64 + 16 * t;
      const uint4 lo = ld_keep_v4(xp), hi = ld_keep_v4(xp + 8);
      w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
      w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
    }
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int e = 8 * (v >> 1) + 2 * (v & 1);
      bfr[gi][2 * v] = elem(w, e) | (elem(w, e + 4) << 16);
      bfr[gi][2 * v + 1] = elem(w, e + 1) | (elem(w, e + 5) << 16);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += bf16lo_to_f32(w[i]) + bf16hi_to_f32(w[i]);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);  // lanes of group r: sum for m = r
    sx[gi][0] = __shfl_sync(0xFFFFFFFFu, s, 8 * t);      // m = 2t
    sx[gi][1] = __shfl_sync(0xFFFFFFFFu, s, 8 * t + 4);  // m = 2t + 1
  }
  if (lane == 0 && warp == 0) SVDQ_ATR(2, 0);

  const size_t row_bytes = (size_t)K / 2;
  // this lane's 16-byte code pieces of a tile: piece q = 32 i + lane is row
  // q / (2 ng), chunk q % (2 ng) of the warp's span (16 rows x 2 ng chunks)
  int pc_row[GPW], pc_src[GPW], pc_dst[GPW];
#pragma unroll
  for (int i = 0; i < GPW; ++i) {
    const int q = 32 * i + lane;
    const int row = q < 32 * ng ? q / (2 * ng) : -1, ch = q - (q / (2 * ng)) * 2 * ng;
    pc_row[i] = row;
    pc_src[i] = 32 * g_begin + 16 * ch;
    pc_dst[i] = row * 128 + ((ch ^ (row & 7)) << 4);
  }
  // asynchronous copies of tile j into stage j % kStages (one commit group per
  // tile, empty past the last tile, so that group counting stays uniform)
  auto issue = [&](int j) {
    if (j < my_tiles) {
      const int n0 = (blockIdx.x + j * gridDim.x) * 16;
      uint8_t* st = slots + (size_t)((j % kStages) * CW + warp) * kWarpStageBytes;
#pragma unroll
      for (int i = 0; i < GPW; ++i) {
        if (pc_row[i] >= 0) {
          const int grow = n0 + pc_row[i];
          cp_async16_cg(st + pc_dst[i], qw + (size_t)min(grow, N - 1) * row_bytes + pc_src[i],
                        grow < N ? 16 : 0);
        }
      }
      if (t < ng) {
        // the 4-byte word holding element i (i & ~1, i | 1): inside the array,
        // whose element count N * G is even
        const int lo_b = n0 + r < N ? 4 : 0, hi_b = n0 + r + 8 < N ? 4 : 0;
        const size_t i_lo = (size_t)min(n0 + r, N - 1) * G + g_begin + t;
        const size_t i_hi = (size_t)min(n0 + r + 8, N - 1) * G + g_begin + t;
        uint32_t* w = reinterpret_cast<uint32_t*>(st + kWarpCodeBytes) + 2 * lane;
        cp_async<4>(w, sc + (i_lo & ~(size_t)1), lo_b);
        cp_async<4>(w + 1, sc + (i_hi & ~(size_t)1), hi_b);
        cp_async<4>(w + 64, zr + (i_lo & ~(size_t)1), lo_b);
        cp_async<4>(w + 65, zr + (i_hi & ~(size_t)1), hi_b);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int a = 0; a < kStages - 1; ++a) issue(a);
  for (int j = 0; j < my_tiles; ++j) {
    issue(j + kStages - 1);
    cp_async_wait<kStages - 1>();  // this lane's copies of tile j have landed
    __syncwarp();                  // ... and every lane's: the code rows are shared
    const int n0 = (blockIdx.x + j * gridDim.x) * 16;
    const uint8_t* st = slots + (size_t)((j % kStages) * CW + warp) * kWarpStageBytes;
    // this lane's scale and zero words (group t of rows r, r + 8) to fp32 once:
    // the value is the half picked by its element index's parity (the same for
    // rows r and r + 8: 8 G is even)
    const uint2 sw = *reinterpret_cast<const uint2*>(st + kWarpCodeBytes + 8 * lane);
    const uint2 zw = *reinterpret_cast<const uint2*>(st + kWarpCodeBytes + 256 + 8 * lane);
    const int sh = ((min(n0 + r, N - 1) * G + g_begin + t) & 1) * 16;
    const float s_lo_own = __half2float(__ushort_as_half((unsigned short)(sw.x >> sh)));
    const float s_hi_own = __half2float(__ushort_as_half((unsigned short)(sw.y >> sh)));
    const float z_lo_own = __half2float(__ushort_as_half((unsigned short)(zw.x >> sh))) + 128.0f;
    const float z_hi_own = __half2float(__ushort_as_half((unsigned short)(zw.y >> sh))) + 128.0f;
    const int b = j % kRed;
    float y[4] = {0.f, 0.f, 0.f, 0.f};  // rows r, r, r+8, r+8; m = 2t, 2t+1, 2t, 2t+1
#pragma unroll
    for (int gi = 0; gi < GPW; ++gi) {
      // the scale and zero of group gi of rows r, r + 8 sit in lane 4 r + gi
      const int src = 4 * r + gi;
      const float s_lo = __shfl_sync(0xFFFFFFFFu, s_lo_own, src);
      const float s_hi = __shfl_sync(0xFFFFFFFFu, s_hi_own, src);
      const float z_lo = __shfl_sync(0xFFFFFFFFu, z_lo_own, src);
      const float z_hi = __shfl_sync(0xFFFFFFFFu, z_hi_own, src);
      if (gi < ng) {
        // bytes 32 gi + 8 t of the warp's span in rows r and r + 8
        const uint8_t* cp = st + (((2 * gi + (t >> 1)) ^ r) << 4) + (t & 1) * 8;
        const uint2 cw0 = *reinterpret_cast<const uint2*>(cp + r * 128);
        const uint2 cw1 = *reinterpret_cast<const uint2*>(cp + (r + 8) * 128);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t c0 = (v >> 1) ? cw0.y : cw0.x;
          const uint32_t c1 = (v >> 1) ? cw1.y : cw1.x;
          const int s0 = 8 * (v & 1);
          mma_bf16_16816(d, nib2_biased(c0, s0), nib2_biased(c1, s0), nib2_biased(c0, s0 + 4),
                         nib2_biased(c1, s0 + 4), bfr[gi][2 * v], bfr[gi][2 * v + 1]);
        }
        y[0] = __fmaf_rn(s_lo, __fmaf_rn(-z_lo, sx[gi][0], d[0]), y[0]);
        y[1] = __fmaf_rn(s_lo, __fmaf_rn(-z_lo, sx[gi][1], d[1]), y[1]);
        y[2] = __fmaf_rn(s_hi, __fmaf_rn(-z_hi, sx[gi][0], d[2]), y[2]);
        y[3] = __fmaf_rn(s_hi, __fmaf_rn(-z_hi, sx[gi][1], d[3]), y[3]);
      }
    }
    // partials of tile j into buffer b once the reduction warp has read it
    bool ok = mbar_wait(&red_empty[b], ((uint32_t)(j / kRed) & 1u) ^ 1u, dev_status, wait_ns) &&
              !abort_flag;
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      abort_flag = 1;
      break;
    }
    if (lane == 0 && warp == 0) SVDQ_ATR(96, j);
    *reinterpret_cast<float2*>(&red[b][warp][r * 8 + 2 * t]) = make_float2(y[0], y[1]);
    *reinterpret_cast<float2*>(&red[b][warp][(r + 8) * 8 + 2 * t]) = make_float2(y[2], y[3]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&red_full[b]);
    if (lane == 0 && warp == 0) SVDQ_ATR(160, j);
  }
  cp_async_wait<0>();  // nothing may land in shared memory after the CTA exits
}

}  // namespace

int awq_max_k() { return 4096; }  // 16 compute warps x 4 groups x 64

cudaError_t launch_awq_gemv(const uint8_t* qweight, const uint16_t* X, const uint16_t* scales,
                            const uint16_t* zeros, const uint16_t* bias, uint16_t* Y, int M,
                            int N, int K, int* dev_status, cudaStream_t stream, int num_sms) {
  if (K > awq_max_k() || K % 64 != 0) return cudaErrorInvalidValue;
  const int G = K / 64;
  void (*kern)(const uint8_t*, const uint16_t*, const uint16_t*, const uint16_t*,
               const uint16_t*, uint16_t*, int, int, int, int*, uint64_t) = nullptr;
  int smem = 0, threads = 0;
#define SVDQ_AWQ_CASE(GPW_, CW_)                  \
  {                                               \
    kern = k_awq_gemv<GPW_, CW_>;                 \
    smem = awq_smem_bytes<GPW_, CW_>();           \
    threads = 32 * (CW_ + 1);                     \
  }
  if (G <= 12) SVDQ_AWQ_CASE(1, 12)
  else if (G <= 24) SVDQ_AWQ_CASE(2, 12)
  else if (G <= 36) SVDQ_AWQ_CASE(3, 12)
  else if (G <= 48) SVDQ_AWQ_CASE(4, 12)  // K = 3072: one 128-byte line per warp and row
  else SVDQ_AWQ_CASE(4, 16)
#undef SVDQ_AWQ_CASE
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles = (N + 15) / 16;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles < num_sms ? tiles : num_sms, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, qweight, X, scales, zeros, bias, Y, M, N, K, dev_status,
                         (uint64_t)kWaitTimeoutNs);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace svdq

#ifdef SVDQ_AWQ_TRACE
// instrumented builds only: where the first 8 CTAs write their timeline
// (512 x u64 per CTA), or nullptr to stop
extern "C" int svdq_awq_trace_set(unsigned long long* p) {
  return (int)cudaMemcpyToSymbol(svdq::g_awq_trace, &p, sizeof(p));
}
#endif
