// svdq_gemm_w4a4: the 4-bit product of the SVDQ W4A4 linear with the
// low-rank up projection and the bias fused into it (dothoosh.com, "How
// Nunchaku Lite halves the VRAM of diffusion models", fused-kernel paragraph:
// the up projection is fused with the 4-bit compute kernel).
//
//   acc  = sum_k dec(a)[m][k] dec(w)[n][k]            tcgen05 kind::mxf4nvf4,
//          + sum_i lora[m][i] L2s[n][i]                 then kind::f16 (bf16),
//                                                     one fp32 TMEM accumulator
//   Y    = bf16( s_T * acc + bias[n] )        with L2s = L2 / s_T (exact: s_T is
//                                             a power of two)
//   or H = bf16( gelu_tanh(Y) )               the GELU variant, for the first
//                                             linear of a transformer MLP
//                                             (dothoosh.com, same article: the
//                                             full engine's GELU/MLP kernels)
//   or the QKV variant: Y's Q and K heads (128 columns each) RMS-normalized
//      and turned pair by pair by the tokens' rotary angles, V as Y (same
//      article, structural rewrites: one fused operator for the QKV
//      projection, the Q/K normalization and the rotary embeddings)
//   or the GELU + quantization variant: H as the GELU variant, quantized as
//      the next linear's input (its e2m1 codes and e4m3 scales, with its
//      inv_lambda) and multiplied by the next linear's L1s on the tensor
//      cores (its low-rank down projection, summed per CTA pair over the
//      pair's run of tiles of one 256-row block; a second kernel adds the
//      runs), H written only on request (same article, the full engine's
//      GELU/MLP kernels; the fused-kernel paragraph: down projection with
//      the quantization)
//
// Persistent kernel in clusters of two CTAs (one CTA per SM) that compute
// together with the tensor cores' CTA-pair MMAs (tcgen05 cta_group::2).  A
// pair walks 256 x BN output tiles (BN = 256, or 128 when N is not a multiple
// of 256), N fastest.  One M = 256 MMA covers the pair's tile: CTA rank c
// holds output rows 128c .. 128c + 127 in its TMEM, its own 128 A rows and
// one half of the tile's W rows (BN/2 of them) in its shared memory; the
// tensor cores of the two SMs exchange the W halves themselves.  So every
// byte a CTA loads is its own: per SM a k tile moves 38 KB (A 16 KB, W half
// 16 KB, block scales 6 KB) for the same 16.8 MFLOP that a lone 128 x 256
// tile would need 54 KB for.
//
// Each CTA's ring (4 slots of 38 KB at BN = 256; 5 for the QKV variant, whose
// epilogue needs no staging area) carries, per output tile,
// its k tiles -- A code tile and its scale chunk, the CTA's half of the W code
// rows, and the scale chunks of all BN W rows (both halves: the MMA of each
// SM needs every column's scales in its own TMEM); 128-byte rows, 128B
// swizzle; the scale layout is already the tensor core's, so scales move as
// plain bulk copies -- and then one slot with the tile's rank-r operands
// (lora rows in the A area, the CTA's half of the L2s rows in the B area,
// K-major, swizzled TMA boxes) plus the tile's bias slice (into a separate
// double buffer that the epilogue releases).
//
// Warp roles (22 warps per CTA; a warp reaches TMEM lanes 32 * (warp % 4)):
//   warp 0     one lane: the producer of this CTA's ring, running ahead
//              across tiles;
//   warp 1     allocates TMEM (collectively with the peer); in the even CTA
//              one lane issues the pair MMAs of each k tile, then the rank-r
//              MMAs into the same accumulator; tcgen05.commit frees the ring
//              slots of both CTAs and finally signals `acc_full` in both;
//   warps 2-5  scale warps, one per TMEM lane quarter: for each k tile they
//              move the block scales from shared memory into this CTA's TMEM
//              with tcgen05.st (registers -> TMEM), keeping that traffic off
//              the MMA issue path, and report to the even CTA's `sf_full`
//              (that report also tells the issuer that this CTA's slot has
//              landed);
//   warps 6-21 the epilogue, four per TMEM lane quarter (one output row per
//              lane, BN/4 columns each): one tcgen05.ld of their columns, and
//              the even CTA's `acc_empty` is told at once -- the single
//              accumulator is held only for that load; then y = s_T * acc +
//              bias rounded to bf16 pairs (QKV: the two warps holding the
//              halves of a head swap their rows' partial sums of squares
//              through shared memory behind a two-warp barrier, then
//              normalize and rotate), and an 8 x 8 (4 x 4 at BN = 128)
//              transpose of 16-byte chunks inside groups of lanes (warp
//              shuffles) turns "one row per lane" into "8 lanes per row": each
//              store instruction writes 4 whole 128-byte row segments.
//
// Block scales in TMEM.  Per 64-wide K step, the 128 x 4 scale chunk of A
// (512 bytes, row r at byte (r%32)*16 + (r/32)*4) occupies 4 columns: every
// lane quarter holds, in lane l, column j, the 4 scales of row l + 32j (the
// layout of tcgen05.cp.32x128b.warpx4).  A scale warp loads chunk row l (16
// bytes) and stores it with one tcgen05.st.32x32b.x4.  B's BN rows take BN/32
// columns the same way, in each CTA of the pair.
//
// Cross-CTA signals are plain mbarrier arrivals on shared::cluster addresses
// (mapa) and tcgen05.commit to each CTA's barrier in turn; no data moves
// between the two shared memories except through the pair MMA.
//
// Every wait is bounded: on timeout the kernel reports SVDQ_DEV_TIMEOUT,
// tells the peer CTA to stop too, stops issuing work, lets the copies and MMAs
// in flight land, frees TMEM and returns.
#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>

#include "act_quant.cuh"
#include "device_common.cuh"
#include "launch.h"

namespace svdq {

namespace {

constexpr int BM = 128;              // output rows per CTA (TMEM lanes); a pair covers 256
constexpr int BK_BYTES = 128;        // one k tile: 256 fp4 values per row
constexpr int KB_PER_TILE = 4;       // 64-wide MMA steps per k tile
constexpr int NUM_THREADS = 22 * 32;
constexpr int SF_WARP0 = 2;   // warps 2..5
constexpr int EPI_WARP0 = 6;  // warps 6..21
constexpr int EPI_WARPS = 16;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_LIMIT = 227 * 1024;  // dynamic shared memory of one CTA
constexpr int kMaxDevices = 64;
// GELU + quantization: at most this many CTA pairs (the scratch holds
// kGqMaxPairs + ceil(M / 256) slots of segment sums)
constexpr int kGqMaxPairs = 128;

constexpr int cmin(int a, int b) { return a < b ? a : b; }

// epilogue kinds: bf16 Y; bf16 gelu_tanh(Y); Y with its Q and K heads
// RMS-normalized and rotated (fused QKV projection)
constexpr int kEpiPlain = 0, kEpiGelu = 1, kEpiQkv = 2, kEpiGeluQuant = 3;
constexpr int kHeadDim = 128;  // QKV epilogue: channels of one head

// RANK2: rank of the next layer's down projection (GELU + quantization
// epilogue only; 0 for the others)
template <int BN, int RANK, int EPI, int RANK2 = 0>
struct Cfg {
  static constexpr int BH = BN / 2;  // W rows held by one CTA of the pair
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = BH * BK_BYTES;
  static constexpr int SFA_BYTES = KB_PER_TILE * 512;
  static constexpr int SFB_BYTES = KB_PER_TILE * 512 * (BN / 128);  // all BN rows
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int LROW = RANK * 2;  // bytes of one rank-r row (bf16)
  static constexpr int LA_BYTES = BM * LROW;
  static constexpr int LB_BYTES = BH * LROW;
  static_assert(LA_BYTES <= A_BYTES && LB_BYTES <= B_BYTES, "rank-r operands fit a ring slot");
  static constexpr int BIAS_BYTES = BN * 2;
  // QKV: per-lane partial sums of squares exchanged by the two warps of a head
  // (two buffers), and one barrier per warp pair
  static constexpr int XSUM_BYTES = EPI == kEpiQkv ? 2 * 16 * 32 * 4 : 0;
  static constexpr int PAIR_BARS = EPI == kEpiQkv ? 8 : 0;
  static constexpr int EPI_COLS = BN / 4;     // columns per epilogue warp
  static constexpr int EPI_CH = EPI_COLS / 8;  // 16-byte output chunks per row and warp
  // plain and GELU epilogues: each warp stages its 32 x EPI_COLS bf16 block in
  // shared memory (the swizzled layout of the output tensor map) and stores it
  // with one TMA store; QKV stores from registers after a lane transpose
  static constexpr bool TMA_OUT = EPI != kEpiQkv;
  static constexpr int OUT_ROW_BYTES = EPI_COLS * 2;                 // 128 or 64
  static constexpr int OUT_WARP_BYTES = 32 * OUT_ROW_BYTES;
  static constexpr int OUT_BYTES = TMA_OUT ? EPI_WARPS * OUT_WARP_BYTES : 0;
  // GELU + quantization: per tile this CTA's half of the next layer's L1s
  // slice (rank2/2 rows x BN columns, [BN/64 chunks][rows][64], 128B swizzle:
  // the B operand of the down-projection MMAs, whose A operand is the staged H
  // tile) and the e4m3 reciprocal table of the quantization.  The per-tile
  // slices (bias, L1s) are single-buffered there, so that four ring stages fit.
  static constexpr bool GQ = EPI == kEpiGeluQuant;
  static constexpr int R2H = RANK2 / 2;
  static constexpr int L1S2_BYTES = GQ ? (BN / 64) * R2H * 128 : 0;
  static constexpr int TAB_BYTES = GQ ? 128 * 8 : 0;
  static constexpr int EBUF = GQ ? 1 : 2;  // buffers of the per-tile epilogue slices
  static constexpr int FIXED_BYTES =
      OUT_BYTES + L1S2_BYTES + TAB_BYTES + EBUF * BIAS_BYTES + XSUM_BYTES;
  // barriers: full[S], empty[S], sf_full[S], bias_empty[2], acc_full,
  // acc_empty, mma_done, pair[PAIR_BARS], and for GELU + quantization h_ready,
  // l2q_full, l2q_empty, l1s2_empty
  static constexpr int GQ_BARS = GQ ? 4 : 0;
  static constexpr int BAR_BYTES_MAX = (3 * 6 + 5 + PAIR_BARS + GQ_BARS) * 8;
  // TMEM columns: accumulator [0, BN), then per stage the scales of A and B
  static constexpr int SF_COLS_A = 4 * KB_PER_TILE;
  static constexpr int SF_COLS_B = 4 * KB_PER_TILE * (BN / 128);
  static constexpr int SF_STAGE_COLS = SF_COLS_A + SF_COLS_B;
  static constexpr int SF_BASE = BN;
  // ring depth: what shared memory (less the fixed areas, the barriers, 16
  // bytes of flags and 1024 bytes of base-alignment slack) and TMEM hold
  static constexpr int STAGES =
      cmin(cmin(6, (SMEM_LIMIT - 1024 - 16 - BAR_BYTES_MAX - FIXED_BYTES) / STAGE_BYTES),
           ((int)TMEM_COLS - SF_BASE - RANK2) / SF_STAGE_COLS);
  // GELU + quantization: the down-projection accumulator after the scales
  static constexpr int L2Q_COL = SF_BASE + STAGES * SF_STAGE_COLS;
  static constexpr int OFF_A = 0;  // slot areas 1024-aligned (swizzle atoms)
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_OUT = OFF_SFB + STAGES * SFB_BYTES;  // 1024-aligned
  static constexpr int OFF_L1S2 = OFF_OUT + OUT_BYTES;  // 1024-aligned
  static constexpr int OFF_TAB = OFF_L1S2 + L1S2_BYTES;
  static constexpr int OFF_BIAS = OFF_TAB + TAB_BYTES;
  static constexpr int OFF_XSUM = OFF_BIAS + EBUF * BIAS_BYTES;
  static constexpr int OFF_BAR = OFF_XSUM + XSUM_BYTES;
  static constexpr int NUM_BARS = 3 * STAGES + 5 + PAIR_BARS + GQ_BARS;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + base alignment slack
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert(SF_BASE + STAGES * SF_STAGE_COLS + RANK2 <= (int)TMEM_COLS, "TMEM budget");
  static_assert(!GQ || (BN == 256 && (RANK2 == 32 || RANK2 == 64)),
                "GELU + quantization: 256-column tiles, next-layer rank 32 or 64");
  static_assert(OFF_L1S2 % 1024 == 0 && (L1S2_BYTES / (BN / 64 > 0 ? BN / 64 : 1)) % 1024 == 0,
                "L1s2 chunks keep the swizzle atoms aligned");
  // the down-projection MMAs of the next layer: kind::f16 bf16, M = 256 over
  // the pair, N = RANK2
  static constexpr uint32_t IDESC_L2Q = (1u << 4) | (1u << 7) | (1u << 10) |
                                        ((uint32_t)(RANK2 >> 3) << 17) |
                                        ((uint32_t)((2 * BM) >> 4) << 24);
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  static_assert(B_BYTES % 1024 == 0, "W half tiles keep the 1024-byte swizzle atoms aligned");
  static constexpr SmemLayout LSW =
      LROW == 128 ? kSwizzle128B : (LROW == 64 ? kSwizzle64B : kSwizzle32B);
  // instruction descriptors of the pair MMAs (kind::mxf4nvf4: E2M1 x E2M1,
  // UE4M3 scales, K-major, M = 256 over the pair, N = BN; kind::f16: bf16 x
  // bf16 -> f32)
  static constexpr uint32_t IDESC_NVF4 = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                         ((uint32_t)((2 * BM) >> 4) << 24);
  static constexpr uint32_t IDESC_BF16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                         ((uint32_t)(BN >> 3) << 17) |
                                         ((uint32_t)((2 * BM) >> 4) << 24);
  static_assert(OFF_OUT % 1024 == 0, "staging areas keep the swizzle atoms aligned");
};

#ifdef SVDQ_GEMM_TRACE
// timeline instrumentation, compiled only into instrumented builds: the first
// 8 CTAs stamp %globaltimer at fixed slots (1024 per CTA)
__device__ unsigned long long* g_gemm_trace = nullptr;
#define SVDQ_TR_SETUP unsigned long long* const trace_ = g_gemm_trace
#define SVDQ_TR(slot, lim, idx)                                                   \
  do {                                                                            \
    if (trace_ && blockIdx.x < 8 && (idx) < (lim))                                \
      trace_[blockIdx.x * 1024 + (slot) + (idx)] = globaltimer_ns();              \
  } while (0)
#else
#define SVDQ_TR_SETUP \
  do {                \
  } while (0)
#define SVDQ_TR(slot, lim, idx) \
  do {                          \
  } while (0)
#endif

SVDQ_DEVINL float ex2_approx(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}

SVDQ_DEVINL float rcp_approx(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// GELU in its tanh form, 0.5 y (1 + tanh(u)) with u = sqrt(2/pi) (y + 0.044715
// y^3), for finite y.  0.5 (1 + tanh(u)) is the logistic function of 2u, so the
// value is y / (1 + 2^t) with t = -2 u log2(e) = y (c1 + c2 y^2): no 1 + tanh
// cancellation for negative y, no overflow (2^t = inf gives y * 0).  Relative
// error about 2^-21 + |t| 2^-23 (ex2 and rcp approximations, 5 roundings),
// far below a bf16 half-ulp where the value is not negligible.
SVDQ_DEVINL float gelu_tanh_f32(float y) {
  constexpr float c1 = -2.302208198144325f;   // -2 sqrt(2/pi) log2(e)
  constexpr float c2 = -0.1029432395800235f;  // c1 * 0.044715
  const float t = y * __fmaf_rn(c2, y * y, c1);
  return y * rcp_approx(1.0f + ex2_approx(t));
}

// y = s_T * acc + bias for 32 accumulator columns (raw fp32 bits in v), as 16
// bf16 pairs (round to nearest even); bias: 32 bf16 in shared memory or nullptr
// (out may alias v: element i of out is written after v[2i], v[2i+1] are read).
// GELU: the pairs hold bf16(gelu(y_b)) of the rounded y_b instead, the value
// an unfused GELU would compute on the bf16 output of this layer.
template <bool GELU>
SVDQ_DEVINL void pack_cols32(const uint32_t* v, float s_T, const uint16_t* bias, uint32_t* out) {
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {
    uint4 bw = make_uint4(0u, 0u, 0u, 0u);
    if (bias) bw = lds128(bias + 8 * c8);
    const uint32_t bb[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 8 * c8 + 2 * i;
      const float y0 = __fmaf_rn(s_T, __uint_as_float(v[e]), bf16lo_to_f32(bb[i]));
      const float y1 = __fmaf_rn(s_T, __uint_as_float(v[e + 1]), bf16hi_to_f32(bb[i]));
      __nv_bfloat162 p = __floats2bfloat162_rn(y0, y1);  // .x (low half) = y0
      if constexpr (GELU) {
        const float2 yb = __bfloat1622float2(p);
        p = __floats2bfloat162_rn(gelu_tanh_f32(yb.x), gelu_tanh_f32(yb.y));
      }
      out[4 * c8 + i] = *reinterpret_cast<const uint32_t*>(&p);
    }
  }
}

// QKV epilogue, after the 8 x 8 chunk transpose: lane t holds, for the 8 rows
// row0 + i (i = 0..7, words pk[4i .. 4i+3]), the 8 columns 8 (t % 8) .. + 7 of
// its warp's 64, i.e. the head channels whose weights start at w and the 4
// channel pairs starting at pair p.  rs_lane is 1/rms of the row the lane held
// before the transpose (row gbase + i comes by a shuffle).  n = (y * rs) * w,
// then pair (a, b) turned by the token's angle: (a cos - b sin, a sin + b cos),
// rounded to bf16 pairs in place.  The 8 lanes sharing a row read its table
// slices side by side (128 contiguous bytes).  One row per iteration, not
// unrolled, so that the table loads are not all held in registers at once:
// the rows rotate through pk[0..3] and are back in place after 8.
SVDQ_DEVINL void qkv_rotate_rows(uint32_t (&pk)[32], float rs_lane, int gbase, const uint16_t* w,
                                 const float* rope_cos, const float* rope_sin, int row0, int M,
                                 int p) {
  const uint4 ww = __ldg(reinterpret_cast<const uint4*>(w));
  const uint32_t wp[4] = {ww.x, ww.y, ww.z, ww.w};
#pragma unroll 1
  for (int i = 0; i < 8; ++i) {
    const float rs = __shfl_sync(0xFFFFFFFFu, rs_lane, gbase + i);
    const size_t off = (size_t)min(row0 + i, M - 1) * (kHeadDim / 2) + p;
    const float4 co = __ldg(reinterpret_cast<const float4*>(rope_cos + off));
    const float4 si = __ldg(reinterpret_cast<const float4*>(rope_sin + off));
    const float cc[4] = {co.x, co.y, co.z, co.w}, sv[4] = {si.x, si.y, si.z, si.w};
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = (bf16lo_to_f32(pk[j]) * rs) * bf16lo_to_f32(wp[j]);
      const float b = (bf16hi_to_f32(pk[j]) * rs) * bf16hi_to_f32(wp[j]);
      const __nv_bfloat162 o = __floats2bfloat162_rn(__fmaf_rn(a, cc[j], -(b * sv[j])),
                                                     __fmaf_rn(a, sv[j], b * cc[j]));
      out[j] = *reinterpret_cast<const uint32_t*>(&o);
    }
#pragma unroll
    for (int k = 0; k < 28; ++k) pk[k] = pk[k + 4];
#pragma unroll
    for (int j = 0; j < 4; ++j) pk[28 + j] = out[j];
  }
}

// Inside each group of CH lanes (CH = 8 or 4), transpose the CH x CH matrix of
// 16-byte chunks (lane = row, chunk index = column): afterwards chunk i of
// lane t holds what was chunk t % CH of lane (t & ~(CH-1)) + i.  log2(CH)
// exchange steps; step d swaps the chunks whose row and column differ in bit d.
template <int CH>
SVDQ_DEVINL void transpose_chunks(uint32_t (&c)[4 * CH], int lane) {
#pragma unroll
  for (int d = 1; d < CH; d <<= 1) {
    const bool hi = (lane & d) != 0;
#pragma unroll
    for (int p = 0; p < CH; ++p) {
      if (p & d) continue;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t lo_w = c[4 * p + k], hi_w = c[4 * (p | d) + k];
        const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, hi ? lo_w : hi_w, d);
        c[4 * p + k] = hi ? got : lo_w;
        c[4 * (p | d) + k] = hi ? hi_w : got;
      }
    }
  }
}

template <int BN, int RANK, int EPI, int RANK2>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_w4a4(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_lora,
                const __grid_constant__ CUtensorMap tm_l2s,
                const __grid_constant__ CUtensorMap tm_y,
                const __grid_constant__ CUtensorMap tm_l1s2, const uint8_t* __restrict__ a_scales,
                const uint8_t* __restrict__ w_scales, float s_T,
                const uint16_t* __restrict__ bias, uint16_t* __restrict__ Y, int M, int N, int K,
                const QkvEpilogue qe, const GeluQuantEpilogue gq, int* dev_status, int test_stall,
                uint64_t wait_ns) {
  static_assert(EPI != kEpiQkv || BN == 2 * kHeadDim, "QKV epilogue: two heads per tile");
  using C = Cfg<BN, RANK, EPI, RANK2>;
  constexpr bool GQ = C::GQ;
  constexpr int STAGES = C::STAGES;
  SVDQ_TR_SETUP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_full = empty + STAGES;       // used in the even CTA
  uint64_t* bias_empty = sf_full + STAGES;  // [2]
  uint64_t* acc_full = bias_empty + 2;
  uint64_t* acc_empty = acc_full + 1;       // used in the even CTA
  uint64_t* mma_done = acc_empty + 1;       // used in the even CTA
  uint64_t* pair_bar = mma_done + 1;        // [PAIR_BARS]
  // GELU + quantization: H staged (even CTA; both CTAs' epilogue warps), the
  // next layer's down projection of a tile done (both CTAs), its accumulator
  // read at the end of a segment (even CTA; the 4 reading warps of both CTAs),
  // the L1s2 buffer free (both CTAs)
  uint64_t* h_ready = pair_bar + C::PAIR_BARS;
  uint64_t* l2q_full = h_ready + 1;
  uint64_t* l2q_empty = l2q_full + 1;
  uint64_t* l1s2_empty = l2q_empty + 1;
  constexpr int EBUF = C::EBUF;  // bias slice buffers
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);  // [0] tmem, [1] abort
  volatile uint32_t* abort_flag = &misc[1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();  // 0 (issues the pair MMAs) or 1
  const int kb_total = K >> 6;               // 64-wide steps
  const int k_tiles = (kb_total + KB_PER_TILE - 1) / KB_PER_TILE;
  const int n_tiles = N / BN;
  const int m_tiles = (M + BM - 1) / BM;
  const int num_ptiles = ((m_tiles + 1) / 2) * n_tiles;  // 256-row pair tiles
  const int pair = (int)blockIdx.x >> 1, n_pairs = (int)gridDim.x >> 1;
  // Pair tiles pt (m pair pt / n_tiles, n tile pt % n_tiles) are dealt out
  // round robin; with GELU + quantization each pair takes one contiguous range
  // of them instead, [pt_begin, pt_begin + my_tiles), so that the next
  // layer's down projection accumulates in TMEM over the n tiles of one m
  // pair (a segment) and is written out once per segment.
  int pt_begin = pair, my_tiles = 0;
  if constexpr (GQ) {
    pt_begin = (int)((long long)pair * num_ptiles / n_pairs);
    my_tiles = (int)((long long)(pair + 1) * num_ptiles / n_pairs) - pt_begin;
  } else {
    my_tiles = pair < num_ptiles ? (num_ptiles - 1 - pair) / n_pairs + 1 : 0;
  }
  auto tile_pt = [&](int j) { return GQ ? pt_begin + j : pair + j * n_pairs; };
  // tile j of this CTA: m tile 2 * (pt / n_tiles) + crank (may lie past M when
  // m_tiles is odd: it is computed on zero-filled rows and not stored)
  auto tile_mn = [&](int j, int& m_tile, int& n_tile) {
    const int pt = tile_pt(j);
    m_tile = 2 * (pt / n_tiles) + (int)crank;
    n_tile = pt % n_tiles;
  };
  // GELU + quantization: first / last tile of a segment
  auto seg_first = [&](int j) { return j == 0 || tile_pt(j) % n_tiles == 0; };
  auto seg_last = [&](int j) { return j == my_tiles - 1 || (tile_pt(j) + 1) % n_tiles == 0; };
  // the even CTA's copy of a barrier, as a shared::cluster address
  auto at_even = [](uint64_t* bar) { return cluster_map(smem_u32(bar), 0u); };
  // stop this CTA and tell the peer to stop too (its waits would otherwise
  // run into their own bounds one after another)
  auto abort_pair = [&]() {
    *abort_flag = 1;
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(
                     cluster_map(smem_u32(&misc[1]), crank ^ 1u)),
                 "r"(1u)
                 : "memory");
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);     // the even CTA's MMA commit
      mbar_init(&sf_full[s], 8);   // the 4 scale warps of each CTA of the pair
    }
    for (int b = 0; b < EBUF; ++b) mbar_init(&bias_empty[b], EPI_WARPS);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * EPI_WARPS);  // the epilogue warps of both CTAs
    mbar_init(mma_done, 1);
    for (int b = 0; b < C::PAIR_BARS; ++b) mbar_init(&pair_bar[b], 2);
    if (GQ) {
      mbar_init(h_ready, 2 * EPI_WARPS);
      mbar_init(l2q_full, 1);
      mbar_init(l2q_empty, 8);  // warps 0-3 of the epilogue, both CTAs
      mbar_init(l1s2_empty, 1);
    }
    misc[1] = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_lora);
    prefetch_tmap(&tm_l2s);
    if (C::TMA_OUT && (!GQ || gq.h_out)) prefetch_tmap(&tm_y);  // (no H: an unused map)
    if (GQ) prefetch_tmap(&tm_l1s2);
  }
  if (GQ && threadIdx.x < 128) {
    // two-term reciprocals of the 127 positive e4m3 values (code 0: zeros)
    const float2 v = threadIdx.x == 0 || threadIdx.x == 127 ? make_float2(0.0f, 0.0f)
                                                            : recip2(e4m3_to_f32(threadIdx.x));
    *reinterpret_cast<float2*>(smem + C::OFF_TAB + 8 * threadIdx.x) = v;
  }
  // both CTAs resident and their barriers initialised before the collective
  // TMEM allocation and before any arrival from the peer
  cluster_sync();
  if (warp == 1) tmem_alloc_pair(&misc[0], TMEM_COLS);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  grid_dep_launch();
  // The weight side is no output of the previous kernel: ask L2 for this
  // CTA's half of the first tile's W rows and their scales now (hints only),
  // while that kernel may still run.
  if (warp == 0 && lane == 0 && my_tiles > 0) {
    int m_tile, n_tile;
    tile_mn(0, m_tile, n_tile);
    const int n0 = n_tile * BN, nh = n0 + (int)crank * C::BH;
    const int kp = min(k_tiles, 2 * STAGES);
    for (int kt = 0; kt < kp; ++kt) tma_prefetch_2d(&tm_b, kt * BK_BYTES, nh);
    for (int h = 0; h < BN / 128; ++h)
      bulk_prefetch_l2(w_scales + (size_t)(n0 / 128 + h) * kb_total * 512,
                       (uint32_t)(min(kb_total, kp * KB_PER_TILE) * 512));
  }
  grid_dep_wait();  // the previous kernel's outputs (our inputs) are complete

  int issued = 0;  // producer lane only: ring slots filled
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !test_stall) {
      for (int j = 0; j < my_tiles && !*abort_flag; ++j) {
        int m_tile, n_tile;
        tile_mn(j, m_tile, n_tile);
        const bool m_valid = m_tile < m_tiles;
        const int m0 = m_tile * BM, n0 = n_tile * BN;
        const int nh = n0 + (int)crank * C::BH;  // this CTA's half of the W rows
        for (int kt = 0; kt <= k_tiles; ++kt) {  // k tiles, then the rank-r slot
          const int s = issued % STAGES;
          const uint32_t ph = (uint32_t)(issued / STAGES) & 1u;
          if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1u, dev_status, wait_ns)) {
            abort_pair();
            break;
          }
          SVDQ_TR(832, 128, issued);
          uint8_t* sa = smem + C::OFF_A + s * C::A_BYTES;
          uint8_t* sb = smem + C::OFF_B + s * C::B_BYTES;
          if (kt == k_tiles) {
            // rank-r operands of tile j (own rows, own half of L2s) and its
            // bias slice (all BN columns: this CTA stores every column)
            // (GELU + quantization: also this CTA's half of the next layer's
            // L1s slice)
            if (bias && !mbar_wait(&bias_empty[j % EBUF], (uint32_t)((j / EBUF) & 1) ^ 1u,
                                   dev_status, wait_ns)) {
              abort_pair();
              break;
            }
            // (GELU + quantization: the previous tile's down projection has
            // read the L1s2 buffer)
            if (GQ && !mbar_wait(l1s2_empty, (uint32_t)(j & 1) ^ 1u, dev_status, wait_ns)) {
              abort_pair();
              break;
            }
            mbar_arrive_expect_tx(&full[s], (uint32_t)(C::LA_BYTES + C::LB_BYTES +
                                                       (bias ? C::BIAS_BYTES : 0) +
                                                       C::L1S2_BYTES));
            tma_load_2d(sa, &tm_lora, &full[s], 0, m0);
            tma_load_2d(sb, &tm_l2s, &full[s], 0, nh);
            if (bias)
              bulk_load(smem + C::OFF_BIAS + (j % EBUF) * C::BIAS_BYTES, bias + n0,
                        (uint32_t)C::BIAS_BYTES, &full[s]);
            if (GQ) {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_2d(smem + C::OFF_L1S2 + c * (C::R2H * 128), &tm_l1s2, &full[s],
                            n0 + 64 * c, (int)crank * C::R2H);
            }
            SVDQ_TR(424, 8, j);
          } else {
            const int nkb = min(KB_PER_TILE, kb_total - kt * KB_PER_TILE);
            // this CTA's A tile (+ its scales, rows inside M), its half of the
            // W rows, and the scales of all BN W rows
            const uint32_t bytes = (uint32_t)(C::A_BYTES + C::B_BYTES +
                                              nkb * 512 * ((m_valid ? 1 : 0) + BN / 128));
            mbar_arrive_expect_tx(&full[s], bytes);
            tma_load_2d(sa, &tm_a, &full[s], kt * BK_BYTES, m0);
            tma_load_2d(sb, &tm_b, &full[s], kt * BK_BYTES, nh);
            if (m_valid)
              bulk_load(smem + C::OFF_SFA + s * C::SFA_BYTES,
                        a_scales + ((size_t)m_tile * kb_total + (size_t)kt * KB_PER_TILE) * 512,
                        (uint32_t)nkb * 512u, &full[s]);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              bulk_load(smem + C::OFF_SFB + s * C::SFB_BYTES + h * KB_PER_TILE * 512,
                        w_scales + ((size_t)(n0 / 128 + h) * kb_total +
                                    (size_t)kt * KB_PER_TILE) * 512,
                        (uint32_t)nkb * 512u, &full[s]);
            SVDQ_TR(0, 128, issued);
          }
          ++issued;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    // The tensor cores queue only about one MMA ahead, so this thread keeps
    // the work between two MMAs short: descriptors are formed by adding to
    // per-ring constants, the ring position advances without division, and
    // the wait for the next ring position runs while the current position's
    // last MMA is still queued.
    if (crank == 0) {  // the whole warp, converged; one elected lane issues
      const uint64_t a_desc0 = smem_desc(smem_u32(smem + C::OFF_A), 16, 1024, kSwizzle128B);
      const uint64_t b_desc0 = smem_desc(smem_u32(smem + C::OFF_B), 16, 1024, kSwizzle128B);
      const uint32_t empty_c0 = cluster_map(smem_u32(empty), 0u);
      const uint32_t empty_c1 = cluster_map(smem_u32(empty), 1u);
      const bool tail_half = (kb_total % KB_PER_TILE) != 0;  // last k tile has 2 MMA steps
      int s = 0;
      uint32_t ph = 0;  // ring position: slot and phase parity
      // frees slot s in both CTAs once the MMAs issued so far have read it
      auto release_slot = [&](int s_) {
        tc_commit_pair_warp2(empty_c0 + 8u * (uint32_t)s_, empty_c1 + 8u * (uint32_t)s_);
      };
      // GELU + quantization: the next layer's down projection of tile t, its
      // staged H (both CTAs' 128 rows, [BN/64 chunks][128 rows][64]) times the
      // L1s2 slice, accumulated over the segment into the RANK2 TMEM columns at
      // L2Q_COL.  It is issued between the k tiles of the following tile, once
      // H is staged (h_ready) and, at a segment's first tile, the previous
      // segment's sums were read (l2q_empty, one phase per segment).
      int l2q_pending = -1, l2q_segs = 0;
      auto l2q_issue = [&](int t) {
        tc_fence_after();
        const uint32_t hb = smem_u32(smem + C::OFF_OUT);
        const uint32_t lb = smem_u32(smem + C::OFF_L1S2);
        const uint32_t acc0 = seg_first(t) ? 0u : 1u;
#pragma unroll
        for (int c = 0; c < BN / 64; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16_pair_warp(
                tmem + (uint32_t)C::L2Q_COL,
                smem_desc(hb + c * (4 * C::OUT_WARP_BYTES) + kk * 32, 16, 1024, kSwizzle128B),
                smem_desc(lb + c * (C::R2H * 128) + kk * 32, 16, 1024, kSwizzle128B),
                C::IDESC_L2Q, (c | kk) != 0 ? 1u : acc0);
        tc_commit_pair_warp2(cluster_map(smem_u32(l2q_full), 0u),
                             cluster_map(smem_u32(l2q_full), 1u));
        tc_commit_pair_warp2(cluster_map(smem_u32(l1s2_empty), 0u),
                             cluster_map(smem_u32(l1s2_empty), 1u));
        if (seg_first(t)) ++l2q_segs;
      };
      // the accumulator of the previous segment has been read (or there is none)
      auto l2q_free = [&](int t, bool block) -> bool {
        if (!seg_first(t)) return true;
        const uint32_t par = (uint32_t)(l2q_segs & 1) ^ 1u;
        return block ? mbar_wait(l2q_empty, par, dev_status, wait_ns) : mbar_test(l2q_empty, par);
      };
      auto l2q_try = [&]() {  // non-blocking
        if (!GQ || l2q_pending < 0) return;
        const int t = l2q_pending;
        const bool r = mbar_test(h_ready, (uint32_t)(t & 1)) && l2q_free(t, false);
        if (__all_sync(0xFFFFFFFFu, r)) {
          l2q_issue(t);
          l2q_pending = -1;
        }
      };
      auto l2q_finish = [&]() -> bool {  // blocking
        if (!GQ || l2q_pending < 0) return true;
        const int t = l2q_pending;
        const bool r = mbar_wait(h_ready, (uint32_t)(t & 1), dev_status, wait_ns) &&
                       l2q_free(t, true);
        if (!__all_sync(0xFFFFFFFFu, r)) return false;
        l2q_issue(t);
        l2q_pending = -1;
        return true;
      };
      // Position (s, ph) is ready when the scale warps of both CTAs have seen
      // their slot land and put its scales in their TMEM (sf_full: the scale
      // warps waited on this CTA's `full` first, so it orders the TMA data too).
      // With GELU + quantization a rank-r slot can wait, through the L1s2
      // buffer, for the previous tile's down projection: while one is
      // pending, the wait keeps trying to issue it.
      auto ready = [&](int s_, uint32_t ph_) -> bool {
        bool ok;
        if (GQ && l2q_pending >= 0) {
          const uint64_t t0 = globaltimer_ns();
          while (true) {
            if (__all_sync(0xFFFFFFFFu, mbar_test(&sf_full[s_], ph_))) {
              ok = true;
              break;
            }
            l2q_try();
            if (globaltimer_ns() - t0 > wait_ns) {
              report_timeout(dev_status);
              ok = false;
              break;
            }
          }
        } else {
          ok = mbar_wait(&sf_full[s_], ph_, dev_status, wait_ns);
        }
        tc_fence_after();
        return __all_sync(0xFFFFFFFFu, ok);
      };
      for (int j = 0; j < my_tiles && !__any_sync(0xFFFFFFFFu, *abort_flag != 0); ++j) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(acc_empty, (uint32_t)(j & 1) ^ 1u, dev_status,
                                                 wait_ns))) {
          abort_pair();
          break;
        }
        tc_fence_after();
        SVDQ_TR(384, 8, j);
        bool ok = ready(s, ph);
        int prev = -1;  // slot whose release waits until the next MMA is queued
        uint64_t ad = a_desc0 + (uint64_t)((s * C::A_BYTES) >> 4);
        uint64_t bd = b_desc0 + (uint64_t)((s * C::B_BYTES) >> 4);
        uint32_t sfa = tmem + (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS);
        for (int kt = 0; kt < k_tiles && ok; ++kt) {
          SVDQ_TR(128, 128, kt + j * (k_tiles + 1));
          const uint32_t sfb = sfa + (uint32_t)C::SF_COLS_A;
          // MMA step kb: K offset 32 bytes per step (2 in the descriptor's
          // 16-byte address units), scale columns 4 (A) and 4 BN/128 (B) per step
          auto mma = [&](int kb, uint32_t acc) {
            tc_mma_nvf4_pair_warp(tmem, ad + (uint64_t)(2 * kb), bd + (uint64_t)(2 * kb),
                                  C::IDESC_NVF4, sfa + 4u * kb, sfb + 4u * (BN / 128) * kb, acc);
          };
          int sn = s + 1;
          uint32_t phn = ph;
          if (sn == STAGES) {
            sn = 0;
            phn ^= 1u;
          }
          // the slow steps (commits, barrier waits) each go where an MMA is
          // already queued: release of the previous slot after this slot's
          // first MMA, the wait for the next position after its second
          mma(0, kt != 0 ? 1u : 0u);
          if (prev >= 0) release_slot(prev);
          l2q_try();
          if (tail_half && kt + 1 == k_tiles) {
            ok = ready(sn, phn);
            mma(1, 1u);
          } else {
            mma(1, 1u);
            ok = ready(sn, phn);
            mma(2, 1u);
            mma(3, 1u);
          }
          SVDQ_TR(256, 128, kt + j * (k_tiles + 1));
          prev = s;
          s = sn;
          ph = phn;
          if (sn == 0) {
            ad = a_desc0;
            bd = b_desc0;
            sfa = tmem + (uint32_t)C::SF_BASE;
          } else {
            ad += (uint64_t)(C::A_BYTES >> 4);
            bd += (uint64_t)(C::B_BYTES >> 4);
            sfa += (uint32_t)C::SF_STAGE_COLS;
          }
        }
        if (ok) {
          // the rank-r slot (the scale warps report it in sf_full too, so that
          // every slot's sf_full completes once per use of the slot); its
          // readiness was awaited during the last k tile
          SVDQ_TR(392, 8, j);
          const uint32_t la = smem_u32(smem + C::OFF_A + s * C::A_BYTES);
          const uint32_t lbp = smem_u32(smem + C::OFF_B + s * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < RANK / 16; ++kk) {
            tc_mma_bf16_pair_warp(tmem, smem_desc(la + kk * 32, 16, 8 * C::LROW, C::LSW),
                                  smem_desc(lbp + kk * 32, 16, 8 * C::LROW, C::LSW),
                                  C::IDESC_BF16, 1u);
            if (kk == 0 && prev >= 0) release_slot(prev);
          }
          release_slot(s);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        } else if (prev >= 0) {
          release_slot(prev);
        }
        if (!ok) abort_pair();
        // fires once every MMA issued so far has completed (in both CTAs)
        tc_commit_pair_warp2(cluster_map(smem_u32(acc_full), 0u),
                             cluster_map(smem_u32(acc_full), 1u));
        if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
        if (GQ) {
          if (!l2q_finish()) {  // the previous tile's, if the k tiles did not fit it in
            abort_pair();
            break;
          }
          l2q_pending = j;
        }
      }
      if (GQ && !__any_sync(0xFFFFFFFFu, *abort_flag != 0) && !l2q_finish()) abort_pair();
      if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) {  // wake both epilogues after an abort
        tc_commit_pair_warp2(cluster_map(smem_u32(acc_full), 0u),
                             cluster_map(smem_u32(acc_full), 1u));
        if (GQ)
          tc_commit_pair_warp2(cluster_map(smem_u32(l2q_full), 0u),
                               cluster_map(smem_u32(l2q_full), 1u));
      }
      // no MMA may still write either TMEM when the pair frees it
      tc_commit_pair_warp(cluster_map(smem_u32(mma_done), 0u));
      mbar_wait(mma_done, 0u, dev_status, wait_ns);
    }
  } else if (warp >= SF_WARP0 && warp < SF_WARP0 + 4) {
    // ------------------------------------------------------------ scale warps
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    int it = 0;
    // after this warp's TMEM stores (if any) are complete: one arrival on the
    // even CTA's sf_full of the slot
    auto report = [&](int s) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(at_even(&sf_full[s]));
    };
    for (int j = 0; j < my_tiles; ++j) {
      bool ok = true;
      for (int kt = 0; kt < k_tiles; ++kt, ++it) {
        const int s = it % STAGES;
        ok = mbar_wait(&full[s], (uint32_t)(it / STAGES) & 1u, dev_status, wait_ns) &&
             !*abort_flag;
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
        if (warp == SF_WARP0 && lane == 0) SVDQ_TR(960, 64, it);
        const int nkb = min(KB_PER_TILE, kb_total - kt * KB_PER_TILE);
        const uint8_t* sfa = smem + C::OFF_SFA + s * C::SFA_BYTES + lane * 16;
        const uint8_t* sfb = smem + C::OFF_SFB + s * C::SFB_BYTES + lane * 16;
        const uint32_t col = lane_base + (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS);
        for (int kb = 0; kb < nkb; ++kb) {
          tmem_st_32x32b_x4(col + kb * 4, lds128(sfa + kb * 512));
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tmem_st_32x32b_x4(col + C::SF_COLS_A + kb * 4 * (BN / 128) + h * 4,
                              lds128(sfb + h * KB_PER_TILE * 512 + kb * 512));
        }
        tmem_st_wait();
        report(s);
        if (warp == SF_WARP0 && lane == 0) SVDQ_TR(448, 128, it);
      }
      if (!ok) {
        abort_pair();
        break;
      }
      // the rank-r slot needs no scales; sf_full still completes once for it,
      // after the slot has been filled (so it cannot run a phase ahead)
      const int s = it % STAGES;
      ok = mbar_wait(&full[s], (uint32_t)(it / STAGES) & 1u, dev_status, wait_ns) &&
           !*abort_flag;
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        abort_pair();
        break;
      }
      report(s);
      ++it;
    }
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue warps
    constexpr int CH = C::EPI_CH;
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int e = warp - EPI_WARP0;
    const int col0 = (e >> 2) * C::EPI_COLS;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    const uint32_t acc_empty_even = at_even(acc_empty);
    // TMA-store epilogue: this warp's staging block; lane l writes row l, its
    // 16-byte chunk c at byte offset o = l * ROW + 16 c XOR-ed with the
    // swizzle of the output tensor map (bits 4.. of o ^= bits 7.. of o)
    uint8_t* stage = smem + C::OFF_OUT + e * C::OUT_WARP_BYTES;
    // QKV: warps e and e ^ 4 hold the two 64-column halves of one head for the
    // same 32 rows; `pid` names the pair, `qk` counts its exchanges
    const int pid = ((e >> 3) << 2) | (e & 3);
    int qk = 0;
    for (int j = 0; j < my_tiles; ++j) {
      int m_tile, n_tile;
      tile_mn(j, m_tile, n_tile);
      const int m0 = m_tile * BM, n0 = n_tile * BN;
      bool ok = mbar_wait(acc_full, (uint32_t)(j & 1), dev_status, wait_ns) && !*abort_flag;
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        abort_pair();
        break;
      }
      tc_fence_after();
      if (warp == EPI_WARP0 && lane == 0) SVDQ_TR(400, 8, j);
      if (warp == EPI_WARP0 + EPI_WARPS - 1 && lane == 0) SVDQ_TR(432, 8, j);
      uint32_t v[C::EPI_COLS];
#pragma unroll
      for (int c = 0; c < C::EPI_COLS / 32; ++c)
        tmem_ld_32x32b_x32(lane_base + (uint32_t)(col0 + 32 * c),
                           *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_even);  // accumulator free for the next tile
      if (warp == EPI_WARP0 && lane == 0) SVDQ_TR(408, 8, j);
      if (warp == EPI_WARP0 + EPI_WARPS - 1 && lane == 0) SVDQ_TR(440, 8, j);
      // the bias slice landed with this tile's rank-r slot (the rank-r MMAs
      // waited for it, through sf_full, before acc_full was signalled)
      const uint16_t* bsm =
          bias ? reinterpret_cast<const uint16_t*>(smem + C::OFF_BIAS + (j % EBUF) * C::BIAS_BYTES)
               : nullptr;
      // bf16 pairs in place: pair i lands in v[i] (read from v[2i], v[2i+1])
#pragma unroll
      for (int c = 0; c < C::EPI_COLS / 32; ++c)
        pack_cols32<EPI == kEpiGelu || GQ>(&v[32 * c], s_T, bsm ? bsm + col0 + 32 * c : nullptr,
                                           &v[16 * c]);
      uint32_t(&pk)[4 * CH] = *reinterpret_cast<uint32_t(*)[4 * CH]>(&v[0]);
      if (bsm) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bias_empty[j % EBUF]);
      }
      if constexpr (GQ) {
        // H = bf16(gelu(Y)) of this lane's row: staged for the down-projection
        // MMAs (and the optional store of H), then quantized as the next
        // layer's input, 4 blocks of 16 columns
        constexpr int swz_mask = 7;  // 128-byte rows, 128B swizzle
        const int row = m0 + 32 * q + lane;
        // the down-projection MMAs read 64-column chunk c as 128 rows in
        // order: lane quarter q of the chunk's warps stages at block 4c + q
        uint8_t* gstage = smem + C::OFF_OUT + ((e >> 2) * 4 + q) * C::OUT_WARP_BYTES;
        // the staging area is free: the previous tile's down projection has
        // read it (l2q_full), and its store of H has left it
        if (j > 0) {
          const bool got =
              mbar_wait(l2q_full, (uint32_t)((j - 1) & 1), dev_status, wait_ns) && !*abort_flag;
          if (!__all_sync(0xFFFFFFFFu, got)) {
            abort_pair();
            break;
          }
        }
        if (gq.h_out && lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int o = lane * C::OUT_ROW_BYTES + 16 * c;
          sts128(gstage + (o ^ (((o >> 7) & swz_mask) << 4)), pk[4 * c], pk[4 * c + 1],
                 pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();  // generic writes, before the MMAs (async proxy) read them
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_cluster(at_even(h_ready));
          if (gq.h_out && m0 + 32 * q < M) {
            tma_store_2d(&tm_y, gstage, n0 + col0, m0 + 32 * q);
            bulk_commit_group();
          }
        }
        // the next layer's activation quantization of the row's 64 columns
        const float2* tabp = reinterpret_cast<const float2*>(smem + C::OFF_TAB);
        const float2 r6 = recip2(6.0f);
        // inv_lambda of the columns: the same 64 floats for every lane (one
        // broadcast load each, from L1 after the first warp)
        const float4* invg = reinterpret_cast<const float4*>(gq.inv_lambda2 + n0 + col0);
        uint2 cw[4];
        uint32_t sw = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = pk[8 * b + i];
          float inv[16];
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const float4 iv = __ldg(invg + 4 * b + i4);
            inv[4 * i4] = iv.x;
            inv[4 * i4 + 1] = iv.y;
            inv[4 * i4 + 2] = iv.z;
            inv[4 * i4 + 3] = iv.w;
          }
          uint32_t sb;
          quant_block16(w, inv, r6, tabp, cw[b], sb);
          sw |= sb << (8 * b);
        }
        if (row < M) {
          uint4* cp = reinterpret_cast<uint4*>(gq.a2_codes + (size_t)row * (N / 2) + (n0 + col0) / 2);
          cp[0] = make_uint4(cw[0].x, cw[0].y, cw[1].x, cw[1].y);
          cp[1] = make_uint4(cw[2].x, cw[2].y, cw[3].x, cw[3].y);
          *reinterpret_cast<uint32_t*>(gq.a2_scales +
                                       ((size_t)(row >> 7) * (N / 64) + (n0 + col0) / 64) * 512 +
                                       (row & 31) * 16 + ((row >> 5) & 3) * 4) = sw;
        }
        // at the segment's last tile, warps 0-3 (one per lane quarter): the
        // segment's down-projection sums of their 32 rows, to scratch slot
        // pair + m pair (256 rows x RANK2 floats; unique: a later pair covers
        // no earlier m pair)
        if (e < 4 && seg_last(j)) {
          const bool got =
              mbar_wait(l2q_full, (uint32_t)(j & 1), dev_status, wait_ns) && !*abort_flag;
          if (!__all_sync(0xFFFFFFFFu, got)) {
            abort_pair();
            break;
          }
          tc_fence_after();
          uint32_t pv[RANK2];
#pragma unroll
          for (int c = 0; c < RANK2 / 32; ++c)
            tmem_ld_32x32b_x32(lane_base + (uint32_t)(C::L2Q_COL + 32 * c),
                               *reinterpret_cast<uint32_t(*)[32]>(&pv[32 * c]));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(at_even(l2q_empty));
          if (row < M) {
            const size_t slot = (size_t)(pair + tile_pt(j) / n_tiles);
            uint4* pp = reinterpret_cast<uint4*>(
                gq.partial + (slot * (2 * BM) + (size_t)crank * BM + 32 * q + lane) * RANK2);
#pragma unroll
            for (int i = 0; i < RANK2 / 4; ++i)
              pp[i] = make_uint4(pv[4 * i], pv[4 * i + 1], pv[4 * i + 2], pv[4 * i + 3]);
          }
        }
      } else if constexpr (C::TMA_OUT) {
        // rows at or past M are clipped by the tensor map (a block wholly past
        // M is not stored at all)
        constexpr int swz_mask = C::OUT_ROW_BYTES == 128 ? 7 : 3;  // 128B / 64B swizzle
        if (lane == 0) bulk_wait_group_read0();  // the previous block left the staging area
        __syncwarp();
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int o = lane * C::OUT_ROW_BYTES + 16 * c;
          sts128(stage + (o ^ (((o >> 7) & swz_mask) << 4)), pk[4 * c], pk[4 * c + 1],
                 pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();  // the generic-proxy writes, before the TMA engine reads them
        __syncwarp();
        if (lane == 0 && m0 + 32 * q < M) {
          tma_store_2d(&tm_y, stage, n0 + col0, m0 + 32 * q);
          bulk_commit_group();
        }
      } else {
        const int gbase = lane & ~(CH - 1), tc = lane & (CH - 1);
        // QKV: 1/rms of this lane's row (before the transpose), used after it
        float rs = 0.0f;
        const int region = n0 < qe.hd ? 0 : (n0 < 2 * qe.hd ? 1 : 2);
        if (region < 2) {  // a Q or K tile
          // sum of squares of this lane's 64 bf16 values (column order); the
          // partner's half arrives through shared memory
          float ss = 0.0f;
#pragma unroll
          for (int i = 0; i < C::EPI_COLS / 2; ++i) {
            const float a = bf16lo_to_f32(v[i]), b = bf16hi_to_f32(v[i]);
            ss = __fmaf_rn(a, a, ss);
            ss = __fmaf_rn(b, b, ss);
          }
          float* xs = reinterpret_cast<float*>(smem + C::OFF_XSUM) + (qk & 1) * EPI_WARPS * 32;
          xs[e * 32 + lane] = ss;
          __syncwarp();
          if (lane == 0) mbar_arrive(&pair_bar[pid]);
          const bool got =
              mbar_wait(&pair_bar[pid], (uint32_t)(qk & 1), dev_status, wait_ns) && !*abort_flag;
          if (!__all_sync(0xFFFFFFFFu, got)) {
            abort_pair();
            break;
          }
          ++qk;
          const float other = xs[(e ^ 4) * 32 + lane];
          const float total = (e & 4) ? other + ss : ss + other;  // lower columns first
          rs = rsqrtf(__fmaf_rn(total, 1.0f / kHeadDim, qe.eps));
        }
        // after the transpose, store i of lane t writes chunk t % CH of row
        // (t & ~(CH-1)) + i: CH consecutive lanes cover one row segment
        transpose_chunks<CH>(pk, lane);
        if (region < 2)
          qkv_rotate_rows(pk, rs, gbase,
                          (region == 0 ? qe.norm_q : qe.norm_k) + (col0 & (kHeadDim - 1)) + 8 * tc,
                          qe.rope_cos, qe.rope_sin, m0 + 32 * q + gbase, M,
                          ((col0 & (kHeadDim - 1)) >> 1) + 4 * tc);
        const int cbase = n0 + col0 + 8 * tc;
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          const int row = m0 + 32 * q + gbase + i;
          if (row < M)
            *reinterpret_cast<uint4*>(Y + (size_t)row * N + cbase) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (warp == EPI_WARP0 && lane == 0) SVDQ_TR(416, 8, j);
    }
    // every TMA store of this warp has completed (and left its staging area)
    if (C::TMA_OUT && lane == 0) bulk_wait_group0();
    // GELU + quantization: the last tile's down projection has read the
    // staging area before the CTA may leave (the even CTA's MMAs read both)
    if (GQ && my_tiles > 0 && !*abort_flag)
      mbar_wait(l2q_full, (uint32_t)((my_tiles - 1) & 1), dev_status, wait_ns);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // an aborted run: loads may still be landing; the CTA must not exit first
    for (int i = max(0, issued - STAGES); i < issued; ++i)
      mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u, nullptr, wait_ns);
  }
  // neither CTA of the pair leaves (or frees TMEM) while the other may still
  // write its shared memory, arrive on its barriers or run MMAs into its TMEM
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// GELU + quantization, second kernel: lora2[m][i] = bf16( the sum, over the
// CTA pairs p that covered m pair mp = m / 256 in ascending order, of
// partial[p + mp][m % 256][i] ).  The pairs' tile ranges are those of the
// GEMM: pair p took pair tiles [p T / P, (p + 1) T / P) (T P < 2^31, checked
// by the caller).  One thread per 4 consecutive outputs of a row.
__device__ __forceinline__ int gq_owner(int t, int num_ptiles, int n_pairs) {
  return (int)(((unsigned)(t + 1) * (unsigned)n_pairs - 1u) / (unsigned)num_ptiles);
}
__global__ void __launch_bounds__(128, 4)
    k_lora_reduce(const float* __restrict__ partial, int M, int rank2, int num_ptiles,
                  int n_pairs, int n_tiles, uint16_t* __restrict__ lora2) {
  grid_dep_launch();
  grid_dep_wait();  // the GEMM's segment sums are complete
  const int quads = rank2 >> 2;
  const int total = M * quads;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += gridDim.x * blockDim.x) {
    const int m = idx / quads, i4 = idx - m * quads, mp = m >> 8;
    const int p_lo = gq_owner(mp * n_tiles, num_ptiles, n_pairs);
    const int p_hi = gq_owner(mp * n_tiles + n_tiles - 1, num_ptiles, n_pairs);
    float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int p = p_lo; p <= p_hi; ++p) {
      // (a pair without tiles wrote nothing)
      if ((unsigned)(p + 1) * (unsigned)num_ptiles / (unsigned)n_pairs ==
          (unsigned)p * (unsigned)num_ptiles / (unsigned)n_pairs)
        continue;
      const float4 v = __ldg(reinterpret_cast<const float4*>(
                                 partial + (((size_t)(p + mp) << 8) + (m & 255)) * rank2) +
                             i4);
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
    *reinterpret_cast<uint2*>(lora2 + (size_t)m * rank2 + 4 * i4) =
        make_uint2((uint32_t)f32_to_bf16_rn(sum.x) | ((uint32_t)f32_to_bf16_rn(sum.y) << 16),
                   (uint32_t)f32_to_bf16_rn(sum.z) | ((uint32_t)f32_to_bf16_rn(sum.w) << 16));
  }
}

template <int BN, int RANK, int EPI, int RANK2 = 0>
cudaError_t launch_t(const GemmMaps& maps, const uint8_t* a_scales, const uint8_t* w_scales,
                     float s_T, const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                     const QkvEpilogue& qe, const GeluQuantEpilogue& gq, int* dev_status,
                     int test_stall, int num_sms, cudaStream_t stream) {
  using C = Cfg<BN, RANK, EPI, RANK2>;
  auto kern = k_gemm_w4a4<BN, RANK, EPI, RANK2>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query below takes the cluster shape only
  // persistent: as many CTA pairs as can be resident at once (a GPC with an
  // odd number of free SMs leaves one idle), at most one per tile pair; the
  // count is queried once per device and instantiation
  static std::atomic<int> max_pairs_of[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return cudaErrorInvalidDevice;
  }
  int max_pairs = max_pairs_of[dev].load(std::memory_order_relaxed);
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms / 2;
    }
    max_pairs = n;  // every caller computes the same value: a plain store is enough
    max_pairs_of[dev].store(n, std::memory_order_relaxed);
  }
  const int m_tiles = (M + BM - 1) / BM;
  const int num_ptiles = ((m_tiles + 1) / 2) * (N / BN);
  int pairs = num_ptiles < max_pairs ? num_ptiles : max_pairs;
  if (EPI == kEpiGeluQuant && pairs > kGqMaxPairs) pairs = kGqMaxPairs;  // scratch slots
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, maps.a_codes, maps.w_codes, maps.lora, maps.l2s, maps.y,
                         maps.l1s2, a_scales, w_scales, s_T, bias, Y, M, N, K, qe, gq, dev_status,
                         test_stall, (uint64_t)(test_stall ? 100000000ull : kWaitTimeoutNs));
  if (e != cudaSuccess) return e;
  if (EPI == kEpiGeluQuant) {
    cudaLaunchConfig_t rc = {};
    const size_t total = (size_t)M * (gq.rank2 / 4);
    // small blocks: one fits on an SM beside a GEMM CTA (registers), so the
    // reduction's blocks wait resident during the GEMM, and the next kernel's
    // GEMM CTAs can start beside them
    const size_t blocks = (total + 127) / 128;
    rc.gridDim = dim3((unsigned)(blocks < 4096 ? blocks : 4096), 1, 1);
    rc.blockDim = dim3(128, 1, 1);
    rc.stream = stream;
    rc.attrs = &attr[1];  // programmatic dependent launch
    rc.numAttrs = 1;
    e = cudaLaunchKernelEx(&rc, k_lora_reduce, (const float*)gq.partial, M, gq.rank2,
                           num_ptiles, pairs, N / BN, gq.lora2);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

// the QKV epilogue exists for two-head tiles only (block_n 256)
template <int BN, int RANK>
cudaError_t launch_qkv_t(const GemmMaps& maps, const uint8_t* a_scales, const uint8_t* w_scales,
                         float s_T, const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                         const QkvEpilogue& qe, const GeluQuantEpilogue& gq, int* dev_status,
                         int test_stall, int num_sms, cudaStream_t stream) {
  if constexpr (BN == 2 * kHeadDim)
    return launch_t<BN, RANK, kEpiQkv>(maps, a_scales, w_scales, s_T, bias, Y, M, N, K, qe, gq,
                                       dev_status, test_stall, num_sms, stream);
  else
    return cudaErrorInvalidValue;
}

// the GELU + quantization epilogue exists for 256-column tiles only
template <int BN, int RANK>
cudaError_t launch_gq_t(const GemmMaps& maps, const uint8_t* a_scales, const uint8_t* w_scales,
                        float s_T, const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                        const QkvEpilogue& qe, const GeluQuantEpilogue& gq, int* dev_status,
                        int test_stall, int num_sms, cudaStream_t stream) {
  if constexpr (BN == 256) {
    if (gq.rank2 == 32)
      return launch_t<BN, RANK, kEpiGeluQuant, 32>(maps, a_scales, w_scales, s_T, bias, Y, M, N,
                                                   K, qe, gq, dev_status, test_stall, num_sms,
                                                   stream);
    if (gq.rank2 == 64)
      return launch_t<BN, RANK, kEpiGeluQuant, 64>(maps, a_scales, w_scales, s_T, bias, Y, M, N,
                                                   K, qe, gq, dev_status, test_stall, num_sms,
                                                   stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm_w4a4(const GemmMaps& maps, int block_n, const uint8_t* a_scales,
                             const uint8_t* w_scales, float w_tensor_scale, const uint16_t* bias,
                             uint16_t* Y, int M, int N, int K, int rank, GemmEpilogue epi,
                             const QkvEpilogue& qe, const GeluQuantEpilogue& gq,
                             int* dev_status, int test_stall, int num_sms, cudaStream_t stream) {
#define SVDQ_GEMM_LAUNCH(BN_, R_, E_)                                                        \
  return launch_t<BN_, R_, E_>(maps, a_scales, w_scales, w_tensor_scale, bias, Y, M, N, K,   \
                               qe, gq, dev_status, test_stall, num_sms, stream)
#define SVDQ_GEMM_CASE(BN_, R_)                                                              \
  if (block_n == BN_ && rank == R_) {                                                        \
    if (epi == GemmEpilogue::kPlain) SVDQ_GEMM_LAUNCH(BN_, R_, kEpiPlain);                   \
    if (epi == GemmEpilogue::kGelu) SVDQ_GEMM_LAUNCH(BN_, R_, kEpiGelu);                     \
    if (epi == GemmEpilogue::kQkv)                                                           \
      return launch_qkv_t<BN_, R_>(maps, a_scales, w_scales, w_tensor_scale, bias, Y, M, N,  \
                                   K, qe, gq, dev_status, test_stall, num_sms, stream);      \
    if (epi == GemmEpilogue::kGeluQuant)                                                     \
      return launch_gq_t<BN_, R_>(maps, a_scales, w_scales, w_tensor_scale, bias, Y, M, N,   \
                                  K, qe, gq, dev_status, test_stall, num_sms, stream);       \
  }
  SVDQ_GEMM_CASE(256, 16)
  SVDQ_GEMM_CASE(256, 32)
  SVDQ_GEMM_CASE(256, 64)
  SVDQ_GEMM_CASE(128, 16)
  SVDQ_GEMM_CASE(128, 32)
  SVDQ_GEMM_CASE(128, 64)
#undef SVDQ_GEMM_CASE
#undef SVDQ_GEMM_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace svdq

#ifdef SVDQ_GEMM_TRACE
// instrumented builds only: where the first 8 CTAs write their timeline
// (1024 x u64 per CTA), or nullptr to stop
extern "C" int svdq_gemm_trace_set(unsigned long long* p) {
  return (int)cudaMemcpyToSymbol(svdq::g_gemm_trace, &p, sizeof(p));
}
#endif
