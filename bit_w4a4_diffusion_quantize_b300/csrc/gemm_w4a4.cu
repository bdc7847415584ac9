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
//
// Persistent kernel: one CTA per SM walks 128 x BN output tiles (BN = 256, or
// 128 when N is not a multiple of 256), N fastest.  Warp roles (16 warps):
//   warp 0     one lane streams the k tiles of each output tile -- A/B code
//              tiles (64-byte rows = 128 codes, 64B swizzle: small stages, so
//              a slot is refilled after two MMAs) and the block-scale chunks
//              (plain bulk copies: the scale layout is already the tensor
//              core's) -- into a STAGES-deep ring, running ahead across tile
//              boundaries; a few k tiles into each tile it also loads that
//              tile's rank-r operands (lora rows and L2s rows, K-major,
//              swizzled TMA boxes) and bias slice;
//   warp 1     allocates TMEM; one lane issues the block-scaled MMAs of each
//              k tile, then the rank-r MMAs into the same accumulator;
//              tcgen05.commit frees smem stages and the rank-r buffer and
//              finally signals `acc_full`;
//   warps 4-7  scale warps, one per TMEM lane quarter: for each k tile they
//              move the block scales from shared memory into TMEM with
//              tcgen05.st (registers -> TMEM), keeping that traffic off the
//              MMA issue path, and signal `sf_full`;
//   warps 8-15 the epilogue, two per TMEM lane quarter (one output row per
//              lane, half of the columns each), in two rounds of 64 columns:
//              tcgen05.ld, y = s_T * acc + bias, bf16, into a 32 x 64 staging
//              box in shared memory (128B swizzle), written out by one TMA
//              store (whole 128-byte lines).  The accumulator is released
//              (`acc_empty`) as soon as the second round is in registers, so
//              the next tile's MMAs overlap the rest of the epilogue.
//
// Block scales in TMEM.  Per 64-wide K step, the 128 x 4 scale chunk of A
// (512 bytes, row r at byte (r%32)*16 + (r/32)*4) occupies 4 columns: every
// lane quarter holds, in lane l, column j, the 4 scales of row l + 32j (the
// layout of tcgen05.cp.32x128b.warpx4).  A scale warp loads chunk row l (16
// bytes) and stores it with one tcgen05.st.32x32b.x4.  B's BN rows take BN/32
// columns the same way.
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
constexpr int BK_BYTES = 64;      // one k tile: 128 fp4 values per row
constexpr int KB_PER_TILE = 2;    // 64-wide MMA steps per k tile
constexpr int NUM_THREADS = 16 * 32;
constexpr int SF_WARP0 = 4;       // warps 4..7
constexpr int EPI_WARP0 = 8;      // warps 8..15
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_BUDGET = 224 * 1024;

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int BN, int RANK>
struct Cfg {
  static constexpr int A_BYTES = BM * BK_BYTES;
  static constexpr int B_BYTES = BN * BK_BYTES;
  static constexpr int SFA_BYTES = KB_PER_TILE * 512;
  static constexpr int SFB_BYTES = KB_PER_TILE * 512 * (BN / 128);
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int LROW = RANK * 2;  // bytes of one rank-r row (bf16)
  static constexpr int LA_BYTES = BM * LROW;
  static constexpr int LB_BYTES = BN * LROW;
  static constexpr int BIAS_BYTES = BN * 2;
  static constexpr int LBUF_BYTES = align_up(LA_BYTES + LB_BYTES, 1024);
  static constexpr int STG_BYTES = 8 * 32 * 128;  // 8 epilogue warps x (32 rows x 64 bf16)
  static constexpr int MISC_BYTES = 512;
  static constexpr int FIXED_BYTES = LBUF_BYTES + 2 * BIAS_BYTES + STG_BYTES + MISC_BYTES;
  static constexpr int STAGES = cmin(8, (SMEM_BUDGET - 1024 - FIXED_BYTES) / STAGE_BYTES);
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_L = align_up(OFF_SFB + STAGES * SFB_BYTES, 1024);
  static constexpr int OFF_STG = OFF_L + LBUF_BYTES;  // 1024-aligned (128B swizzle atoms)
  static constexpr int OFF_BIAS = OFF_STG + STG_BYTES;
  static constexpr int OFF_BAR = OFF_BIAS + 2 * BIAS_BYTES;
  // barriers: full[S], empty[S], sf_full[S], lora_full, lora_empty,
  // bias_empty[2], acc_full, acc_empty
  static constexpr int NUM_BARS = 3 * STAGES + 6;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + base alignment slack
  // TMEM columns: accumulator [0, BN), then per stage the scales of A and B
  static constexpr int SF_COLS_A = 4 * KB_PER_TILE;
  static constexpr int SF_COLS_B = 4 * KB_PER_TILE * (BN / 128);
  static constexpr int SF_STAGE_COLS = SF_COLS_A + SF_COLS_B;
  static constexpr int SF_BASE = BN;
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert(SF_BASE + STAGES * SF_STAGE_COLS <= (int)TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static constexpr SmemLayout LSW =
      LROW == 128 ? kSwizzle128B : (LROW == 64 ? kSwizzle64B : kSwizzle32B);
  // instruction descriptors (kind::mxf4nvf4: E2M1 x E2M1, UE4M3 scales, K-major,
  // M = 128, N = BN; kind::f16: bf16 x bf16 -> f32)
  static constexpr uint32_t IDESC_NVF4 = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                         ((uint32_t)(BM >> 4) << 24);
  static constexpr uint32_t IDESC_BF16 = (1u << 4) | (1u << 7) | (1u << 10) |
                                         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  static constexpr int EPI_COLS = BN / 2;  // columns per epilogue warp
  static constexpr int EPI_ROUNDS = EPI_COLS / 64;
};

#ifdef SVDQ_GEMM_TRACE
// timeline instrumentation, compiled only into instrumented builds: the first
// 8 CTAs stamp %globaltimer at fixed slots (1024 per CTA)
__device__ unsigned long long* g_gemm_trace = nullptr;
#define SVDQ_TR(slot, lim, idx)                                                   \
  do {                                                                            \
    if (g_gemm_trace && blockIdx.x < 8 && (idx) < (lim))                          \
      g_gemm_trace[blockIdx.x * 1024 + (slot) + (idx)] = globaltimer_ns();        \
  } while (0)
#else
#define SVDQ_TR(slot, lim, idx) \
  do {                          \
  } while (0)
#endif

template <int BN, int RANK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_gemm_w4a4(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_lora,
                const __grid_constant__ CUtensorMap tm_l2s,
                const __grid_constant__ CUtensorMap tm_y, const uint8_t* __restrict__ a_scales,
                const uint8_t* __restrict__ w_scales, float s_T,
                const uint16_t* __restrict__ bias, int M, int N, int K, int* dev_status,
                int test_stall, uint64_t wait_ns) {
  using C = Cfg<BN, RANK>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* sf_full = empty + STAGES;
  uint64_t* lora_full = sf_full + STAGES;
  uint64_t* lora_empty = lora_full + 1;
  uint64_t* bias_empty = lora_empty + 1;  // [2]
  uint64_t* acc_full = bias_empty + 2;
  uint64_t* acc_empty = acc_full + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);  // [0] tmem, [1] abort
  volatile uint32_t* abort_flag = &misc[1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb_total = K >> 6;  // 64-wide steps
  const int k_tiles = (kb_total + KB_PER_TILE - 1) / KB_PER_TILE;
  const int n_tiles = N / BN;
  const int num_tiles = ((M + BM - 1) / BM) * n_tiles;
  const int my_tiles =
      (int)blockIdx.x < num_tiles ? (num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  // the rank-r operands of a tile are loaded just before its k tile `k_lora`
  // (or after its last k tile): by then the previous tile's rank-r MMAs, which
  // precede this tile's first MMAs, have freed the single rank-r buffer
  const int k_lora = min(STAGES, k_tiles);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 128);
    }
    mbar_init(lora_full, 1);
    mbar_init(lora_empty, 1);
    mbar_init(&bias_empty[0], 8);
    mbar_init(&bias_empty[1], 8);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 256);
    misc[1] = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_lora);
    prefetch_tmap(&tm_l2s);
    prefetch_tmap(&tm_y);
  }
  if (warp == 1) tmem_alloc(&misc[0], TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  int issued_k = 0, issued_l = 0;  // producer lane only: k tiles / rank-r sets loaded
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && !test_stall) {
      for (int j = 0; j < my_tiles && !*abort_flag; ++j) {
        const int tile = (int)blockIdx.x + j * (int)gridDim.x;
        const int m_tile = tile / n_tiles, n_tile = tile % n_tiles;
        const int m0 = m_tile * BM, n0 = n_tile * BN;
        for (int kt = 0; kt <= k_tiles; ++kt) {
          if (kt == k_lora) {
            // rank-r operands and bias slice of tile j
            if (!mbar_wait(lora_empty, (uint32_t)(j & 1) ^ 1u, dev_status, wait_ns) ||
                (bias && !mbar_wait(&bias_empty[j & 1], (uint32_t)((j >> 1) & 1) ^ 1u,
                                    dev_status, wait_ns))) {
              *abort_flag = 1;
              break;
            }
            uint8_t* lbuf = smem + C::OFF_L;
            mbar_arrive_expect_tx(lora_full, (uint32_t)(C::LA_BYTES + C::LB_BYTES +
                                                        (bias ? C::BIAS_BYTES : 0)));
            tma_load_2d(lbuf, &tm_lora, lora_full, 0, m0);
            tma_load_2d(lbuf + C::LA_BYTES, &tm_l2s, lora_full, 0, n0);
            if (bias)
              bulk_load(smem + C::OFF_BIAS + (j & 1) * C::BIAS_BYTES, bias + n0,
                        (uint32_t)C::BIAS_BYTES, lora_full);
            ++issued_l;
            SVDQ_TR(424, 8, j);
          }
          if (kt == k_tiles) break;
          const int s = issued_k % STAGES;
          const uint32_t ph = (uint32_t)(issued_k / STAGES) & 1u;
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
          SVDQ_TR(0, 128, issued_k);
          ++issued_k;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int it = 0;
      for (int j = 0; j < my_tiles && !*abort_flag; ++j) {
        if (!mbar_wait(acc_empty, (uint32_t)(j & 1) ^ 1u, dev_status, wait_ns)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        SVDQ_TR(384, 8, j);
        bool ok = true;
        for (int kt = 0; kt < k_tiles; ++kt, ++it) {
          const int s = it % STAGES;
          // sf_full: the scale warps saw the stage land and put its scales in TMEM
          if (*abort_flag ||
              !mbar_wait(&sf_full[s], (uint32_t)(it / STAGES) & 1u, dev_status, wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          SVDQ_TR(128, 128, it);
          const int nkb = min(KB_PER_TILE, kb_total - kt * KB_PER_TILE);
          const uint32_t a_base = smem_u32(smem + C::OFF_A + s * C::A_BYTES);
          const uint32_t b_base = smem_u32(smem + C::OFF_B + s * C::B_BYTES);
          const uint32_t sf_col = (uint32_t)(C::SF_BASE + s * C::SF_STAGE_COLS);
          for (int kb = 0; kb < nkb; ++kb)
            tc_mma_nvf4(tmem, smem_desc(a_base + kb * 32, 16, 512, kSwizzle64B),
                        smem_desc(b_base + kb * 32, 16, 512, kSwizzle64B), C::IDESC_NVF4,
                        tmem + sf_col + kb * 4,
                        tmem + sf_col + C::SF_COLS_A + kb * 4 * (BN / 128),
                        (kt | kb) != 0 ? 1u : 0u);
          tc_commit(&empty[s]);
          SVDQ_TR(256, 128, it);
        }
        if (ok && mbar_wait(lora_full, (uint32_t)(j & 1), dev_status, wait_ns)) {
          tc_fence_after();
          SVDQ_TR(392, 8, j);
          const uint32_t la = smem_u32(smem + C::OFF_L);
          const uint32_t lbp = la + C::LA_BYTES;
#pragma unroll
          for (int kk = 0; kk < RANK / 16; ++kk)
            tc_mma_bf16(tmem, smem_desc(la + kk * 32, 16, 8 * C::LROW, C::LSW),
                        smem_desc(lbp + kk * 32, 16, 8 * C::LROW, C::LSW), C::IDESC_BF16, 1u);
          tc_commit(lora_empty);
        } else {
          *abort_flag = 1;
        }
        tc_commit(acc_full);  // fires once every MMA issued so far has completed
        if (*abort_flag) break;
      }
      if (*abort_flag) tc_commit(acc_full);  // wake the epilogue after an abort
    }
  } else if (warp >= SF_WARP0 && warp < SF_WARP0 + 4) {
    // ------------------------------------------------------------ scale warps
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    int it = 0;
    for (int j = 0; j < my_tiles; ++j) {
      bool ok = true;
      for (int kt = 0; kt < k_tiles; ++kt, ++it) {
        const int s = it % STAGES;
        ok = mbar_wait(&full[s], (uint32_t)(it / STAGES) & 1u, dev_status, wait_ns) &&
             !*abort_flag;
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
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
        tc_fence_before();
        mbar_arrive(&sf_full[s]);
        if (warp == SF_WARP0 && lane == 0) SVDQ_TR(448, 128, it);
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
    }
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int col0 = ((warp - EPI_WARP0) >> 2) * C::EPI_COLS;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    uint8_t* stg = smem + C::OFF_STG + (warp - EPI_WARP0) * (32 * 128);
    uint8_t* my_row = stg + lane * 128;
    for (int j = 0; j < my_tiles; ++j) {
      const int tile = (int)blockIdx.x + j * (int)gridDim.x;
      const int m0 = (tile / n_tiles) * BM, n0 = (tile % n_tiles) * BN;
      bool ok = mbar_wait(acc_full, (uint32_t)(j & 1), dev_status, wait_ns) && !*abort_flag;
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      if (warp == EPI_WARP0 && lane == 0) SVDQ_TR(400, 8, j);
      if (warp == EPI_WARP0 + 7 && lane == 0) SVDQ_TR(432, 8, j);
      // the bias slice landed with this tile's rank-r operands (the rank-r MMAs
      // waited for it before acc_full was signalled)
      const uint16_t* bsm =
          bias ? reinterpret_cast<const uint16_t*>(smem + C::OFF_BIAS + (j & 1) * C::BIAS_BYTES)
               : nullptr;
      const bool rows_in = m0 + 32 * q < M;  // some row of this warp's box exists
      // Rounds of 64 columns: load (two 32-column tcgen05.ld), scale, add the
      // bias, pack to bf16 pairs, write the 32 x 64 box into this warp's
      // staging buffer (row `lane`, 16-byte chunk c at (c ^ (row % 8)) * 16)
      // and issue its TMA store.  The accumulator is released right after the
      // last load, before the wait for the previous store to have read the
      // buffer.
#pragma unroll 1
      for (int rd = 0; rd < C::EPI_ROUNDS; ++rd) {
        const int c0 = col0 + rd * 64;
        uint32_t pk[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(lane_base + (uint32_t)(c0 + 32 * h), v);
          tmem_ld_wait();
          if (rd == C::EPI_ROUNDS - 1 && h == 1) {
            tc_fence_before();
            mbar_arrive(acc_empty);
            if (warp == EPI_WARP0 && lane == 0) SVDQ_TR(408, 8, j);
            if (warp == EPI_WARP0 + 7 && lane == 0) SVDQ_TR(440, 8, j);
          }
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint4 bw = make_uint4(0u, 0u, 0u, 0u);
            if (bsm) bw = lds128(bsm + c0 + 32 * h + 8 * c8);
            const uint32_t bb[4] = {bw.x, bw.y, bw.z, bw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = 8 * c8 + 2 * i;
              const float y0 = __fmaf_rn(s_T, __uint_as_float(v[e]), bf16lo_to_f32(bb[i]));
              const float y1 = __fmaf_rn(s_T, __uint_as_float(v[e + 1]), bf16hi_to_f32(bb[i]));
              pk[16 * h + 4 * c8 + i] =
                  (uint32_t)f32_to_bf16_rn(y0) | ((uint32_t)f32_to_bf16_rn(y1) << 16);
            }
          }
        }
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
          sts128(my_row + ((c ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                 pk[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && rows_in) {
          tma_store_2d(&tm_y, stg, n0 + c0, m0 + 32 * q);
          bulk_commit_group();
        }
      }
      if (bsm) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bias_empty[j & 1]);
      }
      if (warp == EPI_WARP0 && lane == 0) SVDQ_TR(416, 8, j);
    }
    if (lane == 0) bulk_wait_group0();  // stores complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // an aborted run: loads may still be landing; the CTA must not exit first
    for (int i = max(0, issued_k - STAGES); i < issued_k; ++i)
      mbar_wait(&full[i % STAGES], (uint32_t)(i / STAGES) & 1u, nullptr, wait_ns);
    if (issued_l > 0) mbar_wait(lora_full, (uint32_t)((issued_l - 1) & 1), nullptr, wait_ns);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int BN, int RANK>
cudaError_t launch_t(const GemmMaps& maps, const uint8_t* a_scales, const uint8_t* w_scales,
                     float s_T, const uint16_t* bias, int M, int N, int K, int* dev_status,
                     int test_stall, int num_sms, cudaStream_t stream) {
  using C = Cfg<BN, RANK>;
  auto kern = k_gemm_w4a4<BN, RANK>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int tiles = ((M + BM - 1) / BM) * (N / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  kern<<<grid, NUM_THREADS, C::SMEM_BYTES, stream>>>(
      maps.a_codes, maps.w_codes, maps.lora, maps.l2s, maps.y, a_scales, w_scales, s_T, bias, M,
      N, K, dev_status, test_stall, test_stall ? 100000000ull : kWaitTimeoutNs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_w4a4(const GemmMaps& maps, int block_n, const uint8_t* a_scales,
                             const uint8_t* w_scales, float w_tensor_scale, const uint16_t* bias,
                             int M, int N, int K, int rank, int* dev_status, int test_stall,
                             int num_sms, cudaStream_t stream) {
#define SVDQ_GEMM_CASE(BN_, R_)                                                              \
  if (block_n == BN_ && rank == R_)                                                          \
    return launch_t<BN_, R_>(maps, a_scales, w_scales, w_tensor_scale, bias, M, N, K,        \
                             dev_status, test_stall, num_sms, stream);
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

#ifdef SVDQ_GEMM_TRACE
// instrumented builds only: where the first 8 CTAs write their timeline
// (1024 x u64 per CTA), or nullptr to stop
extern "C" int svdq_gemm_trace_set(unsigned long long* p) {
  return (int)cudaMemcpyToSymbol(svdq::g_gemm_trace, &p, sizeof(p));
}
#endif
