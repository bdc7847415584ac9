// Device helpers shared by the sm_103a kernels of libsvdq: bf16/e4m3/e2m1
// conversions, cache-hinted loads, mbarrier / TMA / tcgen05 wrappers written
// from the PTX ISA, and bounded waits that report a timeout instead of
// hanging.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#define SVDQ_DEVINL __device__ __forceinline__

namespace svdq {

// Pipeline waits give up after this many nanoseconds (%globaltimer) and
// report SVDQ_DEV_TIMEOUT through the status word.  A healthy wait lasts
// microseconds; this bound only keeps a broken pipeline from hanging.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr int kDevTimeout = 1;

SVDQ_DEVINL uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

SVDQ_DEVINL void report_timeout(int* status) {
  if (status) atomicExch(status, kDevTimeout);
}

// ---------------------------------------------------------------- loads
SVDQ_DEVINL uint4 ld_stream_v4(const void* p) {  // read-once data: bypass L1
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
SVDQ_DEVINL uint4 ld_keep_v4(const void* p) {  // data re-read by other warps
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
SVDQ_DEVINL float4 ld_keep_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// ---------------------------------------------------------------- formats
SVDQ_DEVINL float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
SVDQ_DEVINL float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

SVDQ_DEVINL uint16_t f32_to_bf16_rn(float f) {
  // round to nearest even; NaN kept quiet
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// e4m3 (OCP FN) byte of a non-negative float: nearest, ties to even,
// saturating at 448 (PTX cvt with .satfinite).
SVDQ_DEVINL uint32_t f32_to_e4m3_sat(float v) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(0.0f), "f"(v));
  return (uint32_t)(d & 0xFFu);
}

// value of a non-negative finite e4m3 byte (0x00..0x7E)
SVDQ_DEVINL float e4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  return e == 0 ? (float)m * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight floats -> eight e2m1 codes in one 32-bit word, element 2i in the low
// nibble of byte i (PTX cvt.rn.satfinite.e2m1x2: the first source goes to
// the high nibble).  Round to nearest even, saturating at +-6.
SVDQ_DEVINL uint32_t f32x8_to_e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                     float v5, float v6, float v7) {
  uint32_t out;
  asm("{\n"
      ".reg .b8 q0, q1, q2, q3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n"
      "mov.b32 %0, {q0, q1, q2, q3};\n"
      "}"
      : "=r"(out)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return out;
}

// ---------------------------------------------------------------- warp MMA
// D[16x8] += A[16x16] B[16x8], bf16 inputs, fp32 accumulate (legacy warp MMA;
// used for the rank-r down projection inside the activation kernel).
SVDQ_DEVINL void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// packed fp32 pairs (sm_100+): two IEEE binary32 operations, each rounded to
// nearest even exactly as the scalar instruction would
SVDQ_DEVINL float2 mul2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n.reg .b64 ra, rb, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "mul.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
SVDQ_DEVINL float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n.reg .b64 ra, rb, rc, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "mov.b64 rc, {%6, %7};\nfma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// ---------------------------------------------------------------- shared memory / mbarrier
SVDQ_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SVDQ_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
SVDQ_DEVINL void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
SVDQ_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n.reg .b64 st;\n"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
      : "memory");
}
SVDQ_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n.reg .b64 st;\n"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
// Suspend-time hint of mbarrier.try_wait in ns (0: the instruction's default).
#ifndef SVDQ_TRY_WAIT_HINT_NS
#define SVDQ_TRY_WAIT_HINT_NS 0
#endif
SVDQ_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
#if SVDQ_TRY_WAIT_HINT_NS > 0
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"((uint32_t)SVDQ_TRY_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}
// Non-blocking test of an mbarrier phase (never suspends).
SVDQ_DEVINL bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase.  Returns false (and reports) on timeout.
SVDQ_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                           uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) {
      report_timeout(status);
      return false;
    }
  }
}
SVDQ_DEVINL void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
// 2-D tiled bulk tensor load global -> shared, completion on an mbarrier.
SVDQ_DEVINL void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// hint: bring a 2-D box of a tensor map into L2 (no data comes back)
SVDQ_DEVINL void tma_prefetch_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap),
               "r"(x), "r"(y)
               : "memory");
}
// 3-D tiled bulk tensor load global -> shared, completion on an mbarrier.
SVDQ_DEVINL void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar, int x, int y,
                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
SVDQ_DEVINL void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// ---------------------------------------------------------------- dependent launch
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream finishes.
// grid_dep_wait blocks until that kernel has completed and its writes are
// visible (a no-op otherwise): every global access of the library's kernels
// comes after it, so only set-up work overlaps.  grid_dep_launch lets the
// next kernel on the stream be scheduled early.
SVDQ_DEVINL void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SVDQ_DEVINL void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// ---------------------------------------------------------------- clusters
SVDQ_DEVINL uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of every CTA of the cluster (release/acquire)
SVDQ_DEVINL void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
// hint: bring `bytes` (a multiple of 16, 16-byte aligned) at p into L2; no
// data is returned to the issuing CTA and nothing waits for it
SVDQ_DEVINL void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
// hint: bring the 128-byte line at p into L2 (no data returned)
SVDQ_DEVINL void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// per-thread asynchronous copy global -> shared of 4 or 8 bytes; src_bytes = 0
// writes zeros (nothing is read)
template <int BYTES>
SVDQ_DEVINL void cp_async(void* smem_dst, const void* gsrc, int src_bytes) {
  static_assert(BYTES == 4 || BYTES == 8, "cp.async.ca size");
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(smem_u32(smem_dst)),
               "l"(gsrc), "n"(BYTES), "r"(src_bytes)
               : "memory");
}
// 16 bytes, cached in L2 only (read-once streams)
SVDQ_DEVINL void cp_async16_cg(void* smem_dst, const void* gsrc, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(gsrc), "r"(src_bytes)
               : "memory");
}
SVDQ_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
SVDQ_DEVINL void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// 2-D tiled TMA store of a shared-memory box to global memory (bulk group)
SVDQ_DEVINL void tma_store_2d(const void* tmap, const void* smem_src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
      :
      : "l"(tmap), "r"(smem_u32(smem_src)), "r"(x), "r"(y)
      : "memory");
}
SVDQ_DEVINL void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the source shared memory of every committed bulk store may be reused
SVDQ_DEVINL void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed bulk store has completed
SVDQ_DEVINL void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
SVDQ_DEVINL void sts128(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}

SVDQ_DEVINL void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------- tcgen05
SVDQ_DEVINL void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
SVDQ_DEVINL void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// whole warp: allocate `ncols` TMEM columns, base address written to smem
SVDQ_DEVINL void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SVDQ_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// commit all prior tcgen05 async ops of this thread to an mbarrier (1 arrive)
SVDQ_DEVINL void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// ---- CTA-pair forms (cta_group::2): one MMA spans the TMEM lanes of two SMs.
// Allocation and release are collective: one warp of each CTA of the pair
// executes them, with the same column count, while both CTAs are resident.
SVDQ_DEVINL void tmem_alloc_pair(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
SVDQ_DEVINL void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// shared::cluster address of the object at CTA-local shared address `saddr`
// in CTA `rank` of the cluster
SVDQ_DEVINL uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// one arrive on an mbarrier given by its shared::cluster address (this CTA's
// or the peer's).  Default semantics (release, CTA scope) as for a local
// arrive: what the pair signals this way is the completion of work that is
// already finished where it happened (TMEM stores waited for with
// tcgen05.wait::st, TMA copies whose barrier phase completed, TMEM loads
// waited for with tcgen05.wait::ld).  A cluster-scope release or acquire
// costs about half a microsecond per use on this part.
SVDQ_DEVINL void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// completion of every prior tcgen05 async op of this thread (pair MMAs) as one
// arrive on the mbarrier at shared::cluster address `cluster_addr`
SVDQ_DEVINL void tc_commit_pair(uint32_t cluster_addr) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          cluster_addr)
      : "memory");
}
// pair NVFP4 MMA (issued by one thread of the even CTA): D rows 0-127 in the
// even CTA's TMEM, 128-255 in the odd CTA's; each CTA supplies its own 128 A
// rows and one half of the B rows from its shared memory at the same offsets;
// scale addresses name the same TMEM columns in both CTAs
SVDQ_DEVINL void tc_mma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                  uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                  uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.u32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
SVDQ_DEVINL void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Warp-wide forms of the pair MMA and commit: every lane of a converged warp
// executes them with the same (warp-uniform) operands and one lane, picked by
// elect.sync, issues the instruction.  Kept warp-uniform, the operands stay in
// uniform registers: the issue of a tcgen05 instruction from one divergent
// lane costs about 75 cycles of operand moves, more than the tensor cores
// need to run an NVFP4 MMA when back-to-back issue is what keeps them busy.
SVDQ_DEVINL void tc_mma_nvf4_pair_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p, e;\n"
      "setp.ne.u32 p, %6, 0;\n"
      "elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
SVDQ_DEVINL void tc_mma_bf16_pair_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p, e;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// the same commit to two barriers (one elected lane issues both)
SVDQ_DEVINL void tc_commit_pair_warp2(uint32_t cluster_addr0, uint32_t cluster_addr1) {
  asm volatile(
      "{\n.reg .pred e;\n"
      "elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%1];\n}" ::"r"(
          cluster_addr0),
      "r"(cluster_addr1)
      : "memory");
}
SVDQ_DEVINL void tc_commit_pair_warp(uint32_t cluster_addr) {
  asm volatile(
      "{\n.reg .pred e;\n"
      "elect.sync _|e, 0xffffffff;\n"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(
          cluster_addr)
      : "memory");
}
// block-scaled NVFP4 MMA: D(tmem) (+)= A(smem) x B(smem), scales in TMEM
SVDQ_DEVINL void tc_mma_nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.u32 p, %6, 0;\n"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// bf16 MMA: D(tmem) (+)= A(smem) x B(smem), fp32 accumulate
SVDQ_DEVINL void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                             uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\n"
      "setp.ne.u32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// copy a 32-row x 16-byte matrix from shared memory into TMEM, replicated to
// the four 32-lane quarters (block-scale factors)
SVDQ_DEVINL void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// each thread of the warp loads 32 consecutive fp32 columns of its lane
SVDQ_DEVINL void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
SVDQ_DEVINL void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// each thread of the warp stores 4 consecutive 32-bit columns of its lane
SVDQ_DEVINL void tmem_st_32x32b_x4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
SVDQ_DEVINL void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
SVDQ_DEVINL uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), fixed version field 1 at bit 46, layout
// (swizzle) type in bits 61..63.
enum SmemLayout : uint32_t {
  kSwizzleNone = 0,
  kSwizzle128B = 2,
  kSwizzle64B = 4,
  kSwizzle32B = 6
};
SVDQ_DEVINL uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                               SmemLayout layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= (uint64_t)layout << 61;
  return d;
}

}  // namespace svdq
