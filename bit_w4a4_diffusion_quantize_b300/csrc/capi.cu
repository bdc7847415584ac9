// C ABI of libsvdq, device side: argument validation, the compute-capability
// check (dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion
// models", hardware list: the loader validates the CUDA capability and fails
// with a clear error instead of producing wrong output), TMA descriptor
// encoding and kernel launches.  Every error is detected before anything is
// launched.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/svdq.h"
#include "../../include/svdq_test.h"
#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::atomic<int> state{0};  // 0 unknown, 1 supported, 2 unsupported
  int num_sms = 0;
};
DeviceInfo g_dev[kMaxDevices];

// Compute capability required by the sm_103a kernels.
constexpr int kMajor = 10, kMinor = 3;

// Test hooks, set only through svdq_test_set_hooks (include/svdq_test.h):
// a compute capability to report instead of the device's (10 * major +
// minor; 0 = off), and a GEMM whose loader issues nothing.
std::atomic<int> g_fake_cc{0};
std::atomic<int> g_gemm_stall{0};

svdq_status current_device(int* dev_out, int* num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SVDQ_ERR_CUDA;
  }
  // test hook (svdq_test_set_hooks): pretend the device has another compute
  // capability
  const int fake = g_fake_cc.load(std::memory_order_relaxed);
  if (fake != 0 && fake != 10 * kMajor + kMinor) return SVDQ_ERR_UNSUPPORTED_ARCH;
  DeviceInfo& d = g_dev[dev];
  int st = d.state.load(std::memory_order_acquire);
  if (st == 0) {
    int ma = 0, mi = 0, sms = 0;
    if (cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return SVDQ_ERR_CUDA;
    }
    d.num_sms = sms;
    st = (ma == kMajor && mi == kMinor) ? 1 : 2;
    d.state.store(st, std::memory_order_release);
  }
  if (st != 1) return SVDQ_ERR_UNSUPPORTED_ARCH;
  if (dev_out) *dev_out = dev;
  if (num_sms) *num_sms = d.num_sms;
  return SVDQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool rank_ok(int r) { return r == 16 || r == 32 || r == 64; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library links the CUDA runtime statically and never links libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 2-D row-major tensor of `rows` rows x `inner` elements (row pitch
// `pitch_bytes`), box `box_inner` x `box_rows`, with the given swizzle
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr, uint64_t inner,
               uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows][K/2] bytes of 4-bit codes: box 128 bytes (256 codes) x box_rows,
// 128B swizzle (the GEMM's K-major operand tiles)
bool encode_codes(CUtensorMap* map, const uint8_t* ptr, int rows, int K, int box_rows) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, (uint64_t)K / 2, (uint64_t)rows,
                   (uint64_t)K / 2, 128u, (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// [rows][rank] bf16 rank-r operand: one row per box line, swizzle span = row bytes
bool encode_rank_rows(CUtensorMap* map, const uint16_t* ptr, int rows, int rank, int box_rows) {
  const CUtensorMapSwizzle sw = rank == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : rank == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, ptr, (uint64_t)rank, (uint64_t)rows,
                   (uint64_t)rank * 2, (uint32_t)rank, (uint32_t)box_rows, sw);
}

// svdq_quantize_act and its INT4 form: the same kernel, the quantization
// step and the scale layout picked by `int4`
svdq_status quantize_act_impl(const uint16_t* X_bf16, const float* inv_lambda,
                              const uint16_t* L1s, int M, int K, int rank, uint8_t* a_codes,
                              uint8_t* a_scales, uint16_t* lora_act, int* dev_status,
                              void* stream, bool int4) {
  if (M < 0 || K <= 0 || K % 128 != 0) return SVDQ_ERR_SHAPE;
  if (!rank_ok(rank)) return SVDQ_ERR_RANK;
  if (M == 0) return SVDQ_OK;
  if (!X_bf16 || !inv_lambda || !L1s || !a_codes || !a_scales || !lora_act) return SVDQ_ERR_NULL;
  if (!aligned16(X_bf16) || !aligned16(inv_lambda) || !aligned16(L1s) || !aligned16(a_codes) ||
      !aligned16(a_scales) || !aligned16(lora_act))
    return SVDQ_ERR_ALIGN;
  svdq_status st = current_device(nullptr, nullptr);
  if (st != SVDQ_OK) return st;
  CUtensorMap tm_x, tm_l1s;
  if (!encode_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, X_bf16, (uint64_t)K, (uint64_t)M,
                 (uint64_t)K * 2, 64u, 32u, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tm_l1s, CU_TENSOR_MAP_DATA_TYPE_UINT16, L1s, (uint64_t)K, (uint64_t)rank,
                 (uint64_t)K * 2, 64u, (uint32_t)rank, CU_TENSOR_MAP_SWIZZLE_128B))
    return SVDQ_ERR_CUDA;
  cudaError_t e = svdq::launch_quantize_act(tm_x, tm_l1s, inv_lambda, M, K, rank, a_codes,
                                            a_scales, lora_act, dev_status,
                                            static_cast<cudaStream_t>(stream), int4);
  return e == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* svdq_status_string(svdq_status s) {
  switch (s) {
    case SVDQ_OK: return "SVDQ_OK";
    case SVDQ_ERR_NULL: return "SVDQ_ERR_NULL: a required pointer is NULL";
    case SVDQ_ERR_SHAPE: return "SVDQ_ERR_SHAPE: a size violates the call's shape rules";
    case SVDQ_ERR_ALIGN: return "SVDQ_ERR_ALIGN: a device pointer is not 16-byte aligned";
    case SVDQ_ERR_UNSUPPORTED_ARCH:
      return "SVDQ_ERR_UNSUPPORTED_ARCH: the NVFP4 kernels need a compute capability 10.3 "
             "(B300) device";
    case SVDQ_ERR_CUDA: return "SVDQ_ERR_CUDA: a CUDA call failed";
    case SVDQ_ERR_RANK: return "SVDQ_ERR_RANK: rank not allowed for this call";
    case SVDQ_ERR_VALUE: return "SVDQ_ERR_VALUE: a value argument is out of its domain";
    case SVDQ_ERR_NOMEM: return "SVDQ_ERR_NOMEM: host allocation failed";
  }
  return "unknown svdq_status";
}

svdq_status svdq_check_device(void) { return current_device(nullptr, nullptr); }

svdq_status svdq_quantize_act(const uint16_t* X_bf16, const float* inv_lambda,
                              const uint16_t* L1s, int M, int K, int rank, uint8_t* a_codes,
                              uint8_t* a_scales, uint16_t* lora_act, int* dev_status,
                              void* stream) {
  return quantize_act_impl(X_bf16, inv_lambda, L1s, M, K, rank, a_codes, a_scales, lora_act,
                           dev_status, stream, false);
}

svdq_status svdq_quantize_act_int4(const uint16_t* X_bf16, const float* inv_lambda,
                                   const uint16_t* L1s, int M, int K, int rank, uint8_t* a_codes,
                                   uint16_t* a_scales, uint16_t* lora_act, int* dev_status,
                                   void* stream) {
  return quantize_act_impl(X_bf16, inv_lambda, L1s, M, K, rank, a_codes,
                           reinterpret_cast<uint8_t*>(a_scales), lora_act, dev_status, stream,
                           true);
}

}  // extern "C"

namespace {

svdq_status gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* w_codes,
                      const uint8_t* w_scales, float w_tensor_scale, const uint16_t* lora_act,
                      const uint16_t* L2s, const uint16_t* bias, uint16_t* Y, int M, int N,
                      int K, int rank, svdq::GemmEpilogue epi, const svdq::QkvEpilogue& qe,
                      const svdq::GeluQuantEpilogue& gq, const uint16_t* L1s2,
                      int* dev_status, void* stream) {
  const bool is_gq = epi == svdq::GemmEpilogue::kGeluQuant;
  const bool is_qkv = epi == svdq::GemmEpilogue::kQkv;
  if (M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return SVDQ_ERR_SHAPE;
  if (is_qkv && N % 768 != 0) return SVDQ_ERR_SHAPE;  // Q, K, V: whole pairs of 128-wide heads
  if (is_gq && N % 256 != 0) return SVDQ_ERR_SHAPE;
  if (!rank_ok(rank)) return SVDQ_ERR_RANK;
  if (is_gq && gq.rank2 != 32 && gq.rank2 != 64) return SVDQ_ERR_RANK;
  if (is_qkv && !(std::isfinite(qe.eps) && qe.eps > 0.0f)) return SVDQ_ERR_VALUE;
  {
    // a finite power of two in [2^-100, 2^100]
    int ex = 0;
    const float m = std::frexp(w_tensor_scale, &ex);
    if (!std::isfinite(w_tensor_scale) || m != 0.5f || ex - 1 < -100 || ex - 1 > 100)
      return SVDQ_ERR_VALUE;
  }
  if (M == 0) return SVDQ_OK;
  if (!a_codes || !a_scales || !w_codes || !w_scales || !lora_act || !L2s || (!Y && !is_gq))
    return SVDQ_ERR_NULL;
  if (is_gq && (!gq.inv_lambda2 || !L1s2 || !gq.a2_codes || !gq.a2_scales || !gq.lora2 ||
                !gq.partial))
    return SVDQ_ERR_NULL;
  if (is_gq && gq.scratch_bytes < SVDQ_GELU_QUANT_SCRATCH_BYTES(M, N, gq.rank2))
    return SVDQ_ERR_SHAPE;
  // (the segment bookkeeping multiplies tile counts by the pair count in 32 bits)
  if (is_gq && ((size_t)M + 255) / 256 * (size_t)(N / 256) * 128 >= ((size_t)1 << 31))
    return SVDQ_ERR_SHAPE;
  if (is_qkv && (!qe.norm_q || !qe.norm_k || !qe.rope_cos || !qe.rope_sin))
    return SVDQ_ERR_NULL;
  if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) ||
      !aligned16(w_scales) || !aligned16(lora_act) || !aligned16(L2s) || (Y && !aligned16(Y)) ||
      (bias && !aligned16(bias)))
    return SVDQ_ERR_ALIGN;
  if (is_gq && (!aligned16(gq.inv_lambda2) || !aligned16(L1s2) || !aligned16(gq.a2_codes) ||
                !aligned16(gq.a2_scales) || !aligned16(gq.lora2) || !aligned16(gq.partial)))
    return SVDQ_ERR_ALIGN;
  if (is_qkv && (!aligned16(qe.norm_q) || !aligned16(qe.norm_k) || !aligned16(qe.rope_cos) ||
                 !aligned16(qe.rope_sin)))
    return SVDQ_ERR_ALIGN;
  int sms = 0;
  svdq_status st = current_device(nullptr, &sms);
  if (st != SVDQ_OK) return st;
  const int block_n = (N % 256 == 0) ? 256 : 128;
  svdq::GemmMaps maps;
  if (!encode_codes(&maps.a_codes, a_codes, M, K, 128) ||
      !encode_codes(&maps.w_codes, w_codes, N, K, block_n / 2) ||
      !encode_rank_rows(&maps.lora, lora_act, M, rank, 128) ||
      !encode_rank_rows(&maps.l2s, L2s, N, rank, block_n / 2) ||
      (Y && !encode_2d(&maps.y, CU_TENSOR_MAP_DATA_TYPE_UINT16, Y, (uint64_t)N, (uint64_t)M,
                       (uint64_t)N * 2, (uint32_t)(block_n / 4), 32u,
                       block_n == 256 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B)))
    return SVDQ_ERR_CUDA;
  if (!Y) std::memset(&maps.y, 0, sizeof(maps.y));  // GELU + quantization without H: unused
  if (is_gq) {
    if (!encode_2d(&maps.l1s2, CU_TENSOR_MAP_DATA_TYPE_UINT16, L1s2, (uint64_t)N,
                   (uint64_t)gq.rank2, (uint64_t)N * 2, 64u, (uint32_t)(gq.rank2 / 2),
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return SVDQ_ERR_CUDA;
  } else {
    std::memset(&maps.l1s2, 0, sizeof(maps.l1s2));
  }
  // test hook: the kernel's loader issues nothing, so that its pipeline waits
  // time out after 100 ms (status SVDQ_DEV_TIMEOUT)
  const int test_stall = g_gemm_stall.load(std::memory_order_relaxed) ? 1 : 0;
  cudaError_t e = svdq::launch_gemm_w4a4(maps, block_n, a_scales, w_scales, w_tensor_scale,
                                         bias, Y, M, N, K, rank, epi, qe, gq, dev_status,
                                         test_stall, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
}

}  // namespace

extern "C" {

svdq_status svdq_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales,
                           const uint8_t* w_codes, const uint8_t* w_scales,
                           float w_tensor_scale, const uint16_t* lora_act, const uint16_t* L2s,
                           const uint16_t* bias, uint16_t* Y, int M, int N, int K, int rank,
                           int* dev_status, void* stream) {
  return gemm_w4a4(a_codes, a_scales, w_codes, w_scales, w_tensor_scale, lora_act, L2s, bias, Y,
                   M, N, K, rank, svdq::GemmEpilogue::kPlain, svdq::QkvEpilogue{},
                   svdq::GeluQuantEpilogue{}, nullptr, dev_status, stream);
}

svdq_status svdq_gemm_w4a4_gelu(const uint8_t* a_codes, const uint8_t* a_scales,
                                const uint8_t* w_codes, const uint8_t* w_scales,
                                float w_tensor_scale, const uint16_t* lora_act,
                                const uint16_t* L2s, const uint16_t* bias, uint16_t* H, int M,
                                int N, int K, int rank, int* dev_status, void* stream) {
  return gemm_w4a4(a_codes, a_scales, w_codes, w_scales, w_tensor_scale, lora_act, L2s, bias, H,
                   M, N, K, rank, svdq::GemmEpilogue::kGelu, svdq::QkvEpilogue{},
                   svdq::GeluQuantEpilogue{}, nullptr, dev_status, stream);
}

svdq_status svdq_gemm_w4a4_qkv(const uint8_t* a_codes, const uint8_t* a_scales,
                               const uint8_t* w_codes, const uint8_t* w_scales,
                               float w_tensor_scale, const uint16_t* lora_act,
                               const uint16_t* L2s, const uint16_t* bias,
                               const uint16_t* norm_q, const uint16_t* norm_k,
                               const float* rope_cos, const float* rope_sin, float eps,
                               uint16_t* QKV, int M, int N, int K, int rank, int* dev_status,
                               void* stream) {
  const svdq::QkvEpilogue qe{norm_q, norm_k, rope_cos, rope_sin, eps, N / 3};
  return gemm_w4a4(a_codes, a_scales, w_codes, w_scales, w_tensor_scale, lora_act, L2s, bias,
                   QKV, M, N, K, rank, svdq::GemmEpilogue::kQkv, qe,
                   svdq::GeluQuantEpilogue{}, nullptr, dev_status, stream);
}

svdq_status svdq_gemm_w4a4_gelu_quant(const uint8_t* a_codes, const uint8_t* a_scales,
                                      const uint8_t* w_codes, const uint8_t* w_scales,
                                      float w_tensor_scale, const uint16_t* lora_act,
                                      const uint16_t* L2s, const uint16_t* bias,
                                      const float* inv_lambda2, const uint16_t* L1s2,
                                      int rank2, uint8_t* a2_codes, uint8_t* a2_scales,
                                      uint16_t* lora_act2, uint16_t* H, float* scratch,
                                      size_t scratch_bytes, int M, int N, int K, int rank,
                                      int* dev_status, void* stream) {
  const svdq::GeluQuantEpilogue gq{inv_lambda2, a2_codes, a2_scales, scratch,  H,
                                   lora_act2,   rank2,    scratch_bytes};
  return gemm_w4a4(a_codes, a_scales, w_codes, w_scales, w_tensor_scale, lora_act, L2s, bias, H,
                   M, N, K, rank, svdq::GemmEpilogue::kGeluQuant, svdq::QkvEpilogue{}, gq, L1s2,
                   dev_status, stream);
}

svdq_status svdq_gemm_w4a4_int4(const uint8_t* a_codes, const uint16_t* a_scales,
                                const uint8_t* w_codes, const uint16_t* w_scales,
                                const uint16_t* lora_act, const uint16_t* L2,
                                const uint16_t* bias, uint16_t* Y, int M, int N, int K, int rank,
                                int* dev_status, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return SVDQ_ERR_SHAPE;
  if (!rank_ok(rank)) return SVDQ_ERR_RANK;
  if (M == 0) return SVDQ_OK;
  if (!a_codes || !a_scales || !w_codes || !w_scales || !lora_act || !L2 || !Y)
    return SVDQ_ERR_NULL;
  if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(w_codes) ||
      !aligned16(w_scales) || !aligned16(lora_act) || !aligned16(L2) || !aligned16(Y) ||
      (bias && !aligned16(bias)))
    return SVDQ_ERR_ALIGN;
  svdq_status st = current_device(nullptr, nullptr);
  if (st != SVDQ_OK) return st;
  cudaError_t e = svdq::launch_gemm_int4(a_codes, a_scales, w_codes, w_scales, lora_act, L2, bias,
                                         Y, M, N, K, rank, dev_status,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
}

svdq_status awq_gemv_w4a16(const uint16_t* X_bf16, const uint8_t* qweight,
                           const uint16_t* scales, const uint16_t* zeros, const uint16_t* bias,
                           uint16_t* Y, int M, int N, int K, int group_size, int* dev_status,
                           void* stream) {
  if (M < 1 || M > 8 || N < 8 || N % 8 != 0 || K <= 0 || K % 64 != 0 ||
      K > svdq::awq_max_k() || group_size != 64)
    return SVDQ_ERR_SHAPE;
  if (!X_bf16 || !qweight || !scales || !zeros || !Y) return SVDQ_ERR_NULL;
  if (!aligned16(X_bf16) || !aligned16(qweight) || !aligned16(scales) || !aligned16(zeros) ||
      !aligned16(Y) || (bias && !aligned16(bias)))
    return SVDQ_ERR_ALIGN;
  int sms = 0;
  svdq_status st = current_device(nullptr, &sms);
  if (st != SVDQ_OK) return st;
  cudaError_t e = svdq::launch_awq_gemv(qweight, X_bf16, scales, zeros, bias, Y, M, N, K,
                                        dev_status, static_cast<cudaStream_t>(stream), sms);
  return e == cudaSuccess ? SVDQ_OK : SVDQ_ERR_CUDA;
}

}  // extern "C"

namespace {

// Scratch of svdq_gemm_w4a4_gelu_quant_static: one fixed array in device
// global memory, part of this library's device image (it exists on a device
// once the library's kernels are loaded there), shared by every call on that
// device.  Its address is looked up once per device.
static __device__ __align__(256) float g_gq_static_scratch[SVDQ_GELU_QUANT_STATIC_SCRATCH_BYTES /
                                                           sizeof(float)];
std::atomic<float*> g_gq_static_ptr[kMaxDevices];
std::mutex g_gq_static_mu;

float* gq_static_scratch(int dev) {
  float* p = g_gq_static_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_gq_static_mu);
  p = g_gq_static_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_gq_static_scratch) != cudaSuccess || !a) {
      cudaGetLastError();
      return nullptr;
    }
    p = static_cast<float*>(a);
    g_gq_static_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace

extern "C" svdq_status svdq_gemm_w4a4_gelu_quant_static(
    const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* w_codes,
    const uint8_t* w_scales, float w_tensor_scale, const uint16_t* lora_act, const uint16_t* L2s,
    const uint16_t* bias, const float* inv_lambda2, const uint16_t* L1s2, int rank2,
    uint8_t* a2_codes, uint8_t* a2_scales, uint16_t* lora_act2, uint16_t* H, int M, int N, int K,
    int rank, int* dev_status, void* stream) {
  if (M < 0 || N <= 0 || N % 256 != 0) return SVDQ_ERR_SHAPE;
  if (rank2 != 32 && rank2 != 64) return SVDQ_ERR_RANK;
  if (SVDQ_GELU_QUANT_SCRATCH_BYTES(M, N, rank2) > SVDQ_GELU_QUANT_STATIC_SCRATCH_BYTES)
    return SVDQ_ERR_SHAPE;  // more rows than the static scratch holds
  if (M == 0)
    return svdq_gemm_w4a4_gelu_quant(a_codes, a_scales, w_codes, w_scales, w_tensor_scale,
                                     lora_act, L2s, bias, inv_lambda2, L1s2, rank2, a2_codes,
                                     a2_scales, lora_act2, H, nullptr, 0, M, N, K, rank,
                                     dev_status, stream);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SVDQ_ERR_CUDA;
  }
  // (the architecture check first: the device image holding the array loads
  // only on a supported device)
  svdq_status st = current_device(nullptr, nullptr);
  if (st != SVDQ_OK) return st;
  float* scratch = gq_static_scratch(dev);
  if (!scratch) return SVDQ_ERR_CUDA;
  return svdq_gemm_w4a4_gelu_quant(a_codes, a_scales, w_codes, w_scales, w_tensor_scale,
                                   lora_act, L2s, bias, inv_lambda2, L1s2, rank2, a2_codes,
                                   a2_scales, lora_act2, H, scratch,
                                   SVDQ_GELU_QUANT_STATIC_SCRATCH_BYTES, M, N, K, rank,
                                   dev_status, stream);
}

extern "C" svdq_status svdq_test_set_hooks(int fake_compute_capability, int gemm_stall) {
  if (fake_compute_capability < 0 || (gemm_stall != 0 && gemm_stall != 1)) return SVDQ_ERR_VALUE;
  g_fake_cc.store(fake_compute_capability, std::memory_order_relaxed);
  g_gemm_stall.store(gemm_stall, std::memory_order_relaxed);
  return SVDQ_OK;
}
