/*
 * svdq.h -- C ABI of libsvdq: the SVDQuant W4A4 (NVFP4) linear layer of a
 * diffusion transformer and the AWQ W4A16 modulation GEMV, for NVIDIA B300
 * (compute capability 10.3, sm_103a).
 *
 * What the layer computes (source pages: news articles on "Nunchaku Lite" in
 * Diffusers):
 *   - dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion models",
 *     SVDQuant paragraph: activation outliers are moved into the weights; the
 *     hardest part of each weight matrix becomes a small 16-bit low-rank
 *     branch; the residual is quantized to 4 bit.
 *   - same page, fused-kernel paragraph: the low-rank down projection is fused
 *     with the quantization kernel and the low-rank up projection with the
 *     4-bit compute kernel.
 *   - same page, "quantization_config" block: svdq_w4a4 precision "nvfp4",
 *     group_size 16, rank 32; awq_w4a16 precision "int4", group_size 64;
 *     compute_dtype "bfloat16".
 *   - same page, kernel-family list: svdq_w4a4 for attention/MLP projections,
 *     awq_w4a16 for the precision-sensitive, memory-bound modulation layers.
 *   - same page, hardware list: the loader checks the device's CUDA compute
 *     capability and raises a clear error instead of producing wrong output.
 *   - same page, on the full engine's model-specific fused paths and its
 *     structural rewrites: fused QKV projections whose single operator also
 *     normalizes Q and K and applies the rotary embeddings, and fused
 *     GELU/MLP kernels -- here svdq_gemm_w4a4_qkv and svdq_gemm_w4a4_gelu,
 *     the same 4-bit product with those steps in its epilogue.
 *
 *   Y = Q4(X_hat) Q4(R) s_T + (X L1s) L2 + b,    X_hat = X diag(inv_lambda)
 *
 * Fixed rules (the pages name the formats, not the rounding):
 *   e2m1 codes: nearest value of {0,0.5,1,1.5,2,3,4,6}, ties to the even
 *   code, saturating at 6; the code's sign bit is the input's sign bit.
 *   e4m3 (OCP "FN", bias 7) scales: nearest, ties to even, saturating at 448.
 *   Activation block scale s = RNE_e4m3(amax/6) over 16 consecutive k of
 *   x_hat = fl32(x * inv_lambda[k]); codes RNE_e2m1(x_hat / s) (exact real
 *   quotients); a block whose s is 0 gets codes +0.  Activations carry no
 *   tensor scale.  Weights: see svdq_pack_weights.
 *
 * Conventions
 *   - Every buffer is owned by the caller.  Device calls take device
 *     pointers (from cudaMalloc or a framework allocator) and never allocate
 *     device memory; host calls take host pointers.
 *   - Device calls are asynchronous and ordered on `stream` (a cudaStream_t
 *     passed as void*; NULL is the legacy default stream).  A call that
 *     returns an error status has launched nothing.
 *   - bf16 / fp16 tensors are passed as uint16_t bit patterns.
 *   - `dev_status` (nullable) is a device int the kernels write only on a
 *     device-side condition: SVDQ_DEV_TIMEOUT if an internal pipeline wait
 *     exceeded its bound (the kernel then abandons the tile and returns; the
 *     output is incomplete).  Initialise it to 0; read it after the stream
 *     synchronises.
 *   - Device calls return SVDQ_ERR_UNSUPPORTED_ARCH unless the current device
 *     has compute capability 10.3.
 *   - Device pointers must be 16-byte aligned (SVDQ_ERR_ALIGN otherwise).
 *
 * Data layouts (device calls; the packer writes the weight side)
 *   codes    [rows][K/2] bytes, row-major; element 2i of a row in the low
 *            nibble of byte i, element 2i+1 in the high nibble.
 *   scales   e4m3 bytes of a rows x C matrix (C = K/16) in 512-byte tiles:
 *            rows form 128-row blocks rb = r/128, columns 4-column groups
 *            cb = c/4; tile (rb, cb) starts at byte (rb*(C/4) + cb)*512 and
 *            holds entry (r, c) at byte (r%32)*16 + ((r/32)%4)*4 + c%4.
 *            The buffer holds ceil(rows/128) row blocks
 *            (SVDQ_SCALE_BYTES(rows, K)); padding rows are neither written
 *            nor used.  This is the order in which the tensor core reads
 *            block scales, so the GEMM copies them without reshuffling.
 *   lora     [M][rank] bf16 row-major (lora_act).
 *   L1s      [rank][K] bf16: the K x rank down-projection factor stored
 *            transposed (row i = column i of L1s, k contiguous).
 *   L2s      [N][rank] bf16: the rank x N up-projection factor transposed
 *            and divided by the weight tensor scale, L2s[n][i] = L2[i][n] / s_T
 *            (exact for a power-of-two s_T unless the quotient leaves the bf16
 *            normal range), so that the tensor cores can add the rank-r term
 *            into the same accumulator as the 4-bit product.
 *   Y [M][N] bf16;  bias [N] bf16.
 */
#ifndef SVDQ_H_
#define SVDQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SVDQ_OK = 0,
  SVDQ_ERR_NULL = -1,             /* a required pointer is NULL */
  SVDQ_ERR_SHAPE = -2,            /* a size violates the call's shape rules */
  SVDQ_ERR_ALIGN = -3,            /* a device pointer is not 16-byte aligned */
  SVDQ_ERR_UNSUPPORTED_ARCH = -4, /* current device is not compute capability 10.3 */
  SVDQ_ERR_CUDA = -5,             /* a CUDA runtime/driver call failed */
  SVDQ_ERR_RANK = -6,             /* rank not allowed for this call */
  SVDQ_ERR_VALUE = -7,            /* a value argument is out of its domain */
  SVDQ_ERR_NOMEM = -8             /* host scratch allocation failed (packers) */
} svdq_status;

/* values written to *dev_status by a kernel */
#define SVDQ_DEV_OK 0
#define SVDQ_DEV_TIMEOUT 1

/* byte sizes of the packed buffers */
#define SVDQ_CODE_BYTES(rows, K) ((size_t)(rows) * (size_t)(K) / 2)
#define SVDQ_SCALE_BYTES(rows, K) ((((size_t)(rows) + 127) / 128) * 128 * ((size_t)(K) / 16))
/* device scratch of svdq_gemm_w4a4_gelu_quant: fp32 segment sums of the next
 * layer's down projection, 128 + ceil(M/256) slots of 256 x rank2 (N is not
 * used: every N takes the same) */
#define SVDQ_GELU_QUANT_SCRATCH_BYTES(M, N, rank2) \
  ((128 + ((size_t)(M) + 255) / 256) * 256 * (size_t)(rank2) * 4)

/* Human-readable name of a status code (static string). */
const char* svdq_status_string(svdq_status s);

/* SVDQ_OK if the current CUDA device has compute capability 10.3, else
 * SVDQ_ERR_UNSUPPORTED_ARCH (or SVDQ_ERR_CUDA if no device can be queried).
 * The pages' hardware list: the quantizer validates the compute capability
 * and fails clearly rather than producing wrong output. */
svdq_status svdq_check_device(void);

/* ------------------------------------------------------------------ host */

/* Calibration statistic of the smoothing step: x_absmax[j] = max_m |X[m][j]|
 * over M rows of bf16 activations X [M][K] (host).  M may be 0 (all zeros).
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE (M < 0 or K <= 0). */
svdq_status svdq_calib_absmax(const uint16_t* X_bf16, int64_t M, int64_t K,
                              float* x_absmax);

/* Offline packing of one nn.Linear weight W [N][K] (fp32, host, row-major)
 * into the SVDQ W4A4 form (the SVDQuant paragraph: smoothing, 16-bit low-rank
 * branch, 4-bit residual).  Synchronous, host only, thread-safe; allocates
 * and frees its own host scratch.
 *
 *   lambda_j   = sqrt(x_absmax[j] / max_n |W[n][j]|), 1 if either is 0,
 *                clamped to [2^-20, 2^20];  inv_lambda[j] = fl32(1/lambda_j)
 *   W_hat^T    = diag(1/inv_lambda) W^T  (K x N, float64)
 *   L1 L2      = rank-r truncated SVD of W_hat^T (L1 = U_r S_r, L2 = V_r^T),
 *                by randomized subspace iteration with a Jacobi SVD of the
 *                projected matrix (full Jacobi SVD when min(K, N) is small)
 *   L1s        = bf16(inv_lambda[k] * L1[k][i])   -> out [rank][K] (transposed)
 *   L2b        = bf16(L2)
 *   R[k][n]    = (W[n][k] - sum_{i ascending} L1s[k][i] L2b[i][n]) / inv_lambda[k]
 *                (float64, one rounding per operation, no fused multiply-add)
 *   s_T        = smallest power of two with 6*448*s_T >= max|R| (1 if R == 0),
 *                within [2^-100, 2^100] (SVDQ_ERR_VALUE otherwise)
 *   L2s        = L2b^T / s_T (exact)                 -> out [N][rank]
 *   w_scales   = RNE_e4m3(amax16 / (6 s_T)) per 16 consecutive k of each
 *                output channel n, in the scale tile layout (rows = N)
 *   w_codes    = RNE_e2m1(R[k][n] / (s_b s_T)), [N][K/2] packed
 *
 * Sizes: N % 128 == 0, K % 128 == 0, 1 <= rank <= min(K, N).  Buffers:
 * inv_lambda [K], L1s [rank*K], L2s [N*rank], w_codes SVDQ_CODE_BYTES(N, K),
 * w_scales SVDQ_SCALE_BYTES(N, K), w_tensor_scale [1].
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE, SVDQ_ERR_RANK, SVDQ_ERR_VALUE
 * (non-finite W or x_absmax, or a residual beyond the float range),
 * SVDQ_ERR_NOMEM. */
svdq_status svdq_pack_weights(const float* W, int N, int K, const float* x_absmax,
                              int rank, float* inv_lambda, uint16_t* L1s,
                              uint16_t* L2s, uint8_t* w_codes, uint8_t* w_scales,
                              float* w_tensor_scale);

/* Offline packing of a modulation-layer weight W [N][K] (fp32, host) to AWQ
 * W4A16 (kernel-family list: 4-bit weights, 16-bit activations; config block:
 * int4, group_size 64).  Plain asymmetric group quantization along K, per
 * output channel and group g of 64 consecutive k:
 *   s = fp16((max - min) / 15), z = fp16(-min / s) clamped to +-65504,
 *   q = clamp(RNE(w / s + z), 0, 15)  (float64 before the fp16 roundings);
 *   a group with max == min, or whose s rounds to 0, uses s = 1, z = fp16(-min).
 * Outputs: qweight [N][K/2] bytes (even k in the low nibble), scales and
 * zeros [N][K/64] fp16 bit patterns.
 * Sizes: K % 64 == 0, N >= 1, group_size == 64.
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE, SVDQ_ERR_VALUE (non-finite W). */
svdq_status awq_pack_weights(const float* W, int N, int K, int group_size,
                             uint8_t* qweight, uint16_t* scales, uint16_t* zeros);

/* INT4 variant of the SVDQ W4A4 layer (dothoosh.com, "How Nunchaku Lite
 * halves the VRAM of diffusion models", kernel-family list: svdq_w4a4 in INT4
 * and NVFP4 variants; hardware list: INT4 is the pre-Blackwell format; the
 * config block's int4 group size, 64).  4-bit values are signed integers
 * -8..7 (two's complement nibbles, same byte order as the NVFP4 codes) with
 * one bf16 scale per 64 consecutive k, row-major [rows][K/64]:
 *   s = RNE_bf16(amax64 / 7),  q = clamp(RNE(v / s), -8, 7),
 *   a group whose scale is 0 (or, for activations, not finite) has codes 0.
 * SVDQ_INT4_SCALE_BYTES(rows, K) is the size of a scale buffer. */
#define SVDQ_INT4_SCALE_BYTES(rows, K) ((size_t)(rows) * ((size_t)(K) / 64) * 2)

/* Offline packing, INT4 variant: smoothing, low-rank factors and residual R
 * exactly as svdq_pack_weights, then per output channel and 64-group of R:
 *   w_scales = bf16(amax / 7) (float64 quotient),  w_codes = clamp(RNE(R /
 *   s), -8, 7) (float64 quotient, ties to even).
 * No tensor scale: L2 is bf16(L2) transposed, [N][rank].
 * Sizes: N % 128 == 0, K % 128 == 0, 1 <= rank <= min(K, N).  Buffers:
 * inv_lambda [K], L1s [rank*K], L2 [N*rank], w_codes SVDQ_CODE_BYTES(N, K),
 * w_scales SVDQ_INT4_SCALE_BYTES(N, K) (bf16 bit patterns).
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE, SVDQ_ERR_RANK, SVDQ_ERR_VALUE
 * (non-finite W, x_absmax or residual), SVDQ_ERR_NOMEM. */
svdq_status svdq_pack_weights_int4(const float* W, int N, int K, const float* x_absmax,
                                   int rank, float* inv_lambda, uint16_t* L1s,
                                   uint16_t* L2, uint8_t* w_codes, uint16_t* w_scales);

/* ---------------------------------------------------------------- device */

/* Activation side of the SVDQ linear, one kernel (fused-kernel paragraph:
 * the low-rank down projection runs inside the quantization kernel).
 * Reads X once:
 *   lora_act[m][i] = bf16(sum_k X[m][k] L1s[k][i])   (fp32 accumulation on
 *                    tensor cores; L1s already carries inv_lambda)
 *   x_hat          = fl32(X[m][k] * inv_lambda[k])
 *   a_scales       = RNE_e4m3(amax16(x_hat) / 6)   (scale tile layout, rows = M)
 *   a_codes        = RNE_e2m1(x_hat / s)           ([M][K/2] packed)
 * Inputs: X [M][K] bf16, inv_lambda [K] fp32, L1s [rank][K] bf16.
 * Outputs: a_codes SVDQ_CODE_BYTES(M, K), a_scales SVDQ_SCALE_BYTES(M, K),
 * lora_act [M][rank] bf16.
 * Sizes: M >= 0 (M == 0 launches nothing), K % 128 == 0, rank in {16, 32, 64}.
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE, SVDQ_ERR_RANK, SVDQ_ERR_ALIGN,
 * SVDQ_ERR_UNSUPPORTED_ARCH, SVDQ_ERR_CUDA (launch failure). */
svdq_status svdq_quantize_act(const uint16_t* X_bf16, const float* inv_lambda,
                              const uint16_t* L1s, int M, int K, int rank,
                              uint8_t* a_codes, uint8_t* a_scales,
                              uint16_t* lora_act, int* dev_status, void* stream);

/* The 4-bit product with the low-rank up projection and bias fused in its
 * epilogue (fused-kernel paragraph: up projection fused with the 4-bit
 * compute kernel):
 *   Y = bf16( s_T * sum_k dec(a)[m][k] dec(w)[n][k]
 *             + sum_i lora_act[m][i] L2s[n][i] * s_T + bias[n] )
 * dec(.) = e2m1 value x e4m3 block scale.  tcgen05 block-scaled NVFP4 MMA
 * with fp32 accumulators in tensor memory; operands and scales staged by TMA.
 * The rank-r term is accumulated on the tensor cores into the same fp32
 * accumulator (L2s already carries 1/s_T; s_T must be a power of two, as
 * svdq_pack_weights produces).  Persistent kernel, one CTA per SM.
 * Inputs: activation side as written by svdq_quantize_act (rows = M), weight
 * side as written by svdq_pack_weights (rows = N), bias nullable.
 * Output: Y [M][N] bf16.
 * Sizes: M >= 0 (M == 0 launches nothing), N % 128 == 0, K % 128 == 0,
 * rank in {16, 32, 64}; w_tensor_scale a finite power of two in
 * [2^-100, 2^100] (SVDQ_ERR_VALUE otherwise).
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE, SVDQ_ERR_RANK, SVDQ_ERR_VALUE,
 * SVDQ_ERR_ALIGN, SVDQ_ERR_UNSUPPORTED_ARCH, SVDQ_ERR_CUDA. */
svdq_status svdq_gemm_w4a4(const uint8_t* a_codes, const uint8_t* a_scales,
                           const uint8_t* w_codes, const uint8_t* w_scales,
                           float w_tensor_scale, const uint16_t* lora_act,
                           const uint16_t* L2s, const uint16_t* bias, uint16_t* Y,
                           int M, int N, int K, int rank, int* dev_status,
                           void* stream);

/* svdq_gemm_w4a4 with GELU (tanh form) fused into its epilogue, for the first
 * linear of a transformer MLP (dothoosh.com, "How Nunchaku Lite halves the
 * VRAM of diffusion models": the full engine's fused GELU/MLP kernels):
 *   H = bf16( gelu_tanh( Y ) ),  gelu_tanh(y) = 0.5 y (1 + tanh( sqrt(2/pi)
 *                                               (y + 0.044715 y^3) ))
 * where Y is exactly the bf16 output svdq_gemm_w4a4 returns for the same
 * arguments (GELU acts on the rounded value, as an unfused GELU on that output
 * would); gelu_tanh is evaluated in fp32 (relative error below 2^-16 for
 * |y| <= 8; the values beyond that are y itself or negligible), then rounded to
 * nearest even.  H [M][N] bf16 takes the place of Y; every other argument,
 * size rule and error is that of svdq_gemm_w4a4. */
svdq_status svdq_gemm_w4a4_gelu(const uint8_t* a_codes, const uint8_t* a_scales,
                                const uint8_t* w_codes, const uint8_t* w_scales,
                                float w_tensor_scale, const uint16_t* lora_act,
                                const uint16_t* L2s, const uint16_t* bias, uint16_t* H,
                                int M, int N, int K, int rank, int* dev_status,
                                void* stream);

/* svdq_gemm_w4a4_gelu for the first linear of an MLP whose output feeds the
 * second SVDQ linear, with that second layer's activation side
 * (svdq_quantize_act) fused into the epilogue as well (dothoosh.com, "How
 * Nunchaku Lite halves the VRAM of diffusion models": the full engine's fused
 * GELU/MLP kernels; the fused-kernel paragraph: the down projection runs with
 * the quantization).  With H the bf16 GELU output svdq_gemm_w4a4_gelu returns
 * for the same arguments, the outputs are exactly
 *   a2_codes, a2_scales = those of svdq_quantize_act(H, inv_lambda2, K = N)
 * (bit for bit), and
 *   lora_act2[m][i] = bf16( sum_n H[m][n] L1s2[i][n] )
 * accumulated in fp32 on the tensor cores.  The GEMM's persistent CTA pairs
 * each take one contiguous range of 256 x 256 output tiles (m-pair-major); a
 * pair accumulates the down projection in tensor memory over its tiles of one
 * 256-row block and writes that fp32 segment sum to `scratch`; a second kernel
 * adds the (at most a few) segment sums of each row in ascending pair order
 * and rounds once.  H itself is written to `H` only when `H` is non-null.
 * Inputs: as svdq_gemm_w4a4_gelu; inv_lambda2 [N] fp32 and L1s2 [rank2][N]
 * bf16 of the second layer (svdq_pack_weights of that layer, K = N).
 * Outputs: a2_codes SVDQ_CODE_BYTES(M, N), a2_scales SVDQ_SCALE_BYTES(M, N)
 * (rows past M in the last 128-row tile are not written), lora_act2
 * [M][rank2] bf16, H [M][N] bf16 (nullable).
 * Scratch: `scratch` (device, caller-owned, contents on entry irrelevant, left
 * holding the partial sums) of scratch_bytes >=
 * SVDQ_GELU_QUANT_SCRATCH_BYTES(M, N, rank2) (SVDQ_ERR_SHAPE otherwise).
 * Two kernels on `stream` (the second overlaps the first's tail through
 * programmatic dependent launch).
 * Sizes: N % 256 == 0, rank2 in {32, 64} (SVDQ_ERR_RANK otherwise); everything
 * else as svdq_gemm_w4a4. */
svdq_status svdq_gemm_w4a4_gelu_quant(const uint8_t* a_codes, const uint8_t* a_scales,
                                      const uint8_t* w_codes, const uint8_t* w_scales,
                                      float w_tensor_scale, const uint16_t* lora_act,
                                      const uint16_t* L2s, const uint16_t* bias,
                                      const float* inv_lambda2, const uint16_t* L1s2,
                                      int rank2, uint8_t* a2_codes, uint8_t* a2_scales,
                                      uint16_t* lora_act2, uint16_t* H, float* scratch,
                                      size_t scratch_bytes, int M, int N, int K, int rank,
                                      int* dev_status, void* stream);

/* svdq_gemm_w4a4_gelu_quant without caller scratch: the scratch is a fixed
 * array of SVDQ_GELU_QUANT_STATIC_SCRATCH_BYTES in device global memory that
 * belongs to this library (loaded with its kernels, one per device, never
 * allocated or freed by the call).  This call has no counterpart in the
 * method's description; it exists for callers that cannot allocate device
 * memory at the point of the call: a runtime with a fixed device-memory
 * budget that hands out no scratch, or a loop that must never block on or
 * fail in an allocator.
 * Limits and rules:
 *   - SVDQ_GELU_QUANT_SCRATCH_BYTES(M, N, rank2) must not exceed
 *     SVDQ_GELU_QUANT_STATIC_SCRATCH_BYTES: rank2 32 allows M <= 98304,
 *     rank2 64 allows M <= 32768 (SVDQ_ERR_SHAPE beyond).
 *   - The first call on a device (that device current) looks up the array's
 *     address (cudaGetSymbolAddress, which may load the library's device
 *     code): make one call on each device before any stream capture.
 *     SVDQ_ERR_CUDA if the lookup fails.
 *   - Nothing in the array needs to start at zero: a call writes every part
 *     it later reads.
 *   - Every call on a device uses the same array: two calls whose work
 *     overlaps in time (different streams, or different host threads on
 *     unsynchronised streams) race on it and give wrong results.  Order the
 *     calls on one stream, or use svdq_gemm_w4a4_gelu_quant with separate
 *     scratch buffers.
 * Everything else (arguments, outputs, sizes, errors) is that of
 * svdq_gemm_w4a4_gelu_quant. */
#define SVDQ_GELU_QUANT_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
svdq_status svdq_gemm_w4a4_gelu_quant_static(
    const uint8_t* a_codes, const uint8_t* a_scales, const uint8_t* w_codes,
    const uint8_t* w_scales, float w_tensor_scale, const uint16_t* lora_act,
    const uint16_t* L2s, const uint16_t* bias, const float* inv_lambda2,
    const uint16_t* L1s2, int rank2, uint8_t* a2_codes, uint8_t* a2_scales,
    uint16_t* lora_act2, uint16_t* H, int M, int N, int K, int rank, int* dev_status,
    void* stream);

/* svdq_gemm_w4a4 for a fused Q|K|V projection, with the normalization of Q and
 * K and the rotary embedding in its epilogue (dothoosh.com, "How Nunchaku Lite
 * halves the VRAM of diffusion models", paragraphs on structural rewrites:
 * to_q, to_k, to_v joined along the output dimension in the order Q, K, V, and
 * one fused operator for the projection, the Q/K normalization and the rotary
 * embeddings).  With Y_b the bf16 output svdq_gemm_w4a4 returns for the same
 * arguments and heads of D = 128 columns:
 *   V columns [2N/3, N):    QKV = Y_b
 *   Q columns [0, N/3), K columns [N/3, 2N/3), per token m and head h:
 *     n[c]  = Y_b[c] / sqrt( mean_c Y_b[c]^2 + eps ) * w[c]   (w = norm_q or norm_k)
 *     (QKV[2i], QKV[2i+1]) = bf16( n[2i] cos - n[2i+1] sin, n[2i] sin + n[2i+1] cos ),
 *     cos = rope_cos[m][i], sin = rope_sin[m][i], i = 0 .. 63 (the same for every head)
 * evaluated in fp32 (relative error below 2^-16 of the pair's norm), rounded
 * to nearest even once.
 * Inputs: norm_q, norm_k [128] bf16; rope_cos, rope_sin [M][64] fp32 (16-byte
 * aligned, caller-owned); eps > 0 and finite (SVDQ_ERR_VALUE otherwise: with
 * eps = 0 an all-zero head would give 0 * inf).
 * Output: QKV [M][N] bf16.  Sizes: N % 768 == 0 (SVDQ_ERR_SHAPE otherwise);
 * everything else as svdq_gemm_w4a4. */
svdq_status svdq_gemm_w4a4_qkv(const uint8_t* a_codes, const uint8_t* a_scales,
                               const uint8_t* w_codes, const uint8_t* w_scales,
                               float w_tensor_scale, const uint16_t* lora_act,
                               const uint16_t* L2s, const uint16_t* bias,
                               const uint16_t* norm_q, const uint16_t* norm_k,
                               const float* rope_cos, const float* rope_sin, float eps,
                               uint16_t* QKV, int M, int N, int K, int rank, int* dev_status,
                               void* stream);

/* Activation side of the INT4 variant, one kernel (the same fused pass as
 * svdq_quantize_act: lora_act = bf16(X . L1s) alongside the codes):
 *   x_hat    = fl32(X[m][k] * inv_lambda[k])
 *   a_scales = RNE_bf16( fl32(amax64(x_hat) / 7) )   [M][K/64] bf16 bits
 *   a_codes  = clamp(RNE(x_hat / s), -8, 7)          [M][K/2] packed,
 *              rounded from the exact quotient; codes 0 where s is 0 or inf
 * Inputs, sizes, lora_act and errors as svdq_quantize_act (K % 128 == 0, rank
 * in {16, 32, 64}).  Output buffers: a_codes SVDQ_CODE_BYTES(M, K), a_scales
 * SVDQ_INT4_SCALE_BYTES(M, K), lora_act [M][rank]. */
svdq_status svdq_quantize_act_int4(const uint16_t* X_bf16, const float* inv_lambda,
                                   const uint16_t* L1s, int M, int K, int rank,
                                   uint8_t* a_codes, uint16_t* a_scales, uint16_t* lora_act,
                                   int* dev_status, void* stream);

/* The 4-bit GEMM of the INT4 variant with the low-rank up projection and the
 * bias (the fused-kernel paragraph's second kernel):
 *   Y[m][n] = bf16( sum_g a_s[m][g] w_s[n][g] sum_{k in g} a_q[m][k] w_q[n][k]
 *                   + sum_i lora_act[m][i] L2[n][i] + bias[n] )
 * fp32 accumulation: each group's integer sum is exact, then added with one
 * fma by the (exact) product of its two scales; one rounding to bf16.  B300
 * has no 4-bit integer tensor-core path: every code is an exact f16 value,
 * and each group's sum comes from tcgen05 f16 MMAs into tensor memory.
 * dev_status (nullable device int): SVDQ_DEV_TIMEOUT if an internal pipeline
 * wait exceeded its bound (the output is then incomplete).
 * Inputs: a_codes [M][K/2], a_scales [M][K/64] bf16 (svdq_quantize_act_int4),
 * w_codes [N][K/2], w_scales [N][K/64] bf16, L2 [N][rank] bf16
 * (svdq_pack_weights_int4), lora_act [M][rank] bf16, bias [N] bf16 or NULL.
 * Output: Y [M][N] bf16.
 * Sizes: M >= 0 (M == 0 launches nothing), N % 128 == 0, K % 128 == 0, rank in
 * {16, 32, 64}.
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE, SVDQ_ERR_RANK, SVDQ_ERR_ALIGN,
 * SVDQ_ERR_UNSUPPORTED_ARCH, SVDQ_ERR_CUDA. */
svdq_status svdq_gemm_w4a4_int4(const uint8_t* a_codes, const uint16_t* a_scales,
                                const uint8_t* w_codes, const uint16_t* w_scales,
                                const uint16_t* lora_act, const uint16_t* L2,
                                const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                                int rank, int* dev_status, void* stream);

/* AWQ W4A16 GEMV for the small-M modulation layers (kernel-family list:
 * memory-bound adaLN modulation):
 *   Y[m][n] = bf16( sum_k X[m][k] (q[n][k] - z[n][k/64]) s[n][k/64] + bias[n] )
 * fp32 accumulation.  Streams the 4-bit weights once from HBM.
 * Inputs: X [M][K] bf16; qweight [N][K/2] (even k in the low nibble);
 * scales, zeros [N][K/64] fp16; bias [N] bf16 (nullable).  Output Y [M][N] bf16.
 * Sizes: 1 <= M <= 8, N % 8 == 0 (N >= 8), K % 64 == 0, K <= 4096 (X and its
 * per-group sums stay in registers), group_size == 64.
 * Errors: SVDQ_ERR_NULL, SVDQ_ERR_SHAPE, SVDQ_ERR_ALIGN,
 * SVDQ_ERR_UNSUPPORTED_ARCH, SVDQ_ERR_CUDA. */
svdq_status awq_gemv_w4a16(const uint16_t* X_bf16, const uint8_t* qweight,
                           const uint16_t* scales, const uint16_t* zeros,
                           const uint16_t* bias, uint16_t* Y, int M, int N, int K,
                           int group_size, int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SVDQ_H_ */
