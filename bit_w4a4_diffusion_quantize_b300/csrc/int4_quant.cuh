// The activation quantization of the INT4 variant of the SVDQ W4A4 linear
// (dothoosh.com, "How Nunchaku Lite halves the VRAM of diffusion models",
// kernel-family list: svdq_w4a4 in INT4 and NVFP4 variants), used by
// svdq_quantize_act_int4.
#pragma once

#include <cstdint>

#include "act_quant.cuh"
#include "device_common.cuh"

namespace svdq {

SVDQ_DEVINL float2 add2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n.reg .b64 ra, rb, rd;\nmov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "add.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// One 64-element group of one row, held by the four lanes of a
// quad (16 consecutive elements each; all 32 lanes of the warp call it
// together).  Symmetric signed 4-bit codes:
//   s    = RNE_bf16( fl32(amax64(x_hat) / 7) )      (IEEE division, as written)
//   code = clamp( RNE(x_hat / s), -8, 7 )           exact quotient rounding
// A group whose scale is 0 or not finite gets codes 0.  The code quotient
// uses the two-term reciprocal of s (s has 8 significant bits): for a 24-bit
// x_hat the exact quotient is either a half-integer m itself or more than
// half a binary32 ulp of the quotient away from it (the difference x - m s
// is a multiple of ulp(x_hat), and ulp(x_hat) / s exceeds half an ulp of
// x_hat / s), so the binary32 y lands on the same side of m, and the integer
// rounding of y (adding 1.5 * 2^23 rounds to an integer, ties to even) is
// that of the exact quotient.  Scales below 2^-64 are multiplied, with the
// values, by 2^64 first (exact), so that neither 1/s nor the products leave
// the normal range.  codes: element 2i in the low nibble of byte i (two's
// complement nibbles); sbits: the bf16 bit pattern of s.
SVDQ_DEVINL void quant_group64_int4(const uint32_t (&w)[8], const float (&inv)[16],
                                    uint2& codes, uint32_t& sbits) {
  float2 xh[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    xh[i] = mul2_rn(make_float2(bf16lo_to_f32(w[i]), bf16hi_to_f32(w[i])),
                    make_float2(inv[2 * i], inv[2 * i + 1]));
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(xh[i].x), fabsf(xh[i].y));
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], m[i + 4]);
  float amax = fmaxf(fmaxf(m[0], m[2]), fmaxf(m[1], m[3]));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  const uint32_t sb = f32_to_bf16_rn(__fdiv_rn(amax, 7.0f));
  sbits = sb;
  const float s = __uint_as_float(sb << 16);
  const bool ok = s > 0.0f && s <= 3.402823466e38f;  // 0, inf, NaN: codes 0
  const float f = s < 0x1p-64f ? 0x1p64f : 1.0f;
  const float2 r = recip2(ok ? s * f : 1.0f);
  const float2 ff = make_float2(f, f), rh = make_float2(r.x, r.x), rl = make_float2(r.y, r.y);
  const float2 magic = make_float2(12582912.0f, 12582912.0f);  // 1.5 * 2^23
  uint32_t nib[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 x = mul2_rn(xh[i], ff);
    float2 y = fma2_rn(x, rh, mul2_rn(x, rl));
    y.x = fminf(fmaxf(y.x, -8.0f), 7.0f);
    y.y = fminf(fmaxf(y.y, -8.0f), 7.0f);
    const float2 t = add2_rn(y, magic);  // integer in the low mantissa bits
    nib[2 * i] = __float_as_uint(t.x) & 0xFu;
    nib[2 * i + 1] = __float_as_uint(t.y) & 0xFu;
  }
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lo |= nib[i] << (4 * i);
    hi |= nib[8 + i] << (4 * i);
  }
  const uint32_t keep = ok ? 0xFFFFFFFFu : 0u;
  codes = make_uint2(lo & keep, hi & keep);
}


}  // namespace svdq
