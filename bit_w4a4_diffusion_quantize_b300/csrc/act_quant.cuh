// The activation quantization of the SVDQ W4A4 linear, shared by
// svdq_quantize_act and by the GEMM epilogue that quantizes the next layer's
// input (the first MLP linear, whose GELU output feeds the second):
//
//   x_hat      = fl32( x * inv_lambda )
//   scale byte = RNE_e4m3( amax16(x_hat) / 6 )        exact quotient rounding
//   code       = RNE_e2m1( x_hat / s )                exact quotient rounding
//
// The quotients are rounded as the exact real quotient would be, without a
// division (the derivation is in quantize_act.cu): y = RN(x r_hi + RN(x r_lo))
// with r_hi = RD(1/d), r_lo = RN((1 - r_hi d) / d) lies within 2^-46 of x/d,
// closer than any exact quotient comes to a rounding midpoint of the e2m1 or
// e4m3 grid unless it is that midpoint.
#pragma once

#include <cstdint>

#include "device_common.cuh"

namespace svdq {

// RD(1/d) and RN((1 - RD(1/d) d) / d): the two-term reciprocal of d
SVDQ_DEVINL float2 recip2(float d) {
  const float hi = __frcp_rd(d);
  return make_float2(hi, __fdiv_rn(__fmaf_rn(-hi, d, 1.0f), d));
}

// quantize one 16-element block held by one thread (8 bf16x2 words);
// r6 = recip2(6), tab[code] = recip2(e4m3 value of code) (zeros for code 0).
// The products run as packed fp32 pairs (same roundings as scalar code).
SVDQ_DEVINL void quant_block16(const uint32_t (&w)[8], const float (&inv)[16], float2 r6,
                               const float2* tab, uint2& codes, uint32_t& sbyte) {
  float2 xh[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    xh[i] = mul2_rn(make_float2(bf16lo_to_f32(w[i]), bf16hi_to_f32(w[i])),
                    make_float2(inv[2 * i], inv[2 * i + 1]));
  // amax: a balanced tree (max is exact, so the order does not matter)
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(xh[i].x), fabsf(xh[i].y));
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], m[i + 4]);
  const float amax = fmaxf(fmaxf(m[0], m[2]), fmaxf(m[1], m[3]));
  sbyte = f32_to_e4m3_sat(__fmaf_rn(amax, r6.x, __fmul_rn(amax, r6.y)));
  const float2 r = tab[sbyte];
  const float2 rh = make_float2(r.x, r.x), rl = make_float2(r.y, r.y);
  float2 y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = fma2_rn(xh[i], rh, mul2_rn(xh[i], rl));
  const uint32_t keep = sbyte ? 0xFFFFFFFFu : 0u;  // scale 0: every code +0
  codes.x = f32x8_to_e2m1x8(y[0].x, y[0].y, y[1].x, y[1].y, y[2].x, y[2].y, y[3].x, y[3].y) & keep;
  codes.y = f32x8_to_e2m1x8(y[4].x, y[4].y, y[5].x, y[5].y, y[6].x, y[6].y, y[7].x, y[7].y) & keep;
}


}  // namespace svdq
