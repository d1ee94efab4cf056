// Software exp2 on the FMA pipe.
//
// Method: "FlashAttention-4's Softmax Tricks: A Degree-3 exp2 on the FMA Pipe"
// (section "The emulated exp2") and the KernelWiki page "Software-Emulated
// Exponential". 2^x = 2^floor(x) * 2^frac(x):
//   * x is clamped below at -127 (so -inf and anything <= -127 give +0);
//   * adding 2^23 + 2^22 with round-toward-minus-infinity leaves floor(x) as
//     an integer in the low mantissa bits of the sum;
//   * subtracting the constant back is exact and frac = x - floor(x) in [0, 1);
//   * 2^frac comes from a degree-3 polynomial with constant term 1 in Horner
//     form (3 fused multiply-adds), coefficients as printed on the first page
//     (Sollya fpminimax, relative error);
//   * the sum's bit pattern shifted left by 23 (floor(x) mod 512 in the exponent
//     field) is added to the polynomial's bit pattern with a signed 32-bit add.
// Max relative error ~8.8e-5 on [-20, 8]; results are within one bf16 ulp of
// the exact value there. No operation flushes subnormals.
#pragma once

#include <cstdint>

namespace attn {

__device__ __forceinline__ float exp2_fma(float x) {
  constexpr float kMagic = 12582912.0f;  // 2^23 + 2^22
  float xc = fmaxf(x, -127.0f);
  float rounded;
  asm("add.rm.f32 %0, %1, %2;" : "=f"(rounded) : "f"(xc), "f"(kMagic));
  float back;
  asm("sub.rn.f32 %0, %1, %2;" : "=f"(back) : "f"(rounded), "f"(kMagic));
  float frac;
  asm("sub.rn.f32 %0, %1, %2;" : "=f"(frac) : "f"(xc), "f"(back));
  float p = __fmaf_rn(0.077119089663028717041015625f, frac, 0.227564394474029541015625f);
  p = __fmaf_rn(p, frac, 0.695146143436431884765625f);
  p = __fmaf_rn(p, frac, 1.0f);
  int32_t hi, out;
  asm("shl.b32 %0, %1, 23;" : "=r"(hi) : "r"(__float_as_int(rounded)));
  asm("add.s32 %0, %1, %2;" : "=r"(out) : "r"(hi), "r"(__float_as_int(p)));
  return __int_as_float(out);
}

}  // namespace attn
