/*
 * Scalar C model of the software exp2 -- TEST INFRASTRUCTURE ONLY.
 *
 * Built by the oracle's own build step into oracle/liboracle_exp2.so and used
 * by the tests to check the GPU's software exp2 bit for bit. It shares nothing
 * with the CUDA sources.
 *
 * The algorithm is the one described on "FlashAttention-4's Softmax Tricks",
 * section "The emulated exp2" (and the KernelWiki page "Software-Emulated
 * Exponential"): clamp at -127; add 2^23 + 2^22 rounding toward -inf so that
 * floor(x) sits in the low mantissa bits; recover frac = x - floor(x) exactly;
 * 2^frac by a degree-3 Horner polynomial with fused multiply-adds (printed
 * Sollya coefficients, constant term 1); then add the sum's bit pattern shifted
 * left by 23 to the polynomial's bit pattern as a 32-bit integer.
 *
 * Every float operation here is IEEE binary32 with round-to-nearest-even except
 * the one add in round-toward-minus-infinity, and fmaf() rounds once. Nothing
 * flushes subnormals. Build with -frounding-math -ffp-contract=off.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#pragma STDC FENV_ACCESS ON

static const float kC0 = 1.0f;
static const float kC1 = 0.695146143436431884765625f;
static const float kC2 = 0.227564394474029541015625f;
static const float kC3 = 0.077119089663028717041015625f;
static const float kMagic = 12582912.0f; /* 2^23 + 2^22 */

static float add_toward_neg_inf(float a, float b) {
  int saved = fegetround();
  fesetround(FE_DOWNWARD);
  volatile float va = a, vb = b;
  volatile float r = va + vb;
  fesetround(saved);
  return r;
}

static uint32_t bits_of(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

static float float_of(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

float oracle_exp2_emulated_one(float x) {
  /* max with -127; a NaN input selects -127, like a hardware fmax */
  float xc = (x > -127.0f) ? x : -127.0f;
  float rounded = add_toward_neg_inf(xc, kMagic);
  volatile float back = rounded - kMagic; /* exact */
  float frac = xc - back;                 /* exact, in [0, 1) */
  float p = fmaf(kC3, frac, kC2);
  p = fmaf(p, frac, kC1);
  p = fmaf(p, frac, kC0);
  uint32_t r = (bits_of(rounded) << 23) + bits_of(p); /* wraps mod 2^32 */
  return float_of(r);
}

void oracle_exp2_emulated(const float* x, float* y, long n) {
  for (long i = 0; i < n; ++i) y[i] = oracle_exp2_emulated_one(x[i]);
}
