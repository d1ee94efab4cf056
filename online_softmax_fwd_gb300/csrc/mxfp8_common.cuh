// MXFP8 helpers shared by the quantiser and the block-scaled attention kernel:
// the E8M0 exponent rule, E4M3 packing, the scale-factor atom layout and the
// block-scaled tcgen05 MMA.
//
// Block scaling follows "PyTorch FlashAttention-4 adds MXFP8 block-scaled
// forward and backward for Blackwell" (sections "Quantization along both axes"
// and "Softmax conversion and unroll-KV"): square 32 x 32 blocks for Q, K
// (along d) and V (along the sequence), one E8M0 power-of-two scale per block;
// P is converted online per 32 keys with the scale taken from the exponent and
// mantissa bits of the block's amax (no log2, no division).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace attn {

// E8M0 byte of the smallest power of two 2^e with amax / 2^e <= 448 (the
// largest finite E4M3): with amax = 1.m * 2^E, 448 = 1.75 * 2^8, e = E - 8 when
// 1.m <= 1.75 (mantissa bits <= 0x600000) else E - 7; byte = e + 127. An
// all-zero block gets e = 0. Clamped to the finite E8M0 range.
__device__ __forceinline__ uint32_t e8m0_for_amax(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  if (amax <= 0.f) return 127u;
  int b = static_cast<int>((bits >> 23) & 0xFFu) - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  b = b < 0 ? 0 : (b > 254 ? 254 : b);
  return static_cast<uint32_t>(b);
}

// 2^-e as a float for an E8M0 byte (exact; byte <= 253).
__device__ __forceinline__ float e8m0_inverse(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }

// Four floats -> four E4M3 bytes (round to nearest even, saturating), first
// value in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Four floats -> four E5M2 bytes (round to nearest even, saturating to
// +-57344), first value in the lowest byte.
__device__ __forceinline__ uint32_t pack_e5m2x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Scale-factor atom: 512 bytes holding the E8M0 scales of 128 rows x 4 blocks
// of 32 along the MMA's K dimension; row r, block kb at byte
// (r % 32) * 16 + (r / 32) * 4 + kb. tcgen05.cp 32x128b.warpx4 moves it into 4
// TMEM columns (replicated over the four lane quadrants), where the MMA reads
// the A scale of row m at lane m, column m / 32, and the B scale of column n at
// lane n % 32, column n / 32, byte = the scale-factor id of the instruction.
__host__ __device__ constexpr uint32_t sf_atom_index(uint32_t row, uint32_t kb) {
  return (row % 32u) * 16u + (row / 32u) * 4u + kb;
}

// Shared-memory descriptor of an atom (no swizzle; 8-row core matrices of 16
// bytes, 128 bytes apart).
__device__ __forceinline__ uint64_t sf_atom_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

__device__ __forceinline__ void sf_copy_to_tmem(uint32_t tmem_cols, uint32_t atom_saddr) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem_cols), "l"(sf_atom_desc(atom_saddr))
               : "memory");
}

// Instruction descriptor, kind::mxf8f6f4 with E4M3 B, E4M3 or E5M2 A, E8M0
// scales, fp32 accumulator; a_sf / b_sf pick the scale byte of this K=32 step.
__host__ __device__ constexpr uint32_t idesc_mxf8(int m, int n, bool b_mn_major, uint32_t a_sf, uint32_t b_sf,
                                                  bool a_e5m2 = false, bool a_mn_major = false) {
  return ((b_sf & 3u) << 4)                         // B scale-factor id
         | ((a_e5m2 ? 1u : 0u) << 7)                 // A format: E4M3 0, E5M2 1 (B stays E4M3)
         | ((a_mn_major ? 1u : 0u) << 15)            // A major-ness (shared-memory A only)
         | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
         | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
         | (1u << 23)                                // scale type E8M0
         | (static_cast<uint32_t>(m >> 4) << 24)     // M / 16
         | ((a_sf & 3u) << 29);                      // A scale-factor id
}

// D(tmem) (+)= A(smem) * B(smem), block scaled; scale TMEM addresses must be
// 4-column aligned.
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc,
                                            uint32_t sfa, uint32_t sfb) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
// D(tmem) (+)= A(tmem, 4 E4M3 per column) * B(smem), block scaled.
__device__ __forceinline__ void mma_mxf8_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc,
                                            uint32_t sfa, uint32_t sfb) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

// The same two MMAs with each shared-memory descriptor given as its low word
// and a high word common to both operands (only the low words change from one
// MMA to the next).
__device__ __forceinline__ void mma_mxf8_ss_lo(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t desc_hi,
                                               uint32_t idesc, uint32_t acc, uint32_t sfa, uint32_t sfb) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 ad, bd;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 ad, {%1, %3};\n\tmov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], ad, bd, %4, [%6], [%7], p;\n\t}" ::"r"(d),
      "r"(a_lo), "r"(b_lo), "r"(desc_hi), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void mma_mxf8_ts_lo(uint32_t d, uint32_t a, uint32_t b_lo, uint32_t desc_hi,
                                               uint32_t idesc, uint32_t acc, uint32_t sfa, uint32_t sfb) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], bd, %4, [%6], [%7], p;\n\t}" ::"r"(d),
      "r"(a), "r"(b_lo), "r"(desc_hi), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
      : "memory");
}

// Bulk copy of `bytes` (multiple of 16, 16-byte aligned both sides) global ->
// shared, completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

}  // namespace attn
