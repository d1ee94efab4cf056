// Merge of attention results computed over disjoint sets of keys (a sequence
// split): P partial results (O_p bf16, LSE_p fp32) of the same query rows
// become the result over the union of their keys.
//
// "Lecture 2 - Online Softmax and Numerical Correctness", section "Combining
// two blocks exactly": the merged max is the largest of the parts' maxima and
// the merged sum is the parts' sums brought to it by exp of the max gap. With
// each part's statistics taken as (m_p, l_p) = (LSE_p, 1), which has the same
// log-sum-exp, that is
//     m = max_p LSE_p,   w_p = exp(LSE_p - m),   l = sum_p w_p,
//     O = sum_p w_p O_p / l,   LSE = m + ln l.
// A part with LSE_p = -inf (no keys) has w_p = 0; a row whose parts are all
// -inf gets O = 0 and LSE = -inf.
//
// HBM-bound: per row, P (d bf16 + one fp32) in and d bf16 + one fp32 out. One
// warp per row; lane l holds d/32 consecutive columns, so each part's row is
// one coalesced 128- or 256-byte load for the warp, and up to eight parts'
// rows are in flight before the row's weights are known.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "fwd_dispatch.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;
constexpr int kCombineThreads = 256;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, s));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
  return x;
}

// acc[c] += w * (the CPL bf16 values of x), in fp32
template <int CPL, typename Vec>
__device__ __forceinline__ void accumulate(float (&acc)[CPL], float w, const Vec& x) {
  uint32_t words[CPL / 2];
  if constexpr (CPL == 4) {
    words[0] = x.x;
    words[1] = x.y;
  } else {
    words[0] = x;
  }
#pragma unroll
  for (int c = 0; c < CPL / 2; ++c) {
    acc[2 * c] = __fmaf_rn(w, __uint_as_float(words[c] << 16), acc[2 * c]);
    acc[2 * c + 1] = __fmaf_rn(w, __uint_as_float(words[c] & 0xFFFF0000u), acc[2 * c + 1]);
  }
}

// CPL = columns per lane (d / 32: 2 for d = 64, 4 for d = 128). One row per
// warp at a time: two or four rows per warp (more loads in flight) measured
// the same, so the loads in flight are not what limits it.
template <int CPL>
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const __nv_bfloat16* __restrict__ o_parts,
                                                                       const float* __restrict__ lse_parts,
                                                                       int parts, long long rows,
                                                                       __nv_bfloat16* __restrict__ o,
                                                                       float* __restrict__ lse) {
  constexpr int D = 32 * CPL;
  using Vec = typename std::conditional<CPL == 4, uint2, uint32_t>::type;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kCombineThreads / 32);
  const long long part_step = rows * 32;  // Vec units (d / 32 columns each) between the parts' rows
  for (long long row = static_cast<long long>(blockIdx.x) * (kCombineThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const Vec* src = reinterpret_cast<const Vec*>(o_parts + row * D) + lane;
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;
    float m, l;
    if (parts <= 32) {
      // up to 32 parts: the first eight parts' rows are requested before the
      // LSEs (one per lane) are read and reduced, so the loads overlap that
      Vec x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < parts) x[i] = src[i * part_step];
      const float lp = lane < parts ? lse_parts[static_cast<long long>(lane) * rows + row] : -INFINITY;
      m = warp_max(lp);
      // w_p = exp(LSE_p - m): 1 for the largest part, 0 for a part without keys
      const float w = m == -INFINITY ? 0.f : ex2_mufu((lp - m) * kLog2e);
      l = warp_sum(w);
      for (int c0 = 0; c0 < parts; c0 += 8) {
        if (c0 > 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (c0 + i < parts) x[i] = src[(c0 + i) * part_step];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (c0 + i < parts) {
            // a part without keys is skipped, whatever its O holds
            const float wi = __shfl_sync(0xffffffffu, w, c0 + i);
            if (wi != 0.f) accumulate<CPL>(acc, wi, x[i]);
          }
        }
      }
    } else {
      // more parts: the largest LSE first, 32 parts per step
      float mp = -INFINITY;
      for (int p0 = 0; p0 < parts; p0 += 32) {
        const int p = p0 + lane;
        if (p < parts) mp = fmaxf(mp, lse_parts[static_cast<long long>(p) * rows + row]);
      }
      m = warp_max(mp);
      float lw = 0.f;
      for (int p0 = 0; p0 < parts; p0 += 32) {
        const int p = p0 + lane;
        const float w = (p < parts && m != -INFINITY)
                            ? ex2_mufu((lse_parts[static_cast<long long>(p) * rows + row] - m) * kLog2e)
                            : 0.f;
        lw += w;
        const int np = parts - p0 < 32 ? parts - p0 : 32;
#pragma unroll 4
        for (int i = 0; i < np; ++i) {
          const float wi = __shfl_sync(0xffffffffu, w, i);
          if (wi != 0.f) accumulate<CPL>(acc, wi, src[(p0 + i) * part_step]);
        }
      }
      l = warp_sum(lw);
    }
    Vec* orow = reinterpret_cast<Vec*>(o + row * D) + lane;
    uint32_t out[CPL / 2];
    if (m == -INFINITY) {  // no part has a key for this row
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) out[c] = 0u;
    } else {
      const float inv_l = 1.0f / l;
#pragma unroll
      for (int c = 0; c < CPL / 2; ++c) out[c] = pack_bf16x2(acc[2 * c] * inv_l, acc[2 * c + 1] * inv_l);
    }
    if constexpr (CPL == 4)
      *orow = make_uint2(out[0], out[1]);
    else
      *orow = out[0];
    if (lane == 0) lse[row] = m == -INFINITY ? -INFINITY : m + lg2_mufu(l) * kLn2;
  }
}

}  // namespace

cudaError_t launch_attn_combine(const void* o_parts, const float* lse_parts, int parts, long long rows, int d,
                                void* o, float* lse, int sms, cudaStream_t stream) {
  const long long want = (rows + kCombineThreads / 32 - 1) / (kCombineThreads / 32);
  const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 16;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (d == 128)
    attn_combine_kernel<4><<<grid, kCombineThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o_parts), lse_parts, parts, rows, static_cast<__nv_bfloat16*>(o), lse);
  else
    attn_combine_kernel<2><<<grid, kCombineThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o_parts), lse_parts, parts, rows, static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError();
}

}  // namespace attn
