// The backward pass's small kernels around its main kernels:
//   bwd_prep: D_i = sum_c dO_ic O_ic (fp32 from bf16) and LSE_i log2(e) for
//             every query row, stored negated (the kernel adds them in pairs;
//             rows N .. np-1 of a head get 0), and the fp32 dQ accumulator
//             zeroed;
//   bwd_prep_mxfp8: the same with dO from its E4M3 codes times its blocks'
//             E8M0 scales, stored as -D_i and 8 - LSE_i log2(e) (the MXFP8
//             kernel adds them in pairs; its exp then gives P 2^8, the
//             constant scale of P in E4M3); its accumulator is transposed,
//             [B*H, d, np];
//   bwd_post: dQ = s * accumulator, rounded to bf16 (bwd_post_t: from the
//             transposed accumulator).
// All are bandwidth-bound elementwise passes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_dispatch.h"

namespace attn {

namespace {

// one warp per query row; lane l takes elements [D/32 l, D/32 (l+1))
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ lse2,
                                                       float* __restrict__ dvec, float* __restrict__ dq_acc, int n,
                                                       int np) {
  constexpr int kPer = D / 32;  // 2 or 4 bf16 per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  const long long bh = blockIdx.y;
  if (row >= np) return;
  const size_t prow = static_cast<size_t>(bh) * np + row;
  if (row >= n) {
    if (lane == 0) {
      lse2[prow] = 0.f;
      dvec[prow] = 0.f;
    }
    return;
  }
  const size_t grow = static_cast<size_t>(bh) * n + row;
  float acc = 0.f;
  if constexpr (kPer == 4) {
    const uint2 a = reinterpret_cast<const uint2*>(o + grow * D)[lane];
    const uint2 b = reinterpret_cast<const uint2*>(dout + grow * D)[lane];
    const uint32_t aw[2] = {a.x, a.y}, bw[2] = {b.x, b.y};
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      acc = __fmaf_rn(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc);
      acc = __fmaf_rn(__uint_as_float(aw[e] & 0xFFFF0000u), __uint_as_float(bw[e] & 0xFFFF0000u), acc);
    }
  } else {
    const uint32_t a = reinterpret_cast<const uint32_t*>(o + grow * D)[lane];
    const uint32_t b = reinterpret_cast<const uint32_t*>(dout + grow * D)[lane];
    acc = __fmaf_rn(__uint_as_float(a << 16), __uint_as_float(b << 16), acc);
    acc = __fmaf_rn(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u), acc);
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
  if (lane == 0) {
    dvec[prow] = -acc;
    lse2[prow] = -lse[grow] * 1.4426950408889634f;
  }
  float4* z = reinterpret_cast<float4*>(dq_acc + grow * D);
#pragma unroll
  for (int e = lane; e < D / 4; e += 32) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// The value of an E4M3 code (OCP E4M3FN: sign, 4 exponent bits with bias 7, 3
// mantissa bits; exponent 0 holds the subnormals m 2^-9), exact in fp32.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
  return (code & 0x80u) ? -mag : mag;
}

// one warp per query row (d = 128); lane l takes columns 4l .. 4l + 3, in dO's
// 32-column block l / 8
__global__ void __launch_bounds__(256) bwd_prep_mxfp8_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const uint8_t* __restrict__ do8,
                                                             const uint8_t* __restrict__ do_sf,
                                                             const float* __restrict__ lse, float* __restrict__ lse2,
                                                             float* __restrict__ dvec, float* __restrict__ dq_acc,
                                                             int n, int np) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  const long long bh = blockIdx.y;
  if (row >= np) return;
  const size_t prow = static_cast<size_t>(bh) * np + row;
  // the head's transposed accumulator [128, np] holds 128 np floats: row
  // index r zeroes floats 128 r .. 128 r + 127 of it
  reinterpret_cast<float4*>(dq_acc + prow * 128)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (row >= n) {
    if (lane == 0) {
      lse2[prow] = 0.f;
      dvec[prow] = 0.f;
    }
    return;
  }
  const size_t grow = static_cast<size_t>(bh) * n + row;
  const uint2 a = reinterpret_cast<const uint2*>(o + grow * 128)[lane];
  const uint32_t c = reinterpret_cast<const uint32_t*>(do8 + grow * 128)[lane];
  // the block's E8M0 byte: atom of tile row / 128, row r at byte (r % 32) * 16 + (r / 32) * 4 + block
  const int r = row & 127;
  const uint32_t byte =
      do_sf[(static_cast<size_t>(bh) * (np / 128) + (row >> 7)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + (lane >> 3)];
  const float sc = byte ? __uint_as_float(byte << 23) : __uint_as_float(0x400000u);  // 2^(byte - 127)
  float acc = 0.f;
  acc = __fmaf_rn(e4m3_value(c & 0xFFu) * sc, __uint_as_float(a.x << 16), acc);
  acc = __fmaf_rn(e4m3_value((c >> 8) & 0xFFu) * sc, __uint_as_float(a.x & 0xFFFF0000u), acc);
  acc = __fmaf_rn(e4m3_value((c >> 16) & 0xFFu) * sc, __uint_as_float(a.y << 16), acc);
  acc = __fmaf_rn(e4m3_value(c >> 24) * sc, __uint_as_float(a.y & 0xFFFF0000u), acc);
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
  if (lane == 0) {
    dvec[prow] = -acc;
    lse2[prow] = 8.0f - lse[grow] * 1.4426950408889634f;
  }
}

// dQ[bh, q, c] = bf16(s acc[bh, c, q]) through a 32 x 32 shared-memory tile:
// reads along q, writes along c, both coalesced
__global__ void __launch_bounds__(256) bwd_post_t_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                         int n, int np, float scale) {
  __shared__ float tile[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int q0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  const long long bh = blockIdx.z;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int c = c0 + ty + 8 * k, q = q0 + tx;
    tile[ty + 8 * k][tx] = q < n ? acc[(static_cast<size_t>(bh) * 128 + c) * np + q] : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int q = q0 + ty + 8 * k, c = c0 + tx;
    if (q < n) dq[(static_cast<size_t>(bh) * n + q) * 128 + c] = __float2bfloat16_rn(tile[tx][ty + 8 * k] * scale);
  }
}

// four elements per thread
__global__ void __launch_bounds__(256) bwd_post_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                                                       long long n4, float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[i];
  __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * scale, a.y * scale);
  __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * scale, a.w * scale);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&lo);
  w.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(dq)[i] = w;
}

}  // namespace

cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* lse2, float* dvec,
                            float* dq_acc, long long bh, int n, int np, int d, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(np / 8), static_cast<unsigned>(bh));
  if (d == 128)
    bwd_prep_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                   static_cast<const __nv_bfloat16*>(dout), lse, lse2, dvec, dq_acc,
                                                   n, np);
  else
    bwd_prep_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                  static_cast<const __nv_bfloat16*>(dout), lse, lse2, dvec, dq_acc,
                                                  n, np);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep_mxfp8(const void* o, const void* do8, const void* do_sf, const float* lse, float* lse2,
                                  float* dvec, float* dq_acc, long long bh, int n, int np, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(np / 8), static_cast<unsigned>(bh));
  bwd_prep_mxfp8_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                  static_cast<const uint8_t*>(do8), static_cast<const uint8_t*>(do_sf),
                                                  lse, lse2, dvec, dq_acc, n, np);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post_t(const float* dq_acc, void* dq, long long bh, int n, int np, float scale,
                              cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>((n + 31) / 32), 4, static_cast<unsigned>(bh));
  bwd_post_t_kernel<<<grid, 256, 0, stream>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), n, np, scale);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post(const float* dq_acc, void* dq, long long elems, float scale, cudaStream_t stream) {
  const long long n4 = elems / 4;
  const long long blocks = (n4 + 255) / 256;
  bwd_post_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), n4,
                                                                     scale);
  return cudaGetLastError();
}

}  // namespace attn
