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
#include <type_traits>

#include "bwd_dispatch.h"

namespace attn {

namespace {

// Rows per warp in the preparation kernels: every warp issues the loads of all
// its rows before any arithmetic, so that enough bytes are in flight to keep
// HBM busy. np is a multiple of 128, so a grid of np / 32 CTAs of 8 warps
// covers rows 0 .. np-1 exactly.
constexpr int kPrepRows = 4;

// warp w of CTA x takes rows 4 (8 x + w) .. +3; lane l elements
// [D/32 l, D/32 (l+1)) of each
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ lse2,
                                                       float* __restrict__ dvec, float* __restrict__ dq_acc, int n,
                                                       int np) {
  constexpr int kPer = D / 32;  // 2 or 4 bf16 per lane
  using Chunk = typename std::conditional<kPer == 4, uint2, uint32_t>::type;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * 8 + warp) * kPrepRows;
  const long long bh = blockIdx.y;
  Chunk a[kPrepRows], b[kPrepRows];
  float l[kPrepRows];
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i) {
    if (row0 + i < n) {
      const size_t grow = static_cast<size_t>(bh) * n + row0 + i;
      a[i] = reinterpret_cast<const Chunk*>(o + grow * D)[lane];
      b[i] = reinterpret_cast<const Chunk*>(dout + grow * D)[lane];
      l[i] = lse[grow];
    } else {
      a[i] = Chunk{};
      b[i] = Chunk{};
      l[i] = 0.f;
    }
  }
  float acc[kPrepRows];
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i) {
    acc[i] = 0.f;
    if constexpr (kPer == 4) {
      const uint32_t aw[2] = {a[i].x, a[i].y}, bw[2] = {b[i].x, b[i].y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        acc[i] = __fmaf_rn(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), acc[i]);
        acc[i] = __fmaf_rn(__uint_as_float(aw[e] & 0xFFFF0000u), __uint_as_float(bw[e] & 0xFFFF0000u), acc[i]);
      }
    } else {
      acc[i] = __fmaf_rn(__uint_as_float(a[i] << 16), __uint_as_float(b[i] << 16), acc[i]);
      acc[i] = __fmaf_rn(__uint_as_float(a[i] & 0xFFFF0000u), __uint_as_float(b[i] & 0xFFFF0000u), acc[i]);
    }
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1)
#pragma unroll
    for (int i = 0; i < kPrepRows; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], sh);
  // lane i stores row i's pair; rows N .. np-1 of the head get 0
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i) {
    if (lane == i) {
      const size_t prow = static_cast<size_t>(bh) * np + row0 + i;
      const bool valid = row0 + i < n;
      dvec[prow] = valid ? -acc[i] : 0.f;
      lse2[prow] = valid ? -l[i] * 1.4426950408889634f : 0.f;
    }
  }
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i) {
    if (row0 + i < n) {
      float4* z = reinterpret_cast<float4*>(dq_acc + (static_cast<size_t>(bh) * n + row0 + i) * D);
#pragma unroll
      for (int e = lane; e < D / 4; e += 32) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// The value of an E4M3 code (OCP E4M3FN: sign, 4 exponent bits with bias 7, 3
// mantissa bits; exponent 0 holds the subnormals m 2^-9), exact in fp32.
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
  return (code & 0x80u) ? -mag : mag;
}

// d = 128; warp w of CTA x takes rows 4 (8 x + w) .. +3, lane l columns
// 4l .. 4l + 3 of each, in dO's 32-column block l / 8
__global__ void __launch_bounds__(256) bwd_prep_mxfp8_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const uint8_t* __restrict__ do8,
                                                             const uint8_t* __restrict__ do_sf,
                                                             const float* __restrict__ lse, float* __restrict__ lse2,
                                                             float* __restrict__ dvec, float* __restrict__ dq_acc,
                                                             int n, int np) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * 8 + warp) * kPrepRows;
  const long long bh = blockIdx.y;
  uint2 a[kPrepRows];
  uint32_t c[kPrepRows], byte[kPrepRows];
  float l[kPrepRows];
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i) {
    const int row = row0 + i;
    if (row < n) {
      const size_t grow = static_cast<size_t>(bh) * n + row;
      a[i] = reinterpret_cast<const uint2*>(o + grow * 128)[lane];
      c[i] = reinterpret_cast<const uint32_t*>(do8 + grow * 128)[lane];
      // the block's E8M0 byte: atom of tile row / 128, row r at byte (r % 32) * 16 + (r / 32) * 4 + block
      const int r = row & 127;
      byte[i] = do_sf[(static_cast<size_t>(bh) * (np / 128) + (row >> 7)) * 512 + (r & 31) * 16 + (r >> 5) * 4 +
                      (lane >> 3)];
      l[i] = lse[grow];
    } else {
      a[i] = make_uint2(0u, 0u);
      c[i] = 0u;
      byte[i] = 127u;
      l[i] = 0.f;
    }
  }
  // the head's transposed accumulator [128, np] holds 128 np floats: row
  // index r zeroes floats 128 r .. 128 r + 127 of it
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i)
    reinterpret_cast<float4*>(dq_acc + (static_cast<size_t>(bh) * np + row0 + i) * 128)[lane] =
        make_float4(0.f, 0.f, 0.f, 0.f);
  float acc[kPrepRows];
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i) {
    const float sc = byte[i] ? __uint_as_float(byte[i] << 23) : __uint_as_float(0x400000u);  // 2^(byte - 127)
    acc[i] = __fmaf_rn(e4m3_value(c[i] & 0xFFu) * sc, __uint_as_float(a[i].x << 16), 0.f);
    acc[i] = __fmaf_rn(e4m3_value((c[i] >> 8) & 0xFFu) * sc, __uint_as_float(a[i].x & 0xFFFF0000u), acc[i]);
    acc[i] = __fmaf_rn(e4m3_value((c[i] >> 16) & 0xFFu) * sc, __uint_as_float(a[i].y << 16), acc[i]);
    acc[i] = __fmaf_rn(e4m3_value(c[i] >> 24) * sc, __uint_as_float(a[i].y & 0xFFFF0000u), acc[i]);
  }
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1)
#pragma unroll
    for (int i = 0; i < kPrepRows; ++i) acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], sh);
  // lane i stores row i's pair; rows N .. np-1 of the head get 0
#pragma unroll
  for (int i = 0; i < kPrepRows; ++i) {
    if (lane == i) {
      const size_t prow = static_cast<size_t>(bh) * np + row0 + i;
      const bool valid = row0 + i < n;
      dvec[prow] = valid ? -acc[i] : 0.f;
      lse2[prow] = valid ? 8.0f - l[i] * 1.4426950408889634f : 0.f;
    }
  }
}

// dQ[bh, q, c] = bf16(s acc[bh, c, q]) for 32 queries x all 128 columns per
// CTA, through shared memory: each warp load reads 128 contiguous bytes of an
// accumulator row, each warp store writes one whole 256-byte row of dQ. The
// tile's element (c, q) sits at tile[c][q ^ (c / 4)], which keeps both the
// shared-memory stores (one c, 32 q) and loads (32 c four apart, one q) free
// of bank conflicts.
__global__ void __launch_bounds__(256) bwd_post_t_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                         int n, int np, float scale) {
  __shared__ float tile[128][32];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int q0 = blockIdx.x * 32;
  const long long bh = blockIdx.y;
  // q0 + 31 < np (np is a multiple of 128): every load is inside the head's
  // accumulator, whose rows past N the preparation kernel zeroed
  const float* src = acc + static_cast<size_t>(bh) * 128 * np + q0 + tx;
  float v[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) v[k] = src[static_cast<size_t>(ty + 8 * k) * np];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int cc = ty + 8 * k;
    tile[cc][tx ^ (cc >> 2)] = v[k];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int ql = ty + 8 * j, q = q0 + ql;
    if (q < n) {
      const float x0 = tile[4 * tx][ql ^ tx], x1 = tile[4 * tx + 1][ql ^ tx];
      const float x2 = tile[4 * tx + 2][ql ^ tx], x3 = tile[4 * tx + 3][ql ^ tx];
      __nv_bfloat162 lo = __floats2bfloat162_rn(x0 * scale, x1 * scale);
      __nv_bfloat162 hi = __floats2bfloat162_rn(x2 * scale, x3 * scale);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t*>(&lo);
      w.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(dq + (static_cast<size_t>(bh) * n + q) * 128)[tx] = w;
    }
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
  dim3 grid(static_cast<unsigned>(np / (8 * kPrepRows)), static_cast<unsigned>(bh));
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
  dim3 grid(static_cast<unsigned>(np / (8 * kPrepRows)), static_cast<unsigned>(bh));
  bwd_prep_mxfp8_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(o),
                                                  static_cast<const uint8_t*>(do8), static_cast<const uint8_t*>(do_sf),
                                                  lse, lse2, dvec, dq_acc, n, np);
  return cudaGetLastError();
}

cudaError_t launch_bwd_post_t(const float* dq_acc, void* dq, long long bh, int n, int np, float scale,
                              cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>((n + 31) / 32), static_cast<unsigned>(bh));
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
