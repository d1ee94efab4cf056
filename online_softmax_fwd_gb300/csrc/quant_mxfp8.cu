// MXFP8 quantiser: fp32 [B*H, N, d=128] -> E4M3 payload [B*H, N, 128] plus one
// 512-byte scale-factor atom per 128-row tile, in the layout the block-scaled
// MMA consumes (see mxfp8_common.cuh).
//
// Square 32 x 32 blocks ("PyTorch FlashAttention-4 adds MXFP8 ...", section
// "Quantization along both axes and jagged tensors"): each block's amax gives
// its E8M0 exponent e (smallest power of two with amax / 2^e <= 448); elements
// are multiplied by 2^-e (exact) and rounded to E4M3 (nearest even,
// saturating). Role 0 lays the atom out for the S = Q K^T GEMM (atom row = the
// tile's sequence row, block = d / 32); role 1 for the O = P V GEMM (atom row =
// the d column, block = key block of the tile). Rows past N count as zeros for
// the amax and are not written.
#include <cuda_runtime.h>

#include <cstdint>

#include "mxfp8_common.cuh"

namespace attn {

__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const float* __restrict__ x, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ atoms, int n, int ntiles,
                                                             int role) {
  __shared__ float row_amax[128][4];
  __shared__ uint32_t eb[4][4];  // [row block][d block] E8M0 bytes
  const int tid = threadIdx.x;
  const int r = tid >> 1;        // row within the tile
  const int h = tid & 1;         // columns [64h, 64h + 64)
  const int tile = blockIdx.x;
  const long long bh = blockIdx.y;
  const int row = tile * 128 + r;
  const bool valid = row < n;
  float v[64];
  const float4* src = reinterpret_cast<const float4*>(x + ((bh * n + (valid ? row : 0)) * 128 + 64 * h));
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 f = valid ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a0 = fmaxf(a0, fabsf(v[i]));
    a1 = fmaxf(a1, fabsf(v[32 + i]));
  }
  row_amax[r][2 * h] = a0;
  row_amax[r][2 * h + 1] = a1;
  __syncthreads();
  if (tid < 16) {
    const int rb = tid >> 2, db = tid & 3;
    float m = 0.f;
    for (int i = 0; i < 32; ++i) m = fmaxf(m, row_amax[32 * rb + i][db]);
    eb[rb][db] = e8m0_for_amax(m);
  }
  __syncthreads();
  if (valid) {
    const float s0 = e8m0_inverse(eb[r >> 5][2 * h]);
    const float s1 = e8m0_inverse(eb[r >> 5][2 * h + 1]);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = pack_e4m3x4(v[4 * i] * s0, v[4 * i + 1] * s0, v[4 * i + 2] * s0, v[4 * i + 3] * s0);
#pragma unroll
    for (int i = 8; i < 16; ++i)
      w[i] = pack_e4m3x4(v[4 * i] * s1, v[4 * i + 1] * s1, v[4 * i + 2] * s1, v[4 * i + 3] * s1);
    uint4* dst = reinterpret_cast<uint4*>(q + (bh * n + row) * 128 + 64 * h);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  }
  // the tile's atom: 512 bytes, two per thread
  uint8_t* atom = atoms + (bh * ntiles + tile) * 512;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t p = 2 * tid + k;
    const uint32_t atom_row = (p >> 4) + 32 * ((p & 15) >> 2);
    const uint32_t kb = p & 3;
    atom[p] = static_cast<uint8_t>(role == 0 ? eb[atom_row >> 5][kb] : eb[kb][atom_row >> 5]);
  }
}

cudaError_t launch_mxfp8_quantize(const float* x, uint8_t* q, uint8_t* atoms, long long bh, int n, int role,
                                  cudaStream_t stream) {
  const int ntiles = (n + 127) / 128;
  dim3 grid(ntiles, static_cast<unsigned>(bh));
  mxfp8_quantize_kernel<<<grid, 256, 0, stream>>>(x, q, atoms, n, ntiles, role);
  return cudaGetLastError();
}

}  // namespace attn
