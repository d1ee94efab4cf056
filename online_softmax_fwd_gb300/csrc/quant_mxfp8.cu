// MXFP8 quantiser: fp32 [B*H, N, d=128] -> E4M3 payload [B*H, N, 128] plus one
// 512-byte scale-factor atom per 128-row tile, in the layout the block-scaled
// MMA consumes (see mxfp8_common.cuh).
//
// Square 32 x 32 blocks ("PyTorch FlashAttention-4 adds MXFP8 ...", section
// "Quantization along both axes and jagged tensors"): each block's amax gives
// its E8M0 exponent e (smallest power of two with amax / 2^e <= 448); elements
// are multiplied by 2^-e (exact) and rounded to E4M3 (nearest even,
// saturating). Role 0 lays the atom out for a GEMM that contracts over d (atom
// row = the tile's sequence row, block = d / 32: Q and K in S = Q K^T); role 1
// for one that contracts over the sequence (atom row = the d column, block =
// 32-row block of the tile: V in O = P V). The blocks being square, the E4M3
// payload is the same for both; role 2 writes both atom arrays in one pass,
// role 0's first and role 1's right after it, for a tensor that enters
// products along both axes (Q, K and dO in the backward pass). Rows past N
// count as zeros for the amax and are not written.
#include <cuda_runtime.h>

#include <cstdint>

#include "mxfp8_common.cuh"

namespace attn {

// One CTA per (128-row tile, head), 8 warps; warp w takes rows 16w .. 16w+15
// and lane l columns 4l .. 4l+3 of each, so every load and store of a warp
// covers one whole row (512 bytes in, 128 bytes out).
__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const float* __restrict__ x, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ atoms, int n, int ntiles,
                                                             int role) {
  __shared__ float part_amax[8][4];  // [warp][d block]: amax over the warp's 16 rows
  __shared__ uint32_t eb[4][4];      // [row block][d block] E8M0 bytes
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const long long bh = blockIdx.y;
  const int row0 = tile * 128 + 16 * warp;
  float4 v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int row = row0 + i;
    v[i] = row < n ? reinterpret_cast<const float4*>(x + (bh * n + row) * 128)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
  // d block = lane / 8: reduce over the 8 lanes of the block
#pragma unroll
  for (int sh = 1; sh <= 4; sh <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, sh));
  if ((lane & 7) == 0) part_amax[warp][lane >> 3] = a;
  __syncthreads();
  // a 32-row block spans warps 2 rb and 2 rb + 1
  if (tid < 16) {
    const int rb = tid >> 2, db = tid & 3;
    eb[rb][db] = e8m0_for_amax(fmaxf(part_amax[2 * rb][db], part_amax[2 * rb + 1][db]));
  }
  __syncthreads();
  const float sc = e8m0_inverse(eb[warp >> 1][lane >> 3]);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int row = row0 + i;
    if (row < n)
      reinterpret_cast<uint32_t*>(q + (bh * n + row) * 128)[lane] =
          pack_e4m3x4(v[i].x * sc, v[i].y * sc, v[i].z * sc, v[i].w * sc);
  }
  // the tile's atom(s): 512 bytes each, two bytes per thread
  uint8_t* atom = atoms + (bh * ntiles + tile) * 512;
  uint8_t* atom_t = atoms + ((static_cast<long long>(gridDim.y) + bh) * ntiles + tile) * 512;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t p = 2 * tid + k;
    const uint32_t atom_row = (p >> 4) + 32 * ((p & 15) >> 2);
    const uint32_t kb = p & 3;
    const uint8_t by_row = static_cast<uint8_t>(eb[atom_row >> 5][kb]);  // row = sequence position
    const uint8_t by_col = static_cast<uint8_t>(eb[kb][atom_row >> 5]);  // row = d column
    atom[p] = role == 1 ? by_col : by_row;
    if (role == 2) atom_t[p] = by_col;
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
