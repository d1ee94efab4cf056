// Host-side launchers of the backward pass's kernels (bwd_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

struct BwdArgs;
struct BwdMxArgs;

cudaError_t launch_bwd_prep(const void* o, const void* dout, const float* lse, float* lse2, float* dvec,
                            float* dq_acc, long long bh, int n, int np, int d, cudaStream_t stream);
cudaError_t launch_bwd_post(const float* dq_acc, void* dq, long long elems, float scale, cudaStream_t stream);
// dq: 3-D map over the fp32 dQ accumulator [B*H, N, d], 32-column boxes of 128 rows, 128-byte swizzle
cudaError_t launch_bwd_bf16_d64(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& dout, const CUtensorMap& dq, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_bf16_d128(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dout, const CUtensorMap& dq, const BwdArgs& a, cudaStream_t s);
// MXFP8 (d = 128): D from dO's E4M3 codes and its atoms whose rows are queries,
// stored as -D and 8 - LSE log2 e (P comes out of the exp already scaled by 2^8)
cudaError_t launch_bwd_prep_mxfp8(const void* o, const void* do8, const void* do_sf, const float* lse, float* lse2,
                                  float* dvec, float* dq_acc, long long bh, int n, int np, cudaStream_t stream);
// dQ from the transposed accumulator [B*H, 128, np] (MXFP8)
cudaError_t launch_bwd_post_t(const float* dq_acc, void* dq, long long bh, int n, int np, float scale,
                              cudaStream_t stream);
// q, k, v, dout: 3-D maps over the E4M3 payloads (128 x 128 boxes); dq: over
// the transposed fp32 accumulator, 32 x 32 boxes
cudaError_t launch_bwd_mxfp8_d128(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const CUtensorMap& dout, const CUtensorMap& dq, const BwdMxArgs& a,
                                  cudaStream_t s);

}  // namespace attn
