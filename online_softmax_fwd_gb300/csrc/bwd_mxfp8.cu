// Instantiations of the MXFP8 attention backward kernel (d = 128), causal and not.
#include "bwd_dispatch.h"
#include "bwd_mxfp8.cuh"

namespace attn {

cudaError_t launch_bwd_mxfp8_d128(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const CUtensorMap& dout, const CUtensorMap& dq, const BwdMxArgs& a,
                                  cudaStream_t s) {
  return causal ? launch_bwd_mxfp8<true>(q, k, v, dout, dq, a, s) : launch_bwd_mxfp8<false>(q, k, v, dout, dq, a, s);
}

}  // namespace attn
