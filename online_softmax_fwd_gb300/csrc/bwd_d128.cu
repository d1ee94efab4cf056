// Instantiations of the attention backward kernel, d = 128, causal and not.
#include "bwd_bf16.cuh"
#include "bwd_dispatch.h"

namespace attn {

cudaError_t launch_bwd_bf16_d128(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& dout, const CUtensorMap& dq, const BwdArgs& a, cudaStream_t s) {
  return causal ? launch_bwd_bf16<128, true>(q, k, v, dout, dq, a, s)
                : launch_bwd_bf16<128, false>(q, k, v, dout, dq, a, s);
}

}  // namespace attn
