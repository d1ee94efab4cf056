// The MXFP8 forward kernel (d = 128; MUFU exp2, P scaled per 32 keys from the
// block amax) instantiated to write the rescale log: each row's decision to
// move its running max per key block, and its warp's O correction, for
// checking them against the lagging-max rule of "FlashAttention-4's Softmax
// Tricks", section "Conditional rescaling, and when it's exact".
#include "fwd_dispatch.h"
#include "fwd_mxfp8.cuh"

namespace attn {

cudaError_t launch_fwd_mxfp8_d128_log(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                      const FwdMxArgs& a, const WorkList& wl, int ctas, cudaStream_t s) {
  return causal ? launch_fwd_mxfp8<true, 0, 0, false, true>(q, k, v, a, wl, ctas, s)
                : launch_fwd_mxfp8<false, 0, 0, false, true>(q, k, v, a, wl, ctas, s);
}

}  // namespace attn
