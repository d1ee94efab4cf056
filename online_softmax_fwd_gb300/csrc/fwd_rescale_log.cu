// Instantiations of the bf16 forward kernel that also write the rescale log
// (each row's decision to move its running max, and its warp's O correction,
// per key block), for checking the decisions against the lagging-max rule of
// "FlashAttention-4's Softmax Tricks", section "Conditional rescaling, and
// when it's exact". MUFU exp2 only; not used by the product entry points.
#include "fwd_bf16.cuh"
#include "fwd_dispatch.h"

namespace attn {

cudaError_t launch_fwd_bf16_log(int d, int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const FwdArgs& a, const WorkList& wl, int ctas, cudaStream_t s) {
  if (d == 64)
    return causal ? launch_fwd_bf16<64, true, 0, true>(q, k, v, a, wl, ctas, s)
                  : launch_fwd_bf16<64, false, 0, true>(q, k, v, a, wl, ctas, s);
  return causal ? launch_fwd_bf16<128, true, 0, true>(q, k, v, a, wl, ctas, s)
                : launch_fwd_bf16<128, false, 0, true>(q, k, v, a, wl, ctas, s);
}

}  // namespace attn
