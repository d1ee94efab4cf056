// Instantiations of the bf16 forward kernel for d = 64, causal = 1, one per
// software-exp2 share (0..4 of every 16 score columns).
#include "fwd_bf16.cuh"
#include "fwd_dispatch.h"

namespace attn {

cudaError_t launch_fwd_bf16_d64_c1(int emu16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                   const FwdArgs& a, const WorkList& wl, int ctas, cudaStream_t s) {
  switch (emu16) {
    case 0: return launch_fwd_bf16<64, true, 0>(q, k, v, a, wl, ctas, s);
    case 1: return launch_fwd_bf16<64, true, 1>(q, k, v, a, wl, ctas, s);
    case 2: return launch_fwd_bf16<64, true, 2>(q, k, v, a, wl, ctas, s);
    case 3: return launch_fwd_bf16<64, true, 3>(q, k, v, a, wl, ctas, s);
    case 4: return launch_fwd_bf16<64, true, 4>(q, k, v, a, wl, ctas, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
