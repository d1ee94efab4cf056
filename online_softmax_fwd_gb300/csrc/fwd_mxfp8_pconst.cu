// Instantiations of the MXFP8 forward kernel (d = 128), causal and not, with
// and without a software-exp2 share, P scaled by the constant 2^-8.
#include "fwd_mxfp8.cuh"
#include "fwd_dispatch.h"

namespace attn {

cudaError_t launch_fwd_mxfp8_d128_pconst(int causal, int emu16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const FwdMxArgs& a, const WorkList& wl, int ctas, cudaStream_t s) {
  if (causal) {
    switch (emu16) {
      case 0: return launch_fwd_mxfp8<true, 0, 1>(q, k, v, a, wl, ctas, s);
      case 2: return launch_fwd_mxfp8<true, 2, 1>(q, k, v, a, wl, ctas, s);
      case 4: return launch_fwd_mxfp8<true, 4, 1>(q, k, v, a, wl, ctas, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (emu16) {
    case 0: return launch_fwd_mxfp8<false, 0, 1>(q, k, v, a, wl, ctas, s);
    case 2: return launch_fwd_mxfp8<false, 2, 1>(q, k, v, a, wl, ctas, s);
    case 4: return launch_fwd_mxfp8<false, 4, 1>(q, k, v, a, wl, ctas, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
