// The MXFP8 forward kernel (d = 128) with the unroll-KV schedule and the row
// sum taken after the P hand-over, causal and not (MUFU exp2, P scaled per 32
// keys from the block amax): the opt-in attn_fwd_mxfp8_unroll_kv.
#include "fwd_dispatch.h"
#include "fwd_mxfp8.cuh"

namespace attn {

cudaError_t launch_fwd_mxfp8_d128_ukv(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                      const FwdMxArgs& a, const WorkList& wl, int ctas, cudaStream_t s) {
  return causal ? launch_fwd_mxfp8<true, 0, 0, true>(q, k, v, a, wl, ctas, s)
                : launch_fwd_mxfp8<false, 0, 0, true>(q, k, v, a, wl, ctas, s);
}

}  // namespace attn
