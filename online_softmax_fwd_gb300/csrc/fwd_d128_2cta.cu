// The CTA-pair (tcgen05 cta_group::2) instantiation of the bf16 forward:
// d = 128, non-causal.
#include "fwd_bf16_2cta.cuh"
#include "fwd_dispatch.h"

namespace attn {

cudaError_t launch_fwd_bf16_d128_2cta(const CUtensorMap& q, const CUtensorMap& k_half, const CUtensorMap& v,
                                      const FwdArgs& a, const WorkList& wl, int clusters, cudaStream_t s) {
  return launch_fwd_bf16_2cta(q, k_half, v, a, wl, clusters, s);
}

int fwd_bf16_d128_2cta_max_clusters() { return fwd_bf16_2cta_max_clusters(); }

}  // namespace attn
