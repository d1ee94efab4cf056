// Host-side entry points of the per-(d, causal) kernel instantiation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

struct FwdArgs;
struct WorkList;
struct FwdMxArgs;

cudaError_t launch_fwd_bf16_d64_c0(int emu16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                   const FwdArgs& a, const WorkList& wl, int ctas, cudaStream_t s);
cudaError_t launch_fwd_bf16_d64_c1(int emu16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                   const FwdArgs& a, const WorkList& wl, int ctas, cudaStream_t s);
cudaError_t launch_fwd_bf16_d128_c0(int emu16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                    const FwdArgs& a, const WorkList& wl, int ctas, cudaStream_t s);
cudaError_t launch_fwd_bf16_d128_c1(int emu16, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                    const FwdArgs& a, const WorkList& wl, int ctas, cudaStream_t s);

// the CTA-pair instantiation (d = 128, non-causal; fwd_d128_2cta.cu): k_half is
// a map of K with 64-row boxes; the grid is `clusters` pairs of CTAs
cudaError_t launch_fwd_bf16_d128_2cta(const CUtensorMap& q, const CUtensorMap& k_half, const CUtensorMap& v,
                                      const FwdArgs& a, const WorkList& wl, int clusters, cudaStream_t s);
int fwd_bf16_d128_2cta_max_clusters();

// the rescale-logging instantiations (MUFU exp2 only; fwd_rescale_log.cu)
cudaError_t launch_fwd_bf16_log(int d, int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const FwdArgs& a, const WorkList& wl, int ctas, cudaStream_t s);

cudaError_t launch_fwd_mxfp8_d128(int causal, int emu16, const CUtensorMap& q, const CUtensorMap& k,
                                  const CUtensorMap& v, const FwdMxArgs& a, const WorkList& wl, int ctas,
                                  cudaStream_t s);
cudaError_t launch_fwd_mxfp8_d128_pconst(int causal, int emu16, const CUtensorMap& q, const CUtensorMap& k,
                                         const CUtensorMap& v, const FwdMxArgs& a, const WorkList& wl, int ctas,
                                         cudaStream_t s);
cudaError_t launch_fwd_mxfp8_d128_pconst_e5m2(int causal, int emu16, const CUtensorMap& q, const CUtensorMap& k,
                                              const CUtensorMap& v, const FwdMxArgs& a, const WorkList& wl,
                                              int ctas, cudaStream_t s);
// the unroll-KV schedule (fwd_mxfp8_ukv.cu)
cudaError_t launch_fwd_mxfp8_d128_ukv(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                      const FwdMxArgs& a, const WorkList& wl, int ctas, cudaStream_t s);
// the rescale-logging instantiations (fwd_mxfp8_log.cu)
cudaError_t launch_fwd_mxfp8_d128_log(int causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                      const FwdMxArgs& a, const WorkList& wl, int ctas, cudaStream_t s);
// the merge of partial results over disjoint key sets (combine.cu); o_parts
// [parts, rows, d] bf16, lse_parts [parts, rows] fp32, d = 64 or 128
cudaError_t launch_attn_combine(const void* o_parts, const float* lse_parts, int parts, long long rows, int d,
                                void* o, float* lse, int sms, cudaStream_t stream);
// the bounded-wait self-test (selftest.cu)
cudaError_t launch_wait_timeout_selftest(unsigned int* status, long long limit_cycles, cudaStream_t stream);

cudaError_t launch_mxfp8_quantize(const float* x, uint8_t* q, uint8_t* atoms, long long bh, int n, int role,
                                  cudaStream_t stream);

}  // namespace attn
