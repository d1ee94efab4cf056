// attn_fwd_host without a caller workspace: the staging buffers live in one
// file-scope device array of fixed size (kStaticWorkspaceBytes), looked up
// once per device; nothing is allocated or freed. Calls on a device are
// serialised on that array: each call's work starts after the previous call's
// copies back have finished (an event per device), whatever streams they use.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "attn.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kStaticWorkspaceBytes = size_t(128) << 20;  // 128 MiB

__device__ __align__(256) unsigned char g_host_workspace[kStaticWorkspaceBytes];

struct DeviceState {
  void* workspace = nullptr;
  cudaEvent_t last_done = nullptr;  // the previous call's completion, on its stream
  bool used = false;
  std::mutex mu;
};

DeviceState* state_for_current_device() {
  static DeviceState states[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return &states[dev];
}

}  // namespace

extern "C" {

size_t attn_fwd_host_noalloc_max_workspace(void) { return kStaticWorkspaceBytes; }

attn_status_t attn_fwd_host_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                    int N, int d, int causal, float scale, void* stream) {
  const size_t need = attn_fwd_host_workspace_bytes(B, H, N, d);
  // argument errors and empty problems exactly as attn_fwd_host reports them
  if (need == 0) return attn_fwd_host(q, k, v, o, lse, B, H, N, d, causal, scale, nullptr, 0, stream);
  if (need > kStaticWorkspaceBytes) return ATTN_ERR_UNSUPPORTED;
  DeviceState* st = state_for_current_device();
  if (!st) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(st->mu);
  if (!st->workspace) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_host_workspace) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaEventCreateWithFlags(&st->last_done, cudaEventDisableTiming) != cudaSuccess) return ATTN_ERR_CUDA;
    st->workspace = p;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the shared buffers are free once the previous call has copied its results back
  if (st->used && cudaStreamWaitEvent(s, st->last_done, 0) != cudaSuccess) return ATTN_ERR_CUDA;
  const attn_status_t r =
      attn_fwd_host(q, k, v, o, lse, B, H, N, d, causal, scale, st->workspace, kStaticWorkspaceBytes, stream);
  // attn_fwd_host leaves `stream` waiting for its last copy back (also on failure)
  if (cudaEventRecord(st->last_done, s) != cudaSuccess) return r == ATTN_OK ? ATTN_ERR_CUDA : r;
  st->used = true;
  return r;
}

}  // extern "C"
