// Host-memory entry point: Q, K, V in host memory in, O and LSE in host
// memory out, with the copies and the attention kernels overlapped.
//
// The (batch, head) axis is cut into chunks; chunk i goes through three
// streams -- host->device copy, attention, device->host copy -- with two
// device buffers per tensor, so the copy of chunk i+1 runs while chunk i is
// computed and chunk i-1 is copied back. Every chunk is an independent
// attention problem (heads do not interact), so the result equals one call on
// the whole batch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"

namespace {

constexpr int kBuffers = 2;
constexpr int kMaxDevices = 64;

struct Streams {
  cudaStream_t h2d = nullptr, compute = nullptr, d2h = nullptr;
  bool ok = false;
};

// Three non-blocking streams per device, created once and kept for the
// process (streams are not freed per call).
Streams* device_streams() {
  static Streams table[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  Streams& s = table[dev];
  if (!s.ok) {
    if (cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&s.compute, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking) != cudaSuccess)
      return nullptr;
    s.ok = true;
  }
  return &s;
}

// Heads per chunk: about 6 chunks, at least one head. The copies share one
// host link (~220 GB/s for both directions together on GB300), so the step
// is link-bound; measured on the d128 workloads, 6 chunks beat 4, 8 and 12
// (larger chunks lengthen the unoverlapped first upload and last download,
// smaller ones lower the link's efficiency).
long long chunk_heads(long long bh) { return std::max<long long>(1, (bh + 5) / 6); }

size_t head_bytes(int N, int d) { return static_cast<size_t>(N) * d * 2; }

// per buffer: q, k, v, o (bf16) + lse (fp32), each rounded up to 256 bytes
size_t buffer_bytes(long long heads, int N, int d) {
  auto round = [](size_t x) { return (x + 255) & ~size_t(255); };
  return 4 * round(heads * head_bytes(N, d)) + round(heads * static_cast<size_t>(N) * 4);
}

}  // namespace

extern "C" {

size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  return kBuffers * buffer_bytes(chunk_heads(static_cast<long long>(B) * H), N, d);
}

attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                            int d, int causal, float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return d > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse || !workspace) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
  const long long bh = static_cast<long long>(B) * H;
  const long long ch = chunk_heads(bh);
  const size_t buf_bytes = buffer_bytes(ch, N, d);
  if (workspace_bytes < kBuffers * buf_bytes) return ATTN_ERR_INVALID_ARG;
  // reject bad arguments before any copy: a zero-size attention call runs the
  // same checks (scale, causal, d) and launches nothing
  {
    attn_status_t st = attn_fwd(reinterpret_cast<const void*>(256), reinterpret_cast<const void*>(256),
                                reinterpret_cast<const void*>(256), reinterpret_cast<void*>(256),
                                reinterpret_cast<float*>(256), 0, H, N, d, causal, scale, stream);
    if (st != ATTN_OK) return st;
  }
  Streams* ss = device_streams();
  if (!ss) return ATTN_ERR_CUDA;
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  cudaEvent_t start, loaded[kBuffers], computed[kBuffers], freed[kBuffers], done;
  auto mk = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  bool ok = mk(&start) && mk(&done);
  for (int b = 0; b < kBuffers; ++b) ok = ok && mk(&loaded[b]) && mk(&computed[b]) && mk(&freed[b]);
  if (!ok) return ATTN_ERR_CUDA;
  attn_status_t result = ATTN_OK;
  // everything starts after the work already queued on the caller's stream
  if (cudaEventRecord(start, user) != cudaSuccess || cudaStreamWaitEvent(ss->h2d, start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(ss->compute, start, 0) != cudaSuccess || cudaStreamWaitEvent(ss->d2h, start, 0) != cudaSuccess)
    result = ATTN_ERR_CUDA;
  const size_t hb = head_bytes(N, d);
  auto round = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t t_bytes = round(ch * hb);
  const long long n_chunks = (bh + ch - 1) / ch;
  for (long long c = 0; c < n_chunks && result == ATTN_OK; ++c) {
    const int b = static_cast<int>(c % kBuffers);
    const long long h0 = c * ch;
    const long long nh = std::min<long long>(ch, bh - h0);
    uint8_t* base = static_cast<uint8_t*>(workspace) + b * buf_bytes;
    uint8_t* dq = base;
    uint8_t* dk = base + t_bytes;
    uint8_t* dv = base + 2 * t_bytes;
    uint8_t* dout = base + 3 * t_bytes;
    float* dlse = reinterpret_cast<float*>(base + 4 * t_bytes);
    const size_t off = static_cast<size_t>(h0) * hb;
    const size_t bytes = static_cast<size_t>(nh) * hb;
    // the buffer is free once chunk c - kBuffers has been copied back
    if (c >= kBuffers && cudaStreamWaitEvent(ss->h2d, freed[b], 0) != cudaSuccess) result = ATTN_ERR_CUDA;
    if (result != ATTN_OK) break;
    if (cudaMemcpyAsync(dq, static_cast<const uint8_t*>(q) + off, bytes, cudaMemcpyHostToDevice, ss->h2d) != cudaSuccess ||
        cudaMemcpyAsync(dk, static_cast<const uint8_t*>(k) + off, bytes, cudaMemcpyHostToDevice, ss->h2d) != cudaSuccess ||
        cudaMemcpyAsync(dv, static_cast<const uint8_t*>(v) + off, bytes, cudaMemcpyHostToDevice, ss->h2d) != cudaSuccess ||
        cudaEventRecord(loaded[b], ss->h2d) != cudaSuccess || cudaStreamWaitEvent(ss->compute, loaded[b], 0) != cudaSuccess) {
      result = ATTN_ERR_CUDA;
      break;
    }
    // chunk = nh heads of one "batch" (the layout is [B*H, N, d] either way)
    attn_status_t st = attn_fwd(dq, dk, dv, dout, dlse, 1, static_cast<int>(nh), N, d, causal, scale, ss->compute);
    if (st != ATTN_OK) {
      result = st;
      break;
    }
    if (cudaEventRecord(computed[b], ss->compute) != cudaSuccess || cudaStreamWaitEvent(ss->d2h, computed[b], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(o) + off, dout, bytes, cudaMemcpyDeviceToHost, ss->d2h) != cudaSuccess ||
        cudaMemcpyAsync(lse + static_cast<size_t>(h0) * N, dlse, static_cast<size_t>(nh) * N * 4, cudaMemcpyDeviceToHost,
                        ss->d2h) != cudaSuccess ||
        cudaEventRecord(freed[b], ss->d2h) != cudaSuccess) {
      result = ATTN_ERR_CUDA;
      break;
    }
  }
  // the caller's stream continues after the last copy back
  if (cudaEventRecord(done, ss->d2h) != cudaSuccess || cudaStreamWaitEvent(user, done, 0) != cudaSuccess)
    result = result == ATTN_OK ? ATTN_ERR_CUDA : result;
  // events may be destroyed while pending: their resources are released on completion
  cudaEventDestroy(start);
  cudaEventDestroy(done);
  for (int b = 0; b < kBuffers; ++b) {
    cudaEventDestroy(loaded[b]);
    cudaEventDestroy(computed[b]);
    cudaEventDestroy(freed[b]);
  }
  return result;
}

}  // extern "C"
