// Host-side preparation of a kernel instantiation before its first launch on a
// device: the dynamic shared-memory opt-in and the check that the compiled
// register count is the one the kernel's setmaxnreg split assumes. Both are
// properties of (device, instantiation), so they are done once per device and
// remembered; later launches skip the two runtime calls.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

namespace attn {

constexpr int kSetupMaxDevices = 64;

// Kernel is the instantiation itself (a distinct function pointer gives a
// distinct cache). Returns cudaErrorInvalidConfiguration if the compiled
// register count differs from launch_regs: the setmaxnreg split redistributes
// the registers the CTA is launched with, and an increase asking for more than
// that would wait for ever (setmaxnreg.inc only raises a warp's count,
// setmaxnreg.dec only lowers it).
template <auto Kernel>
cudaError_t kernel_ready(unsigned smem_bytes, int launch_regs) {
  static std::atomic<int> ready[kSetupMaxDevices];
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kSetupMaxDevices;
  if (cached && ready[dev].load(std::memory_order_acquire) == 1) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_bytes));
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, Kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != launch_regs) return cudaErrorInvalidConfiguration;
  if (cached) ready[dev].store(1, std::memory_order_release);
  return cudaSuccess;
}

}  // namespace attn
