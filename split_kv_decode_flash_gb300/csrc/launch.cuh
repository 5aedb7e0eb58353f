// Host-side launch preparation shared by the partial kernels.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"

namespace dattn {

// Checks a kernel's launch register budget (the consumers' setmaxnreg.inc
// waits for registers the producer warpgroup releases, which only completes
// if the launch holds them) and opts it into its dynamic shared memory.  Both
// are properties of the function on a device, so they are done once per
// device: "ready" holds one bit per device id already prepared, and later
// launches skip the two driver calls.
template <typename Kernel>
inline cudaError_t prepare_kernel_once(Kernel kernel, size_t smem, long long regs_needed,
                                       std::atomic<unsigned long long>& ready) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (ready.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  cudaFuncAttributes attr;
  err = cudaFuncGetAttributes(&attr, kernel);
  if (err != cudaSuccess) return err;
  if (static_cast<long long>(attr.numRegs) * kThreads < regs_needed) return cudaErrorInvalidConfiguration;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  ready.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

}  // namespace dattn
