// dattn_run_noalloc: one decode step whose workspace is a fixed device array
// owned by the library instead of a buffer passed by the caller.
//
// Some callers cannot hand over (or create) a device workspace at step time:
// a serving engine that reserves all of HBM for its K/V page pool at start-up
// and forbids later allocations, or a latency-critical loop that cannot take
// the implicit device synchronisation of cudaMalloc / cudaFree or an
// allocator's growth.  For them the workspace lives in a file-scope
// __device__ array of kScratchBytes, created when this library's device code
// is loaded on a GPU and kept until the process exits.  This file calls no
// cudaMalloc, cudaFree or other allocating routine; the decode step itself is
// dattn_run unchanged, pointed at that array.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "plan.h"

namespace {

constexpr size_t kScratchBytes = DATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices];  // device address of g_scratch, per device ordinal

// Device address of the scratch array on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress); later calls reuse it.
dattn_status scratch_of_current_device(void** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) {
    dattn::set_error(std::string("dattn_run_noalloc: cudaGetDevice: ") + cudaGetErrorString(err));
    return DATTN_ECUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    dattn::set_error("dattn_run_noalloc: device ordinal " + std::to_string(dev) + " is not below " +
                     std::to_string(kMaxDevices));
    return DATTN_EUNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_scratch);
    if (err != cudaSuccess || !p) {
      dattn::set_error(std::string("dattn_run_noalloc: cudaGetSymbolAddress of the scratch array: ") +
                       cudaGetErrorString(err));
      return DATTN_ECUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DATTN_OK;
}

}  // namespace

extern "C" dattn_status dattn_run_noalloc(const dattn_plan_t* plan, const dattn_problem* prob,
                                          const dattn_tensors* t, void* stream) {
  if (!plan) {
    dattn::set_error("dattn_run_noalloc: plan is NULL");
    return DATTN_EINVAL;
  }
  const size_t need = static_cast<size_t>(plan->info.workspace_bytes);
  if (need > kScratchBytes) {
    dattn::set_error("dattn_run_noalloc: the plan needs a workspace of " + std::to_string(need) +
                     " bytes but the library's static scratch holds " + std::to_string(kScratchBytes) +
                     " bytes; use dattn_run with a caller-owned workspace");
    return DATTN_EWORKSPACE;
  }
  void* scratch = nullptr;
  const dattn_status st = scratch_of_current_device(&scratch);
  if (st != DATTN_OK) return st;
  // The work list is copied into the scratch by dattn_run on "stream"; it
  // carries the zeroed status word and, for a fused-merge plan, the zeroed
  // per-group completion counters.  Every partial-state slot the merge reads
  // is written by the partial kernel first, so no other part of the previous
  // call's contents needs clearing.
  return dattn_run(plan, prob, t, scratch, kScratchBytes, stream);
}

extern "C" dattn_status dattn_noalloc_status(int32_t* flags, void* stream) {
  if (!flags) {
    dattn::set_error("dattn_noalloc_status: flags is NULL");
    return DATTN_EINVAL;
  }
  void* scratch = nullptr;
  const dattn_status st = scratch_of_current_device(&scratch);
  if (st != DATTN_OK) return st;
  // the status word sits in the work-list header at the start of the array
  return dattn_device_status(scratch, flags, stream);
}
