// rssm_static.cu -- rssm_step for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: engines whose
// allocator has already reserved all device memory and gives out no per-call
// workspace, or C/FFI hosts with no access to a device allocator at all.  For
// them this file keeps the step's scratch in a fixed array compiled into the
// library (RSSM_STEP_STATIC_SCRATCH_BYTES on every GPU that loads it, held
// until the process exits) and runs the ordinary two step kernels on it.
#include <cuda_runtime.h>

#include <mutex>

#include "rssm.h"
#include "rssm_internal.h"

namespace {

// The scratch.  In host code this name is only a stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_step_scratch[RSSM_STEP_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};

// Device address of g_step_scratch on the current device, looked up once per
// device with that device current.
rssm_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RSSM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return RSSM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_step_scratch) != cudaSuccess || !p) return RSSM_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return RSSM_OK;
}

}  // namespace

extern "C" rssm_status rssm_step_static_scratch(const rssm_cache* cache, const void* x, const float* dt,
                                                const float* A, const void* B, const void* C, const float* D,
                                                const float* dt_bias, const int32_t* slot_idx, const int32_t* pnat,
                                                const int32_t* cu_seqlens, int32_t batch, int32_t T, void* out,
                                                void* stream) {
  void* scratch = nullptr;
  const rssm_status st = static_scratch(&scratch);
  if (st != RSSM_OK) return st;
  // Nothing in the scratch has to start at zero: the precompute writes every
  // record and coefficient block the readout then reads.  A step that needs
  // more than the array holds is refused with RSSM_ERR_SCRATCH_TOO_SMALL.
  return rssm_step(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, out, scratch,
                   RSSM_STEP_STATIC_SCRATCH_BYTES, stream);
}
