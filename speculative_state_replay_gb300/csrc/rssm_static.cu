// rssm_static.cu -- rssm_step for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: engines whose
// allocator has already reserved all device memory and gives out no per-call
// workspace, or C/FFI hosts with no access to a device allocator at all.  For
// them this file keeps the step's scratch in a fixed array compiled into the
// library (RSSM_STEP_STATIC_SCRATCH_BYTES on every GPU that loads it, held
// until the process exits) and runs the ordinary two step kernels on it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "rssm.h"
#include "rssm_internal.h"

namespace {

// The scratch.  In host code this name is only a stand-in for the device
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_step_scratch[RSSM_STEP_STATIC_SCRATCH_BYTES];

// The array's device address belongs to a CUDA context (the module is loaded
// per context), so it is cached per context, keyed by the context's unique id
// (cuCtxGetId: ids are never reused within a process, so a context created
// after a device reset, or a non-primary context made current by the caller,
// gets its own lookup).  The driver functions come through the runtime's
// entry-point query: the library does not link libcuda.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

constexpr int kMaxContexts = 64;
std::mutex g_mu;
unsigned long long g_ctx_id[kMaxContexts];
void* g_addr[kMaxContexts];
int g_count = 0;

template <typename F>
F driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(p);
}

// Unique id of the calling thread's current context (0 if none is current).
rssm_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return RSSM_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return RSSM_ERR_CUDA;
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return RSSM_ERR_CUDA;
  return RSSM_OK;
}

// Device address of g_step_scratch in the current context, looked up once per
// context with that context current.
rssm_status static_scratch(void** out) {
  unsigned long long id = 0;
  rssm_status st = current_context_id(&id);
  if (st != RSSM_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  if (id != 0) {
    for (int i = 0; i < g_count; ++i)
      if (g_ctx_id[i] == id) {
        *out = g_addr[i];
        return RSSM_OK;
      }
  }
  void* p = nullptr;
  // binds the runtime to the device's primary context if no context is current yet
  const cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
  if (e != cudaSuccess || !p) return RSSM_ERR_CUDA;
  if (id == 0) {
    st = current_context_id(&id);
    if (st != RSSM_OK) return st;
    if (id == 0) return RSSM_ERR_CUDA;
  }
  if (g_count == kMaxContexts) return RSSM_ERR_UNSUPPORTED;
  g_ctx_id[g_count] = id;
  g_addr[g_count] = p;
  ++g_count;
  *out = p;
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
