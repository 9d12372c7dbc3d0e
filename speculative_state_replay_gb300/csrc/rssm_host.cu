// rssm_host.cu -- C ABI entry points of librssm: argument validation and
// kernel dispatch.  Nothing here reads device data or synchronises the host,
// so every call is stream ordered and capturable in a CUDA graph.
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "rssm.h"
#include "rssm_internal.h"

using namespace rssm;

namespace {

int elem_bytes(int dt) {
  switch (dt) {
    case RSSM_F32: return 4;
    case RSSM_BF16:
    case RSSM_F16: return 2;
    case RSSM_I8:
    case RSSM_E4M3: return 1;
    default: return 0;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rssm_status check_cache(const rssm_cache* c, Cache* out) {
  if (!c) return RSSM_ERR_INVALID_ARGUMENT;
  if (c->dim != kDim || c->dstate != kDstate) return RSSM_ERR_UNSUPPORTED;
  if (c->num_slots < 1 || c->nheads < 1 || c->ngroups < 1 || c->nheads % c->ngroups) return RSSM_ERR_INVALID_ARGUMENT;
  if (c->max_window < 0 || c->npredicted < 1) return RSSM_ERR_INVALID_ARGUMENT;
  const int L = c->max_window + c->npredicted;
  if (L > kMaxL) return RSSM_ERR_UNSUPPORTED;
  const int esz = c->state_dtype == RSSM_NVFP4 ? 0 : elem_bytes(c->state_dtype);  // NVFP4: read format only
  if (!esz) return RSSM_ERR_INVALID_ARGUMENT;
  if (c->rounding != RSSM_ROUND_NEAREST && c->rounding != RSSM_ROUND_STOCHASTIC) return RSSM_ERR_INVALID_ARGUMENT;
  const bool q8 = c->state_dtype == RSSM_I8 || c->state_dtype == RSSM_E4M3;
  if (!c->state || !c->x_cache || !c->B_cache || !c->dt_cache || !c->ring_start || !c->flush_epoch ||
      !c->error_word || (q8 && !c->scale))
    return RSSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(c->state) || !aligned16(c->x_cache) || !aligned16(c->B_cache) || (q8 && !aligned16(c->scale)))
    return RSSM_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(c->dt_cache) & 3u) || (reinterpret_cast<uintptr_t>(c->ring_start) & 3u) ||
      (reinterpret_cast<uintptr_t>(c->flush_epoch) & 3u) || (reinterpret_cast<uintptr_t>(c->error_word) & 3u))
    return RSSM_ERR_INVALID_ARGUMENT;
  const long long H = c->nheads, G = c->ngroups;
  if (c->state_slot_stride < H * kHeadElems || (c->state_slot_stride * esz) % 16) return RSSM_ERR_INVALID_ARGUMENT;
  if (q8 && (c->scale_slot_stride < H * kDim || (c->scale_slot_stride * 4) % 16)) return RSSM_ERR_INVALID_ARGUMENT;
  if (c->x_slot_stride < H * L * kDim || (c->x_slot_stride * 2) % 16) return RSSM_ERR_INVALID_ARGUMENT;
  if (c->B_slot_stride < G * L * kDstate || (c->B_slot_stride * 2) % 16) return RSSM_ERR_INVALID_ARGUMENT;
  if (c->dt_slot_stride < H * L) return RSSM_ERR_INVALID_ARGUMENT;
  if (c->read_state) {
    if (c->read_dtype == RSSM_NVFP4) {
      if (!c->read_sf || !c->read_gs || !aligned16(c->read_state) || !aligned16(c->read_sf) ||
          (reinterpret_cast<uintptr_t>(c->read_gs) & 3u))
        return RSSM_ERR_INVALID_ARGUMENT;
      if (c->read_slot_stride < H * kHeadElems / 2 || c->read_slot_stride % 16) return RSSM_ERR_INVALID_ARGUMENT;
      if (c->read_sf_slot_stride < H * kDim * 8 || c->read_sf_slot_stride % 16) return RSSM_ERR_INVALID_ARGUMENT;
    } else {
      if (c->read_dtype != RSSM_I8 && c->read_dtype != RSSM_E4M3) return RSSM_ERR_INVALID_ARGUMENT;
      if (!c->read_scale || !aligned16(c->read_state) || !aligned16(c->read_scale)) return RSSM_ERR_INVALID_ARGUMENT;
      if (c->read_slot_stride < H * kHeadElems || c->read_slot_stride % 16) return RSSM_ERR_INVALID_ARGUMENT;
      if (c->read_scale_slot_stride < H * kDim || (c->read_scale_slot_stride * 4) % 16)
        return RSSM_ERR_INVALID_ARGUMENT;
    }
  }
  if (out) {
    Cache& v = *out;
    v.S = c->num_slots;
    v.H = c->nheads;
    v.G = c->ngroups;
    v.hpg = c->nheads / c->ngroups;
    v.W = c->max_window;
    v.Tmax = c->npredicted;
    v.L = L;
    v.dtype = c->state_dtype;
    v.rounding = c->rounding;
    v.state = c->state;
    v.state_stride = c->state_slot_stride;
    v.scale = c->scale;
    v.scale_stride = c->scale_slot_stride;
    v.x_cache = static_cast<uint16_t*>(c->x_cache);
    v.x_stride = c->x_slot_stride;
    v.B_cache = static_cast<uint16_t*>(c->B_cache);
    v.B_stride = c->B_slot_stride;
    v.dt_cache = c->dt_cache;
    v.dt_stride = c->dt_slot_stride;
    v.ring_start = c->ring_start;
    v.epoch = c->flush_epoch;
    v.err = c->error_word;
    v.read_state = c->read_state;
    v.read_stride = c->read_state ? c->read_slot_stride : 0;
    v.read_scale = c->read_state ? c->read_scale : nullptr;
    v.read_scale_stride = c->read_state ? c->read_scale_slot_stride : 0;
    v.read_dtype = c->read_state ? c->read_dtype : -1;
    const bool fp4 = c->read_state && c->read_dtype == RSSM_NVFP4;
    v.read_sf = fp4 ? static_cast<uint8_t*>(c->read_sf) : nullptr;
    v.read_sf_stride = fp4 ? c->read_sf_slot_stride : 0;
    v.read_gs = fp4 ? c->read_gs : nullptr;
    if (fp4) v.read_scale = nullptr;
  }
  return RSSM_OK;
}

// SMs the persistent kernels size their grids for: the current device's SM
// count (cached per device), capped by the environment variable
// RSSM_SM_LIMIT when it holds a positive integer (read at every call, so a
// caller can leave SMs to concurrent work; results do not depend on it)
int num_sms() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  int n = dev < 64 ? cache[dev] : 0;
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> g(mu);
    if (dev < 64) cache[dev] = n;
  }
  if (const char* lim = getenv("RSSM_SM_LIMIT")) {
    const long v = strtol(lim, nullptr, 10);
    if (v > 0 && v < n) n = static_cast<int>(v);
  }
  return n;
}

rssm_status step_common(const rssm_cache* cache, const void* x, const float* dt, const float* A, const void* B,
                        const void* C, const float* D, const float* dt_bias, const int32_t* slot_idx,
                        const int32_t* pnat, const int32_t* cu, int32_t batch, int32_t T, void* out, void* scratch,
                        size_t scratch_bytes, StepArgs* a) {
  rssm_status st = check_cache(cache, &a->c);
  if (st != RSSM_OK) return st;
  if (batch < 0 || T < 1) return RSSM_ERR_INVALID_ARGUMENT;
  if (T > cache->npredicted || T > kMaxT) return RSSM_ERR_UNSUPPORTED;
  a->batch = batch;
  if (batch == 0) return RSSM_OK;  // nothing to do; pointers of empty tensors may be NULL
  if (!x || !dt || !A || !B || !C || !D || !dt_bias || !slot_idx || !pnat || !out || !scratch)
    return RSSM_ERR_INVALID_ARGUMENT;
  if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(out) || !aligned16(scratch))
    return RSSM_ERR_INVALID_ARGUMENT;
  const size_t need = step_scratch_bytes(batch, cache->nheads, cache->ngroups, a->c.L, T);
  if (scratch_bytes < need) return RSSM_ERR_SCRATCH_TOO_SMALL;
  a->x = static_cast<const uint16_t*>(x);
  a->dt = dt;
  a->A = A;
  a->B = static_cast<const uint16_t*>(B);
  a->C = static_cast<const uint16_t*>(C);
  a->D = D;
  a->dt_bias = dt_bias;
  a->slot_idx = slot_idx;
  a->pnat = pnat;
  a->cu = cu;
  a->batch = batch;
  a->T = T;
  a->TP = t_pad(T);
  a->KB = ring_pad(a->c.L);
  a->out = static_cast<uint16_t*>(out);
  a->z = nullptr;
  a->flush_mode = 0;
  a->seed = 0;
  a->pnat_rw = nullptr;
  a->fw = nullptr;
  a->rwork = static_cast<unsigned*>(scratch) + 2;  // a word of the scratch head (the flush uses words 0, 1)
  uint8_t* sc = static_cast<uint8_t*>(scratch) + kScratchHead;  // past the flush's ticket word
  a->rows = reinterpret_cast<RowRec*>(sc);
  a->cf = reinterpret_cast<uint16_t*>(sc + step_rows_bytes(batch));
  a->rblk = reinterpret_cast<float*>(sc + step_rows_bytes(batch) +
                                     step_cf_bytes(batch, cache->ngroups, T));
  if (a->c.read_state) {
    // the step never writes S0: its readout (and the C block's operand type,
    // which follows the format it reads) works on the read checkpoint
    a->c.state = a->c.read_state;
    a->c.state_stride = a->c.read_stride;
    a->c.scale = a->c.read_scale;
    a->c.scale_stride = a->c.read_scale_stride;
    a->c.dtype = a->c.read_dtype;
  }
  return RSSM_OK;
}

}  // namespace

extern "C" {

size_t rssm_scratch_bytes(const rssm_cache* cache, int32_t batch, int32_t T) {
  Cache c;
  if (check_cache(cache, &c) != RSSM_OK || batch < 0 || T < 1 || T > kMaxT) return 0;
  const size_t f = flush_scratch_bytes(batch), s = flush_step_scratch_bytes(batch, c.H, c.G, c.L, T);
  return f > s ? f : s;
}

rssm_status rssm_init_state(const rssm_cache* cache, const float* states, const int32_t* slot_idx, int32_t n,
                            uint64_t seed, void* stream) {
  InitArgs a;
  rssm_status st = check_cache(cache, &a.c);
  if (st != RSSM_OK) return st;
  if (n < 0) return RSSM_ERR_INVALID_ARGUMENT;
  if (n == 0) return RSSM_OK;
  if (!states || !slot_idx || !aligned16(states)) return RSSM_ERR_INVALID_ARGUMENT;
  if (n > 65535 * 64) return RSSM_ERR_UNSUPPORTED;
  a.states = states;
  a.ids = slot_idx;
  a.n = n;
  a.seed = seed;
  return launch_init(a, stream) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

namespace {
rssm_status flush_common(const rssm_cache* cache, const float* A, const int32_t* slot_idx, int32_t* pnat,
                         const int32_t* accepted, const int32_t* accept_cu_seqlens, int32_t accept_T,
                         const int32_t* cu_seqlens, int32_t batch, int32_t T, int32_t force, uint64_t seed,
                         void* scratch, size_t scratch_bytes, void* stream) {
  FlushArgs a;
  rssm_status st = check_cache(cache, &a.c);
  if (st != RSSM_OK) return st;
  if (batch < 0 || T < 0 || accept_T < 0 || (force != 0 && force != 1)) return RSSM_ERR_INVALID_ARGUMENT;
  if (batch == 0) return RSSM_OK;
  if (!A || !slot_idx || !pnat || !scratch || !aligned16(scratch)) return RSSM_ERR_INVALID_ARGUMENT;
  if (scratch_bytes < flush_scratch_bytes(batch)) return RSSM_ERR_SCRATCH_TOO_SMALL;
  const int sms = num_sms();
  if (sms <= 0) return RSSM_ERR_CUDA;
  a.A = A;
  a.slot_idx = slot_idx;
  a.pnat = pnat;
  a.cu = cu_seqlens;
  a.batch = batch;
  a.T = T;
  a.force = force;
  a.seed = seed;
  a.accepted = accepted;
  a.acu = accepted ? accept_cu_seqlens : nullptr;
  a.aT = accepted ? accept_T : 0;
  a.ticket = static_cast<unsigned*>(scratch);
  a.count = static_cast<int*>(scratch) + 1;
  a.recs = reinterpret_cast<FlushRec*>(static_cast<uint8_t*>(scratch) + kScratchHead);
  return launch_flush(a, sms, stream) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}
}  // namespace

rssm_status rssm_flush(const rssm_cache* cache, const float* A, const int32_t* slot_idx, int32_t* pnat,
                       const int32_t* cu_seqlens, int32_t batch, int32_t T, int32_t force, uint64_t seed,
                       void* scratch, size_t scratch_bytes, void* stream) {
  return flush_common(cache, A, slot_idx, pnat, nullptr, nullptr, 0, cu_seqlens, batch, T, force, seed, scratch,
                      scratch_bytes, stream);
}

rssm_status rssm_accept_flush(const rssm_cache* cache, const float* A, const int32_t* slot_idx, int32_t* pnat,
                              const int32_t* accepted, const int32_t* accept_cu_seqlens, int32_t accept_T,
                              const int32_t* cu_seqlens, int32_t batch, int32_t T, int32_t force, uint64_t seed,
                              void* scratch, size_t scratch_bytes, void* stream) {
  if (!accepted && batch > 0) return RSSM_ERR_INVALID_ARGUMENT;
  return flush_common(cache, A, slot_idx, pnat, accepted, accept_cu_seqlens, accept_T, cu_seqlens, batch, T, force,
                      seed, scratch, scratch_bytes, stream);
}

rssm_status rssm_step_precompute(const rssm_cache* cache, const void* x, const float* dt, const float* A,
                                 const void* B, const void* C, const float* D, const float* dt_bias,
                                 const int32_t* slot_idx, const int32_t* pnat, const int32_t* cu_seqlens,
                                 int32_t batch, int32_t T, void* out, void* scratch, size_t scratch_bytes,
                                 void* stream) {
  StepArgs a;
  rssm_status st = step_common(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, out, scratch,
                               scratch_bytes, &a);
  if (st != RSSM_OK || batch == 0) return st;
  if (static_cast<long long>(batch) * a.c.G > 0x7fffffffLL) return RSSM_ERR_UNSUPPORTED;
  return launch_precompute(a, stream) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_step_readout_gated(const rssm_cache* cache, const void* x, const float* dt, const float* A,
                                    const void* B, const void* C, const float* D, const float* dt_bias,
                                    const int32_t* slot_idx, const int32_t* pnat, const int32_t* cu_seqlens,
                                    int32_t batch, int32_t T, const void* z, void* out, void* scratch,
                                    size_t scratch_bytes, void* stream) {
  StepArgs a;
  rssm_status st = step_common(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, out, scratch,
                               scratch_bytes, &a);
  if (st != RSSM_OK || batch == 0) return st;
  if (z && !aligned16(z)) return RSSM_ERR_INVALID_ARGUMENT;
  a.z = static_cast<const uint16_t*>(z);
  const int sms = num_sms();
  if (sms <= 0) return RSSM_ERR_CUDA;
  return launch_readout(a, sms, stream) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_step_readout(const rssm_cache* cache, const void* x, const float* dt, const float* A, const void* B,
                              const void* C, const float* D, const float* dt_bias, const int32_t* slot_idx,
                              const int32_t* pnat, const int32_t* cu_seqlens, int32_t batch, int32_t T, void* out,
                              void* scratch, size_t scratch_bytes, void* stream) {
  return rssm_step_readout_gated(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, nullptr,
                                 out, scratch, scratch_bytes, stream);
}

rssm_status rssm_step_gated(const rssm_cache* cache, const void* x, const float* dt, const float* A, const void* B,
                            const void* C, const float* D, const float* dt_bias, const int32_t* slot_idx,
                            const int32_t* pnat, const int32_t* cu_seqlens, int32_t batch, int32_t T, const void* z,
                            void* out, void* scratch, size_t scratch_bytes, void* stream) {
  if (batch > 0 && z && !aligned16(z)) return RSSM_ERR_INVALID_ARGUMENT;  // checked before anything launches
  rssm_status st = rssm_step_precompute(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, out,
                                        scratch, scratch_bytes, stream);
  if (st != RSSM_OK) return st;
  return rssm_step_readout_gated(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, z, out,
                                 scratch, scratch_bytes, stream);
}

rssm_status rssm_step(const rssm_cache* cache, const void* x, const float* dt, const float* A, const void* B,
                      const void* C, const float* D, const float* dt_bias, const int32_t* slot_idx,
                      const int32_t* pnat, const int32_t* cu_seqlens, int32_t batch, int32_t T, void* out,
                      void* scratch, size_t scratch_bytes, void* stream) {
  return rssm_step_gated(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, nullptr, out,
                         scratch, scratch_bytes, stream);
}

namespace {
// validation and arguments of the flush+step call (and of its two halves)
rssm_status flush_step_args(const rssm_cache* cache, const void* x, const float* dt, const float* A, const void* B,
                            const void* C, const float* D, const float* dt_bias, const int32_t* slot_idx,
                            int32_t* pnat, const int32_t* cu_seqlens, int32_t batch, int32_t T, int32_t force,
                            uint64_t seed, void* out, void* scratch, size_t scratch_bytes, StepArgs* a, int* sms) {
  if (force != 0 && force != 1) return RSSM_ERR_INVALID_ARGUMENT;
  if (cache && cache->read_state) return RSSM_ERR_UNSUPPORTED;  // the one-call path keeps one checkpoint
  rssm_status st = step_common(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, out, scratch,
                               scratch_bytes, a);
  if (st != RSSM_OK || batch == 0) return st;
  if (scratch_bytes < flush_step_scratch_bytes(batch, cache->nheads, cache->ngroups, a->c.L, T))
    return RSSM_ERR_SCRATCH_TOO_SMALL;
  if (static_cast<long long>(batch) * a->c.H > (1LL << 30)) return RSSM_ERR_UNSUPPORTED;
  *sms = num_sms();
  if (*sms <= 0) return RSSM_ERR_CUDA;
  a->flush_mode = 1 + force;
  a->seed = seed;
  a->pnat_rw = pnat;
  a->fw = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) +
                                   step_scratch_bytes(batch, cache->nheads, cache->ngroups, a->c.L, T));
  return RSSM_OK;
}
}  // namespace

rssm_status rssm_flush_step_classify(const rssm_cache* cache, const void* x, const float* dt, const float* A,
                                     const void* B, const void* C, const float* D, const float* dt_bias,
                                     const int32_t* slot_idx, int32_t* pnat, const int32_t* cu_seqlens, int32_t batch,
                                     int32_t T, int32_t force, uint64_t seed, void* out, void* scratch,
                                     size_t scratch_bytes, void* stream) {
  StepArgs a;
  int sms = 0;
  rssm_status st = flush_step_args(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, force,
                                   seed, out, scratch, scratch_bytes, &a, &sms);
  if (st != RSSM_OK || batch == 0) return st;
  if (static_cast<long long>(batch) * a.c.G > 0x7fffffffLL) return RSSM_ERR_UNSUPPORTED;
  return launch_precompute(a, stream) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_flush_step_main(const rssm_cache* cache, const void* x, const float* dt, const float* A,
                                 const void* B, const void* C, const float* D, const float* dt_bias,
                                 const int32_t* slot_idx, int32_t* pnat, const int32_t* cu_seqlens, int32_t batch,
                                 int32_t T, int32_t force, uint64_t seed, void* out, void* scratch,
                                 size_t scratch_bytes, void* stream) {
  StepArgs a;
  int sms = 0;
  rssm_status st = flush_step_args(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, force,
                                   seed, out, scratch, scratch_bytes, &a, &sms);
  if (st != RSSM_OK || batch == 0) return st;
  return launch_readout_fold(a, sms, stream) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_flush_step(const rssm_cache* cache, const void* x, const float* dt, const float* A, const void* B,
                            const void* C, const float* D, const float* dt_bias, const int32_t* slot_idx,
                            int32_t* pnat, const int32_t* cu_seqlens, int32_t batch, int32_t T, int32_t force,
                            uint64_t seed, void* out, void* scratch, size_t scratch_bytes, void* stream) {
  rssm_status st = rssm_flush_step_classify(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T,
                                            force, seed, out, scratch, scratch_bytes, stream);
  if (st != RSSM_OK) return st;
  return rssm_flush_step_main(cache, x, dt, A, B, C, D, dt_bias, slot_idx, pnat, cu_seqlens, batch, T, force, seed, out,
                              scratch, scratch_bytes, stream);
}

rssm_status rssm_accept(const rssm_cache* cache, const int32_t* slot_idx, int32_t* pnat, const int32_t* accepted,
                        const int32_t* cu_seqlens, int32_t batch, int32_t T, void* stream) {
  Cache c;
  rssm_status st = check_cache(cache, &c);
  if (st != RSSM_OK) return st;
  if (batch < 0 || T < 0) return RSSM_ERR_INVALID_ARGUMENT;
  if (batch == 0) return RSSM_OK;
  if (!slot_idx || !pnat || !accepted) return RSSM_ERR_INVALID_ARGUMENT;
  return launch_accept(c, slot_idx, pnat, accepted, cu_seqlens, batch, T, stream) == cudaSuccess ? RSSM_OK
                                                                                                   : RSSM_ERR_CUDA;
}

rssm_status rssm_eval_spec_math(const float* in, float* out_exp, float* out_softplus, int64_t n, void* stream) {
  if (n < 0 || (n > 0 && !in)) return RSSM_ERR_INVALID_ARGUMENT;
  if (n == 0) return RSSM_OK;
  return launch_spec_math(in, out_exp, out_softplus, n, stream) == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA;
}

rssm_status rssm_selftest_wait_timeout(uint32_t* error_word, int32_t wait_ms, void* stream) {
  if (!error_word || (reinterpret_cast<uintptr_t>(error_word) & 3u)) return RSSM_ERR_INVALID_ARGUMENT;
  if (wait_ms < 1 || wait_ms > 10000) return RSSM_ERR_INVALID_ARGUMENT;
  return launch_wait_timeout(error_word, static_cast<unsigned>(wait_ms), stream) == cudaSuccess ? RSSM_OK
                                                                                               : RSSM_ERR_CUDA;
}

const char* rssm_status_string(rssm_status s) {
  switch (s) {
    case RSSM_OK: return "ok";
    case RSSM_ERR_INVALID_ARGUMENT: return "invalid argument";
    case RSSM_ERR_UNSUPPORTED: return "unsupported shape";
    case RSSM_ERR_SCRATCH_TOO_SMALL: return "scratch buffer too small";
    case RSSM_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

}  // extern "C"
