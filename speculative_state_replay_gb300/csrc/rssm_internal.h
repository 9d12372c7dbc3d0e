// rssm_internal.h -- structures shared by the host entry points and the
// kernels of librssm.  Not part of the public ABI.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "rssm.h"

namespace rssm {

constexpr int kDim = 64;      // head dim
constexpr int kDstate = 128;  // state dim
constexpr int kHeadElems = kDim * kDstate;
constexpr int kMaxL = 32;     // ring length the kernels are built for (one lane per ring slot)
constexpr int kMaxT = 8;      // draft tokens per step
constexpr int kRStride = 72;  // row stride (floats) of the one-call path's ring-term rows in shared memory
// ring-term block of one (row, head) in the step's scratch: kRDec decay floats
// (decay[t] for t < T, padded), then one 64-float row R[t][.] per token, the
// 32-byte chunk c of row t stored at chunk c ^ t (conflict-free reads of one
// column chunk across the rows); only the row's T_b rows are written and read
constexpr int kRDec = 8;
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr uint32_t kWaitTries = 2000;            // x 1 ms suspend hint: ~2 s bound on an mbarrier wait

// device view of an rssm_cache
struct Cache {
  int S, H, G, hpg, W, Tmax, L;
  int dtype, rounding;
  void* state;
  long long state_stride;
  float* scale;
  long long scale_stride;
  uint16_t* x_cache;
  long long x_stride;
  uint16_t* B_cache;
  long long B_stride;
  float* dt_cache;
  long long dt_stride;
  int* ring_start;
  unsigned* epoch;
  unsigned* err;
  // separate read checkpoint (8-bit codes + row scales, or NVFP4 codes +
  // block scales + per-slot global scale; nearest), or null
  void* read_state;
  long long read_stride;
  float* read_scale;
  long long read_scale_stride;
  int read_dtype;
  uint8_t* read_sf;
  long long read_sf_stride;
  float* read_gs;
};

// one flagged row of a flush (written by the flag kernel), 32 bytes
struct FlushRec {
  int b, s, r, p;
  unsigned epoch;  // epoch of the state this flush writes
  int pad[3];
};

// one row of a step (written by the precompute, read by the readout), 32 bytes.
// r and p are the ring start and live count the step works on: the live
// prefix the outputs replay and, for a row flushed in the same call, the
// prefix the fold folds.
struct RowRec {
  int s, r, p, Tb, tok0;
  int flags;           // bit 0: compute the row's outputs (else zeros for Tb tokens); bit 1: fold its live prefix
  unsigned epoch_new;  // epoch of the checkpoint the fold writes (bit 1 set)
  float gs;            // global scale of the slot's NVFP4 read checkpoint (1 otherwise)
};

// fold weights of one flushed (row, head) in the one-call path's scratch:
// w_j = e^{c_end - c_j} dt'_j for j < p (canonical fp32), then e^{c_end} at 32
constexpr int kFoldW = 40;

struct FlushArgs {
  Cache c;
  const float* A;
  const int* slot_idx;
  int* pnat;
  const int* cu;
  int batch, T, force;
  unsigned long long seed;
  // the previous step's acceptance, applied first (rssm_accept_flush); NULL: none
  const int* accepted;
  const int* acu;  // its sequence bounds (NULL: aT tokens a row)
  int aT;
  unsigned* ticket;  // scratch word: CTAs done with the flush (zero between calls)
  int* count;        // scratch: number of flagged rows (written at the end, for diagnostics)
  FlushRec* recs;    // scratch: flagged rows (written at the end, for diagnostics)
};

struct StepArgs {
  Cache c;
  const uint16_t* x;
  const float* dt;
  const float* A;
  const uint16_t* B;
  const uint16_t* C;
  const float* D;
  const float* dt_bias;
  const int* slot_idx;
  const int* pnat;
  const int* cu;
  int batch, T;
  int TP;  // T padded to 4 or 8
  int KB;  // ring rows padded to a multiple of 4
  uint16_t* out;
  const uint16_t* z;         // output gate [tok][H][64] bf16, or null: y * silu(z) (the readout)
  int flush_mode;            // rssm_flush_step: 1 fold rows with p + T_b > W; 2 every active row; 0 none
  unsigned long long seed;   // stochastic-rounding key of the fold (flush_mode != 0)
  int* pnat_rw;              // pnat, written by the fold's bookkeeping (flush_mode != 0)
  float* fw;                 // scratch [batch][H][kFoldW]: fold weights of flushed rows (flush_mode != 0)
  unsigned* rwork;           // scratch word: the readout's chunk counter, zeroed by the precompute
  RowRec* rows;  // scratch [batch]
  uint16_t* cf;  // scratch [batch][G][8][128]: C rows in the readout's MMA operand type
  float* rblk;   // scratch [batch][H][kRDec + TP*64]: decay[t], then the ring term R[t][d] (chunk-swizzled rows)
};

struct InitArgs {
  Cache c;
  const float* states;
  const int* ids;
  int n;
  unsigned long long seed;
};

__host__ __device__ inline int ring_pad(int L) { return (L + 3) & ~3; }
inline int t_pad(int T) { return T <= 4 ? 4 : 8; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// scratch layout: the first kScratchHead bytes hold the flush's ticket word
// (zero between calls) and count; every other layout starts after them
constexpr size_t kScratchHead = 256;
inline size_t flush_scratch_bytes(int batch) { return kScratchHead + align_up(sizeof(FlushRec) * (size_t)batch, 256); }
inline size_t step_rows_bytes(int batch) { return align_up(sizeof(RowRec) * (size_t)batch, 256); }
inline size_t step_cf_bytes(int batch, int G, int T) {
  (void)T;
  return align_up((size_t)batch * G * 8 * 128 * 2, 256);
}
inline size_t step_rblk_floats(int T) { return kRDec + (size_t)t_pad(T) * kDim; }
// float offset of R[t][d] inside a ring-term block
__host__ __device__ inline int rblk_offset(int t, int d) { return kRDec + t * kDim + ((((d >> 3) ^ t) & 7) << 3) + (d & 7); }
inline size_t step_scratch_bytes(int batch, int H, int G, int L, int T) {
  (void)L;
  const size_t blk = step_rblk_floats(T) * sizeof(float);
  return kScratchHead + step_rows_bytes(batch) + step_cf_bytes(batch, G, T) + align_up(blk * (size_t)batch * H, 256);
}
// the flush+step call: the step's scratch, then the fold weights
inline size_t flush_step_scratch_bytes(int batch, int H, int G, int L, int T) {
  return step_scratch_bytes(batch, H, G, L, T) + align_up((size_t)batch * H * kFoldW * sizeof(float), 256);
}

// launchers (defined in the .cu files); return a cudaError_t as int
int launch_flush(const FlushArgs& a, int num_sms, void* stream);
int launch_precompute(const StepArgs& a, void* stream);
int launch_readout(const StepArgs& a, int num_sms, void* stream);
int launch_readout_fold(const StepArgs& a, int num_sms, void* stream);
int launch_accept(const Cache& c, const int* slot_idx, int* pnat, const int* accepted, const int* cu, int batch,
                  int T, void* stream);
int launch_init(const InitArgs& a, void* stream);
int launch_spec_math(const float* in, float* oexp, float* osp, long long n, void* stream);
int launch_wait_timeout(unsigned* err, unsigned tries, void* stream);

}  // namespace rssm
