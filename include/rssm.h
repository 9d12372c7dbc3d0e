/*
 * rssm.h -- C ABI of librssm, a GB300 (sm_103a) implementation of the
 * ReplaySSM checkpointing selective-state-update for Mamba-2 decode with
 * speculative draft tokens.
 *
 * The op.  Each (slot, head) keeps a checkpoint state S0[dim=64][dstate=128]
 * and head-major ring buffers of the recent inputs (x, B and dt').  A decode
 * step with T draft tokens replays the live ring plus the drafts against S0
 * to produce the outputs, and appends the drafts to the rings; when the live
 * window fills, a flush folds the accepted prefix into a new checkpoint.
 * Sources, cited throughout by page and section:
 *   [FI]   FlashInfer PR #3975 "mamba checkpointing SSU: two-kernel split +
 *          ring-buffer cache for checkpointing SSU" (Description items 1-2,
 *          commit notes).
 *   [vS]   vLLM PR #65660 "WIP: [Mamba] Add separate CuTeDSL ReplaySSM
 *          checkpoints" (Overview, Claims, Details, commit notes).
 *   [vAPI] vLLM API docs for vllm.model_executor.layers.mamba.ops.
 *          replayssm_cutedsl (initialize_replayssm_state,
 *          selective_state_update_replayssm).
 *
 * Conventions shared by every entry point.
 *  - Memory: every pointer is caller-owned device memory unless stated
 *    otherwise; the library never allocates, frees or keeps a pointer after a
 *    call returns.  Temporary storage is a caller-provided `scratch` buffer
 *    of at least rssm_scratch_bytes() bytes ([FI] Description item 1:
 *    caller-provided scratch, allocated like the output, graph safe).  Zero
 *    the buffer once when it is allocated: rssm_flush keeps a counter in its
 *    first 4 bytes that must start at zero, and every call leaves it at zero
 *    (after a call that reported RSSM_ERRBIT_TIMEOUT, zero it again).  The
 *    first 256 bytes are the flush's; no other call writes them.
 *  - Streams: `stream` is a cudaStream_t (NULL = the legacy default
 *    stream).  Every call only enqueues kernels on it: no host
 *    synchronisation and no host read of device data, so calls can be
 *    captured in a CUDA graph ([vAPI] selective_state_update_replayssm: the
 *    call is prepared for graph capture).  Calls on one cache must be ordered
 *    on one stream (or by the caller).
 *  - Grid sizing: the persistent kernels size their grids for the device's
 *    SM count; a positive integer in the environment variable RSSM_SM_LIMIT
 *    (read at every call) caps the count they size for, to leave SMs to
 *    concurrent work.  Work is handed out per (row, head) and each unit is
 *    computed the same way by whichever CTA takes it, so results are the
 *    same bits for every grid size.
 *  - Alignment: all pointers and slot strides must give 16-byte aligned rows
 *    (the kernels move rows with bulk copies); violations return
 *    RSSM_ERR_INVALID_ARGUMENT before anything is launched.
 *  - Slots: slot 0 is a padding slot; rows whose slot id is <= 0 or >= the
 *    number of slots are ignored: their outputs are written as zeros and no
 *    cache byte is touched ([vAPI] module docstring and
 *    initialize_replayssm_state).  Active slot ids in one call must be
 *    unique ([vAPI] selective_state_update_replayssm docstring);
 *    duplicates are undefined behaviour.
 *  - Errors: host-detectable problems return a status before any launch.
 *    Data-dependent problems found on the device (bad pnat, bad cu_seqlens,
 *    bad accepted counts) set bits in cache->error_word (sticky, never
 *    cleared by the library) and the affected row is skipped (outputs 0).
 *    A kernel that gives up waiting on its own pipeline sets
 *    RSSM_ERRBIT_TIMEOUT and returns.
 *
 * Call order of one decode step (the library owns the ring bookkeeping on
 * the device):
 *     rssm_flush   -- rows whose live window would overflow fold their live
 *                     prefix into S0, advance ring_start, reset pnat
 *     rssm_step    -- outputs for the drafts; appends them to the rings
 *     rssm_accept  -- pnat += accepted drafts (after verification)
 * (rssm_accept_flush takes a step's rssm_accept and the next step's
 * rssm_flush in one launch.)
 */
#ifndef RSSM_H
#define RSSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RSSM_OK = 0,
  RSSM_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size/stride/alignment, bad enum */
  RSSM_ERR_UNSUPPORTED = 2,      /* shape outside what the kernels are built for */
  RSSM_ERR_SCRATCH_TOO_SMALL = 3,
  RSSM_ERR_CUDA = 4              /* a CUDA runtime call or launch failed */
} rssm_status;

/* Checkpoint state formats.  8-bit formats carry one FP32 scale per
 * (slot, head, d) row of 128 dstate values ([vS] commit notes: quantised
 * checkpoints with FP32 row scales). */
typedef enum { RSSM_F32 = 0, RSSM_BF16 = 1, RSSM_F16 = 2, RSSM_I8 = 3, RSSM_E4M3 = 4, RSSM_NVFP4 = 5 } rssm_dtype;
/* RSSM_NVFP4 is a read-checkpoint format only (rssm_cache.read_dtype): FP4
 * E2M1 codes (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), two per byte with the
 * even dstate element in the low nibble, one E4M3 scale per 16 consecutive
 * dstate values of a row, one FP32 global scale per slot; a value decodes as
 * e2m1(code) * e4m3(scale) * global ([vAPI] initialize_replayssm_state,
 * NVFP4 branch; the NVFP4 kernels' state_lo / sf_lo / sg_meta arguments). */

/* How a flush or init rounds fp32 values to the state format: nearest
 * (ties to even, saturating) or stochastic with a Philox4x32-7 hash keyed by
 * the seed and countered by (element/4, head, slot, flush epoch).  Both are
 * deterministic functions of the inputs ([vS] Claims; [FI] commit notes on
 * Philox stochastic rounding). */
typedef enum { RSSM_ROUND_NEAREST = 0, RSSM_ROUND_STOCHASTIC = 1 } rssm_rounding;

/* bits of *error_word */
#define RSSM_ERRBIT_PNAT 1u    /* pnat < 0, or pnat + tokens > L (step), or pnat > L (flush) */
#define RSSM_ERRBIT_SEQLEN 2u  /* a row's token count (cu_seqlens) < 0 or > T */
#define RSSM_ERRBIT_ACCEPT 4u  /* accepted < 0 or > the row's token count */
#define RSSM_ERRBIT_TIMEOUT 8u /* a kernel gave up waiting on its own copy pipeline */

/*
 * The cache of all slots.  Layouts follow the ring-buffer cache contract of
 * [FI] Description item 2 (head-major, single-buffered rings) with
 * L = max_window + npredicted.  Strides are in ELEMENTS between consecutive
 * slots and may exceed the dense size ([vAPI] module docstring: cache pages
 * may carry padding between slots).
 */
typedef struct {
  int32_t num_slots;   /* S, including padding slot 0 */
  int32_t nheads;      /* H */
  int32_t ngroups;     /* G; head h uses group h / (H / G) */
  int32_t dim;         /* must be 64 */
  int32_t dstate;      /* must be 128 */
  int32_t max_window;  /* W: a row flushes before a step when pnat + tokens > W */
  int32_t npredicted;  /* max draft tokens per step; L = W + npredicted <= 32 */
  int32_t state_dtype; /* rssm_dtype */
  int32_t rounding;    /* rssm_rounding, used by rssm_flush and rssm_init_state */
  void *state;         int64_t state_slot_stride; /* [slot][H][64][128] of state_dtype */
  float *scale;        int64_t scale_slot_stride; /* [slot][H][64] f32; 8-bit only (else may be NULL) */
  void *x_cache;       int64_t x_slot_stride;     /* bf16 [slot][H][L][64] */
  void *B_cache;       int64_t B_slot_stride;     /* bf16 [slot][G][L][128] */
  float *dt_cache;     int64_t dt_slot_stride;    /* f32 [slot][H][L], post-softplus dt' */
  int32_t *ring_start; /* [slot]: physical position of live token 0 */
  uint32_t *flush_epoch; /* [slot]: number of flushes since init (random counter) */
  uint32_t *error_word;  /* [1]: sticky RSSM_ERRBIT_* bits */
  /* Optional separate read checkpoint ([vS] Overview: an FP16 recurrence
   * checkpoint with stochastic rounding, FP32 flush work, an FP8 read
   * checkpoint, BF16 readout; Claims: read checkpoints use nearest
   * encoding).  8-bit codes of read_dtype with one FP32 scale per (slot,
   * head, d) row, written with nearest rounding from the same fp32 values as
   * the recurrence state `state` -- the FP32 prefill states in
   * rssm_init_state, the fold's fp32 accumulators in rssm_flush -- and read
   * by rssm_step's readout in place of `state`.  With a read checkpoint every
   * fold takes the canonical fp32 order, so both encodings are functions of
   * the inputs bit for bit.  read_state = NULL: no read checkpoint (the
   * step reads `state`); the other read fields are then ignored.
   * rssm_flush_step does not take a read checkpoint (RSSM_ERR_UNSUPPORTED). */
  void *read_state;    int64_t read_slot_stride;       /* 8-bit [slot][H][64][128]; NVFP4: bytes [slot][H][64][64] */
  float *read_scale;   int64_t read_scale_slot_stride; /* f32 [slot][H][64] (8-bit read formats) */
  int32_t read_dtype;                                  /* RSSM_I8, RSSM_E4M3 or RSSM_NVFP4 */
  /* NVFP4 read checkpoint only (else ignored): the E4M3 block scales
   * [slot][H][64][8] (bytes; stride in bytes) and the FP32 global scale of
   * each slot [slot].  rssm_init_state sets a slot's global scale to the
   * largest magnitude of its FP32 prefill state / (6 * 448) (1 for a zero
   * state); the slot's flushes keep it.  Block scale = e4m3 nearest of
   * (block max / (6 * global)), saturating; code = e2m1 nearest of
   * (v * (1 / (global * block scale))) (one rounded reciprocal per block),
   * saturating at 6 (0 where the block scale is 0). */
  void *read_sf;       int64_t read_sf_slot_stride;
  float *read_gs;
} rssm_cache;

/*
 * Bytes of scratch rssm_flush / rssm_step need for `batch` rows of up to T
 * tokens.  The same buffer may serve both calls (they are stream ordered).
 * Returns 0 if the cache description is invalid.
 */
size_t rssm_scratch_bytes(const rssm_cache *cache, int32_t batch, int32_t T);

/*
 * Initialise checkpoints from FP32 prefill states ([vAPI]
 * initialize_replayssm_state): for i < n, states[i] ([H][64][128] f32,
 * contiguous, device) is rounded to the state format (flush epoch 0) into
 * slot slot_idx[i]; that slot's x/B/dt rings are zeroed and its ring_start
 * and flush_epoch set to 0.  Ids <= 0 or >= num_slots are ignored.  The
 * caller sets the rows' pnat to 0.  `seed` keys stochastic rounding.
 */
rssm_status rssm_init_state(const rssm_cache *cache, const float *states, const int32_t *slot_idx, int32_t n,
                            uint64_t seed, void *stream);

/*
 * Flush ([FI] commit notes: the write decision is taken per slot at run time
 * as prev_k + T > max_window; [vS] Details: only the accepted prefix enters
 * the checkpoint).  For every active row b (slot s = slot_idx[b], p =
 * pnat[b] live tokens, T_b tokens this step):
 *   flagged  = force ? 1 : (p + T_b > max_window)
 * and for flagged rows, per head h, with c_j = sum_{i<=j} A[h] dt'_i over the
 * live tokens (fp32, ascending), c_end = c_{p-1} (0 if p = 0):
 *   S0' = e^{c_end} S0 + sum_{j<p} e^{c_end - c_j} dt'_j x_j (outer) B_j
 * computed in fp32 in one canonical order (acc = e^{c_end} S0; then for j
 * ascending acc = fma(e^{c_end-c_j} dt'_j x_j[d], B_j[n], acc)) -- except
 * that 2-byte states with nearest rounding and p >= 9 are folded on the tensor
 * cores (fp32 accumulation from e^{c_end} S0, e^{c_end-c_j} dt'_j x_j[d] split
 * into three bf16 parts that carry all 24 bits of its fp32 value), which
 * differs from the canonical order by summation order only -- rounded to the state format with flush epoch
 * flush_epoch[s] + 1; then ring_start[s] = (ring_start[s] + p) mod L,
 * pnat[b] = 0, flush_epoch[s] += 1.  f32, 8-bit and stochastically rounded
 * checkpoints are therefore a function of the inputs bit for bit.
 *   A        [H] f32 (device)
 *   slot_idx [batch] i32 (device)
 *   pnat     [batch] i32 (device, in/out): live accepted tokens per row
 *   cu_seqlens [batch+1] i32 (device) or NULL: row b has cu[b+1]-cu[b]
 *            tokens (<= T); NULL: every row has T tokens
 *   force    0: flush iff pnat + T_b > max_window; 1: every active row
 */
rssm_status rssm_flush(const rssm_cache *cache, const float *A, const int32_t *slot_idx, int32_t *pnat,
                       const int32_t *cu_seqlens, int32_t batch, int32_t T, int32_t force, uint64_t seed,
                       void *scratch, size_t scratch_bytes, void *stream);

/*
 * The previous step's acceptance and this step's flush in one launch: the
 * same results, bit for bit (pnat, checkpoints, 8-bit scales, rings,
 * ring_start, flush_epoch, error bits), as
 *   rssm_accept(cache, slot_idx, pnat, accepted, accept_cu_seqlens, batch, accept_T, stream)
 *   rssm_flush(cache, A, slot_idx, pnat, cu_seqlens, batch, T, force, seed, scratch, scratch_bytes, stream)
 * A row whose acceptance fails rssm_accept's checks keeps its pnat (and sets
 * the error bit, as rssm_accept does) and is then classified like any other.
 * The decode loop becomes: rssm_accept_flush (the drafts verified after the
 * previous rssm_step), then rssm_step; one launch fewer per step.
 *   accepted          [batch] i32 (device, required)
 *   accept_cu_seqlens [batch+1] i32 (device) or NULL: the previous step's
 *                     sequence bounds (NULL: accept_T tokens a row)
 *   accept_T          the previous step's T
 * The other arguments as in rssm_flush.
 */
rssm_status rssm_accept_flush(const rssm_cache *cache, const float *A, const int32_t *slot_idx, int32_t *pnat,
                              const int32_t *accepted, const int32_t *accept_cu_seqlens, int32_t accept_T,
                              const int32_t *cu_seqlens, int32_t batch, int32_t T, int32_t force, uint64_t seed,
                              void *scratch, size_t scratch_bytes, void *stream);

/*
 * Step: replay/readout and ring append ([FI] Description items 1-2).  For
 * active row b (slot s, p = pnat[b] live tokens, T_b new tokens, token
 * offset tok0 = cu_seqlens[b] or b*T) and head h (group g = h/(H/G)), with
 * the live ring followed by the new tokens as logical tokens k = 0..p+T_b-1:
 *   dt'_k = softplus(dt[tok][h] + dt_bias[h]) for new tokens, dt_cache for live
 *   c_k   = sum_{i<=k} A[h] dt'_i
 *   y_t   = e^{c_{p+t}} (S0 . C_t) + sum_{k<=p+t} e^{c_{p+t}-c_k} dt'_k (C_t . B_k) x_k
 *           + D[h] x_t,                         rounded to bf16
 * then x_t, B_t (once per group) and dt'_t are appended at physical position
 * (ring_start[s] + p + t) mod L.  S0 is never written ([vS] Details).
 *   x   bf16 [tok][H][64]     dt f32 [tok][H]       A, D, dt_bias f32 [H]
 *   B,C bf16 [tok][G][128]    out bf16 [tok][H][64] (written)
 *   slot_idx, pnat [batch] i32 (read only); cu_seqlens as in rssm_flush.
 *   T   tokens per row (max tokens per row with cu_seqlens), 1..min(8, npredicted).
 * Requires p + T_b <= L on the device (guaranteed after rssm_flush).
 */
rssm_status rssm_step(const rssm_cache *cache, const void *x, const float *dt, const float *A, const void *B,
                      const void *C, const float *D, const float *dt_bias, const int32_t *slot_idx,
                      const int32_t *pnat, const int32_t *cu_seqlens, int32_t batch, int32_t T, void *out,
                      void *scratch, size_t scratch_bytes, void *stream);

/*
 * One decode iteration's flush and step in one call, in the shape of the
 * pages' own design ([FI] Description item 1: a precompute, then a persistent
 * main kernel that replays the state and, for rows whose window is full,
 * writes the folded checkpoint in the same pass).  Same results as
 * rssm_flush(cache, A, slot_idx, pnat, cu_seqlens, batch, T, force, seed)
 * followed by rssm_step(...) with the same arguments, except as noted:
 *  - checkpoints, 8-bit scales, rings, ring_start, pnat, flush_epoch and error
 *    bits: the same bits -- every fold here takes the canonical fp32 order
 *    (also for 2-byte states with nearest rounding, which rssm_flush may fold
 *    on the tensor cores);
 *  - outputs: a flushed row's outputs replay its whole live prefix from the
 *    old checkpoint (the fold's fp32 values before their rounding), where the
 *    two calls read the rounded new checkpoint; they agree within the bf16
 *    output tolerance;
 *  - a row with pnat + T_b > L (its new tokens would land on live slots the
 *    fold reads) is refused with RSSM_ERRBIT_PNAT (zero outputs, caches
 *    untouched), where the two calls fold it first.  The decode protocol
 *    (flush -> step -> accept) never produces such a row when max_window >=
 *    npredicted.
 * Each flushed checkpoint is read from HBM once (folded in the stage its
 * outputs are read from) instead of twice.
 *   pnat     [batch] i32 (device, in/out): set to 0 for flushed rows
 *   force, seed as in rssm_flush; scratch of at least rssm_scratch_bytes().
 * A cache with a separate read checkpoint is refused (RSSM_ERR_UNSUPPORTED).
 */
rssm_status rssm_flush_step(const rssm_cache *cache, const void *x, const float *dt, const float *A, const void *B,
                            const void *C, const float *D, const float *dt_bias, const int32_t *slot_idx,
                            int32_t *pnat, const int32_t *cu_seqlens, int32_t batch, int32_t T, int32_t force,
                            uint64_t seed, void *out, void *scratch, size_t scratch_bytes, void *stream);

/*
 * The two halves of rssm_flush_step, exposed for profiling: rssm_flush_step
 * == rssm_flush_step_classify followed by rssm_flush_step_main with the same
 * arguments and scratch.
 *   classify: per (row, group): the flush decision, dt', cumulative A dt', the
 *             C.B contraction and the replay terms over the whole live prefix
 *             (as rssm_step_precompute), the ring appends, and for flushed
 *             rows the fold weights in canonical fp32.
 *   main:     per (row, head): streams S0 once, forms y, folds flushed heads
 *             and writes their checkpoints; the flush's bookkeeping.
 */
rssm_status rssm_flush_step_classify(const rssm_cache *cache, const void *x, const float *dt, const float *A,
                                     const void *B, const void *C, const float *D, const float *dt_bias,
                                     const int32_t *slot_idx, int32_t *pnat, const int32_t *cu_seqlens, int32_t batch,
                                     int32_t T, int32_t force, uint64_t seed, void *out, void *scratch,
                                     size_t scratch_bytes, void *stream);
rssm_status rssm_flush_step_main(const rssm_cache *cache, const void *x, const float *dt, const float *A,
                                 const void *B, const void *C, const float *D, const float *dt_bias,
                                 const int32_t *slot_idx, int32_t *pnat, const int32_t *cu_seqlens, int32_t batch,
                                 int32_t T, int32_t force, uint64_t seed, void *out, void *scratch,
                                 size_t scratch_bytes, void *stream);

/*
 * The two halves of rssm_step, exposed for profiling and for callers that
 * want to place other work between them.  rssm_step == rssm_step_precompute
 * followed by rssm_step_readout with the same arguments and scratch.
 *   precompute: per (row, group): dt', cumulative A dt', C.B contraction,
 *               the decayed replay coefficients applied to the x rows (the
 *               ring term) into scratch; appends B, x and dt' to the rings.
 *   readout:    per (row, head): streams S0 once, forms y.
 */
rssm_status rssm_step_precompute(const rssm_cache *cache, const void *x, const float *dt, const float *A,
                                 const void *B, const void *C, const float *D, const float *dt_bias,
                                 const int32_t *slot_idx, const int32_t *pnat, const int32_t *cu_seqlens,
                                 int32_t batch, int32_t T, void *out, void *scratch, size_t scratch_bytes,
                                 void *stream);
rssm_status rssm_step_readout(const rssm_cache *cache, const void *x, const float *dt, const float *A,
                              const void *B, const void *C, const float *D, const float *dt_bias,
                              const int32_t *slot_idx, const int32_t *pnat, const int32_t *cu_seqlens,
                              int32_t batch, int32_t T, void *out, void *scratch, size_t scratch_bytes,
                              void *stream);

/*
 * rssm_step and rssm_step_readout with Mamba-2's output gate: every output is
 * y_t[d] * silu(z_t[d]) (silu(v) = v / (1 + e^-v)), formed in fp32 before
 * the bf16 rounding; the FlashInfer PR's commit notes list z among the
 * operands its monolithic kernel stages next to x.  z bf16 [tok][H][64]
 * (device, 16-byte aligned; read only), laid out like out; z = NULL gives
 * rssm_step / rssm_step_readout exactly.  Padding and rejected rows still
 * get zeros.  Errors as rssm_step (a misaligned z: RSSM_ERR_INVALID_ARGUMENT,
 * before any launch).  rssm_step_gated == rssm_step_precompute followed by
 * rssm_step_readout_gated.
 */
rssm_status rssm_step_gated(const rssm_cache *cache, const void *x, const float *dt, const float *A, const void *B,
                            const void *C, const float *D, const float *dt_bias, const int32_t *slot_idx,
                            const int32_t *pnat, const int32_t *cu_seqlens, int32_t batch, int32_t T, const void *z,
                            void *out, void *scratch, size_t scratch_bytes, void *stream);
rssm_status rssm_step_readout_gated(const rssm_cache *cache, const void *x, const float *dt, const float *A,
                                    const void *B, const void *C, const float *D, const float *dt_bias,
                                    const int32_t *slot_idx, const int32_t *pnat, const int32_t *cu_seqlens,
                                    int32_t batch, int32_t T, const void *z, void *out, void *scratch,
                                    size_t scratch_bytes, void *stream);

/*
 * Commit verified drafts: pnat[b] += accepted[b] for active rows, so the
 * first accepted[b] tokens appended by the last rssm_step join the live
 * prefix; the rest stay outside it and are overwritten by later appends
 * ([vS] Details: rejected drafts never reach the checkpoint).  accepted
 * [batch] i32 (device), 0 <= accepted[b] <= T_b, else RSSM_ERRBIT_ACCEPT.
 */
rssm_status rssm_accept(const rssm_cache *cache, const int32_t *slot_idx, int32_t *pnat, const int32_t *accepted,
                        const int32_t *cu_seqlens, int32_t batch, int32_t T, void *stream);

/*
 * Diagnostics: the device versions of the fixed-sequence fp32 exp and
 * softplus the flush and the dt' ring use (Cody-Waite reduction with a
 * degree-7 Taylor polynomial; softplus(v) = log1p(exp(v)) via an atanh
 * series, v itself above 20).  in/out_exp/out_softplus are [n] f32 device.
 */
rssm_status rssm_eval_spec_math(const float *in, float *out_exp, float *out_softplus, int64_t n, void *stream);

/*
 * Diagnostics: a self-test of the bounded waits every pipeline kernel uses
 * (a wait that gives up records RSSM_ERRBIT_TIMEOUT and the kernel returns
 * instead of hanging; the pages have no counterpart to this call).  Launches
 * one warp that waits on an mbarrier told to expect 256 bytes of transactions
 * no copy will bring, with the library's wait bounded to about wait_ms
 * milliseconds (1..10000); the wait runs out, RSSM_ERRBIT_TIMEOUT is set in
 * *error_word (device, 4-byte aligned) and the kernel returns.  A genuine
 * bulk copy issued next to it is waited for in full, so nothing is in flight
 * when the kernel ends and the context stays usable.
 */
rssm_status rssm_selftest_wait_timeout(uint32_t *error_word, int32_t wait_ms, void *stream);

const char *rssm_status_string(rssm_status status);

/*
 * rssm_step without a caller scratch buffer.  The pages have no counterpart
 * to this entry point; it exists for callers that cannot allocate device
 * memory -- an engine whose allocator has already reserved the GPU and hands
 * out no per-call workspace, or a C/FFI host with no device allocator.
 *
 * Same arguments, semantics and results as rssm_step, minus scratch and
 * scratch_bytes: the scratch is a fixed array of
 * RSSM_STEP_STATIC_SCRATCH_BYTES bytes compiled into the library, present on
 * every GPU that loads it until the process exits.  A step whose
 * rssm_scratch_bytes() exceeds that size returns RSSM_ERR_SCRATCH_TOO_SMALL
 * and launches nothing.  The call allocates and frees nothing.
 *  - The first call in each CUDA context looks up the array's device address
 *    (once per context, with that context current: the primary context of a
 *    device, a context the caller made current, or the one created after a
 *    device reset each get their own lookup); make that first call before
 *    any stream capture.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind; nothing in it needs to start at zero.  Calls whose kernels
 *    overlap on the GPU (different streams without ordering) race on the
 *    array; order them.
 */
#define RSSM_STEP_STATIC_SCRATCH_BYTES (16u << 20)
rssm_status rssm_step_static_scratch(const rssm_cache *cache, const void *x, const float *dt, const float *A,
                                     const void *B, const void *C, const float *D, const float *dt_bias,
                                     const int32_t *slot_idx, const int32_t *pnat, const int32_t *cu_seqlens,
                                     int32_t batch, int32_t T, void *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* RSSM_H */
