// rssm_flush.cu -- flush (classify + fold + requantise + bookkeeping), init,
// accept.
//
// Flush of the ReplaySSM checkpointing SSU (FlashInfer PR #3975, commit note
// on the persistent path: the write decision prev_k + T > max_window is
// taken per slot at run time; vLLM PR #65660, Details: only the accepted
// prefix enters the checkpoint).  One persistent kernel, flush_kernel:
//   every CTA classifies the rows (p + T_b > max_window, or all under force)
//   and folds its range of (flagged row, head) units:
//       S0' = e^{c_end} S0 + sum_j e^{c_end-c_j} dt'_j x_j (x) B_j
//   in fp32, canonical order, then rounds to the state format; the CTA that
//   finishes classifying last advances the ring bookkeeping (ring_start += p
//   mod L, pnat = 0, epoch += 1) while the folds run.  Under
//   rssm_accept_flush the classification first applies the previous step's
//   acceptance (pnat += accepted, under rssm_accept's checks) and the
//   bookkeeping writes every active row's new pnat.
#include <cuda_runtime.h>

#include <cstring>

#include "rssm_device.cuh"
#include "rssm_readout.cuh"

namespace rssm {

// ---------------------------------------------------------------------------
// classification
// ---------------------------------------------------------------------------
struct RowFlag {
  int flag, s, p;
  int book;  // the acceptance applied: pnat[b] becomes p (0 if flagged)
};

// a row's flush decision: active rows with p + T_b > max_window (all active
// rows under force); rows failing a check set an error bit (when `errors`).
// With an acceptance (rssm_accept_flush) p is first pnat + accepted, under
// rssm_accept's checks (a row failing them keeps its pnat).
__device__ __forceinline__ RowFlag row_flag(const FlushArgs& a, int b, bool errors) {
  const Cache& c = a.c;
  RowFlag f = {0, 0, 0, 0};
  // the row's loads are independent: issue them together (one round trip)
  const int s = a.slot_idx[b];
  int p = a.pnat[b];
  const int Tb = a.cu ? a.cu[b + 1] - a.cu[b] : a.T;
  int acc = 0, Ta = 0;
  if (a.accepted) {
    acc = a.accepted[b];
    Ta = a.acu ? a.acu[b + 1] - a.acu[b] : a.aT;
  }
  if (s < 1 || s >= c.S) return f;
  if (a.accepted) {
    if (Ta < 0 || Ta > a.aT) {
      if (errors) set_error(c.err, RSSM_ERRBIT_SEQLEN);
    } else if (acc < 0 || acc > Ta) {
      if (errors) set_error(c.err, RSSM_ERRBIT_ACCEPT);
    } else if (p < 0 || p + acc > c.L) {
      if (errors) set_error(c.err, RSSM_ERRBIT_PNAT);
    } else {
      p += acc;
      f.book = 1;
    }
  }
  f.s = s;
  f.p = p;
  if (Tb < 0 || Tb > a.T) {
    if (errors) set_error(c.err, RSSM_ERRBIT_SEQLEN);
  } else if (p < 0 || p > c.L) {
    if (errors) set_error(c.err, RSSM_ERRBIT_PNAT);
  } else if (a.force || p + Tb > c.W) {
    f.flag = 1;
  }
  return f;
}

// exclusive prefix of `flag` over the CTA's threads in thread order (every
// thread calls it); `total` gets the CTA's sum
__device__ __forceinline__ int block_excl_scan(int flag, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int wpre = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  int before = 0, tot = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
    const int v = wsum[w];
    if (w < warp) before += v;
    tot += v;
  }
  __syncthreads();  // wsum is reused
  total = tot;
  return before + wpre;
}

// ---------------------------------------------------------------------------
// tensor-core pieces of the fold (2-byte states, nearest rounding)
// ---------------------------------------------------------------------------
// d += A B on one m16n8k16 tile, bf16 operands, fp32 accumulation; a0..a3 =
// A[g][2c..2c+1], A[g+8][2c..], A[g][2c+8..], A[g+8][2c+8..]; b0, b1 =
// B[2c..2c+1][g], B[2c+8..2c+9][g]; d = D[g][2c..2c+1], D[g+8][2c..2c+1]
// (g = lane / 4, c = lane % 4)
__device__ __forceinline__ void mma16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// four 8x8 b16 matrices from shared memory (lane 8i + k gives row k of matrix
// i); lane (g, c) receives row g, columns 2c..2c+1 of each -- with .trans,
// rows 2c..2c+1 of column g
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}
// fp32 pair -> bf16 pair, round to nearest even, low half = first
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// fold kernel
// ---------------------------------------------------------------------------
struct FoldMeta {
  int s, h, p;
  unsigned epoch;
};

struct FoldLayout {
  int ns, KB;
  uint32_t s0_bytes, scale_off, x_off, b_off, dt_off, sc_off, w_off, stage_bytes;
  uint32_t meta_off, rows_off, stages_off, total;
};

// 2-byte states: S0 arrives as the readout's TMA boxes (64 rows x 128 bytes,
// 128-byte swizzle) and the live x and B rows in rows padded by 16 bytes, so
// that 8 rows read at one column (ldmatrix, the tensor-core fold's fragments)
// fall on distinct banks.  Other states: S0 and the rows as stored.
__host__ __device__ constexpr bool fold_2byte(int dtype) { return dtype == RSSM_BF16 || dtype == RSSM_F16; }
__host__ __device__ constexpr int fold_xs(int dtype) { return fold_2byte(dtype) ? kDim + 8 : kDim; }        // x row stride (elements)
__host__ __device__ constexpr int fold_bs(int dtype) { return fold_2byte(dtype) ? kDstate + 8 : kDstate; }  // B row stride (elements)

// barriers | per-stage metadata | the records of the flushed rows this CTA
// folds (up to `maxrows`) | stages; one stage: S0 | 8-bit scales | live x rows
// | live B rows | live dt' | A of the head | the fold weights
__host__ __device__ inline FoldLayout fold_layout(int dtype, int L, int ns, int maxrows) {
  FoldLayout f;
  f.ns = ns;
  f.KB = (L + 3) & ~3;
  const int esz = dtype == RSSM_F32 ? 4 : fold_2byte(dtype) ? 2 : 1;
  const uint32_t align = fold_2byte(dtype) ? 1024u : 128u;  // swizzled TMA boxes need 1024-byte alignment
  f.s0_bytes = kHeadElems * esz;
  uint32_t o = f.s0_bytes;
  f.scale_off = o;
  if (dtype == RSSM_I8 || dtype == RSSM_E4M3) o += 256;
  f.x_off = o;
  o += f.KB * fold_xs(dtype) * 2;
  f.b_off = o;
  o += f.KB * fold_bs(dtype) * 2;
  f.dt_off = o;
  o += f.KB * 4;
  f.sc_off = o;
  o += 16;
  f.w_off = o;  // the fold weights w_j (32 floats) and e^{c_end}, written by the weights warp
  o += 48 * 4;
  f.stage_bytes = (o + align - 1) & ~(align - 1);
  f.meta_off = 256;  // after the barriers
  f.rows_off = 512;
  f.stages_off = (f.rows_off + maxrows * static_cast<uint32_t>(sizeof(FlushRec)) + align - 1) & ~(align - 1);
  f.total = f.stages_off + f.ns * f.stage_bytes + (align == 1024u ? 1024u : 0u);  // + slack to align the base
  return f;
}

// smallest live prefix folded on the tensor cores (2-byte states, nearest
// rounding, no read checkpoint); shorter prefixes take the CUDA-core fold (K
// is padded to 16)
constexpr int kMmaMinP = 9;

// The separate read checkpoint of head h in slot s: the lane's 4 x 8 fp32
// values (the ones the recurrence state was just rounded from) encoded to the
// 8-bit read format with nearest rounding and per-row scales
__device__ __forceinline__ void store_read_checkpoint(const Cache& c, float (&acc)[4][8], int r0, int c0, int lane,
                                                      int s, int h) {
  if (c.read_dtype == RSSM_NVFP4) {  // codes [64][64 bytes] and block scales [64][8] of the head
    uint8_t* rs = static_cast<uint8_t*>(c.read_state) + static_cast<long long>(s) * c.read_stride +
                  static_cast<long long>(h) * (kHeadElems / 2);
    uint8_t* sf = c.read_sf + static_cast<long long>(s) * c.read_sf_stride + h * kDim * 8;
    quantize_store_nvfp4(acc, r0, c0, lane, rs, sf, c.read_gs[s]);
    return;
  }
  uint8_t* rs = static_cast<uint8_t*>(c.read_state) +
                static_cast<long long>(s) * c.read_stride + static_cast<long long>(h) * kHeadElems;
  float* rsc = c.read_scale + static_cast<long long>(s) * c.read_scale_stride + h * kDim;
  if (c.read_dtype == RSSM_I8)
    quantize_store<RSSM_I8>(acc, r0, c0, lane, rs, rsc, RSSM_ROUND_NEAREST, 0u, 0u, 0u, 0ull);
  else
    quantize_store<RSSM_E4M3>(acc, r0, c0, lane, rs, rsc, RSSM_ROUND_NEAREST, 0u, 0u, 0u, 0ull);
}

// Classification, fold, requantisation and bookkeeping of rssm_flush in one
// kernel.  Every CTA classifies all rows (two passes over slot_idx, pnat and
// the sequence bounds) and keeps the records of the flushed rows its range of
// (flushed row, head) units covers; then the producer warp fills the stages,
// the weights warp forms each unit's fold weights and the 8 consumer warps
// fold.  The bookkeeping is written by the CTA that takes the last ticket once
// it has classified (a self-resetting ticket), i.e. after every CTA has read
// the values it replaces; nothing in the kernel reads them afterwards.
constexpr int kWeightsWarp = kConsumerWarps + 1;
constexpr int kFlushThreads = kThreads + 32;

template <int DT>
__global__ void __launch_bounds__(kFlushThreads, 2)
    flush_kernel(const __grid_constant__ CUtensorMap s0map, FlushArgs a, int ns, int maxrows) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  constexpr bool k2B = fold_2byte(DT);
  constexpr int XS = fold_xs(DT), BS = fold_bs(DT);
  uint8_t* smem = k2B ? reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))
                      : smem_raw;
  __shared__ int wsum[kFlushThreads / 32];
  __shared__ int s_last;
  const Cache& c = a.c;
  const FoldLayout lay = fold_layout(DT, c.L, ns, maxrows);
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  const int L = c.L, H = c.H;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 8;
  uint64_t* wready = full + 16;  // the stage's fold weights are in place
  FoldMeta* meta = reinterpret_cast<FoldMeta*>(smem + lay.meta_off);
  FlushRec* rows_s = reinterpret_cast<FlushRec*>(smem + lay.rows_off);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < lay.ns; ++st) {
      mbar_init(&full[st], 1 + 32);  // producer lane 0 + one cp.async arrival per producer lane
      mbar_init(&empty[st], kConsumerWarps);
      mbar_init(&wready[st], 1);
    }
    fence_barrier_init();
  }
  pdl_wait();  // pnat as the previous call left it
  pdl_trigger();
  // pass 1: the number of flushed rows (CTA 0 reports bad rows); the flagged
  // rows' ring start and epoch are prefetched for pass 2
  int count = 0;
  for (int b0 = 0; b0 < a.batch; b0 += kFlushThreads) {
    const int b = b0 + tid;
    const RowFlag f = b < a.batch ? row_flag(a, b, blockIdx.x == 0) : RowFlag{0, 0, 0, 0};
    if (f.flag) {
      asm volatile("prefetch.global.L1 [%0];" ::"l"(c.ring_start + f.s));
      asm volatile("prefetch.global.L1 [%0];" ::"l"(c.epoch + f.s));
    }
    count += __syncthreads_count(f.flag);
  }
  if (count == 0 && !a.accepted) {  // nothing to fold or book (every CTA sees the same count)
    if (blockIdx.x == 0 && tid == 0) *a.count = 0;
    return;
  }
  if (blockIdx.x == 0 && tid == 0) *a.count = count;
  const long long units = static_cast<long long>(count) * H;
  const long long per = units / gridDim.x, rem = units % gridDim.x;
  const long long u0 = blockIdx.x * per + min(static_cast<long long>(blockIdx.x), rem);
  const int nu = static_cast<int>(per + (blockIdx.x < rem ? 1 : 0));
  const int li_first = nu > 0 ? static_cast<int>(u0 / H) : 0;
  if (nu > 0) {
    // pass 2: compacted positions; the records of the rows this CTA folds
    const int li_last = static_cast<int>((u0 + nu - 1) / H);
    int base = 0;
    for (int b0 = 0; b0 < a.batch; b0 += kFlushThreads) {
      const int b = b0 + tid;
      const RowFlag f = b < a.batch ? row_flag(a, b, false) : RowFlag{0, 0, 0, 0};
      int tot = 0;
      const int pos = base + block_excl_scan(f.flag, wsum, tot);
      if (f.flag && pos >= li_first && pos <= li_last) {
        const FlushRec rec{b, f.s, c.ring_start[f.s], f.p, c.epoch[f.s] + 1u, {0, 0, 0}};
        rows_s[pos - li_first] = rec;
        // the flush record of the call: by the CTA that folds the row's head 0
        if (static_cast<long long>(pos) * H >= u0) a.recs[pos] = rec;
      }
      base += tot;
    }
  }
  __syncthreads();  // barriers initialised, records in place, this CTA's reads of pnat, ring_start, epoch done
  // The bookkeeping may replace those values once every CTA has read them: the
  // CTA that takes the last ticket writes it (self-resetting ticket), from the
  // flush records, with its consumer warps -- while its producer issues the
  // first copies (the ticket's round trip is off the producer's path).
  if (warp < kConsumerWarps) {
    if (tid == 0) {
      __threadfence();  // this CTA's records are visible before its ticket
      s_last = atomicInc(a.ticket, gridDim.x - 1) == gridDim.x - 1;
    }
    consumer_sync();
    if (s_last) {
      __threadfence();
      if (a.accepted) {
        // every active row's accepted live count (the flagged rows' 0 below);
        // a thread's rows are loaded before any of them is written
        for (int b0 = tid; b0 < a.batch; b0 += 4 * kConsumerThreads) {
          RowFlag f[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int b = b0 + u * kConsumerThreads;
            f[u] = b < a.batch ? row_flag(a, b, false) : RowFlag{0, 0, 0, 0};
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (f[u].book && !f[u].flag) a.pnat[b0 + u * kConsumerThreads] = f[u].p;
        }
        consumer_sync();  // pnat of the flagged rows is read above before it is reset below
      }
      for (int k = tid; k < count; k += kConsumerThreads) {
        const FlushRec rec = a.recs[k];
        c.ring_start[rec.s] = rec.r + rec.p >= L ? rec.r + rec.p - L : rec.r + rec.p;  // (r + p) mod L
        a.pnat[rec.b] = 0;
        c.epoch[rec.s] = rec.epoch;
      }
    }
  }

  if (nu > 0 && warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    // Lane 0 copies S0 (+ scales) -- 2-byte states as two TMA boxes, others
    // with a 1-D bulk copy -- and the live x and B rows (at most two
    // contiguous segments each) with 1-D bulk copies, except for units folded
    // on the tensor cores, whose rows the lanes copy 16 bytes at a time into
    // padded rows.  The lanes copy the live dt' values and A of the head with
    // cp.async.  Nothing here waits for a load it issued.
    int issued = 0;
    bool ok = true;
    // stage index and phase, and the unit's (flushed row, head), advance by
    // increments: no division on the per-unit path
    int st = 0, li = li_first, h = static_cast<int>(u0 % H);
    uint32_t ph = 0;
    for (int i = 0; i < nu; ++i, h = h + 1 == H ? 0 : h + 1, li += h == 0 ? 1 : 0) {
      if (i > 0 && ++st == lay.ns) {
        st = 0;
        ph ^= 1u;
      }
      const FlushRec rec = rows_s[li - li_first];
      if (i >= lay.ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
        break;
      }
      const int s = rec.s, r = rec.r, p = rec.p, g = h / c.hpg;
      uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
      const float* dg = c.dt_cache + static_cast<long long>(s) * c.dt_stride + static_cast<long long>(h) * L;
      const uint16_t* xg = c.x_cache + static_cast<long long>(s) * c.x_stride + static_cast<long long>(h) * L * kDim;
      const uint16_t* bg = c.B_cache + static_cast<long long>(s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
      // units folded on the tensor cores take their x and B rows padded; the rest as stored
      const bool mma_unit = k2B && c.rounding == RSSM_ROUND_NEAREST && p >= kMmaMinP && !c.read_state;
      if (lane == 0) {
        const uint32_t bytes =
            lay.s0_bytes + (k8bit ? 256u : 0u) + (mma_unit ? 0u : static_cast<uint32_t>(p) * (kDim * 2 + kDstate * 2));
        mbar_expect_tx(&full[st], bytes);
        if constexpr (k2B) {
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) tma_load_3d(sb + bx * 8192, &s0map, bx * 64, h * kDim, s, &full[st]);
        } else {
          const uint8_t* st_g = static_cast<const uint8_t*>(c.state) +
                                (static_cast<long long>(s) * c.state_stride + static_cast<long long>(h) * kHeadElems) * esz;
          bulk_g2s(sb, st_g, lay.s0_bytes, &full[st]);
          if (k8bit)
            bulk_g2s(sb + lay.scale_off, c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim, 256,
                     &full[st]);
        }
        if (!mma_unit) {
          const int n1 = min(p, L - r);
          if (n1 > 0) {
            bulk_g2s(sb + lay.x_off, xg + r * kDim, n1 * kDim * 2, &full[st]);
            bulk_g2s(sb + lay.b_off, bg + r * kDstate, n1 * kDstate * 2, &full[st]);
          }
          if (p > n1) {
            bulk_g2s(sb + lay.x_off + n1 * kDim * 2, xg, (p - n1) * kDim * 2, &full[st]);
            bulk_g2s(sb + lay.b_off + n1 * kDstate * 2, bg, (p - n1) * kDstate * 2, &full[st]);
          }
        }
        cp_async4(sb + lay.sc_off, a.A + h);
      }
      if (mma_unit) {
        // live rows into padded shared rows: x 8 and B 16 chunks of 16 bytes per row
        for (int q = lane; q < p * 8; q += 32) {
          const int j = q >> 3, part = q & 7, pos = r + j >= L ? r + j - L : r + j;
          cp_async16(sb + lay.x_off + (j * XS + part * 8) * 2, xg + pos * kDim + part * 8);
        }
        for (int q = lane; q < p * 16; q += 32) {
          const int j = q >> 4, part = q & 15, pos = r + j >= L ? r + j - L : r + j;
          cp_async16(sb + lay.b_off + (j * BS + part * 8) * 2, bg + pos * kDstate + part * 8);
        }
      }
      if (lane < p) cp_async4(sb + lay.dt_off + lane * 4, dg + (r + lane >= L ? r + lane - L : r + lane));
      cp_async_arrive_noinc(&full[st]);
      if (lane == 0) meta[st] = FoldMeta{s, h, p, rec.epoch};
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
      issued = i + 1;
    }
    if (!ok) {
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      // let copies already in flight land before the CTA can exit
      for (int i = max(0, issued - lay.ns); i < issued; ++i) mbar_wait(&full[i % lay.ns], (i / lay.ns) & 1);
    }
  } else if (nu > 0 && warp == kWeightsWarp) {
    // ---------------- weights warp ----------------
    // Per unit, once the stage has landed: the canonical cumulative sums c_j
    // (sequential fp32, the oracle's order) and the weights w_j = e^{c_end -
    // c_j} dt'_j and e^{c_end}, into the stage for all consumer warps (one warp
    // forms them instead of each of the eight).  The stage is not refilled
    // before the consumers release it, and they read the weights first.
    int st = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nu; ++i) {
      if (i > 0 && ++st == lay.ns) {
        st = 0;
        ph ^= 1u;
      }
      if (!mbar_wait(&full[st], ph)) {
        if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
        break;
      }
      uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
      const int p = meta[st].p;
      const float hA = reinterpret_cast<const float*>(sb + lay.sc_off)[0];
      const float dtj = lane < p ? reinterpret_cast<const float*>(sb + lay.dt_off)[lane] : 0.0f;
      const float aj = lane < p ? __fmul_rn(hA, dtj) : 0.0f;
      float cj = 0.0f;
#pragma unroll 4
      for (int k = 0; k < p; ++k) {
        const float ak = __shfl_sync(0xffffffffu, aj, k);
        if (lane >= k) cj = __fadd_rn(cj, ak);
      }
      const float c_end = p > 0 ? __shfl_sync(0xffffffffu, cj, p - 1) : 0.0f;
      float* wsm = reinterpret_cast<float*>(sb + lay.w_off);
      wsm[lane] = lane < p ? __fmul_rn(spec_exp(__fsub_rn(c_end, cj)), dtj) : 0.0f;
      if (lane == 0) wsm[32] = spec_exp(c_end);
      __syncwarp();
      if (lane == 0) mbar_arrive(&wready[st]);
    }
  } else if (nu > 0) {
  // ---------------- consumer warps: rows 8*warp .. 8*warp+7, each on its own ----------------
  // lane: rows r0..r0+3, columns c0..c0+7
  const int r0 = 8 * warp + 4 * (lane >> 4), c0 = 8 * (lane & 15);
  int st = 0;
  uint32_t ph = 0;
  for (int i = 0; i < nu; ++i) {
    if (i > 0 && ++st == lay.ns) {
      st = 0;
      ph ^= 1u;
    }
    // the stage's copies (observed directly: complete by the time the weights
    // are) and its weights
    if (!mbar_wait(&full[st], ph) || !mbar_wait(&wready[st], ph)) {
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      break;
    }
    const uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
    const FoldMeta m = meta[st];
    const int p = m.p;
    // the weights w_j = e^{c_end - c_j} dt'_j (lane j holds w_j) and
    // decay = e^{c_end}, formed by the weights warp
    const float* wsm = reinterpret_cast<const float*>(sb + lay.w_off);
    const float wj = wsm[lane];
    const float decay = wsm[32];
    if constexpr (k2B) {
      if (c.rounding == RSSM_ROUND_NEAREST && p >= kMmaMinP && !c.read_state) {
        // The fold on the tensor cores: S0' = e^{c_end} S0 + U Bm, U[d][j] =
        // w_j x_j[d] (64 x p), Bm[j][n] = B_j[n] (p x 128), as mma.sync
        // m16n8k16 with fp32 accumulation starting from e^{c_end} S0; U is
        // split into three bf16 parts hi + mid + lo (each the rounded
        // remainder of the previous: 24 significant bits, so U is carried to
        // fp32 precision), B is exact in bf16.  Only the summation order
        // differs from the canonical fp32 chain, which 8-bit and
        // stochastically rounded states need bit for bit.
        // Warp: rows mr..mr+15, columns nb..nb+63 (8 tiles of 8).
        const int g = lane >> 2, cq = lane & 3, mi = lane >> 3, rr = lane & 7;
        const int mr = 16 * (warp & 3), nb = 64 * (warp >> 2);
        const uint32_t sbase = smem_addr(sb);
        float D[8][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          // S0 fragments from the swizzled boxes: matrices (rows mr, mr + 8) x (columns n, n + 8)
          const int d = mr + 8 * (mi & 1) + rr, n = nb + 16 * t + 8 * (mi >> 1);
          uint32_t sv[4];
          ldmatrix_x4(sv, sbase + swizzled_offset<2>(d, n));
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float2 v;
            if constexpr (DT == RSSM_BF16)
              v = make_float2(bf16lo(sv[q]), bf16hi(sv[q]));
            else
              v = h2f2(sv[q]);
            float* dd = &D[2 * t + (q >> 1)][2 * (q & 1)];
            dd[0] = __fmul_rn(decay, v.x);
            dd[1] = __fmul_rn(decay, v.y);
          }
        }
        const uint16_t* xs = reinterpret_cast<const uint16_t*>(sb + lay.x_off);
        const uint32_t bsa = sbase + lay.b_off;
        for (int kb = 0; kb < p; kb += 16) {
          // A fragments: rows mr + g, mr + g + 8; tokens kb + 2cq (+1), kb + 2cq + 8 (+1)
          uint32_t ahi[4], amid[4], alo[4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int rw = 0; rw < 2; ++rw) {  // A rows mr + g (rw = 0) and mr + g + 8
              float u[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int j = kb + 2 * cq + 8 * hh + e;
                const float w = __shfl_sync(0xffffffffu, wj, j & 31);
                u[e] = j < p ? __fmul_rn(w, __uint_as_float(static_cast<uint32_t>(xs[j * XS + mr + g + 8 * rw]) << 16))
                             : 0.0f;
              }
              // u = hi + mid + lo: each part the bf16 rounding of what the
              // previous parts leave (the remainders are exact in fp32)
              const uint32_t hi = bf16x2_rn(u[0], u[1]);
              const float r0 = __fsub_rn(u[0], bf16lo(hi)), r1 = __fsub_rn(u[1], bf16hi(hi));
              const uint32_t mid = bf16x2_rn(r0, r1);
              ahi[2 * hh + rw] = hi;
              amid[2 * hh + rw] = mid;
              alo[2 * hh + rw] = bf16x2_rn(__fsub_rn(r0, bf16lo(mid)), __fsub_rn(r1, bf16hi(mid)));
            }
          }
          // B fragments, two column tiles per ldmatrix: matrices (tokens kb, kb + 8)
          // x (columns n, n + 8); token rows past p read row 0 (their U is 0)
          const int kr = kb + 8 * (mi & 1) + rr;
          const uint32_t rowa = bsa + static_cast<uint32_t>((kr < p ? kr : 0) * BS + 8 * (mi >> 1)) * 2;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint32_t bv[4];
            ldmatrix_x4_trans(bv, rowa + static_cast<uint32_t>(nb + 16 * t) * 2);
            mma16816_bf16(D[2 * t], ahi, bv[0], bv[1]);
            mma16816_bf16(D[2 * t], amid, bv[0], bv[1]);
            mma16816_bf16(D[2 * t], alo, bv[0], bv[1]);
            mma16816_bf16(D[2 * t + 1], ahi, bv[2], bv[3]);
            mma16816_bf16(D[2 * t + 1], amid, bv[2], bv[3]);
            mma16816_bf16(D[2 * t + 1], alo, bv[2], bv[3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
        uint16_t* hs = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(c.state) +
                                                   (static_cast<long long>(m.s) * c.state_stride +
                                                    static_cast<long long>(m.h) * kHeadElems) * esz);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int n = nb + 8 * nt + 2 * cq;
          *reinterpret_cast<uint32_t*>(hs + (mr + g) * kDstate + n) =
              DT == RSSM_BF16 ? cvt_bf16x2_sat(D[nt][0], D[nt][1]) : cvt_f16x2_sat(D[nt][0], D[nt][1]);
          *reinterpret_cast<uint32_t*>(hs + (mr + g + 8) * kDstate + n) =
              DT == RSSM_BF16 ? cvt_bf16x2_sat(D[nt][2], D[nt][3]) : cvt_f16x2_sat(D[nt][2], D[nt][3]);
        }
        continue;
      }
    }
    // acc = e^{c_end} * S0f
    float2 acc[4][4];
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      const int row = r0 + i4;
      float v[8];
      if constexpr (DT == RSSM_F32) {
        const float4* p4 = reinterpret_cast<const float4*>(sb + (row * kDstate + c0) * 4);
        const float4 x0 = p4[0], x1 = p4[1];
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
      } else if constexpr (DT == RSSM_BF16) {
        const uint4 q = *reinterpret_cast<const uint4*>(sb + swizzled_offset<2>(row, c0));
        v[0] = bf16lo(q.x); v[1] = bf16hi(q.x); v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
        v[4] = bf16lo(q.z); v[5] = bf16hi(q.z); v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
      } else if constexpr (DT == RSSM_F16) {
        const uint4 q = *reinterpret_cast<const uint4*>(sb + swizzled_offset<2>(row, c0));
        float2 t0 = h2f2(q.x), t1 = h2f2(q.y), t2 = h2f2(q.z), t3 = h2f2(q.w);
        v[0] = t0.x; v[1] = t0.y; v[2] = t1.x; v[3] = t1.y; v[4] = t2.x; v[5] = t2.y; v[6] = t3.x; v[7] = t3.y;
      } else {
        const uint2 q = *reinterpret_cast<const uint2*>(sb + row * kDstate + c0);
        const float sc = reinterpret_cast<const float*>(sb + lay.scale_off)[row];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t w = e < 4 ? q.x : q.y;
          float code;
          if constexpr (DT == RSSM_I8) {
            // code q as fp32 without a conversion instruction:
            // (2^23 + (q + 128)) - (2^23 + 128), every step exact
            const uint32_t bits = __byte_perm(w ^ 0x80808080u, 0x4B000000u, 0x7540u | (e & 3));
            code = __fsub_rn(__uint_as_float(bits), 8388736.0f);
          } else {
            code = e4m3_to_f32(static_cast<uint8_t>((w >> (8 * (e & 3))) & 0xffu));
          }
          v[e] = __fmul_rn(code, sc);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        acc[i4][q] = make_float2(__fmul_rn(decay, v[2 * q]), __fmul_rn(decay, v[2 * q + 1]));
    }
    // acc[d][n] = fma(u_j[d], B_j[n], acc), j ascending, u_j[d] = w_j x_j[d]
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(sb + lay.x_off);
    const uint16_t* bs = reinterpret_cast<const uint16_t*>(sb + lay.b_off);
#pragma unroll 4
    for (int j = 0; j < p; ++j) {
      const float w = __shfl_sync(0xffffffffu, wj, j);
      const uint2 xw = *reinterpret_cast<const uint2*>(xs + j * kDim + r0);
      const float u0v = __fmul_rn(w, bf16lo(xw.x)), u1v = __fmul_rn(w, bf16hi(xw.x));
      const float u2v = __fmul_rn(w, bf16lo(xw.y)), u3v = __fmul_rn(w, bf16hi(xw.y));
      const uint4 bw = *reinterpret_cast<const uint4*>(bs + j * kDstate + c0);
      const float2 bb[4] = {make_float2(bf16lo(bw.x), bf16hi(bw.x)), make_float2(bf16lo(bw.y), bf16hi(bw.y)),
                            make_float2(bf16lo(bw.z), bf16hi(bw.z)), make_float2(bf16lo(bw.w), bf16hi(bw.w))};
      const float2 uu[4] = {make_float2(u0v, u0v), make_float2(u1v, u1v), make_float2(u2v, u2v), make_float2(u3v, u3v)};
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i4][q] = __ffma2_rn(uu[i4], bb[q], acc[i4][q]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
    float accf[4][8];
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        accf[i4][2 * q] = acc[i4][q].x;
        accf[i4][2 * q + 1] = acc[i4][q].y;
      }
    void* head_state = static_cast<uint8_t*>(c.state) +
                       (static_cast<long long>(m.s) * c.state_stride + static_cast<long long>(m.h) * kHeadElems) * esz;
    float* head_scale = k8bit ? c.scale + static_cast<long long>(m.s) * c.scale_stride + m.h * kDim : nullptr;
    quantize_store<DT>(accf, r0, c0, lane, head_state, head_scale, c.rounding, static_cast<uint32_t>(m.h),
                       static_cast<uint32_t>(m.s), m.epoch, a.seed);
    if (c.read_state) store_read_checkpoint(c, accf, r0, c0, lane, m.s, m.h);
  }
  }

}

// ---------------------------------------------------------------------------
// init: quantise FP32 prefill states, clear rings
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kConsumerThreads) init_quant_kernel(InitArgs a) {
  const Cache& c = a.c;
  const int i = blockIdx.x, h = blockIdx.y;
  const int s = a.ids[i];
  if (s < 1 || s >= c.S) return;
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r0 = 8 * warp + 4 * (lane >> 4), c0 = 8 * (lane & 15);
  const float* src = a.states + (static_cast<long long>(i) * c.H + h) * kHeadElems;
  float acc[4][8];
#pragma unroll
  for (int i4 = 0; i4 < 4; ++i4) {
    const float4* p4 = reinterpret_cast<const float4*>(src + (r0 + i4) * kDstate + c0);
    const float4 x0 = p4[0], x1 = p4[1];
    acc[i4][0] = x0.x; acc[i4][1] = x0.y; acc[i4][2] = x0.z; acc[i4][3] = x0.w;
    acc[i4][4] = x1.x; acc[i4][5] = x1.y; acc[i4][6] = x1.z; acc[i4][7] = x1.w;
  }
  void* head_state = static_cast<uint8_t*>(c.state) +
                     (static_cast<long long>(s) * c.state_stride + static_cast<long long>(h) * kHeadElems) * esz;
  float* head_scale =
      (DT == RSSM_I8 || DT == RSSM_E4M3) ? c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim : nullptr;
  quantize_store<DT>(acc, r0, c0, lane, head_state, head_scale, c.rounding, static_cast<uint32_t>(h),
                     static_cast<uint32_t>(s), 0u, a.seed);
  if (c.read_state) store_read_checkpoint(c, acc, r0, c0, lane, s, h);
}

// NVFP4 read checkpoint: each initialised slot's global scale = the largest
// magnitude of its FP32 prefill state (all heads) / (6 * 448), 1 for a zero
// state.  Three steps: zero the slot's word; per (state, head) the head's
// largest magnitude merged by an integer atomic max on the float's bits (the
// bit patterns of non-negative floats order like their values); the scale.
__global__ void __launch_bounds__(64) init_gs_zero_kernel(InitArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.n) return;
  const int s = a.ids[i];
  if (s >= 1 && s < a.c.S) a.c.read_gs[s] = 0.0f;
}
__global__ void __launch_bounds__(256) init_gs_max_kernel(InitArgs a) {
  const int i = blockIdx.x, h = blockIdx.y;
  const int s = a.ids[i];
  if (s < 1 || s >= a.c.S) return;
  const float4* src = reinterpret_cast<const float4*>(a.states + (static_cast<long long>(i) * a.c.H + h) * kHeadElems);
  float m = 0.0f;
  for (int k = threadIdx.x; k < kHeadElems / 4; k += blockDim.x) {
    const float4 v = src[k];
    m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned*>(a.c.read_gs + s), __float_as_uint(m));
}
__global__ void __launch_bounds__(64) init_gs_scale_kernel(InitArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.n) return;
  const int s = a.ids[i];
  if (s < 1 || s >= a.c.S) return;
  const float m = a.c.read_gs[s];
  a.c.read_gs[s] = m > 0.0f ? __fdiv_rn(m, 2688.0f) : 1.0f;
}

__global__ void __launch_bounds__(256) init_clear_kernel(InitArgs a) {
  const Cache& c = a.c;
  const int s = a.ids[blockIdx.x];
  if (s < 1 || s >= c.S) return;
  const int tid = threadIdx.x + blockIdx.y * blockDim.x, nth = blockDim.x * gridDim.y;
  uint4* xr = reinterpret_cast<uint4*>(c.x_cache + static_cast<long long>(s) * c.x_stride);
  const int nx = c.H * c.L * kDim * 2 / 16;
  for (int k = tid; k < nx; k += nth) xr[k] = make_uint4(0, 0, 0, 0);
  uint4* br = reinterpret_cast<uint4*>(c.B_cache + static_cast<long long>(s) * c.B_stride);
  const int nb = c.G * c.L * kDstate * 2 / 16;
  for (int k = tid; k < nb; k += nth) br[k] = make_uint4(0, 0, 0, 0);
  float* dr = c.dt_cache + static_cast<long long>(s) * c.dt_stride;
  for (int k = tid; k < c.H * c.L; k += nth) dr[k] = 0.0f;
  if (tid == 0) {
    c.ring_start[s] = 0;
    c.epoch[s] = 0u;
  }
}

// ---------------------------------------------------------------------------
// accept: pnat += accepted
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) accept_kernel(Cache c, const int* slot_idx, int* pnat, const int* accepted,
                                                     const int* cu, int batch, int T) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (b >= batch) return;
  // the row's loads are independent: issue them together (one round trip)
  const int s = slot_idx[b];
  const int Tb = cu ? cu[b + 1] - cu[b] : T;
  const int acc = accepted[b];
  const int p = pnat[b];
  if (s < 1 || s >= c.S) return;
  if (Tb < 0 || Tb > T) {
    set_error(c.err, RSSM_ERRBIT_SEQLEN);
    return;
  }
  if (acc < 0 || acc > Tb) {
    set_error(c.err, RSSM_ERRBIT_ACCEPT);
    return;
  }
  if (p < 0 || p + acc > c.L) {
    set_error(c.err, RSSM_ERRBIT_PNAT);
    return;
  }
  pnat[b] = p + acc;
}

__global__ void spec_math_kernel(const float* in, float* oexp, float* osp, long long n) {
  for (long long k = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; k < n;
       k += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float v = in[k];
    if (oexp) oexp[k] = spec_exp(v);
    if (osp) osp[k] = spec_softplus(v);
  }
}

// ---------------------------------------------------------------------------
// self-test of the bounded mbarrier wait: one warp.  Barrier `lost` is told to
// expect 256 bytes of transactions that no copy will bring (the state a stage
// barrier is in when a copy it counts on never lands); its wait runs out after
// `tries` tests and the kernel sets RSSM_ERRBIT_TIMEOUT, as the pipeline
// kernels do.  Barrier `real` counts one genuine 256-byte bulk copy, waited
// for in full, so no copy is in flight when the kernel returns.
// ---------------------------------------------------------------------------
__device__ __align__(16) unsigned char g_wait_probe_src[256];

__global__ void wait_timeout_kernel(unsigned* err, unsigned tries) {
  __shared__ __align__(16) unsigned char buf[256];
  __shared__ __align__(8) uint64_t bars[2];
  uint64_t* lost = &bars[0];
  uint64_t* real = &bars[1];
  if (threadIdx.x == 0) {
    mbar_init(lost, 1);
    mbar_init(real, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  mbar_arrive_expect_tx(lost, 256u);  // nothing will ever complete these bytes
  mbar_arrive_expect_tx(real, 256u);
  bulk_g2s(buf, g_wait_probe_src, 256u, real);
  const bool lost_ok = mbar_wait(lost, 0u, tries);
  const bool real_ok = mbar_wait(real, 0u);  // the genuine copy has landed
  if (!lost_ok || !real_ok) set_error(err, RSSM_ERRBIT_TIMEOUT);
}

int launch_wait_timeout(unsigned* err, unsigned tries, void* stream) {
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, tries);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
template <int DT>
static int launch_flush_t(const FlushArgs& a, int num_sms, cudaStream_t st) {
  // a fixed grid of two CTAs per SM (the number of flushed rows is only known
  // on the device); the rows table holds the most rows one CTA's units span
  const int grid = 2 * num_sms;
  const long long nu_max = (static_cast<long long>(a.batch) * a.c.H + grid - 1) / grid;
  const int maxrows = static_cast<int>(nu_max / a.c.H) + 2;
  int ns = 6;  // as many stages (3..6) as fit 113 KB
  while (ns > 2 && fold_layout(DT, a.c.L, ns, maxrows).total > 113 * 1024) --ns;
  const FoldLayout lay = fold_layout(DT, a.c.L, ns, maxrows);
  if (lay.total > 225 * 1024) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(flush_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(flush_kernel<DT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // 2-byte states: S0 by TMA boxes through the readout's tensor map (unused otherwise)
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (fold_2byte(DT) && !encode_state_map(a.c, &map, 1)) return cudaErrorInvalidValue;
  e = launch_pdl(flush_kernel<DT>, dim3(grid), dim3(kFlushThreads), lay.total, st, map, a, ns, maxrows);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int launch_flush(const FlushArgs& a, int num_sms, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (a.c.dtype) {
    case RSSM_F32: return launch_flush_t<RSSM_F32>(a, num_sms, st);
    case RSSM_BF16: return launch_flush_t<RSSM_BF16>(a, num_sms, st);
    case RSSM_F16: return launch_flush_t<RSSM_F16>(a, num_sms, st);
    case RSSM_I8: return launch_flush_t<RSSM_I8>(a, num_sms, st);
    default: return launch_flush_t<RSSM_E4M3>(a, num_sms, st);
  }
}

int launch_init(const InitArgs& a, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 grid(a.n, a.c.H);
  if (a.c.read_state && a.c.read_dtype == RSSM_NVFP4) {  // the slots' global scales first
    const int nb = (a.n + 63) / 64;
    init_gs_zero_kernel<<<nb, 64, 0, st>>>(a);
    init_gs_max_kernel<<<grid, 256, 0, st>>>(a);
    init_gs_scale_kernel<<<nb, 64, 0, st>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  switch (a.c.dtype) {
    case RSSM_F32: init_quant_kernel<RSSM_F32><<<grid, kConsumerThreads, 0, st>>>(a); break;
    case RSSM_BF16: init_quant_kernel<RSSM_BF16><<<grid, kConsumerThreads, 0, st>>>(a); break;
    case RSSM_F16: init_quant_kernel<RSSM_F16><<<grid, kConsumerThreads, 0, st>>>(a); break;
    case RSSM_I8: init_quant_kernel<RSSM_I8><<<grid, kConsumerThreads, 0, st>>>(a); break;
    default: init_quant_kernel<RSSM_E4M3><<<grid, kConsumerThreads, 0, st>>>(a); break;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  init_clear_kernel<<<dim3(a.n, 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

int launch_accept(const Cache& c, const int* slot_idx, int* pnat, const int* accepted, const int* cu, int batch,
                  int T, void* stream) {
  cudaError_t e = launch_pdl(accept_kernel, dim3((batch + 255) / 256), dim3(256), 0, static_cast<cudaStream_t>(stream),
                             c, slot_idx, pnat, accepted, cu, batch, T);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int launch_spec_math(const float* in, float* oexp, float* osp, long long n, void* stream) {
  const long long blocks = (n + 255) / 256;
  spec_math_kernel<<<static_cast<int>(blocks < 4096 ? blocks : 4096), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      in, oexp, osp, n);
  return cudaGetLastError();
}

}  // namespace rssm
