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
//   mod L, pnat = 0, epoch += 1) while the folds run.
#include <cuda_runtime.h>

#include "rssm_device.cuh"

namespace rssm {

// ---------------------------------------------------------------------------
// classification
// ---------------------------------------------------------------------------
struct RowFlag {
  int flag, s, p;
};

// a row's flush decision: active rows with p + T_b > max_window (all active
// rows under force); rows failing a check set an error bit (when `errors`)
__device__ __forceinline__ RowFlag row_flag(const FlushArgs& a, int b, bool errors) {
  const Cache& c = a.c;
  RowFlag f = {0, 0, 0};
  // the row's loads are independent: issue them together (one round trip)
  const int s = a.slot_idx[b];
  const int p = a.pnat[b];
  const int Tb = a.cu ? a.cu[b + 1] - a.cu[b] : a.T;
  if (s >= 1 && s < c.S) {
    if (Tb < 0 || Tb > a.T) {
      if (errors) set_error(c.err, RSSM_ERRBIT_SEQLEN);
    } else if (p < 0 || p > c.L) {
      if (errors) set_error(c.err, RSSM_ERRBIT_PNAT);
    } else if (a.force || p + Tb > c.W) {
      f = RowFlag{1, s, p};
    }
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
// fold kernel
// ---------------------------------------------------------------------------
struct FoldMeta {
  int s, h, p;
  unsigned epoch;
};

struct FoldLayout {
  int ns, KB;
  uint32_t s0_bytes, scale_off, x_off, b_off, dt_off, sc_off, stage_bytes;
  uint32_t meta_off, rows_off, stages_off, total;
};

// barriers | per-stage metadata | the records of the flushed rows this CTA
// folds (up to `maxrows`) | stages; one stage: S0 (as stored) | 8-bit scales |
// live x rows | live B rows | live dt' | A of the head
__host__ __device__ inline FoldLayout fold_layout(int dtype, int L, int ns, int maxrows) {
  FoldLayout f;
  f.ns = ns;
  f.KB = (L + 3) & ~3;
  const int esz = dtype == RSSM_F32 ? 4 : (dtype == RSSM_BF16 || dtype == RSSM_F16) ? 2 : 1;
  f.s0_bytes = kHeadElems * esz;
  uint32_t o = f.s0_bytes;
  f.scale_off = o;
  if (dtype == RSSM_I8 || dtype == RSSM_E4M3) o += 256;
  f.x_off = o;
  o += f.KB * kDim * 2;
  f.b_off = o;
  o += f.KB * kDstate * 2;
  f.dt_off = o;
  o += f.KB * 4;
  f.sc_off = o;
  o += 16;
  f.stage_bytes = (o + 127) & ~127u;
  f.meta_off = 256;  // after the barriers
  f.rows_off = 512;
  f.stages_off = (f.rows_off + maxrows * static_cast<uint32_t>(sizeof(FlushRec)) + 127) & ~127u;
  f.total = f.stages_off + f.ns * f.stage_bytes;
  return f;
}

// Classification, fold, requantisation and bookkeeping of rssm_flush in one
// kernel.  Every CTA classifies all rows (two passes over slot_idx, pnat and
// the sequence bounds) and keeps the records of the flushed rows its range of
// (flushed row, head) units covers; the producer and consumer warps then fold
// those units.  The bookkeeping is written by the CTA that takes the last ticket
// once it has classified (a self-resetting ticket), i.e. after every CTA has
// read the values it replaces; nothing in the kernel reads them afterwards.
template <int DT>
__global__ void __launch_bounds__(kThreads, 2) flush_kernel(FlushArgs a, int ns, int maxrows) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int wsum[kThreads / 32];
  __shared__ int s_last;
  const Cache& c = a.c;
  const FoldLayout lay = fold_layout(DT, c.L, ns, maxrows);
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  const int L = c.L, H = c.H;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 8;
  FoldMeta* meta = reinterpret_cast<FoldMeta*>(smem + lay.meta_off);
  FlushRec* rows_s = reinterpret_cast<FlushRec*>(smem + lay.rows_off);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < lay.ns; ++st) {
      mbar_init(&full[st], 1 + 32);  // producer lane 0 + one cp.async arrival per producer lane
      mbar_init(&empty[st], kConsumerWarps);
    }
    fence_barrier_init();
  }
  pdl_wait();  // pnat as the previous call left it
  pdl_trigger();
  // pass 1: the number of flushed rows (CTA 0 reports bad rows); the flagged
  // rows' ring start and epoch are prefetched for pass 2
  int count = 0;
  for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
    const int b = b0 + tid;
    const RowFlag f = b < a.batch ? row_flag(a, b, blockIdx.x == 0) : RowFlag{0, 0, 0};
    if (f.flag) {
      asm volatile("prefetch.global.L1 [%0];" ::"l"(c.ring_start + f.s));
      asm volatile("prefetch.global.L1 [%0];" ::"l"(c.epoch + f.s));
    }
    count += __syncthreads_count(f.flag);
  }
  if (count == 0) {  // nothing to fold or book (every CTA sees the same count)
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
    for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
      const int b = b0 + tid;
      const RowFlag f = b < a.batch ? row_flag(a, b, false) : RowFlag{0, 0, 0};
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
  // flush records, while its producer issues the first copies.
  if (tid == 0) {
    __threadfence();  // this CTA's records are visible before its ticket
    s_last = atomicInc(a.ticket, gridDim.x - 1) == gridDim.x - 1;
  }
  __syncthreads();
  if (s_last && tid < kConsumerThreads) {
    __threadfence();
    for (int k = tid; k < count; k += kConsumerThreads) {
      const FlushRec rec = a.recs[k];
      c.ring_start[rec.s] = rec.r + rec.p >= L ? rec.r + rec.p - L : rec.r + rec.p;  // (r + p) mod L
      a.pnat[rec.b] = 0;
      c.epoch[rec.s] = rec.epoch;
    }
  }

  if (nu > 0 && warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    // Lane 0 copies S0 (+ scales) and the live x and B rows (at most two
    // contiguous segments each) with 1-D bulk copies; the lanes copy the live
    // dt' values and A of the head with cp.async.  Nothing here waits for a
    // load it issued: the next unit's flagged-row record is loaded a unit ahead.
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
      if (lane == 0) {
        const uint32_t bytes = lay.s0_bytes + (k8bit ? 256u : 0u) + static_cast<uint32_t>(p) * (kDim * 2 + kDstate * 2);
        mbar_expect_tx(&full[st], bytes);
        const uint8_t* st_g = static_cast<const uint8_t*>(c.state) +
                              (static_cast<long long>(s) * c.state_stride + static_cast<long long>(h) * kHeadElems) * esz;
        bulk_g2s(sb, st_g, lay.s0_bytes, &full[st]);
        if (k8bit) bulk_g2s(sb + lay.scale_off, c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim, 256,
                            &full[st]);
        const uint16_t* xg = c.x_cache + static_cast<long long>(s) * c.x_stride + static_cast<long long>(h) * L * kDim;
        const uint16_t* bg = c.B_cache + static_cast<long long>(s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
        const int n1 = min(p, L - r);
        if (n1 > 0) {
          bulk_g2s(sb + lay.x_off, xg + r * kDim, n1 * kDim * 2, &full[st]);
          bulk_g2s(sb + lay.b_off, bg + r * kDstate, n1 * kDstate * 2, &full[st]);
        }
        if (p > n1) {
          bulk_g2s(sb + lay.x_off + n1 * kDim * 2, xg, (p - n1) * kDim * 2, &full[st]);
          bulk_g2s(sb + lay.b_off + n1 * kDstate * 2, bg, (p - n1) * kDstate * 2, &full[st]);
        }
        cp_async4(sb + lay.sc_off, a.A + h);
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
    if (!mbar_wait(&full[st], ph)) {
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      break;
    }
    const uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
    const FoldMeta m = meta[st];
    const int p = m.p;
    // canonical cumulative sums c_j (sequential fp32) and the weights
    // w_j = e^{c_end - c_j} dt'_j (lane j holds w_j), decay = e^{c_end}
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
    const float wj = lane < p ? __fmul_rn(spec_exp(__fsub_rn(c_end, cj)), dtj) : 0.0f;
    const float decay = spec_exp(c_end);
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
        const uint4 q = *reinterpret_cast<const uint4*>(sb + (row * kDstate + c0) * 2);
        v[0] = bf16lo(q.x); v[1] = bf16hi(q.x); v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
        v[4] = bf16lo(q.z); v[5] = bf16hi(q.z); v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
      } else if constexpr (DT == RSSM_F16) {
        const uint4 q = *reinterpret_cast<const uint4*>(sb + (row * kDstate + c0) * 2);
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
  e = launch_pdl(flush_kernel<DT>, dim3(grid), dim3(kThreads), lay.total, st, a, ns, maxrows);
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
