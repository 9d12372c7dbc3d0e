// rssm_step.cu -- replay/readout of the ReplaySSM checkpointing SSU.
//
// Two kernels, the split of FlashInfer PR #3975 (Description item 1):
//   precompute_kernel  one CTA per (row, group): dt' = softplus(dt + dt_bias)
//       for the new tokens (appended to the dt ring), the cumulative sums
//       c_k = sum_{i<=k} A dt'_i over live ring + new tokens (recomputed, not
//       cached: Description item 2), the C.B contraction CB[t][k] = C_t . B_k
//       once per group, and per head the replay coefficients
//           coef[k][t] = e^{c_{p+t} - c_k} dt'_k CB[t][k]  (+ D on k = p+t)
//       which it applies at once to the head's x rows:
//           R[t][d] = sum_k coef[k][t] x_k[d],   decay[t] = e^{c_{p+t}}
//       written to scratch (the row's T_b rows) with the C rows (in the
//       readout's MMA type).  Appends B, x and dt'.
//   readout_kernel  persistent, one (row, head) unit at a time:
//           y_t[d] = decay[t] (S0[d] . C_t) + R[t][d]
//       streaming S0 once through a multi-stage shared-memory ring filled by
//       TMA (swizzled tensor boxes for S0, 1-D bulk copies for the rest) from
//       a producer warp with mbarriers; 8 consumer warps contract on the
//       tensor cores (mma.sync m16n8k16, f32 accumulation).
#include "rssm_readout.cuh"

namespace rssm {

// ---------------------------------------------------------------------------
// precompute
// ---------------------------------------------------------------------------
// The precompute's inputs all come in through shared memory in one round of
// asynchronous copies, issued as soon as the row's ring start is known; the
// kernel is a short chain of dependent steps per CTA (every CTA of a step fits
// in one wave), so its time is the latency of that chain.  Dynamic shared
// memory, one (row, group):
//   xs [hcm][L][64]        bf16  x rows of a chunk of hcm = min(hpg, 16) of
//                                the group's heads by logical token k (live
//                                ring rows, then new)
//   bs [L][128]            bf16  B rows by logical token k
//   cs [8][128]            bf16  C rows of the new tokens
constexpr int kHeadChunk = 16;
__host__ __device__ inline int head_chunk(int hpg) { return hpg < kHeadChunk ? hpg : kHeadChunk; }
inline size_t precompute_smem(int hpg, int L) {
  return static_cast<size_t>(head_chunk(hpg)) * L * kDim * 2 + static_cast<size_t>(L) * kDstate * 2 + 8 * kDstate * 2;
}


template <int TP>
__global__ void __launch_bounds__(256, TP == 4 ? 4 : 3) precompute_kernel(StepArgs a) {
  extern __shared__ __align__(16) unsigned char psm[];
  __shared__ float CB[TP][kMaxL];
  __shared__ float dts[kHeadChunk][kMaxL];  // dt' of the live tokens; dt of the new ones (before bias, softplus)
  __shared__ float hp[3][kHeadChunk];       // A, D, dt_bias of the chunk's heads
  __shared__ __align__(16) float cfs[8][kMaxL][TP];  // per warp: coef[k][t] of its current head
  __shared__ int meta[7];
  __shared__ __align__(8) uint64_t pbar;  // completion of the chunk's bulk row copies
  const Cache& c = a.c;
  const int b = blockIdx.x / c.G, g = blockIdx.x % c.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = c.L, H = c.H, G = c.G, hpg = c.hpg;
  uint16_t* xs = reinterpret_cast<uint16_t*>(psm);
  uint16_t* bs = xs + head_chunk(hpg) * L * kDim;
  uint16_t* cs = bs + L * kDstate;
  if (tid == 0) {
    mbar_init(&pbar, 1);
    fence_barrier_init();
  }
  pdl_wait();  // the flush's bookkeeping and checkpoints are complete from here on
  pdl_trigger();
  if (warp == 0) {
    // the row's scalars in one round trip, then its ring start
    int v = 0;
    if (lane == 0) v = a.slot_idx[b];
    else if (lane == 1) v = a.pnat[b];
    else if (lane == 2) v = a.cu ? a.cu[b] : b * a.T;
    else if (lane == 3) v = a.cu ? a.cu[b + 1] : (b + 1) * a.T;
    const int s = __shfl_sync(0xffffffffu, v, 0), pn = __shfl_sync(0xffffffffu, v, 1);
    const int tok0 = __shfl_sync(0xffffffffu, v, 2), tok1 = __shfl_sync(0xffffffffu, v, 3);
    if (lane == 0) {
      int Tb = tok1 - tok0, flags = 0, p = 0, r = 0;
      unsigned ep = 0u;
      float gs = 1.0f;
      const bool tb_ok = Tb >= 0 && Tb <= a.T;
      if (s >= 1 && s < c.S) {
        if (!tb_ok) {
          if (g == 0) set_error(c.err, RSSM_ERRBIT_SEQLEN);
        } else if (pn < 0 || pn + Tb > L) {
          if (g == 0) set_error(c.err, RSSM_ERRBIT_PNAT);
        } else {
          p = pn;
          r = c.ring_start[s];
          if (c.dtype == RSSM_NVFP4) gs = c.read_gs[s];
          flags = 1;
          // the one-call path: the flush decision (the flush's rule); the row's
          // outputs still replay its whole live prefix from the old checkpoint
          // and the readout folds that prefix into the new one
          if (a.flush_mode && (a.flush_mode == 2 || pn + Tb > c.W)) {
            flags |= 2;
            ep = c.epoch[s] + 1u;
          }
        }
      }
      if (!tb_ok) Tb = 0;
      meta[0] = s; meta[1] = r; meta[2] = p; meta[3] = Tb; meta[4] = tok0; meta[5] = flags & 1; meta[6] = flags & 2;
      if (g == 0) a.rows[b] = RowRec{s, r, p, Tb, tok0, flags, ep, gs};
      if (blockIdx.x == 0) *a.rwork = 0u;  // the readout's chunk counter
    }
  }
  __syncthreads();
  const int s = meta[0], r = meta[1], p = meta[2], Tb = meta[3], tok0 = meta[4];
  const bool fold = meta[6] != 0;
  if (!meta[5] || (Tb == 0 && !fold)) return;
  const int K = p + Tb;  // logical tokens: p live ring rows, then the Tb new ones
  auto ring = [&](int k) {  // ring slot of logical token k < L
    const int q = r + k;
    return q >= L ? q - L : q;
  };
  uint16_t* bring = c.B_cache + static_cast<long long>(s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
  uint16_t* xslot = c.x_cache + static_cast<long long>(s) * c.x_stride;
  float* dslot = c.dt_cache + static_cast<long long>(s) * c.dt_stride;
  const int n1 = p < L - r ? p : L - r;  // live tokens before the ring wraps
  const bool c_f16 = c.dtype == RSSM_F16 || c.dtype == RSSM_I8 || c.dtype == RSSM_E4M3 || c.dtype == RSSM_NVFP4;
  for (int h0 = 0, ph = 0; h0 < hpg; h0 += kHeadChunk, ph ^= 1) {
    const int hc = hpg - h0 < kHeadChunk ? hpg - h0 : kHeadChunk, hb = g * hpg + h0;
    if (h0) __syncthreads();  // every warp is done with the previous chunk's rows
    // the rows by 1-D bulk copies, counted on pbar: lane hh < hc of warp 0 the
    // x rows of head hb + hh (the live prefix: at most two ring segments; then
    // the new rows), lane 16 the group's B rows, lane 17 its C rows (first chunk)
    if (warp == 0) {
      if (lane == 0) {
        const uint32_t bytes = static_cast<uint32_t>(hc * K * kDim * 2 + (h0 == 0 ? (K + Tb) * kDstate * 2 : 0));
        mbar_arrive_expect_tx(&pbar, bytes);
      }
      __syncwarp();
      if (lane < hc) {
        uint16_t* dst = xs + lane * L * kDim;
        const uint16_t* xh = xslot + static_cast<long long>(hb + lane) * L * kDim;
        if (n1 > 0) bulk_g2s(dst, xh + r * kDim, n1 * kDim * 2, &pbar);
        if (p > n1) bulk_g2s(dst + n1 * kDim, xh, (p - n1) * kDim * 2, &pbar);
        for (int t = 0; t < Tb; ++t)
          bulk_g2s(dst + (p + t) * kDim, a.x + (static_cast<long long>(tok0 + t) * H + hb + lane) * kDim, kDim * 2,
                   &pbar);
      } else if (lane == 16 && h0 == 0) {
        if (n1 > 0) bulk_g2s(bs, bring + r * kDstate, n1 * kDstate * 2, &pbar);
        if (p > n1) bulk_g2s(bs + n1 * kDstate, bring, (p - n1) * kDstate * 2, &pbar);
        for (int t = 0; t < Tb; ++t)
          bulk_g2s(bs + (p + t) * kDstate, a.B + (static_cast<long long>(tok0 + t) * G + g) * kDstate, kDstate * 2,
                   &pbar);
      } else if (lane == 17 && h0 == 0) {
        for (int t = 0; t < Tb; ++t)
          bulk_g2s(cs + t * kDstate, a.C + (static_cast<long long>(tok0 + t) * G + g) * kDstate, kDstate * 2, &pbar);
      }
    }
    for (int idx = tid; idx < hc * 32; idx += 256) {
      const int hh = idx >> 5, k = idx & 31;
      if (k < K) {
        const float* src = k < p ? dslot + static_cast<long long>(hb + hh) * L + ring(k)
                                 : a.dt + static_cast<long long>(tok0 + k - p) * H + hb + hh;
        cp_async4(&dts[hh][k], src);
      }
    }
    if (tid < hc) {
      cp_async4(&hp[0][tid], a.A + hb + tid);
      cp_async4(&hp[1][tid], a.D + hb + tid);
      cp_async4(&hp[2][tid], a.dt_bias + hb + tid);
    }
    cp_async_wait_all();
    if (!mbar_wait(&pbar, static_cast<uint32_t>(ph))) {
      if (tid == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      return;
    }
    __syncthreads();
    // dt' = softplus(dt + dt_bias) of every (head, new token) of the chunk at
    // once (the exact sequence: these values go into the ring), in place
    if (tid < hc * 8) {
      const int hh = tid >> 3, t = tid & 7;
      if (t < Tb) {
        const float v = spec_softplus(__fadd_rn(dts[hh][p + t], hp[2][hh]));
        dts[hh][p + t] = v;
        dslot[static_cast<long long>(hb + hh) * L + ring(p + t)] = v;
      }
    }
    if (h0 == 0) {
      // ring append of the new B rows
      if (tid < Tb * 16) {
        const int t = tid >> 4, q = tid & 15;
        reinterpret_cast<uint4*>(bring + ring(p + t) * kDstate)[q] =
            reinterpret_cast<const uint4*>(bs + (p + t) * kDstate)[q];
      }
      // C.B contraction on the tensor cores: CB[t][k] = sum_n C[t][n] B[k][n]
      // as mma.sync m16n8k16 (M = t, rows >= T_b zero; N = k, one 8-token
      // tile per warp; K = dstate in 8 steps), f32 accumulation of exact bf16
      // products.  Entries with k > p + t are never used.
      if (warp * 8 < K) {
        const int g8 = lane >> 2, c4 = lane & 3;
        const int kr = warp * 8 + g8 < K ? warp * 8 + g8 : K - 1;  // B row (token) of this lane
        const uint32_t* crow = reinterpret_cast<const uint32_t*>(cs + g8 * kDstate);
        const uint32_t* brow = reinterpret_cast<const uint32_t*>(bs + kr * kDstate);
        float d4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t a0 = g8 < Tb ? crow[8 * ks + c4] : 0u, a2 = g8 < Tb ? crow[8 * ks + 4 + c4] : 0u;
          mma_bf16(d4, a0, a2, brow[8 * ks + c4], brow[8 * ks + 4 + c4]);
        }
        if (g8 < TP) {
          CB[g8][warp * 8 + 2 * c4] = d4[0];
          CB[g8][warp * 8 + 2 * c4 + 1] = d4[1];
        }
      }
      // the C block for the readout's tensor-core contraction: [8][128] in the
      // MMA operand type (bf16 for f32/bf16 checkpoints, fp16 otherwise), rows
      // t >= T_b zero; 32-byte quad j of row t is stored at quad j ^ t, so the
      // readout's per-row fragment loads fall on distinct banks
      uint16_t* cbg = a.cf + (static_cast<long long>(b) * G + g) * 8 * kDstate;
      for (int idx = tid; idx < 8 * (kDstate / 2); idx += 256) {
        const int t = idx >> 6, q = idx & 63, n = 2 * q;
        uint32_t w = t < Tb ? reinterpret_cast<const uint32_t*>(cs + t * kDstate)[q] : 0u;
        if (c_f16) {
          const __half2 hv = __floats2half2_rn(bf16lo(w), bf16hi(w));
          w = *reinterpret_cast<const uint32_t*>(&hv);
        }
        reinterpret_cast<uint32_t*>(cbg)[(t * kDstate + 16 * (((n >> 4) ^ t) & 7) + (n & 15)) >> 1] = w;
      }
      __syncthreads();
    }
    // ring appends of the chunk's new x rows: lane hh < hc of warp 1, one bulk
    // copy a row out of shared memory (completed at the end of the chunk)
    if (warp == 1 && lane < hc && Tb > 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      for (int t = 0; t < Tb; ++t)
        bulk_s2g(xslot + (static_cast<long long>(hb + lane) * L + ring(p + t)) * kDim,
                 xs + lane * L * kDim + (p + t) * kDim, kDim * 2);
      bulk_commit();
    }
    if (h0) __syncthreads();  // the chunk's dt' (the first chunk synchronised above)
    for (int hh = warp; hh < hc; hh += 8) {
      const int h = hb + hh;
      const float Ah = hp[0][hh], Dh = hp[1][hh];
      const float dtp = lane < K ? dts[hh][lane] : 0.0f;
      if (fold) {
        // the fold's weights in the flush's canonical fp32 order (they decide
        // stored bits): c_j = sum_{i<=j} A dt'_i sequentially over the live
        // prefix, w_j = e^{c_end - c_j} dt'_j, and e^{c_end}
        const float aj = lane < p ? __fmul_rn(Ah, dtp) : 0.0f;
        float cj = 0.0f;
        for (int k = 0; k < p; ++k) {
          const float ak = __shfl_sync(0xffffffffu, aj, k);
          if (lane >= k) cj = __fadd_rn(cj, ak);
        }
        const float c_end = p > 0 ? __shfl_sync(0xffffffffu, cj, p - 1) : 0.0f;
        float* fwb = a.fw + (static_cast<long long>(b) * H + h) * kFoldW;
        fwb[lane] = lane < p ? __fmul_rn(spec_exp(__fsub_rn(c_end, cj)), dtp) : 0.0f;
        if (lane == 0) fwb[32] = spec_exp(c_end);
      }
      if (Tb == 0) continue;  // nothing to read out (a fold of a row without tokens)
      // inclusive prefix sum of A dt' over the lanes (these sums only feed the
      // outputs, so any summation order is fine here)
      float cum = lane < K ? Ah * dtp : 0.0f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, cum, off);
        if (lane >= off) cum += x;
      }
      float cf[TP];
      float dec[TP];
#pragma unroll
      for (int t = 0; t < TP; ++t) {
        const int kt = p + t < 31 ? p + t : 31;
        const float cpt = __shfl_sync(0xffffffffu, cum, kt);
        float v = 0.0f;
        if (t < Tb && lane <= p + t) {
          v = __expf(cpt - cum) * dtp * CB[t][lane];
          if (lane == p + t) v += Dh;
        }
        cf[t] = v;
        dec[t] = t < Tb ? __expf(cpt) : 0.0f;
      }
      float* blk = a.rblk + (static_cast<long long>(b) * H + h) * (kRDec + TP * kDim);
      if (lane == 0) {
        float4* d4 = reinterpret_cast<float4*>(blk);
        d4[0] = make_float4(dec[0], dec[1], dec[2], dec[3]);
        d4[1] = TP == 8 ? make_float4(dec[TP > 4 ? 4 : 0], dec[TP > 5 ? 5 : 0], dec[TP > 6 ? 6 : 0],
                                      dec[TP > 7 ? 7 : 0])
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
      // ring term of this head: R[t][d] = sum_k coef[k][t] x_k[d]; lane k
      // holds coef[k][.], shared through cfs; lane l accumulates d = 2l, 2l + 1;
      // blocks of 4 tokens at or past T_b are skipped (zero coefficients)
#pragma unroll
      for (int t4 = 0; t4 < TP; t4 += 4)
        *reinterpret_cast<float4*>(&cfs[warp][lane][t4]) = make_float4(cf[t4], cf[t4 + 1], cf[t4 + 2], cf[t4 + 3]);
      __syncwarp();
      float2 R[TP];
#pragma unroll
      for (int t = 0; t < TP; ++t) R[t] = make_float2(0.0f, 0.0f);
      const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs + hh * L * kDim) + lane;
      const bool hi4 = TP > 4 && Tb > 4;
#pragma unroll 4
      for (int k = 0; k < K; ++k) {
        const uint32_t w = xr[k * (kDim / 2)];
        const float2 xv = make_float2(bf16lo(w), bf16hi(w));
#pragma unroll
        for (int t4 = 0; t4 < TP; t4 += 4) {
          if (t4 > 0 && !hi4) continue;
          const float4 cv = *reinterpret_cast<const float4*>(&cfs[warp][k][t4]);
          R[t4 + 0] = __ffma2_rn(make_float2(cv.x, cv.x), xv, R[t4 + 0]);
          R[t4 + 1] = __ffma2_rn(make_float2(cv.y, cv.y), xv, R[t4 + 1]);
          R[t4 + 2] = __ffma2_rn(make_float2(cv.z, cv.z), xv, R[t4 + 2]);
          R[t4 + 3] = __ffma2_rn(make_float2(cv.w, cv.w), xv, R[t4 + 3]);
        }
      }
      // the row's T_b rows, chunk-swizzled (rblk_offset)
#pragma unroll
      for (int t = 0; t < TP; ++t)
        if (t < Tb) *reinterpret_cast<float2*>(blk + rblk_offset(t, 2 * lane)) = R[t];
      __syncwarp();  // cfs is rewritten for the warp's next head
    }
    if (warp == 1 && lane < hc) bulk_wait_all();  // the chunk's x appends are written (xs is reused next)
  }
}

// ---------------------------------------------------------------------------
// the one-call path's fold, from a readout stage
// ---------------------------------------------------------------------------
// Folds the unit's HPU heads in the flush's canonical fp32 order and stores the
// new checkpoints (and 8-bit row scales): for each of the warp's 8 state rows
// (lane: rows r0..r0+3, columns c0..c0+7)
//     acc = e^{c_end} S0f;  acc = fma(w_j x_j[d], B_j[n], acc) for j ascending
// with S0f read from the stage's TMA boxes (the checkpoint the outputs were
// just read from), the weights from the stage's fold area and the live x and B
// rows brought by the consumer threads into the CTA's fold buffer, 8 tokens at
// a time, double buffered (the producer hinted the rows into L2 when it issued
// the unit), then the flush's quantiser -- the operations rssm_flush performs.
// Every consumer warp calls it for the unit; the warps meet at the mbarrier
// fsync (8 arrivals a phase, bounded waits: returns false if a wait ran out,
// with RSSM_ERRBIT_TIMEOUT set; the caller then stops).
template <int DT, int HPU>
__device__ __forceinline__ bool fold_stage(const uint8_t* sb, uint8_t* fbuf, uint64_t* fsync, uint32_t& fph,
                                           const ReadLayout& lay, int fold_kb, const ReadMeta& m, int warp, int lane,
                                           const StepArgs& a) {
  const Cache& c = a.c;
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  static_assert(HPU == 1, "the fold takes one head per unit");
  const int r0 = 8 * warp + 4 * (lane >> 4), c0 = 8 * (lane & 15);
  const int p = m.p, L = c.L, rs = m.r, tid = threadIdx.x;
  const uint16_t* bg = c.B_cache + static_cast<long long>(m.s) * c.B_stride +
                       static_cast<long long>(m.h / c.hpg) * L * kDstate;
  const uint16_t* xg = c.x_cache + static_cast<long long>(m.s) * c.x_stride + static_cast<long long>(m.h) * L * kDim;
  // chunk ch of the live rows into buffer ch & 1: thread t < 64 copies 16 bytes
  // of an x row, 64 <= t < 192 of a B row (rows past the prefix are skipped)
  auto issue = [&](int ch) {
    uint8_t* dst = fbuf + (ch & 1) * kFoldBufOne;
    const int jj = tid < 64 ? tid >> 3 : (tid - 64) >> 4, jt = static_cast<int>(kFoldChunk) * ch + jj;
    if (tid < 192 && jt < p) {
      const int q = rs + jt >= L ? rs + jt - L : rs + jt;  // ring slot of live token jt
      if (tid < 64)
        cp_async16(dst + jj * kDim * 2 + (tid & 7) * 16, xg + q * kDim + (tid & 7) * 8);
      else
        cp_async16(dst + kFoldBufX + jj * kDstate * 2 + ((tid - 64) & 15) * 16, bg + q * kDstate + ((tid - 64) & 15) * 8);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // all consumer warps at one point (each thread's copies waited for first)
  auto cons_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(fsync);
    const bool ok = mbar_wait(fsync, fph);
    fph ^= 1u;
    if (!ok && lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
    return ok;
  };
  const int nch = (p + static_cast<int>(kFoldChunk) - 1) / static_cast<int>(kFoldChunk);
  if (nch > 0) issue(0);
  {
    const int j = 0;
    const float* fw = reinterpret_cast<const float*>(sb + lay.fw_off) + j * kFoldW;
    const float decay = fw[32];
    float2 acc[4][4];
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      const int row = 64 * j + r0 + i4;  // row of the stage's box (two heads' rows for HPU = 2)
      float v[8];
      if constexpr (DT == RSSM_F32) {
        const float4 x0 = *reinterpret_cast<const float4*>(sb + swizzled_offset<4>(row, c0));
        const float4 x1 = *reinterpret_cast<const float4*>(sb + swizzled_offset<4>(row, c0 + 4));
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
      } else if constexpr (DT == RSSM_BF16) {
        const uint4 q = *reinterpret_cast<const uint4*>(sb + swizzled_offset<2>(row, c0));
        v[0] = bf16lo(q.x); v[1] = bf16hi(q.x); v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
        v[4] = bf16lo(q.z); v[5] = bf16hi(q.z); v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
      } else if constexpr (DT == RSSM_F16) {
        const uint4 q = *reinterpret_cast<const uint4*>(sb + swizzled_offset<2>(row, c0));
        const float2 t0 = h2f2(q.x), t1 = h2f2(q.y), t2 = h2f2(q.z), t3 = h2f2(q.w);
        v[0] = t0.x; v[1] = t0.y; v[2] = t1.x; v[3] = t1.y; v[4] = t2.x; v[5] = t2.y; v[6] = t3.x; v[7] = t3.y;
      } else {
        const uint2 q = *reinterpret_cast<const uint2*>(sb + swizzled_offset<1>(row, c0));
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
      for (int q = 0; q < 4; ++q) acc[i4][q] = make_float2(__fmul_rn(decay, v[2 * q]), __fmul_rn(decay, v[2 * q + 1]));
    }
    for (int ch = 0; ch < nch; ++ch) {
      if (ch + 1 < nch) {
        issue(ch + 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      if (!cons_sync()) return false;  // every consumer thread's copies of chunk ch have landed
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(fbuf + (ch & 1) * kFoldBufOne);
      const uint16_t* bs = reinterpret_cast<const uint16_t*>(fbuf + (ch & 1) * kFoldBufOne + kFoldBufX);
      const int jend = min(static_cast<int>(kFoldChunk), p - static_cast<int>(kFoldChunk) * ch);
#pragma unroll 4
    for (int jj = 0; jj < jend; ++jj) {
      const float w = fw[static_cast<int>(kFoldChunk) * ch + jj];
      const uint2 xw = *reinterpret_cast<const uint2*>(xs + jj * kDim + r0);
      const float u0v = __fmul_rn(w, bf16lo(xw.x)), u1v = __fmul_rn(w, bf16hi(xw.x));
      const float u2v = __fmul_rn(w, bf16lo(xw.y)), u3v = __fmul_rn(w, bf16hi(xw.y));
      const uint4 bw = *reinterpret_cast<const uint4*>(bs + jj * kDstate + c0);
      const float2 bb[4] = {make_float2(bf16lo(bw.x), bf16hi(bw.x)), make_float2(bf16lo(bw.y), bf16hi(bw.y)),
                            make_float2(bf16lo(bw.z), bf16hi(bw.z)), make_float2(bf16lo(bw.w), bf16hi(bw.w))};
      const float2 uu[4] = {make_float2(u0v, u0v), make_float2(u1v, u1v), make_float2(u2v, u2v), make_float2(u3v, u3v)};
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i4][q] = __ffma2_rn(uu[i4], bb[q], acc[i4][q]);
    }
      if (!cons_sync()) return false;  // the buffer of chunk ch is refilled by chunk ch + 2
    }
    float accf[4][8];
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        accf[i4][2 * q] = acc[i4][q].x;
        accf[i4][2 * q + 1] = acc[i4][q].y;
      }
    const int h = m.h + j;
    void* head_state = static_cast<uint8_t*>(c.state) +
                       (static_cast<long long>(m.s) * c.state_stride + static_cast<long long>(h) * kHeadElems) * esz;
    float* head_scale = k8bit ? c.scale + static_cast<long long>(m.s) * c.scale_stride + h * kDim : nullptr;
    quantize_store<DT>(accf, r0, c0, lane, head_state, head_scale, c.rounding, static_cast<uint32_t>(h),
                       static_cast<uint32_t>(m.s), m.epoch, a.seed);
  }
  return true;
}

// ---------------------------------------------------------------------------
// readout
// ---------------------------------------------------------------------------
// HPU: heads per unit (2 for 8-bit states when a group has an even number of
// heads: the unit's copies then carry twice the bytes for the same work).
// FOLD (the one-call path, rssm_flush_step): units of rows the precompute
// flagged for a flush also fold their live prefix into a new checkpoint, from
// the same stage the outputs are read from (the outputs replay the whole live
// prefix from the old checkpoint, as an unflushed row's do), and the unit of
// head 0 of such a row writes the flush's bookkeeping.
template <int DT, int TP, int HPU, bool GATE, bool FOLD>
__global__ void __maxnreg__(96) readout_kernel(const __grid_constant__ CUtensorMap s0map, StepArgs a, int ns) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Cache& c = a.c;
  const int fold_kb = FOLD ? ring_pad(c.L) : 0;
  const ReadLayout lay = read_layout(DT, TP, ns, HPU, fold_kb);
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  constexpr bool kFp4 = DT == RSSM_NVFP4;  // an NVFP4 read checkpoint (two state rows per 128-byte box row)
  constexpr int kBox = 8192 * HPU;         // bytes of one column box of S0 (64*HPU rows x 128 bytes)
  constexpr int kNBox = kFp4 ? 1 : esz;    // column boxes per unit
  constexpr int kHeadOff = kFp4 ? 4096 : 8192;  // bytes between the heads of a unit inside a box
  constexpr int kRowsPerHead = kFp4 ? 32 : kDim;  // box rows per head
  const int H = c.H, HU = H / HPU;

  // Units are taken in chunks of consecutive (row, head) pairs: each CTA's
  // first chunk is chunk blockIdx.x (its S0 can be requested before the
  // precompute has finished); later chunks come from a counter the
  // precompute zeroes, so CTAs that stream faster take more of them.  Chunks
  // hold kReadChunk units until about two units per CTA are left, then one
  // (guided sizes: the CTAs finish within about one unit of each other).
  const unsigned units = static_cast<unsigned>(a.batch) * static_cast<unsigned>(HU);
  const unsigned tail = min(units, 2u * gridDim.x);
  const unsigned nbig = (units - tail) / kReadChunk;
  const unsigned big_end = nbig * kReadChunk;
  const unsigned nchunks = nbig + (units - big_end);
  // first unit of chunk ch (< nchunks) and the end of its range
  auto chunk_range = [&](unsigned ch, unsigned& first, unsigned& last) {
    first = ch < nbig ? ch * kReadChunk : big_end + (ch - nbig);
    last = ch < nbig ? first + kReadChunk : first + 1u;
  };

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 8;
  ReadMeta* meta = reinterpret_cast<ReadMeta*>(smem + 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < ns; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumerWarps);
    }
    if (FOLD) mbar_init(full + 16, kConsumerWarps);  // the fold's consumer barrier
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane issues all copies ----------------
    if (lane != 0) return;
    // Before waiting for the precompute: request S0 of the first chunk's
    // units.  S0 is final by now (the precompute waited for the flush before
    // it let this kernel launch) and needs only the slot id, an input of the call.
    unsigned u, cend;
    chunk_range(blockIdx.x, u, cend);
    int b = static_cast<int>(u / HU), h = static_cast<int>(u % HU) * HPU;  // h: the unit's first head
    const int npre = static_cast<int>(cend - u) < ns ? static_cast<int>(cend - u) : ns;
    uint32_t pre = 0u;
    for (int i = 0, pb = b, phh = h; i < npre; ++i, phh = phh + HPU == H ? 0 : phh + HPU, pb += phh == 0 ? 1 : 0) {
      const int s = a.slot_idx[pb];
      if (s >= 1 && s < c.S) {
        uint8_t* sb = smem + lay.stages_off + i * lay.stage_bytes;
        mbar_expect_tx(&full[i], lay.s0_bytes);
#pragma unroll
        for (int bx = 0; bx < kNBox; ++bx)
          tma_load_3d(sb + bx * kBox, &s0map, bx * (128 / esz), phh * kRowsPerHead, s, &full[i]);
        pre |= 1u << i;
      }
    }
    pdl_wait();  // row records, C blocks, ring terms, the chunk counter
    pdl_trigger();
    unsigned next = atomicAdd(a.rwork, 1u);  // the chunk after this one (read at the switch)
    int cur_b = -1, cur_bg = -1;
    RowRec rr = {};
    int issued = 0;
    bool ok = true;
    // per unit: stage index and phase, the (row, head) and the head's group
    // advance by increments (no division on the per-unit path)
    int st = 0, g = h / c.hpg, hh = h % c.hpg;
    uint32_t ph = 0;
    const int rstride = kRDec + TP * kDim;  // floats per ring-term block
    for (int i = 0;; ++i) {
      if (u >= cend) {  // next chunk
        const unsigned ch = gridDim.x + next;
        if (ch >= nchunks) break;
        chunk_range(ch, u, cend);
        b = static_cast<int>(u / HU);
        h = static_cast<int>(u % HU) * HPU;
        g = h / c.hpg;
        hh = h % c.hpg;
        next = atomicAdd(a.rwork, 1u);
      }
      if (i > 0 && ++st == ns) {
        st = 0;
        ph ^= 1u;
      }
      if (i >= ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
        break;
      }
      if (b != cur_b) {
        rr = a.rows[b];
        cur_b = b;
      }
      const bool active = (rr.flags & 1) && rr.Tb > 0;
      const bool fold = FOLD && (rr.flags & 2);
      const int bg = b * c.G + g;
      // the C block is copied only when the (row, group) changes: consumers
      // keep its fragments in registers (flags bit 1 tells them to reload)
      const bool newc = active && bg != cur_bg;
      if (active) cur_bg = bg;
      meta[st] = ReadMeta{b, h, rr.s, rr.r, rr.p, rr.Tb, rr.tok0,
                          (active ? 1 : 0) | (newc ? 2 : 0) | (fold ? 16 : 0), rr.epoch_new,
                          rr.gs, {0, 0}};
      if (active || fold) {
        const int s = rr.s;
        uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
        const bool have_s0 = i < npre && ((pre >> i) & 1u);
        // ring terms: the decay floats and the row's T_b rows of the last head's
        // block (the blocks of the unit's heads are consecutive)
        const uint32_t r_bytes =
            active ? static_cast<uint32_t>(((HPU - 1) * rstride + kRDec + rr.Tb * kDim) * 4) : 0u;
        const int pf = fold ? rr.p : 0;  // live rows the fold reads
        const uint32_t f_bytes = fold ? static_cast<uint32_t>(HPU * kFoldW * 4) : 0u;
        const uint32_t bytes = (have_s0 ? 0u : lay.s0_bytes) + (k8bit ? 256u * HPU : 0u) + (kFp4 ? 512u * HPU : 0u) +
                               (newc ? 8u * kDstate * 2 : 0u) + r_bytes + f_bytes;
        mbar_arrive_expect_tx(&full[st], bytes);
        if (!have_s0) {
#pragma unroll
          for (int bx = 0; bx < kNBox; ++bx)
            tma_load_3d(sb + bx * kBox, &s0map, bx * (128 / esz), h * kRowsPerHead, s, &full[st]);
        }
        if (k8bit)
          bulk_g2s(sb + lay.scale_off, c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim, 256 * HPU,
                   &full[st]);
        if (kFp4)  // the heads' block scales [64 hpu][8]
          bulk_g2s(sb + lay.scale_off, c.read_sf + static_cast<long long>(s) * c.read_sf_stride + h * kDim * 8,
                   512 * HPU, &full[st]);
        if (newc) bulk_g2s(sb + lay.c_off, a.cf + static_cast<long long>(bg) * 8 * kDstate, 8 * kDstate * 2, &full[st]);
        if (active) bulk_g2s(sb + lay.r_off, a.rblk + static_cast<long long>(u) * HPU * rstride, r_bytes, &full[st]);
        if constexpr (FOLD) {
          if (fold) {
            // the fold weights into the stage; the live prefix (at most two
            // contiguous ring segments) of the heads' x rows and the group's B
            // rows hinted into L2 for the consumers' reads
            const int L = c.L, r0 = rr.r, n1 = min(pf, L - r0);
            const uint16_t* xg = c.x_cache + static_cast<long long>(s) * c.x_stride + static_cast<long long>(h) * L * kDim;
            const uint16_t* bgp = c.B_cache + static_cast<long long>(s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
#pragma unroll
            for (int j = 0; j < HPU; ++j) {
              const uint16_t* xj = xg + static_cast<long long>(j) * L * kDim;
              if (n1 > 0) prefetch_l2(xj + r0 * kDim, n1 * kDim * 2);
              if (pf > n1) prefetch_l2(xj, (pf - n1) * kDim * 2);
            }
            if (n1 > 0) prefetch_l2(bgp + r0 * kDstate, n1 * kDstate * 2);
            if (pf > n1) prefetch_l2(bgp, (pf - n1) * kDstate * 2);
            bulk_g2s(sb + lay.fw_off, a.fw + (static_cast<long long>(b) * H + h) * kFoldW, HPU * kFoldW * 4, &full[st]);
            if (h == 0) {
              // the flush's bookkeeping (nothing in this kernel reads it; the
              // outputs use the row records)
              c.ring_start[s] = r0 + pf >= L ? r0 + pf - L : r0 + pf;
              a.pnat_rw[b] = 0;
              c.epoch[s] = rr.epoch_new;
            }
          }
        }
      } else {
        mbar_arrive(&full[st]);
      }
      issued = i + 1;
      ++u;
      if ((h += HPU) == H) {
        h = 0;
        ++b;
        g = 0;
        hh = 0;
      } else if ((hh += HPU) == c.hpg) {
        hh = 0;
        ++g;
      }
    }
    if (ok) {  // end of work for the consumers
      if (++st == ns) {
        st = 0;
        ph ^= 1u;
      }
      if (issued >= ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
      } else {
        meta[st].flags = 8;
        mbar_arrive(&full[st]);
      }
    }
    if (!ok) {
      set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      for (int i = max(0, issued - ns); i < issued; ++i) mbar_wait(&full[i % ns], (i / ns) & 1);
    }
    return;
  }

  // ---------------- consumer warps: state rows 8*warp .. 8*warp+7 ----------------
  const int g = lane >> 2, cq = lane & 3;
  const int d = 8 * warp + g;        // B column (row of S0) this lane loads
  const int dout = 8 * warp + 2 * cq;  // output rows this lane writes (dout, dout + 1)
  uint2 af[8];                          // C block fragments of the current (row, group)
  uint32_t fph = 0;                     // phase of the fold's consumer barrier
  int st = 0;
  uint32_t ph = 0;
  for (int i = 0;; ++i) {
    if (i > 0 && ++st == ns) {
      st = 0;
      ph ^= 1u;
    }
    if (!mbar_wait(&full[st], ph)) {
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      return;
    }
    const ReadMeta m = meta[st];
    if (m.flags & 8) return;  // no more work
    const uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
    if (!(m.flags & (1 | 16))) {
      // inactive or rejected row: zero outputs, no cache update
      for (int idx = lane; idx < m.Tb * 4 * HPU; idx += 32) {
        const int t = idx / (4 * HPU), j = (idx >> 2) % HPU, q = idx & 3;
        *reinterpret_cast<uint32_t*>(a.out + (static_cast<long long>(m.tok0 + t) * H + m.h + j) * kDim + 8 * warp +
                                     2 * q) = 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      continue;
    }
    if constexpr (FOLD) {
      if (!(m.flags & 1)) {  // a fold of a row without tokens: no outputs
        if (!fold_stage<DT, HPU>(sb, smem + lay.fbuf_off, full + 16, fph, lay, fold_kb, m, warp, lane, a)) return;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        continue;
      }
    }
    if (m.flags & 2) load_c_frags(reinterpret_cast<const uint16_t*>(sb + lay.c_off), g, cq, af);
    // output gate (GATE): this lane's z pair per head, requested before the contraction
    uint32_t zw[HPU];
#pragma unroll
    for (int j = 0; j < HPU; ++j) zw[j] = 0u;
    if constexpr (GATE) {
      if (g < m.Tb) {
#pragma unroll
        for (int j = 0; j < HPU; ++j)
          zw[j] = *reinterpret_cast<const uint32_t*>(a.z + (static_cast<long long>(m.tok0 + g) * H + m.h + j) * kDim +
                                                     dout);
      }
    }
    float y[HPU][2];
#pragma unroll
    for (int j = 0; j < HPU; ++j) {  // head m.h + j: rows 64 j .. of the stage's boxes
      float acc[4];
      uint64_t sfrow = 0;
      if constexpr (kFp4) sfrow = *reinterpret_cast<const uint64_t*>(sb + lay.scale_off + (64 * j + d) * 8);
      s0_dot_c<DT, kBox>(sb + j * kHeadOff, af, d, cq, acc, sfrow);
      const float* rb = reinterpret_cast<const float*>(sb + lay.r_off) + j * (kRDec + TP * kDim);
      const float2 rv = g < m.Tb ? *reinterpret_cast<const float2*>(rb + rblk_offset(g, dout)) : make_float2(0.0f, 0.0f);
      const float dec = g < m.Tb ? rb[g] : 0.0f;
      float sc0 = 1.0f, sc1 = 1.0f;
      if constexpr (kFp4) sc0 = sc1 = m.gs;
      if constexpr (k8bit) {
        const float2 scv = *reinterpret_cast<const float2*>(sb + lay.scale_off + j * 256 + dout * 4);
        sc0 = scv.x;
        sc1 = scv.y;
      }
      y[j][0] = fmaf(dec * sc0, acc[0], rv.x);
      y[j][1] = fmaf(dec * sc1, acc[1], rv.y);
      if constexpr (GATE) {  // y * silu(z), silu(v) = v / (1 + e^-v)
        const float z0 = bf16lo(zw[j]), z1 = bf16hi(zw[j]);
        y[j][0] *= z0 / (1.0f + __expf(-z0));
        y[j][1] *= z1 / (1.0f + __expf(-z1));
      }
    }
    if constexpr (FOLD) {
      if (m.flags & 16) {
        if (!fold_stage<DT, HPU>(sb, smem + lay.fbuf_off, full + 16, fph, lay, fold_kb, m, warp, lane, a)) return;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
    if (g < m.Tb) {
#pragma unroll
      for (int j = 0; j < HPU; ++j) {
        const __nv_bfloat162 yv = __floats2bfloat162_rn(y[j][0], y[j][1]);
        *reinterpret_cast<__nv_bfloat162*>(a.out + (static_cast<long long>(m.tok0 + g) * H + m.h + j) * kDim + dout) =
            yv;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
int launch_precompute(const StepArgs& a, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = a.batch * a.c.G;
  const size_t smem = precompute_smem(a.c.hpg, a.c.L);
  // 256-thread CTAs, four per SM at T <= 4 (64 registers, ~55 KB of shared
  // memory at L = 20), three at T <= 8
  auto kern = a.TP == 4 ? precompute_kernel<4> : precompute_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(precompute_smem(kHeadChunk, kMaxL)));
  if (e == cudaSuccess) e = launch_pdl(kern, dim3(grid), dim3(256), smem, st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DT, int TP, int HPU, bool GATE, bool FOLD>
static int launch_readout_t(const StepArgs& a, int num_sms, cudaStream_t st) {
  // as many stages as fit two CTAs per SM (>= 3), else one CTA with up to 8
  const int fold_kb = FOLD ? ring_pad(a.c.L) : 0;
  int ns = 8, ctas = 2;
  for (; ns >= 3; --ns)
    if (read_layout(DT, TP, ns, HPU, fold_kb).total <= 113 * 1024) break;
  if (ns < 3) {
    ctas = 1;
    for (ns = 8; ns > 2; --ns)
      if (read_layout(DT, TP, ns, HPU, fold_kb).total <= 225 * 1024) break;
  }
  const ReadLayout lay = read_layout(DT, TP, ns, HPU, fold_kb);
  CUtensorMap map;
  if (!encode_state_map(a.c, &map, HPU)) return cudaErrorInvalidValue;
  auto kern = readout_kernel<DT, TP, HPU, GATE, FOLD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, lay.total);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  if (occ > ctas) occ = ctas;
  const long long chunks = (static_cast<long long>(a.batch) * (a.c.H / HPU) + kReadChunk - 1) / kReadChunk;
  const long long cap = static_cast<long long>(num_sms) * occ;
  const int grid = static_cast<int>(chunks < cap ? chunks : cap);  // every CTA has a first chunk
  e = launch_pdl(kern, dim3(grid), dim3(kThreads), lay.total, st, map, a, ns);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DT, bool FOLD>
static int launch_readout_dt(const StepArgs& a, int num_sms, cudaStream_t st) {
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3 || DT == RSSM_NVFP4;
  const bool pair = k8bit && a.c.hpg % 2 == 0;
  if constexpr (!FOLD) {
    if (a.z) {
      if (a.TP == 4)
        return pair ? launch_readout_t<DT, 4, 2, true, false>(a, num_sms, st)
                    : launch_readout_t<DT, 4, 1, true, false>(a, num_sms, st);
      return pair ? launch_readout_t<DT, 8, 2, true, false>(a, num_sms, st)
                  : launch_readout_t<DT, 8, 1, true, false>(a, num_sms, st);
    }
  }
  if constexpr (FOLD) {  // one head per unit (a two-head fold does not fit the register budget)
    return a.TP == 4 ? launch_readout_t<DT, 4, 1, false, true>(a, num_sms, st)
                     : launch_readout_t<DT, 8, 1, false, true>(a, num_sms, st);
  } else {
    if (a.TP == 4)
      return pair ? launch_readout_t<DT, 4, 2, false, false>(a, num_sms, st)
                  : launch_readout_t<DT, 4, 1, false, false>(a, num_sms, st);
    return pair ? launch_readout_t<DT, 8, 2, false, false>(a, num_sms, st)
                : launch_readout_t<DT, 8, 1, false, false>(a, num_sms, st);
  }
}

template <bool FOLD>
static int launch_readout_any(const StepArgs& a, int num_sms, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (a.c.dtype) {
    case RSSM_F32: return launch_readout_dt<RSSM_F32, FOLD>(a, num_sms, st);
    case RSSM_BF16: return launch_readout_dt<RSSM_BF16, FOLD>(a, num_sms, st);
    case RSSM_F16: return launch_readout_dt<RSSM_F16, FOLD>(a, num_sms, st);
    case RSSM_I8: return launch_readout_dt<RSSM_I8, FOLD>(a, num_sms, st);
    case RSSM_NVFP4:  // a read-checkpoint format: the one-call path keeps one checkpoint
      if constexpr (FOLD) return cudaErrorInvalidValue;
      else return launch_readout_dt<RSSM_NVFP4, false>(a, num_sms, st);
    default: return launch_readout_dt<RSSM_E4M3, FOLD>(a, num_sms, st);
  }
}

int launch_readout(const StepArgs& a, int num_sms, void* stream) { return launch_readout_any<false>(a, num_sms, stream); }
int launch_readout_fold(const StepArgs& a, int num_sms, void* stream) {
  return launch_readout_any<true>(a, num_sms, stream);
}

}  // namespace rssm
