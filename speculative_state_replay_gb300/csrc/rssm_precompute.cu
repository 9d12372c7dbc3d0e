// rssm_precompute.cu -- the precompute of the ReplaySSM checkpointing SSU
// (FlashInfer PR #3975, Description item 1: the first kernel of the two-kernel
// split), one CTA per (row, group): dt' = softplus(dt + dt_bias) for the new
// tokens (appended to the dt ring), the cumulative sums c_k = sum_{i<=k} A
// dt'_i over live ring + new tokens (recomputed, not cached: Description item
// 2), the C.B contraction CB[t][k] = C_t . B_k once per group, and per head the
// replay coefficients
//     coef[k][t] = e^{c_{p+t} - c_k} dt'_k CB[t][k]  (+ D on k = p+t)
// applied at once to the head's x rows:
//     R[t][d] = sum_k coef[k][t] x_k[d],   decay[t] = e^{c_{p+t}}
// written to scratch (the row's T_b rows) with the C rows (in the readout's
// MMA type).  Appends B, x and dt'.  In the one-call path it also takes the
// flush decision and writes the fold weights of flushed rows.
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

// Replay coefficients and ring term of one head (one warp) for a row with
// T_b <= 2 NP new tokens, taken as NP token pairs; lane k < K holds dt'_k.
//   coef[k][t] = e^{c_{p+t} - c_k} dt'_k CB[t][k] (+ D on k = p + t), k <= p + t
//   R[t][d] = sum_k coef[k][t] x_k[d],  decay[t] = e^{c_{p+t}}
// Lane k puts coef[k][.] in the warp's cfw row k; lane l then accumulates
// d = 2l and 2l + 1 for every pair: (R[2j][d], R[2j+1][d]) += (coef[k][2j],
// coef[k][2j+1]) x_k[d], one f32x2 FMA each.  Writes the T_b rows of the
// row's ring-term block (chunk-swizzled) and its decays.
template <int NP, int TP>
__device__ __forceinline__ void head_ring_term(const float (*CB)[kMaxL], float (*cfw)[TP], const uint32_t* xr,
                                               float* blk, int lane, int p, int Tb, int K, float Ah, float Dh,
                                               float dtp) {
  static_assert(2 * NP <= TP, "token pairs beyond the padded token count");
  // inclusive prefix sum of A dt' over the lanes (these sums only feed the
  // outputs, so any summation order is fine here)
  float cum = lane < K ? Ah * dtp : 0.0f;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float x = __shfl_up_sync(0xffffffffu, cum, off);
    if (lane >= off) cum += x;
  }
  float cf[2 * NP], dec[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) dec[t] = 0.0f;
#pragma unroll
  for (int t = 0; t < 2 * NP; ++t) {
    const int kt = p + t < 31 ? p + t : 31;
    const float cpt = __shfl_sync(0xffffffffu, cum, kt);
    float v = 0.0f;
    if (t < Tb && lane <= p + t) {
      v = __expf(cpt - cum) * dtp * CB[t][lane];
      if (lane == p + t) v += Dh;
    }
    cf[t] = v;
    if (t < Tb) dec[t] = __expf(cpt);
  }
  if (lane == 0) {
    float4* d4 = reinterpret_cast<float4*>(blk);
    d4[0] = make_float4(dec[0], dec[1], dec[2], dec[3]);
    if (TP == 8) d4[1] = make_float4(dec[4], dec[5], dec[6], dec[7]);
  }
#pragma unroll
  for (int j = 0; j < NP; j += 2) {
    if (j + 1 < NP)
      *reinterpret_cast<float4*>(&cfw[lane][2 * j]) = make_float4(cf[2 * j], cf[2 * j + 1], cf[2 * j + 2], cf[2 * j + 3]);
    else
      *reinterpret_cast<float2*>(&cfw[lane][2 * j]) = make_float2(cf[2 * j], cf[2 * j + 1]);
  }
  __syncwarp();
  float2 P0[NP], P1[NP];  // (R[2j][2l], R[2j+1][2l]), (R[2j][2l+1], R[2j+1][2l+1])
#pragma unroll
  for (int j = 0; j < NP; ++j) P0[j] = P1[j] = make_float2(0.0f, 0.0f);
#pragma unroll 2
  for (int k = 0; k < K; ++k) {
    const uint32_t w = xr[k * (kDim / 2)];
    const float x0 = bf16lo(w), x1 = bf16hi(w);
    const float2 X0 = make_float2(x0, x0), X1 = make_float2(x1, x1);
#pragma unroll
    for (int j = 0; j < NP; j += 2) {
      float2 c0, c1;
      if (j + 1 < NP) {
        const float4 c4 = *reinterpret_cast<const float4*>(&cfw[k][2 * j]);
        c0 = make_float2(c4.x, c4.y);
        c1 = make_float2(c4.z, c4.w);
      } else {
        c0 = *reinterpret_cast<const float2*>(&cfw[k][2 * j]);
      }
      P0[j] = __ffma2_rn(c0, X0, P0[j]);
      P1[j] = __ffma2_rn(c0, X1, P1[j]);
      if (j + 1 < NP) {
        P0[j + 1] = __ffma2_rn(c1, X0, P0[j + 1]);
        P1[j + 1] = __ffma2_rn(c1, X1, P1[j + 1]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 2 * NP; ++t)
    if (t < Tb)
      *reinterpret_cast<float2*>(blk + rblk_offset(t, 2 * lane)) =
          t & 1 ? make_float2(P0[t >> 1].y, P1[t >> 1].y) : make_float2(P0[t >> 1].x, P1[t >> 1].x);
  __syncwarp();  // cfw is rewritten for the warp's next head
}


template <int TP>
__global__ void __launch_bounds__(256, TP == 4 ? 4 : 3) precompute_kernel(StepArgs a) {
  extern __shared__ __align__(16) unsigned char psm[];
  __shared__ float CB[TP][kMaxL];
  __shared__ float dts[kHeadChunk][kMaxL];  // dt' of the live tokens; dt of the new ones (before bias, softplus)
  __shared__ float hp[3][kHeadChunk];       // A, D, dt_bias of the chunk's heads
  __shared__ __align__(16) float cfs[8][kMaxL][TP];  // per warp: coef[k][t] of its current head
  __shared__ int meta[7];
  const Cache& c = a.c;
  const int b = blockIdx.x / c.G, g = blockIdx.x % c.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = c.L, H = c.H, G = c.G, hpg = c.hpg;
  uint16_t* xs = reinterpret_cast<uint16_t*>(psm);
  uint16_t* bs = xs + head_chunk(hpg) * L * kDim;
  uint16_t* cs = bs + L * kDstate;
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
  // B and C rows of the group
  for (int idx = tid; idx < K * 16; idx += 256) {
    const int k = idx >> 4, q = idx & 15;
    const uint16_t* src = k < p ? bring + ring(k) * kDstate
                                : a.B + (static_cast<long long>(tok0 + k - p) * G + g) * kDstate;
    cp_async16(bs + k * kDstate + q * 8, src + q * 8);
  }
  if (tid < Tb * 16) {
    const int t = tid >> 4, q = tid & 15;
    cp_async16(cs + t * kDstate + q * 8, a.C + (static_cast<long long>(tok0 + t) * G + g) * kDstate + q * 8);
  }
  const bool c_f16 = c.dtype == RSSM_F16 || c.dtype == RSSM_I8 || c.dtype == RSSM_E4M3 || c.dtype == RSSM_NVFP4;
  for (int h0 = 0; h0 < hpg; h0 += kHeadChunk) {
    const int hc = hpg - h0 < kHeadChunk ? hpg - h0 : kHeadChunk, hb = g * hpg + h0;
    if (h0) __syncthreads();  // every warp is done with the previous chunk's rows
    // x rows: warp w brings the rows of the heads it works on (w, w + 8), 16
    // bytes a lane (per-thread copies: a warp's many small 1-D bulk copies
    // would queue one after another)
    for (int hh = warp; hh < hc; hh += 8) {
      for (int q = lane; q < K * 8; q += 32) {
        const int k = q >> 3, part = q & 7;
        const uint16_t* src = k < p ? xslot + (static_cast<long long>(hb + hh) * L + ring(k)) * kDim
                                    : a.x + (static_cast<long long>(tok0 + k - p) * H + hb + hh) * kDim;
        cp_async16(xs + (hh * L + k) * kDim + part * 8, src + part * 8);
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
    // ring appends of the chunk's new x rows
    for (int idx = tid; idx < hc * 64; idx += 256) {
      const int hh = idx >> 6, t = (idx >> 3) & 7, q = idx & 7;
      if (t < Tb)
        reinterpret_cast<uint4*>(xslot + (static_cast<long long>(hb + hh) * L + ring(p + t)) * kDim)[q] =
            *reinterpret_cast<const uint4*>(xs + (hh * L + p + t) * kDim + q * 8);
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
      float* blk = a.rblk + (static_cast<long long>(b) * H + h) * (kRDec + TP * kDim);
      const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs + hh * L * kDim) + lane;
      const int np = (Tb + 1) >> 1;  // token pairs the row needs
      if (np == 1)
        head_ring_term<1, TP>(CB, cfs[warp], xr, blk, lane, p, Tb, K, Ah, Dh, dtp);
      else if (np == 2 || TP == 4)
        head_ring_term<2, TP>(CB, cfs[warp], xr, blk, lane, p, Tb, K, Ah, Dh, dtp);
      else if (np == 3)
        head_ring_term<(TP > 4 ? 3 : 2), TP>(CB, cfs[warp], xr, blk, lane, p, Tb, K, Ah, Dh, dtp);
      else
        head_ring_term<(TP > 4 ? 4 : 2), TP>(CB, cfs[warp], xr, blk, lane, p, Tb, K, Ah, Dh, dtp);
    }
  }
}

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

}  // namespace rssm
