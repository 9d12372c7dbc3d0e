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
//       written to scratch with the C rows (in the readout's MMA type).
//       Appends B, x and dt'.
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
  __shared__ int meta[6];
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
      const bool tb_ok = Tb >= 0 && Tb <= a.T;
      if (s >= 1 && s < c.S) {
        if (!tb_ok) {
          if (g == 0) set_error(c.err, RSSM_ERRBIT_SEQLEN);
        } else if (pn < 0 || pn + Tb > L) {
          if (g == 0) set_error(c.err, RSSM_ERRBIT_PNAT);
        } else {
          p = pn;
          r = c.ring_start[s];
          flags = 1;
        }
      }
      if (!tb_ok) Tb = 0;
      meta[0] = s; meta[1] = r; meta[2] = p; meta[3] = Tb; meta[4] = tok0; meta[5] = flags;
      if (g == 0) a.rows[b] = RowRec{s, r, p, Tb, tok0, flags, p, 0u};
      if (blockIdx.x == 0) *a.rwork = 0u;  // the readout's chunk counter
    }
  }
  __syncthreads();
  const int s = meta[0], r = meta[1], p = meta[2], Tb = meta[3], tok0 = meta[4];
  if (!meta[5] || Tb == 0) return;
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
  const bool c_f16 = c.dtype == RSSM_F16 || c.dtype == RSSM_I8 || c.dtype == RSSM_E4M3;
  for (int h0 = 0; h0 < hpg; h0 += kHeadChunk) {
    const int hc = hpg - h0 < kHeadChunk ? hpg - h0 : kHeadChunk, hb = g * hpg + h0;
    if (h0) __syncthreads();  // every warp is done with the previous chunk's rows
    // x rows: warp w brings the rows of the heads it works on (w, w + 8), 16 bytes a lane
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
            reinterpret_cast<const uint4*>(xs + (hh * L + p + t) * kDim)[q];
    }
    if (h0) __syncthreads();  // the chunk's dt' (the first chunk synchronised above)
    for (int hh = warp; hh < hc; hh += 8) {
      const int h = hb + hh;
      const float Ah = hp[0][hh], Dh = hp[1][hh];
      const float dtp = lane < K ? dts[hh][lane] : 0.0f;
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
      // ring term of this head: R[t][d] = sum_k coef[k][t] x_k[d]; lane k
      // holds coef[k][.], shared through cfs; lane l accumulates d = 2l, 2l + 1
#pragma unroll
      for (int t4 = 0; t4 < TP; t4 += 4)
        *reinterpret_cast<float4*>(&cfs[warp][lane][t4]) = make_float4(cf[t4], cf[t4 + 1], cf[t4 + 2], cf[t4 + 3]);
      __syncwarp();
      float2 R[TP];
#pragma unroll
      for (int t = 0; t < TP; ++t) R[t] = make_float2(0.0f, 0.0f);
      const uint32_t* xr = reinterpret_cast<const uint32_t*>(xs + hh * L * kDim) + lane;
#pragma unroll 4
      for (int k = 0; k < K; ++k) {
        const uint32_t w = xr[k * (kDim / 2)];
        const float2 xv = make_float2(bf16lo(w), bf16hi(w));
#pragma unroll
        for (int t4 = 0; t4 < TP; t4 += 4) {
          const float4 cv = *reinterpret_cast<const float4*>(&cfs[warp][k][t4]);
          R[t4 + 0] = __ffma2_rn(make_float2(cv.x, cv.x), xv, R[t4 + 0]);
          R[t4 + 1] = __ffma2_rn(make_float2(cv.y, cv.y), xv, R[t4 + 1]);
          R[t4 + 2] = __ffma2_rn(make_float2(cv.z, cv.z), xv, R[t4 + 2]);
          R[t4 + 3] = __ffma2_rn(make_float2(cv.w, cv.w), xv, R[t4 + 3]);
        }
      }
      __syncwarp();  // cfs is rewritten for the warp's next head
      float* blk = a.rblk + (static_cast<long long>(b) * H + h) * (TP * kRStride + TP);
#pragma unroll
      for (int t = 0; t < TP; ++t) reinterpret_cast<float2*>(blk + t * kRStride)[lane] = R[t];
      if (lane == 0) {
#pragma unroll
        for (int t4 = 0; t4 < TP; t4 += 4)
          *reinterpret_cast<float4*>(blk + TP * kRStride + t4) = make_float4(dec[t4], dec[t4 + 1], dec[t4 + 2], dec[t4 + 3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// readout
// ---------------------------------------------------------------------------
// HPU: heads per unit (2 for 8-bit states when a group has an even number of
// heads: the unit's copies then carry twice the bytes for the same work)
template <int DT, int TP, int HPU, bool GATE>
__global__ void __maxnreg__(96) readout_kernel(const __grid_constant__ CUtensorMap s0map, StepArgs a, int ns) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Cache& c = a.c;
  const ReadLayout lay = read_layout(DT, TP, ns, HPU);
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  constexpr int kBox = 8192 * HPU;  // bytes of one column box of S0 (64*HPU rows x 128 bytes)
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
        for (int bx = 0; bx < esz; ++bx) tma_load_3d(sb + bx * kBox, &s0map, bx * (128 / esz), phh * kDim, s, &full[i]);
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
    const int rstride = TP * kRStride + TP;
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
      const int bg = b * c.G + g;
      // the C block is copied only when the (row, group) changes: consumers
      // keep its fragments in registers (flags bit 1 tells them to reload)
      const bool newc = active && bg != cur_bg;
      if (active) cur_bg = bg;
      meta[st] = ReadMeta{b, h, rr.s, rr.r, rr.p, rr.Tb, rr.tok0, (active ? 1 : 0) | (newc ? 2 : 0)};
      if (active) {
        const int s = rr.s;
        uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
        const bool have_s0 = i < npre && ((pre >> i) & 1u);
        const uint32_t bytes =
            (have_s0 ? 0u : lay.s0_bytes) + (k8bit ? 256u * HPU : 0u) + (newc ? 8u * kDstate * 2 : 0u) + lay.r_bytes;
        mbar_arrive_expect_tx(&full[st], bytes);
        if (!have_s0) {
#pragma unroll
          for (int bx = 0; bx < esz; ++bx) tma_load_3d(sb + bx * kBox, &s0map, bx * (128 / esz), h * kDim, s, &full[st]);
        }
        if (k8bit)
          bulk_g2s(sb + lay.scale_off, c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim, 256 * HPU,
                   &full[st]);
        if (newc) bulk_g2s(sb + lay.c_off, a.cf + static_cast<long long>(bg) * 8 * kDstate, 8 * kDstate * 2, &full[st]);
        bulk_g2s(sb + lay.r_off, a.rblk + static_cast<long long>(u) * HPU * rstride, lay.r_bytes, &full[st]);
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
    if (!(m.flags & 1)) {
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
      s0_dot_c<DT, kBox>(sb + j * 8192, af, d, cq, acc);
      const float* rb = reinterpret_cast<const float*>(sb + lay.r_off) + j * (TP * kRStride + TP);
      const float2 rv = g < TP ? *reinterpret_cast<const float2*>(rb + g * kRStride + dout) : make_float2(0.0f, 0.0f);
      const float dec = g < TP ? rb[TP * kRStride + g] : 0.0f;
      float sc0 = 1.0f, sc1 = 1.0f;
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

template <int DT, int TP, int HPU, bool GATE>
static int launch_readout_t(const StepArgs& a, int num_sms, cudaStream_t st) {
  // as many stages as fit two CTAs per SM (>= 3), else one CTA with up to 8
  int ns = 8, ctas = 2;
  for (; ns >= 3; --ns)
    if (read_layout(DT, TP, ns, HPU).total <= 113 * 1024) break;
  if (ns < 3) {
    ctas = 1;
    for (ns = 8; ns > 2; --ns)
      if (read_layout(DT, TP, ns, HPU).total <= 225 * 1024) break;
  }
  const ReadLayout lay = read_layout(DT, TP, ns, HPU);
  CUtensorMap map;
  if (!encode_state_map(a.c, &map, HPU)) return cudaErrorInvalidValue;
  auto kern = readout_kernel<DT, TP, HPU, GATE>;
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

template <int DT>
static int launch_readout_dt(const StepArgs& a, int num_sms, cudaStream_t st) {
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  const bool pair = k8bit && a.c.hpg % 2 == 0;
  if (a.z) {
    if (a.TP == 4)
      return pair ? launch_readout_t<DT, 4, 2, true>(a, num_sms, st) : launch_readout_t<DT, 4, 1, true>(a, num_sms, st);
    return pair ? launch_readout_t<DT, 8, 2, true>(a, num_sms, st) : launch_readout_t<DT, 8, 1, true>(a, num_sms, st);
  }
  if (a.TP == 4)
    return pair ? launch_readout_t<DT, 4, 2, false>(a, num_sms, st) : launch_readout_t<DT, 4, 1, false>(a, num_sms, st);
  return pair ? launch_readout_t<DT, 8, 2, false>(a, num_sms, st) : launch_readout_t<DT, 8, 1, false>(a, num_sms, st);
}

int launch_readout(const StepArgs& a, int num_sms, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (a.c.dtype) {
    case RSSM_F32: return launch_readout_dt<RSSM_F32>(a, num_sms, st);
    case RSSM_BF16: return launch_readout_dt<RSSM_BF16>(a, num_sms, st);
    case RSSM_F16: return launch_readout_dt<RSSM_F16>(a, num_sms, st);
    case RSSM_I8: return launch_readout_dt<RSSM_I8>(a, num_sms, st);
    default: return launch_readout_dt<RSSM_E4M3>(a, num_sms, st);
  }
}

}  // namespace rssm
