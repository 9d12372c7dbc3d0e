// rssm_fused.cu -- rssm_flush_step: one decode iteration's flush and step in
// one pass over the checkpoints.
//
// rssm_flush followed by rssm_step is four kernels in a chain and reads a
// flushed head's checkpoint twice; the precompute and the flush run at a
// small fraction of the bandwidth while the readout waits for them.  Here:
//   classify_kernel  per row: the flush decision with the flush's rule and
//       checks, the ring the step works on after it (p' = 0, r' = r + p for
//       flushed rows; appends land on the same slots either way), the row
//       record, and the zeroed counters of the step kernel.
//   step_kernel      persistent over (row, head) units handed out dynamically
//       in chunks; per CTA three roles on one shared-memory stage ring:
//         producer warp  (one lane issues) S0 by TMA tensor boxes, the unit's
//             ring rows (the live prefix; for a flushed row the pre-flush
//             prefix the fold reads) and new rows of x and B, the C rows, by
//             1-D bulk copies; dt values by plain loads one unit ahead; for a
//             flushed row the fold weights (the flush kernel's operations).
//         prep warp      the step's per-unit replay terms: dt' (fixed-sequence
//             softplus), cumulative sums, C.B on the tensor cores, the decayed
//             coefficients, the ring term R and decay into the stage, the C
//             block in the readout's operand layout; then the ring appends
//             (x, dt' of the head; the group's B rows once every head of the
//             (row, group) has its copy).
//         8 consumer warps  for a flushed unit the fold of their own 8 state
//             rows (canonical fp32 order, u_j[d] formed on the fly), rounded
//             with the flush's quantiser to HBM and, in the TMA box layout,
//             back into the stage; then the tensor-core readout of the stage
//             (readout_kernel's contraction) and y.
// The flush's bookkeeping (ring_start, pnat, epoch) is written by whichever
// CTA takes head 0 of a flushed row; the step reads the row records instead.
#include "rssm_readout.cuh"

namespace rssm {

constexpr int kChunk = 4;  // units per dynamic work grab
constexpr int kPrepWarps = 2;  // take the units of alternate chunks
constexpr int kProducerWarp = kConsumerWarps, kPrepWarp0 = kConsumerWarps + 1;
constexpr int kStepThreads = (kConsumerWarps + 1 + kPrepWarps) * 32;

// ---------------------------------------------------------------------------
// classify
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) classify_kernel(StepArgs a) {
  const Cache& c = a.c;
  pdl_wait();  // pnat, ring_start and epochs as the previous call left them
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0) *a.work = 0u;
  if (b >= a.batch) return;
  for (int g = 0; g < c.G; ++g) a.gdone[static_cast<long long>(b) * c.G + g] = 0u;
  const int L = c.L;
  const int s = a.slot_idx[b], pn = a.pnat[b];
  const int tok0 = a.cu ? a.cu[b] : b * a.T;
  int Tb = a.cu ? a.cu[b + 1] - tok0 : a.T;
  int flags = 0, p = 0, r = 0;
  unsigned ep = 0u;
  const bool tb_ok = Tb >= 0 && Tb <= a.T;
  if (s >= 1 && s < c.S) {
    if (!tb_ok) {
      set_error(c.err, RSSM_ERRBIT_SEQLEN);
    } else if (pn < 0 || pn > L) {
      set_error(c.err, RSSM_ERRBIT_PNAT);  // the flush's check
    } else {
      const int r0 = c.ring_start[s];
      const bool fl = a.flush_mode == 2 || pn + Tb > c.W;
      p = fl ? 0 : pn;
      r = fl ? (r0 + pn >= L ? r0 + pn - L : r0 + pn) : r0;
      if (fl) {
        ep = c.epoch[s] + 1u;
        flags = 2;
      }
      if (p + Tb > L)
        set_error(c.err, RSSM_ERRBIT_PNAT);  // the step's check
      else
        flags |= 1;
    }
  }
  if (!tb_ok) Tb = 0;
  a.rows[b] = RowRec{s, r, p, Tb, tok0, flags, pn, ep};
}

// ---------------------------------------------------------------------------
// step kernel
// ---------------------------------------------------------------------------
struct StepMeta {
  int b, h, s, tok0;
  int Tb;     // tokens of the row (zeros are written for rows without outputs)
  int p;      // live tokens the step reads (0 after a flush)
  int pa;     // ring rows in the stage: the live prefix, or the pre-flush prefix for a fold
  int flags;  // 1 outputs, 2 fold first, 4 new (row, group) for the consumers, 8 no more work,
              // 16 x prep warp: the prep warp that takes the unit
  int r;      // ring start the appends count from
  unsigned epoch;
  int pad[6];
};

struct StepLayout {
  int ns, KX;
  uint32_t s0_bytes, scale_off, c_off, r_off, r_bytes, x_off, b_off, dt_off, sc_off, stage_bytes;
  uint32_t stages_off, prep_off, total;
};

// one stage: S0 boxes | 8-bit scales | C rows (rewritten as the C block) |
// ring term R + decay | x rows | B rows | dt values of the same rows (ring
// dt', then new dt before softplus) | A, D, dt_bias of the head; after the
// stages the prep warp's CB and coefficient tables
__host__ __device__ inline StepLayout step_layout(int dtype, int TP, int L, int Tmax, int ns) {
  StepLayout f;
  f.ns = ns;
  f.KX = (L + Tmax + 3) & ~3;  // ring rows + new rows
  const int esz = dtype == RSSM_F32 ? 4 : (dtype == RSSM_BF16 || dtype == RSSM_F16) ? 2 : 1;
  f.s0_bytes = kHeadElems * esz;
  uint32_t o = f.s0_bytes;
  f.scale_off = o;
  if (dtype == RSSM_I8 || dtype == RSSM_E4M3) o += 256;
  f.c_off = o;
  o += 8 * kDstate * 2;
  f.r_off = o;
  f.r_bytes = (TP * kRStride + TP) * 4;
  o += f.r_bytes;
  f.x_off = o;
  o += f.KX * kDim * 2;
  f.b_off = o;
  o += f.KX * kDstate * 2;
  f.dt_off = o;
  o += f.KX * 4;
  f.sc_off = o;
  o += 16;
  f.stage_bytes = (o + 1023) & ~1023u;  // the swizzled boxes need 1024-byte alignment
  f.stages_off = 1024;                  // barriers and per-stage metadata
  f.prep_off = f.stages_off + ns * f.stage_bytes;
  f.total = f.prep_off + 2 * 2 * 8 * kMaxL * 4 + 1024;  // two prep warps' tables + slack to align the base
  return f;
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int DT, int TP>
__global__ void __launch_bounds__(kStepThreads, 2)
    step_kernel(const __grid_constant__ CUtensorMap s0map, StepArgs a, int ns) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Cache& c = a.c;
  const StepLayout lay = step_layout(DT, TP, c.L, c.Tmax, ns);
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  const int H = c.H, L = c.L, G = c.G, hpg = c.hpg;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // copies landed (+ producer's dt, weights, meta)
  uint64_t* prepped = full + 8;                        // R, decay, C block written
  uint64_t* empty = full + 16;                         // consumers and the prep warps are done with the stage
  StepMeta* meta = reinterpret_cast<StepMeta*>(smem + 256);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < ns; ++st) {
      mbar_init(&full[st], 1 + 32);  // producer lane 0 + one cp.async arrival per producer lane
      mbar_init(&prepped[st], 1);
      mbar_init(&empty[st], kConsumerWarps + kPrepWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // row records and zeroed counters
  pdl_trigger();

  if (warp == kProducerWarp) {
    // ======================= producer warp =======================
    // Nothing on this warp's path waits for a global load it has just issued:
    // chunks of kChunk consecutive units come from a counter grabbed a chunk
    // ahead (with that chunk's row record), and every per-unit value is moved
    // into the stage by the copy engines or per-lane cp.async.
    const unsigned units = static_cast<unsigned>(a.batch) * static_cast<unsigned>(H);
    unsigned raw = 0u;  // lane 0: the answer of the outstanding grab
    auto request = [&]() {
      if (lane == 0) raw = atomicAdd(a.work, static_cast<unsigned>(kChunk));
    };
    request();
    unsigned u = __shfl_sync(0xffffffffu, raw, 0);
    unsigned cend = u < units ? min(u + kChunk, units) : u;
    bool pending = false;
    unsigned nu = units;
    int rec_b = -1, nrec_b = -1;
    RowRec rec = {}, nrec = {};
    if (u < units) {
      request();
      pending = true;
    }
    int i = 0, cur_bg = -1, chunk_no = 0;
    bool ok = true;
    while (u < units) {
      const int b = static_cast<int>(u / static_cast<unsigned>(H)), h = static_cast<int>(u % static_cast<unsigned>(H));
      if (b != rec_b) {  // only when the next chunk's record was not prefetched (or a chunk crosses rows)
        rec = a.rows[b];
        rec_b = b;
      }
      const int st = i % ns;
      const uint32_t ph = (i / ns) & 1;
      if (i >= ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
        break;
      }
      const RowRec rr = rec;
      const int s = rr.s, g = h / hpg;
      const bool fo = (rr.flags & 2) != 0, out = (rr.flags & 1) && rr.Tb > 0;
      const int pa = fo ? rr.p_old : rr.p;
      const int ra = fo ? (rr.r - pa < 0 ? rr.r - pa + L : rr.r - pa) : rr.r;
      const int tn = out ? rr.Tb : 0;  // new rows
      const int bg = b * G + g;
      const bool newc = out && bg != cur_bg;  // C rows (and the C.B products) change with the (row, group)
      if (out) cur_bg = bg;
      uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
      if (fo && h == 0 && lane == 0) {  // the flush's bookkeeping, once per flushed row
        c.ring_start[s] = rr.r;
        a.pnat_rw[b] = 0;
        c.epoch[s] = rr.epoch_new;
      }
      if (fo || out) {
        // lane 0: S0 (+ scales) by TMA and the ring rows of x and B (at most
        // two contiguous segments each) by 1-D bulk copies; all lanes: the new
        // rows, the C rows, the dt values and the head's scalars as cp.async
        // pieces
        const uint16_t* xg = c.x_cache + static_cast<long long>(s) * c.x_stride + static_cast<long long>(h) * L * kDim;
        const uint16_t* bgp = c.B_cache + static_cast<long long>(s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
        const float* dg = c.dt_cache + static_cast<long long>(s) * c.dt_stride + static_cast<long long>(h) * L;
        if (lane == 0) {
          mbar_expect_tx(&full[st], lay.s0_bytes + (k8bit ? 256u : 0u) + static_cast<uint32_t>(pa) * (kDim * 2 + kDstate * 2));
#pragma unroll
          for (int bx = 0; bx < esz; ++bx) tma_load_3d(sb + bx * 8192, &s0map, bx * (128 / esz), h * kDim, s, &full[st]);
          if (k8bit)
            bulk_g2s(sb + lay.scale_off, c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim, 256,
                     &full[st]);
          if (pa > 0) {
            const int n1 = min(pa, L - ra);
            bulk_g2s(sb + lay.x_off, xg + ra * kDim, n1 * kDim * 2, &full[st]);
            bulk_g2s(sb + lay.b_off, bgp + ra * kDstate, n1 * kDstate * 2, &full[st]);
            if (pa > n1) {
              bulk_g2s(sb + lay.x_off + n1 * kDim * 2, xg, (pa - n1) * kDim * 2, &full[st]);
              bulk_g2s(sb + lay.b_off + n1 * kDstate * 2, bgp, (pa - n1) * kDstate * 2, &full[st]);
            }
          }
          float* scl = reinterpret_cast<float*>(sb + lay.sc_off);
          cp_async4(scl, a.A + h);
          cp_async4(scl + 1, a.D + h);
          cp_async4(scl + 2, a.dt_bias + h);
        }
        for (int q = lane; q < tn * 8; q += 32) {
          const int t = q >> 3, part = q & 7;
          cp_async16(sb + lay.x_off + (pa + t) * kDim * 2 + part * 16,
                     a.x + (static_cast<long long>(rr.tok0 + t) * H + h) * kDim + part * 8);
        }
        for (int q = lane; q < tn * 16; q += 32) {
          const int t = q >> 4, part = q & 15;
          const long long row = (static_cast<long long>(rr.tok0 + t) * G + g) * kDstate + part * 8;
          cp_async16(sb + lay.b_off + (pa + t) * kDstate * 2 + part * 16, a.B + row);
          cp_async16(sb + lay.c_off + t * kDstate * 2 + part * 16, a.C + row);
        }
        for (int k = lane; k < pa + tn; k += 32) {
          const float* src = k < pa ? dg + (ra + k >= L ? ra + k - L : ra + k)
                                    : a.dt + static_cast<long long>(rr.tok0 + k - pa) * H + h;
          cp_async4(sb + lay.dt_off + k * 4, src);
        }
      }
      cp_async_arrive_noinc(&full[st]);
      if (lane == 0)
        meta[st] = StepMeta{b, h, s, rr.tok0, rr.Tb, rr.p, pa,
                            (out ? 1 : 0) | (fo ? 2 : 0) | (newc ? 4 : 0) | (chunk_no % kPrepWarps) * 16, rr.r,
                            rr.epoch_new, {0, 0, 0, 0, 0, 0}};
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
      ++i;
      // the next unit; the next chunk's index (and then its row record) were
      // requested a chunk ahead
      ++u;
      if (pending) {
        nu = __shfl_sync(0xffffffffu, raw, 0);
        pending = false;
        if (nu < units) {
          nrec_b = static_cast<int>(nu / static_cast<unsigned>(H));
          nrec = a.rows[nrec_b];
        }
      }
      if (u >= cend) {
        u = nu;
        if (u < units) {
          cend = min(u + kChunk, units);
          rec = nrec;
          rec_b = nrec_b;
          request();
          pending = true;
          ++chunk_no;
        } else {
          cend = u;
        }
      }
    }
    if (ok) {  // end of work for the other roles
      const int st = i % ns;
      const uint32_t ph = (i / ns) & 1;
      if (i >= ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
      } else {
        if (lane == 0) meta[st].flags = 8;
        __syncwarp();
        cp_async_arrive_noinc(&full[st]);
        if (lane == 0) mbar_arrive(&full[st]);
      }
    }
    if (!ok) {
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      // let copies already in flight land before the CTA can exit
      for (int k = max(0, i - ns); k < i; ++k) mbar_wait(&full[k % ns], (k / ns) & 1);
    }
    return;
  }

  if (warp >= kPrepWarp0) {
    // ======================= prep warps =======================
    // Both read every unit's metadata and release every stage; the one named
    // in the unit's flags does the work.
    const int pw = warp - kPrepWarp0;
    float* cbs = reinterpret_cast<float*>(smem + lay.prep_off) + pw * 2 * 8 * kMaxL;  // CB[t][k], [8][32]
    float* cfs = cbs + 8 * kMaxL;                                                    // coef[k][t], [32][TP]
    int my_bg = -1;  // the (row, group) this warp's CB belongs to
    const int g8 = lane >> 2, c4 = lane & 3;
    const bool c_f16 = DT == RSSM_F16 || DT == RSSM_I8 || DT == RSSM_E4M3;
    // the B rows of a (row, group) are appended by the last of its heads to
    // have its ring rows in a stage; the counter's answer is read one unit
    // later, the rows come from the step's inputs
    unsigned pend_landed = 0u;
    int pend = 0, pend_s = 0, pend_g = 0, pend_r = 0, pend_Tb = 0, pend_tok0 = 0;
    auto finish_b = [&]() {
      if (!pend) return;
      const unsigned landed = __shfl_sync(0xffffffffu, pend_landed, 0);
      if (landed == static_cast<unsigned>(hpg - 1)) {
        uint16_t* bring = c.B_cache + static_cast<long long>(pend_s) * c.B_stride + static_cast<long long>(pend_g) * L * kDstate;
        for (int idx = lane; idx < pend_Tb * 16; idx += 32) {
          const int t = idx >> 4, q = idx & 15;
          const int ps = pend_r + t >= L ? pend_r + t - L : pend_r + t;
          reinterpret_cast<uint4*>(bring + ps * kDstate)[q] =
              reinterpret_cast<const uint4*>(a.B + (static_cast<long long>(pend_tok0 + t) * G + pend_g) * kDstate)[q];
        }
      }
      pend = 0;
    };
    for (int i = 0;; ++i) {
      const int st = i % ns;
      const uint32_t ph = (i / ns) & 1;
      if (!mbar_wait(&full[st], ph)) {
        if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
        return;
      }
      finish_b();  // the previous unit's group B rows (also after the last unit)
      const StepMeta m = meta[st];
      if (m.flags & 8) return;
      uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
      if (((m.flags >> 4) & (kPrepWarps - 1)) != pw) {  // the other prep warp's unit
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        continue;
      }
      if (m.flags & 1) {
        const int p = m.p, Tb = m.Tb, K = p + Tb;
        const int base = m.pa - p;  // stage row of logical token 0 (past the fold's rows)
        const float* scl = reinterpret_cast<const float*>(sb + lay.sc_off);
        const float hA = scl[0], hD = scl[1], hbias = scl[2];
        // dt' of the readout tokens: live values as stored, new ones through
        // the fixed-sequence softplus (the values the ring gets); inclusive
        // prefix sums of A dt' (these feed the outputs only: any order)
        float dtv = 0.0f;
        if (lane < K) {
          const float v = reinterpret_cast<const float*>(sb + lay.dt_off)[base + lane];
          dtv = lane < p ? v : spec_softplus(__fadd_rn(v, hbias));
        }
        float cum = lane < K ? hA * dtv : 0.0f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float x = __shfl_up_sync(0xffffffffu, cum, off);
          if (lane >= off) cum += x;
        }
        uint32_t* crow = reinterpret_cast<uint32_t*>(sb + lay.c_off);
        const int bgm = m.b * G + m.h / hpg;
        if (bgm != my_bg) {
          // a new (row, group) for this warp: C.B on the tensor cores (M = t,
          // rows >= T_b zero; N = k, four 8-token tiles as independent chains;
          // K = dstate)
          my_bg = bgm;
          const uint32_t* brow = reinterpret_cast<const uint32_t*>(sb + lay.b_off) + base * (kDstate / 2);
          float d4[4][4];
#pragma unroll
          for (int j = 0; j < 4; ++j) d4[j][0] = d4[j][1] = d4[j][2] = d4[j][3] = 0.0f;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t a0 = g8 < Tb ? crow[g8 * 64 + 8 * ks + c4] : 0u;
            const uint32_t a2 = g8 < Tb ? crow[g8 * 64 + 8 * ks + 4 + c4] : 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (j * 8 < K) {
                const int kr = j * 8 + g8 < K ? j * 8 + g8 : K - 1;
                mma_bf16(d4[j], a0, a2, brow[kr * 64 + 8 * ks + c4], brow[kr * 64 + 8 * ks + 4 + c4]);
              }
            }
          }
          if (g8 < TP) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              cbs[g8 * kMaxL + j * 8 + 2 * c4] = d4[j][0];
              cbs[g8 * kMaxL + j * 8 + 2 * c4 + 1] = d4[j][1];
            }
          }
        }
        if (m.flags & 4) {
          // a new (row, group) for the consumers: the C block in the readout's
          // operand layout in place of the C rows: rows t >= T_b zero, fp16
          // for the fp16-type MMA, 32-byte quad j of row t stored at quad j ^ t
          uint32_t cw[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int idx = lane + 32 * e, t = idx >> 6;
            uint32_t w = t < Tb ? crow[idx] : 0u;
            if (c_f16) {
              const __half2 hv = __floats2half2_rn(bf16lo(w), bf16hi(w));
              w = *reinterpret_cast<const uint32_t*>(&hv);
            }
            cw[e] = w;
          }
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int idx = lane + 32 * e, t = idx >> 6, n = 2 * (idx & 63);
            crow[(t * kDstate + 16 * (((n >> 4) ^ t) & 7) + (n & 15)) >> 1] = cw[e];
          }
          __syncwarp();
        }
        // coefficients coef[k][t] = e^{c_{p+t} - c_k} dt'_k CB[t][k] (+ D on k = p + t), decay
        float cf[TP], dec[TP];
#pragma unroll
        for (int t = 0; t < TP; ++t) {
          const float cpt = __shfl_sync(0xffffffffu, cum, p + t < 31 ? p + t : 31);
          float v = 0.0f;
          if (t < Tb && lane <= p + t) {
            v = __expf(cpt - cum) * dtv * cbs[t * kMaxL + lane];
            if (lane == p + t) v += hD;
          }
          cf[t] = v;
          dec[t] = t < Tb ? __expf(cpt) : 0.0f;
        }
#pragma unroll
        for (int t4 = 0; t4 < TP; t4 += 4)
          *reinterpret_cast<float4*>(&cfs[lane * TP + t4]) = make_float4(cf[t4], cf[t4 + 1], cf[t4 + 2], cf[t4 + 3]);
        __syncwarp();
        // ring term R[t][d] = sum_k coef[k][t] x_k[d], lane l: d = 2l, 2l + 1
        float2 R[TP];
#pragma unroll
        for (int t = 0; t < TP; ++t) R[t] = make_float2(0.0f, 0.0f);
        const uint32_t* xr = reinterpret_cast<const uint32_t*>(sb + lay.x_off) + base * (kDim / 2) + lane;
#pragma unroll 4
        for (int k = 0; k < K; ++k) {
          const uint32_t w = xr[k * (kDim / 2)];
          const float2 xv = make_float2(bf16lo(w), bf16hi(w));
#pragma unroll
          for (int t4 = 0; t4 < TP; t4 += 4) {
            const float4 cv = *reinterpret_cast<const float4*>(&cfs[k * TP + t4]);
            R[t4 + 0] = __ffma2_rn(make_float2(cv.x, cv.x), xv, R[t4 + 0]);
            R[t4 + 1] = __ffma2_rn(make_float2(cv.y, cv.y), xv, R[t4 + 1]);
            R[t4 + 2] = __ffma2_rn(make_float2(cv.z, cv.z), xv, R[t4 + 2]);
            R[t4 + 3] = __ffma2_rn(make_float2(cv.w, cv.w), xv, R[t4 + 3]);
          }
        }
        float* rb = reinterpret_cast<float*>(sb + lay.r_off);
#pragma unroll
        for (int t = 0; t < TP; ++t) reinterpret_cast<float2*>(rb + t * kRStride)[lane] = R[t];
        if (lane == 0) {
#pragma unroll
          for (int t4 = 0; t4 < TP; t4 += 4)
            *reinterpret_cast<float4*>(rb + TP * kRStride + t4) = make_float4(dec[t4], dec[t4 + 1], dec[t4 + 2], dec[t4 + 3]);
        }
        fence_proxy_async_smem();  // these stage writes precede the next copy into the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&prepped[st]);
        // ring appends at (r + p + t) mod L: the head's x rows and dt' now (its
        // ring rows are in the stage), the group's B rows as described above
        const int g = m.h / hpg;
        const int r1 = m.r + p >= L ? m.r + p - L : m.r + p;
        uint16_t* xring = c.x_cache + static_cast<long long>(m.s) * c.x_stride + static_cast<long long>(m.h) * L * kDim;
        const uint4* xnew = reinterpret_cast<const uint4*>(sb + lay.x_off + m.pa * kDim * 2);
        for (int idx = lane; idx < Tb * 8; idx += 32) {
          const int t = idx >> 3, ps = r1 + t >= L ? r1 + t - L : r1 + t;
          reinterpret_cast<uint4*>(xring + ps * kDim)[idx & 7] = xnew[idx];
        }
        const float dnew = __shfl_sync(0xffffffffu, dtv, (p + lane) & 31);
        if (lane < Tb) {
          const int ps = r1 + lane >= L ? r1 + lane - L : r1 + lane;
          c.dt_cache[static_cast<long long>(m.s) * c.dt_stride + static_cast<long long>(m.h) * L + ps] = dnew;
        }
        if (lane == 0) pend_landed = atomicAdd(&a.gdone[static_cast<long long>(m.b) * G + g], 1u);
        pend = 1;
        pend_s = m.s;
        pend_g = g;
        pend_r = r1;
        pend_Tb = Tb;
        pend_tok0 = m.tok0;
        __syncwarp();
      } else {
        if (lane == 0) mbar_arrive(&prepped[st]);
      }
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }

  // ======================= consumer warps: state rows 8*warp .. 8*warp+7 =======================
  const int g = lane >> 2, cq = lane & 3;
  const int d = 8 * warp + g;          // readout: row of S0 this lane loads
  const int dout = 8 * warp + 2 * cq;  // readout: output rows this lane writes
  const int r0 = 8 * warp + 4 * (lane >> 4), c0 = 8 * (lane & 15);  // fold: 4 rows x 8 columns
  uint2 af[8];
  for (int i = 0;; ++i) {
    const int st = i % ns;
    const uint32_t ph = (i / ns) & 1;
    if (!mbar_wait(&full[st], ph)) {
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      return;
    }
    const StepMeta m = meta[st];
    if (m.flags & 8) return;
    uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
    if (m.flags & 2) {
      // ---- fold of this warp's rows: acc = e^{c_end} S0f; then for j
      // ascending acc = fma(u_j[d], B_j[n], acc), u_j[d] = w_j x_j[d] ----
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(sb + lay.x_off);
      const uint16_t* bs = reinterpret_cast<const uint16_t*>(sb + lay.b_off);
      // canonical cumulative sums c_j (sequential fp32) over the pre-flush
      // prefix and the fold weights w_j = e^{c_end - c_j} dt'_j, the flush
      // kernel's operations (lane j holds w_j)
      const int pa = m.pa;
      const float hA = reinterpret_cast<const float*>(sb + lay.sc_off)[0];
      const float dtj = lane < pa ? reinterpret_cast<const float*>(sb + lay.dt_off)[lane] : 0.0f;
      const float aj = lane < pa ? __fmul_rn(hA, dtj) : 0.0f;
      float cj = 0.0f;
      for (int k = 0; k < pa; ++k) {
        const float ak = __shfl_sync(0xffffffffu, aj, k);
        if (lane >= k) cj = __fadd_rn(cj, ak);
      }
      const float c_end = pa > 0 ? __shfl_sync(0xffffffffu, cj, pa - 1) : 0.0f;
      const float wj = lane < pa ? __fmul_rn(spec_exp(__fsub_rn(c_end, cj)), dtj) : 0.0f;
      const float decay = spec_exp(c_end);
      float2 acc[4][4];
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const int row = r0 + i4;
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
            const uint32_t byte = ((e < 4 ? q.x : q.y) >> (8 * (e & 3))) & 0xffu;
            const float code = DT == RSSM_I8 ? static_cast<float>(static_cast<int8_t>(byte)) : e4m3_to_f32(byte);
            v[e] = __fmul_rn(code, sc);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          acc[i4][q] = make_float2(__fmul_rn(decay, v[2 * q]), __fmul_rn(decay, v[2 * q + 1]));
      }
      for (int j = 0; j < pa; ++j) {
        const float w = __shfl_sync(0xffffffffu, wj, j);
        const uint2 xw = *reinterpret_cast<const uint2*>(xs + j * kDim + r0);
        const float u0 = __fmul_rn(w, bf16lo(xw.x)), u1 = __fmul_rn(w, bf16hi(xw.x));
        const float u2 = __fmul_rn(w, bf16lo(xw.y)), u3 = __fmul_rn(w, bf16hi(xw.y));
        const uint4 bw = *reinterpret_cast<const uint4*>(bs + j * kDstate + c0);
        const float2 bb[4] = {make_float2(bf16lo(bw.x), bf16hi(bw.x)), make_float2(bf16lo(bw.y), bf16hi(bw.y)),
                              make_float2(bf16lo(bw.z), bf16hi(bw.z)), make_float2(bf16lo(bw.w), bf16hi(bw.w))};
        const float2 uu[4] = {make_float2(u0, u0), make_float2(u1, u1), make_float2(u2, u2), make_float2(u3, u3)};
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[i4][q] = __ffma2_rn(uu[i4], bb[q], acc[i4][q]);
      }
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
      // the rounded checkpoint to HBM and, in the box layout, over this warp's
      // own rows of the stage (the rows its readout contracts)
      quantize_store<DT, true>(accf, r0, c0, lane, head_state, head_scale, c.rounding, static_cast<uint32_t>(m.h),
                               static_cast<uint32_t>(m.s), m.epoch, a.seed, sb,
                               reinterpret_cast<float*>(sb + lay.scale_off));
      fence_proxy_async_smem();  // these writes precede the next copy into the stage
      __syncwarp();
    }
    float y0 = 0.0f, y1 = 0.0f;
    const bool out = (m.flags & 1) != 0;
    if (out) {
      if (!mbar_wait(&prepped[st], ph)) {
        if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
        return;
      }
      if (m.flags & 4) load_c_frags(reinterpret_cast<const uint16_t*>(sb + lay.c_off), g, cq, af);
      float acc[4];
      s0_dot_c<DT>(sb, af, d, cq, acc);
      const float* rb = reinterpret_cast<const float*>(sb + lay.r_off);
      const float2 rv = g < TP ? *reinterpret_cast<const float2*>(rb + g * kRStride + dout) : make_float2(0.0f, 0.0f);
      const float dec = g < TP ? rb[TP * kRStride + g] : 0.0f;
      float sc0 = 1.0f, sc1 = 1.0f;
      if constexpr (k8bit) {
        const float2 scv = *reinterpret_cast<const float2*>(sb + lay.scale_off + dout * 4);
        sc0 = scv.x;
        sc1 = scv.y;
      }
      y0 = fmaf(dec * sc0, acc[0], rv.x);
      y1 = fmaf(dec * sc1, acc[1], rv.y);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
    if (out) {
      if (g < m.Tb) {
        const __nv_bfloat162 yv = __floats2bfloat162_rn(y0, y1);
        *reinterpret_cast<__nv_bfloat162*>(a.out + (static_cast<long long>(m.tok0 + g) * H + m.h) * kDim + dout) = yv;
      }
    } else {
      // a row without outputs (padding slot, rejected row): zeros for its tokens
      for (int idx = lane; idx < m.Tb * 4; idx += 32) {
        const int t = idx >> 2, q = idx & 3;
        *reinterpret_cast<uint32_t*>(a.out + (static_cast<long long>(m.tok0 + t) * H + m.h) * kDim + 8 * warp +
                                     2 * q) = 0u;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
int launch_classify(const StepArgs& a, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = (a.batch + 127) / 128;
  cudaError_t e = launch_pdl(classify_kernel, dim3(grid), dim3(128), 0, st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DT, int TP>
static int launch_step_t(const StepArgs& a, int num_sms, cudaStream_t st) {
  // as many stages (2..4) as fit two CTAs per SM, else one CTA with up to 6
  int ns = 4, ctas = 2;
  for (; ns >= 2; --ns)
    if (step_layout(DT, TP, a.c.L, a.c.Tmax, ns).total <= 113 * 1024) break;
  if (ns < 2) {
    ctas = 1;
    for (ns = 6; ns > 2; --ns)
      if (step_layout(DT, TP, a.c.L, a.c.Tmax, ns).total <= 225 * 1024) break;
  }
  const StepLayout lay = step_layout(DT, TP, a.c.L, a.c.Tmax, ns);
  CUtensorMap map;
  if (!encode_state_map(a.c, &map)) return cudaErrorInvalidValue;
  auto kern = step_kernel<DT, TP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kStepThreads, lay.total);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  if (occ > ctas) occ = ctas;
  const long long chunks = (static_cast<long long>(a.batch) * a.c.H + kChunk - 1) / kChunk;
  const long long cap = static_cast<long long>(num_sms) * occ;
  const int grid = static_cast<int>(chunks < cap ? chunks : cap);
  e = launch_pdl(kern, dim3(grid), dim3(kStepThreads), lay.total, st, map, a, ns);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int launch_flush_step(const StepArgs& a, int num_sms, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool t4 = a.TP == 4;
  switch (a.c.dtype) {
    case RSSM_F32: return t4 ? launch_step_t<RSSM_F32, 4>(a, num_sms, st) : launch_step_t<RSSM_F32, 8>(a, num_sms, st);
    case RSSM_BF16: return t4 ? launch_step_t<RSSM_BF16, 4>(a, num_sms, st) : launch_step_t<RSSM_BF16, 8>(a, num_sms, st);
    case RSSM_F16: return t4 ? launch_step_t<RSSM_F16, 4>(a, num_sms, st) : launch_step_t<RSSM_F16, 8>(a, num_sms, st);
    case RSSM_I8: return t4 ? launch_step_t<RSSM_I8, 4>(a, num_sms, st) : launch_step_t<RSSM_I8, 8>(a, num_sms, st);
    default: return t4 ? launch_step_t<RSSM_E4M3, 4>(a, num_sms, st) : launch_step_t<RSSM_E4M3, 8>(a, num_sms, st);
  }
}

}  // namespace rssm
