// rssm_fused.cu -- rssm_flush_step: the flush and the step of one decode
// iteration in two kernels.
//
// rssm_flush followed by rssm_step runs four kernels back to back and reads a
// flagged head's checkpoint twice (fold, then readout).  In the combined call
// the precompute (rssm_step.cu, flush_mode != 0) takes the flush decision
// itself with the same rule and works on the ring as the flush leaves it --
// after a flush the new tokens land on the same ring slots as without one --
// and the kernel below takes each (row, head) unit once:
//   * a unit of a flagged row is folded in the shared-memory stage it arrived
//     in (the fold's arithmetic: canonical fp32 order, the same quantiser),
//     written back to HBM, and the rounded checkpoint is also written into
//     the stage in the TMA box layout, so the readout contracts it from there;
//   * every unit is then read out as in readout_kernel.
// The flush's bookkeeping (ring_start, pnat, epoch) is written by whichever
// CTA takes head 0 of a flagged row; nothing else in the call reads those
// words after the precompute.  Units are handed out dynamically in chunks of
// kChunk consecutive heads (a counter in scratch, zeroed by the precompute),
// since a folded unit costs two to three times a plain one.
#include "rssm_readout.cuh"

namespace rssm {

constexpr int kChunk = 4;

struct FusedMeta {
  int b, h, s, p, Tb, tok0;
  int flags;  // 1 read out, 2 fold first, 4 new C block, 8 no more work, 16 append here
  unsigned epoch;
  int r;      // ring start after the flush
};

struct FusedLayout {
  int ns, KB;
  uint32_t s0_bytes, scale_off, c_off, r_off, r_bytes, x_off, b_off, w_off, stage_bytes;
  uint32_t stages_off, uf_off, bf_off, total;
};

// one stage: S0 boxes | 8-bit scales | C block | ring term | live x rows |
// live B rows | fold weights; after the stages the fold's f32 tables
__host__ __device__ inline FusedLayout fused_layout(int dtype, int TP, int L, int ns) {
  FusedLayout f;
  f.ns = ns;
  f.KB = (L + 3) & ~3;
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
  o += f.KB * kDim * 2;
  f.b_off = o;
  o += f.KB * kDstate * 2;
  f.w_off = o;
  o += (f.KB + 4) * 4;
  f.stage_bytes = (o + 1023) & ~1023u;  // the swizzled boxes need 1024-byte alignment
  f.stages_off = 1024;                  // barriers, abort flag, per-stage metadata
  f.uf_off = f.stages_off + ns * f.stage_bytes;
  f.bf_off = f.uf_off + f.KB * kDim * 8;
  f.total = f.bf_off + f.KB * kDstate * 4 + 1024;  // + slack to align the base
  return f;
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int DT, int TP>
__global__ void __launch_bounds__(kThreads, 2)
    flush_readout_kernel(const __grid_constant__ CUtensorMap s0map, StepArgs a, int ns) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Cache& c = a.c;
  const FusedLayout lay = fused_layout(DT, TP, c.L, ns);
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  const int H = c.H, L = c.L;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 128);
  FusedMeta* meta = reinterpret_cast<FusedMeta*>(smem + 256);
  float2* uf2 = reinterpret_cast<float2*>(smem + lay.uf_off);
  float* bfv = reinterpret_cast<float*>(smem + lay.bf_off);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < ns; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // row records, C blocks, ring terms, the work counter; appends done
  pdl_trigger();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp (lane 0 issues the copies) ----------------
    const unsigned units = static_cast<unsigned>(a.batch) * static_cast<unsigned>(H);
    auto grab = [&]() -> unsigned {
      unsigned v = 0u;
      if (lane == 0) v = atomicAdd(a.work, static_cast<unsigned>(kChunk));
      return __shfl_sync(0xffffffffu, v, 0);
    };
    unsigned u = grab();
    unsigned cend = u < units ? min(u + kChunk, units) : u;
    unsigned nbase = u < units ? grab() : units;
    auto advance = [&]() {
      ++u;
      if (u >= cend) {
        u = nbase;
        if (u < units) {
          cend = min(u + kChunk, units);
          nbase = grab();
        } else {
          cend = u;
        }
      }
    };
    // one unit of lookahead: its row record and (for a fold) its live dt' and A
    struct Pre {
      unsigned u;
      int b, h;
      RowRec rr;
      float dtj, Ah;
    };
    int cached_b = -1;
    RowRec cached = {};
    auto fetch = [&](Pre& q) {
      q.u = u;
      q.dtj = 0.0f;
      q.Ah = 0.0f;
      if (u >= units) return;
      q.b = static_cast<int>(u / static_cast<unsigned>(H));
      q.h = static_cast<int>(u % static_cast<unsigned>(H));
      if (q.b != cached_b) {
        cached = a.rows[q.b];
        cached_b = q.b;
      }
      q.rr = cached;
      if (q.rr.flags & 2) {
        const int p = q.rr.p_old;
        const int r_old = q.rr.r - p < 0 ? q.rr.r - p + L : q.rr.r - p;
        const int pos = r_old + lane >= L ? r_old + lane - L : r_old + lane;
        q.dtj = lane < p ? c.dt_cache[static_cast<long long>(q.rr.s) * c.dt_stride +
                                      static_cast<long long>(q.h) * L + pos]
                         : 0.0f;
        q.Ah = a.A[q.h];
      }
    };
    Pre nx;
    fetch(nx);
    int i = 0, cur_bg = -1;
    bool ok = true;
    while (nx.u < units) {
      const Pre cu = nx;
      advance();
      fetch(nx);
      const int st = i % ns;
      const uint32_t ph = (i / ns) & 1;
      if (i >= ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
        break;
      }
      const RowRec& rr = cu.rr;
      const int b = cu.b, h = cu.h, s = rr.s, g = h / c.hpg, bg = b * c.G + g;
      const bool rd = (rr.flags & 1) && rr.Tb > 0, fo = (rr.flags & 2) != 0;
      const bool newc = rd && bg != cur_bg;
      if (rd) cur_bg = bg;
      const int p = fo ? rr.p_old : 0;
      uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
      if (fo && h == 0 && lane == 0) {  // the flush's bookkeeping, once per flagged row
        c.ring_start[s] = rr.r;
        a.pnat_rw[b] = 0;
        c.epoch[s] = rr.epoch_new;
      }
      if (rd || fo) {
        if (lane == 0) {
          const uint32_t bytes = lay.s0_bytes + (k8bit ? 256u : 0u) + (newc ? 8u * kDstate * 2 : 0u) +
                                 (rd ? lay.r_bytes : 0u) + static_cast<uint32_t>(p) * (kDim * 2 + kDstate * 2);
          mbar_expect_tx(&full[st], bytes);
#pragma unroll
          for (int bx = 0; bx < esz; ++bx) tma_load_3d(sb + bx * 8192, &s0map, bx * (128 / esz), h * kDim, s, &full[st]);
          if (k8bit)
            bulk_g2s(sb + lay.scale_off, c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim, 256,
                     &full[st]);
          if (newc)
            bulk_g2s(sb + lay.c_off, a.cf + static_cast<long long>(bg) * 8 * kDstate, 8 * kDstate * 2, &full[st]);
          if (rd)
            bulk_g2s(sb + lay.r_off, a.rblk + (static_cast<long long>(b) * H + h) * (TP * kRStride + TP), lay.r_bytes,
                     &full[st]);
          if (p > 0) {  // the live rows of the ring before the flush: at most two segments
            const int r_old = rr.r - p < 0 ? rr.r - p + L : rr.r - p;
            const uint16_t* xg = c.x_cache + static_cast<long long>(s) * c.x_stride + static_cast<long long>(h) * L * kDim;
            const uint16_t* bgp =
                c.B_cache + static_cast<long long>(s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
            const int n1 = min(p, L - r_old);
            bulk_g2s(sb + lay.x_off, xg + r_old * kDim, n1 * kDim * 2, &full[st]);
            bulk_g2s(sb + lay.b_off, bgp + r_old * kDstate, n1 * kDstate * 2, &full[st]);
            if (p > n1) {
              bulk_g2s(sb + lay.x_off + n1 * kDim * 2, xg, (p - n1) * kDim * 2, &full[st]);
              bulk_g2s(sb + lay.b_off + n1 * kDstate * 2, bgp, (p - n1) * kDstate * 2, &full[st]);
            }
          }
        }
        if (fo) {
          // canonical cumulative sums c_j (sequential fp32) and the fold weights,
          // the same operations as the flush kernel
          const float aj = lane < p ? __fmul_rn(cu.Ah, cu.dtj) : 0.0f;
          float cj = 0.0f;
          for (int k = 0; k < p; ++k) {
            const float ak = __shfl_sync(0xffffffffu, aj, k);
            if (lane >= k) cj = __fadd_rn(cj, ak);
          }
          const float c_end = p > 0 ? __shfl_sync(0xffffffffu, cj, p - 1) : 0.0f;
          float* wv = reinterpret_cast<float*>(sb + lay.w_off);
          if (lane < p) wv[lane] = __fmul_rn(spec_exp(__fsub_rn(c_end, cj)), cu.dtj);
          if (lane == 0) wv[lay.KB] = spec_exp(c_end);
        }
      }
      if (lane == 0)
        meta[st] = FusedMeta{b, h, s, p, rr.Tb, rr.tok0,
                             (rd ? 1 : 0) | (fo ? 2 : 0) | (newc ? 4 : 0) | ((rr.flags & 4) ? 16 : 0), rr.epoch_new,
                             rr.r};
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[st]);
      ++i;
    }
    if (ok) {  // end of work for the consumers
      const int st = i % ns;
      const uint32_t ph = (i / ns) & 1;
      if (i >= ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
      } else {
        if (lane == 0) meta[st] = FusedMeta{0, 0, 0, 0, 0, 0, 8, 0u, 0};
        __syncwarp();
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

  // ---------------- consumer warps: state rows 8*warp .. 8*warp+7 ----------------
  const int g = lane >> 2, cq = lane & 3;
  const int d = 8 * warp + g;          // readout: B column (row of S0) this lane loads
  const int dout = 8 * warp + 2 * cq;  // readout: output rows this lane writes
  const int r0 = 8 * warp + 4 * (lane >> 4), c0 = 8 * (lane & 15);  // fold: 4 rows x 8 columns
  uint2 af[8];
  for (int i = 0;; ++i) {
    const int st = i % ns;
    const uint32_t ph = (i / ns) & 1;
    if (!mbar_wait(&full[st], ph)) {
      *abort_flag = 1;
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
    }
    // every consumer warp passes here for every unit: the abort decision is
    // uniform, and the previous fold is done with the shared tables
    consumer_sync();
    if (*abort_flag) return;
    const FusedMeta m = meta[st];
    if (m.flags & 8) return;
    uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
    if ((m.flags & 16) && warp == 0) {
      // This row's new tokens land on live slots the fold reads, so the
      // precompute left its appends to this kernel.  The unit's live rows are
      // in the stage now: append the head's x rows and dt' (the precompute's
      // exact softplus), and once every head of the (row, group) has its
      // copy, the group's B rows.
      const int g = m.h / c.hpg;
      auto pos = [&](int t) { return m.r + t >= L ? m.r + t - L : m.r + t; };
      uint16_t* xring = c.x_cache + static_cast<long long>(m.s) * c.x_stride + static_cast<long long>(m.h) * L * kDim;
      for (int idx = lane; idx < m.Tb * 8; idx += 32) {
        const int t = idx >> 3, q = idx & 7;
        reinterpret_cast<uint4*>(xring + pos(t) * kDim)[q] =
            reinterpret_cast<const uint4*>(a.x + (static_cast<long long>(m.tok0 + t) * H + m.h) * kDim)[q];
      }
      if (lane < m.Tb)
        c.dt_cache[static_cast<long long>(m.s) * c.dt_stride + static_cast<long long>(m.h) * L + pos(lane)] =
            spec_softplus(__fadd_rn(a.dt[static_cast<long long>(m.tok0 + lane) * H + m.h], a.dt_bias[m.h]));
      unsigned landed = 0u;
      if (lane == 0) landed = atomicAdd(&a.gdone[m.b * c.G + g], 1u);
      landed = __shfl_sync(0xffffffffu, landed, 0);
      if (landed == static_cast<unsigned>(c.hpg - 1)) {
        uint16_t* bring = c.B_cache + static_cast<long long>(m.s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
        for (int idx = lane; idx < m.Tb * 16; idx += 32) {
          const int t = idx >> 4, q = idx & 15;
          reinterpret_cast<uint4*>(bring + pos(t) * kDstate)[q] =
              reinterpret_cast<const uint4*>(a.B + (static_cast<long long>(m.tok0 + t) * c.G + g) * kDstate)[q];
        }
      }
    }
    if (m.flags & 2) {
      // ---- fold: acc = e^{c_end} S0f + sum_j u_j (x) B_j, j ascending ----
      const float* wv = reinterpret_cast<const float*>(sb + lay.w_off);
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(sb + lay.x_off);
      const uint32_t* bs = reinterpret_cast<const uint32_t*>(sb + lay.b_off);
      for (int idx = tid; idx < m.p * kDim; idx += kConsumerThreads) {
        const float uu = __fmul_rn(wv[idx >> 6], bf16f(xs[idx]));
        uf2[idx] = make_float2(uu, uu);
      }
      for (int idx = tid; idx < m.p * (kDstate / 2); idx += kConsumerThreads) {
        const uint32_t wd = bs[idx];
        reinterpret_cast<float2*>(bfv)[idx] = make_float2(bf16lo(wd), bf16hi(wd));
      }
      const float decay = wv[lay.KB];
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
      consumer_sync();  // tables complete
      for (int j = 0; j < m.p; ++j) {
        const float4* up = reinterpret_cast<const float4*>(uf2 + j * kDim + r0);
        const float4 u01 = up[0], u23 = up[1];
        const float4* bp = reinterpret_cast<const float4*>(bfv + j * kDstate + c0);
        const float4 b0 = bp[0], b1 = bp[1];
        const float2 bb[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                              make_float2(b1.z, b1.w)};
        const float2 uu[4] = {make_float2(u01.x, u01.y), make_float2(u01.z, u01.w), make_float2(u23.x, u23.y),
                              make_float2(u23.z, u23.w)};
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
      // the rounded checkpoint to HBM and, in the box layout, over this
      // warp's own rows of the stage (the rows its readout contracts)
      quantize_store<DT, true>(accf, r0, c0, lane, head_state, head_scale, c.rounding, static_cast<uint32_t>(m.h),
                               static_cast<uint32_t>(m.s), m.epoch, a.seed, sb,
                               reinterpret_cast<float*>(sb + lay.scale_off));
      fence_proxy_async_smem();  // these writes precede the next copy into the stage
      __syncwarp();
    }
    float y0 = 0.0f, y1 = 0.0f;
    if (m.flags & 1) {
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
    if (m.flags & 1) {
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

template <int DT, int TP>
static int launch_flush_readout_t(const StepArgs& a, int num_sms, cudaStream_t st) {
  // as many stages (2..4) as fit two CTAs per SM, else one CTA with up to 6
  int ns = 4, ctas = 2;
  for (; ns >= 2; --ns)
    if (fused_layout(DT, TP, a.c.L, ns).total <= 113 * 1024) break;
  if (ns < 2) {
    ctas = 1;
    for (ns = 6; ns > 2; --ns)
      if (fused_layout(DT, TP, a.c.L, ns).total <= 225 * 1024) break;
  }
  const FusedLayout lay = fused_layout(DT, TP, a.c.L, ns);
  CUtensorMap map;
  if (!encode_state_map(a.c, &map)) return cudaErrorInvalidValue;
  auto kern = flush_readout_kernel<DT, TP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, lay.total);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  if (occ > ctas) occ = ctas;
  const long long chunks = (static_cast<long long>(a.batch) * a.c.H + kChunk - 1) / kChunk;
  const long long cap = static_cast<long long>(num_sms) * occ;
  const int grid = static_cast<int>(chunks < cap ? chunks : cap);
  e = launch_pdl(kern, dim3(grid), dim3(kThreads), lay.total, st, map, a, ns);
  return e != cudaSuccess ? e : cudaGetLastError();
}

int launch_flush_readout(const StepArgs& a, int num_sms, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool t4 = a.TP == 4;
  switch (a.c.dtype) {
    case RSSM_F32: return t4 ? launch_flush_readout_t<RSSM_F32, 4>(a, num_sms, st) : launch_flush_readout_t<RSSM_F32, 8>(a, num_sms, st);
    case RSSM_BF16: return t4 ? launch_flush_readout_t<RSSM_BF16, 4>(a, num_sms, st) : launch_flush_readout_t<RSSM_BF16, 8>(a, num_sms, st);
    case RSSM_F16: return t4 ? launch_flush_readout_t<RSSM_F16, 4>(a, num_sms, st) : launch_flush_readout_t<RSSM_F16, 8>(a, num_sms, st);
    case RSSM_I8: return t4 ? launch_flush_readout_t<RSSM_I8, 4>(a, num_sms, st) : launch_flush_readout_t<RSSM_I8, 8>(a, num_sms, st);
    default: return t4 ? launch_flush_readout_t<RSSM_E4M3, 4>(a, num_sms, st) : launch_flush_readout_t<RSSM_E4M3, 8>(a, num_sms, st);
  }
}

}  // namespace rssm
