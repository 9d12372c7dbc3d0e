// rssm_step.cu -- the persistent readout of the ReplaySSM checkpointing SSU
// (FlashInfer PR #3975, Description item 1: the main kernel of the two-kernel
// split), persistent over (row, head) units:
//           y_t[d] = decay[t] (S0[d] . C_t) + R[t][d]
// streaming S0 once through a multi-stage shared-memory ring filled by TMA
// (swizzled tensor boxes for S0, 1-D bulk copies for the rest) from a
// producer warp with mbarriers; 8 consumer warps contract on the tensor cores
// (mma.sync m16n8k16, f32 accumulation).  R and decay come from the
// precompute (rssm_precompute.cu).  The FOLD variant (rssm_flush_step) also
// folds the units of rows flushed in the same call.
#include "rssm_readout.cuh"

namespace rssm {

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
