// rssm_step.cu -- replay/readout of the ReplaySSM checkpointing SSU.
//
// Two kernels, the split of FlashInfer PR #3975 (Description item 1):
//   precompute_kernel  one CTA per (row, group): dt' = softplus(dt + dt_bias)
//       for the new tokens (appended to the dt ring), the cumulative sums
//       c_k = sum_{i<=k} A dt'_i over live ring + new tokens (recomputed, not
//       cached: Description item 2), the C.B contraction CB[t][k] = C_t . B_k
//       once per group, and per head the replay coefficients
//           coef[k][t] = e^{c_{p+t} - c_k} dt'_k CB[t][k]  (+ D on k = p+t)
//       plus decay[t] = e^{c_{p+t}}, written to scratch.  Appends B.
//   readout_kernel  persistent, one (row, head) unit at a time:
//           y_t[d] = decay[t] (S0[d] . C_t) + sum_k coef[k][t] x_k[d]
//       streaming S0 once through a multi-stage shared-memory ring filled by
//       1-D bulk copies (producer warp + mbarriers); 8 consumer warps, 8 lanes
//       per state row pair, packed f32x2 FMAs over dstate, warp-shuffle
//       transpose-reduction over the 8 lanes.  Appends x.
#include <cuda_runtime.h>

#include "rssm_device.cuh"

namespace rssm {

// ---------------------------------------------------------------------------
// precompute
// ---------------------------------------------------------------------------
// swizzled 16-byte chunk index of a converted f32 C row: keeps the lanes of a
// quarter warp of the readout on distinct bank groups for every state layout
__host__ __device__ __forceinline__ int cswz(int m) { return m ^ ((m >> 3) & 3); }

template <int TP>
__global__ void __launch_bounds__(256) precompute_kernel(StepArgs a) {
  __shared__ float Bf[kMaxL][kDstate + 4];
  __shared__ float Cf[TP][kDstate + 4];
  __shared__ float CB[TP][kMaxL];
  __shared__ float dtl[16][kMaxL];  // live dt' of up to 16 heads of the group
  __shared__ int meta[6];
  const Cache& c = a.c;
  const int b = blockIdx.x / c.G, g = blockIdx.x % c.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    const int s = a.slot_idx[b];
    int Tb = a.cu ? a.cu[b + 1] - a.cu[b] : a.T;
    const int tok0 = a.cu ? a.cu[b] : b * a.T;
    int flags = 0, p = 0, r = 0;
    const bool tb_ok = Tb >= 0 && Tb <= a.T;
    if (s >= 1 && s < c.S) {
      if (!tb_ok) {
        if (g == 0) set_error(c.err, RSSM_ERRBIT_SEQLEN);
      } else {
        p = a.pnat[b];
        if (p < 0 || p + Tb > c.L) {
          if (g == 0) set_error(c.err, RSSM_ERRBIT_PNAT);
        } else {
          r = c.ring_start[s];
          flags = 1;
        }
      }
    }
    if (!tb_ok) Tb = 0;
    meta[0] = s; meta[1] = r; meta[2] = p; meta[3] = Tb; meta[4] = tok0; meta[5] = flags;
    if (g == 0) a.rows[b] = RowRec{s, r, p, Tb, tok0, flags, {0, 0}};
  }
  __syncthreads();
  const int s = meta[0], r = meta[1], p = meta[2], Tb = meta[3], tok0 = meta[4];
  if (!meta[5] || Tb == 0) return;
  const int K = p + Tb, L = c.L, H = c.H, G = c.G, hpg = c.hpg;
  uint16_t* bring = c.B_cache + static_cast<long long>(s) * c.B_stride + static_cast<long long>(g) * L * kDstate;
  // independent loads first: B rows (live ring + new), C rows, live dt' of the group's heads
  for (int idx = tid; idx < K * (kDstate / 2); idx += 256) {
    const int k = idx >> 6, q = idx & 63;
    const uint16_t* src = k < p ? bring + ((r + k) % L) * kDstate
                                : a.B + (static_cast<long long>(tok0 + k - p) * G + g) * kDstate;
    const uint32_t w = reinterpret_cast<const uint32_t*>(src)[q];
    Bf[k][2 * q] = bf16lo(w);
    Bf[k][2 * q + 1] = bf16hi(w);
  }
  for (int idx = tid; idx < TP * (kDstate / 2); idx += 256) {
    const int t = idx >> 6, q = idx & 63;
    float2 v = make_float2(0.0f, 0.0f);
    if (t < Tb) {
      const uint32_t w =
          reinterpret_cast<const uint32_t*>(a.C + (static_cast<long long>(tok0 + t) * G + g) * kDstate)[q];
      v = make_float2(bf16lo(w), bf16hi(w));
    }
    Cf[t][2 * q] = v.x;
    Cf[t][2 * q + 1] = v.y;
  }
  const int hl = hpg < 16 ? hpg : 16;
  for (int idx = tid; idx < hl * p; idx += 256) {
    const int hh = idx / p, k = idx % p;
    dtl[hh][k] = c.dt_cache[static_cast<long long>(s) * c.dt_stride + static_cast<long long>(g * hpg + hh) * L +
                            (r + k) % L];
  }
  // ring appends: the new B rows (once per group) and the new x rows of the group's heads
  for (int idx = tid; idx < Tb * 16; idx += 256) {
    const int t = idx >> 4, q = idx & 15;
    const uint4 v = reinterpret_cast<const uint4*>(a.B + (static_cast<long long>(tok0 + t) * G + g) * kDstate)[q];
    reinterpret_cast<uint4*>(bring + ((r + p + t) % L) * kDstate)[q] = v;
  }
  for (int idx = tid; idx < Tb * hpg * 8; idx += 256) {
    const int t = idx / (hpg * 8), rem = idx % (hpg * 8), hh = rem >> 3, q = rem & 7;
    const int h = g * hpg + hh;
    const uint4 v = reinterpret_cast<const uint4*>(a.x + (static_cast<long long>(tok0 + t) * H + h) * kDim)[q];
    uint16_t* dst = c.x_cache + static_cast<long long>(s) * c.x_stride + (static_cast<long long>(h) * L + (r + p + t) % L) * kDim;
    reinterpret_cast<uint4*>(dst)[q] = v;
  }
  __syncthreads();
  // C.B contraction, one warp per (t, k) pair, lanes over dstate
  for (int pr = warp; pr < Tb * K; pr += 8) {
    const int t = pr / K, k = pr % K;
    float v = 0.0f;
    if (k <= p + t) {
#pragma unroll
      for (int n = lane; n < kDstate; n += 32) v = fmaf(Cf[t][n], Bf[k][n], v);
#pragma unroll
      for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    }
    if (lane == 0) CB[t][k] = v;
  }
  // the f32 C block for the readout, 16-byte chunks swizzled
  float* cfg = a.cf + (static_cast<long long>(b) * G + g) * TP * kDstate;
  for (int idx = tid; idx < TP * 32; idx += 256) {
    const int t = idx >> 5, m = idx & 31;
    const float4 v = make_float4(Cf[t][4 * m], Cf[t][4 * m + 1], Cf[t][4 * m + 2], Cf[t][4 * m + 3]);
    *reinterpret_cast<float4*>(cfg + t * kDstate + cswz(m) * 4) = v;
  }
  __syncthreads();
  const int KB = a.KB;
  for (int hh = warp; hh < hpg; hh += 8) {
    const int h = g * hpg + hh;
    const float Ah = a.A[h], Dh = a.D[h];
    float* dtrow = c.dt_cache + static_cast<long long>(s) * c.dt_stride + static_cast<long long>(h) * L;
    float dtp = 0.0f;
    if (lane < p) {
      dtp = hh < 16 ? dtl[hh][lane] : dtrow[(r + lane) % L];
    } else if (lane < K) {
      const int t = lane - p;
      const float v = __fadd_rn(a.dt[static_cast<long long>(tok0 + t) * H + h], a.dt_bias[h]);
      dtp = spec_softplus(v);
      dtrow[(r + p + t) % L] = dtp;
    }
    const float ak = __fmul_rn(Ah, dtp);
    float cum = 0.0f;
    for (int k = 0; k < K; ++k) {
      const float x = __shfl_sync(0xffffffffu, ak, k);
      if (lane >= k) cum = __fadd_rn(cum, x);
    }
    float cf[TP];
    float dec[TP];
#pragma unroll
    for (int t = 0; t < TP; ++t) {
      const int kt = p + t < 31 ? p + t : 31;
      const float cpt = __shfl_sync(0xffffffffu, cum, kt);
      float v = 0.0f;
      if (t < Tb && lane <= p + t) {
        v = expf(cpt - cum) * dtp * CB[t][lane];
        if (lane == p + t) v += Dh;
      }
      cf[t] = v;
      dec[t] = t < Tb ? expf(cpt) : 0.0f;
    }
    float* blk = a.coef + (static_cast<long long>(b) * H + h) * (KB + 1) * TP;
    if (lane < KB) {
#pragma unroll
      for (int t4 = 0; t4 < TP; t4 += 4)
        *reinterpret_cast<float4*>(blk + lane * TP + t4) = make_float4(cf[t4], cf[t4 + 1], cf[t4 + 2], cf[t4 + 3]);
    }
    if (lane == 0) {
#pragma unroll
      for (int t4 = 0; t4 < TP; t4 += 4)
        *reinterpret_cast<float4*>(blk + KB * TP + t4) = make_float4(dec[t4], dec[t4 + 1], dec[t4 + 2], dec[t4 + 3]);
    }
  }
}

// ---------------------------------------------------------------------------
// readout
// ---------------------------------------------------------------------------
struct ReadMeta {
  int b, h, s, r, p, Tb, tok0, flags;
};

struct ReadLayout {
  int ns, KB;
  uint32_t s0_bytes, scale_off, c_off, coef_off, x_off, stage_bytes;
  uint32_t stages_off, total;
};

__host__ __device__ inline ReadLayout read_layout(int dtype, int L, int TP, int ns) {
  ReadLayout f;
  f.ns = ns;
  f.KB = (L + 3) & ~3;
  const int esz = dtype == RSSM_F32 ? 4 : (dtype == RSSM_BF16 || dtype == RSSM_F16) ? 2 : 1;
  f.s0_bytes = kHeadElems * esz;
  uint32_t o = f.s0_bytes;
  f.scale_off = o;
  if (dtype == RSSM_I8 || dtype == RSSM_E4M3) o += 256;
  f.c_off = o;
  o += TP * kDstate * 4;
  f.coef_off = o;
  o += ((f.KB + 1) * TP * 4 + 15) & ~15;
  f.x_off = o;
  o += f.KB * kDim * 2;
  f.stage_bytes = (o + 127) & ~127u;
  f.stages_off = 512;
  f.total = f.stages_off + ns * f.stage_bytes;
  return f;
}

template <int DT>
struct RowChunk;  // 16 bytes of one state row -> float pairs

template <>
struct RowChunk<RSSM_F32> {
  static constexpr int kPairs = 2;
  __device__ __forceinline__ static void get(const uint4& q, float2 (&v)[2]) {
    v[0] = make_float2(__uint_as_float(q.x), __uint_as_float(q.y));
    v[1] = make_float2(__uint_as_float(q.z), __uint_as_float(q.w));
  }
};
template <>
struct RowChunk<RSSM_BF16> {
  static constexpr int kPairs = 4;
  __device__ __forceinline__ static void get(const uint4& q, float2 (&v)[4]) {
    v[0] = make_float2(bf16lo(q.x), bf16hi(q.x));
    v[1] = make_float2(bf16lo(q.y), bf16hi(q.y));
    v[2] = make_float2(bf16lo(q.z), bf16hi(q.z));
    v[3] = make_float2(bf16lo(q.w), bf16hi(q.w));
  }
};
template <>
struct RowChunk<RSSM_F16> {
  static constexpr int kPairs = 4;
  __device__ __forceinline__ static void get(const uint4& q, float2 (&v)[4]) {
    v[0] = h2f2(q.x);
    v[1] = h2f2(q.y);
    v[2] = h2f2(q.z);
    v[3] = h2f2(q.w);
  }
};
__device__ __forceinline__ float i8f(uint32_t x, int k) {
  // byte k of x (sign bit flipped) placed under exponent 2^23, minus 2^23 + 128
  return __uint_as_float(__byte_perm(x, 0x4B000000u, k | (4 << 4) | (5 << 8) | (7 << 12))) - 8388736.0f;
}
template <>
struct RowChunk<RSSM_I8> {
  static constexpr int kPairs = 8;
  __device__ __forceinline__ static void get(const uint4& q, float2 (&v)[8]) {
    const uint32_t w[4] = {q.x ^ 0x80808080u, q.y ^ 0x80808080u, q.z ^ 0x80808080u, q.w ^ 0x80808080u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = make_float2(i8f(w[i], 0), i8f(w[i], 1));
      v[2 * i + 1] = make_float2(i8f(w[i], 2), i8f(w[i], 3));
    }
  }
};
template <>
struct RowChunk<RSSM_E4M3> {
  static constexpr int kPairs = 8;
  __device__ __forceinline__ static void get(const uint4& q, float2 (&v)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xffffu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
      v[2 * i] = __half22float2(__half2(lo));
      v[2 * i + 1] = __half22float2(__half2(hi));
    }
  }
};

// 96 registers: two 9-warp CTAs then fit the per-SMSP register files
template <int DT, int TP>
__global__ void __maxnreg__(96) readout_kernel(StepArgs a, int ns) {
  extern __shared__ __align__(128) uint8_t smem[];
  const Cache& c = a.c;
  const ReadLayout lay = read_layout(DT, c.L, TP, ns);
  constexpr int esz = DT == RSSM_F32 ? 4 : (DT == RSSM_BF16 || DT == RSSM_F16) ? 2 : 1;
  constexpr bool k8bit = DT == RSSM_I8 || DT == RSSM_E4M3;
  constexpr int kEPC = 16 / esz;         // state elements per 16-byte chunk
  constexpr int kRowChunks = 16 / kEPC;  // chunks per lane per row (16 columns per lane)
  constexpr int kRowBytes = kDstate * esz;
  const int H = c.H;

  const long long units = static_cast<long long>(a.batch) * H;
  const long long per = units / gridDim.x, rem = units % gridDim.x;
  const long long u0 = blockIdx.x * per + min(static_cast<long long>(blockIdx.x), rem);
  const int nu = static_cast<int>(per + (blockIdx.x < rem ? 1 : 0));
  if (nu == 0) return;

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

  const int KB = lay.KB;
  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane issues all bulk copies ----------------
    if (lane != 0) return;
    int cur_b = -1;
    RowRec rr = {};
    int issued = 0;
    bool ok = true;
    for (int i = 0; i < nu; ++i) {
      const int st = i % ns;
      const uint32_t ph = (i / ns) & 1;
      if (i >= ns && !mbar_wait(&empty[st], ph ^ 1)) {
        ok = false;
        break;
      }
      const long long u = u0 + i;
      const int b = static_cast<int>(u / H), h = static_cast<int>(u % H);
      if (b != cur_b) {
        rr = a.rows[b];
        cur_b = b;
      }
      meta[st] = ReadMeta{b, h, rr.s, rr.r, rr.p, rr.Tb, rr.tok0, rr.flags};
      if (rr.flags && rr.Tb > 0) {
        const int s = rr.s, r = rr.r, K = rr.p + rr.Tb, g = h / c.hpg;
        uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
        const uint32_t coef_bytes = (KB + 1) * TP * 4;
        const uint32_t bytes = lay.s0_bytes + (k8bit ? 256u : 0u) + TP * kDstate * 4 + coef_bytes + K * kDim * 2;
        mbar_expect_tx(&full[st], bytes);
        bulk_g2s(sb, static_cast<const uint8_t*>(c.state) +
                         (static_cast<long long>(s) * c.state_stride + static_cast<long long>(h) * kHeadElems) * esz,
                 lay.s0_bytes, &full[st]);
        if (k8bit)
          bulk_g2s(sb + lay.scale_off, c.scale + static_cast<long long>(s) * c.scale_stride + h * kDim, 256, &full[st]);
        bulk_g2s(sb + lay.c_off, a.cf + (static_cast<long long>(b) * c.G + g) * TP * kDstate, TP * kDstate * 4,
                 &full[st]);
        bulk_g2s(sb + lay.coef_off, a.coef + (static_cast<long long>(b) * H + h) * (KB + 1) * TP, coef_bytes,
                 &full[st]);
        // live ring + the new rows the precompute appended: logical 0..K-1
        const uint16_t* xg = c.x_cache + static_cast<long long>(s) * c.x_stride + static_cast<long long>(h) * c.L * kDim;
        const int n1 = min(K, c.L - r);
        bulk_g2s(sb + lay.x_off, xg + r * kDim, n1 * kDim * 2, &full[st]);
        if (K > n1) bulk_g2s(sb + lay.x_off + n1 * kDim * 2, xg, (K - n1) * kDim * 2, &full[st]);
      }
      mbar_arrive(&full[st]);
      issued = i + 1;
    }
    if (!ok) {
      set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      for (int i = max(0, issued - ns); i < issued; ++i) mbar_wait(&full[i % ns], (i / ns) & 1);
    }
    return;
  }

  // ---------------- consumer warps (independent; stage barriers only) ----------------
  const int rg = lane >> 3, j = lane & 7;
  const int rho0 = 8 * warp + 2 * rg;
  for (int i = 0; i < nu; ++i) {
    const int st = i % ns;
    const uint32_t ph = (i / ns) & 1;
    if (!mbar_wait(&full[st], ph)) {
      if (lane == 0) set_error(c.err, RSSM_ERRBIT_TIMEOUT);
      return;
    }
    const ReadMeta m = meta[st];
    const uint8_t* sb = smem + lay.stages_off + st * lay.stage_bytes;
    if (!(m.flags && m.Tb > 0)) {
      // inactive or rejected row: zero outputs, no cache update
      for (int idx = tid; idx < m.Tb * (kDim / 2); idx += kConsumerThreads) {
        const int t = idx >> 5, dp = idx & 31;
        reinterpret_cast<uint32_t*>(a.out + (static_cast<long long>(m.tok0 + t) * H + m.h) * kDim)[dp] = 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      continue;
    }
    const int K = m.p + m.Tb;
    // ---- S0 . C_t over this lane's 16 columns of rows rho0, rho0 + 1 ----
    float2 acc[2][TP];
#pragma unroll
    for (int q2 = 0; q2 < 2; ++q2)
#pragma unroll
      for (int t = 0; t < TP; ++t) acc[q2][t] = make_float2(0.0f, 0.0f);
    const float4* Cf4 = reinterpret_cast<const float4*>(sb + lay.c_off);
#pragma unroll
    for (int ch = 0; ch < kRowChunks; ++ch) {
      const int q = j + 8 * ch;  // 16-byte chunk within the row
      const uint4 q0 = *reinterpret_cast<const uint4*>(sb + rho0 * kRowBytes + q * 16);
      const uint4 q1 = *reinterpret_cast<const uint4*>(sb + (rho0 + 1) * kRowBytes + q * 16);
      constexpr int NP = RowChunk<DT>::kPairs;
      float2 v0[NP], v1[NP];
      RowChunk<DT>::get(q0, v0);
      RowChunk<DT>::get(q1, v1);
      const int m0 = q * (kEPC / 4);  // first f32 chunk of C for these columns
#pragma unroll
      for (int t = 0; t < TP; ++t) {
#pragma unroll
        for (int k4 = 0; k4 < kEPC / 4; ++k4) {
          const float4 cv = Cf4[t * (kDstate / 4) + cswz(m0 + k4)];
          const float2 ca = make_float2(cv.x, cv.y), cb = make_float2(cv.z, cv.w);
          acc[0][t] = __ffma2_rn(v0[2 * k4], ca, acc[0][t]);
          acc[0][t] = __ffma2_rn(v0[2 * k4 + 1], cb, acc[0][t]);
          acc[1][t] = __ffma2_rn(v1[2 * k4], ca, acc[1][t]);
          acc[1][t] = __ffma2_rn(v1[2 * k4 + 1], cb, acc[1][t]);
        }
      }
    }
    const float* coef = reinterpret_cast<const float*>(sb + lay.coef_off);
    float vals[2 * TP];
    float sc0 = 1.0f, sc1 = 1.0f;
    if constexpr (k8bit) {
      const float* scl = reinterpret_cast<const float*>(sb + lay.scale_off);
      sc0 = scl[rho0];
      sc1 = scl[rho0 + 1];
    }
#pragma unroll
    for (int t = 0; t < TP; ++t) {
      const float dct = coef[KB * TP + t];
      vals[t] = (acc[0][t].x + acc[0][t].y) * (dct * sc0);
      vals[TP + t] = (acc[1][t].x + acc[1][t].y) * (dct * sc1);
    }
    // ---- ring terms: sum_k coef[k][t] x_k[d], k = j, j+8, ... (x rows in bf16) ----
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(sb + lay.x_off);
    for (int k = j; k < K; k += 8) {
      const uint32_t xw = xs[k * (kDim / 2) + (rho0 >> 1)];
      const float x0 = bf16lo(xw), x1 = bf16hi(xw);
#pragma unroll
      for (int t4 = 0; t4 < TP; t4 += 4) {
        const float4 cv = *reinterpret_cast<const float4*>(coef + k * TP + t4);
        vals[t4 + 0] = fmaf(cv.x, x0, vals[t4 + 0]);
        vals[t4 + 1] = fmaf(cv.y, x0, vals[t4 + 1]);
        vals[t4 + 2] = fmaf(cv.z, x0, vals[t4 + 2]);
        vals[t4 + 3] = fmaf(cv.w, x0, vals[t4 + 3]);
        vals[TP + t4 + 0] = fmaf(cv.x, x1, vals[TP + t4 + 0]);
        vals[TP + t4 + 1] = fmaf(cv.y, x1, vals[TP + t4 + 1]);
        vals[TP + t4 + 2] = fmaf(cv.z, x1, vals[TP + t4 + 2]);
        vals[TP + t4 + 3] = fmaf(cv.w, x1, vals[TP + t4 + 3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage
    // ---- transpose-reduce the 2*TP partial sums over the 8 lanes of a row pair ----
    constexpr int V = 2 * TP;
#pragma unroll
    for (int step = 0; step < 3; ++step) {
      const int mask = 4 >> step;
      const int half = V >> (step + 1);
      const bool upper = (j & mask) != 0;
#pragma unroll
      for (int e = 0; e < half; ++e) {
        const float send = upper ? vals[e] : vals[e + half];
        const float keep = upper ? vals[e + half] : vals[e];
        vals[e] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
      }
    }
    // lane j now holds value index j * (V/8) + e: row rho0 + (j >> 2)
    constexpr int PER = V / 8;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int idx = j * PER + e;
      const int rr = idx / TP, t = idx % TP;
      if (t < m.Tb) {
        const __nv_bfloat16 yv = __float2bfloat16_rn(vals[e]);
        a.out[(static_cast<long long>(m.tok0 + t) * H + m.h) * kDim + rho0 + rr] =
            *reinterpret_cast<const uint16_t*>(&yv);
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
  if (a.TP == 4)
    precompute_kernel<4><<<grid, 256, 0, st>>>(a);
  else
    precompute_kernel<8><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

template <int DT, int TP>
static int launch_readout_t(const StepArgs& a, int num_sms, cudaStream_t st) {
  // as many stages as fit two CTAs per SM (>= 3), else one CTA with up to 6
  int ns = 8, ctas = 2;
  for (; ns >= 3; --ns)
    if (read_layout(DT, a.c.L, TP, ns).total <= 113 * 1024) break;
  if (ns < 3) {
    ctas = 1;
    for (ns = 8; ns > 2; --ns)
      if (read_layout(DT, a.c.L, TP, ns).total <= 225 * 1024) break;
  }
  const ReadLayout lay = read_layout(DT, a.c.L, TP, ns);
  cudaError_t e = cudaFuncSetAttribute(readout_kernel<DT, TP>, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(readout_kernel<DT, TP>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, readout_kernel<DT, TP>, kThreads, lay.total);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  if (occ > ctas) occ = ctas;
  const long long units = static_cast<long long>(a.batch) * a.c.H;
  const long long cap = static_cast<long long>(num_sms) * occ;
  const int grid = static_cast<int>(units < cap ? units : cap);
  readout_kernel<DT, TP><<<grid, kThreads, lay.total, st>>>(a, ns);
  return cudaGetLastError();
}

int launch_readout(const StepArgs& a, int num_sms, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool t4 = a.TP == 4;
  switch (a.c.dtype) {
    case RSSM_F32: return t4 ? launch_readout_t<RSSM_F32, 4>(a, num_sms, st) : launch_readout_t<RSSM_F32, 8>(a, num_sms, st);
    case RSSM_BF16: return t4 ? launch_readout_t<RSSM_BF16, 4>(a, num_sms, st) : launch_readout_t<RSSM_BF16, 8>(a, num_sms, st);
    case RSSM_F16: return t4 ? launch_readout_t<RSSM_F16, 4>(a, num_sms, st) : launch_readout_t<RSSM_F16, 8>(a, num_sms, st);
    case RSSM_I8: return t4 ? launch_readout_t<RSSM_I8, 4>(a, num_sms, st) : launch_readout_t<RSSM_I8, 8>(a, num_sms, st);
    default: return t4 ? launch_readout_t<RSSM_E4M3, 4>(a, num_sms, st) : launch_readout_t<RSSM_E4M3, 8>(a, num_sms, st);
  }
}

}  // namespace rssm
