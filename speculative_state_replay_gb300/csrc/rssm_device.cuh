// rssm_device.cuh -- device building blocks of librssm (sm_103a).
//
// Pipeline primitives (mbarrier, 1-D bulk copies), the fixed-sequence fp32
// exp / softplus, the Philox4x32-7 hash and the checkpoint quantiser.  The
// arithmetic that decides stored bits (dt' in the ring, flushed checkpoints)
// is written with explicit __fmul_rn/__fadd_rn/__fmaf_rn so the compiler
// cannot contract or reorder it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rssm_internal.h"

namespace rssm {

// --------------------------------------------------------------------------
// bit helpers
// --------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ float2 h2f2(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

__device__ __forceinline__ void set_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// --------------------------------------------------------------------------
// mbarrier / bulk-copy primitives (PTX, sm_90+)
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}
// arrive and raise the expected transaction bytes of the current phase in one
// operation (the phase still completes only when those bytes have landed)
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Suspending test: the thread sleeps in hardware until the phase completes or
// about `hint_ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase of an mbarrier: gives up after `tries` suspending
// tests of up to ~1 ms each (about two seconds by default).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t tries = kWaitTries) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < tries; ++i)
    if (mbar_try_wait_for(bar, parity, 1000000u)) return true;
  return false;
}
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Per-thread asynchronous copies global -> shared (16 bytes through L2 only,
// or 4 bytes), all of a thread's copies completed by cp_async_wait_all().
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Arrive on `bar` once every cp.async this thread has issued so far has
// landed, without adding to the barrier's expected count (the barrier is
// initialised to expect this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Programmatic dependent launch.  pdl_wait() returns once the preceding kernel
// in the stream has completed and its writes are visible (immediately when the
// kernel was launched without the attribute); every chain kernel calls it
// before touching memory its predecessors may write.  pdl_trigger() lets the
// next kernel start launching (it still waits before reading our results).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// launch with programmatic stream serialisation (the kernel must call pdl_wait)
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// named barrier over the consumer warps only (the producer warp never joins)
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory"); }

// --------------------------------------------------------------------------
// Fixed-sequence fp32 exp / log1p / softplus.  Methods: Cody-Waite range
// reduction x = k ln2 + r with ln2 split into two floats, degree-7 Taylor
// polynomial of e^r in Horner form, scaling by 2^k; log1p(z) = 2 atanh(s)
// with s = z/(2+z) for small z, else log(w) = e ln2 + 2 atanh((m-1)/(m+1))
// for w = 1 + z = m 2^e plus the correction (z - (w-1))/w.  Coefficients are
// 1/k! and 1/(2k+1) rounded once to float.  Every operation is an IEEE
// round-to-nearest primitive, so the result is a fixed function of x.
// --------------------------------------------------------------------------
__device__ __forceinline__ float spec_exp(float x) {
  if (x != x) return x;
  if (x < -87.0f) return 0.0f;
  if (x > 88.0f) return __uint_as_float(0x7f800000u);
  const float log2e = (float)1.4426950408889634;
  const float ln2_hi = (float)0.6931471805599453;
  const float ln2_lo = (float)(0.6931471805599453 - (double)(float)0.6931471805599453);
  const float kf = rintf(__fmul_rn(x, log2e));
  float r = __fmaf_rn(-kf, ln2_hi, x);
  r = __fmaf_rn(-kf, ln2_lo, r);
  float q = (float)(1.0 / 5040.0);
  q = __fmaf_rn(q, r, (float)(1.0 / 720.0));
  q = __fmaf_rn(q, r, (float)(1.0 / 120.0));
  q = __fmaf_rn(q, r, (float)(1.0 / 24.0));
  q = __fmaf_rn(q, r, (float)(1.0 / 6.0));
  q = __fmaf_rn(q, r, 0.5f);
  q = __fmaf_rn(q, r, 1.0f);
  q = __fmaf_rn(q, r, 1.0f);
  const int k = static_cast<int>(kf);
  return __fmul_rn(q, __uint_as_float(static_cast<uint32_t>(k + 127) << 23));
}

__device__ __forceinline__ float spec_log1p(float z) {
  if (z != z || z == __uint_as_float(0x7f800000u)) return z;
  const float ln2_hi = (float)0.6931471805599453;
  const float ln2_lo = (float)(0.6931471805599453 - (double)(float)0.6931471805599453);
  if (z < 0.25f) {
    const float s = __fdiv_rn(z, __fadd_rn(2.0f, z));
    const float s2 = __fmul_rn(s, s);
    float q = (float)(1.0 / 11.0);
    q = __fmaf_rn(q, s2, (float)(1.0 / 9.0));
    q = __fmaf_rn(q, s2, (float)(1.0 / 7.0));
    q = __fmaf_rn(q, s2, (float)(1.0 / 5.0));
    q = __fmaf_rn(q, s2, (float)(1.0 / 3.0));
    q = __fmul_rn(q, s2);
    const float t = __fmaf_rn(s, q, s);
    return __fadd_rn(t, t);
  }
  const float w = __fadd_rn(1.0f, z);
  const uint32_t wb = __float_as_uint(w);
  int e = static_cast<int>((wb >> 23) & 0xffu) - 127;
  float m = __uint_as_float((wb & 0x7fffffu) | 0x3f800000u);
  if (m > (float)1.4142135623730951) {
    m = __fmul_rn(m, 0.5f);
    e += 1;
  }
  const float f = __fsub_rn(m, 1.0f);
  const float s = __fdiv_rn(f, __fadd_rn(2.0f, f));
  const float s2 = __fmul_rn(s, s);
  float q = (float)(1.0 / 13.0);
  q = __fmaf_rn(q, s2, (float)(1.0 / 11.0));
  q = __fmaf_rn(q, s2, (float)(1.0 / 9.0));
  q = __fmaf_rn(q, s2, (float)(1.0 / 7.0));
  q = __fmaf_rn(q, s2, (float)(1.0 / 5.0));
  q = __fmaf_rn(q, s2, (float)(1.0 / 3.0));
  q = __fmul_rn(q, s2);
  const float t = __fmaf_rn(s, q, s);
  const float logm = __fadd_rn(t, t);
  const float corr = __fdiv_rn(__fsub_rn(z, __fsub_rn(w, 1.0f)), w);
  const float ef = static_cast<float>(e);
  return __fmaf_rn(ef, ln2_hi, __fmaf_rn(ef, ln2_lo, __fadd_rn(logm, corr)));
}

__device__ __forceinline__ float spec_softplus(float v) {
  if (v > 20.0f) return v;
  return spec_log1p(spec_exp(v));
}

// --------------------------------------------------------------------------
// Philox4x32 with 7 rounds (Salmon et al., SC'11): the stochastic-rounding
// hash.  Counter (element/4, head, slot, flush epoch), key = 64-bit seed.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_7(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 7; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// --------------------------------------------------------------------------
// Rounding onto the state formats.  Nearest: ties to even, saturating at
// the largest finite value.  Stochastic: |v| goes to the grid point above
// with probability equal to its fractional distance from the one below,
// using u = (rnd >> 8) 2^-24; all steps are exact (power-of-two scaling).
// --------------------------------------------------------------------------
__device__ __forceinline__ uint16_t round_bf16(float v, bool sr, uint32_t rnd) {
  const uint32_t u = __float_as_uint(v);
  uint32_t r;
  if (sr) {
    const uint32_t low = u & 0xffffu;
    r = (u >> 16) + (((rnd >> 8) < (low << 8)) ? 1u : 0u);
  } else {
    r = (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
  }
  if ((r & 0x7fffu) == 0x7f80u) r = (r & 0x8000u) | 0x7f7fu;  // saturate
  return static_cast<uint16_t>(r);
}

// grid with mbits fraction bits, lowest normal exponent emin: round |v| up or
// down stochastically, saturate at maxf, keep the sign.
__device__ __forceinline__ float sr_grid(float v, int mbits, int emin, float maxf, uint32_t rnd) {
  const float a = fabsf(v);
  int e = static_cast<int>((__float_as_uint(a) >> 23) & 0xffu) - 127;
  e = max(e, emin);
  const int qe = e - mbits;
  const float inv_q = __uint_as_float(static_cast<uint32_t>(127 - qe) << 23);  // 2^-qe
  const float q = __uint_as_float(static_cast<uint32_t>(127 + qe) << 23);      // 2^qe
  const float ratio = __fmul_rn(a, inv_q);
  const float n = floorf(ratio);
  const float f = __fsub_rn(ratio, n);
  const float uu = __fmul_rn(static_cast<float>(rnd >> 8), 5.9604644775390625e-8f);  // 2^-24
  float mag = __fmul_rn(uu < f ? __fadd_rn(n, 1.0f) : n, q);
  mag = fminf(mag, maxf);
  return copysignf(mag, v);
}

__device__ __forceinline__ uint16_t round_f16(float v, bool sr, uint32_t rnd) {
  float g = sr ? sr_grid(v, 10, -14, 65504.0f, rnd) : v;
  __half h = __float2half_rn(g);
  uint16_t bits = *reinterpret_cast<uint16_t*>(&h);
  if ((bits & 0x7fffu) == 0x7c00u) bits = (bits & 0x8000u) | 0x7bffu;  // saturate
  return bits;
}

__device__ __forceinline__ uint8_t round_e4m3(float v, bool sr, uint32_t rnd) {
  float g = sr ? sr_grid(v, 3, -6, 448.0f, rnd) : v;
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(g, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ int8_t round_i8(float v, bool sr, uint32_t rnd) {
  float g;
  if (sr) {
    const float a = fabsf(v);
    const float n = floorf(a);
    const float f = __fsub_rn(a, n);
    const float uu = __fmul_rn(static_cast<float>(rnd >> 8), 5.9604644775390625e-8f);
    g = copysignf(fminf(uu < f ? __fadd_rn(n, 1.0f) : n, 127.0f), v);
  } else {
    g = fminf(fmaxf(rintf(v), -127.0f), 127.0f);
  }
  return static_cast<int8_t>(static_cast<int>(g));
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(hr));
}

// --------------------------------------------------------------------------
// Round-to-nearest-even, saturating at the largest finite value, two at a time
// (the PTX satfinite conversions: RNE first, then clamp to +-max finite).
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cvt_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_bf16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// --------------------------------------------------------------------------
// Checkpoint quantiser for one thread's 4 rows x 8 columns (rows r0..r0+3,
// columns c0..c0+7 of a [64][128] head), the fragment the flush and init
// kernels own.  Lanes sharing rows must be the 16 lanes with equal
// (lane >> 4) of a warp (they hold the 128 columns of those rows).
// 8-bit formats: per-row scale = amax/QMAX (1 for amax < 2^-100), v = acc *
// (1/scale), then nearest or stochastic rounding.  Stochastic rounding draws
// one Philox4x32-7 block per 4 consecutive elements of a row.
// --------------------------------------------------------------------------
__device__ __forceinline__ void row_random(uint32_t (&rnd)[8], int row, int c0, uint32_t h, uint32_t s,
                                           uint32_t epoch, uint64_t seed) {
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t elem = static_cast<uint32_t>(row * 128 + c0 + 4 * q);
    const uint4 w = philox4x32_7(elem >> 2, h, s, epoch, k0, k1);
    rnd[4 * q + 0] = w.x;
    rnd[4 * q + 1] = w.y;
    rnd[4 * q + 2] = w.z;
    rnd[4 * q + 3] = w.w;
  }
}

// Byte offset of state element (row, col) in shared memory laid out as the
// readout's TMA boxes: 64 rows x 128 bytes per box, boxes 8 KiB apart, the
// 16-byte chunk index within a row XOR-ed with (row & 7) (the 128-byte swizzle).
template <int ESZ>
__device__ __forceinline__ uint32_t swizzled_offset(int row, int col) {
  const int byte = col * ESZ;
  return static_cast<uint32_t>((byte >> 7) * 8192 + row * 128 + ((((byte >> 4) & 7) ^ (row & 7)) << 4) + (byte & 15));
}

// Round the lane's 4 x 8 accumulators (rows r0..r0+3, columns c0..c0+7) to
// the state format and store them to the head's checkpoint (and the row
// scales for 8-bit formats).  With kMirror the same bits also go to a
// shared-memory copy of the head in the swizzled box layout (and its scales).
template <int DT, bool kMirror = false>
__device__ __forceinline__ void quantize_store(float (&acc)[4][8], int r0, int c0, int lane, void* head_state,
                                               float* head_scale, int rounding, uint32_t h, uint32_t s,
                                               uint32_t epoch, uint64_t seed, uint8_t* mirror = nullptr,
                                               float* mirror_scale = nullptr) {
  const bool sr = rounding == RSSM_ROUND_STOCHASTIC;
  if constexpr (DT == RSSM_F32) {
    float* st = static_cast<float*>(head_state);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float4* dst = reinterpret_cast<float4*>(st + (r0 + i) * 128 + c0);
      const float4 v0 = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      const float4 v1 = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
      dst[0] = v0;
      dst[1] = v1;
      if constexpr (kMirror) {
        *reinterpret_cast<float4*>(mirror + swizzled_offset<4>(r0 + i, c0)) = v0;
        *reinterpret_cast<float4*>(mirror + swizzled_offset<4>(r0 + i, c0 + 4)) = v1;
      }
    }
  } else if constexpr (DT == RSSM_BF16 || DT == RSSM_F16) {
    uint16_t* st = static_cast<uint16_t*>(head_state);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t wds[4];
      if (!sr) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          wds[q] = DT == RSSM_BF16 ? cvt_bf16x2_sat(acc[i][2 * q], acc[i][2 * q + 1])
                                   : cvt_f16x2_sat(acc[i][2 * q], acc[i][2 * q + 1]);
      } else {
        uint32_t rnd[8];
        row_random(rnd, r0 + i, c0, h, s, epoch, seed);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint16_t lo, hi;
          if constexpr (DT == RSSM_BF16) {
            lo = round_bf16(acc[i][2 * q], true, rnd[2 * q]);
            hi = round_bf16(acc[i][2 * q + 1], true, rnd[2 * q + 1]);
          } else {
            lo = round_f16(acc[i][2 * q], true, rnd[2 * q]);
            hi = round_f16(acc[i][2 * q + 1], true, rnd[2 * q + 1]);
          }
          wds[q] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
      }
      *reinterpret_cast<uint4*>(st + (r0 + i) * 128 + c0) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
      if constexpr (kMirror)
        *reinterpret_cast<uint4*>(mirror + swizzled_offset<2>(r0 + i, c0)) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
    }
  } else {
    constexpr float qmax = (DT == RSSM_I8) ? 127.0f : 448.0f;
    float amax[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float m = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(acc[i][q]));
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      amax[i] = m;
    }
    // lane (lane & 3) of each 16-lane group computes row (lane & 3)'s scale
    const int mine = lane & 3;
    float am = amax[0];
#pragma unroll
    for (int i = 1; i < 4; ++i)
      if (mine == i) am = amax[i];
    const float sc = am < 7.888609052210118e-31f /* 2^-100 */ ? 1.0f : __fdiv_rn(am, qmax);
    const float iv = __frcp_rn(sc);
    float scale[4];
    uint8_t* st = static_cast<uint8_t*>(head_state);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      scale[i] = __shfl_sync(0xffffffffu, sc, (lane & 16) | i);
      const float inv = __shfl_sync(0xffffffffu, iv, (lane & 16) | i);
      uint32_t wds[2] = {0u, 0u};
      if (!sr) {
#pragma unroll
        for (int q = 0; q < 8; q += 2) {
          const float v0 = __fmul_rn(acc[i][q], inv), v1 = __fmul_rn(acc[i][q + 1], inv);
          uint32_t pair;
          if constexpr (DT == RSSM_I8) {
            // round-to-nearest-even onto -127..127 without a conversion
            // instruction: for |v| <= 127, v + 1.5 * 2^23 lies in [2^23, 2^24)
            // where the fp32 grid is the integers, so the addition itself
            // rounds (to even) and the low byte of the sum's bits is the code
            const float t0 = __fadd_rn(fminf(fmaxf(v0, -127.0f), 127.0f), 12582912.0f);
            const float t1 = __fadd_rn(fminf(fmaxf(v1, -127.0f), 127.0f), 12582912.0f);
            pair = __byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x0040u) & 0xffffu;
          } else {
            pair = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3));
          }
          wds[q >> 2] |= pair << (8 * (q & 3));
        }
      } else {
        uint32_t rnd[8];
        row_random(rnd, r0 + i, c0, h, s, epoch, seed);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float v = __fmul_rn(acc[i][q], inv);
          uint32_t code;
          if constexpr (DT == RSSM_I8)
            code = static_cast<uint8_t>(round_i8(v, true, rnd[q]));
          else
            code = round_e4m3(v, true, rnd[q]);
          wds[q >> 2] |= code << (8 * (q & 3));
        }
      }
      *reinterpret_cast<uint2*>(st + (r0 + i) * 128 + c0) = make_uint2(wds[0], wds[1]);
      if constexpr (kMirror)
        *reinterpret_cast<uint2*>(mirror + swizzled_offset<1>(r0 + i, c0)) = make_uint2(wds[0], wds[1]);
    }
    if ((lane & 15) == 0) {
      *reinterpret_cast<float4*>(head_scale + r0) = make_float4(scale[0], scale[1], scale[2], scale[3]);
      if constexpr (kMirror)
        *reinterpret_cast<float4*>(mirror_scale + r0) = make_float4(scale[0], scale[1], scale[2], scale[3]);
    }
  }
}

// --------------------------------------------------------------------------
// NVFP4 read checkpoint: FP4 E2M1 codes (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4,
// 6; code = sign << 3 | magnitude index), one E4M3 scale per 16 consecutive
// dstate values, one FP32 global scale gs per slot.
// --------------------------------------------------------------------------
// E2M1 nearest (ties to the even code), saturating at 6, keeping the sign of
// v (also for values that round to zero): the grid step is 0.5 below 2, 1 in
// [2, 4), 2 from 4 on, so |v| / step (a multiplication by a power of two) and
// the rounding are exact operations.
__device__ __forceinline__ uint32_t e2m1_nearest(float v) {
  const float a = fabsf(v);
  const float inv_q = a < 2.0f ? 2.0f : (a < 4.0f ? 1.0f : 0.5f);
  const float q = a < 2.0f ? 0.5f : (a < 4.0f ? 1.0f : 2.0f);
  const float mag = fminf(__fmul_rn(rintf(__fmul_rn(a, inv_q)), q), 6.0f);  // a grid point
  const uint32_t m = (mag > 0.25f ? 1u : 0u) + (mag > 0.75f ? 1u : 0u) + (mag > 1.25f ? 1u : 0u) +
                     (mag > 1.75f ? 1u : 0u) + (mag > 2.5f ? 1u : 0u) + (mag > 3.5f ? 1u : 0u) +
                     (mag > 5.0f ? 1u : 0u);
  return m | ((__float_as_uint(v) >> 28) & 8u);
}

// Four E2M1 codes (the nibbles of w, lowest first) as two fp16 pairs, exactly:
// the fp16 value of each magnitude has a zero low byte, so its high byte comes
// from an 8-entry table by byte permutation, and the code's sign bit becomes
// the fp16 sign bit.
__device__ __forceinline__ void e2m1x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t mags = __byte_perm(0x3E3C3800u, 0x46444240u, w & 0x7777u);  // high bytes of 0,.5,1,1.5 | 2,3,4,6
  const uint32_t sgn = ((w & 0x8u) << 4) | ((w & 0x80u) << 8) | ((w & 0x800u) << 12) | ((w & 0x8000u) << 16);
  const uint32_t hb = mags | sgn;
  lo = __byte_perm(hb, 0u, 0x1404u);  // (codes 0, 1)
  hi = __byte_perm(hb, 0u, 0x3424u);  // (codes 2, 3)
}

// NVFP4 encoding of the lane's 4 x 8 fp32 values (rows r0..r0+3, columns
// c0..c0+7 of a [64][128] head; lanes 2k and 2k+1 hold the two halves of a
// 16-value block) into the head's codes [64][64 bytes] and block scales
// [64][8]: sf = e4m3 nearest of (block max / (6 gs)), code = e2m1 nearest of
// (v * (1 / (gs * sf))) (0 where sf is 0).
__device__ __forceinline__ void quantize_store_nvfp4(const float (&acc)[4][8], int r0, int c0, int lane,
                                                     uint8_t* head_codes, uint8_t* head_sf, float gs) {
  const float den = __fmul_rn(6.0f, gs);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float m = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(acc[i][q]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    const uint8_t sc = static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(m, den), __NV_SATFINITE, __NV_E4M3));
    const float qs = __fmul_rn(e4m3_to_f32(sc), gs);
    uint32_t word = 0u;
    if (qs > 0.0f) {
      const float inv = __frcp_rn(qs);
#pragma unroll
      for (int q = 0; q < 8; ++q) word |= e2m1_nearest(__fmul_rn(acc[i][q], inv)) << (4 * q);
    }
    *reinterpret_cast<uint32_t*>(head_codes + (r0 + i) * 64 + c0 / 2) = word;
    if (!(lane & 1)) head_sf[(r0 + i) * 8 + c0 / 16] = sc;
  }
}

}  // namespace rssm
