// rssm_readout.cuh -- pieces shared by the readout kernels of librssm: the
// per-stage metadata and shared-memory layout, the tensor-core S0.C
// contraction (mma.sync m16n8k16) over TMA-swizzled S0 boxes, and the tensor
// map over the checkpoint states.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "rssm_device.cuh"

namespace rssm {

// mma.sync m16n8k16 with f32 accumulation and A rows 8..15 zero: D[16x8] +=
// A[16x16] B[16x8] with a0 = A[g][2c..2c+1], a2 = A[g][2c+8..2c+9],
// b0 = B[2c..2c+1][g], b1 = B[2c+8..2c+9][g] (g = lane / 4, c = lane % 4);
// D rows 0..7: d0, d1 = D[g][2c], D[g][2c+1]
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}


// Per (row, head) unit the readout is one small dense contraction on the
// tensor cores, mma.sync m16n8k16 with f32 accumulation:
//     Y^T[t][d] = sum_n Cblk[t][n] S0[d][n]        (M = t, N = d, K = dstate)
//     y_t[d]    = decay_t scale_d Y^T[t][d] + R[t][d]
// where the ring term R (live ring + new tokens) and decay_t come from the
// precompute.  Warp w owns the 8 state rows d = 8w..8w+7 (one n8 tile).  K is
// taken in a permuted order inside each 16-wide step (physical 4c..4c+3 <->
// logical 2c, 2c+1, 2c+8, 2c+9 for lane group c), so every operand fragment is
// one 64-bit shared load; the sum over k is unchanged.  S0 arrives by TMA
// tensor copies with the 128-byte swizzle, which keeps those loads
// conflict-free.
constexpr int kReadChunk = 4;  // (row, head) units per work grab of the readout

// the one-call path's fold rows: two buffers of 8 live tokens, x [8][64] bf16
// then B [8][128] bf16 each
constexpr uint32_t kFoldChunk = 8;
constexpr uint32_t kFoldBufX = kFoldChunk * kDim * 2, kFoldBufOne = kFoldBufX + kFoldChunk * kDstate * 2;
constexpr uint32_t kFoldBuf = 2 * kFoldBufOne;

struct ReadMeta {
  int b, h, s, r, p, Tb, tok0, flags;  // flags: 1 outputs, 2 new C block, 8 no more work, 16 fold
  unsigned epoch;                      // epoch of the checkpoint a fold writes
  float gs;                            // NVFP4: the slot's global scale
  int pad[2];
};

struct ReadLayout {
  int ns;
  uint32_t s0_bytes, scale_off, c_off, r_off, r_bytes, stage_bytes;
  uint32_t fw_off;  // fold area (fold_kb > 0): the heads' fold weights
  uint32_t fbuf_off;  // fold_kb > 0: the CTA's fold-row buffer (two chunks of 8 live tokens' x and B rows)
  uint32_t stages_off, total;
};

// one stage of a unit of `hpu` consecutive heads of one group: S0 as esz
// boxes of 64*hpu rows x 128 bytes | 8-bit scales | C block | ring-term blocks
// [| fold area: the heads' fold weights [hpu][kFoldW]]
__host__ __device__ inline ReadLayout read_layout(int dtype, int TP, int ns, int hpu = 1, int fold_kb = 0) {
  ReadLayout f;
  f.ns = ns;
  const int esz = dtype == RSSM_F32 ? 4 : (dtype == RSSM_BF16 || dtype == RSSM_F16) ? 2 : 1;
  f.s0_bytes = dtype == RSSM_NVFP4 ? kHeadElems / 2 * hpu : kHeadElems * esz * hpu;
  uint32_t o = f.s0_bytes;
  f.scale_off = o;  // 8-bit: row scales [64 hpu] f32; NVFP4: block scales [64 hpu][8] e4m3
  if (dtype == RSSM_I8 || dtype == RSSM_E4M3) o += 256 * hpu;
  if (dtype == RSSM_NVFP4) o += 512 * hpu;
  f.c_off = o;
  o += 8 * kDstate * 2;
  f.r_off = o;
  f.r_bytes = (kRDec + TP * kDim) * 4 * hpu;  // room for the full ring-term blocks (a unit copies its T_b rows)
  o += f.r_bytes;
  f.fw_off = 0;
  if (fold_kb > 0) {
    f.fw_off = o;
    o += hpu * kFoldW * 4;
  }
  f.stage_bytes = (o + 1023) & ~1023u;  // the swizzled boxes need 1024-byte alignment
  f.stages_off = 1024;                  // barriers and per-stage metadata (8 x 48 bytes at 256)
  f.fbuf_off = f.stages_off + ns * f.stage_bytes;
  f.total = f.fbuf_off + (fold_kb > 0 ? kFoldBuf : 0u) + 1024;  // + slack to align the base
  return f;
}

// hint: bring `bytes` (a multiple of 16, 16-byte aligned) at `src` into L2
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// byte offset of (row d, byte k) inside one 64-row x 128-byte swizzled box
__device__ __forceinline__ uint32_t swz(int d, int kbyte) {
  return static_cast<uint32_t>(d * 128 + ((((kbyte >> 4) ^ d) & 7) << 4) + (kbyte & 15));
}

// A fragments of the C block for lane (g, c): row t = g, logical k = 16 ks +
// {2c, 2c+1, 2c+8, 2c+9} (physical 16 ks + 4c .. 4c+3), one 64-bit load per k step
__device__ __forceinline__ void load_c_frags(const uint16_t* cblk, int g, int c, uint2 (&af)[8]) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) af[ks] = *reinterpret_cast<const uint2*>(cblk + g * kDstate + 16 * ((ks ^ g) & 7) + 4 * c);
}

// S0 . C over dstate for state rows d (lane's B column) of this warp; even and
// odd k steps accumulate in separate chains, added at the end
// (BOXB: bytes between the column boxes of a 2- or 4-byte state)
// (NVFP4: sfrow = the 8 block scales of row d)
template <int DT, int BOXB = 8192>
__device__ __forceinline__ void s0_dot_c(const uint8_t* s0, const uint2 (&af)[8], int d, int c, float (&acc)[4],
                                         uint64_t sfrow = 0) {
  float a2[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint2 av = af[ks];
    float(&ac)[4] = a2[ks & 1];
    if constexpr (DT == RSSM_BF16 || DT == RSSM_F16) {
      const int kb = (ks * 16 + 4 * c) * 2;  // byte within the 256-byte row
      const uint2 bv = *reinterpret_cast<const uint2*>(s0 + (kb >> 7) * BOXB + swz(d, kb & 127));
      if constexpr (DT == RSSM_BF16)
        mma_bf16(ac, av.x, av.y, bv.x, bv.y);
      else
        mma_f16(ac, av.x, av.y, bv.x, bv.y);
    } else if constexpr (DT == RSSM_F32) {
      const int kb = (ks * 16 + 4 * c) * 4;
      const float4 f = *reinterpret_cast<const float4*>(s0 + (kb >> 7) * BOXB + swz(d, kb & 127));
      const uint32_t h01 = pack_bf16(f.x, f.y), h23 = pack_bf16(f.z, f.w);
      const uint32_t l01 = pack_bf16(f.x - bf16_lo_f(h01), f.y - bf16_hi_f(h01));
      const uint32_t l23 = pack_bf16(f.z - bf16_lo_f(h23), f.w - bf16_hi_f(h23));
      mma_bf16(a2[0], av.x, av.y, h01, h23);
      mma_bf16(a2[1], av.x, av.y, l01, l23);
    } else if constexpr (DT == RSSM_NVFP4) {
      // rows d and d + 1 share one 128-byte tensor row (64 bytes of codes
      // each); 4 codes = 2 bytes; the block scale of these 16 values is
      // byte ks of the row's 8 (sfrow), applied exactly in fp16
      const uint32_t w = *reinterpret_cast<const uint16_t*>(s0 + swz(d >> 1, (d & 1) * 64 + 8 * ks + 2 * c));
      uint32_t lo, hi;
      e2m1x4_to_f16x2(w, lo, hi);
      const __half_raw sr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>((sfrow >> (8 * ks)) & 0xffu),
                                                    __NV_E4M3);
      const __half2 s2 = __halves2half2(__half(sr), __half(sr));
      const __half2 h01 = __hmul2(*reinterpret_cast<const __half2*>(&lo), s2);
      const __half2 h23 = __hmul2(*reinterpret_cast<const __half2*>(&hi), s2);
      mma_f16(ac, av.x, av.y, *reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(s0 + swz(d, ks * 16 + 4 * c));
      uint32_t b0, b1;
      if constexpr (DT == RSSM_I8) {
        // int8 code q as fp16: (1024 + (q + 128)) - 1152, exact
        const uint32_t u = w ^ 0x80808080u;
        const uint32_t p01 = __byte_perm(u, 0x64646464u, 0x4140), p23 = __byte_perm(u, 0x64646464u, 0x4342);
        const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
        const __half2 h01 = __hsub2(*reinterpret_cast<const __half2*>(&p01), off);
        const __half2 h23 = __hsub2(*reinterpret_cast<const __half2*>(&p23), off);
        b0 = *reinterpret_cast<const uint32_t*>(&h01);
        b1 = *reinterpret_cast<const uint32_t*>(&h23);
      } else {
        const __half2_raw r01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
        const __half2_raw r23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
        b0 = static_cast<uint32_t>(r01.x) | (static_cast<uint32_t>(r01.y) << 16);
        b1 = static_cast<uint32_t>(r23.x) | (static_cast<uint32_t>(r23.y) << 16);
      }
      mma_f16(ac, av.x, av.y, b0, b1);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = a2[0][j] + a2[1][j];
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link)
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// S0 of all slots as a 3-D tensor [slot][H*64 rows][128], boxes of 64 rows x 128 bytes, 128-byte swizzle
// S0 of all slots as a 3-D tensor [slot][H*64 rows][128], boxes of 64*hpu rows
// x 128 bytes, 128-byte swizzle
inline bool encode_state_map(const Cache& c, CUtensorMap* map, int hpu = 1) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  if (c.dtype == RSSM_NVFP4) {
    // codes as [slot][H*32 rows][128 bytes] (two state rows per tensor row);
    // boxes of 32*hpu tensor rows (hpu heads) x 128 bytes, 128-byte swizzle
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(c.H) * 32, static_cast<cuuint64_t>(c.S)};
    const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(c.state_stride)};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(32 * hpu), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c.state, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const int esz = c.dtype == RSSM_F32 ? 4 : (c.dtype == RSSM_BF16 || c.dtype == RSSM_F16) ? 2 : 1;
  const CUtensorMapDataType dt = esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                          : (esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDstate), static_cast<cuuint64_t>(c.H) * kDim,
                              static_cast<cuuint64_t>(c.S)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDstate) * esz, static_cast<cuuint64_t>(c.state_stride) * esz};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(kDim * hpu), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, dt, 3, c.state, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace rssm
