/*
 * rssm_oracle.c -- plain CPU oracle for the ReplaySSM checkpointing
 * selective-state-update (Mamba-2 decode with speculative draft tokens).
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct reference the
 * CUDA library is checked against.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg load it.  It shares no code, header, table
 * or constant generator with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (the pages this follows):
 *   [FI]   FlashInfer PR #3975 "mamba checkpointing SSU: two-kernel split +
 *          ring-buffer cache for checkpointing SSU".
 *   [vS]   vLLM PR #65660 "WIP: [Mamba] Add separate CuTeDSL ReplaySSM
 *          checkpoints".
 *   [vAPI] vLLM API docs, vllm.model_executor.layers.mamba.ops.replayssm_cutedsl.
 *
 * Precision.  The readout y is computed in double from its definition and
 * rounded to bf16 once.  The flush works in fp32, the precision [vS] Overview
 * gives the flush stage, in one canonical order (below) so that 8-bit codes are
 * a function of the inputs alone.  Build with -ffp-contract=off: no a*b+c may
 * be fused behind our back; every fused multiply-add is an explicit fmaf().
 *
 * Pins: every function here is checked by tests/ against something other
 * than itself (brute-force recurrence, library conversions, closed forms,
 * numpy's Philox4x64-10).  The Philox4x32 multipliers are the published
 * constants and have no independent known-answer vector here ("parity
 * unpinned" for those two constants; the round structure is pinned through
 * the 64-bit instantiation of the same code).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define P_DIM 64   /* head dim, [vAPI] module docstring (kernels take head dim 64) */
#define N_DIM 128  /* dstate,   [vAPI] module docstring (state dim 128) */

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_I8 = 3, ORC_E4M3 = 4, ORC_NVFP4 = 5 };
enum { ORC_NEAREST = 0, ORC_STOCHASTIC = 1 };

/* Device-side error bits, sticky.  Same meaning as the library's. */
#define ORC_ERR_PNAT 1u    /* pnat outside what the ring can hold */
#define ORC_ERR_SEQLEN 2u  /* a row's token count < 0 or > T */
#define ORC_ERR_ACCEPT 4u  /* accepted count < 0 or > the row's token count */

typedef struct {
  int32_t num_slots, nheads, ngroups, max_window, npredicted;
  int32_t state_dtype, rounding;
  void *state;       int64_t state_slot_stride; /* elements; [slot][H][64][128] */
  float *scale;      int64_t scale_slot_stride; /* [slot][H][64], 8-bit only */
  uint16_t *x_cache; int64_t x_slot_stride;     /* bf16 [slot][H][L][64] */
  uint16_t *B_cache; int64_t B_slot_stride;     /* bf16 [slot][G][L][128] */
  float *dt_cache;   int64_t dt_slot_stride;    /* f32  [slot][H][L] (dt') */
  int32_t *ring_start;                          /* [slot] */
  uint32_t *flush_epoch;                        /* [slot] */
  uint32_t *error_word;                         /* [1] */
  /* Separate read checkpoint ([vS] Overview: an FP16 recurrence checkpoint
   * with stochastic rounding, FP32 flush work, an 8-bit read checkpoint, BF16
   * readout; Claims: read checkpoints use nearest encoding).  8-bit codes
   * [slot][H][64][128] with FP32 row scales [slot][H][64], encoded to nearest
   * from the same fp32 values as the recurrence state (at init and at every
   * flush); the step's readout reads S0 from them.  read_state = NULL: the
   * step reads the recurrence state itself.                                 */
  void *read_state;  int64_t read_slot_stride;  /* elements (NVFP4: bytes, two codes each) */
  float *read_scale; int64_t read_scale_stride;
  int32_t read_dtype;                           /* ORC_I8, ORC_E4M3 or ORC_NVFP4 */
  /* NVFP4 read checkpoint (read_dtype = ORC_NVFP4; [vAPI]
   * initialize_replayssm_state, NVFP4 branch, and the kernels' state_lo /
   * sf_lo / sg_meta arguments): FP4 E2M1 codes [slot][H][64][64 bytes] in
   * read_state, one E4M3 scale per 16 consecutive dstate values
   * [slot][H][64][8] in read_sf, one FP32 global scale per slot in read_gs
   * (read_scale unused).                                                    */
  uint8_t *read_sf;  int64_t read_sf_stride;    /* bytes */
  float *read_gs;                               /* [slot] */
} orc_cache;

/* ------------------------------------------------------------------------- */
/* bit helpers                                                               */
/* ------------------------------------------------------------------------- */
static inline uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static inline float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static inline void set_err(uint32_t *w, uint32_t bit) {
  if (w) __atomic_fetch_or(w, bit, __ATOMIC_RELAXED);
}

/* ------------------------------------------------------------------------- */
/* Spec math.  dt + dt_bias goes through softplus ([vAPI]
 * selective_state_update_replayssm docstring) and the decays are exponentials
 * of the cumulative A*dt ([FI]
 * Description item 1).  Because dt' is stored in the ring and feeds 8-bit
 * codes, both sides evaluate exp and softplus with one fixed sequence of IEEE
 * fp32 operations, written from textbook methods:
 *   exp:   Cody-Waite reduction x = k ln2 + r (ln2 split in two floats), then
 *          the degree-7 Taylor polynomial of e^r in Horner form, then 2^k.
 *   log1p: log1p(z) = 2 atanh(z / (2 + z)) for small z; otherwise
 *          log(w) = e ln2 + 2 atanh((m-1)/(m+1)) for w = 1 + z = m 2^e, plus
 *          the first-order correction (z - (w - 1)) / w for rounding of w.
 * Coefficients are 1/k! and 1/(2k+1), rounded once to float.               */
/* ------------------------------------------------------------------------- */
static inline float pow2i(int k) { return u2f((uint32_t)(k + 127) << 23); } /* k in [-126,127] */

float orc_spec_exp(float x) {
  if (x != x) return x;
  if (x < -87.0f) return 0.0f;
  if (x > 88.0f) return INFINITY;
  const float log2e = (float)1.4426950408889634;
  const float ln2_hi = (float)0.6931471805599453;
  const float ln2_lo = (float)(0.6931471805599453 - (double)(float)0.6931471805599453);
  float kf = rintf(x * log2e);
  float r = fmaf(-kf, ln2_hi, x);
  r = fmaf(-kf, ln2_lo, r);
  float q = (float)(1.0 / 5040.0);
  q = fmaf(q, r, (float)(1.0 / 720.0));
  q = fmaf(q, r, (float)(1.0 / 120.0));
  q = fmaf(q, r, (float)(1.0 / 24.0));
  q = fmaf(q, r, (float)(1.0 / 6.0));
  q = fmaf(q, r, 0.5f);
  q = fmaf(q, r, 1.0f);
  q = fmaf(q, r, 1.0f);
  return q * pow2i((int)kf);
}

float orc_spec_log1p(float z) {
  if (z != z || z == INFINITY) return z;
  const float ln2_hi = (float)0.6931471805599453;
  const float ln2_lo = (float)(0.6931471805599453 - (double)(float)0.6931471805599453);
  if (z < 0.25f) {
    float s = z / (2.0f + z);
    float s2 = s * s;
    float q = (float)(1.0 / 11.0);
    q = fmaf(q, s2, (float)(1.0 / 9.0));
    q = fmaf(q, s2, (float)(1.0 / 7.0));
    q = fmaf(q, s2, (float)(1.0 / 5.0));
    q = fmaf(q, s2, (float)(1.0 / 3.0));
    q = q * s2;
    float t = fmaf(s, q, s); /* atanh(s) = s + s (s^2/3 + s^4/5 + ...) */
    return t + t;
  }
  float w = 1.0f + z;
  uint32_t wb = f2u(w);
  int e = (int)((wb >> 23) & 0xffu) - 127;
  float m = u2f((wb & 0x7fffffu) | 0x3f800000u);
  if (m > (float)1.4142135623730951) {
    m = m * 0.5f;
    e += 1;
  }
  float f = m - 1.0f;
  float s = f / (2.0f + f);
  float s2 = s * s;
  float q = (float)(1.0 / 13.0);
  q = fmaf(q, s2, (float)(1.0 / 11.0));
  q = fmaf(q, s2, (float)(1.0 / 9.0));
  q = fmaf(q, s2, (float)(1.0 / 7.0));
  q = fmaf(q, s2, (float)(1.0 / 5.0));
  q = fmaf(q, s2, (float)(1.0 / 3.0));
  q = q * s2;
  float t = fmaf(s, q, s);
  float logm = t + t;
  float corr = (z - (w - 1.0f)) / w;
  float ef = (float)e;
  return fmaf(ef, ln2_hi, fmaf(ef, ln2_lo, logm + corr));
}

/* softplus(v) = log(1 + e^v), taken as v itself above 20 (Mamba convention). */
float orc_spec_softplus(float v) {
  if (v > 20.0f) return v;
  return orc_spec_log1p(orc_spec_exp(v));
}

/* ------------------------------------------------------------------------- */
/* Philox counter-based generator (Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11).  One round maps the counter
 * (c0,c1,c2,c3) with key (k0,k1) to (hi(M1*c2)^c1^k0, lo(M1*c2),
 * hi(M0*c0)^c3^k1, lo(M0*c0)); the key is bumped by the Weyl constants
 * before every round but the first.  The stochastic rounding of the pages
 * ([FI] commit notes on Philox rounding; [vS] Claims, where the FP16
 * recurrence checkpoint is rounded with "SR7") is read as Philox4x32 with 7
 * rounds.                                         */
/* ------------------------------------------------------------------------- */
void orc_philox4x32(uint32_t rounds, const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (uint32_t r = 0; r < rounds; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u; /* floor(2^32 (phi - 1)) */
      k1 += 0xBB67AE85u; /* floor(2^32 (sqrt(3) - 1)) */
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The same round structure on 64-bit words; used only to pin the structure
 * against numpy's Philox4x64-10 bit generator. */
void orc_philox4x64(uint32_t rounds, const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
  uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint64_t k0 = key[0], k1 = key[1];
  for (uint32_t r = 0; r < rounds; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B97F4A7C15ull;
      k1 += 0xBB67AE8584CAA73Bull;
    }
    unsigned __int128 p0 = (unsigned __int128)0xD2E7470EE14C6C93ull * c0;
    unsigned __int128 p1 = (unsigned __int128)0xCA5A826395121157ull * c2;
    uint64_t n0 = (uint64_t)(p1 >> 64) ^ c1 ^ k0;
    uint64_t n1 = (uint64_t)p1;
    uint64_t n2 = (uint64_t)(p0 >> 64) ^ c3 ^ k1;
    uint64_t n3 = (uint64_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Random word for element elem = d*128 + n of head h in slot s at flush
 * number `epoch`: counter (elem/4, h, s, epoch), key = the 64-bit seed,
 * word elem%4 of the output block. */
uint32_t orc_sr_word(uint64_t seed, uint32_t elem, uint32_t h, uint32_t s, uint32_t epoch) {
  uint32_t ctr[4] = {elem >> 2, h, s, epoch};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32(7, ctr, key, out);
  return out[elem & 3u];
}

/* ------------------------------------------------------------------------- */
/* Number formats, from their definitions.
 *   bf16: IEEE binary32 with the low 16 fraction bits dropped (7 fraction
 *         bits, exponent range of fp32).
 *   f16:  IEEE binary16 (10 fraction bits, normal exponents -14..15).
 *   e4m3: OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 fraction bits;
 *         subnormals m*2^-9; largest finite 448; S.1111.111 is NaN; no inf.
 *   int8: symmetric codes -127..127.
 * A value is rounded onto a format's grid; then encoded exactly.            */
/* ------------------------------------------------------------------------- */
#define BF16_MAXF ldexpf(255.0f, 120) /* (2 - 2^-7) * 2^127 */
#define F16_MAXF 65504.0f
#define E4M3_MAXF 448.0f

/* quantum of the grid with `mbits` fraction bits and lowest normal exponent
 * `emin` at magnitude a (a = 0 gives the subnormal quantum). */
static float grid_quantum(float a, int mbits, int emin) {
  int e = emin;
  if (a > 0.0f) {
    int fe;
    frexpf(a, &fe); /* a = f 2^fe, f in [0.5, 1) */
    e = fe - 1;
    if (e < emin) e = emin;
  }
  return ldexpf(1.0f, e - mbits);
}

/* round to nearest, ties to even, saturating at maxf (mbits < 0: unit grid) */
static float round_nearest_grid(float v, int mbits, int emin, float maxf) {
  float a = fabsf(v);
  float q = mbits < 0 ? 1.0f : grid_quantum(a, mbits, emin);
  float n = rintf(a / q); /* a/q is exact: q is a power of two */
  float mag = n * q;
  if (mag > maxf) mag = maxf;
  return copysignf(mag, v);
}

/* stochastic rounding: round |v| up to the next grid point with probability
 * equal to the fractional distance, using u = (rnd >> 8) * 2^-24. */
static float round_stochastic_grid(float v, int mbits, int emin, float maxf, uint32_t rnd) {
  float a = fabsf(v);
  float q = mbits < 0 ? 1.0f : grid_quantum(a, mbits, emin);
  float ratio = a / q;   /* exact */
  float n = floorf(ratio);
  float f = ratio - n;   /* exact */
  float u = (float)(rnd >> 8) * (1.0f / 16777216.0f);
  float mag = (u < f ? n + 1.0f : n) * q;
  if (mag > maxf) mag = maxf;
  return copysignf(mag, v);
}

uint16_t orc_bf16_encode(float g) { return (uint16_t)(f2u(g) >> 16); } /* g on the bf16 grid */
float orc_bf16_decode(uint16_t b) { return u2f((uint32_t)b << 16); }

uint16_t orc_f16_encode(float g) { /* g on the f16 grid, |g| <= 65504 */
  uint16_t sign = signbit(g) ? 0x8000u : 0u;
  float a = fabsf(g);
  if (a == 0.0f) return sign;
  int fe;
  frexpf(a, &fe);
  int e = fe - 1;
  if (e < -14) return (uint16_t)(sign | (uint16_t)(a / ldexpf(1.0f, -24)));
  uint32_t mant = (uint32_t)(a / ldexpf(1.0f, e - 10)) - 1024u;
  return (uint16_t)(sign | (uint32_t)(e + 15) << 10 | mant);
}
float orc_f16_decode(uint16_t h) {
  float sign = (h & 0x8000u) ? -1.0f : 1.0f;
  int ex = (h >> 10) & 0x1f, m = h & 0x3ff;
  if (ex == 0x1f) return m ? NAN : sign * INFINITY;
  if (ex == 0) return sign * ldexpf((float)m, -24);
  return sign * ldexpf((float)(1024 + m), ex - 25);
}

uint8_t orc_e4m3_encode(float g) { /* g on the e4m3 grid, |g| <= 448 */
  uint8_t sign = signbit(g) ? 0x80u : 0u;
  float a = fabsf(g);
  if (a == 0.0f) return sign;
  int fe;
  frexpf(a, &fe);
  int e = fe - 1;
  if (e < -6) return (uint8_t)(sign | (uint8_t)(a / ldexpf(1.0f, -9)));
  uint32_t mant = (uint32_t)(a / ldexpf(1.0f, e - 3)) - 8u;
  return (uint8_t)(sign | (uint32_t)(e + 7) << 3 | mant);
}
float orc_e4m3_decode(uint8_t c) {
  float sign = (c & 0x80u) ? -1.0f : 1.0f;
  int ex = (c >> 3) & 0xf, m = c & 0x7;
  if (ex == 0xf && m == 0x7) return NAN;
  if (ex == 0) return sign * ldexpf((float)m, -9);
  return sign * ldexpf((float)(8 + m), ex - 10);
}

/* FP4 E2M1 (OCP microscaling formats): 1 sign, 2 exponent bits (bias 1), 1
 * fraction bit; magnitudes 0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6; no inf or
 * NaN.  Code = sign << 3 | exponent << 1 | fraction.                        */
#define E2M1_MAXF 6.0f
uint8_t orc_e2m1_encode(float g) { /* g on the e2m1 grid, |g| <= 6 */
  uint8_t sign = signbit(g) ? 0x8u : 0u;
  float a = fabsf(g);
  if (a < 1.0f) return (uint8_t)(sign | (uint8_t)(a / 0.5f)); /* 0 or the subnormal 0.5 */
  int fe;
  frexpf(a, &fe);
  int e = fe - 1; /* 0..2 */
  uint32_t frac = (uint32_t)(a / ldexpf(1.0f, e - 1)) - 2u;
  return (uint8_t)(sign | (uint32_t)(e + 1) << 1 | frac);
}
float orc_e2m1_decode(uint8_t c) {
  float sign = (c & 0x8u) ? -1.0f : 1.0f;
  int ex = (c >> 1) & 0x3, m = c & 0x1;
  if (ex == 0) return sign * 0.5f * (float)m;
  return sign * ldexpf((float)(2 + m), ex - 2);
}

/* Round-to-nearest conversions used for plain data (y output, tests). */
uint16_t orc_f32_to_bf16(float v) { return orc_bf16_encode(round_nearest_grid(v, 7, -126, BF16_MAXF)); }
uint16_t orc_f32_to_f16(float v) { return orc_f16_encode(round_nearest_grid(v, 10, -14, F16_MAXF)); }
uint8_t orc_f32_to_e4m3(float v) { return orc_e4m3_encode(round_nearest_grid(v, 3, -6, E4M3_MAXF)); }
uint8_t orc_f32_to_e2m1(float v) { return orc_e2m1_encode(round_nearest_grid(v, 1, 0, E2M1_MAXF)); }

static int dtype_bytes(int dt) {
  switch (dt) {
    case ORC_F32: return 4;
    case ORC_BF16: case ORC_F16: return 2;
    default: return 1;
  }
}
static int dtype_is_8bit(int dt) { return dt == ORC_I8 || dt == ORC_E4M3; }
static int read_dtype_ok(int dt) { return dt == ORC_I8 || dt == ORC_E4M3 || dt == ORC_NVFP4; }

/* ------------------------------------------------------------------------- */
/* NVFP4 read checkpoint of one (slot, head, d) row.  Reading of [vAPI]
 * initialize_replayssm_state (NVFP4 branch): the slot's global scale is the
 * largest magnitude of its FP32 state divided by 6 * 448 (the E2M1 maximum
 * times the E4M3 maximum), 1 for an all-zero state; it is set at init and kept
 * by the slot's later flushes.  Each block of 16 consecutive dstate values
 * takes an E4M3 scale sf = e4m3_nearest(block max / (6 gs)) (saturating at
 * 448), and each value the E2M1 code nearest to v * (1 / (gs * sf)) (one
 * rounded reciprocal per block, as the 8-bit row scales; saturating at 6; a
 * block whose scale rounds to 0 is all zeros).  Decoded value:
 * e2m1(code) * sf * gs.  Nearest rounding throughout ([vS] Claims: read
 * checkpoints use nearest encoding).                                       */
/* ------------------------------------------------------------------------- */
#define NVFP4_BLOCK 16
static void quantize_row_nvfp4(const float *acc, float gs, uint8_t *codes /* 64 bytes */, uint8_t *sf /* 8 */) {
  for (int blk = 0; blk < N_DIM / NVFP4_BLOCK; ++blk) {
    const float *v = acc + blk * NVFP4_BLOCK;
    float bmax = 0.0f;
    for (int i = 0; i < NVFP4_BLOCK; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
    uint8_t sc = orc_f32_to_e4m3(bmax / (6.0f * gs));
    sf[blk] = sc;
    float q = orc_e4m3_decode(sc) * gs;
    float inv = q > 0.0f ? 1.0f / q : 0.0f; /* one reciprocal per block, as the 8-bit row scales */
    for (int i = 0; i < NVFP4_BLOCK; i += 2) {
      uint8_t c0 = 0, c1 = 0;
      if (q > 0.0f) {
        c0 = orc_f32_to_e2m1(v[i] * inv);
        c1 = orc_f32_to_e2m1(v[i + 1] * inv);
      }
      codes[(blk * NVFP4_BLOCK + i) / 2] = (uint8_t)(c0 | c1 << 4); /* even element in the low nibble */
    }
  }
}

/* Exported for direct tests of the NVFP4 row encoder. */
void orc_quantize_rows_nvfp4(const float *acc, int rows, float gs, uint8_t *codes, uint8_t *sf) {
  for (int i = 0; i < rows; ++i) quantize_row_nvfp4(acc + (size_t)i * N_DIM, gs, codes + (size_t)i * 64, sf + (size_t)i * 8);
}

/* The slot's NVFP4 global scale from its FP32 state (all heads). */
float orc_nvfp4_global_scale(const float *state, long n) {
  float m = 0.0f;
  for (long i = 0; i < n; ++i) m = fmaxf(m, fabsf(state[i]));
  return m > 0.0f ? m / (6.0f * 448.0f) : 1.0f;
}

/* ------------------------------------------------------------------------- */
/* Checkpoint quantiser.  [vS] commit notes: quantised checkpoints carry FP32
 * per-row scales; [vAPI] initialize_replayssm_state launches one program per
 * (state, head*64 + d) row.  Reading: one fp32 scale per (slot, head, d) over
 * the 128 dstate values; scale = amax / QMAX (QMAX 127 for int8, 448 for
 * e4m3), an all-zero (or < 2^-100) row gets scale 1 (as the NVFP4 global
 * scale in initialize_replayssm_state falls back to 1 for a zero maximum).
 * Rounding: nearest ([vS] Claims: read checkpoints are encoded to nearest) or
 * stochastic with the Philox word above.                                    */
/* ------------------------------------------------------------------------- */
static void quantize_row(int dtype, int rounding, const float *acc, uint32_t h, uint32_t s, uint32_t d,
                         uint32_t epoch, uint64_t seed, void *dst_row, float *scale_out) {
  int sr = rounding == ORC_STOCHASTIC;
  if (dtype == ORC_F32) {
    memcpy(dst_row, acc, N_DIM * sizeof(float));
    return;
  }
  if (dtype == ORC_BF16 || dtype == ORC_F16) {
    uint16_t *o = (uint16_t *)dst_row;
    int mb = dtype == ORC_BF16 ? 7 : 10, emin = dtype == ORC_BF16 ? -126 : -14;
    float mx = dtype == ORC_BF16 ? BF16_MAXF : F16_MAXF;
    for (int n = 0; n < N_DIM; ++n) {
      float g = sr ? round_stochastic_grid(acc[n], mb, emin, mx, orc_sr_word(seed, d * N_DIM + n, h, s, epoch))
                   : round_nearest_grid(acc[n], mb, emin, mx);
      o[n] = dtype == ORC_BF16 ? orc_bf16_encode(g) : orc_f16_encode(g);
    }
    return;
  }
  /* 8-bit */
  float qmax = dtype == ORC_I8 ? 127.0f : 448.0f;
  float amax = 0.0f;
  for (int n = 0; n < N_DIM; ++n) amax = fmaxf(amax, fabsf(acc[n]));
  float scale = amax < 0x1p-100f ? 1.0f : amax / qmax;
  float inv = 1.0f / scale;
  *scale_out = scale;
  for (int n = 0; n < N_DIM; ++n) {
    float v = acc[n] * inv;
    uint32_t rnd = sr ? orc_sr_word(seed, d * N_DIM + n, h, s, epoch) : 0u;
    if (dtype == ORC_I8) {
      float g = sr ? round_stochastic_grid(v, -1, 0, 127.0f, rnd) : round_nearest_grid(v, -1, 0, 127.0f);
      ((int8_t *)dst_row)[n] = (int8_t)g;
    } else {
      float g = sr ? round_stochastic_grid(v, 3, -6, E4M3_MAXF, rnd) : round_nearest_grid(v, 3, -6, E4M3_MAXF);
      ((uint8_t *)dst_row)[n] = orc_e4m3_encode(g);
    }
  }
}

/* Exported for direct quantiser tests: rows x 128 accumulators of head h,
 * slot s; row i uses d = d0 + i in the random counter. */
void orc_quantize_rows(int dtype, int rounding, const float *acc, int rows, uint32_t d0, uint32_t h, uint32_t s,
                       uint32_t epoch, uint64_t seed, void *codes, float *scales) {
  int eb = dtype_bytes(dtype);
  for (int i = 0; i < rows; ++i)
    quantize_row(dtype, rounding, acc + (size_t)i * N_DIM, h, s, d0 + (uint32_t)i, epoch, seed,
                 (char *)codes + (size_t)i * N_DIM * eb, scales ? scales + i : NULL);
}

/* The fp32 value of state element (d, n) of head h in slot s: exact for
 * float formats; code * scale_d (one rounded multiply) for 8-bit codes. */
static float state_f32(const orc_cache *c, int s, int h, int d, int n) {
  size_t off = (size_t)s * c->state_slot_stride + ((size_t)h * P_DIM + d) * N_DIM + n;
  switch (c->state_dtype) {
    case ORC_F32: return ((const float *)c->state)[off];
    case ORC_BF16: return orc_bf16_decode(((const uint16_t *)c->state)[off]);
    case ORC_F16: return orc_f16_decode(((const uint16_t *)c->state)[off]);
    case ORC_I8: {
      float sc = c->scale[(size_t)s * c->scale_slot_stride + (size_t)h * P_DIM + d];
      return (float)((const int8_t *)c->state)[off] * sc;
    }
    default: {
      float sc = c->scale[(size_t)s * c->scale_slot_stride + (size_t)h * P_DIM + d];
      return orc_e4m3_decode(((const uint8_t *)c->state)[off]) * sc;
    }
  }
}

static void store_state_head(const orc_cache *c, int s, int h, const float *acc /*[64][128]*/, uint32_t epoch,
                             uint64_t seed) {
  int eb = dtype_bytes(c->state_dtype);
  for (int d = 0; d < P_DIM; ++d) {
    size_t off = (size_t)s * c->state_slot_stride + ((size_t)h * P_DIM + d) * N_DIM;
    float *sc = dtype_is_8bit(c->state_dtype) ? &c->scale[(size_t)s * c->scale_slot_stride + (size_t)h * P_DIM + d]
                                              : NULL;
    quantize_row(c->state_dtype, c->rounding, acc + (size_t)d * N_DIM, (uint32_t)h, (uint32_t)s, (uint32_t)d,
                 epoch, seed, (char *)c->state + off * eb, sc);
    if (c->read_state && c->read_dtype == ORC_NVFP4) { /* the read checkpoint: the same fp32 row */
      size_t roff = (size_t)s * c->read_slot_stride + ((size_t)h * P_DIM + d) * (N_DIM / 2);
      size_t soff = (size_t)s * c->read_sf_stride + ((size_t)h * P_DIM + d) * (N_DIM / NVFP4_BLOCK);
      quantize_row_nvfp4(acc + (size_t)d * N_DIM, c->read_gs[s], (uint8_t *)c->read_state + roff, c->read_sf + soff);
    } else if (c->read_state) { /* the read checkpoint: the same fp32 row, nearest */
      size_t roff = (size_t)s * c->read_slot_stride + ((size_t)h * P_DIM + d) * N_DIM;
      quantize_row(c->read_dtype, ORC_NEAREST, acc + (size_t)d * N_DIM, (uint32_t)h, (uint32_t)s, (uint32_t)d,
                   epoch, seed, (uint8_t *)c->read_state + roff,
                   &c->read_scale[(size_t)s * c->read_scale_stride + (size_t)h * P_DIM + d]);
    }
  }
}

/* The fp32 value of S0 element (d, n) the step's readout uses: the read
 * checkpoint's code * scale when there is one, else the recurrence state. */
static float readout_f32(const orc_cache *c, int s, int h, int d, int n) {
  if (!c->read_state) return state_f32(c, s, h, d, n);
  if (c->read_dtype == ORC_NVFP4) {
    size_t row = (size_t)h * P_DIM + d;
    uint8_t byte = ((const uint8_t *)c->read_state)[(size_t)s * c->read_slot_stride + row * (N_DIM / 2) + n / 2];
    uint8_t code = (n & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xfu);
    uint8_t sc = c->read_sf[(size_t)s * c->read_sf_stride + row * (N_DIM / NVFP4_BLOCK) + n / NVFP4_BLOCK];
    return orc_e2m1_decode(code) * orc_e4m3_decode(sc) * c->read_gs[s];
  }
  size_t off = (size_t)s * c->read_slot_stride + ((size_t)h * P_DIM + d) * N_DIM + n;
  float sc = c->read_scale[(size_t)s * c->read_scale_stride + (size_t)h * P_DIM + d];
  if (c->read_dtype == ORC_I8) return (float)((const int8_t *)c->read_state)[off] * sc;
  return orc_e4m3_decode(((const uint8_t *)c->read_state)[off]) * sc;
}

/* ------------------------------------------------------------------------- */
/* Ring buffers.  [FI] Description item 2 (ring-buffer cache contract): with
 * L = max_window + npredicted, live token j of a slot sits at physical
 * position (ring_start + j) mod L for j < pnat, and the i-th new token is
 * appended at (ring_start + pnat + i) mod L.  x_cache is [slot][H][L][64],
 * B_cache [slot][G][L][128], dt_cache [slot][H][L] holding dt' (post
 * softplus).                                                                */
/* ------------------------------------------------------------------------- */
static inline int ring_len(const orc_cache *c) { return c->max_window + c->npredicted; }
static inline uint16_t *x_row(const orc_cache *c, int s, int h, int pos) {
  return c->x_cache + (size_t)s * c->x_slot_stride + ((size_t)h * ring_len(c) + pos) * P_DIM;
}
static inline uint16_t *b_row(const orc_cache *c, int s, int g, int pos) {
  return c->B_cache + (size_t)s * c->B_slot_stride + ((size_t)g * ring_len(c) + pos) * N_DIM;
}
static inline float *dt_at(const orc_cache *c, int s, int h, int pos) {
  return c->dt_cache + (size_t)s * c->dt_slot_stride + (size_t)h * ring_len(c) + pos;
}

/* Row b's token range: cu_seqlens packs rows on the batch side only ([FI]
 * varlen commit note: a row starts at cu_seqlens[b], its token mask uses its
 * own length, cache indexing does not change); without it every row has T. */
static void row_tokens(const int32_t *cu, int b, int T, int *tok0, int *Tb) {
  if (cu) {
    *tok0 = cu[b];
    *Tb = cu[b + 1] - cu[b];
  } else {
    *tok0 = b * T;
    *Tb = T;
  }
}

/* Slot 0 is padding and ids outside [1, S) are ignored ([vAPI] module
 * docstring and initialize_replayssm_state docstring). */
static inline int slot_active(const orc_cache *c, int s) { return s >= 1 && s < c->num_slots; }

static int check_cache(const orc_cache *c) {
  if (!c || c->nheads <= 0 || c->ngroups <= 0 || c->nheads % c->ngroups) return -1;
  if (c->read_state && !read_dtype_ok(c->read_dtype)) return -1;
  if (c->read_state && c->read_dtype != ORC_NVFP4 && !c->read_scale) return -1;
  if (c->read_state && c->read_dtype == ORC_NVFP4 && (!c->read_sf || !c->read_gs)) return -1;
  if (c->max_window < 0 || c->npredicted < 1 || c->max_window + c->npredicted > 256) return -1;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Init ([vAPI] initialize_replayssm_state): quantise FP32 prefill states
 * [n][H][64][128] into the checkpoint of slot ids[i] (flush epoch 0), clear
 * the rings and the slot's ring_start and epoch.  Ids <= 0 or >= S are
 * ignored.                                                                  */
/* ------------------------------------------------------------------------- */
int orc_init_state(const orc_cache *c, const float *states, const int32_t *ids, int32_t n, uint64_t seed) {
  if (check_cache(c)) return -1;
  int H = c->nheads, G = c->ngroups, L = ring_len(c);
  for (int i = 0; i < n; ++i) {
    int s = ids[i];
    if (!slot_active(c, s)) continue;
    if (c->read_state && c->read_dtype == ORC_NVFP4) /* the slot's global scale, from all its heads */
      c->read_gs[s] = orc_nvfp4_global_scale(states + (size_t)i * H * P_DIM * N_DIM, (long)H * P_DIM * N_DIM);
    for (int h = 0; h < H; ++h)
      store_state_head(c, s, h, states + ((size_t)i * H + h) * P_DIM * N_DIM, 0u, seed);
    for (int h = 0; h < H; ++h)
      for (int pos = 0; pos < L; ++pos) {
        memset(x_row(c, s, h, pos), 0, P_DIM * sizeof(uint16_t));
        *dt_at(c, s, h, pos) = 0.0f;
      }
    for (int g = 0; g < G; ++g)
      for (int pos = 0; pos < L; ++pos) memset(b_row(c, s, g, pos), 0, N_DIM * sizeof(uint16_t));
    c->ring_start[s] = 0;
    c->flush_epoch[s] = 0u;
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Flush.  [FI] commit notes (persistent Triton path): the write decision is
 * taken per slot at run time as is_write = (prev_k + T) > max_window, and the
 * write path folds the old tokens into the state by replaying them; [vS]
 * Details: only the accepted prefix may change the canonical checkpoint,
 * rejected drafts never enter it.  For a flagged row
 * with p live tokens:
 *   c_j   = sum_{i<=j} A dt'_i          (sequential fp32, i ascending)
 *   c_end = c_{p-1} (0 if p = 0)
 *   S0'   = e^{c_end} S0 + sum_j e^{c_end - c_j} dt'_j x_j (x) B_j
 * in canonical fp32: acc = spec_exp(c_end) * S0f; for j ascending
 *   acc = fmaf(u_j[d], B_j[n], acc),  u_j[d] = (spec_exp(c_end - c_j) dt'_j) x_j[d];
 * then the quantiser with the slot's new epoch.  Afterwards ring_start
 * advances by p (mod L), pnat = 0, epoch += 1 ([FI] item 2: a flush advances
 * ring_start).  force = 1 flushes every active row.              */
/* ------------------------------------------------------------------------- */
static void flush_unit(const orc_cache *c, int s, int h, int p, int r, float A, uint32_t epoch, uint64_t seed,
                       float *acc /*[64*128] scratch*/) {
  int L = ring_len(c), hpg = c->nheads / c->ngroups, g = h / hpg;
  float cum[256], dtp[256];
  float cval = 0.0f;
  for (int j = 0; j < p; ++j) {
    dtp[j] = *dt_at(c, s, h, (r + j) % L);
    cval = cval + A * dtp[j];
    cum[j] = cval;
  }
  float c_end = p > 0 ? cum[p - 1] : 0.0f;
  float decay = orc_spec_exp(c_end);
  for (int d = 0; d < P_DIM; ++d)
    for (int n = 0; n < N_DIM; ++n) acc[d * N_DIM + n] = decay * state_f32(c, s, h, d, n);
  for (int j = 0; j < p; ++j) {
    float w = orc_spec_exp(c_end - cum[j]) * dtp[j];
    const uint16_t *xr = x_row(c, s, h, (r + j) % L);
    const uint16_t *br = b_row(c, s, g, (r + j) % L);
    for (int d = 0; d < P_DIM; ++d) {
      float u = w * orc_bf16_decode(xr[d]);
      for (int n = 0; n < N_DIM; ++n) acc[d * N_DIM + n] = fmaf(u, orc_bf16_decode(br[n]), acc[d * N_DIM + n]);
    }
  }
  store_state_head(c, s, h, acc, epoch, seed);
}

int orc_flush(const orc_cache *c, const float *A, const int32_t *slot_idx, int32_t *pnat, const int32_t *cu,
              int32_t batch, int32_t T, int32_t force, uint64_t seed, int nthreads) {
  if (check_cache(c) || T < 0 || batch < 0) return -1;
  int H = c->nheads, L = ring_len(c), W = c->max_window;
  int *flag = (int *)calloc((size_t)(batch > 0 ? batch : 1), sizeof(int));
  for (int b = 0; b < batch; ++b) {
    int s = slot_idx[b];
    if (!slot_active(c, s)) continue;
    int tok0, Tb;
    row_tokens(cu, b, T, &tok0, &Tb);
    if (Tb < 0 || Tb > T) { set_err(c->error_word, ORC_ERR_SEQLEN); continue; }
    int p = pnat[b];
    if (p < 0 || p > L) { set_err(c->error_word, ORC_ERR_PNAT); continue; }
    flag[b] = force ? 1 : (p + Tb > W);
  }
  long units = (long)batch * H;
  (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
#endif
  {
    float *acc = (float *)malloc(sizeof(float) * P_DIM * N_DIM);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
    for (long u = 0; u < units; ++u) {
      int b = (int)(u / H), h = (int)(u % H);
      if (!flag[b]) continue;
      int s = slot_idx[b];
      flush_unit(c, s, h, pnat[b], c->ring_start[s], A[h], c->flush_epoch[s] + 1u, seed, acc);
    }
    free(acc);
  }
  for (int b = 0; b < batch; ++b) {
    if (!flag[b]) continue;
    int s = slot_idx[b];
    c->ring_start[s] = (c->ring_start[s] + pnat[b]) % L;
    pnat[b] = 0;
    c->flush_epoch[s] += 1u;
  }
  free(flag);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Step (replay/readout + append).  For row b (slot s, p live tokens, T_b new
 * tokens) and head h, with the live ring followed by the new tokens as one
 * logical sequence k = 0 .. p+T_b-1:
 *   dt'_k = softplus(dt + dt_bias) for new tokens ([vAPI]), dt_cache for live
 *   c_k   = sum_{i<=k} A dt'_i            (sequential fp32; [FI] item 2: the
 *           decay is not cached but recomputed from the dt ring)
 *   y_t   = e^{c_{p+t}} (S0 C_t) + sum_{k<=p+t} e^{c_{p+t}-c_k} dt'_k (C_t.B_k) x_k
 *           + D x_t
 * (the replay of [FI] Description item 1: C.B contraction, cumulative A dt
 * decays, state replay + output projection), evaluated in double and
 * rounded to bf16 once; with an output gate z ([bf16 tok][H][64], nullable),
 * y_t[d] * silu(z_t[d]) in double before that rounding (the gated output of
 * Mamba-2's selective state update; [FI] commit notes list z among the
 * operands the monolithic kernel stages with x).
 * New x, B, dt' are appended at (r + p + t) mod L.
 * Rows whose slot is inactive, or which fail a range check, get y = 0 and
 * touch no cache.                                                           */
/* ------------------------------------------------------------------------- */
int orc_step(const orc_cache *c, const uint16_t *x, const float *dt, const float *A, const uint16_t *B,
             const uint16_t *C, const float *D, const float *dt_bias, const int32_t *slot_idx, const int32_t *pnat,
             const int32_t *cu, int32_t batch, int32_t T, const uint16_t *z, uint16_t *out, double *out_f64,
             int nthreads) {
  if (check_cache(c) || T < 0 || batch < 0) return -1;
  int H = c->nheads, G = c->ngroups, hpg = H / G, L = ring_len(c);
  /* validate rows first (sets the error bits once per row) */
  int *ok = (int *)calloc((size_t)(batch > 0 ? batch : 1), sizeof(int));
  for (int b = 0; b < batch; ++b) {
    int tok0, Tb;
    row_tokens(cu, b, T, &tok0, &Tb);
    int s = slot_idx[b];
    if (!slot_active(c, s)) continue;
    if (Tb < 0 || Tb > T) { set_err(c->error_word, ORC_ERR_SEQLEN); continue; }
    int p = pnat[b];
    if (p < 0 || p + Tb > L) { set_err(c->error_word, ORC_ERR_PNAT); continue; }
    ok[b] = 1;
  }
  long units = (long)batch * H;
  (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
#endif
  {
    float *xk = (float *)malloc(sizeof(float) * 256 * P_DIM);
    float *bk = (float *)malloc(sizeof(float) * 256 * N_DIM);
    float *s0 = (float *)malloc(sizeof(float) * P_DIM * N_DIM);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
    for (long u = 0; u < units; ++u) {
      int b = (int)(u / H), h = (int)(u % H), g = h / hpg;
      int tok0, Tb;
      row_tokens(cu, b, T, &tok0, &Tb);
      if (!ok[b]) {
        if (Tb > 0 && Tb <= T && (cu == NULL || tok0 >= 0))
          for (int t = 0; t < Tb; ++t)
            for (int d = 0; d < P_DIM; ++d) {
              size_t o = ((size_t)(tok0 + t) * H + h) * P_DIM + d;
              out[o] = 0;
              if (out_f64) out_f64[o] = 0.0;
            }
        continue;
      }
      int s = slot_idx[b], p = pnat[b], r = c->ring_start[s], K = p + Tb;
      float dtp[256], cum[256];
      for (int k = 0; k < p; ++k) {
        int pos = (r + k) % L;
        for (int d = 0; d < P_DIM; ++d) xk[k * P_DIM + d] = orc_bf16_decode(x_row(c, s, h, pos)[d]);
        for (int n = 0; n < N_DIM; ++n) bk[k * N_DIM + n] = orc_bf16_decode(b_row(c, s, g, pos)[n]);
        dtp[k] = *dt_at(c, s, h, pos);
      }
      for (int t = 0; t < Tb; ++t) {
        int k = p + t;
        size_t tok = (size_t)(tok0 + t);
        for (int d = 0; d < P_DIM; ++d) xk[k * P_DIM + d] = orc_bf16_decode(x[(tok * H + h) * P_DIM + d]);
        for (int n = 0; n < N_DIM; ++n) bk[k * N_DIM + n] = orc_bf16_decode(B[(tok * G + g) * N_DIM + n]);
        dtp[k] = orc_spec_softplus(dt[tok * H + h] + dt_bias[h]);
      }
      float cv = 0.0f;
      for (int k = 0; k < K; ++k) {
        cv = cv + A[h] * dtp[k];
        cum[k] = cv;
      }
      for (int d = 0; d < P_DIM; ++d)
        for (int n = 0; n < N_DIM; ++n) s0[d * N_DIM + n] = readout_f32(c, s, h, d, n);
      for (int t = 0; t < Tb; ++t) {
        size_t tok = (size_t)(tok0 + t);
        const uint16_t *ct = C + (tok * G + g) * N_DIM;
        double cf[N_DIM];
        for (int n = 0; n < N_DIM; ++n) cf[n] = orc_bf16_decode(ct[n]);
        int kt = p + t;
        double coef[256];
        for (int k = 0; k <= kt; ++k) {
          double cb = 0.0;
          for (int n = 0; n < N_DIM; ++n) cb += cf[n] * (double)bk[k * N_DIM + n];
          coef[k] = exp((double)cum[kt] - (double)cum[k]) * (double)dtp[k] * cb;
        }
        double decay = exp((double)cum[kt]);
        for (int d = 0; d < P_DIM; ++d) {
          double sc = 0.0;
          for (int n = 0; n < N_DIM; ++n) sc += (double)s0[d * N_DIM + n] * cf[n];
          double ring = 0.0;
          for (int k = 0; k <= kt; ++k) ring += coef[k] * (double)xk[k * P_DIM + d];
          double yv = decay * sc + ring + (double)D[h] * (double)xk[kt * P_DIM + d];
          size_t o = (tok * H + h) * P_DIM + d;
          if (z) { /* output gate: y * silu(z), silu(v) = v / (1 + e^-v) */
            double zv = orc_bf16_decode(z[o]);
            yv *= zv / (1.0 + exp(-zv));
          }
          out[o] = orc_f32_to_bf16((float)yv);
          if (out_f64) out_f64[o] = yv;
        }
      }
      /* append the new tokens after the live prefix */
      for (int t = 0; t < Tb; ++t) {
        int pos = (r + p + t) % L;
        size_t tok = (size_t)(tok0 + t);
        memcpy(x_row(c, s, h, pos), x + (tok * H + h) * P_DIM, P_DIM * sizeof(uint16_t));
        *dt_at(c, s, h, pos) = dtp[p + t];
        if (h % hpg == 0) memcpy(b_row(c, s, g, pos), B + (tok * G + g) * N_DIM, N_DIM * sizeof(uint16_t));
      }
    }
    free(xk);
    free(bk);
    free(s0);
  }
  free(ok);
  return 0;
}

/* Commit accepted drafts: the first accepted[b] appended tokens of row b join
 * the live prefix (pnat += accepted).  The rest stay outside the live prefix
 * and are overwritten by later appends ([vS] Details: rejected drafts never
 * reach the canonical state). */
int orc_accept(const orc_cache *c, const int32_t *slot_idx, int32_t *pnat, const int32_t *accepted,
               const int32_t *cu, int32_t batch, int32_t T) {
  if (check_cache(c) || T < 0 || batch < 0) return -1;
  int L = ring_len(c);
  for (int b = 0; b < batch; ++b) {
    int s = slot_idx[b];
    if (!slot_active(c, s)) continue;
    int tok0, Tb;
    row_tokens(cu, b, T, &tok0, &Tb);
    if (Tb < 0 || Tb > T) { set_err(c->error_word, ORC_ERR_SEQLEN); continue; }
    int a = accepted[b];
    if (a < 0 || a > Tb) { set_err(c->error_word, ORC_ERR_ACCEPT); continue; }
    if (pnat[b] < 0 || pnat[b] + a > L) { set_err(c->error_word, ORC_ERR_PNAT); continue; }
    pnat[b] += a;
  }
  return 0;
}

/* vectorised helpers for tests */
void orc_spec_exp_n(const float *x, float *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_spec_exp(x[i]); }
void orc_spec_log1p_n(const float *x, float *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_spec_log1p(x[i]); }
void orc_spec_softplus_n(const float *x, float *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_spec_softplus(x[i]); }
void orc_f32_to_bf16_n(const float *x, uint16_t *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_f32_to_bf16(x[i]); }
void orc_f32_to_f16_n(const float *x, uint16_t *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_f32_to_f16(x[i]); }
void orc_f32_to_e4m3_n(const float *x, uint8_t *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_f32_to_e4m3(x[i]); }
void orc_f16_decode_n(const uint16_t *x, float *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_f16_decode(x[i]); }
void orc_e4m3_decode_n(const uint8_t *x, float *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_e4m3_decode(x[i]); }
void orc_f32_to_e2m1_n(const float *x, uint8_t *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_f32_to_e2m1(x[i]); }
void orc_e2m1_decode_n(const uint8_t *x, float *y, long n) { for (long i = 0; i < n; ++i) y[i] = orc_e2m1_decode(x[i]); }
int orc_have_openmp(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 0;
#endif
}
