// lamp_common.cuh -- shapes, shared-memory layout arithmetic and exact
// 8-bit helpers shared by the LampAttention kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "lamp_ptx.cuh"

namespace lamp {

constexpr int kBM = 128;        // query rows per CTA (one TMEM lane per row)
constexpr int kBN = 64;         // keys per step = one 64-key tile of the method
constexpr int kNC = 32;             // logits per softmax thread per step
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSweepTaus = 8;    // tau values per sweep call
struct SweepCodes {
  int v[kMaxSweepTaus];  // per tau: the smallest sub-block code flagged at it
};

// Kernel parameters (passed by value as a __grid_constant__).
struct FwdParams {
  CUtensorMap tmQ8, tmQ16, tmK8, tmK16, tmV;
  CUtensorMap tmV8;    // FP8 P.V: V8t = fl8(v) as [B, Hkv, D, keys] (keys contiguous)
  void* out;
  float* lse;
  uint8_t* mask;
  unsigned long long* counters;
  uint32_t* records;   // tau-sweep pass: [B, Hq, T, T] tile records
  const float* nq;     // [B, Hq, N]   ||fl8(q_r)||_2 (upper bound)
  const float* nkmax;  // [B, Hkv, T]  max over the tile of ||fl8(k_c)||_2
  const float* nqc;    // [B, Hq, N, D/32] the same per 32-element chunk of d
  const float* nkc;    // [B, Hkv, T, D/32] max over the tile of the chunk norms, + 2^-6
  long long o_stride[3];
  int B, N, Hq, Hkv, T, nqb;
  int window, mask_kind, force, out_f32;
  int q8_in_cta;        // bf16 q: Q8 = fl8(Q16 tile) in shared memory, row norms in the kernel
  float sigma_f;       // softmax scale rounded to float
  double sigma_d;      // softmax scale in double
  double sig18;        // sigma_d * 2^-18 (exact re-derivations: acc * sig18 = A sigma)
  float guard;         // relative bound on |y_tc - y| per unit sigma*|q|*|k|
  float tau_abs;       // flag iff |S8| >= tau_abs (derived from tau)
  uint32_t delta_code; // stage 1 iff P8 code >= delta_code
  uint8_t exp8[256];   // code of fl8(exp(x)) for every E4M3 code x
  unsigned long long timeout_ns;  // a wait gives up after this long
  unsigned int* gabort;           // grid-wide abort word (workspace, zeroed per call)
};

// Pre-pass parameters (see lamp_prep.cu).
struct PrepParams {
  const void* q;
  const void* k;
  const void* v;
  long long qs[3], ks[3], vs[3];  // element strides (B, S, H)
  uint8_t* q8;                    // [B, Hq, N, D]  E4M3
  uint8_t* k8;                    // [B, Hkv, N, D] E4M3
  void* v16;                      // [B, Hkv, N, D] fp16
  void* q16;                      // [B, Hq, N, D]  bf16 (fp32 input only)
  void* k16;                      // [B, Hkv, N, D] bf16 (fp32 input only)
  float* nq;                      // [B, Hq, N]
  float* nkmax;                   // [B, Hkv, T] (zeroed before the launch)
  float* nqc;                     // [B, Hq, N, D/32] chunk norms
  float* nkc;                     // [B, Hkv, T, D/32] max chunk norms + 2^-6 (zeroed before the launch)
  int B, N, Hq, Hkv, T, in_f32;
  int skip_q;   // the fused kernel makes Q8 and the q norms itself
  int skip_kv;  // k / v already prepared (a K/V cache): q rows only
  // division by Hq, Hkv and N as multiply and shift (set by the launcher)
  uint32_t mul_hq, mul_hkv, mul_n;
  int shr_hq, shr_hkv, shr_n;
};

// Byte offset of byte `x` (0 <= x < row_bytes) of row `r` in a K-major
// tile whose rows are `row_bytes` long, stored as 128-byte (or 64-byte when
// row_bytes == 64) swizzled atoms: 8 rows per atom, atoms stacked along the
// rows, columns of atoms (each 128 B of the row) stacked after all rows.
__device__ __forceinline__ uint32_t swz_offset(int r, int x, int rows, int row_bytes) {
  if (row_bytes == 64) {
    int chunk = (x >> 4) ^ ((r >> 1) & 3);
    return (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + chunk * 16 + (x & 15));
  }
  int col = x >> 7, w = x & 127;
  int chunk = (w >> 4) ^ (r & 7);
  return (uint32_t)(col * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + chunk * 16 + (w & 15));
}

// E4M3 codes (low byte: the low element) of fl8(e^x) for the two E4M3 codes
// in x8 (non-positive x); exp8_f16x2 gives their values as f16x2.
__device__ __forceinline__ uint32_t exp8_code2(uint32_t x8) {
  const uint32_t h = e4m3x2_to_f16x2((uint16_t)x8);
  __half2 xv;
  memcpy(&xv, &h, 4);
  const float2 xf = __fmul2_rn(make_float2(__low2float(xv), __high2float(xv)), make_float2(kLog2e, kLog2e));
  return cvt_e4m3x2(ex2_approx(xf.y), ex2_approx(xf.x));
}

// f16x2 values of fl8(e^x) for the two E4M3 codes in x8 (non-positive x):
// e^x in fp32 (ex2 of x log2 e: relative error below 2^-20), then one E4M3
// rounding to nearest even.  Exact for every such code: among the E4M3
// values x <= 0 with e^x >= 2^-11, the one whose e^x lies closest to an E4M3
// rounding boundary is x = -2^-5, at 2^-11 relative -- far beyond the fp32
// error; below 2^-11, e^x rounds to 0 either way.
__device__ __forceinline__ uint32_t exp8_f16x2(uint32_t x8) {
  return e4m3x2_to_f16x2((uint16_t)exp8_code2(x8));
}

// E4M3 value, as f16 bits, of prev + A sigma (chunked logits): A = acc *
// 2^-18 is a chunk's exact dot product, prev the running 8-bit value.  The
// product and the sum are taken in double (the reading's definition; sig18
// = sigma * 2^-18 exactly, so acc * sig18 is the double product A * sigma),
// then rounded to float to odd and to E4M3 (float keeps 24 >= 4 + 2 bits:
// the second rounding is the correctly rounded E4M3 value of the double).
__device__ __forceinline__ uint32_t e4m3_f16_of_chunk_sum(float prev, long long acc, double sig18) {
  const double y = (double)prev + (double)acc * sig18;
  float f = __double2float_rz(y);
  if ((double)f != y) f = __uint_as_float(__float_as_uint(f) | 1u);
  return e4m3x2_to_f16x2(cvt_e4m3x2(0.0f, f)) & 0xFFFFu;
}

// Exact product of two E4M3 codes, times 2^18 (an integer below 2^36): every
// finite code is (significand <= 15) * 2^(shift - 9) with shift in 0..14.
__device__ __forceinline__ long long e4m3_prod_2p18(uint32_t a, uint32_t b) {
  const uint32_t ea = (a >> 3) & 15u, eb = (b >> 3) & 15u;
  const uint32_t ma = ea ? ((a & 7u) | 8u) : (a & 7u);
  const uint32_t mb = eb ? ((b & 7u) | 8u) : (b & 7u);
  const uint32_t sh = (ea ? ea - 1u : 0u) + (eb ? eb - 1u : 0u);
  const long long v = (long long)(ma * mb) << sh;
  return ((a ^ b) & 0x80u) ? -v : v;
}

// E4M3 value, as f16 bits, of the logit with exact dot product acc * 2^-18
// and softmax scale sigma, sig18 = sigma * 2^-18: the product is rounded
// to double precision (one float64 multiply; acc < 2^53 converts exactly),
// which is the reading's y = A sigma, and then to E4M3 (to nearest even,
// saturating to +-448).  The second rounding goes through float32 rounded
// to odd -- truncated, with the last bit set when anything was cut off --
// so that the float32 -> E4M3 rounding to nearest gives the same result as
// one rounding of y (float32 keeps more than two bits beyond E4M3's four).
__device__ __forceinline__ uint32_t e4m3_f16_of_product(long long acc, double sig18) {
  const double y = (double)acc * sig18;
  float f = __double2float_rz(y);
  if ((double)f != y) f = __uint_as_float(__float_as_uint(f) | 1u);
  return e4m3x2_to_f16x2(cvt_e4m3x2(0.0f, f)) & 0xFFFFu;
}

// Host: E4M3 code of the round-to-nearest-even, saturating conversion of a
// double (written from the format definition; NaN -> 0x7F).
inline uint8_t host_e4m3_encode(double x) {
  if (x != x) return 0x7F;
  const uint8_t sign = x < 0 ? 0x80 : 0x00;
  double a = x < 0 ? -x : x;
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int e = 0;
  (void)frexp(a, &e);        // a = f * 2^e, f in [0.5, 1)
  int E = e - 1;             // floor(log2 a)
  if (E < -6) E = -6;
  const double n = nearbyint(ldexp(a, 3 - E));  // RNE at the spacing 2^(E-3)
  int ni = (int)n;
  if (E == -6 && ni < 8) return sign | (uint8_t)ni;   // subnormal
  if (ni == 16) { ni = 8; ++E; }
  if (E > 8 || (E == 8 && ni > 14)) return sign | 0x7E;
  return sign | (uint8_t)(((E + 7) << 3) | (ni - 8));
}

inline double host_e4m3_decode(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return 0.0 / 0.0;
  const double v = e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp((double)m, -9);
  return (c & 0x80) ? -v : v;
}

// exp8 table: code of fl8(exp(x)) for each E4M3 code x.  The double exp is
// far closer than the smallest distance (2^-11 relative) of e^x to an E4M3
// rounding boundary for the codes that matter, so this is correctly rounded.
inline void host_exp8_table(uint8_t* t) {
  for (int c = 0; c < 256; ++c) {
    const double x = host_e4m3_decode((uint8_t)c);
    t[c] = (x != x) ? 0 : host_e4m3_encode(exp(x));
  }
}

// Smallest non-negative E4M3 magnitude whose half-spacing is >= tau
// (+inf if none).  half-spacing(v) = 2^(max(floor(log2 v), -6) - 4), and
// 2^-10 at v = 0.
inline float host_tau_abs(float tau) {
  if (!(tau > 0.0f)) return 0.0f;
  if (tau <= 0x1p-10f) return 0.0f;
  for (int e = -6; e <= 8; ++e) {
    float half = ldexpf(1.0f, e - 4);
    if (half >= tau) return e == -6 ? 0x1p-9f : ldexpf(1.0f, e);
  }
  return __builtin_inff();
}

// tau-sweep records store, per sub-block, log2(largest stage-1 half-ulp8)
// + 11 (1..15; half-ulps of E4M3 run from 2^-10 to 2^4); the sub-block is
// flagged at tau iff its code is >= this (16: never).
inline int host_tau_code(float tau) {
  if (!(tau > 0x1p-10f)) return 1;
  for (int c = 2; c <= 15; ++c)
    if (ldexpf(1.0f, c - 11) >= tau) return c;
  return 16;
}

// Code of the smallest non-negative E4M3 value >= delta (0xFF if none),
// so that P8 >= delta iff code(P8) >= that code (codes of non-negative
// values are ordered like the values).
inline uint32_t host_delta_code(float delta) {
  if (!(delta > 0.0f)) return 0u;
  for (uint32_t c = 0; c <= 0x7E; ++c) {
    uint32_t e = c >> 3, m = c & 7;
    float v = e ? ldexpf(1.0f + m / 8.0f, (int)e - 7) : ldexpf((float)m, -9);
    if (v >= delta) return c;
  }
  return 0xFFu;
}

// ---------------------------------------------------------------- MMA issue
// Shared-memory operand layouts (all 1024-byte aligned):
//   F8 tiles  [rows x D] E4M3, K-major: 128-byte swizzled atom columns of
//             [rows x 128 B] (D = 64: one column of 64-byte swizzled rows).
//   16-bit    [rows x D] BF16/FP16, K-major: D/64 atom columns of
//             [rows x 128 B], 128-byte swizzle.
//   V         [64 keys x D] FP16, MN-major: D/64 regions of [64 keys x 128 B]
//             (64 values of d per key row).
template <int D>
struct Mma {
  static constexpr int F8_ROW = (D == 64) ? 64 : 128;
  // S[128 x 64] (fp32, TMEM) = Q8[128 x D] . K8[64 x D]^T
  static __device__ __forceinline__ void qk8(uint32_t tmem_d, uint32_t q8, uint32_t k8) {
    constexpr uint32_t idesc = make_idesc(0, 0, 0, 128, 64);
    const uint32_t layout = (F8_ROW == 64) ? kLayoutSW64 : kLayoutSW128;
    const uint32_t sbo = (F8_ROW == 64) ? 512u : 1024u;
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
      const int col = (kk * 32) / F8_ROW, off = (kk * 32) % F8_ROW;
      const uint64_t ad = make_sdesc(q8 + col * 128 * 128 + off, 16, sbo, layout);
      const uint64_t bd = make_sdesc(k8 + col * 64 * 128 + off, 16, sbo, layout);
      mma_f8(tmem_d, ad, bd, idesc, kk > 0);
    }
  }
  // Chunked 8-bit logits: S[c][128 x 64] = Q8_c . K8_c^T for each 32-element
  // chunk c of d (one K = 32 instruction each), into its own accumulator 64
  // TMEM columns after the previous one, not summed
  static __device__ __forceinline__ void qk8_chunks(uint32_t tmem_d, uint32_t q8, uint32_t k8) {
    constexpr uint32_t idesc = make_idesc(0, 0, 0, 128, 64);
    const uint32_t layout = (F8_ROW == 64) ? kLayoutSW64 : kLayoutSW128;
    const uint32_t sbo = (F8_ROW == 64) ? 512u : 1024u;
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
      const int col = (kk * 32) / F8_ROW, off = (kk * 32) % F8_ROW;
      const uint64_t ad = make_sdesc(q8 + col * 128 * 128 + off, 16, sbo, layout);
      const uint64_t bd = make_sdesc(k8 + col * 64 * 128 + off, 16, sbo, layout);
      mma_f8(tmem_d + (uint32_t)(kk * 64), ad, bd, idesc, 0u);
    }
  }
  // S16[128 x 64] = Q16[128 x D] . K16[64 x D]^T (BF16)
  static __device__ __forceinline__ void qk16(uint32_t tmem_d, uint32_t q16, uint32_t k16) {
    constexpr uint32_t idesc = make_idesc(1, 1, 0, 128, 64);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int col = kk / 4, off = (kk % 4) * 32;
      const uint64_t ad = make_sdesc(q16 + col * 128 * 128 + off, 16, 1024, kLayoutSW128);
      const uint64_t bd = make_sdesc(k16 + col * 64 * 128 + off, 16, 1024, kLayoutSW128);
      mma_f16(tmem_d, ad, bd, idesc, kk > 0);
    }
  }
  // O[128 x D] (+)= P[128 x 64] . V[64 x D]  (FP16 operands, FP32 accumulation)
  static __device__ __forceinline__ void pv(uint32_t tmem_o, uint32_t pbase, uint32_t vbase, bool acc) {
    constexpr uint32_t idesc_v = make_idesc(0, 0, 1, 128, D);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = make_sdesc(pbase + kk * 32, 16, 1024, kLayoutSW128);
      const uint64_t bd = make_sdesc(vbase + kk * 16 * 128, 64 * 128, 1024, kLayoutSW128);
      mma_f16(tmem_o, ad, bd, idesc_v, acc || kk > 0);
    }
  }
  // O[128 x D] (+)= P8[128 x 64] . V8[64 x D]  (E4M3 operands, FP32
  // accumulation).  Both K-major with 64-byte swizzled rows of 64 keys: the
  // P8 tile [128 rows x 64 keys], V8t [D rows x 64 keys].
  static __device__ __forceinline__ void pv8(uint32_t tmem_o, uint32_t p8base, uint32_t v8base, bool acc) {
    constexpr uint32_t idesc = make_idesc(0, 0, 0, 128, D);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint64_t ad = make_sdesc(p8base + kk * 32, 16, 512, kLayoutSW64);
      const uint64_t bd = make_sdesc(v8base + kk * 32, 16, 512, kLayoutSW64);
      mma_f8(tmem_o, ad, bd, idesc, acc || kk > 0);
    }
  }
};

}  // namespace lamp
