// lamp_fwd.cu -- fused LampAttention forward kernel for sm_103a.
//
// One CTA computes NT query tiles of 128 rows (NT = 2 for d <= 128, 1 for
// d = 256 and for the optional modes at d = 128) of one (batch, query
// head) against their visible 64-key tiles, in ascending key order (the
// running maximum of the method is defined over that order).  The tiles
// share the K/V stages and ping-pong: while the softmax warps of one tile
// work, the tensor core serves the other.  Optional modes (template bits):
// FP8 P.V for the rows of unflagged sub-blocks (P8 . V8, V8 = fl8(v)
// transposed by the pre-pass; P16 . V16 only for steps with a flagged
// sub-block), and 8-bit logits rounded after every 32-element chunk of d
// (one accumulator per chunk, combined on the CUDA cores).
// Warp roles (TPR softmax threads per query row: 2, and 4 with one tile per
// CTA, so that the tile still has 16 softmax warps):
//   warps 4 TPR t .. 4 TPR t + 4 TPR - 1  softmax of tile t: warps
//              4 TPR t + 4 j + w (j < TPR) hold TMEM lanes 32w.. for key
//              columns 64 j / TPR .. of each step.  Per step: 8-bit logits S8 (with an
//              exactness guard: two candidate roundings per logit, settled
//              by a cheap check or an exact integer re-derivation), running
//              max, the two-stage detector, sub-block flags, mask byte +
//              histogram, FP16 P (P8 = fl8(e^x8) computed with an fp32 ex2
//              and one E4M3 rounding, or P16 for the rows of flagged
//              sub-blocks), O rescale in TMEM, the row sum l in registers.
//   warp 4 TPR NT  TMA producer: Q (Q16, and Q8 for fp32 q) of every tile once,
//              then K8/K16/V16 per step into a ring of stages.
//   warp 4 TPR NT + 1 + t  MMA issuer of tile t (the first one also owns TMEM):
//              S = Q8 K8^T (kind::f8f6f4) into the S8 buffer; S16 = Q16 K16^T
//              (kind::f16, BF16) into its own S16 buffer, only for steps with
//              a flagged sub-block -- issued ahead of the decision for the
//              first step and after a flagged step, else once the decision
//              is published; O += P V16 (kind::f16, V MN-major), or in the
//              FP8 P.V mode O += P8 V8 (kind::f8f6f4, both K-major) and,
//              for steps with a flagged sub-block, O += P16 V16.
//
// The method follows "LampAttention: Look-Ahead Mixed-Precision
// FlashAttention for Dedicated Accelerators" (abstract: 8-bit key-query
// products and exponentials, adaptive detection of sensitive sub-blocks,
// 16-bit recompute; Table 1 / Figures 1-8 captions: thresholds delta and
// tau, 16-bit sub-blocks per tile bucketed 0/1/2+).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lamp_common.cuh"

namespace lamp {

// Optional modes of the forward pass (template bits).
constexpr int kOptPV8 = 1;    // FP8 P.V for rows of unflagged sub-blocks
constexpr int kOptChunk = 2;  // 8-bit logits rounded after every 32-element chunk of d

template <int D, int OPT = 0>
struct Cfg {
  static constexpr bool PV8 = (OPT & kOptPV8) != 0;
  static constexpr bool CHUNK = (OPT & kOptChunk) != 0;
  // query tiles of 128 rows per CTA: one at d = 256, and at d = 128 in an
  // optional mode (the FP8 P.V's P8 and V8 tiles leave no room in shared
  // memory for a second tile, the chunked logits' accumulators none in TMEM)
  static constexpr int NT = (D == 256 || (OPT != 0 && D == 128)) ? 1 : 2;
  static constexpr int NS = (D == 256) ? 1 : 2;  // K/V stages
  // softmax threads per query row: two, each with 32 of a step's 64 keys;
  // four (16 keys each) with one query tile per CTA (d = 256, and the
  // optional modes at d = 128), so that the tile still has 16 softmax warps
  // to hide latency with
  static constexpr int TPR = (NT == 1) ? 4 : 2;
  static constexpr int NC = kBN / TPR;                  // logits per softmax thread per step
  static constexpr int SM_THREADS = kBM * TPR;          // softmax threads per tile
  static constexpr int SM_WARPS = NT * SM_THREADS / 32;
  static constexpr int THREADS = 32 * (SM_WARPS + 1 + NT);
  static constexpr int PRODUCER_WARP = SM_WARPS, MMA_WARP = SM_WARPS + 1;  // + t: MMA warp of tile t
  static constexpr int F8_SWZ_ROW = (D == 64) ? 64 : 128;  // swizzle row width of 8-bit tiles
  static constexpr int Q8_BYTES = kBM * D;
  static constexpr int Q16_BYTES = kBM * D * 2;
  static constexpr int QT_BYTES = Q8_BYTES + Q16_BYTES;  // per query tile
  static constexpr int K8_BYTES = kBN * D;
  static constexpr int K16_BYTES = kBN * D * 2;
  static constexpr int V_BYTES = (D / 64) * kBN * 128;
  // FP8 P.V: V8t [D rows x 64 keys] E4M3 after V16 in the stage, and the P8
  // tile [128 rows x 64 keys] after the P16 tile (both 64-byte swizzled)
  static_assert(!(OPT != 0 && D == 256), "no optional mode at d = 256");
  static_assert(!(PV8 && CHUNK), "one optional mode at a time");
  static constexpr int V8_BYTES = PV8 ? kBN * D : 0;
  static constexpr int OFF_V8 = K8_BYTES + K16_BYTES + V_BYTES;  // inside a stage
  static constexpr int STAGE_BYTES = K8_BYTES + K16_BYTES + V_BYTES + V8_BYTES;
  static constexpr int P16_BYTES = kBM * kBN * 2;
  static constexpr int P_BYTES = P16_BYTES + (PV8 ? kBM * kBN : 0);
  static constexpr int OFF_Q = 0;  // tile t: Q8 at t*QT_BYTES, Q16 right after
  static constexpr int OFF_ST = NT * QT_BYTES;
  // one stage (d = 256): a second K8 slot, so the next key's K8 is loaded
  // while the softmax still re-derives from the current one
  static constexpr int OFF_K8B = OFF_ST + NS * STAGE_BYTES;
  static constexpr int OFF_P = OFF_K8B + (NS == 1 ? K8_BYTES : 0);  // tile t at + t*P_BYTES
  static constexpr int OFF_MISC = OFF_P + NT * P_BYTES;
  static constexpr int CH = D / 32;  // 32-element chunks of d (one FP8 MMA instruction each)
  static constexpr int MISC_BYTES = 9216 + 2 * NT * kBM * CH * 4;
  static constexpr int SMEM = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
  // TMEM columns per tile (fp32): O (d values), the 64-column S8 buffer
  // (one per 32-element chunk of d with chunked logits) and the 64-column
  // S16 buffer.  QK16 of a step is computed ahead, while the softmax still
  // works on S8, so the recompute never waits for it.
  static constexpr int O_COLS = D;
  static constexpr int S8_BUFS = CHUNK ? D / 32 : 1;
  static constexpr int S8_OFF = D;
  static constexpr int S16_OFF = D + S8_BUFS * kBN;
  // one K/V stage (d = 256, one tile): two S16 buffers, so QK16 of a step
  // can be issued while the softmax may still read the previous step's S16
  static constexpr int S16_BUFS = (NS == 1) ? 2 : 1;
  static constexpr int TILE_COLS = D + (S8_BUFS + S16_BUFS) * kBN;
  static constexpr int TMEM_COLS = 512;
  static_assert(NT * TILE_COLS <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// misc area (byte offsets inside OFF_MISC); per-tile barriers at + 8 * t
enum : int {
  M_KV_FULL = 0,      // [2 stages]
  M_KV_EMPTY = 16,    // [2 stages][2 tiles] tile t is done with the stage (at + 16 s + 8 t)
  M_Q_FULL = 48,
  M_S_FULL = 56,      // [2 tiles] QK8 result in TMEM
  M_DEC = 72,         // [2 tiles] the softmax has read S8 (the buffer is free)
  M_S16_FULL = 88,    // [2 tiles] QK16 result in TMEM (one tile, d = 256: [2 S16 buffers])
  M_P_FULL = 104,     // [2 tiles] P written, O rescaled, S16 read
  M_PV_DONE = 120,    // [2 tiles]
  M_DRAIN = 136,      // [2 tiles]
  M_TMEM = 152,       // u32 TMEM base address
  M_ABORT = 156,      // u32 abort flag
  M_SFLAG = 160,      // u32 [2 tiles][2 step parities][4 warps] strip bits
  M_Q8_READY = 224,   // [2 tiles] Q8 made from the Q16 tile (bf16 q)
  M_V_FULL = 240,     // one K/V stage: its V part landed
  M_V_EMPTY = 248,    // one K/V stage: its V part is free (P.V done)
  M_EXP8 = 256,       // u8 [256] exp8 table: code of fl8(exp(x)) per code of x
  M_XCH = 512,        // f32 [2 tiles][2 halves][128 rows] values exchanged between a row's two threads
  M_XB = 2560,        // u32 [2 tiles][2 halves][128 rows] bits exchanged between a row's two threads
  M_K8B_FULL = 4608,  // one stage: the second K8 slot landed
  M_K8B_EMPTY = 4616, // one stage: the second K8 slot is free
  M_ANY = 4624,       // u8 [2 tiles][2 step parities]: the step has a flagged sub-block
  M_XLH = 5120,       // f32x2 [2 tiles][2 halves][128 rows] bounds of the tile max exchanged
  M_QG = 9216,        // f32 [2 halves][NT tiles][128 rows][D/32] per-row weights of the exactness bound
};

struct Ctx {
  volatile uint32_t* abort;      // CTA abort flag (shared memory)
  volatile unsigned int* gabort; // grid abort word (global memory)
  unsigned long long timeout_ns;
  unsigned long long* counters;
};

constexpr unsigned long long kDrainNs = 200000000ull;  // 0.2 s for in-flight copies

// Bounded wait: gives up after cx.timeout_ns, or as soon as this CTA or any
// other CTA has given up; on expiry it raises both abort flags and writes
// LAMP_ERR_TIMEOUT into the status counter.  The waiting part suspends in
// hardware; it is inlined (a real call would save live registers to local
// memory around every wait).
__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                           volatile unsigned int* gabort, unsigned long long timeout_ns,
                                           unsigned long long* counters) {
  if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (*abort) return false;
    if (*gabort) { *abort = 1u; return false; }
    if (globaltimer_ns() - t0 > timeout_ns) break;
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  }
  *abort = 1u;
  atomicExch((unsigned int*)gabort, 1u);
  if (counters) atomicExch(&counters[9], 4ull);  // LAMP_ERR_TIMEOUT
  return false;
}

__device__ __forceinline__ bool wait_bar(const Ctx& cx, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, cx.abort, cx.gabort, cx.timeout_ns, cx.counters);
}

// Warp-uniform variant: every lane waits; true only if all lanes succeeded.
__device__ __forceinline__ bool wait_bar_warp(const Ctx& cx, uint32_t bar, uint32_t parity) {
  const bool okl = wait_bar(cx, bar, parity);
  return __all_sync(0xffffffffu, okl);
}

// Wait used only to let this CTA's own copies and MMAs land before exit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kDrainNs) return;
}

__device__ __forceinline__ __half2 as_half2(uint32_t u) {
  __half2 r;
  memcpy(&r, &u, 4);
  return r;
}

__device__ __forceinline__ uint32_t as_u32(__half2 h) {
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

__device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }
__device__ __forceinline__ int imax(int a, int b) { return a > b ? a : b; }

// Visible key range [lo, hi] of global row R (empty if lo > hi).
__device__ __forceinline__ void row_range(const FwdParams& p, int R, int& lo, int& hi) {
  if (R >= p.N) { lo = 1; hi = 0; return; }
  if (p.mask_kind == 0) { lo = 0; hi = p.N - 1; return; }
  hi = R;
  lo = (p.mask_kind == 2) ? imax(0, R - p.window + 1) : 0;
}

// Key-tile range [j_lo, j_hi) of the 128-row query tile starting at row q0
// (empty when q0 >= N).
__device__ __forceinline__ void tile_range(const FwdParams& p, int q0, int& j_lo, int& j_hi) {
  if (q0 >= p.N) { j_lo = 0; j_hi = 0; return; }
  const int last = imin(q0 + kBM - 1, p.N - 1);
  if (p.mask_kind == 0) { j_lo = 0; j_hi = p.T; return; }
  j_hi = last / kBN + 1;
  j_lo = (p.mask_kind == 2) ? imax(0, q0 - p.window + 1) / kBN : 0;
}

// Exact A * 2^18 of (row r of the tile's Q8, key c of the stage's K8): an
// integer dot product of the E4M3 operands in shared memory, D/32 bytes per
// lane (contiguous inside one 16-byte swizzle chunk).  The per-lane sums
// (< 2^39) are split at bit 24 and both parts summed with one warp
// reduction each, so every lane gets the exact total.
template <int D>
__device__ __forceinline__ long long exact_dot(const uint8_t* sQ8, const uint8_t* sK8, int r, int c,
                                               int lane) {
  constexpr int RB = (Cfg<D>::F8_SWZ_ROW == 64) ? 64 : D;
  constexpr int BPL = D / 32;
  const int x = lane * BPL;
  uint32_t q[2] = {0u, 0u}, k[2] = {0u, 0u};
  if (BPL == 8) {
    const uint2 a = *reinterpret_cast<const uint2*>(sQ8 + swz_offset(r, x, kBM, RB));
    const uint2 bb = *reinterpret_cast<const uint2*>(sK8 + swz_offset(c, x, kBN, RB));
    q[0] = a.x; q[1] = a.y; k[0] = bb.x; k[1] = bb.y;
  } else if (BPL == 4) {
    q[0] = *reinterpret_cast<const uint32_t*>(sQ8 + swz_offset(r, x, kBM, RB));
    k[0] = *reinterpret_cast<const uint32_t*>(sK8 + swz_offset(c, x, kBN, RB));
  } else {
    q[0] = *reinterpret_cast<const uint16_t*>(sQ8 + swz_offset(r, x, kBM, RB));
    k[0] = *reinterpret_cast<const uint16_t*>(sK8 + swz_offset(c, x, kBN, RB));
  }
  long long acc = 0;
#pragma unroll
  for (int i = 0; i < BPL; ++i)
    acc += e4m3_prod_2p18((q[i >> 2] >> (8 * (i & 3))) & 0xFFu, (k[i >> 2] >> (8 * (i & 3))) & 0xFFu);
  const int hi = __reduce_add_sync(0xffffffffu, (int)(acc >> 24));
  const unsigned lo = __reduce_add_sync(0xffffffffu, (unsigned)(acc & 0xFFFFFF));
  return (long long)hi * 16777216ll + (long long)lo;
}

// The same for chunk ch of d only (32 elements: lane L takes element
// 32 ch + L; 32 products below 2^36 each, split at bit 24 as above).
template <int D>
__device__ __forceinline__ long long exact_dot_chunk(const uint8_t* sQ8, const uint8_t* sK8, int r, int c, int ch,
                                                     int lane) {
  constexpr int RB = (Cfg<D>::F8_SWZ_ROW == 64) ? 64 : D;
  const int x = ch * 32 + lane;
  const long long acc = e4m3_prod_2p18(sQ8[swz_offset(r, x, kBM, RB)], sK8[swz_offset(c, x, kBN, RB)]);
  const int hi = __reduce_add_sync(0xffffffffu, (int)(acc >> 24));
  const unsigned lo = __reduce_add_sync(0xffffffffu, (unsigned)(acc & 0xFFFFFF));
  return (long long)hi * 16777216ll + (long long)lo;
}

}  // namespace lamp

namespace lamp {

// kMode 0: the forward pass (delta > 0); 1: the forward pass with the first
// stage off (delta = 0); 2 (kSweep): the tau-sweep pass (Figures 1-3 and 8
// sweep tau at fixed delta): only the 8-bit logits, the running max and the
// detector run, and each visited tile gets a record with, per sub-block,
// the largest half-ulp8 of its stage-1 entries (the flag at any tau follows
// from it); no 16-bit recompute, no P.V, no output.

// bf16 q: a softmax thread rounds its part hf (of TPR) of row t of the Q16
// tile to E4M3 (the rounding the pre-pass applies to fp32 values; bf16 ->
// fp32 is exact), writes the codes into the Q8 tile for the tensor core,
// arrives on `rdy` and returns the sum of squares of their values; the sum
// of each 32-element chunk goes to qg_own[chunk] and qg_other[chunk].  Not
// inlined: kept out of the step loop's code, which runs measurably slower
// otherwise.
template <int D, int TPR>
__device__ __noinline__ float q8_from_q16(uint8_t* q8w, int t, int hf, uint32_t rdy, float* qg_own, float* qg_other) {
  using C = Cfg<D>;
  float ss = 0.0f, sc = 0.0f;
  const uint8_t* q16 = q8w + C::Q8_BYTES;
#pragma unroll
  for (int u = 0; u < D / (16 * TPR); ++u) {
    const int cb = hf * (D / TPR) + 16 * u;  // first of the 16 columns
    const uint4 w0 = *reinterpret_cast<const uint4*>(q16 + swz_offset(t, 2 * cb, kBM, 2 * D));
    const uint4 w1 = *reinterpret_cast<const uint4*>(q16 + swz_offset(t, 2 * cb + 16, kBM, 2 * D));
    const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint16_t c = cvt_e4m3x2(__uint_as_float(wd[i] & 0xFFFF0000u), __uint_as_float(wd[i] << 16));
      const __half2 hv = as_half2(e4m3x2_to_f16x2(c));
      const float a0 = __low2float(hv), a1 = __high2float(hv);
      sc = fmaf(a0, a0, fmaf(a1, a1, sc));
      if (i & 1) o[i >> 1] |= (uint32_t)c << 16; else o[i >> 1] = c;
    }
    *reinterpret_cast<uint4*>(q8w + swz_offset(t, cb, kBM, D)) = make_uint4(o[0], o[1], o[2], o[3]);
    if (u & 1) {  // a 32-element chunk done: its sum of squares for both threads of the row
      const int ch = hf * (D / (32 * TPR)) + (u >> 1);
      qg_own[ch] = sc;
      qg_other[ch] = sc;
      ss += sc;
      sc = 0.0f;
    }
  }
  fence_proxy_async_smem();  // visible to the tensor core's reads
  mbar_arrive(rdy);
  return ss;
}

template <int D, int kMode, int kOpt>
__global__ void __launch_bounds__(Cfg<D, kOpt>::THREADS, 1) lamp_fwd_kernel(const __grid_constant__ FwdParams p) {
  constexpr bool kSweep = kMode == 2;
  constexpr bool kNoStage1 = kMode == 1;
  constexpr bool kPV8 = (kOpt & kOptPV8) != 0;
  constexpr bool kChunk = (kOpt & kOptChunk) != 0;
  static_assert(!(kSweep && kOpt != 0), "the sweep pass has no optional mode");
  using C = Cfg<D, kOpt>;
  extern __shared__ uint8_t smem_raw[];
  // align by pointer arithmetic on the __shared__ array so that every access
  // through `smem` stays a shared-memory access
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint8_t* misc = smem + C::OFF_MISC;
  const uint32_t mb = sbase + C::OFF_MISC;
  auto bar = [&](int off) { return mb + (uint32_t)off; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh_count = p.B * p.Hq;
  const int qb = p.nqb - 1 - (int)(blockIdx.x / bh_count);  // longest rows first
  const int bh = blockIdx.x % bh_count;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  const int q0 = qb * kBM * C::NT;  // first row of the CTA
  // key-tile range of each query tile and of the CTA
  int jlo0, jhi0, jlo1 = 0, jhi1 = 0;
  tile_range(p, q0, jlo0, jhi0);
  if (C::NT == 2) tile_range(p, q0 + kBM, jlo1, jhi1);
  const int J0 = (C::NT == 2 && jhi1 > jlo1) ? imin(jlo0, jlo1) : jlo0;
  const int J1 = (C::NT == 2) ? imax(jhi0, jhi1) : jhi0;
  auto JLO = [&](int t) { return t ? jlo1 : jlo0; };
  auto JHI = [&](int t) { return t ? jhi1 : jhi0; };

  Ctx cx;
  cx.abort = (volatile uint32_t*)(misc + M_ABORT);
  cx.gabort = p.gabort;
  cx.timeout_ns = p.timeout_ns;
  cx.counters = p.counters;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(M_S_FULL + 8 * s), 1);
      mbar_init(bar(M_KV_FULL + 8 * s), 1);
      mbar_init(bar(M_KV_EMPTY + 16 * s), 1);
      mbar_init(bar(M_KV_EMPTY + 16 * s + 8), 1);
      mbar_init(bar(M_DEC + 8 * s), 1);
      mbar_init(bar(M_S16_FULL + 8 * s), 1);
      mbar_init(bar(M_P_FULL + 8 * s), C::SM_THREADS);
      mbar_init(bar(M_PV_DONE + 8 * s), 1);
      mbar_init(bar(M_DRAIN + 8 * s), 1);
      mbar_init(bar(M_Q8_READY + 8 * s), C::SM_THREADS);
    }
    mbar_init(bar(M_Q_FULL), 1);
    mbar_init(bar(M_V_FULL), 1);
    mbar_init(bar(M_V_EMPTY), 1);
    mbar_init(bar(M_K8B_FULL), 1);
    mbar_init(bar(M_K8B_EMPTY), 1);
    *(volatile uint32_t*)(misc + M_ABORT) = 0u;
    fence_mbar_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(bar(M_TMEM), C::TMEM_COLS);  // the first MMA warp owns TMEM
  // the exp8 table of codes, for the detector's comparisons with delta
  // (the P8 values themselves are computed, exp8_f16x2)
  if (threadIdx.x < 256) misc[M_EXP8 + threadIdx.x] = p.exp8[threadIdx.x];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *(volatile uint32_t*)(misc + M_TMEM);

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && J1 > J0) {
      prefetch_tmap(&p.tmQ8);
      prefetch_tmap(&p.tmK8);
      if (!kSweep) {  // the sweep pass has no V map
        prefetch_tmap(&p.tmQ16);
        prefetch_tmap(&p.tmK16);
        prefetch_tmap(&p.tmV);
        if (kPV8) prefetch_tmap(&p.tmV8);
      }
      // Q8 comes from the pre-pass, or (bf16 q) the softmax makes it from Q16
      const bool load_q8 = kSweep || !p.q8_in_cta;
      mbar_expect_tx(bar(M_Q_FULL),
                     C::NT * ((load_q8 ? C::Q8_BYTES : 0) + (kSweep ? 0 : C::Q16_BYTES)));
      for (int t = 0; t < C::NT; ++t) {
        const uint32_t qd = sbase + C::OFF_Q + t * C::QT_BYTES;
        for (int c = 0; load_q8 && c < D / C::F8_SWZ_ROW; ++c)
          tma_load_4d(qd + c * kBM * 128, &p.tmQ8, bar(M_Q_FULL), c * C::F8_SWZ_ROW, q0 + t * kBM, h, b);
        if (!kSweep)
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(qd + C::Q8_BYTES + c * kBM * 128, &p.tmQ16, bar(M_Q_FULL), c * 64, q0 + t * kBM, h, b);
      }
      int uses0 = 0, uses1 = 0, uses2 = 0, uses3 = 0;
      uint32_t rel = 0u;  // releases waited for so far, one bit of parity per (tile, stage)
      if (C::NS == 1 && !kSweep) {
        // one stage, filled in parts with their own barriers: K8 in two
        // slots by key parity (KV_FULL / KV_EMPTY and K8B_FULL / K8B_EMPTY,
        // a slot free once the softmax has published its key's step), K16
        // (slot 1 of KV_FULL / KV_EMPTY, free once the key's QK16 is done)
        // and V (V_FULL / V_EMPTY, free once the key's P.V is done).  Order
        // per key j: K16(j), K8(j + 1), V(j) -- each waits for an event
        // earlier than the next one's, so K8 and K16 land a step ahead and
        // only V waits for the P.V.
        const uint32_t st = sbase + C::OFF_ST;
        const int nk = J1 - J0;
        auto load_k8 = [&](int u) {
          const uint32_t fb = (u & 1) ? bar(M_K8B_FULL) : bar(M_KV_FULL);
          const uint32_t dst = (u & 1) ? sbase + C::OFF_K8B : st;
          mbar_expect_tx(fb, C::K8_BYTES);
          for (int c = 0; c < D / C::F8_SWZ_ROW; ++c)
            tma_load_4d(dst + c * kBN * 128, &p.tmK8, fb, c * C::F8_SWZ_ROW, (J0 + u) * kBN, g, b);
          if (u & 1) uses3 = (u >> 1) + 1; else uses0 = (u >> 1) + 1;
        };
        if (nk > 0) load_k8(0);
        for (int u = 0; u < nk && !*cx.abort; ++u) {
          const int key0 = (J0 + u) * kBN;
          if (u >= 1 && !wait_bar(cx, bar(M_KV_EMPTY + 16), (u - 1) & 1)) break;
          mbar_expect_tx(bar(M_KV_FULL + 8), C::K16_BYTES);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(st + C::K8_BYTES + c * kBN * 128, &p.tmK16, bar(M_KV_FULL + 8), c * 64, key0, g, b);
          uses1 = u + 1;
          if (u + 1 < nk) {
            const int v = u + 1;  // its slot held key v - 2
            if (v >= 2 && !wait_bar(cx, (v & 1) ? bar(M_K8B_EMPTY) : bar(M_KV_EMPTY), ((v - 2) >> 1) & 1)) break;
            load_k8(v);
          }
          if (u >= 1 && !wait_bar(cx, bar(M_V_EMPTY), (u - 1) & 1)) break;
          mbar_expect_tx(bar(M_V_FULL), C::V_BYTES);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(st + C::K8_BYTES + C::K16_BYTES + c * kBN * 128, &p.tmV, bar(M_V_FULL), c * 64, key0, g, b);
          uses2 = u + 1;
        }
      }
      for (int j = J0; j < J1 && !*cx.abort && !(C::NS == 1 && !kSweep); ++j) {
        const int s = (j - J0) % C::NS, u = (j - J0) / C::NS;
        bool ok = true;
        if (u >= 1) {  // the stage held key j - NS: wait until every tile is done with it
          // (a tile whose keys start after J0 releases the keys before its
          // first one unused, so that no stage runs two phases ahead of the
          // tile's parity waits)
          const int jr = j - C::NS;
#pragma unroll
          for (int t = 0; t < C::NT; ++t) {
            if (JHI(t) <= JLO(t) || jr >= JHI(t)) continue;
            const uint32_t bit = 1u << (2 * t + s);
            ok = ok && wait_bar(cx, bar(M_KV_EMPTY + 16 * s + 8 * t), (rel & bit) ? 1u : 0u);
            rel ^= bit;
          }
        }
        if (!ok) break;
        const int key0 = j * kBN;
        const uint32_t st = sbase + C::OFF_ST + s * C::STAGE_BYTES;
        const uint32_t fb = bar(M_KV_FULL + 8 * s);
        mbar_expect_tx(fb, kSweep ? C::K8_BYTES : C::STAGE_BYTES);
        for (int c = 0; c < D / C::F8_SWZ_ROW; ++c)
          tma_load_4d(st + c * kBN * 128, &p.tmK8, fb, c * C::F8_SWZ_ROW, key0, g, b);
        if (!kSweep) {
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(st + C::K8_BYTES + c * kBN * 128, &p.tmK16, fb, c * 64, key0, g, b);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(st + C::K8_BYTES + C::K16_BYTES + c * kBN * 128, &p.tmV, fb, c * 64, key0, g, b);
          if (kPV8) tma_load_4d(st + C::OFF_V8, &p.tmV8, fb, key0, 0, g, b);  // V8t rows of d, 64 keys each
        }
        if (s) uses1 = u + 1; else uses0 = u + 1;
      }
      if (*cx.abort) {  // let every load in flight land before the CTA exits
        if (uses0 > 0) drain_wait(bar(M_KV_FULL), (uses0 - 1) & 1);
        if (uses1 > 0) drain_wait(bar(M_KV_FULL + 8), (uses1 - 1) & 1);
        if (uses2 > 0) drain_wait(bar(M_V_FULL), (uses2 - 1) & 1);
        if (uses3 > 0) drain_wait(bar(M_K8B_FULL), (uses3 - 1) & 1);
        drain_wait(bar(M_Q_FULL), 0);
      }
    }
  } else if (warp >= C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuers
    // One warp per query tile, in a fixed order with blocking waits:
    //   QK8(0) QK16(0) | DEC(i-1): QK8(i) | P(i-1): P.V(i-1) QK16(i) | ...
    // QK8(i) goes into the S8 buffer once the softmax has read S8(i-1);
    // QK16(i) into the S16 buffer once the softmax has consumed S16(i-1)
    // (signalled with P(i-1)), ahead of the decision of step i, so a flagged
    // step finds its 16-bit products ready.  After each P.V the tile hands
    // the key's K/V stage back to the producer.
    const int t = warp - C::MMA_WARP;
    const int jlo = JLO(t), n = JHI(t) - JLO(t);
    if (lane == 0 && n > 0) {
      auto stage_of = [&](int j) { return (j - J0) % C::NS; };
      auto kv = [&](int j) { return sbase + C::OFF_ST + stage_of(j) * C::STAGE_BYTES; };
      const uint32_t tm = tmem + t * C::TILE_COLS;
      const uint32_t qbase = sbase + C::OFF_Q + t * C::QT_BYTES;
      // P.V of step i; any16: the step has a flagged sub-block
      auto pv = [&](int i, bool any16) {
        const uint32_t pb = sbase + C::OFF_P + t * C::P_BYTES, vb = kv(jlo + i) + C::K8_BYTES + C::K16_BYTES;
        if constexpr (kPV8) {
          // rows of unflagged sub-blocks: P8 . V8 (the P8 tile is 0 in the
          // flagged rows); rows of flagged ones: P16 . V16, issued only when
          // the step has one (the P16 tile is then 0 in the other rows)
          Mma<D>::pv8(tm, pb + C::P16_BYTES, kv(jlo + i) + C::OFF_V8, i > 0);
          if (any16) Mma<D>::pv(tm, pb, vb, true);
        } else {
          Mma<D>::pv(tm, pb, vb, i > 0);
        }
        mma_commit(bar(M_PV_DONE + 8 * t));
        mma_commit(bar(M_KV_EMPTY + 16 * stage_of(jlo + i) + 8 * t));
      };
      // recompute steps: used, issued ahead and not used, issued after the decision
      uint32_t o_rec = 0, o_spec = 0, o_late = 0;
      auto count = [&](bool dec, bool ahead) {
        o_rec += dec;
        o_spec += ahead && !dec;
        o_late += dec && !ahead;
      };
      bool ok = wait_bar(cx, bar(M_Q_FULL), 0);
      if (ok && !kSweep && p.q8_in_cta) ok = wait_bar(cx, bar(M_Q8_READY + 8 * t), 0);
      // keys of the CTA before this tile's first one (a sliding window's
      // second tile): wait for each to land and hand its stage back unused,
      // so the stage's phases stay in step with this tile's parity waits
      for (int j = J0; ok && j < jlo; ++j) {
        ok = wait_bar(cx, bar(M_KV_FULL + 8 * stage_of(j)), ((j - J0) / C::NS) & 1);
        if (ok) mbar_arrive(bar(M_KV_EMPTY + 16 * stage_of(j) + 8 * t));
      }
      if (kSweep) {
        // QK8 only.  A key's stage is handed back once the softmax has
        // published the step (DEC): its exact re-derivations read K8 from
        // the stage until then.
        for (int i = 0; ok && i < n; ++i) {
          const int j = jlo + i;
          if (i > 0) {
            ok = wait_bar(cx, bar(M_DEC + 8 * t), (i - 1) & 1);
            if (!ok) break;
            mbar_arrive(bar(M_KV_EMPTY + 16 * stage_of(j - 1) + 8 * t));
          }
          ok = wait_bar(cx, bar(M_KV_FULL + 8 * stage_of(j)), ((j - J0) / C::NS) & 1);
          if (!ok) break;
          tc_fence_after();
          Mma<D>::qk8(tm + C::S8_OFF, qbase, kv(j));
          mma_commit(bar(M_S_FULL + 8 * t));
        }
        if (ok && wait_bar(cx, bar(M_DEC + 8 * t), (n - 1) & 1))
          mbar_arrive(bar(M_KV_EMPTY + 16 * stage_of(jlo + n - 1) + 8 * t));
        ok = false;  // nothing more to issue
      }
      if (C::NS == 1 && !kSweep) {
        // One K/V stage (d = 256, one query tile) in three parts (K8 in two
        // slots by key parity, K16, V), each handed back on its own: K8 once
        // the softmax has published the step (its re-derivations read K8
        // until then), K16 once the step's QK16 is done, V after the step's
        // P.V.  QK16(i) goes right
        // after QK8(i), into the S16 buffer of parity i (the softmax may
        // still read the other one); P.V(i - 1) follows once P(i - 1) is in.
        static_assert(C::NS != 1 || (C::NT == 1 && C::S16_BUFS == 2), "one stage: one query tile, two S16 buffers");
        // QK16(i) is issued right after QK8(i) for the first step and when
        // step i - 1 had a flagged sub-block, else once DEC(i) says step i
        // has one (the softmax follows the same rule); a step without flags
        // hands its K16 slot back without one.
        auto any_of = [&](int i) { return *(volatile uint8_t*)(misc + M_ANY + (i & 1)) != 0; };
        auto qk16 = [&](int i) {  // K16 of key jlo + i is in its slot
          // one barrier per S16 buffer: a single one could complete twice
          // (QK16(i), QK16(i + 1)) before the softmax waits for QK16(i),
          // and a parity wait cannot tell those phases apart
          Mma<D>::qk16(tm + C::S16_OFF + (i & 1) * kBN, qbase + C::Q8_BYTES, kv(jlo + i) + C::K8_BYTES);
          mma_commit(bar(M_S16_FULL + 8 * (i & 1)));
          mma_commit(bar(M_KV_EMPTY + 16));  // K16 of key jlo + i
        };
        // step i decided: its QK16 now, or its K16 slot back unused -- in
        // both cases only once the slot's copy has landed (the producer
        // re-arms the slot's barrier for the next key when it gets it back)
        auto decided = [&](int i) -> bool {
          if (!wait_bar(cx, bar(M_KV_FULL + 8), (uint32_t)(jlo + i - J0) & 1u)) return false;
          if (any_of(i)) {
            tc_fence_after();
            qk16(i);
          } else {
            mbar_arrive(bar(M_KV_EMPTY + 16));
          }
          return true;
        };
        bool spec = true;  // QK16 of the current step is issued ahead of its decision (always the first)
        for (int i = 0; ok && i < n; ++i) {
          const int j = jlo + i;
          const uint32_t ph = (uint32_t)(j - J0) & 1u;
          if (i > 0) {
            ok = wait_bar(cx, bar(M_DEC), (i - 1) & 1);
            if (!ok) break;
            mbar_arrive(((i - 1) & 1) ? bar(M_K8B_EMPTY) : bar(M_KV_EMPTY));  // K8 slot of key j - 1
          }
          ok = wait_bar(cx, (i & 1) ? bar(M_K8B_FULL) : bar(M_KV_FULL), (uint32_t)(i >> 1) & 1u);
          if (!ok) break;
          tc_fence_after();
          Mma<D>::qk8(tm + C::S8_OFF, qbase, (i & 1) ? sbase + C::OFF_K8B : kv(j));
          mma_commit(bar(M_S_FULL));
          if (i > 0) {  // the decision of step i - 1, read once QK8(i) is on its way
            count(any_of(i - 1), spec);
            if (!spec) ok = decided(i - 1);
            if (!ok) break;
            spec = any_of(i - 1);
          }
          if (spec) {
            ok = wait_bar(cx, bar(M_KV_FULL + 8), ph);
            if (!ok) break;
            tc_fence_after();
            qk16(i);
          }
          if (i > 0) {
            ok = wait_bar(cx, bar(M_P_FULL), (i - 1) & 1);
            if (ok) ok = wait_bar(cx, bar(M_V_FULL), (ph ^ 1u));
            if (!ok) break;
            tc_fence_after();
            Mma<D>::pv(tm, sbase + C::OFF_P, kv(j - 1) + C::K8_BYTES + C::K16_BYTES, i - 1 > 0);
            mma_commit(bar(M_PV_DONE));
            mma_commit(bar(M_V_EMPTY));  // V of key j - 1
          }
        }
        if (ok) ok = wait_bar(cx, bar(M_DEC), (n - 1) & 1);
        if (ok) count(any_of(n - 1), spec);
        if (ok && !spec) ok = decided(n - 1);
        if (ok) ok = wait_bar(cx, bar(M_P_FULL), (n - 1) & 1);
        if (ok) ok = wait_bar(cx, bar(M_V_FULL), (uint32_t)(jlo + n - 1 - J0) & 1u);
        if (ok) {
          tc_fence_after();
          Mma<D>::pv(tm, sbase + C::OFF_P, kv(jlo + n - 1) + C::K8_BYTES + C::K16_BYTES, n - 1 > 0);
          mma_commit(bar(M_PV_DONE));
        }
        ok = false;
      }
      // The 16-bit products of step i are computed only if the step needs
      // them: ahead of its decision for the first step and when step i - 1
      // had a flagged sub-block (flags come in runs, so the recompute then
      // finds them ready), else once the decision (DEC(i)) says so.  The
      // softmax applies the same rule, so both sides count the same S16
      // phases.
      auto any_of = [&](int i) {  // the decision of step i, published before DEC(i)
        return *(volatile uint8_t*)(misc + M_ANY + 2 * t + (i & 1)) != 0;
      };
      auto qk16 = [&](int i) {
        Mma<D>::qk16(tm + C::S16_OFF, qbase + C::Q8_BYTES, kv(jlo + i) + C::K8_BYTES);
        mma_commit(bar(M_S16_FULL + 8 * t));
      };
      bool spec = true;  // QK16 of the current step is issued ahead of its decision (always the first)
      for (int i = 0; ok && i < n; ++i) {
        const int j = jlo + i;
        if (i > 0) ok = wait_bar(cx, bar(M_DEC + 8 * t), (i - 1) & 1);
        if (ok) ok = wait_bar(cx, bar(M_KV_FULL + 8 * stage_of(j)), ((j - J0) / C::NS) & 1);
        if (!ok) break;
        tc_fence_after();
        if constexpr (kChunk)
          Mma<D>::qk8_chunks(tm + C::S8_OFF, qbase, kv(j));
        else
          Mma<D>::qk8(tm + C::S8_OFF, qbase, kv(j));
        mma_commit(bar(M_S_FULL + 8 * t));
        if (i > 0) {
          // the decision of step i - 1, read once QK8(i) is on its way
          const bool prev = any_of(i - 1);
          count(prev, spec);
          if (prev && !spec) qk16(i - 1);  // step i - 1 decided to recompute: its products now
          spec = prev;
          ok = wait_bar(cx, bar(M_P_FULL + 8 * t), (i - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          pv(i - 1, prev);
        }
        if (spec) qk16(i);
      }
      if (ok) ok = wait_bar(cx, bar(M_DEC + 8 * t), (n - 1) & 1);
      if (ok) {
        count(any_of(n - 1), spec);
        if (any_of(n - 1) && !spec) {
          tc_fence_after();
          qk16(n - 1);
        }
      }
      if (ok) ok = wait_bar(cx, bar(M_P_FULL + 8 * t), (n - 1) & 1);
      if (ok) {
        tc_fence_after();
        pv(n - 1, any_of(n - 1));
      }
      // make sure no MMA of this warp still writes TMEM before it is released
      mma_commit(bar(M_DRAIN + 8 * t));
      drain_wait(bar(M_DRAIN + 8 * t), 0);
      if (p.counters && !kSweep) {
        typedef unsigned long long u64;
        if (o_rec) atomicAdd(&p.counters[10], (u64)o_rec);
        if (o_spec) atomicAdd(&p.counters[11], (u64)o_spec);
        if (o_late) atomicAdd(&p.counters[12], (u64)o_late);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // TPR threads per query row: warps 4 TPR tt + 4 hf + rw (hf < TPR) hold
    // TMEM lanes 32rw.. of tile tt, each for key columns hf NC .. hf NC +
    // NC - 1 of every step; row values are exchanged through shared memory
    // behind a named barrier of the TPR warps.  Every softmax thread of a tile runs every step of
    // the tile, also after a failed wait (its later waits and TMEM accesses
    // are then skipped), so named barriers never miss a participant; waits
    // are warp-uniform so the .sync.aligned TMEM accesses stay converged.
    constexpr int NC = C::NC;             // logits per thread per step
    constexpr int TPR = C::TPR;           // threads per row
    constexpr uint32_t kAll = NC == 32 ? 0xFFFFFFFFu : ((1u << NC) - 1u);  // all NC columns visible
    const int tt = warp / (4 * TPR);      // query tile
    const int hf = (warp >> 2) % TPR;     // column part: keys hf NC .. hf NC + NC - 1 of a step
    const int rw = warp & 3;              // 32-row group of the tile
    const int t = rw * 32 + lane;         // row within the tile == TMEM lane
    const int col0 = hf * NC;
    const int R = q0 + tt * kBM + t;
    const int jlo_t = JLO(tt), nsteps = JHI(tt) - JLO(tt);
    const uint32_t tile_bar = 1 + tt;             // the tile's softmax threads
    const uint32_t pair_bar = 3 + 4 * tt + rw;    // the TPR warps of these 32 rows
    constexpr int kPairThreads = 32 * TPR;
    const uint32_t lane_base = tmem + tt * C::TILE_COLS + ((uint32_t)(rw * 32) << 16);
    const uint8_t* sQ8 = smem + C::OFF_Q + tt * C::QT_BYTES;
    uint8_t* sP = smem + C::OFF_P + tt * C::P_BYTES;
    const uint8_t* tab = misc + M_EXP8;
    float* xch = (float*)(misc + M_XCH) + tt * TPR * kBM;
    uint32_t* xb = (uint32_t*)(misc + M_XB) + tt * TPR * kBM;
    int lo, hi;
    row_range(p, R, lo, hi);
    // key tiles the row sees whole: [jf0, jf1] (empty for a row past the end)
    const int jf0 = (lo + kBN - 1) / kBN, jf1 = (hi + 1) / kBN - 1;
    float m = -INFINITY;
    float l = 0.0f;  // this half's running sum of the (rounded) P values fed to P.V
    bool fail = !(nsteps > 0 && wait_bar_warp(cx, bar(M_Q_FULL), 0));
    float nq = 0.0f;
    // The row's weights of the exactness bound (below): two threads a row
    // keep a copy each in shared memory; four (d = 256) keep them in
    // registers, the shared array then holding the row's chunk sums once.
    float* qg = (float*)(misc + M_QG) + (((TPR == 2 ? hf : 0) * C::NT + tt) * kBM + t) * C::CH;
    float qgr[TPR == 2 ? 1 : C::CH];
    auto QG = [&](int c) -> float& {
      if constexpr (TPR == 2) return qg[c]; else return qgr[c];
    };
    if (!kSweep && p.q8_in_cta) {
      // bf16 q: Q8 and this part's sums of squares from the Q16 tile, per
      // 32-element chunk (into both threads' copies with two threads a
      // row); the row's parts are added for ||fl8(q_r)||
      float ss = 0.0f;
      float* qg_other = (float*)(misc + M_QG) + (((TPR == 2 ? 1 - hf : 0) * C::NT + tt) * kBM + t) * C::CH;
      if (!fail)
        ss = q8_from_q16<D, TPR>(smem + C::OFF_Q + tt * C::QT_BYTES, t, hf, bar(M_Q8_READY + 8 * tt), qg, qg_other);
      xb[hf * kBM + t] = __float_as_uint(ss);
      bar_sync(pair_bar, kPairThreads);
      // upper bounds of the norms: the float sums of squares are rounded up
      float sst = 0.0f;
#pragma unroll
      for (int p2 = 0; p2 < TPR; ++p2) sst += __uint_as_float(xb[p2 * kBM + t]);
      if (R < p.N) nq = sqrtf(sst) * (1.0f + 0x1p-16f);
#pragma unroll
      for (int c = 0; c < C::CH; ++c) QG(c) = sqrtf(qg[c]) * (1.0f + 0x1p-16f);
    } else {
      const size_t row = ((size_t)b * p.Hq + h) * p.N + R;
      if (R < p.N) nq = p.nq[row];
#pragma unroll
      for (int c = 0; c < C::CH; ++c) QG(c) = R < p.N ? p.nqc[row * C::CH + c] : 0.0f;
    }
    // Exactness guard: |A_tc - A| sigma <= G.  Instruction c of the FP8
    // tensor-core chain (K = 32: chunk c of d) aligns the accumulator D_c and
    // its 32 products to their largest exponent E, truncates each to a
    // multiple of 2^(E - 25), sums and truncates the sum to float32, an
    // error below 33 * 2^-25 max(|D_c|, largest product) + 2^-23 |D_c+1|.
    // With x_c = (||q8_c|| + 2^-6)(||k8_c|| + 2^-6) (a product of chunk c, an
    // operand below 2^-6 counting as 2^-6, is at most x_c) and the partial
    // sums |D_c+1| <= P_c = x_0 + ... + x_c (Cauchy-Schwarz per chunk), the
    // chain errs by less than 37 * 2^-25 * sum_c P_c
    // = 37 * 2^-25 * sum_c (C - c) x_c.  The kernel takes the tile's largest
    // ||k8_c|| and the factor 40 (margin for the float roundings of
    // y = A_tc sigma, y -+ G and of this sum); qg holds
    // 40 * 2^-25 (C - c) sigma (||q8_c|| + 2^-6), the pre-pass the key side.
#pragma unroll
    // (chunked logits: each chunk is one instruction with a zero
    // accumulator, its own bound without the chain factor C - c)
    for (int c = 0; c < C::CH; ++c)
      QG(c) = (QG(c) + 0x1p-6f) * (40.0f * 0x1p-25f * (kChunk ? 1.0f : (float)(C::CH - c))) * p.sigma_f;
    const float satq = p.sigma_f * nq * (1.0f + p.guard);
    uint32_t c_h0 = 0, c_h1 = 0, c_h2 = 0, c_strips = 0, c_st1 = 0, c_fl = 0, c_sat = 0, c_fix = 0,
             c_res = 0, c_fmax = 0;  // per-thread counts (a CTA sees at most 2^21 logits per thread slot)
    // S16 phases of the tile so far, and whether this step's QK16 was
    // issued ahead of the decision: for the first step, and when the step
    // before had a flagged sub-block (the MMA warp follows the same rule)
    uint32_t n16 = 0u;
    bool prev_any = true;
    const int qtile = (q0 + tt * kBM) / kBN + (rw >> 1);  // 64-row query tile of this warp
    // this query tile's row of the mask, or of the tau-sweep records
    uint8_t* mrow = nullptr;
    uint32_t* rrow = nullptr;
    if (qtile < p.T) {
      const size_t base = (((size_t)b * p.Hq + h) * p.T + qtile) * p.T;
      if (!kSweep && p.mask) mrow = p.mask + base;
      if (kSweep) rrow = p.records + base;
    }
    const float sig = p.sigma_f;
    const float2 sig2 = make_float2(sig, sig);
    const float T = p.tau_abs;
    const uint32_t dcode = p.delta_code;
    bool done_ok = false;
    const float* nkrow = p.nkmax + ((size_t)b * p.Hkv + g) * p.T;
    const float* nkcrow = p.nkc + ((size_t)b * p.Hkv + g) * p.T * C::CH;
    float nk_next = nsteps > 0 ? nkrow[jlo_t] : 0.0f;

    for (int jj = 0; jj < nsteps; ++jj) {
      const int jt = jlo_t + jj;
      const float nk = nk_next;  // loaded one step ahead
      if (jj + 1 < nsteps) nk_next = nkrow[jt + 1];
      bool rowvis = true;
      uint32_t vm = kAll;  // visible columns of this part (bit c = key k0 + col0 + c)
      if (jt < jf0 || jt > jf1) {  // the row does not see the whole tile
        const int k0 = jt * kBN;
        const int clo = imax(k0, lo), chi = imin(k0 + kBN - 1, hi);
        rowvis = clo <= chi;
        const int a = imax(clo - (k0 + col0), 0), z = imin(chi - (k0 + col0), NC - 1);
        vm = (rowvis && a <= z) ? ((z == 31 ? 0xFFFFFFFFu : ((1u << (z + 1)) - 1u)) & ~((1u << a) - 1u)) : 0u;
      }
      const bool all_full = __all_sync(0xffffffffu, vm == kAll);
      // bound on |A_tc sigma - A sigma| for this row and tile (see qg)
      float G = 0.0f;
#pragma unroll
      for (int c = 0; c < (kChunk ? 0 : C::CH); c += (C::CH >= 4 ? 4 : 2)) {
        if constexpr (C::CH >= 4) {
          const float4 kb = *reinterpret_cast<const float4*>(nkcrow + (size_t)jt * C::CH + c);
          float4 qw;
          if constexpr (TPR == 2)
            qw = *reinterpret_cast<const float4*>(qg + c);
          else
            qw = make_float4(QG(c), QG(c + 1), QG(c + 2), QG(c + 3));
          G = fmaf(qw.x, kb.x, fmaf(qw.y, kb.y, fmaf(qw.z, kb.z, fmaf(qw.w, kb.w, G))));
        } else {
          const float2 kb = *reinterpret_cast<const float2*>(nkcrow + (size_t)jt * C::CH + c);
          const float2 qw = *reinterpret_cast<const float2*>(qg + c);
          G = fmaf(qw.x, kb.x, fmaf(qw.y, kb.y, G));
        }
      }
      // can a logit of this tile reach the 8-bit limit?  (chunked: each of
      // the C roundings may add 1/16, (1 + 1/16)^4 < 1.3)
      const bool satp = satq * nk * (kChunk ? 1.3f : 1.0f) >= 400.0f;

      // ---- S = Q8 K8^T (fp32, TMEM) -> 8-bit logits
      uint32_t s8h[NC / 2];  // S8 pairs as f16x2 (exact values; cl until resolved)
      uint32_t gmx[NC / 8];  // per group of 8: max of the pairs (f16x2)
      uint32_t unc = 0u;     // visible logits whose candidates differ and that may matter
      uint32_t hmx = 0xFC00FC00u;  // f16x2 max of their high candidates ch (-inf: none)
      const float2 gp = make_float2(G, G);
      if (!fail) fail = !wait_bar_warp(cx, bar(M_S_FULL + 8 * tt), jj & 1);
      if constexpr (kChunk) {
        // Chunked logits: a_c = fl8(a_{c-1} + A_c sigma), chunk by chunk.
        // The tensor core's A_c (one K = 32 instruction, zero accumulator)
        // errs by less than 37 * 2^-25 x_c (x_c bounds |A_c| and each
        // product); with sigma's float rounding and the roundings of y and
        // y -+ g, g = qg[c] nkc + 2^-22 |y| bounds |y - (a_{c-1} + A_c sigma)|.
        // Where fl8(y - g) and fl8(y + g) differ, the logit's chunk is
        // re-derived exactly (integer dot product) before the next chunk.
        const uint8_t* sK8c = smem + C::OFF_ST + ((jt - J0) % C::NS) * C::STAGE_BYTES;
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) s8h[i] = 0u;
#pragma unroll 1
        for (int c = 0; c < C::CH; ++c) {
          uint32_t a32[NC];
          if (!fail) {
            tc_fence_after();
            tmem_ld_n(lane_base + C::S8_OFF + c * kBN + col0, a32);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < NC; ++e) a32[e] = 0u;
          }
          float qw = 0.0f;  // QG(c) with constant indices (no local memory)
#pragma unroll
          for (int cc = 0; cc < C::CH; ++cc)
            if (cc == c) qw = QG(cc);
          const float gc = qw * nkcrow[(size_t)jt * C::CH + c];
          uint32_t ucm = 0u;  // logits whose rounding of this chunk is uncertain
#pragma unroll
          for (int i = 0; i < NC / 2; ++i) {
            const __half2 ph = as_half2(s8h[i]);
            const float2 av = make_float2(__uint_as_float(a32[2 * i]), __uint_as_float(a32[2 * i + 1]));
            const float2 y = __ffma2_rn(av, sig2, make_float2(__low2float(ph), __high2float(ph)));
            const float g0 = fmaf(fabsf(y.x), 0x1p-22f, gc), g1 = fmaf(fabsf(y.y), 0x1p-22f, gc);
            const uint16_t cl = cvt_e4m3x2(y.y - g1, y.x - g0), ch = cvt_e4m3x2(y.y + g1, y.x + g0);
            const uint32_t dd = (uint32_t)(cl ^ ch);
            const uint32_t um = ((dd & 0xFFu) ? 0x0000FFFFu : 0u) | ((dd >> 8) ? 0xFFFF0000u : 0u);
            s8h[i] = (e4m3x2_to_f16x2(cl) & ~um) | (s8h[i] & um);  // uncertain: keep a_{c-1}
            ucm |= ((uint32_t)((dd & 0xFFu) != 0u) << (2 * i)) | ((uint32_t)((dd >> 8) != 0u) << (2 * i + 1));
          }
          if (!all_full) ucm &= vm;  // hidden keys take -inf below
          if (fail) ucm = 0u;
          for (;;) {  // one uncertain logit at a time over the warp
            const unsigned who = __ballot_sync(0xffffffffu, ucm != 0u);
            if (!who) break;
            const int src = __ffs(who) - 1;
            const int cb = __shfl_sync(0xffffffffu, ucm ? (__ffs(ucm) - 1) : 0, src);
            const long long acc = exact_dot_chunk<D>(sQ8, sK8c, rw * 32 + src, col0 + cb, c, lane);
            if (lane == src) {
              static_assert(NC == 32 || NC == 16, "the switches below list up to 16 pairs");
              uint32_t w = 0u;
              switch (cb >> 1) {
#define LAMP_GET_CASE(i) \
  case i:                \
    if constexpr (i < NC / 2) w = s8h[i]; \
    break;
                LAMP_GET_CASE(0) LAMP_GET_CASE(1) LAMP_GET_CASE(2) LAMP_GET_CASE(3)
                LAMP_GET_CASE(4) LAMP_GET_CASE(5) LAMP_GET_CASE(6) LAMP_GET_CASE(7)
                LAMP_GET_CASE(8) LAMP_GET_CASE(9) LAMP_GET_CASE(10) LAMP_GET_CASE(11)
                LAMP_GET_CASE(12) LAMP_GET_CASE(13) LAMP_GET_CASE(14) LAMP_GET_CASE(15)
#undef LAMP_GET_CASE
                default: break;
              }
              const __half2 wh = as_half2(w);
              const uint32_t hv = e4m3_f16_of_chunk_sum((cb & 1) ? __high2float(wh) : __low2float(wh), acc, p.sig18);
              const uint32_t keep = (cb & 1) ? 0x0000FFFFu : 0xFFFF0000u;
              const uint32_t put = (hv * 0x00010001u) & ~keep;
              switch (cb >> 1) {
#define LAMP_PUT_CASE(i) \
  case i:                \
    if constexpr (i < NC / 2) s8h[i] = (s8h[i] & keep) | put; \
    break;
                LAMP_PUT_CASE(0) LAMP_PUT_CASE(1) LAMP_PUT_CASE(2) LAMP_PUT_CASE(3)
                LAMP_PUT_CASE(4) LAMP_PUT_CASE(5) LAMP_PUT_CASE(6) LAMP_PUT_CASE(7)
                LAMP_PUT_CASE(8) LAMP_PUT_CASE(9) LAMP_PUT_CASE(10) LAMP_PUT_CASE(11)
                LAMP_PUT_CASE(12) LAMP_PUT_CASE(13) LAMP_PUT_CASE(14) LAMP_PUT_CASE(15)
#undef LAMP_PUT_CASE
                default: break;
              }
              ucm &= ucm - 1u;
            }
            if (lane == 0) ++c_fix;
          }
        }
#pragma unroll
        for (int g4 = 0; g4 < NC / 8; ++g4)
          gmx[g4] = as_u32(__hmax2(__hmax2(as_half2(s8h[4 * g4]), as_half2(s8h[4 * g4 + 1])),
                                   __hmax2(as_half2(s8h[4 * g4 + 2]), as_half2(s8h[4 * g4 + 3]))));
      } else {
      uint32_t a32[NC];
      if (!fail) {
        tc_fence_after();
        tmem_ld_n(lane_base + C::S8_OFF + col0, a32);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int c = 0; c < NC; ++c) a32[c] = 0u;
      }
      // S8 = fl8(A sigma) is one of the E4M3 values from cl = fl8(y - G) to
      // ch = fl8(y + G) (y = A_tc sigma, G bounds the tensor core's error),
      // so it is certain when the two agree -- almost always.  Of the
      // others, only logits that can change m, P8, the detector or the
      // saturation count may need the exact value: m (the running max before
      // this tile) is exact and <= the new max, and a logit whose largest
      // possible value ch is <= m - 6.75 rounds x8 to <= -7 (P8 = 0, below
      // any delta > 0) and is not the maximum.  With delta = 0, or when the
      // tile can reach the 8-bit limit, all count.  A group of 8 logits is
      // looked at only if one of them is uncertain and its largest cl is
      // close enough to m: with cl the lower rounding, y - G is at most cl
      // plus half a gap (<= |cl|/16 + 2^-10), and one more rounding of y + G
      // adds at most |.|/16 + 2^-10, so the exact values are at most
      // cl + 0.13 |cl| + 2.2 G + 2^-8: below m - 6.75 nothing in it counts.
      // Those uncertain logits are resolved once the tile maximum is known.
      {
        // delta = 0 (first stage off): stage 1 holds for every visible entry,
        // so besides the logits near m only those whose candidates lie on
        // both sides of +tau_abs or -tau_abs can move the flag; the sweep
        // pass with delta = 0 needs every |S8|
        const bool tsplit = kNoStage1 && T > 0.0f;
        const float thr = (satp || (kSweep && dcode == 0u)) ? -INFINITY : m - 6.75f;
        const __half2 lthr = __half2half2(__float2half_rd(thr));
        const float c = thr - 2.2f * G - 0x1p-8f;  // cl + 0.13 |cl| > c  <=>  cl > c / 1.13 or c / 0.87
        const __half2 sthr =
            __half2half2(__float2half_rd(kNoStage1 ? -INFINITY : (c >= 0.0f ? 0.884f * c : 1.15f * c)));
        const float2 gm = make_float2(-G, -G);
#pragma unroll
        for (int g4 = 0; g4 < NC / 8; ++g4) {  // 4 pairs at a time, one branch
          uint32_t d4 = 0u, d16[4], ch4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = 4 * g4 + k;
            const float2 av = make_float2(__uint_as_float(a32[2 * i]), __uint_as_float(a32[2 * i + 1]));
            const float2 yl = __ffma2_rn(av, sig2, gm), yh = __ffma2_rn(av, sig2, gp);
            const uint16_t cl = cvt_e4m3x2(yl.y, yl.x), ch = cvt_e4m3x2(yh.y, yh.x);
            s8h[i] = e4m3x2_to_f16x2(cl);
            d16[k] = (uint32_t)(cl ^ ch);
            d4 |= d16[k];
            ch4[k] = ch;
          }
          const __half2 mg = __hmax2(__hmax2(as_half2(s8h[4 * g4]), as_half2(s8h[4 * g4 + 1])),
                                     __hmax2(as_half2(s8h[4 * g4 + 2]), as_half2(s8h[4 * g4 + 3])));
          gmx[g4] = as_u32(mg);
          // rare: a logit near a boundary, maybe relevant (needed by some lane
          // of the warp for about one group in ten on the outlier workload).
          // The vote makes it a warp-uniform branch: a per-lane condition
          // lets the compiler run the body predicated on every group.
          const bool grp_unc = d4 != 0u && __hgt2_mask(mg, sthr) != 0u;
          if (__any_sync(0xffffffffu, grp_unc)) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i = 4 * g4 + k;
              const uint32_t hb = e4m3x2_to_f16x2((uint16_t)ch4[k]);
              const __half2 hh = as_half2(hb);
              uint32_t rel = __hgt2_mask(hh, lthr);
              if (tsplit) {  // T and -T are E4M3 values: exact in f16
                const __half2 tpos = __half2half2(__float2half_rn(T)), tneg = __hneg2(tpos);
                const __half2 hl = as_half2(s8h[i]);
                rel |= (__hlt2_mask(hl, tpos) & __hge2_mask(hh, tpos)) | (__hle2_mask(hl, tneg) & __hgt2_mask(hh, tneg));
              }
              uint32_t u = grp_unc ? rel & (((d16[k] & 0xFFu) ? 0x0000FFFFu : 0u) | ((d16[k] >> 8) ? 0xFFFF0000u : 0u)) : 0u;
              if (!all_full)
                u &= (((vm >> (2 * i)) & 1u) ? 0x0000FFFFu : 0u) | (((vm >> (2 * i + 1)) & 1u) ? 0xFFFF0000u : 0u);
              unc |= ((u & 1u) << (2 * i)) | (((u >> 16) & 1u) << (2 * i + 1));
              hmx = as_u32(__hmax2(as_half2(hmx), as_half2((hb & u) | (0xFC00FC00u & ~u))));
            }
          }
        }
      }
      }  // one rounding of the whole dot product
      if (fail) unc = 0u;
      // hidden keys take -inf: they are never the max and x8 saturates to -448 (P8 = 0)
      if (!all_full) {
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) {
          const uint32_t keep = (((vm >> (2 * i)) & 1u) ? 0x0000FFFFu : 0u) | (((vm >> (2 * i + 1)) & 1u) ? 0xFFFF0000u : 0u);
          s8h[i] = (s8h[i] & keep) | (0xFC00FC00u & ~keep);
        }
      }

      // ---- tile max over both halves.  The largest cl is a lower bound of
      // it and the largest ch of the uncertain logits an upper bound; they
      // agree unless an uncertain logit may be the maximum (rare).
      float2* xlh = (float2*)(misc + M_XLH) + tt * TPR * kBM;
      float lo_row, hi_row;
      {
        __half2 mx;
        if (all_full) {
          mx = as_half2(gmx[0]);
#pragma unroll
          for (int g8 = 1; g8 < NC / 8; ++g8) mx = __hmax2(mx, as_half2(gmx[g8]));
        } else {
          mx = as_half2(s8h[0]);
#pragma unroll
          for (int i = 1; i < NC / 2; ++i) mx = __hmax2(mx, as_half2(s8h[i]));
        }
        const float lo = fmaxf(__low2float(mx), __high2float(mx));
        const __half2 hx = as_half2(hmx);
        const float hi = fmaxf(lo, fmaxf(__low2float(hx), __high2float(hx)));
        xlh[hf * kBM + t] = make_float2(lo, hi);
        bar_sync(pair_bar, kPairThreads);
        lo_row = lo;
        hi_row = hi;
#pragma unroll
        for (int p2 = 0; p2 < TPR; ++p2) {
          if (p2 == hf) continue;
          const float2 o = xlh[p2 * kBM + t];
          lo_row = fmaxf(lo_row, o.x);
          hi_row = fmaxf(hi_row, o.y);
        }
      }
      // Uncertain logits are settled in up to two passes.  Pass 0 (only if
      // an uncertain logit may be a row's maximum; the same decision in both
      // warps of the row group, which hold the same rows): those whose ch
      // exceeds the row's largest cl are re-derived exactly, then the maximum
      // is exchanged again.  Pass 1, with the maximum exact: cl stands for a
      // logit if every value from cl to ch gives the same P8 code (P8 is
      // monotone in S8, so the ends decide), the same side of tau_abs (the
      // flag and the negative-logit scan), the same saturation count and
      // (tau sweep) the same half-ulp8; otherwise it is re-derived too.
      float m_tile = lo_row;
      const bool max_unc = __any_sync(0xffffffffu, hi_row > lo_row);
#pragma unroll 1
      for (int pass = max_unc ? 0 : (__any_sync(0xffffffffu, unc != 0u) ? 1 : 2); pass < 2; ++pass) {
        uint32_t ex = 0u;  // logits to re-derive exactly in this pass
        if (!kSweep && pass == 1) {
          // With the row maximum exact, a row whose own maximum flags it
          // (P8 of the maximum >= delta and the maximum >= tau_abs: a flagged
          // entry) flags its sub-block.  Every row of a sub-block flagged
          // this way takes P16 (from the 16-bit products and the exact m),
          // the sub-block's stage-1 bit comes from the row maxima, and the
          // flag is set whatever its other logits are: their uncertain ones
          // can change nothing except the saturation count (kept when the
          // tile can saturate) and are left unresolved.
          const float mnr = rowvis ? fmaxf(m, m_tile) : m;
          const bool st1m = rowvis && tab[cvt_e4m3x2(0.0f, m_tile - mnr) & 0xFFu] >= dcode;
          const bool rowflag =
              rowvis && (p.force == 1 || (p.force == 0 && st1m && (T <= 0.0f || m_tile >= T)));
          const unsigned bfc = __ballot_sync(0xffffffffu, rowflag);
          const bool sb_flagged = ((lane >> 4) ? (bfc >> 16) : (bfc & 0xFFFFu)) != 0u;
          if (sb_flagged && !satp) unc = 0u;
        }
        if constexpr (kNoStage1) {
          // first stage off: most uncertain logits straddle +-tau_abs, where
          // the comparison of the candidates cannot settle them (measured:
          // half of them); they are re-derived without it
          if (pass == 1) {
            ex = unc;
            unc = 0u;
          }
        }
        uint32_t wor = __reduce_or_sync(0xffffffffu, unc);
        if (wor && !(kNoStage1 && pass == 1)) {
          const float mref = pass == 0 ? lo_row : (rowvis ? fmaxf(m, m_tile) : m);
          const __half2 mh = __float2half2_rn(mref);
          const __half2 tp = __float2half2_rn(T), zero2 = __float2half2_rn(0.0f);
          const float2 gm = make_float2(-G, -G);
          tc_fence_after();
          // one pair of logits at a time (a pair any lane of the warp has an
          // uncertain logit in); both candidates come from the accumulators
#pragma unroll 1
          while (wor) {
            const int i = (__ffs(wor) - 1) >> 1;
            wor &= ~(3u << (2 * i));
            uint32_t ar[2];
            tmem_ld2(lane_base + C::S8_OFF + col0 + 2 * i, ar);
            tmem_wait_ld();
            const uint32_t ub = (unc >> (2 * i)) & 3u;
            if (ub) {
              const float2 av = make_float2(__uint_as_float(ar[0]), __uint_as_float(ar[1]));
              const float2 yl = __ffma2_rn(av, sig2, gm), yh = __ffma2_rn(av, sig2, gp);
              const __half2 ll = as_half2(e4m3x2_to_f16x2(cvt_e4m3x2(yl.y, yl.x)));
              const __half2 hh = as_half2(e4m3x2_to_f16x2(cvt_e4m3x2(yh.y, yh.x)));
              uint32_t sel;  // per half: re-derive
              if (pass == 0) {
                sel = __hgt2_mask(hh, mh);
              } else {
                const __half2 al = __habs2(ll), ah = __habs2(hh);
                const uint32_t xl = cvt_e4m3x2_f16x2(__hsub2(ll, mh)), xh = cvt_e4m3x2_f16x2(__hsub2(hh, mh));
                sel = __hge2_mask(al, tp) ^ __hge2_mask(ah, tp);
                // a sign change between the ends passes |S8| = 0
                const uint32_t straddle = __hlt2_mask(ll, zero2) & __hgt2_mask(hh, zero2);
                if (T > 0.0f) sel |= straddle & __hge2_mask(__hmax2(al, ah), tp);
                if (satp) {
                  const __half2 sat2 = __float2half2_rn(448.0f);
                  sel |= __heq2_mask(al, sat2) ^ __heq2_mask(ah, sat2);
                }
                if constexpr (kSweep) {  // the same half-ulp8: the same binade (all below 2^-6 share one)
                  const __half2 lo6 = __float2half2_rn(0x1p-6f), lo5 = __float2half2_rn(0x1p-5f);
                  const uint32_t e = (as_u32(__hmax2(al, lo6)) ^ as_u32(__hmax2(ah, lo6))) & 0x7C007C00u;
                  sel |= ((e & 0xFFFFu) ? 0x0000FFFFu : 0u) | ((e >> 16) ? 0xFFFF0000u : 0u);
                  sel |= straddle & __hge2_mask(__hmax2(al, ah), lo5);
                }
                if (((xl ^ xh) & 0xFFu) && tab[xl & 0xFFu] != tab[xh & 0xFFu]) sel |= 0x0000FFFFu;
                if (((xl ^ xh) >> 8) && tab[xl >> 8] != tab[xh >> 8]) sel |= 0xFFFF0000u;
              }
              ex |= (ub & ((sel & 1u) | ((sel >> 15) & 2u))) << (2 * i);
            }
          }
          if (pass == 1) c_res += __popc(unc & ~ex);
          else c_fmax += __popc(ex);
          unc = pass == 1 ? 0u : (unc & ~ex);
        }
        // exact re-derivation, one logit at a time over the warp
        if (__any_sync(0xffffffffu, ex != 0u)) {
          const uint8_t* sK8 = (C::NS == 1 && !kSweep && ((jt - J0) & 1))
                                   ? smem + C::OFF_K8B  // the second K8 slot of the one-stage layout
                                   : smem + C::OFF_ST + ((jt - J0) % C::NS) * C::STAGE_BYTES;
          for (;;) {
            const unsigned who = __ballot_sync(0xffffffffu, ex != 0u);
            if (!who) break;
            const int src = __ffs(who) - 1;
            const int cb = __shfl_sync(0xffffffffu, ex ? (__ffs(ex) - 1) : 0, src);
            const long long acc = exact_dot<D>(sQ8, sK8, rw * 32 + src, col0 + cb, lane);
            if (lane == src) {
              const uint32_t hv = e4m3_f16_of_product(acc, p.sig18);
              // replace half (cb & 1) of pair cb >> 1: a switch with constant
              // indices keeps s8h in registers
              static_assert(NC == 32 || NC == 16, "the switch below lists up to 16 pairs");
              const uint32_t keep = (cb & 1) ? 0x0000FFFFu : 0xFFFF0000u;
              const uint32_t put = (hv * 0x00010001u) & ~keep;
              switch (cb >> 1) {
#define LAMP_FIX_CASE(i) \
  case i:                  \
    if constexpr (i < NC / 2) s8h[i] = (s8h[i] & keep) | put; \
    break;
                LAMP_FIX_CASE(0) LAMP_FIX_CASE(1) LAMP_FIX_CASE(2) LAMP_FIX_CASE(3)
                LAMP_FIX_CASE(4) LAMP_FIX_CASE(5) LAMP_FIX_CASE(6) LAMP_FIX_CASE(7)
                LAMP_FIX_CASE(8) LAMP_FIX_CASE(9) LAMP_FIX_CASE(10) LAMP_FIX_CASE(11)
                LAMP_FIX_CASE(12) LAMP_FIX_CASE(13) LAMP_FIX_CASE(14) LAMP_FIX_CASE(15)
#undef LAMP_FIX_CASE
                default: break;
              }
              ex &= ex - 1u;
            }
            if (lane == 0) ++c_fix;
          }
        }
        if (pass == 0) {  // the maximum again, from the exact values (both warps of the row group)
          __half2 mx = as_half2(s8h[0]);
#pragma unroll
          for (int i = 1; i < NC / 2; ++i) mx = __hmax2(mx, as_half2(s8h[i]));
          const float mine = fmaxf(__low2float(mx), __high2float(mx));
          xch[hf * kBM + t] = mine;
          bar_sync(pair_bar, kPairThreads);
          m_tile = mine;
#pragma unroll
          for (int p2 = 0; p2 < TPR; ++p2)
            if (p2 != hf) m_tile = fmaxf(m_tile, xch[p2 * kBM + t]);
        }
      }
      const float m_new = rowvis ? fmaxf(m, m_tile) : m;

      // ---- detector, per row: P8 is monotone in S8, so the tile maximum
      // decides stage 1, and a positive logit >= tau_abs with P8 >= delta
      // exists iff the maximum is one.  Only negative logits <= -tau_abs can
      // flag otherwise; that case is checked element by element.
      bool st1 = false, flg = false;
      if (rowvis) {
        st1 = tab[cvt_e4m3x2(0.0f, m_tile - m_new) & 0xFFu] >= dcode;
        flg = st1 && (T <= 0.0f || m_tile >= T);
      }
      uint32_t scode = 0u;  // sweep pass: code of this row's largest stage-1 half-ulp8
      if constexpr (kSweep) {
        // the stage-1 entries are the visible S8 >= some threshold (P8 is
        // monotone in S8): the largest |S8| among them is the tile maximum,
        // or the smallest of them when it is negative
        flg = false;
        float A = fabsf(m_tile);
        const bool scan = rowvis && st1 && (m_new <= 0.0f || tab[cvt_e4m3x2(0.0f, -m_new) & 0xFFu] >= dcode);
        if (__any_sync(0xffffffffu, scan)) {  // same outcome in both halves
          __half2 mn = __float2half2_rn(0.0f);
          if (scan) {
            const __half2 mh = __float2half2_rn(m_new);
#pragma unroll
            for (int i = 0; i < NC / 2; ++i) {
              const __half2 sv = as_half2(s8h[i]);
              const uint32_t x8 = cvt_e4m3x2_f16x2(__hsub2(sv, mh));
              const bool q0 = ((vm >> (2 * i)) & 1u) && tab[x8 & 0xFFu] >= dcode;
              const bool q1 = ((vm >> (2 * i + 1)) & 1u) && tab[x8 >> 8] >= dcode;
              mn = __hmin2(mn, __halves2half2(q0 ? __low2half(sv) : __float2half(0.0f),
                                              q1 ? __high2half(sv) : __float2half(0.0f)));
            }
          }
          const float mine = fminf(__low2float(mn), __high2float(mn));
          xb[hf * kBM + t] = __float_as_uint(mine);
          bar_sync(pair_bar, kPairThreads);
          float mn_row = mine;
#pragma unroll
          for (int p2 = 0; p2 < TPR; ++p2)
            if (p2 != hf) mn_row = fminf(mn_row, __uint_as_float(xb[p2 * kBM + t]));
          if (scan) A = fmaxf(A, -mn_row);
        }
        if (rowvis && st1) {
          const int e = (int)((__float_as_uint(A) >> 23) & 0xFFu) - 127;  // floor(log2 A), A >= 2^-6
          scode = (uint32_t)((A < 0x1p-6f ? -10 : e - 4) + 11);           // half-ulp8 = 2^(code - 11)
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) scode = max(scode, __shfl_xor_sync(0xffffffffu, scode, o));
      }
      const bool maybe_neg = !kSweep && rowvis && st1 && !flg && T > 0.0f &&
                             tab[cvt_e4m3x2(0.0f, -T - m_new) & 0xFFu] >= dcode;
      if (__any_sync(0xffffffffu, maybe_neg)) {  // same outcome in both halves
        uint32_t mine = 0u;
        if (maybe_neg) {
          const __half2 mh = __float2half2_rn(m_new);
#pragma unroll
          for (int i = 0; i < NC / 2; ++i) {
            const __half2 sv = as_half2(s8h[i]);
            const uint32_t x8 = cvt_e4m3x2_f16x2(__hsub2(sv, mh));
            if (((vm >> (2 * i)) & 1u) && __low2float(sv) <= -T && tab[x8 & 0xFFu] >= dcode) mine = 1u;
            if (((vm >> (2 * i + 1)) & 1u) && __high2float(sv) <= -T && tab[x8 >> 8] >= dcode) mine = 1u;
          }
        }
        xb[hf * kBM + t] = mine;
        bar_sync(pair_bar, kPairThreads);
        uint32_t any_neg = mine;
#pragma unroll
        for (int p2 = 0; p2 < TPR; ++p2)
          if (p2 != hf) any_neg |= xb[p2 * kBM + t];
        if (maybe_neg) flg = any_neg != 0u;
      }
      if (__any_sync(0xffffffffu, rowvis && satp)) {  // warp-uniform: rare
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) {
          const __half2 sv = as_half2(s8h[i]);
          if (rowvis && satp) c_sat += (fabsf(__low2float(sv)) == 448.0f) + (fabsf(__high2float(sv)) == 448.0f);
        }
      }

      // ---- sub-block bits: lanes 0-15 and 16-31 of a warp are two sub-blocks
      unsigned bf = __ballot_sync(0xffffffffu, flg);
      unsigned bv = 0u;
      if (p.force != 0 || hf == 0) bv = __ballot_sync(0xffffffffu, rowvis);
      if (p.force == 1) bf = bv;
      if (p.force == 2) bf = 0u;
      const bool my_flag = ((lane >> 4) ? (bf >> 16) : (bf & 0xFFFFu)) != 0u;
      uint8_t* sflag = misc + M_SFLAG + 32 * tt + 16 * (jj & 1);
      if (hf == 0) {  // the owner of the 64-row query tile needs the sub-block bits
        const unsigned b1 = __ballot_sync(0xffffffffu, st1);
        const uint32_t scode_hi = kSweep ? __shfl_sync(0xffffffffu, scode, 16) : 0u;  // second sub-block's code
        if (lane == 0)
          *(volatile uint32_t*)(sflag + 4 * rw) =
              ((bf & 0xFFFFu) != 0u) | (((bf >> 16) != 0u) << 1) | (((b1 & 0xFFFFu) != 0u) << 2) |
              (((b1 >> 16) != 0u) << 3) | (((bv & 0xFFFFu) != 0u) << 4) | (((bv >> 16) != 0u) << 5) |
              (scode << 8) | (scode_hi << 12);
      }
      // (after a failed wait a thread keeps stepping with its waits skipped,
      // so every thread of the tile reaches every barrier)
      tc_fence_before();  // this thread's S8 reads before the buffer is handed back
      const bool any = bar_red_or(tile_bar, C::SM_THREADS, my_flag);

      if (t == 0 && hf == 0 && !fail) {  // every S8 read is done: the buffer may take the next QK8
        *(volatile uint8_t*)(misc + M_ANY + 2 * tt + (jj & 1)) = any ? 1 : 0;
        mbar_arrive(bar(M_DEC + 8 * tt));
      }
      if (hf == 0 && (rw & 1) == 0 && __any_sync(0xffffffffu, !fail))  // the tile's two owner warps
      if (lane == 0 && !fail) {
        // lane 0 of row groups 0 and 2 owns the 64-row query tile of groups (rw, rw+1)
        const unsigned long long ww = *(volatile unsigned long long*)(sflag + 4 * rw);  // rw even: 8-byte aligned
        const uint32_t w0 = (uint32_t)ww, w1 = (uint32_t)(ww >> 32);
        const uint32_t fl4 = (w0 & 3u) | ((w1 & 3u) << 2);
        const uint32_t st4 = ((w0 >> 2) & 3u) | (((w1 >> 2) & 3u) << 2);
        const uint32_t vs4 = ((w0 >> 4) & 3u) | (((w1 >> 4) & 3u) << 2);
        if (vs4) {
          const int nf = __popc(fl4);
          c_strips += __popc(vs4);
          c_st1 += __popc(st4 & vs4);
          if constexpr (kSweep) {
            ++c_h0;  // counts visited tiles only (no flags in this pass)
            const uint32_t codes = ((w0 >> 8) & 0xFFu) | (((w1 >> 8) & 0xFFu) << 8);
            if (rrow) rrow[jt] = vs4 | (st4 << 4) | (codes << 8);
          } else {
            c_h0 += nf == 0;
            c_h1 += nf == 1;
            c_h2 += nf > 1;
            c_fl += nf;
            if (mrow) mrow[jt] = (uint8_t)(fl4 | (st4 << 4));
          }
        }
      }

      if constexpr (!kSweep) {
      // ---- x8 = fl8(S8 - m) (fp16 difference, then one E4M3 rounding: equal
      // to the single rounding for E4M3 operands), P8 = fl8(e^x8) (exact,
      // exp8_f16x2); rows of flagged sub-blocks take P16 below instead
      uint32_t pw[NC / 2];
      uint32_t pc[kPV8 ? NC / 4 : 1];  // FP8 P.V: the P8 codes, four a word
#pragma unroll
      for (int i = 0; i < NC / 2; ++i) pw[i] = 0u;
#pragma unroll
      for (int i = 0; i < (kPV8 ? NC / 4 : 1); ++i) pc[i] = 0u;
      const bool want_p8 = rowvis && !my_flag;
      if (__any_sync(0xffffffffu, want_p8)) {  // warp-uniform: most warps have only flagged rows
        const __half2 mh = __float2half2_rn(m_new);
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) {
          const __half2 xh = __hsub2(as_half2(s8h[i]), mh);
          const uint32_t c2 = exp8_code2(cvt_e4m3x2_f16x2(xh));
          pw[i] = want_p8 ? e4m3x2_to_f16x2((uint16_t)c2) : 0u;
          if constexpr (kPV8) pc[i >> 1] |= (want_p8 ? c2 : 0u) << (16 * (i & 1));
        }
      }

      // ---- the previous P.V must be done before O is rescaled and P is
      // rewritten; the rescale overlaps this step's QK16 on the tensor core
      if (jj > 0 && !fail) fail = !wait_bar_warp(cx, bar(M_PV_DONE + 8 * tt), (jj - 1) & 1);
      const float alpha = (m_new == m) ? 1.0f : (m == -INFINITY ? 0.0f : ex2_approx((m - m_new) * kLog2e));
      if (!fail && jj > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        tc_fence_after();
        // this part rescales O columns [hf D/TPR, (hf+1) D/TPR)
#pragma unroll 1
        for (int c0 = hf * (D / TPR); c0 < (hf + 1) * (D / TPR); c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                        make_float2(alpha, alpha));
            o[i] = __float_as_uint(v.x);
            o[i + 1] = __float_as_uint(v.y);
          }
          tmem_st32(lane_base + c0, o);
        }
        tmem_wait_st();
      }

      // ---- 16-bit recompute for the rows of flagged sub-blocks
      // (the QK16 of every step is computed; a step without flags skips it)
      // two S16 buffers (one stage): buffer jj & 1 completes every other step
      // (two S16 buffers: n16 counts the phases of each in one half-word)
      const uint32_t s16_bar = C::S16_BUFS == 2 ? bar(M_S16_FULL + 8 * (jj & 1)) : bar(M_S16_FULL + 8 * tt);
      const uint32_t s16_sh = C::S16_BUFS == 2 ? 16u * (uint32_t)(jj & 1) : 0u;
      if (any && !fail) fail = !wait_bar_warp(cx, s16_bar, (n16 >> s16_sh) & 1u);
      n16 += (any || prev_any) ? (1u << s16_sh) : 0u;  // QK16 of this step was issued
      prev_any = any;
      if (any && !fail) {
        tc_fence_after();
        uint32_t r16[NC];
        tmem_ld_n(lane_base + C::S16_OFF + (C::S16_BUFS == 2 ? (jj & 1) * kBN : 0) + col0, r16);
        tmem_wait_ld();
        if (my_flag && rowvis) {
          const float sl2 = sig * kLog2e, ml = m_new * kLog2e;
          const float2 sl22 = make_float2(sl2, sl2), ml2 = make_float2(-ml, -ml);
#pragma unroll
          for (int i = 0; i < NC / 2; ++i) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(r16[2 * i]), __uint_as_float(r16[2 * i + 1])),
                                        sl22, ml2);
            pw[i] = cvt_f16x2_sat(ex2_approx(x.y), ex2_approx(x.x));
          }
          if (!all_full) {
#pragma unroll
            for (int i = 0; i < NC / 2; ++i) {
              if (!((vm >> (2 * i)) & 1u)) pw[i] &= 0xFFFF0000u;
              if (!((vm >> (2 * i + 1)) & 1u)) pw[i] &= 0x0000FFFFu;
            }
          }
        }
      }

      if (!fail) {
        {  // l = alpha l + sum of this half's P (exact fp16 values, fp32 sums)
          float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int i = 0; i < NC / 2; ++i) add_f32_f16x2(ls[2 * (i & 1)], ls[2 * (i & 1) + 1], pw[i]);
          l = fmaf(alpha, l, (ls[0] + ls[1]) + (ls[2] + ls[3]));
        }
        if constexpr (kPV8) {
          // the P8 tile (K-major, 64-byte swizzle; 0 in rows of flagged
          // sub-blocks) and, when the step has a flagged sub-block, the P16
          // tile with P16 in those rows and 0 in the others
#pragma unroll
          for (int k = 0; k < NC / 16; ++k)
            *reinterpret_cast<uint4*>(sP + C::P16_BYTES + swz_offset(t, col0 + 16 * k, kBM, 64)) =
                make_uint4(pc[4 * k], pc[4 * k + 1], pc[4 * k + 2], pc[4 * k + 3]);
          if (any) {
#pragma unroll
            for (int k = 0; k < NC / 8; ++k) {
              const uint4 v4 = my_flag ? make_uint4(pw[4 * k], pw[4 * k + 1], pw[4 * k + 2], pw[4 * k + 3])
                                       : make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(sP + swz_offset(t, 2 * col0 + 16 * k, kBM, 128)) = v4;
            }
          }
        } else {
          // this part of the P row -> shared memory (K-major, 128-byte swizzle)
#pragma unroll
          for (int k = 0; k < NC / 8; ++k) {
            const uint4 v4 = make_uint4(pw[4 * k], pw[4 * k + 1], pw[4 * k + 2], pw[4 * k + 3]);
            *reinterpret_cast<uint4*>(sP + swz_offset(t, 2 * col0 + 16 * k, kBM, 128)) = v4;
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(M_P_FULL + 8 * tt));
      }
      }  // !kSweep
      m = m_new;
      if (jj == nsteps - 1) done_ok = !fail;
    }

    // ---- epilogue: l of the row = sum of both halves; out = O / l, LSE = m + ln l
    xch[hf * kBM + t] = l;
    bar_sync(pair_bar, kPairThreads);
    float lrow = 0.0f;  // the parts in a fixed order: the same sum in every thread of the row
#pragma unroll
    for (int p2 = 0; p2 < TPR; ++p2) lrow += xch[p2 * kBM + t];
    if (kSweep) done_ok = false;  // no output
    if (done_ok) done_ok = wait_bar_warp(cx, bar(M_PV_DONE + 8 * tt), (nsteps - 1) & 1);
    if (done_ok) {
      tc_fence_after();
      const float inv = lrow > 0.0f ? 1.0f / lrow : 0.0f;
      const bool live = R < p.N;
      if (live && hf == 0 && p.lse)
        p.lse[((size_t)b * p.Hq + h) * p.N + R] = lrow > 0.0f ? m + logf(lrow) : -INFINITY;
      char* orow = (char*)p.out + ((size_t)b * p.o_stride[0] + (size_t)R * p.o_stride[1] +
                                   (size_t)h * p.o_stride[2]) * (p.out_f32 ? 4 : 2);
#pragma unroll 1
      for (int c0 = hf * (D / TPR); c0 < (hf + 1) * (D / TPR); c0 += 16) {
        uint32_t o[16];
        tmem_ld16(lane_base + c0, o);
        tmem_wait_ld();
        if (!live) continue;
        if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(orow + (size_t)c0 * 4);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                 __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        } else {
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            __nv_bfloat162 bb = __floats2bfloat162_rn(__uint_as_float(o[2 * i]) * inv,
                                                      __uint_as_float(o[2 * i + 1]) * inv);
            memcpy(&w[i], &bb, 4);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + (size_t)c0 * 2);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    if (p.counters) {
      typedef unsigned long long u64;
      const uint32_t c_tiles = c_h0 + c_h1 + c_h2;
      if (lane == 0 && hf == 0 && (rw & 1) == 0 && c_tiles) {
        atomicAdd(&p.counters[0], (u64)c_tiles);
        if (!kSweep) {
          atomicAdd(&p.counters[1], (u64)c_h0);
          atomicAdd(&p.counters[2], (u64)c_h1);
          atomicAdd(&p.counters[3], (u64)c_h2);
          atomicAdd(&p.counters[6], (u64)c_fl);
        }
        atomicAdd(&p.counters[4], (u64)c_strips);
        atomicAdd(&p.counters[5], (u64)c_st1);
      }
      c_sat = __reduce_add_sync(0xffffffffu, c_sat);
      if (lane == 0 && c_sat) atomicAdd(&p.counters[7], (u64)c_sat);
      if (lane == 0 && c_fix) atomicAdd(&p.counters[8], (u64)c_fix);
      c_res = __reduce_add_sync(0xffffffffu, c_res);
      if (lane == 0 && c_res) atomicAdd(&p.counters[13], (u64)c_res);
      c_fmax = __reduce_add_sync(0xffffffffu, c_fmax);
      if (lane == 0 && c_fmax) atomicAdd(&p.counters[14], (u64)c_fmax);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- launcher
template <int D, int kMode, int kOpt>
static cudaError_t launch_fwd_d(FwdParams p, cudaStream_t st) {
  using C = Cfg<D, kOpt>;
  cudaError_t e =
      cudaFuncSetAttribute(lamp_fwd_kernel<D, kMode, kOpt>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  p.nqb = (p.N + kBM * C::NT - 1) / (kBM * C::NT);
  const unsigned grid = (unsigned)p.nqb * (unsigned)p.B * (unsigned)p.Hq;
  if (grid == 0) return cudaSuccess;
  lamp_fwd_kernel<D, kMode, kOpt><<<grid, C::THREADS, C::SMEM, st>>>(p);
  return cudaGetLastError();
}

template <int D, int kOpt>
static cudaError_t launch_fwd_opt(const FwdParams& p, cudaStream_t st) {
  return p.delta_code == 0u ? launch_fwd_d<D, 1, kOpt>(p, st) : launch_fwd_d<D, 0, kOpt>(p, st);
}

template <int D>
static cudaError_t launch_fwd_mode(const FwdParams& p, cudaStream_t st, bool sweep, int opt) {
  if (sweep) return opt == 0 ? launch_fwd_d<D, 2, 0>(p, st) : cudaErrorInvalidValue;
  if constexpr (D != 256) {
    if (opt == kOptPV8) return launch_fwd_opt<D, kOptPV8>(p, st);
    if (opt == kOptChunk) return launch_fwd_opt<D, kOptChunk>(p, st);
  }
  return opt == 0 ? launch_fwd_opt<D, 0>(p, st) : cudaErrorInvalidValue;
}

// opt: 0, or one of the optional modes (FP8 P.V, chunked logits; d <= 128)
cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t st, bool sweep, int opt) {
  switch (d) {
    case 64: return launch_fwd_mode<64>(p, st, sweep, opt);
    case 128: return launch_fwd_mode<128>(p, st, sweep, opt);
    case 256: return launch_fwd_mode<256>(p, st, sweep, opt);
    default: return cudaErrorInvalidValue;
  }
}

// Histograms of the sweep records for several tau (as sub-block codes):
// hist[4 i .. 4 i + 3] += visited tiles, tiles with 0, 1, 2+ flagged
// sub-blocks at tau i.
__global__ void lamp_sweep_hist_kernel(const uint32_t* __restrict__ rec, long long n, const SweepCodes tcode,
                                       int ntau, unsigned long long* hist) {
  __shared__ unsigned long long acc[kMaxSweepTaus * 4];
  for (int i = threadIdx.x; i < ntau * 4; i += blockDim.x) acc[i] = 0ull;
  __syncthreads();
  uint32_t tot = 0u, h0[kMaxSweepTaus], h1[kMaxSweepTaus], h2[kMaxSweepTaus];
#pragma unroll
  for (int t = 0; t < kMaxSweepTaus; ++t) h0[t] = h1[t] = h2[t] = 0u;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const uint32_t r = rec[i];
    if (!(r & 0xFu)) continue;
    ++tot;
#pragma unroll
    for (int t = 0; t < kMaxSweepTaus; ++t) {
      const int tc = t < ntau ? tcode.v[t] : 16;
      int nf = 0;
#pragma unroll
      for (int sb = 0; sb < 4; ++sb) nf += (((r >> (4 + sb)) & 1u) && (int)((r >> (8 + 4 * sb)) & 0xFu) >= tc) ? 1 : 0;
      h0[t] += nf == 0;
      h1[t] += nf == 1;
      h2[t] += nf >= 2;
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxSweepTaus; ++t) {
    if (t >= ntau) break;
    if (tot) atomicAdd(&acc[4 * t], (unsigned long long)tot);
    if (h0[t]) atomicAdd(&acc[4 * t + 1], (unsigned long long)h0[t]);
    if (h1[t]) atomicAdd(&acc[4 * t + 2], (unsigned long long)h1[t]);
    if (h2[t]) atomicAdd(&acc[4 * t + 3], (unsigned long long)h2[t]);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < ntau * 4; i += blockDim.x)
    if (acc[i]) atomicAdd(&hist[i], acc[i]);
}

cudaError_t launch_sweep_hist(const uint32_t* rec, long long n, const SweepCodes& tcode, int ntau,
                              unsigned long long* hist, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 1216) blocks = 1216;  // 8 per SM
  lamp_sweep_hist_kernel<<<(unsigned)blocks, 256, 0, st>>>(rec, n, tcode, ntau, hist);
  return cudaGetLastError();
}

}  // namespace lamp
