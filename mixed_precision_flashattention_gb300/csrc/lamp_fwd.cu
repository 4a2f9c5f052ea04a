// lamp_fwd.cu -- fused LampAttention forward kernel for sm_103a.
//
// One CTA computes 128 query rows of one (batch, query head) against the
// visible 64-key tiles, in ascending key order (the running maximum of the
// method is defined over that order).  Warp roles:
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t).  Per step:
//              8-bit logits S8 (with an exactness guard), running max,
//              x8 / P8 = fl8(exp(x8)), two-stage detector, sub-block flags,
//              mask byte + histogram, FP16 P (P8, or P16 for flagged rows),
//              O rescale in TMEM.
//   warp 4     TMA producer: Q8/Q16 once, then K8/K16/V16 per step into a
//              ring of stages.
//   warp 5     TMEM owner and MMA issuer: S = Q8 K8^T (kind::f8f6f4),
//              S16 = Q16 K16^T (kind::f16, only when some sub-block of the
//              step is flagged), O += P V16 (kind::f16, V MN-major, plus a
//              block of ones so that column d of O accumulates l = sum P).
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

template <int D>
struct Cfg {
  static constexpr int NS = (D == 256) ? 1 : 2;             // K/V stages
  static constexpr int Q8_ROWB = D;                          // bytes per Q8/K8 row
  static constexpr int F8_SWZ_ROW = (D == 64) ? 64 : 128;    // swizzle row width
  static constexpr int Q8_BYTES = kBM * D;
  static constexpr int Q16_BYTES = kBM * D * 2;
  static constexpr int K8_BYTES = kBN * D;
  static constexpr int K16_BYTES = kBN * D * 2;
  static constexpr int V_REGIONS = D / 64 + 1;              // + block of ones
  static constexpr int V_BYTES = V_REGIONS * kBN * 128;
  static constexpr int STAGE_BYTES = K8_BYTES + K16_BYTES + V_BYTES;
  static constexpr int P_BYTES = kBM * kBN * 2;
  static constexpr int OFF_Q8 = 0;
  static constexpr int OFF_Q16 = OFF_Q8 + Q8_BYTES;
  static constexpr int OFF_ST = OFF_Q16 + Q16_BYTES;
  static constexpr int OFF_P = OFF_ST + NS * STAGE_BYTES;
  static constexpr int OFF_MISC = OFF_P + P_BYTES;
  static constexpr int MISC_BYTES = 3072;
  // + alignment slack; at least 116 KB so that one CTA owns an SM (and all
  // of its TMEM)
  static constexpr int SMEM_USED = OFF_MISC + MISC_BYTES + 1024;
  static constexpr int SMEM = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
  // TMEM columns (fp32): O (d values + 16 columns of l), S ring, S16.
  static constexpr int O_COLS = D + 16;
  static constexpr int S_COL0 = ((O_COLS + 31) / 32) * 32;
  static constexpr int S16_COL = S_COL0 + 2 * kBN;
  // two S16 slots let the MMA warp issue the 16-bit recompute of step j+1
  // speculatively (when step j needed one); d = 256 has room for one
  static constexpr int NSLOT16 = (S16_COL + 2 * kBN <= 512) ? 2 : 1;
  static constexpr bool SPEC16 = NSLOT16 == 2 && NS >= 2;
  static constexpr int TMEM_COLS = 512;
  static_assert(S16_COL + NSLOT16 * kBN <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// misc area (byte offsets inside OFF_MISC)
enum : int {
  M_KV_FULL = 0,      // [2] x 8 B
  M_KV_EMPTY = 16,    // [2]
  M_Q_FULL = 32,
  M_S_FULL = 40,      // [2]
  M_S_EMPTY = 56,     // [2]
  M_REC_REQ = 72,     // [2] per step parity: the decision of step j is published
  M_S16_FULL = 88,    // [2] per S16 slot
  M_S16_EMPTY = 104,  // [2] per S16 slot
  M_P_FULL = 120,
  M_PV_DONE = 128,
  M_DRAIN = 136,
  M_TMEM = 144,       // u32 TMEM base address
  M_ABORT = 148,      // u32 abort flag
  M_REC = 152,        // u32 [2] recompute decision per step parity
  M_SFLAG = 160,      // u32 [2][4] per-warp strip bits
  M_XCH = 256,        // f32 [2][128] per-row values exchanged between the two column halves
  M_EXP8 = 1280,      // u8 [256] exp8 table: code of fl8(exp(x)) per code of x
  M_XB = 1536,        // u32 [2][128] per-row bits exchanged between the two column halves
};

struct Ctx {
  uint32_t misc;                 // shared address of the misc area
  volatile uint32_t* abort;      // CTA abort flag (shared memory)
  volatile unsigned int* gabort; // grid abort word (global memory)
  unsigned long long timeout_ns;
  unsigned long long* counters;
};

constexpr unsigned long long kDrainNs = 200000000ull;  // 0.2 s for in-flight copies

// Bounded wait: gives up after cx.timeout_ns, or as soon as this CTA or any
// other CTA has given up; on expiry it raises both abort flags and writes
// LAMP_ERR_TIMEOUT into the status counter.  The first probe is inline; the
// spinning part is out of line and takes its state by value.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                           volatile unsigned int* gabort, unsigned long long timeout_ns,
                                           unsigned long long* counters) {
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;  // suspended, not spinning
    if (*abort) return false;
    if (*gabort) { *abort = 1u; return false; }
    if (globaltimer_ns() - t0 > timeout_ns) break;
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

// Wait used only to let this CTA's own copies and MMAs land before exit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kDrainNs) return;
}

// Warp-uniform variant: every lane waits; true only if all lanes succeeded.
__device__ __forceinline__ bool wait_bar_warp(const Ctx& cx, uint32_t bar, uint32_t parity) {
  const bool okl = wait_bar(cx, bar, parity);
  return __all_sync(0xffffffffu, okl);
}

__device__ __forceinline__ __half2 as_half2(uint32_t u) {
  __half2 r;
  memcpy(&r, &u, 4);
  return r;
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

// Key-tile range [j_lo, j_hi) of the CTA with first row q0.
__device__ __forceinline__ void tile_range(const FwdParams& p, int q0, int& j_lo, int& j_hi) {
  int last = imin(q0 + kBM - 1, p.N - 1);
  if (p.mask_kind == 0) { j_lo = 0; j_hi = p.T; return; }
  j_hi = last / kBN + 1;
  j_lo = (p.mask_kind == 2) ? imax(0, q0 - p.window + 1) / kBN : 0;
}

// Exact A * 2^18 of (row r, key c): integer dot product of the E4M3
// operands in shared memory, split across the warp (every lane gets the sum).
template <int D>
__device__ long long exact_dot(const uint8_t* sQ8, const uint8_t* sK8, int r, int c, int lane) {
  long long acc = 0;
  for (int t = lane; t < D; t += 32) {
    uint32_t qa = sQ8[swz_offset(r, t, kBM, Cfg<D>::F8_SWZ_ROW == 64 ? 64 : D)];
    uint32_t kb = sK8[swz_offset(c, t, kBN, Cfg<D>::F8_SWZ_ROW == 64 ? 64 : D)];
    acc += (long long)e4m3_to_int512(qa) * (long long)e4m3_to_int512(kb);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) lamp_fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // align by pointer arithmetic on the __shared__ array so that every access
  // through `smem` stays a shared-memory access
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint8_t* sQ8 = smem + C::OFF_Q8;
  uint8_t* sP = smem + C::OFF_P;
  uint8_t* misc = smem + C::OFF_MISC;
  const uint32_t mb = sbase + C::OFF_MISC;
  auto bar = [&](int off) { return mb + (uint32_t)off; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh_count = p.B * p.Hq;
  const int qb = p.nqb - 1 - (int)(blockIdx.x / bh_count);  // longest rows first
  const int bh = blockIdx.x % bh_count;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int g = h / (p.Hq / p.Hkv);
  const int q0 = qb * kBM;
  int j_lo, j_hi;
  tile_range(p, q0, j_lo, j_hi);
  const int nsteps = j_hi - j_lo;

  Ctx cx;
  cx.misc = mb;
  cx.abort = (volatile uint32_t*)(misc + M_ABORT);
  cx.gabort = p.gabort;
  cx.timeout_ns = p.timeout_ns;
  cx.counters = p.counters;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(M_KV_FULL + 8 * s), 1);
      mbar_init(bar(M_KV_EMPTY + 8 * s), 1);
      mbar_init(bar(M_S_FULL + 8 * s), 1);
      mbar_init(bar(M_S_EMPTY + 8 * s), kSoftmaxThreads);
      mbar_init(bar(M_REC_REQ + 8 * s), 1);
    }
    mbar_init(bar(M_Q_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(M_S16_FULL + 8 * s), 1);
      mbar_init(bar(M_S16_EMPTY + 8 * s), kSoftmaxThreads);
    }
    mbar_init(bar(M_P_FULL), kSoftmaxThreads);
    mbar_init(bar(M_PV_DONE), 1);
    mbar_init(bar(M_DRAIN), 1);
    *(volatile uint32_t*)(misc + M_ABORT) = 0u;
    fence_mbar_init();
  }
  if (warp == 9) tmem_alloc(bar(M_TMEM), C::TMEM_COLS);
  // the block of ones that turns column d.. of O into the running sum l
  if (threadIdx.x < kSoftmaxThreads) {
    const uint32_t one2 = 0x3C003C00u;  // two fp16 1.0
    for (int s = 0; s < C::NS; ++s) {
      uint32_t* ones = (uint32_t*)(smem + C::OFF_ST + s * C::STAGE_BYTES + C::K8_BYTES +
                                   C::K16_BYTES + (C::V_REGIONS - 1) * kBN * 128);
      for (int i = threadIdx.x; i < kBN * 128 / 4; i += kSoftmaxThreads) ones[i] = one2;
    }
    misc[M_EXP8 + threadIdx.x] = p.exp8[threadIdx.x];
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *(volatile uint32_t*)(misc + M_TMEM);

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nsteps > 0) {
      prefetch_tmap(&p.tmQ8);
      prefetch_tmap(&p.tmQ16);
      prefetch_tmap(&p.tmK8);
      prefetch_tmap(&p.tmK16);
      prefetch_tmap(&p.tmV);
      mbar_expect_tx(bar(M_Q_FULL), C::Q8_BYTES + C::Q16_BYTES);
      for (int c = 0; c < D / (C::F8_SWZ_ROW); ++c)
        tma_load_4d(sbase + C::OFF_Q8 + c * kBM * 128, &p.tmQ8, bar(M_Q_FULL),
                    c * C::F8_SWZ_ROW, q0, h, b);
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(sbase + C::OFF_Q16 + c * kBM * 128, &p.tmQ16, bar(M_Q_FULL), c * 64, q0, h,
                    b);
      int uses0 = 0, uses1 = 0;
      for (int jj = 0; jj < nsteps && !*cx.abort; ++jj) {
        const int s = jj % C::NS, u = jj / C::NS;
        if (u >= 1 && !wait_bar(cx, bar(M_KV_EMPTY + 8 * s), (u - 1) & 1)) break;
        const int key0 = (j_lo + jj) * kBN;
        const uint32_t st = sbase + C::OFF_ST + s * C::STAGE_BYTES;
        mbar_expect_tx(bar(M_KV_FULL + 8 * s), C::K8_BYTES + C::K16_BYTES + (D / 64) * kBN * 128);
        for (int c = 0; c < D / (C::F8_SWZ_ROW); ++c)
          tma_load_4d(st + c * kBN * 128, &p.tmK8, bar(M_KV_FULL + 8 * s), c * C::F8_SWZ_ROW,
                      key0, g, b);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(st + C::K8_BYTES + c * kBN * 128, &p.tmK16, bar(M_KV_FULL + 8 * s), c * 64,
                      key0, g, b);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(st + C::K8_BYTES + C::K16_BYTES + c * kBN * 128, &p.tmV,
                      bar(M_KV_FULL + 8 * s), c * 64, key0, g, b);
        if (s) uses1 = u + 1; else uses0 = u + 1;
      }
      if (*cx.abort) {  // let every load in flight land before the CTA exits
        if (uses0 > 0) drain_wait(bar(M_KV_FULL), (uses0 - 1) & 1);
        if (uses1 > 0) drain_wait(bar(M_KV_FULL + 8), (uses1 - 1) & 1);
        drain_wait(bar(M_Q_FULL), 0);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nsteps > 0) {
      auto issue_qk8 = [&](int jj) {
        const uint32_t st = sbase + C::OFF_ST + (jj % C::NS) * C::STAGE_BYTES;
        Mma<D>::qk8(tmem + C::S_COL0 + (jj & 1) * kBN, sbase + C::OFF_Q8, st);
        mma_commit(bar(M_S_FULL + 8 * (jj & 1)));
      };
      auto load_and_qk8 = [&](int jj) -> bool {
        const int s = jj % C::NS, u = jj / C::NS;
        if (!wait_bar(cx, bar(M_KV_FULL + 8 * s), u & 1)) return false;
        if (jj >= 2 && !wait_bar(cx, bar(M_S_EMPTY + 8 * (jj & 1)), ((jj - 2) >> 1) & 1))
          return false;
        tc_fence_after();
        issue_qk8(jj);
        return true;
      };
      // 16-bit recompute bookkeeping per S16 slot (slot of step j = j % NSLOT16):
      // a QK16 of step j is issued speculatively when step j-1 needed one
      // (step 0: always), or on demand once step j's decision arrives.
      // per slot: was its last QK16 read (wanted), reads (s16_empty arrivals) expected
      bool wanted0 = false, wanted1 = false;
      int reads0 = 0, reads1 = 0;
      auto issue_qk16 = [&](int j) -> bool {
        const int sl = j % C::NSLOT16;
        const bool wl = sl ? wanted1 : wanted0;
        const int rd = sl ? reads1 : reads0;
        if (wl && !wait_bar(cx, bar(M_S16_EMPTY + 8 * sl), (rd - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t stj = sbase + C::OFF_ST + (j % C::NS) * C::STAGE_BYTES;
        Mma<D>::qk16(tmem + C::S16_COL + sl * kBN, sbase + C::OFF_Q16, stj + C::K8_BYTES);
        mma_commit(bar(M_S16_FULL + 8 * sl));
        if (sl) wanted1 = false; else wanted0 = false;
        return true;
      };
      bool ok = wait_bar(cx, bar(M_Q_FULL), 0);
      bool spec = false;  // QK16 of the current step already issued
      if (ok) ok = load_and_qk8(0);
      if (ok && C::SPEC16) {
        ok = issue_qk16(0);
        spec = true;
      }
      for (int jj = 0; ok && jj < nsteps; ++jj) {
        if (C::NS == 1 && jj > 0) ok = load_and_qk8(jj);
        if (ok && C::NS >= 2 && jj + 1 < nsteps) ok = load_and_qk8(jj + 1);
        if (!ok) break;
        if (!wait_bar(cx, bar(M_REC_REQ + 8 * (jj & 1)), (jj >> 1) & 1)) break;
        const bool want = *(volatile uint32_t*)(misc + M_REC + 4 * (jj & 1)) != 0u;
        const int s = jj % C::NS;
        const uint32_t st = sbase + C::OFF_ST + s * C::STAGE_BYTES;
        if (want && !spec && !issue_qk16(jj)) break;
        if (want) {
          if (jj % C::NSLOT16) { wanted1 = true; ++reads1; } else { wanted0 = true; ++reads0; }
        }
        spec = C::SPEC16 && want && jj + 1 < nsteps;
        if (spec && !issue_qk16(jj + 1)) break;
        // O += P V16 (and l += P 1)
        if (!wait_bar(cx, bar(M_P_FULL), jj & 1)) break;
        tc_fence_after();
        Mma<D>::pv(tmem, sbase + C::OFF_P, st + C::K8_BYTES + C::K16_BYTES, jj > 0);
        mma_commit(bar(M_PV_DONE));
        mma_commit(bar(M_KV_EMPTY + 8 * s));
      }
      // make sure no MMA is still writing TMEM before it is released
      mma_commit(bar(M_DRAIN));
      drain_wait(bar(M_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Two threads per query row: warps w and w+4 own the same 32 rows
    // (TMEM lanes 32*(w%4)..), w < 4 the key columns 0..31 of each step,
    // w >= 4 the columns 32..63.  Every softmax thread runs every step up to
    // the CTA-wide reduction of `fail`, so named barriers never miss a
    // participant; waits are warp-uniform so the .sync.aligned TMEM accesses
    // stay converged.
    const int rw = warp & 3;              // row group
    const int hf = warp >> 2;             // column half
    const int t = rw * 32 + lane;         // query row within the CTA == TMEM lane
    const int col0 = hf * kNC;
    const int R = q0 + t;
    const uint32_t lane_base = tmem + ((uint32_t)(rw * 32) << 16);
    const uint32_t pair_bar = 2 + rw;     // named barrier of warps rw and rw + 4
    float* xch = (float*)(misc + M_XCH);
    uint32_t* xb = (uint32_t*)(misc + M_XB);
    const uint8_t* tab = misc + M_EXP8;
    int lo, hi;
    row_range(p, R, lo, hi);
    float m = -INFINITY;
    float nq = 0.0f;
    if (R < p.N) nq = p.nq[((size_t)b * p.Hq + h) * p.N + R];
    unsigned long long c_tiles = 0, c_h0 = 0, c_h1 = 0, c_h2 = 0, c_strips = 0, c_st1 = 0,
                       c_fl = 0, c_sat = 0, c_fix = 0, c_rec = 0;
    const int qtile = 2 * qb + (rw >> 1);  // 64-row query tile of this warp
    int commits16_0 = 0, commits16_1 = 0;  // QK16 results committed per S16 slot (mirrors the MMA warp)
    bool spec16 = C::SPEC16;    // QK16 of the current step issued speculatively
    unsigned long long c_waste = 0;
    const float sig = p.sigma_f;
    const float2 sig2 = make_float2(sig, sig);
    const float T = p.tau_abs;
    const uint32_t dcode = p.delta_code;
    bool fail = !(nsteps > 0 && wait_bar_warp(cx, bar(M_Q_FULL), 0));
    bool done_ok = false;

    for (int jj = 0; jj < nsteps; ++jj) {
      const int jt = j_lo + jj;
      const int k0 = jt * kBN;
      const int clo = imax(k0, lo), chi = imin(k0 + kBN - 1, hi);
      const bool rowvis = clo <= chi;
      // visible columns of this thread's half (bit c = key k0 + col0 + c)
      uint32_t vm = 0u;
      {
        const int a = imax(clo - (k0 + col0), 0), z = imin(chi - (k0 + col0), kNC - 1);
        if (rowvis && a <= z) vm = (z == 31 ? 0xFFFFFFFFu : ((1u << (z + 1)) - 1u)) & ~((1u << a) - 1u);
      }
      const bool all_full = __all_sync(0xffffffffu, vm == 0xFFFFFFFFu);
      const float nk = p.nkmax[((size_t)b * p.Hkv + g) * p.T + jt];
      const float G = p.guard * sig * nq * nk;

      // ---- S = Q8 K8^T (fp32, TMEM) -> 8-bit logits
      uint32_t a32[kNC];
      if (!fail) fail = !wait_bar_warp(cx, bar(M_S_FULL + 8 * (jj & 1)), (jj >> 1) & 1);
      if (!fail) {
        tc_fence_after();
        tmem_ld32(lane_base + C::S_COL0 + (jj & 1) * kBN + col0, a32);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(M_S_EMPTY + 8 * (jj & 1)));
      } else {
#pragma unroll
        for (int c = 0; c < kNC; ++c) a32[c] = 0u;
      }
      // S8 = fl8(A sigma) is certain unless y = A_tc sigma lies within G of an
      // E4M3 rounding boundary (the two roundings of y -+ G then differ).  Of
      // those, only logits that can change m, P8, the detector or the
      // saturation count need the exact value: m (the running max before
      // this tile) is exact and <= the new max, and a logit whose largest
      // rounding is <= m - 6.75 rounds x8 to <= -7 (P8 = 0, below any
      // delta > 0) and is not the maximum.  With delta = 0 all count.
      uint32_t s8h[kNC / 2];  // S8 pairs as f16x2 (exact)
      uint32_t unc = 0u;      // logits to re-derive exactly
      {
        const float2 gm = make_float2(-G, -G), gp = make_float2(G, G);
        const float thr = m - 6.75f;
#pragma unroll
        for (int g4 = 0; g4 < kNC / 8; ++g4) {  // 4 pairs at a time, one branch
          float2 yh[4];
          uint32_t d4 = 0u, d16[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int i = 4 * g4 + k;
            const float2 av = make_float2(__uint_as_float(a32[2 * i]), __uint_as_float(a32[2 * i + 1]));
            const float2 yl = __ffma2_rn(av, sig2, gm);
            yh[k] = __ffma2_rn(av, sig2, gp);
            const uint16_t cl = cvt_e4m3x2(yl.y, yl.x), ch = cvt_e4m3x2(yh[k].y, yh[k].x);
            s8h[i] = e4m3x2_to_f16x2(cl);
            d16[k] = (uint32_t)(cl ^ ch);
            d4 |= d16[k];
          }
          if (d4 != 0u) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i = 4 * g4 + k;
              const float h0 = yh[k].x, h1 = yh[k].y;
              const bool r0 = dcode == 0u || h0 + 0.125f * fabsf(h0) + 0x1p-8f > thr || fabsf(h0) >= 400.0f;
              const bool r1 = dcode == 0u || h1 + 0.125f * fabsf(h1) + 0x1p-8f > thr || fabsf(h1) >= 400.0f;
              if ((d16[k] & 0xFFu) && r0) unc |= 1u << (2 * i);
              if ((d16[k] >> 8) && r1) unc |= 1u << (2 * i + 1);
            }
          }
        }
      }
      unc &= vm;
      if (fail) unc = 0u;
      if (__any_sync(0xffffffffu, unc != 0u)) {
        const uint8_t* sK8 = smem + C::OFF_ST + (jj % C::NS) * C::STAGE_BYTES;
        for (;;) {
          const unsigned who = __ballot_sync(0xffffffffu, unc != 0u);
          if (!who) break;
          const int src = __ffs(who) - 1;
          const int cb = __shfl_sync(0xffffffffu, unc ? (__ffs(unc) - 1) : 0, src);
          const long long acc = exact_dot<D>(sQ8, sK8, rw * 32 + src, col0 + cb, lane);
          if (lane == src) {
            const float v = e4m3_rne_from_double((double)acc * 0x1p-18 * p.sigma_d);
            const uint32_t hv = (uint32_t)__half_as_ushort(__float2half_rn(v));  // exact
#pragma unroll
            for (int i = 0; i < kNC / 2; ++i)
              if (i == (cb >> 1))
                s8h[i] = (cb & 1) ? ((s8h[i] & 0x0000FFFFu) | (hv << 16)) : ((s8h[i] & 0xFFFF0000u) | hv);
            unc &= unc - 1u;
          }
          if (lane == 0) ++c_fix;
        }
      }
      // hidden keys take -inf: they are never the max and x8 saturates to -448 (P8 = 0)
      if (!all_full) {
#pragma unroll
        for (int i = 0; i < kNC / 2; ++i) {
          const uint32_t keep = (((vm >> (2 * i)) & 1u) ? 0x0000FFFFu : 0u) | (((vm >> (2 * i + 1)) & 1u) ? 0xFFFF0000u : 0u);
          s8h[i] = (s8h[i] & keep) | (0xFC00FC00u & ~keep);
        }
      }

      // ---- tile max over both halves, running max
      float m_tile;
      {
        __half2 mx = as_half2(s8h[0]);
#pragma unroll
        for (int i = 1; i < kNC / 2; ++i) mx = __hmax2(mx, as_half2(s8h[i]));
        const float mine = fmaxf(__low2float(mx), __high2float(mx));
        xch[hf * kBM + t] = mine;
        bar_sync(pair_bar, 64);
        m_tile = fmaxf(mine, xch[(1 - hf) * kBM + t]);
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
      const bool maybe_neg = rowvis && st1 && !flg && T > 0.0f &&
                             tab[cvt_e4m3x2(0.0f, -T - m_new) & 0xFFu] >= dcode;
      if (__any_sync(0xffffffffu, maybe_neg)) {  // same outcome in both halves
        uint32_t mine = 0u;
        if (maybe_neg) {
          const __half2 mh = __float2half2_rn(m_new);
#pragma unroll
          for (int i = 0; i < kNC / 2; ++i) {
            const __half2 sv = as_half2(s8h[i]);
            const uint32_t x8 = cvt_e4m3x2_f16x2(__hsub2(sv, mh));
            if (((vm >> (2 * i)) & 1u) && __low2float(sv) <= -T && tab[x8 & 0xFFu] >= dcode) mine = 1u;
            if (((vm >> (2 * i + 1)) & 1u) && __high2float(sv) <= -T && tab[x8 >> 8] >= dcode) mine = 1u;
          }
        }
        xb[hf * kBM + t] = mine;
        bar_sync(pair_bar, 64);
        if (maybe_neg) flg = (mine | xb[(1 - hf) * kBM + t]) != 0u;
      }
      if (rowvis && sig * nq * nk * (1.0f + p.guard) >= 432.0f) {
#pragma unroll
        for (int i = 0; i < kNC / 2; ++i) {
          const __half2 sv = as_half2(s8h[i]);
          c_sat += (fabsf(__low2float(sv)) == 448.0f) + (fabsf(__high2float(sv)) == 448.0f);
        }
      }

      // ---- sub-block bits: lanes 0-15 and 16-31 of a warp are two sub-blocks
      const unsigned bv = __ballot_sync(0xffffffffu, rowvis);
      const unsigned b1 = __ballot_sync(0xffffffffu, st1);
      const unsigned bf = __ballot_sync(0xffffffffu, flg);
      uint32_t sv[2], s1[2], sf[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        sv[hh] = ((bv >> (16 * hh)) & 0xFFFFu) != 0u;
        s1[hh] = ((b1 >> (16 * hh)) & 0xFFFFu) != 0u;
        sf[hh] = ((bf >> (16 * hh)) & 0xFFFFu) != 0u;
        if (p.force == 1) sf[hh] = sv[hh];
        if (p.force == 2) sf[hh] = 0u;
      }
      const bool my_flag = sf[lane >> 4] != 0u;
      if (lane == 0 && hf == 0)
        *(volatile uint32_t*)(misc + M_SFLAG + 16 * (jj & 1) + 4 * rw) =
            sf[0] | (sf[1] << 1) | (s1[0] << 2) | (s1[1] << 3) | (sv[0] << 4) | (sv[1] << 5);
      const bool any = bar_red_or(1, kSoftmaxThreads, my_flag);
      if (bar_red_or(1, kSoftmaxThreads, fail)) break;  // uniform exit

      if (lane == 0 && hf == 0 && (rw & 1) == 0) {
        // lane 0 of warps 0 and 2 owns the 64-row query tile of row groups (rw, rw+1)
        const uint32_t w0 = *(volatile uint32_t*)(misc + M_SFLAG + 16 * (jj & 1) + 4 * rw);
        const uint32_t w1 = *(volatile uint32_t*)(misc + M_SFLAG + 16 * (jj & 1) + 4 * (rw + 1));
        const uint32_t fl4 = (w0 & 3u) | ((w1 & 3u) << 2);
        const uint32_t st4 = ((w0 >> 2) & 3u) | (((w1 >> 2) & 3u) << 2);
        const uint32_t vs4 = ((w0 >> 4) & 3u) | (((w1 >> 4) & 3u) << 2);
        if (vs4) {
          const int nf = __popc(fl4);
          ++c_tiles;
          if (nf == 0) ++c_h0; else if (nf == 1) ++c_h1; else ++c_h2;
          c_strips += __popc(vs4);
          c_st1 += __popc(st4 & vs4);
          c_fl += nf;
          if (p.mask && qtile < p.T)
            p.mask[(((size_t)b * p.Hq + h) * p.T + qtile) * p.T + jt] = (uint8_t)(fl4 | (st4 << 4));
        }
      }
      if (threadIdx.x == 0) {
        *(volatile uint32_t*)(misc + M_REC + 4 * (jj & 1)) = any ? 1u : 0u;
        mbar_arrive(bar(M_REC_REQ + 8 * (jj & 1)));
        if (any) ++c_rec;
      }

      // ---- x8 = fl8(S8 - m) (fp16 difference, then one E4M3 rounding: equal
      // to the single rounding for E4M3 operands), P8 from the exp8 table;
      // rows of flagged sub-blocks take P16 below instead
      uint32_t pw[kNC / 2];
      if (rowvis && !my_flag) {
        const __half2 mh = __float2half2_rn(m_new);
#pragma unroll
        for (int i = 0; i < kNC / 2; ++i) {
          const __half2 xh = __hsub2(as_half2(s8h[i]), mh);
          const uint32_t x8 = cvt_e4m3x2_f16x2(xh);
          const uint32_t pc = (uint32_t)tab[x8 & 0xFFu] | ((uint32_t)tab[x8 >> 8] << 8);
          pw[i] = e4m3x2_to_f16x2((uint16_t)pc);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kNC / 2; ++i) pw[i] = 0u;
      }

      // ---- 16-bit recompute for the rows of flagged sub-blocks
      {
        const int sl = jj % C::NSLOT16;
        if (spec16 || any) { if (sl) ++commits16_1; else ++commits16_0; }
        const int ncommit = sl ? commits16_1 : commits16_0;
        if (spec16 && !any) ++c_waste;
        spec16 = C::SPEC16 && any && jj + 1 < nsteps;
        if (any && !fail) fail = !wait_bar_warp(cx, bar(M_S16_FULL + 8 * sl), (ncommit - 1) & 1);
        if (any && !fail) {
          tc_fence_after();
          uint32_t r16[kNC];
          tmem_ld32(lane_base + C::S16_COL + sl * kBN + col0, r16);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(M_S16_EMPTY + 8 * sl));
          if (my_flag && rowvis) {
            const float sl2 = sig * kLog2e, ml = m_new * kLog2e;
#pragma unroll
            for (int i = 0; i < kNC / 2; ++i) {
              const float e0 = ex2_approx(fmaf(__uint_as_float(r16[2 * i]), sl2, -ml));
              const float e1 = ex2_approx(fmaf(__uint_as_float(r16[2 * i + 1]), sl2, -ml));
              pw[i] = cvt_f16x2_sat(e1, e0);
            }
            if (!all_full) {
#pragma unroll
              for (int i = 0; i < kNC / 2; ++i) {
                if (!((vm >> (2 * i)) & 1u)) pw[i] &= 0xFFFF0000u;
                if (!((vm >> (2 * i + 1)) & 1u)) pw[i] &= 0x0000FFFFu;
              }
            }
          }
        }
      }

      // ---- the previous P.V must be done before P and O are touched
      if (jj > 0 && !fail) fail = !wait_bar_warp(cx, bar(M_PV_DONE), (jj - 1) & 1);
      if (!fail) {
        tc_fence_after();
        const float alpha =
            (m_new == m) ? 1.0f : (m == -INFINITY ? 0.0f : ex2_approx((m - m_new) * kLog2e));
        if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          constexpr int NCH = C::O_COLS / 16, NCH0 = (NCH + 1) / 2;
          const int cb = hf ? NCH0 : 0, ce = hf ? NCH : NCH0;
#pragma unroll 1
          for (int ch = cb; ch < ce; ++ch) {
            uint32_t o[16];
            tmem_ld16(lane_base + ch * 16, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const float2 v = __fmul2_rn(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                          make_float2(alpha, alpha));
              o[i] = __float_as_uint(v.x);
              o[i + 1] = __float_as_uint(v.y);
            }
            tmem_st16(lane_base + ch * 16, o);
          }
          tmem_wait_st();
        }
        // P row half -> shared memory (K-major, 128-byte swizzle)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v4 = make_uint4(pw[4 * k], pw[4 * k + 1], pw[4 * k + 2], pw[4 * k + 3]);
          *reinterpret_cast<uint4*>(sP + swz_offset(t, (4 * hf + k) * 16, kBM, 128)) = v4;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(M_P_FULL));
      }
      m = m_new;
      if (jj == nsteps - 1) done_ok = !fail;
    }

    // ---- epilogue: out = O / l, LSE = m + ln l (each half writes d/2 columns)
    if (done_ok) done_ok = wait_bar_warp(cx, bar(M_PV_DONE), (nsteps - 1) & 1);
    if (done_ok) {
      tc_fence_after();
      uint32_t lw[16];
      tmem_ld16(lane_base + D, lw);
      tmem_wait_ld();
      const float l = __uint_as_float(lw[0]);
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const bool live = R < p.N;
      if (live && hf == 0 && p.lse)
        p.lse[((size_t)b * p.Hq + h) * p.N + R] = l > 0.0f ? m + logf(l) : -INFINITY;
      char* orow = (char*)p.out + ((size_t)b * p.o_stride[0] + (size_t)R * p.o_stride[1] +
                                   (size_t)h * p.o_stride[2]) * (p.out_f32 ? 4 : 2);
#pragma unroll 1
      for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 16) {
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
      if (lane == 0 && hf == 0 && (rw & 1) == 0 && c_tiles) {
        atomicAdd(&p.counters[0], c_tiles);
        atomicAdd(&p.counters[1], c_h0);
        atomicAdd(&p.counters[2], c_h1);
        atomicAdd(&p.counters[3], c_h2);
        atomicAdd(&p.counters[4], c_strips);
        atomicAdd(&p.counters[5], c_st1);
        atomicAdd(&p.counters[6], c_fl);
      }
      for (int o = 16; o > 0; o >>= 1) c_sat += __shfl_xor_sync(0xffffffffu, c_sat, o);
      if (lane == 0 && c_sat) atomicAdd(&p.counters[7], c_sat);
      if (lane == 0 && c_fix) atomicAdd(&p.counters[8], c_fix);
      if (threadIdx.x == 0 && c_rec) atomicAdd(&p.counters[10], c_rec);
      if (threadIdx.x == 0 && c_waste) atomicAdd(&p.counters[11], c_waste);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, C::TMEM_COLS);
}

}  // namespace lamp

// ---------------------------------------------------------------- launcher
namespace lamp {

template <int D>
static cudaError_t launch_fwd_d(const FwdParams& p, cudaStream_t st) {
  const int smem = Cfg<D>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(lamp_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.nqb * (unsigned)p.B * (unsigned)p.Hq;
  if (grid == 0) return cudaSuccess;
  lamp_fwd_kernel<D><<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams& p, int d, cudaStream_t st) {
  switch (d) {
    case 64: return launch_fwd_d<64>(p, st);
    case 128: return launch_fwd_d<128>(p, st);
    case 256: return launch_fwd_d<256>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lamp
