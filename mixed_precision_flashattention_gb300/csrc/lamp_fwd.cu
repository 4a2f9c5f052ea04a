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
  static constexpr int MISC_BYTES = 1024;
  // + alignment slack; at least 116 KB so that one CTA owns an SM (and all
  // of its TMEM)
  static constexpr int SMEM_USED = OFF_MISC + MISC_BYTES + 1024;
  static constexpr int SMEM = SMEM_USED > 116 * 1024 ? SMEM_USED : 116 * 1024;
  // TMEM columns (fp32): O (d values + 16 columns of l), S ring, S16.
  static constexpr int O_COLS = D + 16;
  static constexpr int S_COL0 = ((O_COLS + 31) / 32) * 32;
  static constexpr int S16_COL = S_COL0 + 2 * kBN;
  static constexpr int TMEM_COLS = 512;
  static_assert(S16_COL + kBN <= TMEM_COLS, "TMEM budget");
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
  M_S16_FULL = 88,
  M_S16_EMPTY = 96,
  M_P_FULL = 104,
  M_PV_DONE = 112,
  M_DRAIN = 120,
  M_TMEM = 128,       // u32 TMEM base address
  M_ABORT = 132,      // u32 abort flag
  M_REC = 136,        // u32 [2] recompute decision per step parity
  M_SFLAG = 144,      // u32 [2][4] per-warp strip bits
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
// LAMP_ERR_TIMEOUT into the status counter.
__device__ __noinline__ bool wait_bar(const Ctx& cx, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0u) {
      if (*cx.abort) return false;
      if (*cx.gabort) { *cx.abort = 1u; return false; }
      if (globaltimer_ns() - t0 > cx.timeout_ns) break;
    }
  }
  *cx.abort = 1u;
  atomicExch((unsigned int*)cx.gabort, 1u);
  if (cx.counters) atomicExch(&cx.counters[9], 4ull);  // LAMP_ERR_TIMEOUT
  return false;
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
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
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
    mbar_init(bar(M_S16_FULL), 1);
    mbar_init(bar(M_S16_EMPTY), kSoftmaxThreads);
    mbar_init(bar(M_P_FULL), kSoftmaxThreads);
    mbar_init(bar(M_PV_DONE), 1);
    mbar_init(bar(M_DRAIN), 1);
    *(volatile uint32_t*)(misc + M_ABORT) = 0u;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(bar(M_TMEM), C::TMEM_COLS);
  // the block of ones that turns column d.. of O into the running sum l
  if (threadIdx.x < kSoftmaxThreads) {
    const uint32_t one2 = 0x3C003C00u;  // two fp16 1.0
    for (int s = 0; s < C::NS; ++s) {
      uint32_t* ones = (uint32_t*)(smem + C::OFF_ST + s * C::STAGE_BYTES + C::K8_BYTES +
                                   C::K16_BYTES + (C::V_REGIONS - 1) * kBN * 128);
      for (int i = threadIdx.x; i < kBN * 128 / 4; i += kSoftmaxThreads) ones[i] = one2;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *(volatile uint32_t*)(misc + M_TMEM);

  if (warp == 4) {
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
      int uses[2] = {0, 0};
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
        uses[s] = u + 1;
      }
      if (*cx.abort) {  // let every load in flight land before the CTA exits
        for (int s = 0; s < C::NS; ++s)
          if (uses[s] > 0) drain_wait(bar(M_KV_FULL + 8 * s), (uses[s] - 1) & 1);
        drain_wait(bar(M_Q_FULL), 0);
      }
    }
  } else if (warp == 5) {
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
      bool ok = wait_bar(cx, bar(M_Q_FULL), 0);
      int nrec = 0;
      for (int jj = 0; ok && jj < nsteps; ++jj) {
        if (C::NS == 1 || jj == 0) ok = load_and_qk8(jj);
        if (ok && C::NS >= 2 && jj + 1 < nsteps) ok = load_and_qk8(jj + 1);
        if (!ok) break;
        // 16-bit recompute of this step, if the softmax warps asked for it
        if (!wait_bar(cx, bar(M_REC_REQ + 8 * (jj & 1)), (jj >> 1) & 1)) break;
        const uint32_t want = *(volatile uint32_t*)(misc + M_REC + 4 * (jj & 1));
        const int s = jj % C::NS;
        const uint32_t st = sbase + C::OFF_ST + s * C::STAGE_BYTES;
        if (want) {
          if (nrec >= 1 && !wait_bar(cx, bar(M_S16_EMPTY), (nrec - 1) & 1)) break;
          tc_fence_after();
          Mma<D>::qk16(tmem + C::S16_COL, sbase + C::OFF_Q16, st + C::K8_BYTES);
          mma_commit(bar(M_S16_FULL));
          ++nrec;
        }
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
    // Every softmax thread runs every step up to the CTA-wide reduction of
    // `fail`, so the named barriers never miss a participant; waits are
    // warp-uniform so the .sync.aligned TMEM accesses stay converged.
    const int t = threadIdx.x;  // query row within the CTA == TMEM lane
    const int R = q0 + t;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    int lo, hi;
    row_range(p, R, lo, hi);
    float m = -INFINITY;
    float nq = 0.0f;
    if (R < p.N) nq = p.nq[((size_t)b * p.Hq + h) * p.N + R];
    unsigned long long c_tiles = 0, c_h0 = 0, c_h1 = 0, c_h2 = 0, c_strips = 0, c_st1 = 0,
                       c_fl = 0, c_sat = 0, c_fix = 0, c_rec = 0;
    const int qtile = 2 * qb + (warp >> 1);  // 64-row query tile of this warp
    int nrec = 0;
    const float sig = p.sigma_f;
    bool fail = !(nsteps > 0 && wait_bar_warp(cx, bar(M_Q_FULL), 0));
    bool done_ok = false;

    for (int jj = 0; jj < nsteps; ++jj) {
      const int jt = j_lo + jj;
      const int k0 = jt * kBN;
      const int clo = imax(k0, lo), chi = imin(k0 + kBN - 1, hi);
      const bool rowvis = clo <= chi;
      const float nk = p.nkmax[((size_t)b * p.Hkv + g) * p.T + jt];
      const float G = p.guard * sig * nq * nk;
      unsigned long long vis = 0ull;
      if (rowvis) {
        const int a = clo - k0, z = chi - k0;  // visible columns a..z of the tile
        vis = (z == 63 ? ~0ull : ((1ull << (z + 1)) - 1ull)) & ~((1ull << a) - 1ull);
      }

      float s8[kBN];
      if (!fail) fail = !wait_bar_warp(cx, bar(M_S_FULL + 8 * (jj & 1)), (jj >> 1) & 1);
      if (!fail) {
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(lane_base + C::S_COL0 + (jj & 1) * kBN, r0);
        tmem_ld32(lane_base + C::S_COL0 + (jj & 1) * kBN + 32, r1);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          s8[c] = __uint_as_float(r0[c]);
          s8[c + 32] = __uint_as_float(r1[c]);
        }
        tc_fence_before();
        mbar_arrive(bar(M_S_EMPTY + 8 * (jj & 1)));
      } else {
#pragma unroll
        for (int c = 0; c < kBN; ++c) s8[c] = 0.0f;
      }

      // S8 = fl8(A * sigma) is certain unless y = A_tc * sigma lies within G
      // of an E4M3 rounding boundary; those logits are re-derived exactly.
      unsigned long long fix = 0ull;
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float y0 = s8[c] * sig, y1 = s8[c + 1] * sig;
        const uint16_t clo2 = cvt_e4m3x2(y1 - G, y0 - G);
        const uint16_t chi2 = cvt_e4m3x2(y1 + G, y0 + G);
        const uint32_t dif = (uint32_t)(clo2 ^ chi2);
        fix |= (unsigned long long)((dif & 0xFFu) != 0u) << c;
        fix |= (unsigned long long)((dif >> 8) != 0u) << (c + 1);
        const __half2 hv = as_half2(e4m3x2_to_f16x2(clo2));
        s8[c] = __low2float(hv);
        s8[c + 1] = __high2float(hv);
      }
      fix &= vis;
      if (fail) fix = 0ull;
      if (__any_sync(0xffffffffu, fix != 0ull)) {
        // Only logits that can change m, P8, the detector bits or the
        // saturation count need the exact value.  mL <= exact running max;
        // if the largest value the logit can round to is <= mL - 6.75, it
        // rounds x8 to <= -7 either way (P8 = 0, below any delta > 0) and is
        // not the maximum.  With the first stage disabled every uncertain
        // logit can move a flag, so all are re-derived.
        float mL = m;
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if ((vis >> c) & 1ull) mL = fmaxf(mL, s8[c]);
        if (p.delta_code != 0u) {
          const float twoG = 2.0f * G;
#pragma unroll
          for (int c = 0; c < kBN; ++c) {
            if ((fix >> c) & 1ull) {
              const float v = s8[c];
              // y - G rounds to v, so fl8(y + G) <= v + 2G + half-spacings <= up
              const float up = v + twoG + 0.25f * (fabsf(v) + twoG) + 0x1p-8f;
              if (up - mL <= -6.75f && fabsf(v) < 416.0f) fix &= ~(1ull << c);
            }
          }
        }
      }
      if (__any_sync(0xffffffffu, fix != 0ull)) {
        const uint8_t* sK8 = smem + C::OFF_ST + (jj % C::NS) * C::STAGE_BYTES;
        unsigned long long pend = fix;
        for (;;) {
          const unsigned who = __ballot_sync(0xffffffffu, pend != 0ull);
          if (!who) break;
          const int src = __ffs(who) - 1;
          const int cc = __shfl_sync(0xffffffffu, pend ? (__ffsll((long long)pend) - 1) : 0, src);
          const long long acc = exact_dot<D>(sQ8, sK8, warp * 32 + src, cc, lane);
          if (lane == src) {
            const float v = e4m3_rne_from_double((double)acc * 0x1p-18 * p.sigma_d);
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c == cc) s8[c] = v;
            pend &= pend - 1ull;
          }
          if (lane == 0) ++c_fix;
        }
      }

      // tile max and running max over the visible keys
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; ++c)
        if ((vis >> c) & 1ull) tmax = fmaxf(tmax, s8[c]);
      const float m_new = rowvis ? fmaxf(m, tmax) : m;

      // x8 = fl8(S8 - m), P8 = fl8(exp(x8)) kept as FP16, detector bits
      uint32_t pw[kBN / 2];
      bool st1 = false, flg = false;
      if (rowvis && !fail) {
        if (sig * nq * nk * (1.0f + p.guard) >= 432.0f) {
#pragma unroll
          for (int c = 0; c < kBN; ++c)
            if (((vis >> c) & 1ull) && fabsf(s8[c]) == 448.0f) ++c_sat;
        }
#pragma unroll
        for (int c = 0; c < kBN; c += 2) {
          const bool v0 = (vis >> c) & 1ull, v1 = (vis >> (c + 1)) & 1ull;
          const float x0 = v0 ? s8[c] - m_new : -448.0f;
          const float x1 = v1 ? s8[c + 1] - m_new : -448.0f;
          const uint16_t x8 = cvt_e4m3x2(x1, x0);
          const __half2 xh = as_half2(e4m3x2_to_f16x2(x8));
          const float e0 = ex2_approx(__low2float(xh) * kLog2e);
          const float e1 = ex2_approx(__high2float(xh) * kLog2e);
          const uint16_t p8 = cvt_e4m3x2(e1, e0);
          uint32_t ph = e4m3x2_to_f16x2(p8);
          const bool s10 = v0 && (uint32_t)(p8 & 0xFFu) >= p.delta_code;
          const bool s11 = v1 && (uint32_t)(p8 >> 8) >= p.delta_code;
          st1 |= s10 | s11;
          flg |= (s10 && fabsf(s8[c]) >= p.tau_abs) | (s11 && fabsf(s8[c + 1]) >= p.tau_abs);
          if (!v0) ph &= 0xFFFF0000u;
          if (!v1) ph &= 0x0000FFFFu;
          pw[c / 2] = ph;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kBN / 2; ++c) pw[c] = 0u;
      }

      // sub-block bits: lanes 0-15 and 16-31 of a warp are two sub-blocks
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
      if (lane == 0)
        *(volatile uint32_t*)(misc + M_SFLAG + 16 * (jj & 1) + 4 * warp) =
            sf[0] | (sf[1] << 1) | (s1[0] << 2) | (s1[1] << 3) | (sv[0] << 4) | (sv[1] << 5);
      const bool any = bar_red_or(1, kSoftmaxThreads, my_flag);
      if (bar_red_or(1, kSoftmaxThreads, fail)) break;  // uniform exit

      if (lane == 0 && (warp & 1) == 0) {
        // lane 0 of warps 0 and 2 owns the 64-row query tile of (warp, warp+1)
        const uint32_t w0 = *(volatile uint32_t*)(misc + M_SFLAG + 16 * (jj & 1) + 4 * warp);
        const uint32_t w1 = *(volatile uint32_t*)(misc + M_SFLAG + 16 * (jj & 1) + 4 * (warp + 1));
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

      // 16-bit recompute for the rows of flagged sub-blocks
      if (any && !fail) {
        fail = !wait_bar_warp(cx, bar(M_S16_FULL), nrec & 1);
        if (!fail) {
          tc_fence_after();
          uint32_t r0[32], r1[32];
          tmem_ld32(lane_base + C::S16_COL, r0);
          tmem_ld32(lane_base + C::S16_COL + 32, r1);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(M_S16_EMPTY));
          ++nrec;
          if (my_flag && rowvis) {
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
              const float a0 = __uint_as_float(c < 32 ? r0[c] : r1[c - 32]);
              const float a1 = __uint_as_float(c + 1 < 32 ? r0[c + 1] : r1[c + 1 - 32]);
              const float e0 = ex2_approx((a0 * sig - m_new) * kLog2e);
              const float e1 = ex2_approx((a1 * sig - m_new) * kLog2e);
              uint32_t ph = cvt_f16x2_sat(e1, e0);
              if (!((vis >> c) & 1ull)) ph &= 0xFFFF0000u;
              if (!((vis >> (c + 1)) & 1ull)) ph &= 0x0000FFFFu;
              pw[c / 2] = ph;
            }
          }
        }
      }

      // the previous P.V must be done before P and O are touched
      if (jj > 0 && !fail) fail = !wait_bar_warp(cx, bar(M_PV_DONE), (jj - 1) & 1);
      if (!fail) {
        tc_fence_after();
        const float alpha =
            (m_new == m) ? 1.0f : (m == -INFINITY ? 0.0f : ex2_approx((m - m_new) * kLog2e));
        if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c0 = 0; c0 < C::O_COLS; c0 += 16) {
            uint32_t o[16];
            tmem_ld16(lane_base + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(lane_base + c0, o);
          }
          tmem_wait_st();
        }
        // P row -> shared memory (K-major, 128-byte swizzle)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint4 v4 = make_uint4(pw[4 * ch], pw[4 * ch + 1], pw[4 * ch + 2], pw[4 * ch + 3]);
          *reinterpret_cast<uint4*>(sP + swz_offset(t, ch * 16, kBM, 128)) = v4;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(M_P_FULL));
      }
      m = m_new;
      if (jj == nsteps - 1) done_ok = !fail;
    }

    // epilogue: out = O / l, LSE = m + ln l
    if (done_ok) done_ok = wait_bar_warp(cx, bar(M_PV_DONE), (nsteps - 1) & 1);
    if (done_ok) {
      tc_fence_after();
      uint32_t lw[16];
      tmem_ld16(lane_base + D, lw);
      tmem_wait_ld();
      const float l = __uint_as_float(lw[0]);
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const bool live = R < p.N;
      if (live && p.lse) p.lse[((size_t)b * p.Hq + h) * p.N + R] = l > 0.0f ? m + logf(l) : -INFINITY;
      char* orow = (char*)p.out + ((size_t)b * p.o_stride[0] + (size_t)R * p.o_stride[1] +
                                   (size_t)h * p.o_stride[2]) * (p.out_f32 ? 4 : 2);
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
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
      if (lane == 0 && (warp & 1) == 0 && c_tiles) {
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
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, C::TMEM_COLS);
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
