// lamp_qkv.cu -- the QKV projection upstream of the attention, with the
// attention's key/value cache written by its epilogue.
//
// y = x W^T for x [T tokens, hidden] and W [(Hq + 2 Hkv) d, hidden] (both
// BF16, K-major), FP32 accumulation in TMEM, y rounded once to BF16 and
// split by columns into q [B, N, Hq, d], k and v [B, N, Hkv, d].  For the
// key columns the epilogue also writes the E4M3 copy of k, the per-chunk
// and per-row norms of that copy (as atomic maxima over each 64-key tile),
// and for the value columns the fp16 copy of v: the same K/V cache the
// attention's pre-pass (lamp_prep.cu) writes; for the query columns it
// writes the E4M3 copy of q and its row and chunk norms, which the fused
// kernel otherwise derives in its CTAs.  The attention call that follows
// runs with kv_prepared = 1 and q_prepared = 1, without a pre-pass.
//
// Tiles of 256 tokens x 256 columns (two heads at d = 128), the column
// tiles of a token tile one after the other, over a persistent grid of CTA
// pairs (clusters of two, one CTA per SM).  The pair computes a tile with
// cta_group::2 MMAs: each CTA holds 128 token rows of x and 128 rows of W
// per K block, so each SM streams half of the W tile it would need alone
// (32 KB per 64-element K block instead of 48).  In each CTA a TMA producer
// warp fills a ring of 6 stages (x 16 KB, W 16 KB, 128-byte swizzle) and
// signals the first CTA's barrier; one thread of the first CTA issues four
// 256 x 256 x 16 kind::f16 MMAs per block into one of two 256-column TMEM
// accumulators (each CTA's TMEM holds its 128 rows; a tile's epilogue
// overlaps the next tile's main loop), and four epilogue warps per CTA read
// them back, one token row per thread.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lamp_common.cuh"
#include "lamp_qkv.cuh"

namespace lamp {

constexpr int kQBM = 128, kQBN = 256, kQBK = 64, kQST = 6;  // kQBM: token rows per CTA
constexpr int kQA = kQBM * kQBK * 2;            // x stage: 16 KB
constexpr int kQB = (kQBN / 2) * kQBK * 2;      // W stage (this CTA's half): 16 KB
constexpr int kQStage = kQA + kQB;
constexpr int kQBar = kQST * kQStage;           // barriers after the stages
constexpr int kQSmem = kQBar + 256 + 1024;      // + barriers, TMEM slot, alignment slack
constexpr int kQThreads = 192;                  // producer, MMA, four epilogue warps

// ---- the CTA-pair forms (cta_group::2) this kernel alone uses
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// TMA load into this CTA's shared memory; completion counted on `bar`, a
// barrier of either CTA of the pair (shared::cluster address)
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(0), "r"(0), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the barrier at shared-memory offset `bar` in both CTAs of the
// pair once the MMAs this thread issued are done
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait of the projection kernel: gives up after timeout_ns (status
// word set to LAMP_ERR_TIMEOUT, 4) or when another thread of the grid gave up.
// Barriers that the other CTA of the pair (or its copies and MMAs) signals
// are waited on with cluster-scope acquire.
__device__ __forceinline__ bool qkv_wait(uint32_t bar, uint32_t parity, const QkvParams& p) {
  for (int i = 0; i < 64; ++i)
    if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (*(volatile unsigned int*)p.abort) return false;
    if (globaltimer_ns() - t0 > p.timeout_ns) break;
    if (mbar_try_wait_cluster(bar, parity)) return true;
    __nanosleep(64);
  }
  atomicExch(p.abort, 1u);
  if (p.counters) atomicExch(&p.counters[9], 4ull);
  return false;
}

// Largest float over the lanes that share `slot` (all lanes when they
// agree, the common case), then one atomic maximum per slot.  The values
// are non-negative, so their bit patterns order like the values.
__device__ __forceinline__ void qkv_atomic_max(float* base, long long slot, float v, bool live) {
  const long long s0 = __shfl_sync(0xffffffffu, slot, 0);
  const bool all_live = __all_sync(0xffffffffu, live);
  if (__all_sync(0xffffffffu, slot == s0) && all_live) {
    const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(v));
    if ((threadIdx.x & 31) == 0) atomicMax((int*)(base + s0), (int)m);
  } else if (live) {
    atomicMax((int*)(base + slot), __float_as_int(v));
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kQThreads, 1)
    lamp_qkv_kernel(const __grid_constant__ QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the same offset in both CTAs: the pair's MMAs address both with one descriptor
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  // barriers: full / empty per stage, and per accumulator: full (MMA ->
  // epilogue) and empty (epilogue -> MMA); the first CTA's full and
  // accumulator-empty barriers serve the pair
  const uint32_t full = sbase + kQBar, empty = full + 8 * kQST, accf = empty + 8 * kQST, acce = accf + 16;
  uint32_t* tslot = (uint32_t*)(smem + kQBar + 8 * (2 * kQST + 4));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: issues the pair's MMAs
  // Persistent: pair c takes tiles c, c + pairs, ...  Tile id -> (token
  // tile, column tile) with the column tiles of a token tile consecutive,
  // so the tiles in flight share a few x tiles and all of W, which stay in L2.
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  const int ntn = (p.ncols + kQBN - 1) / kQBN;
  const int ntiles = ((p.T + 2 * kQBM - 1) / (2 * kQBM)) * ntn;
  const int nkb = p.hidden / kQBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQST; ++s) {
      mbar_init(full + 8 * s, 1);   // first CTA: its producer's arrival; both CTAs' bytes
      mbar_init(empty + 8 * s, 1);  // the pair's MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf + 8 * a, 1);  // the pair's MMA commit
      mbar_init(acce + 8 * a, 8);  // first CTA: one lane of each epilogue warp of both CTAs
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tslot), 2 * kQBN);  // two 256-column accumulators
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *(volatile uint32_t*)tslot;

  if (warp == 0) {
    // ---- TMA producer: this CTA's x rows and W half of each K block
    if (lane == 0) {
      prefetch_tmap(&p.tmX);
      prefetch_tmap(&p.tmW);
      int it = 0;  // K blocks issued so far (over all tiles)
      bool ok = true;
      for (int tile = pair; tile < ntiles && ok; tile += npairs) {
        const int m0 = (tile / ntn) * (2 * kQBM) + (int)rank * kQBM;
        const int n0 = (tile % ntn) * kQBN + (int)rank * (kQBN / 2);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kQST, u = it / kQST;
          if (u > 0 && !qkv_wait(empty + 8 * s, (u - 1) & 1, p)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * kQStage;
          const uint32_t fb = map_to_rank(full + 8 * s, 0);
          if (rank == 0) mbar_expect_tx(full + 8 * s, 2 * kQStage);  // both CTAs' bytes
          tma_load_4d_pair(st, &p.tmX, fb, kb * kQBK, m0);
          tma_load_4d_pair(st + kQA, &p.tmW, fb, kb * kQBK, n0);
        }
      }
      // after a failure, let the copies in flight land before the CTA exits
      if (rank == 0) {
        for (int i = (it > kQST ? it - kQST : 0); i < it; ++i) {
          const int s = i % kQST, u = i / kQST;
          for (int n = 0; n < 100000 && !mbar_try_wait_cluster(full + 8 * s, u & 1); ++n) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer (first CTA): D[256 x 256] (+)= X[256 x 64] . W[256 x 64]^T
    // per block, tile lt of this pair into accumulator lt & 1
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc(1, 1, 0, 2 * kQBM, kQBN);
      bool ok = true;
      int it = 0, lt = 0;
      for (int tile = pair; tile < ntiles && ok; tile += npairs, ++lt) {
        const int a = lt & 1;
        // both CTAs' epilogues have read this accumulator's previous tile
        if (lt >= 2 && !qkv_wait(acce + 8 * a, ((lt >> 1) - 1) & 1, p)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(a * kQBN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kQST, u = it / kQST;
          if (!qkv_wait(full + 8 * s, u & 1, p)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * kQStage;
#pragma unroll
          for (int kk = 0; kk < kQBK / 16; ++kk) {
            const uint64_t ad = make_sdesc(st + kk * 32, 16, 1024, kLayoutSW128);
            const uint64_t bd = make_sdesc(st + kQA + kk * 32, 16, 1024, kLayoutSW128);
            mma_f16_pair(acc, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_pair(empty + 8 * s);
        }
        mma_commit_pair(accf + 8 * a);  // also after a failure: the epilogues must not wait forever
      }
      // the accumulators are released below only once the last MMAs are done
      if (lt > 0) {
        const int a = (lt - 1) & 1;
        for (int n = 0; n < 1000000 && !mbar_try_wait_cluster(accf + 8 * a, ((lt - 1) >> 1) & 1); ++n) {
        }
      }
    }
  } else {
    // ---- epilogue: one token row per thread, this CTA's 128 rows of the tile
    const int quad = warp & 3;  // TMEM lanes 32 quad .. (warp w reads lanes of w % 4)
    const int r = quad * 32 + lane;
    const int D = p.D, CH = D / 32, TT = (p.N + kBN - 1) / kBN;
    bool ok = true;
    int lt = 0;
    for (int tile = pair; tile < ntiles && ok; tile += npairs, ++lt) {
      const int a = lt & 1;
      const int m0 = (tile / ntn) * (2 * kQBM) + (int)rank * kQBM, n0 = (tile % ntn) * kQBN;
      const int t = m0 + r;
      const bool live_row = t < p.T;
      const int b = live_row ? t / p.N : 0, n = live_row ? t - b * p.N : 0;
      ok = qkv_wait(accf + 8 * a, (lt >> 1) & 1, p);
      ok = __all_sync(0xffffffffu, ok);  // warp-uniform: TMEM loads and shuffles below
      if (!ok) break;
      tc_fence_after();
      float ssum = 0.0f;  // sum of squares of the E4M3 query or key row of the current head
#pragma unroll 1
      for (int c0 = 0; c0 < kQBN; c0 += 32) {
        uint32_t acc[32];
        tmem_ld32(tmem + (uint32_t)(a * kQBN) + ((uint32_t)(quad * 32) << 16) + c0, acc);
        tmem_wait_ld();
        if (c0 + 32 == kQBN) {  // the accumulator is read: the MMA thread may reuse it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_to_rank(acce + 8 * a, 0));
        }
        const int col = n0 + c0;
        if (col >= p.ncols) continue;  // warp-uniform
        const int head = col / D, e = col - head * D;
        // round once to BF16 (RNE): the projection's output values
        uint32_t hb[16];
        float vals[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1]));
          memcpy(&hb[i], &h2, 4);
          vals[2 * i] = __low2float(h2);
          vals[2 * i + 1] = __high2float(h2);
        }
        if (head < p.Hq) {
          // E4M3 copy and its norms: one writer per element (upper bounds:
          // the float sums of squares rounded up, as the pre-pass takes them)
          const size_t qrow = ((size_t)b * p.Hq + head) * p.N + n;  // row of the [B, Hq, N, D] copy
          uint32_t c8[8];
          float ss = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint16_t c = cvt_e4m3x2(vals[2 * i + 1], vals[2 * i]);
            const uint32_t hv = e4m3x2_to_f16x2(c);
            __half2 h2;
            memcpy(&h2, &hv, 4);
            const float a0 = __low2float(h2), a1 = __high2float(h2);
            ss = fmaf(a0, a0, fmaf(a1, a1, ss));
            if (i & 1) c8[i >> 1] |= (uint32_t)c << 16; else c8[i >> 1] = c;
          }
          ssum += ss;
          if (live_row) {
            uint4* dst = reinterpret_cast<uint4*>(p.q + (((size_t)b * p.N + n) * p.Hq + head) * D + e);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
            uint4* d8 = reinterpret_cast<uint4*>(p.q8 + qrow * D + e);
            d8[0] = make_uint4(c8[0], c8[1], c8[2], c8[3]);
            d8[1] = make_uint4(c8[4], c8[5], c8[6], c8[7]);
            p.nqc[qrow * CH + e / 32] = sqrtf(ss) * (1.0f + 0x1p-16f);
            if (e + 32 == D) p.nq[qrow] = sqrtf(ssum) * (1.0f + 0x1p-16f);
          }
          if (e + 32 == D) ssum = 0.0f;
        } else if (head < p.Hq + p.Hkv) {
          const int g = head - p.Hq;
          const size_t krow = ((size_t)b * p.Hkv + g) * p.N + n;  // row of the [B, Hkv, N, D] copies
          uint32_t c8[8];
          float ss = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint16_t c = cvt_e4m3x2(vals[2 * i + 1], vals[2 * i]);
            const uint32_t hv = e4m3x2_to_f16x2(c);
            __half2 h2;
            memcpy(&h2, &hv, 4);
            const float a0 = __low2float(h2), a1 = __high2float(h2);
            ss = fmaf(a0, a0, fmaf(a1, a1, ss));
            if (i & 1) c8[i >> 1] |= (uint32_t)c << 16; else c8[i >> 1] = c;
          }
          if (live_row) {
            uint4* dst = reinterpret_cast<uint4*>(p.k + (((size_t)b * p.N + n) * p.Hkv + g) * D + e);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
            uint4* d8 = reinterpret_cast<uint4*>(p.k8 + krow * D + e);
            d8[0] = make_uint4(c8[0], c8[1], c8[2], c8[3]);
            d8[1] = make_uint4(c8[4], c8[5], c8[6], c8[7]);
          }
          // upper bounds of the norms: the float sums of squares rounded up
          const long long ktile = ((long long)b * p.Hkv + g) * TT + n / kBN;
          qkv_atomic_max(p.nkc, ktile * CH + e / 32, sqrtf(ss) * (1.0f + 0x1p-16f) + 0x1p-6f, live_row);
          ssum += ss;
          if (e + 32 == D) {  // the head's last chunk: the whole row
            qkv_atomic_max(p.nk, ktile, sqrtf(ssum) * (1.0f + 0x1p-16f), live_row);
            ssum = 0.0f;
          }
        } else {
          const int g = head - p.Hq - p.Hkv;
          if (live_row) {
            uint4* dst = reinterpret_cast<uint4*>(p.v + (((size_t)b * p.N + n) * p.Hkv + g) * D + e);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
            uint32_t h16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) h16[i] = cvt_f16x2_sat(vals[2 * i + 1], vals[2 * i]);
            uint4* d16 = reinterpret_cast<uint4*>(p.v16 + (((size_t)b * p.Hkv + g) * p.N + n) * D + e);
#pragma unroll
            for (int i = 0; i < 4; ++i) d16[i] = make_uint4(h16[4 * i], h16[4 * i + 1], h16[4 * i + 2], h16[4 * i + 3]);
          }
        }
      }
    }
  }
  // neither CTA leaves (or frees TMEM) while the pair's MMAs, copies or
  // arrivals may still touch its shared memory or TMEM
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 2 * kQBN);
  }
}

cudaError_t launch_qkv(const QkvParams& p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(lamp_qkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)((p.T + 2 * kQBM - 1) / (2 * kQBM)) * ((p.ncols + kQBN - 1) / kQBN);
  if (tiles == 0) return cudaSuccess;
  // persistent: as many CTA pairs as can be resident at once (one CTA per
  // SM; a pair sits in one GPC), tiles strided over them
  static int resident[64];
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int pairs = (dev >= 0 && dev < 64) ? resident[dev] : 0;
  if (pairs <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024);
    cfg.blockDim = dim3(kQThreads);
    cfg.dynamicSmemBytes = kQSmem;
    e = cudaOccupancyMaxActiveClusters(&pairs, (void*)lamp_qkv_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (pairs <= 0) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) resident[dev] = pairs;
  }
  const dim3 grid((unsigned)(2 * (tiles < pairs ? tiles : pairs)));
  lamp_qkv_kernel<<<grid, kQThreads, kQSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace lamp
