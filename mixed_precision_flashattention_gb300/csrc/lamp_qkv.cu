// lamp_qkv.cu -- the QKV projection upstream of the attention, with the
// attention's key/value cache written by its epilogue.
//
// y = x W^T for x [T tokens, hidden] and W [(Hq + 2 Hkv) d, hidden] (both
// BF16, K-major), FP32 accumulation in TMEM, y rounded once to BF16 and
// split by columns into q [B, N, Hq, d], k and v [B, N, Hkv, d].  For the
// key columns the epilogue also writes the E4M3 copy of k, the per-chunk
// and per-row norms of that copy (as atomic maxima over each 64-key tile),
// and for the value columns the fp16 copy of v: the same K/V cache the
// attention's pre-pass (lamp_prep.cu) writes, so the attention call that
// follows runs with kv_prepared = 1 and no pre-pass.
//
// One CTA per 128-token x 256-column tile (two heads at d = 128): a TMA
// producer warp fills a ring of 4 stages of 64-element K blocks (x 16 KB,
// W 32 KB, 128-byte swizzle), one thread of the MMA warp issues four
// 128 x 256 x 16 kind::f16 MMAs per block into a 256-column TMEM
// accumulator, and four epilogue warps read it back, one token row per
// thread.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lamp_common.cuh"
#include "lamp_qkv.cuh"

namespace lamp {

constexpr int kQBM = 128, kQBN = 256, kQBK = 64, kQST = 4;
constexpr int kQA = kQBM * kQBK * 2;            // x stage: 16 KB
constexpr int kQB = kQBN * kQBK * 2;            // W stage: 32 KB
constexpr int kQStage = kQA + kQB;
constexpr int kQBar = kQST * kQStage;           // barriers after the stages
constexpr int kQSmem = kQBar + 128 + 1024;      // + barriers, TMEM slot, alignment slack
constexpr int kQThreads = 192;                  // producer, MMA, four epilogue warps

// Bounded wait of the projection kernel: gives up after timeout_ns (status
// word set to LAMP_ERR_TIMEOUT, 4) or when another thread of the grid gave up.
__device__ __forceinline__ bool qkv_wait(uint32_t bar, uint32_t parity, const QkvParams& p) {
  if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (;;) {
    if (*(volatile unsigned int*)p.abort) return false;
    if (globaltimer_ns() - t0 > p.timeout_ns) break;
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
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

__global__ void __launch_bounds__(kQThreads, 1) lamp_qkv_kernel(const __grid_constant__ QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full = sbase + kQBar, empty = full + 8 * kQST, accf = empty + 8 * kQST;
  uint32_t* tslot = (uint32_t*)(smem + kQBar + 8 * (2 * kQST + 1));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kQBM, n0 = blockIdx.y * kQBN;
  const int nkb = p.hidden / kQBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQST; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, 1);
    }
    mbar_init(accf, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tslot), kQBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *(volatile uint32_t*)tslot;

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      prefetch_tmap(&p.tmX);
      prefetch_tmap(&p.tmW);
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kQST, u = kb / kQST;
        if (u > 0 && !qkv_wait(empty + 8 * s, (u - 1) & 1, p)) break;
        const uint32_t st = sbase + s * kQStage;
        mbar_expect_tx(full + 8 * s, kQStage);
        tma_load_4d(st, &p.tmX, full + 8 * s, kb * kQBK, m0, 0, 0);
        tma_load_4d(st + kQA, &p.tmW, full + 8 * s, kb * kQBK, n0, 0, 0);
        issued = kb + 1;
      }
      // after a failure, let the copies in flight land before the CTA exits
      for (int kb = (issued > kQST ? issued - kQST : 0); kb < issued; ++kb) {
        const int s = kb % kQST, u = kb / kQST;
        for (int it = 0; it < 100000 && !mbar_try_wait(full + 8 * s, u & 1); ++it) {
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: D[128 x 256] (+)= X[128 x 64] . W[256 x 64]^T per block
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(1, 1, 0, kQBM, kQBN);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % kQST, u = kb / kQST;
        ok = qkv_wait(full + 8 * s, u & 1, p);
        if (!ok) break;
        tc_fence_after();
        const uint32_t st = sbase + s * kQStage;
#pragma unroll
        for (int kk = 0; kk < kQBK / 16; ++kk) {
          const uint64_t ad = make_sdesc(st + kk * 32, 16, 1024, kLayoutSW128);
          const uint64_t bd = make_sdesc(st + kQA + kk * 32, 16, 1024, kLayoutSW128);
          mma_f16(tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(empty + 8 * s);
      }
      mma_commit(accf);  // also after a failure: the epilogue must not wait forever
      // the accumulator is released below only once these MMAs are done
      for (int it = 0; it < 1000000 && !mbar_try_wait(accf, 0); ++it) {
      }
    }
  } else {
    // ---- epilogue: one token row per thread
    const int quad = warp & 3;  // TMEM lanes 32 quad .. (warp w reads lanes of w % 4)
    const int r = quad * 32 + lane;
    const int t = m0 + r;
    const bool live_row = t < p.T;
    const int b = live_row ? t / p.N : 0, n = live_row ? t - b * p.N : 0;
    const int D = p.D, CH = D / 32, TT = (p.N + kBN - 1) / kBN;
    bool ok = qkv_wait(accf, 0, p);
    ok = __all_sync(0xffffffffu, ok);  // warp-uniform: TMEM loads and shuffles below
    if (ok) tc_fence_after();
    float ssum = 0.0f;  // sum of squares of the E4M3 key row of the current head
#pragma unroll 1
    for (int c0 = 0; c0 < kQBN; c0 += 32) {
      uint32_t acc[32];
      if (ok) {
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + c0, acc);
        tmem_wait_ld();
      }
      const int col = n0 + c0;
      if (!ok || col >= p.ncols) continue;  // warp-uniform
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
        if (live_row) {
          uint4* dst = reinterpret_cast<uint4*>(p.q + (((size_t)b * p.N + n) * p.Hq + head) * D + e);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hb[4 * i], hb[4 * i + 1], hb[4 * i + 2], hb[4 * i + 3]);
        }
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
        const long long tile = ((long long)b * p.Hkv + g) * TT + n / kBN;
        qkv_atomic_max(p.nkc, tile * CH + e / 32, sqrtf(ss) * (1.0f + 0x1p-16f) + 0x1p-6f, live_row);
        ssum += ss;
        if (e + 32 == D) {  // the head's last chunk: the whole row
          qkv_atomic_max(p.nk, tile, sqrtf(ssum) * (1.0f + 0x1p-16f), live_row);
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
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kQBN);
  }
}

cudaError_t launch_qkv(const QkvParams& p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(lamp_qkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((p.T + kQBM - 1) / kQBM), (unsigned)((p.ncols + kQBN - 1) / kQBN));
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  lamp_qkv_kernel<<<grid, kQThreads, kQSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace lamp
