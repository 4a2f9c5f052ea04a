// lamp_prep.cu -- input pre-pass of the LampAttention forward pass.
//
// Writes, into the workspace, the operand formats the fused kernel reads
// with TMA: Q8 = fl8(q) and K8 = fl8(k) (E4M3, RNE, saturating, taken from
// the input values directly), V16 = fp16(v) (RNE, saturating), BF16 copies
// of fp32 q and k, the row norms ||Q8_r|| and the per-64-key-tile maximum
// of ||K8_c|| (the bound that sizes the exactness guard of the 8-bit
// logits).  HBM-bound.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lamp_common.cuh"

namespace lamp {


template <int D, bool F32>
__device__ __forceinline__ void load_row(const void* base, long long off, int lane, float (&x)[D / 32]) {
  constexpr int E = D / 32;
  if (F32) {
    const float* p = (const float*)base + off + lane * E;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      float2 f = *reinterpret_cast<const float2*>(p + i);
      x[i] = f.x;
      x[i + 1] = f.y;
    }
  } else {
    const __nv_bfloat16* p = (const __nv_bfloat16*)base + off + lane * E;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(p + i);
      x[i] = __low2float(h2);
      x[i + 1] = __high2float(h2);
    }
  }
}

// E4M3 codes of x (pairs), plus the exact sum of squares of their values.
template <int E>
__device__ __forceinline__ float store_e4m3(uint8_t* dst, const float (&x)[E]) {
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const uint16_t c = cvt_e4m3x2(x[i + 1], x[i]);
    *reinterpret_cast<uint16_t*>(dst + i) = c;
    uint32_t h = e4m3x2_to_f16x2(c);
    __half2 hv;
    memcpy(&hv, &h, 4);
    const float a = __low2float(hv), b = __high2float(hv);
    ss = fmaf(a, a, fmaf(b, b, ss));
  }
  return ss;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 16-byte accesses: a lane holds 8 consecutive elements of a row, D/8
// lanes a row, 256/D rows per warp instruction; each warp has all its rows'
// loads in flight before it converts any of them.  Rows are taken in the
// inputs' (b, n, h) order, so the warps of a block read one contiguous
// stretch of the tensor.
template <int D, bool F32>
__device__ __forceinline__ void load8(const void* base, long long off, float (&x)[8]) {
  if (F32) {
    const float4* p = reinterpret_cast<const float4*>((const float*)base + off);
    const float4 a = p[0], c = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>((const __nv_bfloat16*)base + off);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h2;
      memcpy(&h2, &w[i], 4);
      x[2 * i] = __low2float(h2);
      x[2 * i + 1] = __high2float(h2);
    }
  }
}

// rows per warp of the pre-pass (all loads in flight together; d = 256 rows
// are twice as long)
template <int D>
constexpr int kPrepRowsPerWarp = D <= 128 ? 8 : 2;

// Row index -> (batch, position, head) for `heads` heads, in 32-bit
// arithmetic when the row count allows it (64-bit division is slow).
template <bool W64>
__device__ __forceinline__ void split_row(long long row, int heads, int N, int& b, int& n, int& h) {
  if (W64) {
    h = (int)(row % heads);
    const long long bn = row / heads;
    n = (int)(bn % N);
    b = (int)(bn / N);
  } else {
    const uint32_t r = (uint32_t)row, bn = r / (uint32_t)heads;
    h = (int)(r - bn * (uint32_t)heads);
    const uint32_t bb = bn / (uint32_t)N;
    n = (int)(bn - bb * (uint32_t)N);
    b = (int)bb;
  }
}

template <int D, bool F32, bool W64>
__global__ void __launch_bounds__(256) lamp_prep_kernel(const PrepParams p) {
  constexpr int LPR = D / 8;          // lanes per row
  constexpr int RPI = 32 / LPR;       // rows per warp instruction
  constexpr int RPW = kPrepRowsPerWarp<D>;  // rows per warp
  constexpr int NI = RPW / RPI;       // instructions for the warp's rows
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, col = (lane % LPR) * 8;
  const long long nQ = (long long)p.B * p.N * p.Hq, nK = (long long)p.B * p.N * p.Hkv;
  const long long nrows = nQ + (p.v ? 2 : 1) * nK;
  const long long row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW;
  float x[NI][8];
  long long rows[NI];
  int rb[NI], rn[NI], rh[NI];  // (batch, position, head) of each row
#pragma unroll
  for (int it = 0; it < NI; ++it) {
    const long long row = row0 + it * RPI + sub;
    rows[it] = row;
    rb[it] = rn[it] = rh[it] = 0;
    if (row >= nrows) continue;
    const void* src;
    long long off;
    int b, n, h;
    if (row < nQ) {
      split_row<W64>(row, p.Hq, p.N, b, n, h);
      src = p.q;
      off = b * p.qs[0] + n * p.qs[1] + h * p.qs[2];
    } else {
      const bool isk = row < nQ + nK;
      split_row<W64>(isk ? row - nQ : row - nQ - nK, p.Hkv, p.N, b, n, h);
      const long long* st = isk ? p.ks : p.vs;
      src = isk ? p.k : p.v;
      off = b * st[0] + n * st[1] + h * st[2];
    }
    rb[it] = b; rn[it] = n; rh[it] = h;
    load8<D, F32>(src, off + col, x[it]);
  }
#pragma unroll
  for (int it = 0; it < NI; ++it) {
    const long long row = rows[it];
    const bool live = row < nrows;
    const bool isq = row < nQ, isk = !isq && row < nQ + nK;
    const int hh = rh[it], n = rn[it], b = rb[it];
    float ss = 0.0f;
    if (live && (isq || isk)) {
      const size_t o = (((size_t)b * (isq ? p.Hq : p.Hkv) + hh) * p.N + n) * D + col;
      uint32_t c8[2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint16_t c = cvt_e4m3x2(x[it][2 * i + 1], x[it][2 * i]);
        const uint32_t hv = e4m3x2_to_f16x2(c);
        __half2 h2;
        memcpy(&h2, &hv, 4);
        const float a0 = __low2float(h2), a1 = __high2float(h2);
        ss = fmaf(a0, a0, fmaf(a1, a1, ss));
        if (i & 1) c8[i >> 1] |= (uint32_t)c << 16; else c8[i >> 1] = c;
      }
      *reinterpret_cast<uint2*>((isq ? p.q8 : p.k8) + o) = make_uint2(c8[0], c8[1]);
      if (F32) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 bb = __floats2bfloat162_rn(x[it][2 * i], x[it][2 * i + 1]);
          memcpy(&w[i], &bb, 4);
        }
        *reinterpret_cast<uint4*>((__nv_bfloat16*)(isq ? p.q16 : p.k16) + o) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else if (live) {  // v -> fp16
      const size_t o = (((size_t)b * p.Hkv + hh) * p.N + n) * D + col;
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = cvt_f16x2_sat(x[it][2 * i + 1], x[it][2 * i]);
      *reinterpret_cast<uint4*>((__half*)p.v16 + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    // row norm: sum over the row's lanes (all lanes take part in the shuffles)
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (live && (isq || isk) && (lane % LPR) == 0) {
      // upper bound of the norm: the float sum of squares is rounded up
      const float nrm = sqrtf(ss) * (1.0f + 0x1p-16f);
      if (isq) p.nq[((size_t)b * p.Hq + hh) * p.N + n] = nrm;
      else  // non-negative floats order like their bit patterns
        atomicMax((int*)&p.nkmax[((size_t)b * p.Hkv + hh) * p.T + n / kBN], __float_as_int(nrm));
    }
  }
}

template <int D>
static cudaError_t launch_prep_d(const PrepParams& p, cudaStream_t st) {
  const long long rows = (long long)p.B * p.N * (p.Hq + (p.v ? 2LL : 1LL) * p.Hkv);  // no V rows without v
  const long long per_block = 8LL * kPrepRowsPerWarp<D>;  // 8 warps
  const long long blocks = (rows + per_block - 1) / per_block;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  const bool w64 = rows + 64 >= (1LL << 31);
  if (p.in_f32)
    w64 ? lamp_prep_kernel<D, true, true><<<(unsigned)blocks, 256, 0, st>>>(p)
        : lamp_prep_kernel<D, true, false><<<(unsigned)blocks, 256, 0, st>>>(p);
  else
    w64 ? lamp_prep_kernel<D, false, true><<<(unsigned)blocks, 256, 0, st>>>(p)
        : lamp_prep_kernel<D, false, false><<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PrepParams& p, int d, cudaStream_t st) {
  switch (d) {
    case 64: return launch_prep_d<64>(p, st);
    case 128: return launch_prep_d<128>(p, st);
    case 256: return launch_prep_d<256>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lamp
