// lamp_prep.cu -- input pre-pass of the LampAttention forward pass.
//
// Writes, into the workspace, the operand formats the fused kernel reads
// with TMA: Q8 = fl8(q) and K8 = fl8(k) (E4M3, RNE, saturating, taken from
// the input values directly), V16 = fp16(v) (RNE, saturating), BF16 copies
// of fp32 q and k, the row norms ||Q8_r|| and the per-64-key-tile maximum
// of ||K8_c|| (the bound that sizes the exactness guard of the 8-bit
// logits).  HBM-bound: one warp per row, each lane a contiguous slice.
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

template <int D, bool F32>
__global__ void __launch_bounds__(256) lamp_prep_kernel(const PrepParams p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const long long nQ = (long long)p.B * p.N * p.Hq, nK = (long long)p.B * p.N * p.Hkv;
  float x[E];
  if (row < nQ) {
    const int h = (int)(row % p.Hq);
    const long long bn = row / p.Hq;
    const int n = (int)(bn % p.N), b = (int)(bn / p.N);
    load_row<D, F32>(p.q, b * p.qs[0] + n * p.qs[1] + h * p.qs[2], lane, x);
    const size_t o = (((size_t)b * p.Hq + h) * p.N + n) * D + lane * E;
    float ss = warp_sum(store_e4m3<E>(p.q8 + o, x));
    if (F32) {
#pragma unroll
      for (int i = 0; i < E; i += 2)
        *reinterpret_cast<__nv_bfloat162*>((__nv_bfloat16*)p.q16 + o + i) = __floats2bfloat162_rn(x[i], x[i + 1]);
    }
    // upper bound of the norm: the float sum of squares is rounded up
    if (lane == 0) p.nq[((size_t)b * p.Hq + h) * p.N + n] = sqrtf(ss) * (1.0f + 0x1p-16f);
  } else if (row < nQ + nK) {
    const long long r = row - nQ;
    const int g = (int)(r % p.Hkv);
    const long long bn = r / p.Hkv;
    const int n = (int)(bn % p.N), b = (int)(bn / p.N);
    load_row<D, F32>(p.k, b * p.ks[0] + n * p.ks[1] + g * p.ks[2], lane, x);
    const size_t o = (((size_t)b * p.Hkv + g) * p.N + n) * D + lane * E;
    float ss = warp_sum(store_e4m3<E>(p.k8 + o, x));
    if (F32) {
#pragma unroll
      for (int i = 0; i < E; i += 2)
        *reinterpret_cast<__nv_bfloat162*>((__nv_bfloat16*)p.k16 + o + i) = __floats2bfloat162_rn(x[i], x[i + 1]);
    }
    if (lane == 0) {
      const float nk = sqrtf(ss) * (1.0f + 0x1p-16f);
      // non-negative floats order like their bit patterns
      atomicMax((int*)&p.nkmax[((size_t)b * p.Hkv + g) * p.T + n / kBN], __float_as_int(nk));
    }
  } else if (p.v && row < nQ + 2 * nK) {  // (no V rows in the sweep pass: the grid's last block may overhang)
    const long long r = row - nQ - nK;
    const int g = (int)(r % p.Hkv);
    const long long bn = r / p.Hkv;
    const int n = (int)(bn % p.N), b = (int)(bn / p.N);
    load_row<D, F32>(p.v, b * p.vs[0] + n * p.vs[1] + g * p.vs[2], lane, x);
    const size_t o = (((size_t)b * p.Hkv + g) * p.N + n) * D + lane * E;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const uint32_t hh = cvt_f16x2_sat(x[i + 1], x[i]);
      *reinterpret_cast<uint32_t*>((__half*)p.v16 + o + i) = hh;
    }
  }
}

template <int D>
static cudaError_t launch_prep_d(const PrepParams& p, cudaStream_t st) {
  const long long rows = (long long)p.B * p.N * (p.Hq + (p.v ? 2LL : 1LL) * p.Hkv);  // no V rows without v
  const long long blocks = (rows + 7) / 8;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  if (p.in_f32)
    lamp_prep_kernel<D, true><<<(unsigned)blocks, 256, 0, st>>>(p);
  else
    lamp_prep_kernel<D, false><<<(unsigned)blocks, 256, 0, st>>>(p);
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
