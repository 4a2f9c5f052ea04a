// lamp_selftest.cu -- device checks of the tcgen05 building blocks used by
// the fused kernel: the same Mma<D> issue sequences, swizzled shared-memory
// layouts and TMEM read-back, run on caller-given data.
//   which 0: S = A8 . B8^T, A8 [128 x D], B8 [64 x D] E4M3 codes, out [128 x 64]
//   which 1: S = A . B^T,  A [128 x D], B [64 x D] BF16,          out [128 x 64]
//   which 2: O = P . V,    P [128 x 64], V [64 x D] FP16,         out [128 x D]
// and the scalar helpers of the fused kernel: which 3 the exact 8-bit
// re-derivation, which 4 the 8-bit exponential P8 = fl8(e^x), which 5 and 6
// the 8-bit difference x8 = fl8(S8 - m) (5: through the f16 difference the
// P8 path uses, 6: through the fp32 difference the detector uses).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/lamp_attn.h"
#include "lamp_common.cuh"

namespace lamp {

template <int D>
__global__ void __launch_bounds__(128, 1)
    lamp_selftest_kernel(int which, const uint8_t* a, const uint8_t* b, float* out, unsigned int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;                 // up to 128 x 512 B
  uint8_t* sB = smem + 128 * 512;     // up to 64 x 512 B
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t taddr;
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t barp = smem_u32(&bar);
  if (tid == 0) {
    mbar_init(barp, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(&taddr), 512);
  constexpr int F8_ROW = (D == 64) ? 64 : D;
  if (which == 0) {
    for (int i = tid; i < 128 * D; i += 128) sA[swz_offset(i / D, i % D, 128, F8_ROW)] = a[i];
    for (int i = tid; i < 64 * D; i += 128) sB[swz_offset(i / D, i % D, 64, F8_ROW)] = b[i];
  } else if (which == 1) {
    const uint16_t* a16 = (const uint16_t*)a;
    const uint16_t* b16 = (const uint16_t*)b;
    for (int i = tid; i < 128 * D; i += 128)
      *(uint16_t*)(sA + swz_offset(i / D, 2 * (i % D), 128, 2 * D)) = a16[i];
    for (int i = tid; i < 64 * D; i += 128)
      *(uint16_t*)(sB + swz_offset(i / D, 2 * (i % D), 64, 2 * D)) = b16[i];
  } else {
    const uint16_t* p16 = (const uint16_t*)a;
    const uint16_t* v16 = (const uint16_t*)b;
    for (int i = tid; i < 128 * 64; i += 128)
      *(uint16_t*)(sA + swz_offset(i / 64, 2 * (i % 64), 128, 128)) = p16[i];
    for (int i = tid; i < 64 * D; i += 128) {
      const int key = i / D, d = i % D;
      *(uint16_t*)(sB + (d / 64) * 64 * 128 + swz_offset(key, 2 * (d % 64), 64, 128)) = v16[i];
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = taddr;
  if (tid == 0) {
    if (which == 0) Mma<D>::qk8(tmem, smem_u32(sA), smem_u32(sB));
    else if (which == 1) Mma<D>::qk16(tmem, smem_u32(sA), smem_u32(sB));
    else Mma<D>::pv(tmem, smem_u32(sA), smem_u32(sB), false);
    mma_commit(barp);
  }
  bool ok = false;
  for (uint32_t i = 0; i < (1u << 24) && !ok; ++i) ok = mbar_try_wait(barp, 0);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (tid & 31) == 0) atomicExch(status, 4u);
  tc_fence_after();
  const int ncols = which == 2 ? D : 64;
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  for (int c0 = 0; c0 < ncols; c0 += 16) {
    uint32_t r[16];
    tmem_ld16(lane_base + c0, r);
    tmem_wait_ld();
    if (ok)
      for (int i = 0; i < 16; ++i) out[(size_t)tid * ncols + c0 + i] = __uint_as_float(r[i]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void lamp_round_selftest_kernel(const long long* acc, const double* sigma, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t h = e4m3_f16_of_product(acc[i], ldexp(*sigma, -18));
  out[i] = __half2float(__ushort_as_half((unsigned short)h));
}

// out[i] = fl8(e^x) for the E4M3 code codes[i] (x <= 0), as the fused kernel
// computes it (exp8_f16x2)
__global__ void lamp_exp8_selftest_kernel(const uint8_t* codes, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t h = exp8_f16x2((uint32_t)codes[i] * 0x0101u);
  out[i] = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// out[i] = x8 = fl8(S8 - m) for the E4M3 codes s8[i] of S8 and m8[i] of m,
// as the fused kernel computes it: via_f16 -- the f16x2 difference of the
// two values rounded once more to E4M3 (the P8 path); otherwise the fp32
// difference (exact for E4M3 operands) rounded to E4M3 (the detector)
__global__ void lamp_x8_selftest_kernel(const uint8_t* s8, const uint8_t* m8, float* out, int n, bool via_f16) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t sh = e4m3x2_to_f16x2((uint16_t)((uint32_t)s8[i] * 0x0101u));
  const uint32_t mh = e4m3x2_to_f16x2((uint16_t)((uint32_t)m8[i] * 0x0101u));
  __half2 sv, mv;
  memcpy(&sv, &sh, 4);
  memcpy(&mv, &mh, 4);
  uint32_t code;
  if (via_f16) {
    // the kernel holds m as a float and converts it with __float2half2_rn
    const __half2 mk = __float2half2_rn(__low2float(mv));
    code = cvt_e4m3x2_f16x2(__hsub2(sv, mk)) & 0xFFu;
  } else {
    code = cvt_e4m3x2(0.0f, __low2float(sv) - __low2float(mv)) & 0xFFu;
  }
  const uint32_t h = e4m3x2_to_f16x2((uint16_t)code);
  out[i] = __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

template <int D>
static cudaError_t run_selftest(int which, const void* a, const void* b, float* out, unsigned int* status,
                                cudaStream_t st) {
  const int smem = 128 * 512 + 64 * 512 + 64 * 128 + 1024;
  cudaError_t e = cudaFuncSetAttribute(lamp_selftest_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  lamp_selftest_kernel<D><<<1, 128, smem, st>>>(which, (const uint8_t*)a, (const uint8_t*)b, out, status);
  return cudaGetLastError();
}

}  // namespace lamp

extern "C" int lamp_selftest(int which, const void* a, const void* b, float* out, int d, void* stream) {
  if (!a || !b || !out || which < 0 || which > 6) return LAMP_ERR_INVALID_ARG;
  if (which >= 3 ? (d < 1 || d > 65536) : (d != 64 && d != 128 && d != 256)) return LAMP_ERR_UNSUPPORTED;
  int dev = 0, maj = 0, min = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LAMP_ERR_CUDA;
  cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev);
  if (maj != 10 || min != 3) return LAMP_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned int* status = nullptr;
  if (cudaMallocAsync((void**)&status, sizeof(unsigned int), st) != cudaSuccess) return LAMP_ERR_CUDA;
  cudaMemsetAsync(status, 0, sizeof(unsigned int), st);
  cudaError_t e = cudaSuccess;
  if (which == 3) {
    lamp::lamp_round_selftest_kernel<<<(d + 255) / 256, 256, 0, st>>>((const long long*)a, (const double*)b, out, d);
    e = cudaGetLastError();
  } else if (which == 4) {
    lamp::lamp_exp8_selftest_kernel<<<(d + 255) / 256, 256, 0, st>>>((const uint8_t*)a, out, d);
    e = cudaGetLastError();
  } else if (which == 5 || which == 6) {
    lamp::lamp_x8_selftest_kernel<<<(d + 255) / 256, 256, 0, st>>>((const uint8_t*)a, (const uint8_t*)b, out, d,
                                                                   which == 5);
    e = cudaGetLastError();
  } else {
    e = d == 64    ? lamp::run_selftest<64>(which, a, b, out, status, st)
                  : d == 128 ? lamp::run_selftest<128>(which, a, b, out, status, st)
                             : lamp::run_selftest<256>(which, a, b, out, status, st);
  }
  unsigned int hs = 0;
  if (e == cudaSuccess) e = cudaMemcpyAsync(&hs, status, sizeof(hs), cudaMemcpyDeviceToHost, st);
  cudaFreeAsync(status, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return LAMP_ERR_CUDA;
  return hs ? (int)hs : LAMP_OK;
}
