// lamp_prep.cu -- input pre-pass of the LampAttention forward pass.
//
// Writes, into the workspace, the operand formats the fused kernel reads
// with TMA: K8 = fl8(k) (E4M3, RNE, saturating, taken from the input values
// directly), V16 = fp16(v) (RNE, saturating), BF16 copies of fp32 q and k,
// the per-64-key-tile maximum of ||K8_c|| (the bound that sizes the
// exactness guard of the 8-bit logits) and -- for fp32 q, and for the tau
// sweep -- Q8 = fl8(q) with the row norms ||Q8_r||.  For bf16 q the fused
// kernel rounds its own Q tile (skip_q).  HBM-bound.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "lamp_common.cuh"

namespace lamp {

// Each warp takes groups of kPrepRows<D> consecutive rows (rows in the
// inputs' (b, n, h) order, so a group is one contiguous stretch of a tensor
// with the usual strides).  A lane holds 8 consecutive elements of a row:
// D/8 lanes a row, 256/D rows per warp instruction.  The grid is persistent
// (as many blocks as fit on the GPU) and each warp keeps the raw loads of
// its next group in flight while it converts and stores the current one.
template <int D>
constexpr int kPrepRows = D <= 128 ? 4 : 2;

// Division of n < 2^31 by a fixed d < 2^31 as (m n) >> s with
// m = ceil(2^(31+l) / d), s = 31 + l, l = ceil(log2 d): the round-up
// multiplier of Granlund and Montgomery, "Division by Invariant Integers
// using Multiplication" (1994), Theorem 4.2 with N = 31.
__device__ __forceinline__ uint32_t div_inv(uint32_t n, uint32_t m, int s) {
  return (uint32_t)(((unsigned long long)m * n) >> s);
}

static void inv_divisor(int d, uint32_t& m, int& s) {
  int l = 0;
  while ((1LL << l) < d) ++l;
  s = 31 + l;
  m = (uint32_t)(((1ULL << s) + (unsigned long long)d - 1) / (unsigned long long)d);
}

// One lane's share of one row: the raw 16 or 32 input bytes, the kind of
// row (0 q, 1 k, 2 v, -1 none), its output row (b, h, n) -> (b H + h) N + n
// and, for k, its entry of the per-key-tile norm maximum.  In the 32-bit
// variant every offset and index of the launch is below 2^31.
template <bool F32, bool W64>
struct PrepSlot {
  using Off = std::conditional_t<W64, long long, uint32_t>;
  uint4 a, c;  // c only for fp32 input
  int kind;
  Off orow, nki;
};

template <int D, bool F32, bool W64>
__device__ __forceinline__ void prep_issue(const PrepParams& p, long long row, int col, long long nQ, long long nK,
                                           long long nrows, PrepSlot<F32, W64>& s) {
  using Off = typename PrepSlot<F32, W64>::Off;
  s.kind = -1;
  s.orow = s.nki = 0;
  if (row >= nrows) return;
  const bool isq = row < nQ, isk = !isq && row < nQ + nK;
  const long long r = isq ? row : (isk ? row - nQ : row - nQ - nK);
  const int H = isq ? p.Hq : p.Hkv;
  Off b, n, h;
  if (W64) {
    h = (Off)(r % H);
    const long long bn = r / H;
    n = (Off)(bn % p.N);
    b = (Off)(bn / p.N);
  } else {
    const uint32_t ru = (uint32_t)r;
    const uint32_t bn = div_inv(ru, isq ? p.mul_hq : p.mul_hkv, isq ? p.shr_hq : p.shr_hkv);
    h = ru - bn * (uint32_t)H;
    b = div_inv(bn, p.mul_n, p.shr_n);
    n = bn - b * (uint32_t)p.N;
  }
  // strides picked by value (a pointer into the parameters would make
  // every row an indexed constant load)
  const long long s0 = isq ? p.qs[0] : (isk ? p.ks[0] : p.vs[0]);
  const long long s1 = isq ? p.qs[1] : (isk ? p.ks[1] : p.vs[1]);
  const long long s2 = isq ? p.qs[2] : (isk ? p.ks[2] : p.vs[2]);
  const void* src = isq ? p.q : (isk ? p.k : p.v);
  const Off off = b * (Off)s0 + n * (Off)s1 + h * (Off)s2 + (Off)col;
  s.kind = isq ? 0 : (isk ? 1 : 2);
  s.orow = (b * (Off)H + h) * (Off)p.N + n;
  s.nki = (b * (Off)p.Hkv + h) * (Off)p.T + n / kBN;
  if (F32) {
    const uint4* g = reinterpret_cast<const uint4*>((const float*)src + off);
    s.a = g[0];
    s.c = g[1];
  } else {
    s.a = *reinterpret_cast<const uint4*>((const __nv_bfloat16*)src + off);
  }
}

template <int D, bool F32, bool W64>
__device__ __forceinline__ void prep_store(const PrepParams& p, int col, int lane, const PrepSlot<F32, W64>& s) {
  using Off = typename PrepSlot<F32, W64>::Off;
  constexpr int LPR = D / 8;
  float x[8];
  if (F32) {
    const uint32_t w[8] = {s.a.x, s.a.y, s.a.z, s.a.w, s.c.x, s.c.y, s.c.z, s.c.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(w[i]);
  } else {
    const uint32_t w[4] = {s.a.x, s.a.y, s.a.z, s.a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h2;
      memcpy(&h2, &w[i], 4);
      x[2 * i] = __low2float(h2);
      x[2 * i + 1] = __high2float(h2);
    }
  }
  const bool isq = s.kind == 0, isk = s.kind == 1;
  float ss = 0.0f;
  if (isq || isk) {
    const Off o = s.orow * (Off)D + (Off)col;
    uint32_t c8[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t c = cvt_e4m3x2(x[2 * i + 1], x[2 * i]);
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
        const __nv_bfloat162 bb = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        memcpy(&w[i], &bb, 4);
      }
      *reinterpret_cast<uint4*>((__nv_bfloat16*)(isq ? p.q16 : p.k16) + o) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else if (s.kind == 2) {  // v -> fp16
    const Off o = s.orow * (Off)D + (Off)col;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = cvt_f16x2_sat(x[2 * i + 1], x[2 * i]);
    *reinterpret_cast<uint4*>((__half*)p.v16 + o) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  // norms of the row's 32-element chunks (4 lanes each), then of the row;
  // all lanes take part in the shuffles.  Upper bounds: the float sums of
  // squares are rounded up.
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  if ((isq || isk) && (lane % 4) == 0) {
    constexpr int C = D / 32;
    const int c = (lane % LPR) / 4;
    const float nrm = sqrtf(ss) * (1.0f + 0x1p-16f);
    if (isq) p.nqc[s.orow * (Off)C + c] = nrm;
    else  // non-negative floats order like their bit patterns
      atomicMax((int*)&p.nkc[s.nki * (Off)C + c], __float_as_int(nrm + 0x1p-6f));
  }
#pragma unroll
  for (int o = LPR / 2; o > 2; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((isq || isk) && (lane % LPR) == 0) {
    const float nrm = sqrtf(ss) * (1.0f + 0x1p-16f);
    if (isq) p.nq[s.orow] = nrm;
    else
      atomicMax((int*)&p.nkmax[s.nki], __float_as_int(nrm));
  }
}

template <int D, bool F32, bool W64>
__global__ void __launch_bounds__(256) lamp_prep_kernel(const PrepParams p) {
  constexpr int LPR = D / 8;         // lanes per row
  constexpr int RPI = 32 / LPR;      // rows per warp instruction
  constexpr int NI = kPrepRows<D> / RPI;  // instructions per group
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, col = (lane % LPR) * 8;
  const long long nQ = p.skip_q ? 0LL : (long long)p.B * p.N * p.Hq;
  const long long nK = p.skip_kv ? 0LL : (long long)p.B * p.N * p.Hkv;
  const long long nrows = nQ + (p.v ? 2 : 1) * nK;
  const long long ngroups = (nrows + kPrepRows<D> - 1) / kPrepRows<D>;
  const long long stride = (long long)gridDim.x * 8;
  long long g = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  // two sets of slots that take turns (the loop is unrolled by two so
  // neither is copied into the other)
  PrepSlot<F32, W64> sa[NI], sb[NI];
  auto issue = [&](long long grp, PrepSlot<F32, W64>(&s)[NI]) {
#pragma unroll
    for (int it = 0; it < NI; ++it)
      prep_issue<D, F32, W64>(p, grp * kPrepRows<D> + it * RPI + sub, col, nQ, nK, nrows, s[it]);
  };
  auto store = [&](const PrepSlot<F32, W64>(&s)[NI]) {
#pragma unroll
    for (int it = 0; it < NI; ++it) prep_store<D, F32, W64>(p, col, lane, s[it]);
  };
  issue(g, sa);
  while (g < ngroups) {
    issue(g + stride, sb);
    store(sa);
    g += stride;
    if (g >= ngroups) break;
    issue(g + stride, sa);
    store(sb);
    g += stride;
  }
}

template <int D, bool F32, bool W64>
static cudaError_t launch_prep_t(const PrepParams& p, long long ngroups, cudaStream_t st) {
  // blocks that fit on the device at once, per device
  static int fit[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (fit[dev] == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lamp_prep_kernel<D, F32, W64>, 256, 0);
    if (e != cudaSuccess) return e;
    fit[dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  const long long need = (ngroups + 7) / 8;  // 8 warps a block
  const unsigned blocks = (unsigned)(need < fit[dev] ? need : fit[dev]);
  lamp_prep_kernel<D, F32, W64><<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

// largest element offset b s0 + n s1 + h s2 + D of a tensor, or -1 if a
// stride is negative
static long long max_offset(const long long* st, int B, int N, int H, int D) {
  if (st[0] < 0 || st[1] < 0 || st[2] < 0) return -1;
  return (B - 1) * st[0] + (N - 1) * st[1] + (H - 1) * st[2] + D;
}

template <int D>
static cudaError_t launch_prep_d(const PrepParams& p0, cudaStream_t st) {
  PrepParams p = p0;
  // no V rows without v, no K or V rows for prepared keys and values
  const long long rows =
      (long long)p.B * p.N * ((p.skip_q ? 0LL : p.Hq) + (p.skip_kv ? 0LL : (p.v ? 2LL : 1LL) * p.Hkv));
  const long long ngroups = (rows + kPrepRows<D> - 1) / kPrepRows<D>;
  if (ngroups == 0) return cudaSuccess;
  inv_divisor(p.Hq, p.mul_hq, p.shr_hq);
  inv_divisor(p.Hkv, p.mul_hkv, p.shr_hkv);
  inv_divisor(p.N, p.mul_n, p.shr_n);
  // 32-bit offsets when every row index, input offset and output offset of
  // the launch stays below 2^31
  const long long lim = (1LL << 31) - 1;
  const long long oq = max_offset(p.qs, p.B, p.N, p.Hq, D), ok = max_offset(p.ks, p.B, p.N, p.Hkv, D),
                  ov = p.v ? max_offset(p.vs, p.B, p.N, p.Hkv, D) : 0;
  const bool w64 = rows >= lim || (long long)p.B * p.Hq * p.N * D >= lim || oq < 0 || oq >= lim || ok < 0 ||
                   ok >= lim || ov < 0 || ov >= lim;
  if (p.in_f32)
    return w64 ? launch_prep_t<D, true, true>(p, ngroups, st) : launch_prep_t<D, true, false>(p, ngroups, st);
  return w64 ? launch_prep_t<D, false, true>(p, ngroups, st) : launch_prep_t<D, false, false>(p, ngroups, st);
}

// V8t = fl8(v) (E4M3, RNE, saturating, from the input values), transposed
// per (batch, kv head) to [B, Hkv, D, Npad] bytes with the keys contiguous:
// the K-major B operand of the FP8 P.V.  One block per 64 keys x 64
// elements of d of one (batch, kv head), through shared memory: a thread
// loads 16 consecutive elements of one key row and, after the transpose,
// stores 16 consecutive keys of one row of d.  Keys >= N are written as 0.
template <bool F32>
__global__ void __launch_bounds__(256) lamp_v8t_kernel(const void* __restrict__ v, long long vs0, long long vs1,
                                                       long long vs2, uint8_t* __restrict__ v8t, int N, int D,
                                                       int Hkv, int Npad) {
  __shared__ __align__(16) uint8_t tile[64][80];  // [element of d][key], rows padded to 80 bytes
  const int k0 = blockIdx.x * 64, d0 = blockIdx.y * 64, bh = blockIdx.z;
  const int b = bh / Hkv, g = bh - b * Hkv;
  const int tid = threadIdx.x;
  const int kr = tid >> 2, dc = (tid & 3) * 16, key = k0 + kr;
  float x[16];
  if (key < N) {
    const long long off = (long long)b * vs0 + (long long)key * vs1 + (long long)g * vs2 + d0 + dc;
    if constexpr (F32) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(v) + off);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 f = src[i];
        x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
      }
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(v) + off);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 w = src[i];
        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x[8 * i + 2 * j] = __uint_as_float(wd[j] << 16);
          x[8 * i + 2 * j + 1] = __uint_as_float(wd[j] & 0xFFFF0000u);
        }
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.0f;
  }
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const uint16_t c = cvt_e4m3x2(x[i + 1], x[i]);
    tile[dc + i][kr] = (uint8_t)(c & 0xFFu);
    tile[dc + i + 1][kr] = (uint8_t)(c >> 8);
  }
  __syncthreads();
  const int dr = tid >> 2, kc = (tid & 3) * 16;
  *reinterpret_cast<uint4*>(v8t + ((size_t)bh * D + d0 + dr) * (size_t)Npad + k0 + kc) =
      *reinterpret_cast<const uint4*>(&tile[dr][kc]);
}

cudaError_t launch_v8t(const void* v, const int64_t* vs, bool in_f32, uint8_t* v8t, int B, int N, int Hkv, int D,
                       cudaStream_t st) {
  const int T = (N + kBN - 1) / kBN;
  const dim3 grid((unsigned)T, (unsigned)(D / 64), (unsigned)(B * Hkv));
  if (in_f32)
    lamp_v8t_kernel<true><<<grid, 256, 0, st>>>(v, vs[0], vs[1], vs[2], v8t, N, D, Hkv, T * kBN);
  else
    lamp_v8t_kernel<false><<<grid, 256, 0, st>>>(v, vs[0], vs[1], vs[2], v8t, N, D, Hkv, T * kBN);
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
