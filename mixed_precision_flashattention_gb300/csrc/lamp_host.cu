// lamp_host.cu -- lamp_attn_fwd on host buffers: the batch (and, for small
// batches, the kv-head groups) is cut into chunks, and per chunk the
// host->device copies, the forward pass and the device->host copies run on
// their own streams, so the transfers of one chunk overlap the computation
// of its neighbours.  Each chunk has its own device slot while the slots fit
// a 1 GiB budget (else slots are reused, at least two), so a chunk's copy in
// never waits for an earlier chunk's computation.  Consecutive chunks
// compute on four streams (the caller's and three internal ones): every
// chunk holds causal rows that see the whole sequence, whose CTAs take
// about as long as the chunk itself, so the next chunks' CTAs must fill the
// SMs that those leave idle.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/lamp_attn.h"
#include "lamp_common.cuh"

namespace lamp {
namespace {

struct Plan {
  int nb, nh;       // chunks over the batch and over kv-head groups
  int hq_c, hkv_c;  // query and kv heads per chunk
  int nchunks;
  int nslots;       // device slots (chunk c uses slot c % nslots)
  size_t q_bytes, kv_bytes, o_bytes, lse_bytes, ws_bytes, slot_bytes, total;
  lamp_shapes cs;   // shapes of one chunk (dense device layout)
};

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

constexpr int kMinChunks = 16;                     // measured: 16 beat 4, 8 and 32 at the Qwen3-8B shape
constexpr int kMaxSlots = 32;
constexpr size_t kSlotBudget = (size_t)1 << 30;    // device bytes for slots beyond the first two
constexpr int kComputeStreams = 4;                 // the caller's stream + 3 internal ones

// At least kMinChunks chunks when possible: kv-head groups are split (a
// divisor of heads_kv) until batch * groups reaches it.
bool make_plan(const lamp_shapes& s, Plan& p) {
  const int B = s.batch, Hq = s.heads_q, Hkv = s.heads_kv, N = s.seqlen, D = s.head_dim;
  if (B < 1 || N < 1 || Hkv < 1 || Hq < 1 || Hq % Hkv) return false;
  int nh = 1;
  while (B * nh < kMinChunks && nh < Hkv) {
    int next = nh + 1;
    while (next <= Hkv && Hkv % next) ++next;
    if (next > Hkv) break;
    nh = next;
  }
  p.nb = B;
  p.nh = nh;
  p.hkv_c = Hkv / nh;
  p.hq_c = p.hkv_c * (Hq / Hkv);
  p.nchunks = B * nh;
  const size_t ei = s.in_dtype == LAMP_DT_FP32 ? 4 : 2, eo = s.out_dtype == LAMP_DT_FP32 ? 4 : 2;
  p.q_bytes = al256((size_t)N * p.hq_c * D * ei);
  p.kv_bytes = al256((size_t)N * p.hkv_c * D * ei);
  p.o_bytes = al256((size_t)N * p.hq_c * D * eo);
  p.lse_bytes = al256((size_t)p.hq_c * N * 4);
  lamp_shapes& c = p.cs;
  c = s;
  c.batch = 1;
  c.heads_q = p.hq_c;
  c.heads_kv = p.hkv_c;
  const int64_t qs[3] = {(int64_t)N * p.hq_c * D, (int64_t)p.hq_c * D, D};
  const int64_t ks[3] = {(int64_t)N * p.hkv_c * D, (int64_t)p.hkv_c * D, D};
  for (int i = 0; i < 3; ++i) {
    c.q_stride[i] = qs[i];
    c.o_stride[i] = qs[i];
    c.k_stride[i] = ks[i];
    c.v_stride[i] = ks[i];
  }
  c.workspace = nullptr;
  c.workspace_bytes = 0;
  for (int i = 0; i < 3; ++i) c.stage_events[i] = nullptr;
  p.ws_bytes = al256(lamp_attn_workspace_bytes(&c));
  if (p.ws_bytes == 0) return false;
  p.slot_bytes = p.q_bytes + 2 * p.kv_bytes + p.o_bytes + p.lse_bytes + p.ws_bytes;
  const size_t fit = kSlotBudget / p.slot_bytes;
  p.nslots = (int)(fit < 2 ? 2 : (fit > (size_t)kMaxSlots ? kMaxSlots : fit));
  // LAMP_HOST_MAX_SLOTS (>= 2) caps the slots, e.g. to exercise their reuse
  if (const char* e = getenv("LAMP_HOST_MAX_SLOTS")) {
    const int m = atoi(e);
    if (m >= 2 && m < p.nslots) p.nslots = m;
  }
  if (p.nslots > p.nchunks) p.nslots = p.nchunks;
  p.total = (size_t)p.nslots * p.slot_bytes + al256((size_t)p.nchunks * LAMP_NUM_COUNTERS * 8);
  return true;
}

// Sum the per-chunk counters into dst; the status slot keeps the first
// non-zero status.
__global__ void sum_counters_kernel(unsigned long long* dst, const unsigned long long* src, int nchunks) {
  const int i = threadIdx.x;
  if (i >= LAMP_NUM_COUNTERS) return;
  unsigned long long acc = 0;
  for (int c = 0; c < nchunks; ++c) {
    const unsigned long long v = src[(size_t)c * LAMP_NUM_COUNTERS + i];
    if (i == LAMP_CNT_STATUS) {
      if (acc == 0) acc = v;
    } else {
      acc += v;
    }
  }
  dst[i] = acc;
}

// Per device: two copy streams, the internal compute streams and the events
// of one call (per slot: inputs landed, computed, outputs read back; then
// the start and one join per internal stream), created once in the
// device's current context and created anew when that context changes
// (after a cudaDeviceReset the old handles are dropped, not used).  A call
// holds the device's lock from start to end -- it is synchronous -- so
// calls on one device run one after the other.
constexpr int kJoin = 3 * kMaxSlots;
constexpr int kEvents = kJoin + 2 + kComputeStreams;
struct HostCtx {
  std::mutex mu;
  CUcontext ctx = nullptr;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[kComputeStreams - 1] = {};
  cudaEvent_t ev[kEvents] = {};
};
HostCtx g_ctx[64];

using CtxFn = CUresult (*)(CUcontext*);
CUcontext current_context() {
  static CtxFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (CtxFn)f;
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// With c.mu held and the device's primary context current.
bool ctx_ready(HostCtx& c) {
  const CUcontext now = current_context();
  if (!now) return false;
  if (now != c.ctx) {
    c.h2d = c.d2h = nullptr;
    for (auto& s : c.comp) s = nullptr;
    for (auto& e : c.ev) e = nullptr;
    c.ctx = now;
  }
  if (!c.h2d && cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (!c.d2h && cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess) return false;
  for (auto& s : c.comp)
    if (!s && cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return false;
  for (auto& e : c.ev)
    if (!e && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
  return true;
}

}  // namespace
}  // namespace lamp

using namespace lamp;

extern "C" {

size_t lamp_attn_host_buffer_bytes(const lamp_shapes* shapes) {
  if (!shapes) return 0;
  Plan p;
  return make_plan(*shapes, p) ? p.total : 0;
}

int lamp_attn_fwd_host(const void* q, const void* k, const void* v, void* out, float* lse,
                       const lamp_shapes* shapes, int mask_kind, float delta, float tau, lamp_stats* stats,
                       void* dev_buffer, size_t dev_buffer_bytes) {
  // (the device scratch of each chunk is this call's own: nothing prepared in it)
  if (!q || !k || !v || !out || !shapes || shapes->kv_prepared || shapes->q_prepared) return LAMP_ERR_INVALID_ARG;
  const lamp_shapes& s = *shapes;
  const int D = s.head_dim;
  if (D != 64 && D != 128 && D != 256) return LAMP_ERR_UNSUPPORTED;
  // heads and head_dim of the host tensors must be dense (a chunk of heads
  // is then one row segment per sequence position)
  if (s.q_stride[2] != D || s.k_stride[2] != D || s.v_stride[2] != D || s.o_stride[2] != D)
    return LAMP_ERR_INVALID_ARG;
  Plan p;
  if (!make_plan(s, p)) return LAMP_ERR_INVALID_ARG;
  uint8_t* buf = (uint8_t*)dev_buffer;
  if (buf && (dev_buffer_bytes < p.total || ((uintptr_t)buf & 255u))) return LAMP_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LAMP_ERR_CUDA;
  if (cudaSetDevice(dev) != cudaSuccess) return LAMP_ERR_CUDA;  // binds the primary context to this thread
  HostCtx& hc = g_ctx[dev];
  std::lock_guard<std::mutex> lock(hc.mu);
  if (!ctx_ready(hc)) return LAMP_ERR_CUDA;
  const HostCtx& cps = hc;
  cudaEvent_t* ev = hc.ev;
  cudaStream_t sc = (cudaStream_t)s.stream;
  bool own = false;
  if (!buf) {
    if (cudaMallocAsync((void**)&buf, p.total, sc) != cudaSuccess) return LAMP_ERR_CUDA;
    own = true;
  }
  int rc = LAMP_OK;
  auto cuda_ok = [&](cudaError_t e) {
    if (e != cudaSuccess && rc == LAMP_OK) rc = LAMP_ERR_CUDA;
    return e == cudaSuccess;
  };
  unsigned long long* cnt = (unsigned long long*)(buf + (size_t)p.nslots * p.slot_bytes);
  const size_t ei = s.in_dtype == LAMP_DT_FP32 ? 4 : 2, eo = s.out_dtype == LAMP_DT_FP32 ? 4 : 2;
  const int N = s.seqlen, Hq = s.heads_q, Hkv = s.heads_kv;
  const int T = (N + 63) / 64;

  // the other streams start after the work already queued on the caller's
  // stream; chunk c computes on comp[c % kComputeStreams]
  cuda_ok(cudaEventRecord(ev[kJoin], sc));
  cuda_ok(cudaStreamWaitEvent(cps.h2d, ev[kJoin], 0));
  cuda_ok(cudaStreamWaitEvent(cps.d2h, ev[kJoin], 0));
  cudaStream_t comp[kComputeStreams] = {sc};
  for (int i = 1; i < kComputeStreams; ++i) {
    comp[i] = cps.comp[i - 1];
    cuda_ok(cudaStreamWaitEvent(comp[i], ev[kJoin], 0));
  }
  for (int c = 0; c < p.nchunks && rc == LAMP_OK; ++c) {
    const int b = c / p.nh, g0 = (c % p.nh) * p.hkv_c, h0 = g0 * (Hq / Hkv);
    const int slot = c % p.nslots;
    const bool reuse = c >= p.nslots;
    uint8_t* sb = buf + slot * p.slot_bytes;
    uint8_t *dq = sb, *dk = sb + p.q_bytes, *dv = dk + p.kv_bytes, *dout = dv + p.kv_bytes;
    float* dlse = (float*)(dout + p.o_bytes);
    uint8_t* dws = (uint8_t*)dlse + p.lse_bytes;
    cudaEvent_t e_in = ev[3 * slot], e_done = ev[3 * slot + 1], e_out = ev[3 * slot + 2];
    // inputs: the slot's previous chunk must have been computed
    if (reuse) cuda_ok(cudaStreamWaitEvent(cps.h2d, e_done, 0));
    const char* hq = (const char*)q + ((size_t)b * s.q_stride[0] + (size_t)h0 * D) * ei;
    const char* hk = (const char*)k + ((size_t)b * s.k_stride[0] + (size_t)g0 * D) * ei;
    const char* hv = (const char*)v + ((size_t)b * s.v_stride[0] + (size_t)g0 * D) * ei;
    cuda_ok(cudaMemcpy2DAsync(dq, (size_t)p.hq_c * D * ei, hq, (size_t)s.q_stride[1] * ei, (size_t)p.hq_c * D * ei, N,
                              cudaMemcpyHostToDevice, cps.h2d));
    cuda_ok(cudaMemcpy2DAsync(dk, (size_t)p.hkv_c * D * ei, hk, (size_t)s.k_stride[1] * ei, (size_t)p.hkv_c * D * ei,
                              N, cudaMemcpyHostToDevice, cps.h2d));
    cuda_ok(cudaMemcpy2DAsync(dv, (size_t)p.hkv_c * D * ei, hv, (size_t)s.v_stride[1] * ei, (size_t)p.hkv_c * D * ei,
                              N, cudaMemcpyHostToDevice, cps.h2d));
    cuda_ok(cudaEventRecord(e_in, cps.h2d));
    // compute: inputs landed, and the slot's previous outputs were read back
    const cudaStream_t cst = comp[c % kComputeStreams];
    cuda_ok(cudaStreamWaitEvent(cst, e_in, 0));
    if (reuse) cuda_ok(cudaStreamWaitEvent(cst, e_out, 0));
    if (rc != LAMP_OK) break;
    lamp_shapes cs = p.cs;
    cs.stream = cst;
    cs.workspace = dws;
    cs.workspace_bytes = p.ws_bytes;
    lamp_stats st;
    st.counters = (uint64_t*)(cnt + (size_t)c * LAMP_NUM_COUNTERS);
    st.mask = (stats && stats->mask) ? stats->mask + ((size_t)b * Hq + h0) * T * T : nullptr;
    const int r = lamp_attn_fwd(dq, dk, dv, dout, dlse, &cs, mask_kind, delta, tau, &st);
    if (r != LAMP_OK) {
      rc = r;
      break;
    }
    cuda_ok(cudaEventRecord(e_done, cst));
    // outputs back to the host
    cuda_ok(cudaStreamWaitEvent(cps.d2h, e_done, 0));
    char* ho = (char*)out + ((size_t)b * s.o_stride[0] + (size_t)h0 * D) * eo;
    cuda_ok(cudaMemcpy2DAsync(ho, (size_t)s.o_stride[1] * eo, dout, (size_t)p.hq_c * D * eo, (size_t)p.hq_c * D * eo,
                              N, cudaMemcpyDeviceToHost, cps.d2h));
    if (lse)
      cuda_ok(cudaMemcpyAsync(lse + ((size_t)b * Hq + h0) * N, dlse, (size_t)p.hq_c * N * 4, cudaMemcpyDeviceToHost,
                              cps.d2h));
    cuda_ok(cudaEventRecord(e_out, cps.d2h));
  }
  // join: the caller's stream waits for the last read-back, the last copy
  // in and the internal compute streams
  cuda_ok(cudaEventRecord(ev[kJoin + 1], cps.d2h));
  cuda_ok(cudaStreamWaitEvent(sc, ev[kJoin + 1], 0));
  cuda_ok(cudaEventRecord(ev[kJoin], cps.h2d));
  cuda_ok(cudaStreamWaitEvent(sc, ev[kJoin], 0));
  for (int i = 1; i < kComputeStreams; ++i) {
    cuda_ok(cudaEventRecord(ev[kJoin + 1 + i], comp[i]));
    cuda_ok(cudaStreamWaitEvent(sc, ev[kJoin + 1 + i], 0));
  }
  if (rc == LAMP_OK && stats && stats->counters) {
    sum_counters_kernel<<<1, 32, 0, sc>>>((unsigned long long*)stats->counters, cnt, p.nchunks);
    cuda_ok(cudaGetLastError());
  }
  if (own) cuda_ok(cudaFreeAsync(buf, sc));
  // the results are in host memory when the call returns
  cuda_ok(cudaStreamSynchronize(sc));
  return rc;
}

}  // extern "C"
