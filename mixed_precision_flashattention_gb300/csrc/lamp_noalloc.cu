// lamp_noalloc.cu -- lamp_attn_fwd_noalloc: the forward pass with its
// scratch in a fixed, file-scope device array instead of caller- or
// call-allocated workspace.
//
// Who needs it: callers that must not allocate device memory while they
// run -- for example a plug-in inside a host framework that owns all device
// memory through its own pooling allocator (a raw cudaMalloc/cudaFree would
// bypass its accounting and cudaFree synchronises the device), or a
// latency-bound serving loop that has to keep every call free of implicit
// synchronisation.  Such callers pass only inputs and outputs.
//
// Cost: the array (LAMP_NOALLOC_SCRATCH_BYTES) lives on every GPU that
// loads this library, until the process exits.  All calls share it and it
// keeps the last call's contents; the pre-pass rewrites the 8/16-bit copies
// and norms in full and every call clears the parts that must start at zero
// (per-tile key norms, abort word) before its kernels run.  Two calls whose
// work overlaps on the GPU (different streams, or different host threads
// on one device) race on the array: serialise them.
#include <cuda_runtime.h>

#include "../../include/lamp_attn.h"

namespace {

__device__ __align__(256) static unsigned char g_noalloc_scratch[LAMP_NOALLOC_SCRATCH_BYTES];

// Device address of the array on the current device.  In host code the
// array's name only stands in for the symbol; the address comes from
// cudaGetSymbolAddress in the current context, looked up on every call (a
// host-side lookup once the module is loaded), so no address outlives a
// cudaDeviceReset or belongs to another context.
int scratch_on_current_device(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LAMP_ERR_CUDA;
  *out = p;
  return LAMP_OK;
}

}  // namespace

extern "C" int lamp_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                                     const lamp_shapes* shapes, int mask_kind, float delta, float tau,
                                     lamp_stats* stats) {
  if (!shapes || shapes->kv_prepared || shapes->q_prepared) return LAMP_ERR_INVALID_ARG;  // the scratch is this call's own
  const size_t need = lamp_attn_workspace_bytes(shapes);
  if (need == 0) {
    // the same status lamp_attn_fwd gives: shapes that are valid except for
    // the head dimension are unsupported, anything else is an argument error
    lamp_shapes probe = *shapes;
    probe.head_dim = 128;
    return lamp_attn_workspace_bytes(&probe) != 0 ? LAMP_ERR_UNSUPPORTED : LAMP_ERR_INVALID_ARG;
  }
  if (need > (size_t)LAMP_NOALLOC_SCRATCH_BYTES) return LAMP_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != LAMP_OK) return st;
  lamp_shapes s = *shapes;
  s.workspace = scratch;
  s.workspace_bytes = (size_t)LAMP_NOALLOC_SCRATCH_BYTES;
  return lamp_attn_fwd(q, k, v, out, lse, &s, mask_kind, delta, tau, stats);
}
