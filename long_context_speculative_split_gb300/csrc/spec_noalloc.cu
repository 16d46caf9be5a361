// mgd_spec_sample_noalloc: speculative sampling for callers that cannot
// allocate device memory.
//
// Some callers own every byte of device memory through their own pool, or plan
// all memory once at start-up, and may not call cudaMalloc (or any allocating
// routine) on the per-token path: an allocation can synchronise the device,
// can fail late under fragmentation, and would bypass the caller's accounting.
// Such callers cannot provide the caller-owned workspace that mgd_spec_sample
// asks for.  This entry point runs the same kernels with their scratch held in
// a fixed device array that the library owns for the life of the process.
//
// The array (kNoAllocScratchBytes) exists on every GPU that loads the library
// until the process exits.  In host code its name is only a host-side stand-in,
// not a device address, so every call looks the device address up, with the
// call's device current, through cudaGetSymbolAddress: a cheap host-side
// lookup, and never stale (after a device reset the array may live elsewhere).
#include <cuda_runtime.h>

#include <cstdio>

#include "../../include/mgd.h"
#include "internal.h"

namespace mgd {
void record_error(const char *msg);

namespace {

constexpr size_t kNoAllocScratchBytes = MGD_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes % kAlign == 0, "scratch size is a multiple of the alignment");

static __device__ __align__(256) unsigned char g_spec_scratch[kNoAllocScratchBytes];

// Device address of g_spec_scratch on the current device.
cudaError_t scratch_on_current_device(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_spec_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace mgd

extern "C" mgd_status mgd_spec_sample_noalloc(const float *target_logits, const float *draft_logits,
                                              int32_t *draft_tokens, const float *u, int B, int gamma, int V,
                                              int mode, int row, int32_t *out_tokens, int32_t *num_accepted,
                                              void *stream) {
  const mgd::NvtxRange nvtx_range("mgd_spec_sample_noalloc");
  if (B <= 0)  // argument checks only (B == 0 is a no-op); nothing touches the GPU
    return mgd_spec_sample(target_logits, draft_logits, draft_tokens, u, B, gamma, V, mode, row, out_tokens,
                           num_accepted, nullptr, 0, stream);
  const size_t need = mgd_spec_workspace_size(B, gamma, V);
  if (need > mgd::kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "mgd_spec_sample_noalloc: B=%d, gamma=%d, V=%d needs %zu bytes of scratch, more than its fixed %zu; "
             "use mgd_spec_sample with a workspace",
             B, gamma, V, need, mgd::kNoAllocScratchBytes);
    mgd::record_error(msg);
    return MGD_ERR_UNSUPPORTED;
  }
  void *scratch = nullptr;
  const cudaError_t e = mgd::scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "mgd_spec_sample_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    mgd::record_error(msg);
    return MGD_ERR_CUDA;
  }
  return mgd_spec_sample(target_logits, draft_logits, draft_tokens, u, B, gamma, V, mode, row, out_tokens,
                         num_accepted, scratch, mgd::kNoAllocScratchBytes, stream);
}
