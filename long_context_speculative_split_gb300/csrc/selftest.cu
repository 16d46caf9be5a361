// Self-test of the device error path: each bounded wait of the library gives
// up after kWaitLimitNs, raises MGD_DEVERR_TIMEOUT in the workspace's error
// word and lets its kernel return, leaving the context usable.  This kernel
// makes the two kinds of wait the kernels use run out on purpose, one CTA of
// one warp, nothing else touched (and occupy_kernel holds SMs for a while, so a
// test can check that a kernel makes progress with few of its CTAs resident):
//   which = 0: an mbarrier phase that no thread or copy ever completes (the
//              shape of every TMA / MMA / accumulator wait);
//   which = 1: a counter in the workspace that no CTA ever raises (the shape
//              of the SnapKV scorer's wait for the other slices of a pair).
#include "common.cuh"

namespace mgd {
namespace {

__global__ void bounded_wait_selftest(WsHeader *hdr, const unsigned *never_raised, int which) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  const bool done = (which == 0) ? mbar_wait(&bar, 0) : spin_until_geq(never_raised, 1u);
  if (!done) raise_error(hdr, 0x8u);
}

// Holds an SM for `ns` nanoseconds: thread 0 watches the global timer; the CTA's
// dynamic shared memory keeps other kernels' CTAs off the SM meanwhile.
__global__ void occupy_kernel(uint64_t ns) {
  extern __shared__ unsigned char held[];
  if (threadIdx.x != 0) return;
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) __nanosleep(1000);
  held[0] = 0;  // the allocation is used
}

}  // namespace

cudaError_t launch_selftest_occupy(int ctas, int smem_bytes, int usec, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  occupy_kernel<<<ctas, 32, smem_bytes, stream>>>(static_cast<uint64_t>(usec) * 1000u);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int which, void *ws, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(ws, 0, 2 * kAlign, stream);  // header and the counter after it
  if (e != cudaSuccess) return e;
  unsigned char *w = static_cast<unsigned char *>(ws);
  bounded_wait_selftest<<<1, 32, 0, stream>>>(reinterpret_cast<WsHeader *>(w),
                                              reinterpret_cast<const unsigned *>(w + kAlign), which);
  return cudaGetLastError();
}

}  // namespace mgd
