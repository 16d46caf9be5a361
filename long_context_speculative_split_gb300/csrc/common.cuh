// Device-side building blocks shared by the libmgd kernels (sm_103a).
//
// Hand-written inline PTX for: mbarrier pipelines with bounded waits, Tensor
// Memory Accelerator tile loads (cp.async.bulk.tensor), ldmatrix / movmatrix
// fragment shuffles and bf16 mma.sync.  Nothing here is specific to one
// kernel's arithmetic.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "internal.h"

namespace mgd {

// ---------------------------------------------------------------- programmatic dependent launch
// The timed kernels are launched with programmatic stream serialization
// (launch_pdl), so the next kernel in the stream can be scheduled and run its
// set-up while this one finishes.  Each of them lets its dependents launch at
// entry and calls pdl_wait() before it touches global memory: the wait returns
// once the preceding kernel has completed and its writes are visible, and since
// every kernel launched this way waits, completion stays ordered along a chain.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The same launch with a thread-block cluster of `cluster` CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, dim3 cluster, size_t smem,
                                      cudaStream_t stream, Args &&...args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster.x;
  attr[0].val.clusterDim.y = cluster.y;
  attr[0].val.clusterDim.z = cluster.z;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- time / errors
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every spin-wait in this library gives up after this long, raises
// MGD_DEVERR_TIMEOUT and lets the kernel return.  The only waits on other
// CTAs are the SnapKV scorer's (for slices other running CTAs have already
// claimed, microseconds apart), so a correct kernel never comes close.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Error bit of a kernel whose launch clears the header first.
__device__ __forceinline__ void raise_error(WsHeader *hdr, unsigned bit) {
  atomicOr(&hdr->err[1], bit);
}

// Error bit of a self-resetting kernel (no clearing launch before it): the word of
// this call's parity.  seq advances only after every CTA's producer checked in.
__device__ __forceinline__ void raise_error_sr(WsHeader *hdr, unsigned bit) {
  const unsigned s = *reinterpret_cast<volatile unsigned *>(&hdr->seq);
  atomicOr(&hdr->err[s & 1u], bit);
}

// End of one part of a self-resetting call: block `id` (one check-in per block,
// after its claims from next_unit are all done; `claims` of them succeeded).
// The last of `parts` check-ins puts the counters back to zero, clears the
// error word the next call will use and advances seq, so the workspace is ready
// for the next call with no clearing launch in between.  It also checks two
// sums against the values a call started from a ready header produces: the
// successful claims (`expect`) and the block ids of the check-ins, which come
// with the check-in count in one atomic word.  A header left dirty by other use
// (a stale next_unit skips units; a stale count ends the call early; stale
// sums) breaks one of them, and the call raises MGD_DEVERR_STALE_WS unless one
// of its waits timed out (which stops claiming).
__device__ __forceinline__ void call_check_in(WsHeader *hdr, unsigned parts, unsigned id, unsigned claims,
                                              unsigned expect) {
  if (claims) atomicAdd(&hdr->claimed, claims);
  __threadfence();
  const unsigned long long mine = (1ull << 40) + id + 1ull;
  const unsigned long long now = atomicAdd(&hdr->done_ids, mine) + mine;
  if ((now >> 40) == parts) {
    __threadfence();
    volatile unsigned *h = reinterpret_cast<volatile unsigned *>(hdr);
    const unsigned s = h[offsetof(WsHeader, seq) / 4];
    const unsigned got = h[offsetof(WsHeader, claimed) / 4];
    const unsigned long long all_ids = (static_cast<unsigned long long>(parts) * (parts + 1ull)) / 2ull;
    if ((got != expect || (now & ((1ull << 40) - 1ull)) != all_ids) && !(h[s & 1u] & 0x8u))
      atomicOr(&hdr->err[s & 1u], 0x20u);
    h[offsetof(WsHeader, next_unit) / 4] = 0u;
    h[offsetof(WsHeader, next_unit2) / 4] = 0u;
    h[offsetof(WsHeader, claimed) / 4] = 0u;
    *reinterpret_cast<volatile unsigned long long *>(&hdr->done_ids) = 0ull;
    h[(s + 1u) & 1u] = 0u;  // err[(s + 1) & 1]
    h[offsetof(WsHeader, seq) / 4] = s + 1u;
  }
}

// Bounded spin until the counter at p (written by other CTAs) reaches `need`,
// with acquire semantics at GPU scope and a short sleep between polls.
// Returns false after kWaitLimitNs.
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool spin_until_geq(const unsigned *p, unsigned need) {
  if (ld_acquire_gpu(p) >= need) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(p) < need) {
    __nanosleep(64);
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32): results below
// 2^-126 flush to zero, which no softmax sum here can notice.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (the three-input form of PTX max.f32, sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---------------------------------------------------------------- shared memory
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Distributed shared memory of a thread-block cluster: store into the CTA of
// rank `rank` at the place `local` has in this CTA's shared memory, and a
// barrier of every thread of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void st_cluster_f2(const void *local, uint32_t rank, float2 v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local)), "r"(rank));
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(ra), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete may
// be parked by the hardware until it completes or `hint_ns` pass, instead of
// polling; parked warps leave their issue slots to the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_parked(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t kParkNs = 1000000;  // 1 ms per parked try; the overall limit is kWaitLimitNs

// Bounded wait for the phase with the given parity to complete.  Returns false
// (and the caller must unwind) when kWaitLimitNs elapsed first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_parked(bar, parity, kParkNs)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// 4-D tiled load (coordinates innermost first) into shared memory, completion
// counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, uint64_t *bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// L2 eviction-priority policies for loads that carry a cache hint: evict_last
// for data the CTA will read again soon, evict_first for a last read.
// One-dimensional bulk copy global -> shared memory through the TMA unit: both addresses
// 16-byte aligned, `bytes` a multiple of 16; completes as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// tma_load_4d with an L2 cache-hint policy.
__device__ __forceinline__ void tma_load_4d_hint(void *dst, const void *tmap, uint64_t *bar, int c0, int c1, int c2,
                                                 int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}
// 4-D tiled prefetch of a box into L2: no shared memory, nothing to wait for,
// and no memory changed (L2 is the point of coherence, so a prefetch issued
// while another kernel writes the same lines cannot leave a stale copy).
__device__ __forceinline__ void tma_prefetch_l2_4d(const void *tmap, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of 16-byte chunk `c` (0..7) of row `r` inside a tile written by
// TMA with 128-byte swizzling (rows of 128 bytes, tile base 1024-aligned).
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- fragments / mma
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// Transpose an 8x8 b16 matrix held in the standard fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, f32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, f32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Two floats to an f16x2 register (round to nearest; lo in the low half).
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// A bf16x2 register as f16x2: exact for magnitudes in [2^-14, 65504] (a bf16
// value is a float with its low 16 bits zero), gradual underflow below, and
// infinite above.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  return pack_f16(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t *>(&v);
}
// Split two floats into bf16 "hi" parts and the bf16-rounded remainders, so
// that hi + lo carries ~16 significant bits.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t &hi, uint32_t &lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t *>(&h);
  lo = *reinterpret_cast<uint32_t *>(&l);
}

// ---------------------------------------------------------------- tcgen05 (5th-generation tensor cores)
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (the layout of a 64-column TMA box).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;          // leading byte offset (unused for this layout)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;          // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;          // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void umma_f16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16, both
// K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Named barrier over `count` threads (warps of a role group).
__device__ __forceinline__ void named_bar(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float warp_max_xor(float v, int lane_mask_lo, int lane_mask_hi) {
  for (int m = lane_mask_lo; m <= lane_mask_hi; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}
__device__ __forceinline__ float warp_sum_xor(float v, int lane_mask_lo, int lane_mask_hi) {
  for (int m = lane_mask_lo; m <= lane_mask_hi; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

}  // namespace mgd
