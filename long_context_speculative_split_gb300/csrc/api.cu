// extern "C" entry points of libmgd.so (declared in include/mgd.h):
// argument validation, workspace sizing, TMA descriptor encoding and dispatch
// to the kernel launchers.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/mgd.h"
#include "internal.h"

namespace mgd {

namespace {
thread_local std::string g_last_error;

mgd_status fail(mgd_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
mgd_status fail(mgd_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}
mgd_status cuda_fail(cudaError_t e, const char *where) {
  return fail(MGD_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}
mgd_status ok() { return MGD_OK; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// Shared checks of the two attention entry points.
mgd_status check_attention(const void *q, const void *k, const void *v, const int32_t *len, int B, int T, int Hq,
                           int Hkv, int D, int cap, int64_t bstride, int64_t hstride, mgd_dtype in_dtype,
                           const void *out, mgd_dtype out_dtype, const void *ws) {
  if (B < 0) return fail(MGD_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
  if (T < 1 || T > 17) return fail(MGD_ERR_INVALID_ARG, "T must be in [1, 17] (got %d)", T);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(MGD_ERR_INVALID_ARG, "need Hq >= 1, Hkv >= 1 and Hq %% Hkv == 0 (got %d, %d)", Hq, Hkv);
  if (D != 64 && D != 128) return fail(MGD_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", D);
  if (cap < 1) return fail(MGD_ERR_INVALID_ARG, "KV capacity must be >= 1 (got %d)", cap);
  if (in_dtype != MGD_BF16 && in_dtype != MGD_F32) return fail(MGD_ERR_INVALID_ARG, "bad in_dtype %d", in_dtype);
  if (out_dtype != MGD_BF16 && out_dtype != MGD_F32)
    return fail(MGD_ERR_INVALID_ARG, "bad out_dtype %d", out_dtype);
  if (hstride < static_cast<int64_t>(cap) * D)
    return fail(MGD_ERR_INVALID_ARG, "kv_head_stride %lld < capacity * D", static_cast<long long>(hstride));
  if (bstride < hstride * Hkv)
    return fail(MGD_ERR_INVALID_ARG, "kv_batch_stride %lld < Hkv * kv_head_stride", static_cast<long long>(bstride));
  if (B == 0) return ok();
  if (!q || !k || !v || !len || !out || !ws) return fail(MGD_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws))
    return fail(MGD_ERR_INVALID_ARG, "q, k, v, out and ws must be 16-byte aligned");
  if (in_dtype == MGD_BF16 && (hstride % 8 != 0 || bstride % 8 != 0))
    return fail(MGD_ERR_INVALID_ARG, "bf16 KV strides must be multiples of 8 elements");
  return ok();
}

mgd_status run_attention(const void *q, const void *k, const void *v, const int32_t *len, int B, int T, int Hq,
                         int Hkv, int D, int cap, int64_t bstride, int64_t hstride, float scale,
                         mgd_dtype in_dtype, void *out, mgd_dtype out_dtype, float *lse, void *ws,
                         size_t ws_bytes, void *stream) {
  mgd_status s = check_attention(q, k, v, len, B, T, Hq, Hkv, D, cap, bstride, hstride, in_dtype, out, out_dtype, ws);
  if (s != MGD_OK || B == 0) return s;
  AttnArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.kv_len = len;
  a.kv_batch_stride = bstride;
  a.kv_head_stride = hstride;
  a.sm_scale = scale;
  a.out = out;
  a.out_bf16 = (out_dtype == MGD_BF16);
  a.lse = lse;
  a.ws = ws;
  a.stream = static_cast<cudaStream_t>(stream);
  const AttnPlan plan = plan_attention(B, T, Hq, Hkv, D, cap, current_sm_count());
  if (in_dtype == MGD_F32) {
    if (ws_bytes < simt_attention_ws_bytes())
      return fail(MGD_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, simt_attention_ws_bytes());
    cudaError_t e = launch_attention_simt(plan, a);
    return e == cudaSuccess ? ok() : cuda_fail(e, "attention (float32) launch");
  }
  if (ws_bytes < plan.ws_bytes) return fail(MGD_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, plan.ws_bytes);
  CUtensorMap km, vm;
  int r1 = encode_kv_tensor_map(&km, k, B, Hkv, cap, D, bstride, hstride);
  int r2 = encode_kv_tensor_map(&vm, v, B, Hkv, cap, D, bstride, hstride);
  if (r1 != 0 || r2 != 0) return fail(MGD_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d, %d)", r1, r2);
  cudaError_t e = launch_attention_tc(plan, a, km, vm);
  return e == cudaSuccess ? ok() : cuda_fail(e, "attention launch");
}

}  // namespace

namespace {
std::atomic<int> g_pdl{1};
}  // namespace
bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }

// Sets the calling thread's mgd_last_error() text (for entry points defined in
// other translation units).
void record_error(const char *msg) { g_last_error = msg; }

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();  // clear the sticky-free error of a missing device
    return 152;
  }
  return n;
}

int encode_kv_tensor_map(CUtensorMap *map, const void *base, int B, int Hkv, int kv_cap, int D,
                         int64_t batch_stride, int64_t head_stride, unsigned box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return -1;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(kv_cap),
                              static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(head_stride) * 2,
                                 static_cast<cuuint64_t>(batch_stride) * 2};
  const cuuint32_t box[4] = {64, box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

int encode_qwin_tensor_map(CUtensorMap *map, const void *base, int B, int W, int Hq, int D, int G) {
  EncodeFn fn = encode_fn();
  if (!fn || G > 256 || W > 256) return -1;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(W),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2,
                                 static_cast<cuuint64_t>(W) * Hq * D * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(W), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return static_cast<int>(r);
}

}  // namespace mgd

using namespace mgd;

extern "C" {

const char *mgd_status_string(mgd_status s) {
  switch (s) {
    case MGD_OK: return "MGD_OK";
    case MGD_ERR_INVALID_ARG: return "MGD_ERR_INVALID_ARG: invalid argument";
    case MGD_ERR_UNSUPPORTED: return "MGD_ERR_UNSUPPORTED: unsupported configuration";
    case MGD_ERR_WORKSPACE: return "MGD_ERR_WORKSPACE: workspace missing or too small";
    case MGD_ERR_CUDA: return "MGD_ERR_CUDA: CUDA call failed";
  }
  return "unknown mgd_status";
}

const char *mgd_last_error(void) { return g_last_error.c_str(); }

int mgd_version(void) { return 200; }  // 0.2.0: per-sequence budgets, self-resetting attention workspaces

mgd_status mgd_workspace_errors(const void *ws, void *stream, uint32_t *flags) {
  if (!ws || !flags) return fail(MGD_ERR_INVALID_ARG, "null pointer argument");
  uint32_t v[2] = {0u, 0u};  // the two error words of the header: the call's bits are their OR
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(v, ws, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace error words");
  *flags = v[0] | v[1];
  return MGD_OK;
}

mgd_status mgd_selftest_bounded_wait(int which, void *ws, size_t ws_bytes, void *stream) {
  if (!ws) return fail(MGD_ERR_INVALID_ARG, "null workspace");
  if (which != 0 && which != 1) return fail(MGD_ERR_INVALID_ARG, "which must be 0 or 1 (got %d)", which);
  if (ws_bytes < MGD_SELFTEST_WS_BYTES)
    return fail(MGD_ERR_WORKSPACE, "workspace %zu < %u bytes", ws_bytes, MGD_SELFTEST_WS_BYTES);
  cudaError_t e = launch_selftest_wait(which, ws, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "self-test launch");
}

void mgd_set_programmatic_launch(int enable) { g_pdl.store(enable ? 1 : 0, std::memory_order_relaxed); }

mgd_status mgd_selftest_occupy(int ctas, int smem_bytes, int usec, void *stream) {
  if (ctas < 1 || ctas > 65535) return fail(MGD_ERR_INVALID_ARG, "ctas must be in [1, 65535] (got %d)", ctas);
  if (smem_bytes < 1 || smem_bytes > 227 * 1024)
    return fail(MGD_ERR_INVALID_ARG, "smem_bytes must be in [1, 232448] (got %d)", smem_bytes);
  if (usec < 0 || usec > 2000000) return fail(MGD_ERR_INVALID_ARG, "usec must be in [0, 2000000] (got %d)", usec);
  cudaError_t e = launch_selftest_occupy(ctas, smem_bytes, usec, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "occupy launch");
}

size_t mgd_verify_workspace_size(int B, int T, int Hq, int Hkv, int D, int kv_cap) {
  if (B <= 0 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || kv_cap < 1) return kAlign;
  return plan_attention(B, T, Hq, Hkv, D, kv_cap, current_sm_count()).ws_bytes;
}

mgd_status mgd_verify_attn(const void *q, const void *k, const void *v, const int32_t *kv_len, int B, int T, int Hq,
                           int Hkv, int D, int kv_cap, int64_t kv_batch_stride, int64_t kv_head_stride,
                           float sm_scale, mgd_dtype in_dtype, void *out, mgd_dtype out_dtype, float *lse, void *ws,
                           size_t ws_bytes, void *stream) {
  const NvtxRange nvtx_range("mgd_verify_attn");
  return run_attention(q, k, v, kv_len, B, T, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, sm_scale, in_dtype,
                       out, out_dtype, lse, ws, ws_bytes, stream);
}

size_t mgd_draft_workspace_size(int B, int Hq, int Hkv, int D, int k_cap) {
  return mgd_verify_workspace_size(B, 1, Hq, Hkv, D, k_cap);
}

mgd_status mgd_draft_attn(const void *q, const void *k_draft, const void *v_draft, const int32_t *draft_len, int B,
                          int Hq, int Hkv, int D, int k_cap, int64_t kv_batch_stride, int64_t kv_head_stride,
                          float sm_scale, mgd_dtype in_dtype, void *out, mgd_dtype out_dtype, float *lse, void *ws,
                          size_t ws_bytes, void *stream) {
  const NvtxRange nvtx_range("mgd_draft_attn");
  return run_attention(q, k_draft, v_draft, draft_len, B, 1, Hq, Hkv, D, k_cap, kv_batch_stride, kv_head_stride,
                       sm_scale, in_dtype, out, out_dtype, lse, ws, ws_bytes, stream);
}

size_t mgd_snapkv_workspace_size(int B, int Hq, int Hkv, int D, int kv_cap, int W) {
  if (B <= 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || kv_cap < 1 || W < 1) return kAlign;
  return plan_snapkv(B, Hq, Hkv, D, kv_cap, W).ws_bytes;
}

// SnapKV selection with one budget K for every sequence (budgets == nullptr)
// or a per-sequence budget array on the device.
static mgd_status run_snapkv(const void *q_win, const void *k, const void *v, const int32_t *kv_len, int B, int Hq,
                             int Hkv, int D, int kv_cap, int64_t kv_batch_stride, int64_t kv_head_stride, int W,
                             int pool, int K, const int32_t *budgets, float sm_scale, mgd_dtype in_dtype,
                             int32_t *sel_idx, void *k_draft, void *v_draft, int draft_cap, int32_t *draft_len,
                             float *scores, void *ws, size_t ws_bytes, void *stream) {
  if (B < 0) return fail(MGD_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
    return fail(MGD_ERR_INVALID_ARG, "need Hq >= 1, Hkv >= 1 and Hq %% Hkv == 0 (got %d, %d)", Hq, Hkv);
  if (D != 64 && D != 128) return fail(MGD_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", D);
  if (W < 1 || W > 64) return fail(MGD_ERR_UNSUPPORTED, "window W must be in [1, 64] (got %d)", W);
  if (pool < 1 || pool > 63 || pool % 2 == 0)
    return fail(MGD_ERR_INVALID_ARG, "pool kernel must be odd and in [1, 63] (got %d)", pool);
  if (!budgets && K < W) return fail(MGD_ERR_INVALID_ARG, "budget K (%d) must be >= window W (%d)", K, W);
  if (!budgets && draft_cap < K) return fail(MGD_ERR_INVALID_ARG, "draft_cap (%d) must be >= K (%d)", draft_cap, K);
  if (budgets && draft_cap < W) return fail(MGD_ERR_INVALID_ARG, "draft_cap (%d) must be >= W (%d)", draft_cap, W);
  if (kv_cap < 1) return fail(MGD_ERR_INVALID_ARG, "kv_cap must be >= 1");
  if (in_dtype != MGD_BF16 && in_dtype != MGD_F32) return fail(MGD_ERR_INVALID_ARG, "bad in_dtype %d", in_dtype);
  if (kv_head_stride < static_cast<int64_t>(kv_cap) * D)
    return fail(MGD_ERR_INVALID_ARG, "kv_head_stride < capacity * D");
  if (kv_batch_stride < kv_head_stride * Hkv) return fail(MGD_ERR_INVALID_ARG, "kv_batch_stride < Hkv * kv_head_stride");
  if (B == 0) return ok();
  if (!q_win || !k || !v || !kv_len || !sel_idx || !k_draft || !v_draft || !draft_len || !ws)
    return fail(MGD_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q_win) || !aligned16(k) || !aligned16(v) || !aligned16(k_draft) || !aligned16(v_draft) ||
      !aligned16(ws))
    return fail(MGD_ERR_INVALID_ARG, "q_win, k, v, k_draft, v_draft and ws must be 16-byte aligned");
  const int esz = (in_dtype == MGD_F32) ? 4 : 2;
  if ((kv_head_stride * esz) % 16 != 0 || (kv_batch_stride * esz) % 16 != 0)
    return fail(MGD_ERR_INVALID_ARG, "KV strides must be multiples of 16 bytes");
  const SnapPlan plan = plan_snapkv(B, Hq, Hkv, D, kv_cap, W);
  if (ws_bytes < plan.ws_bytes) return fail(MGD_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, plan.ws_bytes);
  SnapArgs a;
  a.q_win = q_win;
  a.k = k;
  a.v = v;
  a.kv_len = kv_len;
  a.kv_batch_stride = kv_batch_stride;
  a.kv_head_stride = kv_head_stride;
  a.pool = pool;
  a.K = budgets ? draft_cap : K;
  a.budgets = budgets;
  a.draft_cap = draft_cap;
  a.sm_scale = sm_scale;
  a.sel_idx = sel_idx;
  a.k_draft = k_draft;
  a.v_draft = v_draft;
  a.draft_len = draft_len;
  a.scores_out = scores;
  a.ws = ws;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (in_dtype == MGD_BF16) {
    CUtensorMap km, qm;
    if (encode_kv_tensor_map(&km, k, B, Hkv, kv_cap, D, kv_batch_stride, kv_head_stride) != 0)
      return fail(MGD_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    // the tcgen05 scorer loads a 128-key tile as two 128-row boxes (its own map); the others
    // take 64-row boxes
    CUtensorMap km128;
    const bool tc05 = snap_tc05_eligible(plan) && sm_scale > 0.f &&
                      encode_qwin_tensor_map(&qm, q_win, B, W, Hq, D, Hq / Hkv) == 0 &&
                      encode_kv_tensor_map(&km128, k, B, Hkv, kv_cap, D, kv_batch_stride, kv_head_stride, 128) == 0;
    e = launch_snapkv(plan, a, 0, tc05 ? &km128 : &km, tc05 ? &qm : nullptr);
  } else {
    e = launch_snapkv(plan, a, 1, nullptr, nullptr);
  }
  return e == cudaSuccess ? ok() : cuda_fail(e, "snapkv launch");
}

mgd_status mgd_snapkv_select(const void *q_win, const void *k, const void *v, const int32_t *kv_len, int B, int Hq,
                             int Hkv, int D, int kv_cap, int64_t kv_batch_stride, int64_t kv_head_stride, int W,
                             int pool, int K, float sm_scale, mgd_dtype in_dtype, int32_t *sel_idx, void *k_draft,
                             void *v_draft, int draft_cap, int32_t *draft_len, float *scores, void *ws,
                             size_t ws_bytes, void *stream) {
  const NvtxRange nvtx_range("mgd_snapkv_select");
  return run_snapkv(q_win, k, v, kv_len, B, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, W, pool, K, nullptr,
                    sm_scale, in_dtype, sel_idx, k_draft, v_draft, draft_cap, draft_len, scores, ws, ws_bytes, stream);
}

mgd_status mgd_snapkv_select_budgets(const void *q_win, const void *k, const void *v, const int32_t *kv_len, int B,
                                     int Hq, int Hkv, int D, int kv_cap, int64_t kv_batch_stride,
                                     int64_t kv_head_stride, int W, int pool, const int32_t *budgets, float sm_scale,
                                     mgd_dtype in_dtype, int32_t *sel_idx, void *k_draft, void *v_draft,
                                     int draft_cap, int32_t *draft_len, float *scores, void *ws, size_t ws_bytes,
                                     void *stream) {
  const NvtxRange nvtx_range("mgd_snapkv_select_budgets");
  if (B > 0 && !budgets) return fail(MGD_ERR_INVALID_ARG, "null budgets");
  return run_snapkv(q_win, k, v, kv_len, B, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, W, pool, W,
                    B > 0 ? budgets : nullptr, sm_scale, in_dtype, sel_idx, k_draft, v_draft, draft_cap, draft_len,
                    scores, ws, ws_bytes, stream);
}

size_t mgd_topk_draft_workspace_size(int B, int Hq, int Hkv, int D, int kv_cap, int draft_cap) {
  if (B <= 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || kv_cap < 1 || draft_cap < 1) return kAlign;
  return align_up(mgd_snapkv_workspace_size(B, Hq, Hkv, D, kv_cap, 1)) +
         mgd_draft_workspace_size(B, Hq, Hkv, D, draft_cap);
}

// Selection (the SnapKV call with the draft query as a one-row window and no
// pooling) into the caller's draft cache, then draft attention over it; the
// workspace holds both calls' scratch one after the other.
mgd_status mgd_topk_draft_attn(const void *q, const void *k, const void *v, const int32_t *kv_len, int B, int Hq,
                               int Hkv, int D, int kv_cap, int64_t kv_batch_stride, int64_t kv_head_stride, int K,
                               float sm_scale, mgd_dtype in_dtype, int32_t *sel_idx, void *k_draft,
                               void *v_draft, int draft_cap, int32_t *draft_len, void *out, mgd_dtype out_dtype,
                               float *lse, void *ws, size_t ws_bytes, void *stream) {
  const NvtxRange nvtx_range("mgd_topk_draft_attn");
  if (K < 1) return fail(MGD_ERR_INVALID_ARG, "budget K must be >= 1 (got %d)", K);
  if (B > 0 && !out) return fail(MGD_ERR_INVALID_ARG, "null pointer argument");
  const size_t need = mgd_topk_draft_workspace_size(B, Hq, Hkv, D, kv_cap, draft_cap);
  if (B > 0 && ws_bytes < need) return fail(MGD_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
  const size_t ws_sel = B > 0 ? align_up(mgd_snapkv_workspace_size(B, Hq, Hkv, D, kv_cap, 1)) : 0;
  mgd_status st = mgd_snapkv_select(q, k, v, kv_len, B, Hq, Hkv, D, kv_cap, kv_batch_stride, kv_head_stride, 1, 1, K,
                                    sm_scale, in_dtype, sel_idx, k_draft, v_draft, draft_cap, draft_len, nullptr,
                                    ws, ws_sel, stream);
  if (st != MGD_OK || B == 0) return st;
  // the attention step's header sits at a shape-dependent offset that a call of
  // another shape may have used as selection scratch: clear it
  cudaError_t e = cudaMemsetAsync(static_cast<unsigned char *>(ws) + ws_sel, 0, kAlign,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "clearing the attention header");
  const int64_t dh = static_cast<int64_t>(draft_cap) * D;
  return mgd_draft_attn(q, k_draft, v_draft, draft_len, B, Hq, Hkv, D, draft_cap, dh * Hkv, dh, sm_scale, in_dtype,
                        out, out_dtype, lse, static_cast<unsigned char *>(ws) + ws_sel, ws_bytes - ws_sel, stream);
}

size_t mgd_spec_workspace_size(int B, int gamma, int V) {
  if (B <= 0 || gamma < 1 || V < 1) return kAlign;
  return plan_spec(B, gamma, V).ws_bytes;
}

mgd_status mgd_spec_sample(const float *target_logits, const float *draft_logits, int32_t *draft_tokens,
                           const float *u, int B, int gamma, int V, int mode, int row, int32_t *out_tokens,
                           int32_t *num_accepted, void *ws, size_t ws_bytes, void *stream) {
  const NvtxRange nvtx_range("mgd_spec_sample");
  if (B < 0) return fail(MGD_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
  if (gamma < 1 || gamma > 16) return fail(MGD_ERR_UNSUPPORTED, "gamma must be in [1, 16] (got %d)", gamma);
  if (V < 1) return fail(MGD_ERR_INVALID_ARG, "V must be >= 1 (got %d)", V);
  if (mode != MGD_VERIFY && mode != MGD_DRAW_DRAFT && mode != MGD_VERIFY_DRAWN)
    return fail(MGD_ERR_INVALID_ARG, "bad mode %d", mode);
  if (mode == MGD_DRAW_DRAFT && row >= gamma) return fail(MGD_ERR_INVALID_ARG, "row %d >= gamma %d", row, gamma);
  if (B == 0) return ok();
  if (!draft_logits || !draft_tokens || !u || !ws) return fail(MGD_ERR_INVALID_ARG, "null pointer argument");
  const bool verify = mode != MGD_DRAW_DRAFT;
  if (verify && (!target_logits || !out_tokens || !num_accepted))
    return fail(MGD_ERR_INVALID_ARG, "MGD_VERIFY and MGD_VERIFY_DRAWN need target_logits, out_tokens and num_accepted");
  if (!aligned16(ws)) return fail(MGD_ERR_INVALID_ARG, "ws must be 16-byte aligned");
  const SpecPlan plan = plan_spec(B, gamma, V);
  if (ws_bytes < plan.ws_bytes) return fail(MGD_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, plan.ws_bytes);
  SpecArgs a;
  a.target = verify ? target_logits : nullptr;
  a.draft = draft_logits;
  a.draft_tokens = draft_tokens;
  a.u = u;
  a.mode = mode;
  a.row = row;
  a.out_tokens = out_tokens;
  a.num_accepted = num_accepted;
  a.ws = ws;
  a.stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_spec(plan, a);
  return e == cudaSuccess ? ok() : cuda_fail(e, "spec_sample launch");
}

mgd_status mgd_streaming_select(const void *k, const void *v, const int32_t *kv_len, int B, int Hkv, int D,
                                int kv_cap, int64_t kv_batch_stride, int64_t kv_head_stride, int sink, int K,
                                mgd_dtype dtype, int32_t *sel_idx, void *k_draft, void *v_draft, int draft_cap,
                                int32_t *draft_len, void *stream) {
  const NvtxRange nvtx_range("mgd_streaming_select");
  if (B < 0) return fail(MGD_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
  if (Hkv < 1 || D < 1 || kv_cap < 1) return fail(MGD_ERR_INVALID_ARG, "need Hkv, D, kv_cap >= 1");
  if (sink < 0 || K < 1 || draft_cap < K)
    return fail(MGD_ERR_INVALID_ARG, "need sink >= 0 and 1 <= K <= draft_cap (got %d, %d, %d)", sink, K, draft_cap);
  if (dtype != MGD_BF16 && dtype != MGD_F32) return fail(MGD_ERR_INVALID_ARG, "bad dtype %d", dtype);
  const int esz = (dtype == MGD_F32) ? 4 : 2;
  if ((D * esz) % 16 != 0) return fail(MGD_ERR_UNSUPPORTED, "rows must be a multiple of 16 bytes");
  if (kv_head_stride < static_cast<int64_t>(kv_cap) * D || kv_batch_stride < kv_head_stride * Hkv)
    return fail(MGD_ERR_INVALID_ARG, "strides smaller than the capacities they hold");
  if ((kv_head_stride * esz) % 16 || (kv_batch_stride * esz) % 16)
    return fail(MGD_ERR_INVALID_ARG, "strides must be multiples of 16 bytes");
  if (B == 0) return ok();
  if (!k || !v || !kv_len || !sel_idx || !k_draft || !v_draft || !draft_len)
    return fail(MGD_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_draft) || !aligned16(v_draft))
    return fail(MGD_ERR_INVALID_ARG, "k, v, k_draft and v_draft must be 16-byte aligned");
  cudaError_t e = launch_streaming_select(k, v, kv_len, B, Hkv, D, esz, kv_cap, kv_batch_stride, kv_head_stride,
                                          sink, K, sel_idx, k_draft, v_draft, draft_cap, draft_len,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "streaming select launch");
}

size_t mgd_commit_workspace_size(int B) {
  (void)B;
  return kAlign;
}

mgd_status mgd_commit_round(const int32_t *num_accepted, int B, int gamma, int Hkv, int D, mgd_dtype dtype,
                            int32_t *kv_len, const void *k, const void *v, int kv_cap, int64_t kv_batch_stride,
                            int64_t kv_head_stride, void *k_draft, void *v_draft, int draft_cap,
                            int64_t draft_batch_stride, int64_t draft_head_stride, int32_t *draft_len, void *ws,
                            size_t ws_bytes, void *stream) {
  const NvtxRange nvtx_range("mgd_commit_round");
  if (B < 0) return fail(MGD_ERR_INVALID_ARG, "B must be >= 0 (got %d)", B);
  if (gamma < 1 || gamma > 16) return fail(MGD_ERR_UNSUPPORTED, "gamma must be in [1, 16] (got %d)", gamma);
  if (Hkv < 1 || D < 1) return fail(MGD_ERR_INVALID_ARG, "need Hkv >= 1 and D >= 1");
  if (dtype != MGD_BF16 && dtype != MGD_F32) return fail(MGD_ERR_INVALID_ARG, "bad dtype %d", dtype);
  const int esz = (dtype == MGD_F32) ? 4 : 2;
  if ((D * esz) % 16 != 0) return fail(MGD_ERR_UNSUPPORTED, "rows must be a multiple of 16 bytes");
  if (kv_cap < 1 || draft_cap < 1) return fail(MGD_ERR_INVALID_ARG, "capacities must be >= 1");
  if (kv_head_stride < static_cast<int64_t>(kv_cap) * D || kv_batch_stride < kv_head_stride * Hkv ||
      draft_head_stride < static_cast<int64_t>(draft_cap) * D || draft_batch_stride < draft_head_stride * Hkv)
    return fail(MGD_ERR_INVALID_ARG, "strides smaller than the capacities they hold");
  if ((kv_head_stride * esz) % 16 || (kv_batch_stride * esz) % 16 || (draft_head_stride * esz) % 16 ||
      (draft_batch_stride * esz) % 16)
    return fail(MGD_ERR_INVALID_ARG, "strides must be multiples of 16 bytes");
  if (B == 0) return ok();
  if (!num_accepted || !kv_len || !k || !v || !k_draft || !v_draft || !draft_len || !ws)
    return fail(MGD_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_draft) || !aligned16(v_draft) || !aligned16(ws))
    return fail(MGD_ERR_INVALID_ARG, "k, v, k_draft, v_draft and ws must be 16-byte aligned");
  if (ws_bytes < kAlign) return fail(MGD_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, kAlign);
  cudaError_t e = launch_commit(num_accepted, B, gamma, Hkv, D, esz, kv_len, k, v, kv_cap, kv_batch_stride,
                                kv_head_stride, k_draft, v_draft, draft_cap, draft_batch_stride, draft_head_stride,
                                draft_len, ws, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "commit launch");
}

}  // extern "C"
