// Internal (not exported) declarations shared by the libmgd translation units:
// workspace layouts, launch plans and the kernel launchers that api.cu calls
// after validating the arguments.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>

namespace mgd {

// Every workspace starts with this 256-byte header.  Kernels either clear it
// ahead of the call (cudaMemsetAsync on the call's stream) or leave it ready
// for the next call themselves (the self-resetting kernels, see call_check_in).
struct WsHeader {
  // MGD_DEVERR_* bits.  Kernels that clear the header before they run raise into
  // err[1].  Kernels that leave the workspace ready for the next call (no clearing
  // launch) raise into err[seq & 1]; the last CTA to check in clears the other word and
  // advances seq.  Either way, after a call err[0] | err[1] holds its bits (a consumer's
  // timeout raised after its CTA checked in shows again after the next call).
  unsigned err[2];
  unsigned next_unit;  // dynamic work counter of persistent kernels
  unsigned next_unit2;
  unsigned seq;  // calls completed by the self-resetting kernels on this workspace
  // Successful claims from next_unit, summed at check-in.  From a zero start a
  // self-resetting call's claims add up to a known count; any other sum means
  // the call started from a header that was not left ready (MGD_DEVERR_STALE_WS).
  unsigned claimed;
  // End-of-call check-ins of the self-resetting kernels, one 64-bit word updated
  // by one atomic per check-in: bits 40..63 count the check-ins, bits 0..39 sum
  // (block index + 1) over them.  The value a check-in gets back therefore says
  // exactly which blocks had checked in: at the last check-in of a call started
  // from a ready header the sum is parts * (parts + 1) / 2.
  unsigned long long done_ids;
  unsigned pad[56];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr size_t kAlign = 256;

// An NVTX range named after the entry point, open for the duration of one call
// (the host-side enqueue).  Without a profiler attached the calls return at once.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

// Whether kernels are launched with programmatic stream serialization
// (mgd_set_programmatic_launch; on by default).
bool pdl_enabled();
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (152 on GB300 when no device is visible,
// so that size queries made without a GPU stay deterministic).
int current_sm_count();

// ------------------------------------------------------------------ attention
// Split-KV plan for the tensor-core attention kernel.  A "pair" is one
// (sequence, KV head, row group); a "unit" is one chunk of C keys of a pair.
struct AttnPlan {
  int B, T, Hq, Hkv, D, kv_cap;
  int G;          // query heads per KV head
  int rows;       // G * T query rows per KV head
  int RG;         // row groups (rows > 32 are split into groups of <= 32)
  int rows_pg;    // rows per group (<= 32)
  int NT;         // n8 tiles per row group = ceil(rows_pg / 8)
  int C;          // keys per unit (multiple of 64)
  int nchunk;     // chunk slots per pair = ceil(kv_cap / C)
  int pairs;      // B * Hkv * RG
  int grid;       // persistent CTAs
  size_t off_tickets, off_part_o, off_part_l, ws_bytes;
};
AttnPlan plan_attention(int B, int T, int Hq, int Hkv, int D, int kv_cap, int sm_count);

struct AttnArgs {
  const void *q;
  const void *k;
  const void *v;
  const int32_t *kv_len;
  int64_t kv_batch_stride, kv_head_stride;
  float sm_scale;
  void *out;
  int out_bf16;
  float *lse;
  void *ws;
  cudaStream_t stream;
};
// bf16 inputs, tensor cores, TMA tiles, persistent split-KV with in-kernel merge.
cudaError_t launch_attention_tc(const AttnPlan &p, const AttnArgs &a, const CUtensorMap &kmap,
                                const CUtensorMap &vmap);
// Any-dtype CUDA-core attention, one CTA per (sequence, KV head).
size_t simt_attention_ws_bytes();
cudaError_t launch_attention_simt(const AttnPlan &p, const AttnArgs &a);

// Encode a 4-D bf16 tensor map over a KV tensor [B, Hkv, kv_cap, D] with
// boxes of 64 columns x box_rows rows and 128-byte swizzling.  Returns a CUDA
// driver status.
int encode_kv_tensor_map(CUtensorMap *map, const void *base, int B, int Hkv, int kv_cap, int D,
                         int64_t batch_stride, int64_t head_stride, unsigned box_rows = 64);

// ------------------------------------------------------------------ SnapKV
// Keys per job of the one-read tcgen05 scorer (12 tiles of 128 keys): small
// enough that the slices open at once (one per resident CTA) mostly stay in L2
// until their pass 2 re-reads them, large enough that the per-job exchange
// stays a small share of the job (measured: 1280 / 1536 / 1792 / 2048 keys).
// Capacities above kSnapMaxSlices * kSnapSliceKeys keys get longer slices, so
// that a pair never has more than 64 slices (a CTA keeps the slices of a pair
// it holds in a 64-bit mask).
constexpr int kSnapSliceKeys = 1536;
constexpr int kSnapMaxSlices = 64;

struct SnapPlan {
  int B, Hq, Hkv, D, kv_cap, W, G, rows, RG;
  int C;       // keys per scoring unit (multiple of 64; a multiple of 128 for the tcgen05 scorer)
  int nchunk;  // ceil(kv_cap / C)
  int pairs;   // B * Hkv
  size_t off_cnt;  // unsigned [2][pairs]: slices published and slices claimed per pair (zeroed with the header)
  int lrows;       // windows of <= 8 rows: logit rows stored per key by pass 1 (4 or 8), else 0
  size_t off_logits;  // float [pairs][kv_cap][lrows] when lrows > 0
  size_t off_part, off_scores, off_pooled, ws_bytes;
};
SnapPlan plan_snapkv(int B, int Hq, int Hkv, int D, int kv_cap, int W);

struct SnapArgs {
  const void *q_win;
  const void *k;
  const void *v;
  const int32_t *kv_len;
  int64_t kv_batch_stride, kv_head_stride;
  int pool, K, draft_cap;
  const int32_t *budgets;  // nullable: per-sequence budgets K_b [B] (device), replacing K
  float sm_scale;
  int32_t *sel_idx;
  void *k_draft;
  void *v_draft;
  int32_t *draft_len;
  float *scores_out;
  void *ws;
  cudaStream_t stream;
};
// kmap: K tensor map (bf16 path); qmap: window-query tensor map, non-null only
// when the tcgen05 scoring kernel is eligible (snap_tc05_eligible).
cudaError_t launch_snapkv(const SnapPlan &p, const SnapArgs &a, int in_f32, const CUtensorMap *kmap,
                          const CUtensorMap *qmap);
bool snap_tc05_eligible(const SnapPlan &p);
cudaError_t launch_snap_score_tc05(const SnapPlan &p, const SnapArgs &a, const CUtensorMap &kmap,
                                   const CUtensorMap &qmap);
// 4-D bf16 tensor map over window queries [B, W, Hq, D] with one box per
// (64 columns, G heads, W rows): the 128-byte-swizzled W*G x 64 tile of a KV head.
int encode_qwin_tensor_map(CUtensorMap *map, const void *base, int B, int W, int Hq, int D, int G);

// ------------------------------------------------------------------ self-test
// One bounded wait that nothing completes (0: an mbarrier phase, 1: a counter
// in the workspace); needs 2 * kAlign bytes of workspace.
cudaError_t launch_selftest_wait(int which, void *ws, cudaStream_t stream);
// `ctas` CTAs, each holding `smem_bytes` of shared memory for `usec` microseconds.
cudaError_t launch_selftest_occupy(int ctas, int smem_bytes, int usec, cudaStream_t stream);

// ------------------------------------------------------------------ sampling
struct SpecPlan {
  int B, gamma, V;
  int split;     // elements per statistics block (and per CTA of the draw kernels)
  int nsplit;    // ceil(V / split)
  int nsub;      // ceil(V / 2048): sub-ranges of a row (one warp each)
  int nrows;     // 2*gamma + 1 rows per sequence (gamma+1 target, gamma draft)
  size_t off_tickets, off_drawn, off_stats, off_sub, ws_bytes;
};
SpecPlan plan_spec(int B, int gamma, int V);

struct SpecArgs {
  const float *target;
  const float *draft;
  int32_t *draft_tokens;
  const float *u;
  int mode, row;
  int32_t *out_tokens;
  int32_t *num_accepted;
  void *ws;
  cudaStream_t stream;
};
cudaError_t launch_spec(const SpecPlan &p, const SpecArgs &a);

// ------------------------------------------------------------------ commit / rollback
cudaError_t launch_commit(const int32_t *num_accepted, int B, int gamma, int Hkv, int D, int esz, int32_t *kv_len,
                          const void *k, const void *v, int kv_cap, int64_t kv_bstride, int64_t kv_hstride,
                          void *k_draft, void *v_draft, int draft_cap, int64_t d_bstride, int64_t d_hstride,
                          int32_t *draft_len, void *ws, cudaStream_t stream);

// ------------------------------------------------------------------ StreamingLLM-style cache
cudaError_t launch_streaming_select(const void *k, const void *v, const int32_t *kv_len, int B, int Hkv, int D,
                                    int esz, int kv_cap, int64_t bstride, int64_t hstride, int sink, int K,
                                    int32_t *sel_idx, void *k_draft, void *v_draft, int draft_cap,
                                    int32_t *draft_len, cudaStream_t stream);

}  // namespace mgd
