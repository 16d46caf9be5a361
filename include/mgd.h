/*
 * mgd.h -- C ABI of libmgd.so: the GPU hot path of self-speculative decoding
 * with a compressed draft KV cache (MagicDec-style), for NVIDIA GB300 (sm_103a).
 *
 * Sources restated here (the pages give the method, never an interface):
 *   [MagicDec] "MAGICDEC: BREAKING THE LATENCY-THROUGHPUT TRADEOFF FOR LONG
 *              CONTEXT GENERATION WITH SPECULATIVE DECODING" (paper notes,
 *              arXiv:2408.11049): quick-read summary, sections 3.1-3.3,
 *              4.1 (Eq. 3), 4.4, appendix A.1.
 *   [SD-Serving] "Wann beschleunigt spekulatives Decoding das LLM-Serving?",
 *              section "Eine Verifizierungsrunde verstehen".
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is CALLER-OWNED DEVICE memory on the current
 *     device.  The library never allocates device memory; scratch space is
 *     the caller's `ws` buffer of at least the size the matching
 *     mgd_*_workspace_size() returns for the same shape.
 *   - A workspace is ZERO-FILLED once before its first use (e.g. one
 *     cudaMemsetAsync after allocating it).  The calls do not clear it per
 *     call: their kernels leave its counters at zero for the next call, which
 *     saves a clearing launch ahead of every launch.  A buffer that served as
 *     scratch for one kind of call (attention, selection, sampling, commit) is
 *     zero-filled again before it serves another kind.  An attention,
 *     selection or commit call that starts from a header in any other state
 *     (its counters not at zero) detects it at its end and raises
 *     MGD_DEVERR_STALE_WS: its outputs are then unspecified, and the workspace
 *     is zero-filled again before the next call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream; nothing synchronises.
 *   - Shape / argument errors are detected on the host before anything is
 *     launched and return MGD_ERR_INVALID_ARG / MGD_ERR_UNSUPPORTED /
 *     MGD_ERR_WORKSPACE; a failed launch returns MGD_ERR_CUDA.  A text for the
 *     last error of the calling thread is available from mgd_last_error().
 *   - Values that live on the device (kv_len, draft_len, token ids) cannot be
 *     checked on the host.  Kernels that meet an out-of-range device value skip
 *     that sequence (its outputs are unspecified) and set a bit in the error
 *     word kept at the start of `ws` (two 32-bit words whose OR is the
 *     call's bits); mgd_workspace_errors() reads it back.
 *   - Element strides are in elements, layouts are row-major, the innermost
 *     dimension (D or V) is contiguous.  Every device pointer must be 16-byte
 *     aligned and bf16 KV strides must be multiples of 8 elements (the K/V
 *     tiles are fetched by the Tensor Memory Accelerator).
 *   - Calls are thread-safe as long as concurrent calls use distinct `ws`.
 *   - B == 0 is a valid no-op.
 */
#ifndef MGD_H_
#define MGD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MGD_OK = 0,
  MGD_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, bad stride, misaligned pointer */
  MGD_ERR_UNSUPPORTED = 2,   /* valid request the kernels do not implement (e.g. D not in {64,128}) */
  MGD_ERR_WORKSPACE = 3,     /* ws NULL or smaller than mgd_*_workspace_size() */
  MGD_ERR_CUDA = 4           /* a CUDA runtime / driver call failed; see mgd_last_error() */
} mgd_status;

typedef enum { MGD_BF16 = 0, MGD_F32 = 1 } mgd_dtype;

typedef enum {
  MGD_VERIFY = 0,        /* accept / reject a whole speculation round */
  MGD_DRAW_DRAFT = 1,    /* draw draft tokens from the draft distributions */
  MGD_VERIFY_DRAWN = 2   /* MGD_VERIFY reusing the draft rows' normalisers left by this round's draws */
} mgd_sample_mode;

/* Bits of the device error word (see mgd_workspace_errors). */
#define MGD_DEVERR_KV_LEN   0x1u   /* kv_len[b] < T, or > kv_cap; or draft_len[b] < 1 or > k_cap */
#define MGD_DEVERR_SNAP_LEN 0x2u   /* kv_len[b] < W or > kv_cap in mgd_snapkv_select; or a budget outside [W, draft_cap] */
#define MGD_DEVERR_TOKEN    0x4u   /* a draft token id outside [0, V) */
#define MGD_DEVERR_TIMEOUT  0x8u   /* a bounded wait inside a kernel gave up (never expected) */
#define MGD_DEVERR_COMMIT   0x10u  /* mgd_commit_round: num_accepted, kv_len or draft_len out of range */
#define MGD_DEVERR_STALE_WS 0x20u  /* a call found its workspace header not ready (not zero-filled, or last
                                      used by another kind of call); its outputs are unspecified */
#define MGD_DEVERR_NOT_DRAWN 0x40u /* MGD_VERIFY_DRAWN: a sequence's gamma draft rows were not all drawn on
                                      this workspace since its last rejection sample; its outputs are
                                      unspecified */

const char *mgd_status_string(mgd_status s);
/* Detail text of the last non-OK status returned on the calling thread ("" if none). */
const char *mgd_last_error(void);
/* Library version, major * 10000 + minor * 100 + patch. */
int mgd_version(void);

/*
 * Reads the device error word of a workspace after the work queued on
 * `stream` finished (this call synchronises `stream`).  *flags receives the
 * OR of MGD_DEVERR_* bits raised by the last call that used `ws`.
 */
mgd_status mgd_workspace_errors(const void *ws, void *stream, uint32_t *flags);

/*
 * Self-test of the device error path.  Every wait inside a libmgd kernel is
 * bounded (2 s); one that gives up raises MGD_DEVERR_TIMEOUT in the
 * workspace's error word and lets its kernel return, so the CUDA context
 * stays usable.  This call launches one small kernel whose wait nothing ever
 * satisfies, so it runs out on purpose:
 *   which = 0: an mbarrier phase that nothing completes (the form of the
 *              TMA, tensor-core and accumulator waits);
 *   which = 1: a workspace counter that no CTA raises (the form of the
 *              SnapKV scorer's wait for the other slices of a pair).
 * Asynchronous on `stream`; the kernel takes about 2 s.  Afterwards
 * mgd_workspace_errors(ws) reports MGD_DEVERR_TIMEOUT.  `ws`: device memory
 * of at least MGD_SELFTEST_WS_BYTES.  Errors: MGD_ERR_INVALID_ARG (null ws,
 * `which` not 0 or 1), MGD_ERR_WORKSPACE (ws_bytes too small), MGD_ERR_CUDA.
 */
#define MGD_SELFTEST_WS_BYTES 512u
mgd_status mgd_selftest_bounded_wait(int which, void *ws, size_t ws_bytes, void *stream);

/*
 * Launch mode of every later call in the process.  By default (enable != 0)
 * the kernels of consecutive calls on one stream are launched with
 * programmatic stream serialization: a kernel may be scheduled, and do set-up
 * that touches no memory, while the previous kernel in the stream finishes; it
 * waits for that kernel's completion (and memory) before any access.  With
 * enable == 0 every kernel is launched plainly, after the previous one ends.
 * Results are the same either way; this switch exists for comparisons.
 */
void mgd_set_programmatic_launch(int enable);

/*
 * Diagnostic: holds SMs for a while, so that a test can run another call on a
 * second stream while few SMs are free (the SnapKV scorer's CTAs wait for one
 * another; this shows that they make progress whatever number of them is
 * resident).  Launches `ctas` CTAs of one warp on `stream`; each holds
 * `smem_bytes` of dynamic shared memory (which keeps other CTAs off its SM when
 * large) and returns after `usec` microseconds of the GPU's global timer.  It
 * waits on nothing else and touches no memory.  Errors: MGD_ERR_INVALID_ARG
 * (ctas outside [1, 65535], smem_bytes outside [1, 232448], usec outside
 * [0, 2000000]), MGD_ERR_CUDA.
 */
mgd_status mgd_selftest_occupy(int ctas, int smem_bytes, int usec, void *stream);

/* ------------------------------------------------------------------------ *
 * Verify attention.  [MagicDec] section 3.2: verifying gamma draft tokens
 * and decoding read the same KV cache, so the target's verify pass is decode
 * attention over T = gamma + 1 query rows per sequence against the full
 * cache (the extra row gives the bonus-token distribution of [SD-Serving]).
 *
 *   q        [B, T, Hq, D]            in_dtype, contiguous
 *   k, v     [B, Hkv, kv_cap, D]      in_dtype; element (b, h, j, d) at
 *                                     b*kv_batch_stride + h*kv_head_stride + j*D + d
 *   kv_len   [B] int32 (device)       rows of sequence b, INCLUDING the T rows
 *                                     being verified; T <= kv_len[b] <= kv_cap
 *   out      [B, T, Hq, D]            out_dtype (MGD_F32 or MGD_BF16)
 *   lse      [B, T, Hq] float32 or NULL: natural-log sum of exp(scores)
 *
 * Query head h reads KV head h / (Hq/Hkv).  Row t sits at position
 * kv_len[b]-T+t and attends to keys 0 .. kv_len[b]-T+t (causal among the
 * appended rows); scores are sm_scale * <q, k>; softmax and accumulation in
 * float32.  The probabilities enter the P V product (bf16 path) as bf16 hi + lo
 * parts, about 16 significant bits; when a KV head has more than 16 query rows
 * (Hq/Hkv * T > 16, e.g. G = 4 and T >= 5) as float16 with V converted to
 * float16 instead (11 significant bits, output rel-L2 about 1e-4 against exact
 * arithmetic): there V entries must lie within the float16 range, |v| <= 65504,
 * or the outputs that read them are not finite.  Supported: D in {64, 128};
 * 1 <= T <= 17 (gamma <= 16, as the sampling and commit calls take);
 * Hq % Hkv == 0.
 * in_dtype MGD_BF16 runs the tensor-core split-KV kernel; MGD_F32 runs a
 * float32 CUDA-core kernel (for float32 inputs; not the timed path).
 * ------------------------------------------------------------------------ */
size_t mgd_verify_workspace_size(int B, int T, int Hq, int Hkv, int D, int kv_cap);
mgd_status mgd_verify_attn(const void *q, const void *k, const void *v, const int32_t *kv_len,
                           int B, int T, int Hq, int Hkv, int D, int kv_cap,
                           int64_t kv_batch_stride, int64_t kv_head_stride, float sm_scale,
                           mgd_dtype in_dtype, void *out, mgd_dtype out_dtype, float *lse,
                           void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * Draft attention.  [MagicDec] quick-read summary and section 4.1 (Eq. 3):
 * the draft is the target model itself reading a compressed KV of budget K,
 * costing T_D(K) per draft step.  One query row per sequence attends to all
 * draft_len[b] rows of the compacted cache (no mask).
 *
 *   q                 [B, Hq, D]              in_dtype (the single draft row)
 *   k_draft, v_draft  [B, Hkv, k_cap, D]      in_dtype, strides as for verify
 *   draft_len         [B] int32 (device)      1 <= draft_len[b] <= k_cap
 *   out [B, Hq, D] out_dtype;  lse [B, Hq] float32 or NULL.
 * Identical arithmetic to mgd_verify_attn with T = 1.
 * ------------------------------------------------------------------------ */
size_t mgd_draft_workspace_size(int B, int Hq, int Hkv, int D, int k_cap);
mgd_status mgd_draft_attn(const void *q, const void *k_draft, const void *v_draft,
                          const int32_t *draft_len, int B, int Hq, int Hkv, int D, int k_cap,
                          int64_t kv_batch_stride, int64_t kv_head_stride, float sm_scale,
                          mgd_dtype in_dtype, void *out, mgd_dtype out_dtype, float *lse,
                          void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * SnapKV draft-cache selection.  [MagicDec] section 4.4 (static selection,
 * SnapKV named) and appendix A.1 (the compressed KV is built at prefill and
 * reused by every draft step).  The pages do not define SnapKV; this call
 * computes the plain reading:
 *   1. window queries q_win[b, w, h] (position kv_len[b]-W+w) attend causally
 *      to keys 0 .. kv_len[b]-W+w; their softmax probabilities are summed over
 *      the W window rows and the G = Hq/Hkv heads of a KV head, for every
 *      prefix key j < kv_len[b]-W;
 *   2. max-pool along the sequence with odd kernel `pool` (stride 1, positions
 *      outside the prefix ignored);
 *   3. keep K_eff = min(K, kv_len[b]) rows: the top K_eff-W prefix positions
 *      (ties -> lower position) plus the W window positions, ascending;
 *   4. gather those K and V rows into the draft cache.
 *
 *   q_win    [B, W, Hq, D] in_dtype;  k, v, kv_len as for mgd_verify_attn
 *            (W <= kv_len[b] <= kv_cap)
 *   sel_idx  [B, Hkv, draft_cap] int32: kept positions, -1 after K_eff
 *   k_draft, v_draft [B, Hkv, draft_cap, D] in_dtype, contiguous; rows after
 *            K_eff are left untouched (draft_cap >= K leaves room for rows
 *            appended while drafting)
 *   draft_len [B] int32: K_eff
 *   scores   [B, Hkv, kv_cap] float32 or NULL: pooled scores of the prefix
 *            positions (entries >= kv_len[b]-W unspecified)
 * Supported: D in {64, 128}; 1 <= W <= 64; 1 <= pool <= 63 and odd; W <= K <= draft_cap.
 * ------------------------------------------------------------------------ */
size_t mgd_snapkv_workspace_size(int B, int Hq, int Hkv, int D, int kv_cap, int W);
mgd_status mgd_snapkv_select(const void *q_win, const void *k, const void *v, const int32_t *kv_len,
                             int B, int Hq, int Hkv, int D, int kv_cap,
                             int64_t kv_batch_stride, int64_t kv_head_stride,
                             int W, int pool, int K, float sm_scale, mgd_dtype in_dtype,
                             int32_t *sel_idx, void *k_draft, void *v_draft, int draft_cap,
                             int32_t *draft_len, float *scores,
                             void *ws, size_t ws_bytes, void *stream);

/*
 * The same selection with a budget per sequence ([MagicDec] section 4.3: in a
 * batch of mixed lengths each sequence may have its own KV budget): step 3
 * keeps K_eff = min(budgets[b], kv_len[b]) rows of sequence b.
 *   budgets  [B] int32 device memory, W <= budgets[b] <= draft_cap; a
 *            sequence whose budget is outside that range is skipped
 *            (sel_idx -1, draft_len 0) and raises MGD_DEVERR_SNAP_LEN.
 * Every other argument, the workspace size and the errors are those of
 * mgd_snapkv_select; host check: draft_cap >= W, budgets not NULL when B > 0.
 */
mgd_status mgd_snapkv_select_budgets(const void *q_win, const void *k, const void *v, const int32_t *kv_len,
                                     int B, int Hq, int Hkv, int D, int kv_cap,
                                     int64_t kv_batch_stride, int64_t kv_head_stride,
                                     int W, int pool, const int32_t *budgets, float sm_scale, mgd_dtype in_dtype,
                                     int32_t *sel_idx, void *k_draft, void *v_draft, int draft_cap,
                                     int32_t *draft_len, float *scores,
                                     void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * Speculative sampling.  [SD-Serving] "Eine Verifizierungsrunde verstehen":
 * candidates are accepted left to right using both distributions; at the
 * first rejection a correction is drawn from the residual target
 * distribution max(0, p - q) (renormalised) and later candidates are
 * dropped; when all are accepted one more token is drawn from the target.
 * The paragraph after it states that this preserves the target distribution.
 *
 *   target_logits [B, gamma+1, V] float32 (verify modes only; may be NULL otherwise)
 *   draft_logits  [B, gamma, V]   float32
 *   draft_tokens  [B, gamma] int32: written by MGD_DRAW_DRAFT, read by the verify modes
 *   u             [B, gamma+1, 3] float32 in [0,1): slot 0 draws the draft
 *                 token of position i, slot 1 is the acceptance test, slot 2
 *                 the correction draw; position gamma uses slot 2 only (bonus)
 *   row           MGD_DRAW_DRAFT: draw only position `row` (0 <= row < gamma),
 *                 or every position when row < 0.  Ignored by the verify modes.
 *   out_tokens    [B, gamma+1] int32 (verify modes): accepted drafts, then the
 *                 correction or bonus token, then -1
 *   num_accepted  [B] int32 (verify modes)
 *
 * p = softmax(target logits), q = softmax(draft logits), temperature 1.
 * Accept position i iff u[b,i,1] * q_i(x_i) < p_i(x_i).  A draw from weights r
 * with uniform u returns the smallest index whose running sum (index order)
 * exceeds u * sum(r), else the last index with r > 0; a residual that sums to
 * zero (rounding only) falls back to p.  Arithmetic in float32.
 * Supported: 1 <= gamma <= 16; 1 <= V < 2^31.
 * ------------------------------------------------------------------------ */
/*
 * Modes.  MGD_DRAW_DRAFT draws position `row` (or every position) of
 * draft_tokens and leaves the drawn rows' softmax statistics (max and sum of
 * exp per 16384-entry chunk) in the workspace.  MGD_VERIFY computes the
 * statistics of all 2*gamma+1 rows itself.  MGD_VERIFY_DRAWN computes only the
 * gamma+1 target rows' and takes the gamma draft rows' from the workspace: it
 * is for a round whose draft rows were all drawn with MGD_DRAW_DRAFT on this
 * workspace, from these draft_logits, since the workspace's last rejection
 * sample (each rejection sample, in either mode, forgets the draws).  A
 * sequence for which that does not hold raises MGD_DEVERR_NOT_DRAWN and gets
 * unspecified outputs.  Both verify modes take the same decisions up to
 * float32 rounding of the normalisers.
 */
size_t mgd_spec_workspace_size(int B, int gamma, int V);
mgd_status mgd_spec_sample(const float *target_logits, const float *draft_logits,
                           int32_t *draft_tokens, const float *u, int B, int gamma, int V,
                           int mode, int row, int32_t *out_tokens, int32_t *num_accepted,
                           void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * StreamingLLM-style draft cache.  [MagicDec] section 5.1 (the end-to-end runs
 * draft over a StreamingLLM-style sparse KV) and 5.2 (SnapKV beats it).  The
 * pages do not define it; this call keeps the first s = min(sink, K_eff)
 * positions (attention sinks) and the last K_eff - s positions,
 * K_eff = min(K, kv_len[b]), ascending, and gathers their rows.
 *   k, v, kv_len as for mgd_verify_attn (1 <= kv_len[b] <= kv_cap);
 *   sel_idx [B, Hkv, draft_cap] int32 (-1 after K_eff); k_draft, v_draft
 *   [B, Hkv, draft_cap, D] contiguous; draft_len [B] = K_eff.
 * Needs no workspace.  A sequence with kv_len outside [1, kv_cap] gets
 * draft_len 0 and no kept rows.  Supported: 0 <= sink; 1 <= K <= draft_cap.
 * ------------------------------------------------------------------------ */
mgd_status mgd_streaming_select(const void *k, const void *v, const int32_t *kv_len, int B, int Hkv, int D,
                                int kv_cap, int64_t kv_batch_stride, int64_t kv_head_stride, int sink, int K,
                                mgd_dtype dtype, int32_t *sel_idx, void *k_draft, void *v_draft, int draft_cap,
                                int32_t *draft_len, void *stream);

/* ------------------------------------------------------------------------ *
 * Dynamic top-K attention drafting (one draft step).  [MagicDec] section 4.4,
 * first bullet (top-K attention reaches very high acceptance with a much
 * smaller budget but is impractical because of its selection cost) and second
 * bullet (dynamic selection searches the KV cache again for every query).
 * The pages give no algorithm; this call is the SnapKV selection above with
 * the draft query itself as a one-row window (W = 1, no pooling), followed by
 * draft attention over the selected rows:
 *   1. the draft query q[b, h] sits at position kv_len[b]-1 (its own K/V row
 *      is the last cache row); its softmax probabilities over keys
 *      0 .. kv_len[b]-1 are summed over the G = Hq/Hkv heads of a KV head;
 *   2. keep K_eff = min(K, kv_len[b]) rows: the newest row plus the top
 *      K_eff-1 earlier positions (ties -> lower position), ascending, and
 *      gather them into k_draft / v_draft;
 *   3. out[b, h] = softmax attention of q[b, h] over the kept rows.
 *   q        [B, Hq, D] in_dtype;  k, v, kv_len as for mgd_verify_attn
 *            (1 <= kv_len[b] <= kv_cap)
 *   sel_idx, k_draft, v_draft, draft_len as for mgd_snapkv_select (outputs;
 *            draft_cap >= K; the draft rows are contiguous)
 *   out      [B, Hq, D] out_dtype;  lse [B, Hq] float32 or NULL (natural log)
 *   ws       mgd_topk_draft_workspace_size(...) bytes
 * Every call reads the whole K cache (the probabilities need each query's
 * normaliser over all keys first; the first pass keeps the G logits of every
 * key, which the key sums then read back instead of K): that is the
 * selection cost.  A sequence with kv_len outside [1, kv_cap] is flagged in
 * the error word at the start of `ws` (MGD_DEVERR_SNAP_LEN, draft_len 0, no
 * kept rows); its out and lse rows are unspecified.
 * Supported: D in {64, 128}; in_dtype bf16 or float32; 1 <= K <= draft_cap.
 * ------------------------------------------------------------------------ */
size_t mgd_topk_draft_workspace_size(int B, int Hq, int Hkv, int D, int kv_cap, int draft_cap);
mgd_status mgd_topk_draft_attn(const void *q, const void *k, const void *v, const int32_t *kv_len, int B, int Hq,
                               int Hkv, int D, int kv_cap, int64_t kv_batch_stride, int64_t kv_head_stride, int K,
                               float sm_scale, mgd_dtype in_dtype, int32_t *sel_idx, void *k_draft,
                               void *v_draft, int draft_cap, int32_t *draft_len, void *out, mgd_dtype out_dtype,
                               float *lse, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * Commit / rollback after a verification round.  [SD-Serving] "Eine
 * Verifizierungsrunde verstehen": candidates after the first rejection are
 * discarded; [MagicDec] appendix A.1: the draft reads the compressed KV built
 * at prefill, so tokens committed since then are appended to it.  The pages
 * give no layout; this call follows the verify convention (kv_len includes the
 * T = gamma + 1 verify rows: the last committed token, then the gamma drafts):
 *   - with n = num_accepted[b], rows kv_len-T .. kv_len-T+n are kept and the
 *     rest rolled back: kv_len[b] -= gamma - n;
 *   - those n + 1 rows (K and V of every KV head) are copied to the draft cache
 *     at draft_len[b] .. draft_len[b] + n, and draft_len[b] += n + 1.
 *   num_accepted [B] int32 (device, e.g. from mgd_spec_sample);
 *   kv_len, draft_len [B] int32, updated in place;
 *   k, v [B, Hkv, kv_cap, D] and k_draft, v_draft [B, Hkv, draft_cap, D] in
 *   `dtype`, strides in elements as for mgd_verify_attn (rows contiguous).
 * A sequence with n outside [0, gamma], kv_len outside [T, kv_cap] or
 * draft_len + n + 1 > draft_cap is left unchanged and flagged
 * (MGD_DEVERR_COMMIT).  Byte copies and integer updates only, in one launch.
 * Like the attention calls, this call does not clear its workspace header:
 * the kernel leaves it ready for the next call, so `ws` is zero-filled once
 * before its first use (and again after serving as any other call's scratch).
 * ------------------------------------------------------------------------ */
size_t mgd_commit_workspace_size(int B);
mgd_status mgd_commit_round(const int32_t *num_accepted, int B, int gamma, int Hkv, int D, mgd_dtype dtype,
                            int32_t *kv_len, const void *k, const void *v, int kv_cap,
                            int64_t kv_batch_stride, int64_t kv_head_stride, void *k_draft, void *v_draft,
                            int draft_cap, int64_t draft_batch_stride, int64_t draft_head_stride,
                            int32_t *draft_len, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------ *
 * Allocation-free speculative sampling.  The papers have no counterpart to
 * this call; it exists for callers that cannot allocate device memory, such
 * as code running under a host framework that owns all device memory through
 * its own pool, or a serving loop whose memory is planned once at start-up
 * and must not call cudaMalloc (which can synchronise the device and fail
 * late) on the per-token path.  Such callers cannot hand mgd_spec_sample a
 * workspace, so this variant keeps its scratch in a fixed device array of
 * MGD_NOALLOC_SCRATCH_BYTES owned by the library: every GPU that loads
 * libmgd.so holds that array until the process exits.
 *
 * Arguments, results and arithmetic are those of mgd_spec_sample without
 * `ws` / `ws_bytes`; inputs and outputs are still caller-provided device
 * memory.  The call allocates nothing.
 *   - Limit: the scratch it needs, mgd_spec_workspace_size(B, gamma, V), must
 *     fit in MGD_NOALLOC_SCRATCH_BYTES (about B * ((2*gamma+1) * ceil(V/16384) * 8
 *     + ceil(V/2048) * 8 + 8) + 768 bytes; e.g. B <= 963 at gamma = 4,
 *     V = 128256); larger requests return MGD_ERR_UNSUPPORTED with an
 *     explanation in mgd_last_error().
 *   - Every call looks up the array's device address on the current device
 *     with cudaGetSymbolAddress (a host-side lookup, so the address is never
 *     stale, e.g. after a device reset).  The first call on a device may also
 *     load the library's device code there; make that first call before any
 *     stream capture.
 *   - Every call shares the one array, which keeps the last call's contents;
 *     each call leaves its counters at zero for the next one (the array is
 *     zero when the library is loaded).  Calls that
 *     overlap on the GPU (different streams or host threads) race on it and
 *     must be serialised by the caller.  The device error word of this
 *     variant is not readable through mgd_workspace_errors.
 * ------------------------------------------------------------------------ */
#define MGD_NOALLOC_SCRATCH_BYTES (1u << 20)
mgd_status mgd_spec_sample_noalloc(const float *target_logits, const float *draft_logits,
                                   int32_t *draft_tokens, const float *u, int B, int gamma, int V,
                                   int mode, int row, int32_t *out_tokens, int32_t *num_accepted,
                                   void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MGD_H_ */
