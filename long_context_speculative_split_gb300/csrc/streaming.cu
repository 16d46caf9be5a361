// StreamingLLM-style draft cache: attention sinks plus the most recent rows.
//
// MagicDec notes, section 5.1 (end-to-end runs draft over a StreamingLLM-style
// sparse KV) and 5.2 (SnapKV beats it).  The pages do not define the cache;
// reading: keep the first s = min(sink, K_eff) positions and the last
// K_eff - s positions, K_eff = min(K, L), ascending, and gather their K / V
// rows.  No scores are computed: one CTA per (sequence, KV head) writes the
// indices and copies the rows with 16-byte vectors.
#include "common.cuh"

namespace mgd {
namespace {

struct StreamParams {
  int Hkv, kv_cap, sink, K, draft_cap, row_bytes;
  int64_t bstride, hstride;  // bytes
};

__global__ void __launch_bounds__(256)
    streaming_select_kernel(const unsigned char *__restrict__ k, const unsigned char *__restrict__ v,
                            const int32_t *__restrict__ kv_len, StreamParams p, int32_t *__restrict__ sel_idx,
                            unsigned char *__restrict__ k_draft, unsigned char *__restrict__ v_draft,
                            int32_t *__restrict__ draft_len) {
  const int b = blockIdx.x / p.Hkv, h = blockIdx.x % p.Hkv;
  const size_t pr = static_cast<size_t>(b) * p.Hkv + h;
  int32_t *sel = sel_idx + pr * p.draft_cap;
  const int L = kv_len[b];
  const bool ok = (L >= 1 && L <= p.kv_cap);
  const int Keff = ok ? min(p.K, L) : 0;
  const int s = min(p.sink, Keff);
  for (int i = threadIdx.x; i < p.draft_cap; i += blockDim.x)
    sel[i] = (i < s) ? i : (i < Keff ? L - Keff + i : -1);
  if (threadIdx.x == 0 && h == 0) draft_len[b] = Keff;
  const int vecs = p.row_bytes / 16;
  const unsigned char *ks = k + b * p.bstride + h * p.hstride;
  const unsigned char *vs = v + b * p.bstride + h * p.hstride;
  unsigned char *kd = k_draft + pr * p.draft_cap * p.row_bytes;
  unsigned char *vd = v_draft + pr * p.draft_cap * p.row_bytes;
  for (int i = threadIdx.x; i < Keff * vecs; i += blockDim.x) {
    const int row = i / vecs, c = i % vecs;
    const int src_row = (row < s) ? row : L - Keff + row;
    const size_t so = static_cast<size_t>(src_row) * p.row_bytes + c * 16;
    const size_t dof = static_cast<size_t>(row) * p.row_bytes + c * 16;
    *reinterpret_cast<uint4 *>(kd + dof) = __ldg(reinterpret_cast<const uint4 *>(ks + so));
    *reinterpret_cast<uint4 *>(vd + dof) = __ldg(reinterpret_cast<const uint4 *>(vs + so));
  }
}

}  // namespace

cudaError_t launch_streaming_select(const void *k, const void *v, const int32_t *kv_len, int B, int Hkv, int D,
                                    int esz, int kv_cap, int64_t bstride, int64_t hstride, int sink, int K,
                                    int32_t *sel_idx, void *k_draft, void *v_draft, int draft_cap,
                                    int32_t *draft_len, cudaStream_t stream) {
  StreamParams p;
  p.Hkv = Hkv;
  p.kv_cap = kv_cap;
  p.sink = sink;
  p.K = K;
  p.draft_cap = draft_cap;
  p.row_bytes = D * esz;
  p.bstride = bstride * esz;
  p.hstride = hstride * esz;
  streaming_select_kernel<<<B * Hkv, 256, 0, stream>>>(
      static_cast<const unsigned char *>(k), static_cast<const unsigned char *>(v), kv_len, p, sel_idx,
      static_cast<unsigned char *>(k_draft), static_cast<unsigned char *>(v_draft), draft_len);
  return cudaGetLastError();
}

}  // namespace mgd
