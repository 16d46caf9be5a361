// Cache bookkeeping after a verification round: keep the accepted rows, roll
// back the rejected ones, and append the kept rows to the draft cache.
//
// "Wann beschleunigt spekulatives Decoding das LLM-Serving?", "Eine
// Verifizierungsrunde verstehen": candidates after the first rejection are
// discarded.  MagicDec notes, appendix A.1: the draft reads the compressed KV
// built at prefill, so the tokens committed since then are appended to it.
// Reading (no layout on the pages): the T = gamma + 1 verify rows sit at
// kv_len - T .. kv_len - 1 (last committed token, then the gamma drafts);
// with n accepted, rows 0..n are kept (kv_len -= gamma - n) and copied to the
// draft cache at draft_len .. draft_len + n (draft_len += n + 1).
//
// One launch, one CTA per sequence: the CTA reads its sequence's lengths,
// copies the kept K and V rows of every KV head (16-byte vectors), and only
// then rewrites those two lengths, so no CTA reads a length another CTA is
// updating.  The workspace header resets itself at the end of the call (no
// clearing launch): the last CTA to check in leaves it ready for the next call.
#include "common.cuh"

namespace mgd {
namespace {

struct CommitParams {
  int B, gamma, Hkv, kv_cap, draft_cap, row_bytes;
  int64_t kv_bstride, kv_hstride, d_bstride, d_hstride;  // bytes
};

__device__ __forceinline__ bool commit_valid(int n, int L, int dl, const CommitParams &p) {
  return n >= 0 && n <= p.gamma && L >= p.gamma + 1 && L <= p.kv_cap && dl >= 0 && dl + n + 1 <= p.draft_cap;
}

__global__ void __launch_bounds__(256)
    commit_kernel(const int32_t *__restrict__ num_accepted, int32_t *__restrict__ kv_len,
                  int32_t *__restrict__ draft_len, const unsigned char *__restrict__ k,
                  const unsigned char *__restrict__ v, unsigned char *__restrict__ kd, unsigned char *__restrict__ vd,
                  CommitParams p, WsHeader *hdr) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x;
  const int n = num_accepted[b], L = kv_len[b], dl = draft_len[b];
  const bool ok = commit_valid(n, L, dl, p);
  if (ok) {
    const int first = L - p.gamma - 1;
    const int vecs = p.row_bytes / 16;
    const int per_head = (n + 1) * vecs;
    for (int i = threadIdx.x; i < p.Hkv * per_head; i += blockDim.x) {
      const int h = i / per_head, r = i - h * per_head;
      const int64_t off = static_cast<int64_t>(r / vecs) * p.row_bytes + (r % vecs) * 16;
      const int64_t src = b * p.kv_bstride + h * p.kv_hstride + static_cast<int64_t>(first) * p.row_bytes + off;
      const int64_t dst = b * p.d_bstride + h * p.d_hstride + static_cast<int64_t>(dl) * p.row_bytes + off;
      *reinterpret_cast<uint4 *>(kd + dst) = *reinterpret_cast<const uint4 *>(k + src);
      *reinterpret_cast<uint4 *>(vd + dst) = *reinterpret_cast<const uint4 *>(v + src);
    }
  }
  __syncthreads();  // every thread has read the lengths above before they change
  if (threadIdx.x == 0) {
    if (ok) {
      kv_len[b] = L - (p.gamma - n);
      draft_len[b] = dl + n + 1;
    } else {
      raise_error_sr(hdr, 0x10u);
    }
    call_check_in(hdr, gridDim.x, blockIdx.x, 0u, 0u);
  }
}

}  // namespace

cudaError_t launch_commit(const int32_t *num_accepted, int B, int gamma, int Hkv, int D, int esz, int32_t *kv_len,
                          const void *k, const void *v, int kv_cap, int64_t kv_bstride, int64_t kv_hstride,
                          void *k_draft, void *v_draft, int draft_cap, int64_t d_bstride, int64_t d_hstride,
                          int32_t *draft_len, void *ws, cudaStream_t stream) {
  CommitParams p;
  p.B = B;
  p.gamma = gamma;
  p.Hkv = Hkv;
  p.kv_cap = kv_cap;
  p.draft_cap = draft_cap;
  p.row_bytes = D * esz;
  p.kv_bstride = kv_bstride * esz;
  p.kv_hstride = kv_hstride * esz;
  p.d_bstride = d_bstride * esz;
  p.d_hstride = d_hstride * esz;
  return launch_pdl(commit_kernel, dim3(B), dim3(256), 0, stream, num_accepted, kv_len, draft_len,
                    static_cast<const unsigned char *>(k), static_cast<const unsigned char *>(v),
                    static_cast<unsigned char *>(k_draft), static_cast<unsigned char *>(v_draft), p,
                    static_cast<WsHeader *>(ws));
}

}  // namespace mgd
