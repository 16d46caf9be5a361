// SnapKV-style static selection of the draft KV cache.
//
// MagicDec notes, section 4.4: static selectors (SnapKV named) gather the
// sparse draft KV once, so drafting pays no per-token search; appendix A.1:
// this compressed KV is built at prefill and reused by every draft step; the
// quick-read summary gives its size as the draft budget K.  The pages do not
// define SnapKV itself; the steps computed here are the plain reading:
//   1. the last W positions are the observation window; each window query
//      attends causally and its softmax probabilities are summed over the W
//      window rows and the G query heads of a KV head, per prefix key;
//   2. max-pool of the scores along the sequence (odd kernel, stride 1);
//   3. the top K_eff - W prefix positions (ties -> lower position) plus the W
//      window positions, K_eff = min(K, L), kept in ascending order;
//   4. the kept K and V rows are gathered into the compacted draft cache.
//
// Kernels:
//   snap_score_tc<PASS>  bf16 tensor-core scoring, one CTA per (sequence, KV
//                        head, row group, key chunk); K tiles arrive through
//                        TMA; pass 1 computes each window row's log-sum-exp,
//                        pass 2 sums the probabilities per prefix key;
//   snap_score_kr<PASS>  the same two passes for windows of <= 32 rows, with
//                        the keys of a tile spread over the warps;
//   snap_score_simt      the same two passes on CUDA cores (float32 inputs);
//   snap_select          max-pool, 3-pass radix select of the K_eff-W-th
//                        largest pooled score, ordered compaction, gather.
// The 128-row bf16 windows at D = 128 (W = 32, G = 4) are scored instead by the
// one-read tcgen05 kernel of snap_tc05.cu (both passes in one launch).
#include <algorithm>

#include "common.cuh"

namespace mgd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kScoreStages = 4;
constexpr int kScoreThreads = 160;  // 4 consumer warps + 1 producer warp
constexpr int kRowsPerCta = 128;    // window rows (w, g) scored per CTA
constexpr int kBoxBytes = 64 * 128;

struct SnapK {
  int W, G, Hq, Hkv, rows, RG, C, nchunk, kv_cap, lrows;
  float sl2;
  size_t off_part, off_scores, off_logits;
};

template <int D>
struct ScoreLayout {
  static constexpr int kBoxes = D / 64;
  static constexpr int kStageBytes = kBoxes * kBoxBytes;
  static constexpr int off_lse = kScoreStages * kStageBytes;  // float [128]
  static constexpr int off_cs = off_lse + kRowsPerCta * 4;     // float [4][64]
  static constexpr int off_bar = off_cs + 4 * 64 * 4;          // uint64 full[], empty[]
  static constexpr int bytes = off_bar + 2 * kScoreStages * 8;
  static constexpr int alloc = bytes + 1024;
};

template <int D, int PASS>
__global__ void __launch_bounds__(kScoreThreads, 2)
    snap_score_tc(const __grid_constant__ CUtensorMap kmap, const __nv_bfloat16 *__restrict__ qw,
                  const int32_t *__restrict__ kv_len, unsigned char *__restrict__ ws, SnapK p) {
  using Lay = ScoreLayout<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *sm_lse = reinterpret_cast<float *>(smem + Lay::off_lse);
  float *sm_cs = reinterpret_cast<float *>(smem + Lay::off_cs);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::off_bar);
  uint64_t *empty = full + kScoreStages;
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  float2 *part = reinterpret_cast<float2 *>(ws + p.off_part);
  float *scores = reinterpret_cast<float *>(ws + p.off_scores);

  const int unit = blockIdx.x;
  const int chunk = unit % p.nchunk;
  const int prg = unit / p.nchunk;
  const int rg = prg % p.RG;
  const int pair = prg / p.RG;
  const int hkv = pair % p.Hkv;
  const int b = pair / p.Hkv;
  const int L = kv_len[b];
  if (L < p.W || L > p.kv_cap) {
    if (threadIdx.x == 0 && chunk == 0 && rg == 0 && hkv == 0) raise_error_sr(hdr, 0x2u);
    return;
  }
  const int kend = (PASS == 1) ? L : L - p.W;
  const int start = chunk * p.C;
  if (start >= kend) return;
  const int end = min(start + p.C, kend);
  const int ntiles = (end - start + 63) / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kScoreStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 4) {  // producer
    if (lane != 0) return;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (!mbar_wait(&empty[stage], phase ^ 1u)) {
        raise_error_sr(hdr, 0x8u);
        for (int s = 0; s < kScoreStages; ++s) mbar_wait(&full[s], phase);
        return;
      }
      mbar_arrive_expect_tx(&full[stage], Lay::kStageBytes);
#pragma unroll
      for (int h = 0; h < Lay::kBoxes; ++h)
        tma_load_4d(smem + stage * Lay::kStageBytes + h * kBoxBytes, &kmap, &full[stage], h * 64, start + 64 * t,
                    hkv, b);
      if (++stage == kScoreStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    return;
  }

  const int gid = lane >> 2, tig = lane & 3;
  constexpr int KK = D / 16;
  // ---- query fragments: A operand rows (mt, half) -> local row warp*32 + mt*16 + half*8 + gid
  uint32_t qa[2][KK][4];
  int pos[2][2];
  float lr[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = rg * kRowsPerCta + warp * 32 + mt * 16 + hf * 8 + gid;
      pos[mt][hf] = -1;
      const __nv_bfloat16 *qr = nullptr;
      if (r < p.rows) {
        const int w = r / p.G, g = r % p.G;
        pos[mt][hf] = L - p.W + w;
        qr = qw + ((static_cast<size_t>(b) * p.W + w) * p.Hq + hkv * p.G + g) * D;
      }
#pragma unroll
      for (int kk = 0; kk < KK; ++kk) {
        const uint32_t x0 = qr ? *reinterpret_cast<const uint32_t *>(qr + 16 * kk + 2 * tig) : 0u;
        const uint32_t x1 = qr ? *reinterpret_cast<const uint32_t *>(qr + 16 * kk + 8 + 2 * tig) : 0u;
        qa[mt][kk][hf] = x0;      // a0 (row gid) / a1 (row gid+8)
        qa[mt][kk][2 + hf] = x1;  // a2 / a3: columns +8
      }
    }
  }
  float m_run[2][2], l_run[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      m_run[mt][hf] = -INFINITY;
      l_run[mt][hf] = 0.f;
    }

  if (PASS == 2) {
    // log2-sum-exp of every window row from the pass-1 partials of all chunks
    const int nch1 = (L + p.C - 1) / p.C;
    if (threadIdx.x < kRowsPerCta) {
      const int rl = threadIdx.x;
      const int r = rg * kRowsPerCta + rl;
      float v = INFINITY;  // padding rows: probability 0
      if (r < p.rows) {
        const float2 *pp = part + (static_cast<size_t>(pair * p.RG + rg) * p.nchunk) * kRowsPerCta + rl;
        float M = -INFINITY;
        for (int c = 0; c < nch1; ++c) M = fmaxf(M, pp[c * kRowsPerCta].x);
        float S = 0.f;
        for (int c = 0; c < nch1; ++c) {
          const float2 x = pp[c * kRowsPerCta];
          if (x.y > 0.f) S += x.y * exp2f(x.x - M);
        }
        v = M + log2f(S);
      }
      sm_lse[rl] = v;
    }
    named_bar(1, 128);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) lr[mt][hf] = sm_lse[warp * 32 + mt * 16 + hf * 8 + gid];
  }

  int stage = 0;
  uint32_t phase = 0;
  for (int t = 0; t < ntiles; ++t) {
    if (!mbar_wait(&full[stage], phase)) {
      raise_error_sr(hdr, 0x8u);
      return;
    }
    const int kt0 = start + 64 * t;
    const uint32_t kbase = smem_addr(smem + stage * Lay::kStageBytes);
    float s[2][8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[mt][nt][c] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
      const int d = 16 * kk + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = 16 * np + (lane & 7) + 8 * (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + (d >> 6) * kBoxBytes + swz128(key, (d & 63) >> 3), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma_bf16_16816(s[mt][2 * np], qa[mt][kk][0], qa[mt][kk][1], qa[mt][kk][2], qa[mt][kk][3], b0, b1);
          mma_bf16_16816(s[mt][2 * np + 1], qa[mt][kk][0], qa[mt][kk][1], qa[mt][kk][2], qa[mt][kk][3], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == kScoreStages) {
      stage = 0;
      phase ^= 1u;
    }

    if (PASS == 1) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          float mx = -INFINITY;
#pragma unroll
          for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int key = kt0 + 8 * nt + 2 * tig + e;
              float v = s[mt][nt][2 * hf + e] * p.sl2;
              if (key > pos[mt][hf]) v = -INFINITY;
              s[mt][nt][2 * hf + e] = v;
              mx = fmaxf(mx, v);
            }
          mx = warp_max_xor(mx, 1, 2);
          const float mn = fmaxf(m_run[mt][hf], mx);
          const float mu = (mn == -INFINITY) ? 0.f : mn;
          float acc = 0.f;
#pragma unroll
          for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) acc += exp2f(s[mt][nt][2 * hf + e] - mu);
          l_run[mt][hf] = l_run[mt][hf] * exp2f(m_run[mt][hf] - mu) + acc;
          m_run[mt][hf] = mn;
        }
    } else {
      // column sums of exp2(s - lse) over this thread's 4 rows, then over the 8 row groups of the warp
      float cs[8][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float acc = 0.f;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) acc += exp2f(s[mt][nt][2 * hf + e] * p.sl2 - lr[mt][hf]);
          cs[nt][e] = warp_sum_xor(acc, 4, 16);
        }
      if (gid == 0) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) sm_cs[warp * 64 + 8 * nt + 2 * tig + e] = cs[nt][e];
      }
      named_bar(1, 128);
      if (threadIdx.x < 64) {
        const int key = kt0 + threadIdx.x;
        if (key < end) {
          const float v = sm_cs[threadIdx.x] + sm_cs[64 + threadIdx.x] + sm_cs[128 + threadIdx.x] +
                          sm_cs[192 + threadIdx.x];
          float *dst = scores + (static_cast<size_t>(b) * p.Hkv + hkv) * p.kv_cap + key;
          if (p.RG == 1)
            *dst = v;
          else
            atomicAdd(dst, v);
        }
      }
      named_bar(1, 128);
    }
  }

  if (PASS == 1) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const float l = warp_sum_xor(l_run[mt][hf], 1, 2);
        if (tig == 0) {
          const int rl = warp * 32 + mt * 16 + hf * 8 + gid;
          part[(static_cast<size_t>(pair * p.RG + rg) * p.nchunk + chunk) * kRowsPerCta + rl] =
              make_float2(m_run[mt][hf], l);
        }
      }
  }
}

// ---------------------------------------------------------------- small windows
// Windows of at most 32 rows (W * G <= 32, e.g. the draft query alone as a
// one-row window): S^T = K Qw^T with the keys on the M side, so each consumer
// warp takes 16 keys of every 64-key tile for all rows (NT n8 row tiles) and a
// short window costs the same per key as a long one.  Pass 1: per row, an
// online (max, sum) over the keys (a max across the 8 key lanes, sums reduced
// at the end); pass 2: per key, the sum over rows of exp2(s - lse_row) (a sum
// across the 4 row lanes).
template <int D>
struct KrLayout {
  static constexpr int kBoxes = D / 64;
  static constexpr int kStageBytes = kBoxes * kBoxBytes;  // 64 keys
  static constexpr int kQStride = D + 8;                  // bf16 per staged row (bank-conflict padding)
  static constexpr int off_q = kScoreStages * kStageBytes;
  static constexpr int off_lse = off_q + 32 * kQStride * 2;  // float [32]
  static constexpr int off_red = off_lse + 32 * 4;           // float2 [4][32]
  static constexpr int off_bar = off_red + 4 * 32 * 8;
  static constexpr int bytes = off_bar + 2 * kScoreStages * 8;
  static constexpr int alloc = bytes + 1024;
};

template <int D, int NT, int PASS>
__global__ void __launch_bounds__(kScoreThreads, 2)
    snap_score_kr(const __grid_constant__ CUtensorMap kmap, const __nv_bfloat16 *__restrict__ qw,
                  const int32_t *__restrict__ kv_len, unsigned char *__restrict__ ws, SnapK p) {
  using Lay = KrLayout<D>;
  constexpr int KK = D / 16;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem + Lay::off_q);
  float *sm_lse = reinterpret_cast<float *>(smem + Lay::off_lse);
  float2 *sm_red = reinterpret_cast<float2 *>(smem + Lay::off_red);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::off_bar);
  uint64_t *empty = full + kScoreStages;
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  float2 *part = reinterpret_cast<float2 *>(ws + p.off_part);
  float *scores = reinterpret_cast<float *>(ws + p.off_scores);

  const int chunk = blockIdx.x % p.nchunk;
  const int pair = blockIdx.x / p.nchunk;  // one row group (rows <= 32)
  const int hkv = pair % p.Hkv;
  const int b = pair / p.Hkv;
  const int L = kv_len[b];
  if (L < p.W || L > p.kv_cap) {
    if (threadIdx.x == 0 && chunk == 0 && hkv == 0) raise_error_sr(hdr, 0x2u);
    return;
  }
  const int kend = (PASS == 1) ? L : L - p.W;
  const int start = chunk * p.C;
  if (start >= kend) return;
  const int end = min(start + p.C, kend);
  const int ntiles = (end - start + 63) / 64;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kScoreStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    fence_mbar_init();
  }
  // window rows r = w * G + g staged in shared memory (zero rows past p.rows)
  for (int i = threadIdx.x; i < 32 * (D / 8); i += kScoreThreads) {
    const int r = i / (D / 8), c = i % (D / 8);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (r < p.rows) {
      const int w = r / p.G, g = r % p.G;
      x = *reinterpret_cast<const uint4 *>(qw + ((static_cast<size_t>(b) * p.W + w) * p.Hq + hkv * p.G + g) * D + 8 * c);
    }
    *reinterpret_cast<uint4 *>(sQ + r * Lay::kQStride + 8 * c) = x;
  }
  if (PASS == 2 && threadIdx.x < 32) {  // log2-sum-exp of every row from the pass-1 partials
    const int r = threadIdx.x;
    float v = INFINITY;  // padding rows: probability 0
    if (r < p.rows) {
      const int nch1 = (L + p.C - 1) / p.C;
      const float2 *pp = part + static_cast<size_t>(pair) * p.nchunk * kRowsPerCta + r;
      float M = -INFINITY;
      for (int c = 0; c < nch1; ++c) M = fmaxf(M, pp[c * kRowsPerCta].x);
      float S = 0.f;
      for (int c = 0; c < nch1; ++c) {
        const float2 x = pp[c * kRowsPerCta];
        if (x.y > 0.f) S += x.y * exp2f(x.x - M);
      }
      v = M + log2f(S);
    }
    sm_lse[r] = v;
  }
  __syncthreads();

  if (warp == 4) {  // producer
    if (lane != 0) return;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (!mbar_wait(&empty[stage], phase ^ 1u)) {
        raise_error_sr(hdr, 0x8u);
        return;
      }
      mbar_arrive_expect_tx(&full[stage], Lay::kStageBytes);
#pragma unroll
      for (int h = 0; h < Lay::kBoxes; ++h)
        tma_load_4d(smem + stage * Lay::kStageBytes + h * kBoxBytes, &kmap, &full[stage], h * 64, start + 64 * t,
                    hkv, b);
      if (++stage == kScoreStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    return;
  }

  const int gid = lane >> 2, tig = lane & 3;
  int lim[NT][2];      // pass 1: last key row (j, e) sees; -1 for padding rows
  float lr[NT][2];     // pass 2: log2-sum-exp of row (j, e)
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 8 * j + 2 * tig + e;
      lim[j][e] = (r < p.rows) ? (L - p.W + r / p.G) : -1;
      lr[j][e] = (PASS == 2) ? sm_lse[r] : 0.f;
      m_run[j][e] = -INFINITY;
      l_run[j][e] = 0.f;
    }
  const uint32_t qaddr = smem_addr(sQ) + 2u * (((lane & 7) + 8 * (lane >> 4)) * Lay::kQStride + 8 * ((lane >> 3) & 1));
  int stage = 0;
  uint32_t phase = 0;
  for (int t = 0; t < ntiles; ++t) {
    if (!mbar_wait(&full[stage], phase)) {
      raise_error_sr(hdr, 0x8u);
      break;  // still meets the end-of-unit barrier below
    }
    const uint32_t kbase = smem_addr(smem + stage * Lay::kStageBytes);
    const int key0 = start + 64 * t + warp * 16;
    float s[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[j][c] = 0.f;
    const int kr = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
      const int d = 16 * kk + 8 * (lane >> 4);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kbase + (d >> 6) * kBoxBytes + swz128(kr, (d & 63) >> 3), a0, a1, a2, a3);
#pragma unroll
      for (int jp = 0; jp < (NT + 1) / 2; ++jp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(qaddr + 2u * (16 * jp * Lay::kQStride + 16 * kk), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * jp], a0, a1, a2, a3, b0, b1);
        if (2 * jp + 1 < NT) mma_bf16_16816(s[2 * jp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == kScoreStages) {
      stage = 0;
      phase ^= 1u;
    }
    const int k_lo = key0 + gid, k_hi = key0 + gid + 8;  // accumulator rows gid / gid + 8
    if (PASS == 1 && NT == 1 && p.lrows > 0 && 2 * tig < p.lrows) {
      // keep this key's logits (rows 2 tig, 2 tig + 1) for the key sums; every
      // window row sees every prefix key, so no mask applies below L - W
      float *lg = reinterpret_cast<float *>(ws + p.off_logits) + static_cast<size_t>(pair) * p.kv_cap * p.lrows;
      const int nprefix = min(end, L - p.W);
      if (k_lo < nprefix)
        *reinterpret_cast<float2 *>(lg + static_cast<size_t>(k_lo) * p.lrows + 2 * tig) =
            make_float2(s[0][0] * p.sl2, s[0][1] * p.sl2);
      if (k_hi < nprefix)
        *reinterpret_cast<float2 *>(lg + static_cast<size_t>(k_hi) * p.lrows + 2 * tig) =
            make_float2(s[0][2] * p.sl2, s[0][3] * p.sl2);
    }
    if (PASS == 1) {
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v0 = (k_lo <= lim[j][e]) ? s[j][e] * p.sl2 : -INFINITY;
          const float v1 = (k_hi <= lim[j][e]) ? s[j][2 + e] * p.sl2 : -INFINITY;
          const float mx = warp_max_xor(fmaxf(v0, v1), 4, 16);
          const float mn = fmaxf(m_run[j][e], mx);
          const float mu = (mn == -INFINITY) ? 0.f : mn;
          l_run[j][e] = l_run[j][e] * ex2(m_run[j][e] - mu) + ex2(v0 - mu) + ex2(v1 - mu);
          m_run[j][e] = mn;
        }
    } else {
      float a_lo = 0.f, a_hi = 0.f;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          a_lo += ex2(s[j][e] * p.sl2 - lr[j][e]);
          a_hi += ex2(s[j][2 + e] * p.sl2 - lr[j][e]);
        }
      a_lo = warp_sum_xor(a_lo, 1, 2);
      a_hi = warp_sum_xor(a_hi, 1, 2);
      if (tig == 0) {
        float *dst = scores + static_cast<size_t>(pair) * p.kv_cap;
        if (k_lo < end) dst[k_lo] = a_lo;
        if (k_hi < end) dst[k_hi] = a_hi;
      }
    }
  }

  if (PASS == 1) {
    // (max, sum) of each row over this warp's keys, then over the 4 warps
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float l = warp_sum_xor(l_run[j][e], 4, 16);
        if (gid == 0) sm_red[warp * 32 + 8 * j + 2 * tig + e] = make_float2(m_run[j][e], l);
      }
    named_bar(1, 128);
    if (threadIdx.x < 8 * NT) {
      const int r = threadIdx.x;
      float M = -INFINITY;
      for (int w = 0; w < 4; ++w) M = fmaxf(M, sm_red[w * 32 + r].x);
      const float mu = (M == -INFINITY) ? 0.f : M;
      float S = 0.f;
      for (int w = 0; w < 4; ++w) {
        const float2 x = sm_red[w * 32 + r];
        if (x.y > 0.f) S += x.y * exp2f(x.x - mu);
      }
      part[(static_cast<size_t>(pair) * p.nchunk + chunk) * kRowsPerCta + r] = make_float2(M, S);
    }
  }
}

// Key sums from the logits pass 1 kept (windows of <= 8 rows): for each prefix
// key j of the chunk, sum over the rows of exp2(logit - lse_row), lse from the
// pass-1 partials.  Streams R floats per key instead of reading K again.
template <int R>
__global__ void __launch_bounds__(256)
    snap_logit_sum(const int32_t *__restrict__ kv_len, unsigned char *__restrict__ ws, SnapK p) {
  __shared__ float sm_nl[R];
  const int chunk = blockIdx.x % p.nchunk;
  const int pair = blockIdx.x / p.nchunk;
  const int b = pair / p.Hkv;
  const int L = kv_len[b];
  if (L < p.W || L > p.kv_cap) return;  // raised by pass 1
  const int start = chunk * p.C, end = min(start + p.C, L - p.W);
  if (start >= end) return;
  if (threadIdx.x < R) {  // minus the log2-sum-exp of every row (padding rows contribute 0)
    const int r = threadIdx.x;
    float v = -INFINITY;
    if (r < p.rows) {
      const int nch1 = (L + p.C - 1) / p.C;
      const float2 *pp = reinterpret_cast<const float2 *>(ws + p.off_part) + static_cast<size_t>(pair) * p.nchunk * kRowsPerCta + r;
      float M = -INFINITY;
      for (int c = 0; c < nch1; ++c) M = fmaxf(M, pp[c * kRowsPerCta].x);
      float S = 0.f;
      for (int c = 0; c < nch1; ++c) {
        const float2 x = pp[c * kRowsPerCta];
        if (x.y > 0.f) S += x.y * exp2f(x.x - M);
      }
      v = -(M + log2f(S));
    }
    sm_nl[r] = v;
  }
  __syncthreads();
  float nl[R];
#pragma unroll
  for (int r = 0; r < R; ++r) nl[r] = sm_nl[r];
  const float4 *lg = reinterpret_cast<const float4 *>(ws + p.off_logits) + static_cast<size_t>(pair) * p.kv_cap * (R / 4);
  float *dst = reinterpret_cast<float *>(ws + p.off_scores) + static_cast<size_t>(pair) * p.kv_cap;
  constexpr int kU = 4;  // keys in flight per thread
  for (int j0 = start + threadIdx.x; j0 < end; j0 += kU * 256) {
    float4 x[kU][R / 4];
#pragma unroll
    for (int u = 0; u < kU; ++u)
#pragma unroll
      for (int h = 0; h < R / 4; ++h) {
        const int j = j0 + u * 256;
        x[u][h] = (j < end) ? lg[static_cast<size_t>(j) * (R / 4) + h] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = j0 + u * 256;
      if (j < end) {
        float acc = 0.f;
#pragma unroll
        for (int h = 0; h < R / 4; ++h)
          acc += (ex2(x[u][h].x + nl[4 * h]) + ex2(x[u][h].y + nl[4 * h + 1])) +
                 (ex2(x[u][h].z + nl[4 * h + 2]) + ex2(x[u][h].w + nl[4 * h + 3]));
        dst[j] = acc;
      }
    }
  }
}

// ---------------------------------------------------------------- CUDA-core scoring
template <typename Tin, int D>
__global__ void __launch_bounds__(256)
    snap_score_simt(const Tin *__restrict__ qw, const Tin *__restrict__ k, const int32_t *__restrict__ kv_len,
                    int64_t bstride, int64_t hstride, unsigned char *__restrict__ ws, SnapK p) {
  extern __shared__ float sm_lse2[];  // [rows]
  __shared__ float red[2][8];
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  float *scores = reinterpret_cast<float *>(ws + p.off_scores);
  const int b = blockIdx.x / p.Hkv, hkv = blockIdx.x % p.Hkv;
  const int L = kv_len[b];
  if (L < p.W || L > p.kv_cap) {
    if (threadIdx.x == 0 && hkv == 0) raise_error_sr(hdr, 0x2u);
    return;
  }
  const Tin *kb = k + b * bstride + hkv * hstride;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = 0; r < p.rows; ++r) {
    const int w = r / p.G, g = r % p.G;
    const int posn = L - p.W + w;
    const Tin *qr = qw + ((static_cast<size_t>(b) * p.W + w) * p.Hq + hkv * p.G + g) * D;
    float m = -INFINITY, l = 0.f;
    for (int j = threadIdx.x; j <= posn; j += 256) {
      float dot = 0.f;
      for (int d = 0; d < D; ++d) dot = fmaf(to_f32(qr[d]), to_f32(kb[static_cast<size_t>(j) * D + d]), dot);
      const float v = dot * p.sl2;
      if (v > m) {
        l = l * exp2f(m - v) + 1.f;
        m = v;
      } else {
        l += exp2f(v - m);
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), l2 = __shfl_xor_sync(0xffffffffu, l, o);
      const float mn = fmaxf(m, m2);
      const float mu = (mn == -INFINITY) ? 0.f : mn;
      l = l * exp2f(m - mu) + l2 * exp2f(m2 - mu);
      m = mn;
    }
    if (lane == 0) {
      red[0][warp] = m;
      red[1][warp] = l;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float M = -INFINITY;
      for (int i = 0; i < 8; ++i) M = fmaxf(M, red[0][i]);
      float S = 0.f;
      for (int i = 0; i < 8; ++i) S += red[1][i] * exp2f(red[0][i] - M);
      sm_lse2[r] = M + log2f(S);
    }
    __syncthreads();
  }
  const int n = L - p.W;
  for (int j = threadIdx.x; j < n; j += 256) {
    float acc = 0.f;
    for (int r = 0; r < p.rows; ++r) {
      const int w = r / p.G, g = r % p.G;
      const Tin *qr = qw + ((static_cast<size_t>(b) * p.W + w) * p.Hq + hkv * p.G + g) * D;
      float dot = 0.f;
      for (int d = 0; d < D; ++d) dot = fmaf(to_f32(qr[d]), to_f32(kb[static_cast<size_t>(j) * D + d]), dot);
      acc += exp2f(dot * p.sl2 - sm_lse2[r]);
    }
    scores[(static_cast<size_t>(b) * p.Hkv + hkv) * p.kv_cap + j] = acc;
  }
}

// ---------------------------------------------------------------- select + gather
constexpr int kSelThreads = 1024;
constexpr int kPoolTile = 4096;     // scores staged in shared memory per pooling step
constexpr int kPoolHalo = 64;       // pool radius up to which the staged path is used
constexpr int kStageLoads = (kPoolTile + 2 * kPoolHalo + kSelThreads - 1) / kSelThreads;
constexpr int kSweepLoads = 8;      // pooled values in flight per thread in a radix pass
constexpr int kCompactLoads = 4;    // 32-position rows in flight per warp in the compaction

struct SelParams {
  int Hkv, W, pool, K, kv_cap, draft_cap, row_bytes;
  int64_t bstride_bytes, hstride_bytes;
  const int32_t *Kb;  // per-sequence budgets (device), or null for K everywhere
  size_t off_cnt;     // the one-read scorer's per-pair counters ([2][pairs]), put back to zero here
  unsigned expect_claims;  // successful work claims the scorer made from a ready header
};

// Exclusive block scan of one unsigned per thread (kSelThreads threads); returns
// the prefix and writes the block total to *total.
__device__ unsigned block_excl_scan(unsigned v, unsigned *sm_warp, unsigned *total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned w = sm_warp[lane];
    unsigned s = w;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sm_warp[lane] = s - w;  // exclusive per-warp offsets
    if (lane == 31) sm_warp[32] = s;
  }
  __syncthreads();
  const unsigned r = sm_warp[warp] + x - v;
  *total = sm_warp[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ void select_pair(const unsigned char *__restrict__ k, const unsigned char *__restrict__ v,
                                            const int32_t *__restrict__ kv_len, const SelParams &sp,
                                            int32_t *__restrict__ sel_idx, unsigned char *__restrict__ k_draft,
                                            unsigned char *__restrict__ v_draft, int32_t *__restrict__ draft_len,
                                            float *__restrict__ scores_out, unsigned char *__restrict__ ws,
                                            size_t off_scores, size_t off_pooled) {
  __shared__ unsigned hist[2048];
  __shared__ unsigned sm_warp[33];
  __shared__ unsigned s_bin, s_above;
  __shared__ float stage[kPoolTile + 2 * kPoolHalo];  // scores of one pooling tile and its halo
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  const int b = blockIdx.x / sp.Hkv, hkv = blockIdx.x % sp.Hkv;
  const int L = kv_len[b];
  const int Kb = sp.Kb ? sp.Kb[b] : sp.K;  // this sequence's budget (MagicDec notes, section 4.3)
  const size_t pr = static_cast<size_t>(b) * sp.Hkv + hkv;
  int32_t *sel = sel_idx + pr * sp.draft_cap;
  if (L < sp.W || L > sp.kv_cap || Kb < sp.W || Kb > sp.draft_cap) {
    for (int i = threadIdx.x; i < sp.draft_cap; i += kSelThreads) sel[i] = -1;
    if (threadIdx.x == 0 && hkv == 0) {
      draft_len[b] = 0;
      raise_error_sr(hdr, 0x2u);
    }
    return;
  }
  const float *s = reinterpret_cast<const float *>(ws + off_scores) + pr * sp.kv_cap;
  float *pooled = reinterpret_cast<float *>(ws + off_pooled) + pr * sp.kv_cap;
  const int n = L - sp.W;
  const int Keff = min(Kb, L);
  const int ktop = Keff - sp.W;
  const int r = sp.pool / 2;

  const bool partial = (ktop > 0 && ktop < n);
  // ---- 1. max-pool (and the optional copy out), with the first radix
  //         pass's histogram of the top 11 bits
  for (int i = threadIdx.x; i < 2048; i += kSelThreads) hist[i] = 0u;
  auto emit = [&](int j, float m) {
    pooled[j] = m;
    if (scores_out) scores_out[pr * sp.kv_cap + j] = m;
    if (partial) atomicAdd(&hist[__float_as_uint(m) >> 21], 1u);
  };
  if (r <= kPoolHalo) {
    // tiles of kPoolTile scores staged in shared memory with their halo (every
    // thread's loads issued together), positions outside the prefix as -inf; the
    // next tile's loads are in flight while the current tile is pooled
    float x[kStageLoads];
    auto load_tile = [&](int t0) {
      const int cnt = min(kPoolTile, n - t0) + 2 * r;
#pragma unroll
      for (int u = 0; u < kStageLoads; ++u) {
        const int i = threadIdx.x + u * kSelThreads, t = t0 - r + i;
        x[u] = (i < cnt && t >= 0 && t < n) ? s[t] : -INFINITY;
      }
    };
    if (n > 0) load_tile(0);
    for (int t0 = 0; t0 < n; t0 += kPoolTile) {
      const int len = min(kPoolTile, n - t0), cnt = len + 2 * r;
      __syncthreads();  // the previous tile's readers are done
#pragma unroll
      for (int u = 0; u < kStageLoads; ++u)
        if (threadIdx.x + u * kSelThreads < cnt) stage[threadIdx.x + u * kSelThreads] = x[u];
      __syncthreads();
      if (t0 + kPoolTile < n) load_tile(t0 + kPoolTile);
      for (int i = threadIdx.x; i < len; i += kSelThreads) {
        float m = stage[i];
        for (int o = 1; o <= 2 * r; ++o) m = fmaxf(m, stage[i + o]);
        emit(t0 + i, m);
      }
    }
  } else {
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += kSelThreads) {
      float m = s[j];
      const int lo = max(0, j - r), hi = min(n - 1, j + r);
      for (int t = lo; t <= hi; ++t) m = fmaxf(m, s[t]);
      emit(j, m);
    }
  }
  __syncthreads();

  // ---- 2. radix select of the ktop-th largest pooled value (scores are >= 0,
  //         so their IEEE bit patterns order like the values)
  unsigned prefix = 0u, mask = 0u, krem = static_cast<unsigned>(ktop);
  if (partial) {
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = (pass == 0) ? 21 : (pass == 1) ? 10 : 0;
      const int nb = (pass == 2) ? 1024 : 2048;
      if (pass > 0) {  // pass 0's histogram came with the pooling
        for (int i = threadIdx.x; i < nb; i += kSelThreads) hist[i] = 0u;
        __syncthreads();
        for (int j0 = threadIdx.x; j0 < n; j0 += kSweepLoads * kSelThreads) {
          unsigned key[kSweepLoads];  // loads issued together, then counted
#pragma unroll
          for (int u = 0; u < kSweepLoads; ++u) {
            const int j = j0 + u * kSelThreads;
            key[u] = (j < n) ? __float_as_uint(pooled[j]) : 0u;
          }
#pragma unroll
          for (int u = 0; u < kSweepLoads; ++u)
            if (j0 + u * kSelThreads < n && (key[u] & mask) == prefix) atomicAdd(&hist[(key[u] >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
      }
      // bins in descending order, two per thread
      const int b_hi = nb - 1 - 2 * threadIdx.x;
      const int b_lo = b_hi - 1;
      const unsigned c_hi = (b_hi >= 0) ? hist[b_hi] : 0u;
      const unsigned c_lo = (b_lo >= 0) ? hist[b_lo] : 0u;
      if (threadIdx.x == 0) {  // set below by the one thread whose bins hold the krem-th value
        s_bin = 0u;
        s_above = 0u;
      }
      unsigned tot;
      const unsigned above = block_excl_scan(c_hi + c_lo, sm_warp, &tot);
      if (b_hi >= 0 && above < krem && krem <= above + c_hi) {
        s_bin = b_hi;
        s_above = above;
      } else if (b_lo >= 0 && above + c_hi < krem && krem <= above + c_hi + c_lo) {
        s_bin = b_lo;
        s_above = above + c_hi;
      }
      __syncthreads();
      prefix |= s_bin << shift;
      mask |= static_cast<unsigned>(nb - 1) << shift;
      krem -= s_above;
      __syncthreads();
    }
  }
  // ---- 3. ordered compaction: position of j = #(greater before j) + min(#(equal before j), krem).
  //         Each warp owns a contiguous segment, read 32 consecutive positions
  //         at a time; ballots order the positions inside a warp and one scan
  //         of the 32 warp totals orders the warps.
  const unsigned tau = prefix;
  const bool keep_all = !partial && ktop >= n;  // ktop >= n keeps the whole prefix, ktop <= 0 none of it
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int wseg = ((n + kSelThreads / 32 - 1) / (kSelThreads / 32) + 31) / 32 * 32;
  const int w0 = min(n, warp * wseg), w1 = min(n, w0 + wseg);
  // keys of positions jb + 32u + lane (u < kCompactLoads), loaded together
  auto load_keys = [&](int jb, unsigned (&key)[kCompactLoads]) {
#pragma unroll
    for (int u = 0; u < kCompactLoads; ++u) {
      const int j = jb + 32 * u + lane;
      key[u] = (partial && j < w1) ? __float_as_uint(pooled[j]) : 0u;
    }
  };
  auto classify = [&](int j, unsigned key, unsigned &gt, unsigned &eq) {
    gt = 0u;
    eq = 0u;
    if (j < w1) {
      if (partial) {
        gt = key > tau ? 1u : 0u;
        eq = key == tau ? 1u : 0u;
      } else {
        gt = keep_all ? 1u : 0u;
      }
    }
  };
  unsigned gt_cnt = 0u, eq_cnt = 0u;
  for (int jb = w0; jb < w1; jb += 32 * kCompactLoads) {
    unsigned key[kCompactLoads];
    load_keys(jb, key);
#pragma unroll
    for (int u = 0; u < kCompactLoads; ++u) {
      unsigned gt, eq;
      classify(jb + 32 * u + lane, key[u], gt, eq);
      gt_cnt += __popc(__ballot_sync(0xffffffffu, gt));
      eq_cnt += __popc(__ballot_sync(0xffffffffu, eq));
    }
  }
  if (lane == 0) {
    hist[warp] = gt_cnt;
    hist[32 + warp] = eq_cnt;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scans of the 32 warp totals
    unsigned g = hist[lane], e = hist[32 + lane];
    unsigned gs = g, es = e;
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned y1 = __shfl_up_sync(0xffffffffu, gs, o);
      const unsigned y2 = __shfl_up_sync(0xffffffffu, es, o);
      if (lane >= o) {
        gs += y1;
        es += y2;
      }
    }
    hist[64 + lane] = gs - g;
    hist[96 + lane] = es - e;
  }
  __syncthreads();
  unsigned g_before = hist[64 + warp], e_before = hist[96 + warp];
  for (int jb = w0; jb < w1; jb += 32 * kCompactLoads) {
    unsigned key[kCompactLoads];
    load_keys(jb, key);
#pragma unroll
    for (int u = 0; u < kCompactLoads; ++u) {
      const int j = jb + 32 * u + lane;
      unsigned gt, eq;
      classify(j, key[u], gt, eq);
      const unsigned gb = __ballot_sync(0xffffffffu, gt), eb = __ballot_sync(0xffffffffu, eq);
      const unsigned gpos = g_before + __popc(gb & lt_mask), epos = e_before + __popc(eb & lt_mask);
      const unsigned dst = gpos + min(epos, krem);  // < ktop whenever the counts are those of the data
      if ((gt || (eq && epos < krem)) && dst < static_cast<unsigned>(ktop)) sel[dst] = j;
      g_before += __popc(gb);
      e_before += __popc(eb);
    }
  }
  for (int w = threadIdx.x; w < sp.W; w += kSelThreads) sel[ktop + w] = n + w;
  for (int i = Keff + threadIdx.x; i < sp.draft_cap; i += kSelThreads) sel[i] = -1;
  if (threadIdx.x == 0 && hkv == 0) draft_len[b] = Keff;
  __syncthreads();

  // ---- 4. gather the kept rows (16-byte vectors)
  const int vecs = sp.row_bytes / 16;
  const unsigned char *ks = k + b * sp.bstride_bytes + hkv * sp.hstride_bytes;
  const unsigned char *vs = v + b * sp.bstride_bytes + hkv * sp.hstride_bytes;
  unsigned char *kd = k_draft + pr * sp.draft_cap * sp.row_bytes;
  unsigned char *vd = v_draft + pr * sp.draft_cap * sp.row_bytes;
  const int total = Keff * vecs;
  for (int i0 = threadIdx.x; i0 < total; i0 += 2 * kSelThreads) {  // 4 loads in flight per thread
    uint4 kx[2], vx[2];
    size_t dst[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = i0 + u * kSelThreads;
      if (i < total) {
        const int row = i / vecs, c = i % vecs;
        // kept positions lie in [0, L); the clamp only guards the reads against a selection
        // whose counts were not those of its data
        const int pos = min(max(sel[row], 0), L - 1);
        const size_t src = static_cast<size_t>(pos) * sp.row_bytes + c * 16;
        dst[u] = static_cast<size_t>(row) * sp.row_bytes + c * 16;
        kx[u] = __ldg(reinterpret_cast<const uint4 *>(ks + src));
        vx[u] = __ldg(reinterpret_cast<const uint4 *>(vs + src));
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (i0 + u * kSelThreads < total) {
        *reinterpret_cast<uint4 *>(kd + dst[u]) = kx[u];
        *reinterpret_cast<uint4 *>(vd + dst[u]) = vx[u];
      }
    }
  }
}

// Steps 2-4 of the selection for one (sequence, KV head) per CTA, and the end
// of the call: each CTA puts its pair's scorer counters back to zero and checks
// in, and the last check-in leaves the workspace header ready for the next
// call (so no clearing launch is needed ahead of a selection).
__global__ void __launch_bounds__(kSelThreads, 2)
    snap_select(const unsigned char *__restrict__ k, const unsigned char *__restrict__ v,
                const int32_t *__restrict__ kv_len, SelParams sp, int32_t *__restrict__ sel_idx,
                unsigned char *__restrict__ k_draft, unsigned char *__restrict__ v_draft,
                int32_t *__restrict__ draft_len, float *__restrict__ scores_out, unsigned char *__restrict__ ws,
                size_t off_scores, size_t off_pooled) {
  pdl_launch_dependents();
  pdl_wait();
  select_pair(k, v, kv_len, sp, sel_idx, k_draft, v_draft, draft_len, scores_out, ws, off_scores, off_pooled);
  if (threadIdx.x == 0) {
    unsigned *cnt = reinterpret_cast<unsigned *>(ws + sp.off_cnt);
    cnt[blockIdx.x] = 0u;              // slices published
    cnt[gridDim.x + blockIdx.x] = 0u;  // slices claimed
    call_check_in(reinterpret_cast<WsHeader *>(ws), gridDim.x, blockIdx.x, 0u, sp.expect_claims);
  }
}

}  // namespace

SnapPlan plan_snapkv(int B, int Hq, int Hkv, int D, int kv_cap, int W) {
  SnapPlan p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.D = D;
  p.kv_cap = kv_cap;
  p.W = W;
  p.G = Hq / Hkv;
  p.rows = p.G * W;
  p.RG = (p.rows + kRowsPerCta - 1) / kRowsPerCta;
  p.pairs = B * Hkv;
  const int slots = 2 * current_sm_count();
  int C = 4096;
  const int cmin = std::max(256, ((kv_cap + 63) / 64 + 63) / 64 * 64);
  while (C > cmin && static_cast<long long>(p.pairs) * p.RG * ((kv_cap + C - 1) / C) < 8LL * slots) C /= 2;
  if (C < cmin) C = cmin;
  if (D == 128 && p.rows == 128 && p.RG == 1) {  // the one-read tcgen05 scorer's slices
    const int per_slice = (kv_cap + kSnapMaxSlices - 1) / kSnapMaxSlices;
    C = std::max(kSnapSliceKeys, (per_slice + 127) / 128 * 128);
  }
  p.C = C;
  p.nchunk = (kv_cap + C - 1) / C;
  p.off_cnt = kAlign;  // [pairs] slices published, then [pairs] slices claimed (one-read tcgen05 scorer)
  size_t off = align_up(p.off_cnt + 2 * sizeof(unsigned) * static_cast<size_t>(p.pairs));
  p.off_part = off;
  off = align_up(off + sizeof(float2) * static_cast<size_t>(p.pairs) * p.RG * p.nchunk * kRowsPerCta);
  p.off_scores = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(p.pairs) * kv_cap);
  p.off_pooled = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(p.pairs) * kv_cap);
  // Windows of at most 8 rows (the draft query alone, for one): pass 1 keeps
  // every prefix key's logits (16 or 32 bytes a key) and the key sums are
  // taken from them, instead of a second read of K (2 * D bytes a key).
  p.lrows = (p.rows <= 4) ? 4 : (p.rows <= 8) ? 8 : 0;
  p.off_logits = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(p.pairs) * kv_cap * p.lrows);
  p.ws_bytes = off;
  return p;
}

cudaError_t launch_snapkv(const SnapPlan &p, const SnapArgs &a, int in_f32, const CUtensorMap *kmap,
                          const CUtensorMap *qmap) {
  // no clearing launch: the select kernel at the end of the call leaves the header and the
  // scorer's counters at zero for the next call (the workspace is zero-filled before first use)
  cudaError_t e = cudaSuccess;
  unsigned char *ws = static_cast<unsigned char *>(a.ws);
  const bool tc05 = !in_f32 && kmap != nullptr && qmap != nullptr && snap_tc05_eligible(p);
  SnapK kp;
  kp.W = p.W;
  kp.G = p.G;
  kp.Hq = p.Hq;
  kp.Hkv = p.Hkv;
  kp.rows = p.rows;
  kp.RG = p.RG;
  kp.C = p.C;
  kp.nchunk = p.nchunk;
  kp.kv_cap = p.kv_cap;
  kp.sl2 = a.sm_scale * kLog2e;
  kp.off_part = p.off_part;
  kp.off_scores = p.off_scores;
  kp.lrows = p.lrows;
  kp.off_logits = p.off_logits;
  if (in_f32 || kmap == nullptr) {  // float32 inputs (bf16 calls always come with the K map)
    if (!in_f32) return cudaErrorInvalidValue;
    const size_t smem = sizeof(float) * p.rows;
    if (p.D == 128)
      snap_score_simt<float, 128><<<p.pairs, 256, smem, a.stream>>>(
          static_cast<const float *>(a.q_win), static_cast<const float *>(a.k), a.kv_len, a.kv_batch_stride,
          a.kv_head_stride, ws, kp);
    else
      snap_score_simt<float, 64><<<p.pairs, 256, smem, a.stream>>>(
          static_cast<const float *>(a.q_win), static_cast<const float *>(a.k), a.kv_len, a.kv_batch_stride,
          a.kv_head_stride, ws, kp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else if (qmap != nullptr && snap_tc05_eligible(p)) {
    e = launch_snap_score_tc05(p, a, *kmap, *qmap);
    if (e != cudaSuccess) return e;
  } else if (p.rows <= 32) {
    const int units = p.pairs * p.nchunk;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q_win);
    const int nt = (p.rows <= 8) ? 1 : (p.rows <= 16) ? 2 : 4;
#define MGD_KR(DD, NTT, PP)                                                                               \
  do {                                                                                                    \
    auto kern = snap_score_kr<DD, NTT, PP>;                                                               \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KrLayout<DD>::alloc);     \
    if (e != cudaSuccess) return e;                                                                       \
    kern<<<units, kScoreThreads, KrLayout<DD>::alloc, a.stream>>>(*kmap, q, a.kv_len, ws, kp);            \
    e = cudaGetLastError();                                                                               \
    if (e != cudaSuccess) return e;                                                                       \
  } while (0)
#define MGD_KR_PASSES(DD, NTT) \
  do {                         \
    MGD_KR(DD, NTT, 1);        \
    MGD_KR(DD, NTT, 2);        \
  } while (0)
    if (nt == 1 && p.lrows > 0) {  // pass 1 keeps the logits; the key sums stream them
      if (p.D == 128) MGD_KR(128, 1, 1);
      else MGD_KR(64, 1, 1);
      if (p.lrows == 4) snap_logit_sum<4><<<units, 256, 0, a.stream>>>(a.kv_len, ws, kp);
      else snap_logit_sum<8><<<units, 256, 0, a.stream>>>(a.kv_len, ws, kp);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    } else if (p.D == 128) {
      if (nt == 1) MGD_KR_PASSES(128, 1);
      else if (nt == 2) MGD_KR_PASSES(128, 2);
      else MGD_KR_PASSES(128, 4);
    } else {
      if (nt == 1) MGD_KR_PASSES(64, 1);
      else if (nt == 2) MGD_KR_PASSES(64, 2);
      else MGD_KR_PASSES(64, 4);
    }
#undef MGD_KR_PASSES
#undef MGD_KR
  } else {
    if (p.RG > 1) {
      e = cudaMemsetAsync(ws + p.off_scores, 0, p.off_pooled - p.off_scores, a.stream);
      if (e != cudaSuccess) return e;
    }
    const int units = p.pairs * p.RG * p.nchunk;
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q_win);
#define MGD_SCORE(DD, PP)                                                                                   \
  do {                                                                                                      \
    auto kern = snap_score_tc<DD, PP>;                                                                      \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ScoreLayout<DD>::alloc);    \
    if (e != cudaSuccess) return e;                                                                         \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,                          \
                             cudaSharedmemCarveoutMaxShared);                                               \
    if (e != cudaSuccess) return e;                                                                         \
    kern<<<units, kScoreThreads, ScoreLayout<DD>::alloc, a.stream>>>(*kmap, q, a.kv_len, ws, kp);           \
    e = cudaGetLastError();                                                                                 \
    if (e != cudaSuccess) return e;                                                                         \
  } while (0)
    if (p.D == 128) {
      MGD_SCORE(128, 1);
      MGD_SCORE(128, 2);
    } else {
      MGD_SCORE(64, 1);
      MGD_SCORE(64, 2);
    }
#undef MGD_SCORE
  }
  SelParams sp;
  sp.Hkv = p.Hkv;
  sp.W = p.W;
  sp.pool = a.pool;
  sp.K = a.K;
  sp.Kb = a.budgets;
  sp.kv_cap = p.kv_cap;
  sp.draft_cap = a.draft_cap;
  sp.row_bytes = p.D * (in_f32 ? 4 : 2);
  sp.bstride_bytes = a.kv_batch_stride * (in_f32 ? 4 : 2);
  sp.hstride_bytes = a.kv_head_stride * (in_f32 ? 4 : 2);
  sp.off_cnt = p.off_cnt;
  sp.expect_claims = tc05 ? static_cast<unsigned>(p.pairs * p.nchunk) : 0u;
  return launch_pdl(snap_select, dim3(p.pairs), dim3(kSelThreads), 0, a.stream, static_cast<const unsigned char *>(a.k),
                    static_cast<const unsigned char *>(a.v), a.kv_len, sp, a.sel_idx,
                    static_cast<unsigned char *>(a.k_draft), static_cast<unsigned char *>(a.v_draft), a.draft_len,
                    a.scores_out, ws, p.off_scores, p.off_pooled);
}

}  // namespace mgd
