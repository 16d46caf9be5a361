// SnapKV window scores on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// MagicDec notes, section 4.4 (SnapKV as the static selector) and appendix A.1
// (selection at prefill).  Steps 1 of the selection (see snapkv.cu): the W
// window queries of a KV head (W * G = 128 rows) attend causally over the
// context; pass 1 gets each row's log-sum-exp, pass 2 sums each prefix key's
// probabilities over the 128 rows.  Both passes are dense contractions
// (2 * 128 * D flop per key), so they run as tcgen05.mma with M = N = 128:
//
//   pass 1: S  = Qw K^T   (TMEM lane = window row, column = key): every thread
//           owns one row and keeps its own online max / sum -- no shuffles;
//   pass 2: S^T = K Qw^T  (TMEM lane = key, column = window row): every thread
//           owns one key and sums exp2(s - lse_row) over the rows in registers.
//
// CTA = 10 warps: warp 0 issues TMA (the 128 window rows once, then 128-key K
// tiles into a 2-stage ring), warp 1 owns the TMEM allocation and one thread
// issues the MMAs (8 k-steps of K = 16 per tile) into a double-buffered
// 2 x 128-column fp32 accumulator, warps 2..9 drain it (tcgen05.ld) as two
// groups of 4 warps taking alternate tiles, one warp per TMEM lane quadrant.
// Operands are K-major bf16 with 128-byte swizzling, exactly the layout TMA
// writes.  Used when W * G == 128 and D == 128 (the Llama-3.1-8B shape with a
// 32-row window); other shapes use the mma.sync kernel in snapkv.cu.
#include "common.cuh"

namespace mgd {
namespace {

constexpr int kT5Keys = 128;
constexpr int kT5Stages = 2;
constexpr int kT5Threads = 320;
constexpr int kT5SoftWarps = 8;
constexpr int kT5Half = 128 * 128;          // one 64-column (128 B) atom column of 128 rows
constexpr int kT5TileBytes = 2 * kT5Half;   // 128 rows x 128 bf16
constexpr uint32_t kT5TmemCols = 256;       // two 128-column accumulators
constexpr float kLog2e = 1.4426950408889634f;

// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16, both
// K-major, M = 128, N = 128.
constexpr uint32_t kIdescM128N128 = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

struct T5Layout {
  static constexpr int off_q = 0;                                   // 32 KB window rows
  static constexpr int off_k = kT5TileBytes;                        // kT5Stages x 32 KB
  static constexpr int off_bar = off_k + kT5Stages * kT5TileBytes;  // 16 mbarriers
  static constexpr int off_tmem = off_bar + 16 * 8;
  static constexpr int off_lse = off_tmem + 16;                     // float [128]
  static constexpr int off_red = off_lse + 128 * 4;                 // float [2][128]
  static constexpr int bytes = off_red + 2 * 128 * 4;
  static constexpr int alloc = bytes + 1024;
};

struct T5Params {
  int W, G, Hq, Hkv, C, nchunk, kv_cap;
  float sl2;
  size_t off_part, off_scores;
};

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

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int PASS>
__global__ void __launch_bounds__(kT5Threads, 2)
    snap_score_tc05(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                    const int32_t *__restrict__ kv_len, unsigned char *__restrict__ ws, T5Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + T5Layout::off_bar);
  uint64_t *q_full = bars + 0;
  uint64_t *full = bars + 1;          // [kT5Stages]
  uint64_t *empty = bars + 3;         // [kT5Stages]
  uint64_t *acc_full = bars + 5;      // [2]
  uint64_t *acc_empty = bars + 7;     // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + T5Layout::off_tmem);
  float *sm_lse = reinterpret_cast<float *>(smem + T5Layout::off_lse);
  float *sm_red = reinterpret_cast<float *>(smem + T5Layout::off_red);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  float2 *part = reinterpret_cast<float2 *>(ws + p.off_part);
  float *scores = reinterpret_cast<float *>(ws + p.off_scores);

  const int chunk = blockIdx.x % p.nchunk;
  const int pair = blockIdx.x / p.nchunk;
  const int hkv = pair % p.Hkv;
  const int b = pair / p.Hkv;
  const int L = kv_len[b];
  if (L < p.W || L > p.kv_cap) {
    if (threadIdx.x == 0 && chunk == 0 && hkv == 0) raise_error(hdr, 0x2u);
    return;
  }
  const int kend = (PASS == 1) ? L : L - p.W;
  const int start = chunk * p.C;
  if (start >= kend) return;
  const int end = min(start + p.C, kend);
  const int ntiles = (end - start + kT5Keys - 1) / kT5Keys;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kT5Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kT5SoftWarps / 2);  // the 4 warps of the group draining buffer a
    }
    fence_mbar_init();
  }
  if (warp == 1) {  // the whole warp allocates the accumulator columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kT5TmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (PASS == 2 && threadIdx.x >= 64 && threadIdx.x < 64 + 128) {
    // log2-sum-exp of each window row from the pass-1 partials of all chunks
    const int r = threadIdx.x - 64;
    const int nch1 = (L + p.C - 1) / p.C;
    const float2 *pp = part + static_cast<size_t>(pair) * p.nchunk * 128 + r;
    float M = -INFINITY;
    for (int c = 0; c < nch1; ++c) M = fmaxf(M, pp[c * 128].x);
    float S = 0.f;
    for (int c = 0; c < nch1; ++c) {
      const float2 x = pp[c * 128];
      if (x.y > 0.f) S += x.y * exp2f(x.x - M);
    }
    sm_lse[r] = M + log2f(S);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      mbar_arrive_expect_tx(q_full, kT5TileBytes);
      for (int h = 0; h < 2; ++h)
        tma_load_4d(smem + T5Layout::off_q + h * kT5Half, &qmap, q_full, 64 * h, hkv * p.G, 0, b);
      int stage = 0;
      uint32_t phase = 0;
      for (int t = 0; t < ntiles && ok; ++t) {
        if (!mbar_wait(&empty[stage], phase ^ 1u)) {
          raise_error(hdr, 0x8u);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], kT5TileBytes);
        unsigned char *st = smem + T5Layout::off_k + stage * kT5TileBytes;
        for (int h = 0; h < 2; ++h)
          for (int kh = 0; kh < 2; ++kh)
            tma_load_4d(st + h * kT5Half + kh * 8192, &kmap, &full[stage], 64 * h, start + t * kT5Keys + 64 * kh, hkv,
                        b);
        if (++stage == kT5Stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      if (!mbar_wait(q_full, 0)) {
        raise_error(hdr, 0x8u);
        ok = false;
      }
      const uint32_t q_base = smem_addr(smem + T5Layout::off_q);
      int stage = 0;
      uint32_t phase = 0;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int a = t & 1;
        const uint32_t aph = (t >> 1) & 1u;
        if (!mbar_wait(&full[stage], phase) || !mbar_wait(&acc_empty[a], aph ^ 1u)) {
          raise_error(hdr, 0x8u);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_base = smem_addr(smem + T5Layout::off_k + stage * kT5TileBytes);
        const uint32_t a_base = (PASS == 1) ? q_base : k_base;
        const uint32_t b_base = (PASS == 1) ? k_base : q_base;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kT5Half + (kk & 3) * 32;
          umma_f16(tmem + a * 128, umma_desc(a_base + off), umma_desc(b_base + off), kIdescM128N128, kk > 0 ? 1u : 0u);
        }
        umma_commit(&empty[stage]);
        umma_commit(&acc_full[a]);
        if (++stage == kT5Stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax warps
    // Two groups of 4 warps take alternate tiles (group g drains accumulator
    // buffer g); warp w of a group reads TMEM lane quadrant w % 4, all 128
    // columns of its lane, in two halves of 64.
    const int qd = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int tl = qd * 32 + lane;  // this thread's TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(qd * 32) << 16) + grp * 128;
    float m_run = -INFINITY, l_run = 0.f;                     // pass 1, exp2 domain
    const int pos = (PASS == 1) ? (L - p.W + tl / p.G) : 0;  // last key visible to window row tl
    for (int t = grp; t < ntiles; t += 2) {
      if (!mbar_wait(&acc_full[grp], (t >> 1) & 1u)) {
        raise_error(hdr, 0x8u);
        break;
      }
      tc_fence_after();
      const int kt0 = start + t * kT5Keys;
      float acc2 = 0.f;  // pass 2: this key's probability sum
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[2][32];
        tmem_ld32(lane_addr + h * 64, v[0]);
        tmem_ld32(lane_addr + h * 64 + 32, v[1]);
        if (h == 1) {  // both halves are in registers: hand the buffer back to the MMA thread
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[grp]);
        }
        if (PASS == 1) {
          // row tl, keys kt0 + 64h + c; the window rows see every key before L - W
          if (kt0 + kT5Keys - 1 > L - p.W) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (kt0 + 64 * h + 32 * i + c > pos) v[i][c] = -INFINITY;
          }
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int c = 0; c < 32; ++c) mx = fmaxf(mx, v[i][c]);
          const float mn = fmaxf(m_run, mx * p.sl2);  // sl2 > 0: the max commutes with the scale
          const float mu = (mn == -INFINITY) ? 0.f : mn;
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int c = 0; c < 32; ++c) acc += ex2(fmaf(v[i][c], p.sl2, -mu));
          l_run = l_run * ex2(m_run - mu) + acc;
          m_run = mn;
        } else {
          // key kt0 + tl, window rows 64h + c
#pragma unroll
          for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
              const float4 lr = *reinterpret_cast<const float4 *>(&sm_lse[64 * h + 32 * i + c]);
              acc2 += ex2(fmaf(v[i][c], p.sl2, -lr.x)) + ex2(fmaf(v[i][c + 1], p.sl2, -lr.y)) +
                      ex2(fmaf(v[i][c + 2], p.sl2, -lr.z)) + ex2(fmaf(v[i][c + 3], p.sl2, -lr.w));
            }
        }
      }
      if (PASS == 2) {
        const int key = kt0 + tl;
        if (key < end) scores[(static_cast<size_t>(b) * p.Hkv + hkv) * p.kv_cap + key] = acc2;
      }
    }
    if (PASS == 1) {
      // combine the two groups' (max, sum) of each row, then write this chunk's partial
      if (grp == 1) {
        sm_red[tl] = m_run;
        sm_red[128 + tl] = l_run;
      }
      named_bar(1, kT5SoftWarps * 32);
      if (grp == 0) {
        const float m2 = sm_red[tl], l2 = sm_red[128 + tl];
        const float mn = fmaxf(m_run, m2);
        const float mu = (mn == -INFINITY) ? 0.f : mn;
        const float l = l_run * exp2f(m_run - mu) + l2 * exp2f(m2 - mu);
        part[(static_cast<size_t>(pair) * p.nchunk + chunk) * 128 + tl] = make_float2(mn, l);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kT5TmemCols) : "memory");
  }
}

}  // namespace

bool snap_tc05_eligible(const SnapPlan &p) { return p.D == 128 && p.rows == 128 && p.RG == 1 && p.C % 128 == 0; }

cudaError_t launch_snap_score_tc05(const SnapPlan &pl, const SnapArgs &a, const CUtensorMap &kmap,
                                   const CUtensorMap &qmap) {
  T5Params kp;
  kp.W = pl.W;
  kp.G = pl.G;
  kp.Hq = pl.Hq;
  kp.Hkv = pl.Hkv;
  kp.C = pl.C;
  kp.nchunk = pl.nchunk;
  kp.kv_cap = pl.kv_cap;
  kp.sl2 = a.sm_scale * kLog2e;
  kp.off_part = pl.off_part;
  kp.off_scores = pl.off_scores;
  const int units = pl.pairs * pl.nchunk;
  unsigned char *ws = static_cast<unsigned char *>(a.ws);
  cudaError_t e;
#define MGD_T5(PP)                                                                                            \
  do {                                                                                                        \
    auto kern = snap_score_tc05<PP>;                                                                          \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T5Layout::alloc);             \
    if (e != cudaSuccess) return e;                                                                           \
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,                            \
                             cudaSharedmemCarveoutMaxShared);                                                 \
    if (e != cudaSuccess) return e;                                                                           \
    kern<<<units, kT5Threads, T5Layout::alloc, a.stream>>>(kmap, qmap, a.kv_len, ws, kp);                     \
    e = cudaGetLastError();                                                                                   \
    if (e != cudaSuccess) return e;                                                                           \
  } while (0)
  MGD_T5(1);
  MGD_T5(2);
#undef MGD_T5
  return cudaSuccess;
}

}  // namespace mgd
